// Split-KV planner: assigns contiguous stretches of (query block, 64-token tile)
// work to units (one 2-SM cluster each), splitting long sequences across units.
// The same function runs in the scheduler kernel (one thread) and on the host
// (mla_plan_host), so the CPU tests exercise exactly the device algorithm.
//
// Background: "MLA inference: two computation paths and FlashMLA", section
// "Decode attention becomes a compute problem" -- with long contexts and small
// batches the KV dimension is split across SMs and the partial results are
// merged; the split plan is precomputed from the context lengths.
#pragma once
#include <cstdint>

#ifndef MLA_HD
#ifdef __CUDACC__
#define MLA_HD __host__ __device__
#else
#define MLA_HD
#endif
#endif

namespace mla {

constexpr int32_t kSchedMagic = 0x4D4C4131;  // "MLA1"
constexpr int kSchedHeader = 8;               // int32 header words
constexpr int kUnitInts = 8;                  // int32 words per unit record
constexpr int kTile = 128;                    // tokens per work tile (two 64-token pages)
// Cost of one piece of work beyond its tiles, in tile units: loading the
// query half and writing the 128 x 256 output half (about one tile of bytes).
constexpr int kPieceFixedCost = 1;

MLA_HD inline int32_t visible_keys(int32_t L, int s_q, int t, int causal) {
  int32_t n = causal ? L - s_q + 1 + t : L;
  if (n < 0) n = 0;
  if (n > L) n = L;
  return n;
}

MLA_HD inline int32_t num_tiles(int32_t visible) { return (visible + kTile - 1) / kTile; }

MLA_HD inline int64_t sched_ints(int num_units, int num_qb) {
  return kSchedHeader + (int64_t)kUnitInts * num_units + 2 * (int64_t)num_qb;
}

// Greedy pass with a per-unit cost budget: walks query blocks in order, filling
// unit after unit; a piece (one query block's tile range inside one unit) costs
// its tiles plus kPieceFixedCost.  Returns false if the work needs more than U
// units.  With write == true it also fills the unit records and num_splits.
MLA_HD inline bool plan_pass(const int32_t* seqlens, int B, int s_q, int causal, int U, int64_t budget, bool write,
                             int32_t* units, int32_t* num_splits) {
  const int NQB = B * s_q;
  int u = 0;
  bool unit_used = false;
  int64_t room = budget;
  for (int qb = 0; qb < NQB; ++qb) {
    const int32_t nt = num_tiles(visible_keys(seqlens[qb / s_q], s_q, qb % s_q, causal));
    int32_t tile = 0, splits = 0;
    while (tile < nt) {
      if (unit_used && room <= kPieceFixedCost) {  // no useful room left: next unit
        if (++u == U) return false;
        room = budget;
        unit_used = false;
      }
      int64_t take = nt - tile;
      if (take > room - kPieceFixedCost) take = room - kPieceFixedCost;
      if (write) {
        int32_t* rec = units + kUnitInts * u;
        if (!unit_used) {
          rec[0] = qb;
          rec[1] = tile;
          rec[4] = splits;
        }
        rec[2] = qb;
        rec[3] = tile + (int32_t)take;
      }
      unit_used = true;
      ++splits;
      tile += (int32_t)take;
      room -= take + kPieceFixedCost;
    }
    if (write) num_splits[qb] = splits;
  }
  return true;
}

// Fills sched (sched_ints(U, B*s_q) int32 words).  Query block qb = b*s_q + t.
// Units hold contiguous ranges in (qb, tile) order; every non-empty query block
// is covered exactly once; a piece never holds zero tiles.  The budget is the
// smallest per-unit cost with which the greedy pass fits in U units (binary
// search; feasibility only improves with a larger budget).
MLA_HD inline void plan_units(const int32_t* seqlens, int B, int s_q, int causal, int U, int32_t* sched) {
  const int NQB = B * s_q;
  int32_t* units = sched + kSchedHeader;
  int32_t* num_splits = units + kUnitInts * U;
  int32_t* split_offset = num_splits + NQB;
  for (int u = 0; u < U; ++u) {
    int32_t* rec = units + kUnitInts * u;
    rec[0] = -1;
    rec[1] = rec[2] = rec[3] = rec[4] = rec[5] = rec[6] = rec[7] = 0;
  }
  for (int qb = 0; qb < NQB; ++qb) num_splits[qb] = 0;
  int64_t total = 0;
  for (int qb = 0; qb < NQB; ++qb) {
    int32_t nt = num_tiles(visible_keys(seqlens[qb / s_q], s_q, qb % s_q, causal));
    if (nt > 0) total += nt + kPieceFixedCost;
  }
  int64_t lo = (total + U - 1) / U;
  if (lo < kPieceFixedCost + 1) lo = kPieceFixedCost + 1;
  int64_t hi = total + kPieceFixedCost + 1;  // one unit takes everything
  if (hi < lo) hi = lo;
  while (lo < hi) {
    const int64_t mid = lo + (hi - lo) / 2;
    if (plan_pass(seqlens, B, s_q, causal, U, mid, false, units, num_splits))
      hi = mid;
    else
      lo = mid + 1;
  }
  plan_pass(seqlens, B, s_q, causal, U, lo, true, units, num_splits);
  int32_t slots = 0;
  for (int qb = 0; qb < NQB; ++qb) {
    split_offset[qb] = slots;
    if (num_splits[qb] > 1) slots += num_splits[qb];
  }
  sched[0] = kSchedMagic;
  sched[1] = U;
  sched[2] = NQB;
  sched[3] = slots;
  sched[4] = (int32_t)lo;  // per-unit budget (diagnostic)
  sched[5] = sched[6] = sched[7] = 0;
}

}  // namespace mla
