// Split-KV planner: assigns contiguous stretches of (work block, 64-token tile)
// work to units, splitting long sequences across units.  A work block is a group
// of G consecutive new tokens of one sequence (G = 1: one query block; G > 1: the
// G tokens share every page, one CTA pair per token in a cluster of 2G CTAs); its
// tiles are those of its last token, which sees the most keys.
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
constexpr int kTile = 64;                     // tokens per work tile (one page)
// Cost of one piece of work beyond its tiles, in tile units: loading the
// 128 x 288 query half, the epilogue writing the 128 x 256 output half, and the
// pipeline refill between pieces -- measured at about six tiles' time per piece
// boundary on GB300 (the plan balances positions, so this is what evens the units).
#ifndef MLA_PIECE_COST
#define MLA_PIECE_COST 6
#endif
constexpr int kPieceFixedCost = MLA_PIECE_COST;

// Keys query token t of a sequence of length L sees.  A negative length (outside the
// contract; the scheduler kernel reports it) sees none.
MLA_HD inline int32_t visible_keys(int32_t L, int s_q, int t, int causal) {
  int32_t n = causal ? L - s_q + 1 + t : L;
  if (n > L) n = L;
  if (n < 0) n = 0;
  return n;
}

MLA_HD inline int32_t num_tiles(int32_t visible) { return (visible + kTile - 1) / kTile; }

// Tiles of work block blk (tokens blk*G .. blk*G + G - 1 of the flattened [B][s_q] order):
// those of its last token.
MLA_HD inline int32_t block_tiles(const int32_t* seqlens, int s_q, int causal, int G, int blk) {
  const int qb_last = blk * G + G - 1;
  return num_tiles(visible_keys(seqlens[qb_last / s_q], s_q, qb_last % s_q, causal));
}

MLA_HD inline int64_t sched_ints(int num_units, int num_qb) {
  return kSchedHeader + (int64_t)kUnitInts * num_units + 2 * (int64_t)num_qb;
}

// Work positions.  Work blocks are laid out one after another on a line of
// cost units: block qb occupies [pos[qb], pos[qb] + kPieceFixedCost + nt[qb]),
// its first kPieceFixedCost units standing for the per-piece overhead and then
// one unit per 64-token tile (tile t at pos[qb] + kPieceFixedCost + t).  With
// B = ceil(total / U), unit u owns the tiles whose positions fall in
// [u*B, (u+1)*B).  Everything below follows in closed form, so the device runs
// each phase in parallel (the prefix sums on one thread).
//
// Phase 1 (per work block): nt[qb] and cost.  (In this and the next phases qb indexes work
// blocks, NQB counts them.)
MLA_HD inline void plan_phase_cost(const int32_t* seqlens, int s_q, int causal, int G, int NQB, int32_t* cost,
                                   int begin, int stride) {
  for (int qb = begin; qb < NQB; qb += stride) {
    const int32_t nt = block_tiles(seqlens, s_q, causal, G, qb);
    cost[qb] = nt > 0 ? nt + kPieceFixedCost : 0;
  }
}

// Largest total of cost positions a plan may have: positions are stored as int32.
constexpr int64_t kMaxPlanPositions = 0x7FFFFFFF;

// Phase 2 (one thread): exclusive prefix sum of cost -> pos (in place); returns the total.
// A total above kMaxPlanPositions leaves pos unusable: the callers then refuse the plan.
MLA_HD inline int64_t plan_phase_scan(int32_t* cost_to_pos, int NQB) {
  int64_t acc = 0;
  for (int qb = 0; qb < NQB; ++qb) {
    const int64_t c = cost_to_pos[qb];
    cost_to_pos[qb] = (int32_t)acc;
    acc += c;
  }
  return acc;
}

MLA_HD inline int64_t plan_budget(int64_t total, int U) {
  int64_t B = (total + U - 1) / U;
  return B < 1 ? 1 : B;
}

// Phase 3 (per unit): the unit record.  pos[] = block start positions.
MLA_HD inline void plan_phase_units(const int32_t* seqlens, int s_q, int causal, int G, int NQB, const int32_t* pos,
                                    int64_t total, int64_t B, int U, int32_t* units, int begin, int stride) {
  for (int u = begin; u < U; u += stride) {
    int32_t* rec = units + kUnitInts * u;
    rec[0] = -1;
    rec[1] = rec[2] = rec[3] = rec[4] = rec[5] = rec[6] = rec[7] = 0;
    const int64_t lo = (int64_t)u * B, hi = lo + B;  // tile positions [lo, hi)
    if (lo >= total) continue;
    // first block whose last tile position >= lo
    int a = 0, b = NQB;
    while (a < b) {
      const int m = (a + b) / 2;
      const int32_t nt = block_tiles(seqlens, s_q, causal, G, m);
      const int64_t last = (int64_t)pos[m] + kPieceFixedCost + nt - 1;
      if (nt > 0 && last >= lo) b = m; else if (nt == 0 && (int64_t)pos[m] > lo) b = m; else a = m + 1;
    }
    // skip empty blocks
    int qb0 = a;
    while (qb0 < NQB && block_tiles(seqlens, s_q, causal, G, qb0) == 0) ++qb0;
    if (qb0 >= NQB) continue;
    const int64_t first0 = (int64_t)pos[qb0] + kPieceFixedCost;
    if (first0 >= hi) continue;  // the range holds only overhead positions
    // last block whose first tile position < hi
    a = qb0;
    b = NQB;
    while (b - a > 1) {
      const int m = (a + b) / 2;
      if ((int64_t)pos[m] + kPieceFixedCost < hi) a = m; else b = m;
    }
    int qb1 = a;
    while (qb1 > qb0 && block_tiles(seqlens, s_q, causal, G, qb1) == 0) --qb1;
    const int32_t nt1 = block_tiles(seqlens, s_q, causal, G, qb1);
    const int64_t t_begin = lo - first0 > 0 ? lo - first0 : 0;
    int64_t t_end = hi - ((int64_t)pos[qb1] + kPieceFixedCost);
    if (t_end > nt1) t_end = nt1;
    const int64_t fu = first0 / B;  // first unit holding a tile of qb0
    rec[0] = qb0;
    rec[1] = (int32_t)t_begin;
    rec[2] = qb1;
    rec[3] = (int32_t)t_end;
    rec[4] = (int32_t)(u - fu);
  }
}

// Phase 4 (per work block): number of units its tiles span, written for each of its G query
// blocks (num_splits is indexed by query block).
MLA_HD inline void plan_phase_splits(const int32_t* seqlens, int s_q, int causal, int G, int NQB, const int32_t* pos,
                                     int64_t B, int32_t* num_splits, int begin, int stride) {
  for (int qb = begin; qb < NQB; qb += stride) {
    const int32_t nt = block_tiles(seqlens, s_q, causal, G, qb);
    int32_t n = 0;
    if (nt > 0) {
      const int64_t first = (int64_t)pos[qb] + kPieceFixedCost;
      n = (int32_t)((first + nt - 1) / B - first / B + 1);
    }
    for (int g = 0; g < G; ++g) num_splits[qb * G + g] = n;
  }
}

// Phase 5 (one thread): slots of the split partials (per query block); header.
MLA_HD inline void plan_phase_finish(int NQB, int U, int G, int64_t B, int32_t* sched) {
  int32_t* num_splits = sched + kSchedHeader + kUnitInts * U;
  int32_t* split_offset = num_splits + NQB;
  int32_t slots = 0;
  for (int qb = 0; qb < NQB; ++qb) {
    split_offset[qb] = slots;
    if (num_splits[qb] > 1) slots += num_splits[qb];
  }
  sched[0] = kSchedMagic;
  sched[1] = U;
  sched[2] = NQB;
  sched[3] = slots;
  sched[4] = (int32_t)B;  // per-unit budget of positions (diagnostic)
  sched[5] = G;           // tokens per work block
  sched[6] = sched[7] = 0;
}

// A refused plan: a header without the magic word, which the decode and combine kernels
// recognise as invalid metadata (they then write nothing).
MLA_HD inline void plan_refuse(int32_t* sched) {
  for (int i = 0; i < kSchedHeader; ++i) sched[i] = 0;
}

// Host twin: all phases in order, one "thread".  The split_offset region of
// sched serves as scratch for the block positions until phase 5 fills it.
// G divides s_q.  Returns false (and writes a refused header) when the lengths
// need more cost positions than an int32 holds.
MLA_HD inline bool plan_units(const int32_t* seqlens, int B_, int s_q, int causal, int G, int U, int32_t* sched) {
  const int NQB = B_ * s_q, NWB = NQB / G;
  int32_t* units = sched + kSchedHeader;
  int32_t* num_splits = units + kUnitInts * U;
  int32_t* pos = num_splits + NQB;
  plan_phase_cost(seqlens, s_q, causal, G, NWB, pos, 0, 1);
  const int64_t total = plan_phase_scan(pos, NWB);
  if (total > kMaxPlanPositions) {
    plan_refuse(sched);
    return false;
  }
  const int64_t B = plan_budget(total, U);
  plan_phase_units(seqlens, s_q, causal, G, NWB, pos, total, B, U, units, 0, 1);
  plan_phase_splits(seqlens, s_q, causal, G, NWB, pos, B, num_splits, 0, 1);
  plan_phase_finish(NQB, U, G, B, sched);
  return true;
}

}  // namespace mla
