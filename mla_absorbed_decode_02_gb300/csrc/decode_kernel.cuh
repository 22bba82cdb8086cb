// Absorbed-MLA decode kernel for sm_103a (tcgen05 + TMA + 2-SM clusters).
//
// Work split.  One work unit = one 2-CTA cluster (two SMs) walking a contiguous
// stretch of (query block, 64-token tile) work from the split plan.  CTA h of
// the pair ("half" h) owns
//   * dims [256h, 256h+256) of the latent and dims [32h, 32h+32) of the RoPE
//     key of every cached token -- it loads only those, one page (64 tokens)
//     per tile, with TMA through the block table (paged gather);
//   * output latent dims [256h, 256h+256): a 128-head x 256 fp32 accumulator
//     in tensor memory.
// Scores need all 576 dims, so each CTA computes a partial score over its 288
// dims (tcgen05.mma, M = 128 heads, N = 64 tokens; the absorbed-query half is
// the A operand in tensor memory, the RoPE-query half in shared memory), and
// the two CTAs swap partial scores through distributed shared memory
// (st.async), encoded as 16-bit block floating point -- one shared exponent per
// (head, 32-token chunk), 16-bit signed mantissas.  Each CTA adds the peer's
// rounded half to its own exact half, runs the online softmax for its output
// half (one thread per head row and 32-token chunk), writes P (bf16) to shared
// memory, and accumulates O_half += P V_half (tcgen05.mma, N = 256, V read
// MN-major from the same shared-memory page the score used).
//
// "MLA inference: two computation paths and FlashMLA", section "Decode
// attention becomes a compute problem": the 128 heads are the M dimension of
// the matrix multiply, a block of KV is staged in shared memory, long
// sequences are split across SMs and merged through their LSE.
//
// Pipelining.  Four 36 KB shared-memory stages (a page stays resident from its
// load through QK, softmax and PV, because the latent is key and value at
// once); two score buffers in tensor memory; two exchange slots per chunk.  The
// MMA warp issues QK ahead of PV.  The softmax warps run one tile ahead on the
// exchange: while they receive tile i and turn it into P, they already encode
// and send tile i+1.
//
// Warp roles (384 threads): warp 0 = TMA producer, warp 1 = MMA issuer,
// warp 2 = tensor-memory allocator, warp 3 idle, warps 4..11 = softmax /
// exchange / epilogue in two warpgroups, one per 32-token half of a tile
// (thread = head row = TMEM lane).
#pragma once
#include "common.cuh"

namespace mla {

constexpr int kThreads = 384;
constexpr int kRows = 128;      // MMA M: head rows (H <= 128, padded with zero queries)
constexpr int kTileTok = 64;    // tokens per work tile (one page)
constexpr int kStages = 4;
constexpr int kChunks = 2;      // 32-token exchange chunks per tile

// shared memory layout (offsets from a 1024-byte aligned base)
constexpr uint32_t kLatBlock = 8192;                  // [64 rows x 128 B]: 64 latent dims of a page
constexpr uint32_t kStageRope = 4 * kLatBlock;        // RoPE half [64 rows x 64 B]
constexpr uint32_t kStageBytes = kStageRope + 4096;   // 36 KB
constexpr uint32_t SM_P = kStages * kStageBytes;      // P: [128 rows x 128 B] bf16, 128-byte swizzle
constexpr uint32_t SM_QR = SM_P + 16384;              // RoPE-query half [128 x 64 B], 64-byte swizzle
constexpr uint32_t SM_X = SM_QR + 8192;               // peer partial scores: [slot][chunk][4][128 rows][16 B]
constexpr uint32_t SM_XE = SM_X + 2 * kChunks * 8192; // peer exponents: [slot][chunk][128 rows] int32
constexpr uint32_t SM_MX = SM_XE + 2 * kChunks * 512; // chunk maxima [2][2][128] f32 + row sums [2][128] f32
constexpr uint32_t SM_BAR = SM_MX + 4096;
constexpr uint32_t kSmemBytes = SM_BAR + 512 + 1024;  // + alignment slack
constexpr uint32_t kXChunkBytes = kRows * (64 + 4);   // bytes one CTA sends the other per chunk

// tensor memory columns
constexpr uint32_t TM_O = 0, TM_S = 256, TM_Q = 384;  // S buffers at 256 and 320

// barrier slots (8 bytes each) inside SM_BAR
enum : uint32_t {
  B_QR_FULL = 0,
  B_QR_EMPTY,
  B_QT_FULL,
  B_P_FULL,
  B_PV_DONE,
  B_DRAIN,
  B_MX,
  B_EPI,
  B_KV_FULL,                        // + stage
  B_KV_EMPTY = B_KV_FULL + kStages,
  B_S_FULL = B_KV_EMPTY + kStages,  // + buffer
  B_S_EMPTY = B_S_FULL + 2,
  B_X_FULL = B_S_EMPTY + 2,         // + 2 * slot + chunk
  B_X_FREE = B_X_FULL + 2 * kChunks,
  kNumBars = B_X_FREE + 2 * kChunks
};
constexpr uint32_t OFF_TMEM_SLOT = kNumBars * 8;
constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4;
static_assert(OFF_ABORT + 4 <= 512, "barrier area");

struct Piece {
  int qb, t0, t1, split;
};

// Walks the pieces (query block, tile range) of one unit record.
struct PieceWalker {
  const int32_t* seqlens;
  int s_q, causal, first_qb, qb, qb_end, tile_begin, tile_end, first_split;
  __device__ bool next(Piece& p) {
    while (qb <= qb_end) {
      const int cur = qb++;
      const int nt = num_tiles(visible_keys(seqlens[cur / s_q], s_q, cur % s_q, causal));
      const int a = (cur == first_qb) ? tile_begin : 0;
      const int b = (cur == qb_end) ? tile_end : nt;
      if (nt > 0 && a < b) {
        p.qb = cur;
        p.t0 = a;
        p.t1 = b;
        p.split = (cur == first_qb) ? first_split : 0;
        return true;
      }
    }
    return false;
  }
};

struct TileInfo {
  int qb, tile, valid, split;
  bool first, last;
};

// Walks the tiles of a unit in order, across its pieces.
struct TileCursor {
  PieceWalker w;
  Piece pc;
  int t, vis;
  bool open;
  __device__ void init(const PieceWalker& pw) {
    w = pw;
    open = false;
  }
  __device__ bool next(TileInfo& ti) {
    if (!open || t >= pc.t1) {
      if (!w.next(pc)) return false;
      open = true;
      t = pc.t0;
      vis = visible_keys(w.seqlens[pc.qb / w.s_q], w.s_q, pc.qb % w.s_q, w.causal);
    }
    ti.qb = pc.qb;
    ti.tile = t;
    ti.valid = min(kTileTok, vis - t * kTileTok);
    ti.split = pc.split;
    ti.first = (t == pc.t0);
    ti.last = (t == pc.t1 - 1);
    ++t;
    return true;
  }
};

__device__ __forceinline__ float pow2f(int p) { return __int_as_float((127 + p) << 23); }  // p in [-126, 127]

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Exponent e (clamped) with |x| < 2^e for the largest |x| of a chunk; the
// 16-bit mantissa of x is then rint(x * 2^(15-e)).
__device__ __forceinline__ int bfp_exponent(float amax) {
  int e = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 126;
  e = e < -60 ? -60 : e;
  e = e > 110 ? 110 : e;
  return e;
}

// Two scaled scores -> two int16 mantissas (round to nearest even, saturating) in one word.
__device__ __forceinline__ uint32_t bfp_pack2(float a, float b) {
  uint32_t w;
  asm("{\n\t.reg .s16 lo, hi;\n\t"
      "cvt.rni.sat.s16.f32 lo, %1;\n\t"
      "cvt.rni.sat.s16.f32 hi, %2;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(w)
      : "f"(a), "f"(b));
  return w;
}
__device__ __forceinline__ void bfp_unpack2(uint32_t w, float& a, float& b) {
  asm("{\n\t.reg .s16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f32.s16 %0, lo;\n\t"
      "cvt.rn.f32.s16 %1, hi;\n\t}"
      : "=f"(a), "=f"(b)
      : "r"(w));
}

__device__ __forceinline__ void st_async_b32(uint32_t cluster_dst, uint32_t v, uint32_t cluster_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(cluster_dst), "r"(v),
               "r"(cluster_bar)
               : "memory");
}

__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_bf16_kernel(const __grid_constant__ DecodeArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t base = smem_addr(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t half = cluster_ctarank(), peer = half ^ 1;
  const int unit = blockIdx.x >> 1;

  // ---- unit record (uniform across the cluster); bail out early on bad metadata
  const int32_t* sched = args.sched;
  if (sched[0] != kSchedMagic || sched[1] != args.num_units || sched[2] != args.num_qb) {
    if (tid == 0) atomicCAS(&g_mla_error, 0, 5);
    return;
  }
  const int32_t* rec = sched + kSchedHeader + kUnitInts * unit;
  if (rec[0] < 0) return;  // no work for this unit (both CTAs take this path)
  const int32_t* num_splits = sched + kSchedHeader + kUnitInts * args.num_units;
  const int32_t* split_offset = num_splits + args.num_qb;

  auto bar = [&](uint32_t i) { return base + SM_BAR + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM_BAR + OFF_ABORT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM_BAR + OFF_TMEM_SLOT);

  if (tid == 0) {
    mbar_init(bar(B_QR_FULL), 1);
    mbar_init(bar(B_QR_EMPTY), 1);
    // softmax-side barriers count one arrival per softmax warp (8), after __syncwarp
    mbar_init(bar(B_QT_FULL), 8);
    mbar_init(bar(B_P_FULL), 8);
    mbar_init(bar(B_MX), 8);
    mbar_init(bar(B_EPI), 8);
    mbar_init(bar(B_PV_DONE), 1);
    mbar_init(bar(B_DRAIN), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_KV_FULL + s), 1);
      mbar_init(bar(B_KV_EMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_S_FULL + s), 1);
      mbar_init(bar(B_S_EMPTY + s), 8);
    }
    for (int c = 0; c < 2 * kChunks; ++c) {
      mbar_init(bar(B_X_FULL + c), 1);
      mbar_init(bar(B_X_FREE + c), 4);  // one arrival per peer softmax warp of that chunk
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // peer barriers initialised before any remote arrive / st.async
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  WaitCtx wc;
  wc.abort_local = abort_flag;
  wc.abort_peer = map_to_rank(smem_addr((const void*)abort_flag), peer);
  wc.timeout_ns = args.timeout_ns;

  PieceWalker walker0;
  walker0.seqlens = args.seqlens;
  walker0.s_q = args.s_q;
  walker0.causal = args.causal;
  walker0.qb = rec[0];
  walker0.first_qb = rec[0];
  walker0.tile_begin = rec[1];
  walker0.qb_end = rec[2];
  walker0.tile_end = rec[3];
  walker0.first_split = rec[4];

  if (warp == 0) {
    // ================================================================ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&args.map_qr);
      prefetch_tensormap(&args.map_kvc);
      prefetch_tensormap(&args.map_kvr);
      const uint64_t pol_kv = l2_policy_evict_first();
      const uint64_t pol_q = l2_policy_evict_last();
      TileCursor cur;
      cur.init(walker0);
      TileInfo ti;
      uint32_t t = 0, piece_no = 0;
      while (cur.next(ti)) {
        if (ti.first) {
          if (piece_no > 0 && !wait_one(bar(B_QR_EMPTY), (piece_no - 1) & 1, wc, kSiteQEmpty)) break;
          mbar_arrive_expect_tx(bar(B_QR_FULL), 8192);
          tma_load_3d(base + SM_QR, &args.map_qr, bar(B_QR_FULL), 32 * half, 0, ti.qb, pol_q);
          ++piece_no;
        }
        const uint32_t st = t % kStages, ph = (t / kStages) & 1;
        if (!wait_one(bar(B_KV_EMPTY + st), ph ^ 1, wc, kSiteKvEmpty)) break;
        mbar_arrive_expect_tx(bar(B_KV_FULL + st), kStageBytes);
        const int b = ti.qb / args.s_q;
        const int page = args.block_table[(int64_t)b * args.max_pages + ti.tile];
        const uint32_t sbase = base + st * kStageBytes;
        for (int blk = 0; blk < 4; ++blk)
          tma_load_2d(sbase + blk * kLatBlock, &args.map_kvc, bar(B_KV_FULL + st), 256 * half + 64 * blk, page * 64,
                      pol_kv);
        tma_load_2d(sbase + kStageRope, &args.map_kvr, bar(B_KV_FULL + st), 512 + 32 * half, page * 64, pol_kv);
        ++t;
      }
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    // Order: QK(t), then PV(t-2): the scores run ahead of the PV products, so the
    // softmax warps find the next tile's scores ready when they need them.
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_bf16_f32(128, 64, 0, 0);
      constexpr uint32_t id_pv = idesc_bf16_f32(128, 256, 0, 1);
      TileCursor cur;
      cur.init(walker0);
      TileInfo ti;
      uint32_t t = 0, piece_no = 0, pv_t = 0;
      bool pv_first[4] = {false, false, false, false};  // first-of-piece flag of tile t, indexed t % 4
      bool ok = true;
      auto issue_pv = [&]() -> bool {
        if (!wait_one(bar(B_P_FULL), pv_t & 1, wc, kSitePFull)) return false;
        tc_fence_after();
        const uint32_t st = pv_t % kStages;
        const uint32_t sbase = base + st * kStageBytes;
        const bool acc = !pv_first[pv_t & 3];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t a = smem_desc(base + SM_P + k * 32, 16, 1024, kSwizzle128B);
          const uint64_t bv = smem_desc(sbase + k * 2048, kLatBlock, 1024, kSwizzle128B);
          mma_bf16_ss(tmem + TM_O, a, bv, id_pv, (acc || k > 0) ? 1u : 0u);
        }
        mma_commit(bar(B_KV_EMPTY + st));
        mma_commit(bar(B_PV_DONE));
        ++pv_t;
        return true;
      };
      while (ok && cur.next(ti)) {
        if (ti.first) {
          if (!(ok = wait_one(bar(B_QR_FULL), piece_no & 1, wc, kSiteQFull))) break;
          if (!(ok = wait_one(bar(B_QT_FULL), piece_no & 1, wc, kSiteQFull))) break;
          ++piece_no;
        }
        const uint32_t st = t % kStages, sb = t & 1;
        if (!(ok = wait_one(bar(B_KV_FULL + st), (t / kStages) & 1, wc, kSiteKvFull))) break;
        if (!(ok = wait_one(bar(B_S_EMPTY + sb), ((t >> 1) & 1) ^ 1, wc, kSiteSEmpty))) break;
        tc_fence_after();
        const uint32_t sbase = base + st * kStageBytes;
        const uint32_t d = tmem + TM_S + 64 * sb;
#pragma unroll
        for (int k = 0; k < 16; ++k)  // latent half: A = query half in tensor memory
          mma_bf16_ts(d, tmem + TM_Q + 8 * k,
                      smem_desc(sbase + (k >> 2) * kLatBlock + (k & 3) * 32, 16, 1024, kSwizzle128B), id_qk,
                      k > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < 2; ++k)  // RoPE half: A = RoPE-query half in shared memory
          mma_bf16_ss(d, smem_desc(base + SM_QR + 32 * k, 16, 512, kSwizzle64B),
                      smem_desc(sbase + kStageRope + 32 * k, 16, 512, kSwizzle64B), id_qk, 1u);
        mma_commit(bar(B_S_FULL + sb));
        if (ti.last) mma_commit(bar(B_QR_EMPTY));
        pv_first[t & 3] = ti.first;
        ++t;
        if (t >= 3 && !(ok = issue_pv())) break;  // PV(t-3) once QK(t-1) is queued
      }
      while (ok && pv_t < t) ok = issue_pv();
      // no MMA may still run when tensor memory is released
      mma_commit(bar(B_DRAIN));
      WaitCtx wd = wc;
      wd.timeout_ns = 100000000ull;
      volatile int no_abort = 0;
      wd.abort_local = &no_abort;
      wd.abort_peer = 0;
      wait_one(bar(B_DRAIN), 0, wd, kSiteDrain);
    }
  } else if (warp >= 4) {
    // ================================================================ softmax / exchange / epilogue
    // Two warpgroups; warpgroup cw handles score columns [32 cw, 32 cw + 32) of every
    // tile (one exchange chunk), O columns [128 cw, 128 cw + 128) for rescale and
    // epilogue, and query columns [64 cw, 64 cw + 64) of tensor memory.
    const int cw = (warp - 4) >> 2;                   // column group
    const int r = ((warp & 3) << 5) | lane;           // head row == TMEM lane
    const int gt = tid - 128;                         // 0..255 across both groups
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    // exchange slot (tile parity) x chunk: data at SM_X + (2 slot + cw) 8 KB, exponents at SM_XE + (2 slot + cw) 512 B
    const uint32_t peer_x = map_to_rank(base + SM_X + cw * 8192, peer);
    const uint32_t peer_xe = map_to_rank(base + SM_XE + cw * 512, peer);
    const uint32_t peer_bar0 = map_to_rank(bar(0), peer);  // the peer's barrier i is at peer_bar0 + 8 i
    const uint32_t my_x = base + SM_X + cw * 8192, my_xe = base + SM_XE + cw * 512;
    const float sl2 = args.scale_log2;
    const int H = args.H;
    bool ok = true;

    // absorbed-query columns of this group -> tensor memory (A operand of the latent score)
    auto load_q_tmem = [&](int qb) {
      uint32_t q[32];
      const uint32_t* src =
          reinterpret_cast<const uint32_t*>(args.q_nope) + ((int64_t)qb * H + r) * 256 + 128 * half + 64 * cw;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (r < H) v = *reinterpret_cast<const uint4*>(src + 32 * c + j);
          q[j] = v.x;
          q[j + 1] = v.y;
          q[j + 2] = v.z;
          q[j + 3] = v.w;
        }
        tmem_st32(tmem + lane_off + TM_Q + 64 * cw + 32 * c, q);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_QT_FULL));
    };

    PieceWalker qwalk = walker0;  // one piece ahead of the score loads: feeds the query loads
    TileCursor cursor;
    cursor.init(walker0);
    uint32_t s_t = 0;     // tiles whose scores were read
    uint32_t x_sent = 0;  // tiles sent to the peer
    uint32_t x_recv = 0;  // tiles received from the peer (== tiles processed)
    uint32_t pieces_done = 0;
    float own_c[32], own_n[32];  // this CTA's exact partial scores (current / next tile)
    uint32_t pk_n[16];           // next tile's partial scores in 16-bit block floating point
    int ex_n = 0;

    // A: this group's score columns of a tile -> registers + block-float encoding
    auto stage_a = [&](const TileInfo& x, float (&own)[32]) -> bool {
      const uint32_t sb = s_t & 1;
      if (!wait_warp(bar(B_S_FULL + sb), (s_t >> 1) & 1, wc, kSiteSFull)) return false;
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32(tmem + lane_off + TM_S + 64 * sb + 32 * cw, v);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_S_EMPTY + sb));
      ++s_t;
      const int valid = x.valid - 32 * cw;
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
      if (valid >= 32) {
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          own[j] = __uint_as_float(v[j]);
          own[j + 1] = __uint_as_float(v[j + 1]);
          own[j + 2] = __uint_as_float(v[j + 2]);
          own[j + 3] = __uint_as_float(v[j + 3]);
          a0 = fmaxf(a0, fabsf(own[j]));
          a1 = fmaxf(a1, fabsf(own[j + 1]));
          a2 = fmaxf(a2, fabsf(own[j + 2]));
          a3 = fmaxf(a3, fabsf(own[j + 3]));
        }
      } else {  // last tile of a sequence: columns past the end are sent as 0 and masked later
#pragma unroll
        for (int j = 0; j < 32; ++j) own[j] = (j < valid) ? __uint_as_float(v[j]) : 0.f;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          a0 = fmaxf(a0, fabsf(own[j]));
          a1 = fmaxf(a1, fabsf(own[j + 1]));
          a2 = fmaxf(a2, fabsf(own[j + 2]));
          a3 = fmaxf(a3, fabsf(own[j + 3]));
        }
      }
      const int e = bfp_exponent(fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)));
      ex_n = e;
      const float k = pow2f(15 - e);
#pragma unroll
      for (int u = 0; u < 16; ++u) pk_n[u] = bfp_pack2(own[2 * u] * k, own[2 * u + 1] * k);
      if (x.last) {  // the query half in tensor memory is free once the last score of its piece exists
        Piece np;
        if (qwalk.next(np)) load_q_tmem(np.qb);
      }
      return true;
    };
    // slot = tile parity, so a send only waits for the peer to have consumed the tile before last
    auto send_chunk = [&]() -> bool {
      const uint32_t slot = x_sent & 1;
      if (!wait_warp(bar(B_X_FREE + 2 * slot + cw), ((x_sent >> 1) & 1) ^ 1, wc, kSiteXFree)) return false;
      const uint32_t full = peer_bar0 + 8 * (B_X_FULL + 2 * slot + cw);
      const uint32_t dst = peer_x + slot * 2 * 8192, dste = peer_xe + slot * 2 * 512;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        st_async_v4(dst + (j * 128 + r) * 16, pk_n[4 * j], pk_n[4 * j + 1], pk_n[4 * j + 2], pk_n[4 * j + 3], full);
      st_async_b32(dste + r * 4, (uint32_t)ex_n, full);
      ++x_sent;
      return true;
    };

    // epilogue of a finished piece (run one tile later, when its last PV is long done)
    bool epi_pending = false;
    int epi_qb = 0, epi_split = 0;
    float epi_m = 0.f, epi_l = 1.f;
    auto epilogue = [&]() -> bool {
      // total row sum = both groups' partial sums
      float* lx = reinterpret_cast<float*>(smem + SM_MX) + 2 * 128 * 2;  // [group][row] after the max buffers
      lx[cw * 128 + r] = epi_l;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_EPI));
      if (!wait_warp(bar(B_EPI), pieces_done & 1, wc, kSitePEmpty)) return false;
      const float ltot = lx[r] + lx[128 + r];
      ++pieces_done;
      const bool split = num_splits[epi_qb] > 1;
      const int slot = split ? split_offset[epi_qb] + epi_split : 0;
      const float inv_l = 1.f / ltot;
      const bool write_row = r < H;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + TM_O + 128 * cw + 32 * c, v);
        tmem_wait_ld();
        if (write_row) {
          const int d0 = 256 * half + 128 * cw + 32 * c;
          if (split || args.out_f32) {
            float* dst = split ? args.o_acc + ((int64_t)slot * H + r) * 512 + d0
                               : reinterpret_cast<float*>(args.out) + ((int64_t)epi_qb * H + r) * 512 + d0;
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(dst + j) =
                  make_float4(__uint_as_float(v[j]) * inv_l, __uint_as_float(v[j + 1]) * inv_l,
                              __uint_as_float(v[j + 2]) * inv_l, __uint_as_float(v[j + 3]) * inv_l);
          } else {
            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(args.out) + ((int64_t)epi_qb * H + r) * 512 + d0;
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              uint4 o;
              o.x = pack_bf16(__uint_as_float(v[j]) * inv_l, __uint_as_float(v[j + 1]) * inv_l);
              o.y = pack_bf16(__uint_as_float(v[j + 2]) * inv_l, __uint_as_float(v[j + 3]) * inv_l);
              o.z = pack_bf16(__uint_as_float(v[j + 4]) * inv_l, __uint_as_float(v[j + 5]) * inv_l);
              o.w = pack_bf16(__uint_as_float(v[j + 6]) * inv_l, __uint_as_float(v[j + 7]) * inv_l);
              *reinterpret_cast<uint4*>(dst + j) = o;
            }
          }
        }
      }
      if (write_row && half == 0 && cw == 0) {
        const float lse = (epi_m + log2f(ltot)) * 0.69314718055994530942f;
        if (split)
          args.lse_acc[(int64_t)slot * H + r] = lse;
        else
          args.lse[(int64_t)epi_qb * H + r] = lse;
      }
      tc_fence_before();
      epi_pending = false;
      return true;
    };

    TileInfo cur, nxt;
    bool have = cursor.next(cur);
    if (have) {
      Piece p0;
      qwalk.next(p0);
      load_q_tmem(p0.qb);
      ok = stage_a(cur, own_c) && send_chunk();
    }
    float m_used = -INFINITY, l = 0.f;  // running max (log2 units) and this group's row sum
    uint32_t kv_t = 0;
    float* mx = reinterpret_cast<float*>(smem + SM_MX);  // [tile parity][group][row] chunk maxima
    while (ok && have) {
      const bool have_n = cursor.next(nxt);
      if (have_n && !(ok = stage_a(nxt, own_n))) break;
      if (cur.first) {
        m_used = -INFINITY;
        l = 0.f;
      }
      // ---- B: the next tile's chunk goes out; receive the peer's half of this tile's chunk
      if (have_n && !(ok = send_chunk())) break;
      const uint32_t rslot = x_recv & 1;
      if (lane == 0 && (warp & 3) == 0) mbar_arrive_expect_tx(bar(B_X_FULL + 2 * rslot + cw), kXChunkBytes);
      if (!(ok = wait_warp<true>(bar(B_X_FULL + 2 * rslot + cw), (x_recv >> 1) & 1, wc, kSiteXFull))) break;
      uint32_t wv[16];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(wv[4 * j]), "=r"(wv[4 * j + 1]), "=r"(wv[4 * j + 2]), "=r"(wv[4 * j + 3])
                     : "r"(my_x + rslot * 2 * 8192 + (j * 128 + r) * 16));
      int pe;
      asm volatile("ld.shared.b32 %0, [%1];" : "=r"(pe) : "r"(my_xe + rslot * 2 * 512 + r * 4));
      const float kp = pow2f(pe - 15);
      const int vc = cur.valid - 32 * cw;
      float sc[32];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        float q0, q1;
        bfp_unpack2(wv[u], q0, q1);
        sc[2 * u] = fmaf(q0, kp, own_c[2 * u]) * sl2;
        sc[2 * u + 1] = fmaf(q1, kp, own_c[2 * u + 1]) * sl2;
      }
      __syncwarp();  // every lane has consumed its part of the slot
      if (lane == 0) mbar_arrive_remote(peer_bar0 + 8 * (B_X_FREE + 2 * rslot + cw));
      if (vc < 32) {
#pragma unroll
        for (int j = 0; j < 32; ++j) sc[j] = (j < vc) ? sc[j] : -INFINITY;
      }
      float c0 = sc[0], c1 = sc[1], c2 = sc[2], c3 = sc[3];
#pragma unroll
      for (int j = 4; j < 32; j += 4) {
        c0 = fmaxf(c0, sc[j]);
        c1 = fmaxf(c1, sc[j + 1]);
        c2 = fmaxf(c2, sc[j + 2]);
        c3 = fmaxf(c3, sc[j + 3]);
      }
      // ---- tile max across the two groups (shared memory, one barrier per tile)
      const uint32_t par = x_recv & 1;
      mx[(par * 2 + cw) * 128 + r] = fmaxf(fmaxf(c0, c1), fmaxf(c2, c3));
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_MX));
      if (!(ok = wait_warp(bar(B_MX), par, wc, kSiteSFull))) break;
      const float cm = fmaxf(mx[(par * 2) * 128 + r], mx[(par * 2 + 1) * 128 + r]);
      float o_alpha = 1.f;
      if (cur.first) {
        m_used = cm;  // finite: token 0 of a piece's first tile is visible
      } else if (cm > m_used + 8.f) {  // lazy rescale: only when the max grows a lot
        o_alpha = exp2f(m_used - cm);
        m_used = cm;
        l *= o_alpha;
      }
      uint32_t pp[16];
      float r0 = 0.f, r1 = 0.f;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const float p0 = exp2f(sc[2 * u] - m_used), p1 = exp2f(sc[2 * u + 1] - m_used);
        pp[u] = pack_bf16(p0, p1);
        r0 += p0;
        r1 += p1;
      }
      l += r0 + r1;
      ++x_recv;
      // ---- C: the previous PV is done -> finish the previous piece, fix O, publish P
      if (kv_t > 0 && !(ok = wait_warp(bar(B_PV_DONE), (kv_t - 1) & 1, wc, kSitePEmpty))) break;
      tc_fence_after();
      if (epi_pending && !(ok = epilogue())) break;
      if (!cur.first && __any_sync(0xffffffffu, o_alpha != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + TM_O + 128 * cw + 32 * c, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * o_alpha);
          tmem_st32(tmem + lane_off + TM_O + 128 * cw + 32 * c, v);
        }
        tmem_wait_st();
      }
      const uint32_t st = kv_t % kStages;
      if (cur.valid < kTileTok) {
        // rows past the sequence end must not reach the PV product (0 * garbage): zero them
        if (!(ok = wait_warp(bar(B_KV_FULL + st), (kv_t / kStages) & 1, wc, kSiteKvFull))) break;
        const uint32_t sbase = base + st * kStageBytes;
        const int nz = (kTileTok - cur.valid) * 4 * 8;  // 16-byte chunks: rows x 4 blocks x 8
        for (int idx = gt; idx < nz; idx += 256) {
          const int row = cur.valid + idx / 32, blk = (idx / 8) & 3, ch = idx & 7;
          asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(sbase + blk * kLatBlock + row * 128 + ch * 16),
                       "r"(0u));
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // this group's 32 P values of the row (K-major, 128-byte swizzle)
        const uint32_t ch = 4 * cw + q;
        const uint32_t a = base + SM_P + r * 128 + ((ch ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(pp[4 * q]), "r"(pp[4 * q + 1]),
                     "r"(pp[4 * q + 2]), "r"(pp[4 * q + 3]));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_P_FULL));
      ++kv_t;
      if (cur.last) {
        epi_pending = true;
        epi_qb = cur.qb;
        epi_split = cur.split;
        epi_m = m_used;
        epi_l = l;
      }
      if (!have_n) break;
      cur = nxt;
#pragma unroll
      for (int u = 0; u < 32; ++u) own_c[u] = own_n[u];
    }
    if (ok && epi_pending) {
      if (wait_warp(bar(B_PV_DONE), (kv_t - 1) & 1, wc, kSitePEmpty)) {
        tc_fence_after();
        epilogue();
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (*abort_flag) drain_delay(200000);  // in-flight TMA / st.async / MMA land before release
  cluster_sync();                        // the peer no longer touches our shared memory
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace mla
