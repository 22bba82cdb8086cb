// Absorbed-MLA decode kernel for sm_103a (tcgen05 + TMA + 2-SM clusters).
//
// Work split.  One work unit = one 2-CTA cluster (two SMs) walking a contiguous
// stretch of (query block, 128-token tile) work from the split plan.  CTA h of
// the pair ("half" h) owns
//   * dims [256h, 256h+256) of the latent and dims [32h, 32h+32) of the RoPE
//     key of every cached token -- it loads only those with TMA (paged gather:
//     each 128-token tile is two 64-token pages found through the block table);
//   * output latent dims [256h, 256h+256): its O accumulator is 128 heads x 256
//     fp32 columns of tensor memory.
// Scores need all 576 dims, so each CTA computes a partial score over its 288
// dims (tcgen05.mma, M = 128 heads, N = 128 tokens; the absorbed-query half
// lives in tensor memory as the A operand, the RoPE-query half in shared
// memory), and the two CTAs swap partial scores through distributed shared
// memory (st.async), encoded as 16-bit block floating point: one shared
// exponent per (head, 32-token chunk), 16-bit signed mantissas.  Both CTAs
// form the same sum rounded(own) + rounded(peer), so their softmax statistics
// agree bit for bit.  Then each CTA runs the online softmax (one thread per
// head row), writes P (bf16) to shared memory, and accumulates
// O_half += P V_half with one more tcgen05.mma (N = 256, V read MN-major from
// the same shared-memory tile the score used).
//
// "MLA inference: two computation paths and FlashMLA", section "Decode
// attention becomes a compute problem": the 128 heads are the M dimension of
// the matrix multiply, a block of KV is staged in shared memory, long
// sequences are split across SMs and merged through their LSE.
//
// Warp roles (256 threads): warp 0 = TMA producer, warp 1 = MMA issuer,
// warp 2 = tensor-memory allocator, warp 3 idle, warps 4..7 = softmax /
// exchange / epilogue (thread = head row = TMEM lane).
#pragma once
#include "common.cuh"

namespace mla {

constexpr int kThreads = 256;
constexpr int kRows = 128;             // MMA M: head rows (H <= 128, padded with zero queries)
constexpr int kTileTok = 128;          // tokens per work tile (two pages)
constexpr int kStages = 2;

// shared memory layout (offsets from a 1024-byte aligned base)
constexpr uint32_t kStageBytes = 73728;           // latent half: 4 blocks x [128 rows x 128 B]; RoPE half [128 x 64 B]
constexpr uint32_t kStageRope = 65536;
constexpr uint32_t kLatBlock = 16384;
constexpr uint32_t SM_P = kStages * kStageBytes;  // P: 2 blocks x [128 rows x 128 B] (tokens 0-63, 64-127)
constexpr uint32_t SM_QR = SM_P + 32768;          // RoPE-query half [128 x 64 B], 64-byte swizzle
constexpr uint32_t SM_X = SM_QR + 8192;           // peer partial scores: [16 chunks][128 rows][16 B] int16 pairs
constexpr uint32_t SM_XE = SM_X + 32768;          // peer exponents: [128 rows][4] int32
constexpr uint32_t SM_BAR = SM_XE + 2048;
constexpr uint32_t kSmemBytes = SM_BAR + 256 + 1024;  // + alignment slack
constexpr uint32_t kXBytes = kRows * (256 + 16);      // bytes one CTA sends the other per tile

// tensor memory columns
constexpr uint32_t TM_O = 0, TM_S = 256, TM_Q = 384;

// barrier slots (8 bytes each) inside SM_BAR
enum : uint32_t {
  B_QR_FULL = 0, B_QR_EMPTY, B_QT_FULL, B_KV_FULL0, B_KV_FULL1, B_KV_EMPTY0, B_KV_EMPTY1, B_S_FULL, B_S_EMPTY,
  B_P_FULL, B_PV_DONE, B_X_FULL, B_X_FREE, B_DRAIN, kNumBars
};
constexpr uint32_t OFF_TMEM_SLOT = kNumBars * 8;
constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4;

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

__device__ __forceinline__ float pow2f(int p) { return __int_as_float((127 + p) << 23); }  // p in [-126, 127]

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Exponent e (clamped) with |x| < 2^e for the largest |x| of a chunk; the
// 16-bit mantissa of x is then rint(x * 2^(15-e)).
__device__ __forceinline__ int bfp_exponent(float amax) {
  int e = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 126;
  e = e < -60 ? -60 : e;
  e = e > 110 ? 110 : e;
  return e;
}

__device__ __forceinline__ int32_t bfp_mant(float x, float k) {
  float y = rintf(x * k);
  y = fminf(fmaxf(y, -32767.f), 32767.f);
  return (int32_t)y;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) mla_decode_bf16_kernel(const __grid_constant__ DecodeArgs args) {
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
    mbar_init(bar(B_QT_FULL), 128);
    mbar_init(bar(B_KV_FULL0), 1);
    mbar_init(bar(B_KV_FULL1), 1);
    mbar_init(bar(B_KV_EMPTY0), 1);
    mbar_init(bar(B_KV_EMPTY1), 1);
    mbar_init(bar(B_S_FULL), 1);
    mbar_init(bar(B_S_EMPTY), 128);
    mbar_init(bar(B_P_FULL), 128);
    mbar_init(bar(B_PV_DONE), 1);
    mbar_init(bar(B_X_FULL), 1);
    mbar_init(bar(B_X_FREE), 128);
    mbar_init(bar(B_DRAIN), 1);
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
      PieceWalker w = walker0;
      Piece pc;
      uint32_t kv_it = 0, piece_no = 0;
      bool ok = true;
      while (ok && w.next(pc)) {
        if (piece_no > 0 && !(ok = wait_one(bar(B_QR_EMPTY), (piece_no - 1) & 1, wc, kSiteQEmpty))) break;
        mbar_arrive_expect_tx(bar(B_QR_FULL), 8192);
        tma_load_3d(base + SM_QR, &args.map_qr, bar(B_QR_FULL), 32 * half, 0, pc.qb, pol_q);
        const int b = pc.qb / args.s_q;
        const int vis = visible_keys(args.seqlens[b], args.s_q, pc.qb % args.s_q, args.causal);
        for (int t = pc.t0; t < pc.t1; ++t) {
          const uint32_t st = kv_it % kStages, ph = (kv_it / kStages) & 1;
          if (!(ok = wait_one(bar(B_KV_EMPTY0 + st), ph ^ 1, wc, kSiteKvEmpty))) break;
          const int npages = (vis - t * kTileTok) > 64 ? 2 : 1;
          mbar_arrive_expect_tx(bar(B_KV_FULL0 + st), npages * (kStageBytes / 2));
          const uint32_t sbase = base + st * kStageBytes;
          for (int pg = 0; pg < npages; ++pg) {
            const int page = args.block_table[(int64_t)b * args.max_pages + 2 * t + pg];
            const int y = page * 64;
            for (int blk = 0; blk < 4; ++blk)
              tma_load_2d(sbase + blk * kLatBlock + pg * 8192, &args.map_kvc, bar(B_KV_FULL0 + st),
                          256 * half + 64 * blk, y, pol_kv);
            tma_load_2d(sbase + kStageRope + pg * 4096, &args.map_kvr, bar(B_KV_FULL0 + st), 512 + 32 * half, y,
                        pol_kv);
          }
          ++kv_it;
        }
        ++piece_no;
      }
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t id_pv = idesc_bf16_f32(128, 256, 0, 1);
      PieceWalker w = walker0;
      Piece pc;
      uint32_t kv_it = 0, s_it = 0, pv_it = 0, piece_no = 0;
      bool ok = true;
      auto issue_pv = [&](uint32_t st, bool accumulate) -> bool {
        if (!wait_one(bar(B_P_FULL), pv_it & 1, wc, kSitePFull)) return false;
        tc_fence_after();
        const uint32_t sbase = base + st * kStageBytes;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t a = smem_desc(base + SM_P + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024, kSwizzle128B);
          const uint64_t bv = smem_desc(sbase + k * 2048, kLatBlock, 1024, kSwizzle128B);
          mma_bf16_ss(tmem + TM_O, a, bv, id_pv, (accumulate || k > 0) ? 1u : 0u);
        }
        mma_commit(bar(B_KV_EMPTY0 + st));
        mma_commit(bar(B_PV_DONE));
        ++pv_it;
        return true;
      };
      while (ok && w.next(pc)) {
        if (!(ok = wait_one(bar(B_QR_FULL), piece_no & 1, wc, kSiteQFull))) break;
        if (!(ok = wait_one(bar(B_QT_FULL), piece_no & 1, wc, kSiteQFull))) break;
        tc_fence_after();
        const int n = pc.t1 - pc.t0;
        uint32_t prev_st = 0;
        for (int i = 0; i < n; ++i) {
          const uint32_t st = kv_it % kStages;
          if (!(ok = wait_one(bar(B_KV_FULL0 + st), (kv_it / kStages) & 1, wc, kSiteKvFull))) break;
          if (!(ok = wait_one(bar(B_S_EMPTY), (s_it & 1) ^ 1, wc, kSiteSEmpty))) break;
          tc_fence_after();
          const uint32_t sbase = base + st * kStageBytes;
#pragma unroll
          for (int k = 0; k < 16; ++k) {  // latent half: A = query half in tensor memory
            const uint64_t bk = smem_desc(sbase + (k >> 2) * kLatBlock + (k & 3) * 32, 16, 1024, kSwizzle128B);
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem + TM_S),
                "r"(tmem + TM_Q + 8 * k), "l"(bk), "r"(id_qk), "r"(k > 0 ? 1u : 0u)
                : "memory");
          }
#pragma unroll
          for (int k = 0; k < 2; ++k) {  // RoPE half: A = RoPE-query half in shared memory
            const uint64_t a = smem_desc(base + SM_QR + 32 * k, 16, 512, kSwizzle64B);
            const uint64_t bk = smem_desc(sbase + kStageRope + 32 * k, 16, 512, kSwizzle64B);
            mma_bf16_ss(tmem + TM_S, a, bk, id_qk, 1u);
          }
          mma_commit(bar(B_S_FULL));
          if (i == n - 1) mma_commit(bar(B_QR_EMPTY));
          ++s_it;
          if (i > 0 && !(ok = issue_pv(prev_st, i - 1 > 0))) break;
          prev_st = st;
          ++kv_it;
        }
        if (!ok) break;
        if (!(ok = issue_pv(prev_st, n - 1 > 0))) break;
        ++piece_no;
      }
      // make sure no MMA is still running when tensor memory is released
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
    const int r = tid - 128;                       // head row == TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t peer_x = map_to_rank(base + SM_X, peer);
    const uint32_t peer_xe = map_to_rank(base + SM_XE, peer);
    const uint32_t peer_x_full = map_to_rank(bar(B_X_FULL), peer);
    const uint32_t peer_x_free = map_to_rank(bar(B_X_FREE), peer);
    const float sl2 = args.scale_log2;
    const int H = args.H;
    PieceWalker w = walker0;
    Piece pc;
    uint32_t s_it = 0, p_it = 0, x_it = 0, kv_it = 0, piece_no = 0;
    bool ok = true;

    // query half -> tensor memory (A operand of the latent part of the score)
    auto load_q_tmem = [&](int qb) {
      uint32_t q[32];
      const uint32_t* src = reinterpret_cast<const uint32_t*>(args.q_nope) +
                            ((int64_t)qb * H + r) * 256 + 128 * half;  // 256 bf16 = 128 words
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (r < H) v = *reinterpret_cast<const uint4*>(src + 32 * c + j);
          q[j] = v.x;
          q[j + 1] = v.y;
          q[j + 2] = v.z;
          q[j + 3] = v.w;
        }
        tmem_st32(tmem + lane_off + TM_Q + 32 * c, q);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_QT_FULL));
    };

    bool have = w.next(pc);
    if (have) load_q_tmem(pc.qb);
    while (ok && have) {
      const int b = pc.qb / args.s_q;
      const int vis = visible_keys(args.seqlens[b], args.s_q, pc.qb % args.s_q, args.causal);
      float m_used = -INFINITY, l = 0.f, lq = 0.f;  // l: exact row sum (for lse); lq: sum of the bf16 weights (for O)
      const int n = pc.t1 - pc.t0;
      Piece nxt;
      bool have_next = false;
      for (int i = 0; i < n; ++i) {
        const int tile = pc.t0 + i;
        const int valid = min(kTileTok, vis - tile * kTileTok);  // >= 1
        // ---- own partial scores
        if (!(ok = wait_warp(bar(B_S_FULL), s_it & 1, wc, kSiteSFull))) break;
        tc_fence_after();
        float s[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + TM_S + 32 * c, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) s[32 * c + j] = __uint_as_float(v[j]);
        }
        tc_fence_before();
        mbar_arrive(bar(B_S_EMPTY));
        ++s_it;
        if (i == n - 1) {  // the query half in tensor memory is free once this score exists
          have_next = w.next(nxt);
          if (have_next) load_q_tmem(nxt.qb);
        }
        // ---- encode (16-bit block floating point per 32-token chunk) and send to the peer
        if (!(ok = wait_warp(bar(B_X_FREE), (x_it & 1) ^ 1, wc, kSiteXFree))) break;
        int ex[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float amax = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) amax = (32 * c + j < valid) ? fmaxf(amax, fabsf(s[32 * c + j])) : amax;
          const int e = bfp_exponent(amax);
          ex[c] = e;
          const float k = pow2f(15 - e), kinv = pow2f(e - 15);
#pragma unroll
          for (int j = 0; j < 32; j += 8) {
            uint32_t wv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int j0 = 32 * c + j + 2 * u;
              const int32_t m0 = (j0 < valid) ? bfp_mant(s[j0], k) : 0;
              const int32_t m1 = (j0 + 1 < valid) ? bfp_mant(s[j0 + 1], k) : 0;
              s[j0] = (float)m0 * kinv;  // own value, rounded exactly as the peer will see it
              s[j0 + 1] = (float)m1 * kinv;
              wv[u] = (uint32_t)(m0 & 0xFFFF) | ((uint32_t)m1 << 16);
            }
            const uint32_t chunk = (32 * c + j) / 8;  // 16-byte chunk index 0..15
            st_async_v4(peer_x + (chunk * 128 + r) * 16, wv[0], wv[1], wv[2], wv[3], peer_x_full);
          }
        }
        st_async_v4(peer_xe + r * 16, (uint32_t)ex[0], (uint32_t)ex[1], (uint32_t)ex[2], (uint32_t)ex[3], peer_x_full);
        if (r == 0) mbar_arrive_expect_tx(bar(B_X_FULL), kXBytes);
        // ---- receive the peer's partial scores and form the full score
        if (!(ok = wait_warp<true>(bar(B_X_FULL), x_it & 1, wc, kSiteXFull))) break;
        {
          uint32_t pe[4];
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(pe[0]), "=r"(pe[1]), "=r"(pe[2]), "=r"(pe[3])
                       : "r"(base + SM_XE + r * 16));
#pragma unroll
          for (int chunk = 0; chunk < 16; ++chunk) {
            uint32_t wv[4];
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(wv[0]), "=r"(wv[1]), "=r"(wv[2]), "=r"(wv[3])
                         : "r"(base + SM_X + (chunk * 128 + r) * 16));
            const float kinv = pow2f((int)pe[chunk >> 2] - 15);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int j0 = chunk * 8 + 2 * u;
              const float p0 = (float)(int32_t)(int16_t)(wv[u] & 0xFFFF) * kinv;
              const float p1 = (float)((int32_t)wv[u] >> 16) * kinv;
              s[j0] = (j0 < valid) ? (s[j0] + p0) * sl2 : -INFINITY;
              s[j0 + 1] = (j0 + 1 < valid) ? (s[j0 + 1] + p1) * sl2 : -INFINITY;
            }
          }
        }
        mbar_arrive_remote(peer_x_free);
        ++x_it;
        // ---- online softmax (log2 domain); O is rescaled only when the max grows by > 8
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 128; ++j) mx = fmaxf(mx, s[j]);
        const bool first = (i == 0);
        const bool resc = !first && (mx > m_used + 8.f);
        const float m_new = (first || resc) ? mx : m_used;
        const float alpha = resc ? exp2f(m_used - m_new) : 1.f;
        m_used = m_new;
        uint32_t pk[64];
        float rs = 0.f, rq = 0.f;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const float p0 = exp2f(s[2 * j] - m_new), p1 = exp2f(s[2 * j + 1] - m_new);
          pk[j] = pack_bf16(p0, p1);
          rs += p0 + p1;
          // O is normalised by the sum of the bf16 weights the PV product saw, so the output
          // is an exact convex combination of the values
          rq += __uint_as_float(pk[j] << 16) + __uint_as_float(pk[j] & 0xFFFF0000u);
        }
        l = l * alpha + rs;
        lq = lq * alpha + rq;
        // ---- previous PV done: P buffer, O and the stage are ours
        if (p_it > 0 && !(ok = wait_warp(bar(B_PV_DONE), (p_it - 1) & 1, wc, kSitePEmpty))) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_off + TM_O + 32 * c, v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
            tmem_st32(tmem + lane_off + TM_O + 32 * c, v);
          }
          tmem_wait_st();
        }
        const uint32_t st = kv_it % kStages;
        if (valid < kTileTok) {
          // rows past the sequence end must not reach the PV product (0 * garbage); zero them
          if (!(ok = wait_warp(bar(B_KV_FULL0 + st), (kv_it / kStages) & 1, wc, kSiteKvFull))) break;
          const uint32_t sbase = base + st * kStageBytes;
          const int nz = (kTileTok - valid) * 4 * 8;  // 16-byte chunks: rows x 4 blocks x 8
          for (int idx = r; idx < nz; idx += 128) {
            const int row = valid + idx / 32, blk = (idx / 8) & 3, ch = idx & 7;
            asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(sbase + blk * kLatBlock + row * 128 + ch * 16),
                         "r"(0u));
          }
        }
        // ---- P row -> shared memory (K-major, 128-byte swizzle)
#pragma unroll
        for (int ch = 0; ch < 16; ++ch) {
          const uint32_t a = base + SM_P + (ch >> 3) * 16384 + r * 128 + ((((uint32_t)ch & 7) ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(pk[4 * ch]), "r"(pk[4 * ch + 1]),
                       "r"(pk[4 * ch + 2]), "r"(pk[4 * ch + 3]));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(B_P_FULL));
        ++p_it;
        ++kv_it;
      }
      if (!ok) break;
      // ---- epilogue: O_half / l -> out (or the split partial), lse
      if (!(ok = wait_warp(bar(B_PV_DONE), (p_it - 1) & 1, wc, kSitePEmpty))) break;
      tc_fence_after();
      const bool split = num_splits[pc.qb] > 1;
      const int slot = split ? split_offset[pc.qb] + pc.split : 0;
      const float inv_l = 1.f / lq;
      const bool write_row = r < H;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + TM_O + 32 * c, v);
        tmem_wait_ld();
        if (write_row) {
          const int d0 = 256 * half + 32 * c;
          if (split) {
            float* dst = args.o_acc + ((int64_t)slot * H + r) * 512 + d0;
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(dst + j) =
                  make_float4(__uint_as_float(v[j]) * inv_l, __uint_as_float(v[j + 1]) * inv_l,
                              __uint_as_float(v[j + 2]) * inv_l, __uint_as_float(v[j + 3]) * inv_l);
          } else if (args.out_f32) {
            float* dst = reinterpret_cast<float*>(args.out) + ((int64_t)pc.qb * H + r) * 512 + d0;
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(dst + j) =
                  make_float4(__uint_as_float(v[j]) * inv_l, __uint_as_float(v[j + 1]) * inv_l,
                              __uint_as_float(v[j + 2]) * inv_l, __uint_as_float(v[j + 3]) * inv_l);
          } else {
            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(args.out) + ((int64_t)pc.qb * H + r) * 512 + d0;
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
      if (write_row && half == 0) {
        const float lse = (m_used + log2f(l)) * 0.69314718055994530942f;
        if (split)
          args.lse_acc[(int64_t)slot * H + r] = lse;
        else
          args.lse[(int64_t)pc.qb * H + r] = lse;
      }
      tc_fence_before();
      ++piece_no;
      pc = nxt;
      have = have_next;
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
