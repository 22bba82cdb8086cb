// Extend (a prefill continuation: s_q new tokens after a cached prefix) by the expand path,
// chunk by chunk ("MLA inference: two computation paths and FlashMLA", sections "Two
// equivalent paths" (path one) and "Which is faster: count new tokens and cached tokens":
// when the prefix is long, expanding all of it at once needs too much memory, so the keys
// and values are expanded a chunk at a time, attended, and the chunks' results merged by
// their log-sum-exp).
//
// Per chunk of C cached rows two kernels run:
//   mla_expand_kernel  K^N[b][h][j] = W_UK[h] c_j and V[b][h][j] = c_j W_UV[h] for the chunk's
//                      rows (bf16, zero rows past the sequence's end), one tcgen05 GEMM per
//                      (128 rows, head): the rows' latent tile stays in shared memory while
//                      the heads' weights stream through it, two 64-deep chunks per TMA box.
// Boxes are large on purpose: one thread issuing TMA copies spends about the same time per
// copy (~0.23 us) whatever its size, so fewer, bigger boxes move more bytes per SM.
//   mla_attend_kernel  per (128 new tokens, head, sequence): S = [q^N, q^R] . [K^N, k^R]^T,
//                      causal mask, online softmax, O += P V over the chunk's 64-key tiles,
//                      then the LSE merge with the result of the chunks before it (float32
//                      accumulators in the workspace); the last chunk writes the bf16 output.
// d_nope = d_v = 128 (DeepSeek-V3's per-head dims), d_c = 512, d_r = 64, pages of 64 rows.
#pragma once
#include "common.cuh"
#include "tma4d.cuh"

namespace mla {

constexpr int kXThreads = 192;                    // warp 0: TMA, warp 1: MMA, warps 2..5: row work
constexpr int kXDim = 128;                        // d_nope = d_v
constexpr uint32_t kXBox = 64 * 128;              // [64 rows][64 bf16], 128-byte swizzle: 8 KB

// ---------------------------------------------------------------- expansion
constexpr int kExRing = 3;                        // weight stages in flight (two 64-deep chunks each)
constexpr uint32_t kExCBytes = 16 * kXBox;        // latent tile: 128 rows x 512 dims (8 chunks of 16 KB)
constexpr uint32_t kExStage = 4 * kXBox;          // two 64-deep chunks of W_UK[h] or W_UV[h]: 32 KB, one box
constexpr uint32_t kExSmem = 1024 + kExCBytes + kExRing * kExStage + 256;

struct ExpandArgs {
  CUtensorMap map_kvc;  // cache rows: bf16 {576, num_pages * 64}, box {64, 64}, 128-byte swizzle
  CUtensorMap map_wuk;  // W_UK: bf16 {64 k, 128 n, 8 k-chunks (128 B apart), H}, box {64, 128, 2, 1}, 128-byte swizzle
  CUtensorMap map_wuv;  // W_UV: bf16 {64 n, 512 k, 2 n-blocks (128 B apart), H}, box {64, 128, 2, 1}, 128-byte swizzle
  const int32_t* block_table;
  const int32_t* seqlens;
  __nv_bfloat16* kn;    // [B][H][C][ld] (first 128 of each row)
  __nv_bfloat16* v;     // [B][H][C][ld]
  int32_t B, H, C, chunk_start, heads_per_cta, s_q, max_pages_per_seq;
  int32_t ld;           // row stride of kn and v, elements: 128 (separate buffers) or 256 (K^N | V rows)
  uint64_t timeout_ns;
};

// A sequence length the extend kernels accept: the s_q new rows are in the cache and every
// row has a block-table entry.  Others are reported in the error word and skipped.
__device__ __forceinline__ bool extend_length_ok(int L, int s_q, int max_pages) {
  const bool ok = L >= s_q && (int64_t)L <= (int64_t)max_pages * 64;
  if (!ok) atomicCAS(&g_mla_error, 0, MLA_ERR_INVALID_ARG);
  return ok;
}

// grid (C / 128, B, H / heads_per_cta)
__global__ void __launch_bounds__(kXThreads, 1) mla_expand_kernel(const __grid_constant__ ExpandArgs args) {
  extern __shared__ uint8_t ex_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ex_smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t base = smem_addr(smem);
  const uint32_t c_base = base, ring = base + kExCBytes;
  const uint32_t bars = ring + kExRing * kExStage;
  // barriers: [0, R) weight full, [R, 2R) weight empty, 2R latent tile full, 2R+1.. accumulator
  // full (2), accumulator empty (2)
  auto W_FULL = [&](int s) { return bars + 8 * s; };
  auto W_EMPTY = [&](int s) { return bars + 8 * (kExRing + s); };
  const uint32_t C_FULL = bars + 8 * (2 * kExRing);
  auto A_FULL = [&](int i) { return bars + 8 * (2 * kExRing + 1 + i); };
  auto A_EMPTY = [&](int i) { return bars + 8 * (2 * kExRing + 3 + i); };
  constexpr int kNumBars = 2 * kExRing + 5;
  static_assert(8 * kNumBars + 16 <= 256, "expansion barrier area");
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kExCBytes + kExRing * kExStage + 8 * kNumBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kExCBytes + kExRing * kExStage + 8 * kNumBars + 8);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.y, h0 = blockIdx.z * args.heads_per_cta, nh = args.heads_per_cta;
  const int rel0 = blockIdx.x * 128, j0 = args.chunk_start + rel0;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(bars + 8 * i, (i >= 2 * kExRing + 3) ? 4 : 1);
    *abort_flag = 0;
    prefetch_tensormap(&args.map_kvc);
    prefetch_tensormap(&args.map_wuk);
    prefetch_tensormap(&args.map_wuv);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait_prerequisites();  // the previous chunk's attention has finished reading the workspace
  const int L = args.seqlens[b];
  const bool active = extend_length_ok(L, args.s_q, args.max_pages_per_seq) && j0 < L;

  WaitCtx wc;
  wc.abort_local = abort_flag;
  wc.abort_peer = 0;
  wc.timeout_ns = args.timeout_ns;
  const int n_it = nh * 8;  // per head: 4 stages of W_UK[h], then 4 of W_UV[h]
  if (active && warp == 0 && lane == 0) {
    const uint64_t keep = l2_policy_evict_last(), stream = l2_policy_evict_first();
    // the 128 rows' latent tile: two pages (the second clamped to the first past the end)
    const int32_t* bt = args.block_table + (int64_t)b * args.max_pages_per_seq;
    const int p0 = bt[j0 / 64], p1 = (j0 + 64 < L) ? bt[j0 / 64 + 1] : p0;
    mbar_arrive_expect_tx(C_FULL, kExCBytes);
    for (int k = 0; k < 8; ++k) {
      tma_load_2d(c_base + k * 2 * kXBox, &args.map_kvc, C_FULL, 64 * k, p0 * 64, stream);
      tma_load_2d(c_base + k * 2 * kXBox + kXBox, &args.map_kvc, C_FULL, 64 * k, p1 * 64, stream);
    }
    for (int it = 0; it < n_it; ++it) {
      const int st = it % kExRing, h = h0 + it / 8, part = (it >> 2) & 1, kp = it & 3;
      if (it >= kExRing && !wait_one(W_EMPTY(st), ((it / kExRing) - 1) & 1, wc, kSiteKvEmpty)) break;
      const uint32_t sb = ring + st * kExStage;
      mbar_arrive_expect_tx(W_FULL(st), kExStage);
      if (part == 0)  // W_UK[h] chunks 2kp, 2kp + 1: [chunk][128 n][64 k]
        tma_load_4d(sb, &args.map_wuk, W_FULL(st), 0, 0, 2 * kp, h, keep);
      else            // W_UV[h] rows 128 kp .. 128 kp + 127: [n block][128 k][64 n]
        tma_load_4d(sb, &args.map_wuv, W_FULL(st), 0, 128 * kp, 0, h, keep);
    }
  } else if (active && warp == 1 && lane == 0) {
    const uint32_t idesc_k = idesc_bf16_f32(128, 128, 0, 0), idesc_v = idesc_bf16_f32(128, 128, 0, 1);
    bool ok = wait_one(C_FULL, 0, wc, kSiteQFull);
    for (int hi = 0; hi < nh && ok; ++hi) {
      const int buf = hi & 1;
      if (hi >= 2 && !(ok = wait_one(A_EMPTY(buf), ((hi >> 1) - 1) & 1, wc, kSiteSEmpty))) break;
      tc_fence_after();
      for (int part = 0; part < 2 && ok; ++part) {
        const uint32_t d = tmem + buf * 256 + part * 128;
        for (int kp = 0; kp < 4; ++kp) {
          const int it = hi * 8 + part * 4 + kp, st = it % kExRing;
          if (!(ok = wait_one(W_FULL(st), (it / kExRing) & 1, wc, kSiteKvFull))) break;
          tc_fence_after();
          const uint32_t sb = ring + st * kExStage;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // latent dims 128 kp + 16 kk
            const uint64_t a = smem_desc(c_base + (2 * kp + (kk >> 2)) * 2 * kXBox + (kk & 3) * 32, 16, 1024, kSwizzle128B);
            if (part == 0)
              mma_bf16_ss(d, a, smem_desc(sb + (kk >> 2) * 2 * kXBox + (kk & 3) * 32, 16, 1024, kSwizzle128B), idesc_k,
                          (kp | kk) ? 1u : 0u);
            else
              mma_bf16_ss(d, a, smem_desc(sb + kk * 2048, 2 * kXBox, 1024, kSwizzle128B), idesc_v, (kp | kk) ? 1u : 0u);
          }
          mma_commit(W_EMPTY(st));
        }
      }
      if (ok) mma_commit(A_FULL(buf));
    }
  } else if (active && warp >= 2) {
    // thread = one of the tile's 128 rows (tensor-memory lane); zero rows past the end
    const int q = warp & 3, r = 32 * q + lane, j = j0 + r;
    const bool valid = j < L;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    for (int hi = 0; hi < nh; ++hi) {
      const int buf = hi & 1, h = h0 + hi;
      if (!wait_warp(A_FULL(buf), (hi >> 1) & 1, wc, kSiteDrain)) break;
      tc_fence_after();
      const int64_t row = ((int64_t)(b * args.H + h) * args.C + rel0 + r) * args.ld;
#pragma unroll 1
      for (int part = 0; part < 2; ++part) {
        __nv_bfloat16* dst = (part ? args.v : args.kn) + row;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t x[32];
          tmem_ld32(tmem + lane_off + buf * 256 + part * 128 + 32 * c, x);
          tmem_wait_ld();
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint4 o = make_uint4(0, 0, 0, 0);
            if (valid) {
              o.x = pack_bf16(__uint_as_float(x[8 * g]), __uint_as_float(x[8 * g + 1]));
              o.y = pack_bf16(__uint_as_float(x[8 * g + 2]), __uint_as_float(x[8 * g + 3]));
              o.z = pack_bf16(__uint_as_float(x[8 * g + 4]), __uint_as_float(x[8 * g + 5]));
              o.w = pack_bf16(__uint_as_float(x[8 * g + 6]), __uint_as_float(x[8 * g + 7]));
            }
            *reinterpret_cast<uint4*>(dst + 32 * c + 8 * g) = o;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(A_EMPTY(buf));
    }
  }
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) drain_delay(200000);  // in-flight copies and MMAs land before release
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- attention over one chunk
constexpr int kAtRing = 4;                               // 64-key tiles in flight
constexpr uint32_t kAtKn = 0, kAtV = 2 * kXBox, kAtKr = 4 * kXBox;  // offsets inside a stage
constexpr uint32_t kAtStage = 5 * kXBox;                 // K^N 16 KB, k^R 8 KB, V 16 KB
constexpr uint32_t kAtP = 2 * kXBox;                     // P: [128 rows][64 keys] bf16, 16 KB
constexpr uint32_t kAtSmem = 1024 + kAtRing * kAtStage + 2 * kAtP + 256;
// tensor-memory columns: O (128), S double buffer (2 x 64), Q = [q^N | q^R] as bf16 pairs (96)
constexpr uint32_t kTxO = 0, kTxS = 128, kTxQ = 256;

struct AttendArgs {
  CUtensorMap map_kvc;  // cache rows (k^R at x = 512): bf16 {576, num_pages * 64}, box {64, 64}, 128-byte swizzle
  CUtensorMap map_kv;   // workspace rows [K^N | V] as bf16 {64, C, 4 blocks (128 B apart), B * H},
                        // box {64, 64, 4, 1}: a tile's keys and values in one copy, 128-byte swizzle
  const __nv_bfloat16* q_nope;  // [B][s_q][H][128]
  const __nv_bfloat16* q_rope;  // [B][s_q][H][64]
  const int32_t* block_table;
  const int32_t* seqlens;
  float* acc_o;                 // [B][s_q][H][128]: merged output of the chunks so far
  float* acc_lse;               // [B][s_q][H]
  __nv_bfloat16* out;           // [B][s_q][H][128]
  float* lse;                   // [B][s_q][H]
  float scale_log2;             // softmax scale times log2(e)
  int32_t B, s_q, H, C, chunk_start, max_pages_per_seq;
  uint64_t timeout_ns;
};

// grid (ceil(s_q / 128), H, B)
__global__ void __launch_bounds__(kXThreads, 1) mla_attend_kernel(const __grid_constant__ AttendArgs args) {
  extern __shared__ uint8_t at_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(at_smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t base = smem_addr(smem);
  const uint32_t p_base = base + kAtRing * kAtStage;
  const uint32_t bars = p_base + 2 * kAtP;
  // barriers: [0, R) KV full, [R, 2R) KV empty, 2R Q full, then S full (2), S free (2),
  // P full (2), PV done (2)
  auto KV_FULL = [&](int s) { return bars + 8 * s; };
  auto KV_EMPTY = [&](int s) { return bars + 8 * (kAtRing + s); };
  const uint32_t Q_FULL = bars + 8 * (2 * kAtRing);
  auto S_FULL = [&](int i) { return bars + 8 * (2 * kAtRing + 1 + i); };
  auto S_FREE = [&](int i) { return bars + 8 * (2 * kAtRing + 3 + i); };
  auto P_FULL = [&](int i) { return bars + 8 * (2 * kAtRing + 5 + i); };
  auto PV_DONE = [&](int i) { return bars + 8 * (2 * kAtRing + 7 + i); };
  constexpr int kNumBars = 2 * kAtRing + 9;
  static_assert(8 * kNumBars + 16 <= 256, "attention barrier area");
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAtRing * kAtStage + 2 * kAtP + 8 * kNumBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kAtRing * kAtStage + 2 * kAtP + 8 * kNumBars + 8);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * 128, h = blockIdx.y, b = blockIdx.z;
  const int s_q = args.s_q, H = args.H;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      const int k = i - 2 * kAtRing;  // Q full, S free and P full take one arrive per row warp
      mbar_init(bars + 8 * i, (k == 0 || (k >= 3 && k <= 6)) ? 4 : 1);
    }
    *abort_flag = 0;
    prefetch_tensormap(&args.map_kvc);
    prefetch_tensormap(&args.map_kv);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait_prerequisites();  // this chunk's keys and values are expanded
  const int L = args.seqlens[b];
  const bool len_ok = extend_length_ok(L, s_q, args.max_pages_per_seq);
  const int cs = args.chunk_start, ce = min(cs + args.C, L);
  const bool in_range = len_ok && cs < L;           // this chunk holds keys of the sequence
  const bool last = in_range && cs + args.C >= L;   // ... and is its last one
  // keys this CTA's rows can see in the chunk: up to L - s_q + (last row), exclusive end
  const int hi_key = min(ce, L - s_q + min(t0 + 127, s_q - 1) + 1);
  const int n = in_range && hi_key > cs ? (hi_key - cs + 63) / 64 : 0;

  WaitCtx wc;
  wc.abort_local = abort_flag;
  wc.abort_peer = 0;
  wc.timeout_ns = args.timeout_ns;
  const int64_t bh = (int64_t)b * H + h;
  if (warp == 0 && lane == 0 && n > 0) {
    const uint64_t pol = l2_policy_evict_first();
    const int32_t* bt = args.block_table + (int64_t)b * args.max_pages_per_seq;
    for (int i = 0; i < n; ++i) {
      const int st = i % kAtRing, key0 = cs + 64 * i, rel = 64 * i;  // row of the chunk's workspace
      if (i >= kAtRing && !wait_one(KV_EMPTY(st), ((i / kAtRing) - 1) & 1, wc, kSiteKvEmpty)) break;
      const uint32_t sb = base + st * kAtStage;
      mbar_arrive_expect_tx(KV_FULL(st), kAtStage);
      tma_load_4d(sb + kAtKn, &args.map_kv, KV_FULL(st), 0, rel, 0, (int)bh, pol);  // K^N, then V
      tma_load_2d(sb + kAtKr, &args.map_kvc, KV_FULL(st), 512, bt[key0 / 64] * 64, pol);
    }
  } else if (warp == 1 && lane == 0 && n > 0) {
    const uint32_t idesc_s = idesc_bf16_f32(128, 64, 0, 0), idesc_o = idesc_bf16_f32(128, 128, 0, 1);
    bool ok = wait_one(Q_FULL, 0, wc, kSiteQFull);
    auto qk = [&](int i) -> bool {
      const int st = i % kAtRing;
      if (!wait_one(KV_FULL(st), (i / kAtRing) & 1, wc, kSiteKvFull)) return false;
      if (i >= 2 && !wait_one(S_FREE(i & 1), ((i >> 1) - 1) & 1, wc, kSiteSEmpty)) return false;
      tc_fence_after();
      const uint32_t sb = base + st * kAtStage, d = tmem + kTxS + 64 * (i & 1);
#pragma unroll
      for (int k = 0; k < 12; ++k) {  // K = 128 (q^N . k^N) + 64 (q^R . k^R), 16 per MMA
        const uint32_t src = k < 8 ? sb + kAtKn + (k >> 2) * kXBox + (k & 3) * 32 : sb + kAtKr + (k - 8) * 32;
        mma_bf16_ts(d, tmem + kTxQ + 8 * k, smem_desc(src, 16, 1024, kSwizzle128B), idesc_s, k > 0 ? 1u : 0u);
      }
      mma_commit(S_FULL(i & 1));
      return true;
    };
    if (ok) ok = qk(0);
    for (int i = 0; i < n && ok; ++i) {
      if (i + 1 < n && !(ok = qk(i + 1))) break;
      if (!(ok = wait_one(P_FULL(i & 1), (i >> 1) & 1, wc, kSitePFull))) break;
      tc_fence_after();
      const uint32_t sb = base + (i % kAtRing) * kAtStage, pb = p_base + (i & 1) * kAtP;
#pragma unroll
      for (int k = 0; k < 4; ++k)  // K = 64 keys, 16 per MMA; V MN-major in two 64-column blocks
        mma_bf16_ss(tmem + kTxO, smem_desc(pb + k * 32, 16, 1024, kSwizzle128B),
                    smem_desc(sb + kAtV + k * 2048, kXBox, 1024, kSwizzle128B), idesc_o, (i | k) ? 1u : 0u);
      mma_commit(KV_EMPTY(i % kAtRing));
      mma_commit(PV_DONE(i & 1));
    }
  } else if (warp >= 2) {
    // thread = query row (tensor-memory lane); row t sees keys 0 .. L - s_q + t
    const int q = warp & 3, r = 32 * q + lane, t = t0 + r;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    const bool row_ok = t < s_q;
    const int lim = row_ok ? L - s_q + t : -1;  // last visible key
    const int64_t row = ((int64_t)b * s_q + (row_ok ? t : 0)) * H + h;
    bool ok = true;
    float m_run = -INFINITY, l_run = 0.f;
    if (n > 0) {
      // Q row -> tensor memory: 64 columns of q^N pairs, 32 of q^R pairs
      uint32_t w[32];
#pragma unroll 1
      for (int c = 0; c < 3; ++c) {
        const uint4* src = c < 2 ? reinterpret_cast<const uint4*>(args.q_nope + row * kXDim + 64 * c)
                                 : reinterpret_cast<const uint4*>(args.q_rope + row * 64);
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const uint4 x = row_ok ? src[g] : make_uint4(0, 0, 0, 0);
          w[4 * g] = x.x;
          w[4 * g + 1] = x.y;
          w[4 * g + 2] = x.z;
          w[4 * g + 3] = x.w;
        }
        tmem_st32(tmem + lane_off + kTxQ + 32 * c, w);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(Q_FULL);

#pragma unroll 1
      for (int i = 0; i < n; ++i) {
        if (!(ok = wait_warp(S_FULL(i & 1), (i >> 1) & 1, wc, kSiteSFull))) break;
        tc_fence_after();
        uint32_t sv[64];
        tmem_ld32(tmem + lane_off + kTxS + 64 * (i & 1), *reinterpret_cast<uint32_t(*)[32]>(sv));
        tmem_ld32(tmem + lane_off + kTxS + 64 * (i & 1) + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(S_FREE(i & 1));
        const int nv = min(max(lim - (cs + 64 * i) + 1, 0), 64);  // visible keys of this tile
        float x[64], mt = -INFINITY;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          x[j] = j < nv ? __uint_as_float(sv[j]) * args.scale_log2 : -INFINITY;
          mt = fmaxf(mt, x[j]);
        }
        // lazy rescale: move the running maximum only when it grows by more than 2^8
        const bool grow = mt > m_run + 8.f;
        if (__any_sync(0xffffffffu, grow) && i > 0) {
          if (!(ok = wait_warp(PV_DONE((i - 1) & 1), ((i - 1) >> 1) & 1, wc, kSitePEmpty))) break;
          tc_fence_after();
          const float f = grow ? ex2_approx(m_run - mt) : 1.f;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + kTxO + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
            tmem_st32(tmem + lane_off + kTxO + 32 * c, o);
          }
          tmem_wait_st();
        }
        if (grow) {
          l_run *= ex2_approx(m_run - mt);  // 0 while nothing was visible
          m_run = mt;
        }
        const float m_use = m_run == -INFINITY ? 0.f : m_run;
        uint32_t pp[32];
        float ls = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float p0 = ex2_approx(x[2 * j] - m_use), p1 = ex2_approx(x[2 * j + 1] - m_use);
          ls += p0 + p1;
          pp[j] = pack_bf16(p0, p1);
        }
        l_run += ls;
        // P buffer i & 1 is free once PV of tile i - 2 has completed
        if (i >= 2 && !(ok = wait_warp(PV_DONE(i & 1), ((i - 2) >> 1) & 1, wc, kSitePEmpty))) break;
        const uint32_t prow = p_base + (i & 1) * kAtP + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(prow + ((uint32_t)(c ^ (r & 7)) << 4)),
                       "r"(pp[4 * c]), "r"(pp[4 * c + 1]), "r"(pp[4 * c + 2]), "r"(pp[4 * c + 3])
                       : "memory");
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(P_FULL(i & 1));
      }
      if (ok) ok = wait_warp(PV_DONE((n - 1) & 1), ((n - 1) >> 1) & 1, wc, kSiteDrain);
      tc_fence_after();
    }
    // ---- merge with the chunks before this one (log-sum-exp weights) and store
    if (ok && in_range) {
      const bool first = args.chunk_start == 0;
      const float lse_c = l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
      const float lse_a = (!first && row_ok) ? args.acc_lse[row] : -INFINITY;
      const float mx = fmaxf(lse_a, lse_c);
      float lse_new = -INFINITY, wa = 0.f, wc_ = 0.f;
      if (mx > -INFINITY) {
        const float ea = expf(lse_a - mx), ec = expf(lse_c - mx);
        lse_new = mx + logf(ea + ec);
        wa = ea / (ea + ec);
        wc_ = ec / (ea + ec) / (l_run > 0.f ? l_run : 1.f);
      }
      const bool write = row_ok && (n > 0 || last);  // an untouched row keeps its accumulator until the last chunk
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        if (n > 0) {
          tmem_ld32(tmem + lane_off + kTxO + 32 * c, o);
          tmem_wait_ld();
        }
        if (!write) continue;
        float y[32];
        const float* a = args.acc_o + row * kXDim + 32 * c;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          const float4 av = wa != 0.f ? *reinterpret_cast<const float4*>(a + j) : make_float4(0.f, 0.f, 0.f, 0.f);
          y[j] = wa * av.x + (wc_ != 0.f ? wc_ * __uint_as_float(o[j]) : 0.f);
          y[j + 1] = wa * av.y + (wc_ != 0.f ? wc_ * __uint_as_float(o[j + 1]) : 0.f);
          y[j + 2] = wa * av.z + (wc_ != 0.f ? wc_ * __uint_as_float(o[j + 2]) : 0.f);
          y[j + 3] = wa * av.w + (wc_ != 0.f ? wc_ * __uint_as_float(o[j + 3]) : 0.f);
        }
        if (last) {
          uint4* dst = reinterpret_cast<uint4*>(args.out + row * kXDim + 32 * c);
#pragma unroll
          for (int g = 0; g < 4; ++g)
            dst[g] = make_uint4(pack_bf16(y[8 * g], y[8 * g + 1]), pack_bf16(y[8 * g + 2], y[8 * g + 3]),
                                pack_bf16(y[8 * g + 4], y[8 * g + 5]), pack_bf16(y[8 * g + 6], y[8 * g + 7]));
        } else {
          float4* dst = reinterpret_cast<float4*>(args.acc_o + row * kXDim + 32 * c);
#pragma unroll
          for (int g = 0; g < 8; ++g) dst[g] = make_float4(y[4 * g], y[4 * g + 1], y[4 * g + 2], y[4 * g + 3]);
        }
      }
      if (write) (last ? args.lse : args.acc_lse)[row] = lse_new;
    }
  }
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) drain_delay(200000);  // in-flight copies and MMAs land before release
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace mla
