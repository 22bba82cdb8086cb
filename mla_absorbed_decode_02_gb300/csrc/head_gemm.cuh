// Per-head projections around the absorbed decode: query absorption (q~ = q^N W_UK, per
// head) before it and the value projection (o = o~ W_UV, per head) after it ("MLA inference:
// two computation paths and FlashMLA", section "Two equivalent paths", path two: W_UK is
// folded into the query, W_UV applied to the latent output).  Both are one batched GEMM
// over heads: C[t, h, :] = A[t, h, :] . W[h], A of K columns per head, W[h] K x N, N columns
// out per head; tcgen05.mma with M = 128 tokens, N = 256 (or N when smaller) output
// columns, K in chunks of 64 staged by TMA.
#pragma once
#include "common.cuh"
#include "tma4d.cuh"

namespace mla {

constexpr int kHgThreads = 128;
constexpr int kHgRows = 128;                                  // tokens per CTA (MMA M)
constexpr int kHgKChunk = 64;                                 // K per stage (128 bytes of bf16)
constexpr int kHgMaxN = 256;                                  // output columns per CTA (MMA N)
constexpr uint32_t kHgABytes = kHgRows * 128;                 // [128 tokens][64 K] bf16, 128-byte swizzle
constexpr uint32_t kHgBBlock = kHgKChunk * 128;               // [64 K rows][64 N] bf16, 128-byte swizzle
constexpr int kHgMaxStages = 6;
constexpr uint32_t kHgTail = 128;                             // barriers, abort flag, tensor-memory slot
constexpr uint32_t kHgSmemMax = 196608 + 1024 + kHgTail;      // up to 192 KB of stages
// Stage of an n_tile-column CTA: the A chunk and n_tile / 64 blocks of W.
__host__ __device__ constexpr uint32_t hg_stage_bytes(int n_tile) { return kHgABytes + (n_tile / 64) * kHgBBlock; }

struct HeadGemmArgs {
  CUtensorMap map_a;  // A: bf16 {K, H, T}, box {64, 1, 128}, 128-byte swizzle
  CUtensorMap map_w;  // W: bf16 {64, K, N / 64 blocks (128 B apart), H}, box {64, 64, n_tile / 64, 1}, 128-byte swizzle
  void* c;            // C: bf16 [T][H][N]
  int32_t T, H, K, N, n_tile, stages;  // stages: K chunks in flight (2..6)
  uint64_t timeout_ns;
};

// grid: (N / n_tile, H, ceil(T / 128)); one CTA of 128 threads.
__global__ void __launch_bounds__(kHgThreads, 1) mla_head_gemm_kernel(const __grid_constant__ HeadGemmArgs args) {
  extern __shared__ uint8_t hg_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(hg_smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t base = smem_addr(smem);
  const int S = args.stages;
  const uint32_t stage_bytes = hg_stage_bytes(args.n_tile), tail = S * stage_bytes;
  // barriers at the tail: [0, S) stage full, [S, 2S) stage empty, [2S] accumulator done
  const uint32_t bars = base + tail;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + tail + 8 * (2 * kHgMaxStages + 1));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + tail + 8 * (2 * kHgMaxStages + 1) + 8);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int n0 = blockIdx.x * args.n_tile, h = blockIdx.y, t0 = blockIdx.z * kHgRows;
  const int nk = args.K / kHgKChunk, nblk = args.n_tile / 64;

  if (tid == 0) {
    for (int i = 0; i < 2 * S + 1; ++i) mbar_init(bars + 8 * i, 1);
    *abort_flag = 0;
    prefetch_tensormap(&args.map_a);
    prefetch_tensormap(&args.map_w);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait_prerequisites();  // the kernel before this one (the decode, for the projection) is done

  WaitCtx wc;
  wc.abort_local = abort_flag;
  wc.abort_peer = 0;
  wc.timeout_ns = args.timeout_ns;
  if (tid == 0) {
    // producer and MMA issuer in one thread: K chunk k into stage k % S
    const uint64_t pol = l2_policy_evict_first();
    const uint32_t idesc = idesc_bf16_f32(128, args.n_tile, 0, 1);
    auto load = [&](int k) {
      const uint32_t st = k % S, sbase = base + st * stage_bytes;
      mbar_arrive_expect_tx(bars + 8 * st, kHgABytes + nblk * kHgBBlock);
      tma_load_3d(sbase, &args.map_a, bars + 8 * st, k * kHgKChunk, h, t0, pol);
      // the stage's n_tile / 64 blocks of W in one copy (a copy costs the issuing thread the same
      // whatever its size)
      tma_load_4d(sbase + kHgABytes, &args.map_w, bars + 8 * st, 0, k * kHgKChunk, n0 / 64, h, pol);
    };
    bool ok = true;
    for (int k = 0; k < nk && k < S; ++k) load(k);
    for (int k = 0; k < nk && ok; ++k) {
      const uint32_t st = k % S, sbase = base + st * stage_bytes, ph = (k / S) & 1;
      if (!(ok = wait_one(bars + 8 * st, ph, wc, kSiteKvFull))) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kHgKChunk / 16; ++kk)
        mma_bf16_ss(tmem, smem_desc(sbase + kk * 32, 16, 1024, kSwizzle128B),
                    smem_desc(sbase + kHgABytes + kk * 2048, kHgBBlock, 1024, kSwizzle128B), idesc,
                    (k > 0 || kk > 0) ? 1u : 0u);
      mma_commit(bars + 8 * (S + st));
      if (k + S < nk) {  // the stage is refilled once its MMAs have read it
        if (!(ok = wait_one(bars + 8 * (S + st), ph, wc, kSiteKvEmpty))) break;
        load(k + S);
      }
    }
    mma_commit(bars + 8 * (2 * S));
  }
  __syncwarp();
  // ---- epilogue: thread = token row = tensor-memory lane; 32 columns per round
  const bool done = wait_warp(bars + 8 * (2 * S), 0, wc, kSiteDrain);
  tc_fence_after();
  const int t = t0 + tid;
  __nv_bfloat16* crow = reinterpret_cast<__nv_bfloat16*>(args.c) + ((int64_t)t * args.H + h) * args.N + n0;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  for (int c = 0; c < args.n_tile / 32 && done; ++c) {
    uint32_t v[32];
    tmem_ld32(tmem + lane_off + 32 * c, v);
    tmem_wait_ld();
    if (t < args.T) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 o;
        o.x = pack_bf16(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1]));
        o.y = pack_bf16(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
        o.z = pack_bf16(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
        o.w = pack_bf16(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
        *reinterpret_cast<uint4*>(crow + 32 * c + 8 * q) = o;
      }
    }
  }
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) drain_delay(200000);  // in-flight copies and MMAs land before release
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace mla
