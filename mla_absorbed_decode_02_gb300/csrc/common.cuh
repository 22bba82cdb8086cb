// Shared device-side pieces of the decode library: the per-device error word,
// bounded waits, and the kernel argument block.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "plan.h"
#include "ptx.cuh"

namespace mla {

// First error seen by any kernel of this library on this device (0 = none).
// Encoding: MLA_ERR_TIMEOUT (4) + 16 * wait site.
__device__ int g_mla_error = 0;

enum WaitSite : int {
  kSiteQEmpty = 1, kSiteKvEmpty, kSiteQFull, kSiteKvFull, kSiteSEmpty, kSitePFull, kSiteSFull,
  kSiteXFree, kSiteXFull, kSitePEmpty, kSiteDrain, kSiteSelftest, kSiteML,
};

struct WaitCtx {
  volatile int* abort_local;   // this CTA's abort flag (shared memory)
  uint32_t abort_peer;         // the peer CTA's abort flag (shared::cluster address), 0 if none
  uint64_t timeout_ns;
};

__device__ __forceinline__ void raise_abort(const WaitCtx& w, int site) {
  atomicCAS(&g_mla_error, 0, 4 + 16 * site);
  *w.abort_local = 1;
  if (w.abort_peer) asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(w.abort_peer), "r"(1) : "memory");
}

// Bounded wait by one thread (the slow path, out of line).  Returns false if
// the CTA is aborting or the wait ran out (then it raises the abort for this
// CTA and its peer).
template <bool kClusterScope = false>
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const WaitCtx& w, int site) {
  auto poll = [&]() { return kClusterScope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (poll()) return true;
    if ((i & 31) == 0) {
      if (*w.abort_local) return false;
      if (globaltimer_ns() - t0 > w.timeout_ns) {
        raise_abort(w, site);
        return false;
      }
    }
  }
}

// Bounded wait by one thread: one inline poll, then the slow path.
template <bool kClusterScope = false>
__device__ __forceinline__ bool wait_one(uint32_t bar, uint32_t parity, const WaitCtx& w, int site) {
  if (kClusterScope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
  return wait_slow<kClusterScope>(bar, parity, w, site);
}

// Bounded wait by a whole warp; the result is the same in every lane.
template <bool kClusterScope = false>
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const WaitCtx& w, int site) {
  const bool ok = wait_one<kClusterScope>(bar, parity, w, site);
  return __all_sync(0xffffffffu, ok);
}

// After an abort: give in-flight asynchronous copies and MMAs time to land
// before shared memory and tensor memory are released.
__device__ __forceinline__ void drain_delay(uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < ns) {
  }
}

struct DecodeArgs {
  CUtensorMap map_qr;    // q^R half: bf16 {64, H, NQB}, box {32, 128, 1}, 64-byte swizzle (FP8 QK:
                         // the same view of the RoPE values inside the 656-byte query rows)
  CUtensorMap map_kvc;   // bf16 cache: latent of 64 rows, box {64 dims, 64 rows}, 128-byte swizzle;
                         // FP8 cache (bytes): the 256 codes of one half, box {256, 64}, no swizzle;
                         // FP8 QK: one 128-code tile, box {128, 64}, 128-byte swizzle
  CUtensorMap map_kvr;   // RoPE key of 64 rows: bf16 box {32 dims, 64 rows} / bytes {64, 64}, 64-byte swizzle
  CUtensorMap map_kvs;   // FP8 cache: the 4 tile scales of 64 rows, box {16 bytes, 64}, no swizzle
  const void* q_nope;    // absorbed queries, bf16 [NQB][H][512] (read by threads into tensor memory);
                         // FP8 QK: 656-byte query rows [NQB][H] (512 codes, 4 scales, RoPE)
  const void* q_rope;    // RoPE queries, bf16 [NQB][H][64] (loaded by TMA; read here only to prefetch into L2)
  const int32_t* block_table;
  const int32_t* seqlens;
  const int32_t* sched;
  void* out;
  float* lse;
  float* o_acc;          // split partials [slots][H][512], normalised
  float* lse_acc;        // [slots][H]
  float scale_log2;      // softmax scale * log2(e)
  int32_t H, s_q, causal, max_pages, out_f32, num_units, num_qb, kv_fp8, qk_fp8;
  int32_t group;         // G: new tokens per work block; a unit is a cluster of 2G CTAs, one pair per token
  uint64_t timeout_ns;
};

}  // namespace mla
