// libmla_decode.so: C ABI (include/mla_decode.h) and the small kernels around
// the decode kernel -- split planning, LSE combine, bounded-wait self test.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/mla_decode.h"
#include "decode_kernel.cuh"
#include "head_gemm.cuh"
#include "extend_kernel.cuh"

namespace mla {

// ----------------------------------------------------------------- split planner (device twin)
// One CTA of 1024 threads runs the planner phases of plan.h (the prefix sums on one thread).
__global__ void __launch_bounds__(1024) mla_sched_kernel(const int32_t* seqlens, int B, int s_q, int causal, int G,
                                                         int U, int32_t* sched) {
  __shared__ int64_t sh_total;
  const int NQB = B * s_q, NWB = NQB / G, tid = threadIdx.x, nt = blockDim.x;
  int32_t* units = sched + kSchedHeader;
  int32_t* num_splits = units + kUnitInts * U;
  int32_t* pos = num_splits + NQB;  // scratch until the last phase (one entry per work block)
  plan_phase_cost(seqlens, s_q, causal, G, NWB, pos, tid, nt);
  // a negative length is outside the contract: reported, and planned as an empty sequence
  for (int b = tid; b < B; b += nt)
    if (seqlens[b] < 0) atomicCAS(&g_mla_error, 0, MLA_ERR_INVALID_ARG);
  __syncthreads();
  if (tid == 0) sh_total = plan_phase_scan(pos, NWB);
  __syncthreads();
  if (sh_total > kMaxPlanPositions) {  // more work positions than an int32 holds: refuse the plan
    if (tid == 0) {
      plan_refuse(sched);
      atomicCAS(&g_mla_error, 0, MLA_ERR_INVALID_ARG);
    }
    return;
  }
  const int64_t total = sh_total, Bq = plan_budget(total, U);
  plan_phase_units(seqlens, s_q, causal, G, NWB, pos, total, Bq, U, units, tid, nt);
  plan_phase_splits(seqlens, s_q, causal, G, NWB, pos, Bq, num_splits, tid, nt);
  __syncthreads();
  if (tid == 0) plan_phase_finish(NQB, U, G, Bq, sched);
}

// ----------------------------------------------------------------- LSE combine of split partials
// out = sum_i exp(lse_i - lse) * out_i, lse = M + ln sum_i exp(lse_i - M), M = max_i lse_i
// (the merge of split-KV partial results, "MLA inference: two computation paths and
// FlashMLA", section "Decode attention becomes a compute problem").  Query blocks that see
// no key get out = 0, lse = -inf.  One CTA of 256 threads per (query block, 16 heads, one
// of Z column slices): the 16 combined LSEs first (two heads per warp, the splits spread
// over 16 lanes), then 16 threads per head stream the slice's float4 columns of every
// split, kNf columns each, the splits dealt round-robin over kG adjacent lanes (summed by
// shuffles at the end), four of a lane's splits in flight together.  The host picks Z (and
// with it kG, kNf) from the splits per query block it expects: long sequences split over
// many units are merged by many more CTAs.
constexpr int kCombineHeads = 16;
template <int kG, int kNf>
__global__ void __launch_bounds__(256) mla_combine_kernel(const int32_t* sched, int U, int NQB, int H,
                                                          const float* o_acc, const float* lse_acc, void* out,
                                                          float* lse, int out_f32) {
  pdl_wait_prerequisites();  // the decode kernel before it in the stream has finished
  // metadata for other params, or a refused plan: nothing to merge (the decode kernel has
  // reported it in the device error word)
  if (sched[0] != kSchedMagic || sched[1] != U || sched[2] != NQB) return;
  constexpr int kW = kNf * 16 / kG;  // float4 columns of a slice (of 128 per head)
  const int qb = blockIdx.x, h0 = blockIdx.y * kCombineHeads, slice = blockIdx.z;
  const int32_t* num_splits = sched + kSchedHeader + kUnitInts * U;
  const int32_t* split_offset = num_splits + NQB;
  const int ns = num_splits[qb];
  if (ns == 1) return;  // the decode kernel wrote this query block's output itself
  const int off = ns > 1 ? split_offset[qb] : 0;
  __shared__ float s_lse[kCombineHeads];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {
    const int hh = 2 * warp + (lane >> 4), h = h0 + hh, sub = lane & 15;
    float M = -INFINITY;
    for (int i = sub; i < ns && h < H; i += 16) M = fmaxf(M, lse_acc[(int64_t)(off + i) * H + h]);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float S = 0.f;
    if (M > -INFINITY)
      for (int i = sub; i < ns && h < H; i += 16) S += expf(lse_acc[(int64_t)(off + i) * H + h] - M);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
    if (sub == 0) s_lse[hh] = M > -INFINITY ? M + logf(S) : -INFINITY;
  }
  __syncthreads();
  const int hh = tid >> 4, h = h0 + hh, sub = tid & 15, g = sub % kG, ci = sub / kG;
  const float L = s_lse[hh];
  const int64_t split_stride = (int64_t)H * 128;  // float4 per split
  const int c0 = kW * slice + ci;                 // first float4 column; then every 16 / kG
  const float4* src = reinterpret_cast<const float4*>(o_acc) + ((int64_t)off * H + (h < H ? h : 0)) * 128 + c0;
  const float* lsrc = lse_acc + (int64_t)off * H + (h < H ? h : 0);
  float4 acc[kNf];
#pragma unroll
  for (int f = 0; f < kNf; ++f) acc[f] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (h < H) {
    for (int i0 = g; i0 < ns; i0 += 4 * kG) {
      float4 v[4][kNf];
      float wgt[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = i0 + k * kG;
        const bool in = i < ns;
        wgt[k] = in ? lsrc[(int64_t)i * H] : -INFINITY;
#pragma unroll
        for (int f = 0; f < kNf; ++f)
          v[k][f] = in ? __ldcs(src + i * split_stride + f * (16 / kG)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float wk = L > -INFINITY ? expf(wgt[k] - L) : 0.f;  // every split empty: out = 0
#pragma unroll
        for (int f = 0; f < kNf; ++f) {
          acc[f].x += wk * v[k][f].x;
          acc[f].y += wk * v[k][f].y;
          acc[f].z += wk * v[k][f].z;
          acc[f].w += wk * v[k][f].w;
        }
      }
    }
  }
#pragma unroll
  for (int o = 1; o < kG; o <<= 1)
#pragma unroll
    for (int f = 0; f < kNf; ++f) {
      acc[f].x += __shfl_xor_sync(0xffffffffu, acc[f].x, o);
      acc[f].y += __shfl_xor_sync(0xffffffffu, acc[f].y, o);
      acc[f].z += __shfl_xor_sync(0xffffffffu, acc[f].z, o);
      acc[f].w += __shfl_xor_sync(0xffffffffu, acc[f].w, o);
    }
  if (h >= H || g != 0) return;
  const int64_t row = (int64_t)qb * H + h;
#pragma unroll
  for (int f = 0; f < kNf; ++f) {
    const int d = 4 * (c0 + f * (16 / kG));
    if (out_f32) {
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + row * 512 + d) = acc[f];
    } else {
      uint2 o;
      o.x = pack_bf16(acc[f].x, acc[f].y);
      o.y = pack_bf16(acc[f].z, acc[f].w);
      *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + row * 512 + d) = o;
    }
  }
  if (ci == 0 && slice == 0) lse[row] = L;
}

// ----------------------------------------------------------------- FP8 cache writer
// bf16 rows [576] (latent 512 + RoPE 64) -> 656-byte FP8 rows: 512 E4M3 codes, the 4
// float32 tile scales, the 64 bf16 RoPE values unchanged.  Per 128-element tile:
// scale = amax / 448 (1 if the tile is all zero), code = E4M3(x / scale) rounded to
// nearest even, the quotient first clamped to the E4M3 range +-448 ("MLA and FP8 MoE
// Serving: Multi-Head Latent Attention at Scale", section "Understanding FP8 Formats:
// E4M3 vs. E5M2").  One warp per token; lane l owns latent elements [16 l, 16 l + 16),
// so a tile is 8 lanes.
// (latent row `tok` at lat + tok * lat_stride, its 64 RoPE values at rope + tok * rope_stride: one
// 576-element cache row, or a query's two arrays)
__global__ void __launch_bounds__(256) mla_quantize_fp8_kernel(const __nv_bfloat16* lat, int64_t lat_stride,
                                                               const __nv_bfloat16* rope, int64_t rope_stride,
                                                               uint8_t* out, int64_t n) {
  const int64_t tok = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (tok >= n) return;
  const __nv_bfloat16* src = lat + tok * lat_stride;
  const __nv_bfloat16* src_r = rope + tok * rope_stride;
  uint8_t* dst = out + tok * 656;
  float x[16];
  {
    const uint4 a = *reinterpret_cast<const uint4*>(src + 16 * lane);
    const uint4 b = *reinterpret_cast<const uint4*>(src + 16 * lane + 8);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = amax > 0.f ? amax / 448.f : 1.f;
  uint32_t codes[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float y = fminf(fmaxf(x[i] / scale, -448.f), 448.f);
    const uint32_t c = (uint32_t)__nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3);
    codes[i >> 2] |= c << (8 * (i & 3));
  }
  *reinterpret_cast<uint4*>(dst + 16 * lane) = make_uint4(codes[0], codes[1], codes[2], codes[3]);
  if ((lane & 7) == 0) *reinterpret_cast<float*>(dst + 512 + 4 * (lane >> 3)) = scale;
  if (lane < 8) *reinterpret_cast<uint4*>(dst + 528 + 16 * lane) = *reinterpret_cast<const uint4*>(src_r + 8 * lane);
}

// ----------------------------------------------------------------- bounded-wait self test
// One CTA waits on a barrier that nothing ever completes; the bounded wait runs
// out, records MLA_ERR_TIMEOUT in the device error word and the kernel returns.
__global__ void mla_wait_selftest_kernel(uint64_t timeout_ns) {
  __shared__ uint64_t barrier_word;
  __shared__ int abort_word;
  const uint32_t b = smem_addr(&barrier_word);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    abort_word = 0;
    fence_mbar_init();
  }
  __syncthreads();
  WaitCtx w;
  w.abort_local = &abort_word;
  w.abort_peer = 0;
  w.timeout_ns = timeout_ns;
  wait_warp(b, 0, w, kSiteSelftest);
}

}  // namespace mla

// =================================================================== host side
namespace {

using namespace mla;

struct DeviceInfo {
  bool ready = false;
  int sm_count = 0;
  int max_clusters[5] = {0, 0, 0, 0, 0};  // [G]: clusters of 2G decode CTAs that fit at once
};
std::mutex g_mu;
DeviceInfo g_dev[64];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int32_t device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MLA_ERR_CUDA;
    for (const void* k : {(const void*)mla_decode_bf16_kernel, (const void*)mla_decode_fp8_kernel,
                          (const void*)mla_decode_bf16_group_kernel, (const void*)mla_decode_fp8_group_kernel,
                          (const void*)mla_decode_fp8qk_kernel})
      if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
        return MLA_ERR_CUDA;
    for (int G = 1; G <= 4; ++G) {  // GPCs hold whole clusters: bigger ones leave SMs idle
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * G * (d.sm_count / (2 * G)), 1, 1);
      cfg.blockDim = dim3(kThreads, 1, 1);
      cfg.dynamicSmemBytes = kSmemBytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2 * G;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, (void*)mla_decode_bf16_kernel, &cfg) != cudaSuccess || n <= 0)
        n = d.sm_count / (2 * G);
      d.max_clusters[G] = n;
    }
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return MLA_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    d.ready = true;
  }
  *out = &d;
  return MLA_OK;
}

int32_t check_params(const mla_decode_params* p) {
  if (!p) return MLA_ERR_INVALID_ARG;
  if (p->batch < 1 || p->num_heads < 1 || p->num_pages < 1 || p->max_pages_per_seq < 1) return MLA_ERR_INVALID_ARG;
  if (p->s_q < 1 || p->page_size < 1 || p->num_units < 0 || p->timeout_us < 0) return MLA_ERR_INVALID_ARG;
  for (int i = 0; i < 3; ++i)
    if (p->reserved[i] != 0) return MLA_ERR_INVALID_ARG;
  if (p->qk_fp8 != 0 && (p->qk_fp8 != 1 || p->kv_dtype != MLA_KV_FP8_E4M3)) return MLA_ERR_INVALID_ARG;
  if (p->token_group < 0 || p->token_group > 4 || (p->token_group > 0 && p->s_q % p->token_group != 0))
    return MLA_ERR_INVALID_ARG;
  if (p->kv_dtype != MLA_KV_BF16 && p->kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (p->out_dtype != MLA_OUT_BF16 && p->out_dtype != MLA_OUT_F32) return MLA_ERR_INVALID_ARG;
  if (p->page_size != 64 || p->s_q > 8 || p->num_heads > 128) return MLA_ERR_UNSUPPORTED;
  if ((int64_t)p->batch * p->s_q > (1 << 24) || (int64_t)p->num_pages * 64 > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  if (p->qk_fp8 && p->token_group > 1) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

// New tokens per work block: the caller's token_group, else 1.  A group of G tokens reads each
// page once instead of G times, but GPCs hold whole clusters: clusters of 4 CTAs fill 144 of
// the 152 SMs, of 8 CTAs 120, so where the decode is bound by the SMs' work rather than by
// DRAM (every s_q >= 2 workload measured) the per-token mode is the faster one.
int resolve_group(const mla_decode_params* p) { return p->token_group > 0 ? p->token_group : 1; }

int32_t resolve_units(const mla_decode_params* p, int32_t* U) {
  if (p->num_units > 0) {
    *U = p->num_units;
    return MLA_OK;
  }
  DeviceInfo* d = nullptr;
  int32_t st = device_info(&d);
  if (st != MLA_OK) return st;
  *U = d->max_clusters[resolve_group(p)];
  return MLA_OK;
}

// Split-partial slots: each unit boundary splits at most one work block, and each split block
// takes one slot per split for each of its G query blocks.
size_t partial_slots(const mla_decode_params* p, int32_t U) {
  return (size_t)p->batch * p->s_q + (size_t)resolve_group(p) * U;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int32_t encode_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* ptr, const uint64_t* dims,
                   const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle sw) {
  cuuint64_t gd[5];
  cuuint64_t gs[4];
  cuuint32_t bx[5], es[5] = {1, 1, 1, 1, 1};
  if (rank < 1 || rank > 5) return MLA_ERR_INVALID_ARG;
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
  CUresult r = g_encode(m, dt, rank, const_cast<void*>(ptr), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_CUDA;
}

// Tensor maps of recent calls.  A decode step calls the library once per layer with the
// same query buffers and, per layer, its own cache pool; encoding the four maps on the host
// every call costs microseconds, so the last few sets are kept, keyed on everything the
// maps encode (device, base pointers, extents, cache format).
struct MapKey {
  int dev;
  const void* q_rope;
  const void* kv;
  int H, NQB, num_pages, kv_dtype, qk8;  // qk8: q_rope is the 656-byte FP8 query rows
  bool operator==(const MapKey& o) const {
    return dev == o.dev && q_rope == o.q_rope && kv == o.kv && H == o.H && NQB == o.NQB &&
           num_pages == o.num_pages && kv_dtype == o.kv_dtype && qk8 == o.qk8;
  }
};
struct MapSet {
  MapKey key;
  bool valid = false;
  CUtensorMap qr, kvc, kvr, kvs;
};
constexpr int kMapCache = 16;
MapSet g_maps[kMapCache];
int g_map_next = 0;

int32_t encode_maps(const MapKey& k, MapSet* m) {
  int32_t st;
  {
    // q^R: its own bf16 array, or (FP8 QK) the 64 bf16 at byte 528 of each 656-byte query row
    const void* q = k.qk8 ? static_cast<const void*>(static_cast<const char*>(k.q_rope) + 528) : k.q_rope;
    const uint64_t row = k.qk8 ? 656 : 64 * 2;
    const uint64_t d[3] = {64, (uint64_t)k.H, (uint64_t)k.NQB};
    const uint64_t s[2] = {row, (uint64_t)k.H * row};
    const uint32_t bx[3] = {32, 128, 1};
    if ((st = encode_map(&m->qr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, d, s, bx, CU_TENSOR_MAP_SWIZZLE_64B)))
      return st;
  }
  if (k.kv_dtype == MLA_KV_BF16) {
    const uint64_t d[2] = {576, (uint64_t)k.num_pages * 64};
    const uint64_t s[1] = {576 * 2};
    const uint32_t bc[2] = {64, 64}, br[2] = {32, 64};
    if ((st = encode_map(&m->kvc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, k.kv, d, s, bc, CU_TENSOR_MAP_SWIZZLE_128B)))
      return st;
    if ((st = encode_map(&m->kvr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, k.kv, d, s, br, CU_TENSOR_MAP_SWIZZLE_64B)))
      return st;
    m->kvs = m->kvr;  // unused
  } else {  // FP8 rows of 656 bytes: 512 codes, 4 float32 scales, 64 bf16 RoPE
    const uint64_t d[2] = {656, (uint64_t)k.num_pages * 64};
    const uint64_t s[1] = {656};
    const uint32_t bc[2] = {256, 64}, bc8[2] = {128, 64}, br[2] = {64, 64}, bs[2] = {16, 64};
    if (k.qk8) {  // one 128-code tile in the swizzled K-major layout the QK MMAs read
      if ((st = encode_map(&m->kvc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, k.kv, d, s, bc8, CU_TENSOR_MAP_SWIZZLE_128B)))
        return st;
    } else if ((st = encode_map(&m->kvc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, k.kv, d, s, bc, CU_TENSOR_MAP_SWIZZLE_NONE))) {
      return st;
    }
    if ((st = encode_map(&m->kvr, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, k.kv, d, s, br, CU_TENSOR_MAP_SWIZZLE_64B)))
      return st;
    if ((st = encode_map(&m->kvs, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, k.kv, d, s, bs, CU_TENSOR_MAP_SWIZZLE_NONE)))
      return st;
  }
  m->key = k;
  m->valid = true;
  return MLA_OK;
}

// The maps for key k into args: from the cache, or encoded now (and cached).
int32_t tensor_maps(const MapKey& k, DecodeArgs* a) {
  std::lock_guard<std::mutex> lk(g_mu);
  const MapSet* hit = nullptr;
  for (const MapSet& m : g_maps)
    if (m.valid && m.key == k) {
      hit = &m;
      break;
    }
  if (!hit) {
    MapSet fresh;
    const int32_t st = encode_maps(k, &fresh);
    if (st != MLA_OK) return st;
    g_maps[g_map_next] = fresh;
    hit = &g_maps[g_map_next];
    g_map_next = (g_map_next + 1) % kMapCache;
  }
  a->map_qr = hit->qr;
  a->map_kvc = hit->kvc;
  a->map_kvr = hit->kvr;
  a->map_kvs = hit->kvs;
  return MLA_OK;
}

}  // namespace

extern "C" {

const char* mla_status_string(int32_t s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
    case MLA_ERR_SCRATCH_LIMIT: return "MLA_ERR_SCRATCH_LIMIT";
    default: return "MLA_ERR_UNKNOWN";
  }
}

int32_t mla_resolve_num_units(const mla_decode_params* p, int32_t* num_units) {
  int32_t st = check_params(p);
  if (st != MLA_OK) return st;
  if (!num_units) return MLA_ERR_INVALID_ARG;
  return resolve_units(p, num_units);
}

int32_t mla_get_workspace_size(const mla_decode_params* p, size_t* sched_bytes, size_t* workspace_bytes) {
  int32_t st = check_params(p);
  if (st != MLA_OK) return st;
  if (!sched_bytes || !workspace_bytes) return MLA_ERR_INVALID_ARG;
  int32_t U = 0;
  if ((st = resolve_units(p, &U)) != MLA_OK) return st;
  const int64_t nqb = (int64_t)p->batch * p->s_q;
  *sched_bytes = sizeof(int32_t) * (size_t)sched_ints(U, (int)nqb);
  const size_t slots = partial_slots(p, U);
  *workspace_bytes = align256(slots * p->num_heads * 512 * sizeof(float)) + align256(slots * p->num_heads * sizeof(float));
  return MLA_OK;
}

int32_t mla_plan_host(const mla_decode_params* p, int32_t num_units, const int32_t* cache_seqlens, void* sched) {
  int32_t st = check_params(p);
  if (st != MLA_OK) return st;
  if (num_units < 1 || !cache_seqlens || !sched) return MLA_ERR_INVALID_ARG;
  for (int b = 0; b < p->batch; ++b)
    if (cache_seqlens[b] < 0) return MLA_ERR_INVALID_ARG;
  return plan_units(cache_seqlens, p->batch, p->s_q, p->causal != 0, resolve_group(p), num_units,
                    static_cast<int32_t*>(sched))
             ? MLA_OK
             : MLA_ERR_INVALID_ARG;
}

int32_t mla_get_scheduler_metadata(const mla_decode_params* p, const int32_t* cache_seqlens, void* sched,
                                   void* stream) {
  int32_t st = check_params(p);
  if (st != MLA_OK) return st;
  if (!cache_seqlens || !sched) return MLA_ERR_INVALID_ARG;
  int32_t U = 0;
  if ((st = resolve_units(p, &U)) != MLA_OK) return st;
  mla_sched_kernel<<<1, 1024, 0, static_cast<cudaStream_t>(stream)>>>(
      cache_seqlens, p->batch, p->s_q, p->causal != 0, resolve_group(p), U, static_cast<int32_t*>(sched));
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int32_t mla_decode_splitkv(const mla_decode_params* p, const void* q_nope_absorbed, const void* q_rope,
                           const void* kv_pages, const int32_t* block_table, const int32_t* cache_seqlens, float scale,
                           void* out, float* lse, const void* sched, void* workspace, void* stream) {
  int32_t st = check_params(p);
  if (st != MLA_OK) return st;
  // (FP8 QK: the query is the FP8 rows alone; q_rope is not read)
  const bool qk8 = p->qk_fp8 != 0;
  const void* ptrs[] = {q_nope_absorbed, qk8 ? q_nope_absorbed : q_rope, kv_pages, block_table, cache_seqlens,
                        out, lse, sched, workspace};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return MLA_ERR_INVALID_ARG;  // the kernel takes row maxima before scaling
  DeviceInfo* dinfo = nullptr;
  if ((st = device_info(&dinfo)) != MLA_OK) return st;
  int32_t U = 0;
  if ((st = resolve_units(p, &U)) != MLA_OK) return st;
  const int H = p->num_heads, NQB = p->batch * p->s_q, G = resolve_group(p);
  const size_t slots = partial_slots(p, U);

  DecodeArgs a;
  std::memset(&a, 0, sizeof a);
  {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    const MapKey key{dev, qk8 ? q_nope_absorbed : q_rope, kv_pages, H, NQB, p->num_pages, p->kv_dtype, qk8 ? 1 : 0};
    if ((st = tensor_maps(key, &a)) != MLA_OK) return st;
  }
  a.kv_fp8 = p->kv_dtype == MLA_KV_FP8_E4M3;
  a.qk_fp8 = qk8 ? 1 : 0;
  a.q_nope = q_nope_absorbed;
  a.q_rope = q_rope;
  a.block_table = block_table;
  a.seqlens = cache_seqlens;
  a.sched = static_cast<const int32_t*>(sched);
  a.out = out;
  a.lse = lse;
  a.o_acc = static_cast<float*>(workspace);
  a.lse_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(slots * H * 512 * sizeof(float)));
  a.scale_log2 = scale * 1.4426950408889634f;
  a.H = H;
  a.s_q = p->s_q;
  a.causal = p->causal != 0;
  a.max_pages = p->max_pages_per_seq;
  a.out_f32 = p->out_dtype == MLA_OUT_F32;
  a.num_units = U;
  a.num_qb = NQB;
  a.group = G;
  a.timeout_ns = (uint64_t)(p->timeout_us > 0 ? p->timeout_us : 2000000) * 1000ull;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * G * U, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = static_cast<cudaStream_t>(stream);
  // one unit = a cluster of 2G CTAs; programmatic dependent launch: the kernel's set-up
  // (barriers, tensor memory) overlaps the end of the kernel before it in the stream, and it
  // waits (griddepcontrol.wait) before reading any global memory
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2 * G;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = qk8      ? cudaLaunchKernelEx(&cfg, mla_decode_fp8qk_kernel, a)
                        : G > 1 ? (a.kv_fp8 ? cudaLaunchKernelEx(&cfg, mla_decode_fp8_group_kernel, a)
                                            : cudaLaunchKernelEx(&cfg, mla_decode_bf16_group_kernel, a))
                                : (a.kv_fp8 ? cudaLaunchKernelEx(&cfg, mla_decode_fp8_kernel, a)
                                            : cudaLaunchKernelEx(&cfg, mla_decode_bf16_kernel, a));
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int32_t mla_combine(const mla_decode_params* p, void* out, float* lse, const void* sched, void* workspace,
                    void* stream) {
  int32_t st = check_params(p);
  if (st != MLA_OK) return st;
  const void* ptrs[] = {out, lse, sched, workspace};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return MLA_ERR_INVALID_ARG;
  int32_t U = 0;
  if ((st = resolve_units(p, &U)) != MLA_OK) return st;
  const int H = p->num_heads, NQB = p->batch * p->s_q;
  const size_t slots = partial_slots(p, U);
  const float* o_acc = static_cast<const float*>(workspace);
  const float* lse_acc =
      reinterpret_cast<const float*>(static_cast<const char*>(workspace) + align256(slots * H * 512 * sizeof(float)));
  // Column slices per (query block, 16 heads): enough CTAs for the splits a query block is
  // expected to have when the units are spread over the query blocks (1 + U / NQB).
  const int expect = 1 + (U + NQB - 1) / NQB;
  const int Z = expect <= 4 ? 4 : expect <= 8 ? 8 : expect <= 16 ? 16 : 32;
  // programmatic dependent launch: this grid is set up while the decode kernel before it
  // drains, and waits (griddepcontrol.wait) for it before reading the partials
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(NQB, (H + kCombineHeads - 1) / kCombineHeads, Z);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int32_t* sc = static_cast<const int32_t*>(sched);
  const int of32 = (int)(p->out_dtype == MLA_OUT_F32);
  cudaError_t e;
  if (Z == 4)
    e = cudaLaunchKernelEx(&cfg, mla_combine_kernel<1, 2>, sc, U, NQB, H, o_acc, lse_acc, out, lse, of32);
  else if (Z == 8)
    e = cudaLaunchKernelEx(&cfg, mla_combine_kernel<1, 1>, sc, U, NQB, H, o_acc, lse_acc, out, lse, of32);
  else if (Z == 16)
    e = cudaLaunchKernelEx(&cfg, mla_combine_kernel<2, 1>, sc, U, NQB, H, o_acc, lse_acc, out, lse, of32);
  else
    e = cudaLaunchKernelEx(&cfg, mla_combine_kernel<4, 1>, sc, U, NQB, H, o_acc, lse_acc, out, lse, of32);
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int32_t mla_decode(const mla_decode_params* p, const void* q_nope_absorbed, const void* q_rope, const void* kv_pages,
                   const int32_t* block_table, const int32_t* cache_seqlens, float scale, void* out, float* lse,
                   const void* sched, void* workspace, void* stream) {
  int32_t st = mla_decode_splitkv(p, q_nope_absorbed, q_rope, kv_pages, block_table, cache_seqlens, scale, out, lse,
                                  sched, workspace, stream);
  if (st != MLA_OK) return st;
  return mla_combine(p, out, lse, sched, workspace, stream);
}

int32_t mla_device_error(int32_t* word, int32_t clear) {
  if (!word) return MLA_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MLA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_mla_error, sizeof v) != cudaSuccess) return MLA_ERR_CUDA;
  *word = v;
  if (clear) {
    int z = 0;
    if (cudaMemcpyToSymbol(g_mla_error, &z, sizeof z) != cudaSuccess) return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

int32_t mla_quantize_kv_fp8(const void* kv_bf16, void* kv_fp8, int64_t num_tokens, void* stream) {
  if (!kv_bf16 || !kv_fp8 || num_tokens < 0 || !aligned16(kv_bf16) || !aligned16(kv_fp8)) return MLA_ERR_INVALID_ARG;
  if (num_tokens == 0) return MLA_OK;
  const int64_t blocks = (num_tokens + 7) / 8;
  if (blocks > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  const __nv_bfloat16* kv = static_cast<const __nv_bfloat16*>(kv_bf16);
  mla_quantize_fp8_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      kv, 576, kv + 512, 576, static_cast<uint8_t*>(kv_fp8), num_tokens);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int32_t mla_quantize_q_fp8(const void* q_nope_absorbed, const void* q_rope, void* q_fp8, int64_t num_rows,
                           void* stream) {
  if (!q_nope_absorbed || !q_rope || !q_fp8 || num_rows < 0) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_nope_absorbed) || !aligned16(q_rope) || !aligned16(q_fp8)) return MLA_ERR_INVALID_ARG;
  if (num_rows == 0) return MLA_OK;
  const int64_t blocks = (num_rows + 7) / 8;
  if (blocks > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  mla_quantize_fp8_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(q_nope_absorbed), 512, static_cast<const __nv_bfloat16*>(q_rope), 64,
      static_cast<uint8_t*>(q_fp8), num_rows);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

// Per-head GEMM C[t, h, :] = A[t, h, :] . W[h] (K x N per head), bf16 in and out, fp32 accumulation.
static int32_t launch_head_gemm(int32_t T, int32_t H, int32_t K, int32_t N, const void* a, const void* w, void* c,
                                void* stream) {
  if (T < 1 || H < 1 || H > 65535 || !a || !w || !c) return MLA_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(w) || !aligned16(c)) return MLA_ERR_INVALID_ARG;
  if (K < 64 || K % 64 != 0 || N < 64 || N % 64 != 0 || K > 4096 || N > 4096) return MLA_ERR_UNSUPPORTED;
  if ((int64_t)T * H * (K > N ? K : N) > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  DeviceInfo* dinfo = nullptr;
  int32_t st = device_info(&dinfo);
  if (st != MLA_OK) return st;
  static bool attr_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MLA_ERR_CUDA;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(mla_head_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kHgSmemMax) !=
        cudaSuccess)
      return MLA_ERR_CUDA;
    attr_set[dev] = true;
  }
  HeadGemmArgs g;
  std::memset(&g, 0, sizeof g);
  {
    const uint64_t d[3] = {(uint64_t)K, (uint64_t)H, (uint64_t)T};
    const uint64_t s[2] = {(uint64_t)K * 2, (uint64_t)H * K * 2};
    const uint32_t bx[3] = {64, 1, (uint32_t)kHgRows};
    if ((st = encode_map(&g.map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a, d, s, bx, CU_TENSOR_MAP_SWIZZLE_128B)))
      return st;
  }
  g.n_tile = N % kHgMaxN == 0 ? kHgMaxN : (N % 128 == 0 ? 128 : 64);
  {  // W [H][K][N] as {64, K rows, N / 64 blocks (128 B apart), H}: a stage's blocks in one box
    const uint64_t d[4] = {64, (uint64_t)K, (uint64_t)(N / 64), (uint64_t)H};
    const uint64_t s[3] = {(uint64_t)N * 2, 128, (uint64_t)K * N * 2};
    const uint32_t bx[4] = {64, (uint32_t)kHgKChunk, (uint32_t)(g.n_tile / 64), 1};
    if ((st = encode_map(&g.map_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, w, d, s, bx, CU_TENSOR_MAP_SWIZZLE_128B)))
      return st;
  }
  g.c = c;
  g.T = T;
  g.H = H;
  g.K = K;
  g.N = N;
  g.timeout_ns = 2000000000ull;
  // K chunks in flight: all of them (up to six, 192 KB) when the grid fits one CTA per SM, two
  // (two CTAs per SM) when it is larger
  const int64_t ctas = (int64_t)(N / g.n_tile) * H * ((T + kHgRows - 1) / kHgRows);
  const int nk = K / kHgKChunk;
  const uint32_t sb = hg_stage_bytes(g.n_tile);
  int stages = ctas <= dinfo->sm_count ? (int)(196608 / sb) : 2;
  stages = stages > kHgMaxStages ? kHgMaxStages : stages;
  stages = stages > nk ? nk : stages;
  g.stages = stages < 2 ? 2 : stages;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(N / g.n_tile, H, (T + kHgRows - 1) / kHgRows);
  cfg.blockDim = dim3(kHgThreads, 1, 1);
  cfg.dynamicSmemBytes = g.stages * sb + 1024 + kHgTail;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_head_gemm_kernel, g) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int32_t mla_absorb_query(int32_t n_tokens, int32_t num_heads, int32_t d_nope, const void* q_nope, const void* w_uk,
                         void* q_absorbed, void* stream) {
  return launch_head_gemm(n_tokens, num_heads, d_nope, 512, q_nope, w_uk, q_absorbed, stream);
}

int32_t mla_project_output(int32_t n_tokens, int32_t num_heads, int32_t d_v, const void* o_latent, const void* w_uv,
                           void* out, void* stream) {
  return launch_head_gemm(n_tokens, num_heads, 512, d_v, o_latent, w_uv, out, stream);
}

// ------------------------------------------------------------------ extend by the expand path
static int32_t check_extend(const mla_extend_params* p) {
  if (!p) return MLA_ERR_INVALID_ARG;
  if (p->batch < 1 || p->s_q < 1 || p->num_heads < 1 || p->num_pages < 1 || p->max_pages_per_seq < 1 ||
      p->max_seqlen < 1 || p->chunk_tokens < 1 || p->timeout_us < 0)
    return MLA_ERR_INVALID_ARG;
  for (int i = 0; i < 5; ++i)
    if (p->reserved[i] != 0) return MLA_ERR_INVALID_ARG;
  if (p->s_q > p->max_seqlen || (int64_t)p->max_seqlen > (int64_t)p->max_pages_per_seq * 64) return MLA_ERR_INVALID_ARG;
  if (p->page_size != 64 || p->d_nope != kXDim || p->d_v != kXDim || p->num_heads > 128 || p->chunk_tokens % 128 != 0)
    return MLA_ERR_UNSUPPORTED;
  if (p->batch > 65535 || (int64_t)p->num_pages * 64 > INT32_MAX || (int64_t)p->batch * p->num_heads > INT32_MAX ||
      (int64_t)p->batch * p->s_q * p->num_heads > INT32_MAX)
    return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

struct ExtendLayout {
  size_t kv, acc_o, acc_lse, total;  // bytes of K^N (and of V), of the output and lse accumulators
};
static ExtendLayout extend_layout(const mla_extend_params* p) {
  ExtendLayout l;
  l.kv = align256((size_t)p->batch * p->num_heads * p->chunk_tokens * kXDim * 2);  // half of the [K^N | V] rows
  l.acc_o = align256((size_t)p->batch * p->s_q * p->num_heads * kXDim * 4);
  l.acc_lse = align256((size_t)p->batch * p->s_q * p->num_heads * 4);
  l.total = 2 * l.kv + l.acc_o + l.acc_lse;
  return l;
}

static void pdl_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, void* stream) {
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg->attrs = attr;
  cfg->numAttrs = 1;
  cfg->stream = static_cast<cudaStream_t>(stream);
}

static int32_t extend_attrs(DeviceInfo** dinfo) {
  int32_t st = device_info(dinfo);
  if (st != MLA_OK) return st;
  static bool attr_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MLA_ERR_CUDA;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(mla_expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kExSmem) != cudaSuccess ||
        cudaFuncSetAttribute(mla_attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAtSmem) != cudaSuccess)
      return MLA_ERR_CUDA;
    attr_set[dev] = true;
  }
  return MLA_OK;
}

static int32_t cache_map(CUtensorMap* m, const void* kv_pages, int32_t num_pages) {
  const uint64_t d[2] = {576, (uint64_t)num_pages * 64};
  const uint64_t s[1] = {576 * 2};
  const uint32_t bx[2] = {64, 64};
  return encode_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv_pages, d, s, bx, CU_TENSOR_MAP_SWIZZLE_128B);
}

// The workspace's [K^N | V] rows (256 values) as {64, C rows, 4 blocks of 64, B * H}.
static int32_t workspace_map(CUtensorMap* m, const void* buf, const mla_extend_params* p) {
  const uint64_t d[4] = {64, (uint64_t)p->chunk_tokens, 4, (uint64_t)p->batch * p->num_heads};
  const uint64_t s[3] = {2 * kXDim * 2, 128, (uint64_t)p->chunk_tokens * 2 * kXDim * 2};
  const uint32_t bx[4] = {64, 64, 4, 1};
  return encode_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, buf, d, s, bx, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Maps and grid of the expansion; the caller sets chunk_start and launches.
static int32_t expand_setup(const mla_extend_params* p, const void* kv_pages, const int32_t* block_table,
                            const int32_t* cache_seqlens, const void* w_uk, const void* w_uv, void* k_nope, void* v,
                            int sm_count, ExpandArgs* a, dim3* grid) {
  std::memset(a, 0, sizeof *a);
  int32_t st;
  if ((st = cache_map(&a->map_kvc, kv_pages, p->num_pages))) return st;
  {  // W_UK [H][128 n][512 k] as {64 k, 128 n, 8 k-chunks, H}: two chunks per box
    const uint64_t d[4] = {64, (uint64_t)kXDim, 8, (uint64_t)p->num_heads};
    const uint64_t s[3] = {512 * 2, 128, (uint64_t)kXDim * 512 * 2};
    const uint32_t bx[4] = {64, 128, 2, 1};
    if ((st = encode_map(&a->map_wuk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, w_uk, d, s, bx, CU_TENSOR_MAP_SWIZZLE_128B)))
      return st;
  }
  {  // W_UV [H][512 k][128 n] as {64 n, 512 k, 2 n-blocks, H}: 128 k rows of both blocks per box
    const uint64_t d[4] = {64, 512, 2, (uint64_t)p->num_heads};
    const uint64_t s[3] = {(uint64_t)kXDim * 2, 128, (uint64_t)512 * kXDim * 2};
    const uint32_t bx[4] = {64, 128, 2, 1};
    if ((st = encode_map(&a->map_wuv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, w_uv, d, s, bx, CU_TENSOR_MAP_SWIZZLE_128B)))
      return st;
  }
  a->block_table = block_table;
  a->seqlens = cache_seqlens;
  a->kn = static_cast<__nv_bfloat16*>(k_nope);
  a->v = static_cast<__nv_bfloat16*>(v);
  a->B = p->batch;
  a->H = p->num_heads;
  a->C = p->chunk_tokens;
  a->s_q = p->s_q;
  a->max_pages_per_seq = p->max_pages_per_seq;
  a->ld = kXDim;  // separate K^N and V buffers (the extend's workspace interleaves them)
  a->timeout_ns = (uint64_t)(p->timeout_us ? p->timeout_us : 2000000) * 1000ull;
  // heads per CTA: as many as keep at least two CTAs per SM busy (the latent tile is loaded once
  // per CTA and reused for all of its heads)
  const int64_t tiles = (int64_t)(p->chunk_tokens / 128) * p->batch;
  int hpc = 1;
  for (int c : {8, 4, 2})
    if (p->num_heads % c == 0 && tiles * (p->num_heads / c) >= 2 * sm_count) {
      hpc = c;
      break;
    }
  a->heads_per_cta = hpc;
  *grid = dim3(p->chunk_tokens / 128, p->batch, p->num_heads / hpc);
  return MLA_OK;
}

static int32_t launch_expand(const ExpandArgs& a, dim3 grid, void* stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kXThreads, 1, 1);
  cfg.dynamicSmemBytes = kExSmem;
  pdl_config(&cfg, attr, stream);
  return cudaLaunchKernelEx(&cfg, mla_expand_kernel, a) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int32_t mla_extend_workspace_size(const mla_extend_params* p, size_t* workspace_bytes) {
  int32_t st = check_extend(p);
  if (st != MLA_OK) return st;
  if (!workspace_bytes) return MLA_ERR_INVALID_ARG;
  *workspace_bytes = extend_layout(p).total;
  return MLA_OK;
}

int32_t mla_expand_kv(const mla_extend_params* p, const void* kv_pages, const int32_t* block_table,
                      const int32_t* cache_seqlens, const void* w_uk, const void* w_uv, int32_t chunk_start,
                      void* k_nope, void* v, void* stream) {
  int32_t st = check_extend(p);
  if (st != MLA_OK) return st;
  if (!kv_pages || !block_table || !cache_seqlens || !w_uk || !w_uv || !k_nope || !v) return MLA_ERR_INVALID_ARG;
  if (!aligned16(kv_pages) || !aligned16(w_uk) || !aligned16(w_uv) || !aligned16(k_nope) || !aligned16(v))
    return MLA_ERR_INVALID_ARG;
  if (chunk_start < 0 || chunk_start % p->chunk_tokens != 0) return MLA_ERR_INVALID_ARG;
  DeviceInfo* dinfo = nullptr;
  if ((st = extend_attrs(&dinfo))) return st;
  ExpandArgs a;
  dim3 grid;
  if ((st = expand_setup(p, kv_pages, block_table, cache_seqlens, w_uk, w_uv, k_nope, v, dinfo->sm_count, &a, &grid)))
    return st;
  a.chunk_start = chunk_start;
  return launch_expand(a, grid, stream);
}

int32_t mla_extend(const mla_extend_params* p, const void* q_nope, const void* q_rope, const void* kv_pages,
                   const int32_t* block_table, const int32_t* cache_seqlens, const void* w_uk, const void* w_uv,
                   float scale, void* out, float* lse, void* workspace, void* stream) {
  int32_t st = check_extend(p);
  if (st != MLA_OK) return st;
  if (!q_nope || !q_rope || !kv_pages || !block_table || !cache_seqlens || !w_uk || !w_uv || !out || !lse ||
      !workspace)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(kv_pages) || !aligned16(w_uk) || !aligned16(w_uv) ||
      !aligned16(out) || !aligned16(lse) || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MLA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < INFINITY)) return MLA_ERR_INVALID_ARG;
  DeviceInfo* dinfo = nullptr;
  if ((st = extend_attrs(&dinfo))) return st;
  const ExtendLayout lay = extend_layout(p);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* kn = ws;                                      // rows [K^N | V] of 256 values
  void* vv = ws + kXDim * 2;
  float* acc_o = reinterpret_cast<float*>(ws + 2 * lay.kv);
  float* acc_lse = reinterpret_cast<float*>(ws + 2 * lay.kv + lay.acc_o);
  ExpandArgs ea;
  dim3 eg;
  if ((st = expand_setup(p, kv_pages, block_table, cache_seqlens, w_uk, w_uv, kn, vv, dinfo->sm_count, &ea, &eg)))
    return st;
  AttendArgs aa;
  std::memset(&aa, 0, sizeof aa);
  aa.map_kvc = ea.map_kvc;
  ea.ld = 2 * kXDim;
  if ((st = workspace_map(&aa.map_kv, kn, p))) return st;
  aa.q_nope = static_cast<const __nv_bfloat16*>(q_nope);
  aa.q_rope = static_cast<const __nv_bfloat16*>(q_rope);
  aa.block_table = block_table;
  aa.seqlens = cache_seqlens;
  aa.acc_o = acc_o;
  aa.acc_lse = acc_lse;
  aa.out = static_cast<__nv_bfloat16*>(out);
  aa.lse = lse;
  aa.scale_log2 = scale * 1.4426950408889634f;
  aa.B = p->batch;
  aa.s_q = p->s_q;
  aa.H = p->num_heads;
  aa.C = p->chunk_tokens;
  aa.max_pages_per_seq = p->max_pages_per_seq;
  aa.timeout_ns = ea.timeout_ns;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((p->s_q + 127) / 128, p->num_heads, p->batch);
  cfg.blockDim = dim3(kXThreads, 1, 1);
  cfg.dynamicSmemBytes = kAtSmem;
  pdl_config(&cfg, attr, stream);
  const int n_chunks = (p->max_seqlen + p->chunk_tokens - 1) / p->chunk_tokens;
  for (int k = 0; k < n_chunks; ++k) {
    ea.chunk_start = aa.chunk_start = k * p->chunk_tokens;
    if ((st = launch_expand(ea, eg, stream))) return st;
    if (cudaLaunchKernelEx(&cfg, mla_attend_kernel, aa) != cudaSuccess) return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

int32_t mla_wait_selftest(int32_t timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 10000000) return MLA_ERR_INVALID_ARG;
  mla_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((uint64_t)timeout_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // extern "C"

// =================================================================== allocation-free decode
// For callers that cannot call cudaMalloc on their decode path: serving engines
// and plugin hosts that reserve all device memory for their own pool allocator
// at start-up (a cudaMalloc would take memory outside that pool, and
// cudaMalloc/cudaFree can synchronise the device in the middle of a step).
// They pass inputs and outputs as usual; the scheduler metadata and the split
// partials live in this fixed array, which every GPU that loads the library
// holds until the process exits.
static __device__ __align__(256) unsigned char g_mla_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

namespace {

void* g_noalloc_ptr[64];  // device address of g_mla_noalloc_scratch per device (guarded by g_mu)

// Set-up, once per device, with that device current: look the array's device
// address up (no allocation).  Runs inside the first mla_decode_noalloc call on
// the device.
int32_t noalloc_scratch(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_noalloc_ptr[dev]) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_mla_noalloc_scratch) != cudaSuccess || a == nullptr) return MLA_ERR_CUDA;
    g_noalloc_ptr[dev] = a;
  }
  *ptr = g_noalloc_ptr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" int32_t mla_decode_noalloc(const mla_decode_params* p, const void* q_nope_absorbed, const void* q_rope,
                                      const void* kv_pages, const int32_t* block_table,
                                      const int32_t* cache_seqlens, float scale, void* out, float* lse,
                                      void* stream) {
  int32_t st = check_params(p);
  if (st != MLA_OK) return st;
  size_t sched_bytes = 0, workspace_bytes = 0;
  if ((st = mla_get_workspace_size(p, &sched_bytes, &workspace_bytes)) != MLA_OK) return st;
  const size_t sched_region = align256(sched_bytes);
  if (sched_region + workspace_bytes > (size_t)MLA_NOALLOC_SCRATCH_BYTES) return MLA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != MLA_OK) return st;
  // The scheduler kernel rewrites all of the metadata, and every split partial is
  // written by the decode kernel before the combine reads it, so nothing in the
  // array has to start at zero.
  void* sched = scratch;
  void* workspace = static_cast<char*>(scratch) + sched_region;
  if ((st = mla_get_scheduler_metadata(p, cache_seqlens, sched, stream)) != MLA_OK) return st;
  return mla_decode(p, q_nope_absorbed, q_rope, kv_pages, block_table, cache_seqlens, scale, out, lse, sched,
                    workspace, stream);
}
