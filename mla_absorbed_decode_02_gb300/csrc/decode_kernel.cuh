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
// (head, tile), 15-bit magnitudes with sign.  Each CTA adds the peer's
// rounded half to its own exact half, runs the online softmax for its output
// half, writes P (bf16) to shared memory, and accumulates O_half += P V_half
// (tcgen05.mma, N = 256, V read MN-major from the same shared-memory page the
// score used).
//
// "MLA inference: two computation paths and FlashMLA", section "Decode
// attention becomes a compute problem": the 128 heads are the M dimension of
// the matrix multiply, a block of KV is staged in shared memory, long
// sequences are split across SMs and merged through their LSE.
//
// Softmax warpgroups.  Two warpgroups take the tiles in turn (warpgroup w owns
// the tiles of parity w, thread = head row = TMEM lane, all 64 columns of the
// row), so the two run their exchange waits and exponentials overlapped, each
// with its own score buffer, exchange slot and P buffer.  The only per-tile
// link between them is the running row maximum (the max of tile t is decided
// from the one of tile t-1, through shared memory); each keeps its own part of
// the row sum and the epilogue adds the two.  The maximum is raised lazily
// (only when a tile's max exceeds it by more than 8 in log2 units), and O is
// rescaled only then.
//
// Pipelining.  Five 36 KB shared-memory stages (a page stays resident from its
// load through QK, softmax and PV, because the latent is key and value at
// once).  QK and PV are issued by two different warps, so the scores of the
// next tiles never wait for the P of the current one.
//
// Warp roles (384 threads): warp 0 = TMA producer, warp 1 = QK issuer, warp 2
// = tensor-memory allocator, warp 3 = PV issuer, warps 4..7 / 8..11 = softmax
// warpgroups 0 / 1.
//
// FP8 QK (opt-in, FP8 cache only; "MLA inference: two computation paths and
// FlashMLA", exercise 2 "An FP8 KV cache": FP8 tensor cores for QK).  The query
// arrives quantised like the cache (E4M3 codes, one float32 scale per 128-dim
// tile).  QK runs on the E4M3 codes straight from the stage (tcgen05.mma
// kind::f8f6f4): one fp32 accumulator per 128-dim tile of this CTA's half and
// one for the RoPE part (bf16), combined by the softmax warpgroups with the
// query and key tile scales.  PV still needs the bf16 latent, so the softmax
// warpgroup of tile t expands page t once it has published P(t) (QK(t) has read
// the codes by then, and it has read the key scales), and PV(t) waits for that.
// Tensor memory then holds one score buffer (three accumulators), not two.
#pragma once
#include <type_traits>

#include "common.cuh"

namespace mla {

constexpr int kThreads = 384;
constexpr int kRows = 128;      // MMA M: head rows (H <= 128, padded with zero queries)
constexpr int kTileTok = 64;    // tokens per work tile (one page)
#ifndef MLA_STAGES
#define MLA_STAGES 5
#endif
constexpr int kStages = MLA_STAGES;

// shared memory layout (offsets from a 1024-byte aligned base)
constexpr uint32_t kLatBlock = 8192;                  // [64 rows x 128 B]: 64 latent dims of a page
constexpr uint32_t kStageRope = 4 * kLatBlock;        // RoPE half [64 rows x 64 B]
constexpr uint32_t kStageBytes = kStageRope + 4096;   // 36 KB
// FP8 cache: this CTA's 256 E4M3 codes of 64 rows land row-major in the upper
// half of the latent area, the 4 tile scales of the 64 rows [64 x 16 B] at its
// start; both are read before the expansion to the bf16 layout overwrites them.
constexpr uint32_t kStageCodes = 2 * kLatBlock;
constexpr uint32_t kStageScales = 0;
constexpr uint32_t kFp8StageTx = 64 * 256 + 4096 + 1024;  // codes + RoPE half + scales
constexpr uint32_t kBf16StageTx = 4 * kLatBlock + 4096;   // latent half + RoPE half
// P / exchange buffer of a tile parity: the peer's partial scores of tile t arrive here
// ([8 column chunks][128 rows][16 B]), are decoded, and P(t) (bf16, same [8][128][16 B]
// layout: K-major without swizzle for PV) is written over them, each thread on its own
// row's chunks; the buffer is handed back to the peer once PV(t) is done.
constexpr uint32_t kPBytes = kRows * 128;
constexpr uint32_t SM_P = kStages * kStageBytes;      // P / exchange [tile parity]
constexpr uint32_t SM_QR = SM_P + 2 * kPBytes;        // RoPE-query half [128 x 64 B], 64-byte swizzle
constexpr uint32_t SM_XE = SM_QR + 8192;              // peer block-float exponents [tile parity][128 rows] u32
constexpr uint32_t SM_ML = SM_XE + 2 * kRows * 4;     // published running max / row sum: [parity][2][128] f32
constexpr uint32_t SM_BAR = SM_ML + 2 * 2 * kRows * 4;
// Tile schedule the TMA producer publishes for the softmax warpgroups: one 32-byte entry per tile
// in a ring of 8 ({qb, valid, split, flags (1 first, 2 last), piece, qb of the next piece or -1,
// qb and split of the previous tile}); entry t is written after stage t-5 is free again, by
// when the reader of entry t-8 has long read it.
constexpr int kTiRing = 8;
constexpr uint32_t SM_TI = SM_BAR + 512;
constexpr uint32_t kSmemBytes = SM_TI + kTiRing * 32 + 1024;  // + alignment slack
constexpr uint32_t kXBytes = kRows * (128 + 4);       // bytes one CTA sends the other per tile

// tensor memory columns
constexpr uint32_t TM_O = 0, TM_S = 256, TM_Q = 384;  // S buffers at 256 and 320
// FP8 QK: one score buffer of three accumulators (latent tiles 2h and 2h + 1 of this half, RoPE)
// and the query codes of this half (256 E4M3 codes: 64 columns)
constexpr uint32_t TM_S8 = 256, TM_Q8 = 448;

// barrier slots (8 bytes each) inside SM_BAR; "[parity]" = + tile parity
enum : uint32_t {
  B_QR_FULL = 0,
  B_QR_EMPTY,
  B_QT_FULL,
  B_DRAIN,                          // + issuer (0 = QK, 1 = PV)
  B_DRAIN_PV,
  B_KV_FULL,                        // + stage
  B_KV_EMPTY = B_KV_FULL + kStages,
  B_K_READY = B_KV_EMPTY + kStages, // + stage: FP8 cache expanded to bf16
  B_S_FULL = B_K_READY + kStages,   // [parity] QK(t) done
  B_S_EMPTY = B_S_FULL + 2,         // [parity] scores of tile t read out
  B_P_FULL = B_S_EMPTY + 2,         // [parity] P(t) written
  B_P_FREE = B_P_FULL + 2,          // [parity] PV(t) done
  B_X_FULL = B_P_FREE + 2,          // [parity] the peer's partial scores of tile t arrived
  B_X_FREE = B_X_FULL + 2,          // [parity] the peer consumed what this CTA sent for tile t
  B_ML = B_X_FREE + 2,              // [parity] running max / row sum of tile t published
  B_TI_FULL = B_ML + 2,             // [t mod 8] tile-schedule entry of tile t published
  B_KV_SHARED = B_TI_FULL + kTiRing, // + stage: (token groups, loading CTA) every pair's PV(t) done
  kNumBars = B_KV_SHARED + kStages
};
constexpr uint32_t OFF_TMEM_SLOT = kNumBars * 8;
constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4;
static_assert(OFF_ABORT + 4 <= 512, "barrier area");
static_assert(kSmemBytes <= 232448, "shared memory");

struct Piece {
  int qb, t0, t1, split;
};

// Walks the pieces (query block, tile range) of one unit record.  The record's ranges are over
// work blocks of `group` tokens; this CTA pair's token is `g` of each block, so its query block
// is blk * group + g, over the block's tiles (a token before the block's last may see none of
// the last one or two).
struct PieceWalker {
  const int32_t* seqlens;
  int s_q, causal, group, g, first_qb, qb, qb_end, tile_begin, tile_end, first_split;
  __device__ bool next(Piece& p) {
    while (qb <= qb_end) {
      const int cur = qb++;
      const int nt = block_tiles(seqlens, s_q, causal, group, cur);
      const int a = (cur == first_qb) ? tile_begin : 0;
      const int b = (cur == qb_end) ? tile_end : nt;
      if (nt > 0 && a < b) {
        p.qb = cur * group + g;
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

// Exponent e (clamped) of a row's block: every |x| of the row is below 2^e (1 - 2^-16)
// (e is the exponent bucket of amax * (1 + 2^-15), one rounding included), so
// rint(x * 2^(14-e)) lies in [-(2^14 - 1), 2^14 - 1].
__device__ __forceinline__ int bfp_exponent(float amax) {
  const float a = fmaf(amax, 3.0517578125e-05f, amax);  // amax * (1 + 2^-15)
  int e = (int)((__float_as_uint(a) >> 23) & 0xFF) - 126;
  e = e < -60 ? -60 : e;
  e = e > 110 ? 110 : e;
  return e;
}

// Packed float pairs (the f32x2 arithmetic of sm_100-class GPUs: one instruction
// for two lanes of a 64-bit register pair).
__device__ __forceinline__ uint64_t pack_b32x2(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  return pack_b32x2(__float_as_uint(lo), __float_as_uint(hi));
}
__device__ __forceinline__ uint64_t splat_f32x2(float v) { return pack_f32x2(v, v); }
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t fadd_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// 2^x on the special-function unit (inputs below -126 give 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Columns >= valid of a row of score pairs -> v.
__device__ __forceinline__ void mask_pairs(uint64_t (&sc)[32], int valid, float v) {
#pragma unroll
  for (int u = 0; u < 32; ++u) {
    float x0, x1;
    unpack_f32x2(sc[u], x0, x1);
    sc[u] = pack_f32x2(2 * u < valid ? x0 : v, 2 * u + 1 < valid ? x1 : v);
  }
}

// Block floating point without conversion instructions, one exponent e per row and
// tile.  Encode: n = rint(x * 2^(14-e)) lies in [-(2^14 - 1), 2^14 - 1]; adding
// 1.5 * 2^23 + 3 * 2^14 in one FMA leaves u = n + 3 * 2^14, which lies in [2^15, 2^16),
// in the low 16 bits of the float, and two such halves are packed into one word.
// Decode: u placed at bits 8..23 under the exponent of 0.5 gives the float
// 1 + (u - 2^15) 2^-15 = 1.5 + n 2^-15 exactly (u >= 2^15 sets the exponent's low bit,
// so every u lands in [1, 2)); the receiver folds it into its own partial with one
// FMA by 2^(e_peer + 1), which leaves the constant bias beta = 3 * 2^e_peer on every
// score of the row -- the softmax only ever sees scores relative to the row max, so
// beta is removed there.  The peer's half is off by at most half a quantum,
// 2^(e_peer - 15); the biased sum, below 2^(e_peer + 3), rounds within 2^(e_peer - 21).
constexpr float kBfpMagic = 12632064.0f;  // 1.5 * 2^23 + 3 * 2^14
__device__ __forceinline__ uint32_t bfp_pack_pair(uint64_t xy, uint64_t k) {
  float a, b;
  unpack_f32x2(ffma_f32x2(xy, k, splat_f32x2(kBfpMagic)), a, b);
  return __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x5410);
}
// The two halves u of w as the floats 1 + (u - 2^15) 2^-15 (u at bits 8..23 of 0x3F000000).
__device__ __forceinline__ uint64_t bfp_unpack_pair(uint32_t w) {
  return pack_b32x2(__byte_perm(w, 0x3F000000u, 0x7104), __byte_perm(w, 0x3F000000u, 0x7324));
}

__device__ __forceinline__ void st_async_b32(uint32_t cluster_dst, uint32_t v, uint32_t cluster_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(cluster_dst), "r"(v),
               "r"(cluster_bar)
               : "memory");
}

// prmt with selector s on (x, 0): a selector nibble with bit 3 set replicates the sign bit of the
// byte it selects (the PTX form; the __byte_perm intrinsic uses only the low 3 bits)
__device__ __forceinline__ uint32_t prmt_sext(uint32_t x, uint32_t s) {
  uint32_t d;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(d) : "r"(x), "r"(s));
  return d;
}

// FP8 cache: this warpgroup thread's share of a stage (i in [0, 128): row i % 64, the 128 codes of
// tile half i / 64) -> bf16 x tile scale, written into the 128-byte-swizzled latent layout the MMAs
// read.  A lane takes its eight 16-code chunks starting at chunk (lane mod 8): the eight lanes of a
// quarter-warp then read eight different bank groups, and (rows consecutive across lanes, the
// layout's row-XOR swizzle) write eight different ones -- no bank conflicts either way.  The codes
// sit in the upper half of the latent area, so every thread of the warpgroup reads its codes before
// any thread writes (named barrier bar_id over the 128 threads).
// kQk8: the codes of each 128-code tile sit in the 128-byte-swizzled K-major layout the QK MMAs
// read (logical chunk c of row r at physical chunk c ^ (r mod 8)); a lane walks logical chunks
// ((j + lane) mod 8) ^ (lane mod 8), which keeps reads and writes conflict-free.  Rows >= valid are
// written as zeros (they must not reach PV).
template <bool kQk8>
__device__ __forceinline__ void expand_fp8_stage(uint32_t sbase, int i, uint32_t half, uint32_t bar_id,
                                                 int valid = 64) {
  const int row = i & 63, part = i >> 6;
  const uint32_t rot = (uint32_t)i & 7;
  auto lchunk = [&](int j) -> uint32_t { return kQk8 ? (((uint32_t)j + rot) & 7) ^ rot : ((uint32_t)j + rot) & 7; };
  uint32_t c[32];  // c[4j .. 4j+3]: codes of logical chunk lchunk(j)
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t addr = kQk8 ? sbase + kStageCodes + part * 8192 + row * 128 + ((lchunk(j) ^ (uint32_t)(row & 7)) << 4)
                               : sbase + kStageCodes + row * 256 + part * 128 + 16 * lchunk(j);
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(c[4 * j]), "=r"(c[4 * j + 1]), "=r"(c[4 * j + 2]), "=r"(c[4 * j + 3])
                 : "r"(addr));
  }
  float scale;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(scale) : "r"(sbase + kStageScales + row * 16 + (2 * half + part) * 4));
  asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory");
  // E4M3 -> bf16 without the conversion units: a code's 7 magnitude bits placed as a bf16's
  // exponent and mantissa give the code's value times 2^-120 exactly (subnormal codes land on
  // bf16 subnormals), the sign bit goes to bit 15; then x 2^120 (exact) and x scale (rounded
  // to bf16) in two packed bf16 multiplies.
  const uint32_t k120 = 0x7B807B80u;  // bf16x2 {2^120, 2^120}
  uint32_t sc2;
  {
    const __nv_bfloat162 s2 = __floats2bfloat162_rn(scale, scale);
    sc2 = *reinterpret_cast<const uint32_t*>(&s2);
  }
  const bool zero_row = kQk8 && row >= valid;
#pragma unroll
  for (int ch = 0; ch < 16; ++ch) {  // 8 codes -> 8 bf16 (16 bytes): output chunk 2 lchunk(j) + k
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      // two codes sign-extended to 16 bits (the byte permute's sign-replicate selectors), shifted so
      // that the magnitude bits sit at bf16 bits 10..4, with the sign kept at bit 15
      const uint32_t z = prmt_sext(c[2 * ch + (q >> 1)], (q & 1) ? 0xB3A2u : 0x9180u);
      const uint32_t y = (z << 4) & 0x87F087F0u;
      uint32_t v;
      asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(v) : "r"(y), "r"(k120));
      asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(o[q]) : "r"(v), "r"(sc2));
      if (kQk8 && zero_row) o[q] = 0u;
    }
    const uint32_t out_ch = 2 * lchunk(ch >> 1) + (ch & 1);
    const uint32_t blk = 2 * part + (out_ch >> 3), chunk = out_ch & 7;
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(sbase + blk * kLatBlock + row * 128 +
                                                              ((chunk ^ (uint32_t)(row & 7)) << 4)),
                 "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3]));
  }
}

__device__ __forceinline__ void mma_e4m3_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
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

// The kernel body, instantiated once per cache format (no code of the other format in the
// instruction stream of either).  kQk8 (FP8 cache only): QK on the E4M3 codes.
template <bool kFp8, bool kGroups, bool kQk8 = false>
__device__ __forceinline__ void decode_body(const DecodeArgs& args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t base = smem_addr(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // a unit is a cluster of 2G CTAs: pair g (ranks 2g, 2g + 1) decodes token g of each work block,
  // the two CTAs of a pair own the two halves of the latent dims
  const uint32_t rank = cluster_ctarank(), half = rank & 1, peer = rank ^ 1;
  const int grp = kGroups ? args.group : 1, g = kGroups ? (int)(rank >> 1) : 0;
  const int unit = blockIdx.x / (2 * grp);

  auto bar = [&](uint32_t i) { return base + SM_BAR + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM_BAR + OFF_ABORT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM_BAR + OFF_TMEM_SLOT);

  if (tid == 0) {
    mbar_init(bar(B_QR_FULL), 1);
    mbar_init(bar(B_QR_EMPTY), 1);
    mbar_init(bar(B_QT_FULL), 4);  // the four warps of the warpgroup that loads the query half
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_DRAIN_PV), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_KV_FULL + s), 1);
      mbar_init(bar(B_KV_EMPTY + s), 1);
      mbar_init(bar(B_K_READY + s), 4);  // the four warps of the warpgroup that expands the stage
    }
    for (int p = 0; p < 2; ++p) {
      mbar_init(bar(B_S_FULL + p), 1);   // MMA commit
      mbar_init(bar(B_S_EMPTY + p), 4);  // one arrival per warp of warpgroup p
      mbar_init(bar(B_P_FULL + p), 4);
      mbar_init(bar(B_P_FREE + p), 1);   // MMA commit
      mbar_init(bar(B_X_FULL + p), 1);   // receiver's expect_tx arrival + the peer's st.async bytes
      mbar_init(bar(B_X_FREE + p), 4);   // one remote arrival per warp of the peer's warpgroup p
      mbar_init(bar(B_ML + p), 4);
    }
    for (int i = 0; i < kTiRing; ++i) mbar_init(bar(B_TI_FULL + i), 1);
    for (int s = 0; s < kStages; ++s) mbar_init(bar(B_KV_SHARED + s), grp);  // one PV commit per pair
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncwarp();  // (warp 0 ran the set-up on one lane: the CTA and cluster barriers below take whole warps)
  __syncthreads();
  cluster_sync();  // peer barriers initialised before any remote arrive / st.async
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The tensor maps are launch parameters, nothing the kernel before this one writes: their
  // fetch overlaps that kernel's end too.
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&args.map_qr);
    prefetch_tensormap(&args.map_kvc);
    prefetch_tensormap(&args.map_kvr);
    if (kFp8) prefetch_tensormap(&args.map_kvs);
  }
  // Everything above touches no other global memory: it runs while the kernel before this one
  // in the stream is still finishing (programmatic dependent launch).  Its writes (the
  // metadata, the inputs) are visible from here on.
  pdl_wait_prerequisites();
  // ---- unit record (uniform across the cluster); bail out early on bad metadata
  const int32_t* sched = args.sched;
  const bool bad_meta = sched[0] != kSchedMagic || sched[1] != args.num_units || sched[2] != args.num_qb ||
                        sched[5] != grp;
  const int32_t* rec = sched + kSchedHeader + kUnitInts * unit;
  if (bad_meta || rec[0] < 0) {  // bad metadata, or no work for this unit (both CTAs take this path)
    if (bad_meta && tid == 0) atomicCAS(&g_mla_error, 0, 5);
    if (warp == 2) tmem_dealloc(tmem, 512);
    return;
  }
  pdl_launch_dependents();  // the combine kernel may start launching; it waits for this grid to finish
  const int32_t* num_splits = sched + kSchedHeader + kUnitInts * args.num_units;
  const int32_t* split_offset = num_splits + args.num_qb;

  WaitCtx wc;
  wc.abort_local = abort_flag;
  wc.abort_peer = map_to_rank(smem_addr((const void*)abort_flag), peer);
  wc.timeout_ns = args.timeout_ns;

  PieceWalker walker0;
  walker0.seqlens = args.seqlens;
  walker0.s_q = args.s_q;
  walker0.causal = args.causal;
  walker0.group = grp;
  walker0.g = g;
  walker0.qb = rec[0];
  walker0.first_qb = rec[0];
  walker0.tile_begin = rec[1];
  walker0.qb_end = rec[2];
  walker0.tile_end = rec[3];
  walker0.first_split = rec[4];
  const int first_qb = rec[0] * grp + g;  // this pair's query block of the unit's first work block

  auto count_tiles = [&]() {  // tiles of this unit
    uint32_t n = 0;
    PieceWalker pw = walker0;
    Piece pc;
    while (pw.next(pc)) n += pc.t1 - pc.t0;
    return n;
  };
  if (warp == 0) {
    // ================================================================ TMA producer
    if (lane == 0) {
      const uint64_t pol_kv = l2_policy_evict_first();
      const uint64_t pol_q = l2_policy_evict_last();
      // one page into stage st: the half of its 64 rows this CTA owns
      auto load_page = [&](uint32_t st, int page) {
        const uint32_t sbase = base + st * kStageBytes;
        if (kFp8) {  // 656-byte rows: codes of this half, its RoPE half, the 4 tile scales
          mbar_arrive_expect_tx(bar(B_KV_FULL + st), kFp8StageTx);
          if (kQk8) {  // the half's two 128-code tiles, each in the swizzled K-major layout QK reads
            tma_load_2d(sbase + kStageCodes, &args.map_kvc, bar(B_KV_FULL + st), 256 * half, page * 64, pol_kv);
            tma_load_2d(sbase + kStageCodes + 8192, &args.map_kvc, bar(B_KV_FULL + st), 256 * half + 128, page * 64,
                        pol_kv);
          } else {
            tma_load_2d(sbase + kStageCodes, &args.map_kvc, bar(B_KV_FULL + st), 256 * half, page * 64, pol_kv);
          }
          tma_load_2d(sbase + kStageRope, &args.map_kvr, bar(B_KV_FULL + st), 528 + 64 * half, page * 64, pol_kv);
          tma_load_2d(sbase + kStageScales, &args.map_kvs, bar(B_KV_FULL + st), 512, page * 64, pol_kv);
        } else {
          mbar_arrive_expect_tx(bar(B_KV_FULL + st), kBf16StageTx);
          for (int blk = 0; blk < 4; ++blk)
            tma_load_2d(sbase + blk * kLatBlock, &args.map_kvc, bar(B_KV_FULL + st), 256 * half + 64 * blk, page * 64,
                        pol_kv);
          tma_load_2d(sbase + kStageRope, &args.map_kvr, bar(B_KV_FULL + st), 512 + 32 * half, page * 64, pol_kv);
        }
      };
      // Token groups: pair 0 loads each page half once into the same half of every pair
      // (multicast); the other pairs only expect the bytes on their own barrier.
      const uint16_t mc_mask = (uint16_t)(0x5555u & ((1u << (2 * grp)) - 1u)) << half;
      auto load_page_group = [&](uint32_t st, int page) {
        const uint32_t sbase = base + st * kStageBytes;
        if (kFp8) {
          mbar_arrive_expect_tx(bar(B_KV_FULL + st), kFp8StageTx);
          if (g != 0) return;
          tma_load_2d_mc(sbase + kStageCodes, &args.map_kvc, bar(B_KV_FULL + st), 256 * half, page * 64, mc_mask, pol_kv);
          tma_load_2d_mc(sbase + kStageRope, &args.map_kvr, bar(B_KV_FULL + st), 528 + 64 * half, page * 64, mc_mask,
                         pol_kv);
          tma_load_2d_mc(sbase + kStageScales, &args.map_kvs, bar(B_KV_FULL + st), 512, page * 64, mc_mask, pol_kv);
        } else {
          mbar_arrive_expect_tx(bar(B_KV_FULL + st), kBf16StageTx);
          if (g != 0) return;
          for (int blk = 0; blk < 4; ++blk)
            tma_load_2d_mc(sbase + blk * kLatBlock, &args.map_kvc, bar(B_KV_FULL + st), 256 * half + 64 * blk,
                           page * 64, mc_mask, pol_kv);
          tma_load_2d_mc(sbase + kStageRope, &args.map_kvr, bar(B_KV_FULL + st), 512 + 32 * half, page * 64, mc_mask,
                         pol_kv);
        }
      };
      // logical page lp of sequence b; a length beyond the block table is reported, and no entry
      // past the row is read
      auto page_of = [&](int b, int lp) {
        if (lp >= args.max_pages) {
          atomicCAS(&g_mla_error, 0, 1);
          lp = args.max_pages - 1;
        }
        return args.block_table[(int64_t)b * args.max_pages + lp];
      };
      // The unit's first tile is (its first query block, its first tile): the planner makes both
      // non-empty.  That page and the block's RoPE-query half go out straight from the unit
      // record, before the walk over the lengths.
      mbar_arrive_expect_tx(bar(B_QR_FULL), 8192);
      tma_load_3d(base + SM_QR, &args.map_qr, bar(B_QR_FULL), 32 * half, 0, first_qb, pol_q);
      if (grp == 1)
        load_page(0, page_of(first_qb / args.s_q, walker0.tile_begin));
      else
        load_page_group(0, page_of(first_qb / args.s_q, walker0.tile_begin));
      TileCursor cur;
      cur.init(walker0);
      TileInfo ti;
      // bf16 cache: the block-table entry of the next tile is read one iteration ahead, so its
      // latency overlaps the wait for a free stage (ragged decode 117.4 against 119.5 us; the FP8
      // kernel measured 1% slower with it and reads the entry when it needs it)
      TileCursor la = cur;
      TileInfo tl;
      int pg_next = -1;
      if (!kFp8 && la.next(tl) && la.next(tl)) pg_next = page_of(tl.qb / args.s_q, tl.tile);  // tile 1
      PieceWalker ahead = walker0;  // one piece ahead of the tile walk
      Piece np;
      ahead.next(np);  // piece 0
      int next_qb = -1, prev_qb = -1, prev_split = 0;
      uint32_t t = 0, piece_no = 0;
      while (cur.next(ti)) {
        if (ti.first) {
          if (piece_no > 0) {
            if (!wait_one(bar(B_QR_EMPTY), (piece_no - 1) & 1, wc, kSiteQEmpty)) break;
            mbar_arrive_expect_tx(bar(B_QR_FULL), 8192);
            tma_load_3d(base + SM_QR, &args.map_qr, bar(B_QR_FULL), 32 * half, 0, ti.qb, pol_q);
          }
          ++piece_no;
          next_qb = ahead.next(np) ? np.qb : -1;
        }
        const uint32_t st = t % kStages, ph = (t / kStages) & 1;
        // the stage is free: here (this CTA's PV of its last tile), or, for the loading pair of a
        // token group, in every pair
        if (t > 0 && !wait_one(bar((grp > 1 && g == 0 ? B_KV_SHARED : B_KV_EMPTY) + st), ph ^ 1, wc, kSiteKvEmpty))
          break;
        {  // the tile's schedule entry for the softmax warpgroups
          const uint32_t e = base + SM_TI + (t % kTiRing) * 32;
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(e), "r"(ti.qb), "r"(ti.valid), "r"(ti.split),
                       "r"((ti.first ? 1 : 0) | (ti.last ? 2 : 0))
                       : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(e + 16), "r"((int)piece_no - 1), "r"(next_qb),
                       "r"(prev_qb), "r"(prev_split)
                       : "memory");
          mbar_arrive(bar(B_TI_FULL + (t % kTiRing)));
          prev_qb = ti.qb;
          prev_split = ti.split;
        }
        if (t > 0) {  // (tile 0's page went out above)
          const int page = kFp8 ? page_of(ti.qb / args.s_q, ti.tile) : pg_next;
          if (grp == 1)
            load_page(st, page);
          else
            load_page_group(st, page);
          if (!kFp8 && la.next(tl)) pg_next = page_of(tl.qb / args.s_q, tl.tile);
        }
        ++t;
      }
      // Token groups: the loading pair's CTAs receive every pair's last PV commits; they stay
      // until those arrived (the barrier phases of the last min(t, stages) tiles).
      if (grp > 1 && g == 0 && !*abort_flag)
        for (uint32_t k = t > kStages ? t - kStages : 0; k < t; ++k)
          if (!wait_one(bar(B_KV_SHARED + k % kStages), (k / kStages) & 1, wc, kSiteKvEmpty)) break;
    }
  } else if (warp == 1 || warp == 3) {
    // ================================================================ MMA issuers
    // warp 1: QK(t) as soon as the page is loaded and its score buffer was read out;
    // warp 3: PV(t) as soon as P(t) is published.  The two touch disjoint tensor
    // memory (scores / O) and only read shared memory.
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_bf16_f32(128, 64, 0, 0);
      constexpr uint32_t id_pv = idesc_bf16_f32(128, 256, 0, 1);
      TileCursor cur;
      cur.init(walker0);
      TileInfo ti;
      uint32_t t = 0, piece_no = 0;
      if (warp == 1) {
        while (cur.next(ti)) {
          if (ti.first) {
            if (!wait_one(bar(B_QR_FULL), piece_no & 1, wc, kSiteQFull)) break;
            if (!wait_one(bar(B_QT_FULL), piece_no & 1, wc, kSiteQFull)) break;
            ++piece_no;
          }
          const uint32_t st = t % kStages, sb = t & 1;
          const uint32_t ready = kFp8 && !kQk8 ? B_K_READY : B_KV_FULL;  // (FP8 QK reads the codes)
          if (!wait_one(bar(ready + st), (t / kStages) & 1, wc, kSiteKvFull)) break;
          if (kQk8) {  // one score buffer: the previous tile's scores must have been read out
            if (t > 0 && !wait_one(bar(B_S_EMPTY + (sb ^ 1)), ((t - 1) >> 1) & 1, wc, kSiteSEmpty))
              break;
          } else if (!wait_one(bar(B_S_EMPTY + sb), ((t >> 1) & 1) ^ 1, wc, kSiteSEmpty)) {
            break;
          }
          tc_fence_after();
          const uint32_t sbase = base + st * kStageBytes;
          if (kQk8) {
            // each 128-code tile into its own accumulator (K = 32 codes per MMA), RoPE into a third
            constexpr uint32_t id_qk8 = idesc_e4m3_f32(128, 64, 0, 0);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_e4m3_ts(tmem + TM_S8 + 64 * (k >> 2), tmem + TM_Q8 + 8 * k,
                          smem_desc(sbase + kStageCodes + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024, kSwizzle128B),
                          id_qk8, (k & 3) ? 1u : 0u);
#pragma unroll
            for (int k = 0; k < 2; ++k)
              mma_bf16_ss(tmem + TM_S8 + 128, smem_desc(base + SM_QR + 32 * k, 16, 512, kSwizzle64B),
                          smem_desc(sbase + kStageRope + 32 * k, 16, 512, kSwizzle64B), id_qk, k > 0 ? 1u : 0u);
          } else {
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
          }
          mma_commit(bar(B_S_FULL + sb));
          if (ti.last) mma_commit(bar(B_QR_EMPTY));
          ++t;
        }
      } else {
        while (cur.next(ti)) {
          const uint32_t pb = t & 1, st = t % kStages;
          if (!wait_one(bar(B_P_FULL + pb), (t >> 1) & 1, wc, kSitePFull)) break;
          // FP8 QK: the page's bf16 latent (V) is written after its QK, by the expansion warpgroup
          if (kQk8 && !wait_one(bar(B_K_READY + st), (t / kStages) & 1, wc, kSiteKvFull)) break;
          tc_fence_after();
          const uint32_t sbase = base + st * kStageBytes;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t a = smem_desc(base + SM_P + pb * kPBytes + k * 4096, 2048, 128, kSwizzleNone);
            const uint64_t bv = smem_desc(sbase + k * 2048, kLatBlock, 1024, kSwizzle128B);
            mma_bf16_ss(tmem + TM_O, a, bv, id_pv, (!ti.first || k > 0) ? 1u : 0u);
          }
          mma_commit(bar(B_KV_EMPTY + st));
          if (grp > 1) mma_commit_mc(bar(B_KV_SHARED + st), (uint16_t)(1u << half));  // the loading CTA
          mma_commit(bar(B_P_FREE + pb));
          ++t;
        }
      }
      // no MMA of this issuer may still run when tensor memory is released
      const uint32_t drain = bar(warp == 1 ? B_DRAIN : B_DRAIN_PV);
      mma_commit(drain);
      WaitCtx wd = wc;
      wd.timeout_ns = 100000000ull;
      volatile int no_abort = 0;
      wd.abort_local = &no_abort;
      wd.abort_peer = 0;
      wait_one(drain, 0, wd, kSiteDrain);
    }
  } else if (warp >= 4) {
    // ================================================================ softmax warpgroups
    const uint32_t w = (uint32_t)(warp - 4) >> 2;  // this warpgroup owns the tiles of parity w
    const int r = ((warp & 3) << 5) | lane;        // head row == TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t peer_bar0 = map_to_rank(bar(0), peer);  // the peer's barrier i is at peer_bar0 + 8 i
    const uint32_t peer_x = map_to_rank(base + SM_P + w * kPBytes, peer);
    const uint32_t peer_xe = map_to_rank(base + SM_XE + w * kRows * 4, peer);
    const uint32_t my_x = base + SM_P + w * kPBytes, my_xe = base + SM_XE + w * kRows * 4;
    float* ml = reinterpret_cast<float*>(smem + SM_ML);  // [parity][0 = max, 1 = row sum][128]
    const float sl2 = args.scale_log2;
    const int H = args.H;
    bool ok = true;

    // absorbed-query half of query block qb -> tensor memory (A operand of the latent score)
    // (all 32 row loads in flight at once: one memory latency)
    auto load_q_tmem = [&](int qb) {
      if (kQk8) {  // this half's 256 E4M3 codes of the 656-byte query row: 64 columns
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(args.q_nope) +
                                                          ((int64_t)qb * H + r) * 656 + 256 * half);
        uint32_t q[64];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (r < H) v = src[j];
          q[4 * j] = v.x;
          q[4 * j + 1] = v.y;
          q[4 * j + 2] = v.z;
          q[4 * j + 3] = v.w;
        }
#pragma unroll
        for (int c = 0; c < 2; ++c)
          tmem_st32(tmem + lane_off + TM_Q8 + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(q + 32 * c));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_QT_FULL));
        return;
      }
      const uint32_t* src = reinterpret_cast<const uint32_t*>(args.q_nope) + ((int64_t)qb * H + r) * 256 + 128 * half;
      uint32_t q[128];
#pragma unroll
      for (int j = 0; j < 128; j += 4) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < H) v = *reinterpret_cast<const uint4*>(src + j);
        q[j] = v.x;
        q[j + 1] = v.y;
        q[j + 2] = v.z;
        q[j + 3] = v.w;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_st32(tmem + lane_off + TM_Q + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(q + 32 * c));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_QT_FULL));
    };

    // Row-per-thread data (tensor memory's layout) <-> whole-row global accesses go through this
    // warp's 4 KB of the warpgroup's P / exchange buffer: 32 rows x 128 bytes, 16-byte chunks
    // XOR-swizzled by row so that both the row-per-lane and the chunk-per-lane passes are
    // conflict-free.  Callers own the buffer at that point (no P for PV in it, no exchange data
    // due).
    const uint32_t stg = my_x + (uint32_t)(warp & 3) * 4096;
    const int row0 = (warp & 3) * 32;  // this warp's first head row
    const int sub = lane >> 3, chk = lane & 7;
    auto stg_row = [&](int row, int c) -> uint32_t { return stg + row * 128 + (((uint32_t)(c ^ (row & 7))) << 4); };

    // absorbed-query half of query block qb -> tensor memory (A operand of the latent score):
    // 128-byte row segments loaded by 8 lanes each, two 32-column blocks in flight at a time
    auto load_q_tmem_staged = [&](int qb) {
      if (kQk8) {  // (a quarter of the bytes: loaded row per thread)
        load_q_tmem(qb);
        return;
      }
      const uint32_t* src = reinterpret_cast<const uint32_t*>(args.q_nope) + (int64_t)qb * H * 256 + 128 * half + 4 * chk;
      auto fetch = [&](uint4 (&g)[8], int k) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int row = row0 + 4 * i + sub;
          g[i] = row < H ? *reinterpret_cast<const uint4*>(src + (int64_t)row * 256 + 32 * k) : make_uint4(0, 0, 0, 0);
        }
      };
      auto put = [&](const uint4 (&g)[8], int k) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(stg_row(4 * i + sub, chk)), "r"(g[i].x), "r"(g[i].y),
                       "r"(g[i].z), "r"(g[i].w)
                       : "memory");
        __syncwarp();
        uint32_t v[32];
#pragma unroll
        for (int c = 0; c < 8; ++c)
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(v[4 * c]), "=r"(v[4 * c + 1]), "=r"(v[4 * c + 2]), "=r"(v[4 * c + 3])
                       : "r"(stg_row(lane, c))
                       : "memory");
        __syncwarp();
        tmem_st32(tmem + lane_off + TM_Q + 32 * k, v);
      };
      uint4 g0[8], g1[8];
      fetch(g0, 0);
      fetch(g1, 1);
      put(g0, 0);
      fetch(g0, 2);
      put(g1, 1);
      fetch(g1, 3);
      put(g0, 2);
      put(g1, 3);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_QT_FULL));
    };

    // epilogue of a finished piece: O / l -> out (or a split partial), lse; whole 128-byte row
    // segments per 8 lanes through the staging buffer
    int epi_qb = 0, epi_split = 0, epi_piece = -1;
    bool epi_pending = false;
    const uint64_t pol_partial = l2_policy_evict_last();
    // (columns: part `part` of `nparts` equal parts of this CTA's 256)
    auto epilogue = [&](float m_fin, float l_tot, int part, int nparts) {
      const bool split = num_splits[epi_qb] > 1;
      const int slot = split ? split_offset[epi_qb] + epi_split : 0;
      const float inv_l = l_tot > 0.f ? 1.f / l_tot : 0.f;  // a token that saw no key: out = 0, lse = -inf
      if (split || args.out_f32) {
        float* dst = (split ? args.o_acc + (int64_t)slot * H * 512 : reinterpret_cast<float*>(args.out) + (int64_t)epi_qb * H * 512) +
                     256 * half + 4 * chk;
#pragma unroll 1
        for (int c = 8 * part / nparts; c < 8 * (part + 1) / nparts; ++c) {  // 32 columns per round
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + TM_O + 32 * c, v);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 8; ++q)
            asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(stg_row(lane, q)),
                         "f"(__uint_as_float(v[4 * q]) * inv_l), "f"(__uint_as_float(v[4 * q + 1]) * inv_l),
                         "f"(__uint_as_float(v[4 * q + 2]) * inv_l), "f"(__uint_as_float(v[4 * q + 3]) * inv_l)
                         : "memory");
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int row = 4 * i + sub;
            float4 o4;
            asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                         : "=f"(o4.x), "=f"(o4.y), "=f"(o4.z), "=f"(o4.w)
                         : "r"(stg_row(row, chk))
                         : "memory");
            if (row0 + row < H) {
              float* d = dst + (int64_t)(row0 + row) * 512 + 32 * c;
              if (split)  // read back by the combine right after this kernel: keep it in L2
                st_global_v4_hint(d, o4, pol_partial);
              else
                *reinterpret_cast<float4*>(d) = o4;
            }
          }
          __syncwarp();
        }
      } else {
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(args.out) + (int64_t)epi_qb * H * 512 + 256 * half + 8 * chk;
#pragma unroll 1
        for (int c = 4 * part / nparts; c < 4 * (part + 1) / nparts; ++c) {  // 64 columns per round
          uint32_t v[2][32];
          tmem_ld32(tmem + lane_off + TM_O + 64 * c, v[0]);
          tmem_ld32(tmem + lane_off + TM_O + 64 * c + 32, v[1]);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t* u = &v[q >> 2][(q & 3) * 8];
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(stg_row(lane, q)),
                         "r"(pack_bf16(__uint_as_float(u[0]) * inv_l, __uint_as_float(u[1]) * inv_l)),
                         "r"(pack_bf16(__uint_as_float(u[2]) * inv_l, __uint_as_float(u[3]) * inv_l)),
                         "r"(pack_bf16(__uint_as_float(u[4]) * inv_l, __uint_as_float(u[5]) * inv_l)),
                         "r"(pack_bf16(__uint_as_float(u[6]) * inv_l, __uint_as_float(u[7]) * inv_l))
                         : "memory");
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int row = 4 * i + sub;
            uint4 o;
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(o.x), "=r"(o.y), "=r"(o.z), "=r"(o.w)
                         : "r"(stg_row(row, chk))
                         : "memory");
            if (row0 + row < H) *reinterpret_cast<uint4*>(dst + (int64_t)(row0 + row) * 512 + 64 * c) = o;
          }
          __syncwarp();
        }
      }
      if (r < H && half == 0 && part == 0) {
        const float lse = (m_fin + log2f(l_tot)) * 0.69314718055994530942f;
        if (split)
          args.lse_acc[(int64_t)slot * H + r] = lse;
        else
          args.lse[(int64_t)epi_qb * H + r] = lse;
      }
      tc_fence_before();
    };

    if (w == 0) load_q_tmem(first_qb);  // piece 0's query half (the planner makes piece 0 non-empty)
    int np_qb = -1;  // query block of the piece after the current tile's (from the schedule)

    float l_mine = 0.f, m_ref = 0.f;  // this warpgroup's part of the row sum, relative to m_ref
    uint32_t slot_dep = 0;            // computed from the last values read from the exchange slot
    int my_piece = -1;                // piece that l_mine belongs to
    // FP8 cache: stage t is expanded to bf16 before QK(t) -- tile 0 by warpgroup 0 and tiles 1 and 2
    // by warpgroup 1 up front, tile t + 3 (the other warpgroup's next) by the warpgroup of tile t
    // right after publishing P(t) -- so QK(t + 3) can run before that warpgroup is done with t + 1.
    const uint32_t n_tiles = count_tiles();
    auto expand_tile = [&](uint32_t tt) -> bool {
      const uint32_t st = tt % kStages;
      if (!wait_warp(bar(B_KV_FULL + st), (tt / kStages) & 1, wc, kSiteKvFull)) return false;
      expand_fp8_stage<false>(base + st * kStageBytes, r, half, 1 + w);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_K_READY + st));
      return true;
    };
    // (warpgroup 1 takes tile 2: warpgroup 0 must not wait for page 2 before tile 0, whose query
    // load for the next piece the loading of page 2 may depend on)
    if (kFp8 && !kQk8) {
#pragma unroll 1
      for (uint32_t tt = w; ok && tt <= 2 * w && tt < n_tiles; ++tt) ok = expand_tile(tt);  // 0 | 1, 2
    }
    TileInfo x{};
    uint32_t t = 0;
    int piece = -1;
    float sq0 = 0.f, sq1 = 0.f;  // FP8 QK: query tile scales of the current tile's token
    int sq_qb = -1;
    // the schedule entry of tile tt: x, piece, np_qb; and the epilogue the tile's warpgroup owes
    // when tt opens a piece (the previous piece ended at tt-1)
    auto read_entry = [&](uint32_t tt) {
      const uint32_t e = base + SM_TI + (tt % kTiRing) * 32;
      int v[8];
      asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]) : "r"(e) : "memory");
      asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]) : "r"(e + 16) : "memory");
      x.qb = v[0];
      x.valid = v[1];
      x.split = v[2];
      x.first = (v[3] & 1) != 0;
      x.last = (v[3] & 2) != 0;
      piece = v[4];
      np_qb = v[5];
      if (x.first && tt > 0) {
        epi_pending = true;
        epi_qb = v[6];
        epi_split = v[7];
        epi_piece = piece - 1;
      }
    };
    // One tile of this warpgroup.  Two instances: the full one for the first and the last tile
    // of a piece (query load for the next piece, the finished piece's epilogue, a partial last
    // page), and a lean one for the tiles in between, which carries none of that code -- the
    // per-tile loop is sensitive to the size of its instruction stream.  (A partial page is
    // always a piece's last tile; the epilogue is always due at a piece's first.)
    auto tile = [&](auto full) -> bool {
      constexpr bool kFull = decltype(full)::value;
          const uint32_t sb = w, ph = (t >> 1) & 1;
          // ---- own partial scores; the score buffer is free again right after the read
          if (!(ok = wait_warp(bar(B_S_FULL + sb), ph, wc, kSiteSFull))) return false;
          tc_fence_after();
          // QK(t) is done: if it was the piece's last, the query half in tensor memory is free.  From
          // tile 2 on, this warpgroup's buffer (P(t-2), read by PV(t-2)) is not handed back for X(t)
          // yet: the load is staged in it.  Before that the buffer may already be receiving.
          bool handed_back = false;
          if (kFull && x.last && np_qb >= 0) {
            if (t < 2) {
              load_q_tmem(np_qb);
            } else {
              if (!(ok = wait_warp(bar(B_P_FREE + sb), ph ^ 1, wc, kSitePEmpty))) return false;
              load_q_tmem_staged(np_qb);
              if (lane == 0) mbar_arrive_remote(peer_bar0 + 8 * (B_X_FREE + sb));
              handed_back = true;
            }
          }
          uint64_t sc[32];  // score pairs: columns (2u, 2u + 1) in pair u
          float beta = 0.f;  // bias the block-float decode leaves on every score of the row
          if constexpr (kQk8) {
            // partial score = sq_0 sk_0 S_0 + sq_1 sk_1 S_1 + S_R, 16 columns at a time; the key scales
            // (this half's two of each row's four) are read from the stage, which this warpgroup
            // overwrites with the page's bf16 latent after P(t)
            const uint32_t st = t % kStages;
            if (!(ok = wait_warp(bar(B_KV_FULL + st), (t / kStages) & 1, wc, kSiteKvFull))) return false;
            const uint32_t scl = base + st * kStageBytes + kStageScales + 8 * half;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t a0[16], a1[16], ar[16];
              tmem_ld16(tmem + lane_off + TM_S8 + 16 * q, a0);
              tmem_ld16(tmem + lane_off + TM_S8 + 64 + 16 * q, a1);
              tmem_ld16(tmem + lane_off + TM_S8 + 128 + 16 * q, ar);
              tmem_wait_ld();
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                float k00, k01, k10, k11;  // (tile 2h, tile 2h + 1) scales of keys 16q + 2u and 16q + 2u + 1
                asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(k00), "=f"(k01) : "r"(scl + (16 * q + 2 * u) * 16));
                asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];"
                             : "=f"(k10), "=f"(k11)
                             : "r"(scl + (16 * q + 2 * u + 1) * 16));
                const float x0 = fmaf(__uint_as_float(a0[2 * u]), sq0 * k00,
                                      fmaf(__uint_as_float(a1[2 * u]), sq1 * k01, __uint_as_float(ar[2 * u])));
                const float x1 = fmaf(__uint_as_float(a0[2 * u + 1]), sq0 * k10,
                                      fmaf(__uint_as_float(a1[2 * u + 1]), sq1 * k11, __uint_as_float(ar[2 * u + 1])));
                sc[8 * q + u] = pack_f32x2(x0, x1);
              }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_S_EMPTY + sb));
          } else {
            uint32_t v0[32], v1[32];
            tmem_ld32(tmem + lane_off + TM_S + 64 * sb, v0);
            tmem_ld32(tmem + lane_off + TM_S + 64 * sb + 32, v1);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_S_EMPTY + sb));
  #pragma unroll
            for (int u = 0; u < 16; ++u) {
              sc[u] = pack_b32x2(v0[2 * u], v0[2 * u + 1]);
              sc[16 + u] = pack_b32x2(v1[2 * u], v1[2 * u + 1]);
            }
          }
          // this warpgroup's buffer held P(t-2): hand it back to the peer once PV(t-2) is done
          // (a relaxed arrive, made to depend on the values read from the buffer)
          if (t >= 2 && !handed_back) {
            if (!(ok = wait_warp(bar(B_P_FREE + sb), ph ^ 1, wc, kSitePEmpty))) return false;
            if (lane == 0) mbar_arrive_remote_relaxed(peer_bar0 + 8 * (B_X_FREE + sb), slot_dep);
          }
          const int valid = x.valid;
          if (kFull && valid < kTileTok) mask_pairs(sc, valid, 0.f);  // columns past the sequence end: sent as 0
          // ---- encode (16-bit block floating point, one exponent per row and tile) and send
          {
            float a[4] = {0.f, 0.f, 0.f, 0.f};
  #pragma unroll
            for (int u = 0; u < 32; ++u) {
              float x0, x1;
              unpack_f32x2(sc[u], x0, x1);
              a[(2 * u) & 3] = fmaxf(a[(2 * u) & 3], fabsf(x0));
              a[(2 * u + 1) & 3] = fmaxf(a[(2 * u + 1) & 3], fabsf(x1));
            }
            const int e = bfp_exponent(fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3])));
            const uint64_t k = splat_f32x2(pow2f(14 - e));
            if (!(ok = wait_warp(bar(B_X_FREE + sb), ph ^ 1, wc, kSiteXFree))) return false;
            const uint32_t full = peer_bar0 + 8 * (B_X_FULL + sb);
  #pragma unroll
            for (int j = 0; j < 8; ++j)  // each 16-byte chunk goes out as soon as it is encoded
              st_async_v4(peer_x + (j * kRows + r) * 16, bfp_pack_pair(sc[4 * j], k), bfp_pack_pair(sc[4 * j + 1], k),
                          bfp_pack_pair(sc[4 * j + 2], k), bfp_pack_pair(sc[4 * j + 3], k), full);
            st_async_b32(peer_xe + r * 4, (uint32_t)e, full);
          }
          // ---- the peer's half of the same scores
          if ((warp & 3) == 0 && lane == 0) mbar_arrive_expect_tx(bar(B_X_FULL + sb), kXBytes);
          if (!(ok = wait_warp<true>(bar(B_X_FULL + sb), ph, wc, kSiteXFull))) return false;
          {
            uint32_t pe;
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(pe) : "r"(my_xe + r * 4));
            slot_dep = pe;
            const float kpf = pow2f((int)pe + 1);
            const uint64_t kp = splat_f32x2(kpf);
            beta = 1.5f * kpf;  // exact
  #pragma unroll
            for (int j = 0; j < 8; ++j) {
              uint32_t wv[4];
              asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                           : "=r"(wv[0]), "=r"(wv[1]), "=r"(wv[2]), "=r"(wv[3])
                           : "r"(my_x + (j * kRows + r) * 16));
              slot_dep ^= wv[0] ^ wv[3];
  #pragma unroll
              for (int q = 0; q < 4; ++q) sc[4 * j + q] = ffma_f32x2(bfp_unpack_pair(wv[q]), kp, sc[4 * j + q]);
            }
          }
          if (kFull && valid < kTileTok) mask_pairs(sc, valid, -INFINITY);
          float cm;
          {
            float c[4];
  #pragma unroll
            for (int q = 0; q < 4; ++q) {
              float x0, x1;
              unpack_f32x2(sc[q], x0, x1);
              c[q] = fmaxf(x0, x1);
            }
  #pragma unroll
            for (int u = 4; u < 32; ++u) {
              float x0, x1;
              unpack_f32x2(sc[u], x0, x1);
              c[u & 3] = fmax3(c[u & 3], x0, x1);
            }
            cm = (fmax3(c[0], c[1], fmaxf(c[2], c[3])) - beta) * sl2;  // log2 units (sl2 > 0)
          }
          // ---- running max: decided from the previous tile's (the other warpgroup's)
          float m_prev = 0.f, l_other = 0.f;
          if (t > 0) {
            if (!(ok = wait_warp(bar(B_ML + (sb ^ 1)), ((t - 1) >> 1) & 1, wc, kSiteML))) return false;
            m_prev = ml[((sb ^ 1) * 2) * kRows + r];
            l_other = ml[((sb ^ 1) * 2 + 1) * kRows + r];
          }
          float m = m_prev, alpha = 1.f;
          if (kFull && x.first) {
            // finite unless this token sees no key of the tile (a token before the last of a group,
            // on the group's last tile): then any finite value, the tile's P is zero
            m = (!kGroups || cm > -INFINITY) ? cm : 0.f;
          } else if (cm > m_prev + 8.f) {
            m = cm;
            alpha = exp2f(m_prev - cm);
          }
          // the finished piece (last tile t-1) takes both warpgroups' row sums at its final max
          float epi_l = 0.f;
          if (kFull && epi_pending) epi_l = l_other + (my_piece == epi_piece ? l_mine * exp2f(m_ref - m_prev) : 0.f);
          // ---- the previous piece's epilogue (O after PV(t-1)), staged in this warpgroup's buffer
          // once every thread has read its exchange data from it; P(t) goes there afterwards
          if (kFull && epi_pending) {
            asm volatile("bar.sync %0, 128;" ::"r"(1 + w) : "memory");
            if (!(ok = wait_warp(bar(B_P_FREE + (sb ^ 1)), ((t - 1) >> 1) & 1, wc, kSitePEmpty))) return false;
            tc_fence_after();
            epilogue(m_prev, epi_l, 0, 1);
            epi_pending = false;
            asm volatile("bar.sync %0, 128;" ::"r"(1 + w) : "memory");
          }
          // ---- exponentials; each thread stores its P row where it read its exchange data (16-byte
          // chunk j of row r at (j * 128 + r) * 16: the K-major layout without swizzle that PV reads),
          // so no thread writes where another still reads
          float rsum;
          {
            const uint64_t s2 = splat_f32x2(sl2), nm = splat_f32x2(-fmaf(beta, sl2, m));
            uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
  #pragma unroll
            for (int j = 0; j < 8; ++j) {
              uint32_t pp[4];
  #pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int u = 4 * j + q;
                float x0, x1;
                unpack_f32x2(ffma_f32x2(sc[u], s2, nm), x0, x1);
                const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                pp[q] = pack_bf16(p0, p1);
                acc[q] = fadd_f32x2(acc[q], pack_f32x2(p0, p1));
              }
              asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(my_x + (j * kRows + r) * 16), "r"(pp[0]),
                           "r"(pp[1]), "r"(pp[2]), "r"(pp[3]));
            }
            float z[8];
            unpack_f32x2(fadd_f32x2(fadd_f32x2(acc[0], acc[1]), fadd_f32x2(acc[2], acc[3])), z[0], z[1]);
            rsum = z[0] + z[1];
          }
          if (piece != my_piece) {
            my_piece = piece;
            l_mine = 0.f;
            m_ref = m;
          }
          l_mine = l_mine * exp2f(m_ref - m) + rsum;
          m_ref = m;
          ml[(sb * 2) * kRows + r] = m;
          ml[(sb * 2 + 1) * kRows + r] = l_mine;
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_ML + sb));
          // ---- a raised running max rescales O (after PV(t-1), before PV(t))
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
            if (!(ok = wait_warp(bar(B_P_FREE + (sb ^ 1)), ((t - 1) >> 1) & 1, wc, kSitePEmpty))) return false;
            tc_fence_after();
  #pragma unroll 1
            for (int c = 0; c < 8; ++c) {
              uint32_t v[32];
              tmem_ld32(tmem + lane_off + TM_O + 32 * c, v);
              tmem_wait_ld();
  #pragma unroll
              for (int jj = 0; jj < 32; ++jj) v[jj] = __float_as_uint(__uint_as_float(v[jj]) * alpha);
              tmem_st32(tmem + lane_off + TM_O + 32 * c, v);
            }
            tmem_wait_st();
          }
          // ---- publish P
          if (kFull && !kQk8 && valid < kTileTok) {
            // rows past the sequence end must not reach the PV product (0 * garbage): zero them
            // (FP8 QK: the expansion warpgroup writes them as zeros)
            const uint32_t sbase = base + (t % kStages) * kStageBytes;
            const int v0 = valid > 0 ? valid : 0;
            const int nz = (kTileTok - v0) * 4 * 8;  // 16-byte chunks: rows x 4 blocks x 8
            for (int idx = r; idx < nz; idx += kRows) {
              const int row = v0 + idx / 32, blk = (idx / 8) & 3, ch = idx & 7;
              asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(sbase + blk * kLatBlock + row * 128 + ch * 16),
                           "r"(0u));
            }
          }
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_P_FULL + sb));
          if (kQk8) {  // FP8 QK: this tile's page to bf16 for PV(t) (QK(t) has read the codes, this
                       // warpgroup the key scales)
            const uint32_t st = t % kStages;
            expand_fp8_stage<true>(base + st * kStageBytes, r, half, 1 + w, valid);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_K_READY + st));
          }
          if (kFp8 && !kQk8 && t + 3 < n_tiles && !(ok = expand_tile(t + 3))) return false;
      return true;
    };
    // this warpgroup's tiles: t = w, w + 2, ...
    for (t = w; ok && t < n_tiles; t += 2) {
      if (!(ok = wait_warp(bar(B_TI_FULL + (t % kTiRing)), (t / kTiRing) & 1, wc, kSiteSFull))) break;
      read_entry(t);
      if (kQk8 && x.qb != sq_qb) {  // this row's two query tile scales (of this half) for the tile's token
        sq_qb = x.qb;
        float2 v = make_float2(0.f, 0.f);
        if (r < H)
          v = *reinterpret_cast<const float2*>(static_cast<const uint8_t*>(args.q_nope) + ((int64_t)x.qb * H + r) * 656 +
                                               512 + 8 * half);
        sq0 = v.x;
        sq1 = v.y;
      }
      if (kQk8 && x.first && np_qb >= 0 && r < H) {  // the next piece's 656-byte query row into L2
        const char* q8 = reinterpret_cast<const char*>(args.q_nope) + ((int64_t)np_qb * H + r) * 656;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(q8 + 256 * half));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(q8 + 256 * half + 128));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(q8 + 512));
      } else if (x.first && np_qb >= 0 && r < H) {  // bring the next piece's query rows into L2 for its load
        const char* qn = reinterpret_cast<const char*>(args.q_nope) + (((int64_t)np_qb * H + r) * 512 + 256 * half) * 2;
        const char* qr = reinterpret_cast<const char*>(args.q_rope) + (((int64_t)np_qb * H + r) * 64 + 32 * half) * 2;
#pragma unroll
        for (int k = 0; k < 4; ++k) asm volatile("prefetch.global.L2 [%0];" ::"l"(qn + 128 * k));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(qr));
      }
      // (the lean instance first: it is the one the loop runs back to back)
      if (__builtin_expect(!(x.first || x.last || (kGroups && x.valid < kTileTok)), 1)) {
        if (!tile(std::false_type{})) {
          ok = false;
          break;
        }
      } else if (!tile(std::true_type{})) {
        ok = false;
        break;
      }
    }
    // the unit's last tile n_tiles-1 (its entry is still in the ring): its piece ends the unit
    t = n_tiles;
    if (ok && t > 0) {
      if (!(ok = wait_warp(bar(B_TI_FULL + ((t - 1) % kTiRing)), ((t - 1) / kTiRing) & 1, wc, kSiteSFull))) t = 0;
      const bool pend = epi_pending;
      read_entry(t - 1);
      epi_pending = pend;
      epi_qb = x.qb;
      epi_split = x.split;
      epi_piece = piece;
    }
    // The unit's last piece: both warpgroups write half of its columns each, from the same final
    // max and row sum (same operands, same operations).  The owner of the last tile t-1 takes the
    // other warpgroup's share from what that one published for tile t-2 (if t-2 is in the piece,
    // i.e. t-1 did not open it; x still describes tile t-1), the other one from what the owner
    // published for t-1.
    if (ok && t > 0) {
      const uint32_t pp = (t - 1) & 1;
      const bool owner = pp == w;
      float m_fin = m_ref, l_tot = 0.f;
      bool go = true;
      if (owner) {
        const uint32_t po = pp ^ 1;
        l_tot = l_mine + (x.first ? 0.f : ml[(po * 2 + 1) * kRows + r] * exp2f(ml[(po * 2) * kRows + r] - m_fin));
      } else {  // epi_pending: the other warpgroup's tile t-1 ended the piece
        go = wait_warp(bar(B_ML + pp), ((t - 1) >> 1) & 1, wc, kSiteML);
        m_fin = ml[(pp * 2) * kRows + r];
        const float l_other = ml[(pp * 2 + 1) * kRows + r];
        l_tot = l_other + (my_piece == epi_piece ? l_mine * exp2f(m_ref - m_fin) : 0.f);
      }
      if (go && wait_warp(bar(B_P_FREE + pp), ((t - 1) >> 1) & 1, wc, kSitePEmpty)) {
        tc_fence_after();
        epilogue(m_fin, l_tot, owner ? 1 : 0, 2);
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncwarp();  // the producer and MMA-issuer warps worked on one lane: reconverge before the barriers
  __syncthreads();
  if (*abort_flag) drain_delay(200000);  // in-flight TMA / st.async / MMA land before release
  cluster_sync();                        // the peer no longer touches our shared memory
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// One pair per new token (clusters of 2 CTAs) and token groups (clusters of 2G CTAs, G > 1) are
// separate instances: the grouped code costs the per-token kernel registers.
__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_bf16_kernel(const __grid_constant__ DecodeArgs args) {
  decode_body<false, false>(args);
}
__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_fp8_kernel(const __grid_constant__ DecodeArgs args) {
  decode_body<true, false>(args);
}
__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_bf16_group_kernel(const __grid_constant__ DecodeArgs args) {
  decode_body<false, true>(args);
}
__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_fp8_group_kernel(const __grid_constant__ DecodeArgs args) {
  decode_body<true, true>(args);
}
// FP8 cache with QK on the E4M3 codes (opt-in): one pair per new token
__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_fp8qk_kernel(const __grid_constant__ DecodeArgs args) {
  decode_body<true, false, true>(args);
}

}  // namespace mla
