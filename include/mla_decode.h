/*
 * mla_decode.h -- C ABI of libmla_decode.so: weight-absorbed Multi-Head Latent
 * Attention decode on GB300 (sm_103a).
 *
 * The operation ("MLA inference: two computation paths and FlashMLA", section
 * "Two equivalent paths", path two; "MLA: what the multi-head latent attention
 * paper actually says", section "The absorbed form: how inference actually
 * works"): every query head h of new token t of sequence b holds an absorbed
 * query q~ (512 dims, W_UK already folded in by the caller) and a RoPE query
 * q^R (64 dims).  Each cached token j holds a 512-dim latent c_j and a 64-dim
 * RoPE key k^R_j shared by all heads (576 numbers per token).  The library
 * computes
 *     s_j = scale * (q~ . c_j + q^R . k^R_j)
 *     out = sum_j softmax(s)_j * c_j        (512 dims, latent space; W_UV is NOT applied)
 *     lse = ln sum_j exp(s_j)               (natural log, scale applied)
 * over the keys the token may see.  The cache is paged, 64 tokens per page,
 * addressed through a per-sequence block table ("FlashMLA: Fast Hopper
 * Decoding for Latent Attention Guide", section "1. Direct Paged Latent
 * Ingestion (512 + 64)"); long sequences are split across SMs and the partial
 * results are merged through their LSE (split-KV, "MLA inference: two
 * computation paths and FlashMLA", section "Decode attention becomes a compute
 * problem"), with the split plan computed on the device from the context
 * lengths (the "scheduling metadata precomputed from context lengths" of the
 * same section).
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" are CUDA device pointers on the current device;
 *     "host" pointers are ordinary host memory.  All device buffers are owned
 *     by the caller; the library never allocates or frees device memory and
 *     never synchronises on the decode path.  Device buffers must be
 *     contiguous in the stated layout and 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls are asynchronous on that stream.
 *   - Return value: an mla_status.  Problems the host can see (null pointers,
 *     bad sizes, unsupported options, a CUDA launch error) are returned at
 *     once and nothing is launched.  Problems only the device can see (a
 *     bounded wait that ran out) are recorded in a per-device error word that
 *     mla_device_error() reads; outputs of such a call are undefined.
 *   - Not thread-safe per (device, stream) for concurrent calls sharing one
 *     workspace.
 */
#ifndef MLA_DECODE_H
#define MLA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned buffer */
  MLA_ERR_UNSUPPORTED = 2,  /* valid request the library does not implement (e.g. H > 128, s_q > 8) */
  MLA_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed (no device, launch failure, ...) */
  MLA_ERR_TIMEOUT = 4,      /* device error word: a bounded wait inside a kernel ran out */
  MLA_ERR_WORKSPACE = 5,    /* scheduler metadata does not match the params (wrong unit count or batch) */
  MLA_ERR_SCRATCH_LIMIT = 6, /* mla_decode_noalloc: the request needs more than MLA_NOALLOC_SCRATCH_BYTES */
} mla_status;

typedef enum {
  MLA_KV_BF16 = 0,          /* page = [64][576] bf16: c (512) then k^R (64); 1152 bytes per token */
  MLA_KV_FP8_E4M3 = 1,      /* page = [64][656 bytes]: 512 E4M3 codes of c, then 4 float32 scales
                               (one per 128-code tile, value = code * scale), then k^R as 64 bf16 */
} mla_kv_dtype;

typedef enum {
  MLA_OUT_BF16 = 0,
  MLA_OUT_F32 = 1,
} mla_out_dtype;

/* Problem description shared by all calls of one decode step. */
typedef struct mla_decode_params {
  int32_t batch;             /* B >= 1 sequences */
  int32_t s_q;               /* new tokens per sequence, 1..8 (MTP / speculative decoding); each
                                new token is its own query block of H rows */
  int32_t num_heads;         /* H, 1..128 query heads */
  int32_t num_pages;         /* physical pages in the pool (>= 1) */
  int32_t page_size;         /* tokens per page; must be 64 */
  int32_t max_pages_per_seq; /* row length of block_table (>= 1) */
  int32_t causal;            /* s_q > 1: nonzero => new token t sees keys 0 .. L_b - s_q + t;
                                zero => every new token sees all L_b keys */
  int32_t kv_dtype;          /* mla_kv_dtype */
  int32_t out_dtype;         /* mla_out_dtype */
  int32_t num_units;         /* work units (one cluster of 2G SMs each, G = the token group); 0 = as
                                many as fit at once */
  int32_t timeout_us;        /* limit of every bounded wait inside the kernels; 0 = 2,000,000 us */
  int32_t token_group;       /* G: new tokens of a sequence decoded together on shared pages: each page
                                is read from memory once for the G tokens (one CTA pair per token, a
                                cluster of 2G CTAs, pages multicast to every pair); 1..4 and dividing
                                s_q; 0 = 1.  Clusters of 4 / 8 CTAs occupy 144 / 120 of GB300's 152 SMs,
                                so G > 1 pays where DRAM, not the SMs, bounds the decode */
  int32_t qk_fp8;            /* FP8 cache only, opt-in (0 or 1): 1 => QK runs on E4M3 codes on the FP8 tensor
                                cores ("MLA inference: two computation paths and FlashMLA", exercise 2
                                "An FP8 KV cache").  The query is then passed quantised like the cache:
                                q_nope_absorbed points to [B][s_q][H][656 bytes] rows written by
                                mla_quantize_q_fp8 (the absorbed query's 512 codes, 4 tile scales, q^R
                                as 64 bf16) and q_rope is not read (may be NULL).  The result is that of
                                attention with the dequantised query (code x scale), not the bf16 one.
                                Needs token_group <= 1; 0 = QK on the bf16-expanded cache */
  int32_t reserved[3];       /* must be zero */
} mla_decode_params;

/*
 * Sizes of the two caller-provided device buffers for a decode with `p`:
 *   *sched_bytes     -- scheduler metadata written by mla_get_scheduler_metadata
 *   *workspace_bytes -- split partials (float32) used by mla_decode
 * Both depend only on p (batch, s_q, num_heads, unit count), never on the
 * context lengths, so buffers can be allocated once and reused.  Needs a CUDA
 * device only when p->num_units == 0 (to count SMs).
 */
int32_t mla_get_workspace_size(const mla_decode_params* p, size_t* sched_bytes, size_t* workspace_bytes);

/*
 * Split plan ("which stretches of KV each SM handles"): reads the per-sequence
 * lengths cache_seqlens (device, int32 [B], each length counts the s_q new
 * tokens) and writes `sched` (device, sched_bytes).  One tiny kernel; no host
 * synchronisation.  Compute it once per decode step and reuse it for every
 * layer that shares the lengths.
 */
int32_t mla_get_scheduler_metadata(const mla_decode_params* p, const int32_t* cache_seqlens, void* sched,
                                   void* stream);

/*
 * The decode.
 *   q_nope_absorbed  device bf16 [B][s_q][H][512]  absorbed query q~ (qk_fp8: the 656-byte rows of
 *                    mla_quantize_q_fp8)
 *   q_rope           device bf16 [B][s_q][H][64]   RoPE query q^R (qk_fp8: not read)
 *   kv_pages         device [num_pages][64][576] bf16, or [num_pages][64][656 bytes] FP8 rows
 *   block_table      device int32 [B][max_pages_per_seq]: physical page of logical page i of
 *                    sequence b; entries past ceil(L_b/64) are never read.  Every entry read
 *                    must be in [0, num_pages).
 *   cache_seqlens    device int32 [B]; L_b includes the s_q new tokens; 0 <= L_b <= 64*max_pages
 *                    (a longer length sets MLA_ERR_INVALID_ARG in the device error word; the
 *                    kernel then reads no block-table entry past the row, and that sequence's
 *                    result is undefined; a negative length sets the same error and is decoded
 *                    as an empty sequence)
 *   scale            softmax scale, finite and > 0 (1/sqrt(192) for DeepSeek-V3 shapes)
 *   out              device [B][s_q][H][512], bf16 or float32 (out_dtype)
 *   lse              device float32 [B][s_q][H]; a token that sees no key gets out = 0, lse = -inf
 *   sched            device, from mla_get_scheduler_metadata with the same p and lengths
 *   workspace        device, workspace_bytes from mla_get_workspace_size
 * Cache rows of the last page past L_b are not used (they may hold any bits).
 */
int32_t mla_decode(const mla_decode_params* p, const void* q_nope_absorbed, const void* q_rope, const void* kv_pages,
                   const int32_t* block_table, const int32_t* cache_seqlens, float scale, void* out, float* lse,
                   const void* sched, void* workspace, void* stream);

/*
 * The two halves of mla_decode, for callers that want to place or time them
 * separately (same arguments and rules as mla_decode):
 *   mla_decode_splitkv -- the decode kernel only: writes out/lse of every query
 *                         token whose keys one unit handled, and the split
 *                         partials (in workspace) of the others;
 *   mla_combine        -- merges the split partials through their LSE into
 *                         out/lse and writes out = 0, lse = -inf for tokens that
 *                         see no key.  Must follow mla_decode_splitkv on the
 *                         same stream with the same p, sched and workspace.
 * mla_decode == mla_decode_splitkv followed by mla_combine.
 */
int32_t mla_decode_splitkv(const mla_decode_params* p, const void* q_nope_absorbed, const void* q_rope,
                           const void* kv_pages, const int32_t* block_table, const int32_t* cache_seqlens, float scale,
                           void* out, float* lse, const void* sched, void* workspace, void* stream);
int32_t mla_combine(const mla_decode_params* p, void* out, float* lse, const void* sched, void* workspace,
                    void* stream);

/*
 * Host-side twin of the split planner (the same code the scheduler kernel runs),
 * for tests and capacity planning.  cache_seqlens and sched are HOST pointers;
 * num_units must be >= 1; sched must hold sched_bytes for that unit count.
 * Layout of sched (int32): [0] = 0x4D4C4131, [1] = units, [2] = B*s_q query blocks,
 * [3] = partial slots used, [4] = per-unit budget of work positions (one per 64-key
 * tile plus a fixed cost per work block; diagnostic), [5] = G, the token group,
 * [6..7] = 0; then per unit 8 ints {wb_begin, tile_begin, wb_end, tile_end (exclusive),
 * first_split, 0, 0, 0} (wb_begin = -1: no work); then num_splits[B*s_q]; then
 * split_offset[B*s_q].  A query block qb = b*s_q + t; a work block wb holds the G query
 * blocks wb*G .. wb*G + G - 1 (G = 1: wb = qb), and its tiles are those of its last
 * token; num_splits is the same for the G query blocks of a work block.
 * Returns MLA_ERR_INVALID_ARG for a negative length, or for lengths whose work
 * positions exceed 2^31 - 1 in total (sched then holds a header without the magic
 * word).  The scheduler kernel (mla_get_scheduler_metadata) reports the same two
 * cases in the device error word: it plans a negative length as an empty sequence,
 * and for the oversized case writes that invalid header, so the decode writes nothing.
 */
int32_t mla_plan_host(const mla_decode_params* p, int32_t num_units, const int32_t* cache_seqlens, void* sched);

/* Unit count mla_decode would use for p on the current device (0 -> as many clusters as fit). */
int32_t mla_resolve_num_units(const mla_decode_params* p, int32_t* num_units);

/*
 * Writes the FP8 form of a bf16 cache ("MLA and FP8 MoE Serving: Multi-Head Latent
 * Attention at Scale", section "Understanding FP8 Formats: E4M3 vs. E5M2"; "MLA inference:
 * two computation paths and FlashMLA", exercise 2 "An FP8 KV Cache"), in the layout
 * MLA_KV_FP8_E4M3 reads.
 *   kv_bf16   device bf16 [num_tokens][576]: latent c (512) then k^R (64)
 *   kv_fp8    device [num_tokens][656 bytes]: 512 E4M3 codes, 4 float32 scales (one per
 *             128-element latent tile), the 64 bf16 RoPE values copied unchanged
 * Per tile: scale = amax / 448 (1 for an all-zero tile); code = E4M3(clamp(x / scale,
 * -448, 448)) rounded to nearest even; the decoded value is code * scale.  num_tokens = 0
 * launches nothing.  Both buffers 16-byte aligned; asynchronous on stream.
 */
int32_t mla_quantize_kv_fp8(const void* kv_bf16, void* kv_fp8, int64_t num_tokens, void* stream);

/*
 * The query of an FP8-QK decode (mla_decode_params.qk_fp8), quantised like a cache row:
 *   q_nope_absorbed  device bf16 [num_rows][512]  absorbed query q~ (num_rows = B * s_q * H)
 *   q_rope           device bf16 [num_rows][64]   RoPE query q^R
 *   q_fp8            device [num_rows][656 bytes]: 512 E4M3 codes of q~, 4 float32 tile scales,
 *                    then q^R copied unchanged as 64 bf16
 * Per 128-element tile: the rule of mla_quantize_kv_fp8.  num_rows = 0 launches nothing.  All
 * buffers 16-byte aligned; asynchronous on stream.
 */
int32_t mla_quantize_q_fp8(const void* q_nope_absorbed, const void* q_rope, void* q_fp8, int64_t num_rows,
                           void* stream);

/*
 * Query absorption ("MLA inference: two computation paths and FlashMLA", section "Two
 * equivalent paths", path two: W_UK is folded into the query; "MLA: what the multi-head
 * latent attention paper actually says", section "The absorbed form: how inference actually
 * works"): for every token t and head h
 *     q_absorbed[t][h][:] = q_nope[t][h][:] . W_UK[h]          (512 = d_c columns)
 *   n_tokens    T >= 1 (B * s_q of a decode step)
 *   num_heads   H, 1..65535
 *   d_nope      per-head no-RoPE query dims (128 in DeepSeek-V3); a multiple of 64, <= 4096
 *   q_nope      device bf16 [T][H][d_nope]
 *   w_uk        device bf16 [H][d_nope][512]
 *   q_absorbed  device bf16 [T][H][512]: the q_nope_absorbed input of mla_decode
 * bf16 inputs, fp32 accumulation on the tensor cores, bf16 output (rounded to nearest even).
 * Buffers 16-byte aligned; asynchronous on stream (a programmatic dependent of the kernel
 * before it).  Unsupported sizes return MLA_ERR_UNSUPPORTED before any launch.
 */
int32_t mla_absorb_query(int32_t n_tokens, int32_t num_heads, int32_t d_nope, const void* q_nope, const void* w_uk,
                         void* q_absorbed, void* stream);

/*
 * Value projection, the last step of the absorbed path (same sections: W_UV applied to the
 * latent output): for every token t and head h
 *     out[t][h][:] = o_latent[t][h][:] . W_UV[h]               (d_v columns)
 *   o_latent    device bf16 [T][H][512]: the out of mla_decode (bf16 output)
 *   w_uv        device bf16 [H][512][d_v]
 *   d_v         per-head value dims (128 in DeepSeek-V3); a multiple of 64, <= 4096
 *   out         device bf16 [T][H][d_v]
 * Same arithmetic, alignment and error rules as mla_absorb_query.
 */
int32_t mla_project_output(int32_t n_tokens, int32_t num_heads, int32_t d_v, const void* o_latent, const void* w_uv,
                           void* out, void* stream);

/*
 * Extend by the expand path, chunk by chunk ("MLA inference: two computation paths and
 * FlashMLA", section "Two equivalent paths", path one, and section "Which is faster: count
 * new tokens and cached tokens": with many new tokens the keys and values are expanded per
 * head and attended as ordinary multi-head attention; a long prefix is expanded a chunk at a
 * time and the chunks' results are merged by their log-sum-exp).  Sequence b has L_b cached
 * rows, the last s_q of them its new tokens; new token t attends to rows 0 .. L_b - s_q + t.
 */
typedef struct mla_extend_params {
  int32_t batch;             /* B >= 1 sequences (<= 65535) */
  int32_t s_q;               /* new tokens per sequence, >= 1, already written into the cache */
  int32_t num_heads;         /* H, 1..128 */
  int32_t d_nope;            /* per-head no-RoPE query/key dims; must be 128 */
  int32_t d_v;               /* per-head value dims; must be 128 */
  int32_t num_pages;         /* physical pages in the pool (>= 1) */
  int32_t page_size;         /* must be 64 */
  int32_t max_pages_per_seq; /* row length of block_table (>= 1) */
  int32_t max_seqlen;        /* an upper bound of every L_b, s_q <= max_seqlen <= 64 * max_pages_per_seq;
                                it fixes the number of chunks, ceil(max_seqlen / chunk_tokens) */
  int32_t chunk_tokens;      /* C: cached rows expanded at a time; a multiple of 128 */
  int32_t timeout_us;        /* limit of every bounded wait inside the kernels; 0 = 2,000,000 us */
  int32_t reserved[5];       /* must be zero */
} mla_extend_params;

/*
 * Size of the device workspace mla_extend needs for p: the expanded keys and values of one
 * chunk (bf16, 2 * B * H * C * 128 * 2 bytes) and the float32 accumulators of the merge
 * (B * s_q * H * 129 * 4 bytes), each rounded up to 256 bytes.  Host only.
 */
int32_t mla_extend_workspace_size(const mla_extend_params* p, size_t* workspace_bytes);

/*
 * The expansion of one chunk (path one's per-head keys and values): for every sequence b,
 * head h and row j of [chunk_start, chunk_start + C)
 *     k_nope[b][h][j - chunk_start][:] = W_UK[h] . c_j      (d_nope values)
 *     v[b][h][j - chunk_start][:]      = c_j . W_UV[h]      (d_v values)
 * with c_j the 512 latent values of cache row j; rows j >= L_b are written as zeros, except
 * whole 128-row tiles at or past L_b, which are not written.
 *   kv_pages      device bf16 [num_pages][64][576] (the MLA_KV_BF16 layout)
 *   block_table   device int32 [B][max_pages_per_seq]; cache_seqlens device int32 [B]
 *                 (a length < s_q or > 64 * max_pages_per_seq sets MLA_ERR_INVALID_ARG in the
 *                 device error word and that sequence is skipped)
 *   w_uk          device bf16 [H][d_nope][512]; w_uv device bf16 [H][512][d_v] (the layouts
 *                 of mla_absorb_query and mla_project_output)
 *   chunk_start   a multiple of chunk_tokens, >= 0
 *   k_nope, v     device bf16 [B][H][chunk_tokens][128]
 * bf16 inputs, fp32 accumulation on the tensor cores, bf16 outputs rounded to nearest even.
 * Buffers 16-byte aligned; asynchronous on stream.
 */
int32_t mla_expand_kv(const mla_extend_params* p, const void* kv_pages, const int32_t* block_table,
                      const int32_t* cache_seqlens, const void* w_uk, const void* w_uv, int32_t chunk_start,
                      void* k_nope, void* v, void* stream);

/*
 * The extend: for each chunk of C rows, mla_expand_kv into the workspace, then attention of
 * every new token over the chunk's rows it may see,
 *     score_j = scale * (q_nope . k^N_j + q_rope . k^R_j)     (k^R_j: the 64 RoPE values of row j)
 * with an online softmax, merged with the chunks before by their log-sum-exp (float32).
 *   q_nope   device bf16 [B][s_q][H][128]; q_rope device bf16 [B][s_q][H][64]
 *   kv_pages, block_table, cache_seqlens, w_uk, w_uv   as for mla_expand_kv
 *   scale    softmax scale, finite and > 0 (1/sqrt(192) for DeepSeek-V3 shapes)
 *   out      device bf16 [B][s_q][H][d_v]: softmax-weighted sum of the values
 *   lse      device float32 [B][s_q][H]: natural log of the sum of exp(score) over the visible rows
 *   workspace  device, mla_extend_workspace_size(p) bytes, 256-byte aligned
 * Keys and values are held in bf16 between the two kernels, P in bf16 for the P.V product.
 * 2 * ceil(max_seqlen / C) launches on stream, each a programmatic dependent of the one before.
 */
int32_t mla_extend(const mla_extend_params* p, const void* q_nope, const void* q_rope, const void* kv_pages,
                   const int32_t* block_table, const int32_t* cache_seqlens, const void* w_uk, const void* w_uv,
                   float scale, void* out, float* lse, void* workspace, void* stream);

/*
 * Device error word of the current device: synchronises the device, writes the
 * word to *word (MLA_OK if none; MLA_ERR_TIMEOUT + 16 * site for a bounded wait that ran
 * out; MLA_ERR_INVALID_ARG for a length beyond the block table; MLA_ERR_WORKSPACE for
 * scheduler metadata that does not match the params) and,
 * if clear != 0, resets it.  Host pointer.
 */
int32_t mla_device_error(int32_t* word, int32_t clear);

/*
 * Failure-path self test: launches one CTA whose bounded wait on a barrier that
 * nothing completes runs out after timeout_us, sets the device error word and
 * returns normally.  The GPU context stays usable.  Read the result with
 * mla_device_error().
 */
int32_t mla_wait_selftest(int32_t timeout_us, void* stream);

/*
 * Allocation-free decode, for callers that cannot call cudaMalloc on their
 * decode path: serving engines and plugin hosts that reserve all device memory
 * for their own pool allocator at start-up (a cudaMalloc would take memory from
 * outside that pool, and cudaMalloc/cudaFree can synchronise the device in the
 * middle of a step).  The paper has no counterpart; it is an interface of this
 * library only.
 *
 * Same inputs, outputs, rules and results as mla_get_scheduler_metadata
 * followed by mla_decode with the same p, but the scheduler metadata and the
 * split partials live in one fixed device array inside the library,
 * MLA_NOALLOC_SCRATCH_BYTES (64 MiB) per GPU, reserved by the CUDA runtime
 * when it loads the library's device code on that GPU and held until the
 * process exits.  It holds
 * align256(sched_bytes) + workspace_bytes of mla_get_workspace_size: with 128
 * heads, batch * s_q plus the unit count up to 255.  A larger request returns
 * MLA_ERR_SCRATCH_LIMIT and launches nothing.  The call itself allocates
 * nothing (no cudaMalloc, cudaFree or allocating library routine).
 *
 * The first call on a device also looks up the array's device address for that
 * device (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.
 *
 * Every call on a device shares the one array, which keeps the last call's
 * contents; nothing in it needs to start at zero.  Calls whose kernels overlap
 * on the GPU (other streams, other host threads) race on the array and give
 * undefined results: order them on one stream or with events.
 */
#define MLA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int32_t mla_decode_noalloc(const mla_decode_params* p, const void* q_nope_absorbed, const void* q_rope,
                           const void* kv_pages, const int32_t* block_table, const int32_t* cache_seqlens,
                           float scale, void* out, float* lse, void* stream);

/* Human-readable name of a status (static string). */
const char* mla_status_string(int32_t status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H */
