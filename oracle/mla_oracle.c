/*
 * Oracle for absorbed-path MLA decode — TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, single-threaded fp64 C.  Only the tests, the smoke check and
 * the CPU-baseline leg of the benchmark call it; the product library never
 * links or loads it, and it shares no code, header or table with the CUDA
 * path.  Every floating-point input is widened exactly to double before any
 * arithmetic (bf16 -> double and E4M3 code * float32 scale -> double are both
 * exact), and everything after that is fp64.
 *
 * What it computes, per query block (b, t) and head h, is the plain
 * definition of the weight-absorbed decode:
 *
 *   s_j   = scale * ( sum_{d < d_c} qn[d] * c_j[d] + sum_{r < d_r} qr[r] * kR_j[r] )
 *           ("MLA inference: two computation paths and FlashMLA", section
 *            "Two equivalent paths": the score is the latent dot product plus
 *            the shared-RoPE dot product, path two)
 *   p_j   = exp(s_j - m) / sum_i exp(s_i - m),  m = max_j s_j   (exact softmax)
 *   out   = sum_j p_j * c_j[0:d_c]            (the latent itself is the value;
 *            same section: "the weighted sum is also taken in latent space")
 *   lse   = m + ln(sum_j exp(s_j - m))         (natural log, scale applied)
 *
 * Key j of sequence b lives at row page*page_size + j % page_size of the
 * pool, page = block_table[b][j / page_size]  (paged KV with block tables,
 * "FlashMLA: Fast Hopper Decoding for Latent Attention Guide", section
 * "1. Direct Paged Latent Ingestion (512 + 64)").
 *
 * Visible keys: cache_seqlens[b] counts the s_q new tokens; with the causal
 * flag, new token t (0-based) sees keys 0 .. L_b - s_q + t (the "k includes
 * the new tokens" convention of the flops(q, k) accounting in section "Which
 * is faster: count new tokens and cached tokens").  Without it every new
 * token sees all L_b keys.  No visible key: out = 0, lse = -inf.
 *
 * Cache row formats (kv_kind):
 *   ORC_KV_F64 : double  [rows][d_c + d_r]
 *   ORC_KV_BF16: bf16    [rows][d_c + d_r]  (raw 16-bit patterns)
 *   ORC_KV_FP8 : bytes   [rows][d_c + 4*(d_c/128) + 2*d_r] =
 *                d_c E4M3 codes | one float32 scale per 128-code tile | d_r bf16
 *                (latent stored as FP8 E4M3 with per-tile scales, RoPE part
 *                kept bf16; E4M3 format from "MLA and FP8 MoE Serving",
 *                section "Understanding FP8 Formats: E4M3 vs. E5M2").
 *
 * Parity status: every function here is pinned by a test under tests/
 * (absorb == expand, split-merge == unsplit, weights sum to one, page
 * permutation invariance, brute force, closed forms, the 256 E4M3 codes).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_KV_F64 0
#define ORC_KV_BF16 1
#define ORC_KV_FP8 2

typedef struct {
  int32_t batch, s_q, num_heads, causal;
  int32_t d_c, d_r;
  int32_t page_size, max_pages_per_seq;
  int32_t kv_kind;
  int32_t reserved;
  double scale;
  const double* q_nope;        /* [batch][s_q][num_heads][d_c] */
  const double* q_rope;        /* [batch][s_q][num_heads][d_r] */
  const void* kv;              /* page pool, format kv_kind */
  const int32_t* block_table;  /* [batch][max_pages_per_seq] */
  const int32_t* seqlens;      /* [batch], includes the s_q new tokens */
} orc_problem;

/* bf16 is the upper half of an IEEE binary32; the widening is exact. */
static double bf16_bits_to_f64(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* E4M3 ("fn" flavour: no infinities, S.1111.111 is NaN, largest finite
 * magnitude 448): exponent bias 7, 3 mantissa bits, subnormals at exponent
 * field 0.  Written from the format definition, not from any library. */
double orc_e4m3_to_f64(uint8_t code) {
  int sign = code >> 7;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

static int64_t fp8_row_bytes(int d_c, int d_r) { return (int64_t)d_c + 4 * (d_c / 128) + 2 * (int64_t)d_r; }

/* Widen cache row `row` (a pool row index) into dst[0 .. d_c+d_r). */
static void widen_row(const orc_problem* P, int64_t row, double* dst) {
  const int D = P->d_c + P->d_r;
  if (P->kv_kind == ORC_KV_F64) {
    const double* src = (const double*)P->kv + row * D;
    for (int d = 0; d < D; ++d) dst[d] = src[d];
  } else if (P->kv_kind == ORC_KV_BF16) {
    const uint16_t* src = (const uint16_t*)P->kv + row * D;
    for (int d = 0; d < D; ++d) dst[d] = bf16_bits_to_f64(src[d]);
  } else {
    const uint8_t* src = (const uint8_t*)P->kv + row * fp8_row_bytes(P->d_c, P->d_r);
    const uint8_t* scales = src + P->d_c;
    const uint8_t* rope = scales + 4 * (P->d_c / 128);
    for (int d = 0; d < P->d_c; ++d) {
      float sc;
      memcpy(&sc, scales + 4 * (d / 128), sizeof sc);
      dst[d] = orc_e4m3_to_f64(src[d]) * (double)sc; /* product of an E4M3 value and a float32 is exact in fp64 */
    }
    for (int r = 0; r < P->d_r; ++r) {
      uint16_t bits;
      memcpy(&bits, rope + 2 * r, sizeof bits);
      dst[P->d_c + r] = bf16_bits_to_f64(bits);
    }
  }
}

static int64_t pool_row(const orc_problem* P, int b, int j) {
  int32_t page = P->block_table[(int64_t)b * P->max_pages_per_seq + j / P->page_size];
  return (int64_t)page * P->page_size + j % P->page_size;
}

/* Number of keys visible to new token t of sequence b. */
int orc_visible_keys(const orc_problem* P, int b, int t) {
  int L = P->seqlens[b];
  int n = P->causal ? L - P->s_q + 1 + t : L;
  if (n < 0) n = 0;
  if (n > L) n = L;
  return n;
}

/*
 * Outputs for query block (b, t) and the n_heads heads listed in `heads`,
 * restricted to keys [k_lo, k_hi) intersected with the visible range
 * (k_hi < 0 means "to the end").  out: [n_heads][d_c], lse: [n_heads].
 * Returns 0, or -1 if a scratch allocation failed.
 */
int orc_decode_rows(const orc_problem* P, int b, int t, int n_heads, const int32_t* heads, int k_lo, int k_hi,
                    double* out, double* lse) {
  const int d_c = P->d_c, d_r = P->d_r, D = d_c + d_r;
  int vis = orc_visible_keys(P, b, t);
  int lo = k_lo < 0 ? 0 : k_lo;
  int hi = (k_hi < 0 || k_hi > vis) ? vis : k_hi;
  int n = hi - lo;
  memset(out, 0, sizeof(double) * (size_t)n_heads * d_c);
  if (n <= 0) {
    for (int i = 0; i < n_heads; ++i) lse[i] = -INFINITY;
    return 0;
  }
  double* w = (double*)malloc(sizeof(double) * (size_t)n_heads * n); /* scores, then weights */
  double* key = (double*)malloc(sizeof(double) * D);
  if (!w || !key) {
    free(w);
    free(key);
    return -1;
  }
  /* scores s_j */
  for (int j = lo; j < hi; ++j) {
    widen_row(P, pool_row(P, b, j), key);
    for (int i = 0; i < n_heads; ++i) {
      int64_t qi = (((int64_t)b * P->s_q + t) * P->num_heads + heads[i]);
      const double* qn = P->q_nope + qi * d_c;
      const double* qr = P->q_rope + qi * d_r;
      double latent = 0.0, rope = 0.0;
      for (int d = 0; d < d_c; ++d) latent += qn[d] * key[d];
      for (int r = 0; r < d_r; ++r) rope += qr[r] * key[d_c + r];
      w[(size_t)i * n + (j - lo)] = P->scale * (latent + rope);
    }
  }
  /* exact softmax and log-sum-exp, per head */
  for (int i = 0; i < n_heads; ++i) {
    double* s = w + (size_t)i * n;
    double m = -INFINITY, l = 0.0;
    for (int j = 0; j < n; ++j)
      if (s[j] > m) m = s[j];
    for (int j = 0; j < n; ++j) l += exp(s[j] - m);
    for (int j = 0; j < n; ++j) s[j] = exp(s[j] - m) / l;
    lse[i] = m + log(l);
  }
  /* out = sum_j p_j c_j */
  for (int j = lo; j < hi; ++j) {
    widen_row(P, pool_row(P, b, j), key);
    for (int i = 0; i < n_heads; ++i) {
      double p = w[(size_t)i * n + (j - lo)];
      double* o = out + (size_t)i * d_c;
      for (int d = 0; d < d_c; ++d) o[d] += p * key[d];
    }
  }
  free(w);
  free(key);
  return 0;
}

/*
 * Merge of partial results computed over disjoint key ranges (the split-KV
 * merge "with LSE", section "Decode attention becomes a compute problem" and
 * the chunked-prefix paragraph of "Which is faster"): with M = max_i lse_i,
 *   lse = M + ln sum_i exp(lse_i - M),  out = sum_i exp(lse_i - lse) * out_i.
 * Parts with lse = -inf (no keys) carry zero weight.  outs: [n_parts][d_c].
 */
void orc_merge(int n_parts, int d_c, const double* outs, const double* lses, double* out, double* lse) {
  double M = -INFINITY;
  for (int i = 0; i < n_parts; ++i)
    if (lses[i] > M) M = lses[i];
  memset(out, 0, sizeof(double) * d_c);
  if (M == -INFINITY) {
    *lse = -INFINITY;
    return;
  }
  double S = 0.0;
  for (int i = 0; i < n_parts; ++i) S += exp(lses[i] - M);
  *lse = M + log(S);
  for (int i = 0; i < n_parts; ++i) {
    double wgt = exp(lses[i] - *lse);
    for (int d = 0; d < d_c; ++d) out[d] += wgt * outs[(size_t)i * d_c + d];
  }
}
