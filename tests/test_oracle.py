"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test is chosen so that a plausible slip in the oracle (a dropped RoPE
term, a wrong sign, a transposed operand, an off-by-one in the causal range,
a wrong page index, a wrong merge weight) fails at least one of them:

* absorb == expand ("MLA inference: two computation paths and FlashMLA",
  section "Two equivalent paths": the two paths give the same output; also
  "FlashMLA: Fast Hopper Decoding for Latent Attention Guide", section
  "Implementation: Simulating FlashMLA Decoding in Python", W_UK/W_UV shaped
  [H, 128, 512]).  The expanded side is textbook multi-head attention in
  numpy fp64, written here independently of the oracle.
* split-merge == unsplit (the LSE merge of split-KV / chunked prefixes).
* weights sum to one, brute force against a dense numpy formula, page
  permutation invariance, and closed forms (uniform weights, one key,
  a dominant key, duplicated keys).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import KV_BF16, KV_F64, KV_FP8, Problem


def paged(keys_per_seq, page_size, rng, extra_pages=3):
    """Scatter dense per-sequence key arrays [L_b, D] into a shuffled page pool."""
    D = keys_per_seq[0].shape[1]
    need = [(k.shape[0] + page_size - 1) // page_size for k in keys_per_seq]
    pool_pages = sum(need) + extra_pages
    perm = rng.permutation(pool_pages)
    pool = rng.standard_normal((pool_pages, page_size, D))  # unused slots hold junk that must never be read
    bt = np.full((len(keys_per_seq), max(need)), -1, np.int32)
    o = 0
    for b, k in enumerate(keys_per_seq):
        for i in range(need[b]):
            p = perm[o]
            o += 1
            bt[b, i] = p
            rows = k[i * page_size:(i + 1) * page_size]
            pool[p, :rows.shape[0]] = rows
    return pool, bt


def dense_reference(qn, qr, keys, scale, s_q, causal):
    """softmax(scale * [qn|qr] K^T) C for one sequence; keys [L, d_c+d_r] dense fp64."""
    d_c = qn.shape[-1]
    L = keys.shape[0]
    q = np.concatenate([qn, qr], axis=-1)            # [s_q, H, D]
    s = scale * np.einsum("thd,jd->thj", q, keys)    # [s_q, H, L]
    if causal:
        for t in range(s_q):
            s[t, :, max(0, L - s_q + 1 + t):] = -np.inf
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    p = e / e.sum(axis=-1, keepdims=True)
    out = np.einsum("thj,jd->thd", p, keys[:, :d_c])
    lse = (m[..., 0] + np.log(e.sum(axis=-1)))
    return out, lse


# ---------------------------------------------------------------- absorb == expand

def rope_rotate(x, pos):
    """Rotate adjacent pairs of the last axis by angle pos / 10000^(2i/d) (decoupled RoPE)."""
    d = x.shape[-1]
    ang = pos[:, None] / 10000 ** (np.arange(0, d, 2) / d)
    x1, x2 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x1 * np.cos(ang) - x2 * np.sin(ang)
    out[..., 1::2] = x1 * np.sin(ang) + x2 * np.cos(ang)
    return out


@pytest.mark.parametrize("H,NOPE,ROPE,DV,DC,L,s_q,page", [
    (4, 8, 4, 8, 16, 6, 6, 4),        # the page's toy shape: all 6 tokens are queries, causal
    (128, 128, 64, 128, 512, 150, 2, 64),  # DeepSeek-V3 shape, two new tokens after 148 cached
    (8, 128, 64, 128, 512, 70, 1, 64),     # single-token decode
])
def test_absorb_equals_expand(H, NOPE, ROPE, DV, DC, L, s_q, page):
    rng = np.random.default_rng(1234 + H + L)
    D = 64
    h = rng.standard_normal((L, D))
    W_q = rng.standard_normal((D, H * (NOPE + ROPE))) / 8
    W_dkv = rng.standard_normal((D, DC)) / 8
    W_kr = rng.standard_normal((D, ROPE)) / 8
    W_uk = rng.standard_normal((H, DC, NOPE)) / 4   # latent -> per-head non-positional key
    W_uv = rng.standard_normal((H, DC, DV)) / 4     # latent -> per-head value
    pos = np.arange(L, dtype=np.float64)
    c = h @ W_dkv                                   # [L, DC] cached latent
    k_r = rope_rotate(h @ W_kr, pos)                # [L, ROPE] cached shared RoPE key
    q = (h @ W_q).reshape(L, H, NOPE + ROPE)
    q_n, q_r = q[..., :NOPE], rope_rotate(q[..., NOPE:].transpose(1, 0, 2), pos).transpose(1, 0, 2)
    scale = 1 / math.sqrt(NOPE + ROPE)
    new = np.arange(L - s_q, L)                     # positions of the new (query) tokens

    # path one: expand K and V per head, ordinary causal multi-head attention
    out1 = np.empty((s_q, H, DV))
    for hh in range(H):
        k = np.concatenate([c @ W_uk[hh], k_r], axis=1)     # [L, NOPE+ROPE]
        v = c @ W_uv[hh]                                    # [L, DV]
        qq = np.concatenate([q_n[new, hh], q_r[new, hh]], axis=1)
        s = scale * qq @ k.T
        s[np.arange(L)[None, :] > new[:, None]] = -np.inf
        p = np.exp(s - s.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        out1[:, hh] = p @ v

    # path two: absorb W_uk into the query, attend over the paged latent cache, apply W_uv last
    q_lat = oracle.absorb_query(q_n[new], W_uk.transpose(0, 2, 1))   # [s_q, H, DC]; W_uk[h]^T is [NOPE, DC]
    pool, bt = paged([np.concatenate([c, k_r], axis=1)], page, rng)
    P = Problem(q_nope=q_lat[None], q_rope=q_r[new][None], kv=pool, kv_kind=KV_F64, block_table=bt,
                seqlens=np.array([L], np.int32), scale=scale, causal=True, page_size=page)
    out_lat, _ = P.full()
    out2 = oracle.project_output(out_lat[0], W_uv)
    np.testing.assert_allclose(out2, out1, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- brute force vs dense formula

@pytest.mark.parametrize("seed", range(6))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 4))
    H = int(rng.integers(1, 5))
    s_q = int(rng.integers(1, 9))
    causal = bool(rng.integers(0, 2))
    d_c, d_r, page = 32, 8, 16
    Ls = rng.integers(s_q, 131, size=B)
    keys = [rng.standard_normal((int(L), d_c + d_r)) for L in Ls]
    pool, bt = paged(keys, page, rng)
    qn = rng.standard_normal((B, s_q, H, d_c))
    qr = rng.standard_normal((B, s_q, H, d_r))
    scale = 1 / math.sqrt(192)
    P = Problem(qn, qr, pool, KV_F64, bt, Ls.astype(np.int32), scale, causal=causal, page_size=page)
    out, lse = P.full()
    for b in range(B):
        ro, rl = dense_reference(qn[b], qr[b], keys[b], scale, s_q, causal)
        np.testing.assert_allclose(out[b], ro, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[b], rl, rtol=1e-13, atol=1e-13)


def test_visible_keys_causal_and_not():
    rng = np.random.default_rng(5)
    keys = [rng.standard_normal((10, 12))]
    pool, bt = paged(keys, 4, rng)
    qn, qr = rng.standard_normal((1, 3, 1, 8)), rng.standard_normal((1, 3, 1, 4))
    Pc = Problem(qn, qr, pool, KV_F64, bt, np.array([10], np.int32), 0.3, causal=True, page_size=4)
    Pn = Problem(qn, qr, pool, KV_F64, bt, np.array([10], np.int32), 0.3, causal=False, page_size=4)
    assert [Pc.visible_keys(0, t) for t in range(3)] == [8, 9, 10]
    assert [Pn.visible_keys(0, t) for t in range(3)] == [10, 10, 10]


# ---------------------------------------------------------------- LSE merge

@pytest.mark.parametrize("seed", range(5))
def test_split_merge_equals_unsplit(seed):
    rng = np.random.default_rng(100 + seed)
    d_c, d_r, page, H = 64, 16, 8, 3
    L = int(rng.integers(1, 300))
    keys = [rng.standard_normal((L, d_c + d_r)) * 2]
    pool, bt = paged(keys, page, rng)
    qn, qr = rng.standard_normal((1, 1, H, d_c)), rng.standard_normal((1, 1, H, d_r))
    P = Problem(qn, qr, pool, KV_F64, bt, np.array([L], np.int32), 0.2, page_size=page)
    ref_out, ref_lse = P.rows(0, 0)
    n_parts = int(rng.integers(1, 8))
    cuts = np.sort(rng.integers(0, L + 1, size=n_parts - 1))
    bounds = [0, *cuts.tolist(), L]                   # may contain empty ranges
    for h in range(H):
        outs, lses = [], []
        for lo, hi in zip(bounds[:-1], bounds[1:]):
            o, l = P.rows(0, 0, heads=[h], k_lo=lo, k_hi=hi)
            outs.append(o[0])
            lses.append(l[0])
        mo, ml = oracle.merge(np.array(outs), np.array(lses))
        np.testing.assert_allclose(mo, ref_out[h], rtol=1e-12, atol=1e-13)
        assert abs(ml - ref_lse[h]) < 1e-12


def test_merge_all_empty_parts():
    out, lse = oracle.merge(np.zeros((3, 5)), np.full(3, -np.inf))
    assert lse == -np.inf and np.all(out == 0)


# ---------------------------------------------------------------- invariants and closed forms

def _simple_problem(rng, L, H=2, d_c=32, d_r=8, page=8, keys=None, qn=None, qr=None, scale=0.25):
    keys = [rng.standard_normal((L, d_c + d_r))] if keys is None else keys
    pool, bt = paged(keys, page, rng)
    qn = rng.standard_normal((1, 1, H, d_c)) if qn is None else qn
    qr = rng.standard_normal((1, 1, H, d_r)) if qr is None else qr
    return Problem(qn, qr, pool, KV_F64, bt, np.array([L], np.int32), scale, page_size=page), keys[0]


def test_weights_sum_to_one():
    rng = np.random.default_rng(7)
    L, d_c, d_r = 97, 32, 8
    keys = rng.standard_normal((L, d_c + d_r)) * 3
    a = rng.standard_normal(d_c)
    keys[:, :d_c] = a                                  # every value row equals a  =>  out == sum_j p_j * a == a
    P, _ = _simple_problem(rng, L, keys=[keys])
    out, _ = P.rows(0, 0)
    np.testing.assert_allclose(out, np.broadcast_to(a, out.shape), rtol=1e-14, atol=1e-14)


def test_zero_query_gives_uniform_weights():
    rng = np.random.default_rng(8)
    L = 130
    P, keys = _simple_problem(rng, L, qn=np.zeros((1, 1, 2, 32)), qr=np.zeros((1, 1, 2, 8)))
    out, lse = P.rows(0, 0)
    np.testing.assert_allclose(out, np.broadcast_to(keys[:, :32].mean(0), out.shape), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, math.log(L), rtol=1e-15)


def test_single_key():
    rng = np.random.default_rng(9)
    P, keys = _simple_problem(rng, 1)
    out, lse = P.rows(0, 0)
    q = np.concatenate([P.q_nope[0, 0], P.q_rope[0, 0]], axis=1)
    np.testing.assert_array_equal(out, np.broadcast_to(keys[0, :32], out.shape))
    np.testing.assert_allclose(lse, 0.25 * q @ keys[0], rtol=1e-14)


def test_dominant_key():
    rng = np.random.default_rng(10)
    L, j0 = 50, 17
    qn = rng.standard_normal((1, 1, 1, 32))
    keys = rng.standard_normal((L, 40))
    keys[j0, :32] = 40 * qn[0, 0, 0] / np.linalg.norm(qn)  # score of key j0 exceeds the rest by > 50
    P, _ = _simple_problem(rng, L, H=1, keys=[keys], qn=qn, qr=np.zeros((1, 1, 1, 8)))
    out, _ = P.rows(0, 0)
    np.testing.assert_allclose(out[0], keys[j0, :32], rtol=1e-12, atol=1e-12)


def test_duplicated_keys_add_ln2():
    rng = np.random.default_rng(11)
    L = 40
    keys = rng.standard_normal((L, 40))
    P1, _ = _simple_problem(rng, L, keys=[keys])
    P2, _ = _simple_problem(rng, 2 * L, keys=[np.concatenate([keys, keys])], qn=P1.q_nope, qr=P1.q_rope)
    o1, l1 = P1.rows(0, 0)
    o2, l2 = P2.rows(0, 0)
    np.testing.assert_allclose(o2, o1, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(l2, l1 + math.log(2), rtol=1e-14)


def test_empty_sequence():
    rng = np.random.default_rng(12)
    pool = rng.standard_normal((2, 8, 40))
    P = Problem(np.ones((1, 1, 2, 32)), np.ones((1, 1, 2, 8)), pool, KV_F64, np.array([[0]], np.int32),
                np.array([0], np.int32), 0.3, page_size=8)
    out, lse = P.rows(0, 0)
    assert np.all(out == 0) and np.all(lse == -np.inf)


def test_page_permutation_invariance():
    rng = np.random.default_rng(13)
    B, H, d_c, d_r, page = 3, 2, 32, 8, 8
    Ls = np.array([5, 64, 41], np.int32)
    keys = [rng.standard_normal((int(L), d_c + d_r)) for L in Ls]
    pool, bt = paged(keys, page, rng)
    qn, qr = rng.standard_normal((B, 1, H, d_c)), rng.standard_normal((B, 1, H, d_r))
    o1, l1 = Problem(qn, qr, pool, KV_F64, bt, Ls, 0.3, page_size=page).full()
    perm = rng.permutation(pool.shape[0])            # new physical position of every page
    pool2 = np.empty_like(pool)
    pool2[perm] = pool
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    o2, l2 = Problem(qn, qr, pool2, KV_F64, bt2, Ls, 0.3, page_size=page).full()
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ---------------------------------------------------------------- cache formats (exact widening)

def test_e4m3_all_codes_against_torch_and_definition():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_f64(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got)) and nan.sum() == 2          # only S.1111.111
    assert np.array_equal(got[~nan], ref[~nan])
    assert oracle.e4m3_to_f64(0x7E) == 448.0 and oracle.e4m3_to_f64(0xFE) == -448.0   # largest finite magnitude
    assert oracle.e4m3_to_f64(0x01) == 2.0 ** -9 and oracle.e4m3_to_f64(0x08) == 2.0 ** -6


def _bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_cache_matches_f64_cache():
    rng = np.random.default_rng(14)
    L, page = 77, 64
    pool_bits = _bf16_bits(rng.standard_normal((3, page, 576)))
    pool_f64 = torch.from_numpy(pool_bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    bt = np.array([[2, 0]], np.int32)
    qn, qr = rng.standard_normal((1, 1, 4, 512)), rng.standard_normal((1, 1, 4, 64))
    a = Problem(qn, qr, pool_bits, KV_BF16, bt, np.array([L], np.int32), 1 / math.sqrt(192)).full()
    b = Problem(qn, qr, pool_f64, KV_F64, bt, np.array([L], np.int32), 1 / math.sqrt(192)).full()
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_fp8_cache_matches_f64_cache():
    import mla_workloads as mw
    rng = np.random.default_rng(15)
    n = 2 * 64
    x = rng.standard_normal((n, 576)).astype(np.float32)
    rows = mw.quantize_fp8_rows(x[:, :512], mw.to_bf16_bits(x[:, 512:]))
    # dequantise with torch (library decode of the codes, times the stored float32 scale)
    codes = torch.from_numpy(rows[:, :512].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    scales = rows[:, 512:528].copy().view(np.float32).astype(np.float64)
    latent = codes * np.repeat(scales, 128, axis=1)
    rope = torch.from_numpy(rows[:, 528:].copy().view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    pool_f64 = np.concatenate([latent, rope], axis=1).reshape(2, 64, 576)
    # the quantiser really used its scale: each tile's largest magnitude maps to the top of the E4M3 range
    assert np.allclose(np.abs(codes.reshape(n, 4, 128)).max(-1), 448.0)
    bt = np.array([[1, 0]], np.int32)
    qn, qr = rng.standard_normal((1, 2, 3, 512)), rng.standard_normal((1, 2, 3, 64))
    L = np.array([100], np.int32)
    a = Problem(qn, qr, rows.reshape(2, 64, 656), KV_FP8, bt, L, 1 / math.sqrt(192)).full()
    b = Problem(qn, qr, pool_f64, KV_F64, bt, L, 1 / math.sqrt(192)).full()
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_fp8_rows_to_f64_matches_the_oracles_cache_decoding():
    """oracle.fp8_rows_to_f64 (the FP8-QK query's decoding) against torch's E4M3 decode times the stored
    scale, and against the C oracle's own decoding of the same rows as an FP8 cache: an FP8-cache
    problem and a float64-cache problem built from fp8_rows_to_f64 of its pool give equal results."""
    import mla_workloads as mw
    rng = np.random.default_rng(21)
    n = 2 * 64
    x = (rng.standard_normal((n, 576)) * np.exp(rng.uniform(-6, 6, (n, 1)))).astype(np.float32)
    x[5, 128:256] = 0.0  # an all-zero tile (scale 1)
    rows = mw.quantize_fp8_rows(x[:, :512], mw.to_bf16_bits(x[:, 512:]))
    lat, rope = oracle.fp8_rows_to_f64(rows.reshape(2, 64, 656))
    codes = torch.from_numpy(rows[:, :512].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    scales = rows[:, 512:528].copy().view(np.float32).astype(np.float64)
    assert np.array_equal(lat.reshape(n, 512), codes * np.repeat(scales, 128, axis=1))
    rope_bits = mw.to_bf16_bits(x[:, 512:])
    assert np.array_equal(rope.reshape(n, 64),
                          torch.from_numpy(rope_bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy())
    assert np.all(lat.reshape(n, 512)[5, 128:256] == 0.0)
    pool_f64 = np.concatenate([lat, rope], axis=2)
    bt = np.array([[1, 0]], np.int32)
    qn, qr = rng.standard_normal((1, 1, 2, 512)), rng.standard_normal((1, 1, 2, 64))
    L = np.array([113], np.int32)
    a = Problem(qn, qr, rows.reshape(2, 64, 656), KV_FP8, bt, L, 1 / math.sqrt(192)).full()
    b = Problem(qn, qr, pool_f64, KV_F64, bt, L, 1 / math.sqrt(192)).full()
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_threads_match_single_thread():
    rng = np.random.default_rng(16)
    Ls = np.array([33, 64, 130, 1], np.int32)
    keys = [rng.standard_normal((int(L), 40)) for L in Ls]
    pool, bt = paged(keys, 8, rng)
    P = Problem(rng.standard_normal((4, 2, 3, 32)), rng.standard_normal((4, 2, 3, 8)), pool, KV_F64, bt, Ls, 0.3,
                page_size=8)
    a = P.full(threads=1)
    b = P.full(threads=3)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---------------------------------------------------------------- the Python marshalling helpers

def test_bf16_widening_all_patterns():
    """oracle.bf16_bits_to_f64 on every one of the 65,536 bf16 bit patterns, against torch's own
    bf16 -> float64 conversion and against the format's definition (sign, 8-bit exponent with bias
    127, 7-bit fraction; exponent 0 = subnormal, 255 = inf / NaN)."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):          # numpy flags the signalling-NaN patterns as it widens them
        got = oracle.bf16_bits_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2 * 127                                   # exponent 255, fraction != 0, both signs
    assert np.array_equal(got[~nan].view(np.uint64), ref[~nan].view(np.uint64))   # bit for bit, -0.0 included
    sign = np.where(bits >> 15, -1.0, 1.0)
    e = ((bits >> 7) & 0xFF).astype(np.int64)
    f = (bits & 0x7F).astype(np.float64)
    defn = np.where(e == 0, sign * f * 2.0 ** -133, sign * (1.0 + f / 128.0) * np.ldexp(1.0, e - 127))
    fin = e < 255
    assert np.array_equal(got[fin], defn[fin])
    assert np.all(np.isinf(got[(e == 255) & (f == 0)]))


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_from_workload_matches_a_problem_built_by_hand(kv_dtype):
    """oracle.from_workload: which array is the absorbed query and which the RoPE query, the cache
    kind, the causal flag, the scale and the page size of a workload all reach the oracle.  The
    hand-built problem widens the queries with torch and, for the FP8 cache, dequantises the codes
    with torch's E4M3 type times the stored float32 tile scale; the results must agree bit for bit.
    Two new tokens, not causal: a dropped causal flag would change the first token's keys."""
    import mla_workloads as mw
    w = mw.make_custom([70, 129, 3], num_heads=4, s_q=2, causal=False, kv_dtype=kv_dtype, seed=61)
    P = oracle.from_workload(w)
    widen = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert P.q_nope.shape == (3, 2, 4, 512) and P.q_rope.shape == (3, 2, 4, 64)
    assert np.array_equal(P.q_nope, widen(w.q_nope)) and np.array_equal(P.q_rope, widen(w.q_rope))
    assert P.causal is False and P.scale == 1 / math.sqrt(192) and P.page_size == 64
    assert np.array_equal(P.block_table, w.block_table) and np.array_equal(P.seqlens, w.seqlens)
    if kv_dtype == "bf16":
        assert P.kv_kind == KV_BF16
        pool = widen(w.kv)
    else:
        assert P.kv_kind == KV_FP8
        rows = w.kv.reshape(-1, mw.FP8_ROW_BYTES)
        codes = torch.from_numpy(rows[:, :512].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        scales = rows[:, 512:528].copy().view(np.float32).astype(np.float64)
        rope = widen(rows[:, 528:].copy().view(np.uint16))
        pool = np.concatenate([codes * np.repeat(scales, 128, axis=1), rope], axis=1).reshape(w.kv.shape[0], 64, 576)
    hand = Problem(widen(w.q_nope), widen(w.q_rope), pool, KV_F64, w.block_table, w.seqlens, 1 / math.sqrt(192),
                   causal=False, page_size=64)
    a, b = P.full(), hand.full()
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # and the flag matters here: the causal reading of the same inputs differs
    c = Problem(widen(w.q_nope), widen(w.q_rope), pool, KV_F64, w.block_table, w.seqlens, 1 / math.sqrt(192),
                causal=True, page_size=64).full()
    assert not np.array_equal(a[1][:, 0], c[1][:, 0])


def test_head_projections_by_loops():
    """oracle.absorb_query / project_output against sums written out element by element."""
    rng = np.random.default_rng(77)
    T, H, K, N = 3, 2, 5, 4
    a = rng.standard_normal((T, H, K))
    w = rng.standard_normal((H, K, N))
    want = np.zeros((T, H, N))
    for t in range(T):
        for h in range(H):
            for n in range(N):
                acc = 0.0
                for k in range(K):
                    acc += a[t, h, k] * w[h, k, n]
                want[t, h, n] = acc
    np.testing.assert_allclose(oracle.absorb_query(a, w), want, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(oracle.project_output(a, w), want, rtol=1e-14, atol=1e-14)
    # head h uses only W[h]: swapping the heads' weights swaps the heads' outputs
    np.testing.assert_allclose(oracle.absorb_query(a, w[::-1])[:, 0], oracle.absorb_query(a[:, ::-1], w)[:, 1])


# ---------------------------------------------------------------- the expand path (extend)

def test_round_bf16_matches_torch_cast():
    """oracle.round_bf16 against torch's float32 -> bf16 cast (round to nearest, ties to even) on
    float32 inputs, where a single rounding is exact: random values, exact ties and one-ulp
    neighbours of ties."""
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(20000) * 2.0 ** rng.integers(-20, 20, 20000)).astype(np.float32)
    bits = x.view(np.uint32)
    ties = ((bits & np.uint32(0xFFFF0000)) | np.uint32(0x8000)).view(np.float32)
    near = np.concatenate([(ties.view(np.uint32) + np.uint32(1)).view(np.float32),
                           (ties.view(np.uint32) - np.uint32(1)).view(np.float32)])
    for v in (x, ties, near, np.float32([0.0, -0.0, 1.0, -3.5])):
        want = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
        np.testing.assert_array_equal(oracle.round_bf16(v.astype(np.float64)), want)


def test_expand_kv_by_loops():
    """oracle.expand_kv against sums written out element by element: k^N_j[n] = sum_c W_UK[h][n][c] c_j[c],
    v_j[n] = sum_c c_j[c] W_UV[h][c][n]."""
    rng = np.random.default_rng(8)
    H, L, DC, NOPE, DV = 2, 3, 5, 4, 3
    c = rng.standard_normal((L, DC))
    w_uk = rng.standard_normal((H, NOPE, DC))
    w_uv = rng.standard_normal((H, DC, DV))
    kn, v = oracle.expand_kv(c, w_uk, w_uv)
    for h in range(H):
        for j in range(L):
            for n in range(NOPE):
                assert abs(kn[h, j, n] - sum(w_uk[h, n, k] * c[j, k] for k in range(DC))) < 1e-13
            for n in range(DV):
                assert abs(v[h, j, n] - sum(c[j, k] * w_uv[h, k, n] for k in range(DC))) < 1e-13


def _bf16_pool(rows_per_seq, rng, extra_pages=2):
    """bf16 bit patterns of per-sequence rows [L_b, 576] scattered over a shuffled page pool."""
    pool, bt = paged(rows_per_seq, 64, rng, extra_pages)
    bits = torch.from_numpy(pool.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return bits, bt


@pytest.mark.parametrize("lengths,s_q", [([70, 150], 1), ([70, 150], 3), ([9, 200], 8), ([40, 40], 40)])
def test_extend_expanded_equals_absorbed_oracle(lengths, s_q):
    """Path one (oracle.extend_expanded, numpy) against path two computed by the C oracle on the
    absorbed queries, then projected by W_UV ("Two equivalent paths": the two paths give the same
    output; the lse is the same quantity on both).  Includes a pure prefill (s_q = L)."""
    rng = np.random.default_rng(sum(lengths) + s_q)
    B, H, NOPE, DC, DR, DV = len(lengths), 4, 128, 512, 64, 128
    rows = [rng.standard_normal((L, DC + DR)) for L in lengths]
    kv, bt = _bf16_pool(rows, rng)
    q_n = rng.standard_normal((B, s_q, H, NOPE))
    q_r = rng.standard_normal((B, s_q, H, DR))
    w_uk = rng.standard_normal((H, NOPE, DC)) / math.sqrt(DC)
    w_uv = rng.standard_normal((H, DC, DV)) / math.sqrt(DC)
    seqlens = np.array(lengths, np.int32)
    scale = 1 / math.sqrt(NOPE + DR)
    out1, lse1 = oracle.extend_expanded(q_n, q_r, kv, bt, seqlens, w_uk, w_uv, scale)
    P = Problem(q_nope=oracle.absorb_query(q_n, w_uk), q_rope=q_r, kv=kv, kv_kind=KV_BF16, block_table=bt,
                seqlens=seqlens, scale=scale, causal=True)
    out_lat, lse2 = P.full()
    np.testing.assert_allclose(out1, oracle.project_output(out_lat, w_uv), rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(lse1, lse2, rtol=0, atol=1e-10)


def test_extend_expanded_closed_forms():
    """One cached row and one query: out = v_0 and lse = the score.  Two equal rows: the same
    output and lse + ln 2."""
    rng = np.random.default_rng(21)
    H, NOPE, DC, DR, DV = 3, 128, 512, 64, 128
    row = rng.standard_normal((1, DC + DR))
    w_uk = rng.standard_normal((H, NOPE, DC)) / 16
    w_uv = rng.standard_normal((H, DC, DV)) / 16
    q_n = rng.standard_normal((1, 1, H, NOPE))
    q_r = rng.standard_normal((1, 1, H, DR))
    kv, bt = _bf16_pool([row], rng)
    c = oracle.bf16_bits_to_f64(kv[bt[0, 0], 0])
    kn, v = oracle.expand_kv(c[None, :DC], w_uk, w_uv)
    out, lse = oracle.extend_expanded(q_n, q_r, kv, bt, np.array([1], np.int32), w_uk, w_uv, 0.1)
    np.testing.assert_allclose(out[0, 0], v[:, 0], rtol=1e-12)
    want_s = 0.1 * (np.einsum("hn,hn->h", q_n[0, 0], kn[:, 0]) + q_r[0, 0] @ c[DC:])
    np.testing.assert_allclose(lse[0, 0], want_s, rtol=1e-12)
    kv2, bt2 = _bf16_pool([np.concatenate([row, row])], rng)
    out2, lse2 = oracle.extend_expanded(q_n, q_r, kv2, bt2, np.array([2], np.int32), w_uk, w_uv, 0.1)
    np.testing.assert_allclose(out2, out, rtol=1e-12)
    np.testing.assert_allclose(lse2, lse + math.log(2), rtol=1e-12)
