"""GPU parity of the opt-in FP8-QK decode (QK on E4M3 codes, tcgen05 kind::f8f6f4) through the C ABI.

The oracle is fed the identically dequantised cache and the identically quantised query: the
query rows come from the input generator's quantiser (the cache writer's rule, applied to the
absorbed query), the oracle decodes them with ``oracle.fp8_rows_to_f64`` (code x scale, exact)
and the GPU decodes the same bytes.  What is left between the two is the kernel's own
arithmetic: fp32 accumulation of the code products and of the tile-scale products, P in bf16,
the 16-bit block-float score exchange -- as on a bf16 cache -- and V, which PV reads as
code x scale rounded to bf16 (relative error up to 2^-9: up to 0.008 on the |v| ~ 4 of these
caches, where a bf16 cache's V is exact).  QK8_TOL is the bf16-cache bound with that rounding
added to the max-abs term.
"""
import os

import numpy as np
import pytest

import mla_workloads as mw
from gpu_util import compare, params_for

pytestmark = pytest.mark.gpu

THREADS = max(1, min(16, os.cpu_count() or 1))
QK8_TOL = dict(max_abs=2e-2, rel_l2=5e-3, lse=1e-3)


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_absorbed_decode_02_gb300.build import build
    build()


def _oracle_problem(w, q8):
    import oracle
    P = oracle.from_workload(w)
    lat, rope = oracle.fp8_rows_to_f64(q8)
    return oracle.Problem(q_nope=lat, q_rope=rope, kv=P.kv, kv_kind=P.kv_kind, block_table=P.block_table,
                          seqlens=P.seqlens, scale=P.scale, causal=P.causal, page_size=P.page_size)


def run_qk8(w, q8, num_units=0):
    """FP8-QK decode of workload w with query rows q8 (uint8 [B, s_q, H, 656]); float64 numpy results."""
    import torch
    from mla_absorbed_decode_02_gb300 import Decoder, mla_device_error
    from gpu_util import to_device
    _, _, kv, bt, seq = to_device(w)
    q = torch.from_numpy(np.ascontiguousarray(q8)).cuda()
    dec = Decoder(params_for(w, num_units, qk_fp8=1))
    dec.plan(seq)
    out, lse = dec.decode(q, None, kv, bt, seq, w.scale)
    torch.cuda.synchronize()
    err = mla_device_error(clear=True)
    assert err == 0, f"device error word {err}"
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def full_check(w, num_units=0, what=""):
    q8 = mw.quantize_query_fp8(w)
    out, lse = run_qk8(w, q8, num_units)
    ref_out, ref_lse = _oracle_problem(w, q8).full(threads=THREADS)
    return compare(out, lse, ref_out, ref_lse, QK8_TOL, what or w.name, out_bf16=w.out_dtype == "bf16")


# ------------------------------------------------------------------ the query quantiser

@pytest.mark.parametrize("n", [1, 7, 8, 1000])
def test_query_quantizer_matches_the_generator_bytes(n):
    """mla_quantize_q_fp8 writes exactly the rows of the generator's quantiser (the FP8 cache rule)."""
    import torch
    from mla_absorbed_decode_02_gb300 import mla_quantize_q_fp8
    rng = np.random.default_rng(n)
    lat = (rng.standard_normal((n, 512)) * np.exp(rng.uniform(-20, 20, (n, 1)))).astype(np.float32)
    lat[0, 256:384] = 0.0  # an all-zero tile: scale 1, codes 0
    qn_bits = mw.to_bf16_bits(lat)
    qr_bits = mw.to_bf16_bits(rng.standard_normal((n, 64)).astype(np.float32))
    want = mw.quantize_fp8_rows((qn_bits.astype(np.uint32) << 16).view(np.float32), qr_bits)
    qn = torch.from_numpy(qn_bits.view(np.int16)).view(torch.bfloat16).cuda()
    qr = torch.from_numpy(qr_bits.view(np.int16)).view(torch.bfloat16).cuda()
    got = torch.zeros((n, 656), dtype=torch.uint8, device="cuda")
    mla_quantize_q_fp8(qn, qr, got, n)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), want)


# ------------------------------------------------------------------ parity

@pytest.mark.parametrize("num_units", [0, 1, 7])
def test_ragged_lengths_and_splits(num_units):
    w = mw.make_custom([1, 63, 64, 65, 700, 2049, 4100], num_heads=128, kv_dtype="fp8", seed=81)
    full_check(w, num_units=num_units, what=f"fp8 qk ragged U={num_units}")


@pytest.mark.parametrize("s_q,causal", [(2, True), (4, False), (8, True)])
def test_several_new_tokens(s_q, causal):
    w = mw.make_custom([9, 130, 1500], num_heads=128, s_q=s_q, causal=causal, kv_dtype="fp8", seed=82 + s_q)
    full_check(w, num_units=5, what=f"fp8 qk s_q={s_q} causal={causal}")


def test_fewer_heads_and_f32_output():
    w = mw.make_custom([77, 640], num_heads=40, kv_dtype="fp8", out_dtype="f32", seed=86)
    full_check(w, num_units=3, what="fp8 qk H=40 f32")


def test_empty_and_short_sequences():
    """Sequences of no key and sequences shorter than s_q (tokens that see no key: out = 0, lse = -inf)."""
    w = mw.make_custom([0, 100, 0, 1, 3], num_heads=32, s_q=4, kv_dtype="fp8", seed=90)
    q8 = mw.quantize_query_fp8(w)
    out, lse = run_qk8(w, q8, num_units=3)
    ref_out, ref_lse = _oracle_problem(w, q8).full(threads=THREADS)
    compare(out, lse, ref_out, ref_lse, QK8_TOL, "fp8 qk empty and short", out_bf16=True)
    assert np.all(lse[0] == -np.inf) and np.all(out[0] == 0) and np.all(lse[2] == -np.inf)


def test_row_garbage_past_the_end_is_ignored():
    """Rows past the sequence end hold NaN codes, NaN scales and NaN RoPE: QK reads them as codes, the
    expansion must write them as zeros and the softmax must mask their scores."""
    w = mw.make_custom([65, 130, 1, 200], num_heads=64, kv_dtype="fp8", seed=87)
    for b, L in enumerate(w.seqlens):
        page = w.block_table[b, (int(L) - 1) // 64]
        w.kv[page, int(L) % 64 or 64:, :] = 0xFF
    full_check(w, num_units=2, what="fp8 qk NaN past the end")


def test_large_query_and_key_scales():
    """Query tiles and cache tiles spanning many binades: the per-tile scales of both sides enter every
    score, so a scale applied to the wrong tile or the wrong key shows up here."""
    w = mw.make_custom([300, 1030], num_heads=128, kv_dtype="fp8", seed=88)
    rng = np.random.default_rng(88)
    lat = (w.q_nope.astype(np.uint32) << 16).view(np.float32)
    lat = lat * np.exp2(rng.integers(-5, 1, size=lat.shape[:-1] + (4,))).repeat(128, axis=-1).astype(np.float32)
    w.q_nope[:] = mw.to_bf16_bits(lat)
    # every cache row's four tile scales times its own powers of two (the codes stay as they are);
    # the logits stay within the range where the block-float exchange meets the LSE bound
    sc = np.ascontiguousarray(w.kv[:, :, 512:528]).view(np.float32)
    sc *= np.exp2(rng.integers(-4, 2, size=sc.shape)).astype(np.float32)
    w.kv[:, :, 512:528] = sc.view(np.uint8)
    full_check(w, num_units=4, what="fp8 qk scaled tiles")


def test_full_size_fp8_mtp2_sampled():
    """The fp8_mtp2 workload (B = 128, s_q = 2, lengths 2,433..16,334) in the benchmark's launch
    configuration; one head from each 32-row group of every (sequence, token), against the oracle."""
    w = mw.make_workload(4)
    q8 = mw.quantize_query_fp8(w)
    out, lse = run_qk8(w, q8)
    P = _oracle_problem(w, q8)
    rng = np.random.default_rng(1404)
    items = [(b, t, [int(g + rng.integers(0, 32)) for g in range(0, w.num_heads, 32)])
             for b in range(w.batch) for t in range(w.s_q)]
    import oracle
    res = {}

    def work(chunk):
        for b, t, heads in chunk:
            res[(b, t)] = (np.asarray(heads),) + P.rows(b, t, heads=np.asarray(heads, np.int32))

    oracle.run_threads(work, items, THREADS)
    got_o = np.concatenate([out[b, t, h] for (b, t), (h, _, _) in res.items()])
    got_l = np.concatenate([lse[b, t, h] for (b, t), (h, _, _) in res.items()])
    ref_o = np.concatenate([o for (h, o, _) in res.values()])
    ref_l = np.concatenate([l for (h, _, l) in res.values()])
    compare(got_o, got_l, ref_o, ref_l, QK8_TOL, "fp8_mtp2 qk sampled", out_bf16=True, raw=True)


def test_allocation_free_entry_point_gives_the_same_bits():
    """mla_decode_noalloc with qk_fp8 runs the same kernels on the same plan as the buffered call."""
    import torch
    from mla_absorbed_decode_02_gb300 import mla_decode_noalloc, mla_device_error
    from gpu_util import to_device
    w = mw.make_custom([33, 700, 1400], num_heads=128, s_q=2, kv_dtype="fp8", seed=89)
    q8 = mw.quantize_query_fp8(w)
    ref_out, ref_lse = run_qk8(w, q8, num_units=76)
    _, _, kv, bt, seq = to_device(w)
    q = torch.from_numpy(np.ascontiguousarray(q8)).cuda()
    out = torch.empty((w.batch, w.s_q, w.num_heads, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.batch, w.s_q, w.num_heads), dtype=torch.float32, device="cuda")
    mla_decode_noalloc(params_for(w, num_units=76, qk_fp8=1), q, None, kv, bt, seq, w.scale, out, lse)
    torch.cuda.synchronize()
    assert mla_device_error(clear=True) == 0
    assert np.array_equal(out.float().cpu().numpy().astype(np.float64), ref_out)
    assert np.array_equal(lse.cpu().numpy().astype(np.float64), ref_lse)
