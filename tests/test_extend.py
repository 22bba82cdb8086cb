"""Extend by the expand path, chunk by chunk, through the C ABI, against the oracle.

mla_expand_kv produces path one's per-head keys and values of one chunk of cached rows and
mla_extend runs the whole chunked extend ("MLA inference: two computation paths and
FlashMLA", sections "Two equivalent paths" (path one) and "Which is faster: count new tokens
and cached tokens": long prefixes are expanded a chunk at a time and the chunks' results
merged by their log-sum-exp).  The oracle is oracle.extend_expanded (float64, unchunked), once
with the expanded keys and values held in bf16 as the kernels hold them (tight bound) and once
exact (bound widened by that rounding)."""
import numpy as np
import pytest

import mla_workloads as mw
from gpu_util import BF16_TOL, compare, half_ulp_bf16

pytestmark = pytest.mark.gpu

# Against the exact float64 expansion, the bf16 keys (relative error <= 2^-9 per element)
# move each score by about 2^-9 * |q^N| |k^N| / sqrt(128) * scale ~ 1e-3 nats at unit-variance
# inputs, which moves the lse by as much and the output by that times |v|.
EXACT_KV_TOL = dict(max_abs=2e-2, rel_l2=1e-2, lse=5e-3)


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_absorbed_decode_02_gb300.build import build
    build()


def _dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _params(x, chunk, max_seqlen=None):
    from mla_absorbed_decode_02_gb300 import MlaExtendParams
    c = x.cache
    return MlaExtendParams.make(c.batch, x.s_q, c.num_heads, c.kv.shape[0], c.block_table.shape[1],
                                int(max_seqlen or c.seqlens.max()), chunk)


def _widen(bits):
    import oracle
    return oracle.bf16_bits_to_f64(bits)


def run_extend(x, chunk, max_seqlen=None):
    import torch
    from mla_absorbed_decode_02_gb300 import mla_device_error, mla_extend, mla_extend_workspace_size
    c = x.cache
    p = _params(x, chunk, max_seqlen)
    ws = torch.empty(mla_extend_workspace_size(p), dtype=torch.uint8, device="cuda")
    out = torch.empty((c.batch, x.s_q, c.num_heads, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((c.batch, x.s_q, c.num_heads), dtype=torch.float32, device="cuda")
    kv = _dev(c.kv)
    bt = torch.from_numpy(c.block_table).cuda()
    seq = torch.from_numpy(c.seqlens).cuda()
    mla_extend(p, _dev(x.q_nope), _dev(x.q_rope), kv, bt, seq, _dev(x.w_uk), _dev(x.w_uv), x.scale, out, lse, ws)
    torch.cuda.synchronize()
    assert mla_device_error(clear=True) == 0
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def oracle_extend(x, round_kv):
    import oracle
    c = x.cache
    return oracle.extend_expanded(_widen(x.q_nope), _widen(x.q_rope), c.kv, c.block_table, c.seqlens,
                                  _widen(x.w_uk), _widen(x.w_uv), x.scale, round_kv=round_kv)


@pytest.mark.parametrize("lengths,H,chunk,starts", [
    ([150, 300], 8, 256, [0, 256]),          # ragged ends inside a 128-row tile, a tile past the end
    ([1000, 64, 777], 16, 512, [0, 512]),    # a sequence shorter than one tile; tiles past its end
    ([3000, 2500], 128, 1024, [0, 2048]),    # 128 heads: several heads per CTA
])
def test_expand_kv_matches_oracle(lengths, H, chunk, starts):
    import torch
    import oracle
    from mla_absorbed_decode_02_gb300 import mla_device_error, mla_expand_kv
    x = mw.make_extend(lengths, s_q=1, num_heads=H, seed=len(lengths) + H)
    c = x.cache
    p = _params(x, chunk)
    kv, bt, seq = _dev(c.kv), torch.from_numpy(c.block_table).cuda(), torch.from_numpy(c.seqlens).cuda()
    w_uk64, w_uv64 = _widen(x.w_uk), _widen(x.w_uv)
    heads = np.unique(np.linspace(0, H - 1, 8).astype(int))
    for cs in starts:
        kn = torch.full((c.batch, H, chunk, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        v = torch.full_like(kn, float("nan"))
        mla_expand_kv(p, kv, bt, seq, _dev(x.w_uk), _dev(x.w_uv), cs, kn, v)
        torch.cuda.synchronize()
        assert mla_device_error(clear=True) == 0
        kn_g = kn.float().cpu().numpy().astype(np.float64)
        v_g = v.float().cpu().numpy().astype(np.float64)
        for b in range(c.batch):
            L = int(c.seqlens[b])
            if cs >= L:
                continue
            hi = min(L, cs + chunk)
            rows = oracle.cache_rows(c.kv, c.block_table, b, L)[cs:hi, :512]
            want_k, want_v = oracle.expand_kv(rows, w_uk64[heads], w_uv64[heads])
            for got, want, name in ((kn_g[b, heads, :hi - cs], want_k, "k^N"), (v_g[b, heads, :hi - cs], want_v, "v")):
                excess = float((np.abs(got - want) - half_ulp_bf16(want)).max())
                print(f"[parity] expand {name} b={b} chunk@{cs}: max excess over bf16 rounding {excess:.3g}")
                assert excess <= 2.0 ** -12 * float(np.abs(want).max()), (name, b, cs, excess)
            # rows past the end inside the last written 128-row tile are zeros
            tail_end = min(cs + chunk, (L + 127) // 128 * 128)
            if tail_end > hi:
                assert np.all(kn_g[b, :, hi - cs:tail_end - cs] == 0) and np.all(v_g[b, :, hi - cs:tail_end - cs] == 0)


@pytest.mark.parametrize("lengths,s_q,H,chunk", [
    ([300, 517], 1, 16, 128),       # one new token (the decode shape), five chunks, ragged tails
    ([700, 129], 7, 16, 256),       # causal block of 7 inside the last chunk
    ([200, 450], 200, 16, 128),     # s_q = L for the first sequence: a pure prefill; 2 query tiles
    ([1300], 130, 32, 512),         # query tile of 2 rows; causal edge across a chunk boundary
    ([64, 640, 1000], 60, 8, 384),  # chunk of 3 tiles; a sequence of exactly one page
])
def test_extend_matches_oracle(lengths, s_q, H, chunk):
    x = mw.make_extend(lengths, s_q=s_q, num_heads=H, seed=sum(lengths) + s_q)
    out, lse = run_extend(x, chunk)
    ref_out, ref_lse = oracle_extend(x, round_kv=True)
    compare(out, lse, ref_out, ref_lse, BF16_TOL, f"extend bf16-held K/V L={lengths} s_q={s_q}", out_bf16=True)
    ref_out, ref_lse = oracle_extend(x, round_kv=False)
    compare(out, lse, ref_out, ref_lse, EXACT_KV_TOL, f"extend exact K/V L={lengths} s_q={s_q}", out_bf16=True)


def test_chunk_size_does_not_change_the_result_beyond_rounding():
    """One chunk for everything, and chunks of 128: both within the bound of the same oracle,
    and close to each other (the merge is exact up to float32 rounding)."""
    x = mw.make_extend([900, 333], s_q=40, num_heads=16, seed=77)
    a_out, a_lse = run_extend(x, 1024)
    b_out, b_lse = run_extend(x, 128)
    ref_out, ref_lse = oracle_extend(x, round_kv=True)
    compare(a_out, a_lse, ref_out, ref_lse, BF16_TOL, "one chunk", out_bf16=True)
    compare(b_out, b_lse, ref_out, ref_lse, BF16_TOL, "chunks of 128", out_bf16=True)
    assert np.abs(a_lse - b_lse).max() < 1e-3


def test_max_seqlen_above_every_length():
    """max_seqlen larger than every length: the extra chunks hold no rows and change nothing."""
    x = mw.make_extend([300, 200], s_q=5, num_heads=16, seed=5)
    bt = x.cache.block_table
    x.cache.block_table = np.pad(bt, ((0, 0), (0, 16 - bt.shape[1])), constant_values=-1)  # entries never read
    out, lse = run_extend(x, 128, max_seqlen=1000)
    ref_out, ref_lse = oracle_extend(x, round_kv=True)
    compare(out, lse, ref_out, ref_lse, BF16_TOL, "max_seqlen 1000", out_bf16=True)


def test_single_token_extend_equals_absorbed_decode_then_projection():
    """s_q = 1: the expand path and the absorbed path (absorb -> decode -> project), both on the
    GPU, give the same output within their combined bf16 rounding ("Two equivalent paths")."""
    import torch
    from mla_absorbed_decode_02_gb300 import Decoder, mla_absorb_query, mla_project_output
    from gpu_util import params_for
    x = mw.make_extend([1500, 90, 4096], s_q=1, num_heads=128, seed=9)
    out_x, lse_x = run_extend(x, 1024)
    c = x.cache
    q_abs = torch.empty((c.batch, 1, c.num_heads, 512), dtype=torch.bfloat16, device="cuda")
    mla_absorb_query(_dev(x.q_nope), _dev(x.w_uk), q_abs)
    dec = Decoder(params_for(c))
    seq = torch.from_numpy(c.seqlens).cuda()
    dec.plan(seq)
    o_lat, lse_d = dec.decode(q_abs, _dev(x.q_rope), _dev(c.kv), torch.from_numpy(c.block_table).cuda(), seq, x.scale)
    o = torch.empty((c.batch, 1, c.num_heads, 128), dtype=torch.bfloat16, device="cuda")
    mla_project_output(o_lat, _dev(x.w_uv), o)
    torch.cuda.synchronize()
    out_a = o.float().cpu().numpy().astype(np.float64)
    rel = float(np.linalg.norm(out_x - out_a) / np.linalg.norm(out_a))
    dl = float(np.abs(lse_x - lse_d.cpu().numpy()).max())
    print(f"[parity] expand path vs absorbed path on the GPU: rel L2 {rel:.3g}, max |d lse| {dl:.3g}")
    assert rel <= 1e-2 and dl <= 5e-3


def test_extend_full_size_sampled_heads():
    """The bench's extend workload (one sequence, 512 new tokens after a 32,768-row prefix, 128
    heads, chunks of 4096 rows: nine chunks merged), run in full; the oracle computes a sample of
    heads spread over the four 32-row lane quarters, every new token."""
    x = mw.make_extend([32768 + 512], s_q=512, num_heads=128, seed=11, nan_tail=False)
    out, lse = run_extend(x, 4096)
    heads = np.array([0, 37, 70, 127])
    sub = mw.ExtendWorkload(cache=x.cache, s_q=x.s_q, q_nope=x.q_nope[:, :, heads], q_rope=x.q_rope[:, :, heads],
                            w_uk=x.w_uk[heads], w_uv=x.w_uv[heads], scale=x.scale)
    ref_out, ref_lse = oracle_extend(sub, round_kv=True)
    compare(out[:, :, heads], lse[:, :, heads], ref_out, ref_lse, BF16_TOL, "extend 512 after 32K, sampled heads",
            out_bf16=True)
