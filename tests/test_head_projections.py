"""The per-head projections around the absorbed decode, through the C ABI, against the oracle.

mla_absorb_query computes q~ = q^N W_UK per head and mla_project_output o = o~ W_UV per head
("MLA inference: two computation paths and FlashMLA", section "Two equivalent paths", path
two).  Each is compared with the oracle's plain definition on the same bf16 inputs; then the
whole absorbed path (absorb -> decode -> project) is compared with textbook multi-head
attention over the expanded keys and values in float64 -- the equality of the two paths that
the same section shows."""
import math

import numpy as np
import pytest

import mla_workloads as mw
from gpu_util import BF16_TOL, compare, oracle_full, params_for, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_absorbed_decode_02_gb300.build import build
    build()


def _bf16(x):
    """float64 array -> (bf16 torch tensor on the GPU, the exact float64 values it holds)."""
    import torch
    bits = mw.to_bf16_bits(np.asarray(x, np.float32))
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    return t, (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _check_gemm(got, ref, what):
    """bf16 output of an fp32-accumulated product: within half a bf16 ulp of the exact value plus
    2^-12 of the largest |ref| (fp32 accumulation over up to 512 terms), and rel L2 within 3e-3."""
    from gpu_util import half_ulp_bf16
    err = np.abs(got - ref)
    excess = float((err - half_ulp_bf16(ref)).max())
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    print(f"[parity] {what}: max excess {excess:.3g}, rel L2 {rel:.3g}")
    assert excess <= 2.0 ** -12 * float(np.abs(ref).max()), (what, excess)
    assert rel <= 3e-3, (what, rel)


@pytest.mark.parametrize("T,d_nope", [(1, 128), (64, 128), (130, 128), (33, 64)])
def test_absorb_query_matches_oracle(T, d_nope):
    import torch
    import oracle
    from mla_absorbed_decode_02_gb300 import mla_absorb_query, mla_device_error
    rng = np.random.default_rng(90 + T)
    H = 128
    q, q64 = _bf16(rng.standard_normal((T, H, d_nope)))
    w, w64 = _bf16(rng.standard_normal((H, d_nope, 512)) / math.sqrt(d_nope))
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    mla_absorb_query(q, w, out)
    torch.cuda.synchronize()
    assert mla_device_error(clear=True) == 0
    _check_gemm(out.float().cpu().numpy().astype(np.float64), oracle.absorb_query(q64, w64), f"absorb T={T}")


@pytest.mark.parametrize("T,d_v", [(1, 128), (64, 128), (200, 128), (17, 192), (5, 512)])
def test_project_output_matches_oracle(T, d_v):
    import torch
    import oracle
    from mla_absorbed_decode_02_gb300 import mla_device_error, mla_project_output
    rng = np.random.default_rng(190 + T + d_v)
    H = 128
    o, o64 = _bf16(rng.standard_normal((T, H, 512)))
    w, w64 = _bf16(rng.standard_normal((H, 512, d_v)) / math.sqrt(512))
    out = torch.empty((T, H, d_v), dtype=torch.bfloat16, device="cuda")
    mla_project_output(o, w, out)
    torch.cuda.synchronize()
    assert mla_device_error(clear=True) == 0
    _check_gemm(out.float().cpu().numpy().astype(np.float64), oracle.project_output(o64, w64), f"project T={T} d_v={d_v}")


def test_absorbed_layer_equals_expanded_attention():
    """q^N, q^R and the latent cache with random W_UK, W_UV: absorb, decode and project on the
    GPU; each stage against the oracle on the inputs it received, and the result against
    expanded multi-head attention (per head: K = [c W_UK[h]^T, k^R], V = c W_UV[h]) in float64.
    The end-to-end tolerance (rel L2 1e-2) allows the two bf16 roundings between the kernels
    (q~ and o~) on top of the decode's own error."""
    import torch
    import oracle
    from mla_absorbed_decode_02_gb300 import (Decoder, mla_absorb_query, mla_device_error, mla_project_output)
    rng = np.random.default_rng(300)
    H, d_nope, d_r, d_v = 128, 128, 64, 128
    w = mw.make_custom([100, 700, 1500, 64], num_heads=H, seed=301)   # the latent cache, pages, block table
    B = w.batch
    q_n, q_n64 = _bf16(rng.standard_normal((B, 1, H, d_nope)))
    w_uk, w_uk64 = _bf16(rng.standard_normal((H, d_nope, 512)) / math.sqrt(512))
    w_uv, w_uv64 = _bf16(rng.standard_normal((H, 512, d_v)) / math.sqrt(512))
    # stage 1: absorption
    q_abs = torch.empty((B, 1, H, 512), dtype=torch.bfloat16, device="cuda")
    mla_absorb_query(q_n, w_uk, q_abs)
    torch.cuda.synchronize()
    q_abs64 = q_abs.float().cpu().numpy().astype(np.float64)
    _check_gemm(q_abs64, oracle.absorb_query(q_n64, w_uk64), "layer: absorb")
    # stage 2: the decode on the absorbed queries the GPU produced
    w.q_nope[:] = q_abs.view(torch.int16).cpu().numpy().view(np.uint16)
    q_nope, q_rope, kv, bt, seq = to_device(w)
    dec = Decoder(params_for(w))
    dec.plan(seq)
    o_lat, lse = dec.decode(q_nope, q_rope, kv, bt, seq, w.scale)
    torch.cuda.synchronize()
    ref_lat, ref_lse = oracle_full(w)
    compare(o_lat.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ref_lat, ref_lse,
            BF16_TOL, "layer: decode", out_bf16=True)
    # stage 3: the value projection of the latent output the GPU produced
    out = torch.empty((B, 1, H, d_v), dtype=torch.bfloat16, device="cuda")
    mla_project_output(o_lat, w_uv, out)
    torch.cuda.synchronize()
    assert mla_device_error(clear=True) == 0
    got = out.float().cpu().numpy().astype(np.float64)
    _check_gemm(got, oracle.project_output(o_lat.float().cpu().numpy().astype(np.float64), w_uv64), "layer: project")
    # end to end: the expanded path (path one) from the same bf16 inputs, in float64
    widen = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    q_r64 = widen(w.q_rope)
    want = np.empty((B, 1, H, d_v))
    for b in range(B):
        L = int(w.seqlens[b])
        rows = widen(np.concatenate([w.kv[w.block_table[b, i]] for i in range((L + 63) // 64)])[:L])
        c, k_r = rows[:, :512], rows[:, 512:]
        for h in range(H):
            k = np.concatenate([c @ w_uk64[h].T, k_r], axis=1)            # [L, d_nope + d_r]
            v = c @ w_uv64[h]                                            # [L, d_v]
            q = np.concatenate([q_n64[b, 0, h], q_r64[b, 0, h]])
            s = w.scale * (k @ q)
            p = np.exp(s - s.max())
            want[b, 0, h] = (p / p.sum()) @ v
    rel = float(np.linalg.norm(got - want) / np.linalg.norm(want))
    print(f"[parity] absorbed layer vs expanded attention: rel L2 {rel:.3g}, max abs {np.abs(got - want).max():.3g}")
    assert rel <= 1e-2
