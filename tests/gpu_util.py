"""Helpers shared by the GPU tests: run the CUDA library on a workload and
compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np

# Tolerances for a bf16 cache (bf16 MMA inputs, fp32 accumulation):
# max |out - ref| <= 1e-2, ||out - ref||_2 / ||ref||_2 <= 5e-3, |lse - ref| <= 1e-3.
BF16_TOL = dict(max_abs=1e-2, rel_l2=5e-3, lse=1e-3)
# FP8 E4M3 latent cache, compared with the oracle fed the identically dequantised cache.
FP8_TOL = dict(max_abs=None, rel_l2=3e-2, lse=None)


def to_device(w, device="cuda"):
    import torch
    q_nope = torch.from_numpy(w.q_nope.view(np.int16)).view(torch.bfloat16).to(device)
    q_rope = torch.from_numpy(w.q_rope.view(np.int16)).view(torch.bfloat16).to(device)
    if w.kv_dtype == "bf16":
        kv = torch.from_numpy(w.kv.view(np.int16)).view(torch.bfloat16).to(device)
    else:
        kv = torch.from_numpy(w.kv).to(device)
    bt = torch.from_numpy(w.block_table).to(device)
    seq = torch.from_numpy(w.seqlens).to(device)
    return q_nope, q_rope, kv, bt, seq


def params_for(w, num_units=0, timeout_us=0, token_group=0, qk_fp8=0):
    from mla_absorbed_decode_02_gb300 import MlaDecodeParams, MLA_KV_BF16, MLA_KV_FP8_E4M3, MLA_OUT_BF16, MLA_OUT_F32
    return MlaDecodeParams.make(w.batch, w.s_q, w.num_heads, w.num_pages, w.block_table.shape[1], causal=w.causal,
                                kv_dtype=MLA_KV_FP8_E4M3 if w.kv_dtype == "fp8" else MLA_KV_BF16,
                                out_dtype=MLA_OUT_F32 if w.out_dtype == "f32" else MLA_OUT_BF16,
                                num_units=num_units, timeout_us=timeout_us, token_group=token_group, qk_fp8=qk_fp8)


def run_gpu(w, num_units=0, token_group=0):
    """Decode workload w with the CUDA library; returns (out float64 numpy, lse float64 numpy, decoder)."""
    import torch
    from mla_absorbed_decode_02_gb300 import Decoder, mla_device_error
    q_nope, q_rope, kv, bt, seq = to_device(w)
    dec = Decoder(params_for(w, num_units, token_group=token_group))
    dec.plan(seq)
    out, lse = dec.decode(q_nope, q_rope, kv, bt, seq, w.scale)
    torch.cuda.synchronize()
    err = mla_device_error(clear=True)
    assert err == 0, f"device error word {err}"
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), dec


def half_ulp_bf16(x):
    """Half the spacing of bf16 numbers at |x| (the rounding error of storing x as bf16)."""
    a = np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** -126)
    return np.ldexp(1.0, (np.floor(np.log2(a)) - 8).astype(np.int64))


def compare(out, lse, ref_out, ref_lse, tol, what="", out_bf16=False, raw=False):
    """Element-wise comparison against the oracle; returns the measured errors.

    max_abs_raw is max |out - ref| itself.  With out_bf16 the output tensor holds bf16
    numbers, and storing the exact result already costs up to half a bf16 ulp (up to
    0.0078 for |out| in [2, 4)); the max-abs bound then applies to the error beyond that,
    |out - ref| - half_ulp(ref) (max_abs).  raw=True bounds max_abs_raw as well: on the
    benchmark workloads |out| is far below 1, where half an ulp is tiny, so the literal
    bound is affordable there."""
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(lse)), f"{what}: -inf pattern of lse differs"
    assert np.all(out[~fin] == 0), f"{what}: tokens with no visible key must give out = 0"
    diff = out - ref_out
    excess = np.abs(diff) - (half_ulp_bf16(ref_out) if out_bf16 else 0.0)
    max_abs = float(excess.max()) if diff.size else 0.0
    max_abs_raw = float(np.abs(diff).max()) if diff.size else 0.0
    denom = float(np.linalg.norm(ref_out))
    rel_l2 = float(np.linalg.norm(diff) / denom) if denom > 0 else float(np.linalg.norm(diff))
    lse_err = float(np.abs(lse[fin] - ref_lse[fin]).max()) if fin.any() else 0.0
    errs = dict(max_abs=max_abs, max_abs_raw=max_abs_raw, rel_l2=rel_l2, lse=lse_err)
    print(f"[parity] {what}: max_abs_raw={max_abs_raw:.3g} max_abs_beyond_bf16_rounding={max_abs:.3g} "
          f"rel_l2={rel_l2:.3g} lse={lse_err:.3g}")
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    if tol.get("max_abs") is not None:
        assert max_abs <= tol["max_abs"], f"{what}: max abs {max_abs:.3g} > {tol['max_abs']} ({errs})"
        if raw:
            assert max_abs_raw <= tol["max_abs"], f"{what}: raw max abs {max_abs_raw:.3g} > {tol['max_abs']} ({errs})"
    assert rel_l2 <= tol["rel_l2"], f"{what}: rel L2 {rel_l2:.3g} > {tol['rel_l2']} ({errs})"
    if tol.get("lse") is not None:
        assert lse_err <= tol["lse"], f"{what}: lse err {lse_err:.3g} > {tol['lse']} ({errs})"
    return errs


def oracle_full(w, threads=8):
    import oracle
    return oracle.from_workload(w).full(threads=threads)


def oracle_sampled(w, items, threads=8):
    """items: list of (b, t, heads) -> dict {(b, t): (heads, out, lse)}"""
    import oracle
    P = oracle.from_workload(w)
    res = {}

    def work(chunk):
        for b, t, heads in chunk:
            o, l = P.rows(b, t, heads=np.asarray(heads, np.int32))
            res[(b, t)] = (np.asarray(heads), o, l)

    oracle.run_threads(work, list(items), threads)
    return res
