"""The allocation-free entry point, mla_decode_noalloc, through the C ABI.

It must give what the entry point with caller-owned buffers gives
(mla_get_scheduler_metadata + mla_decode) on the same inputs, within the bf16
tolerance of the parity tests.  Two calls run in a row on different problems,
because every call reuses the one scratch array inside the library and finds
the previous call's contents there.  The file sorts last so that it also runs
after every other test in the same process."""
import ctypes

import numpy as np
import pytest

import mla_workloads as mw
from gpu_util import BF16_TOL, compare, params_for, to_device


def test_noalloc_rejects_requests_beyond_the_scratch_array():
    # needs no GPU: the size check comes before any CUDA call when the unit count is given
    from mla_absorbed_decode_02_gb300 import MLA_ERR_SCRATCH_LIMIT, MlaDecodeParams, load_library
    from mla_absorbed_decode_02_gb300 import build
    build.build()
    lib = load_library()
    big = MlaDecodeParams.make(batch=4096, s_q=1, num_heads=128, num_pages=1, max_pages_per_seq=1, num_units=76)
    null = None
    assert lib.mla_decode_noalloc(ctypes.byref(big), null, null, null, null, null, 1.0, null, null, null) == MLA_ERR_SCRATCH_LIMIT
    assert lib.mla_status_string(MLA_ERR_SCRATCH_LIMIT).decode() == "MLA_ERR_SCRATCH_LIMIT"


@pytest.mark.gpu
def test_noalloc_matches_the_buffered_entry_point_twice_in_a_row():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_absorbed_decode_02_gb300 import Decoder, mla_decode_noalloc, mla_device_error
    from mla_absorbed_decode_02_gb300.build import build
    build()
    problems = [
        # long and short sequences: several split query blocks, an empty one, a ragged tail
        mw.make_custom([9000, 300, 1, 0, 4097, 12345], seed=21, name="ragged-splits"),
        # a different batch and shape on the second call: the scratch holds the first call's plan
        mw.make_custom([5000, 64, 2100], s_q=2, causal=True, seed=22, name="two-new-tokens"),
    ]
    for w in problems:
        q_nope, q_rope, kv, bt, seq = to_device(w)
        p = params_for(w)
        dec = Decoder(p)
        dec.plan(seq)
        ref_out, ref_lse = dec.decode(q_nope, q_rope, kv, bt, seq, w.scale)
        out, lse = dec.new_outputs()
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        mla_decode_noalloc(p, q_nope, q_rope, kv, bt, seq, w.scale, out, lse)
        torch.cuda.synchronize()
        assert mla_device_error(clear=True) == 0
        compare(out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                ref_out.float().cpu().numpy().astype(np.float64), ref_lse.cpu().numpy().astype(np.float64),
                BF16_TOL, w.name, out_bf16=True)
