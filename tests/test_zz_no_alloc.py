"""The allocation-free entry point, mla_decode_noalloc, through the C ABI.

Some callers cannot allocate device memory while they decode: serving engines and
plugin hosts that hand all device memory to their own pool allocator at start-up.
mla_decode_noalloc serves them from a fixed array inside the library.  It runs
the same kernels on the same plan as mla_get_scheduler_metadata + mla_decode with
caller-owned buffers, so on the same inputs the two give the same bits; one of
the problems is also checked against the fp64 oracle.  Two calls run in a row on
different problems, because every call reuses the one scratch array and finds
the previous call's contents there.  The file sorts last so that it also runs
after every other test in the same process."""
import ctypes

import numpy as np
import pytest

import mla_workloads as mw
from gpu_util import BF16_TOL, compare, oracle_full, params_for, to_device


def _lib():
    from mla_absorbed_decode_02_gb300 import build, load_library
    build.build()
    return load_library()


def test_noalloc_rejects_requests_beyond_the_scratch_array():
    # needs no GPU: the size check comes before any CUDA call when the unit count is given
    from mla_absorbed_decode_02_gb300 import MLA_ERR_SCRATCH_LIMIT, MlaDecodeParams
    lib = _lib()
    big = MlaDecodeParams.make(batch=4096, s_q=1, num_heads=128, num_pages=1, max_pages_per_seq=1, num_units=76)
    null = None
    assert lib.mla_decode_noalloc(ctypes.byref(big), null, null, null, null, null, 1.0, null, null, null) == MLA_ERR_SCRATCH_LIMIT
    assert lib.mla_status_string(MLA_ERR_SCRATCH_LIMIT).decode() == "MLA_ERR_SCRATCH_LIMIT"


@pytest.mark.parametrize("units", [1, 76])
def test_noalloc_capacity_edge(units):
    """At 128 heads the array holds batch * s_q plus the unit count up to 255 partial slots:
    255 fits (checked from the sizes the library reports), 256 is refused before any launch."""
    from mla_absorbed_decode_02_gb300 import (MLA_ERR_SCRATCH_LIMIT, MLA_NOALLOC_SCRATCH_BYTES, MlaDecodeParams,
                                              mla_get_workspace_size)
    lib = _lib()
    fits = MlaDecodeParams.make(batch=255 - units, s_q=1, num_heads=128, num_pages=1, max_pages_per_seq=1,
                                num_units=units)
    sched, work = mla_get_workspace_size(fits)
    assert ((sched + 255) // 256) * 256 + work <= MLA_NOALLOC_SCRATCH_BYTES
    over = MlaDecodeParams.make(batch=256 - units, s_q=1, num_heads=128, num_pages=1, max_pages_per_seq=1,
                                num_units=units)
    sched, work = mla_get_workspace_size(over)
    assert ((sched + 255) // 256) * 256 + work > MLA_NOALLOC_SCRATCH_BYTES
    null = None
    assert lib.mla_decode_noalloc(ctypes.byref(over), null, null, null, null, null, 1.0, null, null, null) == MLA_ERR_SCRATCH_LIMIT


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
    for i, w in enumerate(problems):
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
        # same kernels, same plan: the same bits
        assert torch.equal(out, ref_out), w.name
        assert torch.equal(lse, ref_lse), w.name
        if i == 0:
            o_ref, l_ref = oracle_full(w)
            compare(out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                    o_ref, l_ref, BF16_TOL, w.name, out_bf16=True)
