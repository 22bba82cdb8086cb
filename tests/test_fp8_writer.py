"""The GPU FP8 cache writer (mla_quantize_kv_fp8) against the test-side quantiser
of the workload generator: byte-identical rows (codes, tile scales, RoPE copy)."""
import numpy as np
import pytest

import mla_workloads as mw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_absorbed_decode_02_gb300.build import build
    build()


def test_writer_matches_the_reference_quantiser_bytewise():
    import torch
    from mla_absorbed_decode_02_gb300 import mla_quantize_kv_fp8
    rng = np.random.default_rng(31)
    n = 1000
    x = rng.standard_normal((n, 576), dtype=np.float32) * rng.uniform(0.01, 50.0, size=(n, 1)).astype(np.float32)
    x[3, 128:256] = 0.0          # an all-zero tile: scale 1, codes 0
    x[4, :5] = [1e4, -1e4, 3e-3, -0.0, 7.0]
    bits = mw.to_bf16_bits(x)
    as_f32 = (bits.astype(np.uint32) << 16).view(np.float32)          # the bf16 values, exactly
    ref = mw.quantize_fp8_rows(as_f32[:, :512], bits[:, 512:])
    kv = torch.from_numpy(bits.view(np.int16)).cuda()
    out = torch.empty((n, 656), dtype=torch.uint8, device="cuda")
    mla_quantize_kv_fp8(kv, out, n)
    got = out.cpu().numpy()
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:10]


def test_writer_zero_tokens_is_a_no_op():
    import torch
    from mla_absorbed_decode_02_gb300 import mla_quantize_kv_fp8
    kv = torch.zeros((1, 576), dtype=torch.bfloat16, device="cuda")
    out = torch.full((1, 656), 7, dtype=torch.uint8, device="cuda")
    mla_quantize_kv_fp8(kv, out, 0)
    assert int(out.min()) == 7 and int(out.max()) == 7
