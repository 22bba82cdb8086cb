"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle.

Small cases compare every output element; the full-size benchmark workloads
compare sampled (sequence, head) rows the oracle computes one by one, in the
same launch configuration the benchmark times (default unit count)."""
import math
import os

import numpy as np
import pytest

import mla_workloads as mw
from gpu_util import BF16_TOL, FP8_TOL, compare, oracle_full, oracle_sampled, run_gpu, to_device, params_for

pytestmark = pytest.mark.gpu

THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_absorbed_decode_02_gb300.build import build
    build()


def full_check(w, tol=BF16_TOL, num_units=0, what="", token_group=0):
    out, lse, _ = run_gpu(w, num_units=num_units, token_group=token_group)
    ref_out, ref_lse = oracle_full(w, threads=THREADS)
    return compare(out, lse, ref_out, ref_lse, tol, what or w.name, out_bf16=w.out_dtype == "bf16")


# ------------------------------------------------------------------ the benchmark workloads

def test_workload_tiny_full():
    w = mw.make_workload(0)
    out, lse, _ = run_gpu(w)
    ref_out, ref_lse = oracle_full(w, threads=THREADS)
    errs = compare(out, lse, ref_out, ref_lse, BF16_TOL, w.name, raw=True)
    print("tiny", errs)


@pytest.mark.parametrize("index", [1, 2, 3, 4])
def test_workload_full_size_sampled(index):
    w = mw.make_workload(index)
    out, lse, _ = run_gpu(w)
    rng = np.random.default_rng(1000 + index)
    items = []
    for b in range(w.batch):
        for t in range(w.s_q):
            # one head from each 32-row group (a warp's tensor-memory lanes) of every (sequence, token)
            heads = [int(g + rng.integers(0, 32)) for g in range(0, w.num_heads, 32)]
            items.append((b, t, heads))
    ref = oracle_sampled(w, items, threads=THREADS)
    got_o, got_l, ref_o, ref_l = [], [], [], []
    for (b, t), (heads, o, l) in ref.items():
        got_o.append(out[b, t, heads])
        got_l.append(lse[b, t, heads])
        ref_o.append(o)
        ref_l.append(l)
    errs = compare(np.concatenate(got_o), np.concatenate(got_l), np.concatenate(ref_o), np.concatenate(ref_l),
                   FP8_TOL if w.kv_dtype == "fp8" else BF16_TOL, w.name, out_bf16=True, raw=True)
    print(w.name, errs)


# ------------------------------------------------------------------ ragged tails, splits, head counts

@pytest.mark.parametrize("num_units", [0, 1, 3, 7])
def test_ragged_lengths_and_splits(num_units):
    lens = [1, 63, 64, 65, 127, 128, 129, 255, 256, 257, 1000, 2049]
    w = mw.make_custom(lens, num_heads=128, seed=11, pool_factor=1.3)
    full_check(w, num_units=num_units, what=f"ragged U={num_units}")


@pytest.mark.parametrize("num_units", [9, 20, 40, 76])
def test_combine_column_slicings(num_units):
    """Four long sequences over 9, 20, 40 and 76 units: the combine merges up to ~20 splits per
    query block, with 4, 8, 16 or 32 column slices per (block, 16 heads) and the splits of a
    column dealt over 1, 2 or 4 lanes."""
    w = mw.make_custom([30000, 9000, 20000, 3000], num_heads=128, seed=27)
    full_check(w, num_units=num_units, what=f"combine U={num_units}")


@pytest.mark.parametrize("H", [1, 16, 17, 100, 128])
def test_head_counts(H):
    w = mw.make_custom([130, 7, 700], num_heads=H, seed=12)
    full_check(w, num_units=2, what=f"H={H}")


def test_f32_output():
    w = mw.make_custom([200, 513], num_heads=64, out_dtype="f32", seed=13)
    full_check(w, num_units=3)


@pytest.mark.parametrize("causal", [True, False])
def test_two_new_tokens(causal):
    w = mw.make_custom([2, 3, 128, 129, 600], num_heads=128, s_q=2, causal=causal, seed=14)
    full_check(w, num_units=4, what=f"s_q=2 causal={causal}")


@pytest.mark.parametrize("s_q,causal", [(4, True), (8, True), (8, False)])
def test_up_to_eight_new_tokens(s_q, causal):
    """MTP / speculative decoding: s_q new tokens per sequence, each its own query block.
    Sequences shorter than s_q leave the first causal tokens with no visible key."""
    w = mw.make_custom([1, 3, 8, 9, 65, 300, 1000], num_heads=128, s_q=s_q, causal=causal, seed=40 + s_q)
    full_check(w, num_units=5, what=f"s_q={s_q} causal={causal}")


@pytest.mark.parametrize("s_q,group,kv", [(2, 1, "bf16"), (2, 2, "bf16"), (4, 2, "bf16"), (4, 4, "bf16"),
                                           (6, 3, "bf16"), (2, 2, "fp8"), (4, 4, "fp8")])
@pytest.mark.parametrize("num_units", [1, 3, 40])
def test_token_groups(s_q, group, kv, num_units):
    """G new tokens of a sequence decoded together, each page loaded once into the G CTA pairs
    of a cluster.  Lengths 64k + 1 .. 64k + G - 1 put keys only the later tokens see on the work
    block's last tile (for the earlier tokens a fully masked tile, at 40 units often a piece of
    its own); sequences shorter than s_q leave early tokens no key at all; one is empty."""
    w = mw.make_custom([0, 1, 3, 65, 66, 129, 130, 640, 701], num_heads=64, s_q=s_q, causal=True, kv_dtype=kv,
                       seed=60 + 7 * s_q + group)
    full_check(w, tol=FP8_TOL if kv == "fp8" else BF16_TOL, num_units=num_units, token_group=group,
               what=f"s_q={s_q} G={group} {kv} units={num_units}")


@pytest.mark.parametrize("group,causal", [(2, True), (4, True), (4, False), (2, False)])
def test_token_groups_of_eight_new_tokens(group, causal):
    """s_q = 8 in work blocks of 2 or 4 tokens (several blocks per sequence, each read once by
    its cluster), causal and not."""
    w = mw.make_custom([1, 8, 9, 66, 300, 1000], num_heads=128, s_q=8, causal=causal, seed=80 + group)
    full_check(w, num_units=7, token_group=group, what=f"s_q=8 G={group} causal={causal}")


def test_token_group_plan_on_the_device_matches_the_host():
    import torch
    from mla_absorbed_decode_02_gb300 import Decoder, mla_plan_host
    w = mw.make_workload(4)
    _, _, _, _, seq = to_device(w)
    dec = Decoder(params_for(w, token_group=2))
    dec.plan(seq)
    torch.cuda.synchronize()
    host = mla_plan_host(params_for(w, num_units=dec.num_units, token_group=2), dec.num_units, w.seqlens)
    assert host[5] == 2 and np.array_equal(dec.sched.cpu().numpy(), host)


def test_fp8_cache_four_new_tokens():
    w = mw.make_custom([4, 70, 640], num_heads=64, s_q=4, causal=True, kv_dtype="fp8", seed=49)
    full_check(w, tol=FP8_TOL, num_units=3, what="fp8 s_q=4")


def test_empty_sequences():
    w = mw.make_custom([0, 100, 0, 1], num_heads=32, seed=15)
    out, lse, _ = run_gpu(w, num_units=2)
    ref_out, ref_lse = oracle_full(w)
    compare(out, lse, ref_out, ref_lse, BF16_TOL, "empty", out_bf16=True)
    assert np.all(lse[0] == -np.inf) and np.all(out[0] == 0) and np.all(lse[2] == -np.inf)


def test_length_beyond_the_block_table_is_reported():
    """A length past 64 x max_pages_per_seq breaks the call's contract: the decode reports
    MLA_ERR_INVALID_ARG in the device error word, reads nothing past the block-table row, and
    the other sequences' results are still right."""
    import torch
    from mla_absorbed_decode_02_gb300 import Decoder, MLA_ERR_INVALID_ARG, mla_device_error
    w = mw.make_custom([100, 128], num_heads=128, seed=25)       # block table rows of 2 pages
    ref_out, ref_lse = oracle_full(w)
    q_nope, q_rope, kv, bt, seq = to_device(w)
    seq[1] = 300                                                  # 5 pages, 3 past the row
    dec = Decoder(params_for(w, num_units=3))
    dec.plan(seq)
    out, lse = dec.decode(q_nope, q_rope, kv, bt, seq, w.scale)
    torch.cuda.synchronize()
    assert mla_device_error(clear=True) == MLA_ERR_INVALID_ARG
    compare(out[:1].float().cpu().numpy().astype(np.float64), lse[:1].cpu().numpy().astype(np.float64),
            ref_out[:1], ref_lse[:1], BF16_TOL, "valid sequence next to an overlong one", out_bf16=True)


def test_negative_length_is_reported_and_decoded_as_empty():
    """A negative length breaks the call's contract: the scheduler reports MLA_ERR_INVALID_ARG in
    the device error word and plans the sequence as empty (out = 0, lse = -inf); the other
    sequences' results are still right."""
    import torch
    from mla_absorbed_decode_02_gb300 import Decoder, MLA_ERR_INVALID_ARG, mla_device_error
    w = mw.make_custom([100, 64, 3000], num_heads=128, seed=26)
    ref_out, ref_lse = oracle_full(w)
    q_nope, q_rope, kv, bt, seq = to_device(w)
    seq[1] = -5
    dec = Decoder(params_for(w, num_units=3))
    dec.plan(seq)
    out, lse = dec.decode(q_nope, q_rope, kv, bt, seq, w.scale)
    torch.cuda.synchronize()
    assert mla_device_error(clear=True) == MLA_ERR_INVALID_ARG
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    assert np.all(o[1] == 0) and np.all(l[1] == -np.inf)
    keep = [0, 2]
    compare(o[keep], l[keep], ref_out[keep], ref_lse[keep], BF16_TOL, "valid sequences next to a negative length",
            out_bf16=True)


def test_all_pages_alias_one_physical_page():
    w = mw.make_custom([300, 64, 129], num_heads=128, seed=16)
    w.block_table[w.block_table >= 0] = 0
    full_check(w, num_units=3, what="aliased pages")


def test_zero_query_gives_uniform_average():
    w = mw.make_custom([1000, 77], num_heads=128, seed=17)
    w.q_nope[:] = 0
    w.q_rope[:] = 0
    errs = full_check(w, num_units=2, what="uniform")
    out, lse, _ = run_gpu(w, num_units=2)
    np.testing.assert_allclose(lse[:, 0, 0], np.log(w.seqlens), rtol=0, atol=1e-4)


def test_dominant_key():
    w = mw.make_custom([500, 300], num_heads=128, seed=18)
    # give key 123 of sequence 0 a RoPE key aligned with every head's RoPE query: it dominates
    page = w.block_table[0, 123 // 64]
    qr = w.q_rope.view(np.uint16)
    kr = (qr[0, 0].astype(np.uint32) << 16).view(np.float32).sum(axis=0)   # sum over heads
    big = np.sign(kr) * 8.0
    w.kv[page, 123 % 64, 512:] = mw.to_bf16_bits(big.astype(np.float32))
    full_check(w, num_units=2, what="dominant key")


def _scaled_queries(w, factor):
    """Queries multiplied by a power of two (exact in bf16)."""
    widen = lambda b: (b.astype(np.uint32) << 16).view(np.float32)
    w.q_nope[:] = mw.to_bf16_bits(widen(w.q_nope) * factor)
    w.q_rope[:] = mw.to_bf16_bits(widen(w.q_rope) * factor)
    return w


def _exchange_bound(w):
    """What the score exchange of a CTA pair may cost, from the inputs: each CTA of the pair holds a
    partial score over 256 latent + 32 RoPE dims; the one it receives is rounded to a multiple of
    2^(e-14), e the exponent bucket of the largest |partial| of its row and tile (times 1 + 2^-15),
    so no score is off by more than 2^(e_max - 15) * scale and the LSE, which moves by at most the
    largest score error, neither.  Returns (that bound in nats, the largest |c| of a visible key,
    the widest spread of one row's scores)."""
    widen = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    big, cmax, spread = 0.0, 0.0, 0.0
    for b in range(w.batch):
        L = int(w.seqlens[b])
        if L == 0:
            continue
        rows = widen(np.concatenate([w.kv[w.block_table[b, i]] for i in range((L + 63) // 64)])[:L])
        cmax = max(cmax, float(np.abs(rows[:, :512]).max()))
        for t in range(w.s_q):
            q = np.concatenate([widen(w.q_nope[b, t]), widen(w.q_rope[b, t])], axis=-1)   # [H, 576]
            spread = max(spread, float(np.ptp(rows @ q.T * w.scale, axis=0).max()))
            for h in (0, 1):
                lat, rope = slice(256 * h, 256 * h + 256), slice(512 + 32 * h, 512 + 32 * h + 32)
                part = rows[:, lat] @ q[:, lat].T + rows[:, rope] @ q[:, rope].T
                big = max(big, float(np.abs(part).max()))
    e_max = math.floor(math.log2(big * (1 + 2.0 ** -10))) + 1
    return 2.0 ** (e_max - 15) * w.scale, cmax, spread


@pytest.mark.parametrize("num_units", [0, 3, 7])
def test_high_dynamic_range_logits(num_units):
    """Queries scaled by 8: the scores of a row span more than 100 nats and one key usually
    dominates.  The LSE must stay within what the 16-bit score exchange between the two CTAs of a
    pair can cost (the bound computed from the inputs; about 2.3e-3 nats here), rel L2 within
    5e-3, and max |out - ref| beyond bf16 rounding within 1e-2 plus what rounding P to bf16 for
    the PV product can cost when one key carries all the weight (2^-9 of the largest |c|).
    Ragged lengths, several unit counts (splits merged by the combine)."""
    w = _scaled_queries(mw.make_custom([1, 63, 65, 700, 2049, 4100, 9000], num_heads=128, seed=71), 8.0)
    bound, cmax, spread = _exchange_bound(w)
    assert spread > 100.0
    tol = dict(max_abs=1e-2 + cmax * 2.0 ** -9, rel_l2=5e-3, lse=bound * 1.01 + 2e-5)
    full_check(w, tol=tol, num_units=num_units, what=f"high dynamic range x8 U={num_units}")


@pytest.mark.parametrize("num_units", [0, 3, 7])
def test_large_logits_within_the_stated_tolerance(num_units):
    """Queries scaled by 4 (scores of a row spread over ~50 nats): the LSE within the stated 1e-3
    and rel L2 within 5e-3, max |out - ref| beyond bf16 rounding within 1e-2 plus the bf16 P term."""
    w = _scaled_queries(mw.make_custom([1, 63, 65, 700, 2049, 4100, 9000], num_heads=128, seed=71), 4.0)
    bound, cmax, spread = _exchange_bound(w)
    assert spread > 45.0 and bound < 1.2e-3
    tol = dict(max_abs=1e-2 + cmax * 2.0 ** -9, rel_l2=5e-3, lse=1e-3)
    full_check(w, tol=tol, num_units=num_units, what=f"large logits x4 U={num_units}")


def test_a_million_keys():
    """One sequence of 2^20 cached tokens (16,384 pages, 1.2 GB) beside a 3-token one: the long one is
    split over every unit, so each of its 2 x 76 partials goes through the combine; byte offsets into
    the pool pass 2^30.  One head from each 32-row group, and every head of the short sequence."""
    w = mw.make_custom([1 << 20, 3], num_heads=128, seed=91)
    out, lse, dec = run_gpu(w)
    assert dec.num_units >= 2
    rng = np.random.default_rng(91)
    items = [(0, 0, [int(g + rng.integers(0, 32)) for g in range(0, 128, 32)]), (1, 0, list(range(128)))]
    ref = oracle_sampled(w, items, threads=THREADS)
    got_o = np.concatenate([out[b, t, h] for (b, t), (h, _, _) in ref.items()])
    got_l = np.concatenate([lse[b, t, h] for (b, t), (h, _, _) in ref.items()])
    ref_o = np.concatenate([o for (_, o, _) in ref.values()])
    ref_l = np.concatenate([l for (_, _, l) in ref.values()])
    compare(got_o, got_l, ref_o, ref_l, BF16_TOL, "2^20 keys", out_bf16=True)


def test_long_tail_row_garbage_is_ignored():
    """Cache rows past the sequence end inside the last page hold NaN: they must not leak."""
    w = mw.make_custom([65, 130, 1], num_heads=128, seed=19)
    nan_bf16 = np.uint16(0x7FC0)
    for b, L in enumerate(w.seqlens):
        last = (int(L) - 1) // 64
        page = w.block_table[b, last]
        w.kv[page, int(L) % 64 or 64:, :] = nan_bf16
    full_check(w, num_units=2, what="NaN past the end")


def test_metadata_is_reusable_across_calls():
    """One scheduler metadata serves every call of a step: two decodes with the same
    metadata and workspace give the same bits (and the oracle's result)."""
    import torch
    from mla_absorbed_decode_02_gb300 import Decoder, mla_device_error
    w = mw.make_custom([3000, 40, 5000, 700, 1], num_heads=128, seed=24)
    q_nope, q_rope, kv, bt, seq = to_device(w)
    dec = Decoder(params_for(w, num_units=9))
    dec.plan(seq)
    out1, lse1 = dec.decode(q_nope, q_rope, kv, bt, seq, w.scale)
    out2, lse2 = dec.decode(q_nope, q_rope, kv, bt, seq, w.scale)
    torch.cuda.synchronize()
    assert mla_device_error(clear=True) == 0
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    U, nqb = dec.num_units, w.batch * w.s_q
    assert dec.sched.cpu().numpy()[8 + 8 * U: 8 + 8 * U + nqb].max() > 1   # some block was split
    ref_out, ref_lse = oracle_full(w, threads=THREADS)
    compare(out2.float().cpu().numpy().astype(np.float64), lse2.cpu().numpy().astype(np.float64), ref_out, ref_lse,
            BF16_TOL, "reused metadata", out_bf16=True)


def test_decode_right_after_the_kernel_writing_its_queries():
    """The decode kernel is launched as a programmatic dependent of the kernel before it on
    the stream and starts its set-up early: it must still read the queries that kernel
    writes.  A slow producer (a matmul) writes the queries immediately before the decode;
    the result must be the oracle's for the new queries, not the old ones."""
    import dataclasses
    import torch
    from mla_absorbed_decode_02_gb300 import Decoder, mla_device_error
    w = mw.make_custom([2500, 900, 64, 4100], num_heads=128, seed=31)
    w2 = mw.make_custom([2500, 900, 64, 4100], num_heads=128, seed=32)  # other queries (same shapes)
    w2 = dataclasses.replace(w, q_nope=w2.q_nope, q_rope=w2.q_rope)      # same cache and pages as w
    q_nope, q_rope, kv, bt, seq = to_device(w)
    q2_nope, q2_rope, _, _, _ = to_device(w2)
    dec = Decoder(params_for(w))
    dec.plan(seq)
    dec.decode(q_nope, q_rope, kv, bt, seq, w.scale)  # warm: the old queries' results
    torch.cuda.synchronize()
    # producer: q_nope <- q2_nope through a matmul that takes a while (x @ I, exact for bf16)
    n = q2_nope.numel() // 512
    eye = torch.eye(512, dtype=torch.bfloat16, device=q_nope.device)
    big = torch.randn(8192, 8192, dtype=torch.bfloat16, device=q_nope.device)
    for _ in range(3):
        big = big @ big.T / 100.0  # keep the stream busy before the producer
    q_rope.copy_(q2_rope)
    torch.matmul(q2_nope.view(n, 512), eye, out=q_nope.view(n, 512))
    out, lse = dec.decode(q_nope, q_rope, kv, bt, seq, w.scale)
    torch.cuda.synchronize()
    assert mla_device_error(clear=True) == 0
    ref_out, ref_lse = oracle_full(w2, threads=THREADS)
    compare(out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ref_out, ref_lse,
            BF16_TOL, "decode after its producer", out_bf16=True)


# ------------------------------------------------------------------ FP8 E4M3 latent cache

@pytest.mark.parametrize("num_units", [0, 3])
def test_fp8_cache_ragged(num_units):
    w = mw.make_custom([1, 64, 65, 300, 1000, 2049], num_heads=128, kv_dtype="fp8", seed=21, pool_factor=1.2)
    errs = full_check(w, tol=FP8_TOL, num_units=num_units, what=f"fp8 U={num_units}")
    print("fp8", errs)


def test_fp8_two_new_tokens_causal():
    w = mw.make_custom([2, 129, 700], num_heads=128, s_q=2, causal=True, kv_dtype="fp8", seed=22)
    full_check(w, tol=FP8_TOL, num_units=4, what="fp8 s_q=2")


def test_fp8_every_code_value_reaches_the_output_at_its_dimension():
    """Each query selects one token of a shared page (orthogonal RoPE keys, no latent query; the
    other tokens' scores are 115 nats lower, so their probabilities are exactly 0 in fp32) and
    its output row is that token's dequantised latent row: e4m3(code) x tile scale. Rounding
    allowed: the scale and the product to bf16, the output to bf16, and the selected token's
    P = bf16(p) with p within a few 1e-3 of 1 (the 16-bit block floating point of the score
    exchange is exact to ~2^-15 of the row's largest partial score, here 1600), so
    |out - exact| <= 2^-6 |exact|; a misplaced code bit errs by 12% or more. Every non-NaN
    code value sits at many dimensions of every row, under scales from 2^-120 (bf16
    subnormal results) to 3e4."""
    from oracle import e4m3_to_f64
    T = 64
    w = mw.make_custom([T] * T, num_heads=16, kv_dtype="fp8", seed=24)
    w.block_table[:, 0] = w.block_table[0, 0]          # every sequence reads the same page
    page = int(w.block_table[0, 0])
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)   # 254 values, no NaN
    scales = np.array([1.0, 2.0 ** -120, 0.3716, 1234.5, 2.0 ** -118, 3.0e4, 7.0e-5, 0.1], np.float32)
    sc_of = np.empty((T, 4), np.float32)
    for j in range(T):
        row = np.zeros(mw.FP8_ROW_BYTES, np.uint8)
        row[:512] = codes[(np.arange(512) + 37 * j) % codes.size]
        sc_of[j] = scales[(np.arange(4) + j) % scales.size]
        row[512:528] = sc_of[j].view(np.uint8)
        kr = np.zeros(mw.D_R, np.float32)
        kr[j] = 40.0
        row[528:656] = mw.to_bf16_bits(kr).view(np.uint8)
        w.kv[page, j] = row
    w.q_nope[:] = 0
    qr = np.zeros((T, 1, 16, mw.D_R), np.float32)
    qr[np.arange(T), 0, :, np.arange(T)] = 40.0        # sequence b selects token b
    w.q_rope[:] = mw.to_bf16_bits(qr)
    out, lse, _ = run_gpu(w, num_units=0)
    value = np.array([e4m3_to_f64(c) for c in range(256)])
    for b in range(T):
        exact = value[w.kv[page, b, :512]] * np.repeat(sc_of[b].astype(np.float64), 128)
        got = out[b, 0]                                  # [16 heads, 512]
        err = np.abs(got - exact[None, :])
        bound = np.abs(exact) * 2.0 ** -6 + 2.0 ** -133
        bad = np.argwhere(err > bound[None, :])
        assert bad.size == 0, (f"token {b}: dim {bad[0][1]} code {w.kv[page, b, bad[0][1]]:#04x} "
                               f"got {got[tuple(bad[0])]!r} want {exact[bad[0][1]]!r}")
    assert np.all(np.isfinite(lse))


def test_fp8_row_garbage_past_the_end_is_ignored():
    """FP8 rows past the sequence end hold NaN codes, NaN scales and NaN RoPE: they must not leak."""
    w = mw.make_custom([65, 130, 1], num_heads=64, kv_dtype="fp8", seed=23)
    for b, L in enumerate(w.seqlens):
        page = w.block_table[b, (int(L) - 1) // 64]
        w.kv[page, int(L) % 64 or 64:, :] = 0xFF
    full_check(w, tol=FP8_TOL, num_units=2, what="fp8 NaN past the end")


# ------------------------------------------------------------------ metadata, errors

def test_device_plan_matches_host_plan():
    import torch
    from mla_absorbed_decode_02_gb300 import Decoder, mla_plan_host
    w = mw.make_workload(2)
    _, _, _, _, seq = to_device(w)
    dec = Decoder(params_for(w))
    dec.plan(seq)
    torch.cuda.synchronize()
    host = mla_plan_host(params_for(w, num_units=dec.num_units), dec.num_units, w.seqlens)
    assert np.array_equal(dec.sched.cpu().numpy(), host)


def test_bounded_wait_reports_timeout_and_context_survives():
    import torch
    from mla_absorbed_decode_02_gb300 import mla_wait_selftest, mla_device_error
    mla_device_error(clear=True)
    mla_wait_selftest(20000)
    word = mla_device_error(clear=True)
    assert word % 16 == 4 and word // 16 > 0
    # the context is still usable afterwards
    x = torch.arange(10, device="cuda").sum().item()
    assert x == 45
    assert mla_device_error(clear=True) == 0


def test_unaligned_pointer_rejected():
    import torch
    from mla_absorbed_decode_02_gb300 import MlaError, mla_decode
    w = mw.make_custom([10], num_heads=16, seed=20)
    q_nope, q_rope, kv, bt, seq = to_device(w)
    p = params_for(w, num_units=1)
    buf = torch.empty(100000, dtype=torch.uint8, device="cuda")
    with pytest.raises(MlaError):
        mla_decode(p, q_nope, q_rope, kv, bt, seq, w.scale, buf[1:], buf, buf, buf)
