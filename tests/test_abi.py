"""Host-side tests of the C ABI (no GPU needed): the library builds, loads and
exports every entry point the header declares; argument checks; and the split
planner (the same code the scheduler kernel runs) covers the work exactly once."""
import ctypes
import re

import numpy as np
import pytest

from mla_absorbed_decode_02_gb300 import _lib
from mla_absorbed_decode_02_gb300.build import build
from mla_absorbed_decode_02_gb300._lib import MlaDecodeParams

import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "mla_decode.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "mla_decode" in names and "mla_get_scheduler_metadata" in names and len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert _lib.mla_status_string(0) == "MLA_OK"
    assert _lib.mla_status_string(4) == "MLA_ERR_TIMEOUT"
    assert _lib.mla_status_string(99) == "MLA_ERR_UNKNOWN"


def _p(**kw):
    base = dict(batch=2, s_q=1, num_heads=128, num_pages=10, max_pages_per_seq=5, num_units=4)
    base.update(kw)
    return MlaDecodeParams.make(**base)


def test_workspace_size_without_gpu(lib):
    sb, wb = _lib.mla_get_workspace_size(_p(batch=3, s_q=2, num_units=7))
    assert sb == 4 * (8 + 8 * 7 + 2 * 6)
    slots = 6 + 7
    assert wb >= slots * 128 * 512 * 4 + slots * 128 * 4


@pytest.mark.parametrize("kw,status", [
    (dict(batch=0), _lib.MLA_ERR_INVALID_ARG),
    (dict(num_heads=129), _lib.MLA_ERR_UNSUPPORTED),
    (dict(s_q=9), _lib.MLA_ERR_UNSUPPORTED),
    (dict(page_size=32), _lib.MLA_ERR_UNSUPPORTED),
    (dict(kv_dtype=7), _lib.MLA_ERR_INVALID_ARG),
    (dict(out_dtype=5), _lib.MLA_ERR_INVALID_ARG),
    (dict(num_units=-1), _lib.MLA_ERR_INVALID_ARG),
    (dict(s_q=2, token_group=3), _lib.MLA_ERR_INVALID_ARG),   # must divide s_q
    (dict(s_q=8, token_group=8), _lib.MLA_ERR_INVALID_ARG),   # at most 4 (clusters of 8 CTAs)
    (dict(token_group=-1), _lib.MLA_ERR_INVALID_ARG),
    (dict(qk_fp8=1), _lib.MLA_ERR_INVALID_ARG),                # FP8 QK needs the FP8 cache
    (dict(qk_fp8=2, kv_dtype=_lib.MLA_KV_FP8_E4M3), _lib.MLA_ERR_INVALID_ARG),
    (dict(qk_fp8=1, kv_dtype=_lib.MLA_KV_FP8_E4M3, s_q=2, token_group=2), _lib.MLA_ERR_UNSUPPORTED),
])
def test_bad_params_are_rejected(lib, kw, status):
    with pytest.raises(_lib.MlaError) as e:
        _lib.mla_get_workspace_size(_p(**kw))
    assert e.value.status == status


def test_null_pointers_rejected_before_any_launch(lib):
    with pytest.raises(_lib.MlaError) as e:
        _lib.mla_decode(_p(), None, None, None, None, None, 0.07, None, None, None, None, stream=0)
    assert e.value.status == _lib.MLA_ERR_INVALID_ARG


def test_workspace_of_a_token_group(lib):
    """A token group of G takes G partial slots for each unit boundary."""
    _, wb = _lib.mla_get_workspace_size(_p(batch=3, s_q=4, num_units=7, token_group=2))
    slots = 12 + 2 * 7
    assert wb == _a256(slots * 128 * 512 * 4) + _a256(slots * 128 * 4)


def _a256(x):
    return (x + 255) // 256 * 256


def test_fp8_qk_params_accepted(lib):
    """The FP8-QK decode takes the FP8 cache and no token group; its buffers are those of the
    FP8 decode."""
    kw = dict(batch=3, s_q=2, num_units=7, kv_dtype=_lib.MLA_KV_FP8_E4M3)
    assert _lib.mla_get_workspace_size(_p(qk_fp8=1, **kw)) == _lib.mla_get_workspace_size(_p(**kw))
    assert _lib.mla_get_workspace_size(_p(qk_fp8=1, token_group=1, **kw))


def test_query_quantizer_rejects_bad_arguments(lib):
    import torch
    x = torch.zeros(1024, dtype=torch.uint8)
    for args in ((None, x, x, 1), (x, None, x, 1), (x, x, None, 1), (x, x, x, -1)):
        with pytest.raises(_lib.MlaError) as e:
            _lib.mla_quantize_q_fp8(*args, stream=0)
        assert e.value.status == _lib.MLA_ERR_INVALID_ARG
    _lib.mla_quantize_q_fp8(x, x, x, 0, stream=0)  # no rows: nothing to launch


def test_reserved_must_be_zero(lib):
    p = _p()
    p.reserved[2] = 1
    with pytest.raises(_lib.MlaError):
        _lib.mla_get_workspace_size(p)


# ------------------------------------------------------------------ split planner

TILE = 64
FIX = int(re.search(r"#define MLA_PIECE_COST (\d+)", open(os.path.join(os.path.dirname(os.path.dirname(
    os.path.abspath(__file__))), "mla_absorbed_decode_02_gb300", "csrc", "plan.h")).read()).group(1))


def visible(L, s_q, t, causal):
    n = L - s_q + 1 + t if causal else L
    return max(0, min(n, L))


def decode_plan(sched, B, s_q, causal, seqlens):
    """Expand the metadata into the list of pieces (unit, qb, t0, t1, split_idx).  The unit
    records range over work blocks of G = sched[5] tokens whose tiles are their last token's;
    each work block's piece is one piece of each of its G query blocks.  Returns ntiles per
    query block as the tiles its work block covers."""
    U, nqb, G = sched[1], sched[2], sched[5]
    assert sched[0] == _lib.SCHED_MAGIC and nqb == B * s_q and G >= 1 and s_q % G == 0
    units = sched[8:8 + 8 * U].reshape(U, 8)
    num_splits = sched[8 + 8 * U:8 + 8 * U + nqb]
    offsets = sched[8 + 8 * U + nqb:]
    own = [-(-visible(seqlens[q // s_q], s_q, q % s_q, causal) // TILE) for q in range(nqb)]
    wtiles = [own[w * G + G - 1] for w in range(nqb // G)]   # a work block: its last token's tiles
    assert all(own[w * G + g] <= wtiles[w] for w in range(nqb // G) for g in range(G))
    ntiles = [wtiles[q // G] for q in range(nqb)]
    pieces = []
    for u in range(U):
        wb0, tb, wb1, te, fs = units[u, :5]
        if wb0 < 0:
            continue
        for wb in range(wb0, wb1 + 1):
            a = tb if wb == wb0 else 0
            b = te if wb == wb1 else wtiles[wb]
            if wtiles[wb] > 0 and a < b:
                for g in range(G):
                    pieces.append((u, wb * G + g, a, b, fs if wb == wb0 else 0))
    return pieces, ntiles, num_splits, offsets


@pytest.mark.parametrize("seed", range(16))
def test_plan_covers_every_tile_once(lib, seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 80))
    s_q = int(rng.integers(1, 9))
    causal = bool(rng.integers(0, 2))
    kind = seed % 4
    if kind == 0:
        seqlens = rng.integers(0, 3000, size=B)
    elif kind == 1:
        seqlens = np.full(B, int(rng.integers(1, 9000)))
    elif kind == 2:
        seqlens = np.round(np.exp(rng.uniform(np.log(1), np.log(140000), size=B)))
    else:
        seqlens = rng.choice([0, 1, 2, 127, 128, 129, 65536], size=B)
    seqlens = seqlens.astype(np.int32)
    U = int(rng.choice([1, 2, 3, 7, 19, 76, 148, 500]))
    group = [0, 1, *[g for g in (2, 3, 4) if s_q % g == 0]][seed % (2 + sum(s_q % g == 0 for g in (2, 3, 4)))]
    p = MlaDecodeParams.make(B, s_q, 128, 100, 10, causal=causal, num_units=U, token_group=group)
    sched = _lib.mla_plan_host(p, U, seqlens)
    pieces, ntiles, num_splits, offsets = decode_plan(sched, B, s_q, causal, seqlens)
    # every tile of every query block exactly once, pieces non-empty
    seen = {}
    for u, qb, a, b, si in pieces:
        assert b > a
        for t in range(a, b):
            assert (qb, t) not in seen
            seen[(qb, t)] = u
    assert len(seen) == sum(ntiles)
    # units hold contiguous, increasing stretches of (qb, tile)
    order = [(qb // sched[5], a, qb) for _, qb, a, _, _ in pieces]
    assert order == sorted(order)
    # split bookkeeping: split indices 0..n-1 per query block, slots disjoint
    per_qb = {}
    for u, qb, a, b, si in pieces:
        per_qb.setdefault(qb, []).append(si)
    slots = set()
    for qb in range(B * s_q):
        got = per_qb.get(qb, [])
        assert num_splits[qb] == len(got)
        assert sorted(got) == list(range(len(got)))
        if len(got) > 1:
            for i in range(len(got)):
                s = offsets[qb] + i
                assert s not in slots
                slots.add(s)
    G = sched[5]
    assert G == (group or 1)
    assert sched[3] == len(slots) <= B * s_q + G * U


def test_plan_balances_load(lib):
    seqlens = np.full(32, 4096, np.int32)
    U = 76
    p = MlaDecodeParams.make(32, 1, 128, 2048, 64, num_units=U)
    sched = _lib.mla_plan_host(p, U, seqlens)
    pieces, ntiles, _, _ = decode_plan(sched, 32, 1, True, seqlens)
    load = np.zeros(U)
    for u, qb, a, b, _ in pieces:
        load[u] += (b - a) + FIX
    total = sum(ntiles) + FIX * 32
    budget = -(-total // U)
    assert sched[4] == budget
    assert load.max() <= budget + FIX      # one extra piece overhead at most
    assert (load > 0).sum() >= U - 2


def test_plan_handles_empty_sequences(lib):
    seqlens = np.array([0, 5, 0, 0, 300, 0], np.int32)
    p = MlaDecodeParams.make(6, 1, 128, 10, 5, num_units=3)
    sched = _lib.mla_plan_host(p, 3, seqlens)
    pieces, ntiles, num_splits, _ = decode_plan(sched, 6, 1, True, seqlens)
    assert [num_splits[i] for i in (0, 2, 3, 5)] == [0, 0, 0, 0]
    assert sum(b - a for _, _, a, b, _ in pieces) == sum(ntiles) == -(-5 // TILE) + -(-300 // TILE)


def test_non_positive_scale_is_rejected_before_any_launch(lib):
    from mla_absorbed_decode_02_gb300 import MlaDecodeParams
    p = MlaDecodeParams.make(batch=1, s_q=1, num_heads=128, num_pages=1, max_pages_per_seq=1, num_units=4)
    buf = ctypes.c_void_p(256)  # never dereferenced: the scale check comes first
    for scale in (0.0, -0.07, float("nan"), float("inf")):
        st = lib.mla_decode_splitkv(ctypes.byref(p), buf, buf, buf, buf, buf, scale, buf, buf, buf, buf, None)
        assert st == 1, scale


def test_plan_refuses_negative_lengths(lib):
    """A negative length is outside the contract: the host twin refuses it."""
    p = MlaDecodeParams.make(3, 1, 128, 10, 5, num_units=2)
    with pytest.raises(_lib.MlaError):
        _lib.mla_plan_host(p, 2, np.array([100, -1, 7], np.int32))


def test_plan_refuses_more_positions_than_an_int32_holds(lib):
    """Work positions are int32: lengths that need more than 2^31 - 1 of them in total are refused
    (and the metadata header loses its magic word, so no kernel would use it), where a smaller
    total of the same shape still plans."""
    B = 1 << 17
    p = MlaDecodeParams.make(B, 1, 128, 1 << 20, 1 << 14, num_units=76)
    over = np.full(B, 1 << 20, np.int32)                 # 16384 tiles + 6 each: 2^17 * 16390 > 2^31
    with pytest.raises(_lib.MlaError):
        _lib.mla_plan_host(p, 76, over)
    ok = np.full(B, 1 << 19, np.int32)                   # 8192 tiles + 6 each: below 2^31
    sched = _lib.mla_plan_host(p, 76, ok)
    assert sched[0] == _lib.SCHED_MAGIC and sched[1] == 76 and sched[2] == B


def test_head_projections_reject_bad_arguments_before_any_launch(lib):
    """mla_absorb_query / mla_project_output check their sizes and pointers before touching CUDA."""
    buf = ctypes.c_void_p(256)  # never dereferenced
    odd = ctypes.c_void_p(258)  # not 16-byte aligned
    for f in (lib.mla_absorb_query, lib.mla_project_output):
        assert f(0, 128, 128, buf, buf, buf, None) == _lib.MLA_ERR_INVALID_ARG         # no tokens
        assert f(4, 0, 128, buf, buf, buf, None) == _lib.MLA_ERR_INVALID_ARG           # no heads
        assert f(4, 128, 128, None, buf, buf, None) == _lib.MLA_ERR_INVALID_ARG        # null input
        assert f(4, 128, 128, buf, buf, odd, None) == _lib.MLA_ERR_INVALID_ARG         # misaligned output
        assert f(4, 128, 100, buf, buf, buf, None) == _lib.MLA_ERR_UNSUPPORTED         # width not a multiple of 64


def test_extend_params_are_checked_without_a_gpu(lib):
    """mla_extend_workspace_size validates the extend parameters on the host and sizes the
    workspace: two bf16 [B][H][C][128] buffers and the float32 merge accumulators."""
    ok = dict(batch=2, s_q=5, num_heads=16, num_pages=40, max_pages_per_seq=20, max_seqlen=1000, chunk_tokens=256)
    p = _lib.MlaExtendParams.make(**ok)
    n = ctypes.c_size_t()
    assert lib.mla_extend_workspace_size(ctypes.byref(p), ctypes.byref(n)) == _lib.MLA_OK
    a256 = lambda x: (x + 255) // 256 * 256
    assert n.value == 2 * a256(2 * 16 * 256 * 128 * 2) + a256(2 * 5 * 16 * 128 * 4) + a256(2 * 5 * 16 * 4)
    bad = [(dict(chunk_tokens=200), _lib.MLA_ERR_UNSUPPORTED),      # not a multiple of 128
           (dict(d_v=64), _lib.MLA_ERR_UNSUPPORTED),               # only 128-wide heads
           (dict(num_heads=256), _lib.MLA_ERR_UNSUPPORTED),
           (dict(max_seqlen=20 * 64 + 1), _lib.MLA_ERR_INVALID_ARG),  # longer than the block table
           (dict(s_q=1001), _lib.MLA_ERR_INVALID_ARG),             # more new tokens than rows
           (dict(batch=0), _lib.MLA_ERR_INVALID_ARG),
           (dict(page_size=32), _lib.MLA_ERR_UNSUPPORTED)]
    for kw, status in bad:
        q = _lib.MlaExtendParams.make(**{**ok, **kw})
        assert lib.mla_extend_workspace_size(ctypes.byref(q), ctypes.byref(n)) == status, kw
    q = _lib.MlaExtendParams.make(**ok)
    q.reserved[2] = 1
    assert lib.mla_extend_workspace_size(ctypes.byref(q), ctypes.byref(n)) == _lib.MLA_ERR_INVALID_ARG
    buf = ctypes.c_void_p(256)
    assert lib.mla_extend(ctypes.byref(p), buf, buf, buf, buf, buf, buf, buf, ctypes.c_float(0.1), buf, buf, None,
                          None) == _lib.MLA_ERR_INVALID_ARG                       # no workspace
    assert lib.mla_extend(ctypes.byref(p), buf, buf, buf, buf, buf, buf, buf, ctypes.c_float(0.0), buf, buf, buf,
                          None) == _lib.MLA_ERR_INVALID_ARG                       # scale 0
    assert lib.mla_expand_kv(ctypes.byref(p), buf, buf, buf, buf, buf, 100, buf, buf, None) == \
        _lib.MLA_ERR_INVALID_ARG                                                  # chunk start not a chunk multiple
