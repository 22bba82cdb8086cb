"""fp64 CPU oracle for absorbed-path MLA decode -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product library (``mla_absorbed_decode_02_gb300``) never imports it, and this
package imports nothing from the product: the two share no code.

The arithmetic lives in ``mla_oracle.c`` (plain single-threaded fp64 C, built
with gcc by ``build()``); this module marshals numpy arrays into it and adds
the exact bf16 -> float64 widening of the queries.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB = os.path.join(_HERE, "libmla_oracle.so")

KV_F64, KV_BF16, KV_FP8 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2; no fast-math, so IEEE fp64 semantics hold)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Problem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("s_q", ctypes.c_int32), ("num_heads", ctypes.c_int32), ("causal", ctypes.c_int32),
        ("d_c", ctypes.c_int32), ("d_r", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
        ("kv_kind", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("scale", ctypes.c_double),
        ("q_nope", ctypes.c_void_p), ("q_rope", ctypes.c_void_p), ("kv", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p), ("seqlens", ctypes.c_void_p),
    ]


_lib = None
_lock = threading.Lock()


def bind(path: str):
    """Load an oracle library build (the normal one, or a test's variant of the same source)
    and declare its entry points."""
    lib = ctypes.CDLL(path)
    lib.orc_decode_rows.argtypes = [ctypes.POINTER(_Problem), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                    ctypes.c_void_p]
    lib.orc_decode_rows.restype = ctypes.c_int
    lib.orc_merge.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                              ctypes.c_void_p, ctypes.c_void_p]
    lib.orc_merge.restype = None
    lib.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_to_f64.restype = ctypes.c_double
    lib.orc_visible_keys.argtypes = [ctypes.POINTER(_Problem), ctypes.c_int, ctypes.c_int]
    lib.orc_visible_keys.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
    return _lib


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of raw bf16 patterns (uint16) to float64."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def e4m3_to_f64(code: int) -> float:
    return _load().orc_e4m3_to_f64(int(code) & 0xFF)


def fp8_rows_to_f64(rows: np.ndarray, d_c: int = 512, d_r: int = 64):
    """Rows in the FP8 cache-row layout ("MLA and FP8 MoE Serving: Multi-Head Latent Attention at
    Scale", section "Understanding FP8 Formats: E4M3 vs. E5M2"): d_c E4M3 codes, one float32 scale per
    128 codes, d_r bf16 values -> (latent float64 [..., d_c] = code x scale, exact; RoPE float64
    [..., d_r]).  The same decoding the C oracle applies to an FP8 cache, for rows held elsewhere
    (the quantised query of an FP8-QK decode)."""
    rows = np.ascontiguousarray(rows, dtype=np.uint8)
    lead = rows.shape[:-1]
    assert rows.shape[-1] == d_c + 4 * (d_c // 128) + 2 * d_r
    r = rows.reshape(-1, rows.shape[-1])
    table = np.array([e4m3_to_f64(c) for c in range(256)], np.float64)
    scales = np.ascontiguousarray(r[:, d_c:d_c + 4 * (d_c // 128)]).view(np.float32).astype(np.float64)
    lat = table[r[:, :d_c]] * np.repeat(scales, 128, axis=1)
    rope = bf16_bits_to_f64(np.ascontiguousarray(r[:, d_c + 4 * (d_c // 128):]).view(np.uint16))
    return lat.reshape(*lead, d_c), rope.reshape(*lead, d_r)


@dataclass
class Problem:
    """Inputs in the oracle's terms (numpy, host).

    q_nope: float64 [B, s_q, H, d_c]; q_rope: float64 [B, s_q, H, d_r]
    kv: page pool -- float64 [pages, page_size, d_c+d_r] (KV_F64), uint16 bf16 bits
        [pages, page_size, d_c+d_r] (KV_BF16) or uint8 [pages, page_size, row_bytes] (KV_FP8)
    block_table: int32 [B, max_pages]; seqlens: int32 [B]
    """
    q_nope: np.ndarray
    q_rope: np.ndarray
    kv: np.ndarray
    kv_kind: int
    block_table: np.ndarray
    seqlens: np.ndarray
    scale: float
    causal: bool = True
    page_size: int = 64

    def __post_init__(self):
        self.q_nope = np.ascontiguousarray(self.q_nope, dtype=np.float64)
        self.q_rope = np.ascontiguousarray(self.q_rope, dtype=np.float64)
        self.kv = np.ascontiguousarray(self.kv)
        self.block_table = np.ascontiguousarray(self.block_table, dtype=np.int32)
        self.seqlens = np.ascontiguousarray(self.seqlens, dtype=np.int32)
        B, s_q, H, d_c = self.q_nope.shape
        d_r = self.q_rope.shape[-1]
        assert self.q_rope.shape == (B, s_q, H, d_r)
        assert self.block_table.shape[0] == B and self.seqlens.shape == (B,)
        exp_dtype = {KV_F64: np.float64, KV_BF16: np.uint16, KV_FP8: np.uint8}[self.kv_kind]
        assert self.kv.dtype == exp_dtype, (self.kv.dtype, exp_dtype)
        self._c = _Problem(B, s_q, H, int(bool(self.causal)), d_c, d_r, self.page_size,
                           self.block_table.shape[1], self.kv_kind, 0, float(self.scale),
                           self.q_nope.ctypes.data, self.q_rope.ctypes.data, self.kv.ctypes.data,
                           self.block_table.ctypes.data, self.seqlens.ctypes.data)

    @property
    def shape(self):
        return self.q_nope.shape

    def visible_keys(self, b: int, t: int) -> int:
        return _load().orc_visible_keys(ctypes.byref(self._c), b, t)

    def rows(self, b: int, t: int, heads=None, k_lo: int = 0, k_hi: int = -1):
        """out [n_heads, d_c] and lse [n_heads] for query block (b, t)."""
        B, s_q, H, d_c = self.shape
        heads = np.arange(H, dtype=np.int32) if heads is None else np.ascontiguousarray(heads, dtype=np.int32)
        out = np.empty((len(heads), d_c), np.float64)
        lse = np.empty(len(heads), np.float64)
        rc = _load().orc_decode_rows(ctypes.byref(self._c), b, t, len(heads), heads.ctypes.data, k_lo, k_hi,
                                     out.ctypes.data, lse.ctypes.data)
        if rc != 0:
            raise MemoryError("oracle scratch allocation failed")
        return out, lse

    def full(self, threads: int = 1):
        """out [B, s_q, H, d_c], lse [B, s_q, H]; (b, t) blocks spread over `threads` host threads."""
        B, s_q, H, d_c = self.shape
        out = np.empty((B, s_q, H, d_c), np.float64)
        lse = np.empty((B, s_q, H), np.float64)
        items = [(b, t) for b in range(B) for t in range(s_q)]

        def work(chunk):
            for b, t in chunk:
                out[b, t], lse[b, t] = self.rows(b, t)

        run_threads(work, items, threads)
        return out, lse


def run_threads(fn, items, threads: int):
    """Run fn over round-robin chunks of items on `threads` Python threads (the C call releases the GIL)."""
    threads = max(1, min(threads, len(items)))
    if threads == 1:
        fn(items)
        return
    chunks = [items[i::threads] for i in range(threads)]
    ts = [threading.Thread(target=fn, args=(c,)) for c in chunks]
    for t in ts:
        t.start()
    for t in ts:
        t.join()


def merge(outs: np.ndarray, lses: np.ndarray):
    """LSE merge of partial (out_i [d_c], lse_i) over disjoint key ranges -> (out, lse)."""
    outs = np.ascontiguousarray(outs, dtype=np.float64)
    lses = np.ascontiguousarray(lses, dtype=np.float64)
    n, d_c = outs.shape
    out = np.empty(d_c, np.float64)
    lse = np.empty(1, np.float64)
    _load().orc_merge(n, d_c, outs.ctypes.data, lses.ctypes.data, out.ctypes.data, lse.ctypes.data)
    return out, float(lse[0])


def from_workload(w) -> Problem:
    """Oracle view of a workload produced by ``mla_workloads.make_workload`` (bf16 or FP8 cache)."""
    kind = KV_FP8 if w.kv_dtype == "fp8" else KV_BF16
    return Problem(q_nope=bf16_bits_to_f64(w.q_nope), q_rope=bf16_bits_to_f64(w.q_rope), kv=w.kv, kv_kind=kind,
                   block_table=w.block_table, seqlens=w.seqlens, scale=w.scale, causal=w.causal,
                   page_size=w.page_size)


def absorb_query(q_nope, w_uk) -> np.ndarray:
    """q~[.., h, :] = q^N[.., h, :] W_UK[h]: the query absorption of the absorbed path ("MLA
    inference: two computation paths and FlashMLA", section "Two equivalent paths", path two),
    in float64.  q_nope [..., H, d_nope], w_uk [H, d_nope, d_c] -> [..., H, d_c]."""
    q = np.asarray(q_nope, np.float64)
    w = np.asarray(w_uk, np.float64)
    return np.einsum("...hk,hkn->...hn", q, w, optimize=True)


def project_output(o_latent, w_uv) -> np.ndarray:
    """o[.., h, :] = o~[.., h, :] W_UV[h]: the value projection that ends the absorbed path (same
    section), in float64.  o_latent [..., H, d_c], w_uv [H, d_c, d_v] -> [..., H, d_v]."""
    o = np.asarray(o_latent, np.float64)
    w = np.asarray(w_uv, np.float64)
    return np.einsum("...hk,hkn->...hn", o, w, optimize=True)


# ---------------------------------------------------------------- the expand path (extend)

def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even, returned as float64 (for
    values in bf16's normal range; zero stays zero).  bf16 keeps 8 significant bits: write
    x = m * 2^e with m in [0.5, 1), round m * 2^8 to an integer (numpy rounds halves to even)."""
    m, e = np.frexp(np.asarray(x, np.float64))
    return np.ldexp(np.round(m * 256.0), e - 8)


def cache_rows(kv_bits, block_table, b: int, L: int, page_size: int = 64) -> np.ndarray:
    """Rows 0..L-1 of sequence b's paged bf16 cache, widened to float64: [L, d_c + d_r].
    Row j lives in slot j % page_size of page block_table[b][j // page_size]."""
    n_pages = (L + page_size - 1) // page_size
    pages = np.asarray(block_table[b, :n_pages], np.int64)
    return bf16_bits_to_f64(np.asarray(kv_bits)[pages].reshape(-1, kv_bits.shape[-1])[:L])


def expand_kv(c, w_uk, w_uv):
    """Path one's expansion of cached latent vectors ("MLA inference: two computation paths and
    FlashMLA", section "Two equivalent paths", path one): per head h, the non-positional key
    k^N_j = W_UK[h] c_j and the value v_j = c_j W_UV[h], with W_UK [H, d_nope, d_c] and
    W_UV [H, d_c, d_v] (the layouts of absorb_query / project_output).
    c [L, d_c] -> (k^N [H, L, d_nope], v [H, L, d_v]), float64."""
    c = np.asarray(c, np.float64)
    return (np.einsum("hnc,jc->hjn", np.asarray(w_uk, np.float64), c, optimize=True),
            np.einsum("jc,hcv->hjv", c, np.asarray(w_uv, np.float64), optimize=True))


def extend_expanded(q_nope, q_rope, kv_bits, block_table, seqlens, w_uk, w_uv, scale, page_size=64,
                    d_c=512, round_kv=False):
    """Extend (prefill continuation) by path one ("Two equivalent paths"; section "Which is
    faster: count new tokens and cached tokens"): the s_q new tokens of sequence b are the last
    s_q of its L_b cached rows; query t attends, per head, to keys j <= L_b - s_q + t with key
    [k^N_j, k^R_j] (k^R_j stored in the cache row after the latent) and value v_j, score
    scale * (q^N . k^N_j + q^R . k^R_j).  Plain two-pass softmax in float64.
    round_kv: hold k^N and v as bf16 (the model's activation type) before attending.
    q_nope [B, s_q, H, d_nope], q_rope [B, s_q, H, d_r] float64; kv_bits uint16 bf16 pages
    -> out [B, s_q, H, d_v], lse [B, s_q, H] (natural log of the sum of exp(score))."""
    q_nope = np.asarray(q_nope, np.float64)
    q_rope = np.asarray(q_rope, np.float64)
    B, s_q, H, _ = q_nope.shape
    d_v = np.asarray(w_uv).shape[-1]
    out = np.zeros((B, s_q, H, d_v))
    lse = np.full((B, s_q, H), -np.inf)
    for b in range(B):
        L = int(seqlens[b])
        rows = cache_rows(kv_bits, block_table, b, L, page_size)
        kn, v = expand_kv(rows[:, :d_c], w_uk, w_uv)
        if round_kv:
            kn, v = round_bf16(kn), round_bf16(v)
        s = scale * (np.einsum("thn,hjn->thj", q_nope[b], kn, optimize=True) +
                     np.einsum("thr,jr->thj", q_rope[b], rows[:, d_c:], optimize=True))
        hidden = np.arange(L)[None, :] > (L - s_q + np.arange(s_q))[:, None]      # [s_q, L]
        s[np.broadcast_to(hidden[:, None, :], s.shape)] = -np.inf
        m = s.max(axis=-1, keepdims=True)
        e = np.exp(s - m)
        l = e.sum(axis=-1)
        out[b] = np.einsum("thj,hjv->thv", e / l[..., None], v, optimize=True)
        lse[b] = m[..., 0] + np.log(l)
    return out, lse
