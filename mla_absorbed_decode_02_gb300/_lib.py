"""ctypes binding of libmla_decode.so (names mirror include/mla_decode.h).

Argument marshalling only: tensors go in as raw device pointers, the stream as
the CUDA stream handle.  Every step of the decode runs in the library's
kernels; there is no fallback path -- if the library is missing, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

(MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA, MLA_ERR_TIMEOUT, MLA_ERR_WORKSPACE,
 MLA_ERR_SCRATCH_LIMIT) = range(7)
MLA_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024
MLA_KV_BF16, MLA_KV_FP8_E4M3 = 0, 1
MLA_OUT_BF16, MLA_OUT_F32 = 0, 1
SCHED_MAGIC = 0x4D4C4131

_PKG = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return os.path.join(_PKG, "libmla_decode.so")


class MlaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_status_name(status)} ({status})")


class MlaDecodeParams(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("s_q", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32), ("causal", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("num_units", ctypes.c_int32), ("timeout_us", ctypes.c_int32),
                ("token_group", ctypes.c_int32), ("qk_fp8", ctypes.c_int32), ("reserved", ctypes.c_int32 * 3)]

    @classmethod
    def make(cls, batch, s_q, num_heads, num_pages, max_pages_per_seq, causal=True, kv_dtype=MLA_KV_BF16,
             out_dtype=MLA_OUT_BF16, num_units=0, timeout_us=0, page_size=64, token_group=0, qk_fp8=0):
        return cls(batch, s_q, num_heads, num_pages, page_size, max_pages_per_seq, int(bool(causal)), kv_dtype,
                   out_dtype, num_units, timeout_us, token_group, int(qk_fp8))


class MlaExtendParams(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("s_q", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("d_nope", ctypes.c_int32), ("d_v", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32), ("max_seqlen", ctypes.c_int32),
                ("chunk_tokens", ctypes.c_int32), ("timeout_us", ctypes.c_int32), ("reserved", ctypes.c_int32 * 5)]

    @classmethod
    def make(cls, batch, s_q, num_heads, num_pages, max_pages_per_seq, max_seqlen, chunk_tokens=4096, d_nope=128,
             d_v=128, timeout_us=0, page_size=64):
        return cls(batch, s_q, num_heads, d_nope, d_v, num_pages, page_size, max_pages_per_seq, max_seqlen,
                   chunk_tokens, timeout_us)


def load_library():
    """Load the built library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it with mla_absorbed_decode_02_gb300.build.build()")
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER(MlaDecodeParams)
        X = ctypes.POINTER(MlaExtendParams)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        sig = {
            "mla_get_workspace_size": ([P, ctypes.POINTER(sz), ctypes.POINTER(sz)], i32),
            "mla_get_scheduler_metadata": ([P, vp, vp, vp], i32),
            "mla_decode": ([P, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp], i32),
            "mla_decode_splitkv": ([P, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp], i32),
            "mla_combine": ([P, vp, vp, vp, vp, vp], i32),
            "mla_plan_host": ([P, i32, vp, vp], i32),
            "mla_resolve_num_units": ([P, ctypes.POINTER(i32)], i32),
            "mla_device_error": ([ctypes.POINTER(i32), i32], i32),
            "mla_wait_selftest": ([i32, vp], i32),
            "mla_decode_noalloc": ([P, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp], i32),
            "mla_quantize_kv_fp8": ([vp, vp, ctypes.c_int64, vp], i32),
            "mla_quantize_q_fp8": ([vp, vp, vp, ctypes.c_int64, vp], i32),
            "mla_absorb_query": ([i32, i32, i32, vp, vp, vp, vp], i32),
            "mla_project_output": ([i32, i32, i32, vp, vp, vp, vp], i32),
            "mla_extend_workspace_size": ([X, ctypes.POINTER(sz)], i32),
            "mla_expand_kv": ([X, vp, vp, vp, vp, vp, i32, vp, vp, vp], i32),
            "mla_extend": ([X, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp], i32),
            "mla_status_string": ([i32], ctypes.c_char_p),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
        return lib


def _status_name(status: int) -> str:
    names = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_CUDA",
             4: "MLA_ERR_TIMEOUT", 5: "MLA_ERR_WORKSPACE", 6: "MLA_ERR_SCRATCH_LIMIT"}
    return names.get(status, "MLA_ERR_UNKNOWN")


def _check(status: int, what: str):
    if status != MLA_OK:
        raise MlaError(status, what)


def _ptr(t) -> int:
    if t is None:
        return 0
    return int(t.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    return int(getattr(stream, "cuda_stream", stream))


def mla_status_string(status: int) -> str:
    return load_library().mla_status_string(status).decode()


def mla_get_workspace_size(p: MlaDecodeParams):
    sb, wb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load_library().mla_get_workspace_size(ctypes.byref(p), ctypes.byref(sb), ctypes.byref(wb)),
           "mla_get_workspace_size")
    return sb.value, wb.value


def mla_resolve_num_units(p: MlaDecodeParams) -> int:
    u = ctypes.c_int32()
    _check(load_library().mla_resolve_num_units(ctypes.byref(p), ctypes.byref(u)), "mla_resolve_num_units")
    return u.value


def mla_plan_host(p: MlaDecodeParams, num_units: int, cache_seqlens) -> np.ndarray:
    """Host twin of the split planner; returns the int32 metadata array."""
    seq = np.ascontiguousarray(cache_seqlens, dtype=np.int32)
    nqb = p.batch * p.s_q
    out = np.zeros(8 + 8 * num_units + 2 * nqb, np.int32)
    _check(load_library().mla_plan_host(ctypes.byref(p), num_units, seq.ctypes.data, out.ctypes.data),
           "mla_plan_host")
    return out


def mla_get_scheduler_metadata(p: MlaDecodeParams, cache_seqlens, sched, stream=None):
    _check(load_library().mla_get_scheduler_metadata(ctypes.byref(p), _ptr(cache_seqlens), _ptr(sched),
                                                     _stream(stream)), "mla_get_scheduler_metadata")


def mla_decode(p: MlaDecodeParams, q_nope_absorbed, q_rope, kv_pages, block_table, cache_seqlens, scale: float, out,
               lse, sched, workspace, stream=None):
    _check(load_library().mla_decode(ctypes.byref(p), _ptr(q_nope_absorbed), _ptr(q_rope), _ptr(kv_pages),
                                     _ptr(block_table), _ptr(cache_seqlens), float(scale), _ptr(out), _ptr(lse),
                                     _ptr(sched), _ptr(workspace), _stream(stream)), "mla_decode")


def mla_decode_splitkv(p: MlaDecodeParams, q_nope_absorbed, q_rope, kv_pages, block_table, cache_seqlens,
                       scale: float, out, lse, sched, workspace, stream=None):
    _check(load_library().mla_decode_splitkv(ctypes.byref(p), _ptr(q_nope_absorbed), _ptr(q_rope), _ptr(kv_pages),
                                             _ptr(block_table), _ptr(cache_seqlens), float(scale), _ptr(out),
                                             _ptr(lse), _ptr(sched), _ptr(workspace), _stream(stream)),
           "mla_decode_splitkv")


def mla_combine(p: MlaDecodeParams, out, lse, sched, workspace, stream=None):
    _check(load_library().mla_combine(ctypes.byref(p), _ptr(out), _ptr(lse), _ptr(sched), _ptr(workspace),
                                      _stream(stream)), "mla_combine")


def mla_decode_noalloc(p: MlaDecodeParams, q_nope_absorbed, q_rope, kv_pages, block_table, cache_seqlens,
                       scale: float, out, lse, stream=None):
    """Scheduler metadata + decode with the library's fixed device scratch array
    instead of caller buffers (for callers that cannot allocate device memory)."""
    _check(load_library().mla_decode_noalloc(ctypes.byref(p), _ptr(q_nope_absorbed), _ptr(q_rope), _ptr(kv_pages),
                                             _ptr(block_table), _ptr(cache_seqlens), float(scale), _ptr(out),
                                             _ptr(lse), _stream(stream)), "mla_decode_noalloc")


def mla_quantize_kv_fp8(kv_bf16, kv_fp8, num_tokens: int, stream=None):
    """bf16 cache rows [n, 576] -> 656-byte FP8 rows [n, 656] (codes, tile scales, RoPE)."""
    _check(load_library().mla_quantize_kv_fp8(_ptr(kv_bf16), _ptr(kv_fp8), int(num_tokens), _stream(stream)),
           "mla_quantize_kv_fp8")


def mla_quantize_q_fp8(q_nope_absorbed, q_rope, q_fp8, num_rows: int, stream=None):
    """Query rows for an FP8-QK decode: q~ bf16 [n, 512] and q^R bf16 [n, 64] -> 656-byte rows [n, 656]."""
    _check(load_library().mla_quantize_q_fp8(_ptr(q_nope_absorbed), _ptr(q_rope), _ptr(q_fp8), int(num_rows),
                                             _stream(stream)), "mla_quantize_q_fp8")


def mla_absorb_query(q_nope, w_uk, q_absorbed, stream=None):
    """q_absorbed[t, h] = q_nope[t, h] @ w_uk[h]: q_nope bf16 [..., H, d_nope], w_uk bf16 [H, d_nope, 512],
    q_absorbed bf16 [..., H, 512] (leading dims flattened to tokens)."""
    H, d_nope = int(q_nope.shape[-2]), int(q_nope.shape[-1])
    T = int(q_nope.numel() // (H * d_nope))
    _check(load_library().mla_absorb_query(T, H, d_nope, _ptr(q_nope), _ptr(w_uk), _ptr(q_absorbed), _stream(stream)),
           "mla_absorb_query")


def mla_project_output(o_latent, w_uv, out, stream=None):
    """out[t, h] = o_latent[t, h] @ w_uv[h]: o_latent bf16 [..., H, 512], w_uv bf16 [H, 512, d_v],
    out bf16 [..., H, d_v] (leading dims flattened to tokens)."""
    H = int(o_latent.shape[-2])
    T = int(o_latent.numel() // (H * 512))
    d_v = int(w_uv.shape[-1])
    _check(load_library().mla_project_output(T, H, d_v, _ptr(o_latent), _ptr(w_uv), _ptr(out), _stream(stream)),
           "mla_project_output")


def mla_extend_workspace_size(p: MlaExtendParams) -> int:
    n = ctypes.c_size_t()
    _check(load_library().mla_extend_workspace_size(ctypes.byref(p), ctypes.byref(n)), "mla_extend_workspace_size")
    return n.value


def mla_expand_kv(p: MlaExtendParams, kv_pages, block_table, cache_seqlens, w_uk, w_uv, chunk_start: int, k_nope, v,
                  stream=None):
    """k_nope[b, h, j] = w_uk[h] @ c_j and v[b, h, j] = c_j @ w_uv[h] for cache rows j of one chunk:
    k_nope, v bf16 [B, H, chunk_tokens, 128]."""
    _check(load_library().mla_expand_kv(ctypes.byref(p), _ptr(kv_pages), _ptr(block_table), _ptr(cache_seqlens),
                                        _ptr(w_uk), _ptr(w_uv), int(chunk_start), _ptr(k_nope), _ptr(v),
                                        _stream(stream)), "mla_expand_kv")


def mla_extend(p: MlaExtendParams, q_nope, q_rope, kv_pages, block_table, cache_seqlens, w_uk, w_uv, scale: float,
               out, lse, workspace, stream=None):
    """Extend by the expand path, chunk by chunk: out bf16 [B, s_q, H, 128], lse float32 [B, s_q, H]."""
    _check(load_library().mla_extend(ctypes.byref(p), _ptr(q_nope), _ptr(q_rope), _ptr(kv_pages), _ptr(block_table),
                                     _ptr(cache_seqlens), _ptr(w_uk), _ptr(w_uv), float(scale), _ptr(out), _ptr(lse),
                                     _ptr(workspace), _stream(stream)), "mla_extend")


def mla_device_error(clear: bool = True) -> int:
    w = ctypes.c_int32()
    _check(load_library().mla_device_error(ctypes.byref(w), int(clear)), "mla_device_error")
    return w.value


def mla_wait_selftest(timeout_us: int, stream=None):
    _check(load_library().mla_wait_selftest(int(timeout_us), _stream(stream)), "mla_wait_selftest")


class Decoder:
    """Convenience wrapper: owns the scheduler-metadata and workspace buffers
    (allocated once through torch) for one problem shape."""

    def __init__(self, p: MlaDecodeParams, device=None):
        import torch
        self.p = p
        self.device = torch.device("cuda" if device is None else device)
        sb, wb = mla_get_workspace_size(p)
        self.num_units = mla_resolve_num_units(p)
        self.sched = torch.empty(sb // 4, dtype=torch.int32, device=self.device)
        self.workspace = torch.empty(max(wb, 256) // 4, dtype=torch.float32, device=self.device)

    def plan(self, cache_seqlens, stream=None):
        mla_get_scheduler_metadata(self.p, cache_seqlens, self.sched, stream)

    def new_outputs(self):
        import torch
        p = self.p
        dt = torch.float32 if p.out_dtype == MLA_OUT_F32 else torch.bfloat16
        out = torch.empty((p.batch, p.s_q, p.num_heads, 512), dtype=dt, device=self.device)
        lse = torch.empty((p.batch, p.s_q, p.num_heads), dtype=torch.float32, device=self.device)
        return out, lse

    def decode(self, q_nope_absorbed, q_rope, kv_pages, block_table, cache_seqlens, scale, out=None, lse=None,
               stream=None):
        if out is None or lse is None:
            out, lse = self.new_outputs()
        mla_decode(self.p, q_nope_absorbed, q_rope, kv_pages, block_table, cache_seqlens, scale, out, lse,
                   self.sched, self.workspace, stream)
        return out, lse
