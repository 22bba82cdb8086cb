"""GB300 (sm_103a) weight-absorbed MLA decode.

The compute lives in ``libmla_decode.so`` (hand-written CUDA, C ABI declared in
``include/mla_decode.h``); ``_lib`` is a thin ctypes binding with the same names.
Importing this package does not load the library; the first call does, and it
raises if the library has not been built.
"""
from ._lib import (  # noqa: F401
    MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA, MLA_ERR_TIMEOUT, MLA_ERR_WORKSPACE,
    MLA_ERR_SCRATCH_LIMIT, MLA_KV_BF16, MLA_KV_FP8_E4M3, MLA_NOALLOC_SCRATCH_BYTES, MLA_OUT_BF16, MLA_OUT_F32,
    Decoder, MlaDecodeParams, MlaError, library_path, load_library, mla_absorb_query, mla_combine, mla_decode,
    mla_decode_noalloc, mla_project_output, MlaExtendParams, mla_expand_kv, mla_extend, mla_extend_workspace_size,
    mla_decode_splitkv, mla_device_error, mla_get_scheduler_metadata, mla_get_workspace_size, mla_plan_host,
    mla_quantize_kv_fp8, mla_quantize_q_fp8, mla_resolve_num_units, mla_status_string, mla_wait_selftest,
)
