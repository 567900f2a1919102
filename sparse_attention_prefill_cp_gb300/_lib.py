"""ctypes declarations of libdsa_cp.so (include/dsa_cp.h).  Argument
marshalling only; every step of the path runs in the library's kernels."""
from __future__ import annotations

import ctypes as C
import os

from .build import LIB_PATH

c_stream = C.c_void_p
c_i32p = C.POINTER(C.c_int32)


class LocalMetadata(C.Structure):
    """dsa_cp_local_metadata: device pointers into one int32 buffer."""
    _fields_ = [
        ("scalars", C.c_void_p),
        ("local_query_start_loc", C.c_void_p),
        ("local_seq_lens", C.c_void_p),
        ("local_kv_start_loc", C.c_void_p),
        ("local_req_id", C.c_void_p),
        ("local_req_kv_base", C.c_void_p),
        ("local_token_pos", C.c_void_p),
        ("local_req_pos_base", C.c_void_p),
    ]


# name -> (restype, argtypes), the order of include/dsa_cp.h
SIGNATURES = {
    "dsa_cp_geometry": (C.c_int, [C.c_int32, C.c_int32, c_i32p, c_i32p]),
    "dsa_cp_metadata_sizes": (C.c_int, [C.c_int32, C.c_int32, C.c_int32, C.POINTER(C.c_size_t)]),
    "dsa_cp_metadata_bind": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.POINTER(LocalMetadata)]),
    "dsa_cp_build_local_metadata": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                              C.c_int, C.POINTER(LocalMetadata), c_stream]),
    "dsa_cp_build_local_metadata_compressed": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int32,
                                                         C.c_int32, C.c_int, C.c_int32, C.POINTER(LocalMetadata),
                                                         c_stream]),
    "dsa_cp_split": (C.c_int, [C.c_void_p, C.c_int64, C.c_int32, C.c_int32, C.c_int, C.c_int32, C.c_void_p,
                               c_stream]),
    "dsa_cp_rerange": (C.c_int, [C.c_void_p, C.c_int64, C.c_int32, C.c_int32, C.c_int, C.c_void_p, c_stream]),
    "dsa_cp_split_from_host": (C.c_int, [C.c_void_p, C.c_int64, C.c_int32, C.c_int32, C.c_int, C.c_int32,
                                         C.c_void_p, c_stream]),
    "dsa_cp_rerange_to_host": (C.c_int, [C.c_void_p, C.c_int64, C.c_int32, C.c_int32, C.c_int, C.c_int32,
                                         C.c_void_p, c_stream]),
    "dsa_cp_all_to_all_heads": (C.c_int, [C.c_void_p, C.c_int32, C.c_int64, C.c_int32, C.c_int32, C.c_int,
                                          C.c_void_p, c_stream]),
    "dsa_indexer_topk_workspace_size": (C.c_int, [C.c_int32, C.c_int32, C.c_int32, C.POINTER(C.c_size_t)]),
    "dsa_indexer_topk": (C.c_int, [C.POINTER(LocalMetadata), C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                                   C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                                   C.c_void_p, C.c_size_t, c_stream]),
    "dsa_indexer_topk_rows": (C.c_int, [C.POINTER(LocalMetadata), C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                        C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32,
                                        C.c_int32, C.c_int32, C.c_void_p, C.c_void_p, C.c_size_t, c_stream]),
    "dsa_indexer_topk_noalloc": (C.c_int, [C.POINTER(LocalMetadata), C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                                           C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                           C.c_void_p, c_stream]),
    "dsa_indexer_scores": (C.c_int, [C.POINTER(LocalMetadata), C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                                     C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                     C.c_void_p, c_stream]),
    "dsa_indexer_topk_fp8": (C.c_int, [C.POINTER(LocalMetadata), C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                                       C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                       C.c_void_p, C.c_void_p, C.c_size_t, c_stream]),
    "dsa_indexer_scores_fp8": (C.c_int, [C.POINTER(LocalMetadata), C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                                         C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                         C.c_int32, C.c_void_p, c_stream]),
    "dsa_sparse_attn_prefill": (C.c_int, [C.POINTER(LocalMetadata), C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                          C.c_int32, C.c_void_p, C.c_int32, C.c_void_p, C.c_float, C.c_int32,
                                          C.c_int32, C.c_int32, C.c_void_p, c_stream]),
    "dsa_sparse_attn_prefill_headsharded": (C.c_int, [C.POINTER(LocalMetadata), C.c_int32, C.c_int32, C.c_void_p,
                                                      C.c_void_p, C.c_int32, C.c_void_p, C.c_int32, C.c_void_p,
                                                      C.c_float, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                                      C.c_void_p, c_stream]),
    "dsa_sparse_attn_prefill_flat": (C.c_int, [C.POINTER(LocalMetadata), C.c_int32, C.c_int32, C.c_void_p, C.c_int32,
                                               C.c_void_p, C.c_int32, C.c_void_p, C.c_int32, C.c_void_p, C.c_float,
                                               C.c_int32, C.c_int32, C.c_int32, C.c_void_p, c_stream]),
    "dsa_sparse_attn_prefill_fp8kv": (C.c_int, [C.POINTER(LocalMetadata), C.c_int32, C.c_int32, C.c_void_p,
                                                C.c_int32, C.c_void_p, C.c_int32, C.c_void_p, C.c_int32, C.c_void_p,
                                                C.c_float, C.c_int32, C.c_int32, C.c_int32, C.c_void_p, c_stream]),
    "dsa_sparse_attn_prefill_rows": (C.c_int, [C.POINTER(LocalMetadata), C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                               C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_int32, C.c_void_p,
                                               C.c_int32, C.c_void_p, C.c_float, C.c_int32, C.c_int32, C.c_int32,
                                               C.c_void_p, c_stream]),
    "dsa_swa_index": (C.c_int, [C.POINTER(LocalMetadata), C.c_int32, C.c_int32, C.c_void_p, C.c_int32, C.c_void_p,
                                C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p, c_stream]),
    "dsa_sparse_attn_prefill_swa": (C.c_int, [C.POINTER(LocalMetadata), C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                              C.c_int32, C.c_void_p, C.c_int32, C.c_void_p, C.c_int32, C.c_void_p,
                                              C.c_int32, C.c_void_p, C.c_float, C.c_int32, C.c_int32, C.c_int32,
                                              C.c_void_p, c_stream]),
    "dsa_kv_fp8_row_bytes": (C.c_int, [C.c_int32, C.c_int32, C.POINTER(C.c_size_t)]),
    "dsa_kv_fp8_quantize": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_void_p, c_stream]),
    "dsa_kv_fp8_dequantize": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_void_p, c_stream]),
    "dsa_poll_device_error": (C.c_int, [c_stream]),
    "dsa_poll_device_error_detail": (C.c_int, [c_stream, c_i32p]),
    "dsa_status_string": (C.c_char_p, [C.c_int]),
    "dsa_last_cuda_error": (C.c_char_p, []),
    "dsa_abi_version": (C.c_int32, []),
}

STATUS = {
    0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_SHAPE", 3: "DSA_ERR_UNSUPPORTED",
    4: "DSA_ERR_WORKSPACE", 5: "DSA_ERR_CUDA", 6: "DSA_ERR_DEVICE_TIMEOUT", 7: "DSA_ERR_DEVICE_BOUNDS",
    8: "DSA_ERR_DEVICE_SEQ_LENS",
}

_LIB = None


def load(path: str | None = None) -> C.CDLL:
    """Load libdsa_cp.so (building it first if it is missing).  Raises if the
    library cannot be built or loaded: there is no fallback path."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or LIB_PATH
    if not os.path.exists(p):
        from .build import build
        build()
    lib = C.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _LIB = lib
    return lib


class DSAError(RuntimeError):
    def __init__(self, status: int, where: str, detail=None):
        lib = load()
        msg = lib.dsa_status_string(status).decode()
        if status == 5:
            msg += " -- " + lib.dsa_last_cuda_error().decode()
        if detail is not None:
            msg += f" (site {detail[0]}, detail {detail[1]}, block {detail[2]})"
        super().__init__(f"{where}: {msg}")
        self.status = status
        self.detail = detail


def check(status: int, where: str) -> None:
    if status != 0:
        raise DSAError(status, where)
