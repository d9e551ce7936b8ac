"""ctypes binding of libspecdec_verify.so: argument marshalling only.

Every function here passes device pointers (from torch CUDA tensors) or
host pointers (from pinned CPU tensors) straight to the C ABI declared in
include/specdec_verify.h; all arithmetic happens in the library's kernels.
If the library has not been built the import fails loudly: there is no
other implementation behind these names.
"""
from __future__ import annotations

import ctypes
import os
import re

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libspecdec_verify.so")
HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "specdec_verify.h")

SPECDEC_SAMPLE = 0
SPECDEC_GREEDY = 1
SPECDEC_BF16 = 0
SPECDEC_FP32 = 1
SPECDEC_MAX_GAMMA = 32
SPECDEC_MAX_TREE_NODES = 128

SPECDEC_OK = 0
SPECDEC_ERR_INVALID_ARG = -1
SPECDEC_ERR_UNSUPPORTED = -2
SPECDEC_ERR_WORKSPACE = -3
SPECDEC_ERR_CUDA = -4
SPECDEC_ERR_TIMEOUT = -5
SPECDEC_ERR_TOKEN_RANGE = -6

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_u64 = ctypes.c_uint64
_sz = ctypes.c_size_t

_CORE = [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _u64, _i, _vp, _vp, _vp, _sz, _vp]

_TREE = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _u64, _i, _vp, _vp, _vp, _vp, _sz, _vp]

_SIGNATURES = {
    "specdec_verify_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "specdec_verify": (_i, _CORE),
    "specdec_verify_debug": (_i, _CORE + [_vp] * 6),
    "specdec_verify_timed": (_i, _CORE + [_vp, _vp]),
    "specdec_verify_host_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "specdec_verify_host": (_i, _CORE),
    "specdec_read_status": (_i, [_vp, _vp, ctypes.POINTER(ctypes.c_int32)]),
    "specdec_philox_uniforms": (_i, [_u64, _i, _i, _i, _vp, _vp]),
    "specdec_status_string": (ctypes.c_char_p, [_i]),
    "specdec_verify_noalloc": (_i, _CORE[:14] + [_vp]),
    "specdec_selftest_wait_timeout": (_i, [_vp, _sz, _vp, ctypes.POINTER(ctypes.c_int32)]),
    "specdec_verify_tree_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "specdec_verify_tree": (_i, _TREE),
    "specdec_verify_tree_timed": (_i, _TREE + [_vp, _vp]),
    "specdec_verify_attention_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "specdec_verify_attention": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp, _vp,
                                      _sz, _vp]),
    "specdec_shard_record_bytes": (_sz, [_i, _i]),
    "specdec_shard_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "specdec_shard_score": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _vp,
                                 _sz, _vp]),
    "specdec_shard_accept": (_i, [_vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _u64, _i, _vp,
                                  _vp, _vp, _vp, _sz, _vp]),
    "specdec_shard_draw": (_i, [_vp, _i, _i, _vp, _i, _i, _i, _i, _i, _i, _f, _u64, _i, _vp, _vp,
                                _sz, _vp]),
    "specdec_cluster_head_workspace_size": (_sz, [_i, _i, _i, _i]),
    "specdec_cluster_head": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _u64, _i,
                                  _i, _vp, _vp, _vp, _vp, _sz, _vp]),
}

_lib = None


class SpecdecError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} ({code})")
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m target_model_verify_gb300.build` (nvcc, sm_103a)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/specdec_verify.h declares."""
    with open(HEADER, encoding="utf-8") as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(specdec_\w+)\s*\(", text)))


def status_string(code: int) -> str:
    return lib().specdec_status_string(int(code)).decode()


def _check(code: int, where: str) -> None:
    if code != SPECDEC_OK:
        raise SpecdecError(code, where)


# ------------------------------------------------------------ raw calls --

def specdec_verify_workspace_size(B, gamma, d, V, dtype, mode) -> int:
    return int(lib().specdec_verify_workspace_size(B, gamma, d, V, dtype, mode))


def specdec_verify_host_workspace_size(B, gamma, d, V, dtype, mode) -> int:
    return int(lib().specdec_verify_host_workspace_size(B, gamma, d, V, dtype, mode))


def specdec_verify(*args) -> int:
    return int(lib().specdec_verify(*args))


def specdec_verify_debug(*args) -> int:
    return int(lib().specdec_verify_debug(*args))


def specdec_verify_timed(*args) -> int:
    return int(lib().specdec_verify_timed(*args))


def specdec_verify_host(*args) -> int:
    return int(lib().specdec_verify_host(*args))


def specdec_verify_noalloc(*args) -> int:
    """The verify step with the library's static scratch (no workspace)."""
    return int(lib().specdec_verify_noalloc(*args))


def specdec_verify_tree_workspace_size(B, n_nodes, d, V, dtype, mode) -> int:
    return int(lib().specdec_verify_tree_workspace_size(B, n_nodes, d, V, dtype, mode))


def specdec_verify_tree(*args) -> int:
    """Tree verification (the parent array is a host int32 array)."""
    return int(lib().specdec_verify_tree(*args))


def specdec_verify_tree_timed(*args) -> int:
    return int(lib().specdec_verify_tree_timed(*args))


def specdec_verify_attention_workspace_size(B, n_new, Hq, Hkv, D, Lmax) -> int:
    return int(lib().specdec_verify_attention_workspace_size(B, n_new, Hq, Hkv, D, Lmax))


def specdec_verify_attention(*args) -> int:
    return int(lib().specdec_verify_attention(*args))


def specdec_cluster_head_workspace_size(M, n_c, top_k, max_cluster) -> int:
    return int(lib().specdec_cluster_head_workspace_size(M, n_c, top_k, max_cluster))


def specdec_cluster_head(*args) -> int:
    return int(lib().specdec_cluster_head(*args))


def specdec_shard_record_bytes(B, gamma) -> int:
    return int(lib().specdec_shard_record_bytes(B, gamma))


def specdec_shard_workspace_size(B, gamma, d, V_shard, mode) -> int:
    return int(lib().specdec_shard_workspace_size(B, gamma, d, V_shard, mode))


def specdec_shard_score(*args) -> int:
    return int(lib().specdec_shard_score(*args))


def specdec_shard_accept(*args) -> int:
    return int(lib().specdec_shard_accept(*args))


def specdec_shard_draw(*args) -> int:
    return int(lib().specdec_shard_draw(*args))


def specdec_read_status(workspace_ptr: int, stream_ptr: int) -> int:
    st = ctypes.c_int32(0)
    _check(lib().specdec_read_status(workspace_ptr, stream_ptr, ctypes.byref(st)),
           "specdec_read_status")
    return int(st.value)


def specdec_selftest_wait_timeout(workspace_ptr: int, workspace_bytes: int, stream_ptr: int) -> int:
    """Runs the bounded-wait self-test; returns the status word it left."""
    st = ctypes.c_int32(0)
    _check(lib().specdec_selftest_wait_timeout(workspace_ptr, workspace_bytes, stream_ptr,
                                               ctypes.byref(st)), "specdec_selftest_wait_timeout")
    return int(st.value)


def specdec_philox_uniforms(seed, B, n_pos, purpose, out_ptr, stream_ptr) -> int:
    return int(lib().specdec_philox_uniforms(seed, B, n_pos, purpose, out_ptr, stream_ptr))
