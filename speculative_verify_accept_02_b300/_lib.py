"""Loads libisd.so (the C ABI declared under include/) with ctypes.

There is no fallback: if the library is missing or fails to load, every
entry point raises.
"""
import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(HERE, "libisd.so")

ISD_OK, ISD_ERR_INVALID_ARG, ISD_ERR_UNSUPPORTED, ISD_ERR_WORKSPACE, ISD_ERR_CUDA = range(5)
ISD_DTYPE_BF16, ISD_DTYPE_F32 = 0, 1

# KV commit status bits (ISD_KV_ERR_* of include/isd_kv.h).
ISD_KV_ERR_STATE, ISD_KV_ERR_ACCEPT, ISD_KV_ERR_SLOT, ISD_KV_ERR_POOL, ISD_KV_ERR_CAPACITY = 1, 2, 4, 8, 16
ISD_KV_MAX_SEQS = 1 << 24
ISD_FILTER_MAX_TOP_K = 64

# Every symbol the headers under include/ declare, with (restype, argtypes).
SIGNATURES = {
    "isd_verify_workspace_bytes": (C.c_size_t, [C.c_int, C.c_int, C.c_int, C.c_int]),
    "isd_verify": (C.c_int, [C.c_void_p, C.c_int64, C.c_void_p, C.c_int64, C.c_int, C.c_int,
                             C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_uint64,
                             C.c_uint64, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                             C.c_void_p, C.c_size_t, C.c_void_p]),
    "isd_verify_relaxed": (C.c_int, [C.c_void_p, C.c_int64, C.c_void_p, C.c_int64, C.c_int, C.c_int,
                                     C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_uint64,
                                     C.c_uint64, C.c_float, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                     C.c_void_p, C.c_size_t, C.c_void_p]),
    "isd_verify_propose_workspace_bytes": (C.c_size_t, [C.c_int, C.c_int, C.c_int, C.c_int]),
    "isd_verify_propose": (C.c_int, [C.c_void_p, C.c_int64, C.c_void_p, C.c_int64, C.c_int, C.c_int,
                                     C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_uint64,
                                     C.c_uint64, C.c_float, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                     C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p,
                                     C.c_void_p, C.c_size_t, C.c_void_p]),
    "isd_verify_propose_gumbel": (C.c_int, [C.c_void_p, C.c_int64, C.c_void_p, C.c_int64, C.c_int, C.c_int,
                                            C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_uint64,
                                            C.c_uint64, C.c_float, C.c_void_p, C.c_void_p, C.c_void_p,
                                            C.c_void_p, C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p,
                                            C.c_void_p, C.c_size_t, C.c_void_p]),
    "isd_propose_workspace_bytes": (C.c_size_t, [C.c_int, C.c_int, C.c_int, C.c_int]),
    "isd_propose": (C.c_int, [C.c_void_p, C.c_int64, C.c_int, C.c_int, C.c_void_p, C.c_int,
                              C.c_int, C.c_void_p, C.c_uint64, C.c_uint64, C.c_void_p,
                              C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    "isd_alpha": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p,
                            C.c_void_p]),
    "isd_status_string": (C.c_char_p, [C.c_int]),
    "isd_verify_filtered_workspace_bytes": (C.c_size_t, [C.c_int, C.c_int, C.c_int]),
    "isd_verify_filtered": (C.c_int, [C.c_void_p, C.c_int64, C.c_void_p, C.c_int64, C.c_int, C.c_int,
                                      C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_uint64,
                                      C.c_uint64, C.c_int, C.c_float, C.c_void_p, C.c_void_p, C.c_void_p,
                                      C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    "isd_propose_filtered_workspace_bytes": (C.c_size_t, [C.c_int, C.c_int, C.c_int]),
    "isd_propose_filtered": (C.c_int, [C.c_void_p, C.c_int64, C.c_int, C.c_int, C.c_void_p, C.c_int,
                                       C.c_int, C.c_void_p, C.c_uint64, C.c_uint64, C.c_int, C.c_float,
                                       C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    "isd_decision_uniforms": (C.c_int, [C.c_uint64, C.c_uint64, C.c_void_p, C.c_int, C.c_void_p, C.c_void_p]),
    "isd_debug_verify_stall": (C.c_int, [C.c_void_p, C.c_int64, C.c_void_p, C.c_int64, C.c_int, C.c_int,
                                         C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_uint64,
                                         C.c_uint64, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                         C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t,
                                         C.c_int, C.c_uint64, C.c_void_p]),
    "isd_kv_commit": (C.c_int, [C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                C.c_void_p, C.c_int, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p]),
    "isd_verify_noalloc": (C.c_int, [C.c_void_p, C.c_int64, C.c_void_p, C.c_int64, C.c_int, C.c_int,
                                     C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_uint64,
                                     C.c_uint64, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                     C.c_void_p]),
}

# Size of the library's built-in scratch array (ISD_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 8 << 20


class IsdError(RuntimeError):
    def __init__(self, fn, status, message):
        super().__init__(f"{fn} failed: {message} (status {status})")
        self.status = status


_lib = None


def load():
    """The loaded library (built in-tree by speculative_verify_accept_02_b300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIBRARY):
            raise ImportError(f"{LIBRARY} is missing; build it with "
                              "`python -m speculative_verify_accept_02_b300.build`")
        lib = C.CDLL(LIBRARY)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def check(fn, status):
    if status != ISD_OK:
        msg = load().isd_status_string(status).decode()
        raise IsdError(fn, status, msg)
