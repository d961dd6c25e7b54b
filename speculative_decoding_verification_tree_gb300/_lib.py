"""ctypes binding of libspecverify.so (include/specverify.h).

Argument marshalling only: every step of verification runs in the library's
CUDA kernels.  If the library is missing or fails to load, every call raises;
there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libspecverify.so")

SPEC_OK = 0
SPEC_ERR_ARG = -1
SPEC_ERR_DTYPE = -2
SPEC_ERR_SHAPE = -3
SPEC_ERR_CUDA = -4
SPEC_ERR_WORKSPACE = -5
SPEC_ERR_UNSUPPORTED = -6

SPEC_F32 = 0
SPEC_BF16 = 1
SPEC_DRAFT_LOGITS = 0
SPEC_DRAFT_PROBS = 1

SPEC_MAX_VOCAB = 1 << 24
SPEC_MAX_TOP_K = 128
SPEC_MAX_CHILDREN = 64
SPEC_MAX_TREE_NODES = 1024
SPEC_EAGLE2_MAX_TOPK = 32
SPEC_NOALLOC_MAX_ROWS = 8192
SPEC_NOALLOC_MAX_PARTS = 65536

SPEC_STATUS_NAN = 1
SPEC_STATUS_QZERO_ACCEPT = 2
SPEC_STATUS_RESIDUAL_ZERO = 4
SPEC_STATUS_DRAFT_EXHAUSTED = 8
SPEC_STATUS_CDF_FALLBACK = 16
SPEC_STATUS_BAD_TREE = 32
SPEC_STATUS_TOKEN_RANGE = 64
SPEC_STATUS_TIMEOUT = 128
SPEC_FLAG_TEST_STALL = 0x80000000

SPEC_OP_CHAIN = 1
SPEC_OP_TREE = 2
SPEC_OP_EAGLE2 = 3
SPEC_OP_LMHEAD = 4
SPEC_OP_TREE_LMHEAD = 5


class SpecParams(ctypes.Structure):
    """Mirror of spec_params_t (40 bytes)."""
    _fields_ = [
        ("temperature", ctypes.c_float),
        ("top_k", ctypes.c_int32),
        ("top_p", ctypes.c_float),
        ("draft_kind", ctypes.c_int32),
        ("seed", ctypes.c_uint64),
        ("philox_offset", ctypes.c_uint32),
        ("flags", ctypes.c_uint32),
        ("draft_lse", ctypes.c_void_p),
    ]


assert ctypes.sizeof(SpecParams) == 40

SPEC_STATS_MAX_BINS = 1024
STATS_FIELDS = ("len_hist", "node_tested", "node_accepted", "depth_tested",
                "depth_accepted", "calib_tested", "calib_accepted",
                "calib_conf_sum", "invalid")


class SpecAcceptStats(ctypes.Structure):
    """Mirror of spec_accept_stats_t (nine device pointers)."""
    _fields_ = [(f, ctypes.c_void_p) for f in STATS_FIELDS]

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t

_SIGNATURES = {
    "spec_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "spec_verify_chain": (_I, [_P, _P, _P, _I, _I, _I, _I, _I,
                               ctypes.POINTER(SpecParams), _P, _P, _P, _P,
                               _SZ, _P]),
    "spec_verify_tree": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                              ctypes.POINTER(SpecParams), _P, _P, _P, _P, _P,
                              _SZ, _P]),
    "spec_tree_mask": (_I, [_P, _I, _I, _P, _P, _P]),
    "spec_lm_head": (_I, [_P, _P, _I, _I, _I, ctypes.c_float, _P, _P, _P,
                          _SZ, _P]),
    "spec_verify_tree_lmhead": (_I, [_P, _P, _I, _P, _P, _P, _P, _I, _I, _I,
                                     _I, _I, ctypes.POINTER(SpecParams), _P,
                                     _P, _P, _P, _P, _P, _SZ, _P]),
    "spec_eagle2_expand_rerank": (_I, [_P, _I, _I, _I, _I, _I, _I, _I,
                                       ctypes.POINTER(SpecParams), _P, _P, _P,
                                       _P, _P, _P, _SZ, _P]),
    "spec_get_status": (_I, [_P, ctypes.POINTER(ctypes.c_uint32), _P]),
    "spec_philox_uniforms": (_I, [ctypes.c_uint64, ctypes.c_uint32, _P, _P,
                                  _P, _I, _P, _P]),
    "spec_error_string": (ctypes.c_char_p, [_I]),
    "spec_verify_chain_noalloc": (_I, [_P, _P, _P, _I, _I, _I, _I, _I,
                                       ctypes.POINTER(SpecParams), _P, _P, _P,
                                       _P]),
    "spec_get_status_noalloc": (_I, [ctypes.POINTER(ctypes.c_uint32), _P]),
    "spec_kv_commit": (_I, [_P, _I, _I, _I, ctypes.c_int64, ctypes.c_int64,
                            ctypes.c_int64, ctypes.c_int64, _I, _P, _P, _P, _I,
                            _P, _P]),
    "spec_accept_stats": (_I, [_P, _P, _P, _P, _I, _I, _I,
                               ctypes.POINTER(SpecAcceptStats), _P]),
    "spec_tree_attention": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                 ctypes.c_float, _P, _P]),
    "spec_profile_enable": (_I, [_I]),
    "spec_profile_read": (_I, [_I, ctypes.POINTER(ctypes.c_double),
                               ctypes.POINTER(ctypes.c_int)]),
}

SPEC_PROF_ARGMAX = 0
SPEC_PROF_VERIFY = 1
SPEC_PROF_EXPAND = 2
SPEC_PROF_KV = 3
SPEC_PROF_STATS = 4
SPEC_PROF_ATTN = 5
SPEC_PROF_LMHEAD = 6

EXPORTED = tuple(_SIGNATURES)

_lib = None


class SpecError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        msg = "unknown"
        if _lib is not None:
            msg = _lib.spec_error_string(code).decode()
        super().__init__(f"{fn} failed with {code} ({msg})")


def load(path: str = LIB_PATH):
    """Load (once) and return the library; raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA library not built: {path} is missing.  Run "
            "`python -c 'import __graft_entry__ as g; g.build()'` (or "
            "python -m speculative_decoding_verification_tree_gb300.build).")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def call(name: str, *args) -> int:
    """Call an entry point; raise SpecError on a non-zero return code."""
    rc = getattr(load(), name)(*args)
    if name not in ("spec_workspace_bytes", "spec_error_string") and rc != 0:
        raise SpecError(name, rc)
    return rc


def raw(name: str, *args):
    """Call an entry point and return its result unchecked (tests)."""
    return getattr(load(), name)(*args)
