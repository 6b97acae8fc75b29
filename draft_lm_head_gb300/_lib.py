"""ctypes loader of liblmhead.so and the raw C signatures (include/lmhead.h)."""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblmhead.so")

_c = ctypes
_P = _c.c_void_p
_I = _c.c_int
_I64 = _c.c_int64
_SZ = _c.c_size_t
_F = _c.c_float

# name -> (restype, argtypes); mirrors include/lmhead.h
SIGNATURES = {
    "lmhead_version": (_I, []),
    "lmhead_status_string": (_c.c_char_p, [_I]),
    "lmhead_candidate_count": (_I64, [_I, _I64, _I, _I]),
    "lmhead_workspace_size": (_SZ, [_I, _I64, _I, _I, _I, _I, _I]),
    "lmhead_project_u": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "lmhead_lowrank_score_topk": (_I, [_I, _P, _P, _P, _P, _I64, _I, _I, _I, _I, _I,
                                       _P, _P, _P, _SZ, _P]),
    "lmhead_gather_logits": (_I, [_P, _P, _P, _I64, _I, _I, _I, _P, _P]),
    "lmhead_candidate_softmax": (_I, [_P, _I, _I, _F, _P, _P]),
    "lmhead_two_stage": (_I, [_I, _P, _P, _P, _P, _P, _I64, _I, _I, _I, _I, _I, _F,
                              _P, _P, _P, _P, _SZ, _P]),
    "lmhead_two_stage_profiled": (_I, [_I, _P, _P, _P, _P, _P, _I64, _I, _I, _I, _I, _I, _F,
                                       _P, _P, _P, _P, _SZ, _P, _I, _P]),
    "lmhead_two_stage_launches": (_I, [_I, _I]),
    "lmhead_dense_head": (_I, [_P, _P, _I64, _I, _I, _F, _P, _P, _P]),
    "lmhead_pruned_head": (_I, [_P, _P, _I, _I, _I, _F, _P, _P, _P]),
    "lmhead_last_device_error": (_I, [_P]),
    "lmhead_debug_set_wait_cycles": (_I64, [_I64]),
    "lmhead_shard_workspace_size": (_SZ, [_I64, _I, _I, _I, _I, _I]),
    "lmhead_shard_two_stage": (_I, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I, _I, _I, _I, _I, _F,
                                    _P, _P, _P, _P, _SZ, _P]),
    "lmhead_shard_softmax": (_I, [_P, _I, _P, _I, _I, _F, _P, _P]),
    "lmhead_draft_select": (_I, [_P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]),
    "lmhead_verify_chain": (_I, [_P, _I64, _I, _I, _P, _P, _P, _I, _P, _P, _P, _P, _P]),
    "lmhead_cluster_candidate_count": (_I64, [_I64, _I, _I]),
    "lmhead_cluster_workspace_size": (_SZ, [_I64, _I, _I, _I, _I, _I]),
    "lmhead_cluster_two_stage": (_I, [_P, _P, _P, _P, _I64, _I, _I, _I, _I, _I, _F,
                                      _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "lmhead_two_stage_local_noalloc": (_I, [_P, _P, _P, _P, _P, _I64, _I, _I, _I, _I, _I, _F,
                                            _P, _P, _P, _P]),
}

_lib = None


class LmheadError(RuntimeError):
    """A negative lmhead_status returned by the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def load() -> ctypes.CDLL:
    """Load liblmhead.so once. There is no fallback: a missing library is an
    error (build it with draft_lm_head_gb300.build.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m draft_lm_head_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().lmhead_status_string(status).decode()


def check(status: int, where: str) -> None:
    if status != 0:
        raise LmheadError(status, where)
