"""ctypes view of ``libdynaspec.so`` (the C ABI in ``include/dynaspec.h``).

Loading fails loudly when the library has not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdynaspec.so")

P = ctypes.c_void_p
I = ctypes.c_int
I64 = ctypes.c_int64
U64 = ctypes.c_uint64
F = ctypes.c_float
SZ = ctypes.c_size_t
ST = ctypes.c_int32

# name -> (restype, argtypes); mirrors include/dynaspec.h
SIGNATURES = {
    "ds_status_string": (ctypes.c_char_p, [ST]),
    "ds_version": (I, []),
    "ds_vocab_index": (ST, [P, P, I, I, P, P, P, P]),
    "ds_router_workspace_bytes": (SZ, [I, I]),
    "ds_router_topk": (ST, [P, I, I, P, P, I, P, P, I, I, P, I, I, P, P, I, P, SZ, P, P]),
    "ds_router_create": (ST, [P, P, P, P, P, I, I, I, I, P, I]),
    "ds_router_destroy": (ST, [P]),
    "ds_router_workspace_bytes_h": (SZ, [P, I]),
    "ds_router_topk_h": (ST, [P, P, I, I, P, P, I, P, SZ, P, P]),
    "ds_router_topk_list_b1": (ST, [P, P, I, P, I, P, P, P, P, P, I64, I, P, SZ, P, P]),
    "ds_gathered_head_b1_table": (ST, [P, P, I, I, P, I, P, F, U64, I, P, P, P, P, P, I, P, SZ, P, P]),
    "ds_shortlist_workspace_bytes": (SZ, [I, I]),
    "ds_build_shortlist": (ST, [P, P, I, I, P, I, I, P, P, I64, P, P, P, P, P, SZ, P, P]),
    "ds_head_workspace_bytes": (SZ, [I]),
    "ds_gathered_head": (ST, [P, I, I, P, I, I, P, P, P, I, P, P, P, P, F, U64, I,
                              P, P, P, P, P, I, P, SZ, P, P]),
    "ds_gathered_head_noalloc": (ST, [P, I, I, P, I, I, P, P, P, I, P, P, P, P, F, U64, I,
                                      P, P, P, P, P, I, P, P]),
    "ds_prefetch_rows": (ST, [P, I, I, P, P, I, I, P]),
    "ds_verify_workspace_bytes": (SZ, [I, I, I]),
    "ds_verify": (ST, [P, I, I, I, F, P, I64, P, P, P, P, I, P, P, P, P, P, P, P, SZ, P, P]),
    "ds_verify_tree_workspace_bytes": (SZ, [I, I, I, I]),
    "ds_verify_tree": (ST, [P, I, I, I, I, F, P, P, I64, P, P, P, P, I64, P, I, P, P, P, P, P,
                            P, P, P, P, SZ, P, P]),
    "ds_workspace_bytes": (SZ, [I, I, I, I, I, I, I]),
    "ds_set_wait_budget": (ST, [I64]),
    "ds_kmeans_workspace_bytes": (SZ, [I, I, I]),
    "ds_kmeans_init": (ST, [P, I, I, P, I, P, P, P, P]),
    "ds_kmeans_step": (ST, [P, I, I, I, P, P, P, P, P, P, SZ, P, P]),
    "ds_drafter_standin_workspace_bytes": (SZ, [I, I]),
    "ds_drafter_standin": (ST, [P, P, I, P, P, P, P, P, I, I, P, F, P, P, SZ, P, P]),
    "ds_philox4x32_10": (ST, [P, U64, P, I, P]),
    "ds_event_record": (ST, [P, P]),
    "ds_copy": (ST, [P, P, SZ, P]),
}

_lib = None


class DynaSpecError(RuntimeError):
    pass


def load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python -c 'import dynamic_vocab_draft_gb300.build as b; b.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(status: int, what: str) -> None:
    if status != 0:
        msg = load().ds_status_string(status).decode()
        raise DynaSpecError(f"{what}: {msg} (status {status})")
