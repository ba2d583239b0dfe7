"""ctypes binding of libmla_decode.so (C ABI in include/mla_decode.h).

Argument marshalling only: every computation happens in the library's CUDA kernels.
The library must have been built (``mla_paged_decode_03_gb300.build.build()``); there is
no fallback, and loading fails loudly when the shared object is missing.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

MLA_OK = 0
MLA_ERR_INVALID_ARGUMENT = -1
MLA_ERR_UNSUPPORTED = -2
MLA_ERR_CUDA = -3
MLA_ERR_DEVICE = -4
PAD_SLOT_ID = -1

EXPORTED = ("mla_decode_workspace_size", "mla_decode", "mla_decode_shards", "mla_decode_noalloc",
            "lse_merge", "cp_local_slot", "cp_local_slot_scatter",
            "mla_get_device_status", "mla_set_decode_kernel", "mla_set_rescale_budget",
            "mla_set_wait_limit_ns", "mla_set_test_stall", "mla_last_error",
            "mla_abi_version")

_lock = threading.Lock()
_lib = None


class MlaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


def lib_path() -> str:
    return _build.lib_path()


def load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if not os.path.exists(path):
            raise ImportError(
                f"{path} is missing: build it with mla_paged_decode_03_gb300.build.build() "
                "(there is no CPU or Python fallback)")
        lib = ctypes.CDLL(path)
        c_int, c_i64, c_sz, c_vp, c_f = (ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                                         ctypes.c_void_p, ctypes.c_float)
        lib.mla_decode_workspace_size.restype = c_sz
        lib.mla_decode_workspace_size.argtypes = [c_int, c_int, c_int, c_int]
        # q, kv_cache, block_table, bt_stride, seq_lens, causal_seqlens_global, B, H, q_len,
        # causal, block_size, num_blocks, max_blocks, cp_world | n_shards, cp_rank (not in
        # the shards call), interleave, scale, out, lse, lse_base_e, [workspace, bytes,]
        # stream
        head = [c_vp, c_vp, c_vp, c_i64, c_vp, c_vp, c_int, c_int, c_int, c_int, c_int, c_int,
                c_int]
        lib.mla_decode.restype = c_int
        lib.mla_decode.argtypes = head + [c_int, c_int, c_int, c_f, c_vp, c_vp, c_int, c_vp,
                                          c_sz, c_vp]
        lib.mla_decode_shards.restype = c_int
        lib.mla_decode_shards.argtypes = head + [c_int, c_int, c_f, c_vp, c_vp, c_int, c_vp,
                                                 c_sz, c_vp]
        lib.mla_decode_noalloc.restype = c_int
        lib.mla_decode_noalloc.argtypes = head + [c_int, c_int, c_int, c_f, c_vp, c_vp, c_int,
                                                  c_vp]
        lib.lse_merge.restype = c_int
        lib.lse_merge.argtypes = [c_vp, c_int, c_vp, c_int, c_int, c_int, c_vp, c_vp, c_int,
                                  c_vp]
        lib.cp_local_slot.restype = c_int
        lib.cp_local_slot.argtypes = [c_vp, c_vp, c_i64, c_int, c_int, c_int, c_int, c_int,
                                      c_int, c_int, c_vp, c_vp]
        lib.cp_local_slot_scatter.restype = c_int
        lib.cp_local_slot_scatter.argtypes = [c_vp, c_vp, c_vp, c_i64, c_int, c_int, c_int,
                                              c_int, c_int, c_int, c_int, c_vp, c_int, c_vp,
                                              c_vp]
        lib.mla_get_device_status.restype = c_int
        lib.mla_get_device_status.argtypes = [c_vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.mla_last_error.restype = ctypes.c_char_p
        lib.mla_last_error.argtypes = []
        lib.mla_set_decode_kernel.restype = c_int
        lib.mla_set_decode_kernel.argtypes = [c_int]
        lib.mla_set_rescale_budget.restype = c_int
        lib.mla_set_rescale_budget.argtypes = [c_int]
        lib.mla_set_wait_limit_ns.restype = c_i64
        lib.mla_set_wait_limit_ns.argtypes = [c_i64]
        lib.mla_set_test_stall.restype = c_int
        lib.mla_set_test_stall.argtypes = [c_int]
        lib.mla_abi_version.restype = c_int
        lib.mla_abi_version.argtypes = []
        _lib = lib
        return lib


def check(rc: int) -> None:
    if rc != MLA_OK:
        msg = load().mla_last_error().decode(errors="replace")
        raise MlaError(rc, msg)
