"""GB300-native paged MLA decode with decode-context-parallel (DCP) shards.

Thin PyTorch-facing wrappers over the C ABI of ``libmla_decode.so``:

  mla_decode             one shard's partial attention (out, lse) for q_len-row query
                         blocks, causal or not, any round-robin interleave
  mla_decode_shards      every emulated shard of a step in one launch
  lse_merge              merge shard partials through their LSEs
  cp_local_slot          global position -> this rank's KV slot (PAD_SLOT_ID = -1 otherwise)
  cp_local_slot_scatter  write new KV rows into this rank's pool at those slots

PyTorch provides device memory and the current stream; every step of the computation
runs in the library's CUDA kernels.  All tensors must live on the current CUDA device.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from . import _lib
from ._lib import PAD_SLOT_ID, MlaError  # noqa: F401

D_QK = 576
D_V = 512

__all__ = ["mla_decode", "mla_decode_shards", "lse_merge", "cp_local_slot",
           "cp_local_slot_scatter", "workspace_size", "device_status", "set_decode_kernel",
           "set_rescale_budget", "set_wait_limit_ns", "PAD_SLOT_ID", "MlaError", "D_QK", "D_V"]


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _need(t: torch.Tensor, name: str, dtype, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def workspace_size(B: int, H: int, q_len: int, device=None) -> int:
    """Workspace bytes mla_decode can use for split-KV on ``device``."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    return int(_lib.load().mla_decode_workspace_size(B, H, q_len, sms))


def alloc_workspace(B: int, H: int, q_len: int, device=None) -> torch.Tensor:
    n = workspace_size(B, H, q_len, device)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=dev)


def mla_decode(q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
               seq_lens: torch.Tensor, causal_seqlens_global: Optional[torch.Tensor],
               q_len: int, cp_world: int, cp_rank: int, scale: float,
               out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
               lse_base_e: bool = True, workspace: Optional[torch.Tensor] = None,
               return_lse: bool = True, stream=None, causal: bool = True,
               interleave: int = 1) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """One shard's partial MLA decode.

    q [B, q_len, H, 576] (or [B*q_len, H, 576]) bf16; kv_cache [num_blocks, block_size,
    576] bf16; block_table [B, max_blocks] int32 (row stride may exceed max_blocks);
    seq_lens [B] int32 shard-local counts; causal_seqlens_global [B] int32 global
    lengths (None when cp_world == 1 or the block is non-causal).  ``causal`` False: every
    query row reads the shard's whole local sequence.  ``interleave``: the KV is dealt to
    the ranks in round-robin segments of that many positions.  Returns out [B*q_len, H,
    512] bf16 and lse [B*q_len, H] float32 (natural log, or log2 when lse_base_e is False).
    """
    if q.dim() == 3:
        q = q.view(-1, q_len, q.shape[1], q.shape[2])
    _need(q, "q", torch.bfloat16, 4)
    B, ql, H, D = q.shape
    if ql != q_len or D != D_QK:
        raise ValueError(f"q must be [B, q_len={q_len}, H, {D_QK}], got {tuple(q.shape)}")
    _need(kv_cache, "kv_cache", torch.bfloat16, 3)
    if kv_cache.shape[2] != D_QK:
        raise ValueError("kv_cache must be [num_blocks, block_size, 576]")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or not block_table.is_cuda:
        raise TypeError("block_table must be a 2-D int32 CUDA tensor")
    if block_table.stride(1) != 1:
        raise ValueError("block_table rows must be contiguous")
    _need(seq_lens, "seq_lens", torch.int32, 1)
    if causal_seqlens_global is not None:
        _need(causal_seqlens_global, "causal_seqlens_global", torch.int32, 1)
    if out is None:
        out = torch.empty(B * q_len, H, D_V, dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16)
    if lse is None and return_lse:
        lse = torch.empty(B * q_len, H, dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32)
    if workspace is None:
        workspace = alloc_workspace(B, H, q_len, q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    L = _lib.load()
    rc = L.mla_decode(q.data_ptr(), kv_cache.data_ptr(), block_table.data_ptr(),
                      block_table.stride(0), seq_lens.data_ptr(), _ptr(causal_seqlens_global),
                      B, H, q_len, 1 if causal else 0, kv_cache.shape[1], kv_cache.shape[0],
                      block_table.shape[1], cp_world, cp_rank, int(interleave), float(scale),
                      out.data_ptr(), _ptr(lse), 1 if lse_base_e else 0, workspace.data_ptr(),
                      ws_bytes, _stream(stream))
    _lib.check(rc)
    return out, lse


def mla_decode_shards(q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
                      seq_lens: torch.Tensor, causal_seqlens_global: Optional[torch.Tensor],
                      q_len: int, n_shards: int, scale: float,
                      out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                      lse_base_e: bool = True, workspace: Optional[torch.Tensor] = None,
                      stream=None, causal: bool = True,
                      interleave: int = 1) -> Tuple[torch.Tensor, torch.Tensor]:
    """Every shard of an emulated context-parallel step in one launch: the result equals
    ``mla_decode`` of shard r (rank r of cp_world = n_shards) for each r.

    q [B, q_len, H, 576] bf16; kv_cache [num_blocks, block_size, 576] bf16 holding all
    shards' pages; block_table [n_shards*B, max_blocks] int32, shard-major, page ids into
    kv_cache; seq_lens [n_shards*B] int32 shard-major; causal_seqlens_global [B] int32.
    Returns out [n_shards, B*q_len, H, 512] bf16 and lse [n_shards, B*q_len, H] float32.
    """
    if q.dim() == 3:
        q = q.view(-1, q_len, q.shape[1], q.shape[2])
    _need(q, "q", torch.bfloat16, 4)
    B, ql, H, D = q.shape
    if ql != q_len or D != D_QK:
        raise ValueError(f"q must be [B, q_len={q_len}, H, {D_QK}], got {tuple(q.shape)}")
    _need(kv_cache, "kv_cache", torch.bfloat16, 3)
    if kv_cache.shape[2] != D_QK:
        raise ValueError("kv_cache must be [num_blocks, block_size, 576]")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or not block_table.is_cuda:
        raise TypeError("block_table must be a 2-D int32 CUDA tensor")
    if block_table.stride(1) != 1 or block_table.shape[0] != n_shards * B:
        raise ValueError("block_table must be [n_shards*B, max_blocks] with contiguous rows")
    _need(seq_lens, "seq_lens", torch.int32, 1)
    if seq_lens.shape[0] != n_shards * B:
        raise ValueError("seq_lens must be [n_shards*B]")
    if causal_seqlens_global is not None:
        _need(causal_seqlens_global, "causal_seqlens_global", torch.int32, 1)
    if out is None:
        out = torch.empty(n_shards, B * q_len, H, D_V, dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16)
    if lse is None:
        lse = torch.empty(n_shards, B * q_len, H, dtype=torch.float32, device=q.device)
    _need(lse, "lse", torch.float32)
    if workspace is None:
        workspace = alloc_workspace(n_shards * B, H, q_len, q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    L = _lib.load()
    rc = L.mla_decode_shards(q.data_ptr(), kv_cache.data_ptr(), block_table.data_ptr(),
                             block_table.stride(0), seq_lens.data_ptr(),
                             _ptr(causal_seqlens_global), B, H, q_len, 1 if causal else 0,
                             kv_cache.shape[1], kv_cache.shape[0], block_table.shape[1],
                             n_shards, int(interleave), float(scale), out.data_ptr(),
                             lse.data_ptr(), 1 if lse_base_e else 0, workspace.data_ptr(),
                             ws_bytes, _stream(stream))
    _lib.check(rc)
    return out, lse


def lse_merge(partials: torch.Tensor, lses: torch.Tensor, out: Optional[torch.Tensor] = None,
              out_lse: Optional[torch.Tensor] = None, lse_base_e: bool = True,
              stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Merge partials [n, T, H, 512] (bf16 or float32) with lses [n, T, H] float32 into
    out [T, H, 512] bf16 (and out_lse [T, H] float32 when given)."""
    if partials.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("partials must be bf16 or float32")
    _need(partials, "partials", partials.dtype, 4)
    n, T, H, Dv = partials.shape
    if Dv != D_V:
        raise ValueError("partials must be [n, T, H, 512]")
    _need(lses, "lses", torch.float32, 3)
    if tuple(lses.shape) != (n, T, H):
        raise ValueError("lses must be [n, T, H]")
    if out is None:
        out = torch.empty(T, H, D_V, dtype=torch.bfloat16, device=partials.device)
    _need(out, "out", torch.bfloat16)
    if out_lse is not None:
        _need(out_lse, "out_lse", torch.float32)
    rc = _lib.load().lse_merge(partials.data_ptr(), 1 if partials.dtype == torch.float32 else 0,
                               lses.data_ptr(), n, T, H, out.data_ptr(), _ptr(out_lse),
                               1 if lse_base_e else 0, _stream(stream))
    _lib.check(rc)
    return out, out_lse


def cp_local_slot(positions: torch.Tensor, block_table: torch.Tensor, block_size: int,
                  cp_size: int, cp_rank: int, interleave: int = 1,
                  slots: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Slots int64 [B, N] of positions int64 [B, N] (negative = rejected) on rank
    ``cp_rank``; PAD_SLOT_ID where this rank does not own the position."""
    if positions.dim() == 1:
        positions = positions.view(1, -1)
    _need(positions, "positions", torch.int64, 2)
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or not block_table.is_cuda:
        raise TypeError("block_table must be a 2-D int32 CUDA tensor")
    if block_table.stride(1) != 1:
        raise ValueError("block_table rows must be contiguous")
    B, N = positions.shape
    if block_table.shape[0] != B:
        raise ValueError("block_table must have one row per positions row")
    if slots is None:
        slots = torch.empty_like(positions)
    _need(slots, "slots", torch.int64, 2)
    rc = _lib.load().cp_local_slot(positions.data_ptr(), block_table.data_ptr(),
                                   block_table.stride(0), block_table.shape[1], B, N,
                                   block_size, cp_size, cp_rank, interleave, slots.data_ptr(),
                                   _stream(stream))
    _lib.check(rc)
    return slots


def cp_local_slot_scatter(positions: torch.Tensor, kv_new: torch.Tensor,
                          block_table: torch.Tensor, kv_cache: torch.Tensor, cp_size: int,
                          cp_rank: int, interleave: int = 1,
                          slots: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Writes kv_new [B, N, 576] bf16 into kv_cache [num_blocks, block_size, 576] at the
    slots ``cp_local_slot`` gives positions [B, N] on rank ``cp_rank``; positions the rank
    does not own (and negative ones) write nothing.  Returns kv_cache."""
    if positions.dim() == 1:
        positions = positions.view(1, -1)
    _need(positions, "positions", torch.int64, 2)
    B, N = positions.shape
    _need(kv_new, "kv_new", torch.bfloat16, 3)
    if tuple(kv_new.shape) != (B, N, D_QK):
        raise ValueError(f"kv_new must be [B, N, {D_QK}], got {tuple(kv_new.shape)}")
    _need(kv_cache, "kv_cache", torch.bfloat16, 3)
    if kv_cache.shape[2] != D_QK:
        raise ValueError("kv_cache must be [num_blocks, block_size, 576]")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or not block_table.is_cuda:
        raise TypeError("block_table must be a 2-D int32 CUDA tensor")
    if block_table.stride(1) != 1 or block_table.shape[0] != B:
        raise ValueError("block_table must have one contiguous row per positions row")
    if slots is not None:
        _need(slots, "slots", torch.int64, 2)
    rc = _lib.load().cp_local_slot_scatter(
        positions.data_ptr(), kv_new.data_ptr(), block_table.data_ptr(), block_table.stride(0),
        block_table.shape[1], B, N, kv_cache.shape[1], cp_size, cp_rank, interleave,
        kv_cache.data_ptr(), kv_cache.shape[0], _ptr(slots), _stream(stream))
    _lib.check(rc)
    return kv_cache


KERNEL_AUTO, KERNEL_MMA, KERNEL_TC = 0, 1, 2
BUDGET_AUTO, BUDGET_NARROW, BUDGET_WIDE = 0, 1, 2


def set_decode_kernel(choice: int) -> int:
    """0 = automatic, 1 = warp-level mma.sync kernel, 2 = tcgen05 kernel where it applies.
    Returns the previous choice."""
    rc = _lib.load().mla_set_decode_kernel(int(choice))
    if rc < 0:
        _lib.check(rc)
    return rc


def set_rescale_budget(choice: int) -> int:
    """Lazy-rescale budget of the tcgen05 kernel: 0 = per call, 1 = narrow, 2 = wide.
    Returns the previous choice."""
    rc = _lib.load().mla_set_rescale_budget(int(choice))
    if rc < 0:
        _lib.check(rc)
    return rc


def set_wait_limit_ns(ns: int) -> int:
    """Limit of every bounded on-chip wait of later launches (0 = default, 2 s).  Returns
    the previous setting."""
    rc = _lib.load().mla_set_wait_limit_ns(int(ns))
    if rc < 0:
        _lib.check(int(rc))
    return int(rc)


def set_test_stall(on: bool) -> int:
    """Tests of the timeout path only: make later decode launches wait for an arrival that
    never comes (the wait runs out after the wait limit).  Returns the previous setting."""
    rc = _lib.load().mla_set_test_stall(1 if on else 0)
    if rc < 0:
        _lib.check(rc)
    return rc


def device_status(stream=None) -> int:
    """Waits for the stream, returns and clears the device status bits (0 = clean)."""
    bits = ctypes.c_uint32(0)
    rc = _lib.load().mla_get_device_status(_stream(stream), ctypes.byref(bits))
    if rc not in (_lib.MLA_OK, _lib.MLA_ERR_DEVICE):
        _lib.check(rc)
    return int(bits.value)
