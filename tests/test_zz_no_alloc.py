"""mla_decode_noalloc against mla_decode, through the C ABI.

mla_decode_noalloc exists for callers that cannot allocate device memory on their decode
path -- a runtime whose memory is planned once at start-up, or a host program that links
only the C library and owns no allocator -- but still need split-KV scratch.  It uses a
fixed 64 MiB array inside the library instead of a caller workspace.  Here it must give
the same result as mla_decode with a caller workspace, within the parity tolerances,
on two calls in a row (the array keeps the previous call's contents) -- bit for bit when
that workspace is as large as the array (both then split the keys the same way), and
unlike a call with no workspace at all (which does not split them) -- and must reject a
problem whose scratch would not fit, after the argument checks mla_decode makes.

This file is named to be collected last, so that a run stopping at the first failure
has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import mla_paged_decode_03_gb300 as M
import synth
from mla_paged_decode_03_gb300 import _lib
from step_builder import step_from_workload

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-2
LSE_TOL = 1e-3


SCRATCH_BYTES = 64 << 20


def _noalloc(step, r, out, lse):
    L = _lib.load()
    pool = step.pools[r]
    rc = L.mla_decode_noalloc(
        step.q.data_ptr(), pool.data_ptr(), step.block_table.data_ptr(),
        step.block_table.stride(0), step.seq_lens[r].data_ptr(), step.gseq.data_ptr(),
        step.B, step.H, step.q_len, 1, pool.shape[1], pool.shape[0],
        step.block_table.shape[1], step.cp, r, 1, ctypes.c_float(step.scale), out.data_ptr(),
        lse.data_ptr(), 1 if step.lse_base_e else 0,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc


def _check_close(out, lse, out_ref, lse_ref):
    o = out.float().cpu().numpy()
    orf = out_ref.float().cpu().numpy()
    assert np.all(np.isfinite(o))
    assert float(np.abs(o - orf).max()) <= OUT_TOL
    l, lr = lse.cpu().numpy(), lse_ref.cpu().numpy()
    fin = np.isfinite(lr)
    assert np.array_equal(fin, np.isfinite(l))
    if fin.any():
        assert float(np.abs(l[fin] - lr[fin]).max()) <= LSE_TOL


@pytest.mark.parametrize("name,lengths", [("cp2", None), ("plain", [3000, 700, 4100])])
def test_noalloc_matches_mla_decode_twice(name, lengths):
    M.set_decode_kernel(M.KERNEL_AUTO)
    M.device_status()
    w = synth.make_workload(name, lengths=lengths)
    step = step_from_workload(w, "cuda")
    same_size = torch.empty(SCRATCH_BYTES, dtype=torch.uint8, device="cuda")
    for r in range(step.cp):
        out_ref, lse_ref = M.mla_decode(step.q, step.pools[r], step.block_table,
                                        step.seq_lens[r], step.gseq, step.q_len, step.cp, r,
                                        step.scale, lse_base_e=step.lse_base_e)
        out_ws, lse_ws = M.mla_decode(step.q, step.pools[r], step.block_table,
                                      step.seq_lens[r], step.gseq, step.q_len, step.cp, r,
                                      step.scale, lse_base_e=step.lse_base_e,
                                      workspace=same_size)
        out_none, _ = M.mla_decode(step.q, step.pools[r], step.block_table, step.seq_lens[r],
                                   step.gseq, step.q_len, step.cp, r, step.scale,
                                   lse_base_e=step.lse_base_e,
                                   workspace=torch.empty(0, dtype=torch.uint8, device="cuda"))
        for _ in range(2):                                   # two calls in a row
            out = torch.full_like(out_ref, float("nan"))
            lse = torch.full_like(lse_ref, float("nan"))
            rc = _noalloc(step, r, out, lse)
            assert rc == _lib.MLA_OK, _lib.load().mla_last_error()
            torch.cuda.synchronize()
            _check_close(out, lse, out_ref, lse_ref)
            assert torch.equal(out, out_ws) and torch.equal(lse, lse_ws)
        # the split schedule (and so the scratch) is in use: without any workspace the
        # keys are not split and some output rounds differently
        assert not torch.equal(out, out_none)
    assert M.device_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    # 4096 requests x 128 heads would need far more than 64 MiB of split-KV scratch;
    # the call is refused on the host and launches nothing (the pointers are never used).
    L = _lib.load()
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    p = dummy.data_ptr()
    rc = L.mla_decode_noalloc(p, p, p, 4, p, p, 4096, 128, 1, 1, 64, 4, 4, 1, 0, 1,
                              ctypes.c_float(0.1), p, p, 1, None)
    assert rc == _lib.MLA_ERR_UNSUPPORTED
    assert b"scratch" in L.mla_last_error()
    # a bad argument gets mla_decode's own error before the size is looked at
    rc = L.mla_decode_noalloc(p, p, p, 4, p, p, 4096, 128, 1000, 1, 64, 4, 4, 1, 0, 1,
                              ctypes.c_float(0.1), p, p, 1, None)
    assert rc == _lib.MLA_ERR_UNSUPPORTED and b"q_len" in L.mla_last_error()
    rc = L.mla_decode_noalloc(p, p, p, 4, p, p, 4096, 0, 1, 1, 64, 4, 4, 1, 0, 1,
                              ctypes.c_float(0.1), p, p, 1, None)
    assert rc == _lib.MLA_ERR_INVALID_ARGUMENT
