"""The C-ABI library without a GPU: it loads, exports every symbol the header declares,
and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import mla_paged_decode_03_gb300 as M
from mla_paged_decode_03_gb300 import _lib, build
from mla_paged_decode_03_gb300.dcp import local_seq_lens

import oracle.mla_ref as R

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(build.lib_path()):
        build.build()
    return _lib.load()


def header_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for fn in sorted(os.listdir(inc)):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(inc, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                            text, flags=re.M)
    return sorted(set(names))


def test_header_lists_the_entry_points():
    names = header_functions()
    for n in _lib.EXPORTED:
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_abi_version(lib):
    assert lib.mla_abi_version() >> 16 == 2


def _decode(lib, **kw):
    a = dict(q=16, kv=16, bt=16, bt_stride=4, seq=16, gseq=16, B=1, H=16, q_len=1, causal=1,
             bs=16, num_blocks=4, max_blocks=4, cp=1, rank=0, il=1, scale=0.1, out=16, lse=16,
             base_e=1, ws=None, ws_bytes=0)
    a.update(kw)
    return lib.mla_decode(a["q"], a["kv"], a["bt"], a["bt_stride"], a["seq"], a["gseq"], a["B"],
                          a["H"], a["q_len"], a["causal"], a["bs"], a["num_blocks"],
                          a["max_blocks"], a["cp"], a["rank"], a["il"], a["scale"], a["out"],
                          a["lse"], a["base_e"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(H=0), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(q_len=0), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(q_len=17), _lib.MLA_ERR_UNSUPPORTED),
    (dict(bs=0), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(num_blocks=0), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(max_blocks=5, bt_stride=4), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(cp=2, rank=2), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(cp=0), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(rank=-1), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(scale=float("nan")), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(scale=0.0), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(scale=-0.1), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(q=None), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(out=None), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(cp=2, gseq=None), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(q=24), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(seq=18), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(ws=272, ws_bytes=1024), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(il=0), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(il=3), _lib.MLA_ERR_INVALID_ARGUMENT),          # must divide block_size 16
    (dict(il=32), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(cp=2, gseq=None, causal=1), _lib.MLA_ERR_INVALID_ARGUMENT),
])
def test_decode_rejects(lib, kw, code):
    assert _decode(lib, **kw) == code
    assert lib.mla_last_error().decode()


def test_noncausal_decode_needs_no_global_lengths(lib):
    # accepted by validation: without a GPU the call fails only where it needs the device
    rc = _decode(lib, cp=2, rank=1, gseq=None, causal=0)
    assert rc != _lib.MLA_ERR_INVALID_ARGUMENT, lib.mla_last_error()


def _decode_shards(lib, **kw):
    a = dict(q=16, kv=16, bt=16, bt_stride=4, seq=16, gseq=16, B=1, H=16, q_len=1, causal=1,
             bs=16, num_blocks=4, max_blocks=4, n=2, il=1, scale=0.1, out=16, lse=16, base_e=1,
             ws=None, ws_bytes=0)
    a.update(kw)
    return lib.mla_decode_shards(a["q"], a["kv"], a["bt"], a["bt_stride"], a["seq"], a["gseq"],
                                 a["B"], a["H"], a["q_len"], a["causal"], a["bs"],
                                 a["num_blocks"], a["max_blocks"], a["n"], a["il"], a["scale"],
                                 a["out"], a["lse"], a["base_e"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(n=0), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(n=-3), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(gseq=None), _lib.MLA_ERR_INVALID_ARGUMENT),     # several shards need global lengths
    (dict(B=-1), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(q_len=17), _lib.MLA_ERR_UNSUPPORTED),
    (dict(max_blocks=5, bt_stride=4), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(scale=float("inf")), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(kv=None), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(out=24), _lib.MLA_ERR_INVALID_ARGUMENT),
    (dict(B=1 << 20, H=1 << 8, q_len=16, n=16), _lib.MLA_ERR_UNSUPPORTED),  # rows past 2^31
    (dict(B=20000, n=16), _lib.MLA_ERR_UNSUPPORTED),     # n * B^2 >= 2^32
    (dict(il=5), _lib.MLA_ERR_INVALID_ARGUMENT),
])
def test_decode_shards_rejects(lib, kw, code):
    assert _decode_shards(lib, **kw) == code
    assert lib.mla_last_error().decode().startswith("mla_decode_shards")


def test_decode_shards_empty_batch_is_noop(lib):
    assert _decode_shards(lib, B=0, q=None, out=None) == _lib.MLA_OK


def test_decode_empty_batch_is_noop(lib):
    assert _decode(lib, B=0, q=None, out=None) == _lib.MLA_OK


def test_merge_rejects(lib):
    E = _lib.MLA_ERR_INVALID_ARGUMENT
    assert lib.lse_merge(16, 0, 16, 0, 4, 4, 16, None, 1, None) == E
    assert lib.lse_merge(16, 0, 16, 2, -1, 4, 16, None, 1, None) == E
    assert lib.lse_merge(16, 0, 16, 2, 4, 0, 16, None, 1, None) == E
    assert lib.lse_merge(None, 0, 16, 2, 4, 4, 16, None, 1, None) == E
    assert lib.lse_merge(24, 0, 16, 2, 4, 4, 16, None, 1, None) == E
    assert lib.lse_merge(16, 0, 16, 2, 0, 4, 16, None, 1, None) == _lib.MLA_OK


def test_slot_rejects(lib):
    E = _lib.MLA_ERR_INVALID_ARGUMENT
    f = lib.cp_local_slot
    assert f(16, 16, 4, 4, 1, 8, 16, 2, 2, 1, 16, None) == E        # rank >= cp
    assert f(16, 16, 4, 4, 1, 8, 16, 0, 0, 1, 16, None) == E        # cp 0
    assert f(16, 16, 4, 4, 1, 8, 16, 2, 0, 3, 16, None) == E        # 16 % 3 != 0
    assert f(16, 16, 4, 5, 1, 8, 16, 2, 0, 1, 16, None) == E        # max_blocks > stride
    assert f(None, 16, 4, 4, 1, 8, 16, 2, 0, 1, 16, None) == E
    assert f(12, 16, 4, 4, 1, 8, 16, 2, 0, 1, 16, None) == E        # misaligned int64
    assert f(16, 16, 4, 4, 0, 8, 16, 2, 0, 1, 16, None) == _lib.MLA_OK
    assert f(16, 16, 4, 4, 1 << 16, 1 << 16, 16, 2, 0, 1, 16, None) == _lib.MLA_ERR_UNSUPPORTED


def test_scatter_rejects(lib):
    E = _lib.MLA_ERR_INVALID_ARGUMENT
    f = lib.cp_local_slot_scatter
    # positions, kv_new, block_table, bt_stride, max_blocks, B, N, bs, cp, rank, il,
    # kv_cache, num_blocks, slots, stream
    ok = (16, 16, 16, 4, 4, 1, 8, 16, 2, 0, 1, 16, 4, None, None)

    def call(**kw):
        a = list(ok)
        names = ["pos", "new", "bt", "stride", "maxb", "B", "N", "bs", "cp", "rank", "il", "kv",
                 "nb", "slots", "stream"]
        for k, v in kw.items():
            a[names.index(k)] = v
        return f(*a)

    assert call(rank=2) == E
    assert call(il=3) == E
    assert call(nb=0) == E
    assert call(new=None) == E
    assert call(kv=None) == E
    assert call(new=24) == E                                        # 8-byte aligned only
    assert call(kv=40) == E
    assert call(slots=12) == E
    assert call(N=0) == _lib.MLA_OK


def test_workspace_size_is_pure(lib):
    assert lib.mla_decode_workspace_size(0, 128, 1, 152) == 0
    a = lib.mla_decode_workspace_size(64, 128, 1, 152)
    assert a == lib.mla_decode_workspace_size(64, 128, 1, 152)


def test_local_seq_lens_matches_oracle():
    G = torch.arange(0, 200)
    for cp in (1, 2, 3, 8, 16):
        for il in (1, 2):
            for rank in range(cp):
                got = local_seq_lens(G, cp, rank, il).numpy()
                want = R.ref_local_len(G.numpy(), cp, rank, il)
                assert np.array_equal(got, want)


def test_python_wrappers_refuse_cpu_tensors():
    q = torch.zeros(1, 1, 16, 576, dtype=torch.bfloat16)
    kv = torch.zeros(2, 16, 576, dtype=torch.bfloat16)
    bt = torch.zeros(1, 2, dtype=torch.int32)
    sl = torch.ones(1, dtype=torch.int32)
    with pytest.raises((ValueError, TypeError)):
        M.mla_decode(q, kv, bt, sl, None, 1, 1, 0, 0.1)
