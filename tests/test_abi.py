"""The C-ABI library without a GPU: it loads, exports every symbol include/*.h
declares, and rejects bad arguments on the host before touching CUDA."""

import ctypes
import os
import re

import pytest

import mla_latent_kv_69_b300 as mla
from mla_latent_kv_69_b300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INVALID, UNSUPPORTED = _lib.MLA_ERR_INVALID_ARG, _lib.MLA_ERR_UNSUPPORTED
A = 0x10000          # a fake, 16-byte aligned "device" address (never dereferenced)
MIS = A + 4          # misaligned


def _declared():
    names = set()
    for f in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if f.endswith(".h"):
            hdr = open(os.path.join(ROOT, "include", f)).read()
            names.update(re.findall(r"MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", hdr))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    lib = _lib.get()
    names = _declared()
    assert names == sorted(_lib.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n
    assert lib.mla_abi_version() == 1


def test_status_strings():
    for s in range(7):
        assert _lib.status_string(s).startswith("MLA_")
    assert "unknown" in _lib.status_string(99)


def test_split_range_rule():
    # chunk = 64 * ceil(ceil(L/64)/S); splits are front-loaded, trailing ones may be empty
    assert mla.split_range(4096, 3, 0) == (0, 1408)
    assert mla.split_range(4096, 3, 2) == (2816, 4096)
    assert mla.split_range(100, 4, 0) == (0, 64)
    assert mla.split_range(100, 4, 1) == (64, 100)
    assert mla.split_range(100, 4, 3) == (100, 100)
    assert mla.split_range(0, 2, 1) == (0, 0)
    for L in (1, 63, 64, 65, 1000, 131072):
        for S in (1, 2, 5, 37):
            covered = []
            for s in range(S):
                a, b = mla.split_range(L, S, s)
                assert a <= b and (a == b or a % 64 == 0)
                covered.extend(range(a, b))
            assert covered == list(range(L))
    with pytest.raises(mla.MlaError):
        mla.split_range(10, 0, 0)
    with pytest.raises(mla.MlaError):
        mla.split_range(10, 2, 2)


def test_num_splits_range():
    for B, L, h in [(1, 256, 16), (32, 4096, 128), (4, 131072, 128), (64, 32768, 128), (128, 8192, 128)]:
        S = mla.num_splits(B, L, h)
        assert 1 <= S <= _lib.MLA_MAX_SPLITS
    assert mla.num_splits(4, 0, 128) == 1


def _cache(**kw):
    c = _lib.MlaCache()
    c.dtype, c.page_size, c.data, c.scales, c.block_table = 0, 0, A, None, None
    c.max_pages, c.reserved, c.seq_stride_tokens, c.num_rows = 0, 0, 4096, 32 * 4096
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _decode(c=None, **kw):
    args = dict(q_lat=A, seq_lens=A, B=32, n_h=128, max_len=4096, scale=0.07, S=2, o_part=A, lse_part=A,
                status=None)
    args.update(kw)
    c = _cache() if c is None else c
    return _lib.get().mla_decode_fwd(args["q_lat"], ctypes.byref(c), args["seq_lens"], args["B"], args["n_h"],
                                     args["max_len"], args["scale"], args["S"], args["o_part"], args["lse_part"],
                                     args["status"], None)


def test_decode_rejects_bad_arguments_on_host():
    assert _decode(q_lat=None) == INVALID
    assert _decode(q_lat=MIS) == INVALID
    assert _decode(o_part=None) == INVALID
    assert _decode(B=0) == INVALID
    assert _decode(n_h=96) == UNSUPPORTED
    assert _decode(n_h=0) == INVALID
    assert _decode(S=-1) == INVALID
    assert _decode(S=_lib.MLA_MAX_SPLITS + 1) == INVALID
    assert _decode(scale=0.0) == INVALID
    assert _decode(scale=float("nan")) == INVALID
    assert _decode(max_len=-1) == INVALID
    assert _decode(status=A + 2) == INVALID
    assert _decode(_cache(data=None)) == INVALID
    assert _decode(_cache(dtype=7)) == INVALID
    assert _decode(_cache(reserved=1)) == INVALID
    assert _decode(_cache(scales=A)) == INVALID                     # bf16 with scales
    assert _decode(_cache(dtype=1)) == INVALID                      # fp8 without scales
    assert _decode(_cache(dtype=1, scales=MIS)) == INVALID
    assert _decode(_cache(seq_stride_tokens=100)) == INVALID        # stride < max_seq_len
    assert _decode(_cache(num_rows=1000)) == INVALID                # rows do not cover the batch
    paged = dict(block_table=A, page_size=64, max_pages=64, num_rows=64 * 100)
    assert _decode(_cache(**{**paged, "page_size": 32})) == UNSUPPORTED
    assert _decode(_cache(**{**paged, "max_pages": 10})) == INVALID   # too few pages for max_seq_len
    assert _decode(_cache(**{**paged, "num_rows": 64 * 100 + 3})) == INVALID
    assert _decode(_cache(**{**paged, "block_table": MIS})) == INVALID


def test_other_calls_reject_bad_arguments_on_host():
    L = _lib.get()
    assert L.mla_absorb_q(None, A, A, 1, 128, 10000.0, A, None) == INVALID
    assert L.mla_absorb_q(A, A, A, 1, 128, 0.5, A, None) == INVALID
    assert L.mla_absorb_q(A, A, A, 1, 48, 10000.0, A, None) == UNSUPPORTED
    assert L.mla_absorb_q(A, MIS, A, 1, 128, 10000.0, A, None) == INVALID
    assert L.mla_combine(A, A, 1, 0, 128, A, None, None) == INVALID
    assert L.mla_combine(A, A, 0, 1, 128, A, None, None) == INVALID
    assert L.mla_combine(A, A, 1, 1, 128, None, None, None) == INVALID
    assert L.mla_up_v(A, A, 1, 100, A, None) == UNSUPPORTED
    assert L.mla_up_v(A, None, 1, 128, A, None) == INVALID
    assert L.mla_combine_up_v(A, A, 2, 0, 128, A, A, None, None, None) == INVALID
    assert L.mla_combine_up_v(A, A, 2, 257, 128, A, A, None, None, None) == INVALID
    assert L.mla_combine_up_v(A, A, 0, 3, 128, A, A, None, None, None) == INVALID
    assert L.mla_combine_up_v(A, A, 2, 3, 100, A, A, None, None, None) == UNSUPPORTED
    assert L.mla_combine_up_v(A, A, 2, 3, 128, None, A, None, None, None) == INVALID
    assert L.mla_combine_up_v(A, A, 2, 3, 128, A, None, None, None, None) == INVALID
    assert L.mla_combine_up_v(A, A, 2, 3, 128, A, A, MIS, None, None) == INVALID     # o_lat misaligned
    assert L.mla_combine_up_v(A, A, 2, 3, 128, A, A, None, A + 2, None) == INVALID   # lse misaligned
    assert L.mla_quantize_fp8(A, -1, A, A, None) == INVALID
    assert L.mla_quantize_fp8(MIS, 10, A, A, None) == INVALID
    assert L.mla_quantize_fp8(A, 0, A, A, None) == _lib.MLA_OK      # nothing to do
    assert L.mla_quantize_fp6(A, -1, A, A, None) == INVALID
    assert L.mla_quantize_fp6(MIS, 10, A, A, None) == INVALID
    assert L.mla_quantize_fp6(A, 10, None, A, None) == INVALID
    assert L.mla_quantize_fp6(A, 0, A, A, None) == _lib.MLA_OK      # nothing to do


def test_static_entry_rejects_oversize_before_any_launch():
    # 128 sequences x 256 splits x 128 heads of partials (~8.6 GB) exceed the fixed array
    c = _cache(num_rows=128 * 4096)
    rc = _lib.get().mla_decode_combine_static(A, ctypes.byref(c), A, 128, 128, 4096, 0.07, 256, A, A, None, None)
    assert rc == _lib.MLA_ERR_WORKSPACE
    assert _lib.get().mla_decode_combine_static(None, ctypes.byref(c), A, 32, 128, 4096, 0.07, 2, A, A, None,
                                                None) == INVALID


def test_binding_rejects_a_block_table_without_a_row_per_sequence():
    import torch

    import mla_latent_kv_69_b300 as mla

    data = torch.zeros(4, 64, 576, dtype=torch.bfloat16)
    ok = mla.Cache(data, None, torch.zeros(3, 2, dtype=torch.int32))
    mla._need_table_rows(ok, 3)
    with pytest.raises(ValueError):
        mla._need_table_rows(ok, 4)
    with pytest.raises(ValueError):
        mla._need_table_rows(mla.Cache(data, None, torch.zeros(6, dtype=torch.int32)), 3)


def test_tensors_on_two_devices_are_rejected():
    """Every tensor of a call must sit on one device: the library launches on the current
    device and would otherwise be handed a peer GPU's address."""
    from types import SimpleNamespace

    import torch

    d0 = SimpleNamespace(device=torch.device("cuda", 0))
    d1 = SimpleNamespace(device=torch.device("cuda", 1))
    assert mla._one_device(q_lat=d0, status=None, o_part=d0) == torch.device("cuda", 0)
    assert mla._one_device(x=d1) == torch.device("cuda", 1)
    with pytest.raises(ValueError, match="o_part"):
        mla._one_device(q_lat=d0, o_part=d1)
    with pytest.raises(ValueError, match="cache.block_table"):
        mla._one_device(q_lat=d1, **{"cache.data": d1, "cache.block_table": d0})


def test_stall_hook_rejects_bad_arguments_on_host():
    L = _lib.get()

    def stalled(c=None, status=A, wait_ns=2_000_000, **kw):
        c = _cache() if c is None else c
        return L.mla_test_decode_stalled(A, ctypes.byref(c), A, kw.get("B", 32), 128, 4096, 0.07, 2, A, A, status,
                                         wait_ns, None)

    assert stalled(status=None) == INVALID                          # the status word is where the timeout lands
    assert stalled(_cache(dtype=1, scales=A)) == INVALID            # bf16 kernel only
    assert stalled(wait_ns=10) == INVALID
    assert stalled(wait_ns=3_000_000_000) == INVALID
    assert stalled(B=0) == INVALID                                  # and every check of mla_decode_fwd


def test_cache_append_rejects_bad_arguments_on_host():
    L = _lib.get()

    def append(c=None, h=A, T=4, d=5120, base=10000.0, num_seqs=32, staging=None, status=None):
        c = _cache() if c is None else c
        return L.mla_cache_append(h, A, A, A, A, T, d, base, ctypes.byref(c), num_seqs, staging, status, None)

    assert append(T=0) == _lib.MLA_OK                              # nothing to write
    assert append(h=None) == INVALID
    assert append(h=MIS) == INVALID
    assert append(T=-1) == INVALID
    assert append(d=5000) == UNSUPPORTED                           # not a multiple of 512
    assert append(d=0) == INVALID
    assert append(base=0.5) == INVALID
    assert append(num_seqs=0) == INVALID
    assert append(status=A + 2) == INVALID
    assert append(_cache(dtype=1, scales=A)) == INVALID             # e4m3 needs the staging buffer
    assert append(_cache(dtype=1)) == INVALID                       # ... and scales
    assert append(_cache(scales=A)) == INVALID                      # bf16 with scales
    assert append(_cache(seq_stride_tokens=0)) == INVALID
    paged = dict(block_table=A, page_size=64, max_pages=64, num_rows=64 * 100)
    assert append(_cache(**{**paged, "page_size": 16})) == UNSUPPORTED
    assert append(_cache(**{**paged, "num_rows": 64 * 100 + 1})) == INVALID


def test_rope_spec_is_checked_on_host():
    L = _lib.get()

    def absorb(**kw):
        r = _lib.MlaRope()
        r.base, r.yarn_scale, r.yarn_alpha, r.yarn_beta, r.original_max_pos, r.reserved = 10000.0, 40.0, 1.0, 32.0, 4096, 0
        for k, v in kw.items():
            setattr(r, k, v)
        return L.mla_absorb_q_ex(A, A, A, 1, 128, ctypes.byref(r), None if kw.get("null_out") else A, None)

    assert absorb(base=1.0) == INVALID
    assert absorb(yarn_scale=0.5) == INVALID
    assert absorb(yarn_beta=1.0) == INVALID          # beta must exceed alpha
    assert absorb(yarn_alpha=-1.0) == INVALID
    assert absorb(original_max_pos=0) == INVALID
    assert absorb(reserved=1) == INVALID
    assert L.mla_absorb_q_ex(A, A, A, 1, 128, None, A, None) == INVALID


def test_multi_token_view_rejects_bad_arguments_on_host():
    L = _lib.get()

    def view(c=None, B=4, T=2, max_len=4096, mp=64, out=A):
        c = _cache() if c is None else c
        v = _lib.MlaCache()
        return L.mla_multi_token_view(ctypes.byref(c), A, B, T, max_len, out, A, A, mp, ctypes.byref(v), None)

    assert view(T=0) == INVALID
    assert view(B=40000, T=2) == INVALID                          # B*T beyond the grid limit
    assert view(mp=10) == INVALID                                 # too few pages for max_seq_len
    assert view(out=MIS) == INVALID
    assert view(_cache(seq_stride_tokens=4100, num_rows=32 * 4100)) == UNSUPPORTED   # not whole pages
    assert view(max_len=5000) == INVALID                          # longer than the contiguous stride
