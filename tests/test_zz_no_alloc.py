"""mla_decode_combine_static, the decode-and-merge entry point for callers that cannot
allocate device memory (its split partials live in the library's own fixed device
array): through the C ABI it must give the same o_lat and lse, bit for bit, as
mla_decode_fwd + mla_combine with caller-allocated partials, on two calls in a row with different
shapes (the shared array keeps the previous call's contents). Collected last on
purpose, so a run that stops at the first failure has run every other test."""

import ctypes

import pytest
import torch

import mla_latent_kv_69_b300 as mla
import workloads as W
from mla_cases import Case
from mla_latent_kv_69_b300 import _lib

pytestmark = pytest.mark.gpu


def _static_call(case, q_lat, n_splits, o_lat, lse, status):
    c = case.cache.to_c()
    rc = _lib.get().mla_decode_combine_static(
        q_lat.data_ptr(), ctypes.byref(c), case.seq_lens.data_ptr(), case.B, case.n_h, case.max_len,
        mla.default_scale(), n_splits, o_lat.data_ptr(), lse.data_ptr(), status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.MLA_OK, _lib.status_string(rc)


def _reference(case, q_lat, n_splits):
    o_part, lse_part = mla.decode_fwd(q_lat, case.cache, case.seq_lens, case.max_len, n_splits=n_splits)
    return mla.combine(o_part, lse_part)


def test_static_entry_matches_allocating_path_on_two_calls(cuda_device):
    cases = [
        (Case(W.Workload("na1", n_h=128, batch=32, ctx=4096, seed=21), cuda_device), 0),
        (Case(W.Workload("na2", n_h=64, batch=3, ctx=0, paged=True, seed=22), cuda_device, lens=[700, 1, 130]), 3),
    ]
    for case, n_splits in cases:
        q_lat = mla.absorb_q(case.q, case.w_uk, case.pos)
        o_lat = torch.full((case.B, case.n_h, 512), float("nan"), device=cuda_device)
        lse = torch.full((case.B, case.n_h), float("nan"), device=cuda_device)
        status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
        _static_call(case, q_lat, n_splits, o_lat, lse, status)
        ref_o, ref_lse = _reference(case, q_lat, n_splits)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        # the same kernels on the same split layout: equal bit for bit (a stale value
        # left in the shared array by the previous call would show here)
        torch.testing.assert_close(o_lat, ref_o, rtol=0, atol=0)
        torch.testing.assert_close(lse, ref_lse, rtol=0, atol=0)
