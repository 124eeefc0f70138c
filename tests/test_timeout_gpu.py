"""The decode kernel's bounded waits, run out on purpose through the test hook
mla_test_decode_stalled: the score CTAs issue no loads and the waits that an abort can
end are limited to 2 ms. The kernel has to record MLA_ERR_TIMEOUT, stop both CTAs of
every SM pair, drain what it had started, free its tensor memory and return, leaving the
stream and the context usable: the same decode right after is bit for bit the first.

Nothing is in flight when the first waits run out (no load was issued; the value CTAs'
loads, if any started, are drained), so the abort cannot fault; the waits themselves
are what runs out, not a trap or a bad address."""

import time

import pytest
import torch

import mla_latent_kv_69_b300 as mla
import workloads as W
from mla_cases import Case, bits_to_torch_bf16
from mla_latent_kv_69_b300 import _lib

pytestmark = pytest.mark.gpu

WAIT_NS = 2_000_000


def _decode_merged(q_lat, case, n_splits):
    status = torch.zeros(1, dtype=torch.int32, device=q_lat.device)
    o_part, lse_part = mla.decode_fwd(q_lat, case.cache, case.seq_lens, case.max_len, n_splits=n_splits,
                                      status=status)
    o_lat, lse = mla.combine(o_part, lse_part)
    torch.cuda.synchronize()
    return o_lat, lse, int(status.item())


@pytest.mark.parametrize("paged,n_splits", [(False, 0), (False, 3), (True, 0), (True, 2)])
def test_bounded_waits_run_out_and_the_stream_recovers(cuda_device, paged, n_splits):
    # contiguous with the library schedule: one piece per SM pair; paged: the persistent kernel
    lens = [700, 1500, 64, 2100]
    w = W.Workload("stall", n_h=128, batch=len(lens), ctx=0, paged=paged, seed=71)
    case = Case(w, cuda_device, lens=lens)
    q_lat = bits_to_torch_bf16(W.gen_q_lat(w), cuda_device)
    o_ref, lse_ref, st = _decode_merged(q_lat, case, n_splits)
    assert st == 0

    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    t0 = time.perf_counter()
    mla.test_decode_stalled(q_lat, case.cache, case.seq_lens, case.max_len, status, WAIT_NS, n_splits=n_splits)
    torch.cuda.synchronize()   # returns: every role of every CTA left the kernel
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == _lib.MLA_ERR_TIMEOUT
    assert elapsed < 5.0, elapsed   # a few limits of 2 ms, not the 2 s default

    o_lat, lse, st = _decode_merged(q_lat, case, n_splits)
    assert st == 0
    assert torch.equal(o_lat, o_ref) and torch.equal(lse, lse_ref)


def test_stall_hook_reports_through_status_only(cuda_device):
    """A second stalled call on the same stream after the first: the status word keeps
    the first error, and the launches queue and complete normally."""
    w = W.Workload("stall2", n_h=64, batch=2, ctx=0, seed=72)
    case = Case(w, cuda_device, lens=[300, 129])
    q_lat = bits_to_torch_bf16(W.gen_q_lat(w), cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    for _ in range(2):
        mla.test_decode_stalled(q_lat, case.cache, case.seq_lens, case.max_len, status, WAIT_NS)
    torch.cuda.synchronize()
    assert int(status.item()) == _lib.MLA_ERR_TIMEOUT
