"""mla.DecodeStepGraph: the decode step captured once as a CUDA graph (copies of the
step's inputs from pinned host buffers, the C-ABI calls of decode_step, the copy of o back) gives,
replay after replay, exactly what the eager step gives on the same inputs, and
takes each step's inputs from the host buffers as they are at replay time."""

import numpy as np
import pytest
import torch

import mla_latent_kv_69_b300 as mla
import workloads as W
from mla_cases import Case

pytestmark = pytest.mark.gpu


def _eager_o(case, q, pos, lens):
    d_q = q.to(case.device)
    d_pos = torch.from_numpy(pos).to(case.device)
    d_len = torch.from_numpy(lens).to(case.device)
    out = mla.decode_step(d_q, case.w_uk, case.w_uv, case.cache, d_len, d_pos, case.max_len)
    torch.cuda.synchronize()
    return out["o"].cpu()


@pytest.mark.parametrize("paged", [False, True])
def test_graph_step_equals_eager_step(cuda_device, paged):
    lens = np.array([300, 1000, 65], dtype=np.int32)
    w = W.Workload("graph", n_h=128, batch=len(lens), ctx=0, paged=paged, seed=81)
    case = Case(w, cuda_device, lens=lens)
    g = mla.DecodeStepGraph(case.w_uk, case.w_uv, case.cache, case.B, case.max_len)
    rng = np.random.default_rng(810)
    for step in range(3):
        # a new query each step, and lengths that shrink (a cache view with fewer tokens)
        q = W.bits_to_torch_bf16(W.f32_to_bf16_bits(rng.standard_normal((case.B, case.n_h, 192), dtype=np.float32)),
                                 "cpu")
        cur = np.maximum(lens - 97 * step, 0).astype(np.int32)
        pos = W.positions(cur)
        g.h_q.copy_(q)
        g.h_pos.copy_(torch.from_numpy(pos))
        g.h_seq_lens.copy_(torch.from_numpy(cur))
        g.replay()
        g.synchronize()
        got = g.h_o.clone()   # read right after the step's own event, before anything else syncs
        assert g.done.query()
        ref = _eager_o(case, q, pos, cur)
        assert torch.equal(got, ref), f"step {step}"
