"""Several new query tokens per sequence (mla_multi_token_view + the decode step) against
the oracle's attend_multi, every element: query j of sequence b sits at L_b - T + j and
sees only the tokens up to its own position; a query with no visible token gives 0."""

import numpy as np
import pytest
import torch

import mla_latent_kv_69_b300 as mla
import workloads as W
from mla_cases import Case, assert_within_tolerance, bits_to_torch_bf16, rows_f32
from oracle import mla_oracle as M

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("paged,kv", [(False, "bf16"), (True, "bf16"), (False, "fp8")])
def test_multi_token_decode_every_element(cuda_device, paged, kv):
    T = 4
    lens = [300, 1000, 2, 64]        # the third sequence holds fewer tokens than new queries
    w = W.Workload("multi", n_h=128, batch=len(lens), ctx=0, paged=paged, kv=kv, seed=111)
    case = Case(w, cuda_device, lens=lens, keep_rows=True)
    if not paged:                    # whole 64-row pages per sequence, as the view needs
        stride = 1024
        src = torch.zeros(case.B, stride, 576, dtype=torch.bfloat16, device=cuda_device)
        src[:, :case.source.shape[1]] = case.source
        case.source = src
        case.rebuild_cache()
    qw = w.with_(batch=len(lens) * T)
    q_bits = W.gen_q(qw).reshape(len(lens), T, 128, 192)
    q = bits_to_torch_bf16(q_bits, cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    out = mla.decode_multi(q, case.w_uk, case.w_uv, case.cache, case.seq_lens, case.max_len, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o = out["o"].double().cpu().numpy()
    wk, wv = rows_f32(case.wuk_bits), rows_f32(case.wuv_bits)
    got, ref = [], []
    for b, L in enumerate(lens):
        rows = case.oracle_rows(b)
        r = M.attend_multi(rows_f32(q_bits[b]), rows[:, :512], rows[:, 512:], wk, wv, T=T)
        for j in range(T):
            if L - T + j < 0:
                assert np.all(o[b, j] == 0), (b, j)
            else:
                got.append(o[b, j].ravel())
                ref.append(r["o"][j].ravel())
    assert_within_tolerance(np.concatenate(got), np.concatenate(ref), f"o of every query ({kv}, paged={paged})")
    np.testing.assert_array_equal(out["view_seq_lens"].cpu().numpy().reshape(len(lens), T),
                                  np.maximum(np.array(lens)[:, None] - T + np.arange(T)[None, :] + 1, 0))
