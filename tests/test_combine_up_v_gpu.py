"""mla_combine_up_v (the log-sum-exp merge of the split partials and W_UV in one launch)
against the oracle, every element: o = W_UV · merge(o_part, lse_part), with o_lat and
lse as optional outputs. Cases span one to every slot (MLA_MAX_SPLITS), empty slots
(lse = -inf), a sequence whose slots are all empty, a ragged last batch tile and every
head count; the fused o also agrees with mla_combine followed by mla_up_v."""

import numpy as np
import pytest
import torch

import mla_latent_kv_69_b300 as mla
import workloads as W
from mla_cases import assert_within_tolerance, bits_to_torch_bf16, rows_f32
from oracle import mla_oracle as M

pytestmark = pytest.mark.gpu


def _partials(B, S, n_h, seed, empty_frac=0.25):
    rng = np.random.default_rng(seed)
    o_part = rng.standard_normal((B, S, n_h, 512)).astype(np.float32)
    lse = rng.uniform(-6.0, 6.0, (B, S, n_h)).astype(np.float32)
    lse[rng.random((B, S, n_h)) < empty_frac] = -np.inf
    lse[0] = -np.inf                     # a sequence with no token at all
    if S > 1:
        lse[-1, 1:] = -np.inf            # only the first slot holds tokens
    return o_part, lse


@pytest.mark.parametrize("B,S,n_h", [(1, 1, 128), (37, 2, 128), (5, 5, 64), (33, 18, 16), (3, 256, 32)])
def test_combine_up_v_every_element(cuda_device, B, S, n_h):
    o_part, lse = _partials(B, S, n_h, seed=1000 + B + S)
    w = W.Workload("cuv", n_h=n_h, batch=B, ctx=0, seed=500 + n_h)
    wuv_bits = W.gen_w_uv(w)
    d_o_part = torch.from_numpy(o_part).to(cuda_device)
    d_lse_part = torch.from_numpy(lse).to(cuda_device)
    w_uv = bits_to_torch_bf16(wuv_bits, cuda_device)
    o_lat = torch.full((B, n_h, 512), float("nan"), device=cuda_device)
    lse_out = torch.full((B, n_h), float("nan"), device=cuda_device)
    o, _, _ = mla.combine_up_v(d_o_part, d_lse_part, w_uv, o_lat=o_lat, lse=lse_out)
    o_only, none_lat, none_lse = mla.combine_up_v(d_o_part, d_lse_part, w_uv)
    torch.cuda.synchronize()
    assert none_lat is None and none_lse is None
    assert torch.equal(o, o_only), "o must not depend on whether o_lat and lse are written"

    ref_lat, ref_lse = M.merge_partials(np.moveaxis(o_part, 1, 0), np.moveaxis(lse, 1, 0))   # [B, n_h, ...]
    ref_o = np.einsum("hdj,bhj->bhd", rows_f32(wuv_bits).astype(np.float64), ref_lat)
    assert_within_tolerance(o.double().cpu().numpy(), ref_o, f"o (B={B}, S={S}, n_h={n_h})")
    np.testing.assert_allclose(o_lat.double().cpu().numpy(), ref_lat, rtol=1e-5, atol=1e-5)
    got_lse = lse_out.double().cpu().numpy()
    assert np.array_equal(np.isneginf(got_lse), np.isneginf(ref_lse))
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(got_lse[fin], ref_lse[fin], rtol=0, atol=2e-5)
    # an all-empty sequence: o_lat = 0 and o = 0 exactly
    assert torch.all(o[0] == 0) and torch.all(o_lat[0] == 0)

    # the two-call path on the same partials
    o_lat2, lse2 = mla.combine(d_o_part, d_lse_part)
    o2 = mla.up_v(o_lat2, w_uv)
    torch.cuda.synchronize()
    assert_within_tolerance(o.double().cpu().numpy(), o2.double().cpu().numpy(), "fused vs two calls")

