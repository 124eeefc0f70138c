"""YaRN-extended RoPE on the GPU (mla_absorb_q_ex, mla_cache_append_ex) against the
oracle's yarn_inv_freq, with the pages' setting (scale 40, alpha 1, beta 32) over a 4K
original context, at positions up to 160K: the rotated query and key columns, and a
whole decode step whose query is rotated with the extended frequencies."""

import numpy as np
import pytest
import torch

import mla_latent_kv_69_b300 as mla
import workloads as W
from mla_cases import Case, assert_within_tolerance, bits_to_torch_bf16, rows_f32
from oracle import mla_oracle as M

pytestmark = pytest.mark.gpu

YARN = mla.Yarn()
FREQ = M.yarn_inv_freq(64, 10000.0, YARN.scale, YARN.alpha, YARN.beta, YARN.original_max_pos)


def _bf16_f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def test_absorbed_query_rotation(cuda_device):
    w = W.Workload("yarn_q", n_h=16, batch=8, ctx=0, seed=101)
    q_bits, wuk_bits = W.gen_q(w), W.gen_w_uk(w)
    pos = np.array([0, 1, 4095, 4096, 40000, 131071, 150000, 163839], dtype=np.int32)
    q_lat = mla.absorb_q(bits_to_torch_bf16(q_bits, cuda_device), bits_to_torch_bf16(wuk_bits, cuda_device),
                         torch.from_numpy(pos).to(cuda_device), yarn=YARN)
    plain = mla.absorb_q(bits_to_torch_bf16(q_bits, cuda_device), bits_to_torch_bf16(wuk_bits, cuda_device),
                         torch.from_numpy(pos).to(cuda_device))
    torch.cuda.synchronize()
    got = q_lat.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = M.rope(rows_f32(q_bits)[..., 128:].astype(np.float64), pos[:, None], inv_freq=FREQ)   # [B, n_h, 64]
    err = np.abs(_bf16_f64(got[..., 512:]) - ref)
    # one bf16 rounding (2^-8 relative) plus the fp32 rotation of a reduced angle
    assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 2e-6 * np.abs(rows_f32(q_bits)[..., 128:]).max())
    # the latent part does not depend on the RoPE
    assert torch.equal(q_lat[..., :512], plain[..., :512])
    assert not torch.equal(q_lat[..., 512:], plain[..., 512:])


def test_appended_key_rotation(cuda_device):
    T, B, stride = 24, 3, 8192
    rng = np.random.default_rng(102)
    seq = (np.arange(T) % B).astype(np.int32)
    pos = np.sort(rng.choice(stride, size=T, replace=False)).astype(np.int32)
    rows = torch.zeros(B * stride, 576, dtype=torch.bfloat16, device=cuda_device)
    cache = mla.Cache(rows.view(B, stride, 576))
    h_bits, wd_bits, wk_bits = W.gen_hidden(103, T), W.gen_w_dkv(103), W.gen_w_kr(103)
    h, wd, wk = (bits_to_torch_bf16(x, cuda_device) for x in (h_bits, wd_bits, wk_bits))
    mla.cache_append(h, wd, wk, torch.from_numpy(seq).to(cuda_device), torch.from_numpy(pos).to(cuda_device), cache,
                     yarn=YARN)
    torch.cuda.synchronize()
    got = rows.view(torch.int16).cpu().numpy().view(np.uint16)[seq.astype(np.int64) * stride + pos]
    ref = M.cache_rows(_bf16_f64(h_bits), _bf16_f64(wd_bits), _bf16_f64(wk_bits), pos, inv_freq=FREQ)
    err = np.abs(_bf16_f64(got) - ref)
    assert np.all(err <= 2.0 ** -7 * np.abs(ref) + 1e-3), float(err.max())
    plain = M.cache_rows(_bf16_f64(h_bits), _bf16_f64(wd_bits), _bf16_f64(wk_bits), pos)
    assert np.abs(_bf16_f64(got[:, 512:]) - plain[:, 512:]).max() > 1e-2   # the extension changed the keys


def test_decode_step_with_extended_query(cuda_device):
    lens = [5000, 130]
    w = W.Workload("yarn_step", n_h=64, batch=len(lens), ctx=0, seed=104)
    case = Case(w, cuda_device, lens=lens, keep_rows=True)
    out = mla.decode_step(case.q, case.w_uk, case.w_uv, case.cache, case.seq_lens, case.pos, case.max_len,
                          yarn=YARN)
    torch.cuda.synchronize()
    o = out["o"].double().cpu().numpy()
    got, ref = [], []
    for b in range(case.B):
        rows = case.oracle_rows(b)
        r = M.attend_explicit(rows_f32(case.q_bits[b]), rows[:, :512], rows[:, 512:], rows_f32(case.wuk_bits),
                              rows_f32(case.wuv_bits), pos_q=int(case.pos_np[b]), inv_freq=FREQ)
        got.append(o[b].ravel())
        ref.append(r["o"].ravel())
    assert_within_tolerance(np.concatenate(got), np.concatenate(ref), "o with the YaRN query")
