"""GPU parity of mla_cache_append against the oracle's cache_rows (fp64).

The kernel rounds the fp32 sum of 5120 exact bf16 products once to bf16, so every written
element must be within one bf16 step of the fp64 value and equal to its correctly
rounded value except where the fp32 accumulation crosses a rounding midpoint (a small
fraction). Rows that no token targets must be left as they were."""

import numpy as np
import pytest
import torch

import mla_latent_kv_69_b300 as mla
import workloads as W
from mla_cases import bits_to_torch_bf16
from mla_latent_kv_69_b300 import _lib
from oracle import fp8_e4m3 as F
from oracle import mla_oracle as M

pytestmark = pytest.mark.gpu

D = W.D_MODEL


def _inputs(seed, T, device, d=D):
    h_bits, wd_bits, wk_bits = W.gen_hidden(seed, T, d), W.gen_w_dkv(seed, d), W.gen_w_kr(seed, d)
    dev = [bits_to_torch_bf16(x, device) for x in (h_bits, wd_bits, wk_bits)]
    f64 = [W.bf16_bits_to_f32(x).astype(np.float64) for x in (h_bits, wd_bits, wk_bits)]
    return dev, f64


def _bf16_f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def _bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (normal range)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def _term_sums(h64, wd64, wk64):
    """Sum of |products| behind each element of the rows (before rounding): the scale of
    the fp32 accumulation error. A rotated key element mixes its pair's two sums."""
    c = np.abs(h64) @ np.abs(wd64).T
    k = np.abs(h64) @ np.abs(wk64).T
    kk = k[:, :32] + k[:, 32:]
    return np.concatenate([c, kk, kk], axis=1)


def _check_rows(got_bits, ref, sums, what):
    """Within one bf16 step plus the fp32 accumulation's error (2^-18 of the summed
    magnitudes, some 30x the error of 5120 additions in random order), and the
    correctly rounded value for at least 99% of the elements."""
    got = _bf16_f64(got_bits)
    rounded = _bf16_f64(W.f32_to_bf16_bits(ref.astype(np.float32)))
    err = np.abs(got - ref)
    bound = _bf16_ulp(ref) + 2.0 ** -18 * sums
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert np.all(err <= bound), (f"{what}: element {worst} is off by {err[worst]:.3e} (ref {ref[worst]:.4e}, "
                                  f"bound {bound[worst]:.3e}, summed magnitude {sums[worst]:.3e})")
    exact = np.mean(got == rounded)
    assert exact >= 0.99, f"{what}: only {exact:.4f} of the elements are the correctly rounded value"


@pytest.mark.parametrize("paged", [False, True])
def test_append_bf16_rows(cuda_device, paged):
    rng = np.random.default_rng(91 if paged else 90)
    B, stride = 6, 512
    T = 200 if paged else 37                      # two token tiles in the paged case
    seq = rng.integers(0, B, size=T).astype(np.int32)
    pos = np.zeros(T, dtype=np.int32)
    used = set()
    for t in range(T):                            # distinct destinations
        while True:
            p = int(rng.integers(0, stride))
            if (int(seq[t]), p) not in used:
                used.add((int(seq[t]), p))
                pos[t] = p
                break
    before = rng.standard_normal((B * stride, 576)).astype(np.float32)
    rows = torch.from_numpy(W.f32_to_bf16_bits(before).view(np.int16)).view(torch.bfloat16).to(cuda_device)
    if paged:
        npg = stride // 64
        perm = rng.permutation(B * npg).astype(np.int32)
        bt = perm.reshape(B, npg)
        cache = mla.Cache(rows.view(B * npg, 64, 576), None, torch.from_numpy(bt).to(cuda_device))
        dest = bt[seq, pos // 64].astype(np.int64) * 64 + pos % 64
    else:
        cache = mla.Cache(rows.view(B, stride, 576))
        dest = seq.astype(np.int64) * stride + pos
    (h, wd, wk), (h64, wd64, wk64) = _inputs(5 + paged, T, cuda_device)
    before_bits = rows.view(torch.int16).cpu().numpy().view(np.uint16).copy()
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    mla.cache_append(h, wd, wk, torch.from_numpy(seq).to(cuda_device), torch.from_numpy(pos).to(cuda_device), cache,
                     status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    after = rows.view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1, 576)
    ref = M.cache_rows(h64, wd64, wk64, pos)
    _check_rows(after[dest], ref, _term_sums(h64, wd64, wk64), "written rows")
    untouched = np.ones(after.shape[0], dtype=bool)
    untouched[dest] = False
    np.testing.assert_array_equal(after[untouched], before_bits.reshape(-1, 576)[untouched])


def test_append_bounds_are_reported_and_skipped(cuda_device):
    B, stride, T = 2, 128, 4
    rows = torch.zeros(B * stride, 576, dtype=torch.bfloat16, device=cuda_device)
    cache = mla.Cache(rows.view(B, stride, 576))
    seq = np.array([0, 1, 2, -1], dtype=np.int32)     # sequences 2 and -1 do not exist
    pos = np.array([5, 127, 0, 0], dtype=np.int32)
    (h, wd, wk), (h64, wd64, wk64) = _inputs(7, T, cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    mla.cache_append(h, wd, wk, torch.from_numpy(seq).to(cuda_device), torch.from_numpy(pos).to(cuda_device), cache,
                     status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == _lib.MLA_ERR_DEVICE_BOUNDS
    after = rows.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = M.cache_rows(h64[:2], wd64, wk64, pos[:2])
    _check_rows(after[[5, stride + 127]], ref, _term_sums(h64[:2], wd64, wk64), "valid tokens")
    keep = np.ones(B * stride, dtype=bool)
    keep[[5, stride + 127]] = False
    assert np.all(after[keep] == 0)


def test_append_e4m3_exact_latent(cuda_device):
    """One-hot hidden states make the latent part exact (a column of W_DKV), and a small
    W_KR keeps the row's largest element in that part: the scale and the latent codes
    must then be exactly what the oracle's quantiser gives."""
    T, B, stride = 16, 2, 64
    cols = np.arange(T) * 311 % D
    h_bits = np.zeros((T, D), dtype=np.uint16)
    h_bits[np.arange(T), cols] = W.f32_to_bf16_bits(np.ones(T, dtype=np.float32))
    wd_bits = W.gen_w_dkv(8)
    wk_bits = W.f32_to_bf16_bits(W.bf16_bits_to_f32(W.gen_w_kr(8)) * np.float32(1e-3))
    h, wd, wk = (bits_to_torch_bf16(x, cuda_device) for x in (h_bits, wd_bits, wk_bits))
    codes = torch.zeros(B * stride, 576, dtype=torch.uint8, device=cuda_device)
    scales = torch.zeros(B * stride, dtype=torch.float32, device=cuda_device)
    cache = mla.Cache(codes.view(B, stride, 576), scales.view(B, stride))
    seq = (np.arange(T) % B).astype(np.int32)
    pos = (np.arange(T) // B * 7).astype(np.int32)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    mla.cache_append(h, wd, wk, torch.from_numpy(seq).to(cuda_device), torch.from_numpy(pos).to(cuda_device), cache,
                     status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    dest = seq.astype(np.int64) * stride + pos
    got_codes = codes.cpu().numpy()[dest]
    got_scales = scales.cpu().numpy()[dest]
    ref = M.cache_rows(_bf16_f64(h_bits), _bf16_f64(wd_bits), _bf16_f64(wk_bits), pos)
    ref_bits = W.f32_to_bf16_bits(ref.astype(np.float32))
    assert np.all(np.abs(ref[:, 512:]).max(axis=1) < np.abs(ref[:, :512]).max(axis=1))
    np.testing.assert_array_equal(ref[:, :512], _bf16_f64(ref_bits[:, :512]))   # the latent part is exact
    exp_codes, exp_scales = F.quantize_rows(W.bf16_bits_to_f32(ref_bits))
    np.testing.assert_array_equal(got_scales, exp_scales)
    np.testing.assert_array_equal(got_codes[:, :512], exp_codes[:, :512])
    assert np.all(np.abs(got_codes[:, 512:].astype(int) - exp_codes[:, 512:].astype(int)) <= 1)


def test_append_e4m3_paged(cuda_device):
    rng = np.random.default_rng(93)
    B, npg, T = 3, 4, 50
    seq = (np.arange(T) % B).astype(np.int32)           # distinct destinations
    pos = (np.arange(T) // B * 5).astype(np.int32)
    bt = rng.permutation(B * npg).astype(np.int32).reshape(B, npg)
    codes = torch.zeros(B * npg * 64, 576, dtype=torch.uint8, device=cuda_device)
    scales = torch.zeros(B * npg * 64, dtype=torch.float32, device=cuda_device)
    cache = mla.Cache(codes.view(B * npg, 64, 576), scales.view(B * npg, 64), torch.from_numpy(bt).to(cuda_device))
    (h, wd, wk), (h64, wd64, wk64) = _inputs(9, T, cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    mla.cache_append(h, wd, wk, torch.from_numpy(seq).to(cuda_device), torch.from_numpy(pos).to(cuda_device), cache,
                     status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    dest = bt[seq, pos // 64].astype(np.int64) * 64 + pos % 64
    deq = F.dequantize_rows(codes.cpu().numpy()[dest], scales.cpu().numpy()[dest])
    ref = M.cache_rows(h64, wd64, wk64, pos)
    amax = np.abs(ref).max(axis=1, keepdims=True)
    # e4m3 keeps 3 fraction bits: half a step is 2^-4 relative for normal codes and
    # scale * 2^-10 below them; the bf16 staging adds at most one bf16 step
    tol = 2.0 ** -4 * np.abs(ref) + amax / 448 * 2.0 ** -9 + _bf16_ulp(ref) * 1.01 + \
        2.0 ** -18 * _term_sums(h64, wd64, wk64)
    assert np.all(np.abs(deq - ref) <= tol)
