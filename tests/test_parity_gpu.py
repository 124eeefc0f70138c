"""GPU parity: the library's decode step (all four C-ABI calls) against the fp64 oracle
on the same seeded inputs, within max|gpu-oracle| <= 2e-2·max|oracle| and
sum|gpu-oracle|/sum|oracle| <= 3e-3.

Small cases compare every element; the full-size workloads run in the launch
configuration the benchmark times (automatic split count) and compare sampled
(sequence, head) outputs that the oracle evaluates one by one.
"""

import gc

import numpy as np
import pytest
import torch

import mla_latent_kv_69_b300 as mla
import workloads as W
from mla_cases import Case, assert_within_tolerance, rows_f32
from oracle import fp8_e4m3

pytestmark = pytest.mark.gpu


def _compare(case, out, samples, check_lat=True):
    o = out["o"].double().cpu().numpy()
    o_lat = out["o_lat"].double().cpu().numpy()
    lse = out["lse"].double().cpu().numpy()
    got, ref, got_lat, ref_lat = [], [], [], []
    for b, heads in samples:
        r = case.oracle(b, heads=heads)
        hs = list(range(case.n_h)) if heads is None else list(heads)
        got.append(o[b, hs]); ref.append(r["o"][hs])
        got_lat.append(o_lat[b, hs]); ref_lat.append(r["o_lat"][hs])
        if case.lens[b] > 0:
            np.testing.assert_allclose(lse[b, hs], r["lse"][hs], atol=2e-2, rtol=0)
        else:
            assert np.all(np.isneginf(lse[b, hs]))
    got, ref = np.concatenate([g.ravel() for g in got]), np.concatenate([r.ravel() for r in ref])
    if np.abs(ref).sum() == 0:
        assert np.all(got == 0)
        return
    stats = assert_within_tolerance(got, ref, "o")
    if check_lat:
        assert_within_tolerance(np.concatenate([g.ravel() for g in got_lat]),
                                np.concatenate([r.ravel() for r in ref_lat]), "o_lat")
    return stats


SMALL = [
    ("h128_contig_ragged", W.Workload("s1", n_h=128, batch=3, ctx=0), [1, 100, 700]),
    ("h128_paged_ragged", W.Workload("s2", n_h=128, batch=4, ctx=0, paged=True, seed=3), [65, 130, 1000, 3]),
    ("h128_fp8_ragged", W.Workload("s3", n_h=128, batch=2, ctx=0, kv="fp8", seed=5), [77, 640]),
    ("h128_fp8_paged", W.Workload("s4", n_h=128, batch=2, ctx=0, kv="fp8", paged=True, seed=6), [200, 64]),
    ("h64", W.Workload("s5", n_h=64, batch=2, ctx=0, seed=7), [300, 129]),
    ("h32_paged", W.Workload("s6", n_h=32, batch=2, ctx=0, paged=True, seed=8), [300, 129]),
    ("h16", W.Workload("s7", n_h=16, batch=2, ctx=0, seed=9), [513, 2]),
    ("with_empty_seq", W.Workload("s8", n_h=128, batch=3, ctx=0, seed=10), [0, 191, 64]),
]


@pytest.mark.parametrize("name,w,lens", SMALL, ids=[s[0] for s in SMALL])
@pytest.mark.parametrize("n_splits", [1, 3, 0])
def test_small_cases_every_element(cuda_device, name, w, lens, n_splits):
    case = Case(w, cuda_device, lens=lens, keep_rows=True)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    out = case.run(n_splits=n_splits, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _compare(case, out, [(b, None) for b in range(case.B)])


def test_tiny_workload_every_element(cuda_device):
    case = Case(W.WORKLOADS["tiny_h16_b1_l256"], cuda_device, keep_rows=True)
    out = case.run()
    torch.cuda.synchronize()
    _compare(case, out, [(0, None)])


def _fp8_codes_match(case, b):
    """The GPU quantiser's codes and scales equal the oracle codec's, bit for bit."""
    L = int(case.lens[b])
    codes, scales = fp8_e4m3.quantize_rows(rows_f32(case.rows_of(b)))
    if case.block_table_np is None:
        g_codes = case.cache.data[b, :L].cpu().numpy()
        g_scales = case.cache.scales[b, :L].cpu().numpy()
    else:
        pages = case.block_table_np[b, : (L + 63) // 64]
        g_codes = case.cache.data[torch.from_numpy(pages).long()].reshape(-1, 576)[:L].cpu().numpy()
        g_scales = case.cache.scales[torch.from_numpy(pages).long()].reshape(-1)[:L].cpu().numpy()
    np.testing.assert_array_equal(g_codes, codes)
    np.testing.assert_array_equal(g_scales.view(np.uint32), scales.view(np.uint32))


def test_fp8_quantiser_bit_exact_small(cuda_device):
    for _, w, lens in SMALL:
        if w.kv == "fp8":
            case = Case(w, cuda_device, lens=lens, keep_rows=True)
            for b in range(case.B):
                _fp8_codes_match(case, b)


class _CodesCase(Case):
    """An e4m3 case whose codes and per-token scales are drawn on the host and written
    into the device cache directly; the oracle decodes the same codes."""

    def set_codes(self, b, codes, scales):
        L = len(codes)
        self.cache.data[b, :L] = torch.from_numpy(codes).to(self.device)
        self.cache.scales[b, :L] = torch.from_numpy(scales).to(self.device)
        self.host_codes = getattr(self, "host_codes", {})
        self.host_codes[b] = (codes, scales)

    def oracle_rows(self, b):
        codes, scales = self.host_codes[b]
        return fp8_e4m3.dequantize_rows(codes, scales)


def test_fp8_every_code_through_tensor_cores(cuda_device):
    """Every finite e4m3 code, half of them drawn from the subnormal codes (exponent field
    0), through both contractions of the e4m3 kernel: the code-to-f16 mapping has to be
    exact for normal and subnormal codes alike for the result to stay in tolerance."""
    w = W.Workload("codes", n_h=128, batch=2, ctx=0, kv="fp8", seed=21)
    case = _CodesCase(w, cuda_device, lens=[300, 257])
    rng = np.random.default_rng(2101)
    finite = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    sub = finite[((finite >> 3) & 15) == 0]
    for b, L in enumerate(case.lens):
        L = int(L)
        codes = np.where(rng.random((L, 576)) < 0.5, rng.choice(sub, (L, 576)), rng.choice(finite, (L, 576)))
        scales = (rng.uniform(0.5, 1.0, L) / 448.0).astype(np.float32)
        case.set_codes(b, codes.astype(np.uint8), scales)
    assert mla.decode_kernel("fp8", 128) == "tcgen05_f16_e4m3"
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    out = case.run(n_splits=3, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _compare(case, out, [(b, None) for b in range(case.B)])


FULL = {
    "v2_b32_l4096": lambda c: [(0, None), (c.B - 1, None)],
    "paged_b64_l1k_32k": lambda c: [(int(np.argmin(c.lens)), None), (int(np.argmax(c.lens)), [0, 1, 2, 127]),
                                    (0, list(range(0, 128, 16)))],
    "long_b4_l128k": lambda c: [(0, [0, 77]), (3, [127])],
    "fp8_b128_l8192": lambda c: [(0, list(range(0, 128, 4))), (127, list(range(1, 128, 8)))],
}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_sampled(cuda_device, name):
    w = W.WORKLOADS[name]
    case = Case(w, cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    out = case.run(n_splits=0, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    samples = FULL[name](case)
    _compare(case, out, samples)
    if w.kv == "fp8":
        for b, _ in samples:
            _fp8_codes_match(case, b)
    del case, out
    gc.collect()
    torch.cuda.empty_cache()
