"""GPU properties that hold at any size and need no oracle run: uniform weights for a
zero query (full size, including 128K contexts), split-count invariance, paged ==
contiguous, block-table permutation invariance, constant caches, empty sequences and
the device status word for out-of-pool page ids."""

import gc
import math

import numpy as np
import pytest
import torch

import mla_latent_kv_69_b300 as mla
import workloads as W
from mla_cases import Case, assert_within_tolerance, bits_to_torch_bf16

pytestmark = pytest.mark.gpu


def _latent_values(case: Case) -> list:
    """Per sequence, the cached latents as float64 tensors (dequantised for e4m3)."""
    out = []
    data = case.cache.data
    for b, L in enumerate(case.lens):
        L = int(L)
        if case.block_table is None:
            rows = data[b, :L]
            sc = case.cache.scales[b, :L] if case.cache.scales is not None else None
        else:
            pages = case.block_table[b, : (L + 63) // 64].long()
            rows = data[pages].reshape(-1, 576)[:L]
            sc = case.cache.scales[pages].reshape(-1)[:L] if case.cache.scales is not None else None
        if sc is None:
            v = rows.double()
        else:
            v = rows.view(torch.float8_e4m3fn).double() * sc.double()[:, None]
        out.append(v[:, :512])
    return out


@pytest.mark.parametrize("name", ["v2_b32_l4096", "paged_b64_l1k_32k", "long_b4_l128k", "fp8_b128_l8192"])
def test_zero_query_gives_latent_mean(cuda_device, name):
    case = Case(W.WORKLOADS[name], cuda_device)
    q_lat = torch.zeros(case.B, case.n_h, 576, dtype=torch.bfloat16, device=cuda_device)
    o_part, lse_part = mla.decode_fwd(q_lat, case.cache, case.seq_lens, case.max_len)
    o_lat, lse = mla.combine(o_part, lse_part)
    torch.cuda.synchronize()
    means = torch.stack([v.mean(dim=0) for v in _latent_values(case)])            # [B, 512]
    ref = means[:, None, :].expand(case.B, case.n_h, 512).cpu().numpy()
    assert_within_tolerance(o_lat.double().cpu().numpy(), ref, "o_lat")
    np.testing.assert_allclose(lse.cpu().numpy(), np.log(case.lens.astype(np.float64))[:, None]
                               .repeat(case.n_h, 1), atol=1e-4, rtol=0)
    del case
    gc.collect()
    torch.cuda.empty_cache()


def test_split_count_invariance(cuda_device):
    # Different split counts round P (bf16) against different running maxima, so the
    # results agree to the parity tolerance, not bit for bit.
    case = Case(W.WORKLOADS["v2_b32_l4096"], cuda_device)
    ref = case.run(n_splits=1)["o"].double().cpu().numpy()
    for S in (2, 5, 64, 0):
        o = case.run(n_splits=S)["o"].double().cpu().numpy()
        assert_within_tolerance(o, ref, f"S={S} vs S=1")


def test_paged_equals_contiguous_and_permutation_invariance(cuda_device):
    w = W.Workload("pc", n_h=128, batch=5, ctx_range=(1, 3000), seed=11)
    lens = W.seq_lens(w)
    rows = [W.gen_rows(w, b, int(L)) for b, L in enumerate(lens)]
    stride = int(lens.max())
    contig = bits_to_torch_bf16(W.layout_contiguous(rows, stride), cuda_device)
    bt, pool = W.gen_block_table(w.with_(paged=True), lens)
    paged = bits_to_torch_bf16(W.layout_paged(rows, bt, pool), cuda_device)
    q_lat = bits_to_torch_bf16(W.gen_rows(w, 99, 5 * 128).reshape(5, 128, 576), cuda_device)
    seq = torch.from_numpy(lens).to(cuda_device)
    outs = []
    for cache in (mla.Cache(contig), mla.Cache(paged, None, torch.from_numpy(bt).to(cuda_device))):
        o_part, lse_part = mla.decode_fwd(q_lat, cache, seq, stride, n_splits=3)
        outs.append(mla.combine(o_part, lse_part))
    torch.testing.assert_close(outs[0][0], outs[1][0], rtol=0, atol=0)
    torch.testing.assert_close(outs[0][1], outs[1][1], rtol=0, atol=0)
    # move every page to a new slot and rewrite the block table accordingly
    perm = np.random.default_rng(0).permutation(pool)
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    paged2 = torch.empty_like(paged)
    paged2[torch.from_numpy(perm).long().to(cuda_device)] = paged
    o_part, lse_part = mla.decode_fwd(q_lat, mla.Cache(paged2, None, torch.from_numpy(bt2).to(cuda_device)), seq,
                                      stride, n_splits=3)
    o2 = mla.combine(o_part, lse_part)
    torch.testing.assert_close(o2[0], outs[1][0], rtol=0, atol=0)


def test_constant_cache_returns_projected_row(cuda_device):
    w = W.Workload("cc", n_h=128, batch=2, ctx=0, seed=12)
    case = Case(w, cuda_device, lens=[1000, 5])
    row = case.cache.data[0, 0].clone()
    case.cache.data[:] = row
    out = case.run(n_splits=4)
    torch.cuda.synchronize()
    c = row[:512].double()
    ref = torch.einsum("hdj,j->hd", case.w_uv.double(), c)
    for b in range(2):
        assert_within_tolerance(out["o"][b].double().cpu().numpy(), ref.cpu().numpy(), "o")
        torch.testing.assert_close(out["o_lat"][b].double(), c.expand(128, 512), rtol=1e-5, atol=1e-6)


def test_empty_and_single_token_sequences(cuda_device):
    w = W.Workload("e", n_h=128, batch=3, ctx=0, seed=13)
    case = Case(w, cuda_device, lens=[0, 1, 0])
    out = case.run(n_splits=2)
    torch.cuda.synchronize()
    assert torch.all(out["o"][0] == 0) and torch.all(out["o"][2] == 0)
    assert torch.all(torch.isneginf(out["lse"][0]))
    # a single token: o_lat is exactly that token's latent
    torch.testing.assert_close(out["o_lat"][1], case.cache.data[1, 0, :512].float().expand(128, 512),
                               rtol=1e-6, atol=1e-6)


def test_out_of_pool_page_sets_status_and_is_skipped(cuda_device):
    w = W.Workload("oob", n_h=128, batch=2, ctx=0, paged=True, seed=14)
    case = Case(w, cuda_device, lens=[200, 100])
    bt = case.block_table.clone()
    bt[0, 1] = case.pool_pages + 5          # second page of sequence 0 points outside the pool
    cache = mla.Cache(case.cache.data, None, bt)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    o_part, lse_part = mla.decode_fwd(case.q.new_zeros(2, 128, 576), cache, case.seq_lens, case.max_len,
                                      n_splits=1, status=status)
    o_lat, lse = mla.combine(o_part, lse_part)
    torch.cuda.synchronize()
    assert int(status.item()) == 6          # MLA_ERR_DEVICE_BOUNDS
    # sequence 0 averaged only the 136 tokens on its valid pages
    assert abs(float(lse[0, 0]) - math.log(136)) < 1e-4
    assert abs(float(lse[1, 0]) - math.log(100)) < 1e-4
