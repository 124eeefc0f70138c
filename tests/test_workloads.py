"""The seeded input generator: determinism, per-sequence regeneration, bf16 rounding
(checked against torch's bfloat16 conversion) and the paged layout."""

import numpy as np
import torch

import workloads as W


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10,
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0, -0.0],
                                 dtype=np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(W.f32_to_bf16_bits(x), ref)
    np.testing.assert_array_equal(W.bf16_bits_to_f32(ref), torch.from_numpy(ref.view(np.int16)).view(
        torch.bfloat16).float().numpy())


def test_streams_are_deterministic_and_per_sequence():
    w = W.WORKLOADS["v2_b32_l4096"]
    a = W.gen_rows(w, 3, 100)
    b = W.gen_rows(w, 3, 100)
    np.testing.assert_array_equal(a, b)
    assert not np.array_equal(a, W.gen_rows(w, 4, 100))
    np.testing.assert_array_equal(W.gen_q(w), W.gen_q(w))
    assert W.gen_q(w).shape == (32, 128, 192)
    assert W.gen_w_uk(w).shape == (128, 128, 512)
    assert not np.array_equal(W.gen_w_uk(w), W.gen_w_uv(w))


def test_weight_and_data_statistics():
    w = W.WORKLOADS["tiny_h16_b1_l256"]
    wk = W.bf16_bits_to_f32(W.gen_w_uk(w))
    assert abs(wk.std() - 1 / np.sqrt(512)) < 2e-3 * 1 / np.sqrt(512) * 50
    rows = W.bf16_bits_to_f32(W.gen_rows(w, 0, 256))
    assert abs(rows.std() - 1.0) < 0.02 and abs(rows.mean()) < 0.02


def test_variable_lengths_and_block_table():
    w = W.WORKLOADS["paged_b64_l1k_32k"]
    lens = W.seq_lens(w)
    assert lens.shape == (64,) and lens.min() >= 1024 and lens.max() <= 32768
    bt, pool = W.gen_block_table(w, lens)
    npg = W.pages_per_seq(lens)
    assert pool == int(npg.sum())
    used = np.concatenate([bt[b, :n] for b, n in enumerate(npg)])
    np.testing.assert_array_equal(np.sort(used), np.arange(pool))
    for b, n in enumerate(npg):
        assert np.all(bt[b, n:] == -1)


def test_paged_layout_places_every_token():
    w = W.Workload("t", n_h=16, batch=3, ctx_range=(1, 200), paged=True)
    lens = W.seq_lens(w)
    bt, pool = W.gen_block_table(w, lens)
    rows = [W.gen_rows(w, b, int(L)) for b, L in enumerate(lens)]
    P = W.layout_paged(rows, bt, pool)
    for b, L in enumerate(lens):
        for t in range(int(L)):
            np.testing.assert_array_equal(P[bt[b, t // 64], t % 64], rows[b][t])
        tail = int(L) % 64
        if tail:
            assert np.all(P[bt[b, (int(L) - 1) // 64], tail:] == 0)


def test_cache_bytes():
    assert W.cache_bytes(W.WORKLOADS["v2_b32_l4096"]) == 150_994_944
    assert W.cache_bytes(W.WORKLOADS["long_b4_l128k"]) == 603_979_776
    assert W.cache_bytes(W.WORKLOADS["fp8_b128_l8192"]) == 608_174_080
    assert W.cache_bytes(W.WORKLOADS["tiny_h16_b1_l256"]) == 294_912
