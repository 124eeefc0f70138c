"""GPU parity: the library's decode step (absorb_q, decode_fwd, combine_up_v through the
C ABI) against the fp64 oracle
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
from mla_cases import Case, assert_within_tolerance, bits_to_torch_bf16, lse_tolerance, rows_f32
from oracle import fp8_e4m3, mla_oracle

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
            err = np.abs(lse[b, hs] - r["lse"][hs])
            tol = lse_tolerance(case, b, hs)
            assert np.all(err <= tol), f"lse of sequence {b}: worst error {err.max():.3e}, " \
                                       f"error/bound up to {np.max(err / tol):.2f}"
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
    ("h64_fp8", W.Workload("s9", n_h=64, batch=2, ctx=0, kv="fp8", seed=11), [300, 129]),
    ("h32_fp8_paged", W.Workload("s10", n_h=32, batch=2, ctx=0, kv="fp8", paged=True, seed=12), [513, 70]),
    ("h16_fp8", W.Workload("s11", n_h=16, batch=2, ctx=0, kv="fp8", seed=13), [257, 2]),
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
    assert mla.decode_kernel("fp8", 128) == "tcgen05_e4m3"
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    out = case.run(n_splits=3, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _compare(case, out, [(b, None) for b in range(case.B)])


FULL = {
    "v2_b32_l4096": lambda c: [(0, None), (c.B - 1, None)],
    "paged_b64_l1k_32k": lambda c: [(int(np.argmin(c.lens)), None), (int(np.argmax(c.lens)), [0, 1, 2, 127]),
                                    (0, list(range(0, 128, 16)))],
    "long_b4_l128k": lambda c: [(0, list(range(0, 128, 16))), (1, [5, 64, 101]), (2, [30, 127]),
                                (3, list(range(3, 128, 24)))],
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


# ------------------------------------------------------------------------------------
# The lazy running maximum: a head's maximum is raised only when a tile beats it by more
# than 2^8 (log2 units), and then the value CTA rescales that head's rows of O in TMEM.
# N(0, 1) inputs never trigger it after the first tile, so these cases plant tokens whose
# latent lies along the heads' absorbed queries with growing strength.
# ------------------------------------------------------------------------------------
SPIKES = [(300, 300.0), (700, 600.0), (1600, 1100.0), (2990, 2000.0)]   # (token, strength)


def _absorbed_direction(case, b):
    """Unit vector along sum_h W_UK[h]^T q^C[b, h] (fp64, test-side)."""
    q = rows_f32(case.q_bits[b]).astype(np.float64)
    wk = rows_f32(case.wuk_bits).astype(np.float64)
    g = np.einsum("hd,hdj->j", q[:, :128], wk)
    return g / np.linalg.norm(g)


def _plant_spikes(case, spikes):
    for b in range(case.B):
        g = _absorbed_direction(case, b)
        toks = [t for t, _ in spikes if t < case.lens[b]]
        rows = np.zeros((len(toks), 576), np.float32)
        for k, (t, a) in enumerate(spikes[:len(toks)]):
            rows[k, :512] = a * g
        case.set_rows(b, toks, W.f32_to_bf16_bits(rows))
    case.rebuild_cache()


def _count_rescales(case, b, n_splits):
    """Rescales of O the kernel's schedule performs for sequence b (heads x events),
    replayed on the oracle's scores: per split, per 128-token tile, a head whose tile
    maximum exceeds its running maximum by more than 8 (log2) after the first raise.
    For an e4m3 cache the running maximum is taken over the score plus log2 of the
    token's scale (the log2 weight of the codes)."""
    rows = case.oracle_rows(b)
    q = rows_f32(case.q_bits[b])
    from oracle import mla_oracle
    out = mla_oracle.attend_explicit(q, rows[:, :512], rows[:, 512:], rows_f32(case.wuk_bits),
                                     rows_f32(case.wuv_bits), pos_q=int(case.pos_np[b]), return_p=True)
    with np.errstate(divide="ignore"):
        y = (np.log(out["p"]) + out["lse"][:, None]) / np.log(2.0)
    if case.w.kv == "fp8":
        _, scales = fp8_e4m3.quantize_rows(rows_f32(case.rows_of(b)))
        y = y + np.log2(scales.astype(np.float64))[None, :]
    L = int(case.lens[b])
    events = 0
    for sp in range(n_splits):
        st, en = mla.split_range(L, n_splits, sp)
        m = np.full(case.n_h, -np.inf)
        for t0 in range(st, en, 128):
            mt = y[:, t0:min(t0 + 128, en)].max(axis=1)
            rise = mt > m + 8.0
            events += int(np.sum(rise & np.isfinite(m)))
            m = np.where(rise, mt, m)
    return events


RESCALE = [
    ("bf16_contig", W.Workload("r1", n_h=128, batch=2, ctx=0, seed=41)),
    ("bf16_paged", W.Workload("r2", n_h=128, batch=2, ctx=0, paged=True, seed=42)),
    ("fp8", W.Workload("r3", n_h=128, batch=2, ctx=0, kv="fp8", seed=43)),
    ("fp8_paged_h64", W.Workload("r4", n_h=64, batch=2, ctx=0, kv="fp8", paged=True, seed=44)),
]


@pytest.mark.parametrize("name,w", RESCALE, ids=[r[0] for r in RESCALE])
@pytest.mark.parametrize("n_splits", [1, 3, 0])
def test_running_max_rises_rescale_o(cuda_device, name, w, n_splits):
    case = Case(w, cuda_device, lens=[3000, 2500], keep_rows=True)
    _plant_spikes(case, SPIKES)
    S = n_splits if n_splits else mla.num_splits(case.B, case.max_len, case.n_h)
    events = sum(_count_rescales(case, b, S) for b in range(case.B))
    if n_splits:   # the automatic split count leaves about two tiles per split: no later tile can rise
        # most heads rescale at every planted token after the first in a split
        assert events >= case.n_h, f"the case triggers only {events} rescales"
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    out = case.run(n_splits=n_splits, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _compare(case, out, [(b, None) for b in range(case.B)])


# ------------------------------------------------------------------------------------
# Magnitudes. The e4m3 path works on f16 operands, so rows of very small or very large
# magnitude (per-token scales from 2e-8 to 2e2) and absorbed queries far above f16's
# maximum (65504) or below its normal range must not lose what matters. The decode and
# merge calls are fed a query drawn directly (bf16) and compared with the oracle's
# latent form on the same query; going through the absorption step instead would add the
# bf16 rounding of the absorbed query, whose effect on the scores grows with their spread
# (at a spread of ~30 natural units it alone reaches the tolerance, for any kernel).
# ------------------------------------------------------------------------------------
MAGNITUDES = [   # (row factor, absorbed-query factor); None = per-token factors 10^U(-3, 3)
    (1e-3, 3e3), (1e-2, 500.0), (1e2, 0.05), (1e3, 0.005), (None, 0.005), (1.0, 30.0), (1e-5, 1e5), (1e5, 1e-5),
    (1.0, 1e3),
]


@pytest.mark.parametrize("kv,paged", [("fp8", False), ("fp8", True), ("bf16", False), ("bf16", True)])
def test_row_and_query_magnitudes(cuda_device, kv, paged):
    lens = [300, 257, 700, 129, 900, 450, 200, 333, 520]
    w = W.Workload("mag", n_h=128, batch=len(lens), ctx=0, kv=kv, paged=paged, seed=51)
    case = Case(w, cuda_device, lens=lens, keep_rows=True)
    rng = np.random.default_rng(5100)
    for b, (f, _) in enumerate(MAGNITUDES):
        L = lens[b]
        fac = np.float32(f) if f is not None else (10.0 ** rng.uniform(-3, 3, (L, 1))).astype(np.float32)
        case.set_rows(b, np.arange(L), W.f32_to_bf16_bits(rows_f32(case.rows_of(b)) * fac))
    case.rebuild_cache()
    q_lat_bits = W.f32_to_bf16_bits(rows_f32(W.gen_q_lat(w)) * np.array([g for _, g in MAGNITUDES], np.float32)[:, None, None])
    q_lat = bits_to_torch_bf16(q_lat_bits, cuda_device)
    q64 = rows_f32(q_lat_bits).astype(np.float64)
    for n_splits in (1, 3, 0):
        status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
        o_part, lse_part = mla.decode_fwd(q_lat, case.cache, case.seq_lens, case.max_len, n_splits=n_splits,
                                          status=status)
        o_lat, lse = mla.combine(o_part, lse_part)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        o_lat, lse = o_lat.double().cpu().numpy(), lse.double().cpu().numpy()
        for b in range(case.B):   # one sequence at a time: their outputs differ by 1e8 in size
            ref = mla_oracle.attend_latent(q64[b], case.oracle_rows(b))
            assert_within_tolerance(o_lat[b], ref["o_lat"], f"o_lat, sequence {b}")
            # the query is exact here: the fp32 scores and normaliser leave ~1e-6 relative
            np.testing.assert_allclose(lse[b], ref["lse"], rtol=2e-5, atol=2e-4)
    if kv == "fp8":
        for b in range(case.B):
            _fp8_codes_match(case, b)


@pytest.mark.parametrize("name,lens", [
    # ragged: about 480 tiles on the SM pairs, so pairs walk several pieces of several sequences
    ("many_ragged", list(np.random.default_rng(61).integers(1, 700, size=160))),
    # equal tile counts: each sequence cut into equal pieces (the split plan)
    ("equal_lengths", [5120, 5100, 5080]),
])
def test_paged_persistent_schedule(cuda_device, name, lens):
    """The paged cache under the library schedule runs the persistent kernel: every slot's
    piece of every sequence, merged, against the latent form of the oracle (absorbed query
    drawn directly), every head of every sequence."""
    w = W.Workload("sched", n_h=128, batch=len(lens), ctx=0, paged=True, seed=62)
    case = Case(w, cuda_device, lens=lens, keep_rows=True)
    q_lat_bits = W.gen_q_lat(w)
    q_lat = bits_to_torch_bf16(q_lat_bits, cuda_device)
    q64 = rows_f32(q_lat_bits).astype(np.float64)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    o_part, lse_part = mla.decode_fwd(q_lat, case.cache, case.seq_lens, case.max_len, n_splits=0, status=status)
    o_lat, lse = mla.combine(o_part, lse_part)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o_lat, lse = o_lat.double().cpu().numpy(), lse.double().cpu().numpy()
    got, ref = [], []
    for b in range(case.B):
        r = mla_oracle.attend_latent(q64[b], case.oracle_rows(b))
        got.append(o_lat[b].ravel())
        ref.append(r["o_lat"].ravel())
        np.testing.assert_allclose(lse[b], r["lse"], rtol=2e-5, atol=2e-4)
    assert_within_tolerance(np.concatenate(got), np.concatenate(ref), "o_lat")
