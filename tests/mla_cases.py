"""Helpers for GPU tests: build a workload's device tensors from the seeded generator,
run the library, and evaluate the oracle on chosen (sequence, head) samples."""

from __future__ import annotations

import os

import numpy as np

import workloads as W
from oracle import fp8_e4m3, mla_oracle

MAX_REL = 2e-2      # max|gpu - oracle| <= MAX_REL * max|oracle|
MEAN_REL = 3e-3     # sum|gpu - oracle| / sum|oracle| <= MEAN_REL


bits_to_torch_bf16 = W.bits_to_torch_bf16


def rows_f32(bits: np.ndarray) -> np.ndarray:
    return W.bf16_bits_to_f32(bits)


class Case(W.DeviceInputs):
    """A workload on the device, its cache in the library's format (e4m3 workloads are
    quantised by the library's own cache writer), plus the oracle for any sequence."""

    def __init__(self, w: W.Workload, device, lens=None, keep_rows: bool = False):
        import mla_latent_kv_69_b300 as mla

        super().__init__(w, device, lens=lens, keep_rows=keep_rows)
        if w.kv == "fp8":
            codes, scales = mla.quantize_fp8(self.source)
            self.cache = mla.Cache(codes, scales, self.block_table)
        else:
            self.cache = mla.Cache(self.source, None, self.block_table)

    def rebuild_cache(self):
        """Re-make the library's cache view after `source` changed (re-quantises e4m3)."""
        import mla_latent_kv_69_b300 as mla

        if self.w.kv == "fp8":
            codes, scales = mla.quantize_fp8(self.source)
            self.cache = mla.Cache(codes, scales, self.block_table)
        else:
            self.cache = mla.Cache(self.source, None, self.block_table)

    def set_rows(self, b: int, tokens, rows_bits: np.ndarray):
        """Overwrite cache rows (bf16 bits [len(tokens), 576]) of sequence b on the host
        copy and in the device `source`; call rebuild_cache() afterwards."""
        import torch

        tokens = np.asarray(tokens, dtype=np.int64)
        host = self.rows_of(b).copy()
        host[tokens] = rows_bits
        self.rows[b] = host
        dev_rows = bits_to_torch_bf16(np.ascontiguousarray(rows_bits), self.device)
        if self.block_table_np is None:
            self.source[b, torch.from_numpy(tokens).to(self.device)] = dev_rows
        else:
            pages = self.block_table_np[b, tokens // 64].astype(np.int64)
            self.source[torch.from_numpy(pages).to(self.device), torch.from_numpy(tokens % 64).to(self.device)] = dev_rows

    def scale_queries(self, factor):
        """Multiply the queries by `factor` (a number, or one per sequence), rounded to
        bf16, on the host and the device."""
        f = np.broadcast_to(np.asarray(factor, np.float32), (self.B,))[:, None, None]
        self.q_bits = W.f32_to_bf16_bits(rows_f32(self.q_bits) * f)
        self.q = bits_to_torch_bf16(self.q_bits, self.device)

    def run(self, n_splits: int = 0, status=None, bufs=None):
        import mla_latent_kv_69_b300 as mla

        return mla.decode_step(self.q, self.w_uk, self.w_uv, self.cache, self.seq_lens, self.pos, self.max_len,
                               n_splits=n_splits, status=status, bufs=bufs)

    # ---------------- oracle side ----------------
    def oracle_rows(self, b: int) -> np.ndarray:
        """fp64 cache rows of sequence b as the oracle sees them."""
        src = rows_f32(self.rows_of(b))
        if self.w.kv == "fp8":
            codes, scales = fp8_e4m3.quantize_rows(src)
            return fp8_e4m3.dequantize_rows(codes, scales)
        return src.astype(np.float64)

    def oracle(self, b: int, heads=None):
        rows = self.oracle_rows(b)
        q = rows_f32(self.q_bits[b])
        wk = rows_f32(self.wuk_bits)
        wv = rows_f32(self.wuv_bits)
        return mla_oracle.attend_explicit(q, rows[:, :512], rows[:, 512:], wk, wv, pos_q=int(self.pos_np[b]),
                                          heads=heads)


def lse_tolerance(case, b: int, heads) -> np.ndarray:
    """Per-head bound on |lse_gpu - lse_oracle| from the one rounding the scores carry:
    the absorbed query q_lat = [W_UK^T q^C ‖ RoPE(q^R)] is stored in bf16, an error of at
    most half an ulp (2^-8 relative) per element, uniform and independent, so the error
    of score s_t has std <= 2^-8/sqrt(3) · scale · ||q_lat ⊙ row_t||_2. The lse is a
    softmax-weighted mean of score errors; six of those stds over the worst token bounds
    it, plus 1e-4 for the fp32 normaliser and the exp2 approximation."""
    rows = case.oracle_rows(b)
    if rows.shape[0] == 0:
        return np.zeros(len(heads))
    q = rows_f32(case.q_bits[b]).astype(np.float64)
    wk = rows_f32(case.wuk_bits).astype(np.float64)
    hs = list(heads)
    q_lat = np.concatenate([np.einsum("hd,hdj->hj", q[hs, :128], wk[hs]),
                            mla_oracle.rope(q[hs, 128:], int(case.pos_np[b]))], axis=1)   # [h, 576]
    norms = np.sqrt(np.einsum("hj,tj->ht", q_lat * q_lat, rows * rows)).max(axis=1)
    return 6.0 * 2.0 ** -8 / np.sqrt(3.0) * mla_oracle.default_scale() * norms + 1e-4


def tol_stats(got: np.ndarray, ref: np.ndarray) -> tuple[float, float]:
    err = np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))
    ref_abs = np.abs(np.asarray(ref, np.float64))
    max_rel = err.max() / max(ref_abs.max(), 1e-300)
    mean_rel = err.sum() / max(ref_abs.sum(), 1e-300)
    return float(max_rel), float(mean_rel)


def assert_within_tolerance(got, ref, what=""):
    mx, mn = tol_stats(got, ref)
    log = os.environ.get("MLA_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(f"{os.environ.get('PYTEST_CURRENT_TEST', '?').split(' ')[0]}\t{what}\tmax_rel={mx:.3e}\tmean_rel={mn:.3e}\n")
    assert mx <= MAX_REL and mn <= MEAN_REL, f"{what}: max_rel={mx:.3e} mean_rel={mn:.3e}"
    return mx, mn
