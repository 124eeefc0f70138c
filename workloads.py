"""Seeded synthetic inputs for the MLA latent-cache decode workloads.

This module is shared by the tests, the oracle side and the CUDA side. It holds
no attention, RoPE or quantisation arithmetic: it only draws numbers, rounds them
to bf16 storage and lays rows out in HBM order (contiguous or paged).

Workload shapes follow the model on the pages: 128 heads, d_c = 512, d_h^R = 64,
d_h = 128 ("DeepSeek-V2: A Strong, Economical, and Efficient Mixture-of-Experts
Language Model - 中文验证版", §计算设置 and §方法适配). The pages' own serving workload
(DeepSeek 67B's production prompt/generation length mix, same page §证据) is not
published; uniform context lengths stand in for it.

Recipe (every tensor has its own counter-keyed stream, so any single sequence can
be regenerated alone):
  * stream(tag, *index) = numpy Generator(PCG64(SeedSequence([seed, tag, *index])))
  * q [B, n_h, 192]           ~ N(0, 1)           → bf16 (round to nearest even)
  * cache rows of sequence b  [L_b, 576] ~ N(0,1) → bf16; columns 0..511 are c_KV,
    512..575 the decoupled RoPE key as stored (already rotated at its position)
  * W_UK, W_UV [n_h, 128, 512] ~ N(0, 1/512)      → bf16
  * variable lengths: integers uniform on [lo, hi] inclusive
  * paged layout: 64-token pages; the pool holds exactly sum_b ceil(L_b/64) pages,
    assigned to (b, page) slots by one random permutation; page tails are zero
The query of sequence b sits at position L_b - 1.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

D_NOPE = 128
D_ROPE = 64
D_LATENT = 512
D_ROW = 576
D_Q = 192
PAGE = 64

TAG_Q, TAG_ROWS, TAG_WUK, TAG_WUV, TAG_LENS, TAG_PAGES, TAG_QLAT = 1, 2, 3, 4, 5, 6, 7
TAG_H, TAG_WDKV, TAG_WKR = 8, 9, 10
D_MODEL = 5120   # hidden size ([A] §"8.1T token 预训练配置与 H800 成本账"; [B] §"计算设置")


@dataclass(frozen=True)
class Workload:
    name: str
    n_h: int
    batch: int
    ctx: int = 0                      # uniform context length (when ctx_range is None)
    ctx_range: tuple | None = None    # (lo, hi) inclusive uniform lengths
    paged: bool = False
    kv: str = "bf16"                  # "bf16" | "fp8"
    seed: int = 0
    note: str = ""

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_h16_b1_l256", n_h=16, batch=1, ctx=256,
                 note="tiny decode, 16 heads, one sequence of 256 tokens"),
        Workload("v2_b32_l4096", n_h=128, batch=32, ctx=4096,
                 note="DeepSeek-V2 shape, batch 32, contiguous bf16 cache of 4096 tokens"),
        Workload("paged_b64_l1k_32k", n_h=128, batch=64, ctx_range=(1024, 32768), paged=True,
                 note="V2 shape, batch 64, lengths uniform in [1024, 32768], 64-token pages"),
        Workload("long_b4_l128k", n_h=128, batch=4, ctx=131072,
                 note="V2 shape, batch 4, contiguous bf16 cache of 131072 tokens"),
        Workload("fp8_b128_l8192", n_h=128, batch=128, ctx=8192, kv="fp8",
                 note="V2 shape, batch 128, 8192 tokens, e4m3 cache with a per-token fp32 scale"),
    ]
}
WORKLOAD_ORDER = list(WORKLOADS)


def stream(seed: int, tag: int, *index: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, *index])))


# bf16 storage: round fp32 to the nearest bf16 (ties to even) and keep the 16-bit pattern.
def f32_to_bf16_bits(x) -> np.ndarray:
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return f32_to_bf16_bits(x)


def seq_lens(w: Workload) -> np.ndarray:
    if w.ctx_range is None:
        return np.full(w.batch, w.ctx, dtype=np.int32)
    lo, hi = w.ctx_range
    return stream(w.seed, TAG_LENS).integers(lo, hi, size=w.batch, endpoint=True).astype(np.int32)


def gen_q(w: Workload) -> np.ndarray:
    """bf16 bits [B, n_h, 192]."""
    return _normal_bf16(stream(w.seed, TAG_Q), (w.batch, w.n_h, D_Q))


def gen_q_lat(w: Workload) -> np.ndarray:
    """bf16 bits [B, n_h, 576], N(0, 1): an absorbed query drawn directly, for feeding the
    decode call without the absorption step."""
    return _normal_bf16(stream(w.seed, TAG_QLAT), (w.batch, w.n_h, D_ROW))


def gen_w_uk(w: Workload) -> np.ndarray:
    """bf16 bits [n_h, 128, 512], N(0, 1/512)."""
    return _normal_bf16(stream(w.seed, TAG_WUK), (w.n_h, D_NOPE, D_LATENT), std=1.0 / np.sqrt(512.0))


def gen_w_uv(w: Workload) -> np.ndarray:
    return _normal_bf16(stream(w.seed, TAG_WUV), (w.n_h, D_NOPE, D_LATENT), std=1.0 / np.sqrt(512.0))


def gen_hidden(seed: int, T: int, d: int = D_MODEL) -> np.ndarray:
    """bf16 bits [T, d], N(0, 1): hidden states of new tokens (the cache write's input)."""
    return _normal_bf16(stream(seed, TAG_H), (T, d))


def gen_w_dkv(seed: int, d: int = D_MODEL) -> np.ndarray:
    """bf16 bits [512, d], N(0, 1/d): the down-projection to the latent."""
    return _normal_bf16(stream(seed, TAG_WDKV), (D_LATENT, d), std=1.0 / np.sqrt(d))


def gen_w_kr(seed: int, d: int = D_MODEL) -> np.ndarray:
    """bf16 bits [64, d], N(0, 1/d): the projection to the shared RoPE key."""
    return _normal_bf16(stream(seed, TAG_WKR), (D_ROPE, d), std=1.0 / np.sqrt(d))


def gen_rows(w: Workload, b: int, length: int) -> np.ndarray:
    """bf16 bits [length, 576] for sequence b (c_KV ‖ stored RoPE key)."""
    return _normal_bf16(stream(w.seed, TAG_ROWS, b), (length, D_ROW))


def positions(lens) -> np.ndarray:
    """Query position of each sequence: the newest cached token."""
    return np.maximum(np.asarray(lens, dtype=np.int32) - 1, 0).astype(np.int32)


def pages_per_seq(lens) -> np.ndarray:
    return (np.asarray(lens, dtype=np.int64) + PAGE - 1) // PAGE


def gen_block_table(w: Workload, lens) -> tuple[np.ndarray, int]:
    """(block_table int32 [B, max_pages] with -1 in unused slots, pool page count)."""
    npg = pages_per_seq(lens)
    total = int(npg.sum())
    max_pages = max(int(npg.max()) if len(npg) else 0, 1)
    perm = stream(w.seed, TAG_PAGES).permutation(total).astype(np.int32)
    bt = np.full((len(npg), max_pages), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(npg):
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt, total


# ------------------------------ HBM layouts ---------------------------------------
def layout_contiguous(rows_per_seq, seq_stride: int) -> np.ndarray:
    """[B, seq_stride, 576] uint16 (bf16 bits) with zero tails."""
    B = len(rows_per_seq)
    out = np.zeros((B, seq_stride, D_ROW), dtype=np.uint16)
    for b, r in enumerate(rows_per_seq):
        out[b, : r.shape[0]] = r
    return out


def layout_paged(rows_per_seq, block_table, pool_pages: int, dtype=np.uint16) -> np.ndarray:
    """[pool_pages, 64, W] pool; sequence b's token t lives at page block_table[b, t//64], row t%64."""
    width = rows_per_seq[0].shape[1] if len(rows_per_seq) else D_ROW
    pool = np.zeros((pool_pages, PAGE, width), dtype=dtype)
    for b, r in enumerate(rows_per_seq):
        L = r.shape[0]
        for j in range((L + PAGE - 1) // PAGE):
            seg = r[j * PAGE:(j + 1) * PAGE]
            pool[block_table[b, j], : seg.shape[0]] = seg
    return pool


def layout_paged_1d(vals_per_seq, block_table, pool_pages: int, dtype=np.float32, fill=0) -> np.ndarray:
    """Per-token scalars (e.g. fp8 scales) in the same paged order: [pool_pages, 64]."""
    pool = np.full((pool_pages, PAGE), fill, dtype=dtype)
    for b, v in enumerate(vals_per_seq):
        L = v.shape[0]
        for j in range((L + PAGE - 1) // PAGE):
            seg = v[j * PAGE:(j + 1) * PAGE]
            pool[block_table[b, j], : seg.shape[0]] = seg
    return pool


def cache_bytes(w: Workload, lens=None) -> int:
    """Algorithmic cache bytes one decode step must read: 576 elements per token
    (2 bytes each in bf16; 1 byte each plus a 4-byte scale in fp8)."""
    lens = seq_lens(w) if lens is None else lens
    tokens = int(np.sum(lens, dtype=np.int64))
    per_tok = D_ROW * 2 if w.kv == "bf16" else D_ROW + 4
    return tokens * per_tok


# ------------------------------ device upload ---------------------------------------
def bits_to_torch_bf16(bits: np.ndarray, device):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


class DeviceInputs:
    """A workload's inputs uploaded to one device (torch tensors): q, w_uk, w_uv,
    pos, seq_lens, the bf16 cache rows `source` (contiguous [B, stride, 576] or
    paged [pages, 64, 576]) and the block table. Rows of each generated sequence
    are kept on the host when keep_rows is set."""

    def __init__(self, w: Workload, device, lens=None, keep_rows: bool = False):
        import torch

        self.w = w
        self.device = device
        self.lens = np.asarray(seq_lens(w) if lens is None else lens, dtype=np.int32)
        self.B, self.n_h = w.batch, w.n_h
        self.max_len = int(self.lens.max()) if len(self.lens) else 0
        self.q_bits, self.wuk_bits, self.wuv_bits = gen_q(w), gen_w_uk(w), gen_w_uv(w)
        self.q = bits_to_torch_bf16(self.q_bits, device)
        self.w_uk = bits_to_torch_bf16(self.wuk_bits, device)
        self.w_uv = bits_to_torch_bf16(self.wuv_bits, device)
        self.pos_np = positions(self.lens)
        self.pos = torch.from_numpy(self.pos_np).to(device)
        self.seq_lens = torch.from_numpy(self.lens).to(device)
        self.rows = {}
        if w.paged:
            self.block_table_np, self.pool_pages = gen_block_table(w, self.lens)
            rows = [gen_rows(w, b, int(L)) for b, L in enumerate(self.lens)]
            if keep_rows:
                self.rows = dict(enumerate(rows))
            self.source = bits_to_torch_bf16(layout_paged(rows, self.block_table_np, self.pool_pages), device)
            del rows
            self.block_table = torch.from_numpy(self.block_table_np).to(device)
        else:
            self.block_table_np, self.block_table, self.pool_pages = None, None, 0
            stride = max(self.max_len, 1)
            self.source = torch.zeros(self.B, stride, D_ROW, dtype=torch.bfloat16, device=device)
            for b, L in enumerate(self.lens):
                r = gen_rows(w, b, int(L))
                if keep_rows:
                    self.rows[b] = r
                if L:
                    self.source[b, :L] = bits_to_torch_bf16(r, device)

    def rows_of(self, b: int) -> np.ndarray:
        if b not in self.rows:
            self.rows[b] = gen_rows(self.w, b, int(self.lens[b]))
        return self.rows[b]
