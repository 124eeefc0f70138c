"""B300-native (sm_103a) MLA latent-cache decode: Python binding of libmla_b300.so.

The functions mirror the C ABI in include/mla.h one to one. They only marshal
arguments (shape/dtype/device checks, raw pointers, the current CUDA stream);
every step of the computation runs in the library's CUDA kernels. Buffers are
torch tensors on the GPU; outputs are allocated here when not passed in. All tensors of
a call must live on one CUDA device (ValueError otherwise); the call runs with that
device current, on the given stream or that device's current torch stream.

A decode step of one MLA layer:

    q_lat = absorb_q(q, w_uk, pos)                      # [B, n_h, 576] bf16
    o_part, lse_part = decode_fwd(q_lat, cache, seq_lens, max_seq_len)
    o_lat, lse = combine(o_part, lse_part)              # [B, n_h, 512] fp32
    o = up_v(o_lat, w_uv)                               # [B, n_h, 128] fp32
"""
from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import (MLA_KV_BF16, MLA_KV_FP8_E4M3, MLA_MAX_SPLITS, MlaCache, MlaError, MlaRope, check,
                   status_string)

__all__ = [
    "absorb_q", "decode_fwd", "combine", "up_v", "quantize_fp8", "cache_append", "decode_multi", "num_splits",
    "split_range",
    "decode_kernel",
    "decode_combine_static",
    "compute_dtype",
    "Cache", "Yarn", "MlaError", "status_string", "default_scale", "decode_step", "DecodeStepGraph", "lib_path",
    "MLA_MAX_SPLITS", "test_decode_stalled",
]

D_NOPE, D_ROPE, D_LATENT, D_ROW, D_Q, PAGE = 128, 64, 512, 576, 192, 64


def lib_path() -> str:
    return _lib.LIB_PATH


def default_scale() -> float:
    """1/sqrt(d_h + d_h^R) for the 192-wide query/key pair."""
    return 1.0 / math.sqrt(D_NOPE + D_ROPE)


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device=None) -> int:
    if stream is None:
        if _raw_stream is not None and device is not None and device.index is not None:
            return int(_raw_stream(device.index))   # the device's current torch stream, as a handle
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _one_device(**tensors):
    """The single CUDA device every given tensor lives on (None entries are skipped).

    The library launches on the current device and dereferences every pointer there,
    so a tensor on another GPU would hand a kernel a peer address."""
    dev = None
    for name, t in tensors.items():
        if t is None:
            continue
        d = t.device
        if dev is None:
            dev = d
        elif d != dev:
            raise ValueError(f"{name} is on {d}, but the call's other tensors are on {dev}; "
                             "every tensor of a call must be on one device")
    return dev


def _call(fn: str, device, *args, stream=None):
    """Run one C-ABI call with `device` current, on `stream` (default: that device's
    current torch stream), and raise MlaError on a non-OK status."""
    f = getattr(_lib.get(), fn)
    if device.index is not None and device.index == torch.cuda.current_device():
        check(fn, f(*args, _stream(stream, device)))
        return
    with torch.cuda.device(device):
        check(fn, f(*args, _stream(stream, device)))


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


def _need(t, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _need_table_rows(cache, B):
    bt = cache.block_table
    if bt is not None and (bt.dim() != 2 or bt.shape[0] < B):
        raise ValueError(f"block_table must have a row per sequence: [>= {B}, max_pages]")


@dataclass(frozen=True)
class Yarn:
    """YaRN extension of the decoupled RoPE (mla_rope in include/mla.h); the defaults are
    the pages' setting over a 4K pre-training context."""
    scale: float = 40.0
    alpha: float = 1.0
    beta: float = 32.0
    original_max_pos: int = 4096


def _rope(rope_base: float, yarn: Yarn | None) -> MlaRope:
    r = MlaRope()
    r.base = float(rope_base)
    r.yarn_scale = 1.0 if yarn is None else float(yarn.scale)
    r.yarn_alpha = 0.0 if yarn is None else float(yarn.alpha)
    r.yarn_beta = 0.0 if yarn is None else float(yarn.beta)
    r.original_max_pos = 0 if yarn is None else int(yarn.original_max_pos)
    r.reserved = 0
    return r


@dataclass
class Cache:
    """One layer's latent cache (see mla_cache in include/mla.h).

    data: contiguous [B, stride, 576] or paged [pages, 64, 576]; bf16 or uint8 (e4m3 codes)
    scales: fp32 per row ([B, stride] or [pages, 64]) for e4m3, else None
    block_table: int32 [B, max_pages] for paged, else None
    """
    data: torch.Tensor
    scales: torch.Tensor | None = None
    block_table: torch.Tensor | None = None

    def tensors(self) -> dict:
        """The cache's tensors by name (None where absent), for device checks."""
        return {"cache.data": self.data, "cache.scales": self.scales, "cache.block_table": self.block_table}

    @property
    def dtype_code(self) -> int:
        return MLA_KV_FP8_E4M3 if self.data.dtype in (torch.uint8, torch.float8_e4m3fn) else MLA_KV_BF16

    def to_c(self) -> MlaCache:
        """The C view of the cache, built and checked once per set of tensors (a serving
        loop passes the same cache every step)."""
        key = tuple((id(t), t.data_ptr(), tuple(t.shape), t.dtype) if t is not None else None
                    for t in (self.data, self.scales, self.block_table))
        memo = self.__dict__.get("_c_memo")
        if memo is not None and memo[0] == key:
            return memo[1]
        c = self._build_c()
        self.__dict__["_c_memo"] = (key, c)
        return c

    def _build_c(self) -> MlaCache:
        d = self.data
        if d.dtype not in (torch.bfloat16, torch.uint8, torch.float8_e4m3fn):
            raise TypeError("cache data must be bf16 or uint8/float8_e4m3fn codes")
        if not d.is_cuda or not d.is_contiguous() or d.dim() != 3 or d.shape[-1] != D_ROW:
            raise ValueError("cache data must be a contiguous CUDA tensor [*, *, 576]")
        c = MlaCache()
        c.dtype = self.dtype_code
        c.data = d.data_ptr()
        c.scales = _ptr(self.scales)
        c.num_rows = d.shape[0] * d.shape[1]
        if self.scales is not None:
            _need(self.scales, "scales", torch.float32)
            if self.scales.numel() != c.num_rows:   # the kernels read one scale per row
                raise ValueError(f"scales must hold one fp32 per cache row ({c.num_rows}), got {self.scales.numel()}")
        if self.block_table is not None:
            _need(self.block_table, "block_table", torch.int32)
            if self.block_table.dim() != 2:
                raise ValueError("block_table must be [B, max_pages]")
            if d.shape[1] != PAGE:
                raise ValueError("paged cache data must be [pages, 64, 576]")
            c.block_table = self.block_table.data_ptr()
            c.page_size = PAGE
            c.max_pages = self.block_table.shape[1]
        else:
            c.block_table = None
            c.seq_stride_tokens = d.shape[1]
        return c


def decode_kernel(kv: str, n_h: int) -> str:
    """Name of the decode kernel the library runs for a cache dtype ("bf16"/"fp8") and head count."""
    code = int(_lib.get().mla_decode_kernel(MLA_KV_FP8_E4M3 if kv == "fp8" else MLA_KV_BF16, n_h))
    return {1: "tcgen05_bf16", 2: "tcgen05_e4m3"}.get(code, "invalid")


def compute_dtype(n_h: int, kv: str) -> str:
    """Arithmetic type of the decode kernel's contractions."""
    return {"tcgen05_bf16": "bf16", "tcgen05_e4m3": "e4m3/f16"}.get(decode_kernel(kv, n_h), "?")


def num_splits(B: int, max_seq_len: int, n_h: int) -> int:
    return int(_lib.get().mla_num_splits(B, max_seq_len, n_h))


def split_range(seq_len: int, n_splits: int, split: int) -> tuple[int, int]:
    a, b = ctypes.c_int(), ctypes.c_int()
    check("mla_split_range", _lib.get().mla_split_range(seq_len, n_splits, split, ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def absorb_q(q, w_uk, pos, q_lat=None, rope_base: float = 10000.0, stream=None, yarn: Yarn | None = None):
    B, n_h = q.shape[0], q.shape[1]
    _need(q, "q", torch.bfloat16, (B, n_h, D_Q))
    _need(w_uk, "w_uk", torch.bfloat16, (n_h, D_NOPE, D_LATENT))
    _need(pos, "pos", torch.int32, (B,))
    if q_lat is None:
        q_lat = torch.empty(B, n_h, D_ROW, dtype=torch.bfloat16, device=q.device)
    _need(q_lat, "q_lat", torch.bfloat16, (B, n_h, D_ROW))
    dev = _one_device(q=q, w_uk=w_uk, pos=pos, q_lat=q_lat)
    if yarn is None:
        _call("mla_absorb_q", dev, _ptr(q), _ptr(w_uk), _ptr(pos), B, n_h, float(rope_base), _ptr(q_lat),
              stream=stream)
    else:
        r = _rope(rope_base, yarn)
        _call("mla_absorb_q_ex", dev, _ptr(q), _ptr(w_uk), _ptr(pos), B, n_h, ctypes.byref(r), _ptr(q_lat),
              stream=stream)
    return q_lat


def decode_fwd(q_lat, cache: Cache, seq_lens, max_seq_len: int, softmax_scale: float | None = None,
               n_splits: int = 0, o_part=None, lse_part=None, status=None, stream=None):
    B, n_h = q_lat.shape[0], q_lat.shape[1]
    _need(q_lat, "q_lat", torch.bfloat16, (B, n_h, D_ROW))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    S = n_splits if n_splits > 0 else num_splits(B, max_seq_len, n_h)
    if o_part is None:
        o_part = torch.empty(B, S, n_h, D_LATENT, dtype=torch.float32, device=q_lat.device)
    if lse_part is None:
        lse_part = torch.empty(B, S, n_h, dtype=torch.float32, device=q_lat.device)
    _need(o_part, "o_part", torch.float32, (B, S, n_h, D_LATENT))
    _need(lse_part, "lse_part", torch.float32, (B, S, n_h))
    if status is not None:
        _need(status, "status", torch.int32)
    _need_table_rows(cache, B)
    c = cache.to_c()
    dev = _one_device(q_lat=q_lat, seq_lens=seq_lens, o_part=o_part, lse_part=lse_part, status=status,
                      **cache.tensors())
    scale = default_scale() if softmax_scale is None else float(softmax_scale)
    # n_splits = 0 keeps the library's own schedule (o_part then has S = num_splits() slots)
    _call("mla_decode_fwd", dev, _ptr(q_lat), ctypes.byref(c), _ptr(seq_lens), B, n_h, int(max_seq_len), scale,
          int(n_splits) if n_splits > 0 else 0, _ptr(o_part), _ptr(lse_part), _ptr(status), stream=stream)
    return o_part, lse_part


def test_decode_stalled(q_lat, cache: Cache, seq_lens, max_seq_len: int, status, wait_ns: int,
                        n_splits: int = 0, o_part=None, lse_part=None, stream=None):
    """Test hook (include/mla_test.h): decode_fwd with the cache loads withheld and the
    given wait limit, so the kernel's bounded waits run out and it records
    MLA_ERR_TIMEOUT in `status`. Not part of a decode step."""
    B, n_h = q_lat.shape[0], q_lat.shape[1]
    _need(q_lat, "q_lat", torch.bfloat16, (B, n_h, D_ROW))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    _need(status, "status", torch.int32)
    S = n_splits if n_splits > 0 else num_splits(B, max_seq_len, n_h)
    if o_part is None:
        o_part = torch.empty(B, S, n_h, D_LATENT, dtype=torch.float32, device=q_lat.device)
    if lse_part is None:
        lse_part = torch.empty(B, S, n_h, dtype=torch.float32, device=q_lat.device)
    _need(o_part, "o_part", torch.float32, (B, S, n_h, D_LATENT))
    _need(lse_part, "lse_part", torch.float32, (B, S, n_h))
    _need_table_rows(cache, B)
    c = cache.to_c()
    dev = _one_device(q_lat=q_lat, seq_lens=seq_lens, o_part=o_part, lse_part=lse_part, status=status,
                      **cache.tensors())
    _call("mla_test_decode_stalled", dev, _ptr(q_lat), ctypes.byref(c), _ptr(seq_lens), B, n_h, int(max_seq_len),
          default_scale(), int(n_splits) if n_splits > 0 else 0, _ptr(o_part), _ptr(lse_part), _ptr(status),
          int(wait_ns), stream=stream)
    return o_part, lse_part


def combine(o_part, lse_part, o_lat=None, lse=None, stream=None):
    B, S, n_h = o_part.shape[0], o_part.shape[1], o_part.shape[2]
    _need(o_part, "o_part", torch.float32, (B, S, n_h, D_LATENT))
    _need(lse_part, "lse_part", torch.float32, (B, S, n_h))
    if o_lat is None:
        o_lat = torch.empty(B, n_h, D_LATENT, dtype=torch.float32, device=o_part.device)
    if lse is None:
        lse = torch.empty(B, n_h, dtype=torch.float32, device=o_part.device)
    _need(o_lat, "o_lat", torch.float32, (B, n_h, D_LATENT))
    _need(lse, "lse", torch.float32, (B, n_h))
    dev = _one_device(o_part=o_part, lse_part=lse_part, o_lat=o_lat, lse=lse)
    _call("mla_combine", dev, _ptr(o_part), _ptr(lse_part), B, S, n_h, _ptr(o_lat), _ptr(lse), stream=stream)
    return o_lat, lse


def decode_combine_static(q_lat, cache: Cache, seq_lens, max_seq_len: int, o_lat, lse=None,
                          softmax_scale: float | None = None, n_splits: int = 0, status=None, stream=None):
    """decode_fwd + combine with the split partials in the library's fixed device array
    (see mla_decode_combine_static in include/mla.h); the outputs are the caller's."""
    B, n_h = q_lat.shape[0], q_lat.shape[1]
    _need(q_lat, "q_lat", torch.bfloat16, (B, n_h, D_ROW))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    _need(o_lat, "o_lat", torch.float32, (B, n_h, D_LATENT))
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, n_h))
    if status is not None:
        _need(status, "status", torch.int32)
    _need_table_rows(cache, B)
    c = cache.to_c()
    dev = _one_device(q_lat=q_lat, seq_lens=seq_lens, o_lat=o_lat, lse=lse, status=status, **cache.tensors())
    scale = default_scale() if softmax_scale is None else float(softmax_scale)
    _call("mla_decode_combine_static", dev, _ptr(q_lat), ctypes.byref(c), _ptr(seq_lens), B, n_h,
          int(max_seq_len), scale, int(n_splits), _ptr(o_lat), _ptr(lse), _ptr(status), stream=stream)
    return o_lat, lse


def up_v(o_lat, w_uv, o=None, stream=None):
    B, n_h = o_lat.shape[0], o_lat.shape[1]
    _need(o_lat, "o_lat", torch.float32, (B, n_h, D_LATENT))
    _need(w_uv, "w_uv", torch.bfloat16, (n_h, D_NOPE, D_LATENT))
    if o is None:
        o = torch.empty(B, n_h, D_NOPE, dtype=torch.float32, device=o_lat.device)
    _need(o, "o", torch.float32, (B, n_h, D_NOPE))
    dev = _one_device(o_lat=o_lat, w_uv=w_uv, o=o)
    _call("mla_up_v", dev, _ptr(o_lat), _ptr(w_uv), B, n_h, _ptr(o), stream=stream)
    return o


def combine_up_v(o_part, lse_part, w_uv, o=None, o_lat=None, lse=None, stream=None):
    """combine + up_v in one launch (include/mla.h, mla_combine_up_v): o [B, n_h, 128]
    from the split partials; o_lat and lse are written only when given."""
    B, S, n_h = o_part.shape[0], o_part.shape[1], o_part.shape[2]
    _need(o_part, "o_part", torch.float32, (B, S, n_h, D_LATENT))
    _need(lse_part, "lse_part", torch.float32, (B, S, n_h))
    _need(w_uv, "w_uv", torch.bfloat16, (n_h, D_NOPE, D_LATENT))
    if o is None:
        o = torch.empty(B, n_h, D_NOPE, dtype=torch.float32, device=o_part.device)
    _need(o, "o", torch.float32, (B, n_h, D_NOPE))
    if o_lat is not None:
        _need(o_lat, "o_lat", torch.float32, (B, n_h, D_LATENT))
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, n_h))
    dev = _one_device(o_part=o_part, lse_part=lse_part, w_uv=w_uv, o=o, o_lat=o_lat, lse=lse)
    _call("mla_combine_up_v", dev, _ptr(o_part), _ptr(lse_part), B, S, n_h, _ptr(w_uv), _ptr(o), _ptr(o_lat),
          _ptr(lse), stream=stream)
    return o, o_lat, lse


def cache_append(h, w_dkv, w_kr, seq_ids, pos, cache: Cache, num_seqs: int | None = None,
                 rope_base: float = 10000.0, staging=None, status=None, stream=None, yarn: Yarn | None = None):
    """Write the cache rows of the new tokens (include/mla.h, mla_cache_append):
    row = [W_DKV h ‖ RoPE(W_KR h, pos)] in bf16 at token pos[t] of sequence seq_ids[t].
    h [T, d_model] bf16, w_dkv [512, d_model], w_kr [64, d_model] bf16, seq_ids/pos [T]
    int32. An e4m3 cache needs (or gets allocated here) a bf16 staging buffer [T, 576]."""
    T, d = h.shape[0], h.shape[1]
    _need(h, "h", torch.bfloat16, (T, d))
    _need(w_dkv, "w_dkv", torch.bfloat16, (D_LATENT, d))
    _need(w_kr, "w_kr", torch.bfloat16, (D_ROPE, d))
    _need(seq_ids, "seq_ids", torch.int32, (T,))
    _need(pos, "pos", torch.int32, (T,))
    if num_seqs is None:
        num_seqs = cache.block_table.shape[0] if cache.block_table is not None else cache.data.shape[0]
    if cache.dtype_code == MLA_KV_FP8_E4M3:
        if staging is None:
            staging = torch.empty(T, D_ROW, dtype=torch.bfloat16, device=h.device)
        _need(staging, "staging", torch.bfloat16, (T, D_ROW))
    if status is not None:
        _need(status, "status", torch.int32)
    c = cache.to_c()
    dev = _one_device(h=h, w_dkv=w_dkv, w_kr=w_kr, seq_ids=seq_ids, pos=pos, staging=staging, status=status,
                      **cache.tensors())
    r = _rope(rope_base, yarn)
    _call("mla_cache_append_ex", dev, _ptr(h), _ptr(w_dkv), _ptr(w_kr), _ptr(seq_ids), _ptr(pos), T, d,
          ctypes.byref(r), ctypes.byref(c), int(num_seqs), _ptr(staging), _ptr(status), stream=stream)


def quantize_fp8(rows, codes=None, scales=None, stream=None):
    """rows [..., 576] bf16 → (codes uint8 [..., 576], scales fp32 [...])."""
    if rows.dtype != torch.bfloat16 or rows.shape[-1] != D_ROW:
        raise TypeError("rows must be bf16 [..., 576]")
    lead = tuple(rows.shape[:-1])
    n = int(math.prod(lead))
    if codes is None:
        codes = torch.empty(*lead, D_ROW, dtype=torch.uint8, device=rows.device)
    if scales is None:
        scales = torch.empty(*lead, dtype=torch.float32, device=rows.device)
    _need(rows, "rows", torch.bfloat16)
    _need(codes, "codes", torch.uint8, (*lead, D_ROW))
    _need(scales, "scales", torch.float32, lead)
    dev = _one_device(rows=rows, codes=codes, scales=scales)
    _call("mla_quantize_fp8", dev, _ptr(rows), n, _ptr(codes), _ptr(scales), stream=stream)
    return codes, scales


def quantize_fp6(rows, packed=None, scales=None, stream=None):
    """rows [..., 576] bf16 → (packed uint8 [..., 432], scale bytes uint8 [..., 18]): the
    ~6-bit cache format of include/mla.h, mla_quantize_fp6 (e2m3 codes in 32-element
    blocks sharing a power-of-two scale)."""
    if rows.dtype != torch.bfloat16 or rows.shape[-1] != D_ROW:
        raise TypeError("rows must be bf16 [..., 576]")
    lead = tuple(rows.shape[:-1])
    n = int(math.prod(lead))
    if packed is None:
        packed = torch.empty(*lead, D_ROW * 6 // 8, dtype=torch.uint8, device=rows.device)
    if scales is None:
        scales = torch.empty(*lead, D_ROW // 32, dtype=torch.uint8, device=rows.device)
    _need(rows, "rows", torch.bfloat16)
    _need(packed, "packed", torch.uint8, (*lead, D_ROW * 6 // 8))
    _need(scales, "scales", torch.uint8, (*lead, D_ROW // 32))
    if n == 0:   # empty tensors may have no storage to point at
        return packed, scales
    dev = _one_device(rows=rows, packed=packed, scales=scales)
    _call("mla_quantize_fp6", dev, _ptr(rows), n, _ptr(packed), _ptr(scales), stream=stream)
    return packed, scales


def decode_step(q, w_uk, w_uv, cache: Cache, seq_lens, pos, max_seq_len: int, n_splits: int = 0,
                softmax_scale: float | None = None, rope_base: float = 10000.0, bufs: dict | None = None,
                status=None, stream=None, yarn: Yarn | None = None, latent: bool = True):
    """One decode step: absorb_q, decode_fwd, then combine and up_v as one launch
    (combine_up_v). `bufs` (optional) holds preallocated outputs. With latent=False the
    merged o_lat and lse are not written (None in the result)."""
    bufs = {} if bufs is None else bufs
    q_lat = absorb_q(q, w_uk, pos, q_lat=bufs.get("q_lat"), rope_base=rope_base, stream=stream, yarn=yarn)
    o_part, lse_part = decode_fwd(q_lat, cache, seq_lens, max_seq_len, softmax_scale, n_splits,
                                  o_part=bufs.get("o_part"), lse_part=bufs.get("lse_part"), status=status,
                                  stream=stream)
    o_lat = lse = None
    if latent:
        B, n_h = q_lat.shape[0], q_lat.shape[1]
        o_lat = bufs.get("o_lat")
        if o_lat is None:
            o_lat = torch.empty(B, n_h, D_LATENT, dtype=torch.float32, device=q_lat.device)
        lse = bufs.get("lse")
        if lse is None:
            lse = torch.empty(B, n_h, dtype=torch.float32, device=q_lat.device)
    o, o_lat, lse = combine_up_v(o_part, lse_part, w_uv, o=bufs.get("o"), o_lat=o_lat, lse=lse, stream=stream)
    return dict(q_lat=q_lat, o_part=o_part, lse_part=lse_part, o_lat=o_lat, lse=lse, o=o)


def decode_multi(q, w_uk, w_uv, cache: Cache, seq_lens, max_seq_len: int, n_splits: int = 0,
                 softmax_scale: float | None = None, rope_base: float = 10000.0, status=None, stream=None,
                 yarn: Yarn | None = None):
    """T new query tokens per sequence (include/mla.h, mla_multi_token_view): the last T
    cached tokens of sequence b are its new ones, query j sits at position L_b - T + j and
    sees tokens 0 .. L_b - T + j. q [B, T, n_h, 192] bf16 → dict of the step's outputs
    with o [B, T, n_h, 128]. The library builds a paged view of the cache with one
    sequence per query and runs the decode step on it."""
    B, T, n_h = q.shape[0], q.shape[1], q.shape[2]
    _need(q, "q", torch.bfloat16, (B, T, n_h, D_Q))
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    mp = max((int(max_seq_len) + PAGE - 1) // PAGE, 1)
    dev_t = q.device
    v_lens = torch.empty(B * T, dtype=torch.int32, device=dev_t)
    v_pos = torch.empty(B * T, dtype=torch.int32, device=dev_t)
    v_table = torch.empty(B * T, mp, dtype=torch.int32, device=dev_t)
    c = cache.to_c()
    view = MlaCache()
    dev = _one_device(q=q, seq_lens=seq_lens, **cache.tensors())
    _call("mla_multi_token_view", dev, ctypes.byref(c), _ptr(seq_lens), B, T, int(max_seq_len), _ptr(v_lens),
          _ptr(v_pos), _ptr(v_table), mp, ctypes.byref(view), stream=stream)
    # the same rows as 64-row pages (the view's block table indexes them)
    pages = cache.data.shape[0] * cache.data.shape[1] // PAGE
    v_cache = Cache(cache.data.view(pages, PAGE, D_ROW),
                    None if cache.scales is None else cache.scales.view(pages, PAGE), v_table)
    out = decode_step(q.view(B * T, n_h, D_Q), w_uk, w_uv, v_cache, v_lens, v_pos, max_seq_len, n_splits=n_splits,
                      softmax_scale=softmax_scale, rope_base=rope_base, status=status, stream=stream, yarn=yarn)
    out["o"] = out["o"].view(B, T, n_h, D_NOPE)
    out["view_seq_lens"], out["view_pos"] = v_lens, v_pos
    return out


class DecodeStepGraph:
    """One decode step of one layer, captured once as a CUDA graph and replayed per step.

    A serving loop repeats the same step on the same buffers, so the host work of the
    three calls (argument checks, tensor maps, launches) is paid once, at capture: the
    graph holds the C-ABI calls of decode_step. Each replay queues, on the graph's own
    stream: the copy of the step's inputs from pinned host buffers (`h_q`, `h_pos`,
    `h_seq_lens`, which the caller fills before each step), the graph, and the copy of
    `o` into the pinned host buffer `h_o`. The copies stay outside the graph: copy nodes
    inside a graph moved the same bytes at about half the rate of the stream copies on
    B300. With latent=True the step also writes `bufs["o_lat"]` and `bufs["lse"]`.

        g = DecodeStepGraph(w_uk, w_uv, cache, B, max_seq_len)
        g.h_q.copy_(...); g.h_pos.copy_(...); g.h_seq_lens.copy_(...)
        g.replay(); g.synchronize()          # g.h_o holds o [B, n_h, 128] fp32

    The cache tensors and weights are captured by address: they must stay allocated
    (their contents may change between steps, e.g. appended tokens). max_seq_len bounds
    every later seq_lens, as for decode_fwd.
    """

    def __init__(self, w_uk, w_uv, cache: Cache, B: int, max_seq_len: int, n_splits: int = 0,
                 softmax_scale: float | None = None, rope_base: float = 10000.0, status=None,
                 yarn: Yarn | None = None, latent: bool = False):
        n_h = w_uk.shape[0]
        dev = w_uk.device
        self.device, self.B, self.n_h = dev, B, n_h
        self.h_q = torch.empty(B, n_h, D_Q, dtype=torch.bfloat16).pin_memory()
        self.h_pos = torch.zeros(B, dtype=torch.int32).pin_memory()
        self.h_seq_lens = torch.zeros(B, dtype=torch.int32).pin_memory()
        self.h_o = torch.empty(B, n_h, D_NOPE, dtype=torch.float32).pin_memory()
        self.d_q = torch.zeros(B, n_h, D_Q, dtype=torch.bfloat16, device=dev)
        self.d_pos = torch.zeros(B, dtype=torch.int32, device=dev)
        self.d_seq_lens = torch.zeros(B, dtype=torch.int32, device=dev)
        S = n_splits if n_splits > 0 else num_splits(B, max_seq_len, n_h)
        self.bufs = dict(
            q_lat=torch.empty(B, n_h, D_ROW, dtype=torch.bfloat16, device=dev),
            o_part=torch.empty(B, S, n_h, D_LATENT, dtype=torch.float32, device=dev),
            lse_part=torch.empty(B, S, n_h, dtype=torch.float32, device=dev),
            o=torch.empty(B, n_h, D_NOPE, dtype=torch.float32, device=dev))
        if latent:
            self.bufs["o_lat"] = torch.empty(B, n_h, D_LATENT, dtype=torch.float32, device=dev)
            self.bufs["lse"] = torch.empty(B, n_h, dtype=torch.float32, device=dev)
        self.stream = torch.cuda.Stream(dev)
        self.graph = torch.cuda.CUDAGraph()
        args = (w_uk, w_uv, cache, self.d_seq_lens, self.d_pos, max_seq_len)
        kw = dict(n_splits=n_splits, softmax_scale=softmax_scale, rope_base=rope_base, bufs=self.bufs, status=status,
                  yarn=yarn, latent=latent)
        with torch.cuda.device(dev), torch.cuda.stream(self.stream):
            # one eager step first: every argument check and launch path runs once outside capture
            decode_step(self.d_q, *args, **kw)
            self.stream.synchronize()
            with torch.cuda.graph(self.graph, stream=self.stream):
                decode_step(self.d_q, *args, **kw)
        self.done = torch.cuda.Event()

    def replay(self):
        """Queue one step on the graph's own stream, after the work already queued on the
        caller's current stream (returns at once)."""
        with torch.cuda.device(self.device):
            self.stream.wait_stream(torch.cuda.current_stream(self.device))
            with torch.cuda.stream(self.stream):
                self.d_q.copy_(self.h_q, non_blocking=True)
                self.d_pos.copy_(self.h_pos, non_blocking=True)
                self.d_seq_lens.copy_(self.h_seq_lens, non_blocking=True)
                self.graph.replay()
                self.h_o.copy_(self.bufs["o"], non_blocking=True)
            self.done.record(self.stream)

    def synchronize(self):
        """Wait until the last replayed step's o is in h_o."""
        self.done.synchronize()
