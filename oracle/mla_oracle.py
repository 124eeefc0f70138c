"""fp64 oracle for one MLA decode step over the latent KV cache.

TEST INFRASTRUCTURE ONLY (see the package docstring): the library never imports this.

What is computed, per sequence and per head h, in the explicit (non-absorbed) form
that [A] §"长上下文推理的第一瓶颈" describes — K and V are up-projected from the cached
latent c_KV at attention time:

    K_{h,t} = [ W_UK[h] · c_t  ‖  k^R_t ]        (128 + 64 = 192 wide)
    V_{h,t} =   W_UV[h] · c_t                    (128 wide)
    q_h     = [ q^C_h ‖ RoPE(q^R_h, p_q) ]       (q^C = first 128, q^R = last 64)
    s_{h,t} = (q_h · K_{h,t}) · scale,   scale = 1/sqrt(d_h + d_h^R) = 1/sqrt(192)
    p_{h,t} = exp(s_{h,t} - max_t s) / sum_t exp(s_{h,t} - max_t s)
    o_h     = sum_t p_{h,t} V_{h,t};   lse_h = max_t s + ln sum_t exp(s - max)
    o^lat_h = sum_t p_{h,t} c_t                  (the latent-space output)

Readings where the pages are silent (each also listed in the design notes):

* Storage of the up-projections is [n_h, d_h = 128, d_c = 512]; K = W_UK[h]·c and
  V = W_UV[h]·c are the only orientations whose shapes compose.
* The cached k^R_t is stored already rotated at its own position t (the write-time
  rotation is what lets the compressed path stay position-free, [A] §"解耦 RoPE 与
  YaRN"). ``rope`` rotates raw keys for callers that model the cache write.
* RoPE uses the rotate-half pairing (i, i + 32), θ_i = p · base^(-2i/64),
  base = 10000. The pages name RoPE but print no formula.
* The decode query sits at position p_q = L - 1 (the newest cached token).
* The softmax scale 1/sqrt(192) is not on the pages; it is the scaled-dot-product
  convention for the 192-wide query/key pair.
* An empty context (L = 0) returns o = 0, o^lat = 0 and lse = -inf.
"""

from __future__ import annotations

import math

import numpy as np

D_H = 128        # per-head query/key/value width (2.25 groups · 2 · d_h = 576 ⇒ d_h = 128)
D_C = 512        # latent width d_c ([A] §长上下文推理的第一瓶颈; [B] §方法适配)
D_R = 64         # decoupled RoPE width d_h^R ([A] §解耦 RoPE 与 YaRN; [B] §方法适配)
D_ROW = D_C + D_R  # 576 cached elements per token per layer
ROPE_BASE = 10000.0


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def default_scale() -> float:
    """1/sqrt(d_h + d_h^R): the query/key pair is 128 + 64 = 192 wide."""
    return 1.0 / math.sqrt(D_H + D_R)


# ---------------------------------------------------------------------------------
# RoPE ([A] §"解耦 RoPE 与 YaRN": position is carried only by the 64-wide decoupled
# query/key pair). Rotate-half pairing, written from the rotation definition.
# ---------------------------------------------------------------------------------
def yarn_inv_freq(width: int, base: float, scale: float, alpha: float, beta: float, original_max_pos: int):
    """Per-pair angular frequencies of RoPE extended by YaRN ([A] §"解耦 RoPE 与 YaRN":
    YaRN on the decoupled key with scale 40, α = 1, β = 32; the pages give no formula,
    so this is the published YaRN frequency rule): pair i's plain frequency θ_i turns
    r_i = L_0 θ_i / (2π) times over the original context L_0; pairs that turn more than
    β times keep θ_i, pairs that turn less than α times are slowed to θ_i / scale, and
    in between the frequency moves linearly in r from one to the other."""
    m = width // 2
    i = np.arange(m, dtype=np.float64)
    theta = base ** (-2.0 * i / width)
    if scale == 1.0:
        return theta
    r = original_max_pos * theta / (2.0 * math.pi)
    gamma = np.clip((r - alpha) / (beta - alpha), 0.0, 1.0)     # 0: fully slowed, 1: unchanged
    return (1.0 - gamma) * theta / scale + gamma * theta


def rope(x, pos, base: float = ROPE_BASE, inv_freq=None) -> np.ndarray:
    """Rotate the last axis of ``x`` (width 2m) by position ``pos``.

    Element pair (i, i + m) is rotated by the angle pos · θ_i, θ_i = base^(-2i/(2m))
    unless ``inv_freq`` (the m frequencies, e.g. from yarn_inv_freq) is given:
        x'_i     = x_i cos(pos θ_i) - x_{i+m} sin(pos θ_i)
        x'_{i+m} = x_{i+m} cos(pos θ_i) + x_i sin(pos θ_i)
    ``pos`` broadcasts against ``x.shape[:-1]``.
    """
    x = _f64(x)
    width = x.shape[-1]
    m = width // 2
    if inv_freq is None:
        i = np.arange(m, dtype=np.float64)
        inv_freq = base ** (-2.0 * i / width)
    theta = _f64(pos)[..., None] * _f64(inv_freq)
    c, s = np.cos(theta), np.sin(theta)
    x1, x2 = x[..., :m], x[..., m:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# ---------------------------------------------------------------------------------
# Explicit form: up-project K and V per head, then plain softmax attention.
# ---------------------------------------------------------------------------------
def attend_explicit(q, c_kv, k_rope, w_uk, w_uv, pos_q, scale=None, heads=None,
                    base: float = ROPE_BASE, return_p: bool = False, inv_freq=None):
    """Decode attention of one sequence, explicit (non-absorbed) form.

    q       [n_h, 192]  (q^C ‖ q^R before rotation)
    c_kv    [L, 512]    cached latents
    k_rope  [L, 64]     cached decoupled key, already rotated at its own position
    w_uk    [n_h, 128, 512], w_uv [n_h, 128, 512]
    pos_q   position of the query (the decode token)
    heads   optional iterable of head indices to evaluate (others are left at 0)

    Returns dict with o [n_h,128], lse [n_h], o_lat [n_h,512] (and p [n_h, L]).
    """
    q = _f64(q)
    c = _f64(c_kv)
    kr = _f64(k_rope)
    w_uk = np.asarray(w_uk)
    w_uv = np.asarray(w_uv)
    n_h = q.shape[0]
    L = c.shape[0]
    scale = default_scale() if scale is None else float(scale)
    heads = range(n_h) if heads is None else heads
    q_r = rope(q[:, D_H:], pos_q, base, inv_freq)

    o = np.zeros((n_h, D_H))
    o_lat = np.zeros((n_h, D_C))
    lse = np.full(n_h, -np.inf)
    p_all = np.zeros((n_h, L)) if return_p else None
    if L == 0:
        out = dict(o=o, lse=lse, o_lat=o_lat)
        if return_p:
            out["p"] = p_all
        return out
    for h in heads:
        wk = _f64(w_uk[h])                                  # [128, 512]
        wv = _f64(w_uv[h])                                  # [128, 512]
        K = np.concatenate([c @ wk.T, kr], axis=1)          # [L, 192]: W_UK[h]·c_t ‖ k^R_t
        V = c @ wv.T                                        # [L, 128]: W_UV[h]·c_t
        qh = np.concatenate([q[h, :D_H], q_r[h]])           # [192]
        s = (K @ qh) * scale                                # [L]
        m = s.max()
        e = np.exp(s - m)
        z = e.sum()
        p = e / z
        o[h] = p @ V
        o_lat[h] = p @ c
        lse[h] = m + math.log(z)
        if return_p:
            p_all[h] = p
    out = dict(o=o, lse=lse, o_lat=o_lat)
    if return_p:
        out["p"] = p_all
    return out


def attend_absorbed(q, c_kv, k_rope, w_uk, w_uv, pos_q, scale=None, base: float = ROPE_BASE):
    """The same quantity with W_UK folded into the query and W_UV applied after the
    latent-space weighted sum ([A] §"长上下文推理的第一瓶颈": the up-projections can be
    absorbed so K/V are never expanded). Used only to cross-check the explicit form
    on tiny inputs.
    """
    q = _f64(q)
    c = _f64(c_kv)
    kr = _f64(k_rope)
    n_h = q.shape[0]
    scale = default_scale() if scale is None else float(scale)
    q_r = rope(q[:, D_H:], pos_q, base)
    o = np.zeros((n_h, D_H))
    o_lat = np.zeros((n_h, D_C))
    lse = np.full(n_h, -np.inf)
    if c.shape[0] == 0:
        return dict(o=o, lse=lse, o_lat=o_lat)
    for h in range(n_h):
        q_lat = _f64(w_uk[h]).T @ q[h, :D_H]                # [512]
        s = (c @ q_lat + kr @ q_r[h]) * scale
        m = s.max()
        e = np.exp(s - m)
        p = e / e.sum()
        o_lat[h] = p @ c
        o[h] = _f64(w_uv[h]) @ o_lat[h]
        lse[h] = m + math.log(e.sum())
    return dict(o=o, lse=lse, o_lat=o_lat)


def attend_latent(q_lat, rows, scale=None):
    """Attention of the absorbed query over the cached rows, what the decode and merge
    calls compute from a given absorbed query ([A] §"长上下文推理的第一瓶颈": with W_UK
    folded into the query every head attends directly over the cached latent; the
    decoupled RoPE key is the rows' last 64 columns, [A] §"解耦 RoPE 与 YaRN").

    q_lat   [n_h, 576]  absorbed query: W_UK[h]^T q^C ‖ RoPE(q^R) per head
    rows    [L, 576]    cached rows c_KV ‖ k^R
    Returns dict with o_lat [n_h, 512] = sum_t p_t c_t and lse [n_h].
    """
    q_lat = _f64(q_lat)
    rows = _f64(rows)
    n_h = q_lat.shape[0]
    scale = default_scale() if scale is None else float(scale)
    if rows.shape[0] == 0:
        return dict(o_lat=np.zeros((n_h, D_C)), lse=np.full(n_h, -np.inf))
    s = (q_lat @ rows.T) * scale                          # [n_h, L]
    m = s.max(axis=1)
    e = np.exp(s - m[:, None])
    z = e.sum(axis=1)
    p = e / z[:, None]
    return dict(o_lat=p @ rows[:, :D_C], lse=m + np.log(z))


# ---------------------------------------------------------------------------------
# Several new query tokens per sequence (speculative or chunked decoding). The pages
# describe decoding as each new token attending to every earlier token ([A] §"长上下文推理
# 的第一瓶颈"); with T new tokens cached at the end of a sequence of L tokens, query j
# (0 <= j < T) sits at position L - T + j and attends causally to tokens 0 .. L - T + j.
# ---------------------------------------------------------------------------------
def attend_multi(q, c_kv, k_rope, w_uk, w_uv, T: int, scale=None, base: float = ROPE_BASE, inv_freq=None):
    """q [T, n_h, 192]; c_kv [L, 512], k_rope [L, 64] (the last T rows are the new
    tokens). Returns dict with o [T, n_h, 128], lse [T, n_h], o_lat [T, n_h, 512]; a
    query with no visible token (L - T + j < 0) gets o = o_lat = 0 and lse = -inf."""
    q = _f64(q)
    L = np.asarray(c_kv).shape[0]
    n_h = q.shape[1]
    outs = []
    for j in range(T):
        p = L - T + j
        if p < 0:
            outs.append(dict(o=np.zeros((n_h, D_H)), lse=np.full(n_h, -np.inf), o_lat=np.zeros((n_h, D_C))))
            continue
        outs.append(attend_explicit(q[j], c_kv[:p + 1], k_rope[:p + 1], w_uk, w_uv, pos_q=p, scale=scale, base=base,
                                    inv_freq=inv_freq))
    return {k: np.stack([o[k] for o in outs]) for k in ("o", "lse", "o_lat")}


# ---------------------------------------------------------------------------------
# Writing the cache ([A] §"长上下文推理的第一瓶颈": each token's hidden state is
# down-projected to the latent c_KV, d_c = 512, and only that is cached; [A] §"解耦
# RoPE 与 YaRN": a shared 64-wide key carries the position, rotated where it is made;
# hidden size 5120, [A] §"8.1T token 预训练配置与 H800 成本账" and [B] §"计算设置").
# ---------------------------------------------------------------------------------
def cache_rows(h, w_dkv, w_kr, pos, base: float = ROPE_BASE, inv_freq=None) -> np.ndarray:
    """Cache rows of new tokens, unrounded.

    h      [T, d]     hidden states of the new tokens
    w_dkv  [512, d]   down-projection to the latent:  c_t = W_DKV · h_t
    w_kr   [64, d]    projection to the shared RoPE key: k^R_t = RoPE(W_KR · h_t, pos_t)
    pos    [T]        each token's position in its sequence
    Returns [T, 576] = [c_t ‖ k^R_t].
    """
    h = _f64(h)
    c = h @ _f64(w_dkv).T                                 # [T, 512]
    k_raw = h @ _f64(w_kr).T                              # [T, 64]
    return np.concatenate([c, rope(k_raw, _f64(pos), base, inv_freq)], axis=-1)


# ---------------------------------------------------------------------------------
# Log-sum-exp merge of attention over disjoint token subsets. The exact identity:
# for a partition of the tokens into parts j with normalised outputs o_j and
# log-normalisers lse_j,  lse = ln sum_j exp(lse_j)  and  o = sum_j exp(lse_j - lse) o_j.
# Parts with lse_j = -inf (no tokens) carry zero weight.
# ---------------------------------------------------------------------------------
def merge_partials(o_parts, lse_parts):
    """o_parts [S, ..., W], lse_parts [S, ...] → (o [..., W], lse [...])."""
    o_parts = _f64(o_parts)
    lse_parts = _f64(lse_parts)
    m = np.max(lse_parts, axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - m_safe), 0.0)   # [S, ...]
    z = w.sum(axis=0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, z, 1.0)), -np.inf)
    o = np.einsum("s...,s...w->...w", w, o_parts)
    o = np.where(finite[..., None], o / np.where(finite, z, 1.0)[..., None], 0.0)
    return o, lse


# ---------------------------------------------------------------------------------
# Cache-size arithmetic ([A] §长上下文推理的第一瓶颈; [B] §瓶颈, §方法适配).
# ---------------------------------------------------------------------------------
def mha_cache_elements(n_h: int, d_h: int, layers: int) -> int:
    """Standard MHA caches K and V for every head: 2·n_h·d_h·l elements per token."""
    return 2 * n_h * d_h * layers


def mla_cache_elements(d_c: int, d_r: int, layers: int) -> int:
    """MLA caches the latent and the shared RoPE key: (d_c + d_h^R)·l per token."""
    return (d_c + d_r) * layers


def gqa_equivalent_groups(d_c: int, d_r: int, d_h: int) -> float:
    """GQA with g groups caches 2·g·d_h elements per token per layer."""
    return (d_c + d_r) / (2.0 * d_h)


def mla_cache_bytes(d_c: int, d_r: int, layers: int, tokens: int, batch: int,
                    bits_per_element: float) -> float:
    return mla_cache_elements(d_c, d_r, layers) * tokens * batch * bits_per_element / 8.0
