"""The oracle's pins catch planted mistakes.

Each case rewrites one line of one oracle function (a flipped sign, a swapped operand,
a wrong constant or index), installs the rewritten function in place of the original
for the duration of the case, runs the pin tests of test_oracle.py / test_fp8_codec.py /
test_fp6_codec.py against it, and requires that at least one pin fails. The mistakes are planted only in
this process, on the CPU; the oracle's files are not touched.
"""

import inspect
import textwrap

import numpy as np
import pytest

import test_fp6_codec as P6
import test_fp8_codec as PF
import test_oracle as PO
from oracle import fp6_e2m3 as F6
from oracle import fp8_e4m3 as F
from oracle import mla_oracle as M


def _mutant(func, old: str, new: str):
    """`func` recompiled from its source with the single occurrence of `old` replaced."""
    src = textwrap.dedent(inspect.getsource(func))
    assert src.count(old) == 1, f"{func.__name__}: the planted line must occur exactly once: {old!r}"
    ns = dict(func.__globals__)
    exec(compile(src.replace(old, new), f"<mutant of {func.__name__}>", "exec"), ns)
    return ns[func.__name__]


def _failing_pins(pin_module, extra=()):
    """Names of the pin tests (argument-free ones, plus `extra` zero-argument callables)
    that fail under the current oracle."""
    failed = []
    pins = [(n, f) for n, f in inspect.getmembers(pin_module, inspect.isfunction)
            if n.startswith("test_") and not inspect.signature(f).parameters]
    for name, fn in list(pins) + list(extra):
        try:
            with np.errstate(all="ignore"):
                fn()
        except Exception:   # an assertion or a numerical failure: the mistake is visible
            failed.append(name)
    return failed


ORACLE_MUTANTS = [
    # RoPE: signs, pairing, frequencies, cos/sin roles
    ("rope", "x1 * c - x2 * s", "x1 * c + x2 * s"),
    ("rope", "x2 * c + x1 * s", "x2 * c - x1 * s"),
    ("rope", "inv_freq = base ** (-2.0 * i / width)", "inv_freq = base ** (-1.0 * i / width)"),
    ("rope", "x1, x2 = x[..., :m], x[..., m:]", "x1, x2 = x[..., 0::2], x[..., 1::2]"),
    ("rope", "c, s = np.cos(theta), np.sin(theta)", "c, s = np.sin(theta), np.cos(theta)"),
    # scale
    ("default_scale", "math.sqrt(D_H + D_R)", "math.sqrt(D_H)"),
    # explicit form: which weight makes K and V, the RoPE key, the query position,
    # the scale, the normalisation, the latent output, the log base of lse
    ("attend_explicit", "wk = _f64(w_uk[h])", "wk = _f64(w_uv[h])"),
    ("attend_explicit", "V = c @ wv.T", "V = c @ wk.T"),
    ("attend_explicit", "K = np.concatenate([c @ wk.T, kr], axis=1)", "K = np.concatenate([c @ wk.T, 0.0 * kr], axis=1)"),
    ("attend_explicit", "q_r = rope(q[:, D_H:], pos_q, base, inv_freq)", "q_r = rope(q[:, D_H:], pos_q + 1, base, inv_freq)"),
    ("attend_explicit", "s = (K @ qh) * scale", "s = K @ qh"),
    ("attend_explicit", "p = e / z", "p = e / e.max()"),
    ("attend_explicit", "o_lat[h] = p @ c", "o_lat[h] = e @ c"),
    ("attend_explicit", "lse[h] = m + math.log(z)", "lse[h] = m + math.log2(z)"),
    ("attend_explicit", "qh = np.concatenate([q[h, :D_H], q_r[h]])", "qh = np.concatenate([q[h, :D_H], q[h, D_H:]])"),
    # latent form: the scale, the RoPE key columns, the value columns, the log base
    ("attend_latent", "s = (q_lat @ rows.T) * scale", "s = q_lat @ rows.T"),
    ("attend_latent", "s = (q_lat @ rows.T) * scale", "s = (q_lat[:, :D_C] @ rows[:, :D_C].T) * scale"),
    ("attend_latent", "return dict(o_lat=p @ rows[:, :D_C], lse=m + np.log(z))",
     "return dict(o_lat=p @ rows[:, D_R:], lse=m + np.log(z))"),
    ("attend_latent", "return dict(o_lat=p @ rows[:, :D_C], lse=m + np.log(z))",
     "return dict(o_lat=p @ rows[:, :D_C], lse=m + np.log2(z))"),
    # split merge
    ("merge_partials", "np.exp(lse_parts - m_safe)", "np.exp(m_safe - lse_parts)"),
    ("merge_partials", "o = np.where(finite[..., None], o / np.where(finite, z, 1.0)[..., None], 0.0)",
     "o = np.where(finite[..., None], o, 0.0)"),
    # cache-size arithmetic
    ("mla_cache_elements", "return (d_c + d_r) * layers", "return d_c * layers"),
    ("mha_cache_elements", "return 2 * n_h * d_h * layers", "return n_h * d_h * layers"),
    # writing the cache: which weight, the key's rotation and its position
    ("cache_rows", "c = h @ _f64(w_dkv).T", "c = h @ _f64(w_dkv).T * 1.0001"),
    ("cache_rows", "rope(k_raw, _f64(pos), base, inv_freq)", "rope(k_raw, -_f64(pos), base, inv_freq)"),
    ("cache_rows", "rope(k_raw, _f64(pos), base, inv_freq)", "rope(k_raw, _f64(pos) + 1, base, inv_freq)"),
    ("cache_rows", "rope(k_raw, _f64(pos), base, inv_freq)", "k_raw"),
    # YaRN: the ramp's direction, its end points, the slowed frequency
    ("yarn_inv_freq", "return (1.0 - gamma) * theta / scale + gamma * theta", "return gamma * theta / scale + (1.0 - gamma) * theta"),
    ("yarn_inv_freq", "gamma = np.clip((r - alpha) / (beta - alpha), 0.0, 1.0)", "gamma = np.clip((r - alpha) / beta, 0.0, 1.0)"),
    ("yarn_inv_freq", "r = original_max_pos * theta / (2.0 * math.pi)", "r = original_max_pos * theta"),
    ("yarn_inv_freq", "return (1.0 - gamma) * theta / scale + gamma * theta", "return (1.0 - gamma) * theta * scale + gamma * theta"),
    ("cache_rows", "k_raw = h @ _f64(w_kr).T", "k_raw = h @ _f64(w_dkv[:64]).T"),
    # several new tokens: the query position, what it sees
    ("attend_multi", "p = L - T + j", "p = L - T + j - 1"),
    ("attend_multi", "outs.append(attend_explicit(q[j], c_kv[:p + 1], k_rope[:p + 1], w_uk, w_uv, pos_q=p,",
     "outs.append(attend_explicit(q[j], c_kv, k_rope, w_uk, w_uv, pos_q=p,"),
    ("attend_multi", "if p < 0:", "if p <= 0:"),
]


@pytest.mark.parametrize("fname,old,new", ORACLE_MUTANTS, ids=[f"{m[0]}:{m[2][:28]}" for m in ORACLE_MUTANTS])
def test_oracle_pins_catch_planted_mistake(monkeypatch, fname, old, new):
    assert not _failing_pins(PO), "every pin passes on the unmodified oracle"
    monkeypatch.setattr(M, fname, _mutant(getattr(M, fname), old, new))
    assert _failing_pins(PO), f"no pin notices {fname}: {old!r} -> {new!r}"


def _fp8_param_pins():
    """The parametrised code-value pin, run over its own parameter list."""
    codes = next(m.args[1] for m in PF.test_code_value_definition.pytestmark if m.name == "parametrize")

    def listed_codes():
        for code in codes:
            PF.test_code_value_definition(code)
    return [("test_code_value_definition[listed]", listed_codes)]


FP8_MUTANTS = [
    ("code_value", "v = (1.0 + m / 8.0) * 2.0 ** (e - 7)", "v = (1.0 + m / 8.0) * 2.0 ** (e - 8)"),
    ("code_value", "v = m * 2.0 ** -9", "v = m * 2.0 ** -10"),
    ("code_value", "m = code & 0x7", "m = (code >> 1) & 0x7"),
    ("encode", "take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))", "take_hi = d_hi <= d_lo"),
    ("encode", "(np.signbit(x).astype(np.int64) << 7)", "(np.signbit(x).astype(np.int64) << 6)"),
    ("encode", "return np.where(np.isnan(x), np.uint8(NAN_CODE), code).astype(np.uint8)", "return code"),
    ("quantize_rows", "amax / np.float32(E4M3_MAX)", "amax / np.float32(240.0)"),
]


@pytest.mark.parametrize("fname,old,new", FP8_MUTANTS, ids=[f"{m[0]}:{m[2][:28]}" for m in FP8_MUTANTS])
def test_fp8_pins_catch_planted_mistake(monkeypatch, fname, old, new):
    assert not _failing_pins(PF, _fp8_param_pins())
    mutant = _mutant(getattr(F, fname), old, new)
    monkeypatch.setattr(F, fname, mutant)
    if fname == "code_value":   # the decode table is built from code_value at import
        monkeypatch.setattr(F, "DECODE_TABLE", np.array([mutant(c) for c in range(256)], dtype=np.float64))
        monkeypatch.setattr(F, "_POS", F.DECODE_TABLE[:0x7F].copy())
    assert _failing_pins(PF, _fp8_param_pins()), f"no pin notices {fname}: {old!r} -> {new!r}"



def _fp6_param_pins():
    """The parametrised code-value pin, run over its own parameter list."""
    cases = next(m.args[1] for m in P6.test_code_value_definition.pytestmark if m.name == "parametrize")

    def listed_codes():
        for code, value in cases:
            P6.test_code_value_definition(code, value)
    return [("test_code_value_definition[listed]", listed_codes)]


FP6_MUTANTS = [
    ("code_value", "v = (1.0 + m / 8.0) * 2.0 ** (e - 1)", "v = (1.0 + m / 8.0) * 2.0 ** (e - 2)"),
    ("code_value", "v = m * 2.0 ** -3", "v = m * 2.0 ** -4"),
    ("code_value", "m = code & 0x7", "m = (code >> 1) & 0x7"),
    ("encode", "take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))", "take_hi = d_hi <= d_lo"),
    ("encode", "(np.signbit(x).astype(np.int64) << 5)", "(np.signbit(x).astype(np.int64) << 4)"),
    ("block_exponents", "e.astype(np.int64) - 1 - E2M3_EMAX", "e.astype(np.int64) - E2M3_EMAX"),
    ("quantize_blocks", "(-se)[..., None]", "(1 - se)[..., None]"),
    ("pack", "(c[..., 2] << 12)", "(c[..., 2] << 11)"),
    ("unpack", "(w >> (6 * k)) & 0x3F", "(w >> (6 * k)) & 0x1F"),
]


@pytest.mark.parametrize("fname,old,new", FP6_MUTANTS, ids=[f"{m[0]}:{m[2][:28]}" for m in FP6_MUTANTS])
def test_fp6_pins_catch_planted_mistake(monkeypatch, fname, old, new):
    assert not _failing_pins(P6, _fp6_param_pins())
    mutant = _mutant(getattr(F6, fname), old, new)
    monkeypatch.setattr(F6, fname, mutant)
    if fname == "code_value":   # the decode table is built from code_value at import
        monkeypatch.setattr(F6, "DECODE_TABLE", np.array([mutant(c) for c in range(64)], dtype=np.float64))
        monkeypatch.setattr(F6, "_POS", F6.DECODE_TABLE[:0x20].copy())
    assert _failing_pins(P6, _fp6_param_pins()), f"no pin notices {fname}: {old!r} -> {new!r}"
