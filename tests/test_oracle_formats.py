"""Pins for the oracle's number formats (bf16 rounding, OCP E4M3 encode/decode).

Each check compares the oracle with something other than itself: PyTorch's own
dtype casts (library routines), exact rational arithmetic, brute-force nearest-value
search over the full E4M3 value table, and a hand-worked example.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_value(bits):
    return np.asarray(bits, np.uint32).__lshift__(16).astype(np.uint32).view(np.float32)


def _rand_f32(rng, n, lo_exp, hi_exp):
    """Random fp32 values with uniformly random exponents in [lo_exp, hi_exp)."""
    m = rng.integers(0, 1 << 23, n, dtype=np.uint32)
    e = rng.integers(lo_exp + 127, hi_exp + 127, n, dtype=np.uint32)
    s = rng.integers(0, 2, n, dtype=np.uint32) << 31
    return (s | (e << 23) | m).view(np.float32)


# ----------------------------------------------------------------------------- bf16

def test_bf16_matches_torch_cast_on_float_inputs():
    rng = np.random.default_rng(1)
    v = np.concatenate([
        _rand_f32(rng, 200_000, -126, 127),
        # exact ties: low 16 bits 0x8000, both parities of the kept LSB
        ((rng.integers(0, 1 << 16, 20_000, dtype=np.uint32) << 16) | 0x8000).view(np.float32),
        # fp32 subnormals
        rng.integers(1, 1 << 23, 10_000, dtype=np.uint32).view(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.3895314e38, -3.3895314e38], np.float32),
    ])
    v = v[np.isfinite(v)]
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_from_double(v.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_bf16_from_double_is_exact_nearest_even():
    """Brute force with exact rationals: the result is the nearest bf16, ties to even."""
    rng = np.random.default_rng(2)
    vals = list(rng.standard_normal(1500) * np.exp2(rng.integers(-140, 120, 1500)))
    # exact midpoints between neighbouring bf16 values (both parities)
    for b in rng.integers(0x0001, 0x7F00, 300):
        lo = float(_bf16_value(b)[()])
        hi = float(_bf16_value(b + 1)[()])
        vals.append((lo + hi) / 2)
    got = oracle.bf16_from_double(np.array(vals))
    for v, g in zip(vals, got):
        g = int(g)
        a = Fraction(abs(v))
        cand = [g & 0x7FFF]
        if (g & 0x7FFF) > 0:
            cand.append((g & 0x7FFF) - 1)
        cand.append((g & 0x7FFF) + 1)
        dist = {c: abs(Fraction(float(_bf16_value(c)[()])) - a) for c in cand}
        best = min(dist.values())
        assert dist[g & 0x7FFF] == best, (v, hex(g))
        ties = [c for c in cand if dist[c] == best]
        if len(ties) > 1:
            assert (g & 1) == 0, (v, hex(g))
        assert (g >> 15) == (1 if v < 0 else 0)


def test_bf16_overflow_and_subnormal_edges():
    top = float(_bf16_value(0x7F7F)[()])          # largest finite bf16
    half_ulp = 2.0 ** 127 * 2.0 ** -8
    got = oracle.bf16_from_double(np.array([top, top + half_ulp * 0.999, top + half_ulp,
                                            2.0 ** -133, 2.0 ** -134, 2.0 ** -134 * 1.0001,
                                            -2.0 ** -135]))
    assert [hex(int(g)) for g in got] == ["0x7f7f", "0x7f7f", "0x7f80", "0x1", "0x0", "0x1",
                                          "0x8000"]


# ----------------------------------------------------------------------------- e4m3

def _torch_e4m3_table():
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    return t.numpy()


def test_e4m3_decode_matches_torch_table():
    ref = _torch_e4m3_table()
    got = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.isnan(got).sum() == 2                      # 0x7F and 0xFF only
    np.testing.assert_array_equal(got[~np.isnan(got)], ref[~np.isnan(ref)])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def _nearest_e4m3_bruteforce(v):
    """Nearest finite E4M3 code by exhaustive search; ties to the even code; |v| > 448
    saturates to 448. Works on float64 copies of fp32 inputs (differences are exact)."""
    table = _torch_e4m3_table()[:0x7F]                   # codes 0..0x7E, ascending
    a = np.abs(v.astype(np.float64))
    idx = np.clip(np.searchsorted(table, a), 1, 0x7E)
    lo, hi = idx - 1, idx
    dlo, dhi = a - table[lo], table[hi] - a
    code = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = np.where(a >= 448.0, 0x7E, code)
    return (code | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def test_e4m3_encode_exhaustive_binades():
    # every fp32 pattern in a subnormal binade, a small normal binade, [1, 2) and
    # [256, 512) (which crosses the saturation point), both signs
    for exp in (-10, -7, 0, 8):
        m = np.arange(1 << 23, dtype=np.uint32)
        pos = ((np.uint32(exp + 127) << 23) | m).view(np.float32)
        for v in (pos, -pos):
            np.testing.assert_array_equal(oracle.e4m3_encode(v), _nearest_e4m3_bruteforce(v))


def test_e4m3_encode_random_and_specials():
    rng = np.random.default_rng(3)
    v = np.concatenate([_rand_f32(rng, 2_000_000, -14, 12),
                        np.array([0.0, -0.0, 448.0, -448.0, 464.0, 1e30, -1e30], np.float32)])
    np.testing.assert_array_equal(oracle.e4m3_encode(v), _nearest_e4m3_bruteforce(v))
    inf = oracle.e4m3_encode(np.array([np.inf, -np.inf, np.nan], np.float32))
    assert list(inf) == [0x7E, 0xFE, 0x7F]


def test_e4m3_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(4)
    v = _rand_f32(rng, 1_000_000, -12, 9)
    v = v[np.abs(v) <= 448.0]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(v), ref)


# ----------------------------------------------------------------------------- quantisation

def _torch_quantize(xbits):
    """Independent per-128-group quantisation through PyTorch ops (IEEE fp32 divide and
    multiply, library e4m3 cast after clamping to the finite range)."""
    x = torch.from_numpy(xbits.view(np.int16)).view(torch.bfloat16).float()
    g = x.reshape(*x.shape[:-1], -1, 128)
    amax = g.abs().amax(dim=-1, keepdim=True)
    am = torch.clamp(amax, min=torch.tensor(1e-4, dtype=torch.float32))
    scale = am / 448.0
    inv = torch.tensor(448.0, dtype=torch.float32) / am
    q = torch.clamp(g * inv, -448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return q.reshape(x.shape).numpy(), scale.squeeze(-1).numpy()


def test_quantize_rows_matches_torch_path():
    rng = np.random.default_rng(5)
    x32 = rng.standard_normal((64, 1024)).astype(np.float32)
    x32[3, :128] = 0.0                                  # all-zero group -> amax floor
    x32[4, 128:256] = 1e-7                               # group below the floor
    x32[5] *= 1e3
    xb = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    q, sc = oracle.quantize_rows(xb)
    q_ref, sc_ref = _torch_quantize(xb)
    np.testing.assert_array_equal(q, q_ref)
    np.testing.assert_array_equal(sc.view(np.uint32), sc_ref.view(np.uint32))


def test_quantize_roundtrip_error_bound():
    rng = np.random.default_rng(6)
    x32 = (rng.standard_normal((32, 7168)) * np.exp2(rng.integers(-8, 8, (32, 1)))).astype(np.float32)
    xb = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xf = _bf16_value(xb).astype(np.float64)
    q, sc = oracle.quantize_rows(xb)
    dq = oracle.e4m3_decode(q).reshape(32, 56, 128) * sc[..., None].astype(np.float64)
    xg = xf.reshape(32, 56, 128)
    # half an E4M3 ulp of |x * inv| (in units of the scale), plus slack for the two
    # fp32 roundings of inv and the product
    inv = 448.0 / np.maximum(np.abs(xg).max(-1, keepdims=True), 1e-4)
    a = np.abs(xg) * inv
    ulp = np.exp2(np.maximum(np.floor(np.log2(np.maximum(a, 2.0 ** -9))), -6) - 3)
    bound = (0.5 * ulp * (1 + 2 ** -20) + a * 2 ** -22) * sc[..., None]
    assert np.all(np.abs(dq - xg) <= bound)
    # the amax element of every group maps to +-448 exactly
    amax_pos = np.abs(xg).argmax(-1)
    codes = np.take_along_axis(q.reshape(32, 56, 128), amax_pos[..., None], -1)[..., 0]
    assert np.all((codes & 0x7F) == 0x7E)


def test_quantize_hand_example():
    with open(os.path.join(GOLDEN, "fp8_hand_example.json")) as f:
        g = json.load(f)
    H = g["H"]
    x = np.zeros((1, H), np.uint16)
    for i, b in g["group0_values_bf16_bits"].items():
        x[0, int(i)] = int(b, 16)
    q, sc = oracle.quantize_rows(x)
    expect = np.zeros(H, np.uint8)
    for i, c in g["group0_codes"].items():
        expect[int(i)] = int(c, 16)
    np.testing.assert_array_equal(q[0], expect)
    assert sc[0, 0] == np.float32(g["group0_amax"]) / np.float32(448.0)
    assert sc[0, 1] == np.float32(g["group1_amax_floor"]) / np.float32(448.0)


# ----------------------------------------------------------------------------- scale modes

def _torch_quantize_modes(xbits, mode, tensor_scale=0.0):
    """Power-of-two / per-tensor quantisation through PyTorch ops: fp32 division, exact
    power-of-two rounding via frexp, library e4m3 cast after clamping."""
    x = torch.from_numpy(xbits.view(np.int16)).view(torch.bfloat16).float()
    g = x.reshape(*x.shape[:-1], -1, 128)
    if mode == oracle.SCALE_TENSOR:
        s = torch.tensor(tensor_scale, dtype=torch.float32)
        inv = torch.tensor(1.0, dtype=torch.float32) / s
        scale = s.expand(g.shape[:-1])
    else:
        am = torch.clamp(g.abs().amax(dim=-1, keepdim=True), min=torch.tensor(1e-4))
        s0 = am / 448.0
        m, e = torch.frexp(s0)
        scale = torch.ldexp(torch.ones_like(s0), torch.where(m == 0.5, e - 1, e))
        inv = 1.0 / scale
        scale = scale.squeeze(-1)
    q = torch.clamp(g * inv, -448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return q.reshape(x.shape).numpy(), scale.numpy()


@pytest.mark.parametrize("mode", [1, 2, 3])
def test_scale_modes_match_torch_path(mode):
    rng = np.random.default_rng(8)
    x32 = (rng.standard_normal((48, 1024)) * np.exp2(rng.integers(-10, 10, (48, 1)))).astype(np.float32)
    x32[0, :128] = 0.0
    xb = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ts = 0.0173 if mode == 3 else 0.0
    q, sc = oracle.quantize_rows(xb, mode, ts)
    q_ref, sc_ref = _torch_quantize_modes(xb, mode, ts)
    np.testing.assert_array_equal(q, q_ref)
    if mode == 2:
        # one byte per group: the biased exponent of the power-of-two scale
        np.testing.assert_array_equal(sc.astype(np.float64), np.log2(sc_ref.astype(np.float64)) + 127)
        q1, _ = oracle.quantize_rows(xb, 1)
        np.testing.assert_array_equal(q, q1)           # same codes as the fp32 power-of-two mode
    else:
        np.testing.assert_array_equal(sc.view(np.uint32), sc_ref.astype(np.float32).view(np.uint32))
    if mode in (1, 2):
        s_f = np.exp2(sc.astype(np.float64) - 127) if mode == 2 else sc.astype(np.float64)
        m, _ = np.frexp(s_f)
        assert np.all(m == 0.5)                           # exact powers of two
        amax = np.abs(_bf16_value(xb).reshape(48, 8, 128)).max(-1)
        s0 = np.maximum(amax, np.float32(1e-4)).astype(np.float32) / np.float32(448)
        assert np.all(s_f >= s0) and np.all(s_f / 2 < s0)  # the next power of two up


def test_scale_modes_hand_example():
    with open(os.path.join(GOLDEN, "fp8_scale_modes_hand_example.json")) as f:
        g = json.load(f)
    H = g["H"]
    x = np.zeros((1, H), np.uint16)
    for i, b in g["group0_values_bf16_bits"].items():
        x[0, int(i)] = int(b, 16)
    for mode in (1, 2):
        q, sc = oracle.quantize_rows(x, mode)
        exp = np.zeros(H, np.uint8)
        for i, c in g["pow2_codes"].items():
            exp[int(i)] = int(c, 16)
        np.testing.assert_array_equal(q[0], exp)
        if mode == 1:
            assert sc[0, 0] == g["pow2_scale_group0"]
        else:
            assert sc[0, 0] == g["ue8m0_byte_group0"] and sc[0, 1] == g["ue8m0_byte_group1_zeros"]
    for i, b in g["tensor_extra_value"].items():
        x[0, int(i)] = int(b, 16)
    q, sc = oracle.quantize_rows(x, 3, g["tensor_scale"])
    exp = np.zeros(H, np.uint8)
    for i, c in g["tensor_codes"].items():
        exp[int(i)] = int(c, 16)
    np.testing.assert_array_equal(q[0], exp)
    assert np.all(sc == np.float32(g["tensor_scale"]))
