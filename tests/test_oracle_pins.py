"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each check is chosen so that a plausible slip in the oracle (a wrong rounding
rule, an off-by-one exponent, a swapped sign or cos/sin column, a transposed
head / group index) fails at least one of them:

* E4M3 decode / encode: the OFP8 spec's code points (tests/golden), torch's
  float8_e4m3fn cast (a library routine) over every fp32 pattern in
  [2^-12, 448), brute-force nearest search over the 127 finite magnitudes.
* ceil(log2): exact rational arithmetic (fractions.Fraction) and the defining
  inequality 2^(e-1) < r <= 2^e over a dense sweep of fp32 patterns.
* Rotation: complex multiplication by exp(-i*theta) / exp(+i*theta) in
  complex128 (a library routine), textbook RoPE angles evaluated from the
  positions, cos=0/sin=1 swap, position-0 identity, forward/inverse round trip.
* Whole op: hand-built worked cases whose codes and scales follow from the
  spec by hand, layout fingerprints per (token, group, head), the block-amax
  invariant 224 <= amax/scale <= 448, the dequantisation error bound.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- E4M3 table

def _spec_points():
    pts = []
    with open(os.path.join(GOLDEN, "ofp8_e4m3_points.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            code, val = line.split()
            pts.append((int(code, 16), val))
    return pts


def test_e4m3_decode_matches_spec_points(oracle_lib):
    for code, val in _spec_points():
        got = oracle_lib.e4m3_decode(np.array([code], np.uint8))[0]
        if val == "nan":
            assert np.isnan(got), hex(code)
        elif val == "-0":
            assert got == 0.0 and np.signbit(got), hex(code)
        else:
            assert Fraction(got) == Fraction(val), (hex(code), got, val)


def test_e4m3_decode_matches_torch_for_all_codes(oracle_lib):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle_lib.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_e4m3_roundtrip_every_code(oracle_lib):
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle_lib.e4m3_decode(codes)
    for c, v in zip(codes, vals):
        if np.isnan(v):
            continue
        assert oracle_lib.e4m3_encode_scalar(v) == c, (hex(c), v)


def test_e4m3_encode_matches_torch_dense_sweep(oracle_lib):
    """Every fp32 pattern with magnitude in [2^-12, 448): 174M values, both signs
    on a stride. torch's float8_e4m3fn cast rounds to nearest even there."""
    lo = np.float32(2.0 ** -12).view(np.uint32)
    hi = np.float32(448.0).view(np.uint32)
    step = 1 << 24
    for start in range(int(lo), int(hi), step):
        bits = np.arange(start, min(start + step, int(hi)), dtype=np.uint32)
        v = bits.view(np.float32)
        ours = oracle_lib.e4m3_encode(v)
        ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        bad = np.nonzero(ours != ref)[0]
        assert bad.size == 0, (v[bad[:5]], ours[bad[:5]], ref[bad[:5]])
        neg = -v[::97]
        ours_n = oracle_lib.e4m3_encode(neg)
        ref_n = torch.from_numpy(neg).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(ours_n, ref_n)


def _nearest_even_bruteforce(a: Fraction, mags):
    """Nearest finite E4M3 magnitude to a >= 0 by direct search; ties -> even code."""
    best = None
    for code, m in mags:
        d = abs(a - m)
        if best is None or d < best[0] or (d == best[0] and code % 2 == 0):
            best = (d, code, m)
    return best[1]


def test_e4m3_encode_bruteforce_nearest(oracle_lib):
    codes = np.arange(0x7F, dtype=np.uint8)  # 0x00..0x7E: the 127 finite magnitudes
    mags = [(int(c), Fraction(float(v))) for c, v in zip(codes, oracle_lib.e4m3_decode(codes))]
    rng = np.random.default_rng(1)
    samples = [Fraction(0)]
    # every midpoint between neighbours (the ties), and one fp32 ulp either side
    for (c0, m0), (c1, m1) in zip(mags[:-1], mags[1:]):
        mid = (m0 + m1) / 2
        f = np.float32(float(mid))
        samples += [mid, Fraction(float(np.nextafter(f, np.float32(0)))),
                    Fraction(float(np.nextafter(f, np.float32(1e9))))]
    samples += [Fraction(float(v)) for v in rng.uniform(0, 448, 3000).astype(np.float32)]
    samples += [Fraction(float(v)) for v in
                np.exp2(rng.uniform(-14, 8.8, 3000)).astype(np.float32)]
    for a in samples:
        f = float(a)
        assert Fraction(f) == a  # every sample is an exact double
        want = _nearest_even_bruteforce(a, mags)
        got = oracle_lib.e4m3_encode_scalar(f)
        assert got == want, (f, hex(got), hex(want))
        assert oracle_lib.e4m3_encode_scalar(-f) == (want | 0x80), f


@pytest.mark.parametrize("value,code", [
    (310.0, 0x7A),          # 310 lies between 288 and 320, nearer 320 (S.1111.010)
    (2.0 ** -10, 0x00),     # tie between 0 and 2^-9 -> even (zero)
    (3 * 2.0 ** -10, 0x02), # tie between 2^-9 (odd) and 2*2^-9 (even)
    (460.0, 0x7E),          # above max normal: saturates
    (1e30, 0x7E),
    (float("inf"), 0x7E),
    (float("-inf"), 0xFE),
    (-1e-9, 0x80),          # negative underflow keeps the sign
    (-0.0, 0x80),
    (float("nan"), 0x7F),
    (17.0, 0x58),           # tie 16 | 18 -> 16 (even mantissa), S.1011.000
    (19.0, 0x5A),           # tie 18 | 20 -> 20 (even mantissa), S.1011.010
])
def test_e4m3_encode_worked_cases(oracle_lib, value, code):
    assert oracle_lib.e4m3_encode_scalar(value) == code


def test_e4m3_encode_saturation_and_tiny(oracle_lib):
    v = np.array([448.0, 449.0, 463.99, 464.0, 500.0, 3.4e38, 2.0 ** -11, 2.0 ** -30,
                  1e-45], np.float32)
    got = oracle_lib.e4m3_encode(v)
    assert list(got) == [0x7E] * 6 + [0x00] * 3
    assert list(oracle_lib.e4m3_encode(-v)) == [0xFE] * 6 + [0x80] * 3


# ----------------------------------------------------------------- ceil(log2)

def _ceil_log2_exact(r: float) -> int:
    """Smallest integer e with r <= 2^e, by exact rational comparison."""
    q = Fraction(r)
    e = q.numerator.bit_length() - q.denominator.bit_length() - 1
    while Fraction(2) ** e < q:
        e += 1
    while Fraction(2) ** (e - 1) >= q:
        e -= 1
    return e


def test_ceil_log2_exact_rational(oracle_lib):
    vals = []
    for k in range(-149, 128):
        p = np.float32(2.0 ** k)
        vals += [p, np.nextafter(p, np.float32(0)), np.nextafter(p, np.float32(np.inf))]
    rng = np.random.default_rng(2)
    vals += list(rng.integers(1, 0x7F800000, 20000, dtype=np.uint32).view(np.float32))
    vals = np.array([v for v in vals if np.isfinite(v) and v > 0], np.float32)
    got = oracle_lib.ceil_log2(vals)
    for v, e in zip(vals, got):
        assert e == _ceil_log2_exact(float(v)), (float(v), e)


def test_ceil_log2_defining_inequality_sweep(oracle_lib):
    """2^(e-1) < r <= 2^e for every 61st positive finite fp32 (all binades)."""
    bits = np.arange(1, 0x7F800000, 61, dtype=np.uint32)
    r = bits.view(np.float32)
    e = oracle_lib.ceil_log2(r).astype(np.int64)
    r64 = r.astype(np.float64)
    assert np.all(np.ldexp(1.0, e) >= r64)
    assert np.all(np.ldexp(1.0, e - 1) < r64)


def test_block_scale_closed_forms(oracle_lib):
    for k in range(-60, 100):
        amax = np.float32(448.0 * 2.0 ** k)
        assert oracle_lib.block_scale(np.array([amax]))[0] == np.float32(2.0 ** k)
        up = np.nextafter(amax, np.float32(np.inf))
        assert oracle_lib.block_scale(np.array([up]))[0] == np.float32(2.0 ** (k + 1))
        dn = np.nextafter(amax, np.float32(0))
        assert oracle_lib.block_scale(np.array([dn]))[0] == np.float32(2.0 ** k)


def test_block_scale_is_ceil_pow2_of_rounded_quotient(oracle_lib):
    rng = np.random.default_rng(3)
    amax = np.exp2(rng.uniform(-33, 60, 20000)).astype(np.float32)
    s = oracle_lib.block_scale(amax)
    for a, sc in zip(amax[:4000], s[:4000]):
        raw = np.float32(a) / np.float32(448.0)       # fp32 division, RN-even
        assert Fraction(float(sc)) == Fraction(2) ** _ceil_log2_exact(float(raw))
    # every scale is a power of two: zero mantissa bits
    assert np.all((s.view(np.uint32) & 0x7FFFFF) == 0)


@pytest.mark.parametrize("eps", [1e-10, 1e-4])
def test_zero_block_scale_follows_eps(oracle_lib, eps):
    raw = np.float32(eps) / np.float32(448.0)
    want = Fraction(2) ** _ceil_log2_exact(float(raw))
    codes, scales = oracle_lib.quant_rows(np.zeros((1, 512), np.float32), eps=eps)
    assert np.all(codes == 0)
    assert all(Fraction(float(s)) == want for s in scales[0])
    assert {1e-10: -42, 1e-4: -22}[eps] == _ceil_log2_exact(float(raw))


# ----------------------------------------------------------------- rotation

def _complex_rotate(rows, positions, cache, inverse):
    """(even + i odd) * conj(cos + i sin) for inverse, * (cos + i sin) forward."""
    rows = np.asarray(rows, np.float64)
    cs = np.asarray(cache, np.float64)[np.asarray(positions)]
    z = rows[:, 448::2] + 1j * rows[:, 449::2]
    w = cs[:, :32] + 1j * cs[:, 32:]
    z = z * (np.conj(w) if inverse else w)
    out = rows.copy()
    out[:, 448::2] = z.real
    out[:, 449::2] = z.imag
    return out


@pytest.mark.parametrize("inverse", [True, False])
def test_rotation_matches_complex_multiply(oracle_lib, inverse):
    rng = np.random.default_rng(4)
    R = 400
    rows = (rng.standard_normal((R, 512)) * np.exp2(rng.integers(-6, 7, (R, 1)))).astype(np.float32)
    cache = W.rope_cache(65536).numpy()
    pos = rng.integers(0, 65536, R)
    got = oracle_lib.rope_rows(rows, pos, cache, inverse=inverse).astype(np.float64)
    ref = _complex_rotate(rows, pos, cache, inverse)
    assert np.array_equal(got[:, :448], rows[:, :448].astype(np.float64))
    e = rows[:, 448::2].astype(np.float64)
    o = rows[:, 449::2].astype(np.float64)
    bound = 2.0 ** -22 * (np.abs(e) + np.abs(o))
    assert np.all(np.abs(got[:, 448::2] - ref[:, 448::2]) <= bound)
    assert np.all(np.abs(got[:, 449::2] - ref[:, 449::2]) <= bound)


def test_rotation_matches_textbook_angles(oracle_lib):
    """Forward RoPE rotates pair j by +p*10000^(-j/32), inverse by the negative angle,
    with the angle computed here from the position (not from the cache)."""
    rng = np.random.default_rng(5)
    R = 64
    rows = rng.standard_normal((R, 512)).astype(np.float32)
    pos = rng.integers(0, 4096, R)
    cache = W.rope_cache(4096).numpy()
    theta = 10000.0 ** (-np.arange(32) / 32.0)
    ang = pos[:, None] * theta[None, :]
    z = rows[:, 448::2].astype(np.float64) + 1j * rows[:, 449::2].astype(np.float64)
    for inverse, sign in ((False, 1.0), (True, -1.0)):
        got = oracle_lib.rope_rows(rows, pos, cache, inverse=inverse)
        zr = z * np.exp(1j * sign * ang)
        assert np.allclose(got[:, 448::2], zr.real, atol=2e-6, rtol=0)
        assert np.allclose(got[:, 449::2], zr.imag, atol=2e-6, rtol=0)


def test_rotation_swap_and_identity(oracle_lib):
    rng = np.random.default_rng(6)
    rows = rng.standard_normal((8, 512)).astype(np.float32)
    rows[0, 448:452] = [-0.0, 0.0, 1.5, -2.25]
    swap = np.zeros((1, 64), np.float32)
    swap[0, 32:] = 1.0                         # cos 0, sin 1: rotation by +-90 degrees
    z = np.zeros(8, np.int64)
    inv = oracle_lib.rope_rows(rows, z, swap, inverse=True)
    fwd = oracle_lib.rope_rows(rows, z, swap, inverse=False)
    assert np.array_equal(inv[:, 448::2], rows[:, 449::2])     # e' = o
    assert np.array_equal(inv[:, 449::2], -rows[:, 448::2])    # o' = -e
    assert np.array_equal(fwd[:, 448::2], -rows[:, 449::2])
    assert np.array_equal(fwd[:, 449::2], rows[:, 448::2])
    ident = W.rope_cache(1).numpy()            # position 0: cos 1, sin 0
    for inverse in (True, False):
        out = oracle_lib.rope_rows(rows, z, ident, inverse=inverse)
        assert np.array_equal(out, rows)       # equal as values (+0 == -0)


def test_rotation_round_trip(oracle_lib):
    rng = np.random.default_rng(7)
    rows = rng.standard_normal((256, 512)).astype(np.float32)
    cache = W.rope_cache(65536).numpy()
    pos = rng.integers(0, 65536, 256)
    back = oracle_lib.rope_rows(oracle_lib.rope_rows(rows, pos, cache, False), pos, cache, True)
    norm = np.hypot(rows[:, 448::2], rows[:, 449::2]).repeat(2, axis=1)
    assert np.all(np.abs(back[:, 448:] - rows[:, 448:]) <= 2.0 ** -21 * norm + 1e-30)
    assert np.array_equal(back[:, :448], rows[:, :448])


# ----------------------------------------------------------------- whole op

def _bf16(a):
    return torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16)


def test_worked_case_single_448(oracle_lib):
    x = np.zeros((1, 1, 512), np.float32)
    x[0, 0, 5] = 448.0
    x[0, 0, 130] = -3.0
    codes, scales = oracle_lib.inv_rope_fp8_quant(_bf16(x), torch.zeros(1, dtype=torch.int64),
                                                  W.rope_cache(1), 1)
    assert scales[0, 0, 0] == 1.0                      # 448/448 = 1 = 2^0
    assert codes[0, 0, 5] == 0x7E
    assert scales[0, 0, 1] == 2.0 ** -7                # ceil(log2(3/448)) = -7
    assert codes[0, 0, 130] == 0xFC                    # -3 * 2^7 = -384 = -1.5*2^8
    expect_zero = Fraction(2) ** _ceil_log2_exact(float(np.float32(1e-10) / np.float32(448)))
    assert Fraction(float(scales[0, 0, 2])) == expect_zero
    assert Fraction(float(scales[0, 0, 3])) == expect_zero
    mask = np.ones(512, bool)
    mask[[5, 130]] = False
    assert np.all(codes[0, 0, mask] == 0)


def test_worked_case_exact_grid_block(oracle_lib):
    """A block whose values are E4M3 values times 2^s (max 448*2^s) quantises to
    exactly those codes with scale 2^s, for every s the bf16 range allows."""
    rng = np.random.default_rng(8)
    grid_codes = rng.integers(0, 0x7F, 512).astype(np.uint8)
    grid_codes[[0, 128, 256, 384]] = 0x7E              # each block holds the max
    signs = rng.integers(0, 2, 512).astype(np.uint8) << 7
    grid = oracle_lib.e4m3_decode(grid_codes | signs)
    for s in (-20, -3, 0, 5, 40):
        x = (grid * 2.0 ** s).astype(np.float32).reshape(1, 1, 512)
        assert np.array_equal(_bf16(x).float().numpy(), x)   # bf16-exact
        codes, scales = oracle_lib.inv_rope_fp8_quant(_bf16(x), torch.zeros(1, dtype=torch.int64),
                                                      W.rope_cache(1), 1)
        assert np.all(scales == np.float32(2.0 ** s))
        want = grid_codes | signs
        zero = grid_codes == 0     # a rotated -0 may come back as +0: compare magnitudes
        assert np.array_equal(codes[0, 0][~zero], want[~zero])
        assert np.all(codes[0, 0][zero] & 0x7F == 0)
        assert np.array_equal(codes[0, 0, :448][zero[:448]], signs[:448][zero[:448]])


# A rotated value that lands exactly on a round-to-nearest-even tie of the
# e4m3 grid when each product and the sum are rounded on their own (the op
# order of the inverse-RoPE page, S2): pair 23 of a row at position 5386 of
# the 8192-row theta=10000 cache, block 3's scale fixed at 2^-2 by a 100.
# A fused multiply-add would land just below the tie and give code 3.
TIE_POSITION = 5386
TIE_E, TIE_O = -0.4296875, 0.34375


def tie_row():
    x = np.zeros((1, 1, 512), np.float32)
    x[0, 0, 384] = 100.0
    x[0, 0, 494] = TIE_E
    x[0, 0, 495] = TIE_O
    return x


def test_worked_case_rotation_tie(oracle_lib):
    cache = W.rope_cache(8192)
    c = np.float32(cache[TIE_POSITION, 23].item())
    s = np.float32(cache[TIE_POSITION, 32 + 23].item())
    e, o = np.float32(TIE_E), np.float32(TIE_O)
    even = np.float32(np.float32(e * c) + np.float32(o * s))   # numpy fp32: each op rounded
    scale = 0.25                                                 # 2^ceil(log2(100/448))
    assert Fraction(float(even)) / Fraction(scale) == Fraction(7, 2) * Fraction(1, 2 ** 9)
    fused = np.float32(np.float64(e) * np.float64(c) + np.float64(np.float32(o * s)))
    assert float(fused) / scale < 3.5 * 2.0 ** -9                # the fused value is below the tie
    codes, scales = oracle_lib.inv_rope_fp8_quant(
        _bf16(tie_row()), torch.tensor([TIE_POSITION]), cache, 1)
    assert scales[0, 0, 3] == np.float32(scale)
    assert codes[0, 0, 494] == 4                                 # the tie goes to the even code
    assert codes[0, 0, 384] == 0x7C                              # 100 * 4 = 400 = 1.5625 * 2^8


def test_layout_fingerprint_groups(oracle_lib):
    """Token t, head h filled with 2^(h + 2t - 12): scale 2^(h + 2t - 20); codes all
    equal. The scale of every (t, g, hig*4+b) slot identifies which head landed there."""
    N, H, hpg = 3, 12, 4
    G = H // hpg
    x = np.zeros((N, H, 512), np.float32)
    for t in range(N):
        for h in range(H):
            x[t, h] = 2.0 ** (h + 2 * t - 12)
    codes, scales = oracle_lib.inv_rope_fp8_quant(_bf16(x), torch.zeros(N, dtype=torch.int64),
                                                  W.rope_cache(1), hpg)
    assert codes.shape == (N, G, hpg * 512) and scales.shape == (N, G, hpg * 4)
    for t in range(N):
        for g in range(G):
            for hig in range(hpg):
                h = g * hpg + hig
                for b in range(4):
                    # 2^k / 448 -> ceil(log2) = k - 8 (448 = 1.75 * 2^8)
                    assert scales[t, g, hig * 4 + b] == np.float32(2.0 ** (h + 2 * t - 12 - 8))
    assert np.all(codes == 0x78)   # value / scale = 2^8 = 256 -> S.1111.000


def test_strided_input_and_batch_invariance(oracle_lib):
    spec = W.InverseSpec("t", 24, 6, 3, 4096, "uniform", True, seed=11)
    inp = W.inverse_inputs(spec)
    x = inp["x"]
    c_ref, s_ref = oracle_lib.inv_rope_fp8_quant(x, inp["positions"], inp["cos_sin_cache"], 3)
    # head-major storage viewed token-major: token stride 512, head stride N*512
    xt = x.transpose(0, 1).contiguous().transpose(0, 1)
    c2, s2 = oracle_lib.inv_rope_fp8_quant(xt, inp["positions"], inp["cos_sin_cache"], 3)
    assert np.array_equal(c_ref, c2) and np.array_equal(s_ref, s2)
    # padded heads: a slice of a wider buffer
    wide = torch.zeros(24, 9, 512, dtype=torch.bfloat16)
    wide[:, 2:8] = x
    c3, s3 = oracle_lib.inv_rope_fp8_quant(wide[:, 2:8], inp["positions"], inp["cos_sin_cache"], 3)
    assert np.array_equal(c_ref, c3) and np.array_equal(s_ref, s3)
    # batch invariance: tokens 5..12 alone give the same rows
    c4, s4 = oracle_lib.inv_rope_fp8_quant(x[5:13], inp["positions"][5:13], inp["cos_sin_cache"], 3)
    assert np.array_equal(c_ref[5:13], c4) and np.array_equal(s_ref[5:13], s4)
    # threads do not change anything
    c5, s5 = oracle_lib.inv_rope_fp8_quant(x, inp["positions"], inp["cos_sin_cache"], 3, threads=5)
    assert np.array_equal(c_ref, c5) and np.array_equal(s_ref, s5)


def test_grouping_is_a_view(oracle_lib):
    """With contiguous outputs every heads_per_group gives the same bytes."""
    inp = W.inverse_inputs(W.InverseSpec("t", 4, 24, 1, 4096, "uniform", True, seed=12))
    ref = None
    for hpg in (1, 2, 3, 4, 6, 8, 12, 24):
        c, s = oracle_lib.inv_rope_fp8_quant(inp["x"], inp["positions"], inp["cos_sin_cache"], hpg)
        cur = (c.reshape(4, -1).copy(), s.reshape(4, -1).copy())
        if ref is None:
            ref = cur
        assert np.array_equal(cur[0], ref[0]) and np.array_equal(cur[1], ref[1])


def test_op_invariants(oracle_lib):
    """Whole-op properties on the tiny workload: the rotated rows (pinned above
    against complex multiplication) quantise with 224 <= amax/scale <= 448,
    power-of-two scales, and |decode(code) - y/scale| <= half an E4M3 step."""
    inp = W.inverse_inputs(W.TINY)
    x, pos, cache = inp["x"], inp["positions"], inp["cos_sin_cache"]
    codes, scales = oracle_lib.inv_rope_fp8_quant(x, pos, cache, 8)
    N, H = x.shape[:2]
    rows = x.float().numpy().reshape(N * H, 512)
    y = oracle_lib.rope_rows(rows, np.repeat(pos.numpy(), H), cache.numpy(), True)
    y = y.astype(np.float64)
    sc = scales.reshape(N * H, 4).astype(np.float64)
    assert np.all((scales.view(np.uint32) & 0x7FFFFF) == 0)
    amax = np.abs(y).reshape(N * H, 4, 128).max(axis=2)
    ratio = amax / sc
    assert np.all(ratio <= 448.0 * (1 + 2.0 ** -22)) and np.all(ratio >= 224.0 * (1 - 2.0 ** -22))
    deq = oracle_lib.e4m3_decode(codes.reshape(N * H, 512)).reshape(N * H, 4, 128)
    yb = y.reshape(N * H, 4, 128) / sc[:, :, None]
    # half-step of the E4M3 grid at |v|: 2^(max(floor(log2|v|), -6) - 4)
    ex = np.floor(np.log2(np.maximum(np.abs(yb), 2.0 ** -30)))
    half = np.exp2(np.maximum(ex, -6) - 4)
    assert np.all(np.abs(deq - yb) <= half)
    # the worst case is reached: the bound is not loose by a factor of two
    assert np.max(np.abs(deq - yb) / half) > 0.9


def test_tiny_workload_digest_is_stable(oracle_lib):
    """Regression pin: the committed digest of the oracle's output on the tiny
    workload (written by tests/golden/make_golden.py, which calls only the oracle)."""
    import hashlib
    inp = W.inverse_inputs(W.TINY)
    codes, scales = oracle_lib.inv_rope_fp8_quant(inp["x"], inp["positions"],
                                                  inp["cos_sin_cache"], 8)
    h = hashlib.sha256(codes.tobytes() + scales.tobytes()).hexdigest()
    with open(os.path.join(GOLDEN, "tiny_oracle_digest.txt")) as f:
        want = [l.split()[1] for l in f if l.startswith("inverse")][0]
    assert h == want


# ----------------------------------------------------------------- insert op

def test_insert_placement_and_sentinel(oracle_lib):
    spec = W.InsertSpec("t", 40, 4096, 6, 8, seed=13)
    inp = W.insert_inputs(spec)
    slots = inp["slot_mapping"].clone()
    slots[3] = -1                                    # skipped token
    pad = 64                                         # block stride with padding
    bs = spec.block_size
    k_cache = torch.full((spec.num_blocks, bs * 528 + pad), 0xA5, dtype=torch.uint8)
    out = oracle_lib.rope_fp8_quant_insert(inp["kv"], inp["positions"], inp["cos_sin_cache"],
                                           slots, k_cache, bs)
    rows = inp["kv"].float().numpy()
    y = oracle_lib.rope_rows(rows, inp["positions"].numpy(), inp["cos_sin_cache"].numpy(), False)
    codes, scales = oracle_lib.quant_rows(y)
    touched = np.zeros(out.shape, bool)
    for t, s in enumerate(slots.tolist()):
        if s < 0:
            continue
        b, o = divmod(s, bs)
        rec = out[b, o * 528:(o + 1) * 528]
        touched[b, o * 528:(o + 1) * 528] = True
        assert np.array_equal(rec[:512], codes[t])
        assert np.array_equal(rec[512:].view(np.float32), scales[t])
    assert np.all(out[~touched] == 0xA5)
    # the forward rotation is the +theta one (complex pin)
    ref = _complex_rotate(rows, inp["positions"].numpy(), inp["cos_sin_cache"].numpy(), False)
    assert np.allclose(y, ref, atol=1e-5, rtol=0)


# ----------------------------------------------------------------- next rows: bf16 out, UE8M0

def test_bf16_rounding_matches_torch_dense_sweep(oracle_lib):
    """Round-to-nearest-even fp32 -> bf16 against torch's conversion (a library
    routine) over every 97th fp32 bit pattern, both signs, NaN excluded."""
    for sign in (0, 0x80000000):
        bits = (np.arange(0, 0x7F800001, 97, dtype=np.uint64) | sign).astype(np.uint32)
        v = bits.view(np.float32)
        want = torch.from_numpy(v.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(oracle_lib.f32_to_bf16(v), want)


@pytest.mark.parametrize("bits,want", [
    (0x3F808000, 0x3F80),   # 1 + 2^-8: a tie, to the even neighbour 1.0
    (0x3F818000, 0x3F82),   # 1 + 3*2^-8: a tie, to the even neighbour 1 + 2^-6
    (0x3F808001, 0x3F81),   # just above the tie: up
    (0x7F7FFFFF, 0x7F80),   # the largest finite fp32 rounds to +inf
    (0x7F7F7FFF, 0x7F7F),   # below the last tie: the largest finite bf16
    (0x80000000, 0x8000),   # -0 keeps its sign
    (0x00008000, 0x0000),   # subnormal tie to even (0)
    (0x00018000, 0x0002),   # subnormal tie to even (2)
    (0xFF800000, 0xFF80),   # -inf
])
def test_bf16_rounding_worked_cases(oracle_lib, bits, want):
    v = np.array([bits], np.uint32).view(np.float32)
    assert int(oracle_lib.f32_to_bf16(v)[0]) == want


def test_bf16_rounding_keeps_nan(oracle_lib):
    v = np.array([0x7FC00000, 0xFF800001, 0x7F800001], np.uint32).view(np.float32)
    out = oracle_lib.f32_to_bf16(v)
    assert np.all((out & 0x7F80) == 0x7F80) and np.all((out & 0x007F) != 0)


def test_ue8m0_packing_worked_case(oracle_lib):
    """OCP Microscaling E8M0: value 2^(byte - 127); block b in bits 8b..8b+7."""
    s = np.array([2.0 ** -3, 1.0, 2.0 ** 5, 2.0 ** -42], np.float32)
    assert int(oracle_lib.pack_ue8m0(s)[0]) == (85 << 24) | (132 << 16) | (127 << 8) | 124


def test_ue8m0_decodes_to_every_scale_of_a_run(oracle_lib):
    inp = W.inverse_inputs(W.TINY)
    codes, scales = oracle_lib.inv_rope_fp8_quant(inp["x"], inp["positions"],
                                                  inp["cos_sin_cache"], 8)
    packed = oracle_lib.pack_ue8m0(scales)
    assert packed.shape == (64, 1, 8)
    for b in range(4):
        byte = ((packed >> (8 * b)) & 0xFF).astype(np.int64)
        dec = np.ldexp(1.0, byte - 127)
        assert np.array_equal(dec, scales[..., b::4].astype(np.float64))


def test_inv_rope_bf16_is_the_rotation_rounded(oracle_lib):
    """quantize=False: NoPE dims pass through bit-exactly; the rotated dims are
    torch's bf16 rounding of the (separately pinned) fp32 rotation."""
    spec = W.InverseSpec("bf16", 37, 12, 6, 8192, "uniform", True, seed=11)
    inp = W.inverse_inputs(spec)
    out = oracle_lib.inv_rope_bf16(inp["x"], inp["positions"], inp["cos_sin_cache"], 6)
    assert out.shape == (37, 2, 6 * 512)
    xb = inp["x"].view(torch.int16).numpy().view(np.uint16).reshape(37, 12, 512)
    o = out.reshape(37, 12, 512)
    assert np.array_equal(o[..., :448], xb[..., :448])
    rows = oracle_lib.rope_rows(inp["x"].float().numpy().reshape(-1, 512),
                                np.repeat(inp["positions"].numpy(), 12),
                                inp["cos_sin_cache"], inverse=True)
    want = torch.from_numpy(rows).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(o.reshape(-1, 512), want)


# ----------------------------------------------------------------- next rows: fused q/kv op

def _nearest_bf16_bruteforce(v: float) -> int:
    """Exact nearest bf16 to a double (ties to even) by comparing the candidate
    neighbours with exact rational distances."""
    f = np.float32(v)  # a starting point; the answer is within one bf16 step of it
    b = int(np.array([f], np.float32).view(np.uint32)[0] >> 16)
    best = None
    for c in {b - 1, b, b + 1}:
        if c < 0 or c > 0xFFFF or (c & 0x7F80) == 0x7F80:
            continue
        if (c ^ b) & 0x8000:
            continue
        cv = Fraction(float(np.array([c << 16], np.uint32).view(np.float32)[0]))
        d = abs(cv - Fraction(v))
        key = (d, c & 1)            # nearer first, then the even one
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_f64_to_bf16_bruteforce_and_direct_rounding(oracle_lib):
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.standard_normal(1500) * 10.0 ** rng.integers(-30, 30, 1500),
                        rng.standard_normal(200) * 1e-39])
    # exact bf16 midpoints nudged by far less than an fp32 ulp: rounding through
    # fp32 first would land on the midpoint and tie the wrong way
    mids = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 3 * 2.0 ** -9, 1.5 + 2.0 ** -8])
    v = np.concatenate([v, mids, mids + 2.0 ** -40, mids - 2.0 ** -40, -mids])
    got = oracle_lib.f64_to_bf16(v)
    want = np.array([_nearest_bf16_bruteforce(float(a)) for a in v], np.uint16)
    assert np.array_equal(got, want)
    assert int(oracle_lib.f64_to_bf16(np.array([1 + 2.0 ** -8 + 2.0 ** -40]))[0]) == 0x3F81


def _qnorm_case(x_rows, pos, hq, hpad, cache_rows=64, eps=1e-6):
    n = x_rows.shape[0]
    q = torch.tensor(x_rows, dtype=torch.float32).to(torch.bfloat16)
    kv = torch.zeros(n, 512, dtype=torch.bfloat16)
    k_cache = torch.full((2, 4 * 528), 0xA5, dtype=torch.uint8)
    slots = torch.full((n,), -1, dtype=torch.int64)
    return q, kv, torch.tensor(pos), W.rope_cache(cache_rows), slots, k_cache, eps


def test_qnorm_constant_row_is_unit_and_pads_are_zero(oracle_lib):
    x = np.zeros((2, 3, 512), np.float32)
    x[0, 0] = 0.75
    x[0, 1] = -3.0
    x[0, 2] = 2.0 ** -20
    x[1] = 5.0
    q, kv, pos, cache, slots, kc, eps = _qnorm_case(x, [0, 0], 3, 5, eps=0.0)
    q_out, _ = oracle_lib.qnorm_rope_kv_rope_quant_insert(q, kv, pos, cache, slots, kc, 4, 5,
                                                          norm_eps=0.0)
    assert q_out.shape == (2, 5, 512)
    assert np.all(q_out[0, 0] == 0x3F80) and np.all(q_out[0, 1] == 0xBF80)   # +1, -1
    assert np.all(q_out[0, 2] == 0x3F80) and np.all(q_out[1, :3] == 0x3F80)
    assert np.all(q_out[:, 3:] == 0)                                         # pad heads


def test_qnorm_scale_invariance_and_unit_rms(oracle_lib):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 2, 512)).astype(np.float32)
    x = torch.tensor(x).to(torch.bfloat16).float().numpy()                   # bf16-exact
    q1 = oracle_lib.qnorm_rope_kv_rope_quant_insert(*_qnorm_case(x, [0, 1, 2, 3], 2, 2)[:6], 4,
                                                    2, norm_eps=0.0)[0]
    q2 = oracle_lib.qnorm_rope_kv_rope_quant_insert(*_qnorm_case(x * 8.0, [0, 1, 2, 3], 2, 2)[:6],
                                                    4, 2, norm_eps=0.0)[0]
    assert np.array_equal(q1, q2)
    y = torch.from_numpy(q1.view(np.int16)).view(torch.bfloat16).double().numpy()
    rms = np.sqrt((y ** 2).mean(axis=-1))        # a rotation keeps the norm
    assert np.all(np.abs(rms - 1.0) < 4e-3)


def test_qnorm_rotated_tail_matches_complex_multiplication(oracle_lib):
    rng = np.random.default_rng(9)
    x = torch.tensor(rng.standard_normal((6, 1, 512)), dtype=torch.float32).to(torch.bfloat16)
    pos = [0, 1, 7, 100, 1000, 4095]
    cache = W.rope_cache(4096)
    q, kv, p_, _, slots, kc, _ = _qnorm_case(x.float().numpy(), pos, 1, 1, cache_rows=4096)
    q_out, _ = oracle_lib.qnorm_rope_kv_rope_quant_insert(x, kv, p_, cache, slots, kc, 4, 1,
                                                          norm_eps=1e-6)
    xd = x.double().numpy()[:, 0]
    y = xd / np.sqrt((xd ** 2).mean(axis=-1, keepdims=True) + 1e-6)
    c = cache.double().numpy()[pos]
    z = (y[:, 448::2] + 1j * y[:, 449::2]) * (c[:, :32] + 1j * c[:, 32:])      # rotation by +theta
    got = torch.from_numpy(q_out[:, 0].view(np.int16)).view(torch.bfloat16).double().numpy()
    tol = 2.0 ** -8 * np.maximum(np.abs(z), 2.0 ** -120)                       # half a bf16 step + slack
    assert np.all(np.abs(got[:, 448::2] - z.real) <= tol)
    assert np.all(np.abs(got[:, 449::2] - z.imag) <= tol)
    tol_n = 2.0 ** -8 * np.abs(y[:, :448]) + 1e-30
    assert np.all(np.abs(got[:, :448] - y[:, :448]) <= tol_n)


def test_fused_kv_part_is_the_insert_op(oracle_lib):
    spec = W.InsertSpec("fused", 40, 4096, 4, 16, seed=12)
    inp = W.insert_inputs(spec)
    q = torch.randn(40, 3, 512, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    _, kc = oracle_lib.qnorm_rope_kv_rope_quant_insert(q, inp["kv"], inp["positions"],
                                                       inp["cos_sin_cache"], inp["slot_mapping"],
                                                       inp["k_cache"], 16, 4)
    want = oracle_lib.rope_fp8_quant_insert(inp["kv"], inp["positions"], inp["cos_sin_cache"],
                                            inp["slot_mapping"], inp["k_cache"], 16)
    assert np.array_equal(kc, want)


# ----------------------------------------------------------------- next rows: indexer q op

def _idx_worked(oracle_lib, neox: bool, pos: int):
    """One live pair (j = 5) plus a 224 that fixes the head's scale at 2^-1."""
    j = 5
    i0, i1 = (j, 32 + j) if neox else (2 * j, 2 * j + 1)
    q = np.zeros((1, 1, 128), np.float32)
    q[0, 0, i0] = 1.0
    q[0, 0, 100] = 224.0
    cache = W.rope_cache(4096)
    codes, w = oracle_lib.indexer_q_rope_quant(
        torch.tensor(q).to(torch.bfloat16), torch.tensor([pos]), cache,
        torch.tensor([[3.0]]), 128 ** -0.5, 64 ** -0.5, neox=neox)
    # expected: r0 = cos, r1 = sin of the textbook angle, rounded to fp32 (the
    # cache), then to bf16 (the page's .to(bf16)), divided by the scale 1/2 and
    # encoded by torch's float8 cast (all below 448)
    ang = pos * 10000.0 ** (-j / 32)
    cs = torch.tensor([np.cos(ang), np.sin(ang)], dtype=torch.float64).to(torch.float32)
    vals = (cs.to(torch.bfloat16).float() * 2.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return codes[0, 0], w[0, 0], i0, i1, vals


@pytest.mark.parametrize("neox", [True, False], ids=["neox", "gptj"])
@pytest.mark.parametrize("pos", [0, 1, 3000])
def test_indexer_worked_pair(oracle_lib, neox, pos):
    codes, w, i0, i1, vals = _idx_worked(oracle_lib, neox, pos)
    assert codes[i0] == vals[0] and codes[i1] == vals[1]
    assert codes[100] == 0x7E                                   # 224 * 2 = 448
    rest = np.ones(128, bool)
    rest[[i0, i1, 100]] = False
    assert np.all(codes[rest] & 0x7F == 0)      # zeros (a rotated 0 may carry a - sign)
    exact = 3.0 * 0.5 * 128 ** -0.5 * 64 ** -0.5
    assert abs(float(w) - exact) <= 2 * np.spacing(np.float32(exact))


def test_indexer_scales_and_fold_invariants(oracle_lib):
    gen = torch.Generator().manual_seed(4)
    q = (torch.randn(50, 8, 128, generator=gen) * 3).to(torch.bfloat16)
    pos = torch.randint(0, 4096, (50,), generator=gen)
    wts = torch.rand(50, 8, generator=gen) + 0.5
    codes, w = oracle_lib.indexer_q_rope_quant(q, pos, W.rope_cache(4096), wts, 0.125, 0.25)
    q_scale = w.astype(np.float64) / (wts.double().numpy() * 0.125 * 0.25)
    e = np.round(np.log2(q_scale))
    assert np.allclose(q_scale, 2.0 ** e, rtol=2 ** -22)        # a power of two per head
    dec = oracle_lib.e4m3_decode(codes).reshape(50, 8, 128)
    amax_over_scale = np.abs(dec).max(axis=-1)
    assert np.all(amax_over_scale <= 448) and np.all(amax_over_scale >= 224 - 16)
    # NoPE dims 64..127 are the input exactly scaled: decode * scale == x rounded to e4m3
    x = q.float().numpy()[..., 64:] / (2.0 ** e)[..., None]
    want = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes[..., 64:], want)


# ----------------------------------------------------------------- next rows: grouped FP8 GEMM

def test_gemm_oracle_identity_weights(oracle_lib):
    """Weights = 1.0 (e4m3 0x38) on the diagonal, scale 2^-3: y = dequant(A)[:, :, :n_out] / 8."""
    rng = np.random.default_rng(1)
    a = rng.integers(0, 256, (5, 2, 256)).astype(np.uint8)
    a[(a & 0x7F) == 0x7F] = 0x38
    sa = np.ldexp(1.0, rng.integers(-4, 4, (5, 2, 2))).astype(np.float32)
    w = np.zeros((2, 128, 256), np.uint8)
    w[:, np.arange(128), np.arange(128)] = 0x38
    sw = np.full((2, 1, 2), 0.125, np.float32)
    y = oracle_lib.grouped_fp8_gemm(a, sa, w, sw)
    want = oracle_lib.e4m3_decode(a[..., :128]) * sa[..., :1] / 8
    assert np.array_equal(y, want)


def test_gemm_oracle_brute_force(oracle_lib):
    rng = np.random.default_rng(2)
    a = rng.integers(0, 0x7F, (3, 1, 256)).astype(np.uint8) | (rng.integers(0, 2, (3, 1, 256)) << 7).astype(np.uint8)
    w = rng.integers(0, 0x7F, (1, 128, 256)).astype(np.uint8)
    sa = np.ldexp(1.0, rng.integers(-3, 3, (3, 1, 2))).astype(np.float32)
    sw = np.ldexp(1.0, rng.integers(-3, 3, (1, 1, 2))).astype(np.float32)
    y = oracle_lib.grouped_fp8_gemm(a, sa, w, sw)
    dec = {c: oracle_lib.e4m3_decode(np.array([c], np.uint8))[0] for c in range(256)}
    for m in range(3):
        for n in (0, 5, 127):
            s = sum(dec[int(a[m, 0, k])] * float(sa[m, 0, k // 128]) * dec[int(w[0, n, k])] *
                    float(sw[0, 0, k // 128]) for k in range(256))
            assert y[m, 0, n] == s


def test_ue8m0_decode_special_codes(oracle_lib):
    """OCP MX UE8M0: code 127 is 1.0, 0 is 2^-127, 254 is 2^127, 255 is NaN."""
    v = oracle_lib.ue8m0_decode(np.array([0, 1, 126, 127, 128, 254, 255], np.uint8))
    assert v[0] == math.ldexp(1.0, -127) and v[1] == math.ldexp(1.0, -126)
    assert v[2] == 0.5 and v[3] == 1.0 and v[4] == 2.0 and v[5] == math.ldexp(1.0, 127)
    assert math.isnan(v[6])


def test_gemm_ue8m0_oracle_brute_force(oracle_lib):
    """Scales given as UE8M0 codes: every (row, K block) of A has a distinct
    exponent, so a wrong byte inside the packed word or a wrong word (head) shows.
    Decoding here goes through torch's float8_e4m3fn, not the oracle's decoder."""
    rng = np.random.default_rng(3)
    n, k, n_out = 3, 1024, 256              # two heads of 4 blocks per row, 2 weight row blocks
    a = rng.integers(0, 256, (n, 1, k)).astype(np.uint8)
    a[(a & 0x7F) == 0x7F] = 0x30             # no NaN codes
    w = rng.integers(0, 256, (1, n_out, k)).astype(np.uint8)
    w[(w & 0x7F) == 0x7F] = 0x40
    a_exp = (120 + rng.permutation(8 * n).reshape(n, 1, 8)).astype(np.uint32)   # per (row, block)
    words = np.zeros((n, 1, 2), np.uint32)
    for b in range(4):
        words |= a_exp[..., b::4] << (8 * b)   # block 4h + b in byte b of word h
    w_sf = rng.integers(124, 131, (1, n_out // 128, k // 128)).astype(np.uint8)
    y = oracle_lib.grouped_fp8_gemm_ue8m0(a, words, w, w_sf)
    dec = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    for m in range(n):
        for o in (0, 77, 128, 255):
            terms = []
            for kk in range(k):
                kt = kk // 128
                sa = math.ldexp(1.0, int(a_exp[m, 0, kt]) - 127)
                sw = math.ldexp(1.0, int(w_sf[0, o // 128, kt]) - 127)
                terms.append(dec[a[m, 0, kk]] * sa * dec[w[0, o, kk]] * sw)   # each exact
            # fsum is the correctly rounded sum; the oracle's float64 matmul may
            # round each of its 1024 additions
            exact = math.fsum(terms)
            assert abs(y[m, 0, o] - exact) <= 2.0 ** -42 * math.fsum(abs(t) for t in terms)


def test_gemm_ue8m0_oracle_matches_fp32_scales_of_the_op(oracle_lib):
    """The op's UE8M0 output and its fp32 scales are the same powers of two, so
    the GEMM over either scale encoding gives the same float64 result."""
    spec = W.InverseSpec("g", 6, 8, 8, 4096, "uniform", True, seed=4)
    inp = W.inverse_inputs(spec)
    codes, scales = oracle_lib.inv_rope_fp8_quant(inp["x"], inp["positions"], inp["cos_sin_cache"], 8)
    words = oracle_lib.pack_ue8m0(scales.reshape(6, 1, 32))
    rng = np.random.default_rng(5)
    w = rng.integers(0, 0x7F, (1, 128, 4096)).astype(np.uint8)
    e = rng.integers(122, 132, (1, 1, 32)).astype(np.uint8)
    y_ue = oracle_lib.grouped_fp8_gemm_ue8m0(codes.reshape(6, 1, 4096), words, w, e)
    y_f32 = oracle_lib.grouped_fp8_gemm(codes.reshape(6, 1, 4096), scales.reshape(6, 1, 32), w,
                                        np.ldexp(1.0, e.astype(np.int64) - 127).astype(np.float32))
    assert np.array_equal(y_ue, y_f32)


def _bf16_bits(v):
    return torch.tensor(np.asarray(v, np.float32)).to(torch.bfloat16).view(torch.int16).numpy() \
        .view(np.uint16)


def test_qnorm_weight_of_ones_is_the_weightless_norm(oracle_lib):
    rng = np.random.default_rng(11)
    x = torch.tensor(rng.standard_normal((5, 3, 512)), dtype=torch.float32).to(torch.bfloat16)
    args = _qnorm_case(x.float().numpy(), [0, 3, 9, 27, 81], 3, 3, cache_rows=4096)[:6]
    plain = oracle_lib.qnorm_rope_kv_rope_quant_insert(*args, 4, 3, norm_eps=1e-6)[0]
    ones = oracle_lib.qnorm_rope_kv_rope_quant_insert(*args, 4, 3, norm_eps=1e-6,
                                                      norm_weight=_bf16_bits(np.ones(512)))[0]
    assert np.array_equal(plain, ones)


def test_qnorm_weight_scales_each_dimension_before_the_rotation(oracle_lib):
    """Weight 2^a(k), equal within each rotated pair: rounding to bf16 commutes
    with a power of two, so every output value is the weightless one times
    2^a(k), exactly. The per-dimension pattern pins the weight's indexing, and
    the pair rule pins that it acts before the rotation (a weight applied after
    it would scale the pair's members differently once they mix)."""
    rng = np.random.default_rng(12)
    x = torch.tensor(rng.standard_normal((4, 2, 512)), dtype=torch.float32).to(torch.bfloat16)
    args = _qnorm_case(x.float().numpy(), [1, 5, 50, 500], 2, 2, cache_rows=4096)[:6]
    a = (np.arange(512) // 2) % 4 - 1           # -1..2, constant on each (2j, 2j+1) pair
    w = np.ldexp(1.0, a)
    plain = oracle_lib.qnorm_rope_kv_rope_quant_insert(*args, 4, 2, norm_eps=1e-6)[0]
    got = oracle_lib.qnorm_rope_kv_rope_quant_insert(*args, 4, 2, norm_eps=1e-6,
                                                     norm_weight=_bf16_bits(w))[0]
    to_f = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(to_f(got), to_f(plain) * w)
    # a weight that differs inside a rotated pair is not a per-dimension scaling of
    # the output there (the rotation mixes the pair after the weight)
    w2 = np.ones(512)
    w2[448] = 4.0
    got2 = oracle_lib.qnorm_rope_kv_rope_quant_insert(*args, 4, 2, norm_eps=1e-6,
                                                      norm_weight=_bf16_bits(w2))[0]
    f2, fp = to_f(got2), to_f(plain)
    assert np.array_equal(f2[..., :448], fp[..., :448])
    assert not np.array_equal(f2[..., 449], fp[..., 449])   # the partner moved with it


def test_bit_range_drivers_are_the_scalar_steps(oracle_lib):
    """The bit-pattern range drivers that the exhaustive GPU checks compare
    against add no arithmetic: element by element they equal the pinned
    encoder (on the scaled value) and the pinned block scale (on the eps-clamped
    amax), at chunk edges, around zero, subnormals, 448, infinities and NaNs,
    and with several threads."""
    starts = [0, 0x00000001 - 1, 0x007FFF00, 0x3E5FFF00, 0x43DFFF80, 0x7F7FFF00, 0x7F800000,
              0x80000000, 0x807FFF00, 0xC3DFFF80, 0xFF7FFF00, 0xFFFFFF00]
    for first in starts:
        n = min(256, (1 << 32) - first)
        bits = (np.arange(n, dtype=np.uint64) + first).astype(np.uint32)
        v = bits.view(np.float32)
        for e in (0, -9, 5, 126, -126):
            got = oracle_lib.e4m3_encode_bits_range(first, n, e, threads=3)
            want = oracle_lib.e4m3_encode((v.astype(np.float64) / 2.0 ** e).astype(np.float32)) \
                if e in (0,) else np.array([oracle_lib.e4m3_encode_scalar(float(x) / 2.0 ** e)
                                            for x in v], np.uint8)
            assert np.array_equal(got, want), (hex(first), e)
    for first in (0, 0x0D7FFF00, 0x3F5FFF80, 0x43DFFF80, 0x7F7FFF00):
        n = 256
        amax = (np.arange(n, dtype=np.uint64) + first).astype(np.uint32).view(np.float32)
        for eps in (2.0 ** -100, 1e-10, 1e-4):
            e32 = np.float32(eps)
            got = oracle_lib.block_scale_bits_range(first, n, float(e32), threads=4)
            want = oracle_lib.block_scale(np.maximum(amax, e32))
            assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (hex(first), eps)
    with pytest.raises(oracle_lib.OracleError):
        oracle_lib.e4m3_encode_bits_range(0xFFFFFFF0, 32)
