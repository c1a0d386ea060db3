"""Exhaustive on-device checks of the per-block arithmetic every quantising
kernel runs, against the oracle's independent statement of it.

* The block scale: for EVERY finite non-negative fp32 block amax (all
  2,139,095,040 patterns), the kernels' integer rule on amax's bits gives the
  bits of 2^ceil(log2(fl32(max(amax, eps) / 448))), exactly as the oracle's
  frexp-based ceiling does ("[vllm] vLLM의 GLM5.2 성능 최적화", S1, applied to
  the block absmax of the inverse-RoPE page, S3), at the smallest eps the ABI
  accepts and at the default; and the kernels' inverse scale is its exact
  reciprocal.
* The quantisation: for EVERY fp32 bit pattern (2^32 values), the kernels'
  exact scaling plus cvt.rn.satfinite.e4m3x2 gives the oracle's OFP8
  nearest-even, saturating code (inverse-RoPE page, S3); NaN inputs (outside
  the op's contract) only have to give a NaN code. Other block scales are
  checked on spread-out ranges of patterns.

Both sides evaluate in chunks; the GPU side is the library's test-only entry
points rq_debug_block_scale / rq_debug_quant_codes, which run the kernels' own
device functions.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

FINITE_POSITIVE_END = 0x7F800000        # +inf: patterns below it are the finite amax >= 0
TWO32 = 1 << 32
NAN_RANGES = ((0x7F800001, 0x80000000), (0xFF800001, TWO32))


@pytest.fixture(scope="module")
def rq():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import rope_block_fp8_inverse_b300 as rq
    rq.lib()
    return rq


def _chunks(begin, end, size):
    c = begin
    while c < end:
        yield c, min(size, end - c)
        c += size


@pytest.mark.parametrize("eps", [2.0 ** -100, 1e-10], ids=["eps2^-100", "eps1e-10"])
def test_block_scale_rule_every_finite_amax(rq, eps):
    eps32 = float(np.float32(eps))
    for first, n in _chunks(0, FINITE_POSITIVE_END, 1 << 27):
        s_dev, inv_dev = rq.debug_block_scale(first, n, eps32)
        # the inverse is exact: scale * inv == 1 in float64 (both powers of two)
        assert bool(torch.all(s_dev.double() * inv_dev.double() == 1.0)), \
            f"inverse scale not exact in chunk {first:#010x}"
        s = s_dev.cpu().numpy()
        want = oracle.block_scale_bits_range(first, n, eps32)
        bad = np.flatnonzero(s.view(np.uint32) != want.view(np.uint32))
        assert bad.size == 0, (
            f"scale differs for amax bits {first + int(bad[0]):#010x}: "
            f"kernel {s[bad[0]]!r}, oracle {want[bad[0]]!r} ({bad.size} patterns in chunk)")
        del s_dev, inv_dev


def _compare_codes(first, got, want):
    """Exact for every pattern except NaNs, which only need a NaN code."""
    n = got.size
    mask = np.ones(n, dtype=bool)
    for lo, hi in NAN_RANGES:
        a, b = max(lo, first), min(hi, first + n)
        if a < b:
            mask[a - first:b - first] = False
            nan_codes = got[a - first:b - first]
            assert np.all((nan_codes & 0x7F) == 0x7F), \
                f"a NaN input gave a non-NaN code in [{a:#010x}, {b:#010x})"
    bad = np.flatnonzero((got != want) & mask)
    assert bad.size == 0, (
        f"code differs for fp32 bits {first + int(bad[0]):#010x}: kernel {int(got[bad[0]]):#04x}, "
        f"oracle {int(want[bad[0]]):#04x} ({bad.size} patterns in chunk)")


def test_quant_codes_every_fp32_pattern(rq):
    buf = torch.empty(1 << 28, dtype=torch.uint8, device="cuda")
    for first, n in _chunks(0, TWO32, 1 << 28):
        got = rq.debug_quant_codes(first, n, 0, out=buf).cpu().numpy()
        want = oracle.e4m3_encode_bits_range(first, n, 0)
        _compare_codes(first, got, want)


@pytest.mark.parametrize("scale_exp", [-126, -42, -20, -9, -1, 1, 7, 20, 64, 126])
def test_quant_codes_other_block_scales(rq, scale_exp):
    """Sixteen ranges of 2^22 patterns spread over the whole fp32 space
    (both signs, every binade region), at a block scale of 2^scale_exp."""
    n = 1 << 22
    buf = torch.empty(n, dtype=torch.uint8, device="cuda")
    gen = np.random.default_rng(scale_exp & 0xFFFF)
    starts = [(k << 28) + int(gen.integers(0, (1 << 28) - n)) // 16 * 16 for k in range(16)]
    for first in starts:
        got = rq.debug_quant_codes(first, n, scale_exp, out=buf).cpu().numpy()
        want = oracle.e4m3_encode_bits_range(first, n, scale_exp)
        _compare_codes(first, got, want)


def test_debug_entry_points_reject_bad_arguments(rq):
    lib = rq.lib()
    buf = torch.empty(64, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert lib.rq_debug_quant_codes(0, 17, 0, buf.data_ptr(), st) != 0       # not a multiple of 16
    assert lib.rq_debug_quant_codes(0, 16, 127, buf.data_ptr(), st) != 0     # exponent out of range
    assert lib.rq_debug_quant_codes(TWO32 - 16, 32, 0, buf.data_ptr(), st) != 0  # past 2^32
    f = torch.empty(16, dtype=torch.float32, device="cuda")
    assert lib.rq_debug_block_scale(0, 16, 0.0, f.data_ptr(), f.data_ptr(), st) != 0  # eps
    assert lib.rq_debug_block_scale(0, 0, 1e-10, 0, 0, st) == 0              # empty is fine
