"""CPU checks of the exact reformulations the CUDA kernels use, against the oracle.

The kernels never divide amax by 448 nor take a logarithm: they build the
scale's fp32 bit pattern from amax's bits, ((bits + 0x1fffff) & 0x7f800000) -
(8 << 23), i.e. 2^(E-8) when amax's mantissa field is <= 0x600000 and
2^(E-7) above it, and the inverse scale as (254 << 23) minus that pattern.
This test restates that rule (it is the kernel's formula, not the oracle's)
and compares it with the oracle's definition, 2^ceil(log2(fl32(amax / 448))),
at every binade boundary and over a dense stride of all normal fp32 values
>= 2^-100 (the ABI's smallest eps, so the smallest possible amax).
"""
import numpy as np


def kernel_scale_rule(amax: np.ndarray):
    u = amax.view(np.uint32).astype(np.uint64)
    sbits = (((u + 0x1FFFFF) & 0x7F800000) - (8 << 23)).astype(np.uint32)
    inv = ((254 << 23) - sbits.astype(np.int64)).astype(np.uint32)
    return sbits.view(np.float32), inv.view(np.float32)


def kernel_exponent_rule(amax: np.ndarray) -> np.ndarray:
    s, inv = kernel_scale_rule(amax)
    assert np.all(s.astype(np.float64) * inv.astype(np.float64) == 1.0)
    return ((s.view(np.uint32) >> 23) & 0xFF).astype(np.int64) - 127


def _oracle_exponent(oracle_lib, amax):
    s = oracle_lib.block_scale(amax)
    return ((s.view(np.uint32) >> 23) & 0xFF).astype(np.int64) - 127


def test_scale_exponent_rule_at_binade_boundaries(oracle_lib):
    parts = []
    for E in range(-100, 128):
        lo_bits = (E + 127) << 23
        for m in (0x000000, 0x5FFFFF, 0x600000, 0x600001, 0x7FFFFF):
            c = lo_bits | m
            parts.append(np.arange(max(c - 40, lo_bits), min(c + 41, lo_bits + (1 << 23)),
                                   dtype=np.int64))
    bits = np.unique(np.concatenate(parts))
    bits = bits[bits < 0x7F800000].astype(np.uint32)
    amax = bits.view(np.float32)
    assert np.array_equal(kernel_exponent_rule(amax), _oracle_exponent(oracle_lib, amax))


def test_scale_exponent_rule_dense_sweep(oracle_lib):
    lo = int(np.float32(2.0 ** -100).view(np.uint32))
    step = 1 << 24
    for start in range(lo, 0x7F800000, step * 11):
        bits = np.arange(start, min(start + step, 0x7F800000), 3, dtype=np.uint32)
        amax = bits.view(np.float32)
        assert np.array_equal(kernel_exponent_rule(amax), _oracle_exponent(oracle_lib, amax))
