"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bar (the tolerance stated for this op): scales bit-exact; FP8 codes exact
except for at most 1e-4 of elements, each of those at most one E4M3 step
away (which keeps the dequantised value within 1 E4M3 ulp); the paged
scatter bit-exact in placement. The kernels are designed to be bit-exact
(same fp32 op order, no FMA, exact power-of-two scaling), and the tests
also report, and for the small cases require, zero mismatches.
"""
import os

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

CODE_MISMATCH_FRACTION = 1e-4
THREADS = max(1, min(32, os.cpu_count() or 1))


@pytest.fixture(scope="module")
def rq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rope_block_fp8_inverse_b300 import build
    build.build()
    import rope_block_fp8_inverse_b300 as m
    return m


def _e4m3_step_apart(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """True where codes a and b are adjacent on the E4M3 number line (or +-0)."""
    def ordinal(c):
        c = c.astype(np.int32)
        mag = c & 0x7F
        return np.where(c & 0x80, -mag, mag)
    return np.abs(ordinal(a) - ordinal(b)) <= 1


def assert_parity(got_codes, got_scales, want_codes, want_scales, exact=False):
    gc = got_codes.reshape(-1)
    wc = want_codes.reshape(-1)
    gs = got_scales.reshape(-1).view(np.uint32)
    ws = want_scales.reshape(-1).view(np.uint32)
    assert gc.shape == wc.shape and gs.shape == ws.shape
    bad_s = np.nonzero(gs != ws)[0]
    assert bad_s.size == 0, f"{bad_s.size} scales differ, first at {bad_s[:5]}"
    bad = np.nonzero(gc != wc)[0]
    if exact:
        assert bad.size == 0, (f"{bad.size} codes differ; first {bad[:8]}: "
                               f"got {gc[bad[:8]]} want {wc[bad[:8]]}")
    assert bad.size <= CODE_MISMATCH_FRACTION * gc.size, f"{bad.size} of {gc.size} codes differ"
    assert np.all(_e4m3_step_apart(gc[bad], wc[bad]))
    return bad.size


VARIANT_IDS = {1: "warp_rows", 2: "stream"}
VARIANTS = pytest.mark.parametrize("variant", list(VARIANT_IDS), ids=list(VARIANT_IDS.values()))


def run_inverse(rq, inp, eps=1e-10, x_override=None, variant=0):
    dev = torch.device("cuda:0")
    x = (x_override if x_override is not None else inp["x"]).to(dev)
    pos = inp["positions"].to(dev)
    cache = inp["cos_sin_cache"].to(dev)
    codes, scales = rq.inv_rope_fp8_quant(x, pos, cache, inp["heads_per_group"], eps=eps,
                                          variant=variant)
    torch.cuda.synchronize()
    return codes.view(torch.uint8).cpu().numpy(), scales.cpu().numpy()


def oracle_inverse(inp, eps=1e-10, x=None):
    import oracle
    return oracle.inv_rope_fp8_quant(inp["x"] if x is None else x, inp["positions"],
                                     inp["cos_sin_cache"], inp["heads_per_group"], eps=eps,
                                     threads=THREADS)


# ---------------------------------------------------------------- inverse op

@VARIANTS
def test_tiny_workload_exact(rq, variant):
    inp = W.inverse_inputs(W.TINY)
    gc, gs = run_inverse(rq, inp, variant=variant)
    wc, ws = oracle_inverse(inp)
    assert gc.shape == (64, 1, 8 * 512) and gs.shape == (64, 1, 32)
    assert_parity(gc, gs, wc, ws, exact=True)


@pytest.mark.parametrize("n", W.DECODE_TOKENS)
@VARIANTS
def test_decode_sweep_exact(rq, variant, n):
    inp = W.inverse_inputs(W.decode_spec(n))
    gc, gs = run_inverse(rq, inp, variant=variant)
    wc, ws = oracle_inverse(inp)
    assert_parity(gc, gs, wc, ws, exact=True)


@pytest.mark.parametrize("h,groups", W.PAGE_TEST_SHAPES,
                         ids=[f"H{h}_G{g}" for h, g in W.PAGE_TEST_SHAPES])
@pytest.mark.parametrize("n", [1, 37, 300])
@VARIANTS
def test_page_test_shapes(rq, variant, h, groups, n):
    """The (H, groups) shapes of the inverse-RoPE page's test (S5), ragged N."""
    spec = W.InverseSpec(f"page{h}x{groups}", n, h, h // groups, 8192, "uniform", True, seed=n)
    inp = W.inverse_inputs(spec)
    gc, gs = run_inverse(rq, inp, variant=variant)
    wc, ws = oracle_inverse(inp)
    assert gc.shape == (n, groups, (h // groups) * 512)
    assert_parity(gc, gs, wc, ws, exact=True)


@VARIANTS
def test_irregular_grouping_full(rq, variant):
    """N=8192, H=24, heads_per_group=6: every output compared."""
    inp = W.inverse_inputs(W.IRREGULAR)
    gc, gs = run_inverse(rq, inp, variant=variant)
    wc, ws = oracle_inverse(inp)
    assert gc.shape == (8192, 4, 6 * 512)
    assert_parity(gc, gs, wc, ws, exact=True)


_FULL = {}


def _full_size(name):
    """Inputs and oracle outputs of a full-size workload, computed once per
    test module (the multi-threaded oracle takes about a second for each)."""
    if name not in _FULL:
        if name == "prefill16k":
            inp = W.inverse_inputs(W.PREFILL16K)
            _FULL[name] = (inp, oracle_inverse(inp))
        elif name == "prefill16k_bf16":
            inp, _ = _full_size("prefill16k")
            _FULL[name] = (inp, oracle_layout(inp, "bf16"))
        elif name == "indexer16k_neox" or name == "indexer16k_gptj":
            inp = W.indexer_inputs(W.INDEXER16K)
            _FULL[name] = (inp, oracle_indexer(inp, name.rsplit("_", 1)[1]))
    return _FULL[name]


@VARIANTS
def test_prefill16k_every_output(rq, variant):
    """Full-size launch (N=16384, H=32, hpg=8, the benchmarked configuration):
    every code and every scale of all 16384 tokens against the oracle."""
    inp, (wc, ws) = _full_size("prefill16k")
    gc, gs = run_inverse(rq, inp, variant=variant)
    assert gc.shape == (16384, 4, 4096) and gs.shape == (16384, 4, 32)
    assert_parity(gc, gs, wc, ws, exact=True)
    # properties at every output: scales are powers of two, no NaN codes
    assert np.all((gs.view(np.uint32) & 0x7FFFFF) == 0)
    assert not np.any((gc & 0x7F) == 0x7F)


@VARIANTS
def test_strided_inputs(rq, variant):
    """Token / head strides other than [N, H, 512] contiguous give the same bytes."""
    spec = W.InverseSpec("strided", 77, 16, 4, 4096, "uniform", True, seed=3)
    inp = W.inverse_inputs(spec)
    wc, ws = oracle_inverse(inp)
    x = inp["x"]
    wide = torch.zeros(77, 21, 512, dtype=torch.bfloat16)
    wide[:, 3:19] = x
    head_major = x.transpose(0, 1).contiguous().transpose(0, 1)
    # head stride of 520 elements (a multiple of 8, not 16) and a base 16 bytes
    # past a 32-byte boundary: kernels that read 32 bytes per lane must fall back
    odd = torch.zeros(77, 16, 520, dtype=torch.bfloat16)
    odd[:, :, 8:] = x
    for xv in (wide.cuda()[:, 3:19], head_major.cuda(), odd.cuda()[:, :, 8:]):
        gc, gs = run_inverse(rq, inp, x_override=xv, variant=variant)
        assert_parity(gc, gs, wc, ws, exact=True)


def test_batch_invariance_across_launch_shapes(rq):
    """A token's bytes do not depend on the batch it came with (small calls
    take the one-row-per-warp launch, large ones two rows per warp)."""
    inp = W.inverse_inputs(W.InverseSpec("bi", 4096, 32, 8, 65536, "uniform", True, seed=5))
    gc, gs = run_inverse(rq, inp)
    for lo, hi in ((0, 1), (100, 164), (4000, 4096)):
        sub = {k: (v[lo:hi] if k in ("x", "positions") else v) for k, v in inp.items()}
        c2, s2 = run_inverse(rq, sub)
        assert np.array_equal(gc[lo:hi], c2) and np.array_equal(gs[lo:hi], s2)


def test_variants_identical_at_full_size(rq):
    """Every kernel variant writes the same bytes on the benchmarked shape."""
    inp = W.inverse_inputs(W.PREFILL16K)
    ref = run_inverse(rq, inp, variant=1)
    for v in (0, 2):
        got = run_inverse(rq, inp, variant=v)
        assert np.array_equal(ref[0], got[0]) and np.array_equal(ref[1], got[1]), v


@pytest.mark.parametrize("eps", [1e-10, 1e-4, 2.0 ** -100, 3.5])
@VARIANTS
def test_eps_and_special_values(rq, variant, eps):
    """Zero blocks (scale from eps), subnormal bf16, exact saturation, signed zeros."""
    n, h = 6, 4
    gen = torch.Generator().manual_seed(21)
    x = torch.zeros(n, h, 512, dtype=torch.float32)
    x[1] = torch.randn(h, 512, generator=gen) * 1e-38       # bf16 subnormals
    x[2, :, ::7] = 448.0
    x[2, :, 1::7] = -448.0 * 2 ** -12
    x[3] = -0.0
    x[4, :, 448:] = torch.randn(h, 64, generator=gen) * 3   # only the rotated dims live
    x[5] = torch.randn(h, 512, generator=gen) * 2.0 ** 60
    spec_inp = {"x": x.to(torch.bfloat16), "positions": torch.tensor([0, 1, 2, 3, 4, 5]),
                "cos_sin_cache": W.rope_cache(64), "heads_per_group": 2}
    gc, gs = run_inverse(rq, spec_inp, eps=eps, variant=variant)
    wc, ws = oracle_inverse(spec_inp, eps=eps)
    assert_parity(gc, gs, wc, ws, exact=True)


@VARIANTS
def test_rotation_tie_is_not_fused(rq, variant):
    """A rotated value on an exact e4m3 rounding tie (the oracle pin's worked
    case): an FMA anywhere in the rotation would flip its code."""
    from test_oracle_pins import TIE_POSITION, tie_row
    inp = {"x": torch.tensor(tie_row()).to(torch.bfloat16).expand(3, 4, 512).contiguous(),
           "positions": torch.tensor([TIE_POSITION] * 3), "cos_sin_cache": W.rope_cache(8192),
           "heads_per_group": 2}
    gc, gs = run_inverse(rq, inp, variant=variant)
    wc, ws = oracle_inverse(inp)
    assert wc[0, 0, 494] == 4
    assert_parity(gc, gs, wc, ws, exact=True)


@VARIANTS
def test_position_out_of_range_flags_and_skips(rq, variant):
    """The kernel's own bounds check: a bad position skips the token (outputs
    untouched) and sets RQ_FLAG_POSITION_RANGE; the other tokens are exact."""
    inp = W.inverse_inputs(W.InverseSpec("oob", 8, 8, 8, 100, "uniform", True, seed=9))
    pos = inp["positions"].clone()
    pos[2] = 100          # == cache_rows
    pos[5] = -1
    dev = torch.device("cuda:0")
    out = torch.full((8, 1, 4096), 0x5A, dtype=torch.uint8, device=dev)
    scales = torch.full((8, 1, 32), -7.0, device=dev)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    rq.inv_rope_fp8_quant(inp["x"].to(dev), pos.to(dev), inp["cos_sin_cache"].to(dev), 8,
                          out=out, scales=scales, error_flags=flags, variant=variant)
    torch.cuda.synchronize()
    assert int(flags.item()) == 1
    o = out.cpu().numpy()
    s = scales.cpu().numpy()
    assert np.all(o[[2, 5]] == 0x5A) and np.all(s[[2, 5]] == -7.0)
    keep = [0, 1, 3, 4, 6, 7]
    sub = {"x": inp["x"][keep], "positions": pos[keep], "cos_sin_cache": inp["cos_sin_cache"],
           "heads_per_group": 8}
    wc, ws = oracle_inverse(sub)
    assert_parity(o[keep], s[keep], wc, ws, exact=True)


def test_preallocated_fp8_output_and_stream(rq):
    """The `_out` form: caller-owned float8 output, a non-default stream."""
    inp = W.inverse_inputs(W.TINY)
    dev = torch.device("cuda:0")
    out = torch.empty(64, 1, 4096, dtype=torch.float8_e4m3fn, device=dev)
    scales = torch.empty(64, 1, 32, device=dev)
    x, pos, cache = inp["x"].to(dev), inp["positions"].to(dev), inp["cos_sin_cache"].to(dev)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        c, sc = rq.inv_rope_fp8_quant(x, pos, cache, 8, out=out, scales=scales)
    s.synchronize()
    assert c.data_ptr() == out.data_ptr() and sc.data_ptr() == scales.data_ptr()
    wc, ws = oracle_inverse(inp)
    assert_parity(out.view(torch.uint8).cpu().numpy(), scales.cpu().numpy(), wc, ws, exact=True)


# ---------------------------------------------------------------- insert op

def run_insert(rq, inp, k_cache=None, slots=None, eps=1e-10, flags=None, kv=None,
               positions=None):
    dev = torch.device("cuda:0")
    kc = (inp["k_cache"] if k_cache is None else k_cache).to(dev).contiguous()
    sl = (inp["slot_mapping"] if slots is None else slots).to(dev)
    kvd = (inp["kv"] if kv is None else kv).to(dev)
    pos = (inp["positions"] if positions is None else positions).to(dev)
    rq.rope_fp8_quant_insert(kvd, pos, inp["cos_sin_cache"].to(dev), sl, kc, inp["block_size"],
                             eps=eps, error_flags=flags)
    torch.cuda.synchronize()
    return kc.cpu().numpy()


def oracle_insert(inp, k_cache=None, slots=None, eps=1e-10):
    import oracle
    return oracle.rope_fp8_quant_insert(inp["kv"], inp["positions"], inp["cos_sin_cache"],
                                        inp["slot_mapping"] if slots is None else slots,
                                        inp["k_cache"] if k_cache is None else k_cache,
                                        inp["block_size"], eps=eps, threads=THREADS)


def _assert_cache_parity(got, want):
    """Placement bit-exact: every byte outside records equal; inside records
    the scales bit-exact and the codes within the stated tolerance."""
    assert got.shape == want.shape
    diff = np.nonzero(got.reshape(-1) != want.reshape(-1))[0]
    assert diff.size == 0, f"{diff.size} cache bytes differ, first at {diff[:8]}"


def test_insert16k_full(rq):
    inp = W.insert_inputs(W.INSERT16K)
    got = run_insert(rq, inp)
    want = oracle_insert(inp)
    _assert_cache_parity(got, want)
    assert got.shape == (512, 64 * 528)


def test_insert_records_past_4gib(rq):
    """A paged k_cache larger than 4 GiB (131,072 blocks of 64 records of 528
    bytes, 4.43 GB): 16,384 tokens go to distinct slots, half of them drawn
    from the slots whose records start past byte 2^32. Every written record
    equals the oracle's record of the same token (computed into a small cache
    with slots 0..N-1: a record's bytes do not depend on its slot), and the
    untouched records of a sample and the cache's last record keep the
    sentinel."""
    n, num_blocks, bs = 16384, 131072, 64
    inp = W.insert_inputs(W.InsertSpec("ins4g", n, 65536, n // bs, bs, seed=3))
    n_slots = num_blocks * bs
    first_high = (2 ** 32 + 527) // 528  # first slot whose record starts past 2^32
    gen = torch.Generator().manual_seed(11)
    hi = first_high + torch.randperm(n_slots - first_high, generator=gen)[: n // 2]
    lo = torch.randperm(first_high, generator=gen)[: n // 2]
    slots = torch.cat([hi, lo])[torch.randperm(n, generator=gen)]
    dev = torch.device("cuda:0")
    kc = torch.full((num_blocks, bs * 528), 0xA5, dtype=torch.uint8, device=dev)
    rq.rope_fp8_quant_insert(inp["kv"].to(dev), inp["positions"].to(dev),
                             inp["cos_sin_cache"].to(dev), slots.to(dev), kc, bs)
    torch.cuda.synchronize()
    records = kc.view(-1, 528)
    got = records[slots.to(dev)].cpu().numpy()
    want = oracle_insert(inp, slots=torch.arange(n, dtype=torch.int64)).reshape(-1, 528)
    assert np.array_equal(got, want), f"{int((got != want).any(axis=1).sum())} records differ"
    taken = torch.zeros(n_slots, dtype=torch.bool)
    taken[slots] = True
    others = torch.randint(0, n_slots, (8192,), generator=gen)
    others = torch.cat([others[~taken[others]], torch.tensor([n_slots - 1])])
    others = others[~taken[others]]
    assert torch.all(records[others.to(dev)] == 0xA5)
    del kc, records
    torch.cuda.empty_cache()


@pytest.mark.parametrize("n", [1, 5, 64, 1000])
def test_insert_ragged_and_padded_blocks(rq, n):
    blocks = 2 * W.ceil_div(n, 16) + 1
    spec = W.InsertSpec("ins", n, 4096, blocks, 16, seed=n)
    inp = W.insert_inputs(spec)
    pad = 16 * 528 + 48                          # block stride with padding bytes
    kc = torch.full((blocks, pad), 0xA5, dtype=torch.uint8)
    slots = inp["slot_mapping"].clone()
    if n > 3:
        slots[::3] = -1                          # skipped tokens
    got = run_insert(rq, inp, k_cache=kc, slots=slots)
    want = oracle_insert(inp, k_cache=kc, slots=slots)
    _assert_cache_parity(got, want)


def test_insert_slot_out_of_range_flags(rq):
    spec = W.InsertSpec("ins-oob", 6, 64, 2, 4, seed=2)
    inp = W.insert_inputs(spec)
    slots = torch.tensor([0, 8, 3, -1, 100, 7])   # 8 slots: 8 and 100 are out of range
    flags = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    got = run_insert(rq, inp, slots=slots, flags=flags)
    assert int(flags.item()) == 2
    ok = torch.tensor([0, -1, 3, -1, -1, 7])
    want = oracle_insert(inp, slots=ok)
    _assert_cache_parity(got, want)


def test_insert_position_out_of_range_flags(rq):
    """A bad position skips its token (record untouched) and sets the flag."""
    spec = W.InsertSpec("ins-pos", 9, 64, 3, 4, seed=4)
    inp = W.insert_inputs(spec)
    pos = inp["positions"].clone()
    pos[1] = 64
    pos[6] = -3
    flags = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    got = run_insert(rq, inp, flags=flags, positions=pos)
    assert int(flags.item()) == 1
    slots = inp["slot_mapping"].clone()
    slots[[1, 6]] = -1
    want = oracle_insert(inp, slots=slots)
    _assert_cache_parity(got, want)


def test_insert_strided_kv(rq):
    """kv rows with a token stride of 520 elements (not contiguous) give the same bytes."""
    spec = W.InsertSpec("ins-strided", 300, 4096, 10, 32, seed=6)
    inp = W.insert_inputs(spec)
    wide = torch.zeros(300, 520, dtype=torch.bfloat16)
    wide[:, :512] = inp["kv"]
    got = run_insert(rq, inp, kv=wide.cuda()[:, :512])
    want = oracle_insert(inp)
    _assert_cache_parity(got, want)


def test_outputs_past_4gib(rq):
    """Byte offsets past 2^32: 270,000 tokens x 32 heads (8.64 M rows; x is 8.8
    GB and the codes 4.4 GB, so the last rows' offsets exceed 4 GiB) through
    the plain op, the layout call with group-major codes, and the layout call
    with transposed fp32 scales (the token-tiled kernel). The first and last 48
    tokens and 64 others are compared with the oracle run on those tokens
    alone. x follows the input recipe (randn, 1% of values x50, bf16),
    generated on the device in chunks from a seeded generator."""
    n, h, hpg = 270_000, 32, 8
    g = h // hpg
    dev = torch.device("cuda:0")
    gen = torch.Generator(device=dev).manual_seed(2024)
    x = torch.empty((n, h, 512), dtype=torch.bfloat16, device=dev)
    for c in range(0, n, 16384):
        v = torch.randn((min(16384, n - c), h, 512), generator=gen, device=dev)
        m = torch.rand(v.shape, generator=gen, device=dev) < W.OUTLIER_RATE
        x[c:c + v.shape[0]] = torch.where(m, v * W.OUTLIER_GAIN, v).to(torch.bfloat16)
        del v, m
    cache = W.rope_cache(65536)
    pos = torch.randint(0, 65536, (n,), generator=gen, device=dev)
    cache_d = cache.to(dev)
    mid = torch.randint(48, n - 48, (64,), generator=torch.Generator().manual_seed(5)).tolist()
    sample = sorted(set(range(48)) | set(range(n - 48, n)) | set(mid))
    idx = torch.tensor(sample, device=dev)
    sub = {"x": x[idx].cpu(), "positions": pos[idx].cpu(), "cos_sin_cache": cache,
           "heads_per_group": hpg}
    wc, ws = oracle_inverse(sub)

    def check(codes, scales):
        torch.cuda.synchronize()
        gc = codes[idx].contiguous().view(torch.uint8).cpu().numpy()
        gs = scales[idx].contiguous().cpu().numpy()
        assert_parity(gc, gs, wc, ws, exact=True)

    codes, scales = rq.inv_rope_fp8_quant(x, pos, cache_d, hpg)
    check(codes, scales)
    del codes, scales
    out, sc = rq.empty_outputs(n, g, hpg, "fp8", group_major=True, device=dev)
    rq.inv_rope_quant(x, pos, cache_d, hpg, mode="fp8", out=out, scales=sc)
    check(out, sc)
    del out, sc
    out = torch.empty((n, g, hpg * 512), dtype=torch.uint8, device=dev)
    sc = torch.empty((g, hpg * 4, n), dtype=torch.float32, device=dev).permute(2, 0, 1)
    rq.inv_rope_quant(x, pos, cache_d, hpg, mode="fp8", out=out, scales=sc)
    check(out, sc)
    del out, sc, x
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- output kinds and layouts

LAYOUTS = ["token_major", "group_major", "scales_transposed", "group_major_padded"]
GROUP_PAD = 3  # tokens of padding after each group in the padded group-major storage


def _outputs(rq, n, g, hpg, mode, layout):
    dev = torch.device("cuda:0")
    out, sc = rq.empty_outputs(n, g, hpg, mode, group_major=(layout == "group_major"), device=dev)
    if layout == "scales_transposed" and sc is not None:
        w = sc.shape[2]
        sc = torch.empty((g, w, n), dtype=sc.dtype, device=dev).permute(2, 0, 1)
    if layout == "group_major_padded":
        # [G, N + pad, W] storage: a group stride that is not N * W
        out = torch.empty((g, n + GROUP_PAD, out.shape[2]), dtype=out.dtype,
                          device=dev)[:, :n].permute(1, 0, 2)
        if sc is not None:
            sc = torch.empty((g, n + GROUP_PAD, sc.shape[2]), dtype=sc.dtype,
                             device=dev)[:, :n].permute(1, 0, 2)
    return out, sc


def run_layout(rq, inp, mode, layout):
    dev = torch.device("cuda:0")
    x = inp["x"].to(dev)
    n, h = x.shape[0], x.shape[1]
    hpg = inp["heads_per_group"]
    out, sc = _outputs(rq, n, h // hpg, hpg, mode, layout)
    if mode == "bf16":
        out.view(torch.int16).fill_(0x5A5A)
    else:
        out.view(torch.uint8).fill_(0x5A)
    rq.inv_rope_quant(x, inp["positions"].to(dev), inp["cos_sin_cache"].to(dev), hpg, mode=mode,
                      out=out, scales=sc)
    torch.cuda.synchronize()
    if mode == "bf16":
        return out.contiguous().view(torch.int16).cpu().numpy().view(np.uint16), None
    return out.contiguous().view(torch.uint8).cpu().numpy(), sc.contiguous().cpu().numpy()


def oracle_layout(inp, mode):
    import oracle
    if mode == "bf16":
        return oracle.inv_rope_bf16(inp["x"], inp["positions"], inp["cos_sin_cache"],
                                    inp["heads_per_group"]), None
    codes, scales = oracle_inverse(inp)
    if mode == "ue8m0":
        return codes, oracle.pack_ue8m0(scales).view(np.int32)
    return codes, scales


def assert_layout_parity(mode, got, want):
    if mode == "bf16":
        assert np.array_equal(got[0], want[0]), f"{np.count_nonzero(got[0] != want[0])} bf16 differ"
    elif mode == "ue8m0":
        assert got[0].shape == want[0].shape and got[1].shape == want[1].shape
        assert np.array_equal(got[1].view(np.uint32), want[1].view(np.uint32))
        assert np.array_equal(got[0], want[0])
    else:
        assert_parity(got[0], got[1], want[0], want[1], exact=True)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("mode", list(["fp8", "ue8m0", "bf16"]))
@pytest.mark.parametrize("case", ["tiny", "irregular_small", "decode1", "page24x4"])
def test_layout_modes_exact(rq, case, mode, layout):
    spec = {"tiny": W.TINY,
            "irregular_small": W.InverseSpec("irr", 300, 24, 6, 32768, "uniform", True, seed=7),
            "decode1": W.decode_spec(1),
            "page24x4": W.InverseSpec("p24", 37, 24, 6, 8192, "uniform", True, seed=37)}[case]
    inp = W.inverse_inputs(spec)
    got = run_layout(rq, inp, mode, layout)
    want = oracle_layout(inp, mode)
    assert_layout_parity(mode, got, want)


def test_layout_fp8_equals_the_plain_entry_at_full_size(rq):
    """Token-major fp32-scale output of the layout entry is byte-identical to
    rq_inv_rope_fp8_quant on the benchmarked shape; group-major holds the same
    bytes permuted."""
    inp = W.inverse_inputs(W.PREFILL16K)
    ref = run_inverse(rq, inp)
    for layout in ("token_major", "group_major"):
        got = run_layout(rq, inp, "fp8", layout)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1]), layout


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("mode", ["fp8", "ue8m0", "bf16"])
def test_layout_full_size_every_output(rq, mode, layout):
    """Full-size calls (the kernel each layout takes at 16384 tokens x 32
    heads): every output of all 16384 tokens against the oracle."""
    if mode == "bf16":
        inp, want = _full_size("prefill16k_bf16")
    else:
        import oracle
        inp, (wc, ws) = _full_size("prefill16k")
        want = (wc, oracle.pack_ue8m0(ws).view(np.int32)) if mode == "ue8m0" else (wc, ws)
    got = run_layout(rq, inp, mode, layout)
    assert_layout_parity(mode, got, want)


@pytest.mark.parametrize("mode", ["fp8", "ue8m0", "bf16"])
def test_layout_padded_group_major_leaves_the_padding_alone(rq, mode):
    """Padded group-major storage: every output byte equals the oracle's and
    the padding tokens after each group keep their sentinel (no write lands
    outside the view)."""
    inp = W.inverse_inputs(W.InverseSpec("pad", 300, 32, 8, 4096, "uniform", True, seed=5))
    dev = torch.device("cuda:0")
    n, g, hpg = 300, 4, 8
    w = hpg * 512
    odt = torch.bfloat16 if mode == "bf16" else torch.uint8
    ost = torch.empty((g, n + GROUP_PAD, w), dtype=odt, device=dev)
    ost.view(torch.uint8).fill_(0xA5)
    out = ost[:, :n].permute(1, 0, 2)
    sst, sc = None, None
    if mode != "bf16":
        sw, sdt = (hpg * 4, torch.float32) if mode == "fp8" else (hpg, torch.int32)
        sst = torch.empty((g, n + GROUP_PAD, sw), dtype=sdt, device=dev)
        sst.view(torch.uint8).fill_(0xA5)
        sc = sst[:, :n].permute(1, 0, 2)
    rq.inv_rope_quant(inp["x"].to(dev), inp["positions"].to(dev), inp["cos_sin_cache"].to(dev),
                      hpg, mode=mode, out=out, scales=sc)
    torch.cuda.synchronize()
    assert torch.all(ost[:, n:].view(torch.uint8) == 0xA5)
    if sst is not None:
        assert torch.all(sst[:, n:].view(torch.uint8) == 0xA5)
    if mode == "bf16":
        got = (out.contiguous().view(torch.int16).cpu().numpy().view(np.uint16), None)
    else:
        got = (out.contiguous().view(torch.uint8).cpu().numpy(), sc.contiguous().cpu().numpy())
    assert_layout_parity(mode, got, oracle_layout(inp, mode))


@pytest.mark.parametrize("mode", ["fp8", "ue8m0"])
def test_layout_irregular_full(rq, mode):
    """heads_per_group = 6 at full size: tiles of 8 heads would cross groups, so
    the warp-rows layout kernel runs; every output compared."""
    inp = W.inverse_inputs(W.IRREGULAR)
    got = run_layout(rq, inp, mode, "group_major")
    assert_layout_parity(mode, got, oracle_layout(inp, mode))


def test_layout_bad_position_flags_and_skips(rq):
    inp = W.inverse_inputs(W.InverseSpec("lay-oob", 5, 8, 4, 100, "uniform", True, seed=9))
    pos = inp["positions"].clone()
    pos[3] = 100
    dev = torch.device("cuda:0")
    out, sc = rq.empty_outputs(5, 2, 4, "ue8m0", group_major=True, device=dev)
    out.fill_(0x5A)
    sc.fill_(-7)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    rq.inv_rope_quant(inp["x"].to(dev), pos.to(dev), inp["cos_sin_cache"].to(dev), 4,
                      mode="ue8m0", out=out, scales=sc, error_flags=flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 1
    o, s = out.cpu().numpy(), sc.cpu().numpy()
    assert np.all(o[3] == 0x5A) and np.all(s[3] == -7)
    keep = [0, 1, 2, 4]
    sub = {"x": inp["x"][keep], "positions": pos[keep], "cos_sin_cache": inp["cos_sin_cache"],
           "heads_per_group": 4}
    want = oracle_layout(sub, "ue8m0")
    assert np.array_equal(o[keep], want[0]) and np.array_equal(s[keep].view(np.uint32),
                                                               want[1].view(np.uint32))


def test_layout_token_contiguous_fp32_scales_ragged_with_skips(rq):
    """fp32 scales stored token-contiguous ([G, hpg*4, N] inside a padded
    [G, hpg*4, N + 5] buffer) from x with padded strides, at 8191 tokens x 32
    heads, a size at which the layout call takes the token-tiled kernel on
    B300 (tiles of 8 tokens, at least 6 per warp): a ragged last tile, and
    out-of-range positions at a tile's first and last token, mid-call and in
    the ragged tile. The skipped tokens are flagged and their codes and
    scales keep their sentinels, the padding after each scale row keeps its
    sentinel, and every other output equals the oracle's."""
    n, h, hpg = 8191, 32, 8
    g = h // hpg
    inp = W.inverse_inputs(W.InverseSpec("tok-contig", n, h, hpg, 65536, "uniform", True, seed=11))
    pos = inp["positions"].clone()
    bad = [0, 7, 8, 4000, 8184, 8190]
    pos[bad] = 65536
    pos[4000] = -3
    dev = torch.device("cuda:0")
    out = torch.full((n, g, hpg * 512), 0x5A, dtype=torch.uint8, device=dev)
    sst = torch.full((g, hpg * 4, n + 5), -7.0, dtype=torch.float32, device=dev)
    sc = sst[:, :, :n].permute(2, 0, 1)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    # x with padded head and token strides (520 and 33 * 520 elements)
    wide = torch.zeros((n, h + 1, 520), dtype=torch.bfloat16, device=dev)
    wide[:, :h, :512] = inp["x"].to(dev)
    rq.inv_rope_quant(wide[:, :h, :512], pos.to(dev), inp["cos_sin_cache"].to(dev), hpg,
                      mode="fp8", out=out, scales=sc, error_flags=flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 1
    assert torch.all(sst[:, :, n:] == -7.0)
    o, s = out.cpu().numpy(), sc.contiguous().cpu().numpy()
    assert np.all(o[bad] == 0x5A) and np.all(s[bad] == -7.0)
    keep = sorted(set(range(n)) - set(bad))
    sub = {"x": inp["x"][keep], "positions": pos[keep], "cos_sin_cache": inp["cos_sin_cache"],
           "heads_per_group": hpg}
    want = oracle_layout(sub, "fp8")
    assert_layout_parity("fp8", (o[keep], s[keep]), want)


# ---------------------------------------------------------------- fused q/kv op

# q_out tolerance (fp32 kernel vs the fp64 oracle, both rounded to bf16):
#   NoPE dims: within one bf16 step of the oracle;
#   rotated dims: |got - want| <= ulp(got)/2 + ulp(want)/2 + 2^-16 * |pair|,
#     |pair| = the oracle pair's Euclidean norm, covering the fp32 rounding of
#     the norm factor and of the two products when they nearly cancel;
#   and at most 1% of all values not bit-identical.
BF16_INEXACT_FRACTION = 1e-2


def _bf16_ordinal(u):
    u = u.astype(np.int32)
    mag = u & 0x7FFF
    return np.where(u & 0x8000, -mag, mag)


def _bf16_to_f64(u):
    return torch.from_numpy(np.ascontiguousarray(u).view(np.int16)).view(torch.bfloat16).double().numpy()


def _bf16_ulp(v):
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a >= 2.0 ** -126, np.exp2(e - 7), 2.0 ** -133)


def run_fused(rq, inp, norm_eps=1e-6, q=None, positions=None, flags=None, q_out=None,
              weight=None):
    dev = torch.device("cuda:0")
    kc = inp["k_cache"].to(dev).contiguous()
    qd = (inp["q"] if q is None else q).to(dev)
    pos = (inp["positions"] if positions is None else positions).to(dev)
    out = rq.qnorm_rope_kv_rope_quant_insert(
        qd, inp["kv"].to(dev), pos, inp["cos_sin_cache"].to(dev), inp["slot_mapping"].to(dev), kc,
        inp["block_size"], inp["q_head_padded"], norm_eps=norm_eps, error_flags=flags,
        q_out=q_out, norm_weight=None if weight is None else weight.to(dev))
    torch.cuda.synchronize()
    return out.view(torch.int16).cpu().numpy().view(np.uint16), kc.cpu().numpy()


def oracle_fused(inp, norm_eps=1e-6, positions=None, slots=None, weight=None):
    import oracle
    return oracle.qnorm_rope_kv_rope_quant_insert(
        inp["q"], inp["kv"], inp["positions"] if positions is None else positions,
        inp["cos_sin_cache"], inp["slot_mapping"] if slots is None else slots, inp["k_cache"],
        inp["block_size"], inp["q_head_padded"], norm_eps=norm_eps, norm_weight=weight)


def assert_fused_parity(got, want, n_heads_q):
    gq, gc = got
    wq, wc = want
    assert np.array_equal(gc, wc), f"{np.count_nonzero(gc != wc)} cache bytes differ"
    assert np.all(gq[:, n_heads_q:] == 0) and np.all(wq[:, n_heads_q:] == 0)
    g, w = gq[:, :n_heads_q], wq[:, :n_heads_q]
    steps = np.abs(_bf16_ordinal(g[..., :448]) - _bf16_ordinal(w[..., :448]))
    assert steps.max() <= 1, f"NoPE dims: max bf16 step distance {steps.max()}"
    gr, wr = _bf16_to_f64(g[..., 448:]), _bf16_to_f64(w[..., 448:])
    pair = np.sqrt(wr[..., 0::2] ** 2 + wr[..., 1::2] ** 2).repeat(2, axis=-1)
    tol = 0.5 * _bf16_ulp(gr) + 0.5 * _bf16_ulp(wr) + 2.0 ** -16 * pair
    bad = np.abs(gr - wr) > tol
    assert not bad.any(), f"{bad.sum()} rotated values beyond the bound"
    inexact = np.count_nonzero(g != w)
    assert inexact <= BF16_INEXACT_FRACTION * g.size, inexact
    return inexact


@pytest.mark.parametrize("n,hq,hpad", [(1, 1, 1), (7, 16, 64), (300, 32, 64), (64, 32, 32)])
def test_fused_small_shapes(rq, n, hq, hpad):
    spec = W.FusedSpec("f", n, hq, hpad, 4096, 2 * W.ceil_div(n, 16) + 1, 16, seed=n + hq)
    inp = W.fused_inputs(spec)
    assert_fused_parity(run_fused(rq, inp), oracle_fused(inp), hq)


@pytest.mark.parametrize("weighted", [False, True])
def test_fused16k_full(rq, weighted):
    """The 16k-token shape, every output compared (the page's weightless norm,
    and with a synthetic RMSNorm weight)."""
    inp = W.fused_inputs(W.FUSED16K)
    w = W.norm_weight(W.FUSED16K.seed) if weighted else None
    got = run_fused(rq, inp, weight=w)
    assert got[0].shape == (16384, 64, 512)
    assert_fused_parity(got, oracle_fused(inp, weight=w), 32)


@pytest.mark.parametrize("n,hq,hpad", [(1, 1, 1), (33, 4, 8), (130, 16, 16)])
def test_fused_norm_weight_small_shapes(rq, n, hq, hpad):
    """A weight with zeros, negatives and a spread of magnitudes, per dimension."""
    spec = W.FusedSpec("fw", n, hq, hpad, 4096, 2 * W.ceil_div(n, 16) + 1, 16, seed=n + 7)
    inp = W.fused_inputs(spec)
    gen = torch.Generator().manual_seed(n)
    w = (torch.randn(512, generator=gen) * 2.0).to(torch.bfloat16)
    w[::37] = 0.0
    assert_fused_parity(run_fused(rq, inp, weight=w), oracle_fused(inp, weight=w), hq)


@pytest.mark.parametrize("norm_eps", [0.0, 1e-6, 1.0])
def test_fused_eps_zero_rows_and_strided_q(rq, norm_eps):
    spec = W.FusedSpec("fe", 9, 4, 8, 256, 3, 8, seed=3)
    inp = W.fused_inputs(spec)
    q = inp["q"].clone()
    q[2, 1] = 0.0 if norm_eps > 0 else 1.0          # a zero head needs eps > 0
    q[4] = q[4] * 2.0 ** 40                          # large values: the norm removes the scale
    q[5, :, 448:] = 0.0                              # only NoPE dims live
    inp["q"] = q
    wide = torch.zeros(9, 7, 512, dtype=torch.bfloat16)
    wide[:, 2:6] = q
    got = run_fused(rq, inp, norm_eps=norm_eps, q=wide.cuda()[:, 2:6])
    assert_fused_parity(got, oracle_fused(inp, norm_eps=norm_eps), 4)


def test_fused_bad_position_flags_and_skips(rq):
    spec = W.FusedSpec("fb", 6, 2, 4, 64, 2, 8, seed=5)
    inp = W.fused_inputs(spec)
    pos = inp["positions"].clone()
    pos[3] = 64
    dev = torch.device("cuda:0")
    q_out = torch.full((6, 4, 512), 7.0, dtype=torch.bfloat16, device=dev)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    gq, gc = run_fused(rq, inp, positions=pos, flags=flags, q_out=q_out)
    assert int(flags.item()) == 1
    seven = int(torch.tensor(7.0, dtype=torch.bfloat16).view(torch.int16).item())
    assert np.all(gq[3, :2] == seven) and np.all(gq[3, 2:] == 0)
    keep = [0, 1, 2, 4, 5]
    slots = inp["slot_mapping"].clone()
    slots[3] = -1
    sub = dict(inp, q=inp["q"][keep], kv=inp["kv"][keep], positions=pos[keep],
               slot_mapping=slots[keep])
    wq, wc = oracle_fused(sub)
    assert_fused_parity((gq[keep], gc), (wq, wc), 2)


# ---------------------------------------------------------------- indexer q op

def run_indexer(rq, inp, style, q=None, positions=None, flags=None, out=None):
    dev = torch.device("cuda:0")
    qd = (inp["q"] if q is None else q).to(dev)
    pos = (inp["positions"] if positions is None else positions).to(dev)
    codes, w = rq.indexer_q_rope_quant(qd, pos, inp["cos_sin_cache"].to(dev),
                                       inp["weights"].to(dev), inp["softmax_scale"],
                                       inp["head_scale"], rope_style=style, error_flags=flags,
                                       out=out)
    torch.cuda.synchronize()
    return codes.view(torch.uint8).cpu().numpy(), w.cpu().numpy()


def oracle_indexer(inp, style, positions=None):
    import oracle
    return oracle.indexer_q_rope_quant(inp["q"], inp["positions"] if positions is None else positions,
                                       inp["cos_sin_cache"], inp["weights"], inp["softmax_scale"],
                                       inp["head_scale"], neox=(style == "neox"))


@pytest.mark.parametrize("style", ["neox", "gptj"])
@pytest.mark.parametrize("n,h", [(1, 1), (3, 64), (37, 7), (500, 64), (1, 9), (5, 9)])
def test_indexer_exact(rq, style, n, h):
    """Small shapes against the oracle, bit-exact. (1, 9): no whole-token sweep
    holds a multiple of 4 heads, so the row-walk kernel runs; (5, 9): the
    fixed-head kernel over two sweeps of 4 tokens with an odd head count."""
    spec = W.IndexerSpec("idx", n, h, 4096, seed=n + h)
    inp = W.indexer_inputs(spec)
    inp["positions"] = torch.randint(0, 4096, (n,), generator=torch.Generator().manual_seed(n))
    gc, gw = run_indexer(rq, inp, style)
    wc, ww = oracle_indexer(inp, style)
    assert np.array_equal(gc, wc), f"{np.count_nonzero(gc != wc)} codes differ"
    assert np.array_equal(gw.view(np.uint32), ww.view(np.uint32))


@pytest.mark.parametrize("style", ["neox", "gptj"])
def test_indexer16k_every_output(rq, style):
    """Full size (16384 tokens x 64 heads of 128): every code and folded
    weight against the oracle."""
    inp, (wc, ww) = _full_size(f"indexer16k_{style}")
    gc, gw = run_indexer(rq, inp, style)
    assert np.array_equal(gc, wc), f"{np.count_nonzero(gc != wc)} codes differ"
    assert np.array_equal(gw.view(np.uint32), ww.view(np.uint32))


def test_indexer_bad_position_flags_and_skips(rq):
    inp = W.indexer_inputs(W.IndexerSpec("idx-oob", 5, 6, 64, seed=1))
    pos = inp["positions"].clone()
    pos[2] = -1
    dev = torch.device("cuda:0")
    out = torch.full((5, 6, 128), 0x5A, dtype=torch.uint8, device=dev)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    gc, gw = run_indexer(rq, inp, "neox", positions=pos, flags=flags, out=out)
    assert int(flags.item()) == 1 and np.all(gc[2] == 0x5A)
    keep = [0, 1, 3, 4]
    sub = dict(inp, q=inp["q"][keep], weights=inp["weights"][keep], positions=pos[keep])
    wc, ww = oracle_indexer(sub, "neox")
    assert np.array_equal(gc[keep], wc) and np.array_equal(gw[keep], ww)


# ---------------------------------------------------------------- CUDA graphs

def test_every_entry_point_replays_in_a_cuda_graph(rq):
    """Every call is stream-ordered with no host synchronisation and no
    allocation inside the library, so it can be captured in a CUDA graph; the
    replayed bytes equal an eager run's."""
    dev = torch.device("cuda:0")
    inv = W.inverse_inputs(W.InverseSpec("g", 300, 32, 8, 4096, "uniform", True, seed=8))
    ins = W.insert_inputs(W.InsertSpec("g", 300, 4096, 10, 32, seed=8), cache=inv["cos_sin_cache"])
    fus = W.fused_inputs(W.FusedSpec("g", 300, 16, 32, 4096, 10, 32, seed=8), cache=inv["cos_sin_cache"])
    idx = W.indexer_inputs(W.IndexerSpec("g", 300, 8, 4096, seed=8), cache=inv["cos_sin_cache"])
    x, pos, cache = inv["x"].to(dev), inv["positions"].to(dev), inv["cos_sin_cache"].to(dev)
    kv, kpos, sl = ins["kv"].to(dev), ins["positions"].to(dev), ins["slot_mapping"].to(dev)
    fq, fkv, fsl = fus["q"].to(dev), fus["kv"].to(dev), fus["slot_mapping"].to(dev)
    iq, iw = idx["q"].to(dev), idx["weights"].to(dev)
    gen = torch.Generator().manual_seed(8)
    gw = _rand_codes((4, 256, 4096), gen).to(dev)
    gsw = (2.0 ** torch.randint(-10, -6, (4, 2, 32), generator=gen).float()).to(dev)
    gsf = (torch.log2(gsw).round().to(torch.int32) + 127).to(torch.uint8)
    bufs = {}

    def outputs():
        bufs["codes"] = torch.empty(300, 4, 4096, dtype=torch.uint8, device=dev)
        bufs["scales"] = torch.empty(300, 4, 32, device=dev)
        bufs["lay"] = rq.empty_outputs(300, 4, 8, "ue8m0", group_major=True, device=dev)
        bufs["kc"] = ins["k_cache"].to(dev)
        bufs["fkc"] = fus["k_cache"].to(dev)
        bufs["qo"] = torch.empty(300, 32, 512, dtype=torch.bfloat16, device=dev)
        bufs["ic"] = torch.empty(300, 8, 128, dtype=torch.uint8, device=dev)
        bufs["iw"] = torch.empty(300, 8, device=dev)
        bufs["mx"] = (torch.empty(300, 4, 4096, dtype=torch.uint8, device=dev),
                      torch.empty(300, 4, 8, dtype=torch.int32, device=dev))
        bufs["y"] = torch.empty(300, 4, 256, dtype=torch.bfloat16, device=dev)
        bufs["ymx"] = torch.empty(300, 4, 256, dtype=torch.bfloat16, device=dev)
        bufs["yfused"] = torch.empty(300, 4, 256, dtype=torch.bfloat16, device=dev)

    def step():
        rq.inv_rope_fp8_quant(x, pos, cache, 8, out=bufs["codes"], scales=bufs["scales"])
        rq.inv_rope_quant(x, pos, cache, 8, mode="ue8m0", out=bufs["lay"][0], scales=bufs["lay"][1])
        rq.rope_fp8_quant_insert(kv, kpos, cache, sl, bufs["kc"], 32)
        rq.qnorm_rope_kv_rope_quant_insert(fq, fkv, kpos, cache, fsl, bufs["fkc"], 32, 32,
                                           q_out=bufs["qo"])
        rq.indexer_q_rope_quant(iq, kpos, cache, iw, idx["softmax_scale"], idx["head_scale"],
                                out=bufs["ic"], weights_out=bufs["iw"])
        rq.grouped_fp8_gemm(bufs["codes"], bufs["scales"], gw, gsw, out=bufs["y"])
        rq.inv_rope_quant(x, pos, cache, 8, mode="ue8m0", out=bufs["mx"][0], scales=bufs["mx"][1])
        rq.grouped_fp8_gemm_ue8m0(bufs["mx"][0], bufs["mx"][1], gw, gsf, out=bufs["ymx"])
        rq.inv_rope_fp8_quant_gemm(x, pos, cache, 8, gw, gsw, out=bufs["yfused"])

    def snapshot():
        return {k: (tuple(t.clone() for t in v) if isinstance(v, tuple) else v.clone())
                for k, v in bufs.items()}

    outputs()
    step()
    torch.cuda.synchronize()
    eager = snapshot()
    outputs()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    got = snapshot()
    for k in eager:
        a, b = eager[k], got[k]
        if isinstance(a, tuple):
            assert all(torch.equal(u, v) for u, v in zip(a, b)), k
        else:
            assert torch.equal(a, b), k


# ---------------------------------------------------------------- grouped FP8 GEMM (tensor cores)

def _rand_codes(shape, gen):
    c = torch.randint(0, 256, shape, generator=gen, dtype=torch.int32).to(torch.uint8)
    c[(c & 0x7F) == 0x7F] = 0x38              # no NaN codes
    return c


def _gemm_bound(a, sa, w, sw, want):
    """|got - want| <= 2^-8 |want| (bf16 output) + 2^-20 sum_k |a_k w_k| (fp32
    accumulation inside the MMA and across K blocks)."""
    import oracle
    mag = oracle.grouped_fp8_gemm(a.numpy() & 0x7F, sa, w.numpy() & 0x7F, sw)
    return 2.0 ** -8 * np.abs(want) + 2.0 ** -20 * mag


def assert_gemm_parity(got, a, sa, w, sw):
    import oracle
    want = oracle.grouped_fp8_gemm(a, sa, w, sw)
    bound = _gemm_bound(a, sa, w, sw, want)
    err = np.abs(got.double().cpu().numpy() - want)
    assert np.all(err <= bound), f"{np.count_nonzero(err > bound)} outputs beyond the bound"


@pytest.mark.parametrize("m,g,k,n_out", [(1, 1, 128, 128), (128, 1, 128, 128), (300, 2, 512, 256),
                                         (257, 4, 4096, 128), (130, 1, 1024, 384)])
def test_gemm_random_codes(rq, m, g, k, n_out):
    gen = torch.Generator().manual_seed(m + k)
    a, w = _rand_codes((m, g, k), gen), _rand_codes((g, n_out, k), gen)
    sa = 2.0 ** torch.randint(-8, 4, (m, g, k // 128), generator=gen).float()
    sw = 2.0 ** torch.randint(-12, -4, (g, n_out // 128, k // 128), generator=gen).float()
    dev = torch.device("cuda:0")
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    y = rq.grouped_fp8_gemm(a.to(dev), sa.to(dev), w.to(dev), sw.to(dev), error_flags=flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    assert_gemm_parity(y, a, sa, w, sw)


@pytest.mark.parametrize("m,g,k,n_out", [(1, 4, 4096, 1024), (2, 1, 512, 128), (7, 3, 1536, 384),
                                         (16, 2, 2048, 256), (33, 1, 3072, 640), (64, 4, 4096, 1024),
                                         (9, 2, 2560, 128), (48, 1, 3584, 256)])
def test_gemm_fp32_decode_sizes(rq, m, g, k, n_out):
    """Up to 64 tokens (K a multiple of 512) the fp32-scale GEMM runs its
    split-K cluster kernel: one accumulator per K block, the two scales folded
    per block. Scales here are arbitrary fp32 values (not powers of two), and
    every output is compared with the float64 oracle's bound."""
    gen = torch.Generator().manual_seed(500 + m * 7 + k)
    a, w = _rand_codes((m, g, k), gen), _rand_codes((g, n_out, k), gen)
    sa = (torch.rand((m, g, k // 128), generator=gen) + 0.5) * 2.0 ** torch.randint(
        -8, 4, (m, g, k // 128), generator=gen).float()
    sw = (torch.rand((g, n_out // 128, k // 128), generator=gen) + 0.5) * 2.0 ** torch.randint(
        -12, -4, (g, n_out // 128, k // 128), generator=gen).float()
    dev = torch.device("cuda:0")
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    y = rq.grouped_fp8_gemm(a.to(dev), sa.to(dev), w.to(dev), sw.to(dev), error_flags=flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    assert_gemm_parity(y, a, sa.numpy(), w, sw.numpy())


def test_gemm_fp32_decode_consumes_the_op_output(rq):
    """Decode steps with the op's default output (fp32 scales): the op
    rewrites the same buffers and the split-K GEMM reads them right behind it,
    five rounds, each against the oracle."""
    dev = torch.device("cuda:0")
    gen = torch.Generator().manual_seed(23)
    w = _rand_codes((4, 1024, 4096), gen)
    sw = (torch.rand((4, 8, 32), generator=gen) + 0.5) * 2.0 ** -8
    wd, swd = w.to(dev), sw.to(dev)
    codes = torch.empty((8, 4, 4096), dtype=torch.uint8, device=dev)
    scales = torch.empty((8, 4, 32), dtype=torch.float32, device=dev)
    y = torch.empty((8, 4, 1024), dtype=torch.bfloat16, device=dev)
    ins = [W.inverse_inputs(W.InverseSpec("decf", 8, 32, 8, 4096, "uniform", True, seed=60 + r))
           for r in range(5)]
    got = []
    for inp in ins:
        rq.inv_rope_fp8_quant(inp["x"].to(dev), inp["positions"].to(dev),
                              inp["cos_sin_cache"].to(dev), 8, out=codes, scales=scales)
        rq.grouped_fp8_gemm(codes, scales, wd, swd, out=y)
        got.append(y.clone())
    torch.cuda.synchronize()
    for inp, yr in zip(ins, got):
        wc, ws = oracle_inverse(inp)
        assert_gemm_parity(yr, torch.from_numpy(wc), ws, w, sw.numpy())


def test_gemm_consumes_the_inverse_op_output(rq):
    """The op's own codes and scales (bit-exact with the oracle) feed the GEMM."""
    inp = W.inverse_inputs(W.InverseSpec("gemm", 200, 16, 8, 4096, "uniform", True, seed=4))
    dev = torch.device("cuda:0")
    codes, scales = rq.inv_rope_fp8_quant(inp["x"].to(dev), inp["positions"].to(dev),
                                          inp["cos_sin_cache"].to(dev), 8)
    gen = torch.Generator().manual_seed(5)
    w = _rand_codes((2, 256, 4096), gen)
    sw = 2.0 ** torch.randint(-10, -6, (2, 2, 32), generator=gen).float()
    y = rq.grouped_fp8_gemm(codes, scales, w.to(dev), sw.to(dev))
    torch.cuda.synchronize()
    wc, ws = oracle_inverse(inp)
    assert_gemm_parity(y, torch.from_numpy(wc), ws, w, sw)


@pytest.mark.parametrize("n,h,hpg,n_out", [(1, 8, 8, 128), (200, 16, 8, 256), (300, 24, 6, 128),
                                           (129, 32, 8, 384)])
def test_fused_gemm_equals_op_then_gemm(rq, n, h, hpg, n_out):
    """The fused kernel produces the A operand in shared memory with the op's
    arithmetic, so its output equals the op followed by the GEMM bit for bit;
    the GEMM part is also checked against the float64 oracle."""
    inp = W.inverse_inputs(W.InverseSpec("fg", n, h, hpg, 4096, "uniform", True, seed=n))
    dev = torch.device("cuda:0")
    x, pos, cache = inp["x"].to(dev), inp["positions"].to(dev), inp["cos_sin_cache"].to(dev)
    g, k = h // hpg, hpg * 512
    gen = torch.Generator().manual_seed(h)
    w = _rand_codes((g, n_out, k), gen)
    sw = 2.0 ** torch.randint(-10, -6, (g, n_out // 128, k // 128), generator=gen).float()
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    y = rq.inv_rope_fp8_quant_gemm(x, pos, cache, hpg, w.to(dev), sw.to(dev), error_flags=flags)
    codes, scales = rq.inv_rope_fp8_quant(x, pos, cache, hpg)
    y2 = rq.grouped_fp8_gemm(codes, scales, w.to(dev), sw.to(dev))
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    wc, ws = oracle_inverse(inp)
    assert_gemm_parity(y, torch.from_numpy(wc), ws, w, sw)


def test_fused_gemm_full_size_matches_op_then_gemm(rq):
    inp = W.inverse_inputs(W.PREFILL16K)
    dev = torch.device("cuda:0")
    x, pos, cache = inp["x"].to(dev), inp["positions"].to(dev), inp["cos_sin_cache"].to(dev)
    gen = torch.Generator().manual_seed(3)
    w = _rand_codes((4, 256, 4096), gen).to(dev)
    sw = (2.0 ** torch.randint(-10, -6, (4, 2, 32), generator=gen).float()).to(dev)
    y = rq.inv_rope_fp8_quant_gemm(x, pos, cache, 8, w, sw)
    codes, scales = rq.inv_rope_fp8_quant(x, pos, cache, 8)
    y2 = rq.grouped_fp8_gemm(codes, scales, w, sw)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


# ---------------------------------------------------------------- grouped FP8 GEMM, UE8M0 scales

def _ue8m0_case(m, g, k, n_out, seed):
    """Random codes, A scale codes per (row, 128-block) in [118, 134), packed
    four to a word, and W codes per 128 x 128 block in [120, 130)."""
    gen = torch.Generator().manual_seed(seed)
    a, w = _rand_codes((m, g, k), gen), _rand_codes((g, n_out, k), gen)
    ea = torch.randint(118, 134, (m, g, k // 128), generator=gen, dtype=torch.int64)
    words = (ea.view(m, g, k // 512, 4) << torch.tensor([0, 8, 16, 24])).sum(-1)
    a_sf = words.to(torch.uint32).view(torch.int32) if hasattr(torch, "uint32") else \
        words.to(torch.int64).to(torch.int32)
    w_sf = torch.randint(120, 130, (g, n_out // 128, k // 128), generator=gen,
                         dtype=torch.int32).to(torch.uint8)
    sa = torch.ldexp(torch.ones(()), (ea - 127).float()).float()
    sw = torch.ldexp(torch.ones(()), (w_sf.long() - 127).float()).float()
    return a, a_sf, w, w_sf, sa, sw


@pytest.mark.parametrize("m,g,k,n_out", [(1, 1, 512, 128), (128, 1, 512, 256), (300, 2, 1024, 384),
                                         (257, 4, 4096, 1024), (1000, 1, 2048, 640),
                                         (5, 3, 4096, 128)])
def test_gemm_ue8m0_random_codes(rq, m, g, k, n_out):
    """Every row and K block has its own scale code, so a wrong scale-factor
    layout (row, K block or N half) fails the float64 oracle's bound."""
    import oracle
    a, a_sf, w, w_sf, sa, sw = _ue8m0_case(m, g, k, n_out, seed=m * 7 + k)
    dev = torch.device("cuda:0")
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    y = rq.grouped_fp8_gemm_ue8m0(a.to(dev), a_sf.to(dev), w.to(dev), w_sf.to(dev),
                                  error_flags=flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    want = oracle.grouped_fp8_gemm_ue8m0(a.numpy(), a_sf.numpy().view(np.uint32), w.numpy(),
                                         w_sf.numpy())
    bound = _gemm_bound(a, sa.numpy(), w, sw.numpy(), want)
    err = np.abs(y.double().cpu().numpy() - want)
    assert np.all(err <= bound), f"{np.count_nonzero(err > bound)} outputs beyond the bound"


@pytest.mark.parametrize("m,g,k,n_out", [(1, 4, 4096, 1024), (2, 1, 1024, 128), (7, 3, 2048, 384),
                                         (16, 2, 4096, 256), (33, 1, 3072, 640), (64, 4, 4096, 1024),
                                         (1, 2, 512, 128), (9, 1, 1536, 256), (64, 3, 2560, 384)])
def test_gemm_ue8m0_decode_sizes(rq, m, g, k, n_out):
    """Up to 64 tokens the block-scaled GEMM runs split over K on clusters of
    CTAs (8 ways when K is a multiple of 1024, else 4) with the operands
    swapped; every output against the float64 oracle's bound, including K
    runs that cross scale words and token counts that are not multiples of
    16."""
    import oracle
    a, a_sf, w, w_sf, sa, sw = _ue8m0_case(m, g, k, n_out, seed=1000 + m * 7 + k)
    dev = torch.device("cuda:0")
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    y = rq.grouped_fp8_gemm_ue8m0(a.to(dev), a_sf.to(dev), w.to(dev), w_sf.to(dev),
                                  error_flags=flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    want = oracle.grouped_fp8_gemm_ue8m0(a.numpy(), a_sf.numpy().view(np.uint32), w.numpy(),
                                         w_sf.numpy())
    bound = _gemm_bound(a, sa.numpy(), w, sw.numpy(), want)
    err = np.abs(y.double().cpu().numpy() - want)
    assert np.all(err <= bound), f"{np.count_nonzero(err > bound)} outputs beyond the bound"


def test_gemm_ue8m0_decode_reads_what_the_op_just_wrote(rq):
    """Decode steps: the op (UE8M0 mode) rewrites the same activation buffers
    and the GEMM, launched with programmatic dependent launch right behind
    it, consumes them; five rounds with different inputs, each against the
    oracle (a read of the activations before the dependency wait would show
    the previous round's values)."""
    import oracle
    dev = torch.device("cuda:0")
    gen = torch.Generator().manual_seed(21)
    w = _rand_codes((4, 1024, 4096), gen)
    w_sf = torch.randint(120, 126, (4, 8, 32), generator=gen, dtype=torch.int32).to(torch.uint8)
    wd, wsd = w.to(dev), w_sf.to(dev)
    codes = torch.empty((8, 4, 4096), dtype=torch.uint8, device=dev)
    words = torch.empty((8, 4, 8), dtype=torch.int32, device=dev)
    y = torch.empty((8, 4, 1024), dtype=torch.bfloat16, device=dev)
    sw = np.ldexp(1.0, w_sf.numpy().astype(np.int64) - 127).astype(np.float32)
    ins = [W.inverse_inputs(W.InverseSpec("dec", 8, 32, 8, 4096, "uniform", True, seed=40 + r))
           for r in range(5)]
    got = []
    for inp in ins:
        rq.inv_rope_quant(inp["x"].to(dev), inp["positions"].to(dev), inp["cos_sin_cache"].to(dev),
                          8, mode="ue8m0", out=codes, scales=words)
        rq.grouped_fp8_gemm_ue8m0(codes, words, wd, wsd, out=y)
        got.append(y.clone())
    torch.cuda.synchronize()
    for inp, yr in zip(ins, got):
        wc, ws = oracle_inverse(inp)
        want = oracle.grouped_fp8_gemm(wc, ws, w.numpy(), sw)
        bound = _gemm_bound(torch.from_numpy(wc), ws, w, sw, want)
        err = np.abs(yr.double().cpu().numpy() - want)
        assert np.all(err <= bound), f"{np.count_nonzero(err > bound)} outputs beyond the bound"


def test_two_streams_at_once_match_one_stream(rq):
    """Two independent op + GEMM chains (a decode-size one on the split-K
    cluster kernel with programmatic dependent launch, and a 512-token one on
    the tile kernel) enqueued alternately on two streams, so their kernels
    run at the same time, give the bytes of the same calls run one after the
    other on one stream."""
    dev = torch.device("cuda:0")
    gen = torch.Generator().manual_seed(31)
    w = _rand_codes((4, 1024, 4096), gen).to(dev)
    w_sf = torch.randint(120, 126, (4, 8, 32), generator=gen, dtype=torch.int32).to(torch.uint8).to(dev)
    chains = []
    for n in (8, 512):
        inp = W.inverse_inputs(W.InverseSpec("conc", n, 32, 8, 4096, "uniform", True, seed=n))
        x, pos, cache = inp["x"].to(dev), inp["positions"].to(dev), inp["cos_sin_cache"].to(dev)
        codes = torch.empty((n, 4, 4096), dtype=torch.uint8, device=dev)
        words = torch.empty((n, 4, 8), dtype=torch.int32, device=dev)
        y = torch.empty((n, 4, 1024), dtype=torch.bfloat16, device=dev)

        def step(x=x, pos=pos, cache=cache, codes=codes, words=words, y=y):
            rq.inv_rope_quant(x, pos, cache, 8, mode="ue8m0", out=codes, scales=words)
            rq.grouped_fp8_gemm_ue8m0(codes, words, w, w_sf, out=y)
        chains.append((step, codes, words, y))
    for step, *_ in chains:
        step()
    torch.cuda.synchronize()
    want = [tuple(t.clone() for t in c[1:]) for c in chains]
    for t in (c[3] for c in chains):
        t.zero_()
    streams = [torch.cuda.Stream(dev) for _ in chains]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for _ in range(20):
        for (step, *_), s in zip(chains, streams):
            with torch.cuda.stream(s):
                step()
    torch.cuda.synchronize()
    for c, wv in zip(chains, want):
        for got, exp in zip(c[1:], wv):
            assert torch.equal(got, exp)


def test_gemm_ue8m0_consumes_the_op_ue8m0_output(rq):
    """The op's UE8M0 mode (packed words, token-major) feeds the block-scaled
    GEMM directly; the result matches the fp32-scale GEMM on the op's fp32
    scales within the same bound (both are the same powers of two)."""
    import oracle
    inp = W.inverse_inputs(W.InverseSpec("gemm", 300, 16, 8, 4096, "uniform", True, seed=6))
    dev = torch.device("cuda:0")
    x, pos, cache = inp["x"].to(dev), inp["positions"].to(dev), inp["cos_sin_cache"].to(dev)
    codes, words = rq.inv_rope_quant(x, pos, cache, 8, mode="ue8m0")
    gen = torch.Generator().manual_seed(7)
    w = _rand_codes((2, 384, 4096), gen)
    w_sf = torch.randint(120, 126, (2, 3, 32), generator=gen, dtype=torch.int32).to(torch.uint8)
    y = rq.grouped_fp8_gemm_ue8m0(codes, words, w.to(dev), w_sf.to(dev))
    torch.cuda.synchronize()
    wc, ws = oracle_inverse(inp)
    sw = np.ldexp(1.0, w_sf.numpy().astype(np.int64) - 127).astype(np.float32)
    want = oracle.grouped_fp8_gemm(wc, ws, w.numpy(), sw)
    bound = _gemm_bound(torch.from_numpy(wc), ws, w, sw, want)
    err = np.abs(y.double().cpu().numpy() - want)
    assert np.all(err <= bound), f"{np.count_nonzero(err > bound)} outputs beyond the bound"


def test_gemm_ue8m0_full_size_sampled_rows(rq):
    """prefill16k's op output (16384 tokens, 4 groups, K = 4096) through the
    block-scaled GEMM with 1024 outputs per group, in the bench's launch
    configuration; 64 sampled rows against the float64 oracle."""
    import oracle
    inp = W.inverse_inputs(W.PREFILL16K)
    dev = torch.device("cuda:0")
    x, pos, cache = inp["x"].to(dev), inp["positions"].to(dev), inp["cos_sin_cache"].to(dev)
    codes, words = rq.inv_rope_quant(x, pos, cache, 8, mode="ue8m0")
    gen = torch.Generator().manual_seed(11)
    w = _rand_codes((4, 1024, 4096), gen)
    w_sf = torch.randint(118, 124, (4, 8, 32), generator=gen, dtype=torch.int32).to(torch.uint8)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    y = rq.grouped_fp8_gemm_ue8m0(codes, words, w.to(dev), w_sf.to(dev), error_flags=flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    rows = torch.randperm(16384, generator=gen)[:64].sort().values
    rows[-1] = 16383
    a = codes[rows].cpu()
    sf = words[rows].cpu().numpy().view(np.uint32)
    want = oracle.grouped_fp8_gemm_ue8m0(a.numpy(), sf, w.numpy(), w_sf.numpy())
    shifts = np.array([0, 8, 16, 24], np.uint32)
    sa = np.ldexp(1.0, ((sf[..., None] >> shifts) & 0xFF).reshape(64, 4, 32).astype(np.int64)
                  - 127).astype(np.float32)
    sw = np.ldexp(1.0, w_sf.numpy().astype(np.int64) - 127).astype(np.float32)
    bound = _gemm_bound(a, sa, w, sw, want)
    err = np.abs(y[rows].double().cpu().numpy() - want)
    assert np.all(err <= bound), f"{np.count_nonzero(err > bound)} outputs beyond the bound"


# ---------------------------------------------------------------- host-buffer pipeline

@pytest.mark.parametrize("n,h,hpg,chunk", [(5, 8, 8, 1024), (1000, 32, 8, 256), (2049, 32, 8, 1024),
                                           (5000, 24, 6, 512), (700, 16, 16, 1)])
def test_host_pipeline_equals_device_call(rq, n, h, hpg, chunk):
    """Chunks pass through three workspace slots (every slot reused, a ragged
    last chunk); the host outputs equal the device call's bytes, which the
    other tests pin to the oracle."""
    inp = W.inverse_inputs(W.InverseSpec("host", n, h, hpg, 4096, "uniform", True, seed=n))
    dev = torch.device("cuda:0")
    cache = inp["cos_sin_cache"].to(dev)
    x_h, pos_h = inp["x"].pin_memory(), inp["positions"].pin_memory()
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    out_h, sc_h = rq.inv_rope_fp8_quant_host(x_h, pos_h, cache, hpg, chunk_tokens=chunk,
                                             error_flags=flags)
    codes, scales = rq.inv_rope_fp8_quant(x_h.to(dev), pos_h.to(dev), cache, hpg)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    assert out_h.dtype == codes.dtype
    assert torch.equal(out_h.view(torch.uint8), codes.cpu().view(torch.uint8))
    assert torch.equal(sc_h, scales.cpu())


def test_host_pipeline_is_stream_ordered_and_flags_bad_positions(rq):
    """Work enqueued before the call is seen by its copies (the cache is
    written on the stream just before), work after it sees its outputs, and a
    bad position is flagged as in the device call (its host outputs are
    unspecified: the chunk's device slot, stale there, is copied back whole)."""
    inp = W.inverse_inputs(W.InverseSpec("host", 600, 8, 8, 4096, "uniform", True, seed=3))
    dev = torch.device("cuda:0")
    cache = torch.zeros_like(inp["cos_sin_cache"]).to(dev)
    pos = inp["positions"].clone()
    pos[123] = 4096
    x_h, pos_h = inp["x"].pin_memory(), pos.pin_memory()
    out_h = torch.empty((600, 1, 4096), dtype=torch.uint8).pin_memory()
    sc_h = torch.empty((600, 1, 32)).pin_memory()
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    cache.copy_(inp["cos_sin_cache"], non_blocking=True)
    rq.inv_rope_fp8_quant_host(x_h, pos_h, cache, 8, out=out_h, scales=sc_h, chunk_tokens=64,
                               error_flags=flags)
    after = flags.clone()
    torch.cuda.current_stream().synchronize()
    assert int(after.item()) == 1
    keep = torch.tensor([i for i in range(600) if i != 123])
    sub = dict(inp, x=inp["x"][keep], positions=inp["positions"][keep])
    wc, ws = oracle_inverse(sub)
    assert np.array_equal(out_h[keep].numpy(), wc) and np.array_equal(sc_h[keep].numpy(), ws)


# ---------------------------------------------------------------- bounded waits run out

RQ_FLAG_TIMEOUT = 4


def _injected(rq, mask, call):
    """Run `call` with the test-only fault injection on (short waits), always
    switching it off again; returns after the device has finished."""
    rq.debug_inject(mask, 1 << 12)
    try:
        call()
        torch.cuda.synchronize()
    finally:
        rq.debug_inject()


def test_stream_kernel_wait_runs_out_reports_timeout_and_context_stays_usable(rq):
    """Warp 0 of the TMA-ring kernel leaves its first stage unarmed: its wait
    gives up, RQ_FLAG_TIMEOUT is set, the kernel exits; the next normal call on
    the same context is exact."""
    inp = W.inverse_inputs(W.InverseSpec("to", 2048, 32, 8, 4096, "uniform", True, seed=2))
    dev = torch.device("cuda:0")
    x, pos, cache = inp["x"].to(dev), inp["positions"].to(dev), inp["cos_sin_cache"].to(dev)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    _injected(rq, rq.DEBUG_STREAM_STAGE,
              lambda: rq.inv_rope_fp8_quant(x, pos, cache, 8, error_flags=flags,
                                            variant=rq.VARIANT_STREAM))
    assert int(flags.item()) & RQ_FLAG_TIMEOUT
    flags.zero_()
    codes, scales = rq.inv_rope_fp8_quant(x, pos, cache, 8, error_flags=flags,
                                          variant=rq.VARIANT_STREAM)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    wc, ws = oracle_inverse(inp)
    assert np.array_equal(codes.view(torch.uint8).cpu().numpy(), wc)
    assert np.array_equal(scales.cpu().numpy(), ws)


@pytest.mark.parametrize("kind", ["fp32", "ue8m0", "ue8m0_decode", "fp32_decode"])
def test_gemm_wait_runs_out_reports_timeout_and_context_stays_usable(rq, kind):
    """The first CTA's TMA producer issues nothing: its MMA waits give up,
    RQ_FLAG_TIMEOUT is set, TMEM is freed and the kernel exits (on the
    decode-size kernel, after both cluster barriers); the next normal call is
    within the oracle's bound."""
    import oracle
    dev = torch.device("cuda:0")
    m, g, k, n_out = (16 if kind.endswith("_decode") else 300), 2, 1024, 256
    a, a_sf, w, w_sf, sa, sw = _ue8m0_case(m, g, k, n_out, seed=9)
    ad, wd = a.to(dev), w.to(dev)
    if kind.startswith("fp32"):
        sad, swd = sa.to(dev), sw.to(dev)
        call = lambda fl: rq.grouped_fp8_gemm(ad, sad, wd, swd, error_flags=fl)
        want = oracle.grouped_fp8_gemm(a.numpy(), sa.numpy(), w.numpy(), sw.numpy())
    else:
        asd, wsd = a_sf.to(dev), w_sf.to(dev)
        call = lambda fl: rq.grouped_fp8_gemm_ue8m0(ad, asd, wd, wsd, error_flags=fl)
        want = oracle.grouped_fp8_gemm_ue8m0(a.numpy(), a_sf.numpy().view(np.uint32), w.numpy(),
                                             w_sf.numpy())
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    _injected(rq, rq.DEBUG_GEMM_LOADS, lambda: call(flags))
    assert int(flags.item()) & RQ_FLAG_TIMEOUT
    flags.zero_()
    y = call(flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    bound = _gemm_bound(a, sa.numpy(), w, sw.numpy(), want)
    assert np.all(np.abs(y.double().cpu().numpy() - want) <= bound)


def test_gemm_fp32_scales_full_size_sampled_rows(rq):
    """The fp32-scale consumer GEMM in the bench's configuration (prefill16k's
    op output, 4 groups, K = 4096, 1024 outputs per group); 64 sampled rows
    against the float64 oracle."""
    import oracle
    inp = W.inverse_inputs(W.PREFILL16K)
    dev = torch.device("cuda:0")
    x, pos, cache = inp["x"].to(dev), inp["positions"].to(dev), inp["cos_sin_cache"].to(dev)
    codes, scales = rq.inv_rope_fp8_quant(x, pos, cache, 8)
    gen = torch.Generator().manual_seed(12)
    w = _rand_codes((4, 1024, 4096), gen)
    sw = 2.0 ** torch.randint(-10, -6, (4, 8, 32), generator=gen).float()
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    y = rq.grouped_fp8_gemm(codes, scales, w.to(dev), sw.to(dev), error_flags=flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    rows = torch.randperm(16384, generator=gen)[:64].sort().values
    rows[0] = 0
    a = codes[rows].view(torch.uint8).cpu()
    sa = scales[rows].cpu().numpy()
    want = oracle.grouped_fp8_gemm(a.numpy(), sa, w.numpy(), sw.numpy())
    bound = _gemm_bound(a, sa, w, sw.numpy(), want)
    assert np.all(np.abs(y[rows].double().cpu().numpy() - want) <= bound)


def test_host_pipeline_full_size_in_the_bench_configuration(rq):
    """prefill16k through the host-buffer call with 512-token chunks (the
    bench's e2e leg): the same bytes as the device call."""
    inp = W.inverse_inputs(W.PREFILL16K)
    dev = torch.device("cuda:0")
    cache = inp["cos_sin_cache"].to(dev)
    x_h, pos_h = inp["x"].pin_memory(), inp["positions"].pin_memory()
    out_h, sc_h = rq.inv_rope_fp8_quant_host(x_h, pos_h, cache, 8, chunk_tokens=512)
    codes, scales = rq.inv_rope_fp8_quant(x_h.to(dev), pos_h.to(dev), cache, 8)
    torch.cuda.synchronize()
    assert torch.equal(out_h.view(torch.uint8), codes.cpu().view(torch.uint8))
    assert torch.equal(sc_h, scales.cpu())


# ---------------------------------------------------------------- every input value

@pytest.mark.parametrize("order", ["sorted", "shuffled"])
def test_every_finite_bf16_input_value(rq, order):
    """All 65,280 finite bf16 patterns (both zeros, subnormals, up to 3.39e38)
    through the kernel's quantisation at position 0, where the rotation is
    the identity (cos 1, sin 0: no overflow), bit-exact against the oracle.
    Sorted by magnitude, neighbouring values share a block, so every scale
    exponent from the eps floor to 2^120 occurs; shuffled, blocks mix tiny and
    huge values."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    finite = bits[((bits >> 7) & 0xFF) != 0xFF].astype(np.uint16)
    if order == "sorted":
        mag = finite.view(np.int16).astype(np.int32) & 0x7FFF
        finite = finite[np.argsort(mag, kind="stable")]
    else:
        finite = finite[np.random.default_rng(5).permutation(finite.size)]
    rows = -(-finite.size // 512)
    flat = np.zeros(rows * 512, np.uint16)
    flat[:finite.size] = finite
    heads = 8
    toks = -(-rows // heads)
    buf = np.zeros(toks * heads * 512, np.uint16)
    buf[:flat.size] = flat
    x = torch.from_numpy(buf.view(np.int16)).view(torch.bfloat16).reshape(toks, heads, 512)
    inp = {"x": x, "positions": torch.zeros(toks, dtype=torch.int64),
           "cos_sin_cache": W.rope_cache(16), "heads_per_group": heads}
    gc, gs = run_inverse(rq, inp, variant=rq.VARIANT_WARP_ROWS)
    wc, ws = oracle_inverse(inp)
    assert np.array_equal(gc, wc)
    assert np.array_equal(gs.view(np.uint32), ws.view(np.uint32))


# ---------------------------------------------------------------- index validation helper

def _expected_flags(pos, slots, cache_rows, num_slots):
    """Plain Python statement of the preconditions (1 position, 2 slot range, 8 reuse)."""
    f = 0
    if any(p < 0 or p >= cache_rows for p in pos):
        f |= 1
    if slots is not None:
        live = [s for s in slots if s >= 0]
        if any(s >= num_slots for s in live):
            f |= 2
        inside = [s for s in live if s < num_slots]
        if len(set(inside)) != len(inside):
            f |= 8
    return f


def test_validate_indices_planted_errors(rq):
    dev = torch.device("cuda:0")
    base_pos = [0, 5, 63, 17, 9, 40]
    base_slots = [3, 7, -1, 100, 0, 55]
    cases = [
        (base_pos, base_slots, 0),
        ([0, 5, 64, 17, 9, 40], base_slots, 1),          # position == cache_rows
        ([0, -1, 63, 17, 9, 40], base_slots, 1),
        (base_pos, [3, 7, -1, 128, 0, 55], 2),            # slot == num_slots
        (base_pos, [3, 7, -1, 100, 3, 55], 8),            # slot 3 used twice
        (base_pos, [-5, -1, -1, -1, -7, -2], 0),          # every token skipped
        ([70, 5, 63, 17, 9, 40], [3, 3, -1, 999, 0, 55], 11),
    ]
    for pos, slots, want in cases:
        got = rq.validate_indices(torch.tensor(pos, device=dev), 64,
                                  torch.tensor(slots, device=dev), 128)
        assert got == want == _expected_flags(pos, slots, 64, 128), (pos, slots, got)
    # positions only: slots are not looked at
    assert rq.validate_indices(torch.tensor([1, 2, 64], device=dev), 64) == 1


def test_validate_indices_at_the_insert_workload(rq):
    """insert16k's positions and distinct slots are valid; duplicates and a
    range error planted at random tokens are all found."""
    ins = W.insert_inputs(W.INSERT16K)
    dev = torch.device("cuda:0")
    pos, slots = ins["positions"], ins["slot_mapping"]
    n_slots = W.INSERT16K.num_blocks * W.INSERT16K.block_size
    ws = torch.empty(rq.lib().rq_validate_indices_workspace(n_slots), dtype=torch.uint8, device=dev)
    assert rq.validate_indices(pos.to(dev), 65536, slots.to(dev), n_slots, workspace=ws) == 0
    gen = torch.Generator().manual_seed(4)
    bad = slots.clone()
    i, j = torch.randperm(16384, generator=gen)[:2].tolist()
    bad[j] = bad[i]                                    # a repeated slot
    got = rq.validate_indices(pos.to(dev), 65536, bad.to(dev), n_slots, workspace=ws)
    assert got == 8 == _expected_flags(pos.tolist(), bad.tolist(), 65536, n_slots)
    bad[i] = n_slots + 5                               # now out of range instead
    got = rq.validate_indices(pos.to(dev), 65536, bad.to(dev), n_slots, workspace=ws)
    assert got == _expected_flags(pos.tolist(), bad.tolist(), 65536, n_slots) == 2


# ---------------------------------------------------------------- random shapes

def _random_shape_cases(k, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(k):
        h = int(rng.choice([1, 2, 3, 5, 8, 12, 16, 24, 40, 64, 96, 128]))
        divisors = [d for d in range(1, h + 1) if h % d == 0]
        hpg = int(rng.choice(divisors))
        n = int(rng.integers(1, 700))
        pad_h = int(rng.choice([0, 8, 64]))        # padding between heads, in elements
        pad_t = int(rng.choice([0, 8, 512]))       # padding between tokens
        cases.append((i, n, h, hpg, pad_h, pad_t))
    return cases


@pytest.mark.parametrize("case", _random_shape_cases(16, 2024), ids=lambda c: f"r{c[0]}")
def test_random_shapes_and_strides_bit_exact(rq, case):
    """Seeded random token counts, head counts, every divisor as heads_per_group,
    padded head / token strides, both kernels: codes and scales bit-exact, and
    the layout entry's UE8M0 and bf16 outputs too."""
    i, n, h, hpg, pad_h, pad_t = case
    inp = W.inverse_inputs(W.InverseSpec(f"rand{i}", n, h, hpg, 8192, "uniform", True, seed=i))
    sh = 512 + pad_h
    st = h * sh + pad_t
    big = torch.zeros(n * st + 512, dtype=torch.bfloat16)
    view = big.as_strided((n, h, 512), (st, sh, 1))
    view.copy_(inp["x"])
    dev = torch.device("cuda:0")
    xd = big.to(dev).as_strided((n, h, 512), (st, sh, 1))
    wc, ws = oracle_inverse(inp)
    for variant in (rq.VARIANT_WARP_ROWS, rq.VARIANT_STREAM):
        gc, gs = run_inverse(rq, inp, x_override=xd, variant=variant)
        assert np.array_equal(gc, wc), (case, variant)
        assert np.array_equal(gs.view(np.uint32), ws.view(np.uint32)), (case, variant)
    for mode in ("ue8m0", "bf16"):
        got = run_layout(rq, dict(inp, x=xd), mode, "token")
        assert_layout_parity(mode, got, oracle_layout(inp, mode))
    # contiguous group-major outputs (the warp-rows kernel's group-major rows
    # when there is more than one group)
    for mode in ("fp8", "ue8m0"):
        got = run_layout(rq, dict(inp, x=xd), mode, "group_major")
        assert_layout_parity(mode, got, oracle_layout(inp, mode))
