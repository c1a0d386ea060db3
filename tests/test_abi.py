"""The C-ABI library loads, exports every symbol include/rq.h declares, and
rejects invalid arguments on the host before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

import rope_block_fp8_inverse_b300 as rq
from rope_block_fp8_inverse_b300 import build as rq_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rq.h")

RQ_OK, RQ_ERR_NULL, RQ_ERR_SHAPE, RQ_ERR_ALIGN, RQ_ERR_GROUPING, RQ_ERR_CUDA, RQ_ERR_ARG = range(7)


@pytest.fixture(scope="module")
def lib():
    rq_build.build()
    return rq.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = _declared_functions()
    assert "rq_inv_rope_fp8_quant" in names and "rq_rope_fp8_quant_insert" in names
    assert set(names) == set(rq.ABI_SYMBOLS), (names, sorted(rq.ABI_SYMBOLS))


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(rq.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(raw, name), name


def test_version_and_status_strings(lib):
    assert lib.rq_version() >> 16 == 1
    for code in range(7):
        s = rq.status_string(code)
        assert s and s != "unknown status"
    assert rq.status_string(99) == "unknown status"


# fake, never-dereferenced device addresses: every call below fails host checks first
A16 = 0x7F0000000000
A8 = A16 + 8


def _inv(lib, x=A16, n=4, h=8, st=4096, sh=512, pos=A16, cs=A16, rows=16, hpg=4, eps=1e-10,
         out=A16, sc=A16, flags=None):
    return lib.rq_inv_rope_fp8_quant(x, n, h, st, sh, pos, cs, rows, hpg, eps, out, sc, flags, None)


@pytest.mark.parametrize("kw,status", [
    (dict(n=-1), RQ_ERR_SHAPE),
    (dict(h=0), RQ_ERR_SHAPE),
    (dict(rows=0), RQ_ERR_SHAPE),
    (dict(hpg=0), RQ_ERR_GROUPING),
    (dict(hpg=3), RQ_ERR_GROUPING),
    (dict(h=24, hpg=5), RQ_ERR_GROUPING),
    (dict(eps=0.0), RQ_ERR_ARG),
    (dict(eps=-1.0), RQ_ERR_ARG),
    (dict(eps=float("nan")), RQ_ERR_ARG),
    (dict(eps=float("inf")), RQ_ERR_ARG),
    (dict(eps=1e-35), RQ_ERR_ARG),
    (dict(n=1 << 27, h=16, hpg=4), RQ_ERR_SHAPE),     # N*H >= 2^31
    (dict(x=None), RQ_ERR_NULL),
    (dict(pos=None), RQ_ERR_NULL),
    (dict(cs=None), RQ_ERR_NULL),
    (dict(out=None), RQ_ERR_NULL),
    (dict(sc=None), RQ_ERR_NULL),
    (dict(x=A8), RQ_ERR_ALIGN),
    (dict(st=4100), RQ_ERR_ALIGN),
    (dict(sh=516), RQ_ERR_ALIGN),
    (dict(pos=A16 + 4), RQ_ERR_ALIGN),
    (dict(cs=A8), RQ_ERR_ALIGN),
    (dict(out=A8), RQ_ERR_ALIGN),
    (dict(sc=A8), RQ_ERR_ALIGN),
    (dict(flags=A16 + 2), RQ_ERR_ALIGN),
])
def test_inverse_rejects_bad_arguments(lib, kw, status):
    assert _inv(lib, **kw) == status


def test_inverse_rejects_unknown_variant(lib):
    args = (A16, 4, 8, 4096, 512, A16, A16, 16, 4, 1e-10, A16, A16, None, None)
    assert lib.rq_inv_rope_fp8_quant_ex(*args, 3) == RQ_ERR_ARG
    assert lib.rq_inv_rope_fp8_quant_ex(*args, -1) == RQ_ERR_ARG
    bad = (None,) + args[1:]
    for v in (0, 1, 2):   # known variants reach the pointer checks
        assert lib.rq_inv_rope_fp8_quant_ex(*bad, v) == RQ_ERR_NULL


def test_inverse_empty_batch_is_a_no_op(lib):
    # n_tokens == 0: OK with no launch, even with NULL buffers
    assert _inv(lib, n=0, x=None, pos=None, cs=None, out=None, sc=None) == RQ_OK


def _ins(lib, kv=A16, n=4, skv=512, pos=A16, cs=A16, rows=16, slots=A16, cache=A16, nb=8, bs=64,
         stride=64 * 528, eps=1e-10, flags=None):
    return lib.rq_rope_fp8_quant_insert(kv, n, skv, pos, cs, rows, slots, cache, nb, bs, stride,
                                        eps, flags, None)


@pytest.mark.parametrize("kw,status", [
    (dict(n=-1), RQ_ERR_SHAPE),
    (dict(rows=0), RQ_ERR_SHAPE),
    (dict(nb=0), RQ_ERR_SHAPE),
    (dict(bs=0), RQ_ERR_SHAPE),
    (dict(stride=64 * 528 - 16), RQ_ERR_SHAPE),
    (dict(stride=64 * 528 + 8), RQ_ERR_ALIGN),
    (dict(eps=0.0), RQ_ERR_ARG),
    (dict(kv=None), RQ_ERR_NULL),
    (dict(slots=None), RQ_ERR_NULL),
    (dict(cache=None), RQ_ERR_NULL),
    (dict(kv=A8), RQ_ERR_ALIGN),
    (dict(skv=516), RQ_ERR_ALIGN),
    (dict(slots=A16 + 4), RQ_ERR_ALIGN),
    (dict(cache=A8), RQ_ERR_ALIGN),
])
def test_insert_rejects_bad_arguments(lib, kw, status):
    assert _ins(lib, **kw) == status


def test_insert_empty_batch_is_a_no_op(lib):
    assert _ins(lib, n=0, kv=None, pos=None, cs=None, slots=None, cache=None) == RQ_OK


def test_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(2, 8, 512, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        rq.inv_rope_fp8_quant(x, torch.zeros(2, dtype=torch.int64), torch.zeros(4, 64), 8)


def _lay(lib, mode=0, out=A16, ot=4 * 4096, og=4096, sc=A16, st=128, sg=32, se=1, n=4, h=8,
         hpg=4, x=A16, flags=None):
    return lib.rq_inv_rope_quant_layout(x, n, h, 4096, 512, A16, A16, 16, hpg, 1e-10, mode, out,
                                        ot, og, sc, st, sg, se, flags, None)


@pytest.mark.parametrize("kw,status", [
    (dict(mode=3), RQ_ERR_ARG),
    (dict(mode=-1), RQ_ERR_ARG),
    (dict(hpg=3), RQ_ERR_GROUPING),
    (dict(ot=-16), RQ_ERR_SHAPE),
    (dict(se=-1), RQ_ERR_SHAPE),
    (dict(out=None), RQ_ERR_NULL),
    (dict(sc=None), RQ_ERR_NULL),                 # fp32 scales are required
    (dict(mode=1, sc=None), RQ_ERR_NULL),         # so are UE8M0 words
    (dict(out=A8), RQ_ERR_ALIGN),
    (dict(ot=4 * 4096 + 8), RQ_ERR_ALIGN),
    (dict(og=4104), RQ_ERR_ALIGN),
    (dict(sc=A16 + 2), RQ_ERR_ALIGN),
])
def test_layout_rejects_bad_arguments(lib, kw, status):
    assert _lay(lib, **kw) == status


def test_layout_bf16_needs_no_scales_and_empty_is_a_no_op(lib):
    # bf16 mode ignores scales: with scales NULL it reaches the pointer checks of x
    assert _lay(lib, mode=2, sc=None, x=None) == RQ_ERR_NULL
    assert _lay(lib, n=0, out=None, sc=None, x=None) == RQ_OK


def _fus(lib, q=A16, n=4, hq=8, sqt=4096, sqh=512, kv=A16, skv=512, qo=A16, hpad=8, pos=A16,
         cs=A16, rows=16, slots=A16, cache=A16, nb=8, bs=64, stride=64 * 528, ne=1e-6, qe=1e-10,
         w=None):
    return lib.rq_qnorm_rope_kv_rope_quant_insert(q, n, hq, sqt, sqh, kv, skv, qo, hpad, pos, cs,
                                                  rows, slots, cache, nb, bs, stride, ne, w, qe,
                                                  None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(hpad=7), RQ_ERR_SHAPE),
    (dict(hq=0), RQ_ERR_SHAPE),
    (dict(stride=64 * 528 - 16), RQ_ERR_SHAPE),
    (dict(ne=-1.0), RQ_ERR_ARG),
    (dict(ne=float("inf")), RQ_ERR_ARG),
    (dict(qe=0.0), RQ_ERR_ARG),
    (dict(qo=None), RQ_ERR_NULL),
    (dict(kv=None), RQ_ERR_NULL),
    (dict(qo=A8), RQ_ERR_ALIGN),
    (dict(sqh=516), RQ_ERR_ALIGN),
    (dict(stride=64 * 528 + 8), RQ_ERR_ALIGN),
    (dict(w=A8), RQ_ERR_ALIGN),          # the norm weight is read in 16-byte chunks
])
def test_fused_rejects_bad_arguments(lib, kw, status):
    assert _fus(lib, **kw) == status


def test_fused_empty_batch_is_a_no_op(lib):
    assert _fus(lib, n=0, q=None, kv=None, qo=None, pos=None, cs=None, slots=None,
                cache=None) == RQ_OK


def _idx(lib, q=A16, n=4, h=8, sqt=1024, sqh=128, style=0, w=A16, ss=0.1, hs=0.2, eps=1e-4,
         out=A16, wo=A16):
    return lib.rq_indexer_q_rope_fp8_quant(q, n, h, sqt, sqh, A16, A16, 16, style, w, ss, hs,
                                           eps, out, wo, None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(style=2), RQ_ERR_ARG),
    (dict(eps=0.0), RQ_ERR_ARG),
    (dict(ss=float("nan")), RQ_ERR_ARG),
    (dict(h=0), RQ_ERR_SHAPE),
    (dict(w=None), RQ_ERR_NULL),
    (dict(wo=None), RQ_ERR_NULL),
    (dict(out=A8), RQ_ERR_ALIGN),
    (dict(sqh=132), RQ_ERR_ALIGN),
])
def test_indexer_rejects_bad_arguments(lib, kw, status):
    assert _idx(lib, **kw) == status


def _gemm(lib, a=A16, sa=A16, n=4, g=2, k=512, w=A16, sw=A16, no=256, y=A16):
    return lib.rq_grouped_fp8_gemm(a, sa, n, g, k, w, sw, no, y, None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(k=500), RQ_ERR_SHAPE),
    (dict(no=200), RQ_ERR_SHAPE),
    (dict(g=0), RQ_ERR_SHAPE),
    (dict(n=-1), RQ_ERR_SHAPE),
    (dict(w=None), RQ_ERR_NULL),
    (dict(y=A8), RQ_ERR_ALIGN),
    (dict(a=A8), RQ_ERR_ALIGN),
])
def test_gemm_rejects_bad_arguments(lib, kw, status):
    assert _gemm(lib, **kw) == status


def test_gemm_empty_is_a_no_op(lib):
    assert _gemm(lib, n=0, a=None, sa=None, w=None, sw=None, y=None) == RQ_OK


def _gemm_mx(lib, a=A16, sa=A16, n=4, g=2, k=512, w=A16, sw=A16, no=256, y=A16):
    return lib.rq_grouped_fp8_gemm_ue8m0(a, sa, n, g, k, w, sw, no, y, None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(k=128), RQ_ERR_SHAPE),        # K must hold whole 512-wide heads (one scale word each)
    (dict(k=640), RQ_ERR_SHAPE),
    (dict(k=4608), RQ_ERR_SHAPE),       # at most 4096 (the scale codes' TMEM budget)
    (dict(no=200), RQ_ERR_SHAPE),
    (dict(g=0), RQ_ERR_SHAPE),
    (dict(n=-1), RQ_ERR_SHAPE),
    (dict(sa=None), RQ_ERR_NULL),
    (dict(sw=None), RQ_ERR_NULL),
    (dict(y=A8), RQ_ERR_ALIGN),
    (dict(a=A8), RQ_ERR_ALIGN),
    (dict(sa=A16 + 2), RQ_ERR_ALIGN),
])
def test_gemm_ue8m0_rejects_bad_arguments(lib, kw, status):
    assert _gemm_mx(lib, **kw) == status


def test_gemm_ue8m0_empty_is_a_no_op(lib):
    assert _gemm_mx(lib, n=0, a=None, sa=None, w=None, sw=None, y=None) == RQ_OK


def _host(lib, x=A16, n=4, h=8, pos=A16, cache=A16, rows=64, hpg=8, out=A16, sc=A16, ws=A16,
          wsb=1 << 40, chunk=2):
    return lib.rq_inv_rope_fp8_quant_host(x, n, h, pos, cache, rows, hpg, 1e-10, out, sc, ws, wsb,
                                          chunk, None, None)


def test_host_workspace_size_is_three_aligned_slots(lib):
    a = lambda b: (b + 255) // 256 * 256
    for h, ct in ((8, 1), (32, 1024), (24, 7)):
        slot = a(ct * h * 1024) + a(ct * 8) + a(ct * h * 512) + a(ct * h * 16)
        assert lib.rq_inv_rope_fp8_quant_host_workspace(h, ct) == 3 * slot
    assert lib.rq_inv_rope_fp8_quant_host_workspace(0, 4) == -1
    assert lib.rq_inv_rope_fp8_quant_host_workspace(8, 0) == -1


@pytest.mark.parametrize("kw,status", [
    (dict(chunk=0), RQ_ERR_SHAPE),
    (dict(n=-1), RQ_ERR_SHAPE),
    (dict(hpg=3), RQ_ERR_GROUPING),
    (dict(wsb=1000), RQ_ERR_SHAPE),     # smaller than the three slots
    (dict(x=None), RQ_ERR_NULL),
    (dict(ws=None), RQ_ERR_NULL),
    (dict(sc=None), RQ_ERR_NULL),
    (dict(ws=A16 + 16), RQ_ERR_ALIGN),
])
def test_host_rejects_bad_arguments(lib, kw, status):
    assert _host(lib, **kw) == status


def test_host_empty_batch_is_a_no_op(lib):
    assert _host(lib, n=0, x=None, pos=None, out=None, sc=None, ws=None) == RQ_OK


def test_validate_workspace_is_bitmap_plus_result_word(lib):
    for n in (0, 1, 31, 32, 33, 32768, 10 ** 6):
        bitmap = ((n + 31) // 32 * 4 + 15) // 16 * 16
        assert lib.rq_validate_indices_workspace(n) == bitmap + 16
    assert lib.rq_validate_indices_workspace(-1) == -1


def _val(lib, pos=A16, slots=A16, n=4, rows=64, nslots=128, ws=A16, wsb=1 << 20, res=True):
    out = ctypes.c_uint32(0xDEAD)
    st = lib.rq_validate_indices(pos, slots, n, rows, nslots, ws, wsb,
                                 ctypes.addressof(out) if res else None, None)
    return st, out.value


@pytest.mark.parametrize("kw,status", [
    (dict(n=-1), RQ_ERR_SHAPE),
    (dict(rows=0), RQ_ERR_SHAPE),
    (dict(nslots=0), RQ_ERR_SHAPE),          # slots given, but no cache slots
    (dict(res=False), RQ_ERR_NULL),
    (dict(pos=None), RQ_ERR_NULL),
    (dict(ws=None), RQ_ERR_NULL),
    (dict(wsb=16), RQ_ERR_SHAPE),            # smaller than the bitmap + result word
    (dict(pos=A16 + 4), RQ_ERR_ALIGN),
    (dict(ws=A16 + 8), RQ_ERR_ALIGN),
])
def test_validate_rejects_bad_arguments(lib, kw, status):
    assert _val(lib, **kw)[0] == status


def test_validate_empty_batch_reports_nothing(lib):
    assert _val(lib, n=0, pos=None, slots=None, ws=None) == (RQ_OK, 0)


def test_header_is_plain_c_and_links(tmp_path, lib):
    """include/rq.h compiles as C99 (no C++ in the ABI) and a C program linked
    against librq.so calls the entry points that need no GPU."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi_check.c"
    src.write_text(r"""
#include <stdio.h>
#include <string.h>
#include "rq.h"
int main(void) {
    uint32_t flags = 123;
    int64_t ws = rq_validate_indices_workspace(64);
    rq_status st = rq_validate_indices(NULL, NULL, 0, 16, 0, NULL, 0, &flags, NULL);
    printf("%d %s %lld %d %u\n", rq_version() >> 16, rq_status_string(RQ_ERR_ALIGN),
           (long long)ws, (int)st, flags);
    return rq_inv_rope_fp8_quant(NULL, -1, 1, 0, 0, NULL, NULL, 1, 1, 1e-10f, NULL, NULL, NULL,
                                 NULL) == RQ_ERR_SHAPE ? 0 : 1;
}
""")
    exe = tmp_path / "abi_check"
    libdir = os.path.dirname(rq.LIB_PATH)
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", inc, str(src), "-L", libdir,
                        "-lrq", f"-Wl,-rpath,{libdir}", "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    major, *rest = out.stdout.split()
    assert major == "1" and out.stdout.split()[-3:] == ["32", "0", "0"]
