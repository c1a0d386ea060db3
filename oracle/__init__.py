"""CPU oracle for the inverse-RoPE + block-FP8 quant epilogue (test infrastructure).

This package is the correctness reference the CUDA library is checked
against. Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline / reference leg may import it; the library itself never does.
It shares no code with the CUDA path: the arithmetic lives in ``rq_oracle.c``
(plain scalar C, fp32 as the pages fix it, compiled with FMA contraction off)
and this module only builds it and marshals numpy / torch-CPU arrays.

What it computes, and the page sections each step follows, is stated in the
header of ``rq_oracle.c``. Every function here has a pin in
``tests/test_oracle_*.py`` that checks it against something other than
itself (the OFP8 spec's value table, torch's float8 cast, exact ceil-log2
from float64 frexp, complex multiplication, hand-built worked cases).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rq_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread"]

HEAD_DIM = 512
BLOCKS_PER_HEAD = 4
RECORD_BYTES = 528

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile rq_oracle.c into oracle/_build/liboracle.so (gcc, no CUDA)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *_CFLAGS, _SRC, "-lm", "-o", tmp], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        sig = {
            "rqo_e4m3_encode": (ctypes.c_uint8, [ctypes.c_double]),
            "rqo_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "rqo_ceil_log2": (ctypes.c_int, [ctypes.c_float]),
            "rqo_block_scale": (ctypes.c_float, [ctypes.c_float]),
            "rqo_e4m3_encode_f32_array": (None, [P, i64, P]),
            "rqo_e4m3_decode_array": (None, [P, i64, P]),
            "rqo_ceil_log2_array": (None, [P, i64, P]),
            "rqo_block_scale_array": (None, [P, i64, P]),
            "rqo_block_scale_bits_range": (ctypes.c_int, [ctypes.c_uint32, i64, ctypes.c_float, P,
                                                          ctypes.c_int]),
            "rqo_e4m3_encode_bits_range": (ctypes.c_int, [ctypes.c_uint32, i64, ctypes.c_int, P,
                                                          ctypes.c_int]),
            "rqo_rope_rows": (ctypes.c_int, [P, i64, P, P, i64, ctypes.c_int]),
            "rqo_quant_rows": (None, [P, i64, ctypes.c_float, P, P]),
            "rqo_inv_rope_fp8_quant": (ctypes.c_int, [P, i64, i64, i64, i64, P, P, i64, i64,
                                                      ctypes.c_float, P, P, ctypes.c_int]),
            "rqo_rope_fp8_quant_insert": (ctypes.c_int, [P, i64, i64, P, P, i64, P, P, i64,
                                                         i64, i64, ctypes.c_float, ctypes.c_int]),
            "rqo_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
            "rqo_ue8m0_of_scale": (ctypes.c_uint8, [ctypes.c_float]),
            "rqo_f32_to_bf16_array": (None, [P, i64, P]),
            "rqo_pack_ue8m0_array": (None, [P, i64, P]),
            "rqo_inv_rope_bf16": (ctypes.c_int, [P, i64, i64, i64, i64, P, P, i64, i64, P]),
            "rqo_f64_to_bf16_array": (None, [P, i64, P]),
            "rqo_indexer_q_rope_quant": (ctypes.c_int, [P, i64, i64, i64, i64, P, P, i64,
                                                        ctypes.c_int, P, ctypes.c_float,
                                                        ctypes.c_float, ctypes.c_float, P, P]),
            "rqo_qnorm_rope_kv_rope_quant_insert": (ctypes.c_int, [P, i64, i64, i64, i64, P, i64, P,
                                                                   i64, P, i64, i64, i64, P, P, P,
                                                                   i64, ctypes.c_double, P,
                                                                   ctypes.c_float]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


class OracleError(RuntimeError):
    pass


def _np(a, dtype):
    """Contiguous numpy view/copy of a numpy array or CPU torch tensor."""
    if hasattr(a, "detach"):  # torch tensor
        import torch
        t = a.detach().cpu()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        a = t.numpy()
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        if a.dtype.itemsize == np.dtype(dtype).itemsize and dtype in (np.uint16, np.int16):
            a = a.view(dtype)
        else:
            a = a.astype(dtype)
    return a


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# ------------------------------------------------------------------ scalars

def e4m3_encode(v) -> np.ndarray:
    """OFP8 E4M3 codes of fp32 values (RNE, saturate at 448, NaN -> 0x7F)."""
    v = _np(v, np.float32)
    out = np.empty(v.shape, np.uint8)
    _load().rqo_e4m3_encode_f32_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_encode_scalar(v: float) -> int:
    """E4M3 code of one real value given as a Python float (double)."""
    return int(_load().rqo_e4m3_encode(float(v)))


def e4m3_decode(codes) -> np.ndarray:
    """Real value (float64) of each E4M3 code; NaN for 0x7F / 0xFF."""
    c = _np(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().rqo_e4m3_decode_array(_ptr(c), c.size, _ptr(out))
    return out


def ceil_log2(r) -> np.ndarray:
    """Exact ceil(log2(r)) of positive finite fp32 values."""
    r = _np(r, np.float32)
    out = np.empty(r.shape, np.int32)
    _load().rqo_ceil_log2_array(_ptr(r), r.size, _ptr(out))
    return out


def block_scale(amax) -> np.ndarray:
    """2^ceil(log2(fl32(amax / 448))) for clamped block amax values."""
    a = _np(amax, np.float32)
    out = np.empty(a.shape, np.float32)
    _load().rqo_block_scale_array(_ptr(a), a.size, _ptr(out))
    return out


def block_scale_bits_range(first_bits: int, count: int, eps: float, threads: int = 0) -> np.ndarray:
    """block_scale(max(amax, eps)) for every amax = fp32 bit pattern
    first_bits + i, i < count (first_bits + count <= 2^32), over ``threads``
    threads (0 = all cores). Same arithmetic as block_scale, element by element."""
    out = np.empty(int(count), np.float32)
    st = _load().rqo_block_scale_bits_range(int(first_bits), int(count), float(eps), _ptr(out),
                                            int(threads or os.cpu_count() or 1))
    if st:
        raise OracleError(f"rqo_block_scale_bits_range: status {st}")
    return out


def e4m3_encode_bits_range(first_bits: int, count: int, scale_exp: int = 0,
                           threads: int = 0) -> np.ndarray:
    """E4M3 code of (fp32 bit pattern first_bits + i) / 2^scale_exp for i < count,
    the quantisation step of the op; same arithmetic as e4m3_encode."""
    out = np.empty(int(count), np.uint8)
    st = _load().rqo_e4m3_encode_bits_range(int(first_bits), int(count), int(scale_exp), _ptr(out),
                                            int(threads or os.cpu_count() or 1))
    if st:
        raise OracleError(f"rqo_e4m3_encode_bits_range: status {st}")
    return out


def f32_to_bf16(v) -> np.ndarray:
    """bf16 bit patterns (uint16) of fp32 values, round to nearest, ties to even."""
    v = _np(v, np.float32)
    out = np.empty(v.shape, np.uint16)
    _load().rqo_f32_to_bf16_array(_ptr(v), v.size, _ptr(out))
    return out


def f64_to_bf16(v) -> np.ndarray:
    """bf16 bit patterns of float64 values, rounded once to nearest, ties to even."""
    v = _np(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().rqo_f64_to_bf16_array(_ptr(v), v.size, _ptr(out))
    return out


def pack_ue8m0(scales) -> np.ndarray:
    """Pack [..., 4] power-of-two fp32 block scales into one uint32 per head:
    byte b = UE8M0 code (exponent + 127) of block b's scale."""
    s = _np(scales, np.float32)
    if s.shape[-1] % BLOCKS_PER_HEAD:
        raise OracleError("the last dim must hold whole heads (4 scales each)")
    out = np.empty(s.shape[:-1] + (s.shape[-1] // BLOCKS_PER_HEAD,), np.uint32)
    _load().rqo_pack_ue8m0_array(_ptr(s), out.size, _ptr(out))
    return out


# ------------------------------------------------------------------ row steps

def rope_rows(rows, positions, cos_sin_cache, inverse: bool) -> np.ndarray:
    """Rotate the RoPE tail of fp32 rows [R, 512] (a rotated copy is returned)."""
    y = _np(rows, np.float32).reshape(-1, HEAD_DIM).copy()
    pos = _np(positions, np.int64).reshape(-1)
    cs = _np(cos_sin_cache, np.float32)
    if pos.size != y.shape[0]:
        raise OracleError("one position per row")
    rc = _load().rqo_rope_rows(_ptr(y), y.shape[0], _ptr(pos), _ptr(cs), cs.shape[0],
                               1 if inverse else 0)
    if rc:
        raise OracleError(f"rope_rows status {rc}")
    return y


def quant_rows(rows, eps: float = 1e-10):
    """Block-128 E4M3 quant of fp32 rows [R, 512] -> (codes [R,512] u8, scales [R,4] f32)."""
    y = _np(rows, np.float32).reshape(-1, HEAD_DIM)
    codes = np.empty(y.shape, np.uint8)
    scales = np.empty((y.shape[0], BLOCKS_PER_HEAD), np.float32)
    _load().rqo_quant_rows(_ptr(y), y.shape[0], float(eps), _ptr(codes), _ptr(scales))
    return codes, scales


# ------------------------------------------------------------------ full ops

def inv_rope_fp8_quant(x, positions, cos_sin_cache, heads_per_group: int,
                       eps: float = 1e-10, threads: int = 1):
    """Inverse RoPE + block-FP8 quant of x [N, H, 512] bf16.

    Returns (codes [N, G, hpg*512] uint8, scales [N, G, hpg*4] float32),
    G = H / heads_per_group. ``x`` may be a torch bf16 tensor (any token and
    head strides are honoured) or a uint16 numpy array of bf16 bit patterns.
    """
    if hasattr(x, "detach"):
        # torch tensor: honour its token / head strides, pass its data pointer
        t = x.detach().cpu()
        if t.stride(-1) != 1 or t.shape[-1] != HEAD_DIM:
            raise OracleError("x must be [N, H, 512] with a contiguous last dim")
        n, h = t.shape[0], t.shape[1]
        sx_t, sx_h = t.stride(0), t.stride(1)
        ptr, keep = t.data_ptr(), t
    else:
        arr = _np(x, np.uint16)
        n, h = arr.shape[0], arr.shape[1]
        sx_t, sx_h = arr.shape[1] * arr.shape[2], arr.shape[2]
        ptr, keep = arr.ctypes.data, arr
    pos = _np(positions, np.int64)
    cs = _np(cos_sin_cache, np.float32)
    hpg = int(heads_per_group)
    if hpg < 1 or h % hpg:
        raise OracleError("heads_per_group must divide the head count")
    g = h // hpg
    codes = np.empty((n, g, hpg * HEAD_DIM), np.uint8)
    scales = np.empty((n, g, hpg * BLOCKS_PER_HEAD), np.float32)
    rc = _load().rqo_inv_rope_fp8_quant(ptr, n, h, sx_t, sx_h, _ptr(pos), _ptr(cs), cs.shape[0],
                                        hpg, float(eps), _ptr(codes), _ptr(scales), int(threads))
    del keep
    if rc:
        raise OracleError(f"rqo_inv_rope_fp8_quant status {rc}")
    return codes, scales


def inv_rope_bf16(x, positions, cos_sin_cache, heads_per_group: int) -> np.ndarray:
    """The non-quantising variant: inverse RoPE of x [N, H, 512] bf16 as bf16
    bit patterns, [N, G, hpg*512] uint16."""
    arr = _np(x, np.uint16)
    n, h = arr.shape[0], arr.shape[1]
    pos = _np(positions, np.int64)
    cs = _np(cos_sin_cache, np.float32)
    hpg = int(heads_per_group)
    if hpg < 1 or h % hpg:
        raise OracleError("heads_per_group must divide the head count")
    out = np.empty((n, h // hpg, hpg * HEAD_DIM), np.uint16)
    rc = _load().rqo_inv_rope_bf16(_ptr(arr), n, h, h * HEAD_DIM, HEAD_DIM, _ptr(pos), _ptr(cs),
                                   cs.shape[0], hpg, _ptr(out))
    if rc:
        raise OracleError(f"rqo_inv_rope_bf16 status {rc}")
    return out


def rope_fp8_quant_insert(kv, positions, cos_sin_cache, slot_mapping, k_cache,
                          block_size: int, block_stride_bytes: int | None = None,
                          eps: float = 1e-10, threads: int = 1) -> np.ndarray:
    """Forward RoPE + block-FP8 quant of kv [N, 512] bf16 into a paged cache.

    ``k_cache`` is a uint8 array [num_blocks, block_bytes]; a copy with the
    mapped records written is returned (the input is not modified).
    """
    a = _np(kv, np.uint16)
    n = a.shape[0]
    pos = _np(positions, np.int64)
    cs = _np(cos_sin_cache, np.float32)
    slots = _np(slot_mapping, np.int64)
    cache = _np(k_cache, np.uint8).copy()
    stride = int(block_stride_bytes if block_stride_bytes is not None else cache.shape[1])
    rc = _load().rqo_rope_fp8_quant_insert(_ptr(a), n, a.shape[1], _ptr(pos), _ptr(cs),
                                           cs.shape[0], _ptr(slots), _ptr(cache),
                                           cache.shape[0], int(block_size), stride,
                                           float(eps), int(threads))
    if rc:
        raise OracleError(f"rqo_rope_fp8_quant_insert status {rc}")
    return cache


def qnorm_rope_kv_rope_quant_insert(q, kv, positions, cos_sin_cache, slot_mapping, k_cache,
                                    block_size: int, q_head_padded: int, norm_eps: float = 1e-6,
                                    quant_eps: float = 1e-10, norm_weight=None):
    """The fused q/kv op: q [N, Hq, 512] bf16 is RMS-normalised per head (times
    ``norm_weight`` [512] bf16 when given, before the rotation), forward-rotated
    and written into a zero-padded q_out [N, q_head_padded, 512] (bf16 bit
    patterns, uint16); kv [N, 512] is rotated, quantised and inserted into a
    copy of k_cache. Returns (q_out, k_cache copy)."""
    wt = None
    if norm_weight is not None:
        wt = _np(norm_weight, np.uint16).reshape(-1)
        if wt.size != HEAD_DIM:
            raise OracleError("norm_weight must hold 512 bf16 values")
    qa = _np(q, np.uint16)
    n, hq = qa.shape[0], qa.shape[1]
    a = _np(kv, np.uint16)
    pos = _np(positions, np.int64)
    cs = _np(cos_sin_cache, np.float32)
    slots = _np(slot_mapping, np.int64)
    cache = _np(k_cache, np.uint8).copy()
    q_out = np.empty((n, int(q_head_padded), HEAD_DIM), np.uint16)
    rc = _load().rqo_qnorm_rope_kv_rope_quant_insert(
        _ptr(qa), n, hq, hq * HEAD_DIM, HEAD_DIM, _ptr(a), a.shape[1], _ptr(q_out),
        int(q_head_padded), _ptr(cache), cache.shape[0], int(block_size), cache.shape[1],
        _ptr(slots), _ptr(pos), _ptr(cs), cs.shape[0], float(norm_eps),
        None if wt is None else _ptr(wt), float(quant_eps))
    if rc:
        raise OracleError(f"rqo_qnorm_rope_kv_rope_quant_insert status {rc}")
    return q_out, cache


def indexer_q_rope_quant(q, positions, cos_sin_cache, weights, softmax_scale: float,
                         head_scale: float, neox: bool = True, eps: float = 1e-4):
    """The indexer q op: q [N, H, 128] bf16 -> (codes [N, H, 128] uint8,
    weights_out [N, H] fp32); dims 0..63 rotated (NeoX halves or GPT-J pairs),
    rounded through bf16, one power-of-two scale per head folded into weights."""
    a = _np(q, np.uint16)
    n, h = a.shape[0], a.shape[1]
    if a.shape[2] != 128:
        raise OracleError("indexer heads are 128 wide")
    pos = _np(positions, np.int64)
    cs = _np(cos_sin_cache, np.float32)
    w = _np(weights, np.float32)
    codes = np.empty((n, h, 128), np.uint8)
    wout = np.empty((n, h), np.float32)
    rc = _load().rqo_indexer_q_rope_quant(_ptr(a), n, h, h * 128, 128, _ptr(pos), _ptr(cs),
                                          cs.shape[0], 1 if neox else 0, _ptr(w),
                                          float(softmax_scale), float(head_scale), float(eps),
                                          _ptr(codes), _ptr(wout))
    if rc:
        raise OracleError(f"rqo_indexer_q_rope_quant status {rc}")
    return codes, wout


def grouped_fp8_gemm(a_codes, a_scales, w_codes, w_scales) -> np.ndarray:
    """The grouped FP8 GEMM, exactly in float64: for every group g,
    y[:, g] = sum over 128-wide K blocks of (decode(A) * a_scale) @ (decode(W) * w_scale).T,
    with a_codes [N, G, K], a_scales [N, G, K/128], w_codes [G, n_out, K] and
    w_scales [G, n_out/128, K/128] (one scale per 128 x 128 weight block).
    Decoding uses the oracle's e4m3 decoder; the products and sums use numpy
    float64 matmul (every e4m3 product and the scaled sums of up to 2^22 of
    them are exact or within float64 rounding). Returns [N, G, n_out] float64."""
    ac = _np(a_codes, np.uint8)
    wc = _np(w_codes, np.uint8)
    sa = _np(a_scales, np.float32).astype(np.float64)
    sw = _np(w_scales, np.float32).astype(np.float64)
    n, g, k = ac.shape
    n_out = wc.shape[1]
    a = e4m3_decode(ac).reshape(n, g, k // 128, 128) * sa[..., None]
    w = e4m3_decode(wc).reshape(g, n_out // 128, 128, k // 128, 128) * \
        sw[:, :, None, :, None]
    a = a.reshape(n, g, k)
    w = w.reshape(g, n_out, k)
    return np.einsum("ngk,gok->ngo", a, w)


def ue8m0_decode(codes) -> np.ndarray:
    """Values of UE8M0 scale codes (OCP MX: an 8-bit biased exponent, no sign,
    no mantissa): code e is 2^(e - 127); code 255 is NaN. Returns float64."""
    e = _np(codes, np.uint8).astype(np.int64)
    out = np.ldexp(1.0, e - 127)
    return np.where(e == 255, np.nan, out)


def grouped_fp8_gemm_ue8m0(a_codes, a_sf_words, w_codes, w_sf) -> np.ndarray:
    """The grouped FP8 GEMM with UE8M0 block scales (the scale encoding of the
    inverse-RoPE page's packed-scale output, S3, on both operands):
      a_sf_words [N, G, K/512] uint32: byte b of word (n, g, h) is the code of
                 K block 4h + b of row n in group g (one word per 512-wide head,
                 exactly what the op writes in its UE8M0 mode);
      w_sf       [G, n_out/128, K/128] uint8: one code per 128 x 128 weight block.
    The codes are decoded to their powers of two and the GEMM is then the
    definition of grouped_fp8_gemm. Returns [N, G, n_out] float64."""
    words = _np(a_sf_words, np.uint32)
    n, g, heads = words.shape
    shifts = (8 * np.arange(BLOCKS_PER_HEAD, dtype=np.uint32))
    a_bytes = ((words[..., None] >> shifts) & 0xFF).astype(np.uint8)   # [N, G, heads, 4]
    a_scales = ue8m0_decode(a_bytes.reshape(n, g, heads * BLOCKS_PER_HEAD))
    w_scales = ue8m0_decode(w_sf)
    return grouped_fp8_gemm(a_codes, a_scales, w_codes, w_scales)
