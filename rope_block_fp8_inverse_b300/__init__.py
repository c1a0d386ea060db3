"""B300 (sm_103a) inverse RoPE + block-FP8 quant, and forward RoPE + FP8 paged insert.

Thin Python binding over the C ABI of ``include/rq.h`` (``librq.so``, built
in-tree by ``rope_block_fp8_inverse_b300.build``). This module only checks
and marshals arguments (device pointers, strides, the current CUDA stream);
every arithmetic step runs in the library's CUDA kernels. There is no CPU
path: CPU tensors, or a missing ``librq.so``, raise.

    codes, scales = inv_rope_fp8_quant(x, positions, cos_sin_cache, heads_per_group)
    rope_fp8_quant_insert(kv, positions, cos_sin_cache, slot_mapping, k_cache, block_size)
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["validate_indices", "debug_inject", "debug_block_scale", "debug_quant_codes", "DEBUG_STREAM_STAGE", "DEBUG_GEMM_LOADS", "inv_rope_fp8_quant_host", "host_workspace_bytes", "inv_rope_fp8_quant_gemm", "grouped_fp8_gemm", "grouped_fp8_gemm_ue8m0",
           "indexer_q_rope_quant", "qnorm_rope_kv_rope_quant_insert", "VARIANT_AUTO", "VARIANT_WARP_ROWS", "VARIANT_STREAM", "inv_rope_quant", "OUT_MODES",
           "empty_outputs", "inv_rope_fp8_quant", "rope_fp8_quant_insert", "lib", "RQError", "LIB_PATH",
           "HEAD_DIM", "RECORD_BYTES", "status_string", "ABI_SYMBOLS"]

HEAD_DIM = 512
BLOCKS_PER_HEAD = 4
# kernel variants of the inverse op (rq_inv_variant); all give identical bytes
VARIANT_AUTO, VARIANT_WARP_ROWS, VARIANT_STREAM = 0, 1, 2
RECORD_BYTES = 528
# output kinds of inv_rope_quant (rq_out_mode): fp32 scales, packed UE8M0 scales, bf16 (no quant)
OUT_MODES = {"fp8": 0, "ue8m0": 1, "bf16": 2}
DEFAULT_EPS = 1e-10
# test-only fault injection (rq_debug_inject)
DEBUG_STREAM_STAGE, DEBUG_GEMM_LOADS = 1, 2

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "librq.so")

# every symbol include/rq.h declares, with (restype, argtypes)
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
ABI_SYMBOLS = {
    "rq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "rq_version": (ctypes.c_int, []),
    "rq_inv_rope_fp8_quant": (ctypes.c_int, [_P, _I64, _I64, _I64, _I64, _P, _P, _I64, _I64,
                                             ctypes.c_float, _P, _P, _P, _P]),
    "rq_inv_rope_fp8_quant_ex": (ctypes.c_int, [_P, _I64, _I64, _I64, _I64, _P, _P, _I64, _I64,
                                                ctypes.c_float, _P, _P, _P, _P, ctypes.c_int]),
    "rq_rope_fp8_quant_insert": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _I64, _P, _P, _I64,
                                                _I64, _I64, ctypes.c_float, _P, _P]),
    "rq_qnorm_rope_kv_rope_quant_insert": (ctypes.c_int, [_P, _I64, _I64, _I64, _I64, _P, _I64, _P,
                                                          _I64, _P, _P, _I64, _P, _P, _I64, _I64,
                                                          _I64, ctypes.c_float, _P,
                                                          ctypes.c_float, _P, _P]),
    "rq_indexer_q_rope_fp8_quant": (ctypes.c_int, [_P, _I64, _I64, _I64, _I64, _P, _P, _I64,
                                                   ctypes.c_int, _P, ctypes.c_float, ctypes.c_float,
                                                   ctypes.c_float, _P, _P, _P, _P]),
    "rq_grouped_fp8_gemm": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _P, _P, _I64, _P, _P, _P]),
    "rq_debug_inject": (None, [ctypes.c_uint32, ctypes.c_uint32]),
    "rq_debug_block_scale": (ctypes.c_int, [ctypes.c_uint32, _I64, ctypes.c_float, _P, _P, _P]),
    "rq_debug_quant_codes": (ctypes.c_int, [ctypes.c_uint32, _I64, ctypes.c_int, _P, _P]),
    "rq_validate_indices_workspace": (ctypes.c_int64, [_I64]),
    "rq_validate_indices": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _P, _I64, _P, _P]),
    "rq_validate_indices_noalloc": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _P, _P]),
    "rq_inv_rope_fp8_quant_host_workspace": (ctypes.c_int64, [_I64, _I64]),
    "rq_inv_rope_fp8_quant_host": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _I64, _I64, ctypes.c_float,
                                                  _P, _P, _P, _I64, _I64, _P, _P]),
    "rq_grouped_fp8_gemm_ue8m0": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _P, _P, _I64, _P, _P,
                                                 _P]),
    "rq_inv_rope_fp8_quant_gemm": (ctypes.c_int, [_P, _I64, _I64, _I64, _I64, _P, _P, _I64, _I64,
                                                  ctypes.c_float, _P, _P, _I64, _P, _P, _P]),
    "rq_inv_rope_quant_layout": (ctypes.c_int, [_P, _I64, _I64, _I64, _I64, _P, _P, _I64, _I64,
                                                ctypes.c_float, ctypes.c_int, _P, _I64, _I64, _P,
                                                _I64, _I64, _I64, _P, _P]),
}

_lock = threading.Lock()
_lib = None


class RQError(RuntimeError):
    """A non-zero rq_status from the library."""

    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: status {status} ({status_string(status)})")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded librq.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m rope_block_fp8_inverse_b300.build` (needs nvcc)")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in ABI_SYMBOLS.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
        return _lib


def status_string(status: int) -> str:
    return lib().rq_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != 0:
        raise RQError(status, where)


def _cuda(t: torch.Tensor, name: str, dtype: torch.dtype) -> torch.Tensor:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def inv_rope_fp8_quant(x: torch.Tensor, positions: torch.Tensor, cos_sin_cache: torch.Tensor,
                       heads_per_group: int, eps: float = DEFAULT_EPS,
                       out: torch.Tensor | None = None, scales: torch.Tensor | None = None,
                       error_flags: torch.Tensor | None = None, variant: int = VARIANT_AUTO):
    """Inverse GPT-J RoPE on dims 448..511 + block-128 e4m3 quant with power-of-two scales.

    x: [N, H, 512] bf16 on the GPU (token / head strides free, last dim
    contiguous). Returns ``(out, scales)``: ``out`` [N, G, hpg*512] as
    ``torch.float8_e4m3fn``, ``scales`` [N, G, hpg*4] fp32, G = H / hpg.
    Preallocated ``out`` (uint8 or float8_e4m3fn) / ``scales`` are written in place.
    ``variant`` picks the kernel (VARIANT_*; the default is the warp-rows kernel,
    the faster of the two at every size measured).
    Runs on the current CUDA stream, asynchronously.
    """
    _cuda(x, "x", torch.bfloat16)
    if x.dim() != 3 or x.shape[2] != HEAD_DIM or x.stride(2) != 1:
        raise ValueError("x must be [N, H, 512] with a contiguous last dim")
    n, h = x.shape[0], x.shape[1]
    hpg = int(heads_per_group)
    if hpg < 1 or h % hpg:
        raise ValueError(f"heads_per_group={hpg} must divide H={h}")
    g = h // hpg
    _cuda(positions, "positions", torch.int64)
    _cuda(cos_sin_cache, "cos_sin_cache", torch.float32)
    if positions.shape != (n,) or not positions.is_contiguous():
        raise ValueError("positions must be a contiguous [N] int64 tensor")
    if cos_sin_cache.dim() != 2 or cos_sin_cache.shape[1] != 64 or not cos_sin_cache.is_contiguous():
        raise ValueError("cos_sin_cache must be a contiguous [P, 64] fp32 tensor")
    if out is None:
        out = torch.empty((n, g, hpg * HEAD_DIM), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((n, g, hpg * BLOCKS_PER_HEAD), dtype=torch.float32, device=x.device)
    if out.dtype not in (torch.uint8, torch.float8_e4m3fn) or not out.is_cuda:
        raise TypeError("out must be a uint8 or float8_e4m3fn CUDA tensor")
    if out.numel() != n * h * HEAD_DIM or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of N*H*512 bytes")
    _cuda(scales, "scales", torch.float32)
    if scales.numel() != n * h * BLOCKS_PER_HEAD or not scales.is_contiguous():
        raise ValueError("scales must be a contiguous tensor of N*H*4 floats")
    for t in (positions, cos_sin_cache, out, scales):
        if t.device != x.device:
            raise ValueError("all tensors must be on the same device")
    flags = 0
    if error_flags is not None:
        _cuda(error_flags, "error_flags", torch.int32)
        flags = error_flags.data_ptr()
    with torch.cuda.device(x.device):
        st = lib().rq_inv_rope_fp8_quant_ex(
            x.data_ptr(), n, h, x.stride(0), x.stride(1), positions.data_ptr(),
            cos_sin_cache.data_ptr(), cos_sin_cache.shape[0], hpg, float(eps), out.data_ptr(),
            scales.data_ptr(), flags, _stream(x.device), int(variant))
    _check(st, "rq_inv_rope_fp8_quant")
    return out.view(torch.float8_e4m3fn).view(n, g, hpg * HEAD_DIM), scales.view(n, g, hpg * BLOCKS_PER_HEAD)


def empty_outputs(n: int, groups: int, heads_per_group: int, mode: str = "fp8",
                  group_major: bool = False, device=None):
    """Uninitialised ``(out, scales)`` for :func:`inv_rope_quant`, shaped
    [N, G, hpg*512] / [N, G, hpg*4] (fp8), [N, G, hpg] int32 (ue8m0) or
    [N, G, hpg*512] bf16 with ``scales`` None (bf16). With ``group_major`` the
    storage is [G, N, ...] and the returned tensors are its [N, G, ...] views."""
    if mode not in OUT_MODES:
        raise ValueError(f"mode must be one of {sorted(OUT_MODES)}")
    w = heads_per_group * HEAD_DIM
    dt = torch.bfloat16 if mode == "bf16" else torch.uint8
    sw, sdt = ((heads_per_group * BLOCKS_PER_HEAD, torch.float32) if mode == "fp8"
               else (heads_per_group, torch.int32))

    def alloc(width, dtype):
        if group_major:
            return torch.empty((groups, n, width), dtype=dtype, device=device).permute(1, 0, 2)
        return torch.empty((n, groups, width), dtype=dtype, device=device)
    return alloc(w, dt), (None if mode == "bf16" else alloc(sw, sdt))


def inv_rope_quant(x: torch.Tensor, positions: torch.Tensor, cos_sin_cache: torch.Tensor,
                   heads_per_group: int, mode: str = "fp8", out: torch.Tensor | None = None,
                   scales: torch.Tensor | None = None, eps: float = DEFAULT_EPS,
                   error_flags: torch.Tensor | None = None):
    """Inverse RoPE with a choice of output kind and layout (``rq_inv_rope_quant_layout``).

    ``mode``: "fp8" (e4m3 codes + fp32 block scales), "ue8m0" (codes + one
    int32 per head holding its four UE8M0 scale bytes, block b in bits
    8b..8b+7) or "bf16" (no quantisation: the rotated head as bf16).
    ``out`` is an [N, G, hpg*512] view (uint8 / float8_e4m3fn, or bf16) and
    ``scales`` an [N, G, hpg*4] fp32 or [N, G, hpg] int32 view; any token /
    group strides work (e.g. group-major storage, see :func:`empty_outputs`),
    the last dim must be contiguous for ``out``. Returns ``(out, scales)``.
    """
    if mode not in OUT_MODES:
        raise ValueError(f"mode must be one of {sorted(OUT_MODES)}")
    _cuda(x, "x", torch.bfloat16)
    if x.dim() != 3 or x.shape[2] != HEAD_DIM or x.stride(2) != 1:
        raise ValueError("x must be [N, H, 512] with a contiguous last dim")
    n, h = x.shape[0], x.shape[1]
    hpg = int(heads_per_group)
    if hpg < 1 or h % hpg:
        raise ValueError(f"heads_per_group={hpg} must divide H={h}")
    g = h // hpg
    _cuda(positions, "positions", torch.int64)
    _cuda(cos_sin_cache, "cos_sin_cache", torch.float32)
    if positions.shape != (n,) or not positions.is_contiguous():
        raise ValueError("positions must be a contiguous [N] int64 tensor")
    if cos_sin_cache.dim() != 2 or cos_sin_cache.shape[1] != 64 or not cos_sin_cache.is_contiguous():
        raise ValueError("cos_sin_cache must be a contiguous [P, 64] fp32 tensor")
    if out is None:
        out, sc = empty_outputs(n, g, hpg, mode, device=x.device)
        scales = sc if scales is None else scales
    if mode != "bf16" and scales is None:
        scales = empty_outputs(n, g, hpg, mode, device=x.device)[1]
    want_out = (torch.bfloat16,) if mode == "bf16" else (torch.uint8, torch.float8_e4m3fn)
    if not out.is_cuda or out.dtype not in want_out:
        raise TypeError(f"out must be a CUDA tensor of {want_out}")
    if tuple(out.shape) != (n, g, hpg * HEAD_DIM) or out.stride(2) != 1:
        raise ValueError(f"out must be an [N, G, {hpg * HEAD_DIM}] view with a contiguous last dim")
    isz = out.element_size()
    o_t, o_g = out.stride(0) * isz, out.stride(1) * isz
    s_t = s_g = s_e = 0
    sptr = 0
    if mode != "bf16":
        sdt, sw = (torch.float32, hpg * BLOCKS_PER_HEAD) if mode == "fp8" else (torch.int32, hpg)
        _cuda(scales, "scales", sdt)
        if tuple(scales.shape) != (n, g, sw):
            raise ValueError(f"scales must be an [N, G, {sw}] view")
        s_t, s_g, s_e = scales.stride()
        sptr = scales.data_ptr()
    for t in (positions, cos_sin_cache, out) + ((scales,) if mode != "bf16" else ()):
        if t.device != x.device:
            raise ValueError("all tensors must be on the same device")
    flags = 0
    if error_flags is not None:
        _cuda(error_flags, "error_flags", torch.int32)
        flags = error_flags.data_ptr()
    with torch.cuda.device(x.device):
        st = lib().rq_inv_rope_quant_layout(
            x.data_ptr(), n, h, x.stride(0), x.stride(1), positions.data_ptr(),
            cos_sin_cache.data_ptr(), cos_sin_cache.shape[0], hpg, float(eps), OUT_MODES[mode],
            out.data_ptr(), o_t, o_g, sptr, s_t, s_g, s_e, flags, _stream(x.device))
    _check(st, "rq_inv_rope_quant_layout")
    return out, scales


def rope_fp8_quant_insert(kv: torch.Tensor, positions: torch.Tensor, cos_sin_cache: torch.Tensor,
                          slot_mapping: torch.Tensor, k_cache: torch.Tensor, block_size: int,
                          eps: float = DEFAULT_EPS, error_flags: torch.Tensor | None = None) -> None:
    """Forward GPT-J RoPE + block-128 e4m3 quant of kv [N, 512] bf16, scattered
    into the paged ``k_cache`` [num_blocks, block_bytes] uint8 by ``slot_mapping``.

    Each mapped token's 528-byte record (512 codes then 4 fp32 scales) lands at
    block ``slot // block_size``, byte offset ``(slot % block_size) * 528``;
    negative slots are skipped. Runs on the current CUDA stream.
    """
    _cuda(kv, "kv", torch.bfloat16)
    if kv.dim() != 2 or kv.shape[1] != HEAD_DIM or kv.stride(1) != 1:
        raise ValueError("kv must be [N, 512] with a contiguous last dim")
    n = kv.shape[0]
    _cuda(positions, "positions", torch.int64)
    _cuda(slot_mapping, "slot_mapping", torch.int64)
    _cuda(cos_sin_cache, "cos_sin_cache", torch.float32)
    _cuda(k_cache, "k_cache", torch.uint8)
    if positions.shape != (n,) or not positions.is_contiguous():
        raise ValueError("positions must be a contiguous [N] int64 tensor")
    if slot_mapping.shape != (n,) or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous [N] int64 tensor")
    if cos_sin_cache.dim() != 2 or cos_sin_cache.shape[1] != 64 or not cos_sin_cache.is_contiguous():
        raise ValueError("cos_sin_cache must be a contiguous [P, 64] fp32 tensor")
    if k_cache.dim() != 2 or k_cache.stride(1) != 1:
        raise ValueError("k_cache must be [num_blocks, block_bytes] with contiguous rows")
    if k_cache.shape[1] < int(block_size) * RECORD_BYTES:
        raise ValueError(f"k_cache rows must hold block_size * {RECORD_BYTES} bytes")
    for t in (positions, slot_mapping, cos_sin_cache, k_cache):
        if t.device != kv.device:
            raise ValueError("all tensors must be on the same device")
    flags = 0
    if error_flags is not None:
        _cuda(error_flags, "error_flags", torch.int32)
        flags = error_flags.data_ptr()
    with torch.cuda.device(kv.device):
        st = lib().rq_rope_fp8_quant_insert(
            kv.data_ptr(), n, kv.stride(0), positions.data_ptr(), cos_sin_cache.data_ptr(),
            cos_sin_cache.shape[0], slot_mapping.data_ptr(), k_cache.data_ptr(), k_cache.shape[0],
            int(block_size), k_cache.stride(0), float(eps), flags, _stream(kv.device))
    _check(st, "rq_rope_fp8_quant_insert")


def qnorm_rope_kv_rope_quant_insert(q: torch.Tensor, kv: torch.Tensor, positions: torch.Tensor,
                                    cos_sin_cache: torch.Tensor, slot_mapping: torch.Tensor,
                                    k_cache: torch.Tensor, block_size: int, q_head_padded: int,
                                    norm_eps: float = 1e-6, quant_eps: float = DEFAULT_EPS,
                                    q_out: torch.Tensor | None = None,
                                    error_flags: torch.Tensor | None = None,
                                    norm_weight: torch.Tensor | None = None) -> torch.Tensor:
    """The fused q/kv op (``rq_qnorm_rope_kv_rope_quant_insert``): q [N, Hq, 512]
    bf16 is RMS-normalised per head (times ``norm_weight`` [512] bf16 when given,
    before the rotation), forward-rotated and written to ``q_out``
    [N, q_head_padded, 512] bf16 (pad heads zeroed); kv [N, 512] is rotated,
    quantised and inserted into ``k_cache``. Returns ``q_out``."""
    _cuda(q, "q", torch.bfloat16)
    _cuda(kv, "kv", torch.bfloat16)
    if q.dim() != 3 or q.shape[2] != HEAD_DIM or q.stride(2) != 1:
        raise ValueError("q must be [N, Hq, 512] with a contiguous last dim")
    n, hq = q.shape[0], q.shape[1]
    hpad = int(q_head_padded)
    if hpad < hq:
        raise ValueError("q_head_padded must be >= the q head count")
    if kv.dim() != 2 or kv.shape != (n, HEAD_DIM) or kv.stride(1) != 1:
        raise ValueError("kv must be [N, 512] with a contiguous last dim")
    _cuda(positions, "positions", torch.int64)
    _cuda(slot_mapping, "slot_mapping", torch.int64)
    _cuda(cos_sin_cache, "cos_sin_cache", torch.float32)
    _cuda(k_cache, "k_cache", torch.uint8)
    if positions.shape != (n,) or not positions.is_contiguous():
        raise ValueError("positions must be a contiguous [N] int64 tensor")
    if slot_mapping.shape != (n,) or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous [N] int64 tensor")
    if cos_sin_cache.dim() != 2 or cos_sin_cache.shape[1] != 64 or not cos_sin_cache.is_contiguous():
        raise ValueError("cos_sin_cache must be a contiguous [P, 64] fp32 tensor")
    if k_cache.dim() != 2 or k_cache.stride(1) != 1 or k_cache.shape[1] < int(block_size) * RECORD_BYTES:
        raise ValueError("k_cache must be [num_blocks, >= block_size*528] with contiguous rows")
    if q_out is None:
        q_out = torch.empty((n, hpad, HEAD_DIM), dtype=torch.bfloat16, device=q.device)
    _cuda(q_out, "q_out", torch.bfloat16)
    if tuple(q_out.shape) != (n, hpad, HEAD_DIM) or not q_out.is_contiguous():
        raise ValueError("q_out must be a contiguous [N, q_head_padded, 512] bf16 tensor")
    for t in (kv, positions, slot_mapping, cos_sin_cache, k_cache, q_out):
        if t.device != q.device:
            raise ValueError("all tensors must be on the same device")
    wptr = 0
    if norm_weight is not None:
        _cuda(norm_weight, "norm_weight", torch.bfloat16)
        if norm_weight.numel() != HEAD_DIM or not norm_weight.is_contiguous() or \
                norm_weight.device != q.device:
            raise ValueError("norm_weight must be a contiguous bf16 [512] tensor on q's device")
        wptr = norm_weight.data_ptr()
    flags = 0
    if error_flags is not None:
        _cuda(error_flags, "error_flags", torch.int32)
        flags = error_flags.data_ptr()
    with torch.cuda.device(q.device):
        st = lib().rq_qnorm_rope_kv_rope_quant_insert(
            q.data_ptr(), n, hq, q.stride(0), q.stride(1), kv.data_ptr(), kv.stride(0),
            q_out.data_ptr(), hpad, positions.data_ptr(), cos_sin_cache.data_ptr(),
            cos_sin_cache.shape[0], slot_mapping.data_ptr(), k_cache.data_ptr(), k_cache.shape[0],
            int(block_size), k_cache.stride(0), float(norm_eps), wptr, float(quant_eps), flags,
            _stream(q.device))
    _check(st, "rq_qnorm_rope_kv_rope_quant_insert")
    return q_out


ROPE_STYLES = {"neox": 0, "gptj": 1}


def indexer_q_rope_quant(q: torch.Tensor, positions: torch.Tensor, cos_sin_cache: torch.Tensor,
                         weights: torch.Tensor, softmax_scale: float, head_scale: float,
                         rope_style: str = "neox", eps: float = 1e-4,
                         out: torch.Tensor | None = None, weights_out: torch.Tensor | None = None,
                         error_flags: torch.Tensor | None = None):
    """The indexer q op (``rq_indexer_q_rope_fp8_quant``): q [N, H, 128] bf16 ->
    (codes [N, H, 128] float8_e4m3fn, weights_out [N, H] fp32). Dims 0..63 are
    rotated forward ("neox": dim j with 32 + j, "gptj": 2j with 2j + 1) and
    rounded through bf16; one power-of-two scale per head is folded into
    weights_out = weights * q_scale * softmax_scale * head_scale."""
    if rope_style not in ROPE_STYLES:
        raise ValueError(f"rope_style must be one of {sorted(ROPE_STYLES)}")
    _cuda(q, "q", torch.bfloat16)
    if q.dim() != 3 or q.shape[2] != 128 or q.stride(2) != 1:
        raise ValueError("q must be [N, H, 128] with a contiguous last dim")
    n, h = q.shape[0], q.shape[1]
    _cuda(positions, "positions", torch.int64)
    _cuda(cos_sin_cache, "cos_sin_cache", torch.float32)
    _cuda(weights, "weights", torch.float32)
    if positions.shape != (n,) or not positions.is_contiguous():
        raise ValueError("positions must be a contiguous [N] int64 tensor")
    if cos_sin_cache.dim() != 2 or cos_sin_cache.shape[1] != 64 or not cos_sin_cache.is_contiguous():
        raise ValueError("cos_sin_cache must be a contiguous [P, 64] fp32 tensor")
    if tuple(weights.shape) != (n, h) or not weights.is_contiguous():
        raise ValueError("weights must be a contiguous [N, H] fp32 tensor")
    if out is None:
        out = torch.empty((n, h, 128), dtype=torch.uint8, device=q.device)
    if weights_out is None:
        weights_out = torch.empty((n, h), dtype=torch.float32, device=q.device)
    if out.dtype not in (torch.uint8, torch.float8_e4m3fn) or not out.is_cuda:
        raise TypeError("out must be a uint8 or float8_e4m3fn CUDA tensor")
    if tuple(out.shape) != (n, h, 128) or not out.is_contiguous():
        raise ValueError("out must be a contiguous [N, H, 128] tensor")
    _cuda(weights_out, "weights_out", torch.float32)
    if tuple(weights_out.shape) != (n, h) or not weights_out.is_contiguous():
        raise ValueError("weights_out must be a contiguous [N, H] fp32 tensor")
    for t in (positions, cos_sin_cache, weights, out, weights_out):
        if t.device != q.device:
            raise ValueError("all tensors must be on the same device")
    flags = 0
    if error_flags is not None:
        _cuda(error_flags, "error_flags", torch.int32)
        flags = error_flags.data_ptr()
    with torch.cuda.device(q.device):
        st = lib().rq_indexer_q_rope_fp8_quant(
            q.data_ptr(), n, h, q.stride(0), q.stride(1), positions.data_ptr(),
            cos_sin_cache.data_ptr(), cos_sin_cache.shape[0], ROPE_STYLES[rope_style],
            weights.data_ptr(), float(softmax_scale), float(head_scale), float(eps),
            out.data_ptr(), weights_out.data_ptr(), flags, _stream(q.device))
    _check(st, "rq_indexer_q_rope_fp8_quant")
    return out.view(torch.float8_e4m3fn), weights_out


def grouped_fp8_gemm(a_codes: torch.Tensor, a_scales: torch.Tensor, w_codes: torch.Tensor,
                     w_scales: torch.Tensor, out: torch.Tensor | None = None,
                     error_flags: torch.Tensor | None = None) -> torch.Tensor:
    """Grouped FP8 GEMM on the tensor cores (``rq_grouped_fp8_gemm``): for every
    group g, ``y[:, g] = dequant(a_codes[:, g]) @ dequant(w_codes[g]).T`` in
    fp32, written as bf16 [N, G, n_out]. ``a_codes`` [N, G, K] e4m3 (uint8 or
    float8) with ``a_scales`` [N, G, K/128] fp32 (what inv_rope_fp8_quant
    returns); ``w_codes`` [G, n_out, K] with ``w_scales`` [G, n_out/128, K/128]."""
    for t, name in ((a_codes, "a_codes"), (w_codes, "w_codes")):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype not in (torch.uint8, torch.float8_e4m3fn) or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous uint8 / float8_e4m3fn tensor")
    if a_codes.dim() != 3 or w_codes.dim() != 3:
        raise ValueError("a_codes must be [N, G, K] and w_codes [G, n_out, K]")
    n, g, k = a_codes.shape
    if w_codes.shape[0] != g or w_codes.shape[2] != k:
        raise ValueError("w_codes must be [G, n_out, K] with the codes' G and K")
    n_out = w_codes.shape[1]
    _cuda(a_scales, "a_scales", torch.float32)
    _cuda(w_scales, "w_scales", torch.float32)
    if tuple(a_scales.shape) != (n, g, k // 128) or not a_scales.is_contiguous():
        raise ValueError("a_scales must be a contiguous [N, G, K/128] fp32 tensor")
    if tuple(w_scales.shape) != (g, n_out // 128, k // 128) or not w_scales.is_contiguous():
        raise ValueError("w_scales must be a contiguous [G, n_out/128, K/128] fp32 tensor")
    if out is None:
        out = torch.empty((n, g, n_out), dtype=torch.bfloat16, device=a_codes.device)
    _cuda(out, "out", torch.bfloat16)
    if tuple(out.shape) != (n, g, n_out) or not out.is_contiguous():
        raise ValueError("out must be a contiguous [N, G, n_out] bf16 tensor")
    for t in (a_scales, w_codes, w_scales, out):
        if t.device != a_codes.device:
            raise ValueError("all tensors must be on the same device")
    flags = 0
    if error_flags is not None:
        _cuda(error_flags, "error_flags", torch.int32)
        flags = error_flags.data_ptr()
    with torch.cuda.device(a_codes.device):
        st = lib().rq_grouped_fp8_gemm(a_codes.data_ptr(), a_scales.data_ptr(), n, g, k,
                                       w_codes.data_ptr(), w_scales.data_ptr(), n_out,
                                       out.data_ptr(), flags, _stream(a_codes.device))
    _check(st, "rq_grouped_fp8_gemm")
    return out


def validate_indices(positions: torch.Tensor, cache_rows: int,
                     slot_mapping: torch.Tensor | None = None, num_slots: int = 0,
                     workspace: torch.Tensor | None = None) -> int:
    """Debug helper (``rq_validate_indices``, synchronous): the RQ_FLAG_* bits of
    the device-side preconditions the given indices break (0 = all valid):
    positions in [0, cache_rows); slots negative (skip) or below ``num_slots``
    (= num_blocks * block_size), and no slot used twice. ``workspace``: a CUDA
    uint8 tensor of at least ``rq_validate_indices_workspace(num_slots)`` bytes
    (allocated when None)."""
    _cuda(positions, "positions", torch.int64)
    if positions.dim() != 1 or not positions.is_contiguous():
        raise ValueError("positions must be a contiguous [N] int64 tensor")
    n = positions.shape[0]
    sptr = 0
    if slot_mapping is not None:
        _cuda(slot_mapping, "slot_mapping", torch.int64)
        if tuple(slot_mapping.shape) != (n,) or not slot_mapping.is_contiguous() or \
                slot_mapping.device != positions.device:
            raise ValueError("slot_mapping must be a contiguous [N] int64 tensor on the same device")
        sptr = slot_mapping.data_ptr()
    need = lib().rq_validate_indices_workspace(num_slots if slot_mapping is not None else 0)
    if need < 0:
        raise ValueError("num_slots out of range")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=positions.device)
    _cuda(workspace, "workspace", torch.uint8)
    result = ctypes.c_uint32(0)
    with torch.cuda.device(positions.device):
        st = lib().rq_validate_indices(positions.data_ptr(), sptr, n, int(cache_rows),
                                       int(num_slots), workspace.data_ptr(), workspace.numel(),
                                       ctypes.addressof(result), _stream(positions.device))
    _check(st, "rq_validate_indices")
    return int(result.value)


def debug_inject(mask: int = 0, spin_limit: int = 0) -> None:
    """TEST ONLY (``rq_debug_inject``): make the selected kernels skip one of
    their own copies so that a bounded wait runs out after ``spin_limit`` polls
    and ``RQ_FLAG_TIMEOUT`` is reported; ``debug_inject()`` restores normal
    operation. Applies to later calls from this thread."""
    lib().rq_debug_inject(mask, spin_limit)


def debug_block_scale(first_bits: int, count: int, eps: float, device=None):
    """TEST ONLY (``rq_debug_block_scale``): the kernels' block scale of each
    amax = fp32 bit pattern first_bits + i (i < count), clamped below by
    ``eps``, and its reciprocal, as two CUDA fp32 tensors [count]."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    scales = torch.empty(count, dtype=torch.float32, device=dev)
    inv = torch.empty(count, dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = lib().rq_debug_block_scale(int(first_bits), int(count), float(eps), scales.data_ptr(),
                                        inv.data_ptr(), _stream(dev))
    _check(st, "rq_debug_block_scale")
    return scales, inv


def debug_quant_codes(first_bits: int, count: int, scale_exp: int = 0, out: torch.Tensor | None = None,
                      device=None) -> torch.Tensor:
    """TEST ONLY (``rq_debug_quant_codes``): the e4m3 code the kernels store for
    the fp32 value of bit pattern first_bits + i (i < count, a multiple of 16)
    in a block of scale 2^scale_exp, as a CUDA uint8 tensor [count]."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if out is None:
        out = torch.empty(count, dtype=torch.uint8, device=dev)
    if out.dtype != torch.uint8 or not out.is_cuda or out.numel() < count or not out.is_contiguous():
        raise ValueError("out must be a contiguous CUDA uint8 tensor of at least count bytes")
    with torch.cuda.device(out.device):
        st = lib().rq_debug_quant_codes(int(first_bits), int(count), int(scale_exp), out.data_ptr(),
                                        _stream(out.device))
    _check(st, "rq_debug_quant_codes")
    return out[:count]


def host_workspace_bytes(n_heads: int, chunk_tokens: int) -> int:
    """Device workspace bytes ``inv_rope_fp8_quant_host`` needs (three chunk slots)."""
    n = lib().rq_inv_rope_fp8_quant_host_workspace(n_heads, chunk_tokens)
    if n < 0:
        raise ValueError("n_heads and chunk_tokens must be >= 1 with chunk_tokens * n_heads < 2^31")
    return int(n)


def inv_rope_fp8_quant_host(x: torch.Tensor, positions: torch.Tensor, cos_sin_cache: torch.Tensor,
                            heads_per_group: int, eps: float = DEFAULT_EPS,
                            out: torch.Tensor | None = None, scales: torch.Tensor | None = None,
                            workspace: torch.Tensor | None = None, chunk_tokens: int = 512,
                            error_flags: torch.Tensor | None = None):
    """The inverse op over HOST tensors (``rq_inv_rope_fp8_quant_host``): x [N, H, 512]
    bf16 and positions [N] int64 on the CPU (pinned for the copies to overlap),
    the cos/sin cache on the GPU. The library streams chunks of ``chunk_tokens``
    tokens through ``workspace`` (a CUDA uint8 tensor of at least
    ``host_workspace_bytes(H, chunk_tokens)`` bytes; allocated when None), with
    copy-in, kernels and copy-out of consecutive chunks overlapped. Returns the
    CPU (pinned) ``(out, scales)``, complete once the current CUDA stream of
    the cache's device has synchronised."""
    if not isinstance(x, torch.Tensor) or x.is_cuda or x.dtype != torch.bfloat16:
        raise TypeError("x must be a CPU bf16 tensor")
    if x.dim() != 3 or x.shape[-1] != HEAD_DIM or not x.is_contiguous():
        raise ValueError("x must be a contiguous [N, H, 512] tensor")
    n, h, _ = x.shape
    if not isinstance(positions, torch.Tensor) or positions.is_cuda or \
            positions.dtype != torch.int64 or tuple(positions.shape) != (n,) or \
            not positions.is_contiguous():
        raise ValueError("positions must be a contiguous CPU int64 tensor [N]")
    _cuda(cos_sin_cache, "cos_sin_cache", torch.float32)
    dev = cos_sin_cache.device
    if heads_per_group < 1 or h % heads_per_group:
        raise ValueError("heads_per_group must divide the head count")
    g = h // heads_per_group
    if out is None:
        out = torch.empty((n, g, heads_per_group * HEAD_DIM), dtype=torch.float8_e4m3fn,
                          pin_memory=True)
    if scales is None:
        scales = torch.empty((n, g, heads_per_group * BLOCKS_PER_HEAD), dtype=torch.float32,
                             pin_memory=True)
    for t, name, dts, shape in ((out, "out", (torch.uint8, torch.float8_e4m3fn),
                                 (n, g, heads_per_group * HEAD_DIM)),
                                (scales, "scales", (torch.float32,),
                                 (n, g, heads_per_group * BLOCKS_PER_HEAD))):
        if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype not in dts or \
                tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU {dts[0]} tensor of shape {shape}")
    need = host_workspace_bytes(h, chunk_tokens)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _cuda(workspace, "workspace", torch.uint8)
    if workspace.device != dev:
        raise ValueError("workspace must be on the cache's device")
    flags = 0
    if error_flags is not None:
        _cuda(error_flags, "error_flags", torch.int32)
        flags = error_flags.data_ptr()
    with torch.cuda.device(dev):
        st = lib().rq_inv_rope_fp8_quant_host(
            x.data_ptr(), n, h, positions.data_ptr(), cos_sin_cache.data_ptr(),
            cos_sin_cache.shape[0], heads_per_group, eps, out.data_ptr(), scales.data_ptr(),
            workspace.data_ptr(), workspace.numel(), chunk_tokens, flags, _stream(dev))
    _check(st, "rq_inv_rope_fp8_quant_host")
    return out, scales


def grouped_fp8_gemm_ue8m0(a_codes: torch.Tensor, a_sf: torch.Tensor, w_codes: torch.Tensor,
                           w_sf: torch.Tensor, out: torch.Tensor | None = None,
                           error_flags: torch.Tensor | None = None) -> torch.Tensor:
    """Grouped FP8 GEMM with UE8M0 block scales on the block-scaled tensor-core
    MMA (``rq_grouped_fp8_gemm_ue8m0``). ``a_codes`` [N, G, K] e4m3 with
    ``a_sf`` [N, G, K/512] packed UE8M0 words (int32 / uint32: byte b of word h
    = K block 4h + b, what ``inv_rope_quant(mode="ue8m0")`` writes token-major);
    ``w_codes`` [G, n_out, K] with ``w_sf`` [G, n_out/128, K/128] uint8 codes.
    K a multiple of 512, at most 4096. Returns bf16 [N, G, n_out]."""
    for t, name in ((a_codes, "a_codes"), (w_codes, "w_codes")):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype not in (torch.uint8, torch.float8_e4m3fn) or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous uint8 / float8_e4m3fn tensor")
    if a_codes.dim() != 3 or w_codes.dim() != 3:
        raise ValueError("a_codes must be [N, G, K] and w_codes [G, n_out, K]")
    n, g, k = a_codes.shape
    if w_codes.shape[0] != g or w_codes.shape[2] != k:
        raise ValueError("w_codes must be [G, n_out, K] with the codes' G and K")
    n_out = w_codes.shape[1]
    if not isinstance(a_sf, torch.Tensor) or not a_sf.is_cuda or \
            a_sf.dtype not in (torch.int32, torch.uint32):
        raise TypeError("a_sf must be an int32 / uint32 CUDA tensor")
    _cuda(w_sf, "w_sf", torch.uint8)
    if tuple(a_sf.shape) != (n, g, k // 512) or not a_sf.is_contiguous():
        raise ValueError("a_sf must be a contiguous [N, G, K/512] tensor of packed words")
    if tuple(w_sf.shape) != (g, n_out // 128, k // 128) or not w_sf.is_contiguous():
        raise ValueError("w_sf must be a contiguous [G, n_out/128, K/128] uint8 tensor")
    if out is None:
        out = torch.empty((n, g, n_out), dtype=torch.bfloat16, device=a_codes.device)
    _cuda(out, "out", torch.bfloat16)
    if tuple(out.shape) != (n, g, n_out) or not out.is_contiguous():
        raise ValueError("out must be a contiguous [N, G, n_out] bf16 tensor")
    for t in (a_sf, w_codes, w_sf, out):
        if t.device != a_codes.device:
            raise ValueError("all tensors must be on the same device")
    flags = 0
    if error_flags is not None:
        _cuda(error_flags, "error_flags", torch.int32)
        flags = error_flags.data_ptr()
    with torch.cuda.device(a_codes.device):
        st = lib().rq_grouped_fp8_gemm_ue8m0(a_codes.data_ptr(), a_sf.data_ptr(), n, g, k,
                                             w_codes.data_ptr(), w_sf.data_ptr(), n_out,
                                             out.data_ptr(), flags, _stream(a_codes.device))
    _check(st, "rq_grouped_fp8_gemm_ue8m0")
    return out


def inv_rope_fp8_quant_gemm(x: torch.Tensor, positions: torch.Tensor, cos_sin_cache: torch.Tensor,
                            heads_per_group: int, w_codes: torch.Tensor, w_scales: torch.Tensor,
                            eps: float = DEFAULT_EPS, out: torch.Tensor | None = None,
                            error_flags: torch.Tensor | None = None) -> torch.Tensor:
    """Inverse RoPE + block-FP8 quant fused into the grouped FP8 GEMM
    (``rq_inv_rope_fp8_quant_gemm``): y [N, G, n_out] bf16, bit-identical to
    ``grouped_fp8_gemm(*inv_rope_fp8_quant(x, ...), w_codes, w_scales)``."""
    _cuda(x, "x", torch.bfloat16)
    if x.dim() != 3 or x.shape[2] != HEAD_DIM or x.stride(2) != 1:
        raise ValueError("x must be [N, H, 512] with a contiguous last dim")
    n, h = x.shape[0], x.shape[1]
    hpg = int(heads_per_group)
    if hpg < 1 or h % hpg:
        raise ValueError(f"heads_per_group={hpg} must divide H={h}")
    g, k = h // hpg, hpg * HEAD_DIM
    _cuda(positions, "positions", torch.int64)
    _cuda(cos_sin_cache, "cos_sin_cache", torch.float32)
    if positions.shape != (n,) or not positions.is_contiguous():
        raise ValueError("positions must be a contiguous [N] int64 tensor")
    if cos_sin_cache.dim() != 2 or cos_sin_cache.shape[1] != 64 or not cos_sin_cache.is_contiguous():
        raise ValueError("cos_sin_cache must be a contiguous [P, 64] fp32 tensor")
    if w_codes.dtype not in (torch.uint8, torch.float8_e4m3fn) or not w_codes.is_cuda or \
            not w_codes.is_contiguous() or w_codes.dim() != 3 or w_codes.shape[0] != g or \
            w_codes.shape[2] != k:
        raise ValueError(f"w_codes must be a contiguous [G={g}, n_out, K={k}] e4m3 CUDA tensor")
    n_out = w_codes.shape[1]
    _cuda(w_scales, "w_scales", torch.float32)
    if tuple(w_scales.shape) != (g, n_out // 128, k // 128) or not w_scales.is_contiguous():
        raise ValueError("w_scales must be a contiguous [G, n_out/128, K/128] fp32 tensor")
    if out is None:
        out = torch.empty((n, g, n_out), dtype=torch.bfloat16, device=x.device)
    _cuda(out, "out", torch.bfloat16)
    if tuple(out.shape) != (n, g, n_out) or not out.is_contiguous():
        raise ValueError("out must be a contiguous [N, G, n_out] bf16 tensor")
    for t in (positions, cos_sin_cache, w_codes, w_scales, out):
        if t.device != x.device:
            raise ValueError("all tensors must be on the same device")
    flags = 0
    if error_flags is not None:
        _cuda(error_flags, "error_flags", torch.int32)
        flags = error_flags.data_ptr()
    with torch.cuda.device(x.device):
        st = lib().rq_inv_rope_fp8_quant_gemm(
            x.data_ptr(), n, h, x.stride(0), x.stride(1), positions.data_ptr(),
            cos_sin_cache.data_ptr(), cos_sin_cache.shape[0], hpg, float(eps), w_codes.data_ptr(),
            w_scales.data_ptr(), n_out, out.data_ptr(), flags, _stream(x.device))
    _check(st, "rq_inv_rope_fp8_quant_gemm")
    return out
