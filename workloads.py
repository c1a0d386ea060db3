"""Seeded synthetic inputs shared by the CUDA path's tests / bench and the oracle.

This module only draws inputs; it holds none of the method's arithmetic (no
rotation, no scale, no FP8 encoding). Every tensor is created on the CPU with
a ``torch.Generator`` seeded explicitly, in a fixed draw order:

1. ``x = randn(shape)`` (fp32),
2. where outliers apply: ``m = rand(shape) < 0.01`` and ``x = where(m, 50 x, x)``,
3. ``x`` cast to bf16 (round to nearest even),
4. positions (when drawn), then slots (when drawn).

The cos/sin cache is an input of the op, not part of it: row p holds
``cos(p * theta_j)`` in columns 0..31 and ``sin(p * theta_j)`` in 32..63 with
``theta_j = 10000 ** (-j / 32)``, evaluated in float64 and rounded to fp32
(the RoPE cache layout of the DeepSeek-V4 inverse-RoPE page, S2: cos at
column j, sin at column 32 + j).

Workloads (named by what they are):

* ``tiny``       N=64, H=8, heads_per_group=8, positions U[0,4096), cache 4096 rows.
* ``prefill16k`` N=16384, H=32, heads_per_group=8, positions 0..16383, cache 65536.
* ``decode``     N in {1,...,64}, H=32, heads_per_group=8, no outliers,
                 positions U[0,65536), cache 65536.
* ``irregular``  N=8192, H=24, heads_per_group=6, positions U[0,32768), cache 32768.
* ``insert16k``  kv [16384, 512], positions 0..16383, cache 65536,
                 slots = randperm(512*64)[:N], paged cache 512 blocks x 64 slots x 528 B.
* ``fused16k``   the fused q/kv op: q [16384, 32, 512] (the 32 heads per rank of the
                 DeepSeek-V4-Flash TP2 shape) padded to 64 heads in q_out, with the
                 insert16k kv side; q is drawn before kv from the same generator.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

HEAD_DIM = 512
CACHE_WIDTH = 64
RECORD_BYTES = 528
ROPE_BASE = 10000.0
OUTLIER_RATE = 0.01
OUTLIER_GAIN = 50.0


@dataclass(frozen=True)
class InverseSpec:
    name: str
    n_tokens: int
    n_heads: int
    heads_per_group: int
    cache_rows: int
    positions: str          # "arange" or "uniform"
    outliers: bool
    seed: int = 0


@dataclass(frozen=True)
class InsertSpec:
    name: str
    n_tokens: int
    cache_rows: int
    num_blocks: int
    block_size: int
    seed: int = 0


TINY = InverseSpec("tiny", 64, 8, 8, 4096, "uniform", True)
PREFILL16K = InverseSpec("prefill16k", 16384, 32, 8, 65536, "arange", True)
IRREGULAR = InverseSpec("irregular", 8192, 24, 6, 32768, "uniform", True)
DECODE_TOKENS = (1, 2, 4, 8, 16, 32, 64)
INSERT16K = InsertSpec("insert16k", 16384, 65536, 512, 64)


@dataclass(frozen=True)
class FusedSpec:
    name: str
    n_tokens: int
    n_heads_q: int
    q_head_padded: int
    cache_rows: int
    num_blocks: int
    block_size: int
    seed: int = 0


FUSED16K = FusedSpec("fused16k", 16384, 32, 64, 65536, 512, 64)


@dataclass(frozen=True)
class IndexerSpec:
    name: str
    n_tokens: int
    n_heads: int
    cache_rows: int
    seed: int = 0


# the sparse-attention indexer's q: 64 heads of 128 per token (dims 0..63 rotary)
INDEXER16K = IndexerSpec("indexer16k", 16384, 64, 65536)


def decode_spec(n_tokens: int) -> InverseSpec:
    return InverseSpec(f"decode{n_tokens}", n_tokens, 32, 8, 65536, "uniform", False)


# (H, groups) pairs the inverse-RoPE page's test parametrisation lists (S5);
# heads_per_group = H / groups.
PAGE_TEST_SHAPES = ((64, 8), (32, 4), (128, 8), (24, 4))


def rope_cache(rows: int, base: float = ROPE_BASE) -> torch.Tensor:
    """[rows, 64] fp32 cos/sin cache: cos(p*theta_j) | sin(p*theta_j), float64 then fp32."""
    half = CACHE_WIDTH // 2
    j = torch.arange(half, dtype=torch.float64)
    theta = base ** (-j / half)
    ang = torch.arange(rows, dtype=torch.float64)[:, None] * theta[None, :]
    return torch.cat([torch.cos(ang), torch.sin(ang)], dim=1).to(torch.float32).contiguous()


def _activations(gen: torch.Generator, shape, outliers: bool) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if outliers:
        m = torch.rand(shape, generator=gen) < OUTLIER_RATE
        x = torch.where(m, x * OUTLIER_GAIN, x)
    return x.to(torch.bfloat16)


def inverse_inputs(spec: InverseSpec, cache: torch.Tensor | None = None) -> dict:
    """x [N,H,512] bf16, positions [N] int64, cos_sin_cache [P,64] fp32 (all CPU)."""
    gen = torch.Generator().manual_seed(spec.seed)
    x = _activations(gen, (spec.n_tokens, spec.n_heads, HEAD_DIM), spec.outliers)
    if spec.positions == "arange":
        pos = torch.arange(spec.n_tokens, dtype=torch.int64)
    else:
        pos = torch.randint(0, spec.cache_rows, (spec.n_tokens,), generator=gen,
                            dtype=torch.int64)
    if cache is None:
        cache = rope_cache(spec.cache_rows)
    return {"x": x, "positions": pos, "cos_sin_cache": cache,
            "heads_per_group": spec.heads_per_group}


def insert_inputs(spec: InsertSpec, cache: torch.Tensor | None = None,
                  fill: int = 0xA5) -> dict:
    """kv [N,512] bf16, positions, slot_mapping (distinct), k_cache filled with ``fill``."""
    gen = torch.Generator().manual_seed(spec.seed)
    kv = _activations(gen, (spec.n_tokens, HEAD_DIM), False)
    pos = torch.arange(spec.n_tokens, dtype=torch.int64)
    n_slots = spec.num_blocks * spec.block_size
    slots = torch.randperm(n_slots, generator=gen)[: spec.n_tokens].to(torch.int64)
    if cache is None:
        cache = rope_cache(spec.cache_rows)
    block_bytes = spec.block_size * RECORD_BYTES
    k_cache = torch.full((spec.num_blocks, block_bytes), fill, dtype=torch.uint8)
    return {"kv": kv, "positions": pos, "cos_sin_cache": cache, "slot_mapping": slots,
            "k_cache": k_cache, "block_size": spec.block_size}


def fused_inputs(spec: FusedSpec, cache: torch.Tensor | None = None, fill: int = 0xA5) -> dict:
    """q [N,Hq,512] bf16 (drawn first), then kv, positions 0..N-1, slots and a
    ``fill``-ed paged cache as in insert_inputs."""
    gen = torch.Generator().manual_seed(spec.seed)
    q = _activations(gen, (spec.n_tokens, spec.n_heads_q, HEAD_DIM), False)
    kv = _activations(gen, (spec.n_tokens, HEAD_DIM), False)
    pos = torch.arange(spec.n_tokens, dtype=torch.int64)
    n_slots = spec.num_blocks * spec.block_size
    slots = torch.randperm(n_slots, generator=gen)[: spec.n_tokens].to(torch.int64)
    if cache is None:
        cache = rope_cache(spec.cache_rows)
    k_cache = torch.full((spec.num_blocks, spec.block_size * RECORD_BYTES), fill, dtype=torch.uint8)
    return {"q": q, "kv": kv, "positions": pos, "cos_sin_cache": cache, "slot_mapping": slots,
            "k_cache": k_cache, "block_size": spec.block_size, "q_head_padded": spec.q_head_padded}


def norm_weight(seed: int = 0) -> torch.Tensor:
    """A synthetic RMSNorm weight for the fused q/kv op: 512 bf16 values
    uniform in [0.5, 1.5), from its own generator (seed + 1), so the op's other
    inputs are drawn as without it."""
    gen = torch.Generator().manual_seed(seed + 1)
    return (torch.rand(HEAD_DIM, generator=gen) + 0.5).to(torch.bfloat16)


def indexer_inputs(spec: IndexerSpec, cache: torch.Tensor | None = None) -> dict:
    """q [N,H,128] bf16 N(0,1) + 1% x50 outliers (drawn first), weights [N,H]
    fp32 uniform in [0.5, 1.5), positions 0..N-1."""
    gen = torch.Generator().manual_seed(spec.seed)
    q = _activations(gen, (spec.n_tokens, spec.n_heads, 128), True)
    w = torch.rand((spec.n_tokens, spec.n_heads), generator=gen) + 0.5
    if cache is None:
        cache = rope_cache(spec.cache_rows)
    return {"q": q, "weights": w, "positions": torch.arange(spec.n_tokens, dtype=torch.int64),
            "cos_sin_cache": cache, "softmax_scale": 128 ** -0.5,
            "head_scale": spec.n_heads ** -0.5}


def indexer_bytes(n_tokens: int, n_heads: int) -> int:
    """Algorithmic bytes of one indexer q op: q read (256 B per head), codes
    written (128 B), weight read and written (4 + 4 B), position and one cos/sin
    row read per token."""
    return n_tokens * (n_heads * (256 + 128 + 8) + 8 + CACHE_WIDTH * 4)


def fused_bytes(n_tokens: int, n_heads_q: int, q_head_padded: int) -> int:
    """Algorithmic bytes of one fused q/kv op: q read, every q_out head written
    (pad heads too), plus the insert op's bytes (the cos/sin row serves q and kv)."""
    return n_tokens * (n_heads_q * HEAD_DIM * 2 + q_head_padded * HEAD_DIM * 2) + \
        insert_bytes(n_tokens)


def inverse_bytes(n_tokens: int, n_heads: int, mode: str = "fp8") -> int:
    """Algorithmic HBM bytes of one inverse op: x read, the outputs written
    (codes + 4 fp32 scales per head for "fp8", codes + one packed 4-byte word
    per head for "ue8m0", 512 bf16 values per head for "bf16"), positions and
    one 256-byte cos/sin row read per token."""
    out_per_head = {"fp8": HEAD_DIM + 4 * 4, "ue8m0": HEAD_DIM + 4, "bf16": HEAD_DIM * 2}[mode]
    per_head = HEAD_DIM * 2 + out_per_head
    per_token = 8 + CACHE_WIDTH * 4
    return n_tokens * (n_heads * per_head + per_token)


def insert_bytes(n_tokens: int) -> int:
    """Algorithmic bytes of one insert op: kv read, position + slot + cos/sin row
    read, one 528-byte record written per token."""
    return n_tokens * (HEAD_DIM * 2 + 8 + 8 + CACHE_WIDTH * 4 + RECORD_BYTES)


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)

