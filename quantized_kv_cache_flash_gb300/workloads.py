"""Seeded synthetic workloads for quantized-KV decode attention.

This module only draws random numbers and describes shapes.  It holds none of
the method's arithmetic (no rotation, no codebook, no quantisation, no
attention), so both the CUDA path and the fp64 oracle can be fed from it.

Every stream is drawn from ``numpy.random.Generator(PCG64(SeedSequence(key)))``
with ``key = [1000 + config_number, stream_id, *unit]``, so one (batch, kv-head)
unit can be regenerated on its own without drawing the whole tensor.  Values
are N(0, 1) rounded to fp16; "outlier channels" are 4 distinct channel indices
(drawn once per workload) whose K values are multiplied by 8 for every head and
token.  The shapes follow the attention shapes the pages quote: the tiny
Turbo4Asym parity case (4 query heads over 2 KV heads, from the mlxcel
Turbo4Asym pull request's parity test), Qwen2.5-7B (28/4 heads), Llama-3-8B
(32/8 heads) and a long-context speculative block.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

HEAD_DIM = 128

# stream ids used in the seed key
_S_Q, _S_K, _S_V, _S_OUTLIER, _S_LEN, _S_KNEW, _S_VNEW = range(7)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode-attention workload (shapes, mode, seeds)."""

    number: int            # 1-based position in the workload list
    name: str
    mode: str              # "turbo4_asym" | "turbo3" | "turbo4"
    batch: int
    num_q_heads: int
    num_kv_heads: int
    context: int           # visible context per sequence (max when ragged)
    tq: int = 1            # query rows per sequence (causal within the block)
    context_min: Optional[int] = None   # ragged: lengths ~ U[context_min, context]
    outliers: bool = True  # K has 4 channels scaled x8
    append: int = 0        # tokens appended per sequence inside each step
    prefill_chunk: int = 0 # tokens encoded per sequence as a separately timed chunk
    prompt: bool = False   # a prompt of `tq` tokens appended to an empty cache, then attended
    rot_seed: int = 42

    @property
    def seed(self) -> int:
        return 1000 + self.number

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def ragged(self) -> bool:
        return self.context_min is not None


WORKLOADS = [
    Workload(1, "tiny_turbo4asym_b1_hq4_hkv2_l256", "turbo4_asym", 1, 4, 2, 256,
             outliers=False),
    Workload(2, "qwen25_7b_turbo3_b1_hq28_hkv4_l8192", "turbo3", 1, 28, 4, 8192),
    Workload(3, "turbo4asym_b1_hq28_hkv4_l16384", "turbo4_asym", 1, 28, 4, 16384),
    Workload(4, "llama3_8b_turbo4_b32_hq32_hkv8_l16k_32k_ragged_append1", "turbo4",
             32, 32, 8, 32768, context_min=16384, append=1),
    Workload(5, "long_turbo3_b4_hq32_hkv8_l131072_tq4_prefill4096", "turbo3",
             4, 32, 8, 131072, tq=4, prefill_chunk=4096),
    # the 8K prefill leg of the pages' sweep at Qwen2.5-7B attention shape: an
    # 8192-token prompt appended to an empty cache, then causal attention of
    # all its queries over it
    Workload(6, "qwen25_7b_turbo3_prompt8192_prefill", "turbo3", 1, 28, 4, 8192, tq=8192,
             prompt=True),
]


def by_number(n: int) -> Workload:
    return WORKLOADS[n - 1]


def _rng(w: Workload, stream: int, *unit: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(
        [w.seed, stream, *unit])))


def _normal16(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float32).astype(np.float16)


def lengths(w: Workload) -> np.ndarray:
    """Visible context per sequence (int32 [B]) at the decode step."""
    if not w.ragged:
        return np.full(w.batch, w.context, dtype=np.int32)
    rng = _rng(w, _S_LEN)
    return rng.integers(w.context_min, w.context, size=w.batch, endpoint=True
                        ).astype(np.int32)


def outlier_channels(w: Workload) -> np.ndarray:
    if not w.outliers:
        return np.zeros(0, dtype=np.int64)
    rng = _rng(w, _S_OUTLIER)
    return np.sort(rng.choice(HEAD_DIM, size=4, replace=False))


def query(w: Workload, b: int) -> np.ndarray:
    """q for sequence b: fp16 [Hq, Tq, 128]."""
    return _normal16(_rng(w, _S_Q, b), (w.num_q_heads, w.tq, HEAD_DIM))


def _apply_outliers(w: Workload, x: np.ndarray) -> np.ndarray:
    ch = outlier_channels(w)
    if ch.size:
        x = x.astype(np.float32)
        x[..., ch] *= 8.0
        x = x.astype(np.float16)
    return x


def keys(w: Workload, b: int, h: int, start: int, stop: int) -> np.ndarray:
    """K tokens [start, stop) of unit (b, h): fp16 [stop-start, 128].

    Token t of a unit is always the same value whatever slice is asked for:
    the unit's stream is drawn in fixed blocks of 4096 tokens.
    """
    return _apply_outliers(w, _blocked(w, _S_K, b, h, start, stop))


def values(w: Workload, b: int, h: int, start: int, stop: int) -> np.ndarray:
    """V tokens [start, stop) of unit (b, h): fp16 [stop-start, 128]."""
    return _blocked(w, _S_V, b, h, start, stop)


_BLOCK = 4096


def _blocked(w: Workload, stream: int, b: int, h: int, start: int, stop: int
             ) -> np.ndarray:
    out = np.empty((max(stop - start, 0), HEAD_DIM), dtype=np.float16)
    t = start
    while t < stop:
        blk = t // _BLOCK
        x = _normal16(_rng(w, stream, b, h, blk), (_BLOCK, HEAD_DIM))
        lo = t - blk * _BLOCK
        hi = min(stop - blk * _BLOCK, _BLOCK)
        out[t - start:t - start + hi - lo] = x[lo:hi]
        t += hi - lo
    return out


def query_all(w: Workload) -> np.ndarray:
    """q for all sequences: fp16 [B, Hq, Tq, 128]."""
    return np.stack([query(w, b) for b in range(w.batch)])


def kv_unit(w: Workload, b: int, h: int, stop: int):
    """(K, V) fp16 [stop, 128] each for tokens [0, stop) of unit (b, h)."""
    return keys(w, b, h, 0, stop), values(w, b, h, 0, stop)



_S_RANDCODE, _S_RANDNORM = 7, 8


def random_codes(key: int, rows: int, record_bytes: int) -> np.ndarray:
    """Uniform random bytes [rows, record_bytes]: a packed cache whose every
    code is equally likely (any byte pattern is a valid record)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([key, _S_RANDCODE])))
    return rng.integers(0, 256, size=(rows, record_bytes), dtype=np.uint8)


def random_norms(key: int, rows: int, lo: float = 6.0, hi: float = 16.0) -> np.ndarray:
    """fp16 norms ~ U[lo, hi] (the norm of a 128-dim N(0,1) vector is ~11.3)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([key, _S_RANDNORM])))
    return rng.uniform(lo, hi, size=rows).astype(np.float16)


def random_fp16(key: int, shape, scale: float = 1.0) -> np.ndarray:
    """N(0, scale^2) rounded to fp16."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([key, 9])))
    return (rng.standard_normal(shape, dtype=np.float32) * np.float32(scale)).astype(np.float16)
