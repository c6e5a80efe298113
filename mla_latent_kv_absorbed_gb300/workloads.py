"""Seeded synthetic decode batches for absorbed MLA decode.

This module only draws numbers: it holds none of the attention arithmetic, so
both the fp64 oracle (test infrastructure) and the CUDA path can take their
inputs from it without sharing any of the method's code.

The five workloads follow the decode shapes of the DeepSeek pages:
  * one 576-wide bf16 row per cache slot (512-d latent ``c`` then the 64-d
    RoPE key), "MLA" section of the SGLang attention-backends page;
  * page size 1, so a request's cache is a list of slot numbers held in the
    CSR pair (kv_indptr, kv_indices), "Paged, ragged batches" on the same page;
  * the query already multiplied by W_UK (q_nope, 512-d) plus the 64-d rope
    query, per head.

Recipe (identical for every workload; seed = 20261200 + workload number):
  1. context lengths, drawn as the workload says;
  2. slots: the first nnz entries of ``rng.permutation(pool)``, handed to the
     requests in order (random, non-contiguous, never duplicated);
  3. kv_cache [pool, 576]: N(0,1) in float32, rounded to bf16 (round to
     nearest even), generated in blocks of rows from the same stream;
  4. q_nope [B, H, 512], then 5. q_rope [B, H, 64], same distribution.
sm_scale is 1/sqrt(192) (qk_head_dim 128 + 64 with mscale 1).

bf16 values are kept as their uint16 bit patterns (numpy has no bf16 type).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

KV_LORA_RANK = 512
QK_ROPE_HEAD_DIM = 64
KV_ROW = KV_LORA_RANK + QK_ROPE_HEAD_DIM  # 576
SEED_BASE = 20261200
SM_SCALE = 1.0 / math.sqrt(192.0)

_GEN_ROWS = 1 << 15  # rows per generation block (same stream either way)


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    number: int
    name: str
    batch: int
    heads: int
    pool: int
    lengths: str  # how the context lengths are drawn
    fixed: tuple = ()
    lo: int = 0
    hi: int = 0

    @property
    def seed(self) -> int:
        return SEED_BASE + self.number


WORKLOADS = {
    1: WorkloadSpec(1, "tiny_b4_h16", 4, 16, 512, "fixed", fixed=(1, 7, 33, 100)),
    2: WorkloadSpec(2, "v2lite_b64_h16_u512_4096", 64, 16, 1 << 19, "uniform", lo=512, hi=4096),
    3: WorkloadSpec(3, "v3_b128_h128_l4096", 128, 128, 1 << 19, "fixed", fixed=(4096,) * 128),
    4: WorkloadSpec(4, "ragged_b256_h128_lognormal1500", 256, 128, 1 << 20, "lognormal", lo=16, hi=32768),
    5: WorkloadSpec(5, "long_b2_h128_64k_128k", 2, 128, 1 << 19, "fixed", fixed=(65536, 131072)),
}


@dataclasses.dataclass
class DecodeBatch:
    """One synthetic decode step (all arrays host-side numpy)."""
    spec: Optional[WorkloadSpec]
    heads: int
    lengths: np.ndarray      # int64 [B]
    kv_indptr: np.ndarray    # int32 [B+1]
    kv_indices: np.ndarray   # int32 [nnz]
    kv_cache: np.ndarray     # uint16 bf16 bits [pool, 576]
    q_nope: np.ndarray       # uint16 bf16 bits [B, H, 512]
    q_rope: np.ndarray       # uint16 bf16 bits [B, H, 64]
    sm_scale: float = SM_SCALE

    @property
    def batch(self) -> int:
        return int(self.lengths.shape[0])

    @property
    def nnz(self) -> int:
        return int(self.kv_indptr[-1])

    @property
    def pool(self) -> int:
        return int(self.kv_cache.shape[0])


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bits.

    Inputs here are finite normal draws, so no NaN handling is needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def _normal_bf16(rng: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    out = np.empty((rows, cols), dtype=np.uint16)
    for r0 in range(0, rows, _GEN_ROWS):
        r1 = min(rows, r0 + _GEN_ROWS)
        out[r0:r1] = f32_to_bf16_bits(rng.standard_normal((r1 - r0, cols), dtype=np.float32))
    return out


def draw_lengths(spec: WorkloadSpec, rng: np.random.Generator) -> np.ndarray:
    if spec.lengths == "fixed":
        return np.asarray(spec.fixed, dtype=np.int64)
    if spec.lengths == "uniform":
        return rng.integers(spec.lo, spec.hi + 1, size=spec.batch).astype(np.int64)
    if spec.lengths == "lognormal":
        v = np.exp(rng.normal(math.log(1500.0), 1.0, size=spec.batch))
        return np.clip(np.rint(v), spec.lo, spec.hi).astype(np.int64)
    raise ValueError(spec.lengths)


def make_batch(lengths, heads: int, pool: int, seed: int, spec: Optional[WorkloadSpec] = None,
               rng: Optional[np.random.Generator] = None, slots: str = "permutation") -> DecodeBatch:
    """Build a batch for explicit lengths (the recipe's steps 2-5).

    ``slots="permutation"`` uses the recipe; ``"contiguous"`` hands out slots
    0..nnz-1 in order (used by a few edge tests only).
    """
    rng = rng if rng is not None else np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int64)
    nnz = int(lengths.sum())
    if nnz > pool:
        raise ValueError(f"nnz {nnz} exceeds pool {pool}")
    indptr = np.zeros(lengths.shape[0] + 1, dtype=np.int64)
    np.cumsum(lengths, out=indptr[1:])
    if slots == "permutation":
        indices = rng.permutation(pool)[:nnz].astype(np.int32)
    elif slots == "contiguous":
        indices = np.arange(nnz, dtype=np.int32)
    else:
        raise ValueError(slots)
    kv = _normal_bf16(rng, pool, KV_ROW)
    B = lengths.shape[0]
    qn = _normal_bf16(rng, B * heads, KV_LORA_RANK).reshape(B, heads, KV_LORA_RANK)
    qr = _normal_bf16(rng, B * heads, QK_ROPE_HEAD_DIM).reshape(B, heads, QK_ROPE_HEAD_DIM)
    return DecodeBatch(spec=spec, heads=heads, lengths=lengths, kv_indptr=indptr.astype(np.int32),
                       kv_indices=indices, kv_cache=kv, q_nope=qn, q_rope=qr)


def make_workload(number: int) -> DecodeBatch:
    spec = WORKLOADS[number]
    rng = np.random.default_rng(spec.seed)
    lengths = draw_lengths(spec, rng)
    return make_batch(lengths, spec.heads, spec.pool, spec.seed, spec=spec, rng=rng)


def workload_stats(spec_number: int) -> dict:
    """Lengths-only summary (cheap: draws no cache values)."""
    spec = WORKLOADS[spec_number]
    rng = np.random.default_rng(spec.seed)
    lengths = draw_lengths(spec, rng)
    return {"batch": spec.batch, "heads": spec.heads, "pool": spec.pool,
            "nnz": int(lengths.sum()), "max_len": int(lengths.max()), "min_len": int(lengths.min())}


@dataclasses.dataclass
class HeadProductInputs:
    """Synthetic inputs of the two per-head products around the decode
    (uint16 bf16 bits): the query before absorption and the w_kc / w_vc
    weights split from a kv_b_proj of DeepSeek's shape (128 nope and 128 value
    dims per head, rank 512)."""
    q_pre: np.ndarray   # [B, H, 128]
    w_kc: np.ndarray    # [H, 128, 512]
    w_vc: np.ndarray    # [H, 512, 128]


def make_head_product_inputs(batch: int, heads: int, seed: int) -> HeadProductInputs:
    """N(0,1) queries; weights N(0, 1/fan_in) so the products stay O(1); all
    rounded to bf16.  Draw order: q_pre, w_kc, w_vc."""
    rng = np.random.default_rng(seed)
    q_pre = _normal_bf16(rng, batch * heads, 128).reshape(batch, heads, 128)
    w_kc = f32_to_bf16_bits(rng.standard_normal((heads, 128, 512), dtype=np.float32) / np.float32(math.sqrt(128)))
    w_vc = f32_to_bf16_bits(rng.standard_normal((heads, 512, 128), dtype=np.float32) / np.float32(math.sqrt(512)))
    return HeadProductInputs(q_pre=q_pre, w_kc=w_kc, w_vc=w_vc)


FP8_KV_SCALE = 2.0 ** -5   # cache scale of the synthetic FP8 caches: values about N(0, 1)


def make_fp8_cache(pool: int, seed: int) -> np.ndarray:
    """Synthetic FP8 (E4M3) cache [pool, 576] uint8, built from its bit fields:
    a draw x ~ N(0, 1) * 32 gives the sign and the exponent field
    clip(floor(log2 |x|) + 7, 0, 15); the mantissa field is uniform.  With
    FP8_KV_SCALE the values are then roughly N(0, 1).  The NaN code is
    replaced by the largest finite one."""
    rng = np.random.default_rng(seed)
    out = np.empty((pool, 576), dtype=np.uint8)
    for r0 in range(0, pool, _GEN_ROWS):
        r1 = min(pool, r0 + _GEN_ROWS)
        x = rng.standard_normal((r1 - r0, 576), dtype=np.float32) * 32.0
        m = rng.integers(0, 8, size=x.shape, dtype=np.uint8)
        with np.errstate(divide="ignore"):
            e = np.clip(np.floor(np.log2(np.abs(x))) + 7, 0, 15).astype(np.uint8)
        code = (e << 3) | m
        code = np.where(code == 0x7F, 0x7E, code).astype(np.uint8)
        out[r0:r1] = code | np.where(x < 0, 0x80, 0).astype(np.uint8)
    return out
