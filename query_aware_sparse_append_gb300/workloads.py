"""Seeded synthetic decode workloads for query-aware sparse paged attention.

This module only draws inputs: shapes, random values, ragged lengths, the
physical page permutation behind the block tables, and integer page budgets.
It holds none of the method's arithmetic (no bounds, scores, selection or
attention), so both the CUDA path and the CPU oracle can consume its output.

Workload shapes follow the decode settings the TinyServe pages evaluate on
(TinyLLaMA-, GPT2-345M- and 1.3B-scale models, "TinyServe: Query-Aware Cache
Selection for Efficient LLM Serving", 实验亮点 / abstract, and the edgentiq
post's "Performance and Practicality" model list).  Values are synthetic: the
pages' models and datasets are not available here.

Every random stream is a numpy ``Generator(PCG64)`` seeded from
``SeedSequence([seed, config_id, stream, index])`` so that one sequence can be
regenerated alone (the oracle re-derives single sequences at full size).

Storage dtypes: ``"f32"`` -> numpy float32, ``"f16"`` -> numpy float16,
``"bf16"`` -> numpy uint16 holding bfloat16 bit patterns (round-to-nearest-even
from float32, done by torch's CPU cast).  ``"e4m3"`` (FP8 KV cache) draws its
queries and the K/V values it appends as float16: the cache quantizes them.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

DTYPES = ("f32", "f16", "bf16", "e4m3")


def input_dtype(dtype: str) -> str:
    """Dtype of the queries and of the appended K/V values of a workload."""
    return "f16" if dtype == "e4m3" else dtype

# stream ids inside a SeedSequence
_S_SEQ = 0          # per-sequence q, K, V
_S_LENS = 1         # ragged lengths
_S_PERM = 2         # physical page permutation
_S_SCALE = 3        # per-(head, channel) key scales
_S_PLANT = 4        # planted page positions (per sequence)
_S_APPEND = 5       # extra tokens appended after the prefix (decode-time appends)


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and value recipe of one synthetic decode workload."""

    name: str
    config_id: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    dtype: str
    ctx_min: int                 # context lengths drawn uniformly in [ctx_min, ctx_max]
    ctx_max: int
    budget_kind: str             # "pages" | "permille"
    budget_value: int            # pages, or per-mille of each sequence's page count
    q_std: float = 1.0 / 8.0
    planted_permille: int = 0    # planted pages per sequence = ceil(permille/1000 * N)
    planted_count: int = 0       # or a fixed count (config 1)
    key_channel_lognormal_sigma: float = 0.0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_pages(self) -> int:
        return -(-self.ctx_max // self.page_size)

    def with_budget(self, kind: str, value: int, name: Optional[str] = None) -> "Workload":
        return dataclasses.replace(self, budget_kind=kind, budget_value=value,
                                   name=name or self.name)

    def with_batch(self, batch: int) -> "Workload":
        return dataclasses.replace(self, batch=batch)


# The five decode settings plus the 8K / 12.5% headline case.
CONFIGS = {
    "tiny": Workload("tiny", 1, batch=1, num_q_heads=4, num_kv_heads=4, head_dim=64,
                     page_size=16, dtype="f32", ctx_min=2048, ctx_max=2048,
                     budget_kind="pages", budget_value=16, planted_count=4),
    "tinyllama": Workload("tinyllama", 2, batch=16, num_q_heads=32, num_kv_heads=4,
                          head_dim=64, page_size=16, dtype="f16", ctx_min=4096,
                          ctx_max=4096, budget_kind="permille", budget_value=250,
                          planted_permille=20),
    "gpt2_345m": Workload("gpt2_345m", 3, batch=64, num_q_heads=16, num_kv_heads=16,
                          head_dim=64, page_size=16, dtype="f16", ctx_min=256,
                          ctx_max=1024, budget_kind="pages", budget_value=32),
    "llama_1b3_32k": Workload("llama_1b3_32k", 4, batch=8, num_q_heads=32, num_kv_heads=8,
                              head_dim=128, page_size=32, dtype="bf16", ctx_min=32768,
                              ctx_max=32768, budget_kind="pages", budget_value=128,
                              planted_permille=10, key_channel_lognormal_sigma=0.5),
    "serving_mix": Workload("serving_mix", 5, batch=128, num_q_heads=32, num_kv_heads=4,
                            head_dim=128, page_size=16, dtype="f16", ctx_min=512,
                            ctx_max=16384, budget_kind="permille", budget_value=125),
    "headline_8k": Workload("headline_8k", 6, batch=128, num_q_heads=32, num_kv_heads=4,
                            head_dim=128, page_size=16, dtype="f16", ctx_min=8192,
                            ctx_max=8192, budget_kind="permille", budget_value=125),
    # the headline shapes with an FP8 (E4M3) KV cache
    "headline_8k_e4m3": Workload("headline_8k_e4m3", 7, batch=128, num_q_heads=32, num_kv_heads=4,
                                 head_dim=128, page_size=16, dtype="e4m3", ctx_min=8192,
                                 ctx_max=8192, budget_kind="permille", budget_value=125),
}

SERVING_MIX_BUDGETS_PERMILLE = (50, 125, 250, 500, 1000)


def _rng(seed: int, cfg: Workload, stream: int, index: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(
        [int(seed), int(cfg.config_id), int(stream), int(index)])))


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """Cast float32 samples to the storage dtype (bf16 as uint16 bit patterns)."""
    x = np.asarray(x, dtype=np.float32)
    dtype = input_dtype(dtype)
    if dtype == "f32":
        return x
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype == "bf16":
        import torch
        return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).view(
            torch.int16).numpy().view(np.uint16)
    raise ValueError(dtype)


def widen(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of stored elements."""
    dtype = input_dtype(dtype)
    if dtype == "bf16":
        u = np.asarray(x, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return u.view(np.float32).astype(np.float64)
    return np.asarray(x).astype(np.float64)


def np_storage_dtype(dtype: str):
    return {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}[input_dtype(dtype)]


def seq_lens(cfg: Workload, seed: int = 0) -> np.ndarray:
    """Context length of every sequence (uniform integers, inclusive range)."""
    if cfg.ctx_min == cfg.ctx_max:
        return np.full(cfg.batch, cfg.ctx_max, dtype=np.int32)
    r = _rng(seed, cfg, _S_LENS)
    return r.integers(cfg.ctx_min, cfg.ctx_max + 1, size=cfg.batch).astype(np.int32)


def num_pages(lens: np.ndarray, page_size: int) -> np.ndarray:
    return ((np.asarray(lens, dtype=np.int64) + page_size - 1) // page_size).astype(np.int32)


def budgets(cfg: Workload, lens: np.ndarray) -> np.ndarray:
    """Requested page budget per sequence (integer arithmetic only).

    ``pages``: the fixed count.  ``permille``: ceil(permille * N_b / 1000), at
    least 1.  Clamping to the page count and adding the always-kept pages is
    the method's business, not the workload's.
    """
    n = num_pages(lens, cfg.page_size).astype(np.int64)
    if cfg.budget_kind == "pages":
        return np.full(len(n), cfg.budget_value, dtype=np.int32)
    k = (n * cfg.budget_value + 999) // 1000
    return np.maximum(k, 1).astype(np.int32)


def key_channel_scales(cfg: Workload, seed: int = 0) -> Optional[np.ndarray]:
    """Per-(KV head, channel) key scale ~ LogNormal(0, sigma), shared by all tokens."""
    if cfg.key_channel_lognormal_sigma <= 0:
        return None
    r = _rng(seed, cfg, _S_SCALE)
    return r.lognormal(0.0, cfg.key_channel_lognormal_sigma,
                       size=(cfg.num_kv_heads, cfg.head_dim)).astype(np.float32)


def planted_pages(cfg: Workload, n_pages: int, b: int, seed: int = 0) -> np.ndarray:
    """Logical page ids (distinct, drawn from 1..N-2) whose keys point along q."""
    if cfg.planted_count:
        cnt = cfg.planted_count
    elif cfg.planted_permille:
        cnt = -(-cfg.planted_permille * n_pages // 1000)
    else:
        return np.zeros(0, dtype=np.int32)
    cnt = min(cnt, max(n_pages - 2, 0))
    if cnt == 0:
        return np.zeros(0, dtype=np.int32)
    r = _rng(seed, cfg, _S_PLANT, b)
    return np.sort(r.choice(np.arange(1, n_pages - 1), size=cnt, replace=False)).astype(np.int32)


@dataclasses.dataclass
class SequenceData:
    q: np.ndarray        # [Hq, d] storage dtype
    k: np.ndarray        # [L, Hkv, d] storage dtype
    v: np.ndarray        # [L, Hkv, d] storage dtype
    planted: np.ndarray  # logical page ids


def sequence(cfg: Workload, b: int, length: int, seed: int = 0,
             scales: Optional[np.ndarray] = None) -> SequenceData:
    """q, K and V of sequence ``b`` (regenerable alone).

    q ~ N(0,1) * q_std; K, V ~ N(0,1); keys scaled per (head, channel) when the
    workload has outlier channels.  In a planted page every key of KV head h is
    ``2*sqrt(d) * u_h + noise`` where u_h is the unit vector along the mean of
    the group's normalised queries (noise keeps the channel scale).
    """
    H, Hkv, d, P = cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim, cfg.page_size
    r = _rng(seed, cfg, _S_SEQ, b)
    q = (r.standard_normal((H, d), dtype=np.float32) * np.float32(cfg.q_std))
    q_st = to_storage(q, cfg.dtype)
    k = r.standard_normal((length, Hkv, d), dtype=np.float32)
    v = r.standard_normal((length, Hkv, d), dtype=np.float32)
    if scales is None:
        scales = key_channel_scales(cfg, seed)
    noise_scale = scales if scales is not None else np.ones((Hkv, d), np.float32)
    k *= noise_scale[None]
    n = -(-length // P)
    planted = planted_pages(cfg, n, b, seed)
    if planted.size:
        qs = widen(q_st, cfg.dtype).reshape(Hkv, cfg.group, d)
        qhat = qs / np.linalg.norm(qs, axis=-1, keepdims=True)
        u = qhat.mean(axis=1)
        u /= np.linalg.norm(u, axis=-1, keepdims=True)
        shift = (2.0 * math.sqrt(d) * u).astype(np.float32)  # [Hkv, d]
        for p in planted:
            lo, hi = p * P, min((p + 1) * P, length)
            k[lo:hi] = shift[None] + k[lo:hi]
    return SequenceData(q=q_st, k=to_storage(k, cfg.dtype), v=to_storage(v, cfg.dtype),
                        planted=planted)


def append_tokens(cfg: Workload, b: int, count: int, seed: int = 0,
                  scales: Optional[np.ndarray] = None):
    """Extra K/V tokens [count, Hkv, d] for decode-time append tests."""
    r = _rng(seed, cfg, _S_APPEND, b)
    k = r.standard_normal((count, cfg.num_kv_heads, cfg.head_dim), dtype=np.float32)
    v = r.standard_normal((count, cfg.num_kv_heads, cfg.head_dim), dtype=np.float32)
    if scales is None:
        scales = key_channel_scales(cfg, seed)
    if scales is not None:
        k *= scales[None]
    return to_storage(k, cfg.dtype), to_storage(v, cfg.dtype)


@dataclasses.dataclass
class PagePlan:
    """Physical page assignment: ``block_table[b, j]`` = physical page of logical page j."""

    block_table: np.ndarray   # [B, max_pages] int32, -1 where unassigned
    num_phys_pages: int


def page_plan(cfg: Workload, lens: np.ndarray, seed: int = 0, reserve_tokens: int = 0,
              shuffle: bool = True, spare_pages: int = 0,
              max_pages: Optional[int] = None) -> PagePlan:
    """Give each sequence pages for ``len + reserve_tokens`` tokens out of one pool.

    The pool is randomly permuted (``shuffle``) so that logically adjacent pages
    sit at unrelated physical addresses, as in a paged serving cache.
    """
    need = num_pages(np.asarray(lens) + reserve_tokens, cfg.page_size)
    width = int(max_pages if max_pages is not None else max(int(need.max()), 1))
    total = int(need.sum()) + spare_pages
    order = np.arange(total, dtype=np.int64)
    if shuffle:
        order = _rng(seed, cfg, _S_PERM).permutation(total)
    bt = np.full((len(need), width), -1, dtype=np.int32)
    pos = 0
    for b, n in enumerate(need):
        bt[b, :n] = order[pos:pos + n]
        pos += int(n)
    return PagePlan(block_table=bt, num_phys_pages=total)


def all_sequences(cfg: Workload, lens: Sequence[int], seed: int = 0) -> List[SequenceData]:
    scales = key_channel_scales(cfg, seed)
    return [sequence(cfg, b, int(L), seed, scales) for b, L in enumerate(lens)]
