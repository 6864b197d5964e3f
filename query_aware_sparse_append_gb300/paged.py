"""Load a synthetic workload into a device paged KV cache through the library.

The pools are allocated with torch and filled with ``kv_append`` (the
library's own append kernel, which also builds the page boxes), a group of
sequences per call so that staging buffers stay small.  The CUDA library is
loaded on the first ``load`` call, not at import.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np
import torch

from . import workloads as W

TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
               "e4m3": torch.float16}          # the dtype of q, out and appended K/V
POOL_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
              "e4m3": torch.uint8}             # the dtype of the pools and boxes


def to_torch(x: np.ndarray, dtype: str) -> torch.Tensor:
    """Host tensor sharing the bits of a storage-dtype numpy array."""
    if W.input_dtype(dtype) == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x))


@dataclasses.dataclass
class DeviceWorkload:
    cfg: W.Workload
    lens: np.ndarray              # host lengths
    budgets: np.ndarray           # host page budgets
    plan: W.PagePlan
    seqs: List[W.SequenceData]
    cache: "binding.PagedKVCache" = None
    block_table: torch.Tensor = None
    lens_dev: torch.Tensor = None
    budget_dev: torch.Tensor = None
    q_dev: torch.Tensor = None

    @property
    def max_budget(self) -> int:
        n = W.num_pages(self.lens, self.cfg.page_size)
        k = np.minimum(n, np.maximum(self.budgets, np.minimum(n, 2)))
        return max(2, int(k.max()) if len(k) else 2)


def generate(cfg: W.Workload, seed: int = 0, batch: Optional[int] = None, lens=None,
             budgets=None, shuffle: bool = True, reserve_tokens: int = 0) -> DeviceWorkload:
    """Host side of a workload: lengths, budgets, page plan and per-sequence q/K/V."""
    if batch is not None:
        cfg = cfg.with_batch(batch)
    lens = np.asarray(W.seq_lens(cfg, seed) if lens is None else lens, dtype=np.int32)
    bud = np.asarray(W.budgets(cfg, lens) if budgets is None else budgets, dtype=np.int32)
    width = max(1, int(W.num_pages(lens + reserve_tokens, cfg.page_size).max()))
    plan = W.page_plan(cfg, lens, seed, reserve_tokens=reserve_tokens, shuffle=shuffle,
                       max_pages=width)
    scales = W.key_channel_scales(cfg, seed)
    seqs = [W.sequence(cfg, b, int(L), seed, scales) for b, L in enumerate(lens)]
    return DeviceWorkload(cfg, lens, bud, plan, seqs)


def load(wl: DeviceWorkload, device="cuda", poison: bool = False,
         append_chunks: Optional[List[int]] = None, group: int = 16) -> DeviceWorkload:
    """Allocate the pools and append every sequence's tokens (then q, lengths, budgets).

    poison: fill pools and boxes with NaN first, so that reading any slot or box
    the method must not use corrupts the results visibly.
    append_chunks: several append calls of these token counts instead of one.
    """
    from . import binding as qasa   # loads libqasa.so

    cfg = wl.cfg
    dev = torch.device(device)
    cache = qasa.PagedKVCache.empty(wl.plan.num_phys_pages, cfg.num_kv_heads, cfg.page_size,
                                    cfg.head_dim, POOL_DTYPE[cfg.dtype], dev)
    if poison:
        nan = 0x7F if cfg.dtype == "e4m3" else float("nan")   # E4M3 NaN code
        cache.k_pool.fill_(nan)
        cache.v_pool.fill_(nan)
        cache.page_bounds.fill_(nan)
        if cache.page_scales is not None:
            cache.page_scales.fill_(float("nan"))
    bt = torch.from_numpy(wl.plan.block_table).to(dev)
    B = cfg.batch
    lens = wl.lens.astype(np.int64)
    chunks = append_chunks or [int(lens.max()) if B else 0]
    done = np.zeros(B, dtype=np.int64)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for chunk in chunks:
        for b0 in range(0, B, group):
            b1 = min(B, b0 + group)
            take = np.minimum(lens[b0:b1] - done[b0:b1], chunk).clip(min=0)
            T = int(take.max()) if len(take) else 0
            if T == 0:
                continue
            kn = np.zeros((b1 - b0, T, cfg.num_kv_heads, cfg.head_dim),
                          dtype=W.np_storage_dtype(cfg.dtype))
            vn = np.zeros_like(kn)
            for i, b in enumerate(range(b0, b1)):
                s, t = int(done[b]), int(take[i])
                kn[i, :t] = wl.seqs[b].k[s:s + t]
                vn[i, :t] = wl.seqs[b].v[s:s + t]
            qasa.kv_append(cache, bt[b0:b1].contiguous(),
                           torch.from_numpy(done[b0:b1].astype(np.int32)).to(dev),
                           to_torch(kn, cfg.dtype).to(dev), to_torch(vn, cfg.dtype).to(dev),
                           append_lens=torch.from_numpy(take.astype(np.int32)).to(dev),
                           status=status)
            done[b0:b1] += take
    if not np.array_equal(done, lens):
        raise RuntimeError("append chunks do not cover the sequences")
    torch.cuda.synchronize(dev)
    st = int(status.item())
    if st:
        raise RuntimeError("append reported device errors: %s" % qasa.decode_device_errors(st))
    if B:
        q = np.stack([s.q for s in wl.seqs])
    else:
        q = np.zeros((0, cfg.num_q_heads, cfg.head_dim), W.np_storage_dtype(cfg.dtype))
    wl.cache = cache
    wl.block_table = bt
    wl.lens_dev = torch.from_numpy(wl.lens.astype(np.int32)).to(dev)
    wl.budget_dev = torch.from_numpy(wl.budgets.astype(np.int32)).to(dev)
    wl.q_dev = to_torch(q, cfg.dtype).to(dev).contiguous()
    return wl
