"""Thin ctypes binding of libqasa (see include/qasa.h for every contract).

Argument marshalling only: torch tensors supply device memory and the current
CUDA stream; every step of the computation runs in the library's kernels.
Importing this module loads ``libqasa.so``; a missing library raises at once
(there is no fallback path).
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence, Tuple, Union

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libqasa.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError("libqasa.so is not built (run query_aware_sparse_append_gb300.build.build())")
_lib = ctypes.CDLL(_LIB_PATH)

DTYPE_IDS = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
E4M3 = 3            # FP8 KV: uint8 pools and boxes holding E4M3 codes, plus page_scales
STATUS_OK = 0

DEVERR = {
    0x1: "page id out of range",
    0x2: "seq_len out of range",
    0x4: "budget above max_budget",
    0x8: "bounded wait timed out",
    0x10: "append length out of range",
    0x20: "selected id out of range",
}


class _Cache(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("page_bounds", ctypes.c_void_p), ("num_phys_pages", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("page_scales", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I = ctypes.c_int32
_C = ctypes.POINTER(_Cache)
_lib.qasa_kv_append.argtypes = [_C, _P, _I, _P, _P, _P, _P, _I, _I, _P, _P]
_lib.qasa_kv_append.restype = _I
_lib.qasa_decode_workspace_size.argtypes = [_I, _I, _C, _I]
_lib.qasa_decode_workspace_size.restype = ctypes.c_size_t
_lib.qasa_select_pages.argtypes = [_C, _P, _I, _P, _I, _P, _P, _I, _P, _P, _P, ctypes.c_size_t, _I,
                                   _P, _P]
_lib.qasa_select_pages.restype = _I
_lib.qasa_sparse_attention.argtypes = [_C, _P, _I, _P, _I, _P, _P, _I, _P, ctypes.c_float, _P, _P,
                                       ctypes.c_size_t, _I, _P, _P]
_lib.qasa_sparse_attention.restype = _I
_lib.qasa_sparse_decode_attention.argtypes = [_C, _P, _I, _P, _I, _P, _P, _I, ctypes.c_float, _P,
                                              _P, _P, _P, ctypes.c_size_t, _I, _P, _P]
_lib.qasa_sparse_decode_attention.restype = _I
_lib.qasa_dense_decode_attention.argtypes = [_C, _P, _I, _P, _I, _P, ctypes.c_float, _P, _P,
                                             ctypes.c_size_t, _I, _P, _P]
_lib.qasa_dense_decode_attention.restype = _I
_lib.qasa_sparse_decode_attention_noalloc.argtypes = [_C, _P, _I, _P, _I, _P, _P, _I, ctypes.c_float,
                                                      _P, _P, _P, _I, _P, _P]
_lib.qasa_sparse_decode_attention_noalloc.restype = _I
_lib.qasa_rebuild_page_bounds.argtypes = [_C, _P, _I, _P, _I, _P, _P]
_lib.qasa_rebuild_page_bounds.restype = _I
_lib.qasa_page_attention_mass.argtypes = [_C, _P, _I, _P, _I, _P, ctypes.c_float, _P, _I, _P, _P]
_lib.qasa_page_attention_mass.restype = _I
_lib.qasa_page_hit_rate.argtypes = [_C, _P, _I, _P, _P, _I, _P, _I, _P, _P, _P, _P, _P]
_lib.qasa_page_hit_rate.restype = _I
_lib.qasa_host_decode_workspace_size.argtypes = [_I, _I, _C, _I, _I]
_lib.qasa_host_decode_workspace_size.restype = ctypes.c_size_t
_lib.qasa_sparse_decode_attention_host.argtypes = [_C, _P, _I, _P, _I, _P, _P, _I, ctypes.c_float, _P, _P, _P,
                                                   ctypes.c_size_t, _I, _P, _P]
_lib.qasa_sparse_decode_attention_host.restype = _I
_lib.qasa_host_call_is_direct.argtypes = [_P] * 6
_lib.qasa_host_call_is_direct.restype = _I
_lib.qasa_status_string.argtypes = [_I]
_lib.qasa_status_string.restype = ctypes.c_char_p
_lib.qasa_version.restype = _I
_lib.qasa_debug_trace_bytes.restype = ctypes.c_size_t
_lib.qasa_debug_trace.argtypes = [_P, ctypes.c_size_t]
_lib.qasa_debug_trace.restype = _I

EXPORTED = ("qasa_kv_append", "qasa_decode_workspace_size", "qasa_select_pages",
            "qasa_sparse_attention", "qasa_sparse_decode_attention",
            "qasa_dense_decode_attention", "qasa_sparse_decode_attention_noalloc",
            "qasa_rebuild_page_bounds", "qasa_page_attention_mass", "qasa_page_hit_rate",
            "qasa_host_decode_workspace_size", "qasa_sparse_decode_attention_host",
            "qasa_host_call_is_direct", "qasa_status_string", "qasa_version",
            "qasa_debug_trace_bytes", "qasa_debug_trace")

# trace buffer layout (include/qasa.h)
TRACE_MAX_CTAS = 4096
TRACE_SELECT_EVENTS = 4
TRACE_ATTN_EVENTS = 12


class QasaError(RuntimeError):
    pass


def library_path() -> str:
    return _LIB_PATH


def version() -> int:
    return int(_lib.qasa_version())


def debug_trace(buffer: Optional[torch.Tensor]) -> None:
    """Record per-CTA timestamps of every later selection and attention launch
    into `buffer` (a zeroed int64 device tensor of at least
    debug_trace_bytes() bytes); None turns recording off."""
    if buffer is None:
        _check(_lib.qasa_debug_trace(None, 0), "qasa_debug_trace")
        return
    _check(_lib.qasa_debug_trace(_ptr(buffer), buffer.numel() * buffer.element_size()), "qasa_debug_trace")


def debug_trace_bytes() -> int:
    return int(_lib.qasa_debug_trace_bytes())


def status_string(code: int) -> str:
    return _lib.qasa_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code != STATUS_OK:
        raise QasaError("%s failed: %s (%d)" % (what, status_string(code), code))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _contig(t: torch.Tensor, name: str) -> torch.Tensor:
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t


class PagedKVCache:
    """Device pools of one attention layer (caller-owned memory, library layout).

    k_pool, v_pool : [num_phys_pages, num_kv_heads, page_size, head_dim]
    page_bounds    : [num_phys_pages, num_kv_heads, 2, head_dim]  (lo row, hi row)
    page_scales    : FP8 KV only (uint8 pools holding E4M3 codes):
                     [num_phys_pages, num_kv_heads, 4] float32 (amax of K, amax of V, -, -);
                     queries, outputs and appended K/V are then float16
    """

    def __init__(self, k_pool: torch.Tensor, v_pool: torch.Tensor, page_bounds: torch.Tensor,
                 page_scales: Optional[torch.Tensor] = None):
        if k_pool.shape != v_pool.shape or k_pool.dim() != 4:
            raise ValueError("k_pool and v_pool must share a 4-d shape")
        n, hkv, p, d = k_pool.shape
        if tuple(page_bounds.shape) != (n, hkv, 2, d):
            raise ValueError("page_bounds must be [num_phys_pages, num_kv_heads, 2, head_dim]")
        fp8 = k_pool.dtype == torch.uint8
        if not (k_pool.dtype == v_pool.dtype == page_bounds.dtype) or not (fp8 or k_pool.dtype in DTYPE_IDS):
            raise ValueError("pools must share one of float32 / float16 / bfloat16 / uint8 (E4M3 codes)")
        if fp8:
            if page_scales is None or tuple(page_scales.shape) != (n, hkv, 4) or page_scales.dtype != torch.float32:
                raise ValueError("FP8 pools need page_scales [num_phys_pages, num_kv_heads, 4] float32")
            _contig(page_scales, "page_scales")
        for t, nm in ((k_pool, "k_pool"), (v_pool, "v_pool"), (page_bounds, "page_bounds")):
            _contig(t, nm)
        self.k_pool, self.v_pool, self.page_bounds = k_pool, v_pool, page_bounds
        self.page_scales = page_scales if fp8 else None
        self.num_phys_pages, self.num_kv_heads, self.page_size, self.head_dim = n, hkv, p, d
        self.dtype = k_pool.dtype
        self.is_fp8 = fp8
        self._c = _Cache(k_pool.data_ptr(), v_pool.data_ptr(), page_bounds.data_ptr(), n, hkv, p,
                         d, E4M3 if fp8 else DTYPE_IDS[k_pool.dtype],
                         page_scales.data_ptr() if fp8 else None)

    @classmethod
    def empty(cls, num_phys_pages: int, num_kv_heads: int, page_size: int, head_dim: int,
              dtype=torch.float16, device="cuda") -> "PagedKVCache":
        """dtype float32 / float16 / bfloat16, or torch.uint8 for FP8 (E4M3) KV."""
        shape = (num_phys_pages, num_kv_heads, page_size, head_dim)
        scales = (torch.zeros((num_phys_pages, num_kv_heads, 4), dtype=torch.float32, device=device)
                  if dtype == torch.uint8 else None)
        # K and V carved from one allocation (V right after K): the attention
        # kernel then fetches a page's K and V tiles with a single TMA box
        kv = torch.empty((2,) + shape, dtype=dtype, device=device)
        return cls(kv[0], kv[1],
                   torch.empty((num_phys_pages, num_kv_heads, 2, head_dim), dtype=dtype,
                               device=device), scales)

    @property
    def c_ref(self):
        return ctypes.byref(self._c)


def workspace_size(cache: PagedKVCache, batch: int, num_q_heads: int, max_pages_per_seq: int) -> int:
    return int(_lib.qasa_decode_workspace_size(batch, num_q_heads, cache.c_ref, max_pages_per_seq))


def alloc_workspace(cache: PagedKVCache, batch: int, num_q_heads: int, max_pages_per_seq: int,
                    device=None) -> torch.Tensor:
    n = workspace_size(cache, batch, num_q_heads, max_pages_per_seq)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device or cache.k_pool.device)


def kv_append(cache: PagedKVCache, block_table: torch.Tensor, seq_lens: torch.Tensor,
              k_new: torch.Tensor, v_new: torch.Tensor, append_lens: Optional[torch.Tensor] = None,
              status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Write k_new / v_new [B, T, Hkv, d] after seq_lens (not advanced) and update page boxes."""
    B, T = int(k_new.shape[0]), int(k_new.shape[1])
    _contig(k_new, "k_new"), _contig(v_new, "v_new"), _contig(block_table, "block_table")
    code = _lib.qasa_kv_append(cache.c_ref, _ptr(block_table), int(block_table.shape[1]),
                               _ptr(seq_lens), _ptr(append_lens), _ptr(k_new), _ptr(v_new), B, T,
                               _ptr(status), _stream(stream))
    _check(code, "qasa_kv_append")


def rebuild_page_bounds(cache: PagedKVCache, block_table: torch.Tensor, seq_lens: torch.Tensor,
                        status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Recompute every page box of the batch from the keys in the pool."""
    B = int(seq_lens.shape[0])
    code = _lib.qasa_rebuild_page_bounds(cache.c_ref, _ptr(_contig(block_table, "block_table")),
                                         int(block_table.shape[1]), _ptr(_contig(seq_lens, "seq_lens")), B,
                                         _ptr(status), _stream(stream))
    _check(code, "qasa_rebuild_page_bounds")


def budget_pages(budget: Union[int, float, torch.Tensor], seq_lens: torch.Tensor,
                 page_size: int) -> torch.Tensor:
    """Per-sequence page budget as an int32 device tensor.

    int: that many pages for every sequence.  float in (0, 1]: ceil(fraction *
    N_b) pages (needs the lengths on the host, so a device ``seq_lens`` is
    copied back).  Tensor: used as is.
    """
    if isinstance(budget, torch.Tensor):
        return budget.to(device=seq_lens.device, dtype=torch.int32).contiguous()
    if isinstance(budget, float):
        lens = seq_lens.detach().to("cpu", torch.int64).tolist()
        k = [max(1, math.ceil(budget * ((L + page_size - 1) // page_size) - 1e-9)) for L in lens]
        return torch.tensor(k, dtype=torch.int32, device=seq_lens.device)
    return torch.full((int(seq_lens.shape[0]),), int(budget), dtype=torch.int32,
                      device=seq_lens.device)


def select_pages(cache: PagedKVCache, q: torch.Tensor, block_table: torch.Tensor,
                 seq_lens: torch.Tensor, budget, max_budget: int,
                 selected: Optional[torch.Tensor] = None, scores: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    B, Hq = int(q.shape[0]), int(q.shape[1])
    bud = budget_pages(budget, seq_lens, cache.page_size)
    if selected is None:
        selected = torch.empty((B, cache.num_kv_heads, max_budget), dtype=torch.int32,
                               device=q.device)
    if workspace is None:
        workspace = alloc_workspace(cache, B, Hq, int(block_table.shape[1]))
    code = _lib.qasa_select_pages(cache.c_ref, _ptr(_contig(q, "q")), Hq, _ptr(block_table),
                                  int(block_table.shape[1]), _ptr(seq_lens), _ptr(bud), max_budget,
                                  _ptr(selected), _ptr(scores), _ptr(workspace),
                                  workspace.numel(), B, _ptr(status), _stream(stream))
    _check(code, "qasa_select_pages")
    return selected


def sparse_attention(cache: PagedKVCache, q: torch.Tensor, block_table: torch.Tensor,
                     seq_lens: torch.Tensor, budget, selected: torch.Tensor,
                     scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None,
                     status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    B, Hq = int(q.shape[0]), int(q.shape[1])
    bud = budget_pages(budget, seq_lens, cache.page_size)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = alloc_workspace(cache, B, Hq, int(block_table.shape[1]))
    code = _lib.qasa_sparse_attention(cache.c_ref, _ptr(_contig(q, "q")), Hq, _ptr(block_table),
                                      int(block_table.shape[1]), _ptr(seq_lens), _ptr(bud),
                                      int(selected.shape[-1]), _ptr(selected),
                                      float(scale or 0.0), _ptr(out), _ptr(workspace),
                                      workspace.numel(), B, _ptr(status), _stream(stream))
    _check(code, "qasa_sparse_attention")
    return out


def sparse_decode_attention(cache: PagedKVCache, q: torch.Tensor, block_table: torch.Tensor,
                            seq_lens: torch.Tensor, budget, max_budget: Optional[int] = None,
                            scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                            selected: Optional[torch.Tensor] = None,
                            scores: Optional[torch.Tensor] = None,
                            workspace: Optional[torch.Tensor] = None,
                            status: Optional[torch.Tensor] = None,
                            stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """One decode step: (out [B, Hq, d], selected [B, Hkv, max_budget] ascending, -1 padded)."""
    B, Hq = int(q.shape[0]), int(q.shape[1])
    maxp = int(block_table.shape[1])
    bud = budget_pages(budget, seq_lens, cache.page_size)
    if max_budget is None:
        max_budget = selected.shape[-1] if selected is not None else max(2, maxp)
    if out is None:
        out = torch.empty_like(q)
    if selected is None:
        selected = torch.empty((B, cache.num_kv_heads, max_budget), dtype=torch.int32,
                               device=q.device)
    if workspace is None:
        workspace = alloc_workspace(cache, B, Hq, maxp)
    code = _lib.qasa_sparse_decode_attention(cache.c_ref, _ptr(_contig(q, "q")), Hq,
                                             _ptr(block_table), maxp, _ptr(seq_lens), _ptr(bud),
                                             int(max_budget), float(scale or 0.0), _ptr(out),
                                             _ptr(selected), _ptr(scores), _ptr(workspace),
                                             workspace.numel(), B, _ptr(status), _stream(stream))
    _check(code, "qasa_sparse_decode_attention")
    return out, selected


def sparse_decode_attention_noalloc(cache: PagedKVCache, q: torch.Tensor, block_table: torch.Tensor,
                                    seq_lens: torch.Tensor, budget, max_budget: int,
                                    out: torch.Tensor, selected: torch.Tensor,
                                    scale: Optional[float] = None,
                                    scores: Optional[torch.Tensor] = None,
                                    status: Optional[torch.Tensor] = None, stream=None) -> int:
    """The decode step without a workspace, for callers that cannot allocate
    device memory: the library's fixed device buffer serves as scratch (see
    qasa.h).  The caller passes every input and output; returns the status code
    (QASA_ERR_WORKSPACE when the shape needs more scratch than the buffer)."""
    B, Hq = int(q.shape[0]), int(q.shape[1])
    bud = budget if isinstance(budget, torch.Tensor) else budget_pages(budget, seq_lens, cache.page_size)
    return int(_lib.qasa_sparse_decode_attention_noalloc(
        cache.c_ref, _ptr(_contig(q, "q")), Hq, _ptr(block_table), int(block_table.shape[1]),
        _ptr(seq_lens), _ptr(bud), int(max_budget), float(scale or 0.0), _ptr(out), _ptr(selected),
        _ptr(scores), B, _ptr(status), _stream(stream)))


def alloc_host_workspace(cache: PagedKVCache, batch: int, num_q_heads: int, max_pages_per_seq: int,
                         max_budget: int, device=None) -> torch.Tensor:
    n = int(_lib.qasa_host_decode_workspace_size(batch, num_q_heads, cache.c_ref, max_pages_per_seq, max_budget))
    if batch and not n:
        raise QasaError("unsupported shape for the host-buffer decode step")
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or cache.k_pool.device)


def sparse_decode_attention_host(cache: PagedKVCache, q_host: torch.Tensor, block_table_host: torch.Tensor,
                                 seq_lens_host: torch.Tensor, budget_host: torch.Tensor, max_budget: int,
                                 out_host: torch.Tensor, selected_host: torch.Tensor,
                                 workspace: Optional[torch.Tensor] = None, scale: Optional[float] = None,
                                 status: Optional[torch.Tensor] = None, stream=None) -> int:
    """The decode step with host (preferably pinned) inputs and outputs: the
    kernels access pinned buffers in place where the device can address them,
    else the copies and kernels are enqueued on the stream (synchronise before
    reading either way)."""
    B, Hq = int(q_host.shape[0]), int(q_host.shape[1])
    maxp = int(block_table_host.shape[1])
    if workspace is None:
        workspace = alloc_host_workspace(cache, B, Hq, maxp, max_budget)
    code = _lib.qasa_sparse_decode_attention_host(
        cache.c_ref, _ptr(_contig(q_host, "q_host")), Hq, _ptr(_contig(block_table_host, "block_table_host")), maxp,
        _ptr(_contig(seq_lens_host, "seq_lens_host")), _ptr(_contig(budget_host, "budget_host")), int(max_budget),
        float(scale or 0.0), _ptr(_contig(out_host, "out_host")), _ptr(_contig(selected_host, "selected_host")),
        _ptr(workspace), workspace.numel(), B, _ptr(status), _stream(stream))
    _check(code, "qasa_sparse_decode_attention_host")
    return code


def host_call_is_direct(q_host: torch.Tensor, block_table_host: torch.Tensor, seq_lens_host: torch.Tensor,
                        budget_host: torch.Tensor, out_host: torch.Tensor, selected_host: torch.Tensor) -> bool:
    """True when sparse_decode_attention_host with these buffers lets the
    kernels read and write them in host memory (no copies launched)."""
    return bool(_lib.qasa_host_call_is_direct(*(_ptr(t) for t in (q_host, block_table_host, seq_lens_host,
                                                                  budget_host, out_host, selected_host))))


def dense_decode_attention(cache: PagedKVCache, q: torch.Tensor, block_table: torch.Tensor,
                           seq_lens: torch.Tensor, scale: Optional[float] = None,
                           out: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None,
                           status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    B, Hq = int(q.shape[0]), int(q.shape[1])
    maxp = int(block_table.shape[1])
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = alloc_workspace(cache, B, Hq, maxp)
    code = _lib.qasa_dense_decode_attention(cache.c_ref, _ptr(_contig(q, "q")), Hq,
                                            _ptr(block_table), maxp, _ptr(seq_lens),
                                            float(scale or 0.0), _ptr(out), _ptr(workspace),
                                            workspace.numel(), B, _ptr(status), _stream(stream))
    _check(code, "qasa_dense_decode_attention")
    return out


def page_attention_mass(cache: PagedKVCache, q: torch.Tensor, block_table: torch.Tensor,
                        seq_lens: torch.Tensor, scale: Optional[float] = None,
                        mass: Optional[torch.Tensor] = None,
                        status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Share of the dense attention of each (sequence, KV head) on each page,
    [batch, num_kv_heads, max_pages_per_seq] float32 (pages >= N_b: zero when
    ``mass`` is allocated here, untouched otherwise)."""
    B, Hq = int(q.shape[0]), int(q.shape[1])
    maxp = int(block_table.shape[1])
    if mass is None:
        mass = torch.zeros((B, cache.num_kv_heads, maxp), dtype=torch.float32, device=q.device)
    code = _lib.qasa_page_attention_mass(cache.c_ref, _ptr(_contig(q, "q")), Hq, _ptr(block_table), maxp,
                                         _ptr(seq_lens), float(scale or 0.0), _ptr(_contig(mass, "mass")),
                                         B, _ptr(status), _stream(stream))
    _check(code, "qasa_page_attention_mass")
    return mass


def page_hit_rate(cache: PagedKVCache, mass: torch.Tensor, seq_lens: torch.Tensor,
                  budget_pages: torch.Tensor, selected: torch.Tensor,
                  status: Optional[torch.Tensor] = None, stream=None):
    """(hits int32, covered float32, best float32), each [batch, num_kv_heads]:
    how many selected pages are among the k_b pages of largest mass, the mass
    the selection covers and the largest mass any k_b pages cover."""
    B, Hkv, maxp = (int(x) for x in mass.shape)
    mb = int(selected.shape[2])
    hits = torch.empty((B, Hkv), dtype=torch.int32, device=mass.device)
    covered = torch.empty((B, Hkv), dtype=torch.float32, device=mass.device)
    best = torch.empty((B, Hkv), dtype=torch.float32, device=mass.device)
    code = _lib.qasa_page_hit_rate(cache.c_ref, _ptr(_contig(mass, "mass")), maxp, _ptr(seq_lens),
                                   _ptr(budget_pages), mb, _ptr(_contig(selected, "selected")), B,
                                   _ptr(hits), _ptr(covered), _ptr(best), _ptr(status), _stream(stream))
    _check(code, "qasa_page_hit_rate")
    return hits, covered, best


def decode_device_errors(code: int) -> Sequence[str]:
    return [msg for bit, msg in DEVERR.items() if code & bit]
