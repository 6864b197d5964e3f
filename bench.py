#!/usr/bin/env python3
"""Decode-step benchmark: query-aware sparse paged attention on GB300.

One step = one decode step of one attention layer for the whole batch: score
every page of every (sequence, KV head) against its bounding box, keep the
budget, attend over the kept pages (two kernels, chained with programmatic
dependent launch).  Inputs are resident in HBM before the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Prints one JSON line (rank 0).  Multi-GPU runs (torchrun) are weak scaling:
every rank decodes its own batch (seed offset by rank); no data-path
collective exists.  --impl reference times the CPU oracle on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse decode queries/sec and HBM GB/s (% roofline) at 8K ctx, 12.5% budget"
L2_FLUSH_BYTES = 256 << 20        # written between timed steps (evicts the step's data)
L2_CLEAN_BYTES = 512 << 20        # then read, so the flush's dirty lines are written back
                                  # before the next timed step instead of during it
PROFILE_DIR = os.path.join(ROOT, "profiles")   # attention_<workload>.md: ncu summary of the attention kernel


# ------------------------------------------------------------ distributed

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def rank_seed(seed: int, rank: int) -> int:
    """Each rank decodes its own batch: weak scaling, no shared data."""
    return seed + 1000 * rank


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ------------------------------------------------------------ accounting

def algorithmic_bytes(cfg, lens, budgets):
    """Bytes the method must move per step (and per kernel), per (sequence, KV head):
    select:    N_b*2*d*es (page boxes) + G*d*qs (q) + 4*N_b (block table) + 4*k_b (ids out);
               the first three only where some page is dropped and more than the
               two forced pages are kept (elsewhere the kept set is fixed)
    attention: k_b*2*P*d*es (kept K and V page tiles) + 2*G*d*qs (q, out) + 8*k_b (ids, table)
    es = bytes per stored KV element, qs = bytes per query / output element.
    FP8 KV adds the page scales: 4*N_b (K amax) to the selection, 16*k_b (one
    16-byte scale record per kept page) to the attention.
    """
    es = {"f32": 4, "e4m3": 1}.get(cfg.dtype, 2)
    qs = 4 if cfg.dtype == "f32" else 2
    d, P, G, Hkv = cfg.head_dim, cfg.page_size, cfg.group, cfg.num_kv_heads
    N = (np.asarray(lens, np.int64) + P - 1) // P
    k = np.minimum(N, np.maximum(np.asarray(budgets, np.int64), np.minimum(N, 2)))
    f8 = cfg.dtype == "e4m3"
    # scoring (boxes, q, table) only where the scores decide the kept set
    scored = (k < N) & (k > 2)
    sel = Hkv * (np.where(scored, N * 2 * d * es + G * d * qs + 4 * N + (4 * N if f8 else 0), 0) + 4 * k)
    att = Hkv * (k * 2 * P * d * es + 2 * G * d * qs + 8 * k + (16 * k if f8 else 0))
    dense = Hkv * (N * 2 * P * d * es + 2 * G * d * qs + 4 * N + (16 * N if f8 else 0))
    return int(sel.sum()), int(att.sum()), int(dense.sum())


def rebuild_bytes(cfg, lens):
    """Algorithmic bytes of rebuilding every page box: the valid keys read once,
    the boxes written once, the block-table entries read."""
    import numpy as np
    es = {"f32": 4, "e4m3": 1}.get(cfg.dtype, 2)
    lens = np.asarray(lens, dtype=np.int64)
    n = (lens + cfg.page_size - 1) // cfg.page_size
    return int(cfg.num_kv_heads * cfg.head_dim * es * (lens.sum() + 2 * n.sum()) + 4 * n.sum())


def append_bytes(cfg, lens):
    """Algorithmic bytes of one decode-step append (one token per sequence and
    KV head): the new K and V rows read and written (4*d*es), the page box read
    and written back (4*d*es), the block-table entry and the length (8)."""
    import numpy as np
    es = {"f32": 4, "e4m3": 1}.get(cfg.dtype, 2)
    ins = 4 if cfg.dtype == "f32" else 2          # appended values arrive in the input dtype
    B = int(np.count_nonzero(np.asarray(lens) > 0))
    per = 2 * cfg.head_dim * ins + 2 * cfg.head_dim * es + 4 * cfg.head_dim * es
    if cfg.dtype == "e4m3":
        per += 2 * 16                              # the page's scale record read and written
    return int(B * cfg.num_kv_heads * per + 8 * B)


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def kernel_source_digest():
    """Digest of what the attention kernel is compiled from: attention.cu and the
    device helpers with comments and blank lines dropped, plus the AttnParams
    block of the launch header (other parameter blocks there do not reach it)."""
    import hashlib
    import re
    csrc = os.path.join(ROOT, "query_aware_sparse_append_gb300", "csrc")

    def code(text):
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
        return "\n".join(ln for ln in lines if ln.strip())

    h = hashlib.sha256()
    for name in ("attention.cu", "qasa_device.cuh"):
        with open(os.path.join(csrc, name)) as f:
            h.update(code(f.read()).encode())
    with open(os.path.join(csrc, "qasa_launch.h")) as f:
        text = f.read()
    i = text.index("struct AttnParams")
    h.update(code(text[i:text.index("};", i) + 2]).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload="headline_8k"):
    """DRAM bytes per attention launch from the committed ncu summary, if it was
    taken on the current kernel source and on this workload (else None)."""
    try:
        with open(os.path.join(PROFILE_DIR, "attention_%s.md" % workload)) as f:
            text = f.read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if line.startswith("bench-key "):
            k, _, v = line[len("bench-key "):].partition("=")
            vals[k.strip()] = v.strip()
    if vals.get("source_digest") != kernel_source_digest():
        return None
    if vals.get("workload", "headline_8k") != workload:
        return None
    try:
        return int(vals["dram_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------ clocks

class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons of one GPU
    during the timed region: NVML read-only queries through ctypes every ~2 ms
    from a thread (the region can be a few milliseconds long), else nvidia-smi.
    Nothing here changes any GPU setting."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device):
        self.device = device
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self.note = None
        self._stop = None
        self._thread = None
        self._nvml = None
        self._handle = None

    def _open_nvml(self):
        import ctypes
        import torch
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        handle = ctypes.c_void_p()
        uuid = None
        try:
            uuid = str(torch.cuda.get_device_properties(self.device).uuid)
        except (AttributeError, RuntimeError):
            pass
        ok = False
        if uuid:
            u = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            ok = lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(handle)) == 0
        if not ok:
            count = ctypes.c_uint()
            lib.nvmlDeviceGetCount_v2(ctypes.byref(count))
            if count.value != 1:
                raise OSError("cannot map the CUDA device to an NVML device")
            if lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(handle)) != 0:
                raise OSError("nvmlDeviceGetHandleByIndex failed")
        self._nvml, self._handle = lib, handle
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)

    def _poll(self):
        import ctypes
        lib, h = self._nvml, self._handle
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(float(clk.value))
            if get_reasons(h, ctypes.byref(rs)) == 0:
                for bit, name in self.REASONS.items():
                    if rs.value & bit:
                        self.reasons.add(name)
            self._stop.wait(0.002)

    def __enter__(self):
        import threading
        try:
            self._open_nvml()
        except OSError as e:
            self.note = "nvml unavailable (%s); nvidia-smi fallback" % e
            return self._enter_smi()
        self._stop = threading.Event()
        self._thread = threading.Thread(target=self._poll, daemon=True)
        self._thread.start()
        return self

    def _enter_smi(self):
        self._file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device.index), "--query-gpu=clocks.sm,clocks.max.sm,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self._file, stderr=subprocess.DEVNULL)
        except OSError:
            self._proc = None
        time.sleep(1.0)  # first sample lands before the timed region
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(2)
            try:
                self._nvml.nvmlShutdown()
            except Exception:
                pass
        elif getattr(self, "_proc", None) is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
            self._read_smi()

    def _read_smi(self):
        self._file.flush()
        with open(self._file.name) as f:
            rows = [r.split(",") for r in f.read().strip().splitlines() if r.strip()]
        os.unlink(self._file.name)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                self.samples.append(float(r[0]))
                self.max_mhz = max(self.max_mhz or 0.0, float(r[1]))
            except (ValueError, IndexError):
                continue
            for name, v in zip(names, r[2:6]):
                if v.strip().lower() == "active":
                    self.reasons.add(name)

    def summary(self):
        out = {"sm_mhz": statistics.median(self.samples) if self.samples else None,
               "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
               "samples": len(self.samples)}
        if self.note:
            out["note"] = self.note
        return out


# ------------------------------------------------------------ CPU oracle leg

def oracle_sample(cfg, seed, seconds=15.0, threads=None):
    """Time the CPU oracle (as it stands) on (sequence, KV head) units of the
    workload until `seconds` of work are done; returns queries/s and details.
    Page boxes are built outside the timing, as the GPU path keeps them at
    append time; the timed part is score + select + attend per unit."""
    import oracle
    from query_aware_sparse_append_gb300 import workloads as W
    threads = threads or os.cpu_count() or 1
    oracle.build()
    lens = W.seq_lens(cfg, seed)
    bud = W.budgets(cfg, lens)
    scales = W.key_channel_scales(cfg, seed)
    G, P = cfg.group, cfg.page_size
    units = []
    b = 0
    t_prep = time.time()
    while b < cfg.batch and (len(units) < 4 * threads or time.time() - t_prep < min(5.0, seconds / 3)):
        s = W.sequence(cfg, b, int(lens[b]), seed, scales)
        for h in range(cfg.num_kv_heads):
            K = W.widen(s.k[:, h], cfg.dtype)
            V = W.widen(s.v[:, h], cfg.dtype)
            q = W.widen(s.q[h * G:(h + 1) * G], cfg.dtype)
            if cfg.dtype == "e4m3":      # the cache's codes and scales, as one append writes them
                L = int(lens[b])
                tok = np.arange(L) // P
                kc, ka, klo, khi = oracle.fp8_append_replay(K.astype(np.float32), P, [L])
                vc, va, _, _ = oracle.fp8_append_replay(V.astype(np.float32), P, [L])
                sk, sv = oracle.fp8_scale(ka), oracle.fp8_scale(va)
                K, V = oracle.fp8_dequant(kc, sk[tok]), oracle.fp8_dequant(vc, sv[tok])
                lo, hi = oracle.fp8_dequant(klo, sk), oracle.fp8_dequant(khi, sk)
            else:
                lo, hi = oracle.page_bounds(K, P)
            units.append((q, K, V, lo, hi, int(lens[b]), int(bud[b])))
        b += 1

    def one(u):
        q, K, V, lo, hi, L, k = u
        oracle.decode_unit(q, K, V, lo, hi, L, P, k)
        return 1

    done = 0
    t0 = time.perf_counter()
    while True:
        oracle.run_units(one, units, threads=threads)
        done += len(units)
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    qps = done / cfg.num_kv_heads / el
    # the same units on one core, for a fifth of the time
    done1 = 0
    t1 = time.perf_counter()
    while time.perf_counter() - t1 < seconds / 5:
        one(units[done1 % len(units)])
        done1 += 1
    el1 = time.perf_counter() - t1
    return {"value": qps, "unit": "queries/s", "cores": threads, "kind": "oracle",
            "sample": "%d (sequence, KV head) units of %s (%d sequences) repeated for %.1f s; "
                      "score+select+attend per unit, fp64, page boxes prebuilt"
                      % (done, cfg.name, b, el),
            "single_thread": {"value": done1 / cfg.num_kv_heads / el1, "unit": "queries/s", "cores": 1,
                              "sample": "%d units in %.1f s" % (done1, el1)}}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    from query_aware_sparse_append_gb300 import workloads as W
    cfg = W.CONFIGS[args.config]
    if args.batch:
        cfg = cfg.with_batch(args.batch)
    per_step = max(2.0, 30.0 / max(1, args.steps + args.warmup))
    base = oracle_sample(cfg, args.seed, seconds=per_step * (args.steps + args.warmup))
    v = base["value"]
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "queries/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * cfg.batch / v, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_block(cfg), "cpu_baseline": base,
            "ms_per_step_method": "batch / the sampled rate: the oracle decodes (sequence, KV head) units "
                                  "of this workload for about (steps + warmup) * %.1f s; no per-step timing"
                                  % per_step,
            "e2e": {"value": v, "unit": "queries/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_block(cfg):
    """The workload as both arms describe it (identical keys and values)."""
    return {"workload": cfg.name, "batch": cfg.batch, "ctx": [cfg.ctx_min, cfg.ctx_max],
            "num_q_heads": cfg.num_q_heads, "num_kv_heads": cfg.num_kv_heads,
            "head_dim": cfg.head_dim, "page_size": cfg.page_size,
            "budget": ("%g%% of pages" % (cfg.budget_value / 10.0)
                       if cfg.budget_kind == "permille" else "%d pages" % cfg.budget_value),
            "kv_dtype": cfg.dtype, "physical_pages": "shuffled",
            "l2": "between timed steps a 256 MB write evicts L2, then a 512 MB read leaves it "
                  "clean; the step's bytes also exceed L2"}


# ------------------------------------------------------------ GPU leg

def kept_counts(lens, budgets, page_size, max_budget):
    """Pages kept per sequence (the selection's rule: every page when the budget
    reaches the page count, else max(budget, the forced sink and newest pages))."""
    import numpy as np
    n = (np.asarray(lens, dtype=np.int64) + page_size - 1) // page_size
    b = np.asarray(budgets, dtype=np.int64)
    k = np.where(b >= n, n, np.maximum(b, np.minimum(n, 2)))
    return np.minimum(k, max_budget)


def hit_rate_stats(qasa, wl, budget_dev, budgets, max_budget, sel, mass=None):
    """Page hit rate of the GPU selection against the dense attention mass, both
    computed by the library's kernels.  Returns the summary dict of the JSON line."""
    import numpy as np
    import torch
    cfg = wl.cfg
    qasa.sparse_decode_attention(wl.cache, wl.q_dev, wl.block_table, wl.lens_dev, budget_dev,
                                 max_budget=max_budget, selected=sel)
    mass = qasa.page_attention_mass(wl.cache, wl.q_dev, wl.block_table, wl.lens_dev, mass=mass)
    hits, cov, best = qasa.page_hit_rate(wl.cache, mass, wl.lens_dev, budget_dev, sel)
    torch.cuda.synchronize()
    k = kept_counts(wl.lens, budgets, cfg.page_size, max_budget)
    kk = np.repeat(k[:, None], cfg.num_kv_heads, axis=1).astype(np.float64)
    h, c, b = (x.cpu().numpy().astype(np.float64) for x in (hits, cov, best))
    live = kk > 0
    n = (np.asarray(wl.lens, dtype=np.int64) + cfg.page_size - 1) // cfg.page_size
    return {
        "hit_rate": float(h[live].sum() / kk[live].sum()),
        "covered_mass": float(c[live].mean()),
        "best_mass": float(b[live].mean()),
        "covered_over_best": float((c[live] / np.maximum(b[live], 1e-30)).mean()),
        "kept_fraction": float(k.sum() / max(n.sum(), 1)),
        "units": int(live.sum()),
    }


def run_hit_rate_table(args):
    """One JSON line per (workload, budget): the page hit rate of the selection
    against the dense attention mass, on the synthetic workloads."""
    import numpy as np
    import torch
    from query_aware_sparse_append_gb300 import build
    build.build()
    from query_aware_sparse_append_gb300 import binding as qasa
    from query_aware_sparse_append_gb300 import paged
    from query_aware_sparse_append_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    names = [args.config] if args.config != "all" else list(W.CONFIGS)
    for name in names:
        cfg = W.CONFIGS[name]
        if args.batch:
            cfg = cfg.with_batch(args.batch)
        wl = paged.load(paged.generate(cfg, seed=args.seed), device=dev)
        n = W.num_pages(wl.lens, cfg.page_size).astype(np.int64)
        sweeps = [("own", wl.budgets)] + [
            ("%d permille" % pm, np.maximum((n * pm + 999) // 1000, 1).astype(np.int32))
            for pm in (50, 125, 250, 500)]
        for label, bud in sweeps:
            mb = max(2, int(kept_counts(wl.lens, bud, cfg.page_size, 1 << 30).max()))
            sel = torch.empty((cfg.batch, cfg.num_kv_heads, mb), dtype=torch.int32, device=dev)
            bud_dev = torch.from_numpy(np.ascontiguousarray(bud, dtype=np.int32)).to(dev)
            st = hit_rate_stats(qasa, wl, bud_dev, bud, mb, sel)
            print(json.dumps({"workload": name, "budget": label, "planted_pages": bool(
                cfg.planted_count or cfg.planted_permille), **st}), flush=True)
        del wl
        torch.cuda.empty_cache()
    return 0


def trace_summary(buf, qasa, sel_ctas, att_ctas, raw=False):
    """Percentiles (us, from the earliest recorded stamp) of every trace event
    over the CTAs that recorded it."""
    import numpy as np
    t = buf.cpu().numpy().astype(np.int64)
    nsel = qasa.TRACE_MAX_CTAS * qasa.TRACE_SELECT_EVENTS
    sel = t[:nsel].reshape(qasa.TRACE_MAX_CTAS, qasa.TRACE_SELECT_EVENTS)[:sel_ctas]
    sel = sel[sel[:, 0] > 0]   # CTAs that ran
    att = t[nsel:].reshape(qasa.TRACE_MAX_CTAS, qasa.TRACE_ATTN_EVENTS)[:att_ctas]
    ts, ta = sel[:, :3], np.concatenate([att[:, :8], att[:, 9:11]], axis=1)   # time stamps (not SM ids)
    rec = np.concatenate([ts[ts > 0], ta[ta > 0]])
    if rec.size == 0:
        return {}
    t0 = rec.min()
    names_s = ["start", "scored", "ids_written"]
    names_a = ["start", "prologue_done", "dependency_wait_done", "first_copy_issued", "first_page_consumed",
               "last_copy_issued", "consumers_done", "combiner_done", None, "last_states",
               "last_merged", None]
    out = {}
    for pre, arr, names in (("select.", sel, names_s), ("attn.", att, names_a)):
        for j, nm in enumerate(names):
            if nm is None:
                continue
            v = arr[:, j]
            v = v[v > 0]
            if v.size:
                q = np.percentile((v - t0) / 1000.0, [0, 50, 100])
                out[pre + nm] = [round(float(x), 2) for x in q]
    if raw:
        # per CTA, in launch order: every event (us from t0, null when not reached) and its SM
        def us(a):
            return [round(float((x - t0) / 1000.0), 2) if x > 0 else None for x in a]
        out["raw"] = {"select_sm": sel[:, 3].tolist(), "attn_sm": att[:, 8].tolist()}
        for pre, arr, names in (("select.", sel, names_s), ("attn.", att, names_a)):
            for j, nm in enumerate(names):
                if nm is not None:
                    out["raw"][pre + nm] = us(arr[:, j])
    return out


def run_trace(args):
    """Per-CTA timelines of the decode step's kernels (globaltimer stamps),
    one JSON line per repetition: [min, median, max] over CTAs, in us from the
    first recorded stamp of the step."""
    import torch
    from query_aware_sparse_append_gb300 import build
    build.build()
    from query_aware_sparse_append_gb300 import binding as qasa
    from query_aware_sparse_append_gb300 import paged
    from query_aware_sparse_append_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    cfg = W.CONFIGS[args.config]
    if args.batch:
        cfg = cfg.with_batch(args.batch)
    wl = paged.load(paged.generate(cfg, seed=args.seed), device=dev)
    B, Hq, Hkv = cfg.batch, cfg.num_q_heads, cfg.num_kv_heads
    maxp = wl.block_table.shape[1]
    ws = qasa.alloc_workspace(wl.cache, B, Hq, maxp, device=dev)
    out = torch.empty_like(wl.q_dev)
    sel = torch.empty((B, Hkv, wl.max_budget), dtype=torch.int32, device=dev)
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(L2_CLEAN_BYTES // 4, dtype=torch.int32, device=dev)
    buf = torch.zeros(qasa.debug_trace_bytes() // 8, dtype=torch.int64, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    def step():
        qasa.sparse_decode_attention(wl.cache, wl.q_dev, wl.block_table, wl.lens_dev, wl.budget_dev,
                                     max_budget=wl.max_budget, out=out, selected=sel, workspace=ws)

    for _ in range(args.warmup):
        step()
    for rep in range(args.steps):
        flush_w.zero_()
        flush_r.sum()
        buf.zero_()
        torch.cuda.synchronize(dev)
        qasa.debug_trace(buf)
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        step()
        b_.record()
        torch.cuda.synchronize(dev)
        qasa.debug_trace(None)
        line = {"trace": cfg.name, "rep": rep, "step_us": a.elapsed_time(b_) * 1000.0,
                "form": "one launch" if os.environ.get("QASA_SINGLE_LAUNCH") == "1" else "two launches",
                **trace_summary(buf, qasa, qasa.TRACE_MAX_CTAS, sms, raw=args.trace_raw)}
        print(json.dumps(line), flush=True)
    return 0


def time_steps(fn, steps, flush, stream):
    """Mean CUDA-event time (ms) of `steps` calls of fn, L2 flushed before each."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b_ in ev:
        flush()
        a.record(stream)
        fn()
        b_.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b_) for a, b_ in ev)


def measure_per_config(args, qasa, paged, W, dev, seed, status, with_cpu):
    """The decode step (two launches) and the dense path on the other
    workloads, and on the serving mix at every budget of its sweep: time per
    step, queries/s, algorithmic bytes and their fraction of the measured HBM
    peak, next to the oracle's queries/s on a bounded sample."""
    import numpy as np
    import torch
    peak, _ = measured_peak()
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(L2_CLEAN_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    steps = max(5, args.steps // 2)

    def flush():
        flush_w.zero_()
        flush_r.sum()

    def entry(wcfg, wl, lens, bud, label):
        maxp = wl.block_table.shape[1]
        bud = np.asarray(bud, dtype=np.int32)
        mb = max(2, int(kept_counts(lens, bud, wcfg.page_size, 1 << 30).max()))
        bud_dev = torch.from_numpy(bud).to(dev)
        ws = qasa.alloc_workspace(wl.cache, wcfg.batch, wcfg.num_q_heads, maxp, device=dev)
        out = torch.empty_like(wl.q_dev)
        sel = torch.empty((wcfg.batch, wcfg.num_kv_heads, mb), dtype=torch.int32, device=dev)

        def step():
            qasa.sparse_decode_attention(wl.cache, wl.q_dev, wl.block_table, wl.lens_dev, bud_dev,
                                         max_budget=mb, out=out, selected=sel, workspace=ws, status=status)

        def dense():
            qasa.dense_decode_attention(wl.cache, wl.q_dev, wl.block_table, wl.lens_dev, out=out,
                                        workspace=ws, status=status)

        for _ in range(3):
            step()
            dense()
        ms = time_steps(step, steps, flush, stream)
        dms = time_steps(dense, max(3, steps // 2), flush, stream)
        sb, ab, db = algorithmic_bytes(wcfg, lens, bud)
        e = {"workload": label, "batch": wcfg.batch, "kv_dtype": wcfg.dtype,
             "us_per_step": 1000.0 * ms, "queries_per_s": wcfg.batch / (ms * 1e-3),
             "algorithmic_bytes": sb + ab, "achieved_gbs": (sb + ab) / (ms * 1e-3) / 1e9,
             "frac_of_peak": (sb + ab) / (ms * 1e-3) / 1e9 / peak,
             "kept_fraction": float(kept_counts(lens, bud, wcfg.page_size, 1 << 30).sum() /
                                    max(1, W.num_pages(lens, wcfg.page_size).sum())),
             "dense": {"us_per_step": 1000.0 * dms, "queries_per_s": wcfg.batch / (dms * 1e-3),
                       "algorithmic_bytes": db, "frac_of_peak": db / (dms * 1e-3) / 1e9 / peak}}
        if with_cpu and args.cpu_seconds > 0:
            c = oracle_sample(wcfg, seed, seconds=max(1.0, args.cpu_seconds / 10))
            e["oracle"] = {"queries_per_s": c["value"], "cores": c["cores"], "sample": c["sample"]}
        return e

    out = {}
    for name in ("tiny", "tinyllama", "gpt2_345m", "llama_1b3_32k"):
        wcfg = W.CONFIGS[name]
        wl = paged.load(paged.generate(wcfg, seed=seed), device=dev)
        out[name] = entry(wcfg, wl, wl.lens, wl.budgets, name)
        del wl
        torch.cuda.empty_cache()
    mcfg = W.CONFIGS["serving_mix"]
    wl = paged.load(paged.generate(mcfg, seed=seed), device=dev)
    for pm in W.SERVING_MIX_BUDGETS_PERMILLE:
        bcfg = mcfg.with_budget("permille", pm)
        bud = W.budgets(bcfg, wl.lens)
        out["serving_mix@%d" % pm] = entry(bcfg, wl, wl.lens, bud,
                                           "serving_mix (ragged 512..16384, %g %% budget)" % (pm / 10.0))
    del wl
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, local_rank, world = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)

    from query_aware_sparse_append_gb300 import build
    build.build()
    from query_aware_sparse_append_gb300 import binding as qasa
    from query_aware_sparse_append_gb300 import paged
    from query_aware_sparse_append_gb300 import workloads as W

    cfg = W.CONFIGS[args.config]
    if args.batch:
        cfg = cfg.with_batch(args.batch)
    seed = rank_seed(args.seed, rank)
    wl = paged.load(paged.generate(cfg, seed=seed), device=dev)
    B, Hq, Hkv, d = cfg.batch, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim
    maxp = wl.block_table.shape[1]
    max_budget = wl.max_budget
    ws = qasa.alloc_workspace(wl.cache, B, Hq, maxp, device=dev)
    out = torch.empty_like(wl.q_dev)
    sel = torch.empty((B, Hkv, max_budget), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(L2_CLEAN_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    class _Flush:
        @staticmethod
        def zero_():
            flush_w.zero_()
            flush_r.sum()

    flush = _Flush()

    def step():
        qasa.sparse_decode_attention(wl.cache, wl.q_dev, wl.block_table, wl.lens_dev,
                                     wl.budget_dev, max_budget=max_budget, out=out,
                                     selected=sel, workspace=ws, status=status)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)

    # ---- timed region: K fused decode steps, L2 flushed before each
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with ClockSampler(dev) as clocks:
        barrier(dev)
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        barrier(dev)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = statistics.mean(step_ms)
    ms_all = max_over_ranks(ms, dev)
    st = int(status.item())
    if st:
        raise SystemExit("device errors during the benchmark: %s" % qasa.decode_device_errors(st))

    # ---- the same step launched from a CUDA graph (captured once): the device
    # time without the host's launch path between the start event and the first
    # kernel
    graph_ms = None
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            step()
            torch.cuda.synchronize(dev)
            with torch.cuda.graph(g, stream=cap):
                step()
        torch.cuda.synchronize(dev)
        for _ in range(3):
            g.replay()
        evg = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a, b_ in evg:
            flush.zero_()
            a.record(stream)
            g.replay()
            b_.record(stream)
        torch.cuda.synchronize(dev)
        graph_ms = statistics.mean(a.elapsed_time(b_) for a, b_ in evg)
        del g
    except Exception:   # capture refused: no graph figure
        graph_ms = None

    # ---- per-kernel breakdown (same inputs, the two kernels as separate calls)
    ev3 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        ev3[i][0].record(stream)
        qasa.select_pages(wl.cache, wl.q_dev, wl.block_table, wl.lens_dev, wl.budget_dev,
                          max_budget, selected=sel, workspace=ws, status=status)
        ev3[i][1].record(stream)
        qasa.sparse_attention(wl.cache, wl.q_dev, wl.block_table, wl.lens_dev, wl.budget_dev, sel,
                              out=out, workspace=ws, status=status)
        ev3[i][2].record(stream)
    torch.cuda.synchronize(dev)
    sel_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev3)
    att_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev3)

    # ---- the same step in the other form (one cooperative launch <-> two launches)
    single = os.environ.get("QASA_SINGLE_LAUNCH", "0") == "1"
    os.environ["QASA_SINGLE_LAUNCH"] = "0" if single else "1"
    try:
        for _ in range(3):
            step()
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a, b_ in ev2:
            flush.zero_()
            a.record(stream)
            step()
            b_.record(stream)
        torch.cuda.synchronize(dev)
    finally:
        os.environ["QASA_SINGLE_LAUNCH"] = "1" if single else "0"
    other_ms = statistics.mean(a.elapsed_time(b_) for a, b_ in ev2)

    # ---- dense path (every page), for comparison
    dense_out = torch.empty_like(out)
    evd = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(max(3, args.steps // 2))]
    for a, b_ in evd:
        flush.zero_()
        a.record(stream)
        qasa.dense_decode_attention(wl.cache, wl.q_dev, wl.block_table, wl.lens_dev,
                                    out=dense_out, workspace=ws, status=status)
        b_.record(stream)
    torch.cuda.synchronize(dev)
    dense_ms = statistics.mean(a.elapsed_time(b_) for a, b_ in evd)

    # ---- page hit rate of the selection against the dense attention mass
    # (measured on 16/32-bit caches only)
    hit = hit_rate_stats(qasa, wl, wl.budget_dev, wl.budgets, max_budget, sel) if cfg.dtype != "e4m3" else None

    # ---- one decode-step append (T = 1 per sequence): every sequence's newest
    # token written again at its own position (identical K/V, so the cache and
    # its boxes do not change); L2 flushed before each call
    import numpy as np
    lens_m1 = (wl.lens_dev - 1).clamp(min=0).contiguous()
    kl = np.stack([sq.k[max(int(L) - 1, 0):max(int(L), 1)] for sq, L in zip(wl.seqs, wl.lens)])
    vl = np.stack([sq.v[max(int(L) - 1, 0):max(int(L), 1)] for sq, L in zip(wl.seqs, wl.lens)])
    one_tok = (wl.lens_dev > 0).to(torch.int32).contiguous()   # empty sequences append nothing
    k1 = paged.to_torch(kl, cfg.dtype).to(dev).contiguous()
    v1 = paged.to_torch(vl, cfg.dtype).to(dev).contiguous()
    eva = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(6)]
    for a, b_ in eva:
        flush.zero_()
        a.record(stream)
        qasa.kv_append(wl.cache, wl.block_table, lens_m1, k1, v1, append_lens=one_tok, status=status)
        b_.record(stream)
    torch.cuda.synchronize(dev)
    append_ms = statistics.mean(a.elapsed_time(b_) for a, b_ in eva[1:])

    # ---- bulk rebuild of every page box from the pool (same boxes written back)
    evr = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(5)]
    for a, b_ in evr:
        flush.zero_()
        a.record(stream)
        qasa.rebuild_page_bounds(wl.cache, wl.block_table, wl.lens_dev, status=status)
        b_.record(stream)
    torch.cuda.synchronize(dev)
    rebuild_ms = statistics.mean(a.elapsed_time(b_) for a, b_ in evr[1:])

    # ---- end to end through the C-ABI host-buffer call: per step, q, block
    # table, lengths and budgets come from pinned host memory and the output and
    # kept ids go back to it.  Direct form (the default where the device can
    # address the pinned buffers): the kernels read and write host memory over
    # the CPU-GPU link themselves.  Staged form (QASA_HOST_DIRECT=0): H2D copies,
    # the decode step, D2H copies.  Both are timed; e2e.value is the default.
    q_h = wl.q_dev.cpu().pin_memory()
    lens_h = wl.lens_dev.cpu().pin_memory()
    bud_h = wl.budget_dev.cpu().pin_memory()
    bt_h = wl.block_table.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    sel_h = torch.empty(sel.shape, dtype=sel.dtype).pin_memory()
    host_ws = qasa.alloc_host_workspace(wl.cache, B, Hq, maxp, max_budget, device=dev)

    def time_host_call(direct):
        old = os.environ.get("QASA_HOST_DIRECT")
        os.environ["QASA_HOST_DIRECT"] = "1" if direct else "0"
        try:
            form = "direct" if qasa.host_call_is_direct(q_h, bt_h, lens_h, bud_h, out_h, sel_h) else "staged"

            def e2e_step():
                qasa.sparse_decode_attention_host(wl.cache, q_h, bt_h, lens_h, bud_h, max_budget, out_h, sel_h,
                                                  workspace=host_ws, status=status)

            for _ in range(2):
                e2e_step()
            torch.cuda.synchronize(dev)
            eager = []
            for _ in range(args.steps):
                flush.zero_()
                torch.cuda.synchronize(dev)
                t0 = time.perf_counter()
                e2e_step()
                torch.cuda.synchronize(dev)
                eager.append(1000.0 * (time.perf_counter() - t0))
            # the same call captured once in a CUDA graph (copies and kernels are
            # all stream work; the host buffers stay fixed, a server rewrites them
            # per step)
            mode = "eager"
            try:
                graph = torch.cuda.CUDAGraph()
                cap = torch.cuda.Stream(dev)
                cap.wait_stream(torch.cuda.current_stream(dev))
                with torch.cuda.stream(cap):
                    e2e_step()               # warm the capture stream
                    torch.cuda.synchronize(dev)
                    with torch.cuda.graph(graph, stream=cap):
                        e2e_step()
                torch.cuda.synchronize(dev)
                for _ in range(2):
                    graph.replay()
                torch.cuda.synchronize(dev)
                e2e_step = graph.replay
                mode = "cuda_graph"
            except Exception as exc:         # capture refused: keep the eager number
                mode = "eager (graph capture failed: %s)" % str(exc).splitlines()[0][:120]
            ms = []
            for _ in range(args.steps):
                flush.zero_()
                torch.cuda.synchronize(dev)
                t0 = time.perf_counter()
                e2e_step()
                torch.cuda.synchronize(dev)
                ms.append(1000.0 * (time.perf_counter() - t0))
            return {"transfer": form, "mode": mode, "ms_per_step": max_over_ranks(statistics.mean(ms), dev),
                    "eager_ms_per_step": statistics.mean(eager)}
        finally:
            if old is None:
                del os.environ["QASA_HOST_DIRECT"]
            else:
                os.environ["QASA_HOST_DIRECT"] = old

    e2e_staged = time_host_call(False)
    e2e_default = time_host_call(os.environ.get("QASA_HOST_DIRECT", "1") != "0")
    e2e_mean = e2e_default["ms_per_step"]
    h2d = sum(x.numel() * x.element_size() for x in (q_h, lens_h, bud_h, bt_h))
    d2h = out_h.numel() * out_h.element_size() + sel_h.numel() * sel_h.element_size()

    # ---- every other workload of the method's configurations, and the serving
    # mix at each budget of its sweep, reported next to the headline (each a
    # short timed loop; the oracle on a bounded sample of the same workload)
    per_config = None
    if args.per_config and cfg.name == "headline_8k":
        del ws, flush_w, flush_r
        torch.cuda.empty_cache()
        per_config = measure_per_config(args, qasa, paged, W, dev, seed, status, rank == 0)

    if rank != 0:
        return 0
    sel_b, att_b, dense_b = algorithmic_bytes(cfg, wl.lens, wl.budgets)
    rebuild_b = rebuild_bytes(cfg, wl.lens)
    peak, peak_kind = measured_peak()
    att_gbs = att_b / (att_ms * 1e-3) / 1e9
    step_gbs = (sel_b + att_b) / (ms * 1e-3) / 1e9
    cpu = oracle_sample(cfg, seed, seconds=args.cpu_seconds) if args.cpu_seconds > 0 else None
    line = {
        "metric": METRIC,
        "value": world * B / (ms_all * 1e-3),
        "unit": "queries/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_all,
        "ms_per_step_median": max_over_ranks(statistics.median(step_ms), dev),
        "per_head_queries_per_s": world * B * Hq / (ms_all * 1e-3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": cfg.dtype, "data": "synthetic",
        "config": config_block(cfg),
        "roofline": {"bound": "hbm", "kernel": "attn_kernel (sparse attention over kept pages)",
                     "achieved": att_gbs, "peak": peak, "unit": "GB/s",
                     "frac": att_gbs / peak, "traffic": profiled_traffic(cfg.name),
                     "algorithmic_bytes_per_launch": att_b, "ms_per_launch": att_ms,
                     "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_kind
                     if peak_kind == "measured" else "fallback 6.8 TB/s"},
        "step_hbm": {"achieved_gbs": step_gbs, "frac": step_gbs / peak,
                     "algorithmic_bytes": sel_b + att_b},
        "kernels_ms": {"select_pages": sel_ms, "sparse_attention": att_ms,
                       "select_gbs": sel_b / (sel_ms * 1e-3) / 1e9},
        "step_graph": ({"ms_per_step": graph_ms, "queries_per_s": B / (graph_ms * 1e-3),
                        "note": "the same step replayed from a CUDA graph (L2 flushed before each)"}
                       if graph_ms else None),
        "step_form": "one cooperative launch (score + select + attend)" if single
                     else "two launches (select, then attention)",
        ("two_launch_step" if single else "single_launch_step"):
            {"ms_per_step": other_ms, "queries_per_s": B / (other_ms * 1e-3)},
        "dense": {"ms_per_step": dense_ms, "queries_per_s": B / (dense_ms * 1e-3),
                  "achieved_gbs": dense_b / (dense_ms * 1e-3) / 1e9,
                  "frac": dense_b / (dense_ms * 1e-3) / 1e9 / peak,
                  "speedup_sparse_over_dense": dense_ms / ms},
        "page_hit_rate": hit,
        "serving_mix": (per_config or {}).get("serving_mix@125"),
        "per_config": per_config,
        "decode_append": {"us": 1000.0 * append_ms, "bytes": append_bytes(cfg, wl.lens),
                          "achieved_gbs": append_bytes(cfg, wl.lens) / (append_ms * 1e-3) / 1e9,
                          "frac": append_bytes(cfg, wl.lens) / (append_ms * 1e-3) / 1e9 / peak,
                          "note": "one new token per sequence (T = 1): launch-latency bound"},
        "metadata_rebuild": {"ms": rebuild_ms, "bytes": rebuild_b,
                             "achieved_gbs": rebuild_b / (rebuild_ms * 1e-3) / 1e9,
                             "frac": rebuild_b / (rebuild_ms * 1e-3) / 1e9 / peak},
        "cpu_baseline": cpu,
        "e2e": {"value": world * B / (e2e_mean * 1e-3), "unit": "queries/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, **e2e_default,
                "staged": {**e2e_staged, "queries_per_s": world * B / (e2e_staged["ms_per_step"] * 1e-3)}},
        "gpu_launches": (1 if single else 2) * args.steps,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="headline_8k")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (smaller cases for profiling)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-per-config", "--no-serving-mix", dest="per_config", action="store_false",
                    help="skip the other workloads and the serving-mix budget sweep reported beside the headline")
    ap.add_argument("--hit-rate-table", action="store_true",
                    help="print the page hit rate per workload (--config all) and budget, then exit")
    ap.add_argument("--trace", action="store_true",
                    help="print per-CTA kernel timelines of the decode step (diagnostics), then exit")
    ap.add_argument("--trace-raw", action="store_true",
                    help="with --trace: also print every CTA's events and SM")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="seconds of oracle work for the cpu_baseline (0 to skip)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.hit_rate_table:
        return run_hit_rate_table(args)
    if args.trace:
        return run_trace(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
