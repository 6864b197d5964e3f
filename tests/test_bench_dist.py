"""Host logic of the multi-GPU benchmark on CPU: world_size-2 gloo ranks.

Every rank decodes its own batch (weak scaling): distinct seeds, no data-path
collective; the only collective is the max over ranks of the step time.
"""
import json
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
from query_aware_sparse_append_gb300 import workloads as W


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.dist_env()
        local = 1.5 + 2.0 * rank               # rank 1 is the slow one
        bench.barrier()
        got = bench.max_over_ranks(local)
        seed = bench.rank_seed(7, r)
        lens = W.seq_lens(W.CONFIGS["serving_mix"], seed)
        results[rank] = (r, w, got, seed, int(lens.sum()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time_and_distinct_batches():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(results)
    assert res[0][2] == res[1][2] == 3.5
    assert res[0][1] == res[1][1] == 2
    assert res[0][3] != res[1][3] and res[0][4] != res[1][4]


def test_single_process_max_is_identity():
    assert bench.max_over_ranks(2.25) == 2.25


def test_algorithmic_bytes_of_the_headline_case():
    cfg = W.CONFIGS["headline_8k"]
    lens = W.seq_lens(cfg, 0)
    sel, att, dense = bench.algorithmic_bytes(cfg, lens, W.budgets(cfg, lens))
    # 128 sequences x 4 KV heads: 512 pages of 512-byte boxes; 64 kept 8 KiB page pairs
    units = 128 * 4
    assert sel == units * (512 * 512 + 8 * 128 * 2 + 4 * 512 + 4 * 64)
    assert att == units * (64 * 2 * 16 * 128 * 2 + 2 * 8 * 128 * 2 + 8 * 64)
    assert abs((sel + att) / 1e6 - 407.2) < 0.1
    assert dense > 5 * att


def test_selection_bytes_only_where_scores_decide():
    # one KV head, d 128, fp16, P 16: a unit that keeps every page (k >= N) or
    # only the two forced pages (k = 2) reads no boxes, query or table
    cfg = W.CONFIGS["headline_8k"]
    P, d = cfg.page_size, cfg.head_dim
    lens = [16 * P, 16 * P, 16 * P, 0]
    budgets = [16, 2, 3, 5]
    sel, att, _ = bench.algorithmic_bytes(cfg, lens, budgets)
    H = cfg.num_kv_heads
    scored = 16 * 2 * d * 2 + cfg.group * d * 2 + 4 * 16
    assert sel == H * (4 * 16 + 4 * 2 + (scored + 4 * 3) + 0)
    assert att == H * sum(k * 2 * P * d * 2 + 2 * cfg.group * d * 2 + 8 * k for k in (16, 2, 3, 0))


def test_bench_rejects_short_warmup():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_reference_arm_line(monkeypatch, capsys):
    # the reference arm is the oracle on the host cores: one JSON line with the
    # arm's metric, config and unit, a cpu_baseline describing the run and an
    # e2e with no host-device bytes (the oracle sample is replaced by a stub here)
    calls = []

    def stub(cfg, seed, seconds=15.0, threads=None):
        calls.append((cfg.name, seed, seconds))
        return {"value": 1234.5, "unit": "queries/s", "cores": 3, "kind": "oracle", "sample": "stub"}

    monkeypatch.setattr(bench, "oracle_sample", stub)
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        monkeypatch.delenv(k, raising=False)
    assert bench.main(["--impl", "reference", "--steps", "4", "--warmup", "3"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["value"] == 1234.5 and line["unit"] == "queries/s" and line["higher_is_better"] is True
    assert line["steps"] == 4 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["config"]["workload"] == "headline_8k"
    # the same config block as the GPU arm's line, key for key
    from query_aware_sparse_append_gb300 import workloads as W
    assert line["config"] == bench.config_block(W.CONFIGS["headline_8k"])
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == 1234.5
    assert line["e2e"] == {"value": 1234.5, "unit": "queries/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert calls == [("headline_8k", 0, calls[0][2])] and calls[0][2] >= 2.0 * 7

    # under torchrun only rank 0 runs and prints it
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--gpus", "2"]) == 0
    assert capsys.readouterr().out.strip() == ""
    assert len(calls) == 1


def test_kept_counts_follow_the_oracle_selection():
    # the benchmark's byte model counts the pages the selection keeps; it must
    # agree with the oracle's selection on the count for every length and budget
    import oracle
    rng = np.random.default_rng(5)
    P = 16
    lens = np.concatenate([[0, 1, 15, 16, 17, 32, 33], rng.integers(0, 4000, 60)])
    budgets = np.concatenate([[1, 1, 2, 3, 1, 2, 40], rng.integers(1, 300, 60)])
    k = bench.kept_counts(lens, budgets, P, 1 << 30)
    for L, bud, kk in zip(lens, budgets, k):
        N = oracle.num_pages(L, P)
        scores = rng.standard_normal(N)
        assert len(oracle.select_pages(scores, int(bud))) == kk, (L, bud)
