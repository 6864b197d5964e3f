"""The benchmark reports the attention kernel's ncu DRAM traffic only while the
committed summary was taken on the kernel's current source and on the same
workload: the source digest covers the code the kernel is compiled from
(comments and blank lines aside) and nothing else."""
import os
import shutil

import bench

FILES = ("attention.cu", "qasa_device.cuh", "qasa_launch.h")


def _tree(tmp_path, monkeypatch):
    src = os.path.join(bench.ROOT, "query_aware_sparse_append_gb300", "csrc")
    dst = tmp_path / "query_aware_sparse_append_gb300" / "csrc"
    dst.mkdir(parents=True)
    for n in FILES:
        shutil.copy(os.path.join(src, n), dst / n)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return dst


def _append(path, text):
    with open(path, "a") as f:
        f.write(text)


def test_digest_sees_code_but_not_comments(tmp_path, monkeypatch):
    dst = _tree(tmp_path, monkeypatch)
    d0 = bench.kernel_source_digest()
    _append(dst / "attention.cu", "\n// a remark\n/* a block\n   remark */\n\n")
    _append(dst / "qasa_device.cuh", "\n\n   // another remark\n")
    assert bench.kernel_source_digest() == d0
    _append(dst / "attention.cu", "static const int qasa_probe_constant = 1;\n")
    assert bench.kernel_source_digest() != d0


def test_digest_covers_only_the_attention_parameter_block(tmp_path, monkeypatch):
    dst = _tree(tmp_path, monkeypatch)
    d0 = bench.kernel_source_digest()
    header = (dst / "qasa_launch.h").read_text()
    i = header.index("struct AttnParams")
    # a field added to another parameter block does not reach the attention kernel
    j = header.index("struct SelectParams")
    k = header.index("{", j) + 1
    (dst / "qasa_launch.h").write_text(header[:k] + "\n    int probe_field;" + header[k:])
    assert bench.kernel_source_digest() == d0
    # one added to the attention parameters does
    k = header.index("{", i) + 1
    (dst / "qasa_launch.h").write_text(header[:k] + "\n    int probe_field;" + header[k:])
    assert bench.kernel_source_digest() != d0


def test_traffic_needs_the_current_digest_and_the_same_workload(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILE_DIR", str(tmp_path))
    d = bench.kernel_source_digest()

    def summary(recorded_workload, digest, value="123456"):
        (tmp_path / "attention_headline_8k.md").write_text(
            "# summary\n\nbench-key workload = %s\nbench-key source_digest = %s\n"
            "bench-key dram_bytes_per_launch_full_size = %s\n" % (recorded_workload, digest, value))

    assert bench.profiled_traffic("headline_8k") is None          # no summary
    summary("headline_8k", d)
    assert bench.profiled_traffic("headline_8k") == 123456
    summary("headline_8k", "0" * 16)
    assert bench.profiled_traffic("headline_8k") is None          # taken on other code
    summary("serving_mix", d)
    assert bench.profiled_traffic("headline_8k") is None          # taken on another workload
    summary("headline_8k", d, value="n/a")
    assert bench.profiled_traffic("headline_8k") is None          # unreadable figure
