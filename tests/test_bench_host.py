"""Host logic of bench.py that needs no GPU: the kernel-source hash that decides whether the
committed ncu traffic figure still describes the kernel, and the reading of that figure."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _sources():
    d = os.path.join(ROOT, "tensor_sharded_linear_bias_gb300", "csrc")
    return {f: open(os.path.join(d, f)).read() for f in bench.KERNEL_SOURCES}


def test_hash_ignores_comments_and_blank_lines():
    src = _sources()
    base = bench.kernel_source_hash(lambda f: src[f])
    assert base == bench.kernel_source_hash()
    f0 = bench.KERNEL_SOURCES[0]
    edited = dict(src)
    edited[f0] = "// a new comment line\n\n" + src[f0].replace("\n", "  // trailing note\n", 3)
    assert bench.kernel_source_hash(lambda f: edited[f]) == base


def test_hash_follows_code_changes():
    src = _sources()
    base = bench.kernel_source_hash(lambda f: src[f])
    f1 = bench.KERNEL_SOURCES[1]
    edited = dict(src)
    edited[f1] = src[f1] + "\nconstexpr int kUnusedForTheTest = 1;\n"
    assert bench.kernel_source_hash(lambda f: edited[f]) != base


def test_traffic_read_only_for_the_kernel_it_was_taken_on(monkeypatch):
    """The committed ncu summary's DRAM traffic is reported only while its kernel_source_sha
    equals the current code's hash, and only for its own workload."""
    fields = {}
    for line in open(bench.PROFILE_SUMMARY):
        if line.startswith("- ") and ":" in line:
            k, v = line[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    name = fields["workload"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda read=None: fields["kernel_source_sha"])
    assert bench.profiled_traffic(name) == float(fields["dram_bytes_per_launch"])
    assert bench.profiled_traffic(name + "_other") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda read=None: "0" * 16)
    assert bench.profiled_traffic(name) is None
