"""Host logic of bench.py that needs no GPU: the DRAM traffic of a kernel is reported only while its
sources are the ones the committed ncu counters were taken on, the recorded figures are self-consistent,
and the whole-job throughput counts every replica's tokens; the CPU-baseline sample runs for every
workload kind."""
import os
import re
import sys
from dataclasses import replace

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

TRAFFIC = os.path.join(ROOT, "profiles", "dram_traffic.txt")


def _lines():
    return [l.split() for l in open(TRAFFIC) if l.strip() and not l.startswith("#")]


def test_traffic_file_is_well_formed():
    kernels = {k for k, _ in bench.KERNELS.values()} | {"decode_step_kernel"}
    for parts in _lines():
        assert len(parts) == 6, parts
        kernel, workload, digest, total, rd, wr = parts
        assert kernel in kernels, kernel
        assert re.fullmatch(r"[0-9a-f]{16}", digest), digest
        assert int(total) == int(rd) + int(wr) and int(rd) > 0


def test_traffic_is_reported_only_for_the_recorded_sources():
    kernel, workload, digest, total = _lines()[0][:4]
    assert bench.measured_traffic(kernel, workload, digest) == int(total)
    other = format(int(digest, 16) ^ 1, "016x")
    assert bench.measured_traffic(kernel, workload, other) is None
    assert bench.measured_traffic(kernel, "no_such_workload", digest) is None


def test_source_digest_follows_the_files():
    files = bench.KERNELS[("dense", "fwd")][1]
    d = bench.kernel_source_digest(files)
    assert re.fullmatch(r"[0-9a-f]{16}", d)
    assert d == bench.kernel_source_digest(list(files))
    assert d != bench.kernel_source_digest(files[:1])


def test_whole_job_throughput_counts_every_replica():
    # 4 replicas of 16384 tokens, 10 steps in 2 ms of the slowest rank's time
    assert abs(bench.whole_job_tokens_per_s(4, 16384, 10, 2.0) - 4 * 16384 * 10 / 2e-3) < 1e-6
    assert bench.max_over_ranks(3.5, 1, None) == 3.5


def test_peaks_fall_back_to_the_stated_figures_without_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peaks() == (6800.0, 1900.0, 1700.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6783.1, "bf16_tflops": 1883.2}')
    assert bench.peaks() == (6783.1, 1883.2, 1883.2, "measured")


ALL_WORKLOADS = ["tiny_fp32", "headwise_bf16", "material_bf16", "lowrank_bf16", "qkv_packed_bf16", "static_bf16",
                 "decode_bf16", "proj_qkv_bf16", "lowrank_zproj_bf16"]


def test_the_list_names_every_workload():
    from dynamic_short_convolution_gb300 import inputs

    assert sorted(ALL_WORKLOADS) == sorted(w.name for w in inputs.WORKLOADS.values())


@pytest.mark.parametrize("name", ALL_WORKLOADS)
def test_cpu_baseline_step_runs_for_every_workload(name):
    """The CPU-baseline sample (bench's oracle step) runs on every workload kind, on a few tokens of a
    shortened copy, so the reference arm and the per-row CPU figures cannot fail on the GPU machine."""
    import bench
    import oracle
    from dynamic_short_convolution_gb300 import inputs

    wl = inputs.by_name(name)
    if wl.kind != "decode":
        wl = inputs.shrink(replace(wl, B=1), 16)
    else:
        wl = replace(wl, B=4)
    d = inputs.make(wl)
    bench._oracle_step(oracle, wl, d, 0, 2)
