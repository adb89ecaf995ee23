"""The multi-GPU path of bench.py on CPU: world-size-2 gloo ranks in separate
processes, the way `torch.distributed.run --nproc-per-node 2 bench.py` starts
replicas. Covers the host logic only -- the job time is the largest rank time,
the value counts every replica's tokens, and the reference arm runs and prints
on rank 0 alone -- so no GPU and no NCCL are involved."""
import contextlib
import io
import json
import multiprocessing as mp
import os
import socket
import sys
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bench
    from dynamic_short_convolution_gb300 import inputs

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        local_ms = 10.0 * (rank + 1)  # rank 1 is the slower replica
        job_ms = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
        value = bench.whole_job_tokens_per_s(world, 1000, 5, job_ms)
        wl = inputs.WORKLOADS[1]
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            rc = bench.run_reference(types.SimpleNamespace(steps=1, warmup=0), wl, rank, world)
        dist.barrier()
        out = {"job_ms": job_ms, "value": value, "rc": rc, "printed": buf.getvalue(),
               "global_batch": bench.workload_config(wl, world)["global_batch"], "B": wl.B}
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump(out, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["job_ms"] == 20.0  # the slowest replica's time, on every rank
        assert abs(r["value"] - 2 * 1000 * 5 / 0.020) < 1e-6
        assert r["rc"] == 0
        assert r["global_batch"] == 2 * r["B"]
    assert res[1]["printed"] == ""  # only rank 0 runs and prints the reference arm
    line = json.loads(res[0]["printed"].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["config"]["global_batch"] == 2 * res[0]["B"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
