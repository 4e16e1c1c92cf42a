"""The bench's multi-rank host logic on the CPU (gloo, world size 2).

Each GPU runs an independent replica; the only exchange is the timing
reduction: every rank's timings are reduced by maximum (the slowest replica
sets the job's time), only rank 0 reports, and the whole-job throughput
counts the units of all ranks. The reference arm runs on rank 0 alone.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        # rank 1 is slower on the first timing, rank 0 on the second
        got = bench.max_over_ranks([10.0 + 5 * r, 7.0 - r, 3.0], "cpu", w)
        out.put((r, w, local, got))
    finally:
        dist.destroy_process_group()


def test_timings_reduce_to_the_slowest_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [(r, w, local) for r, w, local, _ in res] == [(0, 2, 0), (1, 2, 1)]
    for _, _, _, got in res:
        assert got == [15.0, 7.0, 3.0]  # every rank sees the job's maxima


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks([1.5, 2.5], "cpu", 1) == [1.5, 2.5]


def test_job_throughput_counts_every_rank():
    # two replicas, 4 calls of 1e12 FLOP each, slowest rank 8 ms in total
    assert bench.job_throughput(2, 4, 1e12, 8.0, 1e12) == pytest.approx(1000.0)
    assert bench.job_throughput(1, 4, 1e12, 8.0, 1e12) == pytest.approx(500.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    args = type("A", (), {"steps": 1, "warmup": 3, "gpus": 2, "impl": "reference",
                          "no_cpu_baseline": True})()
    assert bench.run_reference(args) is None  # other ranks exit without work


def test_source_hash_ignores_comments_only(tmp_path, monkeypatch):
    """Recorded DRAM traffic is keyed by a hash of the kernel code without
    comments and blank lines: documenting a kernel keeps its counters, any
    code change voids them."""
    base = "int f(int x) {\n  return x + 1;\n}\n"
    variants = {
        "a.cu": base,
        "b.cu": "// what f does\n" + base.replace("{\n", "{  // add one\n") + "\n\n/* note\n*/\n",
        "c.cu": base.replace("x + 1", "x + 2"),
    }
    for name, text in variants.items():
        (tmp_path / name).write_text(text)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.source_sha("a.cu") == bench.source_sha("b.cu")
    assert bench.source_sha("a.cu") != bench.source_sha("c.cu")


def test_source_hash_covers_included_headers(tmp_path, monkeypatch):
    """Device code in a header the kernel includes counts as the kernel's code."""
    (tmp_path / "k.cu").write_text('#include "h.cuh"\nint g() { return f(1); }\n')
    (tmp_path / "h.cuh").write_text("int f(int x) { return x + 1; }\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    before = bench.source_sha("k.cu")
    (tmp_path / "h.cuh").write_text("// documented\nint f(int x) { return x + 1; }\n")
    assert bench.source_sha("k.cu") == before
    (tmp_path / "h.cuh").write_text("int f(int x) { return x + 2; }\n")
    assert bench.source_sha("k.cu") != before
