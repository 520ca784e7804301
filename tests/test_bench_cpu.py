"""bench.py host logic without a GPU: the reference arm's JSON line, the
packed end-to-end buffers, and the multi-process path (world size 2 over
gloo, launched by torchrun): rank 0 alone prints, the max-over-ranks
reduction, and clean exits."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _env():
    env = dict(os.environ)
    env["CUDA_VISIBLE_DEVICES"] = ""
    env["OMP_NUM_THREADS"] = "2"
    return env


def test_reference_arm_single_process():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2",
                        "--warmup", "3", "--workload", "tiny"], cwd=ROOT, env=_env(),
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOPS" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["higher_is_better"] is True and d["steps"] == 2 and d["warmup"] == 3
    # `tiny` has one (batch, KV head): the oracle's backward has work for one thread.
    assert d["cpu_baseline"]["cores"] == 1
    assert d["cpu_baseline"]["sample"].startswith("per step: all 1 batches and 2 query heads")


def test_reference_arm_two_ranks_gloo():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", "29533", "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--workload", "tiny"]
    r = subprocess.run(cmd, cwd=ROOT, env=_env(), capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    assert json.loads(lines[0])["n_gpus"] == 2


def _worker(rank, world, port, out):
    # The gloo path under test is the CPU one: hide any GPU of the host before
    # the first CUDA query, so that each rank takes the CPU branch.
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import bench
    w, r = bench._dist_init()
    try:
        val = bench._max_over_ranks(float(rank + 1) * 1.5, w)
        bench._barrier(w)
        out[rank] = (w, r, val)
    finally:
        import torch.distributed as dist
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    import torch.multiprocessing as mp
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, 2, 29541, out), daemon=True)
             for r in range(2)]
    try:
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert [p.exitcode for p in procs] == [0, 0]
        assert out[0] == (2, 0, 3.0) and out[1] == (2, 1, 3.0)
    finally:
        # A rank left waiting for a peer that failed must not outlive the test.
        for p in procs:
            if p.is_alive():
                p.kill()
                p.join(10)
        mgr.shutdown()


def test_packed_buffers_hold_each_tensor_aligned():
    """The end-to-end measurement's packed buffers: every view starts on a
    16-byte boundary (the kernels' TMA maps need it), keeps its shape and
    dtype, and the views cover the buffer in order without overlap."""
    import torch
    sys.path.insert(0, ROOT)
    import bench
    like = [torch.empty((2, 33, 3, 64), dtype=torch.bfloat16), torch.empty((2, 3, 33), dtype=torch.float32),
            torch.empty((2, 33, 1, 64), dtype=torch.bfloat16), torch.empty((5,), dtype=torch.float32)]
    buf, views = bench._packed(like, "cpu")
    assert buf.dtype == torch.uint8
    end = buf.data_ptr()
    for v, t in zip(views, like):
        assert v.shape == t.shape and v.dtype == t.dtype and v.is_contiguous()
        assert v.data_ptr() % 16 == 0 and v.data_ptr() >= end
        end = v.data_ptr() + v.numel() * v.element_size()
    assert end <= buf.data_ptr() + buf.numel()
    for i, v in enumerate(views):
        v.fill_(i + 1)
    for i, v in enumerate(views):
        assert bool((v == i + 1).all())
