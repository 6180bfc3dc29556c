"""The benchmark's multi-rank plumbing on the CPU: two gloo ranks (the GPU
run uses one process per GPU over NCCL the same way). Decode batches are
independent replicas, so the only cross-rank steps are the barrier around
the timed region and the max over ranks of the step time; the reference
arm runs on rank 0 alone."""
import os
import socket

import torch.multiprocessing as mp

import bench
import oracle
from kv_cache_decode_gqa_gb300 import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    ws, r, local = bench.dist_setup()
    d = bench.dist_init(ws, "gloo")
    bench.barrier(d)
    worst = bench.max_over_ranks(d, 1.5 + rank)       # per-rank step times
    class A:
        config = "tiny_gqa"
        steps = 1
        warmup = 0
    ref = bench.run_reference(A, ws, r) if r != 0 else None
    d.barrier()
    d.destroy_process_group()
    q.put((rank, ws, worst, ref))


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q))
             for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ws, worst, ref in res:
        assert ws == 2
        assert worst == 2.5                 # max over both ranks
        assert ref is None                  # only rank 0 runs the oracle


def test_single_process_needs_no_group():
    assert bench.dist_init(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.0) == 3.0


def test_step_bytes_follow_the_size_formula():
    """The bench's KV-read bytes per step are the cache of the visible
    tokens: the size formula 2 n_l n_kv d_h b per token ("KV cache", "The
    size formula") times the visible length."""
    s = W.config("llama2_7b_mha")
    assert bench.kv_bytes_step(s) == oracle.bytes_per_token(
        32, 32, 128, 2) * 4097
    s = W.config("llama31_70b_gqa_fp8")
    assert bench.kv_bytes_step(s) == oracle.bytes_per_token(
        80, 8, 128, 1) * sum(s.seq_lens)


def test_reference_arm_line_shape():
    class A:
        config = "tiny_gqa"
        steps = 1
        warmup = 0
    line = bench.run_reference(A, 1, 0)
    assert line["impl"] == "reference" and line["unit"] == "GB/s"
    assert line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
