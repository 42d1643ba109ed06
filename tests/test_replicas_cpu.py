"""The N-GPU bookkeeping of bench.py on CPU: two gloo ranks (replicas), the
max-over-ranks timing and the whole-job rate; the reference arm on a rank
other than 0 exits without work."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from block_sparse_attention_token_gb300 import replicas
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, local, w = replicas.rank_world()
        replicas.barrier()
        ms_local = 10.0 + 5.0 * rank                    # rank 1 is the slower one
        ms = replicas.max_over_ranks(ms_local)
        rate = replicas.whole_job_rate(1e9, ms, w)
        out.put((r, local, w, ms, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, local, w, ms, rate) in enumerate(res):
        assert (rank, local, w) == (r, r, world)
        assert ms == 15.0                               # the slower rank's time on every rank
        assert rate == pytest.approx(2 * 1e9 / 15e-3)   # both ranks' work over that time


def test_single_process_is_its_own_maximum():
    sys.path.insert(0, ROOT)
    from block_sparse_attention_token_gb300 import replicas
    assert replicas.max_over_ranks(3.5) == 3.5
    assert replicas.whole_job_rate(2.0, 1.0, 1) == 2000.0


def test_reference_arm_on_other_ranks_exits_without_output():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
