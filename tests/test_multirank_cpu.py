"""Multi-rank host logic on CPU with the gloo backend: the benchmark's
replicas are timed by the slowest rank; the vocabulary-parallel exchange
(MAX of m, rescale, SUM of the rest) gives the whole-vocabulary statistics
over 2 or 3 uneven shards; a rank lost before the exchange makes the
survivor's collective fail instead of hang. No GPU involved."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        got = bench.max_over_ranks(10.0 + 7.5 * rank, world, torch.device("cpu"))
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_bench_takes_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(world))
    assert res == {0: 17.5, 1: 17.5}


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1, torch.device("cpu")) == 3.25


def _stats_of(z):
    """Per-token (m, d, z_y, sum z) of a block of logits, base-2 as the library
    defines them (test-side restatement; numpy float64)."""
    import numpy as np
    t = z * np.log2(np.e)
    m = t.max(axis=1)
    d = np.exp2(t - m[:, None]).sum(axis=1)
    return m, d


CUTS = {2: [0, 3, 10], 3: [0, 1, 7, 10]}  # uneven shards of V = 10 (one of width 1)


def _protocol_worker(rank, world, port, q):
    import numpy as np
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from linear_cross_entropy_gemm_gb300 import vocab_parallel as VP
        from oracle import flce_oracle as O
        r = np.random.default_rng(5)
        z = r.standard_normal((6, 10)) * 3.0          # the whole-vocabulary logits
        y = np.array([0, 9, 4, 6, 2, 7])
        cuts = CUTS[world]
        a, b = cuts[rank], cuts[rank + 1]
        zl = z[:, a:b]
        m, d = _stats_of(zl)
        inside = (y >= a) & (y < b)
        zy = np.where(inside, z[np.arange(6), y], 0.0)
        stats = torch.tensor(np.stack([m, d, zy, zl.sum(1)]), dtype=torch.float64)

        def cpu_rescale(s, gmax):  # the kernel's arithmetic, restated for the test
            s[1] *= torch.exp2(s[0] - gmax)
            s[0] = gmax

        def gloo_allreduce(t, op):
            dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)

        VP.merge_stats(stats, gloo_allreduce, cpu_rescale)
        lse = (stats[0] + torch.log2(stats[1])) * np.log(2.0)
        q.put((rank, lse.numpy(), stats[2].numpy(), stats[3].numpy(),
               O.logsumexp_rows(z), z[np.arange(6), y], z.sum(1)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_vocab_parallel_exchange_protocol(world):
    import numpy as np
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_protocol_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for _ in range(world):
        rank, lse, zy, sz, ref_lse, ref_zy, ref_sz = q.get(timeout=10)
        np.testing.assert_allclose(lse, ref_lse, rtol=1e-13)
        np.testing.assert_allclose(zy, ref_zy, rtol=1e-15)
        np.testing.assert_allclose(sz, ref_sz, rtol=1e-13)


# Exit codes of the surviving rank: its outcome travels in the exit status,
# which (unlike a queue's feeder thread) cannot be lost when it exits.
_RETURNED, _RAISED = 10, 11


def _dying_rank_worker(rank, world, port):
    import datetime
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=10))
    if rank == 1:
        os._exit(3)  # leaves between steps, before its exchange
    from linear_cross_entropy_gemm_gb300 import vocab_parallel as VP
    stats = torch.ones(4, 6, dtype=torch.float64)

    def gloo_allreduce(t, op):
        dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)

    def cpu_rescale(s, gmax):
        s[1] *= torch.exp2(s[0] - gmax)
        s[0] = gmax

    try:
        VP.merge_stats(stats, gloo_allreduce, cpu_rescale)
        code = _RETURNED
    except Exception:  # the collective reports the lost peer
        code = _RAISED
    os._exit(code)


def test_vocab_parallel_exchange_reports_a_lost_rank():
    # A rank that exits before the exchange: the survivor's first all-reduce
    # ends with an error (peer gone, or the 10 s process-group timeout), it
    # does not hang and does not return merged statistics.
    world = 2
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_dying_rank_worker, args=(r, world, port))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
    assert all(p.exitcode is not None for p in procs), "a rank hung"
    assert procs[1].exitcode == 3
    assert procs[0].exitcode == _RAISED, f"survivor exit code {procs[0].exitcode}"


@pytest.mark.parametrize("V,world", [(128256, 2), (128256, 8), (262144, 8), (1000, 3), (4096, 16)])
def test_vocabulary_shard_plan(V, world):
    # The bench's vocabulary split: contiguous shards that cover [0, V) in
    # rank order, 256-aligned starts, sizes within 256 of each other (the last
    # also takes the ragged end).
    from linear_cross_entropy_gemm_gb300.vocab_parallel import shard_range
    r = [shard_range(V, world, k) for k in range(world)]
    assert r[0][0] == 0 and r[-1][1] == V
    assert all(r[k][1] == r[k + 1][0] for k in range(world - 1))
    assert all(a % 256 == 0 and b > a for a, b in r)
    sizes = [b - a for a, b in r]
    assert max(sizes) - min(sizes) <= 256 + V % 256
