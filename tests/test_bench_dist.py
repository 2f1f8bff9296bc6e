"""Host logic of the multi-GPU benchmark path, run as two gloo ranks on the CPU: every rank runs the
same per-GPU workload (weak scaling, no data-path collective); the timing is the max over ranks and the
aggregate counts all ranks' work."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, lr = bench.dist_env()
    assert (w, r, lr) == (world, rank, rank)
    bench.barrier(world)
    t = bench.reduce_max(1.0 + rank, world)  # rank 1 is slower
    agg = bench.aggregate_rate(100.0, world, t)
    q.put((rank, t, agg))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, agg in res:
        assert t == 2.0               # max over ranks
        assert agg == pytest.approx(100.0)  # 2 ranks x 100 units / 2 s


def test_banded_flop_accounting():
    import bench
    # brute force sum_t min(t+1, w) against the closed form, including chunk offsets
    for L, w, pos0 in [(64, 16, 0), (64, 64, 0), (100, 7, 0), (50, 10, 30), (10, 100, 5), (1, 1, 0)]:
        assert bench.banded_pairs(L, w, pos0) == sum(min(t + 1, w) for t in range(pos0, pos0 + L))
    assert bench.banded_flops(1, 32, 8192, 128, 1024) == 4 * 32 * 128 * 7864832
    assert bench.banded_flops(2, 32, 32768, 128, 4096) == 4 * 64 * 128 * 125831168


def test_dilated_flop_accounting():
    import bench
    import oracle
    # 4 d per pair of the dilated key sets, against the oracle's brute-force membership
    for L, w, s, r in [(60, 9, 3, 4), (41, 6, 2, 3), (30, 7, 0, 2), (25, 5, 4, 1), (12, 30, 4, 5)]:
        pairs = sum(oracle.is_key_dilated(t, i, w, s, r) for t in range(L) for i in range(t + 1))
        assert bench.dilated_flops(2, 3, L, 16, w, s, r) == 4.0 * 2 * 3 * 16 * pairs
    assert bench.dilated_flops(1, 2, 50, 128, 10, 2, 1) == bench.banded_flops(1, 2, 50, 128, 10)


def test_blocksparse_pairs_counts_the_oracle_key_sets():
    import bench
    import oracle
    import swa_inputs
    for L, w, s, ng, block, r, seed in [(90, 12, 2, 1, 8, 2, 1), (130, 40, 0, 0, 16, 3, 2), (75, 9, 3, 2, 5, 1, 3)]:
        globals_, rand = swa_inputs.bigbird_pattern(L, block, ng, r, seed)
        rd = swa_inputs.rand_blocks_dict(rand)
        g = set(globals_)
        want = sum(1 for t in range(L) for i in range(t + 1) if oracle.is_key_blocksparse(t, i, w, s, g, block, rd))
        assert bench.blocksparse_pairs(L, w, s, globals_, block, rand) == want
    # scattered globals, no random blocks
    g = [3, 4, 20, 51]
    want = sum(1 for t in range(60) for i in range(t + 1) if oracle.is_key_blocksparse(t, i, 10, 2, set(g), 4, None))
    assert bench.blocksparse_pairs(60, 10, 2, g, 4, None) == want
    # no pattern: the banded count
    assert bench.blocksparse_pairs(300, 50, 4, [], 16, None) == bench.banded_pairs(300, 50)


def test_hybrid_flop_accounting():
    import bench
    import oracle
    # 8 d^2 per key that has left the window by the end (= per row with a non-empty state), on top of the band
    for L, w, s in [(50, 10, 2), (9, 10, 2), (40, 3, 0), (64, 64, 4)]:
        n = sum(1 for t in range(L) for i in range(t + 1) if i == t - (w - s) and i >= s and not oracle.is_key(t, i, w, s))
        assert bench.hybrid_flops(2, 3, L, 16, w, s) == bench.banded_flops(2, 3, L, 16, w) + 2 * 3 * n * 8 * 16 * 16
