"""The multi-rank path on CPU: two gloo ranks, as torchrun would start them.

With several GPUs each rank owns a contiguous block of token rows and runs the
fused call on it alone; no data crosses ranks, only the timing barrier and
the max-over-ranks of the measured time.  These tests check that the row
blocks tile the global batch exactly, that the max-over-ranks reduction
returns the slowest rank's time on every rank, and that computing each
rank's block on its own gives the same rows as computing the whole batch
(rows are independent, so no collective is needed).  The per-row results
come from the oracle, on the CPU.

The all-reduce across GPUs (PeerComm) exchanges its ranks' IPC handles through
torch.distributed before any device work: that exchange runs here on gloo
(with stand-in handle bytes), and must give every rank all handles in rank
order.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    import oracle
    import workloads
    from tensor_allreduce_residual_gb300.dist import max_over_ranks, shard_range

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # 1. Row blocks tile [0, total) without gaps or overlaps.
        tiles = {}
        for total in (0, 1, 2, 3, 7, 8192 * world, 8191):
            tiles[total] = shard_range(total, rank, world)
        gathered = [None] * world
        dist.all_gather_object(gathered, tiles)

        # 2. Timing: every rank gets the largest value.
        slowest = max_over_ranks(1.0 + 0.25 * rank)

        # 3. This rank's block, computed alone, against the whole batch.
        glob = workloads.fused_inputs(2, 5, 64, "bf16", partial_dist=("N", 0.0, 0.5),
                                      residual_dist=("N", 0.0, 4.0), bias_dist=("N", 0.0, 0.02),
                                      weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=7)
        b, e = shard_range(glob.tokens, rank, world)
        mine = oracle.residual_rmsnorm([p[b:e].contiguous() for p in glob.partials], glob.bias,
                                       glob.residual[b:e].contiguous(), glob.weight, glob.eps, "bf16")
        whole = oracle.residual_rmsnorm(glob.partials, glob.bias, glob.residual, glob.weight, glob.eps, "bf16")
        same = (torch.equal(mine[0].view(torch.int16), whole[0][b:e].view(torch.int16)) and
                torch.equal(mine[1].view(torch.int16), whole[1][b:e].view(torch.int16)))
        # 4. The peer communicator's handle exchange, in rank order on every rank.
        import tensor_allreduce_residual_gb300 as ar
        handle = bytes([rank + 1]) * ar.AR_IPC_HANDLE_BYTES
        table = ar.gather_handles(handle, dist.all_gather_object, world)
        results[rank] = {"tiles": gathered, "slowest": slowest, "same": same, "handles": table}
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.fixture(scope="module")
def rank_results():
    import oracle
    oracle.build()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, WORLD, port, results)) for r in range(WORLD)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=180)
        codes = [p.exitcode for p in procs]
        for p in procs:
            if p.is_alive():
                p.kill()
        assert codes == [0] * WORLD, f"rank exit codes {codes}"
        return dict(results)


def test_row_blocks_tile_the_batch(rank_results):
    tiles = rank_results[0]["tiles"]
    for total in tiles[0]:
        spans = [tiles[r][total] for r in range(WORLD)]
        assert spans[0][0] == 0 and spans[-1][1] == total
        for (b0, e0), (b1, _) in zip(spans, spans[1:]):
            assert e0 == b1 and b0 <= e0
        sizes = [e - b for b, e in spans]
        assert max(sizes) - min(sizes) <= 1


def test_max_over_ranks_is_the_slowest_rank(rank_results):
    assert [rank_results[r]["slowest"] for r in range(WORLD)] == [1.0 + 0.25 * (WORLD - 1)] * WORLD


def test_each_rank_block_alone_equals_the_whole_batch(rank_results):
    assert all(rank_results[r]["same"] for r in range(WORLD))


def test_peer_handles_are_exchanged_in_rank_order(rank_results):
    want = b"".join(bytes([r + 1]) * 64 for r in range(WORLD))
    assert [rank_results[r]["handles"] for r in range(WORLD)] == [want] * WORLD
