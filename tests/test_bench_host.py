"""Host-side logic of bench.py (no GPU): cross-rank aggregation with a real
world-size-2 gloo process group, clock-log parsing, algorithmic counts."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.dist_init("gloo")
    bench.barrier()
    value, t = bench.aggregate(1000, 0.5 + rank, world)   # rank 1 is the slow one
    q.put((rank, value, t))
    dist.destroy_process_group()


def test_aggregate_uses_all_ranks_tokens_over_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, t in res:
        assert t == pytest.approx(1.5)
        assert value == pytest.approx(2000 / 1.5)


def test_aggregate_single_process():
    assert bench.aggregate(500, 0.25, 1) == (2000.0, 0.25)


def test_parse_clocks():
    text = ("0, 1965, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n"
            "0, 1800, 2070, 1300.5, 0x4, Not Active, Not Active, Not Active, Active\n"
            "0, 1900, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    c = bench.parse_clocks(text)
    assert c["sm_mhz"] == 1900 and c["sm_max_mhz"] == 2070 and c["reasons"] == ["sw_power_cap"]
    assert bench.parse_clocks("") is None


def test_per_token_counts_match_the_stated_totals():
    """The step's algorithmic counts: 16eD + 4eN + 8N + 16 bytes, D(17N + 59)
    FP32-pipe ops and D(2N + 14) MUFU ops per token, i.e. 131,344 B,
    1,355,776 and 188,416 at the Mamba-1.4B shape (D = 4096, N = 16, bf16)."""
    D, N, e = 4096, 16, 2
    c = bench.per_token_counts(D, N, e)
    tot = {k: sum(s[k] for s in c.values()) for k in ("bytes", "fp32", "mufu")}
    assert tot["bytes"] == 16 * e * D + 4 * e * N + 8 * N + 16 == 131344
    assert tot["fp32"] == D * (17 * N + 59) == 1355776
    assert tot["mufu"] == D * (2 * N + 14) == 188416
    # forward only: 6eD + 2eN + 8 bytes, D(4N + 17) FP32, D(N + 6) MUFU
    fwd = {k: c["conv_fwd"][k] + c["scan_fwd"][k] for k in ("bytes", "fp32", "mufu")}
    assert fwd == {"bytes": 6 * e * D + 2 * e * N + 8, "fp32": D * (4 * N + 17), "mufu": D * (N + 6)}
