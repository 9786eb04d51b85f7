"""Host-side pieces of bench.py: byte accounting and the multi-rank timing
reduction (world size 2 over gloo on CPU)."""

import io
import os
import socket
import contextlib

import numpy as np
import torch.multiprocessing as mp

import bench


def test_decode_bytes_by_hand():
    # 2 sequences of 17 and 32 tokens, 4 q / 2 kv heads, d 8, block 16, 2-byte elements
    kv = (17 + 32) * 2 * 8 * 2 * 2
    qo = 2 * 2 * 4 * 8 * 2
    tables = (2 + 2) * 4
    assert bench.decode_bytes([17, 32], 4, 2, 8, 16) == kv + qo + tables + 2 * 4
    assert bench.append_bytes(3, 2, 8) == 2 * 3 * 2 * 8 * 2 * 2 + 24
    assert bench.copy_bytes(5, 2, 16, 8) == 2 * 5 * 2 * 16 * 8 * 2 * 2


def test_unique_bytes_count_shared_blocks_once():
    B = 4
    tables = np.array([[7, 3, 9], [7, 3, 5]])     # two sequences share blocks 7 and 3
    ctx = [10, 11]
    u = bench.unique_decode_bytes(tables, ctx, 2, 1, 8, B)
    tokens = 4 + 4 + 2 + 3                         # blocks 7, 3 full; 9 holds 2; 5 holds 3
    assert u == tokens * 1 * 8 * 2 * 2 + 2 * 2 * 2 * 8 * 2 + (3 + 3) * 4 + 2 * 4
    assert u < bench.decode_bytes(ctx, 2, 1, 8, B)


def test_timed_rows_quantiles_and_rates():
    ms = [float(x) for x in range(1, 12)]          # 1 .. 11 ms
    rows = bench.timed_rows(ms, [0.5, 0.5], None, 6_000_000, 1_000_000, 0)
    d = rows["decode"]
    assert d["ms_p50"] == 6.0 and d["ms_p10"] == 2.0 and d["ms_p90"] == 10.0
    assert d["gbs_at_p50"] == 1.0                  # 6 MB in 6 ms
    assert rows["append"]["ms_p50"] == 0.5 and rows["append"]["gbs_at_p50"] == 2.0
    assert rows["copy"] is None
    one = bench.timed_rows([2.0], [1.0], [4.0], 2e6, 1e6, 4e6)
    assert one["decode"]["ms_p10"] == one["decode"]["ms_p90"] == 2.0
    assert one["copy"]["gbs_at_p50"] == 1.0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench as b
    dist = b.init_dist(world, "gloo")
    got = b.max_over_ranks(1.5 * (rank + 1), dist, "cpu")
    # the reference arm prints on rank 0 only; other ranks leave without work
    buf = io.StringIO()
    if rank == 1:
        with contextlib.redirect_stdout(buf):
            b.reference_arm(b.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"]))
    q.put((rank, got, buf.getvalue()))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_world_size_two():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [3.0, 3.0]
    assert res[1][2] == ""
