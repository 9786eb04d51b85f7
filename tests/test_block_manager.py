"""The product block manager against the oracle's reference manager: identical
tables, slots, copy lists and free lists on the same operation sequences."""

import numpy as np
import pytest

from oracle.block_manager_ref import RefBlockManager
from paged_kv_cache_254_gb300 import BlockManager


def same_state(bm: BlockManager, ref: RefBlockManager):
    assert bm.free_blocks() == ref.free
    assert set(bm.sequences()) == set(ref.blocks)
    for s in ref.blocks:
        assert bm.table(s) == ref.table(s)
        assert bm.length(s) == ref.length[s]
    for b, c in ref.refcount.items():
        assert bm.refcount(b) == c
    assert bm.num_used == len(ref.refcount)


@pytest.mark.parametrize("seed", range(10))
def test_random_operations_match_reference(seed):
    r = np.random.Generator(np.random.PCG64(100 + seed))
    B = int(r.choice([1, 4, 16, 32]))
    NB = int(r.integers(8, 80))
    order = [int(x) for x in r.permutation(NB)]
    bm = BlockManager(NB, B, free_order=order)
    ref = RefBlockManager(B, order)
    live, nid = [], 0
    for _ in range(250):
        op = int(r.integers(0, 5))
        if op == 0 or not live:
            n = int(r.integers(0, 3 * B + 2))
            a = bm.add_sequence(nid, n)
            b = ref.add_sequence(nid, n)
            assert (a is None) == (b is None)
            if a is not None:
                assert a.tolist() == b
                live.append(nid)
            nid += 1
        elif op in (1, 2):
            k = int(r.integers(1, min(4, len(live)) + 1))
            seqs = [int(s) for s in r.choice(live, size=k, replace=bool(r.integers(0, 2)))]
            reqs = [(s, int(r.integers(0, 2 * B + 1))) for s in seqs]
            a = bm.append_slots(reqs)
            b = ref.append_tokens(reqs)
            assert (a is None) == (b is None)
            if a is not None:
                assert a.tolist() == b
        elif op == 3:
            p = int(r.choice(live))
            bm.fork(p, nid)
            ref.fork(p, nid)
            live.append(nid)
            nid += 1
        else:
            s = int(r.choice(live))
            bm.free(s)
            ref.free_seq(s)
            live.remove(s)
        assert bm.take_copies().tolist() == [list(c) for c in ref.take_copies()]
        same_state(bm, ref)


def test_block_tables_and_lengths():
    bm = BlockManager(10, 4, free_order=list(range(10)))
    bm.add_sequence("a", 6)
    bm.add_sequence("b", 1)
    t = bm.block_tables(["b", "a"], 3)
    assert t.dtype == np.int32 and t.tolist() == [[7, -1, -1], [9, 8, -1]]
    assert bm.context_lens(["a", "b"]).tolist() == [6, 1]
    with pytest.raises(ValueError):
        bm.block_tables(["a"], 1)


def test_one_token_requests_and_failure_rollback():
    bm = BlockManager(3, 2, free_order=[0, 1, 2])
    bm.add_sequence(0, 3)
    bm.fork(0, 1)
    snap = bm.snapshot()
    assert bm.append_slots([0, 1, 1, 1]) is None          # needs 3 blocks, 1 free
    assert bm.snapshot() == snap
    # seq 0 holds blocks [2, 1] with 3 tokens; its write at t=3 copies the
    # shared block 1 into the last free block 0; seq 1 then owns block 1 alone
    assert bm.append_slots([0, 1]).tolist() == [0 * 2 + 1, 1 * 2 + 1]
    assert bm.take_copies().tolist() == [[1, 0]]


def test_stats_sharing_and_waste():
    bm = BlockManager(200, 16, seed=3)
    bm.add_sequence(0, 2000)
    for i in range(1, 8):
        bm.fork(0, i)
    st = bm.stats()
    assert st["blocks_used"] == 125
    assert st["logical_blocks"] == 8 * 125
    assert st["sharing_ratio"] == 8.0
    assert st["internal_waste_slots"] == 0
    bm.append_slots(list(range(8)))
    st = bm.stats()
    assert st["blocks_used"] == 125 + 8                     # one new block each (2000 is block-aligned)
    assert st["internal_waste_slots"] == 8 * 15
    assert st["fragmentation"] == 8 * 15 / (133 * 16)


def test_restore_round_trip():
    bm = BlockManager(20, 4, seed=1)
    bm.add_sequence("x", 9)
    bm.fork("x", "y")
    bm.append_slots([("y", 2)])
    bm2 = BlockManager.restore(bm.snapshot())
    assert bm2.snapshot() == bm.snapshot()
    assert bm2.append_slots(["x"]).tolist() == bm.append_slots(["x"]).tolist()


def test_parallel_sampling_flow_matches_reference_at_full_size():
    """The shared-prompt workload driven through both managers: 64 prompts of
    2032 tokens (block 32), 7 forks each, then every sample's tail and new
    token in one request list."""
    from workloads import SAMPLING, make_sampling_case
    case = make_sampling_case(SAMPLING, values=False)
    cfg = SAMPLING
    order = [int(b) for b in np.random.Generator(np.random.PCG64(5)).permutation(case.num_blocks)]
    bm = BlockManager(case.num_blocks, cfg.block_size, free_order=order)
    ref = RefBlockManager(cfg.block_size, order)
    for g in range(cfg.groups):
        assert bm.add_sequence((g, 0), cfg.prompt_len).tolist() == ref.add_sequence((g, 0), cfg.prompt_len)
        for j in range(1, cfg.samples):
            bm.fork((g, 0), (g, j))
            ref.fork((g, 0), (g, j))
    reqs = [((g, j), int(case.tails[g * cfg.samples + j]) + 1) for g in range(cfg.groups)
            for j in range(cfg.samples)]
    assert bm.append_slots(reqs).tolist() == ref.append_tokens(reqs)
    copies = bm.take_copies()
    assert copies.tolist() == [list(c) for c in ref.take_copies()]
    assert copies.shape == (cfg.groups * (cfg.samples - 1), 2)
    same_state(bm, ref)
    for g in range(cfg.groups):
        rows = [bm.table((g, j)) for j in range(cfg.samples)]
        assert all(r[:63] == rows[0][:63] for r in rows)            # 63 full prompt blocks shared
        assert len({r[63] for r in rows}) == cfg.samples               # the half-full one: 7 copies + original


def test_shared_prefix_groups_found_from_forks():
    from oracle.attention import check_prefix_groups
    B = 4
    bm = BlockManager(200, B, seed=2)
    bm.add_sequence("solo", 9)
    bm.add_sequence("p", 10)                       # 2 full blocks + 2 tokens
    for c in ("c1", "c2"):
        bm.fork("p", c)
    bm.append_slots([("p", 3), ("c1", 1), ("c2", 6)])   # each diverges in block 2
    bm.add_sequence("q", 8)                        # exactly 2 full blocks
    bm.fork("q", "q1")
    bm.append_slots([("q1", 1)])
    bm.add_sequence("tail", 3)
    seqs = ["solo", "p", "c1", "c2", "q", "q1", "tail"]
    starts, prefix = bm.shared_prefix_groups(seqs)
    assert starts.tolist() == [1, 4, 6] and prefix.tolist() == [2, 2]
    tables = bm.block_tables(seqs, 8)
    assert check_prefix_groups(tables, bm.context_lens(seqs), starts, prefix, B)
    assert bm.shared_prefix_groups(["solo", "tail"])[1].size == 0


def test_shared_prefix_groups_fill_gaps():
    bm = BlockManager(100, 4, seed=3)
    for name in ("a", "x", "b"):
        bm.add_sequence(name, 8)
    bm.fork("a", "a2")
    bm.fork("b", "b2")
    starts, prefix = bm.shared_prefix_groups(["a", "a2", "x", "b", "b2"])
    assert starts.tolist() == [0, 2, 3, 5] and prefix.tolist() == [2, 0, 2]
