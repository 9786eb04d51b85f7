"""Pins for the reference block manager: a hand-worked walkthrough of the
pages' BlockManager sketch, the pages' sharing numbers, and invariants under
random operation sequences."""

import json
import os

import numpy as np
import pytest

from oracle.block_manager_ref import RefBlockManager
from oracle.kv_ops import slot_of

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def check_invariants(bm: RefBlockManager):
    count = {}
    for seq, blocks in bm.blocks.items():
        assert len(blocks) == -(-bm.length[seq] // bm.B)
        for b in blocks:
            count[b] = count.get(b, 0) + 1
    assert count == bm.refcount                      # refcount = table entries pointing at b
    assert len(set(bm.free)) == len(bm.free)         # no duplicates
    assert not (set(bm.free) & set(bm.refcount))     # free and used are disjoint
    assert len(bm.free) + len(bm.refcount) == bm.num_blocks
    for seq in bm.blocks:                            # internal waste < B per sequence
        assert len(bm.blocks[seq]) * bm.B - bm.length[seq] < bm.B


def test_walkthrough_matches_hand_derivation():
    with open(os.path.join(GOLDEN, "block_manager_walkthrough.json")) as f:
        spec = json.load(f)
    bm = RefBlockManager(spec["block_size"], spec["free_order"])
    for step in spec["steps"]:
        op = step["op"]
        if op == "add":
            slots = bm.add_sequence(step["seq"], step["tokens"])
        elif op == "fork":
            bm.fork(step["parent"], step["child"])
            slots = None
        elif op == "append":
            slots = bm.append_tokens([(s, n) for s, n in step["requests"]])
        elif op == "free":
            bm.free_seq(step["seq"])
            slots = None
        if "expect_slots" in step:
            assert slots == step["expect_slots"]
        if "expect_copies" in step:
            assert [list(c) for c in bm.take_copies()] == step["expect_copies"]
        if "expect_tables" in step:
            assert {s: bm.table(s) for s in step["expect_tables"]} == step["expect_tables"]
        if "expect_free" in step:
            assert bm.free == step["expect_free"]
        if "expect_refcount" in step:
            for b, c in step["expect_refcount"].items():
                assert bm.refcount[int(b)] == c
        check_invariants(bm)


def test_allocation_failure_changes_nothing():
    bm = RefBlockManager(4, list(range(3)))
    assert bm.add_sequence("a", 9) == [8, 9, 10, 11, 4, 5, 6, 7, 0]
    before = (list(bm.free), dict(bm.refcount), {k: list(v) for k, v in bm.blocks.items()}, dict(bm.length))
    assert bm.append_tokens([("a", 3), ("a", 1)]) is None     # would need a 4th block
    assert (bm.free, bm.refcount, bm.blocks, bm.length) == before
    assert bm.add_sequence("b", 1) is None
    assert "b" not in bm.blocks


def test_prefix_sharing_saves_the_pages_figure():
    # letsbuildsolutions "Production Considerations": a 2000-token system
    # prompt shared by 100 concurrent requests saves about 200,000 tokens of
    # pages.
    B = 16
    bm = RefBlockManager(B, list(range(200)))
    bm.add_sequence(0, 2000)
    for i in range(1, 100):
        bm.fork(0, i)
    logical = sum(len(v) for v in bm.blocks.values()) * B
    physical = len(bm.refcount) * B
    saved = logical - physical
    assert saved == 99 * 2000
    assert abs(saved - 200_000) / 200_000 < 0.011
    check_invariants(bm)


def test_parallel_sampling_saves_over_half_the_prompt():
    # ontq section 3: sharing prompt blocks across parallel samples cuts
    # prompt memory by over 50%, copying only the block that diverges.
    B, S = 32, 8
    bm = RefBlockManager(B, list(range(400)))
    bm.add_sequence(0, 2032)
    for i in range(1, S):
        bm.fork(0, i)
    assert bm.append_tokens([(i, 1) for i in range(S)]) is not None
    copies = bm.take_copies()
    assert len(copies) == S - 1                          # the half-full last block, S-1 times
    assert all(src == bm.table(S - 1)[63] for src, _ in copies)
    prompt_physical = 64 + (S - 1)
    assert 1 - prompt_physical / (S * 64) > 0.5
    check_invariants(bm)


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_keep_invariants(seed):
    r = np.random.Generator(np.random.PCG64(seed))
    B = int(r.choice([2, 4, 16]))
    NB = 60
    bm = RefBlockManager(B, list(r.permutation(NB)))
    live = []
    next_id = 0
    written = {}   # slot -> (seq, position) of the latest live writer
    for _ in range(300):
        op = r.integers(0, 4)
        if op == 0 or not live:
            n = int(r.integers(1, 3 * B))
            if bm.add_sequence(next_id, n) is not None:
                live.append(next_id)
            next_id += 1
        elif op == 1:
            reqs = [(int(s), int(r.integers(1, B + 2))) for s in r.choice(live, size=min(3, len(live)), replace=False)]
            bm.append_tokens(reqs)
        elif op == 2:
            parent = int(r.choice(live))
            bm.fork(parent, next_id)
            live.append(next_id)
            next_id += 1
        else:
            s = int(r.choice(live))
            bm.free_seq(s)
            live.remove(s)
        bm.take_copies()
        check_invariants(bm)
        # slot rule agrees with the table for every live token
        for s in live:
            t = bm.length[s] - 1
            assert slot_of(bm.table(s), t, B) // B == bm.table(s)[-1]
    for s in list(live):
        bm.free_seq(s)
    assert sorted(bm.free) == list(range(NB))
