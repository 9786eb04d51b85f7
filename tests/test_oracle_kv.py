"""Pins for the oracle's append / copy / slot rules, and a check that the
attention pins catch plausible planted mistakes in the oracle."""

import numpy as np
import pytest

import oracle.attention as att
from oracle.attention import decode_ref, gather_sequence, unpaged_ref
from oracle.kv_ops import append_ref, copy_ref, slot_of


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def test_slot_rule_worked_example():
    # block table formula: i = floor(t / B), j = t mod B; slot = table[i] * B + j
    row = [5, 2, 9]
    assert slot_of(row, 0, 16) == 80
    assert slot_of(row, 17, 16) == 2 * 16 + 1
    assert slot_of(row, 47, 16) == 9 * 16 + 15


def test_append_then_gather_reads_the_new_rows():
    r = _rng(1)
    NB, Hkv, B, d = 10, 3, 4, 8
    kp = r.integers(-30000, 30000, size=(NB, Hkv, B, d)).astype(np.int16)
    vp = r.integers(-30000, 30000, size=(NB, Hkv, B, d)).astype(np.int16)
    row = [7, 2, 4]
    ts = [0, 5, 9, 11]
    kn = r.integers(-30000, 30000, size=(len(ts), Hkv, d)).astype(np.int16)
    vn = r.integers(-30000, 30000, size=(len(ts), Hkv, d)).astype(np.int16)
    slots = [slot_of(row, t, B) for t in ts]
    k2, v2 = append_ref(kp, vp, kn, vn, slots, B)
    for kh in range(Hkv):
        K, V = gather_sequence(k2.astype(np.float64), v2.astype(np.float64), row, 12, kh, B)
        for i, t in enumerate(ts):
            np.testing.assert_array_equal(K[t], kn[i, kh])
            np.testing.assert_array_equal(V[t], vn[i, kh])
    # everything else untouched
    mask = np.ones((NB, B), dtype=bool)
    for s in slots:
        mask[s // B, s % B] = False
    np.testing.assert_array_equal(k2.transpose(0, 2, 1, 3)[mask], kp.transpose(0, 2, 1, 3)[mask])
    np.testing.assert_array_equal(v2.transpose(0, 2, 1, 3)[mask], vp.transpose(0, 2, 1, 3)[mask])


def test_append_skips_negative_slots():
    r = _rng(2)
    kp = r.integers(-9, 9, size=(4, 2, 4, 8)).astype(np.int16)
    kn = r.integers(-9, 9, size=(2, 2, 8)).astype(np.int16)
    k2, v2 = append_ref(kp, kp, kn, kn, [-1, -5], 4)
    np.testing.assert_array_equal(k2, kp)
    np.testing.assert_array_equal(v2, kp)


def test_copy_reads_state_before_the_call():
    r = _rng(3)
    kp = r.integers(-9999, 9999, size=(6, 2, 4, 8)).astype(np.int16)
    vp = r.integers(-9999, 9999, size=(6, 2, 4, 8)).astype(np.int16)
    k2, v2 = copy_ref(kp, vp, [(1, 4), (4, 5), (2, 2)])
    np.testing.assert_array_equal(k2[4], kp[1])
    np.testing.assert_array_equal(k2[5], kp[4])      # the old block 4, not the new one
    np.testing.assert_array_equal(v2[5], vp[4])
    for b in (0, 1, 2, 3):
        np.testing.assert_array_equal(k2[b], kp[b])
        np.testing.assert_array_equal(v2[b], vp[b])


# -- the attention pins catch planted mistakes --------------------------------

def _pins_pass():
    """A condensed run of the attention pins: paged vs un-paged layout (built
    by reshaping whole blocks), a one-token context, and GQA head mapping."""
    from tests.test_oracle import build_paged
    r = _rng(4)
    ok = True
    for ctx, B in [(37, 16), (5, 4)]:
        Hq, Hkv, d = 4, 2, 8
        nblk = -(-ctx // B)
        table = r.permutation(nblk + 4)[:nblk]
        Kc = r.standard_normal((ctx, Hkv, d))
        Vc = r.standard_normal((ctx, Hkv, d))
        q = r.standard_normal((Hq, d))
        kp, vp = build_paged(Kc, Vc, table, nblk + 4, B)
        got = decode_ref(q[None], kp, vp, table[None], np.array([ctx]), 0.3)[0]
        want = unpaged_ref(q, Kc, Vc, 0.3)
        ok &= bool(np.allclose(got, want, rtol=1e-12, atol=1e-13))
    return ok


@pytest.mark.parametrize("mutant", ["offset_as_block", "block_from_offset", "skip_scale", "kv_swapped",
                                    "wrong_group"])
def test_planted_oracle_mistakes_are_caught(monkeypatch, mutant):
    assert _pins_pass()
    if mutant == "offset_as_block":
        monkeypatch.setattr(att, "physical_location",
                            lambda row, t, B: (int(row[t // B]), (t + 1) % B))
    elif mutant == "block_from_offset":
        monkeypatch.setattr(att, "physical_location",
                            lambda row, t, B: (int(row[t % B % len(row)]), t // B % B))
    elif mutant == "skip_scale":
        orig = att.softmax_weights
        monkeypatch.setattr(att, "softmax_weights", lambda q, K, scale: orig(q, K, 1.0))
    elif mutant == "kv_swapped":
        orig = att.gather_sequence
        monkeypatch.setattr(att, "gather_sequence",
                            lambda kp, vp, row, ctx, kh, B: orig(kp, vp, row, ctx, kh, B)[::-1])
    elif mutant == "wrong_group":
        orig = att.gather_sequence
        monkeypatch.setattr(att, "gather_sequence",
                            lambda kp, vp, row, ctx, kh, B: orig(kp, vp, row, ctx, (kh + 1) % kp.shape[1], B))
    assert not _pins_pass()
