"""Host-side integer logic of the oracle (offsets, seam bodies, LPT) against
hand-worked examples and brute force, and the seeded input recipe."""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import schedule as sch
from linear_attn_state_gb300 import synth


def test_offsets_and_bodies():
    assert sch.offsets_from_lengths([3, 0, 5]) == [0, 3, 3, 8]
    assert sch.validate_offsets([0, 3, 3, 8], 8)
    assert not sch.validate_offsets([1, 3], 3)
    assert not sch.validate_offsets([0, 5, 4], 4)
    assert not sch.validate_offsets([0, 3, 8], 9)
    assert sch.body_ranges([0, 3, 3, 20], 8) == [(3, 3), (3, 3), (11, 20)]
    with pytest.raises(ValueError):
        sch.offsets_from_lengths([2, -1])


def test_lpt_hand_examples(golden_dir):
    with open(os.path.join(golden_dir, "lpt_hand_example.json")) as f:
        gold = json.load(f)
    for case in (gold, gold["second_case"], gold["third_case"], gold["fourth_case"]):
        off = sch.offsets_from_lengths(case["lengths"])
        order, worker = sch.lpt_schedule(off, case["seam_w"], case["n_streams"], case["n_workers"])
        assert order == case["order"]
        assert worker == case["worker"]


def test_lpt_graham_bound_against_brute_force():
    """Greedy LPT's makespan is within 4/3 - 1/(3m) of the optimum (Graham 1969);
    the optimum is found by brute force on tiny instances."""
    rng = np.random.default_rng(0)
    for _ in range(40):
        n = int(rng.integers(1, 8))
        m = int(rng.integers(1, 4))
        lengths = [int(x) for x in rng.integers(0, 20, n)]
        off = sch.offsets_from_lengths(lengths)
        order, worker = sch.lpt_schedule(off, 0, 1, m)
        assert sorted(order) == list(range(n))
        costs = [lengths[i] for i in order]
        assert costs == sorted(costs, reverse=True)
        loads = [0] * m
        for i in range(n):
            loads[worker[i]] += lengths[i]
        best = min(max(sum(lengths[i] for i in range(n) if a[i] == w) for w in range(m))
                   for a in itertools.product(range(m), repeat=n))
        assert max(loads) <= (4 / 3 - 1 / (3 * m)) * best + 1e-9


def _schedule_checks(golden_dir):
    """The schedule pins as one function; returns the names that fail."""
    failed = []
    for name, pin in (("bodies", test_offsets_and_bodies),
                      ("hand", lambda: test_lpt_hand_examples(golden_dir)),
                      ("graham", test_lpt_graham_bound_against_brute_force)):
        try:
            pin()
        except Exception:  # noqa: BLE001 - any failure of a pin catches the mutant
            failed.append(name)
    return failed


def test_schedule_planted_mistakes_are_caught(golden_dir, monkeypatch):
    """Mistakes planted into the oracle's schedule (shortest first, ties to the
    highest worker id, stream-major tie-break, the seam window left in the
    cost) each fail one of the schedule pins."""
    assert _schedule_checks(golden_dir) == []
    base_bodies = sch.body_ranges

    def lpt_variant(key, tie_high=False, bodies=None):
        def f(offsets, seam_w, n_streams, n_workers):
            br = (bodies or sch.body_ranges)(offsets, seam_w)
            items = sorted(((b - a, seg, s) for seg, (a, b) in enumerate(br)
                            for s in range(n_streams)), key=key)
            loads = [0] * n_workers
            worker = [0] * len(items)
            for cost, seg, s in items:
                best = min(range(n_workers), key=lambda w: (loads[w], -w if tie_high else w))
                worker[seg * n_streams + s] = best
                loads[best] += cost
            return [seg * n_streams + s for (_, seg, s) in items], worker
        return f

    lpt = lambda it: (-it[0], it[1], it[2])  # noqa: E731
    shortest_first = lpt_variant(lambda it: (it[0], it[1], it[2]))
    ties_high = lpt_variant(lpt, tie_high=True)
    stream_major = lpt_variant(lambda it: (-it[0], it[2], it[1]))
    seam_in_cost = lpt_variant(lpt, bodies=lambda offs, w: base_bodies(offs, 0))
    # the variant with the pages' reading reproduces the oracle
    with monkeypatch.context() as m:
        m.setattr(sch, "lpt_schedule", lpt_variant(lpt))
        assert _schedule_checks(golden_dir) == []

    def seam_not_capped(offsets, seam_w):
        return [(int(a) + int(seam_w), int(b)) for a, b in zip(offsets, offsets[1:])]

    for attr, mutant in (("lpt_schedule", shortest_first), ("lpt_schedule", ties_high),
                         ("lpt_schedule", stream_major), ("lpt_schedule", seam_in_cost),
                         ("body_ranges", seam_not_capped)):
        with monkeypatch.context() as m:
            m.setattr(sch, attr, mutant)
            assert _schedule_checks(golden_dir), getattr(mutant, "__name__", attr)
    assert sch.body_ranges is base_bodies


def test_cold_long_lengths_recipe():
    L = synth.cold_long_lengths()
    assert L.sum() == 131072
    assert (L[:-1] >= 128).all() and (L[:-1] <= 8192).all()
    assert 128 <= L[-1] <= 8192 + 127
    assert 60 <= len(L) <= 250
    assert np.array_equal(L, synth.cold_long_lengths())


def test_small_workload_recipe():
    p = synth.gdn_small()
    assert p.k.dtype == synth.torch.float32 and tuple(p.k.shape) == (1024, 1, 64)
    assert list(p.offsets) == [0, 256, 512, 768, 1024]
    kn = p.k.double().norm(dim=-1)
    assert float((kn - 1).abs().max()) < 1e-6
    a = p.log_alpha.double().exp()
    assert float(a.max()) < 1.0 and float(a.median()) > 0.9
    assert float(p.beta.min()) >= 0.0 and float(p.beta.max()) < 1.0
    p2 = synth.gdn_small()
    assert synth.torch.equal(p.k, p2.k) and synth.torch.equal(p.log_alpha, p2.log_alpha)


def test_decay_heads_recipe():
    r, g = synth.decay_heads()
    gam = np.exp(r.log_alpha.double().numpy())
    assert np.allclose(gam, 1 - 2.0 ** (-5 - np.arange(8)), rtol=1e-6)
    assert tuple(g.log_alpha.shape) == (8192, 8, 128)
    assert r.k.dtype == synth.torch.bfloat16


def test_split_pieces_hand_example():
    """lengths [10, 3, 0, 7], seam window 2, pieces of at most 4 tokens, worked
    by hand: segment 0 [0,10) -> window [0,2), body pieces [2,6) [6,10);
    segment 1 [10,13) -> window [10,12), body [12,13); segment 2 is empty;
    segment 3 [13,20) -> window [13,15), body [15,19) [19,20)."""
    off, body = sch.split_pieces([0, 10, 13, 13, 20], 2, 4)
    assert off == [0, 2, 6, 10, 12, 13, 15, 19, 20]
    assert body == [[1, 2], [4], [], [6, 7]]


def test_split_pieces_invariants():
    """On random segmentations: the pieces tile [0, n_tok) in order, every body
    piece is at most piece_tokens long, each segment's body pieces tile exactly
    its body range, and the other pieces are exactly the seam windows."""
    rng = np.random.default_rng(31)
    for _ in range(50):
        lengths = rng.integers(0, 40, rng.integers(1, 12)).tolist()
        w, P = int(rng.integers(0, 6)), int(rng.integers(1, 9))
        offs = sch.offsets_from_lengths(lengths)
        poff, body = sch.split_pieces(offs, w, P)
        assert poff[0] == 0 and poff[-1] == offs[-1]
        assert all(b > a for a, b in zip(poff, poff[1:]))
        used = set()
        for (a, b), mine in zip(sch.body_ranges(offs, w), body):
            covered = [(poff[i], poff[i + 1]) for i in mine]
            assert all(y - x <= P for x, y in covered)
            if mine:
                assert covered[0][0] == a and covered[-1][1] == b
                assert all(covered[i][1] == covered[i + 1][0] for i in range(len(covered) - 1))
            else:
                assert a == b
            used.update(mine)
        windows = [(x, x + min(w, y - x)) for x, y in zip(offs, offs[1:]) if min(w, y - x) > 0]
        others = [(poff[i], poff[i + 1]) for i in range(len(poff) - 1) if i not in used]
        assert others == windows


def test_split_pieces_planted_mistakes():
    """A cut that keeps the window in the first piece, or cuts past the body's
    end, breaks the hand example."""
    def keep_window(offsets, seam_w, P):
        out, body = [0], []
        for a, b in zip(offsets, offsets[1:]):
            mine, pos = [], a
            while pos < b:
                mine.append(len(out) - 1)
                pos = min(pos + P, b)
                out.append(pos)
            body.append(mine)
        return out, body

    def past_end(offsets, seam_w, P):
        out, body = [0], []
        for a, b in zip(offsets, offsets[1:]):
            w = min(seam_w, b - a)
            if w > 0:
                out.append(a + w)
            mine, pos = [], a + w
            while pos < b:
                mine.append(len(out) - 1)
                pos = pos + P
                out.append(pos)
            body.append(mine)
        return out, body
    want = ([0, 2, 6, 10, 12, 13, 15, 19, 20], [[1, 2], [4], [], [6, 7]])
    for bad in (keep_window, past_end):
        assert bad([0, 10, 13, 13, 20], 2, 4) != want
