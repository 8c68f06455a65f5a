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
    for case in (gold, gold["second_case"]):
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
