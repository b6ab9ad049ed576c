"""The seeded input generators (CPU): deterministic, the stated
distributions, and slot arenas that hold each adapter where the table says."""

import numpy as np
import torch

from workloads import WORKLOADS, distinct_ids, make_inputs, make_slot_inputs, prefill_ids, zipf_ids


def test_inputs_are_deterministic_and_copies_differ():
    wl = WORKLOADS["tiny"]
    a, b, c = make_inputs(wl, "cpu"), make_inputs(wl, "cpu"), make_inputs(wl, "cpu", copy=1)
    assert torch.equal(a.x["x"], b.x["x"]) and torch.equal(a.A[0], b.A[0]) and torch.equal(a.y0[0], b.y0[0])
    assert not torch.equal(a.x["x"], c.x["x"])
    assert torch.equal(a.ids, c.ids)


def test_value_distributions_match_the_stated_variances():
    wl = WORKLOADS["7b_proj_distinct"]
    inp = make_inputs(wl, "cpu")
    h, r = 4096, 16
    for t, var in ((inp.x["x"], 1.0), (inp.A[0], 1.0 / h), (inp.B[0], 1.0 / r), (inp.y0[0], 1.0)):
        v = t.float().var().item()
        assert abs(v / var - 1.0) < 0.05, (v, var)


def test_id_patterns():
    d = distinct_ids(32, 64)
    assert np.unique(d).size == 32 and d.min() >= 0 and d.max() < 64
    z = zipf_ids(256, 1000, 0.8, seed=0)
    assert 120 < np.unique(z).size < 220
    p = prefill_ids()
    lens = np.diff(np.flatnonzero(np.diff(np.concatenate([[-1], p, [-2]]))))
    assert p.size == 6224 and lens.size == 8 and lens.min() >= 128 and lens.max() <= 2048
    assert np.all(np.diff(p) >= 0)  # requests laid out in ascending adapter order


def test_slot_inputs_place_adapters_at_their_slots():
    ids = np.array([0, 2, 2, 1], np.int32)
    rank_of = np.array([8, 16, 32], np.int32)
    si = make_slot_inputs(64, 48, ids, rank_of, n_slots=5, r_max=32, device="cpu")
    slots = si.slot_of.numpy()
    assert np.unique(slots).size == 3 and slots.min() >= 0 and slots.max() < 5
    assert torch.equal(si.rank_of, torch.from_numpy(rank_of))
    for a, r in enumerate(rank_of):
        A = si.A_arena[int(slots[a]), : 64 * r].float()
        B = si.B_arena[int(slots[a]), : r * 48].float()
        # adapter blocks have the LoRA variances; the rest of the slot is N(0, 1) junk
        assert A.var().item() < 0.1 and abs(B.var().item() * r - 1.0) < 0.5
    again = make_slot_inputs(64, 48, ids, rank_of, n_slots=5, r_max=32, device="cpu")
    assert torch.equal(si.A_arena, again.A_arena) and torch.equal(si.slot_of, again.slot_of)
