"""The CPU oracle against its pins (CPU only)."""

import numpy as np
import pytest

import oracle
from tests import _pins
from workloads import WORKLOADS, make_inputs



@pytest.mark.parametrize("pin", _pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


# planted mistakes: each must break at least one pin
MUTANTS = {
    1: "scale dropped",
    2: "B indexed transposed",
    3: "wrong adapter slab",
    4: "last term of the h_in sum dropped",
    5: "sign of the delta flipped",
    6: "unstable segmentation",
    7: "empty adapters kept as segments",
    8: "slot stride from the adapter's rank",
    9: "slot adapters read at the slot capacity's rank",
    10: "backbone W indexed transposed",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda k: MUTANTS[k].replace(" ", "_"))
def test_planted_mistake_is_caught(mutant):
    caught = []
    for pin in _pins.ALL_PINS:
        try:
            pin(mutant=mutant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {mutant} ({MUTANTS[mutant]})"


def test_threads_bit_identical():
    rng = np.random.default_rng(3)
    x, A, B, y0, ids = _pins.rand_problem(rng, 33, 5, 64, 40, 8, p_invalid=0.1)
    y1, v1 = oracle.sgmv_ref(x, A, B, ids, 1.0, y0, threads=1, want_v=True)
    y4, v4 = oracle.sgmv_ref(x, A, B, ids, 1.0, y0, threads=4, want_v=True)
    assert np.array_equal(y1, y4) and np.array_equal(v1, v4)


def test_invalid_ids_leave_rows_unchanged():
    rng = np.random.default_rng(4)
    x, A, B, y0, ids = _pins.rand_problem(rng, 20, 4, 32, 24, 8)
    ids[[2, 5, 11]] = [-1, 4, 1000]
    y = oracle.sgmv_ref(x, A, B, ids, 1.0, y0)
    from workloads import f32_from_bf16_bits

    assert np.array_equal(y[[2, 5, 11]], f32_from_bf16_bits(y0[[2, 5, 11]]))
    seg = oracle.lora_segment_ref(ids, 4)
    assert seg["n_invalid"] == 3
    assert seg["perm"][-3:].tolist() == [2, 5, 11]


def test_oracle_f32_error_within_f64_budget_at_largest_h_in():
    """The fp32 oracle's own error at h_in = 28672 (largest projection) is far
    below the parity tolerance 1e-2 + 1e-2*|y|."""
    rng = np.random.default_rng(5)
    x, A, B, y0, ids = _pins.rand_problem(rng, 2, 2, 28672, 64, 16)
    y32 = oracle.sgmv_ref(x, A, B, ids, 1.0, y0)
    y64 = oracle.sgmv_ref(x, A, B, ids, 1.0, y0, f64=True)
    err = np.abs(y32 - y64)
    assert np.all(err <= 1e-4 + 1e-4 * np.abs(y64)), err.max()


def test_segmentation_of_every_workload_is_a_stable_sort():
    for name, wl in WORKLOADS.items():
        ids = wl.ids()
        seg = oracle.lora_segment_ref(ids, wl.P)
        assert np.array_equal(seg["perm"], np.argsort(ids, kind="stable")), name
        S = seg["num_segments"]
        assert S == len(np.unique(ids))
        assert np.all(np.diff(seg["seg_adapter"][:S]) > 0)


def test_tiny_workload_end_to_end_cpu():
    wl = WORKLOADS["tiny"]
    inp = make_inputs(wl, "cpu")
    y = oracle.sgmv_ref(inp.x["x"], inp.A[0], inp.B[0], inp.ids.numpy(), wl.scale, inp.y0[0])
    y64 = oracle.sgmv_ref(inp.x["x"], inp.A[0], inp.B[0], inp.ids.numpy(), wl.scale, inp.y0[0], f64=True)
    assert y.shape == (16, 256)
    assert np.all(np.abs(y - y64) <= 1e-5 + 1e-5 * np.abs(y64))
    seg = oracle.lora_segment_ref(inp.ids.numpy(), 4)
    assert seg["seg_offsets"].tolist() == [0, 1, 4, 9, 16]


def test_compact_pool_twins_have_the_same_segments():
    """The compact-pool twins of the 70B decode batches relabel the ids in
    order: the oracle's permutation and segment offsets are unchanged."""
    for r in (8, 16):
        full, comp = WORKLOADS[f"70b_decode_r{r}"], WORKLOADS[f"70b_decode_r{r}_compact"]
        a = oracle.lora_segment_ref(full.ids(), full.P)
        b = oracle.lora_segment_ref(comp.ids(), comp.P)
        S = a["num_segments"]
        assert S == b["num_segments"] == comp.P
        assert np.array_equal(a["perm"], b["perm"])
        assert np.array_equal(a["seg_offsets"][:S + 1], b["seg_offsets"][:S + 1])
