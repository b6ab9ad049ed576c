"""Slot arenas with adapters of mixed ranks through sgmv_multi_slots, against
the oracle on the same bytes.  Adapters sit in shuffled slots whose unused
parts hold random junk, so a wrong slot stride or a read past an adapter's
rank shows up as a parity failure."""

import numpy as np
import pytest
import torch

import adapter_gemm_02_b300 as lsg
import oracle
from tests._gpu import THREADS, assert_within_tol, check_segments
from tests._pins import place_adapters, slot_problem

pytestmark = pytest.mark.gpu


def _dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


class SlotCase:
    """One projection's arenas, inputs and oracle."""

    def __init__(self, rng, n, P, n_slots, h_in, h_out, r_max, ranks, ids=None, p_invalid=0.0):
        (self.x, self.A, self.B, self.slots, self.rank_of, _, _, self.y0, ids0) = slot_problem(
            rng, n, P, n_slots, h_in, h_out, r_max, ranks, p_invalid=p_invalid)
        self.ids = ids0 if ids is None else np.asarray(ids, np.int32)
        self.r_max, self.mask, self.n_slots = r_max, lsg.rank_mask(ranks), n_slots
        self.xd, self.Ad, self.Bd = _dev(self.x), _dev(self.A), _dev(self.B)
        self.yd = _dev(self.y0)

    def table(self, slots=None, rank_of=None, mask=None):
        s = self.slots if slots is None else slots
        r = self.rank_of if rank_of is None else rank_of
        return lsg.SlotTable(torch.from_numpy(np.asarray(s, np.int32)).cuda(),
                             torch.from_numpy(np.asarray(r, np.int32)).cuda(), self.n_slots, self.r_max,
                             self.mask if mask is None else mask)

    def ref(self, scale, slots=None, rank_of=None, mask=None):
        return oracle.sgmv_slots_ref(self.x, self.A, self.B, self.slots if slots is None else slots,
                                     self.rank_of if rank_of is None else rank_of, self.r_max,
                                     self.mask if mask is None else mask, self.ids, scale, self.y0,
                                     threads=THREADS)


def _run(cases, scales, P, table=None, expect_err=0):
    ids = cases[0].ids
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P, err_flag=err)
    check_segments(seg, ids, P)
    tab = table if table is not None else cases[0].table()
    projs = [(c.xd, c.Ad, c.Bd, c.yd, s) for c, s in zip(cases, scales)]
    lsg.sgmv_multi_slots(projs, tab, seg, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == expect_err


@pytest.mark.parametrize("h_in,h_out", [(1024, 2056), (136, 520)])
def test_decode_mixed_ranks(h_in, h_out):
    """Short segments (tiles of 4 tokens), every rank in one launch."""
    rng = np.random.default_rng(h_in + h_out)
    P = 20
    c = SlotCase(rng, 48, P, 29, h_in, h_out, 64, [8, 16, 32, 64])
    _run([c], [0.75], P)
    assert_within_tol(c.yd, c.ref(0.75))


def test_longer_segments_mixed_ranks_r_max_32():
    """Tiles of 16 tokens, segments of 1 to 200 tokens (long ones included:
    slot arenas keep them on the split-K kernel); slots of capacity 32."""
    rng = np.random.default_rng(3)
    P = 6
    lens = [200, 1, 17, 64, 33, 90]
    ids = np.concatenate([np.full(l, a, np.int32) for a, l in enumerate(lens)])
    c = SlotCase(rng, ids.size, P, 11, 512, 384, 32, [8, 16, 32], ids=ids)
    _run([c], [1.5], P)
    assert_within_tol(c.yd, c.ref(1.5))


def test_layer_of_seven_projections_two_ranks():
    """7 projections x 2 ranks = 14 (projection, rank) pairs: the call splits
    into launches of 4 projections; every output checked.  One id names the
    same slot and rank in every projection's arenas."""
    rng = np.random.default_rng(4)
    P, n, n_slots = 9, 40, 12
    base = SlotCase(rng, n, P, n_slots, 256, 256, 64, [16, 64])
    cases = [base]
    for h_in, h_out in [(256, 256), (256, 256), (256, 256), (256, 704), (256, 704), (704, 256)]:
        c = SlotCase(rng, n, P, n_slots, h_in, h_out, 64, [16, 64], ids=base.ids)
        c.slots, c.rank_of = base.slots, base.rank_of
        c.A, c.B, _, _ = place_adapters(rng, base.slots, base.rank_of, n_slots, h_in, h_out, 64)
        c.Ad, c.Bd = _dev(c.A), _dev(c.B)
        cases.append(c)
    scales = [0.5, 1.0, 0.25, 2.0, 0.125, 0.75, 1.0]
    _run(cases, scales, P)
    for i, (c, s) in enumerate(zip(cases, scales)):
        assert_within_tol(c.yd, c.ref(s), f"projection {i}")


def test_single_rank_through_the_slot_table():
    """One rank in the mask: the single-rank kernel, reading slots through the table."""
    rng = np.random.default_rng(5)
    P = 16
    c = SlotCase(rng, 64, P, 40, 2048, 1024, 64, [32])
    _run([c], [1.0], P)
    assert_within_tol(c.yd, c.ref(1.0))


def test_invalid_slot_and_rank_are_flagged_and_skipped():
    rng = np.random.default_rng(6)
    P = 8
    c = SlotCase(rng, 40, P, 10, 512, 256, 32, [8, 16])
    c.ids[:4] = [1, 2, 3, 4]
    slots = c.slots.copy()
    rank_of = c.rank_of.copy()
    slots[1] = 10        # outside the arena
    slots[2] = -3
    rank_of[3] = 32      # not in the mask
    rank_of[4] = 24      # not a rank
    y0 = c.yd.clone()
    _run([c], [1.0], P, table=c.table(slots, rank_of), expect_err=-4)
    ref = c.ref(1.0, slots, rank_of)
    bad = np.isin(c.ids, [1, 2, 3, 4])
    assert torch.equal(c.yd[torch.from_numpy(bad).cuda()], y0[torch.from_numpy(bad).cuda()])
    assert_within_tol(c.yd, ref)


def test_relocated_adapters_give_the_same_result():
    """The same adapters in other slots (as after an eviction and reload)."""
    rng = np.random.default_rng(7)
    P = 12
    c = SlotCase(rng, 36, P, 16, 1024, 1024, 64, [8, 64])
    y_first = c.yd.clone()
    _run([c], [1.0], P)
    out1 = c.yd.clone()
    new = rng.permutation(c.n_slots)[:P].astype(np.int32)
    A2, B2 = c.A.copy(), c.B.copy()
    A2[new], B2[new] = c.A[c.slots], c.B[c.slots]
    c.A, c.B, c.Ad, c.Bd = A2, B2, _dev(A2), _dev(B2)
    c.yd = y_first.clone()
    _run([c], [1.0], P, table=c.table(slots=new))
    assert torch.equal(c.yd, out1)
