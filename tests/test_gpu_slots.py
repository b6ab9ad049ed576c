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


def _pinned(bits: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory()


def test_loader_fills_slots_from_pinned_host_and_device_memory():
    """Empty arenas filled only by lora_slot_copy on a loader stream (sources in
    pinned host memory for even adapters, device memory for odd ones), table
    entries by lora_slot_assign; the compute stream waits for the loader's
    event.  Arena bytes must equal the layout's, outputs the oracle's."""
    rng = np.random.default_rng(8)
    P, n, n_slots, h_in, h_out, r_max = 6, 30, 8, 512, 768, 64
    ranks = [8, 16, 32, 64]
    slots = rng.permutation(n_slots)[:P].astype(np.int32)
    rank_of = rng.choice(ranks, P).astype(np.int32)
    A_ref, B_ref, As, Bs = place_adapters(rng, slots, rank_of, n_slots, h_in, h_out, r_max)
    A_gpu = torch.zeros(n_slots, h_in * r_max, dtype=torch.bfloat16, device="cuda")
    B_gpu = torch.zeros(n_slots, r_max * h_out, dtype=torch.bfloat16, device="cuda")
    # the oracle sees the same arenas, with zeros where nothing was copied
    A_exp, B_exp = np.zeros_like(A_ref), np.zeros_like(B_ref)
    for a in range(P):
        r = int(rank_of[a])
        A_exp[slots[a], : h_in * r] = A_ref[slots[a], : h_in * r]
        B_exp[slots[a], : r * h_out] = B_ref[slots[a], : r * h_out]
    table = lsg.SlotTable(torch.full((P,), -1, dtype=torch.int32, device="cuda"),
                          torch.zeros(P, dtype=torch.int32, device="cuda"), n_slots, r_max, lsg.rank_mask(ranks))
    loader = torch.cuda.Stream()
    keep = []
    with torch.cuda.stream(loader):
        for a in range(P):
            src = _pinned if a % 2 == 0 else _dev
            As_t, Bs_t = src(As[a]), src(Bs[a])
            keep += [As_t, Bs_t]
            lsg.lora_slot_copy([(A_gpu, B_gpu, As_t, Bs_t)], n_slots, r_max, int(slots[a]), int(rank_of[a]))
            lsg.lora_slot_assign(table, a, int(slots[a]), int(rank_of[a]))
    done = torch.cuda.Event()
    done.record(loader)
    torch.cuda.current_stream().wait_event(done)
    x = _dev(_b_normal(rng, (n, h_in)))
    y0 = _b_normal(rng, (n, h_out))
    y = _dev(y0)
    ids = rng.integers(0, P, n).astype(np.int32)
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lsg.sgmv_multi_slots([(x, A_gpu, B_gpu, y, 1.0)], table, seg, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(A_gpu.cpu().view(torch.int16).numpy().view(np.uint16), A_exp)
    assert np.array_equal(B_gpu.cpu().view(torch.int16).numpy().view(np.uint16), B_exp)
    assert np.array_equal(table.slot_of.cpu().numpy(), slots)
    ref = oracle.sgmv_slots_ref(x.cpu(), A_exp, B_exp, slots, rank_of, r_max, lsg.rank_mask(ranks), ids, 1.0, y0,
                                threads=THREADS)
    assert_within_tol(y, ref)


def _b_normal(rng, shape):
    from workloads import bf16_bits_from_f32

    return bf16_bits_from_f32(rng.standard_normal(shape).astype(np.float32))


def test_evicted_adapter_is_flagged_and_its_rows_untouched():
    rng = np.random.default_rng(9)
    P = 5
    c = SlotCase(rng, 25, P, 6, 256, 512, 16, [8, 16])
    c.ids[:3] = 2
    tab = c.table()
    lsg.lora_slot_assign(tab, 2, -1)
    y0 = c.yd.clone()
    _run([c], [1.0], P, table=tab, expect_err=-4)
    slots = c.slots.copy()
    slots[2] = -1
    rows = torch.from_numpy(c.ids == 2).cuda()
    assert torch.equal(c.yd[rows], y0[rows])
    assert_within_tol(c.yd, c.ref(1.0, slots=slots))


def test_load_on_a_second_stream_while_sgmv_runs():
    """SGMV over adapters 0..P-2 on the compute stream while adapter P-1 is
    copied into a free slot on a loader stream: both results are exact."""
    rng = np.random.default_rng(10)
    P, n_slots, h, r_max = 8, 10, 2048, 32
    c = SlotCase(rng, 64, P, n_slots, h, h, r_max, [16, 32], ids=rng.integers(0, P - 1, 64).astype(np.int32))
    tab = c.table()
    lsg.lora_slot_assign(tab, P - 1, -1)
    free = int(np.setdiff1d(np.arange(n_slots), c.slots)[0])
    A_new = _pinned(_b_normal(rng, (h, 32)))
    B_new = _pinned(_b_normal(rng, (32, h)))
    torch.cuda.synchronize()
    loader = torch.cuda.Stream()
    with torch.cuda.stream(loader):
        lsg.lora_slot_copy([(c.Ad, c.Bd, A_new, B_new)], n_slots, r_max, free, 32)
    _run([c], [0.5], P, table=tab)
    loader.synchronize()
    slots = c.slots.copy()
    slots[P - 1] = -1
    assert_within_tol(c.yd, c.ref(0.5, slots=slots))
    got = c.Ad[free, : h * 32].cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, A_new.view(torch.int16).numpy().view(np.uint16).reshape(-1))


@pytest.mark.parametrize("r_max,ranks", [(64, [8, 16, 32, 64]), (32, [16, 32])])
def test_prefill_segments_in_slot_arenas(r_max, ranks):
    """Long contiguous segments of ranks 16/32/64 go to one tensor-tile launch
    per rank, rank-8 ones and short ones to the split-K kernel; a long segment
    whose slot is invalid is left to the split-K kernel, which flags it."""
    rng = np.random.default_rng(50 + r_max)
    P, n_slots, h_in, h_out = 7, 10, 512, 640
    lens = [300, 3, 130, 64, 200, 40, 90]
    ids = np.concatenate([np.full(l, a, np.int32) for a, l in enumerate(lens)])
    c = SlotCase(rng, ids.size, P, n_slots, h_in, h_out, r_max, ranks, ids=ids)
    # every rank of the mask on some long segment
    for a, rk in zip([0, 2, 4, 6], (ranks * 2)[:4]):
        c.rank_of[a] = rk
    c.A, c.B, _, _ = place_adapters(rng, c.slots, c.rank_of, n_slots, h_in, h_out, r_max)
    c.Ad, c.Bd = _dev(c.A), _dev(c.B)
    slots = c.slots.copy()
    slots[4] = n_slots  # invalid slot on a 200-token segment
    y0 = c.yd.clone()
    _run([c], [0.5], P, table=c.table(slots=slots), expect_err=-4)
    rows = torch.from_numpy(c.ids == 4).cuda()
    assert torch.equal(c.yd[rows], y0[rows])
    assert_within_tol(c.yd, c.ref(0.5, slots=slots))


def test_prefill_one_rank_slot_table_matches_contiguous_pool():
    """A one-rank slot table over a permuted pool gives the same bits as the
    contiguous pool through the tensor-tile kernel."""
    rng = np.random.default_rng(60)
    P, n_slots, h_in, h_out, r = 4, 6, 1024, 768, 64
    ids = np.concatenate([np.full(l, a, np.int32) for a, l in enumerate([700, 260, 128, 513])])
    c = SlotCase(rng, ids.size, P, n_slots, h_in, h_out, r, [r], ids=ids)
    y_ref = c.yd.clone()
    _run([c], [1.0], P)
    # the same adapters as a contiguous pool
    A = torch.stack([c.Ad[int(c.slots[a])].view(h_in, r) for a in range(P)])
    B = torch.stack([c.Bd[int(c.slots[a])].view(r, h_out) for a in range(P)])
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P)
    lsg.sgmv_fused(c.xd, A.contiguous(), B.contiguous(), seg, y_ref, 1.0)
    torch.cuda.synchronize()
    assert torch.equal(c.yd, y_ref)
