"""Pins that tie the CPU oracle to something other than itself.

Each pin raises AssertionError when the oracle (or a variant of it with a
planted mistake, selected by `mutant`) disagrees with:
  - hand-worked examples stored under tests/golden/ (with their derivation),
  - brute force (dense W = A.B in fp64; Python's stable sort),
  - a library routine in the special case of one adapter (torch.matmul),
  - invariants: B = 0 leaves y unchanged, permuting tokens permutes outputs,
    linearity in s, and the rank-1 closed form y = y0 + s*h_in*c*d;
  - for slot arenas of mixed ranks: the dense fp64 product per adapter, the
    contiguous-pool oracle on zero-padded adapters, and relocation of slots.
"""

from __future__ import annotations

import itertools
import json
import os

import numpy as np
import torch

import oracle
from workloads import bf16_bits_from_f32, f32_from_bf16_bits

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
U32 = 2.0 ** -24  # unit roundoff of fp32


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _b(a):
    return bf16_bits_from_f32(np.asarray(a, dtype=np.float32))


def rand_problem(rng, n, P, h_in, h_out, r, p_invalid=0.0, scale_x=1.0):
    x = _b(rng.standard_normal((n, h_in)) * scale_x)
    A = _b(rng.standard_normal((P, h_in, r)) / np.sqrt(h_in))
    B = _b(rng.standard_normal((P, r, h_out)) / np.sqrt(r))
    y0 = _b(rng.standard_normal((n, h_out)))
    ids = rng.integers(0, P, n).astype(np.int32)
    if p_invalid > 0:
        bad = rng.random(n) < p_invalid
        ids[bad] = rng.choice([-1, P, P + 7], bad.sum())
    return x, A, B, y0, ids


def dense_f64(x, A, B, ids, s, y0):
    """Brute force: y = y0 + s * x . (A[a].B[a]) with the dense product W
    formed first (the other association), all in fp64."""
    xf, Af, Bf, yf = (f32_from_bf16_bits(t).astype(np.float64) for t in (x, A, B, y0))
    out = yf.copy()
    for i, a in enumerate(ids):
        if 0 <= a < A.shape[0]:
            W = Af[a] @ Bf[a]
            out[i] = yf[i] + s * (xf[i] @ W)
    return out


def f32_bound(x, A, B, ids, s, y0):
    """Forward error bound of the fp32 per-token oracle around the exact
    result: (h_in + r + 3) * u * (|y0| + |s| * (|x|.|A|).|B|)."""
    xf, Af, Bf, yf = (np.abs(f32_from_bf16_bits(t).astype(np.float64)) for t in (x, A, B, y0))
    h_in, r = A.shape[1], A.shape[2]
    M = yf.copy()
    for i, a in enumerate(ids):
        if 0 <= a < A.shape[0]:
            M[i] = yf[i] + abs(s) * ((xf[i] @ Af[a]) @ Bf[a])
    return (h_in + r + 3) * U32 * M * 1.01


# ------------------------------------------------------------------ pins

def pin_golden_segment(mutant=0):
    g = _golden("segment_handworked.json")
    out = oracle.lora_segment_ref(g["ids"], g["P"], mutant=mutant)
    assert out["perm"].tolist() == g["perm"]
    assert out["seg_offsets"].tolist() == g["seg_offsets"]
    assert out["seg_adapter"].tolist() == g["seg_adapter"]
    assert out["num_segments"] == g["num_segments"]
    assert out["n_invalid"] == g["n_invalid"]


def pin_golden_sgmv(mutant=0):
    g = _golden("sgmv_handworked.json")
    x, A, B, y0 = _b(g["x"]), _b(g["A"]), _b(g["B"]), _b(g["y0"])
    ids = np.array(g["ids"], np.int32)
    y, v = oracle.sgmv_ref(x, A, B, ids, g["s"], y0, want_v=True, mutant=mutant)
    assert np.array_equal(y, np.array(g["y"], np.float32)), y
    assert np.array_equal(v, np.array(g["v"], np.float32)), v
    y64 = oracle.sgmv_ref(x, A, B, ids, g["s"], y0, f64=True, mutant=mutant)
    assert np.array_equal(y64, np.array(g["y"], np.float64))


def _bruteforce_segment(ids, P):
    n = len(ids)
    key = [a if 0 <= a < P else P for a in ids]
    perm = sorted(range(n), key=lambda i: key[i])  # Python's sort is stable
    segs = sorted({a for a in key if a < P})
    offs = [perm.index(next(i for i in perm if key[i] == a)) for a in segs]
    n_valid = sum(k < P for k in key)
    ms = min(n, P)
    offs = offs + [n_valid] * (ms + 1 - len(offs))
    sad = segs + [-1] * (ms - len(segs))
    return perm, offs, sad, len(segs)


def pin_segment_bruteforce(mutant=0):
    # exhaustive over all id lists of length <= 5 from {-1, 0, 1, 2} with P = 3
    for n in range(0, 6):
        for ids in itertools.product([-1, 0, 1, 2], repeat=n):
            perm, offs, sad, S = _bruteforce_segment(list(ids), 3)
            out = oracle.lora_segment_ref(np.array(ids, np.int32), 3, mutant=mutant)
            assert out["perm"].tolist() == perm, (ids, out["perm"], perm)
            assert out["seg_offsets"].tolist() == offs, (ids, out["seg_offsets"], offs)
            assert out["seg_adapter"].tolist() == sad, (ids,)
            assert out["num_segments"] == S
    rng = np.random.default_rng(7)
    for _ in range(50):
        n = int(rng.integers(1, 200))
        P = int(rng.integers(1, 40))
        ids = rng.integers(-2, P + 2, n).astype(np.int32)
        perm, offs, sad, S = _bruteforce_segment(ids.tolist(), P)
        out = oracle.lora_segment_ref(ids, P, mutant=mutant)
        assert out["perm"].tolist() == perm
        assert out["seg_offsets"].tolist() == offs
        assert out["seg_adapter"].tolist() == sad
        assert out["num_segments"] == S


def pin_dense_bruteforce(mutant=0):
    rng = np.random.default_rng(11)
    for n, P, h_in, h_out, r in [(16, 4, 64, 48, 8), (5, 3, 24, 40, 4), (9, 2, 64, 64, 3), (1, 1, 8, 8, 1)]:
        x, A, B, y0, ids = rand_problem(rng, n, P, h_in, h_out, r, p_invalid=0.15)
        s = float(rng.choice([0.5, 1.0, 2.0, -1.25]))
        ref = dense_f64(x, A, B, ids, s, y0)
        y64 = oracle.sgmv_ref(x, A, B, ids, s, y0, f64=True, mutant=mutant)
        assert np.allclose(y64, ref, rtol=1e-12, atol=1e-12)
        y32 = oracle.sgmv_ref(x, A, B, ids, s, y0, mutant=mutant)
        assert np.all(np.abs(y32 - ref) <= f32_bound(x, A, B, ids, s, y0)), np.max(np.abs(y32 - ref))


def pin_single_adapter_matmul(mutant=0):
    rng = np.random.default_rng(12)
    n, h_in, h_out, r, s = 12, 96, 80, 16, 1.5
    x, A, B, y0, _ = rand_problem(rng, n, 1, h_in, h_out, r)
    ids = np.zeros(n, np.int32)
    t = lambda a: torch.from_numpy(f32_from_bf16_bits(a).astype(np.float64))
    ref = (t(y0) + s * torch.matmul(torch.matmul(t(x), t(A)[0]), t(B)[0])).numpy()
    y64 = oracle.sgmv_ref(x, A, B, ids, s, y0, f64=True, mutant=mutant)
    assert np.allclose(y64, ref, rtol=1e-12, atol=1e-12)
    y32 = oracle.sgmv_ref(x, A, B, ids, s, y0, mutant=mutant)
    assert np.all(np.abs(y32 - ref) <= f32_bound(x, A, B, ids, s, y0))


def pin_zero_B(mutant=0):
    rng = np.random.default_rng(13)
    x, A, B, y0, ids = rand_problem(rng, 10, 3, 40, 24, 8)
    B[:] = 0
    y = oracle.sgmv_ref(x, A, B, ids, 3.0, y0, mutant=mutant)
    assert np.array_equal(y, f32_from_bf16_bits(y0))


def pin_permutation(mutant=0):
    rng = np.random.default_rng(14)
    x, A, B, y0, ids = rand_problem(rng, 20, 5, 48, 32, 8)
    y = oracle.sgmv_ref(x, A, B, ids, 0.75, y0, mutant=mutant)
    p = rng.permutation(20)
    yp = oracle.sgmv_ref(x[p], A, B, ids[p], 0.75, y0[p], mutant=mutant)
    assert np.array_equal(yp, y[p])


def pin_linear_in_s(mutant=0):
    rng = np.random.default_rng(15)
    x, A, B, y0, ids = rand_problem(rng, 8, 3, 32, 16, 4)
    y0 = np.zeros_like(y0)
    y1 = oracle.sgmv_ref(x, A, B, ids, 1.0, y0, mutant=mutant)
    y2 = oracle.sgmv_ref(x, A, B, ids, 2.0, y0, mutant=mutant)
    ym = oracle.sgmv_ref(x, A, B, ids, -1.0, y0, mutant=mutant)
    assert np.array_equal(y2, 2 * y1)
    assert np.array_equal(ym, -y1)
    # and the delta is not trivially zero
    assert np.any(y1 != 0)


def pin_rank1_closed_form(mutant=0):
    # r = 1, A = c, B = d, x = 1: y = y0 + s*h_in*c*d (powers of two: exact)
    n, P, h_in, h_out = 4, 2, 64, 16
    c, d, s = 0.25, 2.0, 0.5
    x = _b(np.ones((n, h_in)))
    A = _b(np.full((P, h_in, 1), c))
    B = _b(np.full((P, 1, h_out), d))
    y0 = _b(np.arange(n * h_out).reshape(n, h_out) * 0.5)
    ids = np.array([0, 1, 1, 0], np.int32)
    y = oracle.sgmv_ref(x, A, B, ids, s, y0, mutant=mutant)
    assert np.array_equal(y, f32_from_bf16_bits(y0) + np.float32(s * h_in * c * d))


# ------------------------------------------------------------------ slot arenas, mixed ranks

def slot_problem(rng, n, P, n_slots, h_in, h_out, r_max, ranks, p_invalid=0.0):
    """Adapters of the given ranks placed in shuffled slots of r_max capacity;
    the unused part of every slot holds random junk, so that reading past an
    adapter's rank or at the wrong slot stride changes the result."""
    slots = rng.permutation(n_slots)[:P].astype(np.int32)
    rank_of = rng.choice(ranks, P).astype(np.int32)
    A_ar, B_ar, As, Bs = place_adapters(rng, slots, rank_of, n_slots, h_in, h_out, r_max)
    x = _b(rng.standard_normal((n, h_in)))
    y0 = _b(rng.standard_normal((n, h_out)))
    ids = rng.integers(0, P, n).astype(np.int32)
    if p_invalid > 0:
        bad = rng.random(n) < p_invalid
        ids[bad] = rng.choice([-1, P], bad.sum())
    return x, A_ar, B_ar, slots, rank_of, As, Bs, y0, ids


def place_adapters(rng, slots, rank_of, n_slots, h_in, h_out, r_max):
    """Arenas of n_slots slots (random junk) with adapter a, rank rank_of[a],
    written at the start of slot slots[a]; returns the arenas and the
    adapters' A [h_in][r] and B [r][h_out]."""
    A_ar = _b(rng.standard_normal((n_slots, h_in * r_max)))
    B_ar = _b(rng.standard_normal((n_slots, r_max * h_out)))
    As, Bs = [], []
    for a in range(len(slots)):
        r = int(rank_of[a])
        A = _b(rng.standard_normal((h_in, r)) / np.sqrt(h_in))
        B = _b(rng.standard_normal((r, h_out)) / np.sqrt(r))
        A_ar[slots[a], : h_in * r] = A.reshape(-1)
        B_ar[slots[a], : r * h_out] = B.reshape(-1)
        As.append(A)
        Bs.append(B)
    return A_ar, B_ar, As, Bs


def _mask(ranks):
    m = 0
    for r in ranks:
        m |= 1 << (int(r).bit_length() - 4)
    return m


def pin_golden_slots(mutant=0):
    """Hand-worked slot-arena example with its derivation (tests/golden)."""
    g = _golden("slots_handworked.json")
    y = oracle.sgmv_slots_ref(_b(g["x"]), _b(g["A_arena"]), _b(g["B_arena"]), g["slot_of"], g["rank_of"],
                              g["r_max"], _mask(g["ranks_allowed"]), np.array(g["ids"], np.int32), g["s"],
                              _b(g["y0"]), mutant=mutant)
    assert np.array_equal(y, np.array(g["y"], np.float32)), y


def pin_slots_dense_bruteforce(mutant=0):
    """Mixed ranks in shuffled slots against y0 + s * x . (A_a . B_a) in fp64
    (the other association), within the fp32 forward error bound."""
    rng = np.random.default_rng(21)
    for n, P, n_slots, h_in, h_out, r_max, ranks in [(24, 5, 9, 64, 40, 64, [8, 16, 32, 64]),
                                                       (10, 3, 3, 32, 48, 32, [8, 32]),
                                                       (7, 4, 6, 16, 24, 16, [8, 16])]:
        x, A_ar, B_ar, slots, rank_of, As, Bs, y0, ids = slot_problem(rng, n, P, n_slots, h_in, h_out, r_max,
                                                                      ranks, p_invalid=0.1)
        s = float(rng.choice([0.5, -1.5, 2.0]))
        xf, yf = (f32_from_bf16_bits(t).astype(np.float64) for t in (x, y0))
        ref, bound = yf.copy(), np.zeros_like(yf)
        for i, a in enumerate(ids):
            if 0 <= a < P:
                Af, Bf = (f32_from_bf16_bits(t).astype(np.float64) for t in (As[a], Bs[a]))
                ref[i] = yf[i] + s * (xf[i] @ (Af @ Bf))
                mag = np.abs(yf[i]) + abs(s) * ((np.abs(xf[i]) @ np.abs(Af)) @ np.abs(Bf))
                bound[i] = (h_in + Af.shape[1] + 3) * U32 * mag * 1.01
        y = oracle.sgmv_slots_ref(x, A_ar, B_ar, slots, rank_of, r_max, _mask(ranks), ids, s, y0, mutant=mutant)
        assert np.all(np.abs(y - ref) <= bound), np.max(np.abs(y - ref) - bound)


def pin_slots_zero_padding(mutant=0):
    """Each adapter zero-padded to rank r_max in a contiguous pool gives the
    same values through the (separately pinned) contiguous-pool oracle: the
    extra ranks add exact zeros after the real terms."""
    rng = np.random.default_rng(22)
    n, P, n_slots, h_in, h_out, r_max = 30, 6, 8, 48, 56, 64
    ranks = [8, 16, 32, 64]
    x, A_ar, B_ar, slots, rank_of, As, Bs, y0, ids = slot_problem(rng, n, P, n_slots, h_in, h_out, r_max, ranks)
    A_pad = np.zeros((P, h_in, r_max), np.uint16)
    B_pad = np.zeros((P, r_max, h_out), np.uint16)
    for a in range(P):
        r = int(rank_of[a])
        A_pad[a, :, :r] = As[a]
        B_pad[a, :r, :] = Bs[a]
    y = oracle.sgmv_slots_ref(x, A_ar, B_ar, slots, rank_of, r_max, _mask(ranks), ids, 1.25, y0, mutant=mutant)
    ref = oracle.sgmv_ref(x, A_pad, B_pad, ids, 1.25, y0)
    assert np.array_equal(y, ref)


def pin_slots_invalid_entries(mutant=0):
    """A slot outside the arena, a rank that is not allowed, above the slot
    capacity or not a LoRA rank, and an id outside the table: y = y0."""
    rng = np.random.default_rng(23)
    n, P, n_slots, h_in, h_out, r_max = 16, 7, 8, 32, 24, 32
    x, A_ar, B_ar, slots, rank_of, As, Bs, y0, ids = slot_problem(rng, n, P, n_slots, h_in, h_out, r_max, [8, 16])
    slots[1], slots[2] = n_slots, -1
    rank_of[3], rank_of[4], rank_of[5] = 32, 64, 12  # 32 not in the mask; 64 > r_max; 12 no rank
    ids[:8] = [0, 1, 2, 3, 4, 5, 6, P]
    y, bad = oracle.sgmv_slots_ref(x, A_ar, B_ar, slots, rank_of, r_max, _mask([8, 16]), ids, 1.0, y0,
                                   mutant=mutant, return_invalid=True)
    y0f = f32_from_bf16_bits(y0)
    rows_bad = np.isin(ids, [1, 2, 3, 4, 5, P])
    assert bad == int(rows_bad.sum())
    assert np.array_equal(y[rows_bad], y0f[rows_bad])
    assert not np.array_equal(y[~rows_bad], y0f[~rows_bad])


def pin_slots_relocation(mutant=0):
    """Moving adapters to other slots (and the table with them) changes nothing."""
    rng = np.random.default_rng(24)
    n, P, n_slots, h_in, h_out, r_max = 20, 5, 9, 40, 32, 32
    x, A_ar, B_ar, slots, rank_of, As, Bs, y0, ids = slot_problem(rng, n, P, n_slots, h_in, h_out, r_max,
                                                                  [8, 16, 32])
    y = oracle.sgmv_slots_ref(x, A_ar, B_ar, slots, rank_of, r_max, 7, ids, 0.5, y0, mutant=mutant)
    new = rng.permutation(n_slots)[:P].astype(np.int32)
    A2 = _b(rng.standard_normal(A_ar.shape))
    B2 = _b(rng.standard_normal(B_ar.shape))
    A2[new], B2[new] = A_ar[slots], B_ar[slots]
    y2 = oracle.sgmv_slots_ref(x, A2, B2, new, rank_of, r_max, 7, ids, 0.5, y0, mutant=mutant)
    assert np.array_equal(y, y2)


# ------------------------------------------------------------------ backbone GEMM with the LoRA delta

def pin_gemm_lora_zero_W(mutant=0):
    """W = 0 leaves exactly the delta the (pinned) SGMV oracle computes on y0 = 0."""
    rng = np.random.default_rng(31)
    x, A, B, y0, ids = rand_problem(rng, 12, 4, 48, 40, 8, p_invalid=0.2)
    W = np.zeros((48, 40), np.uint16)
    y = oracle.gemm_lora_ref(x, W, A, B, ids, 1.5, mutant=mutant)
    ref = oracle.sgmv_ref(x, A, B, ids, 1.5, np.zeros_like(y0))
    assert np.array_equal(y, ref)


def pin_gemm_lora_dense(mutant=0):
    """Against y = x.(W + s*A_a.B_a) in fp64 (the dense association), within
    the fp32 forward error bound; invalid ids give the plain product x.W."""
    rng = np.random.default_rng(32)
    for n, P, h_in, h_out, r in [(10, 3, 64, 48, 8), (6, 2, 40, 24, 16)]:
        x, A, B, _, ids = rand_problem(rng, n, P, h_in, h_out, r, p_invalid=0.2)
        W = _b(rng.standard_normal((h_in, h_out)) / np.sqrt(h_in))
        s = float(rng.choice([0.5, -2.0, 1.0]))
        y = oracle.gemm_lora_ref(x, W, A, B, ids, s, mutant=mutant)
        xf, Wf, Af, Bf = (f32_from_bf16_bits(t).astype(np.float64) for t in (x, W, A, B))
        ref = xf @ Wf
        mag = np.abs(xf) @ np.abs(Wf)
        for i, a in enumerate(ids):
            if 0 <= a < P:
                ref[i] += s * (xf[i] @ (Af[a] @ Bf[a]))
                mag[i] += abs(s) * ((np.abs(xf[i]) @ np.abs(Af[a])) @ np.abs(Bf[a]))
        bound = (h_in + r + 3) * U32 * mag * 1.01
        assert np.all(np.abs(y - ref) <= bound), np.max(np.abs(y - ref) - bound)


ALL_PINS = [
    pin_golden_segment,
    pin_golden_sgmv,
    pin_segment_bruteforce,
    pin_dense_bruteforce,
    pin_single_adapter_matmul,
    pin_zero_B,
    pin_permutation,
    pin_linear_in_s,
    pin_rank1_closed_form,
    pin_golden_slots,
    pin_slots_dense_bruteforce,
    pin_slots_zero_padding,
    pin_slots_invalid_entries,
    pin_slots_relocation,
    pin_gemm_lora_zero_W,
    pin_gemm_lora_dense,
]
