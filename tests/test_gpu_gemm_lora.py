"""gemm_lora: the backbone projection with the LoRA delta, the expand fused
into the GEMM's accumulator (y = x . W + s * (x . A[a]) . B[a], y written
once), against the oracle's definition of the same (oracle.gemm_lora_ref).

Bar: |y - y_ref| <= 1e-2 + 1e-2*|y_ref| elementwise, x . W ~ N(0, 1) (W drawn
with variance 1/h_in); small-integer inputs bit-exact."""

import numpy as np
import pytest
import torch

import adapter_gemm_02_b300 as lsg
import oracle
from tests._gpu import THREADS, assert_within_tol, check_segments
from workloads import bf16_bits_from_f32, normal_bf16, seed_for

pytestmark = pytest.mark.gpu


def _bf16(a) -> torch.Tensor:
    bits = bf16_bits_from_f32(np.asarray(a, np.float32))
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def _problem(name, ids, P, h_in, h_out, r):
    n = ids.size
    x = normal_bf16((n, h_in), 1.0, seed_for(name, "x"), "cuda")
    W = normal_bf16((h_in, h_out), 1.0 / h_in, seed_for(name, "W"), "cuda")
    A = normal_bf16((P, h_in, r), 1.0 / h_in, seed_for(name, "A"), "cuda")
    B = normal_bf16((P, r, h_out), 1.0 / r, seed_for(name, "B"), "cuda")
    return x, W, A, B


def _run(x, W, A, B, ids, P, s):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P, err_flag=err)
    check_segments(seg, ids, P)
    y = torch.full((ids.size, W.shape[1]), float("nan"), dtype=torch.bfloat16, device="cuda")
    lsg.gemm_lora(x, W, A, B, seg, y, s, err_flag=err)
    torch.cuda.synchronize()
    return y, int(err.item())


def _ref(x, W, A, B, ids, s, rows=None):
    rows = np.arange(ids.size) if rows is None else np.asarray(rows)
    ridx = torch.from_numpy(rows.astype(np.int64)).cuda()
    return oracle.gemm_lora_ref(x.index_select(0, ridx).cpu(), W.cpu(), A.cpu(), B.cpu(), ids[rows], s,
                                threads=THREADS)


def _requests(lens, adapters, interleave=False):
    if not interleave:
        return np.concatenate([np.full(l, a, np.int32) for l, a in zip(lens, adapters)])
    queues = [list(np.full(l, a, np.int32)) for l, a in zip(lens, adapters)]
    out = []
    while any(queues):
        for qu in queues:
            if qu:
                out.append(qu.pop())
    return np.asarray(out, np.int32)


@pytest.mark.parametrize("r", [8, 16, 64])
def test_prefill_requests_every_row(r):
    """Sorted prefill requests (contiguous rows, ragged last column tile)."""
    ids = _requests([300, 129, 64, 211], [3, 0, 5, 1])
    P, h_in, h_out = 6, 1024, 1000
    x, W, A, B = _problem(f"gl_prefill_{r}", ids, P, h_in, h_out, r)
    y, err = _run(x, W, A, B, ids, P, 0.5)
    assert err == 0
    assert_within_tol(y, _ref(x, W, A, B, ids, 0.5))


@pytest.mark.parametrize("r", [16, 32])
def test_interleaved_short_and_invalid_every_row(r):
    """Interleaved long requests (gathered rows), short segments (their delta
    added by the split-K kernel after the GEMM) and invalid ids (y = x . W,
    flagged)."""
    rng = np.random.default_rng(r)
    ids = np.concatenate([_requests([200, 150, 90], [2, 7, 4], interleave=True),
                          rng.integers(0, 9, 40).astype(np.int32), np.array([-1, 9, 12], np.int32)])
    ids = ids[rng.permutation(ids.size)]
    P, h_in, h_out = 9, 768, 1280
    x, W, A, B = _problem(f"gl_mixed_{r}", ids, P, h_in, h_out, r)
    y, err = _run(x, W, A, B, ids, P, 1.25)
    assert err == -4
    assert_within_tol(y, _ref(x, W, A, B, ids, 1.25))


@pytest.mark.parametrize("n,interleave,r", [(2100, False, 64), (2100, True, 16), (3072, True, 32), (2100, False, 8)])
def test_units_of_two_token_tiles_every_row(n, interleave, r):
    """Batches large enough for units of two token tiles (256 tokens x 256
    columns) on every SM.  2100 tokens over 20 column tiles: 17 tiles, 180
    pairs, so one whole wave of pairs and the 32 pairs left over split into
    single tiles, the last tile ragged and without a partner; 3072 tokens: 240
    pairs, the 92 left over fill more than half a wave and stay pairs.
    Requests sorted (contiguous rows) or interleaved (gathered rows), with
    short segments and an invalid id; every row against the oracle."""
    rng = np.random.default_rng(n + r)
    lens = [n // 3, n // 4, n // 5, n // 8]
    lens.append(n - 31 - sum(lens))
    ids = np.concatenate([_requests(lens, [4, 1, 7, 2, 5], interleave),
                          rng.integers(0, 9, 30).astype(np.int32), np.array([-1], np.int32)])
    if interleave:
        ids = ids[rng.permutation(ids.size)]
    P, h_in, h_out = 9, 512, 5120
    x, W, A, B = _problem(f"gl_pairs_{n}_{r}", ids, P, h_in, h_out, r)
    y, err = _run(x, W, A, B, ids, P, 0.75)
    assert err == -4
    assert_within_tol(y, _ref(x, W, A, B, ids, 0.75))


@pytest.mark.parametrize("h_in,h_out", [(768, 576), (1000, 1000)])
def test_padded_rows_and_partial_column_tiles(h_in, h_out):
    """x and y with row strides past their widths (y's padding must stay
    untouched by the box stores), and a last column tile that runs past h_out:
    576 = 9 x 64 (W as one 3-D box per stage, its blocks past h_out read as
    zeros) or 1000 (W by 64-column boxes, the last one partly past h_out).
    h_in = 1000: the last k-block is partial (x columns and W rows past h_in
    read as zeros, in the GEMM and in the shrink)."""
    ids = _requests([300, 200, 100, 40], [2, 0, 3, 1])
    n, P, r = ids.size, 4, 32
    ldx, ldy = h_in + 64, h_out + 136
    x_full = normal_bf16((n, ldx), 1.0, seed_for(f"gl_pad_{h_in}_{h_out}", "x"), "cuda")
    x = x_full[:, :h_in]
    W = normal_bf16((h_in, h_out), 1.0 / h_in, seed_for(f"gl_pad_{h_in}_{h_out}", "W"), "cuda")
    A = normal_bf16((P, h_in, r), 1.0 / h_in, seed_for(f"gl_pad_{h_in}_{h_out}", "A"), "cuda")
    B = normal_bf16((P, r, h_out), 1.0 / r, seed_for(f"gl_pad_{h_in}_{h_out}", "B"), "cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P, err_flag=err)
    y_full = torch.full((n, ldy), 7.0, dtype=torch.bfloat16, device="cuda")
    y = y_full[:, :h_out]
    lsg.gemm_lora(x, W, A, B, seg, y, 1.5, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert bool((y_full[:, h_out:] == 7.0).all())
    assert_within_tol(y, _ref(x, W, A, B, ids, 1.5))


@pytest.mark.parametrize("interleave", [False, True])
def test_many_long_segments_per_unit_every_row(interleave):
    """Segments of 64-130 tokens: each 128-token window overlaps two or three
    of them, so a unit of two tiles carries four to six long-segment expands
    (each with its own operand and B tile slot) after its main loop; 2048
    tokens over 20 column tiles make 160 units of two tiles (one whole wave
    and single tiles after it).  Every row against the oracle."""
    rng = np.random.default_rng(11 + int(interleave))
    lens, total = [], 0
    while total < 2048 - 130:
        lens.append(int(rng.integers(64, 131)))
        total += lens[-1]
    lens.append(2048 - total)
    P = len(lens) + 2
    adapters = rng.permutation(P)[:len(lens)]
    ids = _requests(lens, adapters, interleave)
    h_in, h_out, r = 512, 5120, 16
    x, W, A, B = _problem(f"gl_many_{int(interleave)}", ids, P, h_in, h_out, r)
    y, err = _run(x, W, A, B, ids, P, 0.8)
    assert err == 0
    assert_within_tol(y, _ref(x, W, A, B, ids, 0.8))


def test_decode_batch_every_row():
    """A decode batch (every segment short): the GEMM writes x . W and the
    split-K kernel adds every token's delta."""
    ids = np.random.default_rng(3).integers(0, 64, 96).astype(np.int32)
    P, h_in, h_out = 64, 1024, 768
    x, W, A, B = _problem("gl_decode", ids, P, h_in, h_out, 16)
    y, err = _run(x, W, A, B, ids, P, 1.0)
    assert err == 0
    assert_within_tol(y, _ref(x, W, A, B, ids, 1.0))


def test_exact_arithmetic_is_bit_exact():
    """Small-integer inputs: every sum is exact in fp32 and every result an
    integer exact in bf16, so the fused path equals the oracle bit for bit."""
    rng = np.random.default_rng(17)
    ids = _requests([260, 130, 70], [1, 0, 2], interleave=True)
    n, P, h_in, h_out, r = ids.size, 3, 512, 768, 32
    x = rng.choice([-1.0, 0.0, 1.0], (n, h_in), p=[0.2, 0.6, 0.2])
    W = rng.choice([-1.0, 0.0, 1.0], (h_in, h_out), p=[0.03, 0.94, 0.03])
    A = rng.choice([-1.0, 0.0, 1.0], (P, h_in, r), p=[0.02, 0.96, 0.02])
    B = rng.choice([-1.0, 0.0, 1.0], (P, r, h_out), p=[0.1, 0.8, 0.1])
    xt, Wt, At, Bt = _bf16(x), _bf16(W), _bf16(A), _bf16(B)
    y_ref = oracle.gemm_lora_ref(xt.cpu(), Wt.cpu(), At.cpu(), Bt.cpu(), ids, 2.0, threads=THREADS)
    assert np.all(np.abs(y_ref) <= 256) and np.all(y_ref == np.round(y_ref))
    y, err = _run(xt, Wt, At, Bt, ids, P, 2.0)
    assert err == 0
    assert np.array_equal(y.float().cpu().numpy(), y_ref)


def test_llama2_13b_q_projection_full_size():
    """The Llama2-13B prefill batch (8 requests, 6224 tokens) through the q
    projection (5120 -> 5120, r=64): tile-edge and random rows against the
    oracle, every row against fp32 torch.matmul of the same definition."""
    from workloads import prefill_ids

    ids = prefill_ids()
    P, h, r = 32, 5120, 64
    x, W, A, B = _problem("gl_13b_q", ids, P, h, h, r)
    y, err = _run(x, W, A, B, ids, P, 1.0)
    assert err == 0
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(0, ids.size, 127), [ids.size - 1], rng.integers(0, ids.size, 24)]))
    assert_within_tol(y[torch.from_numpy(rows).cuda()], _ref(x, W, A, B, ids, 1.0, rows))
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        full = x.float() @ W.float()
        idt = torch.from_numpy(ids).cuda()
        for a in np.unique(ids):
            sel = (idt == int(a)).nonzero().squeeze(1)
            full[sel] += (x[sel].float() @ A[a].float()) @ B[a].float()
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    assert_within_tol(y, full.cpu().numpy(), "all rows vs fp32 matmul")
