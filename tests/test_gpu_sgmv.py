"""SGMV kernels on the GPU against the oracle (through the C ABI binding).

Bar: |y - y_ref| <= 1e-2 + 1e-2*|y_ref| elementwise; exact-arithmetic inputs
and permutations bit-exact; segmentation bit-exact."""

import numpy as np
import pytest
import torch

import adapter_gemm_02_b300 as lsg
import oracle
from tests._gpu import Run, assert_within_tol, check_segments, oracle_rows
from workloads import WORKLOADS, bf16_bits_from_f32, make_inputs

pytestmark = pytest.mark.gpu


def _bf16(a: np.ndarray, device="cuda") -> torch.Tensor:
    bits = bf16_bits_from_f32(np.asarray(a, np.float32))
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(device)


def _torch_fp32_reference(x, A, B, ids: np.ndarray, s, y0):
    """Full-size cross-check with fp32 torch.matmul per adapter (no TF32)."""
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        out = y0.float().clone()
        idt = torch.from_numpy(ids).to(x.device)
        for a in np.unique(ids):
            rows = (idt == int(a)).nonzero().squeeze(1)
            out[rows] = y0[rows].float() + s * ((x[rows].float() @ A[a].float()) @ B[a].float())
        return out.cpu().numpy()
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


# ------------------------------------------------------------ the five workloads

def test_tiny():
    r = Run(WORKLOADS["tiny"])
    check_segments(r.seg, r.ids, 4)
    assert int(r.err.cpu()[0]) == 0
    assert_within_tol(r.y(0), r.ref(0))


@pytest.mark.parametrize("pattern", ["same", "distinct", "zipf"])
def test_7b_projection(pattern):
    r = Run(WORKLOADS[f"7b_proj_{pattern}"])
    check_segments(r.seg, r.ids, 64)
    assert int(r.err.cpu()[0]) == 0
    assert_within_tol(r.y(0), r.ref(0))


def test_7b_layer_all_projections():
    wl = WORKLOADS["7b_layer"]
    r = Run(wl)
    check_segments(r.seg, r.ids, wl.P)
    assert int(r.err.cpu()[0]) == 0
    for i, p in enumerate(wl.projs):
        assert_within_tol(r.y(i), r.ref(i), p.name)


@pytest.mark.parametrize("name", ["13b_prefill", "13b_prefill_interleaved"])
def test_13b_prefill_every_row(name):
    """All 6224 rows of all seven projections against the oracle (the
    oracle's threaded entry point), plus an extra cross-check of every row
    against fp32 torch.matmul; the requests sorted (contiguous rows) and
    interleaved (every segment's rows gathered)."""
    wl = WORKLOADS[name]
    r = Run(wl)
    check_segments(r.seg, r.ids, wl.P)
    assert int(r.err.cpu()[0]) == 0
    for i, p in enumerate(wl.projs):
        assert_within_tol(r.y(i), r.ref(i), p.name)
    for i, p in enumerate(wl.projs):
        full = _torch_fp32_reference(r.inp.x[p.x_key], r.inp.A[i], r.inp.B[i], r.ids, wl.scale, r.y0[i])
        assert_within_tol(r.y(i), full, p.name + " (all rows vs fp32 matmul)")
    del r
    torch.cuda.empty_cache()


@pytest.mark.parametrize("rank", [8, 16, 32, 64])
def test_70b_decode(rank):
    """All 256 rows of all seven projections against the oracle."""
    wl = WORKLOADS[f"70b_decode_r{rank}"]
    r = Run(wl)
    check_segments(r.seg, r.ids, wl.P)
    assert int(r.err.cpu()[0]) == 0
    for i, p in enumerate(wl.projs):
        assert_within_tol(r.y(i), r.ref(i), p.name)
    del r
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mixed", [False, True], ids=["one_adapter", "16_requests"])
def test_13b_projection_4096_tokens(mixed):
    """The largest prefill point of the batch-size curve: one Llama2-13B
    projection (5120 -> 5120, r=64) over 4096 tokens, of one adapter or of 16
    requests of 256 tokens with their own adapters; every row."""
    from workloads import Proj, Workload

    n, P = 4096, 32
    wl = Workload("curve_pre", (Proj("proj", 5120, 5120, "x"),), 64, P, n, 1.0, lambda: None, "", "curve_pre")
    ids = np.repeat(np.arange(16, dtype=np.int32), n // 16) if mixed else np.zeros(n, np.int32)
    r = Run(wl, ids=ids)
    check_segments(r.seg, r.ids, P)
    assert int(r.err.cpu()[0]) == 0
    assert_within_tol(r.y(0), r.ref(0))


# ------------------------------------------------------------ shrink / expand

@pytest.mark.parametrize("name", ["tiny", "7b_proj_same", "7b_proj_distinct", "7b_proj_zipf"])
def test_shrink_then_expand(name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl, "cuda")
    x, A, B, y = inp.x["x"], inp.A[0], inp.B[0], inp.y0[0]
    y0 = y.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seg = lsg.lora_segment(inp.ids, wl.P, err_flag=err)
    v = lsg.sgmv_shrink(x, A, seg, err_flag=err)
    lsg.sgmv_expand(v, B, seg, y, wl.scale, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.cpu()[0]) == 0
    ids = inp.ids.cpu().numpy()
    y_ref, v_ref = oracle.sgmv_ref(x.cpu(), A.cpu(), B.cpu(), ids, wl.scale, y0.cpu(), want_v=True)
    # v: fp32 sums in another order; bound 2*(h_in+2)*u*sum|x*A|
    xa = (x.float().abs() @ A.float().abs().permute(1, 0, 2).reshape(A.shape[1], -1)).cpu().numpy()
    xa = xa.reshape(x.shape[0], A.shape[0], A.shape[2])[np.arange(x.shape[0]), ids]
    vb = 2 * (A.shape[1] + 2) * 2.0 ** -24 * xa + 1e-30
    assert np.all(np.abs(v.cpu().numpy() - v_ref) <= vb)
    assert_within_tol(y, y_ref)


# ------------------------------------------------------------ exactness, invariants

def _int_problem(rng, n, P, h_in, h_out, r):
    x = rng.choice([-1.0, 0.0, 1.0], (n, h_in), p=[0.25, 0.5, 0.25])
    pa = min(0.05, 20.0 / h_in)  # about 40 nonzeros per column of A: small exact sums
    A = rng.choice([-1.0, 0.0, 1.0], (P, h_in, r), p=[pa, 1 - 2 * pa, pa])
    B = rng.choice([-1.0, 0.0, 1.0], (P, r, h_out), p=[0.1, 0.8, 0.1])
    y0 = rng.integers(-8, 9, (n, h_out)).astype(np.float64)
    ids = rng.integers(0, P, n).astype(np.int32)
    return x, A, B, y0, ids


@pytest.mark.parametrize("shape", [(40, 6, 256, 256, 8), (32, 64, 4096, 4096, 16), (9, 3, 1000, 2056, 64),
                                   (128, 16, 8192, 1024, 32)])
def test_exact_arithmetic_is_bit_exact(shape):
    n, P, h_in, h_out, r = shape
    rng = np.random.default_rng(sum(shape))
    x, A, B, y0, ids = _int_problem(rng, n, P, h_in, h_out, r)
    s = 2.0
    xt, At, Bt, yt = _bf16(x), _bf16(A), _bf16(B), _bf16(y0)
    y_ref = oracle.sgmv_ref(xt.cpu(), At.cpu(), Bt.cpu(), ids, s, yt.cpu())
    assert np.all(np.abs(y_ref) <= 256) and np.all(y_ref == np.round(y_ref))  # integers, exact in bf16
    assert np.any(y_ref != yt.float().cpu().numpy())  # the delta is not trivially zero
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P)
    lsg.sgmv_fused(xt, At, Bt, seg, yt, s)
    assert np.array_equal(yt.float().cpu().numpy(), y_ref)


def test_permuting_tokens_permutes_outputs_bit_exactly():
    rng = np.random.default_rng(21)
    n, P, h_in, h_out, r = 48, 12, 4096, 4096, 16
    x = rng.standard_normal((n, h_in))
    A = rng.standard_normal((P, h_in, r)) / 64
    B = rng.standard_normal((P, r, h_out)) / 4
    y0 = rng.standard_normal((n, h_out))
    ids = rng.integers(0, P, n).astype(np.int32)
    perm = rng.permutation(n)
    At, Bt = _bf16(A), _bf16(B)
    outs = []
    for order in (np.arange(n), perm):
        yt = _bf16(y0[order])
        seg = lsg.lora_segment(torch.from_numpy(ids[order].copy()).cuda(), P)
        lsg.sgmv_fused(_bf16(x[order]), At, Bt, seg, yt, 1.0)
        outs.append(yt.cpu())
    assert torch.equal(outs[1], outs[0][torch.from_numpy(perm)])


def test_repeated_calls_are_deterministic():
    wl = WORKLOADS["7b_layer"]
    a = Run(wl)
    b = Run(wl)
    for i in range(len(wl.projs)):
        assert torch.equal(a.y(i), b.y(i))


def test_zero_B_and_zero_scale_leave_y_unchanged():
    wl = WORKLOADS["7b_proj_zipf"]
    inp = make_inputs(wl, "cuda")
    y0 = inp.y0[0].clone()
    seg = lsg.lora_segment(inp.ids, wl.P)
    lsg.sgmv_fused(inp.x["x"], inp.A[0], torch.zeros_like(inp.B[0]), seg, inp.y0[0], 1.0)
    lsg.sgmv_fused(inp.x["x"], inp.A[0], inp.B[0], seg, inp.y0[0], 0.0)
    torch.cuda.synchronize()
    assert torch.equal(inp.y0[0].float(), y0.float())


def test_linear_in_scale():
    wl = WORKLOADS["7b_proj_distinct"]
    inp = make_inputs(wl, "cuda")
    seg = lsg.lora_segment(inp.ids, wl.P)
    outs = []
    for s in (1.0, 2.0):
        y = torch.zeros_like(inp.y0[0])
        lsg.sgmv_fused(inp.x["x"], inp.A[0], inp.B[0], seg, y, s)
        outs.append(y.float())
    # y(2s) = bf16(2*d) = 2*bf16(d) exactly (scaling by 2 commutes with rounding)
    assert torch.equal(outs[1], 2 * outs[0])


# ------------------------------------------------------------ shapes and edges

SHAPES = [  # n, P, h_in, h_out, r
    (5, 3, 8, 8, 8), (37, 9, 24, 40, 16), (19, 4, 200, 1000, 32), (50, 6, 1000, 200, 64),
    (40, 16, 4104, 2056, 16), (64, 8, 11008, 4096, 16), (33, 2, 4096, 11008, 64), (300, 40, 512, 520, 8),
    (1, 1, 64, 64, 16), (100, 3, 256, 256, 32), (100, 100, 512, 512, 8),
]


@pytest.mark.parametrize("shape", SHAPES, ids=["x".join(map(str, s)) for s in SHAPES])
def test_ragged_shapes_padded_rows_and_guard_bands(shape):
    n, P, h_in, h_out, r = shape
    rng = np.random.default_rng(n + 31 * h_in + 7 * h_out + r)
    pad_x, pad_y = 8, 16
    x = _bf16(rng.standard_normal((n, h_in + pad_x)))[:, :h_in]
    A = _bf16(rng.standard_normal((P, h_in, r)) / np.sqrt(h_in))
    B = _bf16(rng.standard_normal((P, r, h_out)) / np.sqrt(r))
    ybuf = _bf16(rng.standard_normal((n + 2, h_out + pad_y)))  # one guard row each side + guard columns
    y = ybuf[1:-1, :h_out]
    before = ybuf.clone()
    ids = rng.integers(0, P, n).astype(np.int32)
    if shape == (100, 3, 256, 256, 32):
        ids[:] = 2  # all tokens one adapter
    if shape == (100, 100, 512, 512, 8):
        ids = rng.permutation(100).astype(np.int32)  # every token its own adapter
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P)
    lsg.sgmv_fused(x, A, B, seg, y, 1.25)
    torch.cuda.synchronize()
    after = ybuf.cpu()
    assert torch.equal(after[0], before[0].cpu()) and torch.equal(after[-1], before[-1].cpu())
    assert torch.equal(after[:, h_out:], before[:, h_out:].cpu())
    y_ref = oracle_rows(x, A, B, ids, 1.25, before[1:-1, :h_out])
    assert_within_tol(y, y_ref)


def test_invalid_adapter_ids_are_skipped_and_flagged():
    rng = np.random.default_rng(8)
    n, P, h = 64, 10, 1024
    ids = rng.integers(0, P, n).astype(np.int32)
    ids[[3, 17, 40]] = [-1, P, 1 << 20]
    x = _bf16(rng.standard_normal((n, h)))
    A = _bf16(rng.standard_normal((P, h, 16)) / 32)
    B = _bf16(rng.standard_normal((P, 16, h)) / 4)
    y = _bf16(rng.standard_normal((n, h)))
    y0 = y.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P, err_flag=err)
    check_segments(seg, ids, P)
    lsg.sgmv_fused(x, A, B, seg, y, 1.0, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.cpu()[0]) == -4
    y_ref = oracle_rows(x, A, B, ids, 1.0, y0)
    assert torch.equal(y[[3, 17, 40]], y0[[3, 17, 40]])
    assert_within_tol(y, y_ref)


def test_corrupt_segment_record_is_flagged_not_trapped():
    rng = np.random.default_rng(9)
    n, P, h = 16, 4, 256
    ids = np.repeat(np.arange(4, dtype=np.int32), 4)
    x = _bf16(rng.standard_normal((n, h)))
    A = _bf16(rng.standard_normal((P, h, 8)) / 16)
    B = _bf16(rng.standard_normal((P, 8, h)) / 3)
    y = _bf16(rng.standard_normal((n, h)))
    y0 = y.clone()
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P)
    torch.cuda.synchronize()
    seg.seg_adapter[1] = 77          # segment 1 names a slab outside the pool
    seg.perm[9] = 1000               # and one permutation entry is out of range
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lsg.sgmv_fused(x, A, B, seg, y, 1.0, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.cpu()[0]) == -4
    assert torch.equal(y[4:8], y0[4:8])  # segment 1's rows untouched
    ok = np.r_[0:4, 8:9, 10:16]
    y_ref = oracle_rows(x, A, B, ids, 1.0, y0)
    assert_within_tol(y[torch.from_numpy(ok).cuda()], y_ref[ok])


def test_zero_tokens_is_a_noop():
    seg = lsg.Segments.empty(0, 4)
    lsg.lora_segment(torch.zeros(0, dtype=torch.int32, device="cuda"), 4, out=seg)
    x = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    A = torch.zeros(4, 64, 16, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(4, 16, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    lsg.sgmv_fused(x, A, B, seg, y, 1.0)
    torch.cuda.synchronize()


def test_host_validation_raises():
    x = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    A = torch.zeros(4, 64, 12, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(4, 12, 64, dtype=torch.bfloat16, device="cuda")
    seg = lsg.lora_segment(torch.zeros(4, dtype=torch.int32, device="cuda"), 4)
    with pytest.raises(RuntimeError, match="UNSUPPORTED"):
        lsg.sgmv_fused(x, A, B, seg, x.clone(), 1.0)


@pytest.mark.parametrize("name", ["7b_proj_distinct", "7b_proj_zipf", "7b_layer", "70b_decode_r16"])
def test_one_call_and_two_calls_agree_bit_for_bit(name):
    """The benchmark's call (segmentation inside the launch for small
    batches) and the two-call path compute the same bits at full size."""
    wl = WORKLOADS[name]
    a = Run(wl, one_call=True)
    b = Run(wl, one_call=False)
    assert int(a.err.item()) == 0 and int(b.err.item()) == 0
    assert torch.equal(a.seg.perm, b.seg.perm) and torch.equal(a.seg.seg_offsets, b.seg.seg_offsets)
    for i in range(len(wl.projs)):
        assert torch.equal(a.y(i), b.y(i)), f"projection {i}"
