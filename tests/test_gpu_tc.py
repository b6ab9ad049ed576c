"""Long-segment (prefill) batches through sgmv_fused / sgmv_multi /
sgmv_shrink / sgmv_expand against the oracle.  Segments of at least 64 tokens
take the tensor-tile kernel: tiles of contiguous rows by whole-tile tensor
copies, others (tokens of one adapter spread over the batch) by four-row
gathers through the permutation; short segments take the split-K kernel in
the same call, so these batches exercise the split of one batch between the
two and the edges of the 128-token tiles."""

import numpy as np
import pytest
import torch

import adapter_gemm_02_b300 as lsg
from tests._gpu import assert_within_tol, check_segments, oracle_rows
from workloads import bf16_bits_from_f32

pytestmark = pytest.mark.gpu


def _bf16(a: np.ndarray) -> torch.Tensor:
    bits = bf16_bits_from_f32(np.asarray(a, np.float32))
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def _mixed_ids(rng):
    """Contiguous runs of 300 (adapter 0), 5 (1), 77 (3), 128 (4), 64 (5) and
    63 (6) tokens, plus 140 tokens of adapter 2 interleaved with 140 of adapter
    7 (long but not contiguous)."""
    ids = [np.full(300, 0), np.full(5, 1)]
    inter = np.empty(280, np.int64)
    inter[0::2], inter[1::2] = 2, 7
    ids += [inter, np.full(77, 3), np.full(128, 4), np.full(64, 5), np.full(63, 6)]
    return np.concatenate(ids).astype(np.int32)


@pytest.mark.parametrize("r", [8, 16, 32, 64])
@pytest.mark.parametrize("h_in,h_out", [(520, 1000), (1024, 384), (136, 2056)])
def test_mixed_long_short_interleaved(r, h_in, h_out):
    rng = np.random.default_rng(r * 1000 + h_in + h_out)
    ids = _mixed_ids(rng)
    n, P = ids.size, 9
    x = _bf16(rng.standard_normal((n, h_in)))
    A = _bf16(rng.standard_normal((P, h_in, r)) / np.sqrt(h_in))
    B = _bf16(rng.standard_normal((P, r, h_out)) / np.sqrt(r))
    y = _bf16(rng.standard_normal((n, h_out)))
    y0 = y.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P, err_flag=err)
    check_segments(seg, ids, P)
    lsg.sgmv_fused(x, A, B, seg, y, 0.75, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_within_tol(y, oracle_rows(x, A, B, ids, 0.75, y0))


def test_shuffled_prefill_requests_and_padded_rows():
    """Requests stored in a shuffled order with padded row strides: each
    request's tokens stay contiguous, segments gather them."""
    rng = np.random.default_rng(5)
    lens = [200, 96, 131, 64, 40]
    adapters = [3, 1, 3, 0, 2]  # adapter 3 has two requests: its segment is not contiguous
    ids = np.concatenate([np.full(l, a, np.int32) for l, a in zip(lens, adapters)])
    n, P, h_in, h_out, r = ids.size, 4, 640, 1152, 64
    x = _bf16(rng.standard_normal((n, h_in + 16)))[:, :h_in]
    A = _bf16(rng.standard_normal((P, h_in, r)) / np.sqrt(h_in))
    B = _bf16(rng.standard_normal((P, r, h_out)) / np.sqrt(r))
    ybuf = _bf16(rng.standard_normal((n + 2, h_out + 24)))
    y = ybuf[1:-1, :h_out]
    before = ybuf.clone()
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P)
    lsg.sgmv_fused(x, A, B, seg, y, 1.5)
    torch.cuda.synchronize()
    after = ybuf.cpu()
    assert torch.equal(after[0], before[0].cpu()) and torch.equal(after[-1], before[-1].cpu())
    assert torch.equal(after[:, h_out:], before[:, h_out:].cpu())
    assert_within_tol(y, oracle_rows(x, A, B, ids, 1.5, before[1:-1, :h_out]))


def test_multi_projection_prefill_with_chunked_outputs():
    """Seven projections, one of them wide enough to be split into column
    chunks, shared inputs as in a transformer layer."""
    rng = np.random.default_rng(11)
    ids = np.concatenate([np.full(190, 2, np.int32), np.full(70, 0, np.int32), np.full(3, 1, np.int32)])
    n, P, r, h, inter = ids.size, 3, 32, 512, 11264
    shapes = [(h, h, "a"), (h, h, "a"), (h, h, "a"), (h, h, "o"), (h, inter, "m"), (h, inter, "m"), (inter, h, "d")]
    xs = {"a": _bf16(rng.standard_normal((n, h))), "o": _bf16(rng.standard_normal((n, h))),
          "m": _bf16(rng.standard_normal((n, h))), "d": _bf16(rng.standard_normal((n, inter)))}
    projs, refs = [], []
    for hi, ho, key in shapes:
        A = _bf16(rng.standard_normal((P, hi, r)) / np.sqrt(hi))
        B = _bf16(rng.standard_normal((P, r, ho)) / np.sqrt(r))
        y = _bf16(rng.standard_normal((n, ho)))
        refs.append((xs[key], A, B, y.clone()))
        projs.append((xs[key], A, B, y, 1.0))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P, err_flag=err)
    lsg.sgmv_multi(projs, seg, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for i, ((x, A, B, y0), p) in enumerate(zip(refs, projs)):
        assert_within_tol(p[3], oracle_rows(x, A, B, ids, 1.0, y0), f"projection {i}")


def test_long_segment_with_invalid_adapter_is_skipped_and_flagged():
    rng = np.random.default_rng(12)
    ids = np.concatenate([np.full(150, 1, np.int32), np.full(100, 9, np.int32), np.full(70, 0, np.int32)])
    n, P, h_in, h_out, r = ids.size, 3, 256, 384, 16
    x = _bf16(rng.standard_normal((n, h_in)))
    A = _bf16(rng.standard_normal((P, h_in, r)) / 16)
    B = _bf16(rng.standard_normal((P, r, h_out)) / 4)
    y = _bf16(rng.standard_normal((n, h_out)))
    y0 = y.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P, err_flag=err)
    lsg.sgmv_fused(x, A, B, seg, y, 1.0, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == -4
    assert torch.equal(y[150:250], y0[150:250])
    assert_within_tol(y, oracle_rows(x, A, B, ids, 1.0, y0))


def test_exact_arithmetic_prefill_is_bit_exact():
    """Small-integer inputs: every product and sum is exact in fp32 and the
    results are integers exact in bf16, so the tensor-tile path must equal
    the oracle bit for bit."""
    rng = np.random.default_rng(13)
    ids = np.concatenate([np.full(260, 0, np.int32), np.full(130, 1, np.int32)])
    n, P, h_in, h_out, r = ids.size, 2, 1024, 640, 64
    x = rng.choice([-1.0, 0.0, 1.0], (n, h_in), p=[0.25, 0.5, 0.25])
    A = rng.choice([-1.0, 0.0, 1.0], (P, h_in, r), p=[0.02, 0.96, 0.02])
    B = rng.choice([-1.0, 0.0, 1.0], (P, r, h_out), p=[0.1, 0.8, 0.1])
    y0 = rng.integers(-8, 9, (n, h_out)).astype(np.float64)
    xt, At, Bt, yt = _bf16(x), _bf16(A), _bf16(B), _bf16(y0)
    import oracle

    y_ref = oracle.sgmv_ref(xt.cpu(), At.cpu(), Bt.cpu(), ids, 2.0, yt.cpu())
    assert np.all(np.abs(y_ref) <= 256) and np.all(y_ref == np.round(y_ref))
    assert np.any(y_ref != yt.float().cpu().numpy())
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P)
    lsg.sgmv_fused(xt, At, Bt, seg, yt, 2.0)
    assert np.array_equal(yt.float().cpu().numpy(), y_ref)


@pytest.mark.parametrize("r", [16, 64])
def test_small_prefill_batches_split_over_a_cluster(r):
    """A few 128-token tiles of one wide projection: the items are shared by
    the CTAs of a cluster (split-K shrink, split-N expand, partial v summed
    across the cluster), with ragged tiles and a segment below the tile size."""
    rng = np.random.default_rng(40 + r)
    ids = np.concatenate([np.full(300, 1, np.int32), np.full(70, 0, np.int32)])
    n, P, h_in, h_out = ids.size, 2, 1024, 2048
    x = _bf16(rng.standard_normal((n, h_in)))
    A = _bf16(rng.standard_normal((P, h_in, r)) / np.sqrt(h_in))
    B = _bf16(rng.standard_normal((P, r, h_out)) / np.sqrt(r))
    y = _bf16(rng.standard_normal((n, h_out)))
    y0 = y.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P, err_flag=err)
    lsg.sgmv_fused(x, A, B, seg, y, 0.5, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_within_tol(y, oracle_rows(x, A, B, ids, 0.5, y0))


def test_many_items_take_one_cta_per_item():
    """Ten tiles x eight projections fill the machine without a cluster."""
    rng = np.random.default_rng(41)
    ids = np.concatenate([np.full(l, a, np.int32) for a, l in [(0, 500), (2, 380), (1, 320)]])
    n, P, r, h = ids.size, 3, 32, 256
    projs, refs = [], []
    x = _bf16(rng.standard_normal((n, h)))
    for i in range(8):
        A = _bf16(rng.standard_normal((P, h, r)) / np.sqrt(h))
        B = _bf16(rng.standard_normal((P, r, 512)) / np.sqrt(r))
        y = _bf16(rng.standard_normal((n, 512)))
        refs.append((A, B, y.clone()))
        projs.append((x, A, B, y, 0.25 * (i + 1)))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P, err_flag=err)
    lsg.sgmv_multi(projs, seg, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for i, ((A, B, y0), p) in enumerate(zip(refs, projs)):
        assert_within_tol(p[3], oracle_rows(x, A, B, ids, p[4], y0), f"projection {i}")


def _interleaved_requests(rng, lens, adapters):
    """Requests of the given lengths and adapters whose tokens are dealt out
    round robin over the batch (no segment's rows are contiguous)."""
    queues = [list(np.full(l, a, np.int32)) for l, a in zip(lens, adapters)]
    ids = []
    while any(queues):
        for qu in queues:
            if qu:
                ids.append(qu.pop())
    return np.asarray(ids, np.int32)


@pytest.mark.parametrize("r", [8, 16, 64])
def test_interleaved_prefill_requests_every_row(r):
    """A prefill batch of 1,664 tokens whose eight requests' tokens are
    interleaved: every segment is long and gathered; every row checked."""
    rng = np.random.default_rng(70 + r)
    lens = [300, 128, 257, 190, 64, 333, 200, 192]
    ids = _interleaved_requests(rng, lens, [5, 0, 7, 2, 6, 1, 3, 4])
    n, P, h_in, h_out = ids.size, 8, 1024, 1536
    x = _bf16(rng.standard_normal((n, h_in)))
    A = _bf16(rng.standard_normal((P, h_in, r)) / np.sqrt(h_in))
    B = _bf16(rng.standard_normal((P, r, h_out)) / np.sqrt(r))
    y = _bf16(rng.standard_normal((n, h_out)))
    y0 = y.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P, err_flag=err)
    check_segments(seg, ids, P)
    lsg.sgmv_fused(x, A, B, seg, y, 0.5, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_within_tol(y, oracle_rows(x, A, B, ids, 0.5, y0))


def _chunked_requests(lens, adapters, g):
    """Requests dealt out round robin in chunks of g tokens: each segment is a
    sequence of runs of contiguous rows."""
    left = list(lens)
    ids = []
    while any(left):
        for k, a in enumerate(adapters):
            t = min(g, left[k])
            ids.extend([a] * t)
            left[k] -= t
    return np.asarray(ids, np.int32)


@pytest.mark.parametrize("r", [16, 64])
@pytest.mark.parametrize("g", [96, 128, 160])
def test_requests_in_runs_every_row(r, g):
    """Requests in runs of g tokens: tiles inside one run move by whole-tile
    copies, tiles that straddle two runs gather their rows; every row is
    compared with the oracle, and the last run ends at the batch's last row."""
    rng = np.random.default_rng(90 + r + g)
    lens = [400, 256, 333, 129]
    ids = _chunked_requests(lens, [3, 0, 2, 1], g)
    n, P, h_in, h_out = ids.size, 4, 704, 1088
    x = _bf16(rng.standard_normal((n, h_in)))
    A = _bf16(rng.standard_normal((P, h_in, r)) / np.sqrt(h_in))
    B = _bf16(rng.standard_normal((P, r, h_out)) / np.sqrt(r))
    y = _bf16(rng.standard_normal((n, h_out)))
    y0 = y.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P, err_flag=err)
    check_segments(seg, ids, P)
    lsg.sgmv_fused(x, A, B, seg, y, 0.5, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_within_tol(y, oracle_rows(x, A, B, ids, 0.5, y0))


def test_exact_arithmetic_gathered_prefill_is_bit_exact():
    """Small-integer inputs on interleaved long segments: exact sums, so the
    gathered tensor-tile path equals the oracle bit for bit."""
    rng = np.random.default_rng(71)
    ids = _interleaved_requests(rng, [260, 200, 130], [1, 0, 2])
    n, P, h_in, h_out, r = ids.size, 3, 1024, 640, 64
    x = rng.choice([-1.0, 0.0, 1.0], (n, h_in), p=[0.25, 0.5, 0.25])
    A = rng.choice([-1.0, 0.0, 1.0], (P, h_in, r), p=[0.02, 0.96, 0.02])
    B = rng.choice([-1.0, 0.0, 1.0], (P, r, h_out), p=[0.1, 0.8, 0.1])
    y0 = rng.integers(-8, 9, (n, h_out)).astype(np.float64)
    xt, At, Bt, yt = _bf16(x), _bf16(A), _bf16(B), _bf16(y0)
    import oracle

    y_ref = oracle.sgmv_ref(xt.cpu(), At.cpu(), Bt.cpu(), ids, 2.0, yt.cpu())
    assert np.all(np.abs(y_ref) <= 256) and np.all(y_ref == np.round(y_ref))
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P)
    lsg.sgmv_fused(xt, At, Bt, seg, yt, 2.0)
    assert np.array_equal(yt.float().cpu().numpy(), y_ref)


@pytest.mark.parametrize("r", [8, 16, 64])
@pytest.mark.parametrize("gathered", [False, True], ids=["contiguous", "gathered"])
def test_shrink_then_expand_long_segments(r, gathered):
    """Standalone shrink (v to device memory) and expand (v from device
    memory) on prefill segments: v within the fp32 summation bound of the
    oracle's v, y within the parity tolerance."""
    import oracle

    rng = np.random.default_rng(80 + r + gathered)
    lens, ads = [400, 128, 77, 300], [2, 0, 3, 1]
    ids = _interleaved_requests(rng, lens, ads) if gathered else \
        np.concatenate([np.full(l, a, np.int32) for l, a in zip(lens, ads)])
    n, P, h_in, h_out = ids.size, 4, 2048, 1024
    x = _bf16(rng.standard_normal((n, h_in)))
    A = _bf16(rng.standard_normal((P, h_in, r)) / np.sqrt(h_in))
    B = _bf16(rng.standard_normal((P, r, h_out)) / np.sqrt(r))
    y = _bf16(rng.standard_normal((n, h_out)))
    y0 = y.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seg = lsg.lora_segment(torch.from_numpy(ids).cuda(), P, err_flag=err)
    v = lsg.sgmv_shrink(x, A, seg, err_flag=err)
    lsg.sgmv_expand(v, B, seg, y, 1.5, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    y_ref, v_ref = oracle.sgmv_ref(x.cpu(), A.cpu(), B.cpu(), ids, 1.5, y0.cpu(), want_v=True)
    xa = (x.float().abs() @ A.float().abs().permute(1, 0, 2).reshape(h_in, -1)).cpu().numpy()
    xa = xa.reshape(n, P, r)[np.arange(n), ids]
    vb = 2 * (h_in + 2) * 2.0 ** -24 * xa + 1e-30
    assert np.all(np.abs(v.cpu().numpy() - v_ref) <= vb)
    assert_within_tol(y, y_ref)
