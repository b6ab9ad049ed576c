"""sgmv_multi_segment: segmentation and SGMV in one call (one launch for
batches of up to 128 tokens over pools of up to 1024 adapters).  The written segmentation must equal the oracle's bit for
bit, y must match the oracle, and the result must be bit-identical to the
two-call path (lora_segment, then sgmv_fused / sgmv_multi)."""

import numpy as np
import pytest
import torch

import adapter_gemm_02_b300 as lsg
from tests._gpu import assert_within_tol, check_segments, oracle_rows
from workloads import bf16_bits_from_f32, zipf_ids

pytestmark = pytest.mark.gpu


def _bf16(a):
    bits = bf16_bits_from_f32(np.asarray(a, np.float32))
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def _problem(rng, ids, P, h_in, h_out, r):
    n = ids.size
    x = _bf16(rng.standard_normal((n, h_in)))
    A = _bf16(rng.standard_normal((P, h_in, r)) / np.sqrt(h_in))
    B = _bf16(rng.standard_normal((P, r, h_out)) / np.sqrt(r))
    y = _bf16(rng.standard_normal((n, h_out)))
    return x, A, B, y


CASES = {
    "tiny": (np.array([3, 1, 0, 2, 3, 3, 1, 0, 2, 2, 3, 1, 3, 2, 3, 3], np.int32), 4, 256, 256, 8),
    "one_token": (np.array([5], np.int32), 8, 512, 512, 16),
    "distinct_32_of_64": (np.random.default_rng(0).choice(64, 32, replace=False).astype(np.int32), 64, 1024, 1024, 16),
    "zipf_256_of_1000": (zipf_ids(256, 1000, 0.8, seed=3), 1000, 512, 768, 32),
    "invalid_ids": (np.array([2, -1, 0, 7, 2, 9, 1, 1, -5, 0], np.int32), 7, 256, 384, 64),
    "limit_128_of_1024": (np.random.default_rng(1).integers(0, 1024, 128).astype(np.int32), 1024, 128, 256, 16),
    "over_limit_129": (np.random.default_rng(4).integers(0, 300, 129).astype(np.int32), 300, 128, 256, 16),
    "over_limit_1024_of_4096": (np.random.default_rng(1).integers(0, 4096, 1024).astype(np.int32), 4096, 128, 256,
                                16),
    "over_limit_tokens": (np.random.default_rng(2).integers(0, 40, 1500).astype(np.int32), 40, 128, 128, 16),
    "over_limit_pool": (np.random.default_rng(3).integers(0, 5000, 64).astype(np.int32), 5000, 128, 128, 8),
    "prefill_long_segments": (np.repeat(np.array([1, 0], np.int32), [300, 200]), 2, 512, 640, 32),
    "all_invalid": (np.array([3, 3, -1, 7, 3], np.int32), 3, 256, 256, 16),
    "one_adapter_pool": (np.zeros(37, np.int32), 1, 512, 256, 32),
    # up to 64 tokens the kernel ranks ids in registers: duplicates, invalid
    # ids and both sizes of that path
    "rank_sort_32_dups": (np.random.default_rng(5).integers(-1, 6, 32).astype(np.int32), 5, 256, 256, 16),
    "rank_sort_33": (np.random.default_rng(6).integers(0, 9, 33).astype(np.int32), 9, 256, 256, 16),
    "rank_sort_64_dups_invalid": (np.where(np.random.default_rng(7).random(64) < 0.1, 40,
                                           np.random.default_rng(8).integers(0, 12, 64)).astype(np.int32),
                                  12, 256, 512, 32),
    "rank_sort_64_distinct": (np.random.default_rng(9).permutation(200)[:64].astype(np.int32), 200, 256, 256, 8),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_one_call_matches_oracle_and_two_calls(name):
    ids, P, h_in, h_out, r = CASES[name]
    rng = np.random.default_rng(len(name))
    x, A, B, y = _problem(rng, ids, P, h_in, h_out, r)
    y0 = y.clone()
    y2 = y.clone()
    d_ids = torch.from_numpy(ids).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seg = lsg.sgmv_fused_segment(x, A, B, d_ids, y, 0.75, err_flag=err)
    torch.cuda.synchronize()
    expect_err = -4 if np.any((ids < 0) | (ids >= P)) else 0
    assert int(err.item()) == expect_err
    check_segments(seg, ids, P)
    # the two-call path on the same inputs gives the same bits
    err2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    seg2 = lsg.lora_segment(d_ids, P, err_flag=err2)
    lsg.sgmv_fused(x, A, B, seg2, y2, 0.75, err_flag=err2)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    rows = np.arange(ids.size) if ids.size <= 512 else np.random.default_rng(9).choice(ids.size, 256, replace=False)
    assert_within_tol(y[torch.from_numpy(rows).cuda()], oracle_rows(x, A, B, ids, 0.75, y0, rows))


def test_multi_projection_one_call():
    rng = np.random.default_rng(77)
    ids = zipf_ids(64, 128, 1.0, seed=5)
    P, r, h, inter = 128, 16, 256, 704
    d_ids = torch.from_numpy(ids).cuda()
    xa = _bf16(rng.standard_normal((ids.size, h)))
    projs, refs = [], []
    for i, (hi, ho) in enumerate([(h, h), (h, h), (h, inter)]):
        A = _bf16(rng.standard_normal((P, hi, r)) / np.sqrt(hi))
        B = _bf16(rng.standard_normal((P, r, ho)) / np.sqrt(r))
        y = _bf16(rng.standard_normal((ids.size, ho)))
        refs.append(y.clone())
        projs.append((xa, A, B, y, 1.0 + i))
    seg = lsg.sgmv_multi_segment(projs, d_ids, P)
    torch.cuda.synchronize()
    check_segments(seg, ids, P)
    for i, ((x, A, B, y, s), y0) in enumerate(zip(projs, refs)):
        assert_within_tol(y, oracle_rows(x, A, B, ids, s, y0), f"projection {i}")


def test_zero_tokens_writes_an_empty_segmentation():
    rng = np.random.default_rng(3)
    x, A, B, y = _problem(rng, np.zeros(1, np.int32), 4, 256, 256, 16)
    ids = torch.zeros(0, dtype=torch.int32, device="cuda")
    seg = lsg.Segments.empty(0, 4, "cuda")
    seg.num_segments.fill_(-1)
    lsg.sgmv_multi_segment([(x[:0], A, B, y[:0], 1.0)], ids, 4, out=seg)
    torch.cuda.synchronize()
    assert int(seg.num_segments.item()) == 0
    assert int(seg.seg_offsets[0].item()) == 0
