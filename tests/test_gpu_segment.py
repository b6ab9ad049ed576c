"""lora_segment on the GPU against the oracle: bit-exact."""

import numpy as np
import pytest
import torch

import adapter_gemm_02_b300 as lsg
from tests._gpu import check_segments
from workloads import WORKLOADS

pytestmark = pytest.mark.gpu


def _run(ids: np.ndarray, P: int):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seg = lsg.lora_segment(torch.from_numpy(ids.astype(np.int32)).cuda(), P, err_flag=err)
    ref = check_segments(seg, ids, P)
    return seg, ref, int(err.cpu()[0])


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_segment_every_workload(name):
    wl = WORKLOADS[name]
    _, ref, err = _run(wl.ids(), wl.P)
    assert err == 0 and ref["n_invalid"] == 0


CASES = [
    (0, 4, 0.0), (1, 1, 0.0), (2, 3, 0.0), (31, 64, 0.0), (32, 64, 0.0), (33, 5, 0.0), (64, 1, 0.0),
    # up to 256 tokens: the rank sort, whatever the pool
    (100, 1000, 0.05), (200, 3, 0.2), (255, 1000, 0.0), (256, 1000, 0.1), (256, 70000, 0.0),
    (257, 1000, 0.05), (1000, 7, 0.0), (6224, 32, 0.0), (20000, 300, 0.01), (70000, 100, 0.0),
    (5000, 25000, 0.0),   # largest pool whose histograms stay in shared memory
    (3000, 60000, 0.02),  # histograms in the workspace
]


@pytest.mark.parametrize("n,P,p_bad", CASES, ids=[f"n{c[0]}_P{c[1]}" for c in CASES])
def test_segment_fuzz(n, P, p_bad):
    rng = np.random.default_rng(n * 7919 + P)
    ids = rng.integers(0, P, n).astype(np.int32)
    if p_bad:
        bad = rng.random(n) < p_bad
        ids[bad] = rng.choice([-1, P, P + 3, -1000], int(bad.sum()))
    seg, ref, err = _run(ids, P)
    if ref["n_invalid"]:
        assert err == -4  # LORA_ERR_BAD_ADAPTER_ID
    else:
        assert err == 0


def test_segment_skewed_and_degenerate():
    rng = np.random.default_rng(3)
    for ids, P in [
        (np.zeros(500, np.int32), 10),                          # one segment
        (np.arange(300, dtype=np.int32)[::-1].copy(), 300),     # every token its own adapter, reversed
        (np.repeat(np.arange(5, dtype=np.int32), 100)[::-1].copy(), 5),
        (rng.choice(1000, 4096, p=(lambda p: p / p.sum())(np.arange(1, 1001) ** -1.2)).astype(np.int32), 1000),
        (np.full(77, 99, np.int32), 100),                      # only the last adapter
        (np.full(50, -1, np.int32), 8),                        # every id invalid: no segment
        (np.arange(256, dtype=np.int32)[::-1].copy(), 256),   # 256 tokens, 256 segments, reversed
    ]:
        _run(ids, P)


def test_segment_n0_writes_empty_record():
    seg = lsg.Segments.empty(0, 4)
    seg.num_segments.fill_(-5)
    seg.seg_offsets.fill_(-5)
    lsg.lora_segment(torch.zeros(0, dtype=torch.int32, device="cuda"), 4, out=seg)
    torch.cuda.synchronize()
    assert int(seg.num_segments.cpu()[0]) == 0
    assert int(seg.seg_offsets.cpu()[0]) == 0


def test_segment_repeated_calls_reuse_outputs():
    rng = np.random.default_rng(5)
    seg = lsg.Segments.empty(128, 50)
    for _ in range(3):
        ids = rng.integers(0, 50, 128).astype(np.int32)
        lsg.lora_segment(torch.from_numpy(ids).cuda(), 50, out=seg)
        check_segments(seg, ids, 50)
