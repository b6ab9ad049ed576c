"""Helpers of the GPU parity tests: run the CUDA path through the binding and
the oracle on the same bytes, compare."""

from __future__ import annotations

import os

import numpy as np
import torch

import adapter_gemm_02_b300 as lsg
import oracle
from workloads import make_inputs

TOL_ABS = 1e-2  # parity bar: |y - y_ref| <= 1e-2 + 1e-2 * |y_ref|, elementwise
TOL_REL = 1e-2
THREADS = max(1, min(32, os.cpu_count() or 1))


def assert_within_tol(y_gpu: torch.Tensor, y_ref: np.ndarray, what: str = "y") -> None:
    yg = y_gpu.float().cpu().numpy().astype(np.float64)
    yr = np.asarray(y_ref, dtype=np.float64)
    assert yg.shape == yr.shape, (yg.shape, yr.shape)
    err = np.abs(yg - yr)
    bound = TOL_ABS + TOL_REL * np.abs(yr)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} elements out of tolerance; worst at {i}: "
                             f"gpu={yg[i]} ref={yr[i]}")


def check_segments(seg: lsg.Segments, ids: np.ndarray, P: int) -> dict:
    """GPU segmentation must equal the oracle's bit for bit."""
    ref = oracle.lora_segment_ref(ids, P)
    torch.cuda.synchronize()
    n = ids.size
    ms = min(n, P)
    assert int(seg.num_segments.cpu()[0]) == ref["num_segments"]
    if n:
        assert np.array_equal(seg.perm.cpu().numpy()[:n], ref["perm"])
    assert np.array_equal(seg.seg_offsets.cpu().numpy()[: ms + 1], ref["seg_offsets"])
    if ms:
        assert np.array_equal(seg.seg_adapter.cpu().numpy()[:ms], ref["seg_adapter"])
    return ref


def gather_pools(A: torch.Tensor, B: torch.Tensor, ids: np.ndarray):
    """Slabs of the adapters `ids` uses (host copies) and ids renumbered
    into them; invalid ids stay invalid."""
    P = A.shape[0]
    valid = (ids >= 0) & (ids < P)
    used = np.unique(ids[valid])
    if used.size == 0:
        used = np.zeros(1, np.int64)
    idx = torch.from_numpy(used.astype(np.int64)).to(A.device)
    As, Bs = A.index_select(0, idx).cpu(), B.index_select(0, idx).cpu()
    remap = np.full(ids.shape, -1, np.int32)
    remap[valid] = np.searchsorted(used, ids[valid]).astype(np.int32)
    return As, Bs, remap


def oracle_rows(x, A, B, ids: np.ndarray, scale: float, y0, rows=None):
    """Oracle y for the tokens `rows` (all when None)."""
    rows = np.arange(ids.size) if rows is None else np.asarray(rows)
    sub = ids[rows]
    As, Bs, remap = gather_pools(A, B, sub)
    ridx = torch.from_numpy(rows.astype(np.int64)).to(x.device)
    xs = x.index_select(0, ridx).cpu()
    ys = y0.index_select(0, ridx).cpu()
    return oracle.sgmv_ref(xs, As, Bs, remap, scale, ys, threads=THREADS)


class Run:
    """One workload through the call the benchmark times (sgmv_multi_segment:
    segmentation and SGMV, one launch for small batches), or, with
    one_call=False, through lora_segment + sgmv_fused / sgmv_multi."""

    def __init__(self, wl, ids=None, copy=0, one_call=True):
        self.wl = wl
        self.inp = make_inputs(wl, "cuda", copy=copy, ids=ids)
        self.ids = self.inp.ids.cpu().numpy()
        self.y0 = [y.clone() for y in self.inp.y0]
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        projs = [(self.inp.x[p.x_key], self.inp.A[i], self.inp.B[i], self.inp.y0[i], wl.scale)
                 for i, p in enumerate(wl.projs)]
        if one_call:
            self.seg = lsg.sgmv_multi_segment(projs, self.inp.ids, wl.P, err_flag=self.err)
            torch.cuda.synchronize()
            return
        self.seg = lsg.lora_segment(self.inp.ids, wl.P, err_flag=self.err)
        if len(projs) == 1:
            x, A, B, y, s = projs[0]
            lsg.sgmv_fused(x, A, B, self.seg, y, s, err_flag=self.err)
        else:
            lsg.sgmv_multi(projs, self.seg, err_flag=self.err)
        torch.cuda.synchronize()

    def y(self, i):
        return self.inp.y0[i]

    def ref(self, i, rows=None):
        p = self.wl.projs[i]
        return oracle_rows(self.inp.x[p.x_key], self.inp.A[i], self.inp.B[i], self.ids, self.wl.scale,
                           self.y0[i], rows)
