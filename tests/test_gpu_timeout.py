"""Bounded waits that run out.  Every wait inside the kernels gives up after a
time limit, records LORA_ERR_TIMEOUT in err_flag and lets the kernel finish;
the context stays usable.  A test build of the library (20 ms limit, hooks
that make a kernel withhold one signal, so that the wait for it can never
complete) is run in a child process:
  1  the decode kernel's producer withholds its end-of-work marker,
  2  CTA 1 of every decode cluster withholds its partial v from its peers,
  3  the tensor-tile kernel withholds its first expand accumulator,
  4  the backbone GEMM (gemm_lora) withholds its first completed accumulators.
Each must end with -7 in err_flag; afterwards, with nothing withheld, the
same process computes a fused SGMV that matches the oracle."""

import os
import subprocess
import sys

import pytest

from adapter_gemm_02_b300 import build as lib_build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import ctypes, sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
import adapter_gemm_02_b300.lora_sgmv as m
lib = m.load_library(sys.argv[2])
lib.lora_test_withhold.restype = ctypes.c_int
lib.lora_test_withhold.argtypes = [ctypes.c_int]
import oracle
from workloads import WORKLOADS, make_inputs

def decode_case():
    wl = WORKLOADS["7b_proj_distinct"]  # 32 tokens of 32 adapters, clusters of 8 CTAs
    inp = make_inputs(wl, "cuda")
    return inp.x["x"], inp.A[0], inp.B[0], inp.y0[0], inp.ids, wl.P

def prefill_case():
    rng = np.random.default_rng(1)
    ids = np.concatenate([np.full(300, 1, np.int32), np.full(70, 0, np.int32)])
    P, h, r = 2, 512, 16
    bf = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).cuda()
    x = bf(rng.standard_normal((ids.size, h)))
    A = bf(rng.standard_normal((P, h, r)) / np.sqrt(h))
    B = bf(rng.standard_normal((P, r, h)) / np.sqrt(r))
    y = bf(rng.standard_normal((ids.size, h)))
    return x, A, B, y, torch.from_numpy(ids).cuda(), P

def gemm_case():
    rng = np.random.default_rng(2)
    ids = np.concatenate([np.full(300, 1, np.int32), np.full(90, 0, np.int32), rng.integers(0, 2, 20).astype(np.int32)])
    P, h_in, h_out, r = 2, 512, 768, 16
    bf = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).cuda()
    x = bf(rng.standard_normal((ids.size, h_in)))
    W = bf(rng.standard_normal((h_in, h_out)) / np.sqrt(h_in))
    A = bf(rng.standard_normal((P, h_in, r)) / np.sqrt(h_in))
    B = bf(rng.standard_normal((P, r, h_out)) / np.sqrt(r))
    return x, W, A, B, torch.from_numpy(ids).cuda(), P

def run_gemm(what):
    x, W, A, B, ids, P = gemm_case()
    assert lib.lora_test_withhold(what) == 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seg = m.lora_segment(ids, P, err_flag=err)
    y = torch.zeros(ids.shape[0], W.shape[1], dtype=torch.bfloat16, device="cuda")
    m.gemm_lora(x, W, A, B, seg, y, 0.5, err_flag=err)
    torch.cuda.synchronize()
    return int(err.item()), (x, W, A, B, y, ids)

def run(case, what):
    x, A, B, y, ids, P = case()
    y0 = y.clone()
    assert lib.lora_test_withhold(what) == 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seg = m.lora_segment(ids, P, err_flag=err)
    m.sgmv_fused(x, A, B, seg, y, 1.0, err_flag=err)
    torch.cuda.synchronize()
    return int(err.item()), (x, A, B, y, y0, ids)

for what, case in ((1, decode_case), (2, decode_case), (3, prefill_case)):
    e, _ = run(case, what)
    print("withheld", what, "err", e, flush=True)
    assert e == -7, (what, e)
e, _ = run_gemm(4)
print("withheld", 4, "err", e, flush=True)
assert e == -7, (4, e)
for case in (decode_case, prefill_case):
    e, (x, A, B, y, y0, ids) = run(case, 0)
    assert e == 0, e
    ref = oracle.sgmv_ref(x.cpu(), A.cpu(), B.cpu(), ids.cpu().numpy(), 1.0, y0.cpu())
    got = y.float().cpu().numpy()
    assert np.all(np.abs(got - ref) <= 1e-2 + 1e-2 * np.abs(ref))
e, (x, W, A, B, y, ids) = run_gemm(0)
assert e == 0, e
ref = oracle.gemm_lora_ref(x.cpu(), W.cpu(), A.cpu(), B.cpu(), ids.cpu().numpy(), 0.5)
got = y.float().cpu().numpy()
assert np.all(np.abs(got - ref) <= 1e-2 + 1e-2 * np.abs(ref))
print("context usable after the time-outs", flush=True)
'''


def test_wait_that_runs_out_reports_timeout_and_context_stays_usable():
    if lib_build.stale(lib_build.TEST_HOOKS_LIB):
        lib_build.build_test_hooks()
    out = subprocess.run([sys.executable, "-c", CHILD, ROOT, lib_build.TEST_HOOKS_LIB], capture_output=True,
                         text=True, timeout=600)
    assert out.returncode == 0, out.stdout + out.stderr[-3000:]
    assert "context usable after the time-outs" in out.stdout
