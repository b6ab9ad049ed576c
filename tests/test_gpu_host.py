"""The whole step from host memory (sgmv_multi_host): pinned host ids, x and
y, pools on the GPU, against the oracle."""

import numpy as np
import pytest
import torch

import adapter_gemm_02_b300 as lsg
import oracle
from tests._gpu import THREADS, assert_within_tol
from workloads import bf16_bits_from_f32

pytestmark = pytest.mark.gpu


def _host(a: np.ndarray) -> torch.Tensor:
    bits = bf16_bits_from_f32(np.asarray(a, np.float32))
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory()


def _dev(a: np.ndarray) -> torch.Tensor:
    return _host(a).cuda()


def test_single_projection_with_padded_host_rows():
    rng = np.random.default_rng(31)
    n, P, h_in, h_out, r = 40, 12, 1024, 520, 16
    ids = rng.integers(0, P, n).astype(np.int32)
    ids[5] = P  # invalid: row untouched, flagged
    x = _host(rng.standard_normal((n, h_in + 24)))
    A = _dev(rng.standard_normal((P, h_in, r)) / np.sqrt(h_in))
    B = _dev(rng.standard_normal((P, r, h_out)) / np.sqrt(r))
    y = _host(rng.standard_normal((n, h_out + 8)))
    y0 = y.clone()
    ids_h = torch.from_numpy(ids).pin_memory()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lsg.sgmv_multi_host([(x[:, :h_in], A, B, y[:, :h_out], 0.5)], ids_h, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == -4
    assert torch.equal(y[:, h_out:], y0[:, h_out:])
    assert torch.equal(y[5], y0[5])
    ref = oracle.sgmv_ref(x[:, :h_in], A.cpu(), B.cpu(), ids, 0.5, y0[:, :h_out], threads=THREADS)
    assert_within_tol(y[:, :h_out], ref)


def test_layer_with_shared_inputs_and_workspace_reuse():
    """q/k/v share one host x (one device copy); the workspace of the first
    call serves the second."""
    rng = np.random.default_rng(32)
    n, P, h, inter, r = 48, 6, 256, 640, 32
    ids = rng.integers(0, P, n).astype(np.int32)
    ids_h = torch.from_numpy(ids).pin_memory()
    xa = _host(rng.standard_normal((n, h)))
    xm = _host(rng.standard_normal((n, h)))
    shapes = [(xa, h, h), (xa, h, h), (xa, h, h), (xm, h, inter), (xm, h, inter)]
    projs, refs = [], []
    for i, (x, hi, ho) in enumerate(shapes):
        A = _dev(rng.standard_normal((P, hi, r)) / np.sqrt(hi))
        B = _dev(rng.standard_normal((P, r, ho)) / np.sqrt(r))
        y = _host(rng.standard_normal((n, ho)))
        projs.append((x, A, B, y, 1.0 + i))
        refs.append(y.clone())
    ws = lsg.sgmv_multi_host(projs, ids_h)
    torch.cuda.synchronize()
    for i, ((x, A, B, y, s), y0) in enumerate(zip(projs, refs)):
        assert_within_tol(y, oracle.sgmv_ref(x, A.cpu(), B.cpu(), ids, s, y0, threads=THREADS), f"proj {i}")
    # second step on the updated y, same workspace
    refs2 = [p[3].clone() for p in projs]
    lsg.sgmv_multi_host(projs, ids_h, workspace=ws)
    torch.cuda.synchronize()
    for i, ((x, A, B, y, s), y0) in enumerate(zip(projs, refs2)):
        assert_within_tol(y, oracle.sgmv_ref(x, A.cpu(), B.cpu(), ids, s, y0, threads=THREADS), f"step 2 proj {i}")


@pytest.mark.parametrize("n", [1, 127, 128, 129, 300])
def test_ids_in_the_launch_or_copied(n):
    """Batches of up to 128 tokens are segmented inside the launch and take
    their ids from the launch's parameters, read when the call is made (so the
    host ids may be rewritten as soon as it returns); larger ones copy the ids
    to the workspace on the stream and segment them first.  Both sides of the
    limit, with an invalid id, against the oracle."""
    rng = np.random.default_rng(40 + n)
    P, h_in, h_out, r = 24, 512, 768, 16
    ids = rng.integers(0, P, n).astype(np.int32)
    ids[n // 2] = -1  # invalid: row untouched, flagged
    x = _host(rng.standard_normal((n, h_in)))
    A = _dev(rng.standard_normal((P, h_in, r)) / np.sqrt(h_in))
    B = _dev(rng.standard_normal((P, r, h_out)) / np.sqrt(r))
    y = _host(rng.standard_normal((n, h_out)))
    y0 = y.clone()
    ids_h = torch.from_numpy(ids.copy()).pin_memory()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lsg.sgmv_multi_host([(x, A, B, y, 0.75)], ids_h, err_flag=err)
    if n <= 128:
        ids_h.fill_(0)  # the launch carries its own copy of the ids
    torch.cuda.synchronize()
    assert int(err.item()) == -4
    assert torch.equal(y[n // 2], y0[n // 2])
    ref = oracle.sgmv_ref(x, A.cpu(), B.cpu(), ids, 0.75, y0, threads=THREADS)
    assert_within_tol(y, ref)
