"""lora_segment_noalloc, for callers that cannot allocate device memory (a
framework owns the allocator, memory was planned up front, or a plugin gets
only its input and output buffers): called through the C ABI, its output must
equal lora_segment's bit for bit (segmentation is integer work), on two calls
in a row, including a pool large enough that the library's own device scratch
array replaces lora_segment's workspace.  Kept in its own file so that it runs
after every other test."""

import ctypes

import numpy as np
import pytest
import torch

import adapter_gemm_02_b300 as lsg

pytestmark = pytest.mark.gpu


def _noalloc(lib, ids: torch.Tensor, P: int, out: lsg.Segments, err: torch.Tensor) -> int:
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.lora_segment_noalloc(ctypes.c_void_p(ids.data_ptr()), ids.numel(), P,
                                    ctypes.c_void_p(out.perm.data_ptr()),
                                    ctypes.c_void_p(out.seg_offsets.data_ptr()),
                                    ctypes.c_void_p(out.seg_adapter.data_ptr()),
                                    ctypes.c_void_p(out.num_segments.data_ptr()),
                                    ctypes.c_void_p(err.data_ptr()), stream)


@pytest.mark.parametrize("n,P", [(3000, 60000), (256, 1000), (6224, 32)])
def test_noalloc_equals_lora_segment_on_two_calls_in_a_row(n, P):
    lib = lsg.load_library()
    # the first case needs the device scratch path (lora_segment would take a workspace)
    if P == 60000:
        assert lsg.lora_segment_workspace_bytes(n, P) > 0
    rng = np.random.default_rng(n + P)
    out = lsg.Segments.empty(n, P)
    # warm-up call: with CUDA's lazy module loading, the first call in a
    # context loads the library module that holds the scratch array, which
    # reserves its 8 MiB then (a module load, not an allocation by the call)
    warm_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _noalloc(lib, torch.zeros(n, dtype=torch.int32, device="cuda"), P, out, warm_err) == 0
    torch.cuda.synchronize()
    for call in range(2):
        ids_np = rng.integers(0, P, n).astype(np.int32)
        ids_np[rng.random(n) < 0.01] = -1  # a few invalid ids as well
        ids = torch.from_numpy(ids_np).cuda()
        err_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
        ref = lsg.lora_segment(ids, P, err_flag=err_ref)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out.num_segments.fill_(-7)
        torch.cuda.synchronize()
        # the call allocates no device memory: neither the driver's free memory
        # nor torch's allocator moves across it
        free0, torch0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        assert _noalloc(lib, ids, P, out, err) == 0
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] >= free0, call
        assert torch.cuda.memory_allocated() == torch0, call
        ms = min(n, P)
        assert int(out.num_segments.item()) == int(ref.num_segments.item()), call
        assert torch.equal(out.perm[:n], ref.perm[:n]), call
        assert torch.equal(out.seg_offsets[: ms + 1], ref.seg_offsets[: ms + 1]), call
        assert torch.equal(out.seg_adapter[:ms], ref.seg_adapter[:ms]), call
        assert int(err.item()) == int(err_ref.item()), call


def test_noalloc_rejects_pools_beyond_its_scratch():
    lib = lsg.load_library()
    n, P = 300, 70000  # needs more than the 8 MiB scratch (batches of <= 256 tokens need none)
    ids = torch.zeros(n, dtype=torch.int32, device="cuda")
    out = lsg.Segments.empty(n, P)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _noalloc(lib, ids, P, out, err) == -5  # LORA_ERR_WORKSPACE, nothing launched
