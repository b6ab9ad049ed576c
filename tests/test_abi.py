"""The C ABI library loads and exports every symbol its header declares, and
its host-side argument checks answer without touching a GPU (CPU only)."""

import ctypes
import glob
import os
import re

import pytest

import adapter_gemm_02_b300 as lsg
from adapter_gemm_02_b300 import build as lbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        for m in re.finditer(r"LORA_API\s+[\w\s\*]+?\b(\w+)\s*\(", src):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    if lbuild.stale():
        lbuild.build()
    return lsg.load_library()


def test_header_declares_the_boundary():
    assert _declared_symbols() == set(lsg.SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_symbols():
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings(lib):
    assert lib.lora_abi_version() == 2
    for code, name in lsg.STATUS.items():
        assert lib.lora_status_str(code).decode().startswith(name)
    assert lib.lora_status_str(12345) == b"unknown status"


def test_segment_workspace_sizes(lib):
    # histograms fit shared memory for pools up to ~25k adapters
    assert lsg.lora_segment_workspace_bytes(256, 1000) == 0
    assert lsg.lora_segment_workspace_bytes(6224, 32) == 0
    assert lsg.lora_segment_workspace_bytes(100, 60000) == 0  # up to 256 tokens: ranked, no histogram
    big = lsg.lora_segment_workspace_bytes(300, 60000)
    assert big >= 2 * 60001 * 4 and big % 4 == 0
    assert lsg.lora_segment_workspace_bytes(-1, 10) == 0


def _seg_struct(n=4, ms=4, ptrs=True):
    p = 256 if ptrs else 0
    return lsg.lora_sgmv.LoraSegments(p, p, p, p, n, ms)


def test_host_validation_without_gpu(lib):
    """Every check below fails before any CUDA call is made."""
    P = ctypes.c_void_p
    s = _seg_struct()
    # lora_segment: negative n, no adapters, null outputs
    assert lib.lora_segment(P(16), -1, 4, P(16), P(16), P(16), P(16), None, 0, None, None) == -1
    assert lib.lora_segment(P(16), 4, 0, P(16), P(16), P(16), P(16), None, 0, None, None) == -1
    assert lib.lora_segment(P(16), 4, 4, P(16), None, P(16), P(16), None, 0, None, None) == -1
    # huge pool: workspace required
    assert lib.lora_segment(P(16), 300, 60000, P(16), P(16), P(16), P(16), None, 0, None, None) == -5
    # sgmv_*: null segmentation, unsupported rank, bad widths, misalignment, ld < width
    assert lib.sgmv_fused(P(256), 64, P(256), P(256), 4, 64, 64, 16, 1.0, None, P(256), 64, None, None) == -1
    assert lib.sgmv_fused(P(256), 64, P(256), P(256), 4, 64, 64, 12, 1.0, ctypes.byref(s), P(256), 64, None,
                          None) == -3
    assert lib.sgmv_fused(P(256), 64, P(256), P(256), 4, 60, 64, 16, 1.0, ctypes.byref(s), P(256), 64, None,
                          None) == -3
    assert lib.sgmv_fused(P(258), 64, P(256), P(256), 4, 64, 64, 16, 1.0, ctypes.byref(s), P(256), 64, None,
                          None) == -2
    assert lib.sgmv_fused(P(256), 68, P(256), P(256), 4, 64, 64, 16, 1.0, ctypes.byref(s), P(256), 64, None,
                          None) == -2
    assert lib.sgmv_fused(P(256), 32, P(256), P(256), 4, 64, 64, 16, 1.0, ctypes.byref(s), P(256), 64, None,
                          None) == -1
    assert lib.sgmv_fused(P(256), 64, P(256), P(256), 0, 64, 64, 16, 1.0, ctypes.byref(s), P(256), 64, None,
                          None) == -1
    bad = _seg_struct(ptrs=False)
    assert lib.sgmv_fused(P(256), 64, P(256), P(256), 4, 64, 64, 16, 1.0, ctypes.byref(bad), P(256), 64, None,
                          None) == -1
    # n_tokens == 0 is a no-op
    zero = _seg_struct(n=0, ms=0, ptrs=False)
    assert lib.sgmv_fused(P(256), 64, P(256), P(256), 4, 64, 64, 16, 1.0, ctypes.byref(zero), P(256), 64, None,
                          None) == 0
    assert lib.sgmv_shrink(P(256), 64, P(256), 4, 64, 16, ctypes.byref(s), None, None, None) == -1
    assert lib.sgmv_shrink(P(256), 64, P(256), 4, 64, 16, ctypes.byref(s), P(260), None, None) == -2
    assert lib.sgmv_expand(P(256), P(256), 4, 16, 64, 1.0, ctypes.byref(s), P(256), 63, None, None) == -1
    # multi: too many projections
    arr = (lsg.lora_sgmv.LoraProj * 9)()
    assert lib.sgmv_multi(arr, 9, 4, 16, ctypes.byref(s), None, None) == -3
    assert lib.sgmv_multi(arr, 0, 4, 16, ctypes.byref(s), None, None) == -1


def test_slot_table_validation_without_gpu(lib):
    """sgmv_multi_slots rejects bad tables before any CUDA call."""
    P = ctypes.c_void_p
    s = _seg_struct()
    arr = (lsg.lora_sgmv.LoraProj * 1)()
    arr[0] = lsg.lora_sgmv.LoraProj(256, 256, 256, 256, 64, 64, 64, 64, 1.0)
    T = lsg.lora_sgmv.LoraSlotTable

    def call(tab, n_proj=1, seg=s):
        return lib.sgmv_multi_slots(arr, n_proj, None if tab is None else ctypes.byref(tab), ctypes.byref(seg),
                                    None, None)

    assert call(None) == -1
    assert call(T(256, 256, 4, 8, 64, 0b1111), n_proj=0) == -1
    assert call(T(256, 256, 4, 8, 64, 0b1111), n_proj=9) == -3
    assert call(T(0, 256, 4, 8, 64, 0b0010)) == -1          # slot_of missing
    assert call(T(256, 258, 4, 8, 64, 0b0010)) == -2        # rank_of misaligned
    assert call(T(256, 256, 4, 0, 64, 0b0010)) == -1        # no slots
    assert call(T(256, 256, 4, 8, 48, 0b0010)) == -3        # r_max not a rank
    assert call(T(256, 256, 4, 8, 16, 0b0100)) == -3        # rank 32 above r_max 16
    assert call(T(256, 256, 4, 8, 64, 0)) == -3             # empty mask
    assert call(T(256, 256, 4, 8, 64, 0b10000)) == -3       # unknown rank bit
    assert call(T(256, 256, 0, 8, 64, 0b0010)) == -1        # no adapters
    assert call(T(256, 256, 4, 1 << 20, 64, 0b0010)) == -3  # arena rows beyond the tensor-map range
    zero = _seg_struct(n=0, ms=0, ptrs=False)
    assert call(T(256, 256, 4, 8, 64, 0b1010), seg=zero) == 0


def test_slot_loader_validation_without_gpu(lib):
    """lora_slot_copy / lora_slot_assign reject bad arguments before any CUDA call."""
    S = lsg.lora_sgmv.LoraSlotSrc
    arr = (S * 1)()
    arr[0] = S(256, 256, 256, 256, 64, 64)
    assert lib.lora_slot_copy(None, 1, 4, 16, 0, 16, None) == -1
    assert lib.lora_slot_copy(arr, 0, 4, 16, 0, 16, None) == -1
    assert lib.lora_slot_copy(arr, 1, 4, 16, 4, 16, None) == -1     # slot outside
    assert lib.lora_slot_copy(arr, 1, 4, 16, -1, 16, None) == -1
    assert lib.lora_slot_copy(arr, 1, 4, 16, 0, 32, None) == -3     # rank above r_max
    assert lib.lora_slot_copy(arr, 1, 4, 24, 0, 8, None) == -3      # r_max not a rank
    bad = (S * 1)()
    bad[0] = S(256, 264, 256, 256, 64, 64)
    assert lib.lora_slot_copy(bad, 1, 4, 16, 0, 16, None) == -2      # B arena misaligned
    bad[0] = S(256, 256, 0, 256, 64, 64)
    assert lib.lora_slot_copy(bad, 1, 4, 16, 0, 16, None) == -1      # no source
    bad[0] = S(256, 256, 256, 256, 60, 64)
    assert lib.lora_slot_copy(bad, 1, 4, 16, 0, 16, None) == -3      # width
    P = ctypes.c_void_p
    assert lib.lora_slot_assign(None, P(256), 4, 0, 0, 16, None) == -1
    assert lib.lora_slot_assign(P(256), P(258), 4, 0, 0, 16, None) == -2
    assert lib.lora_slot_assign(P(256), P(256), 4, 4, 0, 16, None) == -1   # adapter outside
    assert lib.lora_slot_assign(P(256), P(256), 4, 0, -2, 16, None) == -1  # slot below -1
    assert lib.lora_slot_assign(P(256), P(256), 4, 0, 1, 12, None) == -3   # not a rank


def test_host_step_validation_without_gpu(lib):
    """sgmv_multi_host: workspace sizing and argument checks without a GPU."""
    P = ctypes.c_void_p
    arr = (lsg.lora_sgmv.LoraProj * 2)()
    arr[0] = lsg.lora_sgmv.LoraProj(4096, 256, 256, 8192, 64, 64, 64, 64, 1.0)
    arr[1] = lsg.lora_sgmv.LoraProj(4096, 256, 256, 16384, 64, 128, 64, 128, 1.0)  # same host x
    need = lib.sgmv_multi_host_workspace_bytes(arr, 2, 32, 8)
    # ids, perm, offsets, adapters, count, one x (shared), two y; 256-byte aligned pieces
    assert need == 256 * 5 + 32 * 64 * 2 + 32 * 64 * 2 + 32 * 128 * 2
    assert lib.sgmv_multi_host_workspace_bytes(arr, 9, 32, 8) == 0
    assert lib.sgmv_multi_host(arr, 2, 8, 16, None, 32, P(256), need, None, None) == -1   # no ids
    assert lib.sgmv_multi_host(arr, 2, 8, 12, P(64), 32, P(256), need, None, None) == -3  # rank
    assert lib.sgmv_multi_host(arr, 2, 8, 16, P(64), 32, P(256), need - 1, None, None) == -5
    assert lib.sgmv_multi_host(arr, 2, 8, 16, P(64), 32, None, need, None, None) == -5
    assert lib.sgmv_multi_host(arr, 2, 8, 16, P(64), 32, P(272), need, None, None) == -2
    assert lib.sgmv_multi_host(arr, 2, 8, 16, P(64), 0, None, 0, None, None) == 0       # empty batch
    bad = (lsg.lora_sgmv.LoraProj * 1)()
    bad[0] = lsg.lora_sgmv.LoraProj(4096, 256, 256, 8192, 60, 64, 64, 64, 1.0)          # ldx < h_in
    assert lib.sgmv_multi_host(bad, 1, 8, 16, P(64), 32, P(256), need, None, None) == -1


def test_one_call_step_validation_without_gpu(lib):
    """sgmv_multi_segment rejects bad arguments before any CUDA call."""
    P = ctypes.c_void_p
    arr = (lsg.lora_sgmv.LoraProj * 1)()
    arr[0] = lsg.lora_sgmv.LoraProj(256, 256, 256, 256, 64, 64, 64, 64, 1.0)
    f = lib.sgmv_multi_segment
    ok = (P(256), 32, P(256), P(256), P(256), P(256), None, 0, None, None)
    assert f(arr, 0, 8, 16, *ok) == -1
    assert f(arr, 9, 8, 16, *ok) == -3
    assert f(arr, 1, 8, 12, *ok) == -3                                                        # rank
    assert f(arr, 1, 0, 16, *ok) == -1                                                        # no adapters
    assert f(arr, 1, 8, 16, None, 32, P(256), P(256), P(256), P(256), None, 0, None, None) == -1  # no ids
    assert f(arr, 1, 8, 16, P(258), 32, P(256), P(256), P(256), P(256), None, 0, None, None) == -2
    big = (P(256), 300, P(256), P(256), P(256), P(256), None, 0, None, None)  # > 256 tokens: histograms
    assert f(arr, 1, 60000, 16, *big) == -5                                                   # workspace
    bad = (lsg.lora_sgmv.LoraProj * 1)()
    bad[0] = lsg.lora_sgmv.LoraProj(258, 256, 256, 256, 64, 64, 64, 64, 1.0)                 # x misaligned
    assert f(bad, 1, 8, 16, *ok) == -2


def test_product_path_fails_loudly_without_library(tmp_path):
    from adapter_gemm_02_b300 import lora_sgmv

    saved = lora_sgmv._lib
    try:
        lora_sgmv._lib = None
        with pytest.raises(RuntimeError, match="missing"):
            lora_sgmv.load_library(str(tmp_path / "nope.so"))
    finally:
        lora_sgmv._lib = saved


def test_product_never_imports_the_oracle():
    for path in glob.glob(os.path.join(ROOT, "adapter_gemm_02_b300", "**", "*"), recursive=True):
        if path.endswith((".py", ".cu", ".cuh", ".h")):
            src = open(path).read()
            assert "import oracle" not in src and "from oracle" not in src, path
            assert "sgmv_oracle" not in src, path
