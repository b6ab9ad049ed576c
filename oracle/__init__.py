"""CPU oracle for multi-LoRA SGMV -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package's smoke check and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
binding) never imports, links or calls it, and this package never imports
the product.

The arithmetic lives in ``sgmv_oracle.c`` (plain C, one IEEE operation at a
time, built with ``-ffp-contract=off``); this module compiles it with gcc and
marshals numpy arrays to it.  What it computes and the readings it takes are
stated in the C file's header.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sgmv_oracle.c")
_LIB = os.path.join(_HERE, "libsgmv_oracle.so")
_loaded = {}

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared", "-std=c11"]


def build(out: Optional[str] = None, mutant: int = 0) -> str:
    """Compile the oracle; returns the path of the shared library."""
    out = out or _LIB
    cmd = ["gcc", *CFLAGS, f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", out + ".tmp"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _needs_build(path: str) -> bool:
    return (not os.path.exists(path)) or os.path.getmtime(path) < os.path.getmtime(_SRC)


def load(mutant: int = 0) -> ctypes.CDLL:
    """Load (building first if stale) the oracle, or a planted-mistake variant."""
    if mutant in _loaded:
        return _loaded[mutant]
    if mutant == 0:
        path = _LIB
        if _needs_build(path):
            build(path)
    else:
        path = os.path.join(tempfile.gettempdir(), f"libsgmv_oracle_mutant{mutant}_{os.getpid()}.so")
        build(path, mutant)
    lib = ctypes.CDLL(path)
    i32, i64, p = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    lib.oracle_lora_segment.restype = i32
    lib.oracle_lora_segment.argtypes = [p, i32, i32, i32, p, p, p, p]
    lib.oracle_sgmv_f32.restype = i32
    lib.oracle_sgmv_f32.argtypes = [p, i64, p, p, p, i32, i32, i32, i32, i32, ctypes.c_float, p, i64, p, p, i32]
    lib.oracle_sgmv_f64.restype = i32
    lib.oracle_sgmv_f64.argtypes = [p, i64, p, p, p, i32, i32, i32, i32, i32, ctypes.c_double, p, i64, p, p, i32]
    lib.oracle_sgmv_slots_f32.restype = i32
    lib.oracle_sgmv_slots_f32.argtypes = [p, i64, p, p, p, p, i32, i32, ctypes.c_uint32, p, i32, i32, i32, i32,
                                          ctypes.c_float, p, i64, p, i32]
    lib.oracle_gemm_lora_f32.restype = i32
    lib.oracle_gemm_lora_f32.argtypes = [p, i64, p, p, p, p, i32, i32, i32, i32, i32, ctypes.c_float, p, i32]
    lib.oracle_mutant.restype = i32
    assert lib.oracle_mutant() == mutant
    _loaded[mutant] = lib
    return lib


def bits(a) -> np.ndarray:
    """bf16 data as a C-contiguous uint16 array of bit patterns. Accepts a
    uint16 numpy array or a CPU torch.bfloat16 tensor."""
    if isinstance(a, np.ndarray):
        assert a.dtype == np.uint16, a.dtype
        return np.ascontiguousarray(a)
    import torch  # local: the oracle's C path does not need torch

    assert a.dtype == torch.bfloat16, a.dtype
    return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def lora_segment_ref(ids, P: int, max_segments: Optional[int] = None, mutant: int = 0) -> dict:
    """Stable segmentation of token indices by adapter id (see the C file)."""
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    n = int(ids.size)
    ms = min(n, P) if max_segments is None else int(max_segments)
    perm = np.empty(n, np.int32)
    offs = np.empty(ms + 1, np.int32)
    sad = np.empty(max(ms, 1), np.int32)
    ns = np.zeros(1, np.int32)
    n_bad = load(mutant).oracle_lora_segment(_ptr(ids), n, int(P), ms, _ptr(perm), _ptr(offs), _ptr(sad), _ptr(ns))
    return dict(perm=perm, seg_offsets=offs, seg_adapter=sad[:ms], num_segments=int(ns[0]), n_invalid=int(n_bad))


def sgmv_ref(x, A_pool, B_pool, ids, s: float, y0, *, threads: int = 1, f64: bool = False,
             want_v: bool = False, mutant: int = 0):
    """y = y0 + s*((x.A[a_i]).B[a_i]) per token, unrounded.

    x: [n, >=h_in] bf16; A_pool: [P, h_in, r]; B_pool: [P, r, h_out];
    ids: int32 [n]; y0: [n, >=h_out].  Returns y ([n, h_out], fp32 or fp64)
    and, with want_v, v ([n, r]) as well."""
    xb, Ab, Bb, yb = bits(x), bits(A_pool), bits(B_pool), bits(y0)
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    P, h_in, r = Ab.shape
    P2, r2, h_out = Bb.shape
    assert P2 == P and r2 == r
    n = int(ids.size)
    assert xb.ndim == 2 and xb.shape[0] == n and xb.shape[1] >= h_in
    assert yb.ndim == 2 and yb.shape[0] == n and yb.shape[1] >= h_out
    dt = np.float64 if f64 else np.float32
    y = np.empty((n, h_out), dt)
    v = np.zeros((n, r), dt) if want_v else None
    lib = load(mutant)
    fn = lib.oracle_sgmv_f64 if f64 else lib.oracle_sgmv_f32
    fn(_ptr(xb), xb.shape[1], _ptr(Ab), _ptr(Bb), _ptr(ids), n, P, h_in, h_out, r, float(s),
       _ptr(yb), yb.shape[1], _ptr(y), _ptr(v) if want_v else None, int(threads))
    return (y, v) if want_v else y


def sgmv_slots_ref(x, A_arena, B_arena, slot_of, rank_of, r_max: int, rank_mask: int, ids, s: float, y0, *,
                   threads: int = 1, mutant: int = 0, return_invalid: bool = False):
    """The delta over slot arenas with adapters of mixed ranks (see the C file).

    x: [n, >=h_in] bf16; A_arena: [n_slots, h_in*r_max]; B_arena:
    [n_slots, r_max*h_out]; slot_of, rank_of: int32 [P]; ids: int32 [n];
    y0: [n, >=h_out].  Returns y ([n, h_out] fp32, unrounded)."""
    xb, Ab, Bb, yb = bits(x), bits(A_arena), bits(B_arena), bits(y0)
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    slot_of = np.ascontiguousarray(np.asarray(slot_of, dtype=np.int32))
    rank_of = np.ascontiguousarray(np.asarray(rank_of, dtype=np.int32))
    assert slot_of.shape == rank_of.shape and slot_of.ndim == 1
    P = int(slot_of.size)
    n = int(ids.size)
    n_slots = Ab.shape[0]
    assert Ab.ndim == 2 and Bb.ndim == 2 and Bb.shape[0] == n_slots
    assert Ab.shape[1] % r_max == 0 and Bb.shape[1] % r_max == 0
    h_in, h_out = Ab.shape[1] // r_max, Bb.shape[1] // r_max
    assert xb.shape[0] == n and xb.shape[1] >= h_in and yb.shape[0] == n and yb.shape[1] >= h_out
    y = np.empty((n, h_out), np.float32)
    bad = load(mutant).oracle_sgmv_slots_f32(_ptr(xb), xb.shape[1], _ptr(Ab), _ptr(Bb), _ptr(slot_of),
                                             _ptr(rank_of), n_slots, int(r_max), int(rank_mask), _ptr(ids), n, P,
                                             h_in, h_out, float(s), _ptr(yb), yb.shape[1], _ptr(y), int(threads))
    return (y, int(bad)) if return_invalid else y


def gemm_lora_ref(x, W, A_pool, B_pool, ids, s: float, *, threads: int = 1, mutant: int = 0):
    """y = x.W + s*((x.A[a_i]).B[a_i]) per token, unrounded fp32 (see the C file).

    x: [n, >=h_in] bf16; W: [h_in, h_out]; A_pool: [P, h_in, r];
    B_pool: [P, r, h_out]; ids: int32 [n].  Returns y [n, h_out]."""
    xb, Wb, Ab, Bb = bits(x), bits(W), bits(A_pool), bits(B_pool)
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    P, h_in, r = Ab.shape
    h_in2, h_out = Wb.shape
    assert h_in2 == h_in and Bb.shape == (P, r, h_out)
    n = int(ids.size)
    assert xb.ndim == 2 and xb.shape[0] == n and xb.shape[1] >= h_in
    y = np.empty((n, h_out), np.float32)
    load(mutant).oracle_gemm_lora_f32(_ptr(xb), xb.shape[1], _ptr(Wb), _ptr(Ab), _ptr(Bb), _ptr(ids), n, P, h_in,
                                      h_out, r, float(s), _ptr(y), int(threads))
    return y
