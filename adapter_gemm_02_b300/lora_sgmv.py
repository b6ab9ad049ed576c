"""Python binding of liblora_sgmv.so (argument marshalling only).

Every function has the name of the C entry point it calls and passes
torch tensors' device pointers and the current CUDA stream.  All arithmetic
runs in the library's CUDA kernels; there is no fallback: a missing library
raises at import of the first call, a non-OK status raises RuntimeError.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblora_sgmv.so")
_lib: Optional[ctypes.CDLL] = None

LORA_MAX_PROJ = 8
STATUS = {
    0: "LORA_OK", -1: "LORA_ERR_INVALID_ARG", -2: "LORA_ERR_MISALIGNED", -3: "LORA_ERR_UNSUPPORTED",
    -4: "LORA_ERR_BAD_ADAPTER_ID", -5: "LORA_ERR_WORKSPACE", -6: "LORA_ERR_CUDA", -7: "LORA_ERR_TIMEOUT",
}
# exported symbols declared in include/lora_sgmv.h
SYMBOLS = ("lora_status_str", "lora_abi_version", "lora_segment_workspace_bytes", "lora_segment",
           "lora_segment_noalloc", "sgmv_shrink", "sgmv_expand", "sgmv_fused", "sgmv_multi", "sgmv_multi_slots",
           "lora_slot_copy", "lora_slot_assign", "sgmv_multi_host_workspace_bytes", "sgmv_multi_host",
           "sgmv_multi_segment", "gemm_lora_workspace_bytes", "gemm_lora")
NOALLOC_SCRATCH_BYTES = 8 << 20


class LoraSegments(ctypes.Structure):
    _fields_ = [("perm", ctypes.c_void_p), ("seg_offsets", ctypes.c_void_p), ("seg_adapter", ctypes.c_void_p),
                ("num_segments", ctypes.c_void_p), ("n_tokens", ctypes.c_int32), ("max_segments", ctypes.c_int32)]


class LoraProj(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("A_pool", ctypes.c_void_p), ("B_pool", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("ldx", ctypes.c_int64), ("ldy", ctypes.c_int64),
                ("h_in", ctypes.c_int32), ("h_out", ctypes.c_int32), ("scale", ctypes.c_float)]


class LoraSlotTable(ctypes.Structure):
    _fields_ = [("slot_of", ctypes.c_void_p), ("rank_of", ctypes.c_void_p), ("n_adapters", ctypes.c_int32),
                ("n_slots", ctypes.c_int32), ("r_max", ctypes.c_int32), ("rank_mask", ctypes.c_uint32)]


class LoraSlotSrc(ctypes.Structure):
    _fields_ = [("A_arena", ctypes.c_void_p), ("B_arena", ctypes.c_void_p), ("A_src", ctypes.c_void_p),
                ("B_src", ctypes.c_void_p), ("h_in", ctypes.c_int32), ("h_out", ctypes.c_int32)]


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load liblora_sgmv.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing; build it with `python -m adapter_gemm_02_b300.build`")
    lib = ctypes.CDLL(path)
    p, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.lora_status_str.restype = ctypes.c_char_p
    lib.lora_status_str.argtypes = [ctypes.c_int]
    lib.lora_abi_version.restype = ctypes.c_int
    lib.lora_abi_version.argtypes = []
    lib.lora_segment_workspace_bytes.restype = sz
    lib.lora_segment_workspace_bytes.argtypes = [i32, i32]
    lib.lora_segment.restype = ctypes.c_int
    lib.lora_segment.argtypes = [p, i32, i32, p, p, p, p, p, sz, p, p]
    lib.lora_segment_noalloc.restype = ctypes.c_int
    lib.lora_segment_noalloc.argtypes = [p, i32, i32, p, p, p, p, p, p]
    lib.sgmv_shrink.restype = ctypes.c_int
    lib.sgmv_shrink.argtypes = [p, i64, p, i32, i32, i32, ctypes.POINTER(LoraSegments), p, p, p]
    lib.sgmv_expand.restype = ctypes.c_int
    lib.sgmv_expand.argtypes = [p, p, i32, i32, i32, ctypes.c_float, ctypes.POINTER(LoraSegments), p, i64, p, p]
    lib.sgmv_fused.restype = ctypes.c_int
    lib.sgmv_fused.argtypes = [p, i64, p, p, i32, i32, i32, i32, ctypes.c_float, ctypes.POINTER(LoraSegments),
                               p, i64, p, p]
    lib.sgmv_multi.restype = ctypes.c_int
    lib.sgmv_multi.argtypes = [ctypes.POINTER(LoraProj), i32, i32, i32, ctypes.POINTER(LoraSegments), p, p]
    lib.sgmv_multi_slots.restype = ctypes.c_int
    lib.sgmv_multi_slots.argtypes = [ctypes.POINTER(LoraProj), i32, ctypes.POINTER(LoraSlotTable),
                                     ctypes.POINTER(LoraSegments), p, p]
    lib.sgmv_multi_host_workspace_bytes.restype = sz
    lib.sgmv_multi_host_workspace_bytes.argtypes = [ctypes.POINTER(LoraProj), i32, i32, i32]
    lib.sgmv_multi_host.restype = ctypes.c_int
    lib.sgmv_multi_host.argtypes = [ctypes.POINTER(LoraProj), i32, i32, i32, p, i32, p, sz, p, p]
    lib.sgmv_multi_segment.restype = ctypes.c_int
    lib.sgmv_multi_segment.argtypes = [ctypes.POINTER(LoraProj), i32, i32, i32, p, i32, p, p, p, p, p, sz, p, p]
    lib.gemm_lora_workspace_bytes.restype = sz
    lib.gemm_lora_workspace_bytes.argtypes = [i32, i32]
    lib.gemm_lora.restype = ctypes.c_int
    lib.gemm_lora.argtypes = [p, i64, p, p, p, i32, i32, i32, i32, ctypes.c_float, ctypes.POINTER(LoraSegments), p,
                              i64, p, sz, p, p]
    lib.lora_slot_copy.restype = ctypes.c_int
    lib.lora_slot_copy.argtypes = [ctypes.POINTER(LoraSlotSrc), i32, i32, i32, i32, i32, p]
    lib.lora_slot_assign.restype = ctypes.c_int
    lib.lora_slot_assign.argtypes = [p, p, i32, i32, i32, i32, p]
    _lib = lib
    return lib


def _check(status: int, what: str) -> None:
    if status != 0:
        msg = load_library().lora_status_str(status).decode()
        raise RuntimeError(f"{what} failed: {msg} ({status})")


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _req(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def _rows(t: torch.Tensor, name: str) -> int:
    """Leading dimension of a row-major [n, width] matrix with unit column stride."""
    if t.stride(1) != 1 and t.shape[1] > 1:
        raise ValueError(f"{name} must have unit column stride")
    return t.stride(0) if t.shape[0] > 1 else max(t.stride(0), t.shape[1])


def _pool(t: torch.Tensor, name: str) -> None:
    _req(t, name, torch.bfloat16, 3)
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous [n_adapters, ., .]")


@dataclass
class Segments:
    """Device-side segmentation (output of lora_segment)."""
    perm: torch.Tensor          # int32 [n]
    seg_offsets: torch.Tensor   # int32 [max_segments + 1]
    seg_adapter: torch.Tensor   # int32 [max_segments]
    num_segments: torch.Tensor  # int32 [1]
    n_tokens: int
    max_segments: int
    n_adapters: int

    def __post_init__(self):
        self._c = LoraSegments(self.perm.data_ptr(), self.seg_offsets.data_ptr(), self.seg_adapter.data_ptr(),
                               self.num_segments.data_ptr(), self.n_tokens, self.max_segments)

    @property
    def c_struct(self) -> LoraSegments:
        return self._c

    @staticmethod
    def empty(n_tokens: int, n_adapters: int, device="cuda") -> "Segments":
        ms = min(n_tokens, n_adapters)
        i32 = dict(dtype=torch.int32, device=device)
        return Segments(torch.empty(max(n_tokens, 1), **i32), torch.empty(ms + 1, **i32),
                        torch.empty(max(ms, 1), **i32), torch.empty(1, **i32), n_tokens, ms, n_adapters)


def lora_segment_workspace_bytes(n_tokens: int, n_adapters: int) -> int:
    return int(load_library().lora_segment_workspace_bytes(n_tokens, n_adapters))


def lora_segment(ids: torch.Tensor, n_adapters: int, *, out: Optional[Segments] = None,
                 workspace: Optional[torch.Tensor] = None, err_flag: Optional[torch.Tensor] = None,
                 stream=None) -> Segments:
    """Stable grouping of tokens by adapter id (see include/lora_sgmv.h)."""
    lib = load_library()
    _req(ids, "ids", torch.int32, 1)
    n = ids.shape[0]
    seg = out if out is not None else Segments.empty(n, n_adapters, ids.device)
    if seg.n_tokens != n or seg.n_adapters != n_adapters:
        raise ValueError("out was sized for another batch")
    need = lora_segment_workspace_bytes(n, n_adapters)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=ids.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.lora_segment(_ptr(ids.contiguous()), n, n_adapters, _ptr(seg.perm), _ptr(seg.seg_offsets),
                            _ptr(seg.seg_adapter), _ptr(seg.num_segments), _ptr(workspace), ws_bytes,
                            _ptr(err_flag), _stream(stream)), "lora_segment")
    return seg


def lora_segment_noalloc(ids: torch.Tensor, n_adapters: int, out: Segments, *,
                         err_flag: Optional[torch.Tensor] = None, stream=None) -> Segments:
    """lora_segment without a workspace: large pools use the library's own
    8 MiB device scratch array, so the call allocates nothing (the outputs
    `out` are the caller's).  Calls that overlap on the GPU race on that array."""
    lib = load_library()
    _req(ids, "ids", torch.int32, 1)
    n = ids.shape[0]
    if out.n_tokens != n or out.n_adapters != n_adapters:
        raise ValueError("out was sized for another batch")
    _check(lib.lora_segment_noalloc(_ptr(ids), n, n_adapters, _ptr(out.perm), _ptr(out.seg_offsets),
                                    _ptr(out.seg_adapter), _ptr(out.num_segments), _ptr(err_flag),
                                    _stream(stream)), "lora_segment_noalloc")
    return out


def sgmv_shrink(x: torch.Tensor, A_pool: torch.Tensor, seg: Segments, *, v: Optional[torch.Tensor] = None,
                err_flag: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """v[i] = x[i] . A[a_i] in fp32."""
    lib = load_library()
    _req(x, "x", torch.bfloat16, 2)
    _pool(A_pool, "A_pool")
    P, h_in, r = A_pool.shape
    if x.shape[1] != h_in:
        raise ValueError("x width != h_in")
    if v is None:
        v = torch.zeros(x.shape[0], r, dtype=torch.float32, device=x.device)
    _req(v, "v", torch.float32, 2)
    _check(lib.sgmv_shrink(_ptr(x), _rows(x, "x"), _ptr(A_pool), P, h_in, r, ctypes.byref(seg.c_struct),
                           _ptr(v), _ptr(err_flag), _stream(stream)), "sgmv_shrink")
    return v


def sgmv_expand(v: torch.Tensor, B_pool: torch.Tensor, seg: Segments, y: torch.Tensor, scale: float, *,
                err_flag: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """y[i] += scale * v[i] . B[a_i] (in place)."""
    lib = load_library()
    _req(v, "v", torch.float32, 2)
    _pool(B_pool, "B_pool")
    _req(y, "y", torch.bfloat16, 2)
    P, r, h_out = B_pool.shape
    if y.shape[1] != h_out or v.shape[1] != r:
        raise ValueError("shape mismatch")
    if not v.is_contiguous():
        raise ValueError("v must be contiguous")
    _check(lib.sgmv_expand(_ptr(v), _ptr(B_pool), P, r, h_out, float(scale), ctypes.byref(seg.c_struct),
                           _ptr(y), _rows(y, "y"), _ptr(err_flag), _stream(stream)), "sgmv_expand")
    return y


def sgmv_fused(x: torch.Tensor, A_pool: torch.Tensor, B_pool: torch.Tensor, seg: Segments, y: torch.Tensor,
               scale: float, *, err_flag: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """y[i] += scale * (x[i] . A[a_i]) . B[a_i] in one launch (in place)."""
    lib = load_library()
    _req(x, "x", torch.bfloat16, 2)
    _req(y, "y", torch.bfloat16, 2)
    _pool(A_pool, "A_pool")
    _pool(B_pool, "B_pool")
    P, h_in, r = A_pool.shape
    _, r2, h_out = B_pool.shape
    if r2 != r or x.shape[1] != h_in or y.shape[1] != h_out or B_pool.shape[0] != P:
        raise ValueError("shape mismatch")
    _check(lib.sgmv_fused(_ptr(x), _rows(x, "x"), _ptr(A_pool), _ptr(B_pool), P, h_in, h_out, r, float(scale),
                          ctypes.byref(seg.c_struct), _ptr(y), _rows(y, "y"), _ptr(err_flag), _stream(stream)),
           "sgmv_fused")
    return y


def make_projs(projs: Sequence) -> "ctypes.Array":
    """Host array of lora_proj from (x, A_pool, B_pool, y, scale) tuples."""
    arr = (LoraProj * len(projs))()
    for i, (x, A, B, y, s) in enumerate(projs):
        _req(x, "x", torch.bfloat16, 2)
        _req(y, "y", torch.bfloat16, 2)
        _pool(A, "A_pool")
        _pool(B, "B_pool")
        if A.shape[2] != B.shape[1] or x.shape[1] != A.shape[1] or y.shape[1] != B.shape[2]:
            raise ValueError(f"projection {i}: shape mismatch")
        arr[i] = LoraProj(x.data_ptr(), A.data_ptr(), B.data_ptr(), y.data_ptr(), _rows(x, "x"), _rows(y, "y"),
                          A.shape[1], B.shape[2], float(s))
    return arr


def sgmv_multi(projs: Sequence, seg: Segments, *, err_flag: Optional[torch.Tensor] = None, stream=None,
               c_projs=None) -> None:
    """sgmv_fused over up to 8 projections sharing `seg`, in one launch.
    projs: sequence of (x, A_pool, B_pool, y, scale)."""
    lib = load_library()
    if not 1 <= len(projs) <= LORA_MAX_PROJ:
        raise ValueError("1..8 projections")
    arr = c_projs if c_projs is not None else make_projs(projs)
    P, _, r = projs[0][1].shape
    _check(lib.sgmv_multi(arr, len(projs), P, r, ctypes.byref(seg.c_struct), _ptr(err_flag), _stream(stream)),
           "sgmv_multi")


def rank_mask(ranks) -> int:
    """Bit c set for each rank 8 << c in `ranks`."""
    m = 0
    for r in ranks:
        if r not in (8, 16, 32, 64):
            raise ValueError(f"rank {r} not in (8, 16, 32, 64)")
        m |= 1 << (int(r).bit_length() - 4)
    return m


@dataclass
class SlotTable:
    """Where each adapter of the batch lives in slot arenas, and its rank
    (device int32 tables of n_adapters entries)."""
    slot_of: torch.Tensor  # int32 [n_adapters]
    rank_of: torch.Tensor  # int32 [n_adapters]
    n_slots: int
    r_max: int
    rank_mask: int

    def __post_init__(self):
        _req(self.slot_of, "slot_of", torch.int32, 1)
        _req(self.rank_of, "rank_of", torch.int32, 1)
        if self.slot_of.shape != self.rank_of.shape:
            raise ValueError("slot_of and rank_of differ in length")
        self._c = LoraSlotTable(self.slot_of.data_ptr(), self.rank_of.data_ptr(), self.slot_of.shape[0],
                                int(self.n_slots), int(self.r_max), int(self.rank_mask))

    @property
    def n_adapters(self) -> int:
        return self.slot_of.shape[0]

    @property
    def c_struct(self) -> LoraSlotTable:
        return self._c


def make_slot_projs(projs: Sequence, table: SlotTable) -> "ctypes.Array":
    """Host array of lora_proj from (x, A_arena, B_arena, y, scale) tuples;
    A_arena is [n_slots, h_in * r_max], B_arena [n_slots, r_max * h_out]."""
    arr = (LoraProj * len(projs))()
    for i, (x, A, B, y, s) in enumerate(projs):
        _req(x, "x", torch.bfloat16, 2)
        _req(y, "y", torch.bfloat16, 2)
        _req(A, "A_arena", torch.bfloat16, 2)
        _req(B, "B_arena", torch.bfloat16, 2)
        h_in, h_out = x.shape[1], y.shape[1]
        if not (A.is_contiguous() and B.is_contiguous()):
            raise ValueError(f"projection {i}: arenas must be contiguous")
        if tuple(A.shape) != (table.n_slots, h_in * table.r_max) or \
                tuple(B.shape) != (table.n_slots, table.r_max * h_out):
            raise ValueError(f"projection {i}: arena shapes do not match n_slots / r_max / widths")
        arr[i] = LoraProj(x.data_ptr(), A.data_ptr(), B.data_ptr(), y.data_ptr(), _rows(x, "x"), _rows(y, "y"),
                          h_in, h_out, float(s))
    return arr


def sgmv_multi_slots(projs: Sequence, table: SlotTable, seg: Segments, *, err_flag: Optional[torch.Tensor] = None,
                     stream=None, c_projs=None) -> None:
    """sgmv_multi over slot arenas, adapters of mixed ranks (include/lora_sgmv.h).
    projs: sequence of (x, A_arena, B_arena, y, scale)."""
    lib = load_library()
    if not 1 <= len(projs) <= LORA_MAX_PROJ:
        raise ValueError("1..8 projections")
    if seg.n_adapters != table.n_adapters:
        raise ValueError("segmentation and slot table disagree on n_adapters")
    arr = c_projs if c_projs is not None else make_slot_projs(projs, table)
    _check(lib.sgmv_multi_slots(arr, len(projs), ctypes.byref(table.c_struct), ctypes.byref(seg.c_struct),
                                _ptr(err_flag), _stream(stream)), "sgmv_multi_slots")


def sgmv_fused_slots(x: torch.Tensor, A_arena: torch.Tensor, B_arena: torch.Tensor, table: SlotTable,
                     seg: Segments, y: torch.Tensor, scale: float, *, err_flag: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
    """One projection of sgmv_multi_slots (in place on y)."""
    sgmv_multi_slots([(x, A_arena, B_arena, y, scale)], table, seg, err_flag=err_flag, stream=stream)
    return y


def make_slot_srcs(srcs: Sequence, r_max: int) -> "ctypes.Array":
    """Host array of lora_slot_src from (A_arena, B_arena, A_src, B_src)
    tuples: arenas [n_slots, h_in*r_max] / [n_slots, r_max*h_out] on the GPU,
    sources A [h_in, rank] / B [rank, h_out], contiguous, in pinned host or
    device memory."""
    arr = (LoraSlotSrc * len(srcs))()
    for i, (Aa, Ba, As, Bs) in enumerate(srcs):
        _req(Aa, "A_arena", torch.bfloat16, 2)
        _req(Ba, "B_arena", torch.bfloat16, 2)
        for t, nm in ((As, "A_src"), (Bs, "B_src")):
            if t.dtype != torch.bfloat16 or t.dim() != 2 or not t.is_contiguous():
                raise ValueError(f"{nm} must be a contiguous 2-D bf16 tensor")
            if not t.is_cuda and not t.is_pinned():
                raise ValueError(f"{nm} in host memory must be pinned (asynchronous copy)")
        h_in, rank = As.shape
        rank2, h_out = Bs.shape
        if rank2 != rank or Aa.shape[1] != h_in * r_max or Ba.shape[1] != r_max * h_out:
            raise ValueError(f"source {i}: shapes do not match the arenas")
        arr[i] = LoraSlotSrc(Aa.data_ptr(), Ba.data_ptr(), As.data_ptr(), Bs.data_ptr(), h_in, h_out)
    return arr


def lora_slot_copy(srcs: Sequence, n_slots: int, r_max: int, slot: int, rank: int, *, stream=None,
                   c_srcs=None) -> None:
    """Copy one adapter's matrices into `slot` of each arena pair (stream-ordered)."""
    lib = load_library()
    arr = c_srcs if c_srcs is not None else make_slot_srcs(srcs, r_max)
    _check(lib.lora_slot_copy(arr, len(arr), int(n_slots), int(r_max), int(slot), int(rank), _stream(stream)),
           "lora_slot_copy")


def lora_slot_assign(table: SlotTable, adapter: int, slot: int, rank: int = 0, *, stream=None) -> None:
    """slot_of[adapter] = slot, rank_of[adapter] = rank on the GPU (slot -1 evicts)."""
    lib = load_library()
    _check(lib.lora_slot_assign(_ptr(table.slot_of), _ptr(table.rank_of), table.n_adapters, int(adapter), int(slot),
                                int(rank), _stream(stream)), "lora_slot_assign")


def make_host_projs(projs: Sequence) -> "ctypes.Array":
    """Host array of lora_proj for sgmv_multi_host from (x_host, A_pool,
    B_pool, y_host, scale) tuples: x_host [n, >=h_in] and y_host [n, >=h_out]
    bf16 CPU tensors (pinned, for an asynchronous call), pools on the GPU."""
    arr = (LoraProj * len(projs))()
    for i, (x, A, B, y, s) in enumerate(projs):
        for t, nm in ((x, "x_host"), (y, "y_host")):
            if t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 2:
                raise ValueError(f"{nm} must be a 2-D bf16 CPU tensor")
            if not t.is_pinned():
                raise ValueError(f"{nm} must be pinned (asynchronous copies)")
        _pool(A, "A_pool")
        _pool(B, "B_pool")
        if A.shape[2] != B.shape[1] or x.shape[1] < A.shape[1] or y.shape[1] < B.shape[2]:
            raise ValueError(f"projection {i}: shape mismatch")
        arr[i] = LoraProj(x.data_ptr(), A.data_ptr(), B.data_ptr(), y.data_ptr(), _rows(x, "x"), _rows(y, "y"),
                          A.shape[1], B.shape[2], float(s))
    return arr


def sgmv_multi_host_workspace_bytes(c_projs, n_tokens: int, n_adapters: int) -> int:
    return int(load_library().sgmv_multi_host_workspace_bytes(c_projs, len(c_projs), int(n_tokens),
                                                              int(n_adapters)))


def sgmv_multi_host(projs: Sequence, ids_host: torch.Tensor, *, workspace: Optional[torch.Tensor] = None,
                    err_flag: Optional[torch.Tensor] = None, stream=None, c_projs=None) -> torch.Tensor:
    """The whole step from host memory (include/lora_sgmv.h): ids_host int32
    [n] and the projections' x / y pinned CPU tensors, pools on the GPU; y is
    updated in place in host memory once the stream reaches the end of the
    call.  Returns the device workspace (reuse it for the next call)."""
    lib = load_library()
    if not 1 <= len(projs) <= LORA_MAX_PROJ:
        raise ValueError("1..8 projections")
    if ids_host.is_cuda or ids_host.dtype != torch.int32 or ids_host.dim() != 1 or not ids_host.is_pinned():
        raise ValueError("ids_host must be a pinned 1-D int32 CPU tensor")
    arr = c_projs if c_projs is not None else make_host_projs(projs)
    P, _, r = projs[0][1].shape
    n = ids_host.shape[0]
    if workspace is None:
        need = sgmv_multi_host_workspace_bytes(arr, n, P)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=projs[0][1].device)
    # (a given workspace that is too small: LORA_ERR_WORKSPACE from the library)
    _check(lib.sgmv_multi_host(arr, len(arr), P, r, _ptr(ids_host), n, _ptr(workspace), workspace.numel(),
                               _ptr(err_flag), _stream(stream)), "sgmv_multi_host")
    return workspace


def sgmv_multi_segment(projs: Sequence, ids: torch.Tensor, n_adapters: int, *, out: Optional[Segments] = None,
                       workspace: Optional[torch.Tensor] = None, err_flag: Optional[torch.Tensor] = None,
                       stream=None, c_projs=None) -> Segments:
    """lora_segment + sgmv_multi as one call (one launch for small batches):
    returns the segmentation, written into `out` when given."""
    lib = load_library()
    _req(ids, "ids", torch.int32, 1)
    if not 1 <= len(projs) <= LORA_MAX_PROJ:
        raise ValueError("1..8 projections")
    n = ids.shape[0]
    seg = out if out is not None else Segments.empty(n, n_adapters, ids.device)
    if seg.n_tokens != n or seg.n_adapters != n_adapters:
        raise ValueError("out was sized for another batch")
    arr = c_projs if c_projs is not None else make_projs(projs)
    r = projs[0][1].shape[2]
    need = lora_segment_workspace_bytes(n, n_adapters)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=ids.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.sgmv_multi_segment(arr, len(arr), int(n_adapters), int(r), _ptr(ids), n, _ptr(seg.perm),
                                  _ptr(seg.seg_offsets), _ptr(seg.seg_adapter), _ptr(seg.num_segments),
                                  _ptr(workspace), ws_bytes, _ptr(err_flag), _stream(stream)), "sgmv_multi_segment")
    return seg


def sgmv_fused_segment(x: torch.Tensor, A_pool: torch.Tensor, B_pool: torch.Tensor, ids: torch.Tensor,
                       y: torch.Tensor, scale: float, *, out: Optional[Segments] = None,
                       err_flag: Optional[torch.Tensor] = None, stream=None) -> Segments:
    """One projection of sgmv_multi_segment (y updated in place)."""
    return sgmv_multi_segment([(x, A_pool, B_pool, y, scale)], ids, A_pool.shape[0], out=out, err_flag=err_flag,
                              stream=stream)


def gemm_lora_workspace_bytes(n_tokens: int, r: int) -> int:
    return int(load_library().gemm_lora_workspace_bytes(int(n_tokens), int(r)))


def gemm_lora(x: torch.Tensor, W: torch.Tensor, A_pool: torch.Tensor, B_pool: torch.Tensor, seg: Segments,
              y: torch.Tensor, scale: float, *, workspace: Optional[torch.Tensor] = None,
              err_flag: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """y = x . W + scale * (x . A[a_i]) . B[a_i] with the expand fused into the
    backbone GEMM (y written, not accumulated).  W: [h_in, h_out] bf16."""
    lib = load_library()
    _req(x, "x", torch.bfloat16, 2)
    _req(y, "y", torch.bfloat16, 2)
    _req(W, "W", torch.bfloat16, 2)
    _pool(A_pool, "A_pool")
    _pool(B_pool, "B_pool")
    P, h_in, r = A_pool.shape
    if tuple(W.shape) != (h_in, y.shape[1]) or not W.is_contiguous():
        raise ValueError("W must be a contiguous [h_in, h_out] tensor")
    if x.shape[1] != h_in or B_pool.shape != (P, r, y.shape[1]):
        raise ValueError("shape mismatch")
    need = gemm_lora_workspace_bytes(x.shape[0], r)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _check(lib.gemm_lora(_ptr(x), _rows(x, "x"), _ptr(W), _ptr(A_pool), _ptr(B_pool), P, h_in, y.shape[1], r,
                         float(scale), ctypes.byref(seg.c_struct), _ptr(y), _rows(y, "y"), _ptr(workspace),
                         workspace.numel() * workspace.element_size(), _ptr(err_flag), _stream(stream)), "gemm_lora")
    return y
