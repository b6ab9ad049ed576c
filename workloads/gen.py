"""Seeded synthetic inputs shaped like Llama2 multi-LoRA serving batches.

Value distributions (the second parameter of N(.,.) is a variance):
  x ~ N(0, 1), A ~ N(0, 1/h_in), B ~ N(0, 1/r), y0 ~ N(0, 1),
each drawn in fp32 and rounded to bf16 with round-to-nearest-even.
Adapter-id patterns: shuffled fixed segment lengths, one adapter for all
tokens, all-distinct adapters, finite Zipf(alpha) over the pool
(p(k) proportional to k^-alpha for rank k = 1..P, rank k -> adapter k-1),
and prefill requests of uniform random prompt lengths sorted by adapter.

Punica: Multi-Tenant LoRA Serving (research.elamur.ai summary), "Key points":
rank is far below the hidden size (16 vs 4096), and the evaluation uses
Llama2 7B/13B/70B; the projection shapes below are those models' q/k/v/o
(h -> h), gate/up (h -> intermediate) and down (intermediate -> h).
"""

from __future__ import annotations

import math
import zlib
from dataclasses import dataclass, field
from typing import Callable, Dict, List, Optional

import numpy as np
import torch

# hidden size, MLP intermediate size
LLAMA_DIMS = {"7b": (4096, 11008), "13b": (5120, 13824), "70b": (8192, 28672)}


@dataclass(frozen=True)
class Proj:
    name: str
    h_in: int
    h_out: int
    x_key: str  # projections with the same x_key read the same input rows


@dataclass(frozen=True)
class Workload:
    name: str
    projs: tuple
    r: int
    P: int
    n: int
    scale: float
    ids_fn: Callable[[], np.ndarray] = field(compare=False)
    description: str = ""
    data_name: str = ""  # seeds the values; workloads sharing it share x, pools, y0

    @property
    def seed_name(self) -> str:
        return self.data_name or self.name

    def ids(self) -> np.ndarray:
        ids = np.asarray(self.ids_fn(), dtype=np.int32)
        assert ids.shape == (self.n,)
        return ids


def llama_projs(model: str) -> tuple:
    h, inter = LLAMA_DIMS[model]
    return (
        Proj("q", h, h, "attn"),
        Proj("k", h, h, "attn"),
        Proj("v", h, h, "attn"),
        Proj("o", h, h, "o"),
        Proj("gate", h, inter, "mlp"),
        Proj("up", h, inter, "mlp"),
        Proj("down", inter, h, "down"),
    )


# ---------------------------------------------------------------- adapter ids

def tiny_ids(seed: int = 0) -> np.ndarray:
    """16 tokens in 4 segments of lengths 1,3,5,7 (adapter k gets length
    (1,3,5,7)[k]), the id list shuffled per token."""
    base = np.repeat(np.arange(4, dtype=np.int32), [1, 3, 5, 7])
    return base[np.random.default_rng(seed).permutation(base.size)]


def same_ids(n: int, P: int, seed: int = 0) -> np.ndarray:
    a = int(np.random.default_rng(seed).integers(P))
    return np.full(n, a, dtype=np.int32)


def distinct_ids(n: int, P: int, seed: int = 0) -> np.ndarray:
    return np.random.default_rng(seed).choice(P, n, replace=False).astype(np.int32)


def zipf_ids(n: int, P: int, alpha: float, seed: int = 0) -> np.ndarray:
    k = np.arange(1, P + 1, dtype=np.float64)
    p = k ** (-alpha)
    p /= p.sum()
    return np.random.default_rng(seed).choice(P, n, p=p).astype(np.int32)


def compact_ids(ids: np.ndarray) -> np.ndarray:
    """Ids relabelled 0..k-1 in increasing order of the original ids (the
    stable sort by adapter and its segments are unchanged)."""
    return np.unique(ids, return_inverse=True)[1].astype(np.int32)


def prefill_ids(n_requests: int = 8, P: int = 32, lo: int = 128, hi: int = 2048,
                seed: int = 0, interleave: bool = False) -> np.ndarray:
    """Prefill batch: request i has a prompt of L_i ~ U{lo..hi} tokens and its
    own adapter (distinct, drawn from the pool); requests are laid out in
    ascending adapter order, so the batch is already sorted by adapter.  With
    interleave, the requests' tokens are dealt out round robin instead (same
    ids, no request's rows contiguous)."""
    rng = np.random.default_rng(seed)
    lengths = rng.integers(lo, hi + 1, n_requests)
    adapters = rng.choice(P, n_requests, replace=False)
    order = np.argsort(adapters, kind="stable")
    if not interleave:
        return np.concatenate([np.full(lengths[i], adapters[i], dtype=np.int32) for i in order])
    left = [int(lengths[i]) for i in order]
    out = []
    while any(left):
        for k, i in enumerate(order):
            if left[k]:
                out.append(adapters[i])
                left[k] -= 1
    return np.asarray(out, dtype=np.int32)


# ---------------------------------------------------------------- workloads

def _mk(name, projs, r, P, n, scale, ids_fn, desc, data_name="") -> Workload:
    return Workload(name, tuple(projs), r, P, n, scale, ids_fn, desc, data_name)


def _build_workloads() -> Dict[str, Workload]:
    w: Dict[str, Workload] = {}
    w["tiny"] = _mk("tiny", [Proj("proj", 256, 256, "x")], 8, 4, 16, 2.0, tiny_ids,
                    "h_in=h_out=256, r=8, pool 4, 16 tokens in segments of 1,3,5,7, s=2")
    h7, _ = LLAMA_DIMS["7b"]
    p7 = [Proj("proj", h7, h7, "x")]
    w["7b_proj_same"] = _mk("7b_proj_same", p7, 16, 64, 32, 1.0, lambda: same_ids(32, 64),
                            "Llama2-7B decode projection 4096->4096, r=16, 32 tokens, pool 64, one adapter",
                            "7b_proj")
    w["7b_proj_distinct"] = _mk("7b_proj_distinct", p7, 16, 64, 32, 1.0, lambda: distinct_ids(32, 64),
                                "Llama2-7B decode projection 4096->4096, r=16, 32 tokens, pool 64, 32 distinct adapters",
                                "7b_proj")
    w["7b_proj_zipf"] = _mk("7b_proj_zipf", p7, 16, 64, 32, 1.0, lambda: zipf_ids(32, 64, 1.0),
                            "Llama2-7B decode projection 4096->4096, r=16, 32 tokens, pool 64, Zipf(1.0) ids",
                            "7b_proj")
    w["7b_layer"] = _mk("7b_layer", llama_projs("7b"), 16, 128, 64, 1.0, lambda: zipf_ids(64, 128, 1.0),
                        "Llama2-7B decode layer, 7 projections, r=16, 64 tokens, pool 128, Zipf(1.0), unsorted")
    ids13 = prefill_ids()
    w["13b_prefill"] = _mk("13b_prefill", llama_projs("13b"), 64, 32, int(ids13.size), 1.0,
                           prefill_ids,
                           "Llama2-13B prefill, 7 projections, r=64, 8 requests of U[128,2048] tokens, "
                           "8 adapters of pool 32, sorted by adapter")
    w["13b_prefill_interleaved"] = _mk("13b_prefill_interleaved", llama_projs("13b"), 64, 32, int(ids13.size), 1.0,
                                       lambda: prefill_ids(interleave=True),
                                       "Llama2-13B prefill, 7 projections, r=64, the 8 requests of the prefill batch "
                                       "with their tokens interleaved round robin (rows gathered per segment)",
                                       "13b_prefill")
    ids13s = prefill_ids(n_requests=2)
    w["13b_prefill_small"] = _mk("13b_prefill_small", llama_projs("13b"), 64, 32, int(ids13s.size),
                                 1.0, lambda: prefill_ids(n_requests=2),
                                 "Llama2-13B prefill, 7 projections, r=64, 2 requests of U[128,2048] tokens, "
                                 "2 adapters of pool 32, sorted by adapter (a smaller case of the 8-request batch)")
    h13, _ = LLAMA_DIMS["13b"]
    w["13b_proj_2048"] = _mk("13b_proj_2048", [Proj("proj", h13, h13, "x")], 64, 32, 2048, 1.0,
                             lambda: same_ids(2048, 32),
                             "Llama2-13B prefill projection 5120->5120, r=64, one request of 2048 tokens, pool 32 "
                             "(a few 128-token tiles: the cluster-split case)")
    for r in (8, 16, 32, 64):
        nm = f"70b_decode_r{r}"
        w[nm] = _mk(nm, llama_projs("70b"), r, 1000, 256, 1.0, lambda: zipf_ids(256, 1000, 0.8),
                    f"Llama2-70B decode, 7 projections, r={r}, 256 tokens, pool 1000, Zipf(0.8)")
    # the same launches over a pool of only the adapters the batch uses (the
    # ids relabelled in order, so segments and bytes moved are unchanged): a
    # device footprint small enough for a profiler capture
    n_used = int(np.unique(zipf_ids(256, 1000, 0.8)).size)
    for r in (8, 16):
        nm = f"70b_decode_r{r}_compact"
        w[nm] = _mk(nm, llama_projs("70b"), r, n_used, 256, 1.0, lambda: compact_ids(zipf_ids(256, 1000, 0.8)),
                    f"the 70b_decode_r{r} batch over a pool of its {n_used} adapters (ids relabelled in order)")
    return w


WORKLOADS = _build_workloads()


def workload(name: str) -> Workload:
    return WORKLOADS[name]


# ---------------------------------------------------------------- values

def seed_for(*parts) -> int:
    """Stable 31-bit seed from a tuple of names/ints (same on every host)."""
    return zlib.crc32("/".join(str(p) for p in parts).encode()) & 0x7FFFFFFF


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); returns
    the 16-bit patterns as uint16. Finite inputs only."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(shape, var: float, seed: int, device="cpu") -> torch.Tensor:
    """bf16 tensor of N(0, var) draws (fp32 draw, RNE rounding)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if var != 1.0:
        t.mul_(math.sqrt(var))
    return t.to(torch.bfloat16)


@dataclass
class Inputs:
    wl: Workload
    ids: torch.Tensor                 # int32 [n]
    x: Dict[str, torch.Tensor]        # x_key -> bf16 [n, h_in]
    A: List[torch.Tensor]             # per projection bf16 [P, h_in, r]
    B: List[torch.Tensor]             # per projection bf16 [P, r, h_out]
    y0: List[torch.Tensor]            # per projection bf16 [n, h_out]


def make_inputs(wl: Workload, device="cpu", copy: int = 0,
                ids: Optional[np.ndarray] = None) -> Inputs:
    """Materialise a workload on `device`. `copy` selects an independent
    draw of the same distributions (used to rotate buffers)."""
    ids_np = wl.ids() if ids is None else np.asarray(ids, dtype=np.int32)
    n = ids_np.size
    dev_ids = torch.from_numpy(ids_np.copy()).to(device)
    xs: Dict[str, torch.Tensor] = {}
    for p in wl.projs:
        if p.x_key not in xs:
            xs[p.x_key] = normal_bf16((n, p.h_in), 1.0, seed_for(wl.seed_name, "x", p.x_key, copy), device)
    A, B, Y = [], [], []
    for i, p in enumerate(wl.projs):
        A.append(normal_bf16((wl.P, p.h_in, wl.r), 1.0 / p.h_in, seed_for(wl.seed_name, "A", p.name, copy), device))
        B.append(normal_bf16((wl.P, wl.r, p.h_out), 1.0 / wl.r, seed_for(wl.seed_name, "B", p.name, copy), device))
        Y.append(normal_bf16((n, p.h_out), 1.0, seed_for(wl.seed_name, "y0", p.name, copy), device))
    return Inputs(wl, dev_ids, xs, A, B, Y)


@dataclass
class SlotInputs:
    ids: torch.Tensor       # int32 [n]
    x: torch.Tensor         # bf16 [n, h_in]
    A_arena: torch.Tensor   # bf16 [n_slots, h_in * r_max]
    B_arena: torch.Tensor   # bf16 [n_slots, r_max * h_out]
    y0: torch.Tensor        # bf16 [n, h_out]
    slot_of: torch.Tensor   # int32 [P]
    rank_of: torch.Tensor   # int32 [P]


def make_slot_inputs(h_in: int, h_out: int, ids: np.ndarray, rank_of: np.ndarray, n_slots: int, r_max: int,
                     device="cpu", copy: int = 0, name: str = "slots") -> SlotInputs:
    """Slot arenas for adapters of the given ranks (A ~ N(0, 1/h_in), B ~
    N(0, 1/r) at the start of a shuffled slot each, the rest of the arena
    N(0, 1) junk), with x ~ N(0, 1) and y0 ~ N(0, 1) rows for the tokens `ids`."""
    P = int(len(rank_of))
    rng = np.random.default_rng(seed_for(name, "slots", copy))
    slots = rng.permutation(n_slots)[:P].astype(np.int32)
    A_ar = normal_bf16((n_slots, h_in * r_max), 1.0, seed_for(name, "A_junk", copy), device)
    B_ar = normal_bf16((n_slots, r_max * h_out), 1.0, seed_for(name, "B_junk", copy), device)
    for a in range(P):
        r = int(rank_of[a])
        A_ar[int(slots[a]), : h_in * r] = normal_bf16((h_in * r,), 1.0 / h_in, seed_for(name, "A", a, copy), device)
        B_ar[int(slots[a]), : r * h_out] = normal_bf16((r * h_out,), 1.0 / r, seed_for(name, "B", a, copy), device)
    ids_np = np.asarray(ids, dtype=np.int32)
    n = ids_np.size
    return SlotInputs(torch.from_numpy(ids_np.copy()).to(device),
                      normal_bf16((n, h_in), 1.0, seed_for(name, "x", copy), device), A_ar, B_ar,
                      normal_bf16((n, h_out), 1.0, seed_for(name, "y0", copy), device),
                      torch.from_numpy(slots).to(device), torch.from_numpy(np.asarray(rank_of, np.int32)).to(device))


def make_backbone_weights(wl: Workload, device="cpu", copy: int = 0) -> List[torch.Tensor]:
    """Synthetic backbone weights W [h_in][h_out] per projection, N(0, 1/h_in)
    (so x . W ~ N(0, 1) for x ~ N(0, 1)), rounded to bf16."""
    return [normal_bf16((p.h_in, p.h_out), 1.0 / p.h_in, seed_for(wl.seed_name, "W", p.name, copy), device)
            for p in wl.projs]
