"""B300 (sm_103a) multi-LoRA SGMV: y[i] += s * (x[i] . A[a_i]) . B[a_i] for a
batch whose tokens name adapters of an HBM-resident pool.

The compute lives in liblora_sgmv.so (hand-written CUDA kernels behind a C
ABI, declared in include/lora_sgmv.h); this package is its thin binding.
"""

from .lora_sgmv import (  # noqa: F401
    LIB_PATH,
    LORA_MAX_PROJ,
    STATUS,
    SYMBOLS,
    Segments,
    SlotTable,
    gemm_lora,
    gemm_lora_workspace_bytes,
    load_library,
    lora_segment,
    lora_segment_noalloc,
    lora_segment_workspace_bytes,
    lora_slot_assign,
    lora_slot_copy,
    make_host_projs,
    make_projs,
    make_slot_projs,
    make_slot_srcs,
    rank_mask,
    sgmv_expand,
    sgmv_fused,
    sgmv_fused_slots,
    sgmv_multi,
    sgmv_multi_host,
    sgmv_multi_host_workspace_bytes,
    sgmv_multi_segment,
    sgmv_fused_segment,
    sgmv_multi_slots,
    sgmv_shrink,
)

__all__ = [
    "Segments", "load_library", "lora_segment", "lora_segment_noalloc", "lora_segment_workspace_bytes", "sgmv_shrink", "sgmv_expand",
    "sgmv_fused", "sgmv_multi", "make_projs", "SlotTable", "rank_mask", "make_slot_projs", "sgmv_multi_slots",
    "sgmv_fused_slots", "lora_slot_copy", "lora_slot_assign", "make_slot_srcs",
    "sgmv_multi_host", "sgmv_multi_host_workspace_bytes", "make_host_projs", "sgmv_multi_segment",
    "sgmv_fused_segment", "gemm_lora", "gemm_lora_workspace_bytes",
]
