// C ABI of liblora_sgmv.so: argument checks on the host, then one launch per
// call on the caller's stream.  Declarations and contracts: include/lora_sgmv.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "internal.h"

namespace lsg {

lora_status cuda_status(cudaError_t e) { return e == cudaSuccess ? LORA_OK : LORA_ERR_CUDA; }

namespace {

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool rank_ok(int r) { return r == 8 || r == 16 || r == 32 || r == 64; }
bool width_ok(int h) { return h >= 8 && (h % 8) == 0; }

lora_status check_seg(const lora_segments* seg, int n_adapters) {
  if (seg == nullptr || n_adapters < 1) return LORA_ERR_INVALID_ARG;
  if (seg->n_tokens < 0) return LORA_ERR_INVALID_ARG;
  if (seg->n_tokens == 0) return LORA_OK;
  if (!seg->perm || !seg->seg_offsets || !seg->seg_adapter || !seg->num_segments) return LORA_ERR_INVALID_ARG;
  if (seg->max_segments < 1 || seg->max_segments > seg->n_tokens) return LORA_ERR_INVALID_ARG;
  if (!al4(seg->perm) || !al4(seg->seg_offsets) || !al4(seg->seg_adapter) || !al4(seg->num_segments))
    return LORA_ERR_MISALIGNED;
  return LORA_OK;
}

lora_status check_proj(const lora_bf16* x, int64_t ldx, const lora_bf16* A, const lora_bf16* B, lora_bf16* y,
                       int64_t ldy, int h_in, int h_out, bool need_x, bool need_y) {
  if (need_x) {
    if (!x || !A) return LORA_ERR_INVALID_ARG;
    if (!width_ok(h_in)) return LORA_ERR_UNSUPPORTED;
    if (ldx < h_in) return LORA_ERR_INVALID_ARG;
    if (!al16(x) || !al16(A) || (ldx % 8) != 0) return LORA_ERR_MISALIGNED;
  }
  if (need_y) {
    if (!y || !B) return LORA_ERR_INVALID_ARG;
    if (!width_ok(h_out)) return LORA_ERR_UNSUPPORTED;
    if (ldy < h_out) return LORA_ERR_INVALID_ARG;
    if (!al16(y) || !al16(B) || (ldy % 8) != 0) return LORA_ERR_MISALIGNED;
  }
  return LORA_OK;
}

}  // namespace
}  // namespace lsg

using namespace lsg;

extern "C" {

const char* lora_status_str(int s) {
  switch (s) {
    case LORA_OK: return "LORA_OK";
    case LORA_ERR_INVALID_ARG: return "LORA_ERR_INVALID_ARG: invalid argument";
    case LORA_ERR_MISALIGNED: return "LORA_ERR_MISALIGNED: pointer or leading dimension not 16-byte aligned";
    case LORA_ERR_UNSUPPORTED: return "LORA_ERR_UNSUPPORTED: rank or width not supported";
    case LORA_ERR_BAD_ADAPTER_ID:
      return "LORA_ERR_BAD_ADAPTER_ID: adapter id, permutation entry, slot or rank out of range";
    case LORA_ERR_WORKSPACE: return "LORA_ERR_WORKSPACE: workspace missing or too small";
    case LORA_ERR_CUDA: return "LORA_ERR_CUDA: CUDA runtime error";
    case LORA_ERR_TIMEOUT: return "LORA_ERR_TIMEOUT: a bounded wait in a kernel ran out";
    default: return "unknown status";
  }
}

int lora_abi_version(void) { return LORA_SGMV_ABI_VERSION; }

#ifdef LSG_TEST_HOOKS
// Test builds only (not declared in the public header): which signal the
// kernels withhold, so that a bounded wait runs out (see internal.h).
LORA_API lora_status lora_test_withhold(int what) {
  lora_status s = test_withhold_cc(what);
  if (s == LORA_OK) s = test_withhold_tc(what);
  return s != LORA_OK ? s : test_withhold_gl(what);
}
#endif

size_t lora_segment_workspace_bytes(int32_t n_tokens, int32_t n_adapters) {
  if (n_tokens < 0 || n_adapters < 1) return 0;
  return seg_plan(n_tokens, n_adapters).ws_bytes;
}

lora_status lora_segment(const int32_t* ids, int32_t n_tokens, int32_t n_adapters, int32_t* perm,
                         int32_t* seg_offsets, int32_t* seg_adapter, int32_t* num_segments, void* workspace,
                         size_t workspace_bytes, int32_t* err_flag, lora_stream_t stream) {
  if (n_tokens < 0 || n_adapters < 1) return LORA_ERR_INVALID_ARG;
  if (!seg_offsets || !num_segments) return LORA_ERR_INVALID_ARG;
  if (n_tokens > 0 && (!ids || !perm || !seg_adapter)) return LORA_ERR_INVALID_ARG;
  const SegPlan pl = seg_plan(n_tokens, n_adapters);
  if (pl.gmem && (workspace == nullptr || workspace_bytes < pl.ws_bytes)) return LORA_ERR_WORKSPACE;
  if (pl.gmem && !al4(workspace)) return LORA_ERR_MISALIGNED;
  return launch_segment(ids, n_tokens, n_adapters, perm, seg_offsets, seg_adapter, num_segments,
                        static_cast<int32_t*>(workspace), err_flag, reinterpret_cast<cudaStream_t>(stream));
}

lora_status sgmv_shrink(const lora_bf16* x, int64_t ldx, const lora_bf16* A_pool, int32_t n_adapters,
                        int32_t h_in, int32_t r, const lora_segments* seg, float* v, int32_t* err_flag,
                        lora_stream_t stream) {
  lora_status s = check_seg(seg, n_adapters);
  if (s != LORA_OK) return s;
  if (!rank_ok(r)) return LORA_ERR_UNSUPPORTED;
  if (seg->n_tokens == 0) return LORA_OK;
  s = check_proj(x, ldx, A_pool, nullptr, nullptr, 0, h_in, 0, true, false);
  if (s != LORA_OK) return s;
  if (!v) return LORA_ERR_INVALID_ARG;
  if (!al16(v)) return LORA_ERR_MISALIGNED;
  SgmvCall c{};
  c.mode = kModeShrink;
  c.proj[0] = ProjArgs{x, A_pool, nullptr, nullptr, ldx, 0, h_in, 0, 1.0f};
  c.n_proj = 1;
  c.r = r;
  c.n_adapters = n_adapters;
  c.seg = *seg;
  c.v_out = v;
  c.err_flag = err_flag;
  return launch_sgmv_cc(c, reinterpret_cast<cudaStream_t>(stream));
}

lora_status sgmv_expand(const float* v, const lora_bf16* B_pool, int32_t n_adapters, int32_t r, int32_t h_out,
                        float scale, const lora_segments* seg, lora_bf16* y, int64_t ldy, int32_t* err_flag,
                        lora_stream_t stream) {
  lora_status s = check_seg(seg, n_adapters);
  if (s != LORA_OK) return s;
  if (!rank_ok(r)) return LORA_ERR_UNSUPPORTED;
  if (seg->n_tokens == 0) return LORA_OK;
  s = check_proj(nullptr, 0, nullptr, B_pool, y, ldy, 0, h_out, false, true);
  if (s != LORA_OK) return s;
  if (!v) return LORA_ERR_INVALID_ARG;
  if (!al16(v)) return LORA_ERR_MISALIGNED;
  SgmvCall c{};
  c.mode = kModeExpand;
  c.proj[0] = ProjArgs{nullptr, nullptr, B_pool, y, 0, ldy, 0, h_out, scale};
  c.n_proj = 1;
  c.r = r;
  c.n_adapters = n_adapters;
  c.seg = *seg;
  c.v_in = v;
  c.err_flag = err_flag;
  return launch_sgmv_cc(c, reinterpret_cast<cudaStream_t>(stream));
}

lora_status sgmv_multi(const lora_proj* projs, int32_t n_proj, int32_t n_adapters, int32_t r,
                       const lora_segments* seg, int32_t* err_flag, lora_stream_t stream) {
  if (!projs || n_proj < 1) return LORA_ERR_INVALID_ARG;
  if (n_proj > LORA_MAX_PROJ) return LORA_ERR_UNSUPPORTED;
  lora_status s = check_seg(seg, n_adapters);
  if (s != LORA_OK) return s;
  if (!rank_ok(r)) return LORA_ERR_UNSUPPORTED;
  if (seg->n_tokens == 0) return LORA_OK;
  SgmvCall c{};
  c.mode = kModeFused;
  for (int i = 0; i < n_proj; ++i) {
    const lora_proj& q = projs[i];
    s = check_proj(q.x, q.ldx, q.A_pool, q.B_pool, q.y, q.ldy, q.h_in, q.h_out, true, true);
    if (s != LORA_OK) return s;
    c.proj[i] = ProjArgs{q.x, q.A_pool, q.B_pool, q.y, q.ldx, q.ldy, q.h_in, q.h_out, q.scale};
  }
  c.n_proj = n_proj;
  c.r = r;
  c.n_adapters = n_adapters;
  c.seg = *seg;
  c.err_flag = err_flag;
  return launch_sgmv_cc(c, reinterpret_cast<cudaStream_t>(stream));
}

lora_status sgmv_multi_slots(const lora_proj* projs, int32_t n_proj, const lora_slot_table* table,
                             const lora_segments* seg, int32_t* err_flag, lora_stream_t stream) {
  if (!projs || n_proj < 1 || !table) return LORA_ERR_INVALID_ARG;
  if (n_proj > LORA_MAX_PROJ) return LORA_ERR_UNSUPPORTED;
  const lora_slot_table& t = *table;
  lora_status s = check_seg(seg, t.n_adapters);
  if (s != LORA_OK) return s;
  if (!t.slot_of || !t.rank_of || t.n_slots < 1) return LORA_ERR_INVALID_ARG;
  if (!al4(t.slot_of) || !al4(t.rank_of)) return LORA_ERR_MISALIGNED;
  if (!rank_ok(t.r_max)) return LORA_ERR_UNSUPPORTED;
  if (t.rank_mask == 0 || (t.rank_mask >> 4) != 0) return LORA_ERR_UNSUPPORTED;
  for (int c = 0; c < 4; ++c)
    if ((t.rank_mask & (1u << c)) && (8 << c) > t.r_max) return LORA_ERR_UNSUPPORTED;
  if (seg->n_tokens == 0) return LORA_OK;
  SgmvCall c{};
  c.mode = kModeFused;
  for (int i = 0; i < n_proj; ++i) {
    const lora_proj& q = projs[i];
    s = check_proj(q.x, q.ldx, q.A_pool, q.B_pool, q.y, q.ldy, q.h_in, q.h_out, true, true);
    if (s != LORA_OK) return s;
    // tensor-map rows: n_slots * h_in * r_max / 8 (A as rank-8 rows) and n_slots * r_max (B)
    const int64_t cells = static_cast<int64_t>(t.n_slots) * t.r_max * std::max(q.h_in, q.h_out);
    if (cells >= (int64_t{1} << 31)) return LORA_ERR_UNSUPPORTED;
    c.proj[i] = ProjArgs{q.x, q.A_pool, q.B_pool, q.y, q.ldx, q.ldy, q.h_in, q.h_out, q.scale};
  }
  c.n_proj = n_proj;
  c.r = t.r_max;
  c.n_adapters = t.n_adapters;
  c.seg = *seg;
  c.err_flag = err_flag;
  c.slot_of = t.slot_of;
  c.rank_of = t.rank_of;
  c.n_slots = t.n_slots;
  c.r_max = t.r_max;
  c.rank_mask = t.rank_mask;
  return launch_sgmv_cc(c, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace lsg {
namespace {

// Device workspace of a host-memory step: ids, segmentation, histogram
// workspace, one x per distinct host x, one y per projection (each 256-byte
// aligned, rows packed at ld = width).
struct HostPlan {
  size_t ids, perm, offs, adap, nseg, hist, total;
  size_t x[kMaxProj], y[kMaxProj];
  int x_of[kMaxProj];  // projection -> index of its distinct x
};

size_t al256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

HostPlan host_plan(const lora_proj* projs, int n_proj, int n, int P) {
  HostPlan h{};
  const int ms = std::min(n, P);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = al256(o + bytes);
    return at;
  };
  h.ids = take(static_cast<size_t>(n) * 4);
  h.perm = take(static_cast<size_t>(n) * 4);
  h.offs = take(static_cast<size_t>(ms + 1) * 4);
  h.adap = take(static_cast<size_t>(std::max(ms, 1)) * 4);
  h.nseg = take(4);
  h.hist = take(seg_plan(n, P).ws_bytes);
  for (int i = 0; i < n_proj; ++i) {
    h.x_of[i] = i;
    for (int j = 0; j < i; ++j)
      if (projs[j].x == projs[i].x && projs[j].h_in == projs[i].h_in) {
        h.x_of[i] = h.x_of[j];
        break;
      }
    if (h.x_of[i] == i) h.x[i] = take(static_cast<size_t>(n) * projs[i].h_in * 2);
  }
  for (int i = 0; i < n_proj; ++i) h.y[i] = take(static_cast<size_t>(n) * projs[i].h_out * 2);
  h.total = o;
  return h;
}

}  // namespace
}  // namespace lsg

extern "C" {

size_t sgmv_multi_host_workspace_bytes(const lora_proj* projs, int32_t n_proj, int32_t n_tokens,
                                       int32_t n_adapters) {
  if (!projs || n_proj < 1 || n_proj > LORA_MAX_PROJ || n_tokens < 0 || n_adapters < 1) return 0;
  return host_plan(projs, n_proj, n_tokens, n_adapters).total;
}

lora_status sgmv_multi_host(const lora_proj* projs, int32_t n_proj, int32_t n_adapters, int32_t r,
                            const int32_t* ids_host, int32_t n_tokens, void* workspace, size_t workspace_bytes,
                            int32_t* err_flag, lora_stream_t stream) {
  if (!projs || n_proj < 1 || n_adapters < 1 || n_tokens < 0) return LORA_ERR_INVALID_ARG;
  if (n_proj > LORA_MAX_PROJ) return LORA_ERR_UNSUPPORTED;
  if (!rank_ok(r)) return LORA_ERR_UNSUPPORTED;
  if (n_tokens == 0) return LORA_OK;
  if (!ids_host) return LORA_ERR_INVALID_ARG;
  for (int i = 0; i < n_proj; ++i) {
    const lora_proj& q = projs[i];
    // host x / y: widths and leading dimensions only (no device alignment rule)
    if (!q.x || !q.y || !q.A_pool || !q.B_pool) return LORA_ERR_INVALID_ARG;
    if (!width_ok(q.h_in) || !width_ok(q.h_out)) return LORA_ERR_UNSUPPORTED;
    if (q.ldx < q.h_in || q.ldy < q.h_out) return LORA_ERR_INVALID_ARG;
    if (!al16(q.A_pool) || !al16(q.B_pool)) return LORA_ERR_MISALIGNED;
  }
  const HostPlan h = host_plan(projs, n_proj, n_tokens, n_adapters);
  if (!workspace || workspace_bytes < h.total) return LORA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LORA_ERR_MISALIGNED;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto at = [&](size_t off) { return ws + off; };
  int32_t* ids = reinterpret_cast<int32_t*>(at(h.ids));
  const size_t n = static_cast<size_t>(n_tokens);
  // rows of width w with leading dimension ld: one flat copy when they are
  // contiguous (ld == w), else a 2-D copy
  auto copy_rows = [&](void* dst, size_t dld, const void* src, size_t sld, size_t w) {
    if (dld == w && sld == w) return cudaMemcpyAsync(dst, src, w * n, cudaMemcpyDefault, st);
    return cudaMemcpy2DAsync(dst, dld, src, sld, w, n, cudaMemcpyDefault, st);
  };
  for (int i = 0; i < n_proj; ++i) {
    const lora_proj& q = projs[i];
    if (h.x_of[i] == i && copy_rows(at(h.x[i]), q.h_in * 2, q.x, q.ldx * 2, q.h_in * 2) != cudaSuccess)
      return LORA_ERR_CUDA;
    if (copy_rows(at(h.y[i]), q.h_out * 2, q.y, q.ldy * 2, q.h_out * 2) != cudaSuccess) return LORA_ERR_CUDA;
  }
  lora_segments seg{};
  seg.perm = reinterpret_cast<int32_t*>(at(h.perm));
  seg.seg_offsets = reinterpret_cast<int32_t*>(at(h.offs));
  seg.seg_adapter = reinterpret_cast<int32_t*>(at(h.adap));
  seg.num_segments = reinterpret_cast<int32_t*>(at(h.nseg));
  seg.n_tokens = n_tokens;
  seg.max_segments = std::min(n_tokens, n_adapters);
  // segmentation inside the SGMV launch when the batch is small (else its own kernel first)
  SgmvCall c{};
  c.ids = ids;
  c.ids_host = ids_host;  // in the launch's parameters, or copied to ids, as the launch needs them
  c.seg_hist = seg_plan(n_tokens, n_adapters).gmem ? reinterpret_cast<int32_t*>(at(h.hist)) : nullptr;
  c.mode = kModeFused;
  for (int i = 0; i < n_proj; ++i) {
    const lora_proj& q = projs[i];
    c.proj[i] = ProjArgs{reinterpret_cast<const uint16_t*>(at(h.x[h.x_of[i]])), q.A_pool, q.B_pool,
                         reinterpret_cast<uint16_t*>(at(h.y[i])), q.h_in, q.h_out, q.h_in, q.h_out, q.scale};
  }
  c.n_proj = n_proj;
  c.r = r;
  c.n_adapters = n_adapters;
  c.seg = seg;
  c.err_flag = err_flag;
  const lora_status s = launch_sgmv_cc(c, st);
  if (s != LORA_OK) return s;
  for (int i = 0; i < n_proj; ++i) {
    const lora_proj& q = projs[i];
    if (copy_rows(q.y, q.ldy * 2, at(h.y[i]), q.h_out * 2, q.h_out * 2) != cudaSuccess) return LORA_ERR_CUDA;
  }
  return LORA_OK;
}

lora_status sgmv_multi_segment(const lora_proj* projs, int32_t n_proj, int32_t n_adapters, int32_t r,
                               const int32_t* ids, int32_t n_tokens, int32_t* perm, int32_t* seg_offsets,
                               int32_t* seg_adapter, int32_t* num_segments, void* workspace, size_t workspace_bytes,
                               int32_t* err_flag, lora_stream_t stream) {
  if (!projs || n_proj < 1 || n_tokens < 0 || n_adapters < 1) return LORA_ERR_INVALID_ARG;
  if (n_proj > LORA_MAX_PROJ) return LORA_ERR_UNSUPPORTED;
  if (!rank_ok(r)) return LORA_ERR_UNSUPPORTED;
  if (!seg_offsets || !num_segments) return LORA_ERR_INVALID_ARG;
  if (n_tokens > 0 && (!ids || !perm || !seg_adapter)) return LORA_ERR_INVALID_ARG;
  if (!al4(seg_offsets) || !al4(num_segments) || (n_tokens > 0 && (!al4(ids) || !al4(perm) || !al4(seg_adapter))))
    return LORA_ERR_MISALIGNED;
  const SegPlan pl = seg_plan(n_tokens, n_adapters);
  if (pl.gmem && (workspace == nullptr || workspace_bytes < pl.ws_bytes)) return LORA_ERR_WORKSPACE;
  if (pl.gmem && !al4(workspace)) return LORA_ERR_MISALIGNED;
  if (n_tokens == 0)
    return launch_segment(ids, 0, n_adapters, perm, seg_offsets, seg_adapter, num_segments, nullptr, err_flag,
                          reinterpret_cast<cudaStream_t>(stream));
  SgmvCall c{};
  c.mode = kModeFused;
  for (int i = 0; i < n_proj; ++i) {
    const lora_proj& q = projs[i];
    lora_status s = check_proj(q.x, q.ldx, q.A_pool, q.B_pool, q.y, q.ldy, q.h_in, q.h_out, true, true);
    if (s != LORA_OK) return s;
    c.proj[i] = ProjArgs{q.x, q.A_pool, q.B_pool, q.y, q.ldx, q.ldy, q.h_in, q.h_out, q.scale};
  }
  c.n_proj = n_proj;
  c.r = r;
  c.n_adapters = n_adapters;
  c.seg = lora_segments{perm, seg_offsets, seg_adapter, num_segments, n_tokens, std::min(n_tokens, n_adapters)};
  c.err_flag = err_flag;
  c.ids = ids;
  c.seg_hist = pl.gmem ? static_cast<int32_t*>(workspace) : nullptr;
  return launch_sgmv_cc(c, reinterpret_cast<cudaStream_t>(stream));
}

size_t gemm_lora_workspace_bytes(int32_t n_tokens, int32_t r) {
  if (n_tokens < 0 || !rank_ok(r)) return 0;
  return static_cast<size_t>(kGlVParts) * n_tokens * r * sizeof(float);
}

lora_status gemm_lora(const lora_bf16* x, int64_t ldx, const lora_bf16* W, const lora_bf16* A_pool,
                      const lora_bf16* B_pool, int32_t n_adapters, int32_t h_in, int32_t h_out, int32_t r, float scale,
                      const lora_segments* seg, lora_bf16* y, int64_t ldy, void* workspace, size_t workspace_bytes,
                      int32_t* err_flag, lora_stream_t stream) {
  lora_status s = check_seg(seg, n_adapters);
  if (s != LORA_OK) return s;
  if (!rank_ok(r)) return LORA_ERR_UNSUPPORTED;
  if (seg->n_tokens == 0) return LORA_OK;
  s = check_proj(x, ldx, A_pool, B_pool, y, ldy, h_in, h_out, true, true);
  if (s != LORA_OK) return s;
  if (!W) return LORA_ERR_INVALID_ARG;
  if (!al16(W)) return LORA_ERR_MISALIGNED;
  if (!workspace || workspace_bytes < gemm_lora_workspace_bytes(seg->n_tokens, r)) return LORA_ERR_WORKSPACE;
  if (!al16(workspace)) return LORA_ERR_MISALIGNED;
  GemmLoraCall c{};
  c.x = x;
  c.ldx = ldx;
  c.W = W;
  c.A_pool = A_pool;
  c.B_pool = B_pool;
  c.n_adapters = n_adapters;
  c.h_in = h_in;
  c.h_out = h_out;
  c.r = r;
  c.scale = scale;
  c.seg = *seg;
  c.y = y;
  c.ldy = ldy;
  c.v = static_cast<float*>(workspace);
  c.err_flag = err_flag;
  return launch_gemm_lora(c, reinterpret_cast<cudaStream_t>(stream));
}

lora_status sgmv_fused(const lora_bf16* x, int64_t ldx, const lora_bf16* A_pool, const lora_bf16* B_pool,
                       int32_t n_adapters, int32_t h_in, int32_t h_out, int32_t r, float scale,
                       const lora_segments* seg, lora_bf16* y, int64_t ldy, int32_t* err_flag,
                       lora_stream_t stream) {
  lora_proj q{x, A_pool, B_pool, y, ldx, ldy, h_in, h_out, scale};
  return sgmv_multi(&q, 1, n_adapters, r, seg, err_flag, stream);
}

}  // extern "C"
