/*
 * Plain CPU oracle for multi-LoRA SGMV.  TEST INFRASTRUCTURE ONLY: it is used
 * by the tests, by the package's smoke check and by the benchmark's CPU
 * baseline.  The product path never links, loads or calls it.
 *
 * What it computes (Punica: Serving Multiple LoRA Finetuned LLM as One,
 * "How It Works": a LoRA finetune adds two small matrices A and B to a weight
 * W; Punica: Multi-Tenant LoRA Serving, "Summary": the per-adapter low-rank
 * additions are computed together for a batch of requests with mixed
 * adapters, requests of the same adapter grouped; "Interesting ideas" I2: the
 * batch is sorted by adapter so that same-adapter rows form segments):
 *
 *   segmentation:  stable sort of the token indices by adapter id
 *   delta:         y[i,:] = y0[i,:] + s * ((x[i,:] . A[a_i]) . B[a_i])
 *
 * Readings taken where the pages are silent:
 *  - the scale s multiplies the expanded product, after the B contraction;
 *  - the association is (x.A).B (shrink to rank r, then expand);
 *  - A[a] is [h_in][r] row-major, B[a] is [r][h_out] row-major, pools are
 *    contiguous slabs (adapter id = slab index); x is [n][ldx], y0 [n][ldy0];
 *  - v = x.A is kept in fp32, the result is returned unrounded (fp32 here,
 *    fp64 in the twin);
 *  - segments come in ascending adapter id, empty adapters have none, ties
 *    keep token order (stable);
 *  - an id outside [0, P) belongs to no segment; such tokens are listed after
 *    all valid ones, in token order, and their rows are left unchanged.
 *
 * Floating point: every operation is a separate IEEE fp32 (or fp64) operation
 * in the order written; build with -ffp-contract=off and without fast-math so
 * that no FMA contraction or reassociation changes the rounding.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Deliberate mistakes, compiled in only by the test that checks that the pins
 * catch them (ORACLE_MUTANT=k).  0 = the oracle as it stands. */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

int oracle_abi_version(void) { return 1; }
int oracle_mutant(void) { return ORACLE_MUTANT; }

/*
 * Segmentation by counting sort (histogram, exclusive scan, stable scatter).
 * Outputs: perm[n]; seg_offsets[max_segments+1]; seg_adapter[max_segments];
 * *num_segments.  Entries past the last segment are filled with n_valid
 * (offsets) and -1 (adapters).  Returns the number of invalid ids.
 */
int oracle_lora_segment(const int32_t* ids, int32_t n, int32_t P, int32_t max_segments,
                        int32_t* perm, int32_t* seg_offsets, int32_t* seg_adapter,
                        int32_t* num_segments) {
  /* bucket P collects invalid ids so that they land after every valid one */
  int64_t* cnt = (int64_t*)calloc((size_t)P + 1, sizeof(int64_t));
  int64_t* pos = (int64_t*)calloc((size_t)P + 1, sizeof(int64_t));
  int32_t n_invalid = 0;
  for (int32_t i = 0; i < n; ++i) {
    int32_t a = ids[i];
    int32_t key = (a >= 0 && a < P) ? a : P;
    if (key == P) ++n_invalid;
    cnt[key] += 1;
  }
  int64_t run = 0;
  for (int32_t a = 0; a <= P; ++a) {
    pos[a] = run;
    run += cnt[a];
  }
  int32_t S = 0;
  for (int32_t a = 0; a < P; ++a) {
#if ORACLE_MUTANT == 7 /* empty adapters kept as segments */
    if (S < max_segments) {
#else
    if (cnt[a] > 0) {
#endif
      seg_adapter[S] = a;
      seg_offsets[S] = (int32_t)pos[a];
      ++S;
    }
  }
  int32_t n_valid = n - n_invalid;
  seg_offsets[S] = n_valid;
  for (int32_t s = S + 1; s <= max_segments; ++s) seg_offsets[s] = n_valid;
  for (int32_t s = S; s < max_segments; ++s) seg_adapter[s] = -1;
  *num_segments = S;
#if ORACLE_MUTANT == 6 /* unstable: walk the tokens backwards */
  for (int32_t i = n - 1; i >= 0; --i) {
#else
  for (int32_t i = 0; i < n; ++i) {
#endif
    int32_t a = ids[i];
    int32_t key = (a >= 0 && a < P) ? a : P;
    perm[pos[key]++] = i;
  }
  free(cnt);
  free(pos);
  return n_invalid;
}

/*
 * One token of the fp32 oracle: v[k] = sum_j x[j]*A[j][k] (j ascending),
 * d[c] = sum_k v[k]*B[k][c] (k ascending), y[c] = y0[c] + s*d[c].
 */
static void token_f32(const uint16_t* xi, const uint16_t* A, const uint16_t* B,
                      const uint16_t* y0i, int32_t h_in, int32_t h_out, int32_t r,
                      float s, float* yi, float* vi, float* vtmp) {
  for (int32_t k = 0; k < r; ++k) {
    float acc = 0.0f;
#if ORACLE_MUTANT == 4 /* drops the last term of the h_in sum */
    for (int32_t j = 0; j < h_in - 1; ++j) {
#else
    for (int32_t j = 0; j < h_in; ++j) {
#endif
      float p = bf16_to_f32(xi[j]) * bf16_to_f32(A[(int64_t)j * r + k]);
      acc = acc + p;
    }
    vtmp[k] = acc;
  }
  for (int32_t c = 0; c < h_out; ++c) {
    float d = 0.0f;
    for (int32_t k = 0; k < r; ++k) {
#if ORACLE_MUTANT == 2 /* transposed B index */
      float p = vtmp[k] * bf16_to_f32(B[((int64_t)c * r + k) % ((int64_t)r * h_out)]);
#else
      float p = vtmp[k] * bf16_to_f32(B[(int64_t)k * h_out + c]);
#endif
      d = d + p;
    }
#if ORACLE_MUTANT == 1 /* scale dropped */
    float sd = d;
#elif ORACLE_MUTANT == 5 /* sign of the delta flipped */
    float sd = -(s * d);
#else
    float sd = s * d;
#endif
    yi[c] = bf16_to_f32(y0i[c]) + sd;
  }
  if (vi)
    for (int32_t k = 0; k < r; ++k) vi[k] = vtmp[k];
}

/* Same steps in fp64 (inputs widened exactly). */
static void token_f64(const uint16_t* xi, const uint16_t* A, const uint16_t* B,
                      const uint16_t* y0i, int32_t h_in, int32_t h_out, int32_t r,
                      double s, double* yi, double* vi, double* vtmp) {
  for (int32_t k = 0; k < r; ++k) {
    double acc = 0.0;
    for (int32_t j = 0; j < h_in; ++j)
      acc = acc + (double)bf16_to_f32(xi[j]) * (double)bf16_to_f32(A[(int64_t)j * r + k]);
    vtmp[k] = acc;
  }
  for (int32_t c = 0; c < h_out; ++c) {
    double d = 0.0;
    for (int32_t k = 0; k < r; ++k) d = d + vtmp[k] * (double)bf16_to_f32(B[(int64_t)k * h_out + c]);
    yi[c] = (double)bf16_to_f32(y0i[c]) + s * d;
  }
  if (vi)
    for (int32_t k = 0; k < r; ++k) vi[k] = vtmp[k];
}

static int adapter_of(const int32_t* ids, int32_t i, int32_t P) {
  int32_t a = ids[i];
#if ORACLE_MUTANT == 3 /* wrong adapter slab */
  a = (a >= 0 && a < P) ? (a + 1) % P : a;
#endif
  return a;
}

/*
 * Per-token fp32 oracle (no segments are used: the grouping changes only the
 * order of work, not the result).  x: [n][ldx] bf16 bits; A_pool: [P][h_in][r];
 * B_pool: [P][r][h_out]; y0: [n][ldy0]; y: [n][h_out] fp32; v: [n][r] fp32 or
 * NULL.  Tokens with an invalid id get y = y0 and v untouched.  Returns the
 * number of invalid ids.
 */
int oracle_sgmv_f32(const uint16_t* x, int64_t ldx, const uint16_t* A_pool, const uint16_t* B_pool,
                    const int32_t* ids, int32_t n, int32_t P, int32_t h_in, int32_t h_out, int32_t r,
                    float s, const uint16_t* y0, int64_t ldy0, float* y, float* v, int32_t n_threads) {
  int32_t n_invalid = 0;
  for (int32_t i = 0; i < n; ++i) n_invalid += !(ids[i] >= 0 && ids[i] < P);
  if (n_threads < 1) n_threads = 1;
#pragma omp parallel num_threads(n_threads)
  {
    float* vtmp = (float*)malloc(sizeof(float) * (size_t)(r > 0 ? r : 1));
#pragma omp for schedule(static)
    for (int32_t i = 0; i < n; ++i) {
      int32_t a = adapter_of(ids, i, P);
      float* yi = y + (int64_t)i * h_out;
      const uint16_t* y0i = y0 + (int64_t)i * ldy0;
      if (!(a >= 0 && a < P)) {
        for (int32_t c = 0; c < h_out; ++c) yi[c] = bf16_to_f32(y0i[c]);
        continue;
      }
      token_f32(x + (int64_t)i * ldx, A_pool + (int64_t)a * h_in * r, B_pool + (int64_t)a * r * h_out,
                y0i, h_in, h_out, r, s, yi, v ? v + (int64_t)i * r : NULL, vtmp);
    }
    free(vtmp);
  }
  return n_invalid;
}

/* fp64 twin of oracle_sgmv_f32 (same arguments, double outputs). */
int oracle_sgmv_f64(const uint16_t* x, int64_t ldx, const uint16_t* A_pool, const uint16_t* B_pool,
                    const int32_t* ids, int32_t n, int32_t P, int32_t h_in, int32_t h_out, int32_t r,
                    double s, const uint16_t* y0, int64_t ldy0, double* y, double* v, int32_t n_threads) {
  int32_t n_invalid = 0;
  for (int32_t i = 0; i < n; ++i) n_invalid += !(ids[i] >= 0 && ids[i] < P);
  if (n_threads < 1) n_threads = 1;
#pragma omp parallel num_threads(n_threads)
  {
    double* vtmp = (double*)malloc(sizeof(double) * (size_t)(r > 0 ? r : 1));
#pragma omp for schedule(static)
    for (int32_t i = 0; i < n; ++i) {
      int32_t a = ids[i];
      double* yi = y + (int64_t)i * h_out;
      const uint16_t* y0i = y0 + (int64_t)i * ldy0;
      if (!(a >= 0 && a < P)) {
        for (int32_t c = 0; c < h_out; ++c) yi[c] = (double)bf16_to_f32(y0i[c]);
        continue;
      }
      token_f64(x + (int64_t)i * ldx, A_pool + (int64_t)a * h_in * r, B_pool + (int64_t)a * r * h_out,
                y0i, h_in, h_out, r, s, yi, v ? v + (int64_t)i * r : NULL, vtmp);
    }
    free(vtmp);
  }
  return n_invalid;
}

/*
 * Slot arenas with adapters of mixed ranks (the pool layout of the slot-table
 * entry point).  Adapter a lives in slot slot_of[a] with rank rank_of[a]; its
 * A is [h_in][rank] row-major at A_arena + slot*h_in*r_max and its B is
 * [rank][h_out] row-major at B_arena + slot*r_max*h_out.  An entry is valid
 * when 0 <= a < P, 0 <= slot < n_slots, the rank is 8, 16, 32 or 64, is at
 * most r_max and has its bit (rank 8 << c: bit c) in rank_mask.  Each valid
 * token takes the same steps as oracle_sgmv_f32 with its adapter's rank;
 * any other token gets y = y0.  Returns the number of tokens that are not
 * valid.
 */
static int slot_rank_valid(int32_t rk, int32_t r_max, uint32_t rank_mask) {
  int32_t c = rk == 8 ? 0 : rk == 16 ? 1 : rk == 32 ? 2 : rk == 64 ? 3 : -1;
  return c >= 0 && rk <= r_max && ((rank_mask >> c) & 1u);
}

int oracle_sgmv_slots_f32(const uint16_t* x, int64_t ldx, const uint16_t* A_arena, const uint16_t* B_arena,
                          const int32_t* slot_of, const int32_t* rank_of, int32_t n_slots, int32_t r_max,
                          uint32_t rank_mask, const int32_t* ids, int32_t n, int32_t P, int32_t h_in,
                          int32_t h_out, float s, const uint16_t* y0, int64_t ldy0, float* y, int32_t n_threads) {
  int32_t n_invalid = 0;
  if (n_threads < 1) n_threads = 1;
#pragma omp parallel num_threads(n_threads) reduction(+ : n_invalid)
  {
    float* vtmp = (float*)malloc(sizeof(float) * (size_t)(r_max > 0 ? r_max : 1));
#pragma omp for schedule(static)
    for (int32_t i = 0; i < n; ++i) {
      int32_t a = ids[i];
      float* yi = y + (int64_t)i * h_out;
      const uint16_t* y0i = y0 + (int64_t)i * ldy0;
      int ok = a >= 0 && a < P;
      int32_t sl = ok ? slot_of[a] : -1, rk = ok ? rank_of[a] : 0;
      ok = ok && sl >= 0 && sl < n_slots && slot_rank_valid(rk, r_max, rank_mask);
      if (!ok) {
        n_invalid += 1;
        for (int32_t c = 0; c < h_out; ++c) yi[c] = bf16_to_f32(y0i[c]);
        continue;
      }
#if ORACLE_MUTANT == 8 /* slot stride taken from the adapter's rank instead of the slot capacity */
      const uint16_t* A = A_arena + (int64_t)sl * h_in * rk;
      const uint16_t* B = B_arena + (int64_t)sl * rk * h_out;
#else
      const uint16_t* A = A_arena + (int64_t)sl * h_in * r_max;
      const uint16_t* B = B_arena + (int64_t)sl * r_max * h_out;
#endif
#if ORACLE_MUTANT == 9 /* every adapter read at the slot capacity's rank */
      rk = r_max;
#endif
      token_f32(x + (int64_t)i * ldx, A, B, y0i, h_in, h_out, rk, s, yi, NULL, vtmp);
    }
    free(vtmp);
  }
  return n_invalid;
}

/*
 * The backbone projection with its LoRA delta, as a GEMM epilogue would
 * produce it (Punica: Multi-Tenant LoRA Serving, "Summary": the backbone runs
 * as one GEMM and the per-adapter low-rank additions are computed beside it):
 *
 *   y[i,:] = x[i,:] . W + s * ((x[i,:] . A[a_i]) . B[a_i])
 *
 * W is [h_in][h_out] row-major.  Per token: base[c] = sum_j x[j]*W[j][c]
 * (j ascending, fp32), the delta d[c] with the same steps as
 * oracle_sgmv_f32, y[c] = base[c] + s*d[c] (unrounded fp32).  A token whose
 * id is outside [0, P) gets y = base.  Returns the number of such tokens.
 */
int oracle_gemm_lora_f32(const uint16_t* x, int64_t ldx, const uint16_t* W, const uint16_t* A_pool,
                         const uint16_t* B_pool, const int32_t* ids, int32_t n, int32_t P, int32_t h_in,
                         int32_t h_out, int32_t r, float s, float* y, int32_t n_threads) {
  int32_t n_invalid = 0;
  if (n_threads < 1) n_threads = 1;
#pragma omp parallel num_threads(n_threads) reduction(+ : n_invalid)
  {
    float* v = (float*)malloc(sizeof(float) * (size_t)(r > 0 ? r : 1));
#pragma omp for schedule(static)
    for (int32_t i = 0; i < n; ++i) {
      const uint16_t* xi = x + (int64_t)i * ldx;
      float* yi = y + (int64_t)i * h_out;
      const int32_t a = ids[i];
      const int ok = a >= 0 && a < P;
      n_invalid += !ok;
      const uint16_t* A = ok ? A_pool + (int64_t)a * h_in * r : NULL;
      const uint16_t* B = ok ? B_pool + (int64_t)a * r * h_out : NULL;
      if (ok)
        for (int32_t k = 0; k < r; ++k) {
          float acc = 0.0f;
          for (int32_t j = 0; j < h_in; ++j) acc = acc + bf16_to_f32(xi[j]) * bf16_to_f32(A[(int64_t)j * r + k]);
          v[k] = acc;
        }
      for (int32_t c = 0; c < h_out; ++c) {
        float base = 0.0f;
        for (int32_t j = 0; j < h_in; ++j) {
#if ORACLE_MUTANT == 10 /* W indexed transposed */
          const float w = bf16_to_f32(W[((int64_t)c * h_in + j) % ((int64_t)h_in * h_out)]);
#else
          const float w = bf16_to_f32(W[(int64_t)j * h_out + c]);
#endif
          base = base + bf16_to_f32(xi[j]) * w;
        }
        if (ok) {
          float d = 0.0f;
          for (int32_t k = 0; k < r; ++k) d = d + v[k] * bf16_to_f32(B[(int64_t)k * h_out + c]);
          yi[c] = base + s * d;
        } else {
          yi[c] = base;
        }
      }
    }
    free(v);
  }
  return n_invalid;
}
