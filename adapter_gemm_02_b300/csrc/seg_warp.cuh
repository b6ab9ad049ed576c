// Segmentation of a small batch by one warp, in shared memory, inside the
// SGMV launch (the one-launch step: segmentation and SGMV together).
//
// Punica: Multi-Tenant LoRA Serving (research.elamur.ai summary),
// "Interesting ideas" I2: the batch is sorted by adapter so that same-adapter
// tokens form segments.  The result is the one lora_segment computes: a
// stable counting sort of the token indices by adapter id, segments of the
// non-empty adapters in ascending id, ids outside [0, P) after every valid
// token and in no segment.
#pragma once

#include <cstdint>

namespace lsg {

__device__ __forceinline__ int seg_warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += o;
  }
  return v;
}

struct WarpSegOut {
  int S;        // segments
  int n_valid;  // tokens with a valid id
  bool bad;     // (lane-local) an invalid id was seen by this lane
};

// ids[0..n) (global) -> ids_s[n], cnt[P+1] (scratch: per-key cursors),
// perm_s[n], offs_s[S+1], adap_s[S] (shared memory).  Executed by a full warp.
__device__ inline WarpSegOut warp_segment(const int32_t* ids, int n, int P, int32_t* ids_s, int32_t* cnt,
                                          int32_t* perm_s, int32_t* offs_s, int32_t* adap_s, int lane) {
  WarpSegOut o{0, 0, false};
  for (int i = lane; i < n; i += 32) ids_s[i] = ids[i];
  for (int a = lane; a <= P; a += 32) cnt[a] = 0;
  __syncwarp();
  // histogram: equal keys of a 32-token group are counted by their leader
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    const bool act = i < n;
    const unsigned am = __ballot_sync(0xffffffffu, act);
    if (act) {
      const int id = ids_s[i];
      const int key = (id >= 0 && id < P) ? id : P;
      o.bad |= key == P;
      const unsigned peers = __match_any_sync(am, key);
      if (lane == __ffs(peers) - 1) cnt[key] += __popc(peers);
    }
    __syncwarp();
  }
  // exclusive scan over the keys (segment starts) and compaction of the
  // non-empty adapters: lane l owns the contiguous keys [l*per, (l+1)*per)
  const int per = (P + 1 + 31) / 32;
  const int k0 = min(P + 1, lane * per), k1 = min(P + 1, k0 + per);
  int tot = 0, ne = 0;
  for (int a = k0; a < k1; ++a) {
    const int c = cnt[a];
    tot += c;
    ne += (a < P && c > 0);
  }
  const int tot_incl = seg_warp_incl_scan(tot, lane), ne_incl = seg_warp_incl_scan(ne, lane);
  int run = tot_incl - tot, idx = ne_incl - ne;
  for (int a = k0; a < k1; ++a) {
    const int c = cnt[a];
    cnt[a] = run;
    if (a < P && c > 0) {
      adap_s[idx] = a;
      offs_s[idx] = run;
      ++idx;
    }
    run += c;
  }
  const int S = __shfl_sync(0xffffffffu, ne_incl, 31);
  __syncwarp();
  o.S = S;
  o.n_valid = cnt[P];
  if (lane == 0) offs_s[S] = o.n_valid;
  // stable scatter: groups in token order, equal keys ranked by lane
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    const bool act = i < n;
    const unsigned am = __ballot_sync(0xffffffffu, act);
    if (act) {
      const int id = ids_s[i];
      const int key = (id >= 0 && id < P) ? id : P;
      const unsigned peers = __match_any_sync(am, key);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int b = cnt[key];
      perm_s[b + rank] = i;
      __syncwarp(am);
      if (lane == __ffs(peers) - 1) cnt[key] = b + __popc(peers);
    }
    __syncwarp();
  }
  return o;
}

// The same result for n <= 32*E tokens (E <= 2) without shared-memory
// scratch: lane l holds tokens l and l+32 in registers, and each token's
// place in the stable order is the number of tokens that sort before it
// (a smaller id, or the same id and a smaller index), counted by comparing it
// with every token through warp shuffles.  The first token of each valid id
// starts a segment; a segment's index is the number of segment-starting
// tokens with a smaller id.  Ids outside [0, P) sort as P (after every valid
// token, in token order).  perm_s[n], offs_s[S+1], adap_s[S] in shared memory.
// idv[e]: the id of token e*32 + lane, already loaded by the caller.
template <int E>
__device__ __forceinline__ WarpSegOut warp_segment_rank(const int (&idv)[2], int n, int P, int32_t* perm_s,
                                                        int32_t* offs_s, int32_t* adap_s, int lane) {
  constexpr int kPad = 0x7fffffff;  // lanes past n: after every token
  int key[E];
  bool bad = false;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = e * 32 + lane;
    key[e] = kPad;
    if (i < n) {
      const int id = idv[e];
      const bool ok = id >= 0 && id < P;
      key[e] = ok ? id : P;
      bad |= !ok;
    }
  }
  int before[E], same_before[E];
#pragma unroll
  for (int e = 0; e < E; ++e) before[e] = same_before[e] = 0;
#pragma unroll
  for (int f = 0; f < E; ++f) {
#pragma unroll 8
    for (int src = 0; src < 32; ++src) {
      const int kj = __shfl_sync(0xffffffffu, key[f], src);
      const int j = f * 32 + src;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        before[e] += kj < key[e];
        same_before[e] += (kj == key[e]) & (j < e * 32 + lane);
      }
    }
  }
  int S = 0, n_valid = 0;
  unsigned lead[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    lead[e] = __ballot_sync(0xffffffffu, key[e] < P && same_before[e] == 0);
    S += __popc(lead[e]);
    n_valid += __popc(__ballot_sync(0xffffffffu, key[e] < P));
  }
  int seg[E];
#pragma unroll
  for (int e = 0; e < E; ++e) seg[e] = 0;
#pragma unroll
  for (int f = 0; f < E; ++f) {
#pragma unroll 8
    for (int src = 0; src < 32; ++src) {
      const int kj = __shfl_sync(0xffffffffu, key[f], src);
      const int lj = (lead[f] >> src) & 1;
#pragma unroll
      for (int e = 0; e < E; ++e) seg[e] += lj & (kj < key[e]);
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = e * 32 + lane;
    if (i < n) perm_s[before[e] + same_before[e]] = i;
    if (key[e] < P && same_before[e] == 0) {
      adap_s[seg[e]] = key[e];
      offs_s[seg[e]] = before[e];
    }
  }
  if (lane == 0) offs_s[S] = n_valid;
  __syncwarp();
  return WarpSegOut{S, n_valid, bad};
}

}  // namespace lsg
