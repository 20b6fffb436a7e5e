// routing.cuh -- routing building blocks shared by the prefill routing
// kernel (route.cu) and the decode GEMVs (decode.cu): the order-preserving
// logit key, the block scan, one token's top-k with renormalised gates, and
// the whole routing of up to 8 tokens inside one CTA's shared memory.
//
// Routing (page "Lily Beats MLX-LM 1.35x on Decode: Perplexity's Rust+Metal
// Engine for Apple Silicon", sections "Model structure and three workload
// shapes" and "Prefill: fusing dequantisation and keeping routing
// GPU-resident"): per token the k experts with the largest logits (ties to
// the lower id), gates = softmax over the kept logits; per expert the count
// of (token, slot) pairs, the exclusive prefix scan of the counts, the pairs
// scattered into expert-contiguous rows (stable by pair index t*k + j) and
// the block map of tiles of at most BM rows per expert.
#pragma once
#include "common.cuh"

namespace lily {

constexpr int kMaxE = 256, kMaxK = 8;

// Order-preserving key of a logit: larger key = ranks first.  -0 and +0 map
// to the same key; a NaN maps to 0, below every number.
__device__ __forceinline__ uint32_t logit_key(float v) {
  if (v != v) return 0u;
  uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

// Exclusive scan of one int per thread over 256 threads: the whole block, or
// with NAMED the first 256 threads of a larger block (named barrier 1).
template <bool NAMED = false>
__device__ int block_exclusive_scan(int v, int* tmp /* [8] */) {
  auto sync = [] {
    if (NAMED)
      named_sync(1, kRouteThreads);
    else
      __syncthreads();
  };
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) tmp[warp] = incl;
  sync();
  if (warp == 0) {
    int w = (lane < kRouteThreads / 32) ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    if (lane < kRouteThreads / 32) tmp[lane] = w;  // inclusive warp totals
  }
  sync();
  int base = (warp > 0) ? tmp[warp - 1] : 0;
  int out = base + incl - v;
  sync();
  return out;
}

// Top-k of one token by one warp: lane l holds the logits of experts
// l + 32c in lv[c] (c < E/32 rounded up).  On return lane j < k holds the
// j-th expert (by logit desc, id asc) and its gate.  Returns whether a logit
// of the token was NaN.
__device__ __forceinline__ bool warp_topk(const float (&lv)[kMaxE / 32], int E, int k, int& my_id,
                                          float& my_gate) {
  const int lane = threadIdx.x & 31;
  uint32_t key[kMaxE / 32];
  uint32_t avail = 0;
  bool saw_nan = false;
#pragma unroll
  for (int c = 0; c < kMaxE / 32; ++c) {
    const int e = lane + 32 * c;
    key[c] = 0;
    if (e < E) {
      saw_nan |= (lv[c] != lv[c]);
      key[c] = logit_key(lv[c]);
      avail |= 1u << c;
    }
  }
  float my_logit = 0.f;
  my_id = 0;
  for (int j = 0; j < k; ++j) {
    // lane-local best: largest key, lowest id on ties (c ascending = id ascending)
    uint32_t bk = 0;
    int bc = -1;
#pragma unroll
    for (int c = 0; c < kMaxE / 32; ++c)
      if ((avail >> c) & 1u)
        if (bc < 0 || key[c] > bk) { bk = key[c]; bc = c; }
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bc >= 0 ? bk : 0u);
    const uint32_t cand = (bc >= 0 && bk == kmax) ? (uint32_t)(lane + 32 * bc) : 0xFFFFFFFFu;
    const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
    if ((int)(win & 31u) == lane) avail &= ~(1u << (win >> 5));
    if (lane == j) { my_logit = key_logit(kmax); my_id = (int)win; }
  }
  // gates: softmax over the kept logits; entries equal to the largest weigh 1
  const float lmax = __shfl_sync(0xffffffffu, my_logit, 0);
  float wgt = 0.f;
  if (lane < k) wgt = (my_logit == lmax) ? 1.f : expf(my_logit - lmax);
  float z = wgt;
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  my_gate = lane < k ? wgt / z : 0.f;
  return __any_sync(0xffffffffu, saw_nan);
}

// warp_topk for NT tokens at once (lv[i] the logits of token i, as above):
// the same selection, with the NT tokens' rounds interleaved so that their
// reduction latencies overlap.  Returns a bit mask of the tokens with a NaN
// logit.
template <int NT>
__device__ __forceinline__ uint32_t warp_topk_multi(const float (&lv)[NT][kMaxE / 32], int E,
                                                    int k, int (&my_id)[NT],
                                                    float (&my_gate)[NT]) {
  const int lane = threadIdx.x & 31;
  uint32_t key[NT][kMaxE / 32];
  uint32_t avail[NT];
  uint32_t nan_mask = 0;
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    avail[i] = 0;
    bool saw_nan = false;
#pragma unroll
    for (int c = 0; c < kMaxE / 32; ++c) {
      const int e = lane + 32 * c;
      key[i][c] = 0;
      if (e < E) {
        saw_nan |= (lv[i][c] != lv[i][c]);
        key[i][c] = logit_key(lv[i][c]);
        avail[i] |= 1u << c;
      }
    }
    if (__any_sync(0xffffffffu, saw_nan)) nan_mask |= 1u << i;
  }
  float my_logit[NT];
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    my_logit[i] = 0.f;
    my_id[i] = 0;
  }
  for (int j = 0; j < k; ++j) {
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      // lane-local best: largest key, lowest id on ties (c ascending = id ascending)
      uint32_t bk = 0;
      int bc = -1;
#pragma unroll
      for (int c = 0; c < kMaxE / 32; ++c)
        if ((avail[i] >> c) & 1u)
          if (bc < 0 || key[i][c] > bk) {
            bk = key[i][c];
            bc = c;
          }
      const uint32_t kmax = __reduce_max_sync(0xffffffffu, bc >= 0 ? bk : 0u);
      const uint32_t cand = (bc >= 0 && bk == kmax) ? (uint32_t)(lane + 32 * bc) : 0xFFFFFFFFu;
      const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
      if ((int)(win & 31u) == lane) avail[i] &= ~(1u << (win >> 5));
      if (lane == j) {
        my_logit[i] = key_logit(kmax);
        my_id[i] = (int)win;
      }
    }
  }
  // gates: softmax over the kept logits; entries equal to the largest weigh 1
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    const float lmax = __shfl_sync(0xffffffffu, my_logit[i], 0);
    float wgt = 0.f;
    if (lane < k) wgt = (my_logit[i] == lmax) ? 1.f : expf(my_logit[i] - lmax);
    float z = wgt;
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    my_gate[i] = lane < k ? wgt / z : 0.f;
  }
  return nan_mask;
}

// ------------------------------------------------------------- small T
// One tile slot of a decode step: slot 0 is the shared expert (all T rows,
// weight 1), slot i >= 1 is block-map tile i-1.  row0 is the slot's first row
// in the expert-sorted order of the rows (the shared rows follow the P
// routed ones); tok / gate give each row's token and gate.
constexpr int kSlotRows = 8;
struct DecSlot {
  int expert, row0, rows, pad;
  int tok[kSlotRows];
  float gate[kSlotRows];
};
constexpr int kMaxSlots = 1 + kSlotRows * kMaxK;  // T <= 8: P <= 64 routed tiles
// Decode plan in global memory: the slot count, padded to 16 bytes, then the
// slots (every DecSlot is 80 bytes, five 16-byte words).
struct DecPlan {
  int nslots, pad[3];
  DecSlot slot[kMaxSlots];
};
static_assert(sizeof(DecSlot) == 80 && sizeof(DecPlan) % 16 == 0, "plan layout");

// Routing of T <= 8 tokens by the first kRouteThreads threads of a CTA, from
// the logits `lg` ([T][E], shared memory): the slots of the step into
// `slots` / *nslots and, when `out` is given, the routing outputs (ids,
// gates, counts, offsets, perm, inv, block map, n_tiles) to global memory.
// With T <= 8 <= BM every touched expert is exactly one tile, so everything
// follows from counting over the P = T*k <= 64 pairs: pair p's row is
// #{q : e_q < e_p} + #{q < p : e_q == e_p} (stable by pair index), the first
// pair of an expert leads it, and its slot is 1 + the number of leaders of
// smaller experts.  Synchronises on named barrier 1 only (three times).
// BM (tile rows) is at least 16 > T, so it does not enter.
__device__ __forceinline__ void small_routing(const float* lg, int T, int E, int k, int BM,
                                              DecSlot* slots, int* nslots, const RouteArgs* out,
                                              uint32_t* status) {
  __shared__ int s_e[kSlotRows * kMaxK];      // expert of pair p = t * k + j
  __shared__ float s_g[kSlotRows * kMaxK];    // its gate
  __shared__ int s_perm[kSlotRows * kMaxK];   // pair at sorted position
  __shared__ int s_lead[kSlotRows * kMaxK];   // 1 if pair p leads its expert
  const int P = T * k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < T) {
    const int t = warp;
    float lv[kMaxE / 32];
#pragma unroll
    for (int c = 0; c < kMaxE / 32; ++c) {
      const int e = lane + 32 * c;
      lv[c] = e < E ? lg[(size_t)t * E + e] : 0.f;
    }
    int my_id;
    float my_gate;
    const bool nan = warp_topk(lv, E, k, my_id, my_gate);
    if (nan && lane == 0) set_status(status, LILY_STATUS_NAN_LOGIT);
    if (lane < k) {
      s_e[t * k + lane] = my_id;
      s_g[t * k + lane] = my_gate;
      if (out) {
        out->ids[(size_t)t * k + lane] = my_id;
        out->gates[(size_t)t * k + lane] = my_gate;
      }
    }
  }
  named_sync(1, kRouteThreads);
  // pair p: its row, whether it leads its expert (no earlier pair of it),
  // and its expert's count
  int p_pos = 0, p_cnt = 0;
  const int p = threadIdx.x;
  if (p < P) {
    const int e = s_e[p];
    int below = 0, before = 0, cnt = 0;
    for (int q = 0; q < P; ++q) {
      const int eq = s_e[q];
      below += eq < e;
      before += (eq == e) & (q < p);
      cnt += eq == e;
    }
    p_pos = below + before;
    p_cnt = cnt;
    s_perm[p_pos] = p;
    s_lead[p] = before == 0;
    if (out) {
      out->perm[p_pos] = p;
      out->inv[p] = p_pos;
    }
  }
  // counts and offsets of every expert
  if (out && threadIdx.x < E) {
    const int e = threadIdx.x;
    int cnt = 0, off = 0;
    for (int q = 0; q < P; ++q) {
      cnt += s_e[q] == e;
      off += s_e[q] < e;
    }
    out->counts[e] = cnt;
    out->offsets[e] = off;
    if (e == 0) out->offsets[E] = P;
  }
  named_sync(1, kRouteThreads);
  // the leader of each expert writes its slot (and block-map tile): slot 1 +
  // the number of leaders of smaller experts
  int nlead = 0;
  for (int q = 0; q < P; ++q) nlead += s_lead[q];
  if (p < P && s_lead[p]) {
    int leaders_below = 0;
    for (int q = 0; q < P; ++q) leaders_below += (s_e[q] < s_e[p]) & s_lead[q];
    const int p_slot = 1 + leaders_below;
    DecSlot& sl = slots[p_slot];
    const int row0 = p_pos;  // a leader is its expert's first row
    const int rows = min(p_cnt, kSlotRows);
    sl.expert = s_e[p];
    sl.row0 = row0;
    sl.rows = rows;
    for (int n = 0; n < kSlotRows; ++n) {
      const int pp = n < rows ? s_perm[row0 + n] : 0;
      sl.tok[n] = n < rows ? pp / k : 0;
      sl.gate[n] = n < rows ? s_g[pp] : 0.f;
    }
    if (out) {
      out->block_map[2 * (p_slot - 1)] = s_e[p];
      out->block_map[2 * (p_slot - 1) + 1] = row0;
    }
  }
  if (threadIdx.x == 0) {
    *nslots = 1 + nlead;
    DecSlot& sl = slots[0];
    sl.expert = E;
    sl.row0 = P;
    sl.rows = T;
    for (int n = 0; n < kSlotRows; ++n) {
      sl.tok[n] = n < T ? n : 0;
      sl.gate[n] = n < T ? 1.f : 0.f;
    }
    if (out) *out->n_tiles = nlead;
  }
  if (out)
    for (int i = nlead + threadIdx.x; i < out->cap; i += kRouteThreads) {
      out->block_map[2 * i] = -1;
      out->block_map[2 * i + 1] = -1;
    }
  named_sync(1, kRouteThreads);
}

}  // namespace lily
