// lily_oracle.cpp -- plain, slow, single-threaded FP64 CPU oracle for the
// W4 MoE expert layer.
//
// TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
// load this file: only the test suite, the smoke check and the benchmark's
// CPU-baseline leg use it.  It shares no code, header, table or constant with
// the CUDA library; the two meet only through the seeded input tensors.
//
// Sources (pages about Perplexity's Lily engine):
//   [MS]  "Lily Beats MLX-LM 1.35x on Decode: Perplexity's Rust+Metal Engine
//          for Apple Silicon", section "Model structure and three workload shapes"
//   [PF]  same page, section "Prefill: fusing dequantisation and keeping
//          routing GPU-resident"
//   [UQ]  "Revolutionizing Local AI Inference on Apple Silicon", section
//          "Understanding the Qwen3.6-35B-A3B Model"
//
// What it computes (the plain definition; every value in double):
//   logits   L[t][e] = sum_i x[t][i] * Wr[e][i] + b_r[e]          ([MS], [UQ]:
//            "a router scores 256 experts")
//   top-k    per token, experts ranked by (logit desc, id asc), first k kept;
//            gates g_j = exp(L_j - L_max) / sum_sel exp(L_i - L_max), i.e. the
//            full softmax renormalised over the kept k
//   routing  histogram -> exclusive prefix scan -> stable scatter -> block
//            map ([PF]: "routing histogram, prefix scan, scatter, and block map")
//   dequant  w = scale * q + bias, every 64 consecutive input-dim weights share
//            one bf16 scale and one bf16 bias ([MS]: "groupwise affine 4-bit")
//   expert   SwiGLU FFN: h = silu(Wg x) * (Wu x),  o = Wd h
//   layer    y[t] = sum_j g[t][j] * FFN_{ids[t][j]}(x[t]) + FFN_shared(x[t])
//            ([MS]: the shared expert "processes every token regardless of
//            routing"; it carries weight 1)
//
// Readings where the pages are silent (each listed in the design notes):
//   * nibble order: byte j of a weight row holds element 2j in bits 0-3 and
//     element 2j+1 in bits 4-7; rows are output features, groups run along
//     the input dimension.
//   * ties in top-k go to the lower expert id; -0.0 equals +0.0; a NaN logit
//     ranks below every number and is counted (the GPU sets an error flag).
//   * selected logits equal to the largest selected logit weigh exactly 1 in
//     the gate softmax, so an all -inf or a +inf selection stays defined.
//   * within an expert group, pairs keep ascending pair index t*k + j.
//   * block map: for e ascending, tiles of at most BM rows; unused entries -1.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <algorithm>

namespace {

// bf16 is the top half of an IEEE binary32; widening is exact.
double bf16_to_double(uint16_t h) {
  uint32_t bits = (uint32_t)h << 16;
  float f;
  std::memcpy(&f, &bits, sizeof f);
  return (double)f;
}

// The 4-bit code of element c in a packed row (low nibble = even element).
int nibble(const uint8_t* row, int c) {
  uint8_t byte = row[c / 2];
  return (c % 2 == 0) ? (byte & 0xF) : (byte >> 4);
}

// "a ranks before b" for (logit desc, id asc); NaN ranks last.
bool ranks_before(float la, int ia, float lb, int ib) {
  bool na = std::isnan(la), nb = std::isnan(lb);
  if (na != nb) return nb;          // the number ranks before the NaN
  if (!na && la != lb) return la > lb;
  return ia < ib;                   // equal (incl. -0 == +0) or both NaN
}

double silu(double v) { return v / (1.0 + std::exp(-v)); }

}  // namespace

extern "C" {

// Explicit dequantisation of one packed matrix: R rows (output features) by
// C input-dim elements.  q is [R][C/2] bytes, s and b are [R][C/64] bf16.
// w[r][c] = s[r][c/64] * q[r][c] + b[r][c/64].
int orc_dequant(int R, int C, const uint8_t* q, const uint16_t* s,
                const uint16_t* b, double* w) {
  if (R < 0 || C <= 0 || C % 64 != 0) return -1;
  const int G = C / 64;
  for (int r = 0; r < R; ++r) {
    const uint8_t* qrow = q + (size_t)r * (C / 2);
    for (int c = 0; c < C; ++c) {
      double scale = bf16_to_double(s[(size_t)r * G + c / 64]);
      double bias = bf16_to_double(b[(size_t)r * G + c / 64]);
      w[(size_t)r * C + c] = scale * (double)nibble(qrow, c) + bias;
    }
  }
  return 0;
}

// Router logits in double: L[t][e] = sum_i x[t][i] * Wr[e][i] (+ b_r[e]).
// Also returns A[t][e] = sum_i |x[t][i] * Wr[e][i]|, the scale of the
// rounding error any fp32 evaluation of the same sum may carry.
int orc_router_logits(int T, int d, int E, const uint16_t* x, const float* wr,
                      const float* br, double* logits, double* abs_sum) {
  if (T < 0 || d <= 0 || E <= 0) return -1;
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      double acc = 0.0, mag = 0.0;
      for (int i = 0; i < d; ++i) {
        double p = bf16_to_double(x[(size_t)t * d + i]) * (double)wr[(size_t)e * d + i];
        acc += p;
        mag += std::fabs(p);
      }
      if (br) acc += (double)br[e];
      logits[(size_t)t * E + e] = acc;
      if (abs_sum) abs_sum[(size_t)t * E + e] = mag;
    }
  }
  return 0;
}

// Size of the block map: ceil(P/BM) + min(E, P) entries of (expert, row_begin).
int orc_block_map_cap(int T, int E, int k, int BM) {
  long P = (long)T * k;
  return (int)((P + BM - 1) / BM + std::min<long>(E, P));
}

// Routing from given fp32 logits [T][E].
//   ids[T][k], gates[T][k] (double), counts[E], offsets[E+1], perm[P], inv[P],
//   block_map[cap][2] (expert, row_begin; -1 past n_tiles), *n_tiles, *n_nan.
int orc_route(int T, int E, int k, int BM, const float* logits, int32_t* ids,
              double* gates, int32_t* counts, int32_t* offsets, int32_t* perm,
              int32_t* inv, int32_t* block_map, int cap, int32_t* n_tiles,
              int32_t* n_nan) {
  if (T < 0 || E <= 0 || k <= 0 || k > E || BM <= 0) return -1;
  if (cap < orc_block_map_cap(T, E, k, BM)) return -2;
  const int P = T * k;
  int nan_count = 0;

  // Top-k selection per token: k passes, each taking the best unused expert.
  std::vector<char> used(E);
  for (int t = 0; t < T; ++t) {
    const float* L = logits + (size_t)t * E;
    for (int e = 0; e < E; ++e) nan_count += std::isnan(L[e]) ? 1 : 0;
    std::fill(used.begin(), used.end(), 0);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (used[e]) continue;
        if (best < 0 || ranks_before(L[e], e, L[best], best)) best = e;
      }
      used[best] = 1;
      ids[t * k + j] = best;
    }
    // Gates: softmax over the selected logits, shifted by the largest one.
    double lmax = (double)L[ids[t * k]];
    std::vector<double> w(k);
    double z = 0.0;
    for (int j = 0; j < k; ++j) {
      double l = (double)L[ids[t * k + j]];
      w[j] = (l == lmax) ? 1.0 : std::exp(l - lmax);
      z += w[j];
    }
    for (int j = 0; j < k; ++j) gates[t * k + j] = w[j] / z;
  }

  // Histogram: counts[e] = number of (token, slot) pairs routed to e.
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int p = 0; p < P; ++p) counts[ids[p]] += 1;

  // Exclusive prefix scan; offsets[E] = P.
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];

  // Stable scatter: pairs visited in ascending pair index.
  std::vector<int32_t> next(offsets, offsets + E);
  for (int p = 0; p < P; ++p) {
    int pos = next[ids[p]]++;
    perm[pos] = p;
    inv[p] = pos;
  }

  // Block map: for each expert in ascending id, ceil(count/BM) tiles.
  int nt = 0;
  for (int e = 0; e < E; ++e) {
    for (int r = offsets[e]; r < offsets[e + 1]; r += BM) {
      block_map[2 * nt + 0] = e;
      block_map[2 * nt + 1] = r;
      ++nt;
    }
  }
  for (int i = nt; i < cap; ++i) {
    block_map[2 * i + 0] = -1;
    block_map[2 * i + 1] = -1;
  }
  *n_tiles = nt;
  if (n_nan) *n_nan = nan_count;
  return 0;
}

// One expert's SwiGLU FFN on one row, all matrices already dequantised:
// Wg, Wu are [F][d], Wd is [d][F]; out[d] = Wd (silu(Wg x) * (Wu x)).
static void ffn_row(int d, int F, const double* Wg, const double* Wu,
                    const double* Wd, const double* x, double* h, double* out) {
  for (int f = 0; f < F; ++f) {
    double g = 0.0, u = 0.0;
    for (int i = 0; i < d; ++i) {
      g += Wg[(size_t)f * d + i] * x[i];
      u += Wu[(size_t)f * d + i] * x[i];
    }
    h[f] = silu(g) * u;
  }
  for (int o = 0; o < d; ++o) {
    double acc = 0.0;
    for (int f = 0; f < F; ++f) acc += Wd[(size_t)o * F + f] * h[f];
    out[o] = acc;
  }
}

// MoE layer output for a subset of tokens.
//   x[T][d] bf16; packed weights of E+1 experts (index E = shared expert):
//   gq,uq [E+1][F][d/2], gs,gb,us,ub [E+1][F][d/64],
//   dq [E+1][d][F/2], ds,db [E+1][d][F/64];
//   ids[T][k] and gates[T][k] from orc_route;
//   rows[nrows] token indices; y[nrows][d] receives
//   y = sum_j gates[t][j] * FFN_{ids[t][j]}(x[t]) + FFN_E(x[t]).
// Each needed expert is dequantised once (explicitly, into double) and then
// applied to every selected row that uses it.
int orc_moe_rows(int T, int d, int E, int k, int F, const uint16_t* x,
                 const uint8_t* gq, const uint16_t* gs, const uint16_t* gb,
                 const uint8_t* uq, const uint16_t* us, const uint16_t* ub,
                 const uint8_t* dq, const uint16_t* ds, const uint16_t* db,
                 const int32_t* ids, const double* gates, int nrows,
                 const int32_t* rows, double* y) {
  if (T < 0 || d <= 0 || d % 64 || F <= 0 || F % 64 || E <= 0 || k <= 0 || k > E)
    return -1;
  for (int r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= T) return -2;

  std::vector<double> Wg((size_t)F * d), Wu((size_t)F * d), Wd((size_t)d * F);
  std::vector<double> xr(d), h(F), o(d);
  std::fill(y, y + (size_t)nrows * d, 0.0);

  // Which experts the selected rows need (the shared expert always).
  std::vector<char> needed(E + 1, 0);
  needed[E] = 1;
  for (int r = 0; r < nrows; ++r)
    for (int j = 0; j < k; ++j) {
      int e = ids[(size_t)rows[r] * k + j];
      if (e < 0 || e >= E) return -3;
      needed[e] = 1;
    }

  const size_t gsz = (size_t)F * d;  // elements of a gate/up matrix
  for (int e = 0; e <= E; ++e) {
    if (!needed[e]) continue;
    orc_dequant(F, d, gq + (size_t)e * gsz / 2, gs + (size_t)e * gsz / 64,
                gb + (size_t)e * gsz / 64, Wg.data());
    orc_dequant(F, d, uq + (size_t)e * gsz / 2, us + (size_t)e * gsz / 64,
                ub + (size_t)e * gsz / 64, Wu.data());
    orc_dequant(d, F, dq + (size_t)e * gsz / 2, ds + (size_t)e * gsz / 64,
                db + (size_t)e * gsz / 64, Wd.data());
    for (int r = 0; r < nrows; ++r) {
      int t = rows[r];
      double weight = 0.0;
      if (e == E) {
        weight = 1.0;  // shared expert: every token, weight 1
      } else {
        for (int j = 0; j < k; ++j)
          if (ids[(size_t)t * k + j] == e) weight += gates[(size_t)t * k + j];
        if (weight == 0.0) continue;  // this row does not use expert e
      }
      for (int i = 0; i < d; ++i) xr[i] = bf16_to_double(x[(size_t)t * d + i]);
      ffn_row(d, F, Wg.data(), Wu.data(), Wd.data(), xr.data(), h.data(), o.data());
      for (int i = 0; i < d; ++i) y[(size_t)r * d + i] += weight * o[i];
    }
  }
  return 0;
}

// The whole layer from scratch: double logits, rounded to fp32 for routing,
// then orc_route and orc_moe_rows over every token.  Used as the timed CPU
// baseline.  ids/gates/y are outputs ([T][k], [T][k], [T][d]).
int orc_moe_layer(int T, int d, int E, int k, int F, int BM, const uint16_t* x,
                  const float* wr, const float* br,
                  const uint8_t* gq, const uint16_t* gs, const uint16_t* gb,
                  const uint8_t* uq, const uint16_t* us, const uint16_t* ub,
                  const uint8_t* dq, const uint16_t* ds, const uint16_t* db,
                  int32_t* ids, double* gates, double* y) {
  if (T <= 0) return -1;
  std::vector<double> L((size_t)T * E);
  std::vector<float> Lf((size_t)T * E);
  int rc = orc_router_logits(T, d, E, x, wr, br, L.data(), nullptr);
  if (rc) return rc;
  for (size_t i = 0; i < L.size(); ++i) Lf[i] = (float)L[i];
  int P = T * k, cap = orc_block_map_cap(T, E, k, BM), nt = 0, nn = 0;
  std::vector<int32_t> counts(E), offsets(E + 1), perm(P), inv(P), bmap(2 * (size_t)cap);
  rc = orc_route(T, E, k, BM, Lf.data(), ids, gates, counts.data(), offsets.data(),
                 perm.data(), inv.data(), bmap.data(), cap, &nt, &nn);
  if (rc) return rc;
  std::vector<int32_t> rows(T);
  for (int t = 0; t < T; ++t) rows[t] = t;
  return orc_moe_rows(T, d, E, k, F, x, gq, gs, gb, uq, us, ub, dq, ds, db, ids,
                      gates, T, rows.data(), y);
}

// Unit-weight RMSNorm in double: out[t][i] = x[t][i] / sqrt(mean_i x^2 + eps).
int orc_rmsnorm(int T, int d, const float* x, double eps, double* out) {
  if (T < 0 || d <= 0) return -1;
  for (int t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int i = 0; i < d; ++i) ss += (double)x[(size_t)t * d + i] * (double)x[(size_t)t * d + i];
    double inv = 1.0 / std::sqrt(ss / d + eps);
    for (int i = 0; i < d; ++i) out[(size_t)t * d + i] = (double)x[(size_t)t * d + i] * inv;
  }
  return 0;
}

}  // extern "C"
