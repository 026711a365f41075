// moe_oracle.cpp -- fp64 CPU oracle of the top-k SwiGLU MoE layer.
//
// TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
// benchmark's CPU-baseline leg; never by the product path. Shares nothing
// with the CUDA library. The header states what each entry point computes
// and which page passage it follows.
//
// Structure: the plain definition, one assignment (token t, rank j, expert e)
// at a time, in the order the layer is described on the clip "Mixture-of-
// Kittens: Cursor open-sources an MoE training megakernel" (key flowchart:
// router top-k -> dispatch -> expert FFN + SwiGLU -> combine -> weighted sum;
// key point 2 for the mirrored backward rounds). Threads only split
// independent outputs (tokens, or rows of a weight gradient); each output
// element is accumulated by one thread in a fixed order.

#include "moe_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---- element access ------------------------------------------------------

inline double bf16_to_double(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;  // bf16 = high half of fp32
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

struct F64View {
  const double* p;
  double operator[](size_t i) const { return p[i]; }
};
struct BF16View {
  const uint16_t* p;
  double operator[](size_t i) const { return bf16_to_double(p[i]); }
};

// ---- static work split over threads --------------------------------------

template <class Fn>
void parallel_for(int64_t n, int threads, Fn fn) {
  if (threads <= 0) threads = static_cast<int>(std::thread::hardware_concurrency());
  if (threads <= 0) threads = 1;
  if (n <= 0) return;
  if (threads > n) threads = static_cast<int>(n);
  if (threads == 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  std::vector<std::thread> pool;
  pool.reserve(threads);
  for (int w = 0; w < threads; ++w) {
    int64_t lo = n * w / threads, hi = n * (w + 1) / threads;
    pool.emplace_back([lo, hi, &fn] {
      for (int64_t i = lo; i < hi; ++i) fn(i);
    });
  }
  for (auto& th : pool) th.join();
}

inline double sigmoid(double g) { return 1.0 / (1.0 + std::exp(-g)); }

struct Shape {
  int64_t N;
  int32_t H, I, E, k;
};

// One expert applied to one token (forward): g = Wg[e] x, u = Wu[e] x,
// a = silu(g) * u, ye = Wd[e] a.
template <class V>
void expert_forward(const Shape& s, const V& x, const V& wg, const V& wu,
                    const V& wd, int64_t t, int32_t e, double* g, double* u,
                    double* a, double* ye) {
  const size_t H = s.H, I = s.I;
  const size_t xo = static_cast<size_t>(t) * H;
  const size_t wo = static_cast<size_t>(e) * I * H;
  for (size_t i = 0; i < I; ++i) {
    double gs = 0.0, us = 0.0;
    for (size_t h = 0; h < H; ++h) {
      double xv = x[xo + h];
      gs += wg[wo + i * H + h] * xv;
      us += wu[wo + i * H + h] * xv;
    }
    g[i] = gs;
    u[i] = us;
    a[i] = gs * sigmoid(gs) * us;
  }
  const size_t wdo = static_cast<size_t>(e) * H * I;
  for (size_t h = 0; h < H; ++h) {
    double acc = 0.0;
    for (size_t i = 0; i < I; ++i) acc += wd[wdo + h * I + i] * a[i];
    ye[h] = acc;
  }
}

// One expert, one token (backward), given dye = dL/dye:
//   da = Wd[e]^T dye
//   dg = da * u * s * (1 + g (1 - s)),  du = da * g * s,  s = sigmoid(g)
//   dxe = Wg[e]^T dg + Wu[e]^T du
template <class V>
void expert_backward(const Shape& s, const V& wg, const V& wu, const V& wd,
                     int32_t e, const double* g, const double* u,
                     const double* dye, double* da, double* dg, double* du,
                     double* dxe) {
  const size_t H = s.H, I = s.I;
  const size_t wdo = static_cast<size_t>(e) * H * I;
  for (size_t i = 0; i < I; ++i) da[i] = 0.0;
  for (size_t h = 0; h < H; ++h) {
    double d = dye[h];
    for (size_t i = 0; i < I; ++i) da[i] += wd[wdo + h * I + i] * d;
  }
  for (size_t i = 0; i < I; ++i) {
    double sg = sigmoid(g[i]);
    dg[i] = da[i] * u[i] * sg * (1.0 + g[i] * (1.0 - sg));
    du[i] = da[i] * g[i] * sg;
  }
  const size_t wo = static_cast<size_t>(e) * I * H;
  for (size_t h = 0; h < H; ++h) dxe[h] = 0.0;
  for (size_t i = 0; i < I; ++i) {
    double a1 = dg[i], a2 = du[i];
    for (size_t h = 0; h < H; ++h)
      dxe[h] += wg[wo + i * H + h] * a1 + wu[wo + i * H + h] * a2;
  }
}

bool shape_ok(const Shape& s) {
  return s.N >= 0 && s.H > 0 && s.I > 0 && s.E > 0 && s.k > 0 && s.k <= s.E;
}

template <class V>
int forward_impl(const Shape& s, const V& x, const V& wg, const V& wu,
                 const V& wd, const int32_t* ids, const double* w, double* y,
                 double* ye_out, int threads) {
  if (!shape_ok(s)) return ORC_ERR_ARG;
  for (int64_t a = 0; a < s.N * s.k; ++a)
    if (ids[a] < 0 || ids[a] >= s.E) return ORC_ERR_ARG;
  parallel_for(s.N, threads, [&](int64_t t) {
    std::vector<double> g(s.I), u(s.I), a(s.I), ye(s.H);
    double* yt = y + t * s.H;
    for (int32_t h = 0; h < s.H; ++h) yt[h] = 0.0;
    for (int32_t j = 0; j < s.k; ++j) {
      const int64_t aidx = t * s.k + j;
      expert_forward(s, x, wg, wu, wd, t, ids[aidx], g.data(), u.data(),
                     a.data(), ye.data());
      const double wj = w[aidx];
      for (int32_t h = 0; h < s.H; ++h) yt[h] += wj * ye[h];
      if (ye_out)
        std::memcpy(ye_out + aidx * s.H, ye.data(), sizeof(double) * s.H);
    }
  });
  return ORC_OK;
}

// Per-assignment backward quantities for the listed tokens: dx rows, dw,
// and (optionally) the vectors the weight gradients need.
template <class V, class VD>
void token_backward(const Shape& s, const V& x, const V& wg, const V& wu,
                    const V& wd, const int32_t* ids, const double* w,
                    const VD& dy, int64_t t, double* yt, double* dxt,
                    double* dwt, double* keep_a, double* keep_dye,
                    double* keep_dg, double* keep_du) {
  std::vector<double> g(s.I), u(s.I), a(s.I), ye(s.H), dye(s.H), da(s.I),
      dg(s.I), du(s.I), dxe(s.H);
  if (yt)
    for (int32_t h = 0; h < s.H; ++h) yt[h] = 0.0;
  for (int32_t h = 0; h < s.H; ++h) dxt[h] = 0.0;
  for (int32_t j = 0; j < s.k; ++j) {
    const int64_t aidx = t * s.k + j;
    const int32_t e = ids[aidx];
    expert_forward(s, x, wg, wu, wd, t, e, g.data(), u.data(), a.data(),
                   ye.data());
    const double wj = w[aidx];
    if (yt)
      for (int32_t h = 0; h < s.H; ++h) yt[h] += wj * ye[h];
    double dwa = 0.0;
    for (int32_t h = 0; h < s.H; ++h) {
      double dyv = dy[static_cast<size_t>(t) * s.H + h];
      dye[h] = wj * dyv;        // reverse-combine: dL/dye = w * dy
      dwa += dyv * ye[h];       // dL/dw = <dy, ye>
    }
    dwt[j] = dwa;
    expert_backward(s, wg, wu, wd, e, g.data(), u.data(), dye.data(),
                    da.data(), dg.data(), du.data(), dxe.data());
    for (int32_t h = 0; h < s.H; ++h) dxt[h] += dxe[h];  // reverse-dispatch
    if (keep_a) std::memcpy(keep_a + aidx * s.I, a.data(), sizeof(double) * s.I);
    if (keep_dye) std::memcpy(keep_dye + aidx * s.H, dye.data(), sizeof(double) * s.H);
    if (keep_dg) std::memcpy(keep_dg + aidx * s.I, dg.data(), sizeof(double) * s.I);
    if (keep_du) std::memcpy(keep_du + aidx * s.I, du.data(), sizeof(double) * s.I);
  }
}

template <class V>
int backward_impl(const Shape& s, const V& x, const V& wg, const V& wu,
                  const V& wd, const int32_t* ids, const double* w, const V& dy,
                  double* dx, double* dwg, double* dwu, double* dwd, double* dw,
                  int threads) {
  if (!shape_ok(s)) return ORC_ERR_ARG;
  const int64_t A = s.N * s.k;
  for (int64_t a = 0; a < A; ++a)
    if (ids[a] < 0 || ids[a] >= s.E) return ORC_ERR_ARG;
  std::vector<double> keep_a(static_cast<size_t>(A) * s.I),
      keep_dye(static_cast<size_t>(A) * s.H), keep_dg(static_cast<size_t>(A) * s.I),
      keep_du(static_cast<size_t>(A) * s.I);
  parallel_for(s.N, threads, [&](int64_t t) {
    token_backward(s, x, wg, wu, wd, ids, w, dy, t, nullptr, dx + t * s.H,
                   dw + t * s.k, keep_a.data(), keep_dye.data(), keep_dg.data(),
                   keep_du.data());
  });
  // Assignments of each expert in ascending token order.
  std::vector<std::vector<int64_t>> of_e(s.E);
  for (int64_t a = 0; a < A; ++a) of_e[ids[a]].push_back(a);
  const int64_t H = s.H, I = s.I;
  // dWg[e][i][:] and dWu[e][i][:] : one (e, i) row per work item.
  parallel_for(static_cast<int64_t>(s.E) * I, threads, [&](int64_t r) {
    const int64_t e = r / I, i = r % I;
    double* rg = dwg + (e * I + i) * H;
    double* ru = dwu + (e * I + i) * H;
    for (int64_t h = 0; h < H; ++h) rg[h] = ru[h] = 0.0;
    for (int64_t a : of_e[e]) {
      const int64_t t = a / s.k;
      const double cg = keep_dg[a * I + i], cu = keep_du[a * I + i];
      for (int64_t h = 0; h < H; ++h) {
        double xv = x[static_cast<size_t>(t * H + h)];
        rg[h] += cg * xv;
        ru[h] += cu * xv;
      }
    }
  });
  // dWd[e][h][:] = sum over assignments of dye[h] * a[:].
  parallel_for(static_cast<int64_t>(s.E) * H, threads, [&](int64_t r) {
    const int64_t e = r / H, h = r % H;
    double* rd = dwd + (e * H + h) * I;
    for (int64_t i = 0; i < I; ++i) rd[i] = 0.0;
    for (int64_t a : of_e[e]) {
      const double c = keep_dye[a * H + h];
      const double* av = keep_a.data() + a * I;
      for (int64_t i = 0; i < I; ++i) rd[i] += c * av[i];
    }
  });
  return ORC_OK;
}

double round_half_even(double q) {  // q >= 0, few significant bits
  double fl = std::floor(q);
  double d = q - fl;
  if (d > 0.5) return fl + 1.0;
  if (d < 0.5) return fl;
  return (std::fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

}  // namespace

extern "C" {

int orc_route_topk(int64_t N, int32_t E, int32_t k, const float* logits,
                   const float* bias, int32_t* ids, double* w) {
  if (N < 0 || E <= 0 || k <= 0 || k > E) return ORC_ERR_ARG;
  std::vector<float> z(E);
  std::vector<int32_t> order(E);
  for (int64_t t = 0; t < N; ++t) {
    for (int32_t e = 0; e < E; ++e) {
      float b = bias ? bias[e] : 0.0f;
      volatile float zz = logits[t * E + e] + b;  // one IEEE fp32 add
      z[e] = zz;
      if (std::isnan(z[e])) return ORC_ERR_NAN;
    }
    for (int32_t e = 0; e < E; ++e) order[e] = e;
    // Larger z first; equal z keep ascending expert index (stable sort).
    std::stable_sort(order.begin(), order.end(),
                     [&](int32_t a, int32_t b) { return z[a] > z[b]; });
    const double zmax = z[order[0]];
    double denom = 0.0;
    for (int32_t j = 0; j < k; ++j) denom += std::exp(static_cast<double>(z[order[j]]) - zmax);
    for (int32_t j = 0; j < k; ++j) {
      ids[t * k + j] = order[j];
      w[t * k + j] = std::exp(static_cast<double>(z[order[j]]) - zmax) / denom;
    }
  }
  return ORC_OK;
}

int orc_router_logits(int64_t N, int32_t H, int32_t E, const uint16_t* x, const uint16_t* wr,
                      double* logits, int threads) {
  if (N < 0 || H <= 0 || E <= 0) return ORC_ERR_ARG;
  // logits[t][e] = sum_h x[t][h] * Wr[e][h], every product and sum in fp64
  parallel_for(N, threads, [&](int64_t t) {
    for (int32_t e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int32_t h = 0; h < H; ++h)
        acc += bf16_to_double(x[t * H + h]) * bf16_to_double(wr[static_cast<int64_t>(e) * H + h]);
      logits[t * E + e] = acc;
    }
  });
  return ORC_OK;
}

int orc_router_backward(int64_t N, int32_t H, int32_t E, int32_t k, const uint16_t* x,
                        const uint16_t* wr, const int32_t* ids, const double* w,
                        const double* dw, double* dz, double* dwr, double* dx, int threads) {
  if (N < 0 || H <= 0 || E <= 0 || k <= 0 || k > E) return ORC_ERR_ARG;
  for (int64_t a = 0; a < N * k; ++a)
    if (ids[a] < 0 || ids[a] >= E) return ORC_ERR_ARG;
  // w = softmax over the k selected logits z_j: dL/dz_j = w_j (dL/dw_j - sum_i w_i dL/dw_i)
  for (int64_t t = 0; t < N; ++t) {
    double s = 0.0;
    for (int32_t j = 0; j < k; ++j) s += w[t * k + j] * dw[t * k + j];
    for (int32_t j = 0; j < k; ++j) dz[t * k + j] = w[t * k + j] * (dw[t * k + j] - s);
  }
  // logits = x Wr^T: dWr[e] = sum over (t, j) routed to e of dz[t,j] x[t]; dx[t] = sum_j dz[t,j] Wr[ids[t,j]]
  parallel_for(E, threads, [&](int64_t e) {
    for (int32_t h = 0; h < H; ++h) dwr[e * H + h] = 0.0;
    for (int64_t a = 0; a < N * k; ++a)
      if (ids[a] == e)
        for (int32_t h = 0; h < H; ++h) dwr[e * H + h] += dz[a] * bf16_to_double(x[(a / k) * H + h]);
  });
  parallel_for(N, threads, [&](int64_t t) {
    for (int32_t h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int32_t j = 0; j < k; ++j)
        acc += dz[t * k + j] * bf16_to_double(wr[static_cast<int64_t>(ids[t * k + j]) * H + h]);
      dx[t * H + h] = acc;
    }
  });
  return ORC_OK;
}

int orc_build_schedule(int64_t N, int32_t k, int32_t E, int32_t tile_m,
                       const int32_t* ids, int32_t* counts, int32_t* offsets,
                       int32_t* pad_offsets, int32_t* slot_of,
                       int32_t* src_of_row, int64_t rows_cap, int32_t* tiles,
                       int64_t tiles_cap, int32_t* n_tiles) {
  return orc_build_schedule_padded(N, k, E, tile_m, tile_m, ids, counts, offsets, pad_offsets,
                                   slot_of, src_of_row, rows_cap, tiles, tiles_cap, n_tiles);
}

int orc_build_schedule_padded(int64_t N, int32_t k, int32_t E, int32_t tile_m, int32_t pad_m,
                              const int32_t* ids, int32_t* counts, int32_t* offsets,
                              int32_t* pad_offsets, int32_t* slot_of,
                              int32_t* src_of_row, int64_t rows_cap, int32_t* tiles,
                              int64_t tiles_cap, int32_t* n_tiles) {
  if (N < 0 || k <= 0 || E <= 0 || tile_m <= 0 || pad_m <= 0 || pad_m % tile_m != 0)
    return ORC_ERR_ARG;
  const int64_t A = N * k;
  for (int32_t e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t a = 0; a < A; ++a) {
    if (ids[a] < 0 || ids[a] >= E) return ORC_ERR_ARG;
    counts[ids[a]] += 1;
  }
  offsets[0] = 0;
  pad_offsets[0] = 0;
  for (int32_t e = 0; e < E; ++e) {
    offsets[e + 1] = offsets[e] + counts[e];
    const int32_t padded = (counts[e] + pad_m - 1) / pad_m * pad_m;
    pad_offsets[e + 1] = pad_offsets[e] + padded;
  }
  const int64_t rows = pad_offsets[E];
  const int64_t nt = rows / tile_m;
  if (rows > rows_cap || nt > tiles_cap) return ORC_ERR_ARG;
  for (int64_t r = 0; r < rows; ++r) src_of_row[r] = -1;
  std::vector<int32_t> seen(E, 0);
  for (int64_t t = 0; t < N; ++t)
    for (int32_t j = 0; j < k; ++j) {
      const int64_t a = t * k + j;
      const int32_t e = ids[a];
      const int32_t row = pad_offsets[e] + seen[e];
      seen[e] += 1;
      slot_of[a] = row;
      src_of_row[row] = static_cast<int32_t>(a);
    }
  int64_t i = 0;
  for (int32_t e = 0; e < E; ++e)
    for (int32_t r0 = pad_offsets[e]; r0 < pad_offsets[e + 1]; r0 += tile_m) {
      tiles[3 * i + 0] = e;
      tiles[3 * i + 1] = r0;
      tiles[3 * i + 2] = std::max(0, std::min(tile_m, pad_offsets[e] + counts[e] - r0));
      ++i;
    }
  *n_tiles = static_cast<int32_t>(i);
  return ORC_OK;
}

int orc_forward_f64(int64_t N, int32_t H, int32_t I, int32_t E, int32_t k,
                    const double* x, const double* wg, const double* wu,
                    const double* wd, const int32_t* ids, const double* w,
                    double* y, double* ye_out, int threads) {
  Shape s{N, H, I, E, k};
  return forward_impl(s, F64View{x}, F64View{wg}, F64View{wu}, F64View{wd}, ids,
                      w, y, ye_out, threads);
}

int orc_forward_bf16(int64_t N, int32_t H, int32_t I, int32_t E, int32_t k,
                     const uint16_t* x, const uint16_t* wg, const uint16_t* wu,
                     const uint16_t* wd, const int32_t* ids, const double* w,
                     double* y, double* ye_out, int threads) {
  Shape s{N, H, I, E, k};
  return forward_impl(s, BF16View{x}, BF16View{wg}, BF16View{wu}, BF16View{wd},
                      ids, w, y, ye_out, threads);
}

int orc_backward_f64(int64_t N, int32_t H, int32_t I, int32_t E, int32_t k,
                     const double* x, const double* wg, const double* wu,
                     const double* wd, const int32_t* ids, const double* w,
                     const double* dy, double* dx, double* dwg, double* dwu,
                     double* dwd, double* dw, int threads) {
  Shape s{N, H, I, E, k};
  return backward_impl(s, F64View{x}, F64View{wg}, F64View{wu}, F64View{wd}, ids,
                       w, F64View{dy}, dx, dwg, dwu, dwd, dw, threads);
}

int orc_backward_bf16(int64_t N, int32_t H, int32_t I, int32_t E, int32_t k,
                      const uint16_t* x, const uint16_t* wg, const uint16_t* wu,
                      const uint16_t* wd, const int32_t* ids, const double* w,
                      const uint16_t* dy, double* dx, double* dwg, double* dwu,
                      double* dwd, double* dw, int threads) {
  Shape s{N, H, I, E, k};
  return backward_impl(s, BF16View{x}, BF16View{wg}, BF16View{wu}, BF16View{wd},
                       ids, w, BF16View{dy}, dx, dwg, dwu, dwd, dw, threads);
}

int orc_tokens_bf16(int64_t N, int32_t H, int32_t I, int32_t E, int32_t k,
                    const uint16_t* x, const uint16_t* wg, const uint16_t* wu,
                    const uint16_t* wd, const int32_t* ids, const double* w,
                    const uint16_t* dy, int64_t n_tok, const int64_t* tok,
                    double* y, double* dx, double* dw, int threads) {
  Shape s{N, H, I, E, k};
  if (!shape_ok(s) || n_tok < 0) return ORC_ERR_ARG;
  for (int64_t r = 0; r < n_tok; ++r) {
    if (tok[r] < 0 || tok[r] >= N) return ORC_ERR_ARG;
    for (int32_t j = 0; j < k; ++j)
      if (ids[tok[r] * k + j] < 0 || ids[tok[r] * k + j] >= E) return ORC_ERR_ARG;
  }
  parallel_for(n_tok, threads, [&](int64_t r) {
    token_backward(s, BF16View{x}, BF16View{wg}, BF16View{wu}, BF16View{wd}, ids,
                   w, BF16View{dy}, tok[r], y + r * H, dx + r * H, dw + r * k,
                   nullptr, nullptr, nullptr, nullptr);
  });
  return ORC_OK;
}

int orc_expert_wgrad_bf16(int64_t N, int32_t H, int32_t I, int32_t E,
                          int32_t k, const uint16_t* x, const uint16_t* wg,
                          const uint16_t* wu, const uint16_t* wd,
                          const int32_t* ids, const double* w,
                          const uint16_t* dy, int32_t e, int64_t n_i,
                          const int32_t* i_list, int64_t n_h,
                          const int32_t* h_list, double* dwg_rows,
                          double* dwu_rows, double* dwd_rows, int threads) {
  Shape s{N, H, I, E, k};
  if (!shape_ok(s) || e < 0 || e >= E) return ORC_ERR_ARG;
  for (int64_t r = 0; r < n_i; ++r)
    if (i_list[r] < 0 || i_list[r] >= I) return ORC_ERR_ARG;
  for (int64_t r = 0; r < n_h; ++r)
    if (h_list[r] < 0 || h_list[r] >= H) return ORC_ERR_ARG;
  std::vector<int64_t> mine;  // assignments routed to e, ascending token
  for (int64_t a = 0; a < N * k; ++a)
    if (ids[a] == e) mine.push_back(a);
  const int64_t M = static_cast<int64_t>(mine.size());
  std::vector<double> keep_a(M * I), keep_dye(M * H), keep_dg(M * I), keep_du(M * I);
  parallel_for(M, threads, [&](int64_t m) {
    const int64_t a = mine[m], t = a / k;
    std::vector<double> g(I), u(I), av(I), ye(H), da(I), dxe(H);
    expert_forward(s, BF16View{x}, BF16View{wg}, BF16View{wu}, BF16View{wd}, t, e,
                   g.data(), u.data(), av.data(), ye.data());
    double* dye = keep_dye.data() + m * H;
    for (int32_t h = 0; h < H; ++h)
      dye[h] = w[a] * bf16_to_double(dy[static_cast<size_t>(t) * H + h]);
    expert_backward(s, BF16View{wg}, BF16View{wu}, BF16View{wd}, e, g.data(),
                    u.data(), dye, da.data(), keep_dg.data() + m * I,
                    keep_du.data() + m * I, dxe.data());
    std::memcpy(keep_a.data() + m * I, av.data(), sizeof(double) * I);
  });
  BF16View xv{x};
  parallel_for(n_i, threads, [&](int64_t r) {
    const int64_t i = i_list[r];
    double* rg = dwg_rows + r * H;
    double* ru = dwu_rows + r * H;
    for (int32_t h = 0; h < H; ++h) rg[h] = ru[h] = 0.0;
    for (int64_t m = 0; m < M; ++m) {
      const int64_t t = mine[m] / k;
      const double cg = keep_dg[m * I + i], cu = keep_du[m * I + i];
      for (int32_t h = 0; h < H; ++h) {
        double xx = xv[static_cast<size_t>(t) * H + h];
        rg[h] += cg * xx;
        ru[h] += cu * xx;
      }
    }
  });
  parallel_for(n_h, threads, [&](int64_t r) {
    const int64_t h = h_list[r];
    double* rd = dwd_rows + r * I;
    for (int32_t i = 0; i < I; ++i) rd[i] = 0.0;
    for (int64_t m = 0; m < M; ++m) {
      const double c = keep_dye[m * H + h];
      for (int32_t i = 0; i < I; ++i) rd[i] += c * keep_a[m * I + i];
    }
  });
  return ORC_OK;
}

uint8_t orc_e4m3_encode(double v) {
  const uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
  double a = std::fabs(v);
  if (std::isnan(v)) return 0x7F;
  if (a >= 448.0) return sign | 0x7E;  // saturate (largest finite E4M3)
  if (a < std::ldexp(1.0, -6)) {
    // Subnormal range: multiples of 2^-9. A result of 8 quanta is 2^-6,
    // whose code (exponent field 1, mantissa 0) is also 8.
    double m = round_half_even(a * 512.0);
    return sign | static_cast<uint8_t>(m);
  }
  int ex;
  std::frexp(a, &ex);        // a = f * 2^ex, f in [0.5, 1)
  int e = ex - 1;            // floor(log2 a), in [-6, 8]
  double m = round_half_even(std::ldexp(a, 3 - e));  // in [8, 16]
  if (m == 16.0) {
    m = 8.0;
    e += 1;
  }
  int code = ((e + 7) << 3) | (static_cast<int>(m) - 8);
  if (code > 0x7E) code = 0x7E;  // 480 would round into the NaN code
  return sign | static_cast<uint8_t>(code);
}

double orc_e4m3_decode(uint8_t code) {
  const double sgn = (code & 0x80) ? -1.0 : 1.0;
  const int e = (code >> 3) & 0xF, m = code & 0x7;
  if (e == 15 && m == 7) return std::nan("");
  if (e == 0) return sgn * std::ldexp(static_cast<double>(m), -9);
  return sgn * std::ldexp(static_cast<double>(8 + m), e - 10);
}

int orc_mxfp8_quantize(int64_t rows, int64_t cols, const uint16_t* src,
                       uint8_t* q, uint8_t* scale) {
  if (rows < 0 || cols < 0 || cols % 32 != 0) return ORC_ERR_ARG;
  const int64_t nb = cols / 32;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < nb; ++b) {
      const uint16_t* blk = src + r * cols + b * 32;
      double amax = 0.0;
      for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(bf16_to_double(blk[i])));
      int code = 0;
      if (amax > 0.0) {
        int ex;
        std::frexp(amax, &ex);
        const int shared_exp = (ex - 1) - 8;  // floor(log2 amax) - emax(E4M3)
        code = std::min(254, std::max(0, shared_exp + 127));
      }
      scale[r * nb + b] = static_cast<uint8_t>(code);
      for (int i = 0; i < 32; ++i)
        q[r * cols + b * 32 + i] =
            orc_e4m3_encode(std::ldexp(bf16_to_double(blk[i]), 127 - code));
    }
  return ORC_OK;
}

// ---------------------------------------------------------------------------
// MXFP8 layer: every operand of every GEMM is quantised to MXFP8 along that
// GEMM's K (1x32 blocks, E8M0 scale, E4M3 elements; the rule of
// orc_mxfp8_quantize) and dequantised exactly; products are summed in fp64.
// An intermediate is first rounded to bf16 (where the layer stores it) and
// then quantised. Token-axis blocks (weight gradients) hold 32 consecutive
// assignments of one expert in slot order (ascending token) and restart at
// each expert; a short last block is padded with zeros.

int orc_mxfp8_quantize(int64_t rows, int64_t cols, const uint16_t* src, uint8_t* q,
                       uint8_t* scale);

namespace {

double round_bf16(double v) {
  float f = static_cast<float>(v);  // correctly rounded fp64 -> fp32
  uint32_t u;
  std::memcpy(&u, &f, 4);
  // fp32 -> bf16 round to nearest even (finite values)
  u = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

// Quantise-dequantise one block of n <= 32 values (each exactly a bf16 value).
void qdq_block(double* v, int n) {
  double amax = 0.0;
  for (int i = 0; i < n; ++i) amax = std::max(amax, std::fabs(v[i]));
  int code = 0;
  if (amax > 0.0) {
    int ex;
    std::frexp(amax, &ex);
    code = std::min(254, std::max(0, (ex - 1) - 8 + 127));
  }
  for (int i = 0; i < n; ++i)
    v[i] = orc_e4m3_decode(orc_e4m3_encode(std::ldexp(v[i], 127 - code))) *
           std::ldexp(1.0, code - 127);
}

// Quantise-dequantise a vector along its length in blocks of 32.
void qdq_vec(double* v, int64_t n) {
  for (int64_t b = 0; b < n; b += 32) qdq_block(v + b, static_cast<int>(std::min<int64_t>(32, n - b)));
}

}  // namespace

extern "C" int orc_mxfp8_weights(int32_t H, int32_t I, int32_t E, const uint16_t* wg,
                                 const uint16_t* wu, const uint16_t* wd, int quantize,
                                 double* wg_h, double* wu_h, double* wd_i, double* wd_h,
                                 double* wg_i, double* wu_i, int threads) {
  if (H <= 0 || I <= 0 || E <= 0) return ORC_ERR_ARG;
  const int64_t HI = static_cast<int64_t>(H) * I;
  // Weights as each GEMM reads them:
  //   gate/up forward: rows of Wg[e], Wu[e] along H;  down forward: rows of Wd[e] along I;
  //   down backward (dA = Wd^T dye): columns of Wd[e] along H;
  //   gate/up backward (dxe = Wg^T dg + Wu^T du): columns of Wg[e], Wu[e] along I.
  parallel_for(E, threads, [&](int64_t e) {
    auto q = [quantize](double* v, int64_t n) { if (quantize) qdq_vec(v, n); };
    const int64_t o = e * HI;
    for (int64_t i = o; i < o + HI; ++i) {
      wg_h[i] = wg_i[i] = bf16_to_double(wg[i]);
      wu_h[i] = wu_i[i] = bf16_to_double(wu[i]);
      wd_i[i] = wd_h[i] = bf16_to_double(wd[i]);
    }
    std::vector<double> col(std::max(H, I));
    for (int32_t i = 0; i < I; ++i) {           // Wg/Wu [e][i][:] along H
      q(&wg_h[o + static_cast<int64_t>(i) * H], H);
      q(&wu_h[o + static_cast<int64_t>(i) * H], H);
    }
    for (int32_t h = 0; h < H; ++h) q(&wd_i[o + static_cast<int64_t>(h) * I], I);  // Wd [e][h][:]
    for (int32_t i = 0; i < I; ++i) {           // Wd [e][:][i] along H
      for (int32_t h = 0; h < H; ++h) col[h] = wd_h[o + static_cast<int64_t>(h) * I + i];
      q(col.data(), H);
      for (int32_t h = 0; h < H; ++h) wd_h[o + static_cast<int64_t>(h) * I + i] = col[h];
    }
    for (int32_t h = 0; h < H; ++h) {           // Wg/Wu [e][:][h] along I
      for (int32_t i = 0; i < I; ++i) col[i] = wg_i[o + static_cast<int64_t>(i) * H + h];
      q(col.data(), I);
      for (int32_t i = 0; i < I; ++i) wg_i[o + static_cast<int64_t>(i) * H + h] = col[i];
      for (int32_t i = 0; i < I; ++i) col[i] = wu_i[o + static_cast<int64_t>(i) * H + h];
      q(col.data(), I);
      for (int32_t i = 0; i < I; ++i) wu_i[o + static_cast<int64_t>(i) * H + h] = col[i];
    }
  });
  return ORC_OK;
}

extern "C" int orc_layer_mxfp8(int64_t N, int32_t H, int32_t I, int32_t E, int32_t k,
                               const uint16_t* x, const uint16_t* wg, const uint16_t* wu,
                               const uint16_t* wd, const int32_t* ids, const double* w,
                               const uint16_t* dy, int quantize, double* y, double* dx,
                               double* dwg, double* dwu, double* dwd, double* dw,
                               int threads) {
  if (H <= 0 || I <= 0 || E <= 0) return ORC_ERR_ARG;
  const int64_t n = static_cast<int64_t>(E) * H * I;
  std::vector<double> wg_h(n), wu_h(n), wd_i(n), wd_h(n), wg_i(n), wu_i(n);
  const int st = orc_mxfp8_weights(H, I, E, wg, wu, wd, quantize, wg_h.data(), wu_h.data(),
                                   wd_i.data(), wd_h.data(), wg_i.data(), wu_i.data(), threads);
  if (st != ORC_OK) return st;
  return orc_layer_mxfp8_prepared(N, H, I, E, k, x, wg_h.data(), wu_h.data(), wd_i.data(),
                                  wd_h.data(), wg_i.data(), wu_i.data(), ids, w, dy, quantize,
                                  y, dx, dwg, dwu, dwd, dw, threads);
}

extern "C" int orc_layer_mxfp8_prepared(int64_t N, int32_t H, int32_t I, int32_t E, int32_t k,
                                        const uint16_t* x, const double* wg_h,
                                        const double* wu_h, const double* wd_i,
                                        const double* wd_h, const double* wg_i,
                                        const double* wu_i, const int32_t* ids, const double* w,
                                        const uint16_t* dy, int quantize, double* y, double* dx,
                                        double* dwg, double* dwu, double* dwd, double* dw,
                                        int threads) {
  return orc_layer_mxfp8_trace(N, H, I, E, k, x, wg_h, wu_h, wd_i, wd_h, wg_i, wu_i, ids, w, dy,
                               quantize, 0, y, dx, dwg, dwu, dwd, dw, nullptr, nullptr, threads);
}

extern "C" int orc_layer_mxfp8_trace(int64_t N, int32_t H, int32_t I, int32_t E, int32_t k,
                                     const uint16_t* x, const double* wg_h, const double* wu_h,
                                     const double* wd_i, const double* wd_h, const double* wg_i,
                                     const double* wu_i, const int32_t* ids, const double* w,
                                     const uint16_t* dy, int quantize, int gu_bf16, double* y,
                                     double* dx, double* dwg, double* dwu, double* dwd, double* dw,
                                     double* dg_rows, double* du_rows, int threads) {
  if (N < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || k > E) return ORC_ERR_ARG;
  const int64_t A = N * k;
  for (int64_t a = 0; a < A; ++a)
    if (ids[a] < 0 || ids[a] >= E) return ORC_ERR_ARG;
  auto q = [quantize](double* v, int64_t n) { if (quantize) qdq_vec(v, n); };
  auto rb = [quantize](double v) { return quantize ? round_bf16(v) : v; };
  const int64_t HI = static_cast<int64_t>(H) * I;
  // Per-assignment forward and backward.
  std::vector<double> G(A * I), U(A * I), Ab(A * I), DYe(A * H), DG(A * I), DU(A * I), YE(A * H);
  parallel_for(N, threads, [&](int64_t t) {
    std::vector<double> xq(H), aq(I), dq(H), da(I), gq(I), uq(I);
    for (int32_t h = 0; h < H; ++h) xq[h] = bf16_to_double(x[t * H + h]);
    q(xq.data(), H);                                                   // Xe rows along H
    for (int32_t h = 0; h < H; ++h) { y[t * H + h] = 0.0; dx[t * H + h] = 0.0; }
    for (int32_t j = 0; j < k; ++j) {
      const int64_t a = t * k + j;
      const int32_t e = ids[a];
      const int64_t o = e * HI;
      for (int32_t i = 0; i < I; ++i) {
        double gs = 0.0, us = 0.0;
        for (int32_t h = 0; h < H; ++h) {
          gs += wg_h[o + static_cast<int64_t>(i) * H + h] * xq[h];
          us += wu_h[o + static_cast<int64_t>(i) * H + h] * xq[h];
        }
        G[a * I + i] = gs;
        U[a * I + i] = us;
        Ab[a * I + i] = rb(gs * sigmoid(gs) * us);                     // Act, stored bf16
        aq[i] = Ab[a * I + i];
      }
      q(aq.data(), I);                                                 // Act rows along I
      double dwa = 0.0;
      for (int32_t h = 0; h < H; ++h) {
        double acc = 0.0;
        for (int32_t i = 0; i < I; ++i) acc += wd_i[o + static_cast<int64_t>(h) * I + i] * aq[i];
        YE[a * H + h] = acc;
        y[t * H + h] += w[a] * acc;                                    // combine
        const double dyv = bf16_to_double(dy[t * H + h]);
        dwa += dyv * acc;
        DYe[a * H + h] = rb(w[a] * dyv);                               // dYe, stored bf16
        dq[h] = DYe[a * H + h];
      }
      dw[a] = dwa;
      q(dq.data(), H);                                                 // dYe rows along H
      for (int32_t i = 0; i < I; ++i) {
        double acc = 0.0;
        for (int32_t h = 0; h < H; ++h) acc += wd_h[o + static_cast<int64_t>(h) * I + i] * dq[h];
        da[i] = acc;
      }
      for (int32_t i = 0; i < I; ++i) {
        // gu_bf16 (diagnostic, off in every parity test): G and U as the
        // bf16 values a layer that stores them reads back
        const double g = gu_bf16 ? round_bf16(G[a * I + i]) : G[a * I + i];
        const double u = gu_bf16 ? round_bf16(U[a * I + i]) : U[a * I + i];
        const double sg = sigmoid(g);
        DG[a * I + i] = rb(da[i] * u * sg * (1.0 + g * (1.0 - sg)));  // dG, dU stored bf16
        DU[a * I + i] = rb(da[i] * g * sg);
        gq[i] = DG[a * I + i];
        uq[i] = DU[a * I + i];
      }
      q(gq.data(), I);                                                 // dG, dU rows along I
      q(uq.data(), I);
      if (dg_rows && du_rows)
        for (int32_t i = 0; i < I; ++i) {
          dg_rows[a * I + i] = gq[i];
          du_rows[a * I + i] = uq[i];
        }
      for (int32_t h = 0; h < H; ++h) {
        double acc = 0.0;
        for (int32_t i = 0; i < I; ++i)
          acc += wg_i[o + static_cast<int64_t>(i) * H + h] * gq[i] +
                 wu_i[o + static_cast<int64_t>(i) * H + h] * uq[i];
        dx[t * H + h] += acc;                                          // reverse-dispatch
      }
    }
  });
  // Weight gradients: contraction over each expert's assignments (slot order),
  // each operand column quantised along that axis in blocks of 32.
  std::vector<std::vector<int64_t>> of_e(E);
  for (int64_t a = 0; a < A; ++a) of_e[ids[a]].push_back(a);
  parallel_for(E, threads, [&](int64_t e) {
    const std::vector<int64_t>& as = of_e[e];
    const int64_t M = static_cast<int64_t>(as.size());
    const int64_t o = e * HI;
    std::vector<double> c1(M), c2(M);
    // token-axis quantised operands, column by column
    std::vector<double> dyeT(H * M), actT(I * M), dgT(I * M), duT(I * M), xeT(H * M);
    for (int32_t h = 0; h < H; ++h) {
      for (int64_t m = 0; m < M; ++m) c1[m] = DYe[as[m] * H + h];
      q(c1.data(), M);
      for (int64_t m = 0; m < M; ++m) c2[m] = bf16_to_double(x[(as[m] / k) * H + h]);
      q(c2.data(), M);
      for (int64_t m = 0; m < M; ++m) { dyeT[h * M + m] = c1[m]; xeT[h * M + m] = c2[m]; }
    }
    for (int32_t i = 0; i < I; ++i) {
      for (int64_t m = 0; m < M; ++m) c1[m] = Ab[as[m] * I + i];
      q(c1.data(), M);
      for (int64_t m = 0; m < M; ++m) actT[i * M + m] = c1[m];
      for (int64_t m = 0; m < M; ++m) c1[m] = DG[as[m] * I + i];
      q(c1.data(), M);
      for (int64_t m = 0; m < M; ++m) dgT[i * M + m] = c1[m];
      for (int64_t m = 0; m < M; ++m) c1[m] = DU[as[m] * I + i];
      q(c1.data(), M);
      for (int64_t m = 0; m < M; ++m) duT[i * M + m] = c1[m];
    }
    for (int32_t h = 0; h < H; ++h)
      for (int32_t i = 0; i < I; ++i) {
        double acc = 0.0;
        for (int64_t m = 0; m < M; ++m) acc += dyeT[h * M + m] * actT[i * M + m];
        dwd[o + static_cast<int64_t>(h) * I + i] = acc;
      }
    for (int32_t i = 0; i < I; ++i)
      for (int32_t h = 0; h < H; ++h) {
        double ag = 0.0, au = 0.0;
        for (int64_t m = 0; m < M; ++m) {
          ag += dgT[i * M + m] * xeT[h * M + m];
          au += duT[i * M + m] * xeT[h * M + m];
        }
        dwg[o + static_cast<int64_t>(i) * H + h] = ag;
        dwu[o + static_cast<int64_t>(i) * H + h] = au;
      }
  });
  return ORC_OK;
}

// The MXFP8 weight gradients of expert e at sampled entries, by the steps of
// orc_layer_mxfp8 restricted to what those entries read. Each of e's
// assignments (ascending token) needs its Xe and dYe rows quantised along H
// (whole rows) and, for each listed i, G, U, Act, dAct, dG and dU; each
// listed column then goes through the token-axis quantisation of its own
// column (blocks of 32 assignments from the start of e's list), and the
// contraction runs over the assignments in the same order. Results equal
// orc_layer_mxfp8's dwg[e][i][h], dwu[e][i][h] and dwd[e][h][i] at
// i = i_list[r], h = h_list[c]: dwg, dwu [n_i][n_h], dwd [n_h][n_i].
int orc_expert_wgrad_mxfp8(int64_t N, int32_t H, int32_t I, int32_t E, int32_t k,
                           const uint16_t* x, const uint16_t* wg, const uint16_t* wu,
                           const uint16_t* wd, const int32_t* ids, const double* w,
                           const uint16_t* dy, int32_t e, int64_t n_i, const int32_t* i_list,
                           int64_t n_h, const int32_t* h_list, int quantize, double* dwg,
                           double* dwu, double* dwd, int threads) {
  if (N < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || k > E || e < 0 || e >= E)
    return ORC_ERR_ARG;
  for (int64_t r = 0; r < n_i; ++r)
    if (i_list[r] < 0 || i_list[r] >= I) return ORC_ERR_ARG;
  for (int64_t c = 0; c < n_h; ++c)
    if (h_list[c] < 0 || h_list[c] >= H) return ORC_ERR_ARG;
  auto q = [quantize](double* v, int64_t n) { if (quantize) qdq_vec(v, n); };
  auto rb = [quantize](double v) { return quantize ? round_bf16(v) : v; };
  const int64_t o = static_cast<int64_t>(e) * H * I;
  // the weight rows and columns the listed i read, quantised as the layer reads them
  std::vector<double> wgr(n_i * H), wur(n_i * H), wdc(n_i * H);
  for (int64_t r = 0; r < n_i; ++r) {
    const int64_t i = i_list[r];
    for (int32_t h = 0; h < H; ++h) {
      wgr[r * H + h] = bf16_to_double(wg[o + i * H + h]);               // Wg[e][i][:]
      wur[r * H + h] = bf16_to_double(wu[o + i * H + h]);
      wdc[r * H + h] = bf16_to_double(wd[o + static_cast<int64_t>(h) * I + i]);  // Wd[e][:][i]
    }
    q(&wgr[r * H], H);
    q(&wur[r * H], H);
    q(&wdc[r * H], H);
  }
  std::vector<int64_t> as;  // e's assignments in slot order
  for (int64_t a = 0; a < N * k; ++a) {
    if (ids[a] < 0 || ids[a] >= E) return ORC_ERR_ARG;
    if (ids[a] == e) as.push_back(a);
  }
  const int64_t M = static_cast<int64_t>(as.size());
  std::vector<double> Ab(M * n_i), DG(M * n_i), DU(M * n_i), DYe(M * n_h), Xb(M * n_h);
  parallel_for(M, threads, [&](int64_t m) {
    const int64_t a = as[m], t = a / k;
    std::vector<double> xq(H), dq(H);
    for (int32_t h = 0; h < H; ++h) {
      xq[h] = bf16_to_double(x[t * H + h]);
      dq[h] = rb(w[a] * bf16_to_double(dy[t * H + h]));              // dYe, stored bf16
    }
    for (int64_t c = 0; c < n_h; ++c) {
      DYe[m * n_h + c] = dq[h_list[c]];
      Xb[m * n_h + c] = xq[h_list[c]];
    }
    q(xq.data(), H);                                                  // Xe rows along H
    q(dq.data(), H);                                                  // dYe rows along H
    for (int64_t r = 0; r < n_i; ++r) {
      double gs = 0.0, us = 0.0, da = 0.0;
      for (int32_t h = 0; h < H; ++h) {
        gs += wgr[r * H + h] * xq[h];
        us += wur[r * H + h] * xq[h];
      }
      for (int32_t h = 0; h < H; ++h) da += wdc[r * H + h] * dq[h];
      const double sg = sigmoid(gs);
      Ab[m * n_i + r] = rb(gs * sg * us);                             // Act, stored bf16
      DG[m * n_i + r] = rb(da * us * sg * (1.0 + gs * (1.0 - sg)));   // dG, dU stored bf16
      DU[m * n_i + r] = rb(da * gs * sg);
    }
  });
  // token-axis quantisation, one listed column at a time
  auto column = [&](const std::vector<double>& src, int64_t stride, int64_t col) {
    std::vector<double> v(M);
    for (int64_t m = 0; m < M; ++m) v[m] = src[m * stride + col];
    q(v.data(), M);
    return v;
  };
  std::vector<std::vector<double>> actT(n_i), dgT(n_i), duT(n_i), dyeT(n_h), xeT(n_h);
  for (int64_t r = 0; r < n_i; ++r) {
    actT[r] = column(Ab, n_i, r);
    dgT[r] = column(DG, n_i, r);
    duT[r] = column(DU, n_i, r);
  }
  for (int64_t c = 0; c < n_h; ++c) {
    dyeT[c] = column(DYe, n_h, c);
    xeT[c] = column(Xb, n_h, c);
  }
  for (int64_t r = 0; r < n_i; ++r)
    for (int64_t c = 0; c < n_h; ++c) {
      double ag = 0.0, au = 0.0, ad = 0.0;
      for (int64_t m = 0; m < M; ++m) {
        ag += dgT[r][m] * xeT[c][m];
        au += duT[r][m] * xeT[c][m];
        ad += dyeT[c][m] * actT[r][m];
      }
      dwg[r * n_h + c] = ag;
      dwu[r * n_h + c] = au;
      dwd[c * n_i + r] = ad;
    }
  return ORC_OK;
}

}  // extern "C"
