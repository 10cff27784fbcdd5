// CPU oracle of the MoE layer with top-k routing and one shared expert, in
// plain C++ with fp64 arithmetic.
//
// TEST INFRASTRUCTURE ONLY.  Only the tests, __graft_entry__.smoke() and the
// benchmark's CPU-baseline / reference leg may load this library.  It shares
// no code with the CUDA path (not even the bf16 decoder).
//
// Plain, slow and obviously correct: every quantity is computed from its
// definition with fp64 accumulation, on fp64 copies of the bf16 inputs, in the
// order of the layer's steps; nothing is rounded to bf16.  Rows, experts or
// tokens are split over std::thread workers; no blocking, fusion or
// reordering of any sum.  The layer, as read from the Olmo-core DDP MoE pages
// ("Olmo-core DDP MoE examples" README, "Production throughput runs": top-4
// routing, one shared expert, learned vs random routing; "Interpreting the
// eight-layer DDP vs FSDP comparison": capacity factor, router, shared-branch
// mixing; "Olmo-core 3 Opens Large MoE Training", "Technical Deep Dive":
// experts stay resident, tokens are routed to them):
//
//   router    l[t,e] = fp32(sum_c x[t,c] W_r[e,c]) + b[e]   (fp32 add)
//   top-k     the k experts first in the order (l descending, e ascending)
//   gates     g[t,s] = exp(l_s - l_0) / sum_{j in S} exp(l_j - l_0)
//   rank      rank(t,s) = #{t' < t : idx[t,s] is among t''s experts}
//   capacity  kept iff capacity <= 0 or rank < capacity (no renormalisation)
//   permute   counts, offsets = exclusive prefix sum, row = offsets[e] + rank
//   expert    a = x W_g[e]^T, u = x W_u[e]^T, h = silu(a) u, o = h W_d[e]^T
//   shared    s[t] = the same SwiGLU with the shared weights, weight 1
//   combine   y[t] = s[t] + sum_{s kept} g[t,s] o[row(t,s)]
// and the backward of every step for an upstream gradient dY.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <thread>
#include <vector>

namespace {

int g_threads = 0;  // 0: std::thread::hardware_concurrency()

int n_workers() {
  int n = g_threads > 0 ? g_threads : static_cast<int>(std::thread::hardware_concurrency());
  return n > 0 ? n : 1;
}

// fn(i) for i in [0, n), split into contiguous chunks over the workers
void parallel_for(long long n, const std::function<void(long long)>& fn) {
  const int w = static_cast<int>(std::min<long long>(n_workers(), n));
  if (w <= 1) {
    for (long long i = 0; i < n; ++i) fn(i);
    return;
  }
  std::vector<std::thread> pool;
  const long long chunk = (n + w - 1) / w;
  for (int p = 0; p < w; ++p) {
    const long long lo = p * chunk, hi = std::min(n, lo + chunk);
    if (lo >= hi) break;
    pool.emplace_back([lo, hi, &fn] {
      for (long long i = lo; i < hi; ++i) fn(i);
    });
  }
  for (auto& t : pool) t.join();
}

double sigmoid(double a) { return 1.0 / (1.0 + std::exp(-a)); }

// out[i, j] = sum_c A[i, c] B[j, c]   (A [n, K], B [m, K], both row-major)
void matmul_abt(const double* A, const double* B, long long n, long long m, long long K, double* out) {
  parallel_for(n, [&](long long i) {
    for (long long j = 0; j < m; ++j) {
      double acc = 0.0;
      for (long long c = 0; c < K; ++c) acc += A[i * K + c] * B[j * K + c];
      out[i * m + j] = acc;
    }
  });
}

// out[i, j] = sum_c A[i, c] B[c, j]   (A [n, K], B [K, m])
void matmul_ab(const double* A, const double* B, long long n, long long m, long long K, double* out) {
  parallel_for(n, [&](long long i) {
    for (long long j = 0; j < m; ++j) out[i * m + j] = 0.0;
    for (long long c = 0; c < K; ++c) {
      const double a = A[i * K + c];
      for (long long j = 0; j < m; ++j) out[i * m + j] += a * B[c * m + j];
    }
  });
}

// out[i, j] = sum_r A[r, i] B[r, j]   (A [n_rows, m1], B [n_rows, m2]) -> [m1, m2]
void matmul_atb(const double* A, const double* B, long long n_rows, long long m1, long long m2, double* out) {
  parallel_for(m1, [&](long long i) {
    for (long long j = 0; j < m2; ++j) out[i * m2 + j] = 0.0;
    for (long long r = 0; r < n_rows; ++r) {
      const double a = A[r * m1 + i];
      for (long long j = 0; j < m2; ++j) out[i * m2 + j] += a * B[r * m2 + j];
    }
  });
}

// SwiGLU on n rows: a = x Wg^T, u = x Wu^T, h = silu(a) u, o = h Wd^T
void swiglu_fwd(const double* x, const double* Wg, const double* Wu, const double* Wd, long long n, int d, int H,
                double* a, double* u, double* h, double* o) {
  matmul_abt(x, Wg, n, H, d, a);
  matmul_abt(x, Wu, n, H, d, u);
  for (long long i = 0; i < n * H; ++i) h[i] = a[i] * sigmoid(a[i]) * u[i];
  matmul_abt(h, Wd, n, d, H, o);
}

// Backward of o = (silu(x Wg^T) u) Wd^T for upstream dO [n, d]:
// dh = dO Wd, dWd = dO^T h, da = dh u sig(a) (1 + a (1 - sig(a))),
// du = dh silu(a), dx = da Wg + du Wu, dWg = da^T x, dWu = du^T x
void swiglu_bwd(const double* x, const double* Wg, const double* Wu, const double* Wd, const double* a,
                const double* u, const double* h, const double* dO, long long n, int d, int H, double* dx,
                double* dWg, double* dWu, double* dWd) {
  std::vector<double> dh(n * H), da(n * H), du(n * H), tmp(n * d);
  matmul_ab(dO, Wd, n, H, d, dh.data());
  matmul_atb(dO, h, n, d, H, dWd);
  for (long long i = 0; i < n * H; ++i) {
    const double sg = sigmoid(a[i]);
    da[i] = dh[i] * u[i] * sg * (1.0 + a[i] * (1.0 - sg));
    du[i] = dh[i] * a[i] * sg;
  }
  matmul_ab(da.data(), Wg, n, d, H, dx);
  matmul_ab(du.data(), Wu, n, d, H, tmp.data());
  for (long long i = 0; i < n * d; ++i) dx[i] += tmp[i];
  matmul_atb(da.data(), x, n, H, d, dWg);
  matmul_atb(du.data(), x, n, H, d, dWu);
}

}  // namespace

extern "C" {

__attribute__((visibility("default"))) void orc_set_threads(int n) { g_threads = n; }
__attribute__((visibility("default"))) int orc_threads(void) { return n_workers(); }

// bf16 bit patterns -> fp64: the 16 bits are the high half of an IEEE binary32
// (sign, 8-bit exponent, 7-bit mantissa); every bf16 value is exact in fp64.
__attribute__((visibility("default"))) void orc_bf16_to_f64(const uint16_t* src, long long n, double* dst) {
  for (long long i = 0; i < n; ++i) {
    const uint32_t bits = static_cast<uint32_t>(src[i]) << 16;
    float f;
    std::memcpy(&f, &bits, sizeof(f));
    dst[i] = static_cast<double>(f);
  }
}

// Router logits: fp32 rounding of the fp64 product, then the fp32 bias add.
__attribute__((visibility("default"))) void orc_router_logits(const double* x, const double* W_r, const float* bias,
                                                              int T, int d, int E, float* logits) {
  std::vector<double> l(static_cast<size_t>(T) * E);
  matmul_abt(x, W_r, T, E, d, l.data());
  for (long long t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      float v = static_cast<float>(l[t * E + e]);
      if (bias) v = v + bias[e];
      logits[t * E + e] = v;
    }
}

// Top-k and gates from logits [T,E] given as fp64 values (fp32 logits passed
// exactly): expert e before e' iff l_e > l_e' or (l_e == l_e' and e < e').
__attribute__((visibility("default"))) void orc_route_topk(const double* logits, int T, int E, int k, int32_t* idx,
                                                           double* gates) {
  parallel_for(T, [&](long long t) {
    const double* l = logits + t * E;
    std::vector<int> order(E);
    for (int e = 0; e < E; ++e) order[e] = e;
    std::stable_sort(order.begin(), order.end(), [l](int p, int q) { return l[p] > l[q]; });
    const double m = l[order[0]];
    double den = 0.0;
    std::vector<double> ex(k);
    for (int s = 0; s < k; ++s) {
      const double v = std::exp(l[order[s]] - m);
      ex[s] = std::isnan(v) ? 0.0 : v;  // -inf - (-inf) only if every selected logit is -inf
      den += ex[s];
    }
    for (int s = 0; s < k; ++s) {
      idx[t * k + s] = order[s];
      gates[t * k + s] = ex[s] / den;
    }
  });
}

// Histogram, capacity, exclusive prefix sum, row maps.  Returns R.
__attribute__((visibility("default"))) long long orc_permute(const int32_t* idx, int T, int E, int k, int capacity,
                                                             int64_t* counts_raw, int64_t* counts, int64_t* offsets,
                                                             int64_t* rank, int64_t* row_of_slot,
                                                             int64_t* slot_of_row) {
  for (int e = 0; e < E; ++e) counts_raw[e] = 0;
  for (long long t = 0; t < T; ++t)  // token order: the rank is the count so far
    for (int s = 0; s < k; ++s) {
      const int e = idx[t * k + s];
      rank[t * k + s] = counts_raw[e]++;
    }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) {
    counts[e] = capacity > 0 ? std::min<int64_t>(counts_raw[e], capacity) : counts_raw[e];
    offsets[e + 1] = offsets[e] + counts[e];
  }
  for (long long i = 0; i < static_cast<long long>(T) * k; ++i) {
    const int e = idx[i];
    const bool kept = capacity <= 0 || rank[i] < capacity;
    row_of_slot[i] = kept ? offsets[e] + rank[i] : -1;
    if (kept) slot_of_row[row_of_slot[i]] = i;
  }
  return offsets[E];
}

// Whole forward.  Routing from logits_in (fp64 values, e.g. given fp32
// logits), else from the router (exact_router: logits kept in fp64, plus the
// bias; else fp32 as in orc_router_logits).  gates_in overrides the gates
// (finite differences), identity replaces every routed expert by o = x.
// Buffers are sized for the dropless maximum R = T*k rows.  Returns R.
__attribute__((visibility("default"))) long long orc_layer_forward(
    int T, int d, int E, int k, int H, int Hs, int capacity, const double* x, const double* W_r, const float* bias,
    const double* logits_in, int exact_router, const double* gates_in, int identity, const double* W_g,
    const double* W_u, const double* W_d, const double* Ws_g, const double* Ws_u, const double* Ws_d,
    double* logits, int32_t* idx, double* gates, int64_t* counts_raw, int64_t* counts, int64_t* offsets,
    int64_t* rank, int64_t* row_of_slot, int64_t* slot_of_row, double* x_perm, double* a, double* u, double* h,
    double* o, double* a_s, double* u_s, double* h_s, double* s_out, double* y) {
  const long long TE = static_cast<long long>(T) * E;
  if (logits_in) {
    for (long long i = 0; i < TE; ++i) logits[i] = logits_in[i];
  } else if (exact_router) {
    matmul_abt(x, W_r, T, E, d, logits);
    if (bias)
      for (long long t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) logits[t * E + e] += static_cast<double>(bias[e]);
  } else {
    std::vector<float> l32(TE);
    orc_router_logits(x, W_r, bias, T, d, E, l32.data());
    for (long long i = 0; i < TE; ++i) logits[i] = l32[i];
  }
  orc_route_topk(logits, T, E, k, idx, gates);
  if (gates_in)
    for (long long i = 0; i < static_cast<long long>(T) * k; ++i) gates[i] = gates_in[i];
  const long long R = orc_permute(idx, T, E, k, capacity, counts_raw, counts, offsets, rank, row_of_slot,
                                  slot_of_row);
  for (long long r = 0; r < R; ++r) {
    const long long t = slot_of_row[r] / k;
    std::memcpy(x_perm + r * d, x + t * d, sizeof(double) * d);
  }
  // routed experts, one at a time, each over its own rows
  for (int e = 0; e < E; ++e) {
    const long long r0 = offsets[e], n = offsets[e + 1] - offsets[e];
    if (n == 0) continue;
    if (identity) {
      std::memcpy(o + r0 * d, x_perm + r0 * d, sizeof(double) * n * d);
      continue;
    }
    const long long w = static_cast<long long>(e) * H * d;
    swiglu_fwd(x_perm + r0 * d, W_g + w, W_u + w, W_d + w, n, d, H, a + r0 * H, u + r0 * H, h + r0 * H, o + r0 * d);
  }
  // shared expert on every token
  if (Hs > 0) {
    swiglu_fwd(x, Ws_g, Ws_u, Ws_d, T, d, Hs, a_s, u_s, h_s, s_out);
  }
  // combine
  parallel_for(T, [&](long long t) {
    for (int c = 0; c < d; ++c) y[t * d + c] = Hs > 0 ? s_out[t * d + c] : 0.0;
    for (int s = 0; s < k; ++s) {
      const long long row = row_of_slot[t * k + s];
      if (row < 0) continue;
      const double g = gates[t * k + s];
      for (int c = 0; c < d; ++c) y[t * d + c] += g * o[row * d + c];
    }
  });
  return R;
}

// Whole backward for upstream dY [T,d], given the forward's results.
// learned: the router product's gradients dW_r and the router term of dx.
__attribute__((visibility("default"))) void orc_layer_backward(
    int T, int d, int E, int k, int H, int Hs, const double* x, const double* W_r, int learned, const double* W_g,
    const double* W_u, const double* W_d, const double* Ws_g, const double* Ws_u, const double* Ws_d,
    const double* dY, const int32_t* idx, const double* gates, const int64_t* offsets, const int64_t* row_of_slot,
    const double* x_perm, const double* a, const double* u, const double* h, const double* o, const double* a_s,
    const double* u_s, const double* h_s, double* dO, double* dgates, double* dx_perm, double* dW_g, double* dW_u,
    double* dW_d, double* dx_s, double* dWs_g, double* dWs_u, double* dWs_d, double* dlogits, double* dW_r,
    double* dx) {
  const long long R = offsets[E];
  // combine backward: dO[row] = g dY[t]; dgates = <dY[t], o[row]>, 0 if dropped
  parallel_for(T, [&](long long t) {
    for (int s = 0; s < k; ++s) {
      const long long row = row_of_slot[t * k + s];
      double dg = 0.0;
      if (row >= 0) {
        const double g = gates[t * k + s];
        for (int c = 0; c < d; ++c) {
          dO[row * d + c] = g * dY[t * d + c];
          dg += dY[t * d + c] * o[row * d + c];
        }
      }
      dgates[t * k + s] = dg;
    }
  });
  // experts
  const long long wsz = static_cast<long long>(H) * d;
  for (long long i = 0; i < static_cast<long long>(E) * wsz; ++i) {
    dW_g[i] = 0.0;
    dW_u[i] = 0.0;
    dW_d[i] = 0.0;
  }
  for (int e = 0; e < E; ++e) {
    const long long r0 = offsets[e], n = offsets[e + 1] - offsets[e];
    if (n == 0) continue;
    const long long w = e * wsz;
    swiglu_bwd(x_perm + r0 * d, W_g + w, W_u + w, W_d + w, a + r0 * H, u + r0 * H, h + r0 * H, dO + r0 * d, n, d,
               H, dx_perm + r0 * d, dW_g + w, dW_u + w, dW_d + w);
  }
  if (Hs > 0) swiglu_bwd(x, Ws_g, Ws_u, Ws_d, a_s, u_s, h_s, dY, T, d, Hs, dx_s, dWs_g, dWs_u, dWs_d);
  // router: softmax over the selection; dropped slots (dgates = 0) stay in it
  parallel_for(T, [&](long long t) {
    double sgd = 0.0;
    for (int s = 0; s < k; ++s) sgd += gates[t * k + s] * dgates[t * k + s];
    for (int e = 0; e < E; ++e) dlogits[t * E + e] = 0.0;
    for (int s = 0; s < k; ++s)
      dlogits[t * E + idx[t * k + s]] = gates[t * k + s] * (dgates[t * k + s] - sgd);
  });
  if (learned) matmul_atb(dlogits, x, T, E, d, dW_r);
  // unpermute reduce + shared + router term
  parallel_for(T, [&](long long t) {
    for (int c = 0; c < d; ++c) {
      double v = Hs > 0 ? dx_s[t * d + c] : 0.0;
      for (int s = 0; s < k; ++s) {
        const long long row = row_of_slot[t * k + s];
        if (row >= 0) v += dx_perm[row * d + c];
      }
      if (learned)
        for (int e = 0; e < E; ++e) v += dlogits[t * E + e] * W_r[static_cast<long long>(e) * d + c];
      dx[t * d + c] = v;
    }
  });
  (void)R;
}

}  // extern "C"
