// fab_oracle.cpp -- plain fp64 CPU oracle for the fused attention backward pass.
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct statement
// of what the GPU library computes.  Only the test suite, the smoke check and
// the benchmark's CPU-baseline leg may load it.  It shares no code, header,
// table or helper with the CUDA library, and the CUDA library never calls it.
//
// What it computes (sources, by page and section):
//  * Forward, per (batch b, query head h, query n): the "reference forward
//    attention in plain R" of the ggmlR test file test-flash-attn-back.R
//    (function attn_ref): scores s_m = scale * q.k_m, plus the additive mask
//    column mask[, n]; a row with no finite score is skipped (output 0);
//    otherwise e_m = exp(s_m - max finite s), non-finite scores give 0,
//    p = e / sum(e), out = sum_m p_m v_m.  The query head h reads key/value
//    head h / (H/Hkv) (contiguous groups, "hk <- (h - 1) %/% rk2 + 1").
//  * LSE: the log of the softmax denominator in the labml "Flash Attention"
//    page, section "Forward pass" (L_i = sum_j e^{S_ij}); stored as
//    max + log(sum exp(s - max)), and +inf for a row with no finite score.
//  * Backward: labml "Flash Attention", section "Backward pass":
//    dV_j = sum_i P_ij dO_i;  dP_ij = dO_i V_j^T;
//    dS_ij = P_ij dP_ij - P_ij sum_k P_ik dP_ik;  dQ_i = scale sum_j dS_ij K_j;
//    dK_j = scale sum_i dS_ij Q_i.  The per-row term sum_k P_ik dP_ik is the
//    D_i of the same section, computed here from its first (definitional)
//    form; oracle_di_rowdot computes its last form, dO_i . O_i.
//  * Packed result: the ggml_flash_attn_back constructor (PowerInfer ggml.c):
//    offs_q = 0, offs_k = PAD(elem_q*4, 16), offs_v = offs_k + PAD(elem_k*4,
//    16), end = offs_v + PAD(elem_v*4, 16); and the ggmlR packing test
//    ("the packed gradients occupy disjoint, in-bounds slices"): the whole
//    buffer is zeroed, then each slice written, so padding stays 0.
//
// Layouts are ggml ne order (ne[0] contiguous):
//   q [DK,N,H,B]   k [DK,M,Hkv,B]   v [DV,M,Hkv,B]
//   d, out [DV,H,N,B] (the forward output's permuted shape)
//   mask [M,N] (mask[m + M*n] is added to the score of query n, key m;
//               shared by all heads and batches)
//   lse, di [N,H,B]
// Causal (top-left): query n attends keys m <= n.
//
// Threads: work units are (b, hk) pairs.  A unit owns dK/dV of its key/value
// head and dQ/out/lse/di of the query heads in its group, so units write
// disjoint memory and need no locks.

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

struct Shape {
  int64_t B, H, Hkv, N, M, DK, DV;
};

struct Problem {
  Shape s;
  const double* q;
  const double* k;
  const double* v;
  const double* d;     // may be null for forward-only
  const double* mask;  // may be null
  int causal;
  double scale;
  // outputs (any may be null)
  double* out;
  double* lse;
  double* di;
  double* dq;
  double* dk;
  double* dv;
  // query rows [n_begin, n_end) are computed (all rows by default)
  int64_t n_begin;
  int64_t n_end;
};

inline int64_t at_q(const Shape& s, int64_t i, int64_t n, int64_t h, int64_t b) {
  return i + s.DK * (n + s.N * (h + s.H * b));
}
inline int64_t at_k(const Shape& s, int64_t i, int64_t m, int64_t hk, int64_t b) {
  return i + s.DK * (m + s.M * (hk + s.Hkv * b));
}
inline int64_t at_v(const Shape& s, int64_t i, int64_t m, int64_t hk, int64_t b) {
  return i + s.DV * (m + s.M * (hk + s.Hkv * b));
}
inline int64_t at_o(const Shape& s, int64_t i, int64_t h, int64_t n, int64_t b) {
  return i + s.DV * (h + s.H * (n + s.N * b));
}
inline int64_t at_row(const Shape& s, int64_t n, int64_t h, int64_t b) {
  return n + s.N * (h + s.H * b);
}

// One query row (b, h, n): forward, and when P.d is given, its backward
// contributions.  Scratch vectors have length M.
void one_row(const Problem& P, int64_t b, int64_t h, int64_t n, std::vector<double>& sc,
             std::vector<double>& p, std::vector<double>& dp) {
  const Shape& s = P.s;
  const int64_t hk = h / (s.H / s.Hkv);
  const double inf = std::numeric_limits<double>::infinity();

  // scores (attn_ref: s <- scale * q.k ; s <- s + mask[, n])
  bool any_finite = false;
  double mx = -inf;
  for (int64_t m = 0; m < s.M; ++m) {
    if (P.causal && m > n) {
      sc[m] = -inf;
      continue;
    }
    double dot = 0.0;
    for (int64_t i = 0; i < s.DK; ++i) dot += P.q[at_q(s, i, n, h, b)] * P.k[at_k(s, i, m, hk, b)];
    double x = P.scale * dot;
    if (P.mask) x += P.mask[m + s.M * n];
    sc[m] = x;
    if (std::isfinite(x)) {
      any_finite = true;
      if (x > mx) mx = x;
    }
  }

  if (!any_finite) {  // attn_ref: "if (all(!is.finite(s))) next" -> output row stays 0
    if (P.out)
      for (int64_t i = 0; i < s.DV; ++i) P.out[at_o(s, i, h, n, b)] = 0.0;
    if (P.lse) P.lse[at_row(s, n, h, b)] = inf;
    if (P.di) P.di[at_row(s, n, h, b)] = 0.0;
    if (P.dq)
      for (int64_t i = 0; i < s.DK; ++i) P.dq[at_q(s, i, n, h, b)] = 0.0;
    return;
  }

  // softmax with the max finite score subtracted; non-finite scores give 0
  double sum = 0.0;
  for (int64_t m = 0; m < s.M; ++m) {
    const double e = std::isfinite(sc[m]) ? std::exp(sc[m] - mx) : 0.0;
    p[m] = e;
    sum += e;
  }
  for (int64_t m = 0; m < s.M; ++m) p[m] /= sum;
  if (P.lse) P.lse[at_row(s, n, h, b)] = mx + std::log(sum);

  if (P.out) {
    for (int64_t i = 0; i < s.DV; ++i) P.out[at_o(s, i, h, n, b)] = 0.0;
    for (int64_t m = 0; m < s.M; ++m) {
      if (p[m] == 0.0) continue;
      for (int64_t i = 0; i < s.DV; ++i) P.out[at_o(s, i, h, n, b)] += p[m] * P.v[at_v(s, i, m, hk, b)];
    }
  }

  if (!P.d) return;

  // dP_m = dO_n . V_m ;  D_n = sum_m P_m dP_m
  double Dn = 0.0;
  for (int64_t m = 0; m < s.M; ++m) {
    if (p[m] == 0.0) {
      dp[m] = 0.0;
      continue;
    }
    double acc = 0.0;
    for (int64_t i = 0; i < s.DV; ++i) acc += P.d[at_o(s, i, h, n, b)] * P.v[at_v(s, i, m, hk, b)];
    dp[m] = acc;
    Dn += p[m] * acc;
  }
  if (P.di) P.di[at_row(s, n, h, b)] = Dn;

  // dS_m = P_m dP_m - P_m D_n, then the three gradient sums
  if (P.dq)
    for (int64_t i = 0; i < s.DK; ++i) P.dq[at_q(s, i, n, h, b)] = 0.0;
  for (int64_t m = 0; m < s.M; ++m) {
    if (p[m] == 0.0) continue;
    const double ds = p[m] * dp[m] - p[m] * Dn;
    if (P.dq)
      for (int64_t i = 0; i < s.DK; ++i)
        P.dq[at_q(s, i, n, h, b)] += P.scale * ds * P.k[at_k(s, i, m, hk, b)];
    if (P.dk)
      for (int64_t i = 0; i < s.DK; ++i)
        P.dk[at_k(s, i, m, hk, b)] += P.scale * ds * P.q[at_q(s, i, n, h, b)];
    if (P.dv)
      for (int64_t i = 0; i < s.DV; ++i) P.dv[at_v(s, i, m, hk, b)] += p[m] * P.d[at_o(s, i, h, n, b)];
  }
}

// A unit is (b, hk): every query head of the group and every query row.
void run_unit(const Problem& P, int64_t unit) {
  const Shape& s = P.s;
  const int64_t b = unit / s.Hkv, hk = unit % s.Hkv;
  const int64_t rk2 = s.H / s.Hkv;
  if (P.dk)
    for (int64_t m = 0; m < s.M; ++m)
      for (int64_t i = 0; i < s.DK; ++i) P.dk[at_k(s, i, m, hk, b)] = 0.0;
  if (P.dv)
    for (int64_t m = 0; m < s.M; ++m)
      for (int64_t i = 0; i < s.DV; ++i) P.dv[at_v(s, i, m, hk, b)] = 0.0;
  std::vector<double> sc(s.M), p(s.M), dp(s.M);
  for (int64_t h = hk * rk2; h < (hk + 1) * rk2; ++h)
    for (int64_t n = P.n_begin; n < P.n_end; ++n) one_row(P, b, h, n, sc, p, dp);
}

int check_shape(const int64_t* dims, Shape* s) {
  if (!dims) return 1;
  *s = Shape{dims[0], dims[1], dims[2], dims[3], dims[4], dims[5], dims[6]};
  if (s->B <= 0 || s->H <= 0 || s->Hkv <= 0 || s->N <= 0 || s->M <= 0 || s->DK <= 0 || s->DV <= 0)
    return 1;
  if (s->H % s->Hkv != 0) return 1;  // ne2 % kvne2 == 0 in the ggml constructor
  return 0;
}

void run_units(const Problem& P, const int64_t* units, int64_t n_units, int n_threads) {
  const int64_t total = P.s.B * P.s.Hkv;
  std::vector<int64_t> list;
  if (units && n_units > 0) {
    list.assign(units, units + n_units);
  } else {
    list.resize(total);
    for (int64_t u = 0; u < total; ++u) list[u] = u;
  }
  if (n_threads <= 0) n_threads = (int)std::thread::hardware_concurrency();
  if (n_threads <= 0) n_threads = 1;
  if ((int64_t)n_threads > (int64_t)list.size()) n_threads = (int)list.size();
  std::atomic<int64_t> next{0};
  auto worker = [&]() {
    for (;;) {
      const int64_t i = next.fetch_add(1);
      if (i >= (int64_t)list.size()) break;
      run_unit(P, list[i]);
    }
  };
  if (n_threads <= 1) {
    worker();
    return;
  }
  std::vector<std::thread> pool;
  for (int t = 0; t < n_threads; ++t) pool.emplace_back(worker);
  for (auto& t : pool) t.join();
}

inline int64_t pad16(int64_t bytes) { return (bytes + 15) / 16 * 16; }

}  // namespace

extern "C" {

// dims = {B, H, Hkv, N, M, DK, DV}.  Returns 0 on success, 1 on bad shape.
// Forward only: out [DV,H,N,B], lse [N,H,B] (either may be null).
int oracle_forward(const double* q, const double* k, const double* v, const double* mask, int causal,
                   double scale, const int64_t* dims, double* out, double* lse, int n_threads) {
  Shape s;
  if (check_shape(dims, &s)) return 1;
  Problem P{s, q, k, v, nullptr, mask, causal, scale, out, lse, nullptr, nullptr, nullptr, nullptr, 0, s.N};
  run_units(P, nullptr, 0, n_threads);
  return 0;
}

// Forward and analytic backward.  Every output pointer may be null.  When
// `units` is non-null, only those (b*Hkv + hk) units are computed; the rest of
// each output is left as the caller initialised it.  Only query rows
// [n_begin, n_end) are visited: their out/lse/di/dQ rows are exact, and dK/dV
// hold the contributions of those rows alone (exact for keys that no other
// query attends, e.g. keys >= n_begin under a causal mask when n_end = N).
int oracle_backward(const double* q, const double* k, const double* v, const double* d, const double* mask,
                    int causal, double scale, const int64_t* dims, double* dq, double* dk, double* dv,
                    double* out, double* lse, double* di, const int64_t* units, int64_t n_units,
                    int64_t n_begin, int64_t n_end, int n_threads) {
  Shape s;
  if (check_shape(dims, &s)) return 1;
  if (!d) return 1;
  for (int64_t i = 0; units && i < n_units; ++i)
    if (units[i] < 0 || units[i] >= s.B * s.Hkv) return 1;
  if (n_begin < 0 || n_end > s.N || n_begin > n_end) return 1;
  Problem P{s, q, k, v, d, mask, causal, scale, out, lse, di, dq, dk, dv, n_begin, n_end};
  run_units(P, units, n_units, n_threads);
  return 0;
}

// D_i = dO_i . O_i (the last form of D_i in the labml backward section), for
// every row of d and out [DV,H,N,B]; di is [N,H,B].
int oracle_di_rowdot(const double* d, const double* out, const int64_t* dims, double* di) {
  Shape s;
  if (check_shape(dims, &s)) return 1;
  for (int64_t b = 0; b < s.B; ++b)
    for (int64_t h = 0; h < s.H; ++h)
      for (int64_t n = 0; n < s.N; ++n) {
        double acc = 0.0;
        for (int64_t i = 0; i < s.DV; ++i) acc += d[at_o(s, i, h, n, b)] * out[at_o(s, i, h, n, b)];
        di[at_row(s, n, h, b)] = acc;
      }
  return 0;
}

// Byte offsets of the packed [dQ | dK | dV] f32 result (ggml constructor).
int oracle_packed_layout(const int64_t* dims, int64_t* off_k, int64_t* off_v, int64_t* end) {
  Shape s;
  if (check_shape(dims, &s)) return 1;
  const int64_t tsize = 4;  // GGML_TYPE_F32
  const int64_t elem_q = s.DK * s.N * s.H * s.B;
  const int64_t elem_k = s.DK * s.M * s.Hkv * s.B;
  const int64_t elem_v = s.DV * s.M * s.Hkv * s.B;
  const int64_t offs_q = 0;
  const int64_t offs_k = offs_q + pad16(elem_q * tsize);
  const int64_t offs_v = offs_k + pad16(elem_k * tsize);
  *off_k = offs_k;
  *off_v = offs_v;
  *end = offs_v + pad16(elem_v * tsize);
  return 0;
}

// Packs the three gradients into `packed` (end/4 doubles): zero everything,
// then write each slice at its offset.
int oracle_pack(const int64_t* dims, const double* dq, const double* dk, const double* dv, double* packed) {
  int64_t off_k, off_v, end;
  if (oracle_packed_layout(dims, &off_k, &off_v, &end)) return 1;
  const Shape s{dims[0], dims[1], dims[2], dims[3], dims[4], dims[5], dims[6]};
  const int64_t nq = s.DK * s.N * s.H * s.B, nk = s.DK * s.M * s.Hkv * s.B, nv = s.DV * s.M * s.Hkv * s.B;
  for (int64_t i = 0; i < end / 4; ++i) packed[i] = 0.0;
  for (int64_t i = 0; i < nq; ++i) packed[i] = dq[i];
  for (int64_t i = 0; i < nk; ++i) packed[off_k / 4 + i] = dk[i];
  for (int64_t i = 0; i < nv; ++i) packed[off_v / 4 + i] = dv[i];
  return 0;
}

}  // extern "C"
