// gdn_oracle.cpp -- plain fp64 CPU oracle of the Gated DeltaNet (GDN) token mixer.
//
// TEST INFRASTRUCTURE ONLY.  This file is the independent reference that the CUDA
// library is checked against.  Only the test suite, the smoke check and the CPU
// baseline leg of the benchmark load it.  It shares no code, header, table or
// constant with the CUDA library, and it never calls into it.
//
// What is computed (one GDN layer's token mixer, per token, in this order):
//   a2  causal depthwise conv over the raw [Q|K|V] channels, then SiLU
//       (layer_struct.rs, Qwen3SsmLayer fields conv1d_k / conv1d_l2norm_f32_k);
//   a3  per-key-head L2 norm of q and k, q additionally scaled by q_scale
//       (layer_struct.rs, conv1d_l2norm_f32_k and l2_norm_k);
//   a1  gates: alpha = exp(-exp(A_log) * softplus(a + dt_bias)), beta = sigmoid(b)
//       (layer_struct.rs, ba_gates_k / compute_gdn_gates_k);
//   a4  gated delta rule on a per-value-head state S (d_v x d_k):
//           S_t = alpha_t * S_{t-1} * (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
//           o_t = S_t q_t
//       (layer_struct.rs, gdn_f32_k);
//   a7  Z-gated RMSNorm over d_v: y = o / sqrt(mean(o^2) + eps) * w * SiLU(z)
//       (layer_struct.rs, gated_rms_norm_f32_k); with OrcDims::norm_gate = 1 the gate is
//       sigmoid(z) instead of SiLU(z), the reading taken of the gdn_norm_sigmoid models
//       (layer_struct.rs, the gated_rms_norm_f32_strided_k field), which the pages name
//       as a model flag without printing the formula.
// A separate routine, orc_chunked, writes out the chunked (WY / UT-transform) form of
// the same recurrence (layer_struct.rs, the FLA chunked prefill fields
// gdn_prefill_fla_recompute_wu_k, gdn_prefill_fla_chunk_delta_h_k,
// gdn_prefill_fla_chunk_fwd_o_k).  It is used only to check the algebra that a chunked
// kernel relies on against the token loop.
//
// Storage conventions (readings of the pages, listed in the design notes):
//   * a row of raw QKV holds [Q | K | V]: Q = H_k heads x d_k, K = H_k x d_k,
//     V = H_v x d_v, each head's channels contiguous (layer_struct.rs, the
//     Qwen3SsmLayer doc: the QKVZ projection is turned into [Q | K | V | Z]);
//   * value head h reads key head h / (H_v / H_k);
//   * the state of one value head is stored as H[i][j] = S[j][i], i over d_k and
//     j over d_v, i.e. h_state_bytes = nv * kd * vd values in [H_v][d_k][d_v] order
//     (layer_struct.rs, the h_state_bytes / conv_state_bytes comment);
//   * the conv state of a channel holds its last d_conv raw inputs, oldest first;
//     w[c][d_conv-1] multiplies the newest input.
//
// Everything is double precision.  No blocking, fusion or reordering beyond what the
// definitions above state.  One option changes storage, not arithmetic: with
// OrcDims::h_fp16 set, the state is kept in a half-width pool (layer_struct.rs, the FP16
// h-state variants gdn_f16_norm_k and gdn_wyn_f16_table_k): after every token the stored
// state is rounded to the nearest IEEE binary16 value, while o is formed from the
// unrounded update.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// softplus(x) = log(1 + exp(x)), evaluated as max(x, 0) + log1p(exp(-|x|)) so that
// large |x| neither overflows nor loses the small term.
double softplus(double x) { return (x > 0.0 ? x : 0.0) + std::log1p(std::exp(-std::fabs(x))); }

double sigmoid(double x) { return 1.0 / (1.0 + std::exp(-x)); }

double silu(double x) { return x * sigmoid(x); }

}  // namespace

extern "C" {

// Shape and scalar parameters of one GDN layer.  Mirrors nothing in the CUDA library.
struct OrcDims {
  int32_t n_k_heads;  // H_k
  int32_t n_v_heads;  // H_v (a multiple of H_k)
  int32_t d_k;
  int32_t d_v;
  int32_t d_conv;     // conv width W
  double q_scale;     // multiplies q after its L2 norm
  double l2_eps;      // q <- q / sqrt(sum q^2 + l2_eps)
  double norm_eps;    // gated RMSNorm epsilon
  int32_t h_fp16;     // 1: the state is stored as binary16 after every token
  int32_t norm_gate;  // 0: y gated by SiLU(z); 1: gated by sigmoid(z)
};

// Rounds x to the nearest IEEE 754 binary16 value, ties to even, returned as a double.
// binary16 has an 11-bit significand: numbers in [2^(e-1), 2^e) are spaced 2^(e-11) for
// e - 1 >= -14, and below 2^-14 (subnormals) the spacing stays 2^-24.  The largest finite
// value is 65504; anything that rounds above it is infinite.
double orc_round_fp16(double x) {
  if (!std::isfinite(x) || x == 0.0) return x;
  const double ax = std::fabs(x);
  int e = 0;
  std::frexp(ax, &e);  // ax = f 2^e, f in [0.5, 1)
  const int ex = (e - 11 < -24) ? -24 : e - 11;
  const double step = std::ldexp(1.0, ex);
  double r = std::nearbyint(ax / step) * step;  // the default mode: nearest, ties to even
  if (r > 65504.0) r = INFINITY;
  return std::copysign(r, x);
}

int32_t orc_conv_dim(const OrcDims* d) {
  return 2 * d->n_k_heads * d->d_k + d->n_v_heads * d->d_v;
}

double orc_softplus(double x) { return softplus(x); }

// a1: gates for T tokens and H_v heads.  a, b: [T][H_v]; A_log, dt_bias: [H_v].
void orc_gates(int32_t T, int32_t n_v_heads, const double* a, const double* b,
               const double* A_log, const double* dt_bias, double* alpha, double* beta) {
  for (int32_t t = 0; t < T; ++t) {
    for (int32_t h = 0; h < n_v_heads; ++h) {
      const double x = a[(int64_t)t * n_v_heads + h] + dt_bias[h];
      alpha[(int64_t)t * n_v_heads + h] = std::exp(-std::exp(A_log[h]) * softplus(x));
      beta[(int64_t)t * n_v_heads + h] = sigmoid(b[(int64_t)t * n_v_heads + h]);
    }
  }
}

// a2: causal depthwise conv + SiLU over T tokens of C channels.
//   w: [C][W]; state: [C][W] in/out (last W raw inputs, oldest first);
//   x: [T][C] raw inputs; out: [T][C] = SiLU(sum_j w[c][j] * window[j]);
//   state_snap (nullable): [T][C][W], the state after each token.
void orc_conv(int32_t T, int32_t C, int32_t W, const double* w, double* state,
              const double* x, double* out, double* state_snap) {
  for (int32_t t = 0; t < T; ++t) {
    for (int32_t c = 0; c < C; ++c) {
      double* s = state + (int64_t)c * W;
      // The oldest input leaves, the new one enters at the end.
      for (int32_t j = 0; j + 1 < W; ++j) s[j] = s[j + 1];
      s[W - 1] = x[(int64_t)t * C + c];
      double acc = 0.0;
      for (int32_t j = 0; j < W; ++j) acc += w[(int64_t)c * W + j] * s[j];
      out[(int64_t)t * C + c] = silu(acc);
    }
    if (state_snap)
      std::memcpy(state_snap + (int64_t)t * C * W, state, sizeof(double) * (size_t)C * W);
  }
}

// a3: split conv outputs into q, k, v and L2-normalise q and k per key head.
//   xc: [T][conv_dim]; qn, kn: [T][H_k][d_k]; v: [T][H_v][d_v].
void orc_l2norm_split(const OrcDims* d, int32_t T, const double* xc, double* qn, double* kn,
                      double* v) {
  const int32_t Hk = d->n_k_heads, dk = d->d_k, Hv = d->n_v_heads, dv = d->d_v;
  const int32_t C = orc_conv_dim(d);
  for (int32_t t = 0; t < T; ++t) {
    const double* row = xc + (int64_t)t * C;
    for (int32_t h = 0; h < Hk; ++h) {
      const double* q = row + h * dk;
      const double* k = row + Hk * dk + h * dk;
      double sq = 0.0, sk = 0.0;
      for (int32_t i = 0; i < dk; ++i) {
        sq += q[i] * q[i];
        sk += k[i] * k[i];
      }
      const double rq = d->q_scale / std::sqrt(sq + d->l2_eps);
      const double rk = 1.0 / std::sqrt(sk + d->l2_eps);
      for (int32_t i = 0; i < dk; ++i) {
        qn[((int64_t)t * Hk + h) * dk + i] = q[i] * rq;
        kn[((int64_t)t * Hk + h) * dk + i] = k[i] * rk;
      }
    }
    for (int32_t h = 0; h < Hv; ++h)
      for (int32_t j = 0; j < dv; ++j)
        v[((int64_t)t * Hv + h) * dv + j] = row[2 * Hk * dk + h * dv + j];
  }
}

// a4 for one token and one value head, on H[i][j] = S[j][i]:
//   u = S k;  S <- alpha * (S - beta * u k^T) + beta * v k^T;  o = S q.
// The middle line is S (I - beta k k^T) expanded by distributivity.
void orc_delta_step(int32_t dk, int32_t dv, double* H, const double* q, const double* k,
                    const double* v, double alpha, double beta, double* o) {
  std::vector<double> u(dv, 0.0);
  for (int32_t j = 0; j < dv; ++j) {
    double acc = 0.0;
    for (int32_t i = 0; i < dk; ++i) acc += H[(int64_t)i * dv + j] * k[i];
    u[j] = acc;
  }
  for (int32_t i = 0; i < dk; ++i)
    for (int32_t j = 0; j < dv; ++j) {
      double& s = H[(int64_t)i * dv + j];
      s = alpha * (s - beta * u[j] * k[i]) + beta * v[j] * k[i];
    }
  for (int32_t j = 0; j < dv; ++j) {
    double acc = 0.0;
    for (int32_t i = 0; i < dk; ++i) acc += H[(int64_t)i * dv + j] * q[i];
    o[j] = acc;
  }
}

// a4 over T tokens for all value heads of one sequence.
//   qn, kn: [T][H_k][d_k]; v: [T][H_v][d_v]; alpha, beta: [T][H_v];
//   H: [H_v][d_k][d_v] in/out; o: [T][H_v][d_v];
//   H_snap (nullable): [T][H_v][d_k][d_v], the state after each token.
// Value heads are independent, so they may run on separate threads.
void orc_recurrence(const OrcDims* d, int32_t T, const double* qn, const double* kn,
                    const double* v, const double* alpha, const double* beta, double* H,
                    double* o, double* H_snap) {
  const int32_t Hk = d->n_k_heads, Hv = d->n_v_heads, dk = d->d_k, dv = d->d_v;
  const int32_t G = Hv / Hk;
  const int64_t hsz = (int64_t)dk * dv;
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t h = 0; h < Hv; ++h) {
    const int32_t kh = h / G;
    double* Hh = H + h * hsz;
    for (int32_t t = 0; t < T; ++t) {
      orc_delta_step(dk, dv, Hh, qn + ((int64_t)t * Hk + kh) * dk, kn + ((int64_t)t * Hk + kh) * dk,
                     v + ((int64_t)t * Hv + h) * dv, alpha[(int64_t)t * Hv + h],
                     beta[(int64_t)t * Hv + h], o + ((int64_t)t * Hv + h) * dv);
      if (d->h_fp16)
        for (int64_t e = 0; e < hsz; ++e) Hh[e] = orc_round_fp16(Hh[e]);
      if (H_snap) std::memcpy(H_snap + ((int64_t)t * Hv + h) * hsz, Hh, sizeof(double) * hsz);
    }
  }
}

// a7: Z-gated RMSNorm.  o: [T][H_v][d_v]; z: [T][H_v*d_v]; w: [d_v]; y: [T][H_v*d_v].
// gate 0 multiplies by SiLU(z), gate 1 by sigmoid(z).
void orc_gated_rmsnorm(int32_t T, int32_t n_v_heads, int32_t dv, const double* o,
                       const double* z, const double* w, double eps, int32_t gate, double* y) {
  for (int64_t r = 0; r < (int64_t)T * n_v_heads; ++r) {
    const double* orow = o + r * dv;
    double ss = 0.0;
    for (int32_t j = 0; j < dv; ++j) ss += orow[j] * orow[j];
    const double inv = 1.0 / std::sqrt(ss / dv + eps);
    for (int32_t j = 0; j < dv; ++j) {
      const double zj = z[r * dv + j];
      y[r * dv + j] = orow[j] * inv * w[j] * (gate ? sigmoid(zj) : silu(zj));
    }
  }
}

// The whole mixer for T consecutive tokens of ONE sequence: a2 -> a3 -> a1 -> a4 -> a7.
//   qkv: [T][conv_dim] raw; z: [T][H_v*d_v]; a, b: [T][H_v];
//   conv_w: [conv_dim][W]; A_log, dt_bias: [H_v]; norm_w: [d_v];
//   conv_state: [conv_dim][W] in/out; H: [H_v][d_k][d_v] in/out;
//   y: [T][H_v*d_v]; o (nullable): [T][H_v][d_v] core output before the norm;
//   H_snap (nullable): [T][H_v][d_k][d_v]; conv_snap (nullable): [T][conv_dim][W].
void orc_mixer(const OrcDims* d, int32_t T, const double* qkv, const double* z, const double* a,
               const double* b, const double* conv_w, const double* A_log,
               const double* dt_bias, const double* norm_w, double* conv_state, double* H,
               double* y, double* o, double* H_snap, double* conv_snap) {
  if (T <= 0) return;
  const int32_t Hk = d->n_k_heads, Hv = d->n_v_heads, dk = d->d_k, dv = d->d_v, W = d->d_conv;
  const int32_t C = orc_conv_dim(d);
  std::vector<double> xc((size_t)T * C), qn((size_t)T * Hk * dk), kn((size_t)T * Hk * dk),
      v((size_t)T * Hv * dv), alpha((size_t)T * Hv), beta((size_t)T * Hv), ob;
  double* out_o = o;
  if (!out_o) {
    ob.resize((size_t)T * Hv * dv);
    out_o = ob.data();
  }
  orc_conv(T, C, W, conv_w, conv_state, qkv, xc.data(), conv_snap);
  orc_l2norm_split(d, T, xc.data(), qn.data(), kn.data(), v.data());
  orc_gates(T, Hv, a, b, A_log, dt_bias, alpha.data(), beta.data());
  orc_recurrence(d, T, qn.data(), kn.data(), v.data(), alpha.data(), beta.data(), H, out_o,
                 H_snap);
  orc_gated_rmsnorm(T, Hv, dv, out_o, z, norm_w, d->norm_eps, d->norm_gate, y);
}

// Rounds a double to the nearest bfloat16 value (ties to even), returned as double.
// Used only by the chunked form's optional operand-rounding emulation.
static double round_bf16(double x) {
  float f = (float)x;
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) return (double)f;  // inf / nan unchanged
  u = u + 0x7fffu + ((u >> 16) & 1u);
  u &= 0xffff0000u;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// The chunked form of a4, chunk length Cn, for all value heads of one sequence.  Within
// a chunk (local rows r, s = 0..L-1, L <= Cn), with g_r = sum_{s<=r} log(alpha_s):
//   A    = strict_lower( beta_r (k_r . k_s) exp(g_r - g_s) )
//   Tm   = (I + A)^{-1}                      (forward substitution)
//   Wm   = Tm diag(beta exp(g)) K,   Um = Tm diag(beta) V
//   Dl   = Um - Wm H0                         (H0 = S0^T, [d_k][d_v])
//   O    = diag(exp(g)) Q H0 + (lower_incl(Q K^T exp(g_r - g_s))) Dl
//   H_L  = exp(g_{L-1}) H0 + (diag(exp(g_{L-1} - g)) K)^T Dl
// Every decay ratio is formed as exp(g_r - g_s) with r >= s, never as a quotient.
// round_operands != 0 rounds both operands of every matrix product to bf16 first.
void orc_chunked(const OrcDims* d, int32_t T, int32_t Cn, const double* qn, const double* kn,
                 const double* v, const double* alpha, const double* beta, double* H, double* o,
                 int32_t round_operands) {
  const int32_t Hk = d->n_k_heads, Hv = d->n_v_heads, dk = d->d_k, dv = d->d_v;
  const int32_t G = Hv / Hk;
  auto rnd = [&](double x) { return round_operands ? round_bf16(x) : x; };
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t h = 0; h < Hv; ++h) {
    const int32_t kh = h / G;
    double* H0 = H + (int64_t)h * dk * dv;
    std::vector<double> g(Cn), A((size_t)Cn * Cn), Tm((size_t)Cn * Cn), Wm((size_t)Cn * dk),
        Um((size_t)Cn * dv), Dl((size_t)Cn * dv), Hn((size_t)dk * dv);
    for (int32_t t0 = 0; t0 < T; t0 += Cn) {
      const int32_t L = (T - t0 < Cn) ? (T - t0) : Cn;
      auto K = [&](int32_t r, int32_t i) { return kn[((int64_t)(t0 + r) * Hk + kh) * dk + i]; };
      auto Q = [&](int32_t r, int32_t i) { return qn[((int64_t)(t0 + r) * Hk + kh) * dk + i]; };
      auto V = [&](int32_t r, int32_t j) { return v[((int64_t)(t0 + r) * Hv + h) * dv + j]; };
      auto al = [&](int32_t r) { return alpha[(int64_t)(t0 + r) * Hv + h]; };
      auto be = [&](int32_t r) { return beta[(int64_t)(t0 + r) * Hv + h]; };
      double acc = 0.0;
      for (int32_t r = 0; r < L; ++r) {
        acc += std::log(al(r));
        g[r] = acc;
      }
      // A (strictly lower).
      for (int32_t r = 0; r < L; ++r)
        for (int32_t s = 0; s < L; ++s) {
          double val = 0.0;
          if (s < r) {
            double kk = 0.0;
            for (int32_t i = 0; i < dk; ++i) kk += rnd(K(r, i)) * rnd(K(s, i));
            val = be(r) * kk * std::exp(g[r] - g[s]);
          }
          A[(size_t)r * Cn + s] = val;
        }
      // Tm = (I + A)^{-1}: solve (I + A) X = I column by column, forward substitution.
      for (int32_t c = 0; c < L; ++c)
        for (int32_t r = 0; r < L; ++r) {
          double val = (r == c) ? 1.0 : 0.0;
          for (int32_t s = 0; s < r; ++s) val -= A[(size_t)r * Cn + s] * Tm[(size_t)s * Cn + c];
          Tm[(size_t)r * Cn + c] = val;
        }
      // Wm, Um.
      for (int32_t r = 0; r < L; ++r) {
        for (int32_t i = 0; i < dk; ++i) {
          double sacc = 0.0;
          for (int32_t s = 0; s < L; ++s)
            sacc += rnd(Tm[(size_t)r * Cn + s]) * rnd(be(s) * std::exp(g[s]) * K(s, i));
          Wm[(size_t)r * dk + i] = sacc;
        }
        for (int32_t j = 0; j < dv; ++j) {
          double sacc = 0.0;
          for (int32_t s = 0; s < L; ++s)
            sacc += rnd(Tm[(size_t)r * Cn + s]) * rnd(be(s) * V(s, j));
          Um[(size_t)r * dv + j] = sacc;
        }
      }
      // Dl = Um - Wm H0.
      for (int32_t r = 0; r < L; ++r)
        for (int32_t j = 0; j < dv; ++j) {
          double sacc = 0.0;
          for (int32_t i = 0; i < dk; ++i) sacc += rnd(Wm[(size_t)r * dk + i]) * rnd(H0[(int64_t)i * dv + j]);
          Dl[(size_t)r * dv + j] = Um[(size_t)r * dv + j] - sacc;
        }
      // O.
      for (int32_t r = 0; r < L; ++r) {
        std::vector<double> P(L, 0.0);
        for (int32_t s = 0; s <= r; ++s) {
          double qk = 0.0;
          for (int32_t i = 0; i < dk; ++i) qk += rnd(Q(r, i)) * rnd(K(s, i));
          P[s] = qk * std::exp(g[r] - g[s]);
        }
        for (int32_t j = 0; j < dv; ++j) {
          double qh = 0.0;
          for (int32_t i = 0; i < dk; ++i) qh += rnd(Q(r, i)) * rnd(H0[(int64_t)i * dv + j]);
          double pd = 0.0;
          for (int32_t s = 0; s <= r; ++s) pd += rnd(P[s]) * rnd(Dl[(size_t)s * dv + j]);
          o[((int64_t)(t0 + r) * Hv + h) * dv + j] = std::exp(g[r]) * qh + pd;
        }
      }
      // H at the end of the chunk.
      const double gl = g[L - 1];
      for (int32_t i = 0; i < dk; ++i)
        for (int32_t j = 0; j < dv; ++j) {
          double sacc = 0.0;
          for (int32_t s = 0; s < L; ++s)
            sacc += rnd(std::exp(gl - g[s]) * K(s, i)) * rnd(Dl[(size_t)s * dv + j]);
          Hn[(size_t)i * dv + j] = std::exp(gl) * H0[(int64_t)i * dv + j] + sacc;
        }
      std::memcpy(H0, Hn.data(), sizeof(double) * (size_t)dk * dv);
    }
  }
}

// Several independent sequences through orc_mixer, one thread per sequence.  Every
// pointer is an array of n per-sequence pointers; T[i] is sequence i's token count.
// o, H_snap and conv_snap may be NULL (the whole array) or hold NULL entries.
void orc_mixer_batch(const OrcDims* d, int32_t n, const int32_t* T, const double* const* qkv,
                     const double* const* z, const double* const* a, const double* const* b,
                     const double* conv_w, const double* A_log, const double* dt_bias,
                     const double* norm_w, double* const* conv_state, double* const* H,
                     double* const* y, double* const* o, double* const* H_snap,
                     double* const* conv_snap) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t i = 0; i < n; ++i)
    orc_mixer(d, T[i], qkv[i], z[i], a[i], b[i], conv_w, A_log, dt_bias, norm_w, conv_state[i],
              H[i], y[i], o ? o[i] : nullptr, H_snap ? H_snap[i] : nullptr,
              conv_snap ? conv_snap[i] : nullptr);
}

int32_t orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

// Threads the batch routine uses from now on (n >= 1); no effect without OpenMP.
void orc_set_threads(int32_t n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

}  // extern "C"
