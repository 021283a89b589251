// Plain CPU oracle for the speculative-decoding verification sampler.
//
// TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
// and the benchmark's CPU-baseline leg may build, load or call this file.  It
// shares no code, header, table or constant with the CUDA library: it is a
// slow, double-precision restatement of the rule, written to be checked by eye
// against the pages.
//
// Sources (page title, section):
//   [SD]  "Decodificación Especulativa y EAGLE" (Phase 10 - Lesson 25),
//         sections "El Concepto", "La Regla de Exactitud", "Caso codicioso",
//         "Aceleración Esperada".
//   [SON] "Accelerating Sonar through speculation", section
//         "Decodificación especulativa" (n drafted -> at most n+1 emitted).
//
// Readings of points the pages leave open (the same list is kept in the
// design notes):
//   * u_t = uniforms[b,t] drives the accept test at position t; the bonus draw
//     (every draft accepted) uses uniforms[b,n_b]; the replacement draw at a
//     rejected position uses uniforms_resample[b].  One final draw per request.
//   * The accept test is the strict "u < p(x)/q(x)", evaluated as
//     log u + log q(x) < log p(x).  q(x)=0 with p(x)>0 accepts; p(x)=0 rejects.
//   * T = 0 selects the greedy rule on the raw target logits; the draft logits
//     are not read.  The same T divides both target and draft logits.
//   * argmax ties resolve to the lowest index.
//   * Inverse CDF: the token is the smallest i with w_i > 0 and C_i > u*W,
//     C_i = w_0 + ... + w_i.  If rounding leaves no such i, the last i with
//     w_i > 0 is taken.  A zero-weight token is never emitted.
//   * If the residual mass W is exactly 0 at a rejected position (possible only
//     through rounding), the replacement is drawn from p itself with the same
//     uniform.
//   * Rows after a request's draft length are never read.
//   * out_tokens holds the j accepted drafts, then the final token, then -1.
//
// Everything is computed in IEEE double.  bf16 logits are widened exactly.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

constexpr int kF32 = 0;
constexpr int kBF16 = 1;

// near-tie / condition flags reported per request
constexpr int kTieAccept = 1;       // |u - p/q| < 1e-4 at an evaluated position
constexpr int kTieCdf = 2;          // u*W within 1e-4*W of an edge of the chosen CDF bucket
constexpr int kPrecisionBand = 4;   // u*W within kEdgeAbs of such an edge, but not within 1e-4*W
constexpr int kResFallback = 8;     // residual mass exactly 0: drawn from p instead
constexpr int kBadInput = 16;       // request rejected as invalid

constexpr double kTieBand = 1e-4;
// Absolute floor of the CDF-edge band, in units of probability mass.  If
// every p_i and q_i carries a relative error of at most 1e-5 (the tolerance
// fixed for normalised probabilities computed in fp32), a cumulative edge
// C_i = sum_{k<=i} (p_k - q_k)+ and the draw target u*W move relative to one
// another by at most 1e-5 * sum_k (p_k + q_k) = 2e-5.
constexpr double kEdgeAbs = 2e-5;

double widen(const void* base, int dtype, size_t idx) {
  if (dtype == kF32) return static_cast<double>(static_cast<const float*>(base)[idx]);
  uint32_t bits = static_cast<uint32_t>(static_cast<const uint16_t*>(base)[idx]) << 16;
  float f;
  std::memcpy(&f, &bits, sizeof f);
  return static_cast<double>(f);
}

// One row of V logits, widened to double.
void load_row(const void* base, int dtype, size_t row, int V, std::vector<double>& z) {
  z.resize(V);
  const size_t off = row * static_cast<size_t>(V);
  for (int i = 0; i < V; ++i) z[i] = widen(base, dtype, off + i);
}

// Neumaier's compensated summation (Neumaier 1974), used for every long sum.
struct CompSum {
  double s = 0.0, c = 0.0;
  void add(double x) {
    double t = s + x;
    if (std::fabs(s) >= std::fabs(x)) c += (s - t) + x; else c += (x - t) + s;
    s = t;
  }
  double value() const { return s + c; }
};

// Temperature softmax of one row: p_i = exp((z_i - zmax)/T) / S,
// S = sum_i exp((z_i - zmax)/T).  Returns false for a row with no finite
// maximum (all -inf, +inf or NaN): the distribution is undefined there.
bool softmax_T(const std::vector<double>& z, double T, std::vector<double>& p,
               double& zmax, double& S) {
  const int V = static_cast<int>(z.size());
  zmax = -std::numeric_limits<double>::infinity();
  for (int i = 0; i < V; ++i) if (z[i] > zmax) zmax = z[i];
  if (!std::isfinite(zmax)) return false;
  p.resize(V);
  CompSum acc;
  for (int i = 0; i < V; ++i) {
    p[i] = std::exp((z[i] - zmax) / T);
    acc.add(p[i]);
  }
  S = acc.value();
  for (int i = 0; i < V; ++i) p[i] /= S;
  return true;
}

// Greedy rule: index of the largest raw logit, lowest index on ties.
int argmax_lowest(const std::vector<double>& z) {
  int best = 0;
  for (int i = 1; i < static_cast<int>(z.size()); ++i)
    if (z[i] > z[best]) best = i;
  return best;
}

// Near-tie class of a draw whose target u*W fell in the bucket [lo, hi):
// kTieCdf when an edge with a bucket beyond it lies within 1e-4*W of the
// target, kPrecisionBand when one lies within kEdgeAbs only, else 0.  The
// edge below the first positive weight (0) and above the last (W) have no
// bucket beyond them, so no rounding can move the draw across them.  W = 1
// (a draw from p) makes the relative band the wider one.
int edge_flag(double target, double lo, double hi, double W, bool lo_inner, bool hi_inner) {
  double d = std::numeric_limits<double>::infinity();
  if (lo_inner) d = std::min(d, std::fabs(target - lo));
  if (hi_inner) d = std::min(d, std::fabs(target - hi));
  if (d < kTieBand * W) return kTieCdf;
  if (d < kEdgeAbs) return kPrecisionBand;
  return 0;
}

// Inverse-CDF draw from non-negative weights w with total W and uniform u:
// the smallest i with w_i > 0 and w_0 + ... + w_i > u*W.  *flag gets the
// near-tie class of the chosen bucket (edge_flag).  Returns -1 only when
// every weight is zero.  W must be the same compensated sum of w the loop
// forms, so for u < 1 the target u*W < W is always passed; the "last
// positive weight" return below is a guard for rounding the loop cannot
// reach with such a W.
int inverse_cdf(const std::vector<double>& w, double W, double u, int* flag) {
  const double target = u * W;
  int first_pos = -1, final_pos = -1;
  for (int i = 0; i < static_cast<int>(w.size()); ++i) {
    if (w[i] > 0.0) {
      if (first_pos < 0) first_pos = i;
      final_pos = i;
    }
  }
  CompSum cum;
  int last_pos = -1;
  double last_lo = 0.0, last_hi = 0.0;
  for (int i = 0; i < static_cast<int>(w.size()); ++i) {
    if (!(w[i] > 0.0)) continue;
    const double lo = cum.value();
    cum.add(w[i]);
    const double hi = cum.value();
    last_pos = i; last_lo = lo; last_hi = hi;
    if (hi > target) {
      *flag = edge_flag(target, lo, hi, W, i != first_pos, i != final_pos);
      return i;
    }
  }
  if (last_pos >= 0)
    *flag = edge_flag(target, last_lo, last_hi, W, last_pos != first_pos, false);
  return last_pos;
}

double comp_total(const std::vector<double>& w) {
  CompSum acc;
  for (double x : w) acc.add(x);
  return acc.value();
}

struct Args {
  const void* target;
  const void* draft;
  int dtype;
  const int32_t* draft_tokens;
  const int32_t* draft_len;
  const float* temperature;
  const float* uniforms;
  const float* uniforms_resample;
  int B, K, V;
  int32_t* accepted_len;
  int32_t* out_tokens;
  int32_t* flags;
  double* row_info;   // [B, K+1, kRowInfo] or null
};

constexpr int kRowInfo = 10;

bool row_has_finite_max(const void* base, int dtype, size_t row, int V) {
  double m = -std::numeric_limits<double>::infinity();
  const size_t off = row * static_cast<size_t>(V);
  for (int i = 0; i < V; ++i) {
    const double z = widen(base, dtype, off + i);
    if (z > m) m = z;
  }
  return std::isfinite(m);
}

// Checks the per-request inputs the rule depends on; fills n on success.
bool request_valid(const Args& a, int b, int* n_out) {
  const int n = a.draft_len ? a.draft_len[b] : a.K;
  if (n < 1 || n > a.K) return false;
  const double T = a.temperature[b];
  if (!(T >= 0.0) || !std::isfinite(T)) return false;
  if (T > 0.0 && a.draft == nullptr) return false;
  for (int t = 0; t < n; ++t) {
    const int x = a.draft_tokens[static_cast<size_t>(b) * a.K + t];
    if (x < 0 || x >= a.V) return false;
  }
  for (int t = 0; t <= n; ++t) {
    const double u = a.uniforms[static_cast<size_t>(b) * (a.K + 1) + t];
    if (!(u >= 0.0 && u < 1.0)) return false;
  }
  const double ur = a.uniforms_resample[b];
  if (!(ur >= 0.0 && ur < 1.0)) return false;
  // A sampled request needs a finite maximum in every row it uses (target
  // rows t <= n, draft rows t < n), whether or not the scan reaches them.
  if (T > 0.0) {
    for (int t = 0; t <= n; ++t)
      if (!row_has_finite_max(a.target, a.dtype, (static_cast<size_t>(b) * (a.K + 1) + t), a.V))
        return false;
    for (int t = 0; t < n; ++t)
      if (!row_has_finite_max(a.draft, a.dtype, (static_cast<size_t>(b) * a.K + t), a.V))
        return false;
  }
  *n_out = n;
  return true;
}

void write_outputs(const Args& a, int b, int j, const std::vector<int>& tokens, int flags) {
  a.accepted_len[b] = j;
  int32_t* out = a.out_tokens + static_cast<size_t>(b) * (a.K + 1);
  for (int t = 0; t <= a.K; ++t) out[t] = t < static_cast<int>(tokens.size()) ? tokens[t] : -1;
  if (a.flags) a.flags[b] = flags;
}

// One request, following the rule in the order the pages give it.
void verify_request(const Args& a, int b, std::vector<double>& zp, std::vector<double>& zq,
                    std::vector<double>& p, std::vector<double>& q, std::vector<double>& w) {
  int n = 0;
  if (!request_valid(a, b, &n)) {
    write_outputs(a, b, -1, {}, kBadInput);
    return;
  }
  const double T = a.temperature[b];
  const int32_t* x = a.draft_tokens + static_cast<size_t>(b) * a.K;
  const float* u = a.uniforms + static_cast<size_t>(b) * (a.K + 1);
  const size_t trow0 = static_cast<size_t>(b) * (a.K + 1);
  const size_t drow0 = static_cast<size_t>(b) * a.K;
  std::vector<int> tokens;
  int flags = 0;

  if (T == 0.0) {
    // Greedy case: accept while argmax(p) equals the draft; at the first
    // mismatch (or after the last draft) emit argmax(p) and stop.
    for (int t = 0; t <= n; ++t) {
      load_row(a.target, a.dtype, trow0 + t, a.V, zp);
      const int g = argmax_lowest(zp);
      if (t < n && g == x[t]) { tokens.push_back(x[t]); continue; }
      tokens.push_back(g);
      write_outputs(a, b, t, tokens, flags);
      return;
    }
  }

  double zmax_p, S_p, zmax_q, S_q;
  for (int t = 0; t < n; ++t) {
    load_row(a.target, a.dtype, trow0 + t, a.V, zp);
    load_row(a.draft, a.dtype, drow0 + t, a.V, zq);
    if (!softmax_T(zp, T, p, zmax_p, S_p) || !softmax_T(zq, T, q, zmax_q, S_q)) {
      write_outputs(a, b, -1, {}, kBadInput);
      return;
    }
    // log p(x_t), log q(x_t) straight from the logits: no underflow.
    const double logp = (zp[x[t]] - zmax_p) / T - std::log(S_p);
    const double logq = (zq[x[t]] - zmax_q) / T - std::log(S_q);
    const double ut = u[t];
    const double ratio = std::exp(logp - logq);
    if (std::fabs(ut - ratio) < kTieBand) flags |= kTieAccept;
    if (std::log(ut) + logq < logp) {          // r < p(x)/q(x): accept x_t
      tokens.push_back(x[t]);
      continue;
    }
    // Rejected: replacement ~ (p - q)+ / ||(p - q)+||_1, then stop.
    w.resize(a.V);
    for (int i = 0; i < a.V; ++i) w[i] = std::max(p[i] - q[i], 0.0);
    double W = comp_total(w);
    if (!(W > 0.0)) {
      flags |= kResFallback;
      w = p;
      W = comp_total(w);
    }
    int edge = 0;
    const int tok = inverse_cdf(w, W, a.uniforms_resample[b], &edge);
    flags |= edge;
    tokens.push_back(tok);
    write_outputs(a, b, t, tokens, flags);
    return;
  }
  // Every draft accepted: bonus token from p at position n.
  load_row(a.target, a.dtype, trow0 + n, a.V, zp);
  if (!softmax_T(zp, T, p, zmax_p, S_p)) {
    write_outputs(a, b, -1, {}, kBadInput);
    return;
  }
  int edge = 0;
  const int tok = inverse_cdf(p, comp_total(p), u[n], &edge);
  flags |= edge;
  tokens.push_back(tok);
  write_outputs(a, b, n, tokens, flags);
}

// Per-row quantities for parity of probabilities: every row a request needs
// (target rows t <= n, draft rows t < n when T > 0), not only those before
// the first rejection.  Layout per row (double):
//   0 zmax_p  1 S_p  2 log p(x_t)  3 zmax_q  4 S_q  5 log q(x_t)
//   6 W (residual mass sum (p-q)+ at t < n; sum p at t = n)
//   7 the final-draw token this row would give (residual with the resample
//     uniform at t < n, bonus with u[n] at t = n; greedy: argmax)
//   8 near-tie class of that draw (kTieCdf, kPrecisionBand or 0)
//   9 accept-test near-tie flag
// Rows a request does not need hold NaN.
void row_stats_request(const Args& a, int b, std::vector<double>& zp, std::vector<double>& zq,
                       std::vector<double>& p, std::vector<double>& q, std::vector<double>& w) {
  const double nan = std::numeric_limits<double>::quiet_NaN();
  double* info = a.row_info + static_cast<size_t>(b) * (a.K + 1) * kRowInfo;
  for (int i = 0; i < (a.K + 1) * kRowInfo; ++i) info[i] = nan;
  int n = 0;
  if (!request_valid(a, b, &n)) return;
  const double T = a.temperature[b];
  const int32_t* x = a.draft_tokens + static_cast<size_t>(b) * a.K;
  const float* u = a.uniforms + static_cast<size_t>(b) * (a.K + 1);
  const size_t trow0 = static_cast<size_t>(b) * (a.K + 1);
  const size_t drow0 = static_cast<size_t>(b) * a.K;
  for (int t = 0; t <= n; ++t) {
    double* r = info + t * kRowInfo;
    load_row(a.target, a.dtype, trow0 + t, a.V, zp);
    if (T == 0.0) {
      const int g = argmax_lowest(zp);
      r[0] = zp[g];
      r[7] = g;
      r[8] = 0.0;
      r[9] = 0.0;
      continue;
    }
    double zmax_p, S_p, zmax_q, S_q;
    if (!softmax_T(zp, T, p, zmax_p, S_p)) continue;
    r[0] = zmax_p;
    r[1] = S_p;
    if (t == n) {
      int edge = 0;
      const double W = comp_total(p);
      r[6] = W;
      r[7] = inverse_cdf(p, W, u[n], &edge);
      r[8] = edge;
      continue;
    }
    load_row(a.draft, a.dtype, drow0 + t, a.V, zq);
    if (!softmax_T(zq, T, q, zmax_q, S_q)) continue;
    r[2] = (zp[x[t]] - zmax_p) / T - std::log(S_p);
    r[3] = zmax_q;
    r[4] = S_q;
    r[5] = (zq[x[t]] - zmax_q) / T - std::log(S_q);
    r[9] = std::fabs(u[t] - std::exp(r[2] - r[5])) < kTieBand ? 1.0 : 0.0;
    w.resize(a.V);
    for (int i = 0; i < a.V; ++i) w[i] = std::max(p[i] - q[i], 0.0);
    double W = comp_total(w);
    r[6] = W;
    int edge = 0;
    if (!(W > 0.0)) { w = p; W = comp_total(w); edge = kResFallback; }
    int e2 = 0;
    r[7] = inverse_cdf(w, W, a.uniforms_resample[b], &e2);
    r[8] = edge | e2;
  }
}

// ---------------------------------------------------------------- draft-side sampler
//
// "Decodificación Especulativa y EAGLE", sections "La Configuración de Dos
// Modelos" and "Desarrolla": the draft model proposes each token by sampling
// x ~ softmax(z / T) from its logits at temperature T (its top token at
// T = 0).  One row per request; the uniform u drives the inverse CDF.

void sample_row(const void* logits, int dtype, size_t row, int V, double T, double u,
                std::vector<double>& z, std::vector<double>& p, int32_t* token, int32_t* flag) {
  load_row(logits, dtype, row, V, z);
  if (T == 0.0) {
    *token = argmax_lowest(z);
    *flag = 0;
    return;
  }
  double zmax, S;
  if (!softmax_T(z, T, p, zmax, S)) {
    *token = -1;
    *flag = kBadInput;
    return;
  }
  int edge = 0;
  *token = inverse_cdf(p, comp_total(p), u, &edge);
  *flag = edge;
}

// ---------------------------------------------------------------- one-hot draft
//
// "Accelerating Sonar through speculation", section "Objetivo-Borrador": the
// draft proposes its top token, so the distribution x was drawn from is the
// point mass q = 1{x}.  The rule of "La Regla de Exactitud" with that q:
// accept x_t iff u_t < p_t(x_t) / 1; at the first rejection j draw from
// (p_j - 1{x_j})+ / ||.||_1, which is p_j with x_j removed and renormalised
// (p_j(x_j) - 1 <= 0); if every draft is accepted, the bonus token from p_n.

void onehot_request(const Args& a, int b, std::vector<double>& zp, std::vector<double>& p,
                    std::vector<double>& w) {
  const int n = a.draft_len ? a.draft_len[b] : a.K;
  const double T = a.temperature[b];
  bool ok = n >= 1 && n <= a.K && T >= 0.0 && std::isfinite(T);
  const int32_t* x = a.draft_tokens + static_cast<size_t>(b) * a.K;
  const float* u = a.uniforms + static_cast<size_t>(b) * (a.K + 1);
  for (int t = 0; ok && t < n; ++t) ok = x[t] >= 0 && x[t] < a.V;
  for (int t = 0; ok && t <= n; ++t) ok = u[t] >= 0.0f && u[t] < 1.0f;
  ok = ok && a.uniforms_resample[b] >= 0.0f && a.uniforms_resample[b] < 1.0f;
  const size_t trow0 = static_cast<size_t>(b) * (a.K + 1);
  if (ok && T > 0.0)
    for (int t = 0; t <= n; ++t) ok = ok && row_has_finite_max(a.target, a.dtype, trow0 + t, a.V);
  if (!ok) {
    write_outputs(a, b, -1, {}, kBadInput);
    return;
  }
  std::vector<int> tokens;
  int flags = 0;
  if (T == 0.0) {   // the greedy rule, as for any draft ("Caso codicioso")
    for (int t = 0; t <= n; ++t) {
      load_row(a.target, a.dtype, trow0 + t, a.V, zp);
      const int g = argmax_lowest(zp);
      if (t < n && g == x[t]) { tokens.push_back(x[t]); continue; }
      tokens.push_back(g);
      write_outputs(a, b, t, tokens, 0);
      return;
    }
  }
  double zmax, S;
  for (int t = 0; t < n; ++t) {
    load_row(a.target, a.dtype, trow0 + t, a.V, zp);
    softmax_T(zp, T, p, zmax, S);
    const double logp = (zp[x[t]] - zmax) / T - std::log(S);
    if (std::fabs(u[t] - std::exp(logp)) < kTieBand) flags |= kTieAccept;
    if (std::log(static_cast<double>(u[t])) < logp) {   // u < p(x) / q(x), q(x) = 1
      tokens.push_back(x[t]);
      continue;
    }
    w = p;
    w[x[t]] = 0.0;   // (p - 1{x})+
    double W = comp_total(w);
    if (!(W > 0.0)) {   // only through rounding: p(x) = 1 cannot be rejected
      flags |= kResFallback;
      w = p;
      W = comp_total(w);
    }
    int edge = 0;
    tokens.push_back(inverse_cdf(w, W, a.uniforms_resample[b], &edge));
    write_outputs(a, b, t, tokens, flags | edge);
    return;
  }
  load_row(a.target, a.dtype, trow0 + n, a.V, zp);
  softmax_T(zp, T, p, zmax, S);
  int edge = 0;
  tokens.push_back(inverse_cdf(p, comp_total(p), u[n], &edge));
  write_outputs(a, b, n, tokens, flags | edge);
}

// ---------------------------------------------------------------- greedy token tree
//
// "Decodificación Especulativa y EAGLE", section "Verificación de Atención en
// Árvore", and "Accelerating Sonar through speculation", section "EAGLE":
// the draft proposes a tree of tokens, the target scores every node in one
// pass, and the longest path the target agrees with is kept.  The greedy
// reading of "agrees" (section "Caso codicioso"): node i, with parent
// parents[i] < i and token tokens[i], is accepted iff its parent is accepted
// and argmax(p at the parent) = tokens[i]; node 0 is the root (the last
// verified token) and always accepted.  The deepest accepted node (lowest
// index among equally deep ones) ends the path; the emitted tokens are the
// path's tokens and then argmax(p at that node).

int tree_request(const void* target, int dtype, const int32_t* parents, const int32_t* tokens,
                 int n, int N, int V, size_t row0, int32_t* out_tokens, int32_t* path_nodes,
                 std::vector<double>& z) {
  for (int i = 0; i < N; ++i) out_tokens[i] = path_nodes[i] = -1;
  if (n < 1 || n > N || parents[0] != -1) return -1;
  for (int i = 1; i < n; ++i)
    if (parents[i] < 0 || parents[i] >= i || tokens[i] < 0 || tokens[i] >= V) return -1;
  std::vector<int> g(n), depth(n, 0);
  std::vector<char> acc(n, 0);
  for (int i = 0; i < n; ++i) {
    load_row(target, dtype, row0 + i, V, z);
    g[i] = argmax_lowest(z);
  }
  acc[0] = 1;
  int best = 0;
  for (int i = 1; i < n; ++i) {
    const int par = parents[i];
    acc[i] = acc[par] && tokens[i] == g[par];
    if (acc[i]) {
      depth[i] = depth[par] + 1;
      if (depth[i] > depth[best]) best = i;
    }
  }
  // the path from the root to `best`, root excluded
  std::vector<int> path;
  for (int v = best; v != 0; v = parents[v]) path.push_back(v);
  const int L = static_cast<int>(path.size());
  path_nodes[0] = 0;
  for (int k = 0; k < L; ++k) {
    const int v = path[L - 1 - k];
    out_tokens[k] = tokens[v];
    path_nodes[k + 1] = v;
  }
  out_tokens[L] = g[best];
  return L;
}

template <class F>
void for_requests(const Args& a, int nthreads, F body) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > a.B) nthreads = a.B;
  auto work = [&](int lo, int hi) {
    std::vector<double> zp, zq, p, q, w;
    for (int b = lo; b < hi; ++b) body(a, b, zp, zq, p, q, w);
  };
  if (nthreads == 1) { work(0, a.B); return; }
  std::vector<std::thread> pool;
  for (int k = 0; k < nthreads; ++k) {
    const int lo = static_cast<int>(static_cast<long long>(a.B) * k / nthreads);
    const int hi = static_cast<int>(static_cast<long long>(a.B) * (k + 1) / nthreads);
    pool.emplace_back(work, lo, hi);
  }
  for (auto& th : pool) th.join();
}

bool shape_ok(int B, int K, int V) { return B >= 1 && K >= 1 && V >= 1; }

}  // namespace

extern "C" {

int oracle_version(void) { return 1; }

// Verification sampler on host buffers.  Logits: target [B,K+1,V],
// draft [B,K,V] (may be null when every temperature is 0), dtype 0=f32 1=bf16
// (bf16 passed as raw uint16).  flags [B] (may be null) receives the near-tie
// bitmask.  Returns 0 on success, 1 on a bad shape or null pointer.
int oracle_verify_sample(const void* target_logits, const void* draft_logits, int dtype,
                         const int32_t* draft_tokens, const int32_t* draft_len,
                         const float* temperature, const float* uniforms,
                         const float* uniforms_resample, int B, int K, int V,
                         int32_t* accepted_len, int32_t* out_tokens, int32_t* flags,
                         int nthreads) {
  if (!shape_ok(B, K, V) || !target_logits || !draft_tokens || !temperature || !uniforms ||
      !uniforms_resample || !accepted_len || !out_tokens || (dtype != kF32 && dtype != kBF16))
    return 1;
  Args a{target_logits, draft_logits, dtype, draft_tokens, draft_len, temperature, uniforms,
         uniforms_resample, B, K, V, accepted_len, out_tokens, flags, nullptr};
  for_requests(a, nthreads, verify_request);
  return 0;
}

// Per-row probabilities and per-row final-draw candidates (layout above).
int oracle_row_stats(const void* target_logits, const void* draft_logits, int dtype,
                     const int32_t* draft_tokens, const int32_t* draft_len,
                     const float* temperature, const float* uniforms,
                     const float* uniforms_resample, int B, int K, int V, double* row_info,
                     int nthreads) {
  if (!shape_ok(B, K, V) || !target_logits || !draft_tokens || !temperature || !uniforms ||
      !uniforms_resample || !row_info || (dtype != kF32 && dtype != kBF16))
    return 1;
  Args a{target_logits, draft_logits, dtype, draft_tokens, draft_len, temperature, uniforms,
         uniforms_resample, B, K, V, nullptr, nullptr, nullptr, row_info};
  for_requests(a, nthreads, row_stats_request);
  return 0;
}

// Draft-side sampler on host buffers: logits [R, V] (dtype 0 = f32, 1 = bf16
// as raw uint16), temperature [R] (0 = top token), uniforms [R] in [0, 1).
// tokens [R] get the drawn tokens (-1 for an unusable row), flags [R] (may
// be null) the near-tie flags of each draw.  Returns 0, or 1 on bad
// arguments.
int oracle_sample_draft(const void* logits, int dtype, const float* temperature,
                        const float* uniforms, int R, int V, int32_t* tokens, int32_t* flags,
                        int nthreads) {
  if (R < 1 || V < 1 || !logits || !temperature || !uniforms || !tokens ||
      (dtype != kF32 && dtype != kBF16))
    return 1;
  auto work = [&](int lo, int hi) {
    std::vector<double> z, p;
    for (int r = lo; r < hi; ++r) {
      int32_t flag = 0;
      const double T = temperature[r];
      const double u = uniforms[r];
      if (!(T >= 0.0) || !std::isfinite(T) || !(u >= 0.0 && u < 1.0)) {
        tokens[r] = -1;
        flag = kBadInput;
      } else {
        sample_row(logits, dtype, static_cast<size_t>(r), V, T, u, z, p, tokens + r, &flag);
      }
      if (flags) flags[r] = flag;
    }
  };
  if (nthreads < 1) nthreads = 1;
  if (nthreads > R) nthreads = R;
  std::vector<std::thread> pool;
  for (int k = 0; k < nthreads; ++k)
    pool.emplace_back(work, static_cast<int>(static_cast<long long>(R) * k / nthreads),
                      static_cast<int>(static_cast<long long>(R) * (k + 1) / nthreads));
  for (auto& th : pool) th.join();
  return 0;
}

// The verification rule for a draft that proposes its top token (q one-hot
// at the drafted token; no draft logits).  Same arguments and outputs as
// oracle_verify_sample without draft_logits.
int oracle_verify_onehot(const void* target_logits, int dtype, const int32_t* draft_tokens,
                         const int32_t* draft_len, const float* temperature,
                         const float* uniforms, const float* uniforms_resample, int B, int K,
                         int V, int32_t* accepted_len, int32_t* out_tokens, int32_t* flags,
                         int nthreads) {
  if (!shape_ok(B, K, V) || !target_logits || !draft_tokens || !temperature || !uniforms ||
      !uniforms_resample || !accepted_len || !out_tokens || (dtype != kF32 && dtype != kBF16))
    return 1;
  Args a{target_logits, nullptr, dtype, draft_tokens, draft_len, temperature, uniforms,
         uniforms_resample, B, K, V, accepted_len, out_tokens, flags, nullptr};
  for_requests(a, nthreads, [](const Args& aa, int b, std::vector<double>& zp,
                               std::vector<double>&, std::vector<double>& p,
                               std::vector<double>&, std::vector<double>& w) {
    onehot_request(aa, b, zp, p, w);
  });
  return 0;
}

// Greedy verification of a token tree: target_logits [B, N, V] (row i of a
// request: the target's logits at tree node i), parents [B, N] (parents[0] =
// -1, parents[i] < i), tokens [B, N] (node i's drafted token; tokens[0]
// unused), n_nodes [B] in 1..N (nodes >= n_nodes ignored).  accepted_len [B]
// = the accepted path's length (-1 for an unusable tree); out_tokens [B, N]
// = the path's tokens, then the target's argmax at its last node, then -1;
// path_nodes [B, N] = 0, then the path's node indices, then -1.
int oracle_tree_greedy(const void* target_logits, int dtype, const int32_t* parents,
                       const int32_t* tokens, const int32_t* n_nodes, int B, int N, int V,
                       int32_t* accepted_len, int32_t* out_tokens, int32_t* path_nodes,
                       int nthreads) {
  if (B < 1 || N < 1 || V < 1 || !target_logits || !parents || !tokens || !n_nodes ||
      !accepted_len || !out_tokens || !path_nodes || (dtype != kF32 && dtype != kBF16))
    return 1;
  auto work = [&](int lo, int hi) {
    std::vector<double> z;
    for (int b = lo; b < hi; ++b) {
      const size_t o = static_cast<size_t>(b) * N;
      accepted_len[b] = tree_request(target_logits, dtype, parents + o, tokens + o, n_nodes[b],
                                     N, V, o, out_tokens + o, path_nodes + o, z);
    }
  };
  if (nthreads < 1) nthreads = 1;
  if (nthreads > B) nthreads = B;
  std::vector<std::thread> pool;
  for (int k = 0; k < nthreads; ++k)
    pool.emplace_back(work, static_cast<int>(static_cast<long long>(B) * k / nthreads),
                      static_cast<int>(static_cast<long long>(B) * (k + 1) / nthreads));
  for (auto& th : pool) th.join();
  return 0;
}

// Post-accept insert ("Accelerating Sonar through speculation", sections
// "Programación MTP para un solo token" and "Inferencia con decodificación
// especulativa": a kernel writes the next step's tokens on the device, so
// the host need not read the accepted lengths).  For request b with
// j = accepted_len[b]: the j + 1 emitted tokens out_tokens[b, 0..j] are
// appended to its token history at history[b, seq_lens[b]..] and
// seq_lens[b] grows by j + 1; next_tokens[b] = out_tokens[b, j] (the next
// step's input); cu_emitted[b + 1] = cu_emitted[b] + j + 1 and the emitted
// tokens of all requests are packed, in request order, at packed[cu_emitted[b]..].
// A request with j outside [0, K] emits nothing (status 1); one whose
// history would overflow L emits nothing (status 2); both get
// next_tokens[b] = -1 and keep their history and length.
int oracle_insert_accepted(const int32_t* accepted_len, const int32_t* out_tokens, int B, int K1,
                           int32_t* seq_lens, int32_t* history, int L, int32_t* next_tokens,
                           int32_t* cu_emitted, int32_t* packed, int32_t* status) {
  if (B < 1 || K1 < 1 || L < 1 || !accepted_len || !out_tokens || !seq_lens || !history ||
      !next_tokens || !cu_emitted || !packed || !status)
    return 1;
  cu_emitted[0] = 0;
  for (int b = 0; b < B; ++b) {
    const int j = accepted_len[b];
    const int32_t* out = out_tokens + static_cast<size_t>(b) * K1;
    int emitted = 0;
    if (j < 0 || j >= K1) {
      status[b] = 1;
      next_tokens[b] = -1;
    } else if (seq_lens[b] < 0 || seq_lens[b] + j + 1 > L) {
      status[b] = 2;
      next_tokens[b] = -1;
    } else {
      status[b] = 0;
      emitted = j + 1;
      for (int i = 0; i <= j; ++i) {
        history[static_cast<size_t>(b) * L + seq_lens[b] + i] = out[i];
        packed[cu_emitted[b] + i] = out[i];
      }
      seq_lens[b] += emitted;
      next_tokens[b] = out[j];
    }
    cu_emitted[b + 1] = cu_emitted[b] + emitted;
  }
  return 0;
}

}  // extern "C"
