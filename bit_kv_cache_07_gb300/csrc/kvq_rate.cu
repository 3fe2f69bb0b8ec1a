// kvq_rate.cu -- per-head (K, V) bit allocation (RateQuant summary,
// "Methodology" 1-4): the distortion of this cache's quantizer measured per
// head on calibration tokens (a GPU kernel, kvq_append.cu), the
// distortion-rate fit D(b) = alpha * beta^-b per component, the continuous
// reverse water-filling optimum, and the greedy marginal-gain allocation on
// the bit widths the kernels support.  The allocation itself is host code:
// a handful of components per layer, once per model.
#include <cmath>
#include <cstring>
#include <vector>

#include "kvq_internal.cuh"

using namespace kvq;

namespace {

constexpr int kLadder[3] = {2, 4, 8};  // bit widths of the uniform kernels

// ln D = ln alpha - b ln beta by ordinary least squares over the ladder
// (centred sums).
void fit_component(const double* D, double* alpha, double* beta) {
  double mb = 0.0, my = 0.0;
  for (int i = 0; i < 3; ++i) {
    mb += kLadder[i] / 3.0;
    my += std::log(D[i]) / 3.0;
  }
  double sxy = 0.0, sxx = 0.0;
  for (int i = 0; i < 3; ++i) {
    const double dx = kLadder[i] - mb;
    sxy += dx * (std::log(D[i]) - my);
    sxx += dx * dx;
  }
  const double slope = sxy / sxx;  // -ln beta
  *beta = std::exp(-slope);
  *alpha = std::exp(my - slope * mb);
}

double model(double alpha, double beta, int b) { return alpha * std::pow(beta, -(double)b); }

}  // namespace

extern "C" {

kvq_status kvq_rate_allocate(int32_t n, const double* distortion, const double* weights, int32_t total_bits,
                             int32_t* bits_out, double* alpha_out, double* beta_out, double* waterfill_out) {
  if (n < 1 || !distortion || !bits_out) return KVQ_ERR_INVALID_ARG;
  if (total_bits < 2 * n) return KVQ_ERR_INVALID_ARG;
  std::vector<double> a(n), be(n), w(n);
  for (int i = 0; i < n; ++i) {
    const double* D = distortion + 3 * (size_t)i;
    if (!(D[0] > 0.0 && D[1] > 0.0 && D[2] > 0.0) || !std::isfinite(D[0] + D[1] + D[2])) return KVQ_ERR_INVALID_ARG;
    w[i] = weights ? weights[i] : 1.0;
    if (!(w[i] > 0.0) || !std::isfinite(w[i])) return KVQ_ERR_INVALID_ARG;
    fit_component(D, &a[i], &be[i]);
    if (!(be[i] > 1.0)) return KVQ_ERR_INVALID_ARG;  // distortion must fall with bits
    if (alpha_out) alpha_out[i] = a[i];
    if (beta_out) beta_out[i] = be[i];
  }
  if (waterfill_out) {
    // b_i(lambda) = (ln(w_i alpha_i ln beta_i) - ln lambda) / ln beta_i sums to the budget
    auto total_at = [&](double ll) {
      double t = 0.0;
      for (int i = 0; i < n; ++i) t += (std::log(w[i] * a[i] * std::log(be[i])) - ll) / std::log(be[i]);
      return t;
    };
    double lo = -1000.0, hi = 1000.0;  // total_at falls as ln lambda grows
    for (int it = 0; it < 400; ++it) {
      const double mid = 0.5 * (lo + hi);
      (total_at(mid) > total_bits ? lo : hi) = mid;
    }
    const double ll = 0.5 * (lo + hi);
    for (int i = 0; i < n; ++i) waterfill_out[i] = (std::log(w[i] * a[i] * std::log(be[i])) - ll) / std::log(be[i]);
  }
  // greedy: everyone at the ladder's bottom, then the affordable step with
  // the largest weighted model-distortion drop per added bit (ties: the
  // lower index), until no step fits
  std::vector<int> lvl(n, 0);
  int used = 2 * n;
  for (;;) {
    int pick = -1;
    double best = 0.0;
    for (int i = 0; i < n; ++i) {
      if (lvl[i] == 2) continue;
      const int b0 = kLadder[lvl[i]], b1 = kLadder[lvl[i] + 1];
      if (used + b1 - b0 > total_bits) continue;
      const double g = w[i] * (model(a[i], be[i], b0) - model(a[i], be[i], b1)) / (double)(b1 - b0);
      if (pick < 0 || g > best) {
        pick = i;
        best = g;
      }
    }
    if (pick < 0) break;
    used += kLadder[lvl[pick] + 1] - kLadder[lvl[pick]];
    ++lvl[pick];
  }
  for (int i = 0; i < n; ++i) bits_out[i] = kLadder[lvl[i]];
  return KVQ_OK;
}

kvq_status kvq_measure_distortion(const kvq_config* cfg, const uint16_t* k, const uint16_t* v, int32_t n_tokens,
                                  int32_t bits, void* workspace, uint64_t ws_bytes, double* mse_out,
                                  kvq_stream_t stream) {
  if (!cfg) return KVQ_ERR_INVALID_ARG;
  kvq_config c = *cfg;  // measured with the config's layout, at `bits` for K and V
  if (c.k_bits == 3 || c.k_bits == 16) return KVQ_ERR_UNSUPPORTED;
  if (bits != 2 && bits != 4 && bits != 8) return KVQ_ERR_UNSUPPORTED;
  c.k_bits = c.v_bits = bits;
  kvq_layout L;
  kvq_status st = kvq_layout_query(&c, &L);
  if (st != KVQ_OK) return st;
  if (!k || !v || !mse_out || n_tokens < 1) return KVQ_ERR_INVALID_ARG;
  if (((uintptr_t)k | (uintptr_t)v) % 16 || (uintptr_t)mse_out % 8) return KVQ_ERR_INVALID_ARG;
  AppendParams p;
  std::memset(&p, 0, sizeof(p));
  if (make_geometry_for(&c, &p.geo) != KVQ_OK) return KVQ_ERR_INVALID_ARG;
  p.k_new = k;
  p.v_new = v;
  p.n_new = n_tokens;
  p.hadamard_c = (float)(1.0 / std::sqrt((double)kHeadDim));
  const uint64_t need = (uint64_t)p.geo.NS * kHeadDim * 4;
  float* knorm = nullptr;
  if (p.geo.knorm) {
    if (!workspace || ws_bytes < need || (uintptr_t)workspace % 16) return KVQ_ERR_WORKSPACE;
    knorm = reinterpret_cast<float*>(workspace);
  }
  const cudaError_t e = launch_distortion(p, n_tokens, bits, knorm, mse_out, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // extern "C"
