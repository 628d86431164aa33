// Analytic operating-point report ("Speculative Decoding Part 1: 도입 전에
// 확인해야 할 것들", VESSL AI blog, section "속도 향상을 결정하는 방정식" and the
// section on the compute theorem) on the host, and the measured acceptance
// statistics of a verification on the device.
#include <cmath>
#include <limits>

#include "spec_internal.cuh"

namespace spec {
namespace {

// E[tau] = sum_{k=0}^{gamma} alpha^k, accumulated from the largest term
// down (alpha^k decreases in k) with a running power.
double expected_tau(double alpha, int gamma) {
  double pw = 1.0;
  double terms_hi = 0.0, comp = 0.0;   // compensated sum (Neumaier)
  for (int k = 0; k <= gamma; ++k) {
    const double t = terms_hi + pw;
    comp += (std::fabs(terms_hi) >= std::fabs(pw)) ? (terms_hi - t) + pw : (pw - t) + terms_hi;
    terms_hi = t;
    pw *= alpha;
  }
  return terms_hi + comp;
}

double speedup(double alpha, double c, int gamma) { return expected_tau(alpha, gamma) / (c * gamma + 1.0); }

// alpha^{g+1} (c - (c g + 1) ln alpha) - c: strictly decreasing in g.
double stationarity(double alpha, double c, double g) {
  return std::pow(alpha, g + 1.0) * (c - (c * g + 1.0) * std::log(alpha)) - c;
}

}  // namespace

// Sums of one verification's acceptance statistics (one CTA, fixed order).
__global__ void __launch_bounds__(NT) acceptance_stats_kernel(int B, int gamma, const float* alpha,
                                                              const int* vlen, const int* acc,
                                                              double* out) {
  __shared__ float shf[72];
  DdSum sa, st;
  float na = 0.f, nr = 0.f;
  for (int b = threadIdx.x; b < B; b += NT) {
    const int n = acc[b];
    if (n < 0) continue;                       // request flagged invalid by the verification
    const int L = vlen[b];
    for (int j = 0; j < L && j < gamma; ++j) {
      sa.add(alpha[(size_t)b * gamma + j]);
      na += 1.f;
    }
    st.add((float)(n + 1));
    nr += 1.f;
  }
  const df A = block_sum_df(sa.value(), shf);
  const df Tt = block_sum_df(st.value(), shf);
  const float NA = block_sum(na, shf), NR = block_sum(nr, shf);
  if (threadIdx.x == 0) {
    out[0] = dd_to_double(A);
    out[1] = (double)NA;
    out[2] = dd_to_double(Tt);
    out[3] = (double)NR;
  }
}

}  // namespace spec

using namespace spec;

extern "C" {

int32_t spec_operating_point(const spec_op_args* a, spec_op_result* o) {
  if (!a || !o) return SPEC_EINVAL;
  if (!(a->alpha >= 0.0 && a->alpha <= 1.0) || !(a->c > 0.0) || !(a->c_hat >= 0.0) || a->gamma < 1 ||
      a->gamma_max < a->gamma || a->gamma_max > 100000)
    return SPEC_EINVAL;
  const double alpha = a->alpha, c = a->c;
  spec_op_result r;
  r.expected_tau = expected_tau(alpha, a->gamma);
  r.speedup = r.expected_tau / (c * a->gamma + 1.0);
  r.speedup_gamma1 = (1.0 + alpha) / (c + 1.0);
  r.bound = alpha >= 1.0 ? 1.0 / c : std::fmin(1.0 / c, 1.0 / (1.0 - alpha));
  r.gamma_star = 1;
  r.speedup_star = speedup(alpha, c, 1);
  for (int g = 2; g <= a->gamma_max; ++g) {
    const double s = speedup(alpha, c, g);
    if (s > r.speedup_star) {
      r.speedup_star = s;
      r.gamma_star = g;
    }
  }
  // real root of the stationarity condition by bisection
  if (alpha <= 0.0) {
    r.gamma_continuous = 0.0;
  } else if (alpha >= 1.0) {
    r.gamma_continuous = std::numeric_limits<double>::infinity();   // S grows without end
  } else if (stationarity(alpha, c, 0.0) <= 0.0) {
    r.gamma_continuous = 0.0;
  } else {
    double lo = 0.0, hi = 1.0;
    while (stationarity(alpha, c, hi) > 0.0 && hi < 1e12) hi *= 2.0;
    for (int it = 0; it < 200; ++it) {
      const double mid = 0.5 * (lo + hi);
      (stationarity(alpha, c, mid) > 0.0 ? lo : hi) = mid;
    }
    r.gamma_continuous = 0.5 * (lo + hi);
  }
  r.compute_ratio = (a->gamma * a->c_hat + a->gamma + 1.0) / r.expected_tau;
  r.gains = r.speedup > 1.0 ? 1 : 0;
  *o = r;
  return SPEC_OK;
}

int32_t spec_acceptance_stats(int32_t B, int32_t gamma, const float* alpha, const int32_t* verify_len,
                              const int32_t* accept_len, double* out, spec_stream_t stream) {
  if (B < 1 || gamma < 1 || !alpha || !verify_len || !accept_len || !out) return SPEC_EINVAL;
  acceptance_stats_kernel<<<1, NT, 0, reinterpret_cast<cudaStream_t>(stream)>>>(B, gamma, alpha, verify_len,
                                                                                accept_len, out);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

}  // extern "C"
