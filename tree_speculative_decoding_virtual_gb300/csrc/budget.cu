// Hardware-aware tree budget.
//
// "Resumo Técnico: BASTION", Methodology 3 (hardware-aware online budget
// controller): the verification latency T_verify(N) is estimated with a
// roofline model of memory bandwidth and compute, calibrated with observed
// run times (the scale absorbs fusion, the offset launch and scheduling
// overhead); the tree grows until the estimated speed-up
// S(N) = A_hat(T_N) * L_AR / C(N) starts to decrease.
//
// Two host functions (the cost model and its least-squares calibration) and
// one kernel that makes the per-step choice on the device, straight from the
// path scores the best-first builder wrote, so the chosen size never
// round-trips through the host.

#include <cmath>

#include "tsd_common.cuh"

namespace tsd {
namespace {

constexpr int kSelectThreads = 256;  // >= kMaxNodes + 1

// One block per sequence: the row's path scores and the cost table are staged
// in shared memory with coalesced loads, then one thread walks them in fp32
// (the rounding of every step is fixed, so the choice is reproducible): A_hat
// is a running sum of the non-root path scores in insertion order; S(n) <
// S(n-1) is tested without dividing, as A_hat(n) * C(n-1) < A_hat(n-1) * C(n);
// the chosen size is the last n before S first decreases (ties continue),
// else N_max.
__global__ void __launch_bounds__(kSelectThreads)
budget_select_kernel(const float *__restrict__ rho, int B, int N_max,
                     const float *__restrict__ cost, float l_ar, int32_t *__restrict__ n_opt,
                     float *__restrict__ s_opt) {
  __shared__ float s_r[kMaxNodes], s_c[kMaxNodes + 1];
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, t = threadIdx.x;
  for (int n = t; n < N_max; n += kSelectThreads) s_r[n] = rho[(size_t)b * N_max + n];
  for (int n = t; n <= N_max; n += kSelectThreads) s_c[n] = cost[n];
  __syncthreads();
  if (t != 0) return;
  float a_prev = 0.f, c_prev = s_c[1];
  int best = 1;
#pragma unroll 8
  for (int n = 2; n <= N_max; ++n) {
    const float a = __fadd_rn(a_prev, s_r[n - 1]);
    const float c = s_c[n];
    if (__fmul_rn(a, c_prev) < __fmul_rn(a_prev, c)) break;
    a_prev = a;
    c_prev = c;
    best = n;
  }
  n_opt[b] = best;
  if (s_opt) s_opt[b] = __fdiv_rn(__fmul_rn(a_prev, l_ar), c_prev);
}

}  // namespace
}  // namespace tsd

TSD_API int tsd_verify_step_cost(int B, int Hq, int Hkv, int D, const int32_t *prefix_len, int V,
                                 int D_max, int N, double hbm_gbs, double tc_tflops,
                                 double *bytes, double *flops, double *t_us) {
  if (B < 1 || Hq < 1 || Hkv < 1 || D < 1 || V < 1 || D_max < 0 || N < 1 || !prefix_len ||
      !(hbm_gbs > 0.0) || !(tc_tflops > 0.0) || !std::isfinite(hbm_gbs) ||
      !std::isfinite(tc_tflops))
    return TSD_ERR_ARG;
  long long sum_p = 0;
  for (int b = 0; b < B; ++b) {
    if (prefix_len[b] < 0) return TSD_ERR_ARG;
    sum_p += prefix_len[b];
  }
  const long long W = (N + 31) / 32;
  const long long n = N, bb = B;
  const long long tables =
      4 * (bb * n + bb + bb * (n + 1) * (D_max + 1) + bb * n + bb * n * W + bb);
  const long long kv = 2LL * 2 * Hkv * D * (sum_p + bb * n);      // K and V, bf16
  const long long q_out = 2LL * 2 * bb * n * Hq * D;              // q and out, bf16
  const long long lse = 4LL * bb * n * Hq;
  const long long logits = 4LL * bb * n * V;
  const long long commit = 2LL * 2 * 2 * Hkv * D * bb * D_max;    // read + write of K and V
  const long long nbytes = tables + kv + q_out + lse + logits + commit;
  const long long keys = n * sum_p + bb * n * (D_max + 1);
  const double f = 4.0 * D * Hq * (double)keys;
  const double t = std::fmax((double)nbytes / (hbm_gbs * 1e9), f / (tc_tflops * 1e12)) * 1e6;
  if (bytes) *bytes = (double)nbytes;
  if (flops) *flops = f;
  if (t_us) *t_us = t;
  return TSD_OK;
}

TSD_API int tsd_budget_calibrate(const double *t_roof, const double *t_meas, int count,
                                 double *alpha, double *beta) {
  if (!t_roof || !t_meas || !alpha || !beta || count < 2) return TSD_ERR_ARG;
  double xm = 0.0, ym = 0.0;
  for (int i = 0; i < count; ++i) {
    if (!std::isfinite(t_roof[i]) || !std::isfinite(t_meas[i])) return TSD_ERR_ARG;
    xm += t_roof[i];
    ym += t_meas[i];
  }
  xm /= count;
  ym /= count;
  double sxx = 0.0, sxy = 0.0;
  for (int i = 0; i < count; ++i) {
    sxx += (t_roof[i] - xm) * (t_roof[i] - xm);
    sxy += (t_roof[i] - xm) * (t_meas[i] - ym);
  }
  if (!(sxx > 0.0)) return TSD_ERR_ARG;
  *alpha = sxy / sxx;
  *beta = ym - *alpha * xm;
  return TSD_OK;
}

TSD_API int tsd_budget_select(const float *rho, int B, int N_max, const float *cost, float l_ar,
                              int32_t *n_opt, float *s_opt, tsd_stream_t stream) {
  using namespace tsd;
  if (B < 0) return TSD_ERR_ARG;
  if (N_max < 1 || N_max > kMaxNodes || B > 65535) return TSD_ERR_LIMIT;
  if (B == 0) return TSD_OK;
  if (!rho || !cost || !n_opt || !(l_ar > 0.0) || !std::isfinite(l_ar)) return TSD_ERR_ARG;
  if (launch(budget_select_kernel, dim3(B), dim3(kSelectThreads), 0, as_cuda(stream), rho, B,
             N_max, cost, l_ar, n_opt, s_opt) != cudaSuccess)
    return TSD_ERR_CUDA;
  return TSD_OK;
}
