// Confidence head and hardware-aware prefix scheduler ("[논문리뷰] DSpark:
// Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
// Generation", sections 2.1 "Confidence Head" and 2.2 "Hardware-Aware Prefix
// Scheduler").
//
//   confidence_kernel     c_{r,k} = sigmoid(w^T [h_k; W1[x_{k-1}]]): one CTA
//                         per draft row; the dot product in Dot2 (double-float)
//                         and the logistic in double-float, rounded once to
//                         fp32 -- the nearest float of the exact value except
//                         within ~1e-13 of a rounding midpoint.
//   schedule_rank_kernel  a_{r,j} = running fp32 product of c_{r,1..j}, and
//                         the position of every candidate (r, j) in the global
//                         order (a descending, then r, then j).  A request's
//                         a is non-increasing in j, so each row of every other
//                         request contributes a prefix of its entries; the
//                         count is a branch-free compare over the two rows.
//                         One CTA per request.  Writes the candidates'
//                         increments of tau (units of 2^-36, floor) in sorted
//                         order.
//   schedule_select_kernel  one CTA: prefix sums of the sorted increments give
//                         tau after each admission; Theta = tau * SPS(B) in
//                         float64; the first admission that lowers Theta (or
//                         needs a batch beyond the cost table) stops the
//                         search; l_r = how many of request r's candidates are
//                         ranked before the stop.
//
// tau in integer units makes the sum independent of its order, so the
// parallel scan and a sequential walk over the sorted candidates take the
// same decisions from the same fp32 survival values.
#include "spec_internal.cuh"

namespace spec {

constexpr int CONF_THREADS = 128;    // one CTA per draft row
constexpr int RANK_THREADS = 128;
constexpr int SEL_THREADS = 1024;
constexpr float TAU_SCALE_F = 68719476736.0f;   // 2^36
constexpr double TAU_UNIT_D = 1.0 / 68719476736.0;

// 8 consecutive elements widened to fp32 (16-byte aligned).
__device__ __forceinline__ void load8(const bf16* p, float* o) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = __uint_as_float(w[i] << 16);
    o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void load8(const float* p, float* o) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

template <class DT>
__global__ void __launch_bounds__(CONF_THREADS)
    confidence_kernel(int R, int gamma, int d, int V, int r, const DT* __restrict__ hidden,
                      const DT* __restrict__ W1, const float* __restrict__ w,
                      const int* __restrict__ anchor, const int* __restrict__ tokens,
                      float* __restrict__ conf, uint32_t* status) {
  __shared__ df s_tab[DD_EXP_TAB];
  __shared__ df s_part[CONF_THREADS / 32];
  const int row = blockIdx.x;
  const int b = row / gamma, k = row - b * gamma;
  const int prev = k == 0 ? __ldg(anchor + b) : __ldg(tokens + row - 1);
  if (prev < 0 || prev >= V) {             // uniform over the CTA
    if (threadIdx.x == 0) {
      conf[row] = __int_as_float(0x7fffffff);
      set_status(status, SPEC_DEV_BAD_TOKEN);
    }
    return;
  }
  if (threadIdx.x < DD_EXP_TAB) dd_exp_table_entry(s_tab, threadIdx.x);
  DdDot acc;
  float x[8], y[8];
  const DT* h = hidden + (size_t)row * d;
#pragma unroll 4
  for (int i = threadIdx.x * 8; i < d; i += CONF_THREADS * 8) {
    load8(h + i, x);
    load8(w + i, y);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc.add(x[e], y[e]);
  }
  const DT* emb = W1 + (size_t)prev * r;
  for (int i = threadIdx.x * 8; i < r; i += CONF_THREADS * 8) {
    load8(emb + i, x);
    load8(w + d + i, y);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc.add(x[e], y[e]);
  }
  const df zw = warp_sum_df(acc.value());
  if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = zw;
  __syncthreads();
  if (threadIdx.x == 0) {
    df z = s_part[0];
#pragma unroll
    for (int i = 1; i < CONF_THREADS / 32; ++i) z = dd_add(z, s_part[i]);
    float c;
    if (!isfinite(z.hi)) {
      c = __int_as_float(0x7fffffff);
      set_status(status, SPEC_DEV_BAD_CONF);
    } else {
      const df sg = dd_sigmoid(z, s_tab);
      c = rn_add(sg.hi, sg.lo);
    }
    conf[row] = c;
  }
}

// A confidence outside [0, 1] (or NaN) is flagged and counts as 0.
__device__ __forceinline__ float conf_clean(float c) { return (c >= 0.f && c <= 1.f) ? c : 0.f; }
__device__ __forceinline__ unsigned long long tau_units(float a) {
  return __float2ull_rd(__fmul_rn(a, TAU_SCALE_F));   // exact scaling, then floor
}

template <int G>
__global__ void __launch_bounds__(RANK_THREADS)
    schedule_rank_kernel(int R, int gamma, const float* __restrict__ conf, float* __restrict__ survival,
                         int* __restrict__ rank, unsigned long long* __restrict__ sorted_units,
                         uint32_t* status) {
  __shared__ float s_a[G];
  __shared__ int s_cnt[RANK_THREADS / 32][G];
  const int r = blockIdx.x;
  if (threadIdx.x == 0) {
    float a = 1.f;
    bool bad = false;
    for (int j = 0; j < gamma; ++j) {
      const float c = conf[(size_t)r * gamma + j];
      const float cc = conf_clean(c);
      bad |= !(cc == c);
      a = __fmul_rn(a, cc);
      s_a[j] = a;
      survival[(size_t)r * gamma + j] = a;
    }
    if (bad) set_status(status, SPEC_DEV_BAD_CONF);
  }
  __syncthreads();
  float own[G];
  int cnt[G];
#pragma unroll
  for (int j = 0; j < G; ++j) {
    own[j] = j < gamma ? s_a[j] : 2.f;     // padding: never counted against
    cnt[j] = 0;
  }
  for (int q = threadIdx.x; q < R; q += RANK_THREADS) {
    if (q == r) continue;                  // own row: exactly j candidates precede (r, j)
    const bool before = q < r;             // equal a: the lower request goes first
    float cq[G];
#pragma unroll
    for (int jj = 0; jj < G; ++jj) cq[jj] = jj < gamma ? __ldg(conf + (size_t)q * gamma + jj) : 0.f;
    float a = 1.f;
#pragma unroll
    for (int jj = 0; jj < G; ++jj) {
      a = __fmul_rn(a, conf_clean(cq[jj]));
      const float aq = jj < gamma ? a : -1.f;
#pragma unroll
      for (int j = 0; j < G; ++j) cnt[j] += (aq > own[j]) | (before & (aq == own[j]));
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < G; ++j) {
    int v = cnt[j];
    for (int m = 16; m; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    if (lane == 0) s_cnt[warp][j] = v;
  }
  __syncthreads();
  if (threadIdx.x < gamma) {
    const int j = threadIdx.x;
    int pos = j;
#pragma unroll
    for (int wv = 0; wv < RANK_THREADS / 32; ++wv) pos += s_cnt[wv][j];
    rank[(size_t)r * gamma + j] = pos;
    sorted_units[pos] = tau_units(s_a[j]);
  }
}

__device__ __forceinline__ unsigned long long block_excl_scan_u64(unsigned long long v,
                                                                  unsigned long long* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long incl = v;
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    unsigned long long s = lane < nw ? sh[lane] : 0ull;
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += t;
    }
    sh[lane] = s;   // inclusive warp totals
  }
  __syncthreads();
  const unsigned long long base = warp ? sh[warp - 1] : 0ull;
  __syncthreads();
  return base + incl - v;
}

__global__ void __launch_bounds__(SEL_THREADS)
    schedule_select_kernel(int R, int gamma, const double* __restrict__ sps, int sps_len,
                           const int* __restrict__ rank, const unsigned long long* __restrict__ su,
                           int* __restrict__ ell, long long* __restrict__ totals,
                           double* __restrict__ theta_out) {
  __shared__ unsigned long long s_scan[32];
  __shared__ int s_min[32];
  __shared__ unsigned long long s_sum[32];
  const int N = R * gamma;
  const int seg = (N + SEL_THREADS - 1) / SEL_THREADS;
  const int k0 = min(N, (int)threadIdx.x * seg), k1 = min(N, k0 + seg);
  unsigned long long loc = 0;
  for (int k = k0; k < k1; ++k) loc += su[k];
  const unsigned long long tau0 = (unsigned long long)R << 36;
  unsigned long long tau = tau0 + block_excl_scan_u64(loc, s_scan);
  // first k in this segment whose admission stops the search; key = 4 k + reason
  int key = 4 * N;
  double th = R + k0 < sps_len ? ((double)tau * TAU_UNIT_D) * sps[R + k0] : 0.0;
  for (int k = k0; k < k1; ++k) {
    if (R + k + 1 >= sps_len) { key = 4 * k + 2; break; }
    const unsigned long long nt = tau + su[k];
    const double nth = ((double)nt * TAU_UNIT_D) * sps[R + k + 1];
    if (nth < th) { key = 4 * k + 1; break; }
    tau = nt;
    th = nth;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int m = 16; m; m >>= 1) key = min(key, __shfl_xor_sync(0xffffffffu, key, m));
  if (lane == 0) s_min[warp] = key;
  __syncthreads();
  key = s_min[0];
  for (int wv = 1; wv < SEL_THREADS / 32; ++wv) key = min(key, s_min[wv]);
  const int mstar = key >> 2;
  // tau after mstar admissions
  unsigned long long part = 0;
  for (int k = k0; k < min(k1, mstar); ++k) part += su[k];
  for (int m = 16; m; m >>= 1) part += __shfl_xor_sync(0xffffffffu, part, m);
  if (lane == 0) s_sum[warp] = part;
  __syncthreads();
  for (int q = threadIdx.x; q < R; q += SEL_THREADS) {
    int l = 0;
    for (int j = 0; j < gamma; ++j) l += rank[(size_t)q * gamma + j] < mstar;
    ell[q] = l;
  }
  if (threadIdx.x == 0) {
    unsigned long long t = tau0;
    for (int wv = 0; wv < SEL_THREADS / 32; ++wv) t += s_sum[wv];
    totals[0] = R + mstar;
    totals[1] = (long long)t;
    totals[2] = mstar;
    totals[3] = key & 3;
    theta_out[0] = ((double)t * TAU_UNIT_D) * sps[R + mstar];
  }
}

template <class DT>
cudaError_t launch_confidence(int R, int gamma, int d, int V, int r, const void* hidden, const void* W1,
                              const float* w, const int* anchor, const int* tokens, float* conf,
                              uint32_t* status, cudaStream_t st) {
  confidence_kernel<DT><<<R * gamma, CONF_THREADS, 0, st>>>(
      R, gamma, d, V, r, static_cast<const DT*>(hidden), static_cast<const DT*>(W1), w, anchor, tokens,
      conf, status);
  return cudaGetLastError();
}
template cudaError_t launch_confidence<float>(int, int, int, int, int, const void*, const void*,
                                              const float*, const int*, const int*, float*, uint32_t*,
                                              cudaStream_t);
template cudaError_t launch_confidence<bf16>(int, int, int, int, int, const void*, const void*,
                                             const float*, const int*, const int*, float*, uint32_t*,
                                             cudaStream_t);

cudaError_t launch_schedule_rank(int R, int gamma, const float* conf, float* survival, int* rank,
                                 unsigned long long* sorted_units, uint32_t* status, cudaStream_t st) {
  if (gamma <= 4)
    schedule_rank_kernel<4><<<R, RANK_THREADS, 0, st>>>(R, gamma, conf, survival, rank, sorted_units, status);
  else if (gamma <= 8)
    schedule_rank_kernel<8><<<R, RANK_THREADS, 0, st>>>(R, gamma, conf, survival, rank, sorted_units, status);
  else
    schedule_rank_kernel<16><<<R, RANK_THREADS, 0, st>>>(R, gamma, conf, survival, rank, sorted_units, status);
  return cudaGetLastError();
}

cudaError_t launch_schedule_select(int R, int gamma, const double* sps, int sps_len, const int* rank,
                                   const unsigned long long* sorted_units, int* ell, long long* totals,
                                   double* theta, cudaStream_t st) {
  schedule_select_kernel<<<1, SEL_THREADS, 0, st>>>(R, gamma, sps, sps_len, rank, sorted_units, ell, totals,
                                                    theta);
  return cudaGetLastError();
}

}  // namespace spec
