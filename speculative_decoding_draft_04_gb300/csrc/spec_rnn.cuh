// Gate phase of the RNN head ("[논문리뷰] DSpark", section 1.2, "RNN head"):
// before the bias tiles of draft step k, every request's factor row
// a_k = tanh(W_o z) and next state s_{k+1} = sigma(W_g z) s_k +
// (1 - sigma(W_g z)) tanh(W_c z), z = [s_k; W1[x_k]; h], each rounded to the
// storage type.  The h block arrives as its three projections (hproj); the
// recurrent weights Wr = [W^s | W^e] are [3r][2r] (rows g, c, o).
//
// Certified rounding: each pre-activation is a fixed-order fp32 FMA sum with
// the standard bound gamma_n * sum |terms| on its error; the fp32 tanh and
// logistic add a few ulps.  When the interval [y - err, y + err] of a result
// rounds to one bfloat16 value, that value is the rounding of the exact
// result; otherwise (a rounding midpoint inside the interval, about 1% of the
// outputs) a warp recomputes the row's pre-activations as Dot2 double-float
// dot products and takes the double-float logistic / tanh, correctly rounded.
// fp32 storage always takes the double-float route (no fp32 estimate can
// certify an fp32 rounding).
#pragma once

#include "spec_internal.cuh"

namespace spec {

__device__ __forceinline__ float st_widen(float x) { return x; }
__device__ __forceinline__ float st_widen(bf16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void st_store_df(float* p, df v) { *p = rn_add(v.hi, v.lo); }
__device__ __forceinline__ void st_store_df(bf16* p, df v) {
  *reinterpret_cast<uint16_t*>(p) = dd_to_bf16_bits(v);
}

// The bf16 value every point of [y - e, y + e] rounds to, or -1 if the
// interval holds a rounding midpoint.  The half-width is widened by the
// rounding of y -/+ e itself.
__device__ __forceinline__ int certify_bf16(float y, float e) {
  const float w = e + fabsf(y) * 2.4e-7f + 1e-37f;
  const uint16_t lo = f32_to_bf16_bits(__fsub_rd(y, w)), hi = f32_to_bf16_bits(__fadd_ru(y, w));
  return lo == hi ? (int)lo : -1;
}

// gamma_n = n u / (1 - n u), u = 2^-24
__device__ __forceinline__ float gamma_n(int n) {
  const float nu = (float)n * 5.9604645e-8f;
  return nu / (1.0f - nu);
}

// Eight consecutive bf16 values (16-byte aligned) widened to float.
__device__ __forceinline__ void unpack8(uint4 v, float* z) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    z[2 * j] = __uint_as_float(w[j] << 16);
    z[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
  }
}

// Gates of draft step k for the state indices i = blockIdx + G t; (request,
// index) pairs strided over the threads.  `dsm` holds the fallback list
// (one int per pair at most).
template <typename DT>
__device__ void rnn_gates_body(const Shape& sh, int k, const DT* __restrict__ W1, const int* anchor,
                               const int* tokens, const RnnParams& rp, unsigned char* dsm) {
  const int r = sh.r, K = 2 * r, B = sh.B;
  const int G = gridDim.x;
  const int nI = (r - (int)blockIdx.x + G - 1) / G;
  if (nI <= 0) return;
  const DT* Wr = (const DT*)rp.Wr;
  DT* arows = (DT*)rp.arows + (size_t)k * B * r;
  const DT* s_in = (const DT*)rp.state + (size_t)(k & 1) * B * r;
  DT* s_out = (DT*)rp.state + (size_t)((k + 1) & 1) * B * r;
  const bool last = k == sh.gamma - 1;
  int* list = reinterpret_cast<int*>(dsm);
  __shared__ int s_n;
  __shared__ df s_tab[DD_EXP_TAB];
  __syncthreads();
  if (threadIdx.x == 0) s_n = 0;
  if (threadIdx.x < DD_EXP_TAB) dd_exp_table_entry(s_tab, threadIdx.x);
  __syncthreads();
  for (int p = threadIdx.x; p < nI * B; p += NT) {
    const int il = p / B, b = p - il * B, i = blockIdx.x + G * il;
    int need = last ? 1 : 3;                   // bit 0: a, bit 1: the next state
    if constexpr (sizeof(DT) == 2) {           // bf16: fp32 estimates can certify
      const int x = (k == 0) ? anchor[b] : __ldcg(tokens + (size_t)b * sh.gamma + k - 1);
      const DT* e = W1 + (size_t)min(max(x, 0), sh.V - 1) * r;
      const DT* s = s_in + (size_t)b * r;
      float acc[3][4], mag[3][4];
#pragma unroll
      for (int g = 0; g < 3; ++g)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[g][c] = mag[g][c] = 0.f;
      for (int t0 = (k == 0 ? r : 0); t0 < K; t0 += 8) {   // s_0 = 0
        float z[8], w[3][8];
        unpack8(t0 < r ? __ldcg(reinterpret_cast<const uint4*>(s + t0))
                       : __ldg(reinterpret_cast<const uint4*>(e + (t0 - r))), z);
#pragma unroll
        for (int g = 0; g < 3; ++g)
          unpack8(__ldg(reinterpret_cast<const uint4*>(Wr + (size_t)(g * r + i) * K + t0)), w[g]);
#pragma unroll
        for (int g = 0; g < 3; ++g)
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            acc[g][j & 3] = __fmaf_rn(w[g][j], z[j], acc[g][j & 3]);
            mag[g][j & 3] = __fmaf_rn(fabsf(w[g][j]), fabsf(z[j]), mag[g][j & 3]);
          }
      }
      const float* hp = rp.hproj + ((size_t)b * sh.gamma + k) * 3 * r;
      const float gam = gamma_n(K / 4 + 4);   // 4 chains of K/4 FMAs, 2 merges, + hproj
      float pre[3], err[3];
#pragma unroll
      for (int g = 0; g < 3; ++g) {
        const float h = hp[g * r + i];
        pre[g] = __fadd_rn(__fadd_rn(__fadd_rn(acc[g][0], acc[g][1]), __fadd_rn(acc[g][2], acc[g][3])), h);
        const float m = (mag[g][0] + mag[g][1]) + (mag[g][2] + mag[g][3]) + fabsf(h);
        err[g] = gam * m * 1.0001f;            // also covers the magnitude sum's rounding
      }
      // a = tanh(pre_o): |tanh'| <= 1; the fp32 tanh is within a few ulps
      const float a = tanhf(pre[2]);
      const int abits = certify_bf16(a, err[2] + fabsf(a) * 5e-7f);
      if (abits >= 0) {
        *reinterpret_cast<uint16_t*>(arows + (size_t)b * r + i) = (uint16_t)abits;
        need &= ~1;
      }
      if (!last) {
        const float gv = 1.0f / (1.0f + expf(-pre[0]));
        const float cv = tanhf(pre[1]);
        const float sv = (k == 0) ? 0.f : st_widen(s[i]);
        const float one_g = __fsub_rn(1.0f, gv);
        const float snew = __fadd_rn(__fmul_rn(gv, sv), __fmul_rn(one_g, cv));
        // propagated: logistic slope <= 1/4, tanh slope <= 1, a few ulps each;
        // the update's own four roundings: 6u of its terms
        const float dg = 0.25f * err[0] + gv * 5e-7f;
        const float dc = err[1] + fabsf(cv) * 5e-7f;
        const float ds = (fabsf(sv) + fabsf(cv)) * dg + one_g * dc +
                         3.6e-7f * (fabsf(gv * sv) + fabsf(one_g * cv));
        const int sbits = certify_bf16(snew, ds);
        if (sbits >= 0) {
          *reinterpret_cast<uint16_t*>(s_out + (size_t)b * r + i) = (uint16_t)sbits;
          need &= ~2;
        }
      }
    }
    if (need) list[atomicAdd(&s_n, 1)] = (p << 2) | need;
  }
  __syncthreads();
  // ---- double-float recomputation of the uncertified outputs, one warp each
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = s_n;
  for (int q = warp; q < n; q += NT / 32) {
    const int p = list[q] >> 2, need = list[q] & 3;
    const int il = p / B, b = p - il * B, i = blockIdx.x + G * il;
    const int x = (k == 0) ? anchor[b] : __ldcg(tokens + (size_t)b * sh.gamma + k - 1);
    const DT* e = W1 + (size_t)min(max(x, 0), sh.V - 1) * r;
    const DT* s = s_in + (size_t)b * r;
    DdDot d[3];
    for (int t = lane; t < K; t += 32) {
      const float z = t < r ? (k == 0 ? 0.f : st_widen(s[t])) : st_widen(e[t - r]);
#pragma unroll
      for (int g = 0; g < 3; ++g) d[g].add(st_widen(Wr[(size_t)(g * r + i) * K + t]), z);
    }
    const float* hp = rp.hproj + ((size_t)b * sh.gamma + k) * 3 * r;
    df pre[3];
#pragma unroll
    for (int g = 0; g < 3; ++g) pre[g] = dd_add_f(warp_sum_df(d[g].value()), hp[g * r + i]);
    if (lane == 0) {
      if (need & 1) st_store_df(arows + (size_t)b * r + i, dd_tanh(pre[2], s_tab));
      if (need & 2) {
        const df gv = dd_sigmoid(pre[0], s_tab);
        const df cv = dd_tanh(pre[1], s_tab);
        const float sv = (k == 0) ? 0.f : st_widen(s[i]);
        const df snew = dd_add(dd_mul_f(gv, sv), dd_mul(dd_add_f(dd_neg(gv), 1.0f), cv));
        st_store_df(s_out + (size_t)b * r + i, snew);
      }
    }
  }
}

}  // namespace spec
