// Gate phase of the RNN head ("[논문리뷰] DSpark", section 1.2, "RNN head"):
// before the bias tiles of draft step k, every request's factor row
// a_k = tanh(W_o z) and next state s_{k+1} = sigma(W_g z) s_k +
// (1 - sigma(W_g z)) tanh(W_c z), z = [s_k; W1[x_k]; h], each rounded to the
// storage type.  The h block arrives as its three projections (hproj); the
// recurrent weights Wr = [W^s | W^e] are [3r][2r] (rows g, c, o).
//
// Certified rounding: each pre-activation is a fixed-order fp32 FMA sum whose
// error is bounded a posteriori by 2^-24 times the sum of the magnitudes of all
// its intermediate results; the fp32 tanh and logistic add a few ulps.  When the interval [y - err, y + err] of a result
// rounds to one bfloat16 value, that value is the rounding of the exact
// result; otherwise (a rounding midpoint inside the interval, about 1% of the
// outputs) a warp recomputes the row's pre-activations as Dot2 double-float
// dot products and takes the double-float logistic / tanh, correctly rounded.
// fp32 storage always takes the double-float route (no fp32 estimate can
// certify an fp32 rounding).
#pragma once

#include "spec_gemm.cuh"

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

// Requests whose gate inputs are staged in shared memory at a time (bf16).
constexpr int RNN_STAGE_ROWS = 128;

// Eight consecutive bf16 values (16-byte aligned) widened to float.
__device__ __forceinline__ void unpack8(uint4 v, float* z) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    z[2 * j] = __uint_as_float(w[j] << 16);
    z[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
  }
}

// Double-float recomputation of one (request, index)'s uncertified outputs by
// a warp: the three pre-activations as Dot2 sums over z = [s; W1[x]] (s read
// from `srow`, zero at k = 0; the embedding from `erow`) with the gate rows
// w + g * wstride, then the double-float logistic / tanh, correctly rounded.
template <typename DT, typename WT>
__device__ void gate_recompute(int r, int need, const DT* srow, bool s_zero, const DT* erow, const WT* w,
                               size_t wstride, const float* hp, int i, DT* a_out, DT* s_out,
                               const df* tab) {
  const int lane = threadIdx.x & 31;
  DdDot d[3];
  for (int t = lane; t < 2 * r; t += 32) {
    const float z = t < r ? (s_zero ? 0.f : st_widen(srow[t])) : st_widen(erow[t - r]);
#pragma unroll
    for (int g = 0; g < 3; ++g) d[g].add(st_widen(w[g * wstride + t]), z);
  }
  df pre[3];
#pragma unroll
  for (int g = 0; g < 3; ++g) pre[g] = dd_add_f(warp_sum_df(d[g].value()), hp[g * r + i]);
  if (lane == 0) {
    if (need & 1) st_store_df(a_out, dd_tanh(pre[2], tab));
    if (need & 2) {
      const df gv = dd_sigmoid(pre[0], tab);
      const df cv = dd_tanh(pre[1], tab);
      const float sv = s_zero ? 0.f : st_widen(srow[i]);
      st_store_df(s_out, dd_add(dd_mul_f(gv, sv), dd_mul(dd_add_f(dd_neg(gv), 1.0f), cv)));
    }
  }
}

// Gates of draft step k for the state indices i = blockIdx + G t; (request,
// index) pairs strided over the threads.  `dsm` holds the fallback list
// (one int per pair at most).
template <typename DT>
__device__ void rnn_gates_body(const Shape& sh, int k, const DT* __restrict__ W1, const int* anchor,
                               const int* tokens, const RnnParams& rp, unsigned char* dsm,
                               uint32_t* status) {
  const int r = sh.r, K = 2 * r, B = sh.B;
  const int G = gridDim.x;
  const int nI = (r - (int)blockIdx.x + G - 1) / G;
  if (nI <= 0) return;
  const DT* Wr = (const DT*)rp.Wr;
  DT* arows = (DT*)rp.arows + (size_t)k * B * r;
  const DT* s_in = (const DT*)rp.state + (size_t)k * B * r;        // s_k
  DT* s_out = (DT*)rp.state + (size_t)(k + 1) * B * r;              // s_{k+1}
  const bool last = k == sh.gamma - 1;
  int* list = reinterpret_cast<int*>(dsm);        // fp32: the whole list; bf16: after the stage
  __shared__ int s_n;
  __shared__ df s_tab[DD_EXP_TAB];
  __syncthreads();
  if (threadIdx.x == 0) s_n = 0;
  if (threadIdx.x < DD_EXP_TAB) dd_exp_table_entry(s_tab, threadIdx.x);
  __syncthreads();
  if constexpr (sizeof(DT) == 2) {
    // bf16: fp32 estimates certify the roundings.  The CTA's Wr rows and the
    // inputs z = [s; W1[x]] of up to RB requests at a time are staged in
    // shared memory by cp.async (all loads in flight at once).
    constexpr int RB = RNN_STAGE_ROWS;
    float* w_s = reinterpret_cast<float*>(dsm);                   // [nI][3][K], widened
    bf16* z_s = reinterpret_cast<bf16*>(w_s + (size_t)nI * 3 * K);   // [RB][K]
    list = reinterpret_cast<int*>(z_s + (size_t)RB * K);
    const int cpr = K / 8;                                        // 16-byte pieces per row
    for (int q = threadIdx.x; q < nI * 3 * cpr; q += NT) {
      const int row = q / cpr, piece = q - row * cpr;
      const int il = row / 3, g = row - il * 3, i = blockIdx.x + G * il;
      float wv[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(Wr + (size_t)(g * r + i) * K + piece * 8)), wv);
      float4* dst = reinterpret_cast<float4*>(w_s + (size_t)row * K + piece * 8);
      dst[0] = make_float4(wv[0], wv[1], wv[2], wv[3]);
      dst[1] = make_float4(wv[4], wv[5], wv[6], wv[7]);
    }
    __shared__ int s_x[RB];
    for (int b0 = 0; b0 < B; b0 += RB) {
      const int nb = min(RB, B - b0);
      // the group's previous tokens first (one load each, all in flight)
      for (int bl = threadIdx.x; bl < nb; bl += NT) {
        const int b = b0 + bl;
        const int x = (k == 0) ? anchor[b] : __ldcg(tokens + (size_t)b * sh.gamma + k - 1);
        s_x[bl] = min(max(x, 0), sh.V - 1);
      }
      __syncthreads();
      for (int q = threadIdx.x; q < nb * cpr; q += NT) {
        const int bl = q / cpr, piece = q - bl * cpr, b = b0 + bl, t0 = piece * 8;
        const DT* src;
        bool valid = true;
        if (t0 < r) {
          src = s_in + (size_t)b * r + t0;
          valid = k > 0;                                          // s_0 = 0: zero fill
        } else {
          src = W1 + (size_t)s_x[bl] * r + (t0 - r);
        }
        cp_async16(z_s + (size_t)bl * K + t0, valid ? src : W1, valid);
      }
      cp_async_commit();
      cp_async_wait_all();
      __syncthreads();
      for (int p = threadIdx.x; p < nI * nb; p += NT) {
        const int il = p / nb, bl = p - il * nb, b = b0 + bl, i = blockIdx.x + G * il;
        int need = last ? 1 : 3;                 // bit 0: a, bit 1: the next state
        const bf16* z = z_s + (size_t)bl * K;
        const float* wg = w_s + (size_t)il * 3 * K;
        float acc[3][4], mag[3][4];
#pragma unroll
        for (int g = 0; g < 3; ++g)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[g][c] = mag[g][c] = 0.f;
        for (int t0 = (k == 0 ? r : 0); t0 < K; t0 += 8) {
          float zz[8], w[3][8];
          unpack8(*reinterpret_cast<const uint4*>(z + t0), zz);
#pragma unroll
          for (int g = 0; g < 3; ++g) {
            const float4 w0 = *reinterpret_cast<const float4*>(wg + g * K + t0);
            const float4 w1 = *reinterpret_cast<const float4*>(wg + g * K + t0 + 4);
            w[g][0] = w0.x; w[g][1] = w0.y; w[g][2] = w0.z; w[g][3] = w0.w;
            w[g][4] = w1.x; w[g][5] = w1.y; w[g][6] = w1.z; w[g][7] = w1.w;
          }
#pragma unroll
          for (int g = 0; g < 3; ++g)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              acc[g][j & 3] = __fmaf_rn(w[g][j], zz[j], acc[g][j & 3]);
              mag[g][j & 3] += fabsf(acc[g][j & 3]);
            }
        }
        // A posteriori bound: every FMA or addition rounds once, by at most
        // u |its result|, and the local errors add up -- so u times the sum of
        // all intermediate results bounds the total (u = 2^-24).
        const float* hp = rp.hproj + ((size_t)b * sh.gamma + k) * 3 * r;
        float pre[3], err[3];
#pragma unroll
        for (int g = 0; g < 3; ++g) {
          const float h = hp[g * r + i];
          const float c01 = __fadd_rn(acc[g][0], acc[g][1]), c23 = __fadd_rn(acc[g][2], acc[g][3]);
          const float c = __fadd_rn(c01, c23);
          pre[g] = __fadd_rn(c, h);
          const float m = (mag[g][0] + mag[g][1]) + (mag[g][2] + mag[g][3]) + fabsf(c01) + fabsf(c23) +
                          fabsf(c) + fabsf(pre[g]);
          err[g] = 5.9604645e-8f * m * 1.001f + 1e-36f;   // 1.001: the magnitudes' own sum
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
          const float sv = (k == 0) ? 0.f : __bfloat162float(z[i]);
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
        if (need) list[atomicAdd(&s_n, 1)] = ((il * B + b) << 2) | need;
      }
      __syncthreads();
      // this group's uncertified outputs, from the staged rows
      const int n = s_n;
      for (int q = threadIdx.x >> 5; q < n; q += NT / 32) {
        const int p = list[q] >> 2, need = list[q] & 3;
        const int il = p / B, b = p - il * B, i = blockIdx.x + G * il, bl = b - b0;
        gate_recompute(r, need, (const DT*)(z_s + (size_t)bl * K), k == 0,
                           (const DT*)(z_s + (size_t)bl * K + r), w_s + (size_t)il * 3 * K,
                           (size_t)K, rp.hproj + ((size_t)b * sh.gamma + k) * 3 * r, i,
                           arows + (size_t)b * r + i, s_out + (size_t)b * r + i, s_tab);
      }
      __syncthreads();                           // z_s is restaged for the next group
      if (threadIdx.x == 0) {
        if (n) atomicAdd(status + 3, (uint32_t)n);   // recomputed outputs
        s_n = 0;
      }
    }
    return;
  } else {
    for (int p = threadIdx.x; p < nI * B; p += NT) list[atomicAdd(&s_n, 1)] = (p << 2) | (last ? 1 : 3);
  }
  __syncthreads();
  // ---- fp32 storage: every output in double-float, one warp each
  const int warp = threadIdx.x >> 5;
  const int n = s_n;
  if (threadIdx.x == 0 && n) atomicAdd(status + 3, (uint32_t)n);   // recomputed outputs
  for (int q = warp; q < n; q += NT / 32) {
    const int p = list[q] >> 2, need = list[q] & 3;
    const int il = p / B, b = p - il * B, i = blockIdx.x + G * il;
    const int x = (k == 0) ? anchor[b] : __ldcg(tokens + (size_t)b * sh.gamma + k - 1);
    gate_recompute(r, need, s_in + (size_t)b * r, k == 0, W1 + (size_t)min(max(x, 0), sh.V - 1) * r,
                       Wr + (size_t)i * K, (size_t)r * K, rp.hproj + ((size_t)b * sh.gamma + k) * 3 * r, i,
                       arows + (size_t)b * r + i, s_out + (size_t)b * r + i, s_tab);
  }
}

}  // namespace spec
