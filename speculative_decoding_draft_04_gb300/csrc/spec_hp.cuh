// Extended-precision re-decision: shared device code (see spec_refine.cu for
// the method and its sources).  Data written by other CTAs of the same launch
// (queued items, block sums) is read through L2 (ld.global.cg) so the bodies
// also serve the persistent draft kernel.
#pragma once

#include "spec_gemm.cuh"

namespace spec {

// HpItem is 40 bytes, so array elements are only 8-byte aligned: load it with
// 8-byte accesses.
static_assert(sizeof(HpItem) == 40 && alignof(HpItem) == 8, "HpItem layout");
__device__ __forceinline__ HpItem ldcg_item(const HpItem* p) {
  HpItem h;
  const int2* q = reinterpret_cast<const int2*>(p);
  const int2 a = __ldcg(q), b = __ldcg(q + 1), c = __ldcg(q + 2);
  h.b = a.x; h.j = a.y; h.kind = b.x; h.prev = b.y;
  h.u = __int_as_float(c.x);
  h.fast_token = c.y;
  h.shift_q = __ldcg(&p->shift_q);
  h.shift_p = __ldcg(&p->shift_p);
  return h;
}

__device__ __forceinline__ void init_exp_table(double* tab) {
  if (threadIdx.x < 32) tab[threadIdx.x] = exp2((double)threadIdx.x / 32.0);
}

// e^x, |relative error| ~ 1e-15 for -745 < x < 700.
__device__ __forceinline__ double exp_tang(double x, const double* tab) {
  if (!(x > -745.0)) return 0.0;
  const double LN2 = 0.6931471805599453094172321;
  const double kd = rint(x * (32.0 / LN2));
  const double r = fma(-kd, LN2 / 32.0, x);
  const int k = (int)kd;
  const int j = k & 31;
  const int n = (k - j) >> 5;
  double p = 1.0 / 720.0;
  p = fma(p, r, 1.0 / 120.0);
  p = fma(p, r, 1.0 / 24.0);
  p = fma(p, r, 1.0 / 6.0);
  p = fma(p, r, 0.5);
  p = fma(p, r, 1.0);
  p = fma(p, r, 1.0);
  return ldexp(tab[j] * p, n);
}

// Tempered draft logit (U[v] + W1[x] W2[:, v]) / T with the bias as an
// error-free double-float sum.  `a` holds W1[x] widened to float.
template <typename DT>
__device__ __forceinline__ double hp_logit_q(const float* a, const DT* __restrict__ W2, int V, int r,
                                             const DT* __restrict__ Urow, int v, double invTd) {
  constexpr int UN = 16;                      // r % 16 == 0; loads run one batch ahead
  float s = 0.f, c = 0.f;
  float cur[UN];
#pragma unroll
  for (int u = 0; u < UN; ++u) cur[u] = ldf(W2 + (size_t)u * V + v);
  for (int i0 = 0; i0 < r; i0 += UN) {
    float nxt[UN];
    const bool more = i0 + UN < r;
#pragma unroll
    for (int u = 0; u < UN; ++u) nxt[u] = more ? ldf(W2 + (size_t)(i0 + UN + u) * V + v) : 0.f;
#pragma unroll
    for (int u = 0; u < UN; ++u) {
      const float w = cur[u];
      const float p = __fmul_rn(a[i0 + u], w);
      const float pe = fmaf(a[i0 + u], w, -p);   // 0 for bf16 operands
      float t, e;
      two_sum(s, p, t, e);
      s = t;
      c = __fadd_rn(c, __fadd_rn(e, pe));
    }
#pragma unroll
    for (int u = 0; u < UN; ++u) cur[u] = nxt[u];
  }
  return ((double)ldf(Urow + v) + ((double)s + (double)c)) * invTd;
}
// Same bias, W2 column `col` of a shared-memory slab [r][ld].
template <typename DT>
__device__ __forceinline__ double hp_logit_q_smem(const float* a, const DT* slab, int ld, int col,
                                                  int r, float Uv, double invTd) {
  float s = 0.f, c = 0.f;
  for (int i = 0; i < r; ++i) {
    const float w = tof(slab[(size_t)i * ld + col]);
    const float p = __fmul_rn(a[i], w);
    const float pe = fmaf(a[i], w, -p);
    float t, e;
    two_sum(s, p, t, e);
    s = t;
    c = __fadd_rn(c, __fadd_rn(e, pe));
  }
  return ((double)Uv + ((double)s + (double)c)) * invTd;
}
template <typename DT>
__device__ __forceinline__ double hp_logit_p(const DT* __restrict__ Trow, int v, double invTd) {
  return (double)ldf(Trow + v) * invTd;
}

// Exclusive prefix (double) of one value per thread, thread order.
__device__ __forceinline__ double block_excl_scan_d(double v, double* total, double* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  double inc = v;
  for (int d = 1; d < 32; d <<= 1) {
    double o = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += o;
  }
  __syncthreads();
  if (lane == 31) sh[w] = inc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double run = 0.0;
    for (int q = 0; q < NT / 32; ++q) {
      double t = sh[q];
      sh[q] = run;
      run += t;
    }
    sh[NT / 32] = run;
  }
  __syncthreads();
  double within = __shfl_up_sync(0xffffffffu, inc, 1);
  if (lane == 0) within = 0.0;
  double ex = sh[w] + within;
  *total = sh[NT / 32];
  __syncthreads();
  return ex;
}


template <typename DT>
struct ItemCtx {
  const DT* Urow;
  const DT* Trow;
  double invTd;
};

template <typename DT>
__device__ __forceinline__ ItemCtx<DT> item_ctx(const Shape& sh, const HpRows& R, const HpItem& it) {
  ItemCtx<DT> c;
  c.Urow = (const DT*)R.U + ((size_t)it.b * sh.gamma + (it.kind == HP_BONUS ? 0 : it.j)) * sh.V;
  c.Trow = (const DT*)R.target + ((size_t)it.b * (sh.gamma + 1) + it.j) * sh.V;
  c.invTd = 1.0 / (double)R.temp[it.b];
  return c;
}

// unnormalised extended-precision weights of entry v for an item
template <typename DT>
__device__ __forceinline__ void hp_weights(const Shape& sh, const HpRows& R, const HpItem& it,
                                           const ItemCtx<DT>& c, const float* a, const double* tab,
                                           int v, double& eq, double& ep) {
  eq = 0.0;
  ep = 0.0;
  if (v >= sh.V) return;
  if (it.kind != HP_BONUS)
    eq = exp_tang(hp_logit_q<DT>(a, (const DT*)R.W2, sh.V, sh.r, c.Urow, v, c.invTd) - it.shift_q, tab);
  if (it.kind != HP_DRAFT) ep = exp_tang(hp_logit_p<DT>(c.Trow, v, c.invTd) - it.shift_p, tab);
}

// Same weights with the W2 columns of block `blk` staged in `slab` ([r][HPB]).
template <typename DT>
__device__ __forceinline__ void hp_weights_slab(const Shape& sh, const HpItem& it,
                                                const ItemCtx<DT>& c, const float* a,
                                                const DT* slab, const double* tab, int v,
                                                double& eq, double& ep) {
  eq = 0.0;
  ep = 0.0;
  if (v >= sh.V) return;
  if (it.kind != HP_BONUS)
    eq = exp_tang(hp_logit_q_smem<DT>(a, slab, HPB, v % HPB, sh.r, ldf(c.Urow + v), c.invTd) -
                      it.shift_q, tab);
  if (it.kind != HP_DRAFT) ep = exp_tang(hp_logit_p<DT>(c.Trow, v, c.invTd) - it.shift_p, tab);
}

// Totals over the item's block sums, identical in every kernel (fixed order).
__device__ __forceinline__ double item_total(const double* sums, int HB, int col, double* shd) {
  double s = 0.0;
  for (int q = threadIdx.x; q < HB; q += NT) s += __ldcg(sums + (size_t)q * 3 + col);
  return block_sum_d(s, shd);
}

// Block sums of the n queued items' weights (phase 0) or residuals (phase 1),
// grid-stride over (item, block of HPB columns).  `dsm` holds r*HPB elements.
template <typename DT>
__device__ void hp_sums_body(const Shape& sh, const HpRows& R, const Ws& ws, int phase, int n,
                             unsigned char* dsm) {
  DT* slab = reinterpret_cast<DT*>(dsm);        // [r][HPB] W2 columns of one block
  __shared__ double tab[32];
  __shared__ double shd[40];
  __shared__ float s_a[256];
  init_exp_table(tab);
  __syncthreads();
  for (int w = blockIdx.x; w < n * sh.HB; w += gridDim.x) {
    const int item = w / sh.HB, blk = w - item * sh.HB;
    const HpItem it = ldcg_item(ws.items + item);
    if (phase == 1 && it.kind != HP_RESID) continue;
    __syncthreads();
    if (it.kind != HP_BONUS) {
      for (int i = threadIdx.x; i < sh.r; i += NT) s_a[i] = ldf((const DT*)R.W1 + (size_t)it.prev * sh.r + i);
      stage_w2_slab<DT>(slab, (const DT*)R.W2, sh.V, 0, sh.r, blk * HPB, HPB);
    }
    __syncthreads();
    const ItemCtx<DT> c = item_ctx<DT>(sh, R, it);
    const int v = blk * HPB + threadIdx.x;
    double eq, ep;
    hp_weights_slab<DT>(sh, it, c, s_a, slab, tab, v, eq, ep);
    double* sums = ws.hpsum + (size_t)item * sh.HB * 3;
    if (phase == 0) {
      double A = block_sum_d(it.kind == HP_DRAFT ? eq : ep, shd);
      double Bq = block_sum_d(eq, shd);
      if (threadIdx.x == 0) {
        sums[(size_t)blk * 3 + 0] = A;
        sums[(size_t)blk * 3 + 1] = Bq;
      }
    } else {
      const double Zp = item_total(sums, sh.HB, 0, shd);
      const double Zq = item_total(sums, sh.HB, 1, shd);
      double rr = (v < sh.V) ? fmax(0.0, ep / Zp - eq / Zq) : 0.0;
      double C = block_sum_d(rr, shd);
      if (threadIdx.x == 0) sums[(size_t)blk * 3 + 2] = C;
    }
  }
}

// Re-decide the n queued items: one CTA per item (grid-stride).
template <typename DT>
__device__ void hp_decide_body(const Shape& sh, const HpRows& R, const Ws& ws, int n, int* tokens,
                               float* q_tok, double* lse_q, int* out_tokens, uint32_t* status,
                               unsigned char* dsm) {
  DT* slab = reinterpret_cast<DT*>(dsm);        // [r][HPB] W2 columns of the crossing block
  __shared__ double tab[32];
  __shared__ double shd[40];
  __shared__ float s_a[256];
  __shared__ int s_blk, s_tok;
  __shared__ double s_pref, s_val;
  init_exp_table(tab);
  __syncthreads();
  for (int item = blockIdx.x; item < n; item += gridDim.x) {
    const HpItem it = ldcg_item(ws.items + item);
    const double* sums = ws.hpsum + (size_t)item * sh.HB * 3;
    const bool resid = it.kind == HP_RESID;
    double Zp = item_total(sums, sh.HB, 0, shd);
    double Zq = resid ? item_total(sums, sh.HB, 1, shd) : 0.0;
    double Zc = resid ? item_total(sums, sh.HB, 2, shd) : 0.0;
    // residual with no mass: draw from p (a probability-zero event)
    const bool empty = resid && !(Zc > 0.0);
    const int col = (resid && !empty) ? 2 : 0;
    const double Z = (resid && !empty) ? Zc : Zp;
    const double target = (double)it.u * Z;
    // crossing block
    const int per = (sh.HB + NT - 1) / NT;
    const int q0 = threadIdx.x * per, q1 = min(q0 + per, sh.HB);
    double loc = 0.0;
    for (int q = q0; q < q1; ++q) loc += __ldcg(sums + (size_t)q * 3 + col);
    double tot;
    double ex = block_excl_scan_d(loc, &tot, shd);
    if (threadIdx.x == 0) { s_blk = 0x7fffffff; s_tok = 0x7fffffff; }
    __syncthreads();
    int myb = -1;
    double mypref = 0.0;
    if (ex <= target && ex + loc > target) {
      double run = ex;
      for (int q = q0; q < q1; ++q) {
        double nx = run + __ldcg(sums + (size_t)q * 3 + col);
        if (nx > target) { myb = q; mypref = run; atomicMin(&s_blk, q); break; }
        run = nx;
      }
    }
    __syncthreads();
    if (myb >= 0 && myb == s_blk) s_pref = mypref;
    __syncthreads();
    bool fallback = false;
    if (s_blk == 0x7fffffff) {
      fallback = true;
      if (threadIdx.x == 0) {
        int q = sh.HB - 1;
        while (q > 0 && !(__ldcg(sums + (size_t)q * 3 + col) > 0.0)) --q;
        double run = 0.0;
        for (int t = 0; t < q; ++t) run += __ldcg(sums + (size_t)t * 3 + col);
        s_blk = q;
        s_pref = run;
      }
      __syncthreads();
    }
    const int blk = s_blk;
    // recompute the block
    if (it.kind != HP_BONUS) {
      for (int i = threadIdx.x; i < sh.r; i += NT) s_a[i] = ldf((const DT*)R.W1 + (size_t)it.prev * sh.r + i);
      stage_w2_slab<DT>(slab, (const DT*)R.W2, sh.V, 0, sh.r, blk * HPB, HPB);
    }
    __syncthreads();
    const ItemCtx<DT> c = item_ctx<DT>(sh, R, it);
    const int v = blk * HPB + threadIdx.x;
    double eq, ep;
    hp_weights_slab<DT>(sh, it, c, s_a, slab, tab, v, eq, ep);
    double val;
    if (it.kind == HP_DRAFT) val = eq;
    else if (resid && !empty) val = (v < sh.V) ? fmax(0.0, ep / Zp - eq / Zq) : 0.0;
    else val = ep;
    double btot;
    double bex = block_excl_scan_d(val, &btot, shd);
    const double tin = target - s_pref;
    if (val > 0.0 && bex <= tin && bex + val > tin) atomicMin(&s_tok, (int)threadIdx.x);
    __syncthreads();
    if (s_tok == 0x7fffffff) {
      // rounding left no crossing inside the block: last positive entry
      fallback = true;
      __syncthreads();
      if (threadIdx.x == 0) s_tok = -1;
      __syncthreads();
      if (val > 0.0) atomicMax(&s_tok, (int)threadIdx.x);
      __syncthreads();
      if (s_tok < 0) {
        if (threadIdx.x == 0) s_tok = 0;
        __syncthreads();
      }
    }
    if ((int)threadIdx.x == s_tok) s_val = val;
    __syncthreads();
    if (threadIdx.x == 0) {
      const int tok = blk * HPB + s_tok;
      if (it.kind == HP_DRAFT) {
        const size_t o = (size_t)it.b * sh.gamma + it.j;
        tokens[o] = tok;
        q_tok[o] = (float)(s_val / Z);
        lse_q[o] = it.shift_q + log(Z);
      } else {
        out_tokens[(size_t)it.b * (sh.gamma + 1) + it.j] = tok;
      }
      if (status) {
        atomicAdd(status + 1, 1u);
        if (tok != it.fast_token) atomicAdd(status + 2, 1u);
        atomicOr(status, (uint32_t)SPEC_DEV_REFINED);
      }
    }
    (void)fallback;
    __syncthreads();
  }
}

}  // namespace spec
