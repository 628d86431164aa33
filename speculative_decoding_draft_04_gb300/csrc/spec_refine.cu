// Extended-precision re-decision of near-boundary draws.
//
// The first pass (spec_draft.cu, spec_verify.cu) decides every draw in single
// precision and measures how far the uniform lies from the nearest CDF
// breakpoint.  Draws closer than the first pass's error band are re-decided
// here with per-vocabulary-entry weights accurate to ~1e-15:
//   - transition bias W1[x] W2 as an exact double-float sum (bf16 x bf16
//     products are exact in fp32; fp32 products are split with an FMA;
//     partial sums are carried error-free with TwoSum),
//   - logits and exponentials in double precision; the exponential uses
//     the table-driven method of P. T. P. Tang, "Table-driven implementation
//     of the exponential function in IEEE floating-point arithmetic", ACM
//     TOMS 15(2), 1989 (32-entry table of 2^(j/32), degree-6 polynomial on
//     |r| <= ln2/64), which needs far fewer double operations than a general
//     libm-style exp -- GB300's double rate is low.
//
//   hp_sums_kernel    grid-stride over (item, block of HPB columns): block sums
//                     of the item's unnormalised weights (phase 0), or of the
//                     residual max(0, p - q) once the normalisers are known
//                     (phase 1, residual items only).
//   hp_decide_kernel  one CTA per item: crossing block from the block sums,
//                     recompute that block, scan, write the token.
//   slow_verify_kernel one CTA per request whose ratio test itself was near
//                     its boundary: re-runs that request's verification with
//                     extended-precision normalisers (rare).
#include "spec_gemm.cuh"

namespace spec {

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
  for (int q = threadIdx.x; q < HB; q += NT) s += sums[(size_t)q * 3 + col];
  return block_sum_d(s, shd);
}

template <typename DT>
__global__ void __launch_bounds__(NT) hp_sums_kernel(Shape sh, HpRows R, Ws ws, int phase) {
  extern __shared__ __align__(16) unsigned char dsm[];
  DT* slab = reinterpret_cast<DT*>(dsm);        // [r][HPB] W2 columns of one block
  __shared__ double tab[32];
  __shared__ double shd[40];
  __shared__ float s_a[256];
  const int n = min((int)ws.ctrl[CTRL_ITEMS], ws.max_items);
  if (n == 0) return;
  init_exp_table(tab);
  __syncthreads();
  for (int w = blockIdx.x; w < n * sh.HB; w += gridDim.x) {
    const int item = w / sh.HB, blk = w - item * sh.HB;
    const HpItem it = ws.items[item];
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

template <typename DT>
__global__ void __launch_bounds__(NT) hp_decide_kernel(Shape sh, HpRows R, Ws ws, int* tokens,
                                                       float* q_tok, double* lse_q,
                                                       int* out_tokens, uint32_t* status) {
  extern __shared__ __align__(16) unsigned char dsm[];
  DT* slab = reinterpret_cast<DT*>(dsm);        // [r][HPB] W2 columns of the crossing block
  __shared__ double tab[32];
  __shared__ double shd[40];
  __shared__ float s_a[256];
  __shared__ int s_blk, s_tok;
  __shared__ double s_pref, s_val;
  const int n = min((int)ws.ctrl[CTRL_ITEMS], ws.max_items);
  if (n == 0) return;
  init_exp_table(tab);
  __syncthreads();
  for (int item = blockIdx.x; item < n; item += gridDim.x) {
    const HpItem it = ws.items[item];
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
    for (int q = q0; q < q1; ++q) loc += sums[(size_t)q * 3 + col];
    double tot;
    double ex = block_excl_scan_d(loc, &tot, shd);
    if (threadIdx.x == 0) { s_blk = 0x7fffffff; s_tok = 0x7fffffff; }
    __syncthreads();
    int myb = -1;
    double mypref = 0.0;
    if (ex <= target && ex + loc > target) {
      double run = ex;
      for (int q = q0; q < q1; ++q) {
        double nx = run + sums[(size_t)q * 3 + col];
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
        while (q > 0 && !(sums[(size_t)q * 3 + col] > 0.0)) --q;
        double run = 0.0;
        for (int t = 0; t < q; ++t) run += sums[(size_t)t * 3 + col];
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

// ---------------------------------------------------------------- slow path
// One CTA re-verifies one request whose ratio test sat inside its error band.
template <typename DT>
__device__ double row_total(const Shape& sh, const HpRows& R, const HpItem& it, const float* a,
                            const double* tab, double* shd) {
  const ItemCtx<DT> c = item_ctx<DT>(sh, R, it);
  double s = 0.0;
  for (int v = threadIdx.x; v < sh.V; v += NT) {
    double eq, ep;
    hp_weights<DT>(sh, R, it, c, a, tab, v, eq, ep);
    s += (it.kind == HP_DRAFT) ? eq : ep;
  }
  return block_sum_d(s, shd);
}

template <typename DT>
__global__ void __launch_bounds__(NT) slow_verify_kernel(
    Shape sh, HpRows R, Ws ws, const int* __restrict__ anchor, const int* __restrict__ dtok,
    const double* __restrict__ lse_q, const int* __restrict__ vlen,
    const float* __restrict__ u_acc, const float* __restrict__ u_fin, int* accept_len,
    int* out_tokens, uint32_t* status) {
  __shared__ double tab[32];
  __shared__ double shd[40];
  __shared__ float s_a[256];
  __shared__ int s_tok;
  const int nslow = min((int)ws.ctrl[CTRL_SLOW], sh.B);
  if (nslow == 0) return;
  init_exp_table(tab);
  __syncthreads();
  for (int q = blockIdx.x; q < nslow; q += gridDim.x) {
    const int b = ws.slow[q];
    const int L = vlen[b];
    const uint32_t flags = (uint32_t)ws.vflags[b] >> 8;
    const uint32_t acc = ws.accbits[b];
    const double invTd = 1.0 / (double)R.temp[b];
    int n = L;
    int nhp = 0;
    for (int j = 0; j < L; ++j) {
      bool accept = (acc >> j) & 1u;
      if ((flags >> j) & 1u) {
        ++nhp;
        const int x = dtok[(size_t)b * sh.gamma + j];
        const int prev = j == 0 ? anchor[b] : dtok[(size_t)b * sh.gamma + j - 1];
        HpItem ip; ip.b = b; ip.j = j; ip.kind = HP_BONUS; ip.prev = prev; ip.u = 0.f;
        ip.fast_token = -1; ip.shift_q = lse_q[(size_t)b * sh.gamma + j];
        ip.shift_p = ws.lse_p[(size_t)b * (sh.gamma + 1) + j];
        HpItem iq = ip; iq.kind = HP_DRAFT;
        __syncthreads();
        for (int i = threadIdx.x; i < sh.r; i += NT) s_a[i] = ldf((const DT*)R.W1 + (size_t)prev * sh.r + i);
        __syncthreads();
        const double Zp = row_total<DT>(sh, R, ip, s_a, tab, shd);
        const double Zq = row_total<DT>(sh, R, iq, s_a, tab, shd);
        const ItemCtx<DT> c = item_ctx<DT>(sh, R, iq);
        const double lp = hp_logit_p<DT>(c.Trow, x, invTd) - ip.shift_p - log(Zp);
        const double lq = hp_logit_q<DT>(s_a, (const DT*)R.W2, sh.V, sh.r, c.Urow, x, invTd) -
                          iq.shift_q - log(Zq);
        const double ratio = exp(lp - lq);
        const bool nacc = (double)u_acc[(size_t)b * sh.gamma + j] < ratio;
        if (nacc != accept && threadIdx.x == 0 && status) atomicAdd(status + 2, 1u);
        accept = nacc;
      }
      if (!accept) { n = j; break; }
    }
    // final draw in extended precision
    const int row = n;
    const bool resid = n < L;
    HpItem ip; ip.b = b; ip.j = row; ip.kind = HP_BONUS; ip.u = u_fin[b]; ip.fast_token = -1;
    ip.prev = row == 0 ? anchor[b] : dtok[(size_t)b * sh.gamma + row - 1];
    ip.shift_p = ws.lse_p[(size_t)b * (sh.gamma + 1) + row];
    ip.shift_q = resid ? lse_q[(size_t)b * sh.gamma + row] : 0.0;
    HpItem iq = ip; iq.kind = HP_DRAFT;
    __syncthreads();
    if (resid)
      for (int i = threadIdx.x; i < sh.r; i += NT) s_a[i] = ldf((const DT*)R.W1 + (size_t)ip.prev * sh.r + i);
    __syncthreads();
    const double Zp = row_total<DT>(sh, R, ip, s_a, tab, shd);
    const double Zq = resid ? row_total<DT>(sh, R, iq, s_a, tab, shd) : 1.0;
    const ItemCtx<DT> c = item_ctx<DT>(sh, R, iq);
    // total residual mass
    double Zr = 0.0;
    if (resid) {
      double s = 0.0;
      for (int v = threadIdx.x; v < sh.V; v += NT) {
        double eq, ep;
        HpItem ir = ip; ir.kind = HP_RESID; ir.shift_q = iq.shift_q;
        hp_weights<DT>(sh, R, ir, c, s_a, tab, v, eq, ep);
        s += fmax(0.0, ep / Zp - eq / Zq);
      }
      Zr = block_sum_d(s, shd);
    }
    const bool use_r = resid && Zr > 0.0;
    const double Z = use_r ? Zr : Zp;
    const double target = (double)ip.u * Z;
    double run = 0.0;
    if (threadIdx.x == 0) s_tok = 0x7fffffff;
    __syncthreads();
    int last_pos = -1;
    for (int v0 = 0; v0 < sh.V; v0 += NT) {
      const int v = v0 + threadIdx.x;
      double eq = 0.0, ep = 0.0;
      HpItem ir = ip; ir.kind = resid ? HP_RESID : HP_BONUS; ir.shift_q = iq.shift_q;
      hp_weights<DT>(sh, R, ir, c, s_a, tab, v, eq, ep);
      double val = use_r ? ((v < sh.V) ? fmax(0.0, ep / Zp - eq / Zq) : 0.0) : ep;
      double tot;
      double ex = block_excl_scan_d(val, &tot, shd);
      if (val > 0.0 && run + ex <= target && run + ex + val > target) atomicMin(&s_tok, v);
      if (val > 0.0) last_pos = v;
      __syncthreads();
      if (s_tok != 0x7fffffff) break;
      run += tot;
    }
    // no crossing found means rounding left the total at u*Z: last positive entry
    __shared__ int s_last;
    if (threadIdx.x == 0) s_last = -1;
    __syncthreads();
    atomicMax(&s_last, last_pos);
    __syncthreads();
    if (threadIdx.x == 0) {
      const int tok = s_tok != 0x7fffffff ? s_tok : max(s_last, 0);
      int* out = out_tokens + (size_t)b * (sh.gamma + 1);
      for (int j = 0; j < n; ++j) out[j] = dtok[(size_t)b * sh.gamma + j];
      out[n] = tok;
      for (int j = n + 1; j <= sh.gamma; ++j) out[j] = -1;
      accept_len[b] = n;
      if (status) {
        atomicAdd(status + 3, 1u);
        atomicAdd(status + 1, (uint32_t)(nhp + 1));
        atomicOr(status, (uint32_t)SPEC_DEV_REFINED);
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- launchers
template <typename DT>
cudaError_t launch_hp_sums(const Shape& sh, const HpRows& R, const Ws& ws, int phase, int grid,
                           cudaStream_t st) {
  const size_t smem = (size_t)sh.r * HPB * sizeof(DT);
  cudaError_t e = cudaFuncSetAttribute(hp_sums_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  hp_sums_kernel<DT><<<grid, NT, smem, st>>>(sh, R, ws, phase);
  return cudaGetLastError();
}
template <typename DT>
cudaError_t launch_hp_decide(const Shape& sh, const HpRows& R, const Ws& ws, int* tokens,
                             float* q_tok, double* lse_q, int* out_tokens, uint32_t* status,
                             int grid, cudaStream_t st) {
  const size_t smem = (size_t)sh.r * HPB * sizeof(DT);
  cudaError_t e = cudaFuncSetAttribute(hp_decide_kernel<DT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  hp_decide_kernel<DT><<<grid, NT, smem, st>>>(sh, R, ws, tokens, q_tok, lse_q, out_tokens, status);
  return cudaGetLastError();
}
template <typename DT>
cudaError_t launch_slow_verify(const Shape& sh, const HpRows& R, const Ws& ws, const int* anchor,
                               const int* dtok, const double* lse_q, const int* vlen,
                               const float* u_acc, const float* u_fin, int* accept_len,
                               int* out_tokens, uint32_t* status, int grid, cudaStream_t st) {
  slow_verify_kernel<DT><<<grid, NT, 0, st>>>(sh, R, ws, anchor, dtok, lse_q, vlen, u_acc, u_fin,
                                              accept_len, out_tokens, status);
  return cudaGetLastError();
}

#define SPEC_INST(DT)                                                                            \
  template cudaError_t launch_hp_sums<DT>(const Shape&, const HpRows&, const Ws&, int, int,     \
                                          cudaStream_t);                                        \
  template cudaError_t launch_hp_decide<DT>(const Shape&, const HpRows&, const Ws&, int*, float*, \
                                            double*, int*, uint32_t*, int, cudaStream_t);       \
  template cudaError_t launch_slow_verify<DT>(const Shape&, const HpRows&, const Ws&, const int*, \
                                              const int*, const double*, const int*,           \
                                              const float*, const float*, int*, int*, uint32_t*, \
                                              int, cudaStream_t);
SPEC_INST(float)
SPEC_INST(bf16)
#undef SPEC_INST

}  // namespace spec
