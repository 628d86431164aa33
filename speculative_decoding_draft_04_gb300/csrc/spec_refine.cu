// Extended-precision re-decision of near-boundary draws.
//
// The first pass (spec_draft.cu, spec_verify.cu) decides every draw in single
// precision and measures how far the uniform lies from the nearest CDF
// breakpoint.  Draws closer than the first pass's error band are re-decided
// here with per-vocabulary-entry weights accurate to ~1e-13, all in
// double-float arithmetic (spec_df.cuh) because GB300's fp64 rate is low:
//   - transition bias W1[x] W2 as a compensated (Kahan) sum of the products
//     (bf16 x bf16 products are exact in fp32; fp32 products carry their FMA
//     remainder),
//   - logits in double-float, exponentials by a double-float version of the
//     table-driven method of P. T. P. Tang, "Table-driven implementation of
//     the exponential function in IEEE floating-point arithmetic", ACM TOMS
//     15(2), 1989 (64-entry table of 2^(j/64), |r| <= ln2/128),
//   - block sums and scans in double-float, in a fixed order.
//
//   hp_sums_kernel    grid-stride over (item, block of HPB columns): block sums
//                     of the item's unnormalised weights (phase 0), or of the
//                     residual max(0, p - q) once the normalisers are known
//                     (phase 1, residual items only; the weights of the first
//                     items are kept from phase 0).  The CTA that completes an
//                     item's last block of its final pass re-decides it:
//                     crossing chunk from the chunk sums, that chunk
//                     recomputed and scanned, token written.
//   slow_verify_kernel one CTA per request whose ratio test itself was near
//                     its boundary: re-runs that request's verification with
//                     extended-precision normalisers (rare: the uniform must
//                     lie within a relative 1e-6 of the ratio).
#include "spec_hp.cuh"

namespace spec {

// Block sums of the verification's queued items; the CTA that completes an
// item's last block of its final pass re-decides it (writes out_tokens).
template <typename DT>
__global__ void __launch_bounds__(NT) hp_sums_kernel(Shape sh, HpRows R, Ws ws, int phase,
                                                     int* out_tokens, uint32_t* status) {
  extern __shared__ __align__(16) unsigned char dsm[];
  const int n = min((int)ws.ctrl[CTRL_ITEMS], ws.max_items);
  if (n == 0) return;
  hp_sums_body<DT>(sh, R, ws, phase, n, dsm, true, nullptr, nullptr, nullptr, status, out_tokens);
}

// ---------------------------------------------------------------- slow path
// One CTA re-verifies one request whose ratio test sat inside its error band.
template <typename DT>
__device__ df row_total(const Shape& sh, const HpRows& R, const HpItem& it, const ItemCtx<DT>& c,
                        const float* a, const df* tab, float* shf) {
  df s = {0.f, 0.f};
  for (int v = threadIdx.x; v < sh.V; v += NT) {
    df eq, ep;
    hp_weights<DT>(sh, R, it, c, a, tab, v, eq, ep);
    s = dd_add(s, (it.kind == HP_DRAFT) ? eq : ep);
  }
  return block_sum_df(s, shf);
}

template <typename DT>
__global__ void __launch_bounds__(NT) slow_verify_kernel(
    Shape sh, HpRows R, Ws ws, const int* __restrict__ anchor, const int* __restrict__ dtok,
    const double* __restrict__ lse_q, const int* __restrict__ vlen,
    const float* __restrict__ u_acc, const float* __restrict__ u_fin, int* accept_len,
    int* out_tokens, uint32_t* status) {
  __shared__ df tab[DD_EXP_TAB];
  __shared__ float shf[72];
  __shared__ float s_a[256];
  __shared__ df s_rc;
  __shared__ int s_tok, s_last;
  const int nslow = min((int)ws.ctrl[CTRL_SLOW], sh.B);
  if (nslow == 0) return;
  hp_table(tab);
  __syncthreads();
  for (int q = blockIdx.x; q < nslow; q += gridDim.x) {
    const int b = ws.slow[q];
    const int L = vlen[b];
    const uint32_t flags = (uint32_t)ws.vflags[b] >> 8;
    const uint32_t acc = ws.accbits[b];
    int n = L;
    int nhp = 0;
    for (int j = 0; j < L; ++j) {
      bool accept = (acc >> j) & 1u;
      if ((flags >> j) & 1u) {
        ++nhp;
        const int x = dtok[(size_t)b * sh.gamma + j];
        const int prev = factor_row(sh, b, j, j == 0 ? anchor[b] : dtok[(size_t)b * sh.gamma + j - 1]);
        HpItem ip; ip.b = b; ip.j = j; ip.kind = HP_BONUS; ip.prev = prev; ip.u = 0.f;
        ip.fast_token = -1; ip.shift_q = lse_q[(size_t)b * sh.gamma + j];
        ip.shift_p = ws.lse_p[(size_t)b * (sh.gamma + 1) + j];
        HpItem iq = ip; iq.kind = HP_DRAFT;
        __syncthreads();
        for (int i = threadIdx.x; i < sh.r; i += NT) s_a[i] = ldf((const DT*)R.W1 + (size_t)prev * sh.r + i);
        __syncthreads();
        const ItemCtx<DT> c = item_ctx<DT>(sh, R, iq);
        const double Zp = dd_to_double(row_total<DT>(sh, R, ip, c, s_a, tab, shf));
        const double Zq = dd_to_double(row_total<DT>(sh, R, iq, c, s_a, tab, shf));
        const df lpx = dd_add(dd_mul_f(c.invT, ldf(c.Trow + x)), c.nsp);
        const df lqx = dd_add(
            dd_mul(dd_add_f(hp_bias<DT>(s_a, (const DT*)R.W2, sh.V, sh.r, x), ldf(c.Urow + x)), c.invT),
            c.nsq);
        const double lp = dd_to_double(lpx) - log(Zp);
        const double lq = dd_to_double(lqx) - log(Zq);
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
    ip.prev = factor_row(sh, b, row, row == 0 ? anchor[b] : dtok[(size_t)b * sh.gamma + row - 1]);
    ip.shift_p = ws.lse_p[(size_t)b * (sh.gamma + 1) + row];
    ip.shift_q = resid ? lse_q[(size_t)b * sh.gamma + row] : 0.0;
    HpItem iq = ip; iq.kind = HP_DRAFT;
    HpItem ir = ip; ir.kind = resid ? HP_RESID : HP_BONUS;
    __syncthreads();
    if (resid)
      for (int i = threadIdx.x; i < sh.r; i += NT) s_a[i] = ldf((const DT*)R.W1 + (size_t)ip.prev * sh.r + i);
    __syncthreads();
    const ItemCtx<DT> c = item_ctx<DT>(sh, R, ir);
    const df Zp = row_total<DT>(sh, R, ip, c, s_a, tab, shf);
    const df Zq = resid ? row_total<DT>(sh, R, iq, c, s_a, tab, shf) : df{1.f, 0.f};
    const df izp = shared_recip(Zp, &s_rc);
    const df izq = shared_recip(Zq, &s_rc);
    // total residual mass
    double Zr = 0.0;
    if (resid) {
      df s = {0.f, 0.f};
      for (int v = threadIdx.x; v < sh.V; v += NT) {
        df eq, ep;
        hp_weights<DT>(sh, R, ir, c, s_a, tab, v, eq, ep);
        s = dd_add(s, hp_resid(ep, eq, izp, izq));
      }
      Zr = dd_to_double(block_sum_df(s, shf));
    }
    const bool use_r = resid && Zr > 0.0;
    const double Z = use_r ? Zr : dd_to_double(Zp);
    const double target = (double)ip.u * Z;
    double run = 0.0;
    if (threadIdx.x == 0) s_tok = 0x7fffffff;
    __syncthreads();
    int last_pos = -1;
    for (int v0 = 0; v0 < sh.V; v0 += NT) {
      const int v = v0 + threadIdx.x;
      df eq = {0.f, 0.f}, ep = {0.f, 0.f};
      hp_weights<DT>(sh, R, ir, c, s_a, tab, v, eq, ep);
      const df val = use_r ? ((v < sh.V) ? hp_resid(ep, eq, izp, izq) : df{0.f, 0.f}) : ep;
      df tot;
      const double ex = dd_to_double(block_excl_scan_df(val, &tot, shf));
      const double vd = dd_to_double(val);
      if (vd > 0.0 && run + ex <= target && run + ex + vd > target) atomicMin(&s_tok, v);
      if (vd > 0.0) last_pos = v;
      __syncthreads();
      if (s_tok != 0x7fffffff) break;
      run += dd_to_double(tot);
    }
    // no crossing found means rounding left the total at u*Z: last positive entry
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
cudaError_t launch_hp_sums(const Shape& sh, const HpRows& R, const Ws& ws, int phase, int* out_tokens,
                           uint32_t* status, int grid, cudaStream_t st) {
  const size_t smem = (size_t)sh.r * HPB * sizeof(DT);
  cudaError_t e = cudaFuncSetAttribute(hp_sums_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  hp_sums_kernel<DT><<<grid, NT, smem, st>>>(sh, R, ws, phase, out_tokens, status);
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
  template cudaError_t launch_hp_sums<DT>(const Shape&, const HpRows&, const Ws&, int, int*,    \
                                          uint32_t*, int, cudaStream_t);                        \
  template cudaError_t launch_slow_verify<DT>(const Shape&, const HpRows&, const Ws&, const int*, \
                                              const int*, const double*, const int*,           \
                                              const float*, const float*, int*, int*, uint32_t*, \
                                              int, cudaStream_t);
SPEC_INST(float)
SPEC_INST(bf16)
#undef SPEC_INST

}  // namespace spec
