// Verify side: the lossless acceptance step ("Speculative Decoding Part 1",
// VESSL AI blog, section "알고리즘": ratio tests of all positions after one
// target pass, first reject n, correction token from normalize(relu(p_n -
// q_n)) or bonus token from p_L; section "수락 규칙": residual distribution
// and alpha = sum_v min(p, q)), with a per-request verify length L_b
// (DSpark review, section 2.2).
//
//   verify_prep_kernel   validate requests, pack the draft rows (b, j < L_b)
//                        densely (prefix sum of L_b), reset counters.
//   target_stats_kernel  one CTA per target row j <= L_b: logsumexp of t/T by
//                        streaming the row once (per-slice max-referenced sums
//                        merged online); the bonus row also keeps its slice sums.
//   verify_tile_kernel   packed draft rows x vocabulary slices: recompute the
//                        Markov bias tile on the tensor path, form q and p in
//                        registers and reduce sum min(p, q), sum max(0, p - q)
//                        and the error-estimate sums per slice.
//   verify_final_kernel  one CTA per request: alpha, ratio tests and first
//                        reject (warp ballot), then the correction or bonus
//                        draw (crossing slice from the slice sums, that slice
//                        recomputed and scanned).  Near-boundary draws are queued
//                        for extended-precision re-decision (spec_refine.cu).
#include <cstring>

#include "spec_tile_tc.cuh"
#include "spec_tmap.cuh"

namespace spec {

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ df fast_two_sum(float a, float b) {
  float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
// c * t for float c and double-float t
__device__ __forceinline__ df mul_f_df(float c, df t) {
  float p = __fmul_rn(c, t.hi);
  float e = fmaf(c, t.hi, -p);
  e = fmaf(c, t.lo, e);
  return fast_two_sum(p, e);
}
__device__ __forceinline__ float exp_df(df g) { return __fmul_rn(expf(g.hi), __fadd_rn(1.0f, g.lo)); }
// Factor turning exp(x) (x relative to reference c) into a normalised
// probability: exp(c/T - lse) with 1/T and -lse carried as double-float.
__device__ __forceinline__ float norm_factor(float c, df invT, df nlse) {
  return exp_df(df_add(mul_f_df(c, invT), nlse));
}
__device__ __forceinline__ df d2df(double x) {
  float h = (float)x;
  return {h, (float)(x - (double)h)};
}

// Unnormalised verification weights relative to a slice reference c, with
// s2 = log2(e) / T folded in: q = 2^(((U - c) + bias) s2), p = 2^((t - c) s2)
// (one hardware exp2 each).  The tile epilogue and the final draw's slice
// recompute use these same two expressions.
constexpr float LOG2E_F = 1.44269504f;
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float vq(float u, float c, float bias, float s2) {
  return ex2_approx(__fmul_rn(__fadd_rn(__fsub_rn(u, c), bias), s2));
}
__device__ __forceinline__ float vp(float t, float c, float s2) {
  return ex2_approx(__fmul_rn(__fsub_rn(t, c), s2));
}

// 8 consecutive values (16-byte aligned)
__device__ __forceinline__ void load8(const bf16* p, float* v) {
  uint4 q = *reinterpret_cast<const uint4*>(p);
  const bf16* h = reinterpret_cast<const bf16*>(&q);
#pragma unroll
  for (int e = 0; e < 8; ++e) v[e] = __bfloat162float(h[e]);
}
__device__ __forceinline__ void load8(const float* p, float* v) {
  float4 a = *reinterpret_cast<const float4*>(p);
  float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// ---------------------------------------------------------------- prep
__global__ void __launch_bounds__(NT) verify_prep_kernel(
    Shape sh, const int* __restrict__ anchor, const float* __restrict__ temp,
    const int* __restrict__ dtok, const double* __restrict__ lse_q, const int* __restrict__ vlen,
    Ws ws, uint32_t* status, int* accept_len, int* out_tokens, float* alpha, float* p_tok) {
  __shared__ int s_w[NT / 32 + 1];
  const int per = (sh.B + NT - 1) / NT;
  const int b0 = threadIdx.x * per, b1 = min(b0 + per, sh.B);
  int local = 0;
  for (int b = b0; b < b1; ++b) {
    const int L = vlen[b];
    uint32_t bits = 0;
    if (L < 0 || L > sh.gamma) bits |= SPEC_DEV_BAD_LEN;
    if (!temp_ok(temp[b])) bits |= SPEC_DEV_BAD_TEMP;
    const int a = anchor[b];
    if (a < 0 || a >= sh.V) bits |= SPEC_DEV_BAD_TOKEN;
    if (!(bits & SPEC_DEV_BAD_LEN)) {
      // all of the row's tokens loaded at once (independent loads)
      int xs[MAX_GAMMA];
#pragma unroll
      for (int j = 0; j < MAX_GAMMA; ++j) xs[j] = j < L ? dtok[(size_t)b * sh.gamma + j] : 0;
#pragma unroll
      for (int j = 0; j < MAX_GAMMA; ++j)
        if (xs[j] < 0 || xs[j] >= sh.V) bits |= SPEC_DEV_BAD_TOKEN;
    }
    ws.vflags[b] = bits ? 1 : 0;
    ws.accbits[b] = 0;
    if (bits) {
      set_status(status, bits);
      accept_len[b] = -1;
      for (int j = 0; j <= sh.gamma; ++j) out_tokens[(size_t)b * (sh.gamma + 1) + j] = -1;
      for (int j = 0; j < sh.gamma; ++j) {
        alpha[(size_t)b * sh.gamma + j] = NAN;
        if (p_tok) p_tok[(size_t)b * sh.gamma + j] = NAN;
      }
    } else {
      local += L;
    }
  }
  // exclusive scan of the per-thread counts
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int inc = local;
  for (int d = 1; d < 32; d <<= 1) {
    int o = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += o;
  }
  if (lane == 31) s_w[w] = inc;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int q = 0; q < NT / 32; ++q) {
      int t = s_w[q];
      s_w[q] = run;
      run += t;
    }
    s_w[NT / 32] = run;
  }
  __syncthreads();
  int run = s_w[w] + inc - local;
  for (int b = b0; b < b1; ++b) {
    ws.rowptr[b] = run;
    if (ws.vflags[b] & 1) continue;
    const int L = vlen[b];
    const df it = dd_recip(temp[b]);
    const int a = anchor[b];
    int xs[MAX_GAMMA];
    double lq[MAX_GAMMA];
#pragma unroll
    for (int j = 0; j < MAX_GAMMA; ++j) {
      xs[j] = j < L ? dtok[(size_t)b * sh.gamma + j] : 0;
      lq[j] = j < L ? lse_q[(size_t)b * sh.gamma + j] : 0.0;
    }
#pragma unroll
    for (int j = 0; j < MAX_GAMMA; ++j) {
      if (j < L) {
        ws.prow[run + j] = make_int2(b, j);
        ws.prevtok[run + j] = factor_row(sh, b, j, j == 0 ? a : xs[j - 1 < 0 ? 0 : j - 1]);
        const df nlq = d2df(-lq[j]);
        ws.rowc[run + j] = make_float4(it.hi, it.lo, nlq.hi, nlq.lo);
      }
    }
    run += L;
  }
  if (threadIdx.x == NT - 1) {
    ws.rowptr[sh.B] = s_w[NT / 32];
    ws.ctrl[CTRL_NPACKED] = s_w[NT / 32];
    ws.ctrl[CTRL_ITEMS] = 0;
    ws.ctrl[CTRL_BAR_COUNT] = 0;       // the re-decision launch's grid barrier
    ws.ctrl[CTRL_ABORT] = 0;
    ws.ctrl[CTRL_SLOW] = 0;
  }
  // per-item block counters of the re-decision passes start at zero
  for (int i = threadIdx.x; i < ws.max_items; i += NT) ws.hpcnt[i] = 0u;
}

// ---------------------------------------------------------------- target statistics
// Merge of per-thread log-sum-exp partials (reference m, sum acc of
// exp((x - m)/T)) over the block; returns (M, Z) to every thread.
__device__ __forceinline__ void lse_merge(float& m, df& acc, float invT, float* sh) {
  auto comb = [&](float m2, df a2) {
    const float mn = fmaxf(m, m2);
    if (mn == -INFINITY) return;
    const df x = m == -INFINITY ? df{0.f, 0.f} : df_mulf(acc, expf(fast_tx(m, mn, invT)));
    const df y = m2 == -INFINITY ? df{0.f, 0.f} : df_mulf(a2, expf(fast_tx(m2, mn, invT)));
    acc = df_add(x, y);
    m = mn;
  };
  for (int o = 16; o; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const df a2 = shfl_xor_df(acc, o);
    comb(m2, a2);
  }
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) { sh[3 * w] = m; sh[3 * w + 1] = acc.hi; sh[3 * w + 2] = acc.lo; }
  __syncthreads();
  if (w == 0) {
    m = lane < NT / 32 ? sh[3 * lane] : -INFINITY;
    acc = lane < NT / 32 ? df{sh[3 * lane + 1], sh[3 * lane + 2]} : df{0.f, 0.f};
    for (int o = 16; o; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const df a2 = shfl_xor_df(acc, o);
      comb(m2, a2);
    }
    if (lane == 0) { sh[0] = m; sh[1] = acc.hi; sh[2] = acc.lo; }
  }
  __syncthreads();
  m = sh[0];
  acc = {sh[1], sh[2]};
  __syncthreads();
}

// One CTA per target row j <= L_b of request b: its logsumexp; the bonus row
// (j = L_b) also writes the per-VB-slice partials (c, s, p2) its draw needs.
// 8 consecutive values from a raw 16-byte word of bf16 data.
__device__ __forceinline__ void unpack8(const uint4& q, float* v) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    v[2 * e] = bf_lo(w[e]);
    v[2 * e + 1] = bf_hi(w[e]);
  }
}

template <typename DT>
__global__ void __launch_bounds__(NT, 3) target_stats_kernel(Shape sh, const DT* __restrict__ target,
                                                          const float* __restrict__ temp,
                                                          const int* __restrict__ vlen, Ws ws) {
  __shared__ float s_m[3 * (NT / 32)];
  __shared__ df s_tab[DD_EXP_TAB];
  const int j = blockIdx.x, b = blockIdx.y;
  if (ws.vflags[b] & 1) return;
  const int L = vlen[b];
  if (j > L) return;
  if (threadIdx.x < DD_EXP_TAB) dd_exp_table_entry(s_tab, threadIdx.x);
  const float T = temp[b];
  const float invT = 1.0f / T;
  const DT* row = target + ((size_t)b * (sh.gamma + 1) + j) * sh.V;
  float mref = -INFINITY;
  df acc = {0.f, 0.f};
  if (j == L) {
    // bonus row: GS threads (8 columns each) per VB-column slice; every lane
    // runs the same trip count (full-warp shuffles); UNR slices' loads issued
    // before any is reduced
    // (bf16 rows keep the raw 16-byte words of 8 slices in flight; fp32 rows
    // load 4 slices at a time)
    constexpr int GS = VB / 8, NG = NT / GS, UNR = sizeof(DT) == 2 ? 8 : 4;
    const int hw = threadIdx.x / GS, hl = threadIdx.x % GS;
    for (int base = 0; base < sh.NSV; base += NG * UNR) {
      uint4 raw[sizeof(DT) == 2 ? UNR : 1];
      float fv[sizeof(DT) == 2 ? 1 : UNR][8];
      bool ok[UNR];
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const int s = base + hw + NG * u;
        const int n = s * VB + hl * 8;
        ok[u] = s < sh.NSV && n < sh.V;
        if constexpr (sizeof(DT) == 2) {
          if (ok[u]) raw[u] = __ldcs(reinterpret_cast<const uint4*>(row + n));
        } else {
          if (ok[u]) load8(row + n, fv[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const int s = base + hw + NG * u;
        float vv[8];
        if constexpr (sizeof(DT) == 2) {
          if (ok[u]) unpack8(raw[u], vv);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) vv[e] = fv[u][e];
        }
        float (&vals_u)[8] = vv;
        float c = -INFINITY;
        if (ok[u])
#pragma unroll
          for (int e = 0; e < 8; ++e) c = fmaxf(c, vals_u[e]);
#pragma unroll
        for (int m = GS / 2; m; m >>= 1) c = fmaxf(c, __shfl_xor_sync(0xffffffffu, c, m));
        float ssum = 0.f, p2 = 0.f;
        if (ok[u])
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float wv = __expf(fast_tx(vals_u[e], c, invT));
            ssum = __fadd_rn(ssum, wv);
            p2 = fmaf(wv, wv, p2);
          }
#pragma unroll
        for (int m = GS / 2; m; m >>= 1) {
          ssum += __shfl_xor_sync(0xffffffffu, ssum, m);
          p2 += __shfl_xor_sync(0xffffffffu, p2, m);
        }
        if (s >= sh.NSV || hl != 0) continue;        // one lane per group accumulates
        ws.bpart[(size_t)b * sh.NSV + s] = make_float4(c, ssum, p2, 0.f);
        if (c > mref) {
          if (mref != -INFINITY) acc = df_mulf(acc, expf(fast_tx(mref, c, invT)));
          mref = c;
          acc = df_addf(acc, ssum);
        } else {
          acc = df_addf(acc, __fmul_rn(ssum, expf(fast_tx(c, mref, invT))));
        }
      }
    }
  } else {
    // other rows: per-thread online max and compensated sum over 16-byte
    // chunks strided by the block (coalesced), UNR chunks' loads in flight
    // (five CTAs per SM keep every row of a cycle resident at once)
    constexpr int UNR = sizeof(DT) == 2 ? 8 : 4;
    const int nch = sh.V / 8;
    for (int c0 = threadIdx.x; c0 < nch; c0 += NT * UNR) {
      uint4 raw[sizeof(DT) == 2 ? UNR : 1];
      float fv[sizeof(DT) == 2 ? 1 : UNR][8];
      bool ok[UNR];
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const int c = c0 + NT * u;
        ok[u] = c < nch;
        if constexpr (sizeof(DT) == 2) {
          if (ok[u]) raw[u] = __ldcs(reinterpret_cast<const uint4*>(row + (size_t)c * 8));
        } else {
          if (ok[u]) load8(row + (size_t)c * 8, fv[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        if (!ok[u]) continue;
        float vals_u[8];
        if constexpr (sizeof(DT) == 2) {
          unpack8(raw[u], vals_u);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) vals_u[e] = fv[u][e];
        }
        float c = vals_u[0];
#pragma unroll
        for (int e = 1; e < 8; ++e) c = fmaxf(c, vals_u[e]);
        if (c > mref) {
          if (mref != -INFINITY) acc = df_mulf(acc, expf(fast_tx(mref, c, invT)));
          mref = c;
        }
        float ssum = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ssum = __fadd_rn(ssum, __expf(fast_tx(vals_u[e], mref, invT)));
        acc = df_addf(acc, ssum);
      }
    }
  }
  lse_merge(mref, acc, invT, s_m);
  if (threadIdx.x == 0) {
    // lse = M / T + log Z (double-float steps; fp64 only to assemble the result)
    const double lse = dd_to_double(dd_mul_f(dd_recip(T), mref)) + dd_log(acc, s_tab);
    ws.lse_p[(size_t)b * (sh.gamma + 1) + j] = lse;
    const df nlp = d2df(-lse);
    ws.rowp[(size_t)b * (sh.gamma + 1) + j] = make_float2(nlp.hi, nlp.lo);
  }
}

// ---------------------------------------------------------------- alpha / residual tiles
template <typename DT, int BM, int PATH>
__global__ void __launch_bounds__(NT) verify_tile_kernel(Shape sh, const DT* __restrict__ target,
                                                         const DT* __restrict__ U,
                                                         const DT* __restrict__ W1,
                                                         const DT* __restrict__ W2, Ws ws,
                                                         uint32_t* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int s_tok[BM];
  __shared__ size_t s_offu[BM], s_offt[BM];
  const int P = (int)ws.ctrl[CTRL_NPACKED];
  const int slice = blockIdx.x, m0 = blockIdx.y * BM, n0 = slice * BN;
  if (m0 >= P) return;
  const int nrows = min(BM, P - m0);
  for (int m = threadIdx.x; m < BM; m += NT) {
    if (m < nrows) {
      const int2 bj = ws.prow[m0 + m];
      s_tok[m] = ws.prevtok[m0 + m];
      s_offu[m] = ((size_t)bj.x * sh.gamma + bj.y) * sh.V;
      s_offt[m] = ((size_t)bj.x * (sh.gamma + 1) + bj.y) * sh.V;
    } else {
      s_tok[m] = 0;
      s_offu[m] = 0;
      s_offt[m] = 0;
    }
  }
  static_assert(PATH == 0 || PATH == 1, "the tensor-memory path is verify_tiles_tc_kernel");
  (void)status;
  DT *Us, *Ts;
  float* stage;
  int su;
  {
    const TileLayout<DT> lay(BM, sh.r, true);
    DT* As = reinterpret_cast<DT*>(smem_raw + lay.offA);
    DT* Wsm = reinterpret_cast<DT*>(smem_raw + lay.offW);
    Us = reinterpret_cast<DT*>(smem_raw + lay.offU);
    Ts = reinterpret_cast<DT*>(smem_raw + lay.offT);
    stage = reinterpret_cast<float*>(smem_raw + lay.offStage);
    su = lay.su;
    __syncthreads();
    load_A_rows<DT>(As, lay.sa, W1, s_tok, nrows, BM, sh.r);
    load_W2_tile<DT>(Wsm, lay.sw, W2, sh.V, n0, sh.r);
    load_X_rows<DT>(Us, lay.su, U, s_offu, nrows, BM, sh.V, n0);
    load_X_rows<DT>(Ts, lay.su, target, s_offt, nrows, BM, sh.V, n0);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    bias_tile<DT, BM, PATH == 0>(As, lay.sa, Wsm, lay.sw, sh.r, stage);
    __syncthreads();
  }

  // epilogue: TPR threads per row, COLS columns each; one partial per
  // VB-column slice (SPL threads share a slice, or a thread covers CPT slices)
  constexpr int TPR = NT / BM, COLS = BN / TPR;
  constexpr int SPAN = COLS < VB ? COLS : VB;
  constexpr int CPT = COLS / SPAN, SPL = VB / SPAN;
  constexpr int SS = TileLayout<DT>::SS;
  const int m = threadIdx.x / TPR, part = threadIdx.x % TPR;
  const bool rowok = m < nrows;
  const int p = m0 + m;
  float4 rc = make_float4(1.f, 0.f, 0.f, 0.f);
  float2 rp = make_float2(0.f, 0.f);
  if (rowok) {
    const int2 bj = ws.prow[p];
    rc = ws.rowc[p];
    rp = ws.rowp[(size_t)bj.x * (sh.gamma + 1) + bj.y];
  }
  const float invT = rc.x;
  const DT* urow = Us + (size_t)m * su;
  const DT* trow = Ts + (size_t)m * su;
  const float* brow = stage + m * SS;
#pragma unroll
  for (int q = 0; q < CPT; ++q) {
    const int cbeg = part * COLS + q * SPAN;
    const int cend = min(cbeg + SPAN, sh.V - n0);
    float cU = -INFINITY, cT = -INFINITY;
    for (int i = cbeg; i < cend; ++i) {
      cU = fmaxf(cU, tof(urow[i]));
      cT = fmaxf(cT, tof(trow[i]));
    }
    cU = group_max<SPL>(cU);
    cT = group_max<SPL>(cT);
    const float Fq = norm_factor(cU, {rc.x, rc.y}, {rc.z, rc.w});
    const float Fp = norm_factor(cT, {rc.x, rc.y}, {rp.x, rp.y});
    float al = 0.f, p2 = 0.f, q2 = 0.f;
    Kahan kr;
    const float s2 = __fmul_rn(invT, LOG2E_F);
    for (int i = cbeg; i < cend; ++i) {
      const float qv = __fmul_rn(vq(tof(urow[i]), cU, brow[i], s2), Fq);
      const float pv = __fmul_rn(vp(tof(trow[i]), cT, s2), Fp);
      al += fminf(pv, qv);
      kr.add(fmaxf(0.f, __fsub_rn(pv, qv)));
      p2 = fmaf(pv, pv, p2);
      q2 = fmaf(qv, qv, q2);
    }
    al = group_sum<SPL>(al);
    const df res = group_sum_df<SPL>(kr.value());
    p2 = group_sum<SPL>(p2);
    q2 = group_sum<SPL>(q2);
    const int vs = (n0 + cbeg) / VB;
    if (rowok && part % SPL == 0 && vs < sh.NSV)
      ws.vpart[(size_t)p * sh.NSV + vs] = make_float4(al, df_d(res), p2, q2);
  }
}

// ---------------------------------------------------------------- tensor-memory tiles
// Verification tiles on the warp-specialised engine (spec_tile_tc.cuh), VB =
// 64 columns per tile: the packed draft rows p = (b, j < L_b) in request
// tiles of 128, their previous tokens' W1 rows as the A operand, and per row
// the slice partial (sum min(p, q), sum max(0, p - q), sum p^2, sum q^2).
struct VerifyEpi {
  static constexpr bool kHelpGather = false;
  const Shape& sh;
  const bf16* U;
  const bf16* T;
  const Ws& ws;
  int P;              // packed rows

  __device__ int token(int mt, int m) const {
    const int p = mt * TC_M + m;
    return p < P ? min(max(ws.prevtok[p], 0), sh.NA - 1) : -1;
  }
  // Row offsets of the producer lane's rows (lane + 32 i) for request tile
  // `cmt`, refreshed when the request tile changes.
  mutable int cmt = -1;
  mutable size_t offu[TC_M / 32], offt[TC_M / 32];
  __device__ void rows_of(int mt, int lane) const {
    if (mt == cmt) return;
    cmt = mt;
#pragma unroll
    for (int i = 0; i < TC_M / 32; ++i) {
      const int p = mt * TC_M + lane + 32 * i;
      offu[i] = offt[i] = ~(size_t)0;
      if (p < P) {
        const int2 bj = ws.prow[p];
        offu[i] = ((size_t)bj.x * sh.gamma + bj.y) * sh.V;
        offt[i] = ((size_t)bj.x * (sh.gamma + 1) + bj.y) * sh.V;
      }
    }
  }
  // U and target rows of the tile's 128 packed rows (lane: rows lane + 32 i),
  // VT = 64 columns = 8 chunks of 16 bytes each, 128-byte swizzle; U at xb,
  // the target rows 16 KB further.  Then the next tile's row segments are
  // prefetched into L2 (one 128-byte line per row and tensor).
  __device__ void load_x(int mt, int sl, unsigned char* xb, uint64_t* full, int lane, int nmt,
                         int nsl) const {
    rows_of(mt, lane);
    const int n0 = sl * VT;
#pragma unroll
    for (int i = 0; i < TC_M / 32; ++i) {
      const int m = lane + 32 * i;
      const bool rv = offu[i] != ~(size_t)0;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int n = n0 + 8 * c;
        const bool valid = rv && n < sh.V;
        unsigned char* dst = xb + m * 128 + ((c ^ (m & 7)) << 4);
        cp_async16(dst, valid ? U + offu[i] + n : U, valid);
        cp_async16(dst + TC_M * 128, valid ? T + offt[i] + n : T, valid);
      }
    }
    cp_async_arrive(full);
    if (nmt >= 0) {
      rows_of(nmt, lane);
      const int m0 = nsl * VT;
      if (m0 < sh.V) {
#pragma unroll
        for (int i = 0; i < TC_M / 32; ++i) {
          if (offu[i] == ~(size_t)0) continue;
          asm volatile("prefetch.global.L2 [%0];\n" ::"l"(U + offu[i] + m0));
          asm volatile("prefetch.global.L2 [%0];\n" ::"l"(T + offt[i] + m0));
        }
      }
    }
  }
  // Row m, epilogue group grp: the VB = 32 columns [32 grp, 32 grp + 32) of
  // the tile, in four groups of 8 (one 16-byte chunk of U and of the target
  // row, 8 accumulator columns).  Every thread of the warp runs the whole body
  // (the tensor-memory loads are warp-collective); rows beyond the packed
  // count compute on zeros and skip the store.
  __device__ void epilogue(int mt, int sl, int m, const unsigned char* xb, uint32_t trow, int grp) const {
    const int p = mt * TC_M + m;
    const bool rowok = p < P;
    const int c0 = sl * VT + VB * grp;                       // first column of the slice
    const int nval = rowok ? min(VB, sh.V - c0) : 0;
    float4 rc = make_float4(1.f, 0.f, 0.f, 0.f);
    float2 rp = make_float2(0.f, 0.f);
    if (rowok) {
      const int2 bj = ws.prow[p];
      rc = ws.rowc[p];
      rp = ws.rowp[(size_t)bj.x * (sh.gamma + 1) + bj.y];
    }
    const float s2 = __fmul_rn(rc.x, LOG2E_F);
    const unsigned char* ux = xb + m * 128;
    const unsigned char* tx = xb + TC_M * 128 + m * 128;
    auto chunk = [&](const unsigned char* base, int g) { return lds128(base + (((4 * grp + g) ^ (m & 7)) << 4)); };
    // slice references: the largest U and t of the slice's valid columns
    float cU = -INFINITY, cT = -INFINITY;
    if (nval == VB) {
      __nv_bfloat162 mu = __float2bfloat162_rn(-INFINITY), mtt = mu;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const uint4 a = chunk(ux, g), t = chunk(tx, g);
        const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wt[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          mu = __hmax2(mu, *reinterpret_cast<const __nv_bfloat162*>(&wa[e]));
          mtt = __hmax2(mtt, *reinterpret_cast<const __nv_bfloat162*>(&wt[e]));
        }
      }
      cU = fmaxf(__low2float(mu), __high2float(mu));
      cT = fmaxf(__low2float(mtt), __high2float(mtt));
    } else {
      for (int i = 0; i < nval; ++i) {
        const uint4 a = chunk(ux, i >> 3), t = chunk(tx, i >> 3);
        const int e = i & 7;
        const uint32_t wa = (e >> 1) == 0 ? a.x : (e >> 1) == 1 ? a.y : (e >> 1) == 2 ? a.z : a.w;
        const uint32_t wt = (e >> 1) == 0 ? t.x : (e >> 1) == 1 ? t.y : (e >> 1) == 2 ? t.z : t.w;
        cU = fmaxf(cU, (e & 1) ? bf_hi(wa) : bf_lo(wa));
        cT = fmaxf(cT, (e & 1) ? bf_hi(wt) : bf_lo(wt));
      }
    }
    const float Fq = norm_factor(cU, {rc.x, rc.y}, {rc.z, rc.w});
    const float Fp = norm_factor(cT, {rc.x, rc.y}, {rp.x, rp.y});
    float al[2] = {0.f, 0.f}, p2[2] = {0.f, 0.f}, q2[2] = {0.f, 0.f};
    Kahan kr[2];
#pragma unroll 1
    for (int g = 0; g < 4; ++g) {
      float bias[8];
      tc_ld8_issue(trow + (uint32_t)(VB * grp + 8 * g), bias);
      const uint4 a = chunk(ux, g), t = chunk(tx, g);
      tc_wait_ld();
      const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wt[4] = {t.x, t.y, t.z, t.w};
      const int nv = nval - 8 * g;                           // valid columns in this group
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (e < nv) {
          const float uv = (e & 1) ? bf_hi(wa[e >> 1]) : bf_lo(wa[e >> 1]);
          const float tv = (e & 1) ? bf_hi(wt[e >> 1]) : bf_lo(wt[e >> 1]);
          const float qv = __fmul_rn(vq(uv, cU, bias[e], s2), Fq);
          const float pv = __fmul_rn(vp(tv, cT, s2), Fp);
          al[e & 1] += fminf(pv, qv);
          kr[e & 1].add(fmaxf(0.f, __fsub_rn(pv, qv)));
          p2[e & 1] = fmaf(pv, pv, p2[e & 1]);
          q2[e & 1] = fmaf(qv, qv, q2[e & 1]);
        }
      }
    }
    if (rowok && nval > 0)
      ws.vpart[(size_t)p * sh.NSV + c0 / VB] =
          make_float4(al[0] + al[1], df_d(df_add(kr[0].value(), kr[1].value())), p2[0] + p2[1], q2[0] + q2[1]);
  }
};

struct VtParams {
  TpMaps maps;        // w2 only
  Shape sh;
  const bf16* target;
  const bf16* U;
  const bf16* W1;
  Ws ws;
  uint32_t* status;
};

// One CTA per SM (384 threads: two epilogue groups); each takes a contiguous
// run of the (request tile, VT-column slice) tiles of the packed rows (the
// count is read on the device).
constexpr int VT_THREADS = 384;
__global__ void __launch_bounds__(VT_THREADS, 1) verify_tiles_tc_kernel(const __grid_constant__ VtParams P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ uint64_t s_bar[TB_COUNT];
  __shared__ uint32_t s_holder;
  __shared__ int s_tok[TC_M];
  __shared__ int s_fail;
  const Shape& sh = P.sh;
  const int Pk = (int)P.ws.ctrl[CTRL_NPACKED];
  const int nsl = (sh.V + VT - 1) / VT;
  const int n_tiles = nsl * ((Pk + TC_M - 1) / TC_M);
  const int G = (int)gridDim.x, c = (int)blockIdx.x;
  const int per = n_tiles / G, rem = n_tiles % G;
  const int t0 = c * per + min(c, rem), n = per + (c < rem ? 1 : 0);
  if (n <= 0) return;
  if (threadIdx.x == 0) {
    tp_init(s_bar, 32, 2);
    s_fail = 0;
  }
  if (threadIdx.x < 32) tc_alloc(&s_holder, 2 * VT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  TpState st{s_holder, s_bar, &s_fail, 0u, 0u};
  const VerifyEpi e{sh, P.U, P.target, P.ws, Pk};   // (its row cache is per thread)
  const bool ok = tp_run<VT, VerifyEpi, 2>(e, sh, P.maps, P.W1, nsl, t0, 1, n, smem_raw, st, s_tok);
  if (!ok && threadIdx.x == 0) set_status(P.status, SPEC_DEV_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) tc_dealloc(st.tmem, 2 * VT);
}

// ---------------------------------------------------------------- finalize
template <typename DT>
__global__ void __launch_bounds__(NT) verify_final_kernel(
    Shape sh, const DT* __restrict__ target, const DT* __restrict__ U, const DT* __restrict__ W1,
    const DT* __restrict__ W2, const int* __restrict__ anchor, const float* __restrict__ temp,
    const int* __restrict__ dtok, const float* __restrict__ q_tok, const double* __restrict__ lse_q,
    const int* __restrict__ vlen, const float* __restrict__ u_acc, const float* __restrict__ u_fin,
    int* accept_len, int* out_tokens, float* alpha, float* p_tok, float* diag, uint32_t* status,
    Ws ws, Eps eps) {
  extern __shared__ __align__(16) unsigned char dsm[];
  DT* slab = reinterpret_cast<DT*>(dsm);      // [r][VB] W2 slab of the crossing slice
  __shared__ float sh_f[72];
  __shared__ float s_a[256];
  __shared__ float s_part[NT / VB][VB];
  __shared__ float s_w[VB];
  __shared__ int s_n, s_slice, s_tok, s_slow;
  __shared__ float s_pref[2], s_lo, s_hi;
  __shared__ df s_tab[DD_EXP_TAB];

  const int b = blockIdx.x;
  if (ws.vflags[b] & 1) return;
  if (threadIdx.x < DD_EXP_TAB) dd_exp_table_entry(s_tab, threadIdx.x);
  __syncthreads();
  const int L = vlen[b];
  const int rp = ws.rowptr[b];
  const float T = temp[b];
  const float invT = 1.0f / T;
  const df invTdf = dd_recip(T);
  // (fp32 and double-float only below: GB300's fp64 rate is low)

  // ---- alpha_j = sum over slices (double-float, fixed order): every row's
  // per-thread sums first (all loads independent), then one reduction of all
  // rows at once (warp shuffles, then one pass over the warps' partials)
  {
    df a[MAX_GAMMA];
#pragma unroll
    for (int j = 0; j < MAX_GAMMA; ++j) a[j] = {0.f, 0.f};
    for (int s = threadIdx.x; s < sh.NSV; s += NT)
#pragma unroll
      for (int j = 0; j < MAX_GAMMA; ++j)
        if (j < L) a[j] = df_addf(a[j], ws.vpart[(size_t)(rp + j) * sh.NSV + s].x);
    __shared__ df s_al[NT / 32][MAX_GAMMA];
#pragma unroll
    for (int j = 0; j < MAX_GAMMA; ++j) {
      const df t = warp_sum_df(a[j]);
      if ((threadIdx.x & 31) == 0) s_al[threadIdx.x >> 5][j] = t;
    }
    __syncthreads();
    if (threadIdx.x < sh.gamma) {
      const int j = threadIdx.x;
      df t = s_al[0][j];
      for (int w = 1; w < NT / 32; ++w) t = df_add(t, s_al[w][j]);
      alpha[(size_t)b * sh.gamma + j] = j < L ? (float)df_d(t) : NAN;
    }
  }

  // ---- ratio tests and first reject (warp 0, lane j)
  if (threadIdx.x < 32) {
    const int j = threadIdx.x;
    bool acc = true, near = false;
    if (j < L) {
      const int x = dtok[(size_t)b * sh.gamma + j];
      const float tx = ldf(target + ((size_t)b * (sh.gamma + 1) + j) * sh.V + x);
      const float2 nlp = ws.rowp[(size_t)b * (sh.gamma + 1) + j];       // -lse_p
      const float pt = dd_exp(dd_add(dd_mul_f(invTdf, tx), df{nlp.x, nlp.y}), s_tab).hi;
      const float ratio = __fdiv_rn(pt, q_tok[(size_t)b * sh.gamma + j]);
      const float u = u_acc[(size_t)b * sh.gamma + j];
      acc = u < ratio;
      near = fabsf(u - ratio) <= eps.scale * eps.ratio * ratio;
      if (p_tok) p_tok[(size_t)b * sh.gamma + j] = pt;
    } else if (j < sh.gamma && p_tok) {
      p_tok[(size_t)b * sh.gamma + j] = NAN;
    }
    const uint32_t accm = __ballot_sync(0xffffffffu, acc);
    const uint32_t nearm = __ballot_sync(0xffffffffu, near);
    const uint32_t rej = ~accm & ((L >= 32) ? 0xffffffffu : ((1u << L) - 1u));
    const int n = rej ? (__ffs(rej) - 1) : L;
    const uint32_t upto = (n >= 31) ? 0xffffffffu : ((2u << n) - 1u);
    if (j == 0) {
      s_n = n;
      s_slow = (nearm & upto) != 0;
      if (s_slow) {
        ws.accbits[b] = accm;
        atomicOr(&ws.vflags[b], (int)((nearm & upto) << 8));
        uint32_t q = atomicAdd(&ws.ctrl[CTRL_SLOW], 1u);
        ws.slow[q] = b;
      }
    }
  }
  __syncthreads();
  if (s_slow) return;   // the extended-precision slow path owns this request
  const int n = s_n;
  const bool resid = n < L;
  const int row = n;                 // draft/target row of the final draw
  const float4* VP = ws.vpart + (size_t)(rp + row) * sh.NSV;
  const float4* BP = ws.bpart + (size_t)b * sh.NSV;

  // ---- slice masses of the final distribution
  const int per = (sh.NSV + NT - 1) / NT;
  const int s0 = threadIdx.x * per, s1 = min(s0 + per, sh.NSV);
  float cM = -INFINITY;
  if (!resid) {
    for (int s = s0; s < s1; ++s) cM = fmaxf(cM, BP[s].x);
    cM = block_max(cM, sh_f);
  }
  df loc = {0.f, 0.f};
  float e2 = 0.f, m2 = 0.f;
  for (int s = s0; s < s1; ++s) {
    float wsl;
    if (resid) {
      const float4 v = VP[s];
      wsl = v.y;
      e2 += v.z + v.w;
    } else {
      const float4 v = BP[s];
      const float f = expf(fast_tx(v.x, cM, invT));
      wsl = __fmul_rn(v.y, f);
      e2 = fmaf(v.z * f, f, e2);
    }
    loc = df_addf(loc, wsl);
    m2 = fmaf(wsl, wsl, m2);
  }
  df Zdf;
  const df excl = block_excl_scan_df(loc, &Zdf, sh_f);
  e2 = block_sum(e2, sh_f);
  m2 = block_sum(m2, sh_f);
  const float u = u_fin[b];
  const df tgt = dd_mul_f(Zdf, u);
  bool fallback = !(Zdf.hi > 0.f);

  if (threadIdx.x == 0) s_slice = 0x7fffffff;
  __syncthreads();
  int my_slice = -1;
  df my_pref = {0.f, 0.f};
  if (!fallback && s0 < s1 && dd_le(excl, tgt) && !dd_le(df_add(excl, loc), tgt)) {
    df run = excl;
    for (int s = s0; s < s1; ++s) {
      float wsl = resid ? VP[s].y : __fmul_rn(BP[s].y, expf(fast_tx(BP[s].x, cM, invT)));
      df nxt = df_addf(run, wsl);
      if (!dd_le(nxt, tgt)) {
        my_slice = s;
        my_pref = run;
        atomicMin(&s_slice, s);
        break;
      }
      run = nxt;
    }
  }
  __syncthreads();
  if (my_slice >= 0 && my_slice == s_slice) { s_pref[0] = my_pref.hi; s_pref[1] = my_pref.lo; }
  __syncthreads();
  if (s_slice == 0x7fffffff) {
    fallback = true;
    if (threadIdx.x == 0) {
      int sl = sh.NSV - 1;
      while (sl > 0 && !((resid ? VP[sl].y : BP[sl].y) > 0.f)) --sl;
      df run = {0.f, 0.f};
      for (int s = 0; s < sl; ++s)
        run = df_addf(run, resid ? VP[s].y : __fmul_rn(BP[s].y, expf(fast_tx(BP[s].x, cM, invT))));
      s_slice = sl;
      s_pref[0] = run.hi;
      s_pref[1] = run.lo;
    }
    __syncthreads();
  }
  const int sl = s_slice;
  const int n0 = sl * VB;
  const df pref = {s_pref[0], s_pref[1]};
  const int prev = factor_row(sh, b, row, row == 0 ? anchor[b] : dtok[(size_t)b * sh.gamma + row - 1]);

  // ---- recompute the crossing slice
  const DT* trow = target + ((size_t)b * (sh.gamma + 1) + row) * sh.V;
  const DT* urow = U + ((size_t)b * sh.gamma + (resid ? row : 0)) * sh.V;
  float w = 0.f, fslice = 1.f;
  if (resid) {
    // the slice's U and target values and the factor row are requested before
    // the W2 columns are staged
    const bool lane_in = threadIdx.x < VB && n0 + (int)threadIdx.x < sh.V;
    const float u_pre = lane_in ? ldf(urow + n0 + threadIdx.x) : -INFINITY;
    const float t_pre = lane_in ? ldf(trow + n0 + threadIdx.x) : -INFINITY;
    const float a_pre = (int)threadIdx.x < sh.r ? ldf(W1 + (size_t)prev * sh.r + threadIdx.x) : 0.f;
    issue_w2_slab<DT>(slab, W2, sh.V, 0, sh.r, n0, VB);
    if ((int)threadIdx.x < sh.r) s_a[threadIdx.x] = a_pre;
    cp_async_wait_all();
    __syncthreads();
    const int col = threadIdx.x % VB, grp = threadIdx.x / VB;
    const int kg = sh.r / (NT / VB);            // r % 16 == 0
    float acc = 0.f;
    for (int i = grp * kg; i < grp * kg + kg; ++i) acc = fmaf(s_a[i], tof(slab[i * VB + col]), acc);
    s_part[grp][col] = acc;
    __syncthreads();
    float uv = -INFINITY, tv = -INFINITY, bias = 0.f;
    if (threadIdx.x < VB && n0 + (int)threadIdx.x < sh.V) {
      bias = s_part[0][threadIdx.x];
#pragma unroll
      for (int g = 1; g < NT / VB; ++g) bias = __fadd_rn(bias, s_part[g][threadIdx.x]);
      uv = u_pre;
      tv = t_pre;
    }
    const float cU = block_max(uv, sh_f);
    const float cT = block_max(tv, sh_f);
    const float4 rc = ws.rowc[rp + row];
    const float2 rpp = ws.rowp[(size_t)b * (sh.gamma + 1) + row];
    const float Fq = norm_factor(cU, {rc.x, rc.y}, {rc.z, rc.w});
    const float Fp = norm_factor(cT, {rc.x, rc.y}, {rpp.x, rpp.y});
    if (threadIdx.x < VB && n0 + (int)threadIdx.x < sh.V) {
      const float s2 = __fmul_rn(rc.x, LOG2E_F);
      const float q = __fmul_rn(vq(uv, cU, bias, s2), Fq);
      const float pv = __fmul_rn(vp(tv, cT, s2), Fp);
      w = fmaxf(0.f, __fsub_rn(pv, q));
    }
  } else {
    const float4 v = BP[sl];
    fslice = expf(fast_tx(v.x, cM, invT));
    if (threadIdx.x < VB && n0 + (int)threadIdx.x < sh.V)
      w = __expf(fast_tx(ldf(trow + n0 + threadIdx.x), v.x, invT));
  }
  if (threadIdx.x < VB) s_w[threadIdx.x] = w;
  __syncthreads();
  // in-slice target in slice units
  const df tin = dd_mul(dd_add(tgt, dd_neg(pref)), dd_recip(fslice));
  df wtot;
  const df wex = block_excl_scan_df(df_make(threadIdx.x < VB ? w : 0.f), &wtot, sh_f);
  if (threadIdx.x == 0) s_tok = 0x7fffffff;
  __syncthreads();
  df my_lo = {0.f, 0.f}, my_hi = {0.f, 0.f};
  bool claim = false;
  if (!fallback && threadIdx.x < VB && w > 0.f) {
    my_lo = wex;
    my_hi = df_addf(wex, w);
    if (dd_le(my_lo, tin) && !dd_le(my_hi, tin)) { claim = true; atomicMin(&s_tok, (int)threadIdx.x); }
  }
  __syncthreads();
  if (claim && (int)threadIdx.x == s_tok) {
    s_lo = dd_add(tin, dd_neg(my_lo)).hi;
    s_hi = dd_add(my_hi, dd_neg(tin)).hi;
  }
  __syncthreads();
  if (s_tok == 0x7fffffff) {
    fallback = true;
    if (threadIdx.x == 0) {
      int t = VB - 1;
      while (t > 0 && !(s_w[t] > 0.f)) --t;
      s_tok = t;
      s_lo = 0.f;
      s_hi = 0.f;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const int tok = n0 + s_tok;
    int* out = out_tokens + (size_t)b * (sh.gamma + 1);
    for (int j = 0; j < n; ++j) out[j] = dtok[(size_t)b * sh.gamma + j];
    out[n] = tok;
    for (int j = n + 1; j <= sh.gamma; ++j) out[j] = -1;
    accept_len[b] = n;
    const float Zs = Zdf.hi > 0.f ? Zdf.hi : 1.0f;
    const float scale = __fdiv_rn(fslice, Zs);                 // slice units -> probability
    const float dmargin = fminf(s_lo, s_hi) * scale;
    const float band = eps.scale * (__fdiv_rn(eps.elem * sqrtf(e2) + eps.slice * sqrtf(m2) +
                                                  (resid ? eps.norm : 0.f),
                                              Zs) +
                                    eps.abs_);
    if (diag) {
      diag[(size_t)b * 4 + 0] = s_lo * scale;
      diag[(size_t)b * 4 + 1] = s_hi * scale;
      diag[(size_t)b * 4 + 2] = band;
      diag[(size_t)b * 4 + 3] = (float)tok;
    }
    if (fallback || dmargin <= band) {
      uint32_t it = atomicAdd(&ws.ctrl[CTRL_ITEMS], 1u);
      if ((int)it < ws.max_items) {
        HpItem h;
        h.b = b; h.j = row; h.kind = resid ? HP_RESID : HP_BONUS; h.prev = prev; h.u = u;
        h.fast_token = tok;
        h.shift_q = resid ? lse_q[(size_t)b * sh.gamma + row] : 0.0;
        h.shift_p = ws.lse_p[(size_t)b * (sh.gamma + 1) + row];
        ws.items[it] = h;
      } else {
        set_status(status, SPEC_DEV_OVERFLOW);
      }
    }
  }
}

// ---------------------------------------------------------------- launchers
cudaError_t launch_verify_prep(const Shape& sh, const int* anchor, const float* temp,
                               const int* dtok, const double* lse_q, const int* vlen, const Ws& ws,
                               uint32_t* status, int* accept_len, int* out_tokens, float* alpha,
                               float* p_tok, cudaStream_t st) {
  verify_prep_kernel<<<1, NT, 0, st>>>(sh, anchor, temp, dtok, lse_q, vlen, ws, status, accept_len,
                                       out_tokens, alpha, p_tok);
  return cudaGetLastError();
}

template <typename DT>
cudaError_t launch_target_stats(const Shape& sh, const void* target, const float* temp,
                                const int* vlen, const Ws& ws, cudaStream_t st) {
  dim3 grid(sh.gamma + 1, sh.B);
  target_stats_kernel<DT><<<grid, NT, 0, st>>>(sh, (const DT*)target, temp, vlen, ws);
  return cudaGetLastError();
}

template <typename DT, int BM, int PATH>
static cudaError_t launch_vtile(const Shape& sh, const DT* target, const DT* U, const DT* W1,
                                const DT* W2, const Ws& ws, uint32_t* status, cudaStream_t st) {
  const size_t smem = TileLayout<DT>(BM, sh.r, true).total;
  auto kern = verify_tile_kernel<DT, BM, PATH>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int pmax = sh.B * sh.gamma;
  dim3 grid(sh.NS, (pmax + BM - 1) / BM);
  kern<<<grid, NT, smem, st>>>(sh, target, U, W1, W2, ws, status);
  return cudaGetLastError();
}

// The tensor-memory verification tiles: one CTA per SM (fewer for small
// problems), W2 through its TMA map.
static cudaError_t launch_vtiles_tc(const Shape& sh, const bf16* target, const bf16* U,
                                    const bf16* W1, const bf16* W2, const Ws& ws, uint32_t* status,
                                    cudaStream_t st) {
  VtParams P;
  memset(&P.maps, 0, sizeof(P.maps));
  cudaError_t e = encode_w2_map(sh, W2, &P.maps.w2);
  if (e != cudaSuccess) return e;
  P.sh = sh;
  P.target = target;
  P.U = U;
  P.W1 = W1;
  P.ws = ws;
  P.status = status;
  const size_t smem = TpLayout(sh.r, VT).total;
  e = cudaFuncSetAttribute(verify_tiles_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, nsm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  const int max_tiles = ((sh.V + VT - 1) / VT) * ((sh.B * sh.gamma + TC_M - 1) / TC_M);
  const int G = nsm < max_tiles ? nsm : max_tiles;
  verify_tiles_tc_kernel<<<G, VT_THREADS, smem, st>>>(P);
  return cudaGetLastError();
}

template <typename DT>
cudaError_t launch_verify_tile(const Shape& sh, const void* target, const void* U, const void* W1,
                               const void* W2, const Ws& ws, int path, uint32_t* status,
                               cudaStream_t st) {
  const DT* t = (const DT*)target;
  const DT* u = (const DT*)U;
  const DT* w1 = (const DT*)W1;
  const DT* w2 = (const DT*)W2;
  const int pmax = sh.B * sh.gamma;
  const int BM = pmax <= 32 ? 32 : (pmax <= 64 ? 64 : 128);
#define SPEC_VT(BMV, P) launch_vtile<DT, BMV, P>(sh, t, u, w1, w2, ws, status, st)
  if (path == 0 || sizeof(DT) == 4) {
    if (BM == 32) return SPEC_VT(32, 0);
    if (BM == 64) return SPEC_VT(64, 0);
    return SPEC_VT(128, 0);
  }
  if constexpr (sizeof(DT) == 2) {
    if (path == 2 && sh.r % 64 == 0) return launch_vtiles_tc(sh, t, u, w1, w2, ws, status, st);
  }
  if (BM == 32) return SPEC_VT(32, 1);
  if (BM == 64) return SPEC_VT(64, 1);
  return SPEC_VT(128, 1);
#undef SPEC_VT
}

template <typename DT>
cudaError_t launch_verify_final(const Shape& sh, const void* target, const void* U, const void* W1,
                                const void* W2, const int* anchor, const float* temp,
                                const int* dtok, const float* q_tok, const double* lse_q,
                                const int* vlen, const float* u_acc, const float* u_fin,
                                int* accept_len, int* out_tokens, float* alpha, float* p_tok,
                                float* diag, uint32_t* status, const Ws& ws, const Eps& eps,
                                cudaStream_t st) {
  const size_t smem = (size_t)sh.r * VB * sizeof(DT);
  cudaError_t e = cudaFuncSetAttribute(verify_final_kernel<DT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  verify_final_kernel<DT><<<sh.B, NT, smem, st>>>(
      sh, (const DT*)target, (const DT*)U, (const DT*)W1, (const DT*)W2, anchor, temp, dtok, q_tok,
      lse_q, vlen, u_acc, u_fin, accept_len, out_tokens, alpha, p_tok, diag, status, ws, eps);
  return cudaGetLastError();
}

#define SPEC_INST(DT)                                                                              \
  template cudaError_t launch_target_stats<DT>(const Shape&, const void*, const float*, const int*, \
                                               const Ws&, cudaStream_t);                          \
  template cudaError_t launch_verify_tile<DT>(const Shape&, const void*, const void*, const void*, \
                                              const void*, const Ws&, int, uint32_t*, cudaStream_t); \
  template cudaError_t launch_verify_final<DT>(                                                   \
      const Shape&, const void*, const void*, const void*, const void*, const int*, const float*, \
      const int*, const float*, const double*, const int*, const float*, const float*, int*, int*, \
      float*, float*, float*, uint32_t*, const Ws&, const Eps&, cudaStream_t);
SPEC_INST(float)
SPEC_INST(bf16)
#undef SPEC_INST

}  // namespace spec
