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
#include "spec_tc.cuh"

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
    if (!(bits & SPEC_DEV_BAD_LEN))
      for (int j = 0; j < L; ++j) {
        const int x = dtok[(size_t)b * sh.gamma + j];
        if (x < 0 || x >= sh.V) bits |= SPEC_DEV_BAD_TOKEN;
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
    for (int j = 0; j < L; ++j) {
      ws.prow[run + j] = make_int2(b, j);
      ws.prevtok[run + j] = j == 0 ? anchor[b] : dtok[(size_t)b * sh.gamma + j - 1];
      const df nlq = d2df(-lse_q[(size_t)b * sh.gamma + j]);
      ws.rowc[run + j] = make_float4(it.hi, it.lo, nlq.hi, nlq.lo);
    }
    run += L;
  }
  if (threadIdx.x == NT - 1) {
    ws.rowptr[sh.B] = s_w[NT / 32];
    ws.ctrl[CTRL_NPACKED] = s_w[NT / 32];
    ws.ctrl[CTRL_ITEMS] = 0;
    ws.ctrl[CTRL_SLOW] = 0;
  }
}

// ---------------------------------------------------------------- target statistics
template <typename DT>
__global__ void __launch_bounds__(NT) target_stats_kernel(Shape sh, const DT* __restrict__ target,
                                                          const float* __restrict__ temp,
                                                          const int* __restrict__ vlen, Ws ws) {
  __shared__ float s_c[NT / 16], s_hi[NT / 16], s_lo[NT / 16];
  __shared__ df s_tab[DD_EXP_TAB];
  const int j = blockIdx.x, b = blockIdx.y;
  if (ws.vflags[b] & 1) return;
  const int L = vlen[b];
  if (j > L) return;
  if (threadIdx.x < DD_EXP_TAB) dd_exp_table_entry(s_tab, threadIdx.x);
  const float T = temp[b];
  const float invT = 1.0f / T;
  const DT* row = target + ((size_t)b * (sh.gamma + 1) + j) * sh.V;
  const bool bonus = j == L;
  const int hw = threadIdx.x >> 4, hl = threadIdx.x & 15;
  float cref = -INFINITY;
  df acc = {0.f, 0.f};
  // every lane runs the same trip count (full-warp shuffles below)
  for (int base = 0; base < sh.NS; base += NT / 16) {
    const int s = base + hw;
    const bool sv = s < sh.NS;
    const int n = s * BN + hl * 8;
    const bool valid = sv && n < sh.V;
    float vals[8];
    if (valid) load8(row + n, vals);
    float c = -INFINITY;
    if (valid)
#pragma unroll
      for (int e = 0; e < 8; ++e) c = fmaxf(c, vals[e]);
#pragma unroll
    for (int m = 8; m; m >>= 1) c = fmaxf(c, __shfl_xor_sync(0xffffffffu, c, m));
    float ssum = 0.f, p2 = 0.f;
    if (valid)
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float wv = __expf(fast_tx(vals[e], c, invT));
        ssum = __fadd_rn(ssum, wv);
        p2 = fmaf(wv, wv, p2);
      }
#pragma unroll
    for (int m = 8; m; m >>= 1) {
      ssum += __shfl_xor_sync(0xffffffffu, ssum, m);
      p2 += __shfl_xor_sync(0xffffffffu, p2, m);
    }
    if (!sv) continue;
    if (bonus && hl == 0) ws.bpart[(size_t)b * sh.NS + s] = make_float4(c, ssum, p2, 0.f);
    if (c > cref) {
      if (cref != -INFINITY) acc = df_mulf(acc, expf(fast_tx(cref, c, invT)));
      cref = c;
      acc = df_addf(acc, ssum);
    } else {
      acc = df_addf(acc, __fmul_rn(ssum, expf(fast_tx(c, cref, invT))));
    }
  }
  if (hl == 0) {
    s_c[hw] = cref;
    s_hi[hw] = acc.hi;
    s_lo[hw] = acc.lo;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = -INFINITY;
    for (int h = 0; h < NT / 16; ++h) M = fmaxf(M, s_c[h]);
    df Z = {0.f, 0.f};
    for (int h = 0; h < NT / 16; ++h)
      if (s_c[h] != -INFINITY) Z = df_add(Z, df_mulf({s_hi[h], s_lo[h]}, expf(fast_tx(s_c[h], M, invT))));
    // lse = M / T + log Z (double-float steps; fp64 only to assemble the result)
    const double lse = dd_to_double(dd_mul_f(dd_recip(T), M)) + dd_log(Z, s_tab);
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
  DT *Us, *Ts;
  float* stage;
  int su;
  if constexpr (PATH == 2) {
    static_assert(BM == TC_M, "tensor-memory path uses 128-row tiles");
    unsigned char* smem = align1k(smem_raw);
    const TcLayout lay(sh.r, true);
    bf16* As = reinterpret_cast<bf16*>(smem + lay.offA);
    bf16* Wsm = reinterpret_cast<bf16*>(smem + lay.offW);
    Us = reinterpret_cast<DT*>(smem + lay.offU);
    Ts = reinterpret_cast<DT*>(smem + lay.offT);
    stage = reinterpret_cast<float*>(smem + lay.offStage);
    su = BN + 8;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + lay.offBar);
    uint32_t* holder = reinterpret_cast<uint32_t*>(smem + lay.offBar + 8);
    if (threadIdx.x == 0) mbar_init(bar, 1);
    if (threadIdx.x < 32) tc_alloc(holder, TC_TMEM_COLS);
    __syncthreads();
    tc_load_A(As, reinterpret_cast<const bf16*>(W1), s_tok, nrows, sh.r);
    tc_load_W2(Wsm, reinterpret_cast<const bf16*>(W2), sh.V, n0, sh.r);
    load_X_rows<DT>(Us, su, U, s_offu, nrows, BM, sh.V, n0);
    load_X_rows<DT>(Ts, su, target, s_offt, nrows, BM, sh.V, n0);
    cp_async_commit();
    cp_async_wait_all();
    fence_async_shared();
    tc_fence_before();
    __syncthreads();
    const uint32_t taddr = *holder;
    const bool ok = bias_tile_tc(As, Wsm, sh.r, taddr, bar, 0, stage);
    if (!ok) {
      if (threadIdx.x == 0) set_status(status, SPEC_DEV_TIMEOUT);
      mbar_wait(bar, 0, 1u << 22);
    }
    __syncthreads();
    if (threadIdx.x < 32) tc_dealloc(taddr, TC_TMEM_COLS);
    if (!ok) return;
    __syncthreads();
  } else {
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

  constexpr int TPR = NT / BM, COLS = BN / TPR;
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
  const int cbeg = part * COLS;
  const int cend = min(cbeg + COLS, sh.V - n0);
  const DT* urow = Us + (size_t)m * su;
  const DT* trow = Ts + (size_t)m * su;
  const float* brow = stage + m * SS;
  float cU = -INFINITY, cT = -INFINITY;
  for (int i = cbeg; i < cend; ++i) {
    cU = fmaxf(cU, tof(urow[i]));
    cT = fmaxf(cT, tof(trow[i]));
  }
  cU = group_max<TPR>(cU);
  cT = group_max<TPR>(cT);
  const float Fq = norm_factor(cU, {rc.x, rc.y}, {rc.z, rc.w});
  const float Fp = norm_factor(cT, {rc.x, rc.y}, {rp.x, rp.y});
  float al = 0.f, p2 = 0.f, q2 = 0.f;
  Kahan kr;
  for (int i = cbeg; i < cend; ++i) {
    const float q = __fmul_rn(__expf(fast_x(tof(urow[i]), cU, brow[i], invT)), Fq);
    const float pv = __fmul_rn(__expf(fast_tx(tof(trow[i]), cT, invT)), Fp);
    al += fminf(pv, q);
    kr.add(fmaxf(0.f, __fsub_rn(pv, q)));
    p2 = fmaf(pv, pv, p2);
    q2 = fmaf(q, q, q2);
  }
  al = group_sum<TPR>(al);
  df res = group_sum_df<TPR>(kr.value());
  p2 = group_sum<TPR>(p2);
  q2 = group_sum<TPR>(q2);
  if (rowok && part == 0) ws.vpart[(size_t)p * sh.NS + slice] = make_float4(al, df_d(res), p2, q2);
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
  DT* slab = reinterpret_cast<DT*>(dsm);      // [r][BN] W2 slab of the crossing slice
  __shared__ float sh_f[72];
  __shared__ float s_a[256];
  __shared__ float s_part[2][BN];
  __shared__ float s_w[BN];
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

  // ---- alpha_j = sum over slices (double-float, fixed order)
  for (int j = 0; j < sh.gamma; ++j) {
    df a = {0.f, 0.f};
    if (j < L)
      for (int s = threadIdx.x; s < sh.NS; s += NT) a = df_addf(a, ws.vpart[(size_t)(rp + j) * sh.NS + s].x);
    a = block_sum_df(a, sh_f);
    if (threadIdx.x == 0) alpha[(size_t)b * sh.gamma + j] = j < L ? (float)df_d(a) : NAN;
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
  const float4* VP = ws.vpart + (size_t)(rp + row) * sh.NS;
  const float4* BP = ws.bpart + (size_t)b * sh.NS;

  // ---- slice masses of the final distribution
  const int per = (sh.NS + NT - 1) / NT;
  const int s0 = threadIdx.x * per, s1 = min(s0 + per, sh.NS);
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
      int sl = sh.NS - 1;
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
  const int n0 = sl * BN;
  const df pref = {s_pref[0], s_pref[1]};
  const int prev = row == 0 ? anchor[b] : dtok[(size_t)b * sh.gamma + row - 1];

  // ---- recompute the crossing slice
  const DT* trow = target + ((size_t)b * (sh.gamma + 1) + row) * sh.V;
  const DT* urow = U + ((size_t)b * sh.gamma + (resid ? row : 0)) * sh.V;
  float w = 0.f, fslice = 1.f;
  if (resid) {
    for (int i = threadIdx.x; i < sh.r; i += NT) s_a[i] = ldf(W1 + (size_t)prev * sh.r + i);
    stage_w2_slab<DT>(slab, W2, sh.V, 0, sh.r, n0, BN);
    const int col = threadIdx.x % BN, half = threadIdx.x / BN;
    const int kh = sh.r / 2;
    float acc = 0.f;
    for (int i = half * kh; i < half * kh + kh; ++i) acc = fmaf(s_a[i], tof(slab[i * BN + col]), acc);
    s_part[half][col] = acc;
    __syncthreads();
    float uv = -INFINITY, tv = -INFINITY, bias = 0.f;
    if (threadIdx.x < BN && n0 + (int)threadIdx.x < sh.V) {
      bias = __fadd_rn(s_part[0][threadIdx.x], s_part[1][threadIdx.x]);
      uv = ldf(urow + n0 + threadIdx.x);
      tv = ldf(trow + n0 + threadIdx.x);
    }
    const float cU = block_max(uv, sh_f);
    const float cT = block_max(tv, sh_f);
    const float4 rc = ws.rowc[rp + row];
    const float2 rpp = ws.rowp[(size_t)b * (sh.gamma + 1) + row];
    const float Fq = norm_factor(cU, {rc.x, rc.y}, {rc.z, rc.w});
    const float Fp = norm_factor(cT, {rc.x, rc.y}, {rpp.x, rpp.y});
    if (threadIdx.x < BN && n0 + (int)threadIdx.x < sh.V) {
      const float q = __fmul_rn(__expf(fast_x(uv, cU, bias, invT)), Fq);
      const float pv = __fmul_rn(__expf(fast_tx(tv, cT, invT)), Fp);
      w = fmaxf(0.f, __fsub_rn(pv, q));
    }
  } else {
    const float4 v = BP[sl];
    fslice = expf(fast_tx(v.x, cM, invT));
    if (threadIdx.x < BN && n0 + (int)threadIdx.x < sh.V)
      w = __expf(fast_tx(ldf(trow + n0 + threadIdx.x), v.x, invT));
  }
  if (threadIdx.x < BN) s_w[threadIdx.x] = w;
  __syncthreads();
  // in-slice target in slice units
  const df tin = dd_mul(dd_add(tgt, dd_neg(pref)), dd_recip(fslice));
  df wtot;
  const df wex = block_excl_scan_df(df_make(threadIdx.x < BN ? w : 0.f), &wtot, sh_f);
  if (threadIdx.x == 0) s_tok = 0x7fffffff;
  __syncthreads();
  df my_lo = {0.f, 0.f}, my_hi = {0.f, 0.f};
  bool claim = false;
  if (!fallback && threadIdx.x < BN && w > 0.f) {
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
      int t = BN - 1;
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
  const size_t smem = PATH == 2 ? TcLayout(sh.r, true).total : TileLayout<DT>(BM, sh.r, true).total;
  auto kern = verify_tile_kernel<DT, BM, PATH>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int pmax = sh.B * sh.gamma;
  dim3 grid(sh.NS, (pmax + BM - 1) / BM);
  kern<<<grid, NT, smem, st>>>(sh, target, U, W1, W2, ws, status);
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
    if (path == 2 && sh.r % 64 == 0) return SPEC_VT(128, 2);
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
  const size_t smem = (size_t)sh.r * BN * sizeof(DT);
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
