// Draft side: DSpark's sequential stage with the Markov head ("[논문리뷰]
// DSpark ...", section 1.2: p_k(v | x_0, x_<k) = softmax(U_k + B_k),
// B(x_{k-1}, .) = W1[x_{k-1}] W2; sampled left to right), tempered by T_b.
// The whole draft is one cooperative launch that walks the gamma steps; each
// step has three phases separated by grid barriers:
//
//   tiles     (request tile, slice of BN columns) pairs strided over the CTAs.
//             Gathers W1[x_{k-1}] rows, computes the bias tile, adds U_k,
//             scales by 1/T and writes per (request, slice) the softmax partial
//             (c, m, s, q2): c = max U over the slice, m = max of
//             x = ((U-c)+bias)/T, s = sum exp(x-m), q2 = sum exp(x-m)^2, plus
//             the masses of the slice's four 32-column chunks.  The
//             full-vocabulary logits never leave the SM.
//   sampling  one CTA per request: merges the slice partials into the
//             normaliser, finds the slice and then the 32-column chunk where
//             the running mass crosses u * Z, recomputes that chunk's weights
//             and scans them for the token (smallest v with F(v) > u).
//             Decisions within the first pass's error band of a CDF breakpoint
//             are queued for re-decision in extended precision.
//   re-decision  (only when the step queued draws) the two extended-precision
//             phases of spec_hp.cuh.
#include <cstring>

#include "spec_tile_tc.cuh"
#include "spec_hp.cuh"
#include "spec_rnn.cuh"
#include "spec_tmap.cuh"

namespace spec {

// One (request tile, slice) of draft step k on the SIMT (PATH 0, fp32 FMAs)
// or warp-MMA (PATH 1, mma.sync) bias tile; the tensor-memory path is the
// pipelined engine below.  Tokens written by other CTAs of the same launch are
// read through L2.
template <typename DT, int BM, int PATH>
__device__ void draft_tile_body(const Shape& sh, int k, int slice, int mtile, const DT* __restrict__ U,
                                const DT* __restrict__ W1, const DT* __restrict__ W2,
                                const int* __restrict__ anchor, const int* tokens,
                                const float* __restrict__ temp, const Ws& ws,
                                unsigned char* smem_raw) {
  static_assert(PATH == 0 || PATH == 1, "tensor-memory tiles use the pipelined engine");
  __shared__ int s_tok[BM];
  __shared__ size_t s_off[BM];
  const int m0 = mtile * BM, n0 = slice * BN;
  const int nrows = min(BM, sh.B - m0);
  __syncthreads();      // previous use of the shared buffers is finished
  for (int m = threadIdx.x; m < BM; m += NT) {
    int t = 0;
    if (m < nrows) {
      int b = m0 + m;
      t = (k == 0) ? anchor[b] : __ldcg(tokens + (size_t)b * sh.gamma + k - 1);
      t = factor_row(sh, b, k, min(max(t, 0), sh.V - 1));   // bad tokens: reported by the sampler
      s_off[m] = ((size_t)b * sh.gamma + k) * sh.V;
    } else {
      s_off[m] = 0;
    }
    s_tok[m] = t;
  }
  DT* Us;
  float* stage;
  int su;
  {
    const TileLayout<DT> lay(BM, sh.r, false);
    DT* As = reinterpret_cast<DT*>(smem_raw + lay.offA);
    DT* Wsm = reinterpret_cast<DT*>(smem_raw + lay.offW);
    Us = reinterpret_cast<DT*>(smem_raw + lay.offU);
    stage = reinterpret_cast<float*>(smem_raw + lay.offStage);
    su = lay.su;
    __syncthreads();
    load_A_rows<DT>(As, lay.sa, W1, s_tok, nrows, BM, sh.r);
    load_W2_tile<DT>(Wsm, lay.sw, W2, sh.V, n0, sh.r);
    load_X_rows<DT>(Us, lay.su, U, s_off, nrows, BM, sh.V, n0);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    bias_tile<DT, BM, PATH == 0>(As, lay.sa, Wsm, lay.sw, sh.r, stage);
    __syncthreads();
  }

  // ---- epilogue: TPR threads per row, each COLS consecutive columns; one
  // partial per CW-column chunk (two threads share a chunk when COLS < CW)
  constexpr int TPR = NT / BM, COLS = BN / TPR;
  constexpr int SS = TileLayout<DT>::SS;
  constexpr int SPAN = COLS < CW ? COLS : CW;        // columns of one chunk in this thread
  constexpr int CPT = COLS / SPAN;                   // chunk pieces per thread
  const int m = threadIdx.x / TPR, part = threadIdx.x % TPR;
  const bool rowok = m < nrows;
  const int b = m0 + m;
  const float invT = rowok ? 1.0f / temp[b] : 1.0f;
  const DT* urow = Us + (size_t)m * su;
  const float* brow = stage + m * SS;
#pragma unroll
  for (int q = 0; q < CPT; ++q) {
    const int cb = part * COLS + q * SPAN;
    const int ce = min(cb + SPAN, sh.V - n0);        // valid columns of this piece
    float c = -INFINITY;
    for (int i = cb; i < ce; ++i) c = fmaxf(c, tof(urow[i]));
    if constexpr (SPAN < CW) c = fmaxf(c, __shfl_xor_sync(0xffffffffu, c, 1));
    float xm = -INFINITY;
    for (int i = cb; i < ce; ++i) xm = fmaxf(xm, fast_x(tof(urow[i]), c, brow[i], invT));
    if constexpr (SPAN < CW) xm = fmaxf(xm, __shfl_xor_sync(0xffffffffu, xm, 1));
    Kahan ks;
    float q2 = 0.f;
    for (int i = cb; i < ce; ++i) {
      const float w = fast_w(fast_x(tof(urow[i]), c, brow[i], invT), xm);
      ks.add(w);
      q2 = fmaf(w, w, q2);
    }
    df sdf = ks.value();
    if constexpr (SPAN < CW) {
      sdf = df_add(sdf, df{__shfl_xor_sync(0xffffffffu, sdf.hi, 1), __shfl_xor_sync(0xffffffffu, sdf.lo, 1)});
      q2 += __shfl_xor_sync(0xffffffffu, q2, 1);
    }
    const int chunk = (n0 + cb) / CW;
    const bool owner = SPAN == CW || (part & 1) == 0;
    if (rowok && owner && chunk < sh.NC)
      ws.dpart[(size_t)b * sh.NC + chunk] = make_float4(c, xm, (float)df_d(sdf), q2);
  }
}

// ---------------------------------------------------------------- tensor-memory tiles
// Partial (c, m, s, q2) of one CW-column chunk of a row from its packed bf16
// logits `u` (16 words) and its bias row `x` (overwritten with the tempered
// logits); `nv` valid columns.  Four interleaved max / Kahan / square-sum
// chains keep the dependent-latency per column low.
template <bool FULL>
__device__ __forceinline__ float4 chunk_partial(const uint4 (&u)[4], float (&x)[32], int nv, float invT) {
  auto uval = [&](int i) {
    const uint4 q = u[i >> 3];
    const uint32_t w = ((i >> 1) & 3) == 0 ? q.x : ((i >> 1) & 3) == 1 ? q.y : ((i >> 1) & 3) == 2 ? q.z : q.w;
    return (i & 1) ? bf_hi(w) : bf_lo(w);
  };
  float c4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (FULL || i < nv) c4[i & 3] = fmaxf(c4[i & 3], uval(i));
  const float c = fmaxf(fmaxf(c4[0], c4[1]), fmaxf(c4[2], c4[3]));
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    x[i] = fast_x(uval(i), c, x[i], invT);
    if (FULL || i < nv) m4[i & 3] = fmaxf(m4[i & 3], x[i]);
  }
  const float xm = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
  Kahan k4[4];
  float q4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    if (FULL || i < nv) {
      const float w = fast_w(x[i], xm);
      k4[i & 3].add(w);
      q4[i & 3] = fmaf(w, w, q4[i & 3]);
    }
  }
  const df s = df_add(df_add(k4[0].value(), k4[1].value()), df_add(k4[2].value(), k4[3].value()));
  return make_float4(c, xm, (float)df_d(s), (q4[0] + q4[1]) + (q4[2] + q4[3]));
}

// Draft step k on the warp-specialised engine of spec_tile_tc.cuh: the W1 row
// of each request's previous token, and the epilogue of one tile row.
struct DraftEpi {
  static constexpr bool kHelpGather = true;   // epilogue warps help gather the A rows
  const Shape& sh;
  int k;
  const int* anchor;
  const int* tokens;
  const float* temp;
  float4* dpart;
  const CUtensorMap* umap;   // U as [B][gamma][V] (a __grid_constant__ parameter)

  // the U_k tile of (mt, sl): two 64-column TMA boxes of 128 rows
  __device__ void load_x(int mt, int sl, unsigned char* xb, uint64_t* full, int lane, int, int) const {
    if (lane != 0) return;
    const int n0 = sl * BN, m0 = mt * TC_M;
    mbar_expect_tx(full, (uint32_t)(TC_M * BN * 2));
    tma_load_3d(xb, umap, n0, k, m0, full);
    tma_load_3d(xb + TC_M * 128, umap, n0 + 64, k, m0, full);
  }
  // W1 row of row m of request tile mt (-1: no such request; its A row is zero)
  __device__ int token(int mt, int m) const {
    const int b = mt * TC_M + m;
    if (b >= sh.B) return -1;
    if (sh.rnn) return k * sh.B + b;
    const int t = (k == 0) ? anchor[b] : __ldcg(tokens + (size_t)b * sh.gamma + k - 1);
    return min(max(t, 0), sh.V - 1);          // bad tokens are reported by the sampler
  }
  // Row m of tile (mt, sl): the partials of the slice's four chunks, from the
  // U row in `ub` (swizzled) and the accumulator row at TMEM address `trow`;
  // two chunks per TMEM wait.
  __device__ void epilogue(int mt, int sl, int m, const unsigned char* ub, uint32_t trow, int) const {
    const int b = mt * TC_M + m;
    const bool rowok = b < sh.B;
    const int n0 = sl * BN;
    const float invT = rowok ? 1.0f / temp[b] : 1.0f;
#pragma unroll 1
    for (int pr = 0; pr < 2; ++pr) {
      float x0[32], x1[32];
      tc_ld32_issue(trow + (uint32_t)(64 * pr), x0);
      tc_ld32_issue(trow + (uint32_t)(64 * pr + 32), x1);
      uint4 u0[4], u1[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        u0[j] = lds128(tp_uchunk(ub, m, 8 * pr + j));
        u1[j] = lds128(tp_uchunk(ub, m, 8 * pr + 4 + j));
      }
      tc_wait_ld();
      const int cb = n0 + 64 * pr;
      const int nv0 = min(CW, sh.V - cb), nv1 = min(CW, sh.V - cb - CW);
      float4 p0 = make_float4(0.f, 0.f, 0.f, 0.f), p1 = p0;
      if (nv1 >= CW) {
        p0 = chunk_partial<true>(u0, x0, CW, invT);
        p1 = chunk_partial<true>(u1, x1, CW, invT);
      } else {
        if (nv0 > 0) p0 = chunk_partial<false>(u0, x0, nv0, invT);
        if (nv1 > 0) p1 = chunk_partial<false>(u1, x1, nv1, invT);
      }
      if (rowok) {
        float4* o = dpart + (size_t)b * sh.NC + cb / CW;
        if (nv0 > 0) o[0] = p0;
        if (nv1 > 0) o[1] = p1;
      }
    }
  }
};

// Weighted chunk mass relative to the row's largest chunk reference, in units
// of exp(reference logit):  f = exp((c - cM)/T + (m - mM)).
__device__ __forceinline__ float chunk_factor(float4 p, float cM, float mM, float invT) {
  float a = __fadd_rn(__fmul_rn(__fsub_rn(p.x, cM), invT), __fsub_rn(p.y, mM));
  return expf(a);
}

// Draw token x_{k+1} of request b from its chunk partials (one CTA): merge
// the chunk masses (double-float), find the chunk where the running mass
// crosses u*Z, recompute that chunk's CW weights and scan them.  Queues the
// draw on `counter` / ws.items when it lies inside the error band.  `dsm`
// holds an r x CW W2 slab.  Partials and tokens written by other CTAs of the
// same launch are read through L2.

template <typename DT>
__device__ void draft_sample_body(const Shape& sh, int k, int b, const DT* __restrict__ U,
                                  const DT* __restrict__ W1, const DT* __restrict__ W2,
                                  const int* __restrict__ anchor, const float* __restrict__ temp,
                                  const float* __restrict__ u_draft, int* tokens, float* q_tok,
                                  double* lse_q, float* diag, uint32_t* status, const Ws& ws,
                                  const Eps& eps, uint32_t* counter, unsigned char* dsm) {
  DT* slab = reinterpret_cast<DT*>(dsm);      // [r][CW] W2 columns of the crossing chunk
  __shared__ float sh_f[72];
  __shared__ float s_a[256];
  __shared__ float s_part[NT / CW][CW];
  __shared__ int s_slice, s_tok;
  __shared__ float4 s_pm;
  __shared__ float s_pref[2], s_lo, s_hi, s_wtok;
  __shared__ df s_tab[DD_EXP_TAB];

  __syncthreads();      // previous use of the shared buffers is finished
  if (threadIdx.x < DD_EXP_TAB) dd_exp_table_entry(s_tab, threadIdx.x);
  const size_t ok = (size_t)b * sh.gamma + k;
  const int prev = (k == 0) ? anchor[b] : __ldcg(tokens + ok - 1);
  const float T = temp[b];
  if (prev < 0 || prev >= sh.V || !temp_ok(T)) {
    if (threadIdx.x == 0) {
      tokens[ok] = -1;
      q_tok[ok] = NAN;
      lse_q[ok] = NAN;
      set_status(status, (prev < 0 || prev >= sh.V) ? SPEC_DEV_BAD_TOKEN : SPEC_DEV_BAD_TEMP);
      if (diag) for (int q = 0; q < 4; ++q) diag[ok * 4 + q] = NAN;
    }
    return;
  }
  const int arow = factor_row(sh, b, k, prev);
  // the factor row (r <= NT entries, one per thread): loaded now, stored to
  // shared memory only when the crossing chunk's dot product needs it
  const float a_reg = (int)threadIdx.x < sh.r ? ldf(W1 + (size_t)arow * sh.r + threadIdx.x) : 0.f;
  const float invT = 1.0f / T;
  const float4* P = ws.dpart + (size_t)b * sh.NC;

  // ---- this thread's contiguous range of chunks (the first 8 kept in registers)
  const int per = (sh.NC + NT - 1) / NT;
  const int s0 = threadIdx.x * per, s1 = min(s0 + per, sh.NC);
  float4 pv[8];
  float best = -INFINITY;
  int bidx = 0;
  for (int s = s0, q = 0; s < s1; ++s, ++q) {
    const float4 p = __ldcg(P + s);
    if (q < 8) pv[q] = p;
    const float key = fmaf(p.x, invT, p.y);
    if (key > best) { best = key; bidx = s; }
  }
  // reference chunk: lowest index attaining the largest c/T + m
  {
    const float bmax = block_max(best, sh_f);
    int cand = (best == bmax) ? bidx : 0x7fffffff;
    for (int m = 16; m; m >>= 1) cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, m));
    if ((threadIdx.x & 31) == 0) reinterpret_cast<int*>(sh_f)[32 + (threadIdx.x >> 5)] = cand;
    __syncthreads();
    if (threadIdx.x == 0) {
      int c2 = 0x7fffffff;
      for (int w = 0; w < NT / 32; ++w) c2 = min(c2, reinterpret_cast<int*>(sh_f)[32 + w]);
      s_slice = c2;
    }
    __syncthreads();
    // the owner of the reference chunk passes its partial on
    const int rs = s_slice;
    if (rs >= s0 && rs < s1) s_pm = (rs - s0 < 8) ? pv[rs - s0] : __ldcg(P + rs);
    __syncthreads();
  }
  const float4 PM = s_pm;
  const float cM = PM.x, mM = PM.y;

  // ---- chunk masses (double-float), normaliser and error-estimate sums
  df loc = {0.f, 0.f};
  float q2 = 0.f, m2 = 0.f;
  for (int s = s0, q = 0; s < s1; ++s, ++q) {
    const float4 p = (q < 8) ? pv[q] : __ldcg(P + s);
    const float f = chunk_factor(p, cM, mM, invT);
    const float w = p.z * f;
    loc = df_addf(loc, w);
    q2 = fmaf(p.w * f, f, q2);
    m2 = fmaf(w, w, m2);
  }
  df Zdf;
  const df excl = block_excl_scan_df(loc, &Zdf, sh_f);
  q2 = block_sum(q2, sh_f);
  m2 = block_sum(m2, sh_f);
  // (fp32 and double-float only below: GB300's fp64 rate is low)
  const float u = u_draft[ok];
  const df target = dd_mul_f(Zdf, u);

  // ---- crossing chunk: first s with prefix_incl(s) > target
  if (threadIdx.x == 0) s_slice = 0x7fffffff;
  __syncthreads();
  int my_slice = -1;
  df my_pref = {0.f, 0.f};
  if (s0 < s1 && dd_le(excl, target) && !dd_le(df_add(excl, loc), target)) {
    df run = excl;
    for (int s = s0, q = 0; s < s1; ++s, ++q) {
      const float4 p = (q < 8) ? pv[q] : __ldcg(P + s);
      const df nxt = df_addf(run, p.z * chunk_factor(p, cM, mM, invT));
      if (!dd_le(nxt, target)) {
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
  bool fallback = false;
  if (s_slice == 0x7fffffff) {
    // rounding left the total at or below u*Z: last chunk with mass
    fallback = true;
    if (threadIdx.x == 0) {
      int sl = sh.NC - 1;
      while (sl > 0 && !(__ldcg(P + sl).z > 0.f)) --sl;
      df run = {0.f, 0.f};
      for (int s = 0; s < sl; ++s) {
        const float4 p = __ldcg(P + s);
        run = df_addf(run, p.z * chunk_factor(p, cM, mM, invT));
      }
      s_slice = sl;
      s_pref[0] = run.hi;
      s_pref[1] = run.lo;
    }
    __syncthreads();
  }
  const int sl = s_slice;
  const df pref = {s_pref[0], s_pref[1]};
  const float4 PS = __ldcg(P + sl);
  const float fS = chunk_factor(PS, cM, mM, invT);
  const int n0 = sl * CW;

  // ---- recompute the chunk's CW weights: 8 k-groups x CW columns (the U
  // values of the chunk are requested before the W2 columns are staged)
  const float u_reg =
      (threadIdx.x < 32 && n0 + (int)threadIdx.x < sh.V) ? ldf(U + ok * sh.V + n0 + threadIdx.x) : 0.f;
  issue_w2_slab<DT>(slab, W2, sh.V, 0, sh.r, n0, CW);
  if ((int)threadIdx.x < sh.r) s_a[threadIdx.x] = a_reg;
  cp_async_wait_all();
  __syncthreads();
  {
    const int col = threadIdx.x % CW, grp = threadIdx.x / CW;
    const int kg = sh.r / (NT / CW);           // r % 16 == 0, so r / 8 is whole
    float acc = 0.f;
    for (int i = grp * kg; i < grp * kg + kg; ++i) acc = fmaf(s_a[i], tof(slab[i * CW + col]), acc);
    s_part[grp][col] = acc;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int v = n0 + lane;
    float w = 0.f;
    if (v < sh.V) {
      float bias = s_part[0][lane];
#pragma unroll
      for (int g = 1; g < NT / CW; ++g) bias = __fadd_rn(bias, s_part[g][lane]);
      w = fast_w(fast_x(u_reg, PS.x, bias, invT), PS.y);
    }
    // target inside the chunk, in the chunk's units: (u Z - prefix) / fS
    const df tin = dd_mul(dd_add(target, dd_neg(pref)), dd_recip(fS));
    // inclusive double-float scan across the warp
    df inc = df_make(w);
    for (int d = 1; d < 32; d <<= 1) {
      const df o = shfl_up_df(inc, d);
      if (lane >= d) inc = df_add(inc, o);
    }
    df ex = shfl_up_df(inc, 1);
    if (lane == 0) ex = {0.f, 0.f};
    const bool claim = w > 0.f && dd_le(ex, tin) && !dd_le(inc, tin);
    const uint32_t cl = __ballot_sync(0xffffffffu, claim);
    const uint32_t pos = __ballot_sync(0xffffffffu, w > 0.f);
    int t;
    float dlo = 0.f, dhi = 0.f;
    if (cl) {
      t = __ffs(cl) - 1;
      dlo = __shfl_sync(0xffffffffu, dd_add(tin, dd_neg(ex)).hi, t);
      dhi = __shfl_sync(0xffffffffu, dd_add(inc, dd_neg(tin)).hi, t);
    } else {
      fallback = true;
      t = pos ? 31 - __clz(pos) : 0;           // last entry with mass
    }
    const float wt = __shfl_sync(0xffffffffu, w, t);
    if (lane == 0) {
      s_tok = t;
      s_lo = dlo;
      s_hi = dhi;
      s_wtok = wt;
    }
  }
  __syncthreads();
  if (s_lo == 0.f && s_hi == 0.f) fallback = true;
  if (threadIdx.x == 0) {
    const int tok = n0 + s_tok;
    const float Zf = Zdf.hi;
    const float scale = __fdiv_rn(fS, Zf);                 // chunk units -> probability
    const float dmargin = fminf(s_lo, s_hi) * scale;
    const float band = eps.scale * (eps.elem * __fdiv_rn(sqrtf(q2), Zf) +
                                    eps.slice * __fdiv_rn(sqrtf(m2), Zf) + eps.abs_);
    // lse = cM / T + mM + log Z
    const df ref = dd_add_f(dd_mul_f(dd_recip(T), cM), mM);
    const double lse = dd_to_double(ref) + dd_log(Zdf, s_tab);
    int wtok = tok;                   // the token written until a re-decision
    if (fallback || dmargin <= band) {
      uint32_t it = atomicAdd(counter, 1u);
      if ((int)it < ws.max_items) {
        if (eps.perturb != 0.f) wtok = tok + 1 < sh.V ? tok + 1 : 0;   // test hook
        HpItem h;
        h.b = b; h.j = k; h.kind = HP_DRAFT; h.prev = arow; h.u = u; h.fast_token = wtok;
        h.shift_q = lse; h.shift_p = 0.0;
        ws.items[it] = h;
      } else {
        set_status(status, SPEC_DEV_OVERFLOW);
      }
    }
    tokens[ok] = wtok;
    q_tok[ok] = s_wtok * scale;
    lse_q[ok] = lse;
    if (diag) {
      diag[ok * 4 + 0] = s_lo * scale;
      diag[ok * 4 + 1] = s_hi * scale;
      diag[ok * 4 + 2] = band;
      diag[ok * 4 + 3] = (float)tok;
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------- kernel
struct DraftParams {
  TpMaps maps;       // tensor-memory path only
  Shape sh;
  const void* U;
  const void* W1;
  const void* W2;
  const int* anchor;
  const float* temp;
  const float* u_draft;
  int* tokens;
  float* q_tok;
  double* lse_q;
  float* diag;
  uint32_t* status;
  Ws ws;
  Eps eps;
  RnnParams rnn;     // RNN head (sh.rnn): gates before each step's tiles
};

// The whole draft in one cooperative launch: for each step k, [the RNN head's
// gate phase and a grid barrier,] the tile phase (tiles strided over the CTAs,
// then the previous step's near-boundary draws re-decided by the CTAs as they
// finish their tiles), a grid barrier, the sampling phase (requests strided
// over the CTAs) and a grid barrier; then the last step's re-decisions and,
// if a re-decision changed a token, the steps after it again with their
// re-decisions in place.  Tensor memory is allocated once per CTA.
template <typename DT, int BM, int PATH>
__global__ void __launch_bounds__(NT, 1) draft_persistent_kernel(const __grid_constant__ DraftParams P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ uint64_t s_bar[TB_COUNT];
  __shared__ uint32_t s_holder;
  __shared__ int s_tok[TC_M];
  __shared__ int s_fail;
  const Shape& sh = P.sh;
  const DT* U = (const DT*)P.U;
  // factor rows of the bias: W1 (Markov head) or the RNN head's a_k rows
  const DT* W1 = sh.rnn ? (const DT*)P.rnn.arows : (const DT*)P.W1;
  const DT* W2 = (const DT*)P.W2;
  uint32_t* ctrl = P.ws.ctrl;
  TpState st{0u, s_bar, &s_fail, 0u, 0u};
  if constexpr (PATH == 2) {
    if (threadIdx.x == 0) {
      tp_init(s_bar, 1);
      s_fail = 0;
      tma_prefetch_map(&P.maps.u);
    }
    if (threadIdx.x < 32) tc_alloc(&s_holder, TP_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    st.tmem = s_holder;
  }
  uint32_t gen = 0u;                         // grid barriers passed (thread 0)
  const HpRows R{P.U, P.U, W1, P.W2, P.temp};
  const int n_mt = (sh.B + BM - 1) / BM;
  const int n_tiles = sh.NS * n_mt;
  const uint32_t G = gridDim.x;
  unsigned long long* tr = (P.ws.trace && blockIdx.x == 0 && threadIdx.x == 0) ? P.ws.trace : nullptr;
  int n_prev = 0;          // draws the previous step queued for re-decision
  uint32_t hp_base = 0;    // units taken from CTRL_HPNEXT so far (the same in every CTA)
  // One draft step.  Deferred (the first pass over the steps): the previous
  // step's queued draws are re-decided in this step's tile phase by CTAs that
  // have finished their own tiles, taking units from a shared counter; this
  // step's are left for the next.  A re-decision that changes a token marks
  // the later steps of that request for a redo.  Not deferred (the redo):
  // this step's draws are re-decided behind one more grid barrier.
  auto run_step = [&](int k, bool deferred) -> bool {
    bool ok = true;
    if (sh.rnn) {
      rnn_gates_body<DT>(sh, k, (const DT*)P.W1, P.anchor, P.tokens, P.rnn, smem_raw, P.status);
      if (!grid_sync(ctrl, G, gen, P.status)) return false;
    }
    if (tr) tr[k * TRACE_SLOTS + 0] = globaltimer_ns();
    if constexpr (PATH == 2) {
      const DraftEpi e{sh, k, P.anchor, P.tokens, P.temp, P.ws.dpart, &P.maps.u};
      const int n = (int)blockIdx.x < n_tiles ? (n_tiles - (int)blockIdx.x + (int)G - 1) / (int)G : 0;
      unsigned long long* ttr = (P.ws.trace && blockIdx.x == 0)
                                    ? P.ws.trace + (MAX_GAMMA + k) * TRACE_SLOTS : nullptr;
      ok = tp_run<BN>(e, sh, P.maps, reinterpret_cast<const bf16*>(W1), sh.NS, (int)blockIdx.x,
                      (int)G, n, smem_raw, st, s_tok, ttr);
      if (!ok && threadIdx.x == 0) set_status(P.status, SPEC_DEV_TIMEOUT);
    } else {
      for (int t = blockIdx.x; t < n_tiles; t += G)
        draft_tile_body<DT, BM, PATH>(sh, k, t % sh.NS, t / sh.NS, U, W1, W2, P.anchor, P.tokens,
                                      P.temp, P.ws, smem_raw);
    }
    if (!ok) {
      if (threadIdx.x == 0) atomicExch(ctrl + CTRL_ABORT, 1u);
      return false;
    }
    if (deferred && n_prev > 0) {
      hp_sums_body<DT>(sh, R, P.ws, 0, n_prev, smem_raw, true, P.tokens, P.q_tok, P.lse_q, P.status,
                       nullptr, ctrl + CTRL_HPNEXT, hp_base, ctrl + CTRL_REDO);
      hp_base += (uint32_t)(n_prev * sh.HB) + G;
    }
    if (tr) tr[k * TRACE_SLOTS + 1] = globaltimer_ns();
    if (!grid_sync(ctrl, G, gen, P.status)) return false;
    if (tr) tr[k * TRACE_SLOTS + 2] = globaltimer_ns();
    for (int b = blockIdx.x; b < sh.B; b += G)
      draft_sample_body<DT>(sh, k, b, U, W1, W2, P.anchor, P.temp, P.u_draft, P.tokens, P.q_tok,
                            P.lse_q, P.diag, P.status, P.ws, P.eps, ctrl + CTRL_STEP0 + k,
                            smem_raw);
    if (tr) tr[k * TRACE_SLOTS + 3] = globaltimer_ns();
    if (!grid_sync(ctrl, G, gen, P.status)) return false;
    if (tr) tr[k * TRACE_SLOTS + 4] = globaltimer_ns();
    const int n = min((int)__ldcg(ctrl + CTRL_STEP0 + k), P.ws.max_items);
    n_prev = deferred ? n : 0;
    if (!deferred && n > 0) {
      hp_sums_body<DT>(sh, R, P.ws, 0, n, smem_raw, true, P.tokens, P.q_tok, P.lse_q, P.status);
      if (tr) tr[k * TRACE_SLOTS + 5] = globaltimer_ns();
      if (!grid_sync(ctrl, G, gen, P.status)) return false;
    }
    if (tr) {
      tr[k * TRACE_SLOTS + 6] = globaltimer_ns();
      tr[k * TRACE_SLOTS + 7] = (unsigned long long)n;
    }
    return true;
  };
  bool good = true;
  for (int k = 0; k < sh.gamma && good; ++k) good = run_step(k, true);
  if (good && n_prev > 0) {
    // the last step's draws, then the redo of every step after the earliest
    // changed token (all requests: the others recompute the same values)
    hp_sums_body<DT>(sh, R, P.ws, 0, n_prev, smem_raw, true, P.tokens, P.q_tok, P.lse_q, P.status);
    good = grid_sync(ctrl, G, gen, P.status);
  }
  if (good) {
    const uint32_t redo = __ldcg(ctrl + CTRL_REDO);
    const int k0 = sh.gamma - (int)redo + 1;            // first step to redo
    if (redo > 0 && k0 < sh.gamma) {
      if (blockIdx.x == 0 && threadIdx.x == 0)
        for (int k = k0; k < sh.gamma; ++k) ctrl[CTRL_STEP0 + k] = 0u;
      good = grid_sync(ctrl, G, gen, P.status);
      for (int k = k0; k < sh.gamma && good; ++k) good = run_step(k, false);
    }
  }
  if constexpr (PATH == 2) {
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) tc_dealloc(st.tmem, TP_TMEM_COLS);
  }
}

// ---------------------------------------------------------------- launcher
template <typename DT, int BM, int PATH>
static cudaError_t launch_persist(const DraftParams& P, int nsm, cudaStream_t st) {
  size_t smem = PATH == 2 ? TpLayout(P.sh.r, BN).total : TileLayout<DT>(BM, P.sh.r, false).total;
  const size_t slab = (size_t)P.sh.r * HPB * sizeof(DT);    // re-decision W2 slab (> sampler's)
  smem = smem > slab ? smem : slab;
  const int n_tiles = P.sh.NS * ((P.sh.B + BM - 1) / BM);
  int G = nsm;                             // one CTA per SM (all must be co-resident)
  G = G < n_tiles ? G : n_tiles;
  G = G > P.sh.B ? G : (P.sh.B < nsm ? P.sh.B : nsm);
  G = G < 1 ? 1 : G;
  if (P.sh.rnn) {
    // gate phase of a CTA with nI state indices: its Wr rows and a stage of
    // RNN_STAGE_ROWS requests' inputs (bf16), then one fallback-list int per
    // (request, index)
    const size_t B = P.sh.B, K = 2 * (size_t)P.sh.r, nI = (P.sh.r + G - 1) / G;
    const size_t stage = sizeof(DT) == 2 ? nI * 3 * K * sizeof(float) + RNN_STAGE_ROWS * K * sizeof(DT) : 0;
    const size_t need = stage + nI * B * sizeof(int);
    smem = smem > need ? smem : need;
  }
  auto kern = draft_persistent_kernel<DT, BM, PATH>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, P);
}

// Whole draft in one cooperative launch (the control words must be zeroed).
template <typename DT>
cudaError_t launch_draft_persistent(const Shape& sh, const void* U, const void* W1, const void* W2,
                                    const int* anchor, const float* temp, const float* u_draft,
                                    int* tokens, float* q_tok, double* lse_q, float* diag,
                                    uint32_t* status, const Ws& ws, const Eps& eps, int path,
                                    int nsm, cudaStream_t st, const RnnParams* rnn) {
  DraftParams P;
  memset(&P.maps, 0, sizeof(P.maps));
  memset(&P.rnn, 0, sizeof(P.rnn));
  if (rnn) P.rnn = *rnn;
  P.sh = sh;
  P.U = U;
  P.W1 = W1;
  P.W2 = W2;
  P.anchor = anchor;
  P.temp = temp;
  P.u_draft = u_draft;
  P.tokens = tokens;
  P.q_tok = q_tok;
  P.lse_q = lse_q;
  P.diag = diag;
  P.status = status;
  P.ws = ws;
  P.eps = eps;
  const int BM = sh.B <= 32 ? 32 : (sh.B <= 64 ? 64 : 128);
  if (path == 0 || sizeof(DT) == 4) {
    if (BM == 32) return launch_persist<DT, 32, 0>(P, nsm, st);
    if (BM == 64) return launch_persist<DT, 64, 0>(P, nsm, st);
    return launch_persist<DT, 128, 0>(P, nsm, st);
  }
  if constexpr (sizeof(DT) == 2) {
    if (path == 2 && sh.r % 64 == 0) {
      cudaError_t e = encode_u_map(sh, U, &P.maps.u);
      if (e == cudaSuccess) e = encode_w2_map(sh, W2, &P.maps.w2);
      if (e != cudaSuccess) return e;
      return launch_persist<DT, 128, 2>(P, nsm, st);
    }
  }
  if (BM == 32) return launch_persist<DT, 32, 1>(P, nsm, st);
  if (BM == 64) return launch_persist<DT, 64, 1>(P, nsm, st);
  return launch_persist<DT, 128, 1>(P, nsm, st);
}

template cudaError_t launch_draft_persistent<float>(const Shape&, const void*, const void*,
                                                    const void*, const int*, const float*,
                                                    const float*, int*, float*, double*, float*,
                                                    uint32_t*, const Ws&, const Eps&, int, int,
                                                    cudaStream_t, const RnnParams*);
template cudaError_t launch_draft_persistent<bf16>(const Shape&, const void*, const void*,
                                                   const void*, const int*, const float*,
                                                   const float*, int*, float*, double*, float*,
                                                   uint32_t*, const Ws&, const Eps&, int, int,
                                                   cudaStream_t, const RnnParams*);

}  // namespace spec
