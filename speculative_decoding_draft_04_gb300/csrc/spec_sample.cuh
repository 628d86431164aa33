// Draft-side device code shared by the two persistent draft kernels
// (spec_draft.cu, spec_draft_slice.cu): the per-chunk softmax partial of the
// first pass and the sampler that turns a request's chunk partials into its
// next token (DSpark review, section 1.2: p_k = softmax(U_k + B_k) sampled
// left to right, B = W1[x_{k-1}] W2; tempered by T_b).
#pragma once

#include "spec_tile_tc.cuh"
#include "spec_hp.cuh"

namespace spec {

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

// Weighted chunk mass relative to the row's largest chunk reference, in units
// of exp(reference logit):  f = exp((c - cM)/T + (m - mM)).
__device__ __forceinline__ float chunk_factor(float4 p, float cM, float mM, float invT) {
  float a = __fadd_rn(__fmul_rn(__fsub_rn(p.x, cM), invT), __fsub_rn(p.y, mM));
  return expf(a);
}

// Draw token x_{k+1} of request b from its chunk partials (one CTA): merge
// the chunk masses (double-float), find the chunk where the running mass
// crosses u*Z, recompute that chunk's CW weights and scan them.  Queues the
// draw at ws.items[atomicAdd(counter, 1)] (at most `cap` entries; beyond
// that SPEC_DEV_OVERFLOW) when it lies inside the error band.  `dsm` holds an
// r x CW W2 slab.  Partials and tokens written by other CTAs of the same
// launch are read through L2.  HOOK_PERTURB (a test build of the kernel)
// makes every queued draw first write the next token, so that the
// re-decision has a token to correct.

template <typename DT, int HOOK>
__device__ void draft_sample_body(const Shape& sh, int k, int b, const DT* __restrict__ U,
                                  const DT* __restrict__ W1, const DT* __restrict__ W2,
                                  const int* __restrict__ anchor, const float* __restrict__ temp,
                                  const float* __restrict__ u_draft, int* tokens, float* q_tok,
                                  double* lse_q, float* diag, uint32_t* status, const Ws& ws,
                                  const Eps& eps, uint32_t* counter, int cap, unsigned char* dsm,
                                  unsigned long long* str = nullptr, DT* abuf = nullptr) {
  DT* slab = reinterpret_cast<DT*>(dsm);      // [r][CW] W2 columns of the crossing chunk
  __shared__ float s_rkey[NT / 32];
  __shared__ int s_ridx[NT / 32];
  __shared__ float4 s_wsum[NT / 32];
  __shared__ int s_cross;
  __shared__ float s_a[256];
  __shared__ float s_part[NT / CW][CW];
  __shared__ int s_tok;
  __shared__ float4 s_pm, s_ps;
  __shared__ float s_pref[2], s_lo, s_hi, s_wtok;
  __shared__ df s_tab[DD_EXP_TAB];

  __syncthreads();      // previous use of the shared buffers is finished
  unsigned long long* tstamp = (str && threadIdx.x == 0) ? str : nullptr;
  if (tstamp) tstamp[0] = globaltimer_ns();
  const size_t ok = (size_t)b * sh.gamma + k;
  const float4* P = ws.dpart + (size_t)b * sh.NC;
  // ---- this thread's contiguous range of chunks (the first 8 kept in
  // registers): their loads are issued first, so they overlap the token's
  // and the exponential table's set-up
  const int per = (sh.NC + NT - 1) / NT;
  const int s0 = threadIdx.x * per, s1 = min(s0 + per, sh.NC);
  float4 pv[8];
#pragma unroll
  for (int q = 0; q < 8; ++q)
    if (s0 + q < s1) pv[q] = __ldcg(P + s0 + q);
  const int prev = (k == 0) ? anchor[b] : __ldcg(tokens + ok - 1);
  const float T = temp[b];
  const float u = u_draft[ok];               // (requested early: its latency overlaps the merge)
  if (threadIdx.x < DD_EXP_TAB) dd_exp_table_entry(s_tab, threadIdx.x);
  if (prev < 0 || prev >= sh.V || !temp_ok(T)) {
    if (threadIdx.x == 0) {
      tokens[ok] = -1;
      q_tok[ok] = NAN;
      lse_q[ok] = NAN;
      set_status(status, (prev < 0 || prev >= sh.V) ? SPEC_DEV_BAD_TOKEN : SPEC_DEV_BAD_TEMP);
      if (diag) for (int q = 0; q < 4; ++q) diag[ok * 4 + q] = NAN;
    }
    // the next step's A row of this request: zeros (its outputs are invalid)
    if (abuf && (int)threadIdx.x * 8 < sh.r)
      *reinterpret_cast<uint4*>(abuf + (size_t)b * sh.r + threadIdx.x * 8) = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const int arow = factor_row(sh, b, k, prev);
  // the factor row (r <= NT entries, one per thread): loaded now, stored to
  // shared memory only when the crossing chunk's dot product needs it
  const float a_reg = (int)threadIdx.x < sh.r ? ldf(W1 + (size_t)arow * sh.r + threadIdx.x) : 0.f;
  const float invT = 1.0f / T;

  float best = -INFINITY;
  int bidx = 0;
  // (the first 8 chunks from registers with compile-time indices, the rest,
  // for vocabularies beyond 8 x 32 x 256 columns, from L2)
#pragma unroll
  for (int q = 0; q < 8; ++q)
    if (s0 + q < s1) {
      const float key = fmaf(pv[q].x, invT, pv[q].y);
      if (key > best) { best = key; bidx = s0 + q; }
    }
  for (int s = s0 + 8; s < s1; ++s) {
    const float4 p = __ldcg(P + s);
    const float key = fmaf(p.x, invT, p.y);
    if (key > best) { best = key; bidx = s; }
  }
  // reference chunk: lowest index attaining the largest c/T + m (a selection,
  // so every thread reaches the same one): warp butterflies, then every
  // thread combines the eight warp winners in warp order; its owner passes
  // the partial on
  {
    float key = best;
    int idx = s0 < s1 ? bidx : 0x7fffffff;
#pragma unroll
    for (int m = 16; m; m >>= 1) {
      const float k2 = __shfl_xor_sync(0xffffffffu, key, m);
      const int i2 = __shfl_xor_sync(0xffffffffu, idx, m);
      if (k2 > key || (k2 == key && i2 < idx)) { key = k2; idx = i2; }
    }
    if ((threadIdx.x & 31) == 0) {
      s_rkey[threadIdx.x >> 5] = key;
      s_ridx[threadIdx.x >> 5] = idx;
    }
    if (threadIdx.x == 0) s_cross = 0x7fffffff;
    __syncthreads();
    float kb = s_rkey[0];
    int rs = s_ridx[0];
#pragma unroll
    for (int w = 1; w < NT / 32; ++w) {
      const float k2 = s_rkey[w];
      const int i2 = s_ridx[w];
      if (k2 > kb || (k2 == kb && i2 < rs)) { kb = k2; rs = i2; }
    }
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (rs == s0 + q && rs < s1) s_pm = pv[q];
    if (rs >= s0 + 8 && rs < s1) s_pm = __ldcg(P + rs);
    __syncthreads();
  }
  const float4 PM = s_pm;
  const float cM = PM.x, mM = PM.y;
  if (tstamp) tstamp[1] = globaltimer_ns();

  // ---- chunk masses (double-float), normaliser and error-estimate sums
  df loc = {0.f, 0.f};
  float q2 = 0.f, m2 = 0.f;
  float wv[8];                       // the chunk masses kept for the crossing search
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    wv[q] = 0.f;
    if (s0 + q < s1) {
      const float f = chunk_factor(pv[q], cM, mM, invT);
      wv[q] = pv[q].z * f;
      loc = df_addf(loc, wv[q]);
      q2 = fmaf(pv[q].w * f, f, q2);
      m2 = fmaf(wv[q], wv[q], m2);
    }
  }
  for (int s = s0 + 8; s < s1; ++s) {
    const float4 p = __ldcg(P + s);
    const float f = chunk_factor(p, cM, mM, invT);
    const float w = p.z * f;
    loc = df_addf(loc, w);
    q2 = fmaf(p.w * f, f, q2);
    m2 = fmaf(w, w, m2);
  }
  // exclusive scan of the masses with their total, and the two error sums,
  // with one barrier: warp scans by shuffles, then every thread adds the
  // eight warp totals in warp order (so all hold the same total)
  df Zdf;
  const df excl = block_scan1_df2(loc, &Zdf, q2, m2, s_wsum);
  // (fp32 and double-float only below: GB300's fp64 rate is low)
  const df target = dd_mul_f(Zdf, u);

  // ---- crossing chunk: first s with prefix_incl(s) > target (s_cross was
  // reset before the barrier of the reference step)
  int my_slice = -1;
  df my_pref = {0.f, 0.f};
  float4 my_ps = make_float4(0.f, 0.f, 0.f, 0.f);
  if (s0 < s1 && dd_le(excl, target) && !dd_le(df_add(excl, loc), target)) {
    df run = excl;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (my_slice < 0 && s0 + q < s1) {
        const df nxt = df_addf(run, wv[q]);
        if (!dd_le(nxt, target)) {
          my_slice = s0 + q;
          my_pref = run;
          my_ps = pv[q];
        } else {
          run = nxt;
        }
      }
    }
    for (int s = s0 + 8; s < s1 && my_slice < 0; ++s) {
      const float4 p = __ldcg(P + s);
      const df nxt = df_addf(run, p.z * chunk_factor(p, cM, mM, invT));
      if (!dd_le(nxt, target)) {
        my_slice = s;
        my_pref = run;
        my_ps = p;
      } else {
        run = nxt;
      }
    }
    if (my_slice >= 0) atomicMin(&s_cross, my_slice);
  }
  __syncthreads();
  if (my_slice >= 0 && my_slice == s_cross) {
    s_pref[0] = my_pref.hi;
    s_pref[1] = my_pref.lo;
    s_ps = my_ps;                     // the crossing chunk's partial, passed on chip
  }
  __syncthreads();
  bool fallback = false;
  if (s_cross == 0x7fffffff) {
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
      s_cross = sl;
      s_pref[0] = run.hi;
      s_pref[1] = run.lo;
      s_ps = __ldcg(P + sl);
    }
    __syncthreads();
  }
  const int sl = s_cross;
  const df pref = {s_pref[0], s_pref[1]};
  const float4 PS = s_ps;
  if (tstamp) tstamp[2] = globaltimer_ns();
  const float fS = chunk_factor(PS, cM, mM, invT);
  const int n0 = sl * CW;

  // (the next step's A row is fetched by warp 0 as soon as the token is known)
  const bool early_row = abuf != nullptr && !sh.rnn && k + 1 < sh.gamma;
  uint4 arow_v = make_uint4(0u, 0u, 0u, 0u);
  // ---- recompute the chunk's CW weights: 8 k-groups x CW columns (the U
  // values of the chunk are requested before the W2 columns are staged)
  const float u_reg =
      (threadIdx.x < 32 && n0 + (int)threadIdx.x < sh.V) ? ldf(U + ok * sh.V + n0 + threadIdx.x) : 0.f;
  issue_w2_slab<DT>(slab, W2, sh.V, 0, sh.r, n0, CW);
  if ((int)threadIdx.x < sh.r) s_a[threadIdx.x] = a_reg;
  cp_async_wait_all();
  __syncthreads();
  if (tstamp) tstamp[3] = globaltimer_ns();
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
    // the next step's A row W1[token]: requested now, stored to `abuf` below
    // (its latency overlaps the band and logsumexp of thread 0)
    if constexpr (sizeof(DT) == 2 && HOOK != HOOK_PERTURB) {
      if (early_row && lane * 8 < sh.r)
        arow_v = __ldg(reinterpret_cast<const uint4*>(W1 + (size_t)(n0 + t) * sh.r + lane * 8));
    }
  }
  __syncthreads();
  if (tstamp) tstamp[4] = globaltimer_ns();
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
      if ((int)it < cap) {
        if constexpr (HOOK == HOOK_PERTURB) wtok = tok + 1 < sh.V ? tok + 1 : 0;
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
    s_tok = wtok;                     // the token written (for the prefetch below)
    if (diag) {
      diag[ok * 4 + 0] = s_lo * scale;
      diag[ok * 4 + 1] = s_hi * scale;
      diag[ok * 4 + 2] = band;
      diag[ok * 4 + 3] = (float)tok;
    }
  }
  __syncthreads();
  if (tstamp) tstamp[5] = globaltimer_ns();
  // the next step's A operand row of this request: W1[x_{k+1}] copied into
  // `abuf` (row b), which the next tile phase loads by TMA; without `abuf`
  // the row is only brought into L2 for the next step's gather
  if (!sh.rnn && k + 1 < sh.gamma) {
    const int t = s_tok;
    if (sizeof(DT) == 2 && HOOK != HOOK_PERTURB && early_row) {
      if (threadIdx.x < 32 && (int)threadIdx.x * 8 < sh.r)
        *reinterpret_cast<uint4*>(abuf + (size_t)b * sh.r + threadIdx.x * 8) = arow_v;
    } else if (abuf) {
      if ((int)threadIdx.x * 8 < sh.r && t >= 0 && t < sh.V)
        *reinterpret_cast<uint4*>(abuf + (size_t)b * sh.r + threadIdx.x * 8) =
            __ldg(reinterpret_cast<const uint4*>(W1 + (size_t)t * sh.r + threadIdx.x * 8));
    } else if ((int)threadIdx.x * 128 < sh.r * (int)sizeof(DT) && t >= 0 && t < sh.V) {
      asm volatile("prefetch.global.L2 [%0];\n" ::"l"(reinterpret_cast<const char*>(W1 + (size_t)t * sh.r) +
                                                      threadIdx.x * 128));
    }
  }
}

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
  int slK;           // slice-resident kernel: chunks of CW columns per CTA
};


}  // namespace spec
