// Tree drafting and tree verification ("Speculative Decoding Part 1", VESSL AI
// blog, section "gamma 재배분: 체인 대신 트리"), with DSpark's Markov head
// drafting every node.
//
//   tree_select_kernel   one CTA per request: survival a_s = fp32 product of the
//                        slot factors from the root down, then the top-n slots
//                        (ties: shallower, then lower index) by a comparison
//                        count -- closed under prefixes because a child's a
//                        never exceeds its parent's.
//   tree_plan_kernel     one CTA per request: the depth level at which each
//                        node (the root and every selected slot) is drafted --
//                        its depth when it has selected children, else none.
//   tree_chunks_kernel   per depth level, 16 CTAs per node of that level, each a
//                        share of the vocabulary: the node's draft logits (U row
//                        of its depth + W1[x] W2, over T) in double-float, as
//                        32-column chunk partials.
//   tree_draft_kernel    per depth level, one CTA per node of that level: the
//                        chunk partials merged, then each selected child drawn
//                        by inverse CDF with its own uniform (crossing chunk,
//                        its 32 weights recomputed and scanned).
//   tree_vrow_kernel,    verification, one pair of launches per depth level: S
//   tree_vstep_kernel    CTAs per request compute the draft logits row of the
//                        request's current node (when it has selected children);
//                        then one CTA per request takes one step of its walk from
//                        the root: target logits of the node, recursive rejection
//                        over the node's candidates (ratio u < r(x)/q(x),
//                        r <- normalize(max(0, r - q)) after a rejection); the
//                        first accepted child is the next level's node, otherwise
//                        the final token is drawn from r and the walk ends.
//
// Every weight, sum and scan is a double-float (transition bias as a
// compensated sum of exact products), so the decisions agree with a float64
// computation except within ~1e-12 of a boundary.  This is the direct
// formulation: it spends ~r double-float multiply-adds per vocabulary entry
// and node (spread over many CTAs per node) and is not tiled onto the tensor
// cores.
#include "spec_hp.cuh"

namespace spec {

constexpr int TREE_MAX_SLOTS = 256;

// ---------------------------------------------------------------- selection
__global__ void __launch_bounds__(NT) tree_select_kernel(int B, int N, int gamma, const int* parent,
                                                         const float* conf, int n, float* survival,
                                                         uint8_t* mask, float* expected,
                                                         uint32_t* status) {
  __shared__ float s_a[TREE_MAX_SLOTS];
  __shared__ int s_d[TREE_MAX_SLOTS];
  __shared__ int s_bad;
  const int b = blockIdx.x;
  const int* par = parent + (size_t)b * N;
  if (threadIdx.x == 0) {
    int bad = 0;
    for (int s = 0; s < N; ++s) {        // parents precede children: one pass
      const int p = par[s];
      const float c = conf[(size_t)b * N + s];
      const float cc = (c >= 0.f && c <= 1.f) ? c : 0.f;
      if (!(cc == c)) bad |= SPEC_DEV_BAD_CONF;
      if (p < -1 || p >= s) {
        bad |= SPEC_DEV_BAD_TREE;
        s_d[s] = 1;
        s_a[s] = 0.f;
      } else {
        s_d[s] = p < 0 ? 1 : s_d[p] + 1;
        s_a[s] = p < 0 ? cc : __fmul_rn(s_a[p], cc);
        if (s_d[s] > gamma) bad |= SPEC_DEV_BAD_TREE;
      }
      survival[(size_t)b * N + s] = s_a[s];
    }
    s_bad = bad;
    if (bad) set_status(status, (uint32_t)bad);
  }
  __syncthreads();
  const bool invalid = s_bad & SPEC_DEV_BAD_TREE;
  float sum = 0.f;
  for (int s = threadIdx.x; s < N; s += NT) {
    const float a = s_a[s];
    const int d = s_d[s];
    int rank = 0;
    for (int t = 0; t < N; ++t) {
      const float at = s_a[t];
      rank += (at > a) | ((at == a) & ((s_d[t] < d) | ((s_d[t] == d) & (t < s))));
    }
    const bool take = !invalid && rank < n;
    mask[(size_t)b * N + s] = take ? 1 : 0;
    if (take) sum += a;
  }
  sum = block_sum(sum, reinterpret_cast<float*>(s_d));   // s_d no longer needed
  if (threadIdx.x == 0 && expected) expected[b] = sum;
}

// ---------------------------------------------------------------- block helpers
// Block reductions for a CTA of T threads (T / 32 warps; `sh` holds 2 T / 32
// floats and is free again when they return).  Every thread combines the warp
// results in warp order, so all hold the same value.
template <int T>
__device__ __forceinline__ float tblock_max(float v, float* sh) {
  v = warp_max(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = sh[0];
  for (int q = 1; q < T / 32; ++q) m = fmaxf(m, sh[q]);
  __syncthreads();
  return m;
}
template <int T>
__device__ __forceinline__ df tblock_sum_df(df v, float* sh) {
  v = warp_sum_df(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    sh[2 * (threadIdx.x >> 5)] = v.hi;
    sh[2 * (threadIdx.x >> 5) + 1] = v.lo;
  }
  __syncthreads();
  df t = {0.f, 0.f};
  for (int q = 0; q < T / 32; ++q) t = dd_add(t, df{sh[2 * q], sh[2 * q + 1]});
  __syncthreads();
  return t;
}
// Exclusive scan with the block total.
template <int T>
__device__ __forceinline__ df tblock_excl_scan_df(df v, df* total, float* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  df inc = v;
  for (int d = 1; d < 32; d <<= 1) {
    const df o = shfl_up_df(inc, d);
    if (lane >= d) inc = df_add(inc, o);
  }
  __syncthreads();
  if (lane == 31) {
    sh[2 * w] = inc.hi;
    sh[2 * w + 1] = inc.lo;
  }
  df within = shfl_up_df(inc, 1);
  if (lane == 0) within = {0.f, 0.f};
  __syncthreads();
  df off = {0.f, 0.f}, tot = {0.f, 0.f};
  for (int q = 0; q < T / 32; ++q) {
    if (q == w) off = tot;
    tot = df_add(tot, df{sh[2 * q], sh[2 * q + 1]});
  }
  __syncthreads();
  *total = tot;
  return df_add(off, within);
}

// ---------------------------------------------------------------- node rows
// Logits of one node row over the vocabulary into `out` (double-float pairs):
// draft (U_row + W1[f] W2) / T, or target t_row / T when a == nullptr.
template <typename DT, int T = NT>
__device__ void row_logits(const TreeShape& ts, const DT* urow, const DT* W2, const float* a, df invT,
                           float2* out) {
  for (int v = threadIdx.x; v < ts.V; v += T) {
    df l;
    if (a) {
      const df bias = hp_bias<DT>(a, W2, ts.V, ts.r, v);
      l = dd_mul(dd_add_f(bias, ldf(urow + v)), invT);
    } else {
      l = dd_mul_f(invT, ldf(urow + v));
    }
    out[v] = make_float2(l.hi, l.lo);
  }
}

// Largest logit (its hi part) and the normaliser sum exp(l - m).
template <int T = NT>
__device__ void row_norm(int V, const float2* l, const df* tab, float* shf, float& m, df& Z) {
  float mx = -INFINITY;
  for (int v = threadIdx.x; v < V; v += T) mx = fmaxf(mx, __ldcg(l + v).x);
  m = tblock_max<T>(mx, shf);
  df s = {0.f, 0.f};
  for (int v = threadIdx.x; v < V; v += T) {
    const float2 x = __ldcg(l + v);
    s = dd_add(s, dd_exp(dd_add_f(df{x.x, x.y}, -m), tab));
  }
  Z = tblock_sum_df<T>(s, shf);
}

// Probability of entry v of a row (logits l, shift m, 1/Z).
__device__ __forceinline__ df row_prob(const float2* l, int v, float m, df iz, const df* tab) {
  const float2 x = __ldcg(l + v);
  return dd_mul(dd_exp(dd_add_f(df{x.x, x.y}, -m), tab), iz);
}

// The running distribution r after i rejections at a node: r_0 = p, r_{k+1} =
// max(0, r_k - q) / Z_{k+1} (r_k kept when Z_{k+1} = 0).  izr[k] = 1/Z_{k+1},
// or zero for a kept step.
__device__ __forceinline__ df resid_prob(const float2* lp, const float2* lq, int v, float mp, df izp,
                                         float mq, df izq, const df* izr, int i, const df* tab) {
  df r = row_prob(lp, v, mp, izp, tab);
  if (i == 0) return r;
  const df q = row_prob(lq, v, mq, izq, tab);
  for (int k = 0; k < i; ++k) {
    if (izr[k].hi == 0.f) continue;
    const df d = dd_add(r, dd_neg(q));
    r = d.hi > 0.f ? dd_mul(d, izr[k]) : df{0.f, 0.f};
  }
  return r;
}

// Inverse CDF of an unnormalised row given by `weight(v)`: the smallest v with
// running sum > target (double-float), else the last v with weight > 0.
// Per-thread contiguous ranges, block scan, then the crossing thread's walk.
template <int T, class F>
__device__ int row_draw(int V, df target, F weight, float* shf, int* s_sel, df* s_w) {
  const int per = (V + T - 1) / T;
  const int v0 = min(V, (int)threadIdx.x * per), v1 = min(V, v0 + per);
  df loc = {0.f, 0.f};
  int lastpos = -1;
  for (int v = v0; v < v1; ++v) {
    const df w = weight(v);
    if (w.hi > 0.f) lastpos = v;
    loc = dd_add(loc, w);
  }
  df tot;
  const df ex = tblock_excl_scan_df<T>(loc, &tot, shf);
  if (threadIdx.x == 0) { s_sel[0] = 0x7fffffff; s_sel[1] = -1; }
  __syncthreads();
  if (v0 < v1 && dd_le(ex, target) && !dd_le(dd_add(ex, loc), target)) {
    df run = ex;
    for (int v = v0; v < v1; ++v) {
      const df w = weight(v);
      const df nx = dd_add(run, w);
      if (w.hi > 0.f && !dd_le(nx, target)) {
        atomicMin(&s_sel[0], v);
        break;
      }
      run = nx;
    }
  }
  if (lastpos >= 0) atomicMax(&s_sel[1], lastpos);
  __syncthreads();
  const int tok = s_sel[0] != 0x7fffffff ? s_sel[0] : max(s_sel[1], 0);
  (void)s_w;
  __syncthreads();
  return tok;
}

// ---------------------------------------------------------------- drafting
// Chunk partials of a draft row: for each 32-column chunk c in [c_lo, c_hi), (m_c, s_c) with
// m_c the chunk's largest logit (hi part) and s_c = sum exp(l - m_c), one warp
// per chunk.  l = (U_row + W1[x] W2) / T in double-float.
template <typename DT>
__device__ void draft_row_chunks(const TreeShape& ts, const DT* urow, const DT* W2, const float* a,
                                 df invT, const df* tab, float4* chunks, int c_lo, int c_hi) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int c = c_lo + warp; c < c_hi; c += NT / 32) {
    const int v = c * 32 + lane;
    df l = {-INFINITY, 0.f};
    if (v < ts.V) l = dd_mul(dd_add_f(hp_bias<DT>(a, W2, ts.V, ts.r, v), ldf(urow + v)), invT);
    const float mc = warp_max(l.hi);
    const df w = v < ts.V ? dd_exp(dd_add_f(l, -mc), tab) : df{0.f, 0.f};
    const df sc = warp_sum_df(w);
    if (lane == 0) chunks[c] = make_float4(mc, sc.hi, sc.lo, 0.f);
  }
}

// Mass of chunk c relative to the row's largest logit m: s_c e^{m_c - m}.
__device__ __forceinline__ df chunk_mass(const float4* chunks, int c, float m, const df* tab) {
  const float4 p = __ldcg(chunks + c);
  return dd_mul(df{p.y, p.z}, dd_exp(two_sum_df(p.x, -m), tab));
}

// Node index (b, n): n = 0 the root, n = 1 + s slot s; plan[b][n] = the level
// at which the node is drafted, -1 for none.
__global__ void __launch_bounds__(NT) tree_plan_kernel(TreeShape ts, const int* parent, const uint8_t* mask,
                                                       int8_t* plan) {
  const int b = blockIdx.x;
  const int* par = parent + (size_t)b * ts.N;
  const uint8_t* msk = mask + (size_t)b * ts.N;
  for (int n = threadIdx.x; n <= ts.N; n += NT) {
    const int node = n - 1;
    // depth of the node (root 0; parents checked to precede their children)
    int d = 0, ok = node < 0 || msk[node];
    for (int p = node; p >= 0 && ok; p = par[p]) {
      if (par[p] < -1 || par[p] >= p || ++d > ts.gamma) ok = 0;
    }
    int kids = 0;
    for (int s = node + 1; s < ts.N && ok; ++s) kids += (par[s] == node) & (msk[s] != 0);
    plan[(size_t)b * (ts.N + 1) + n] = (int8_t)((ok && kids > 0) ? d : -1);
  }
}

// S CTAs per node slot: CTA part of the nodes drafted at `level` computes the
// chunk partials of its share of the vocabulary.  (Nodes with a bad token or
// temperature are left to tree_draft_kernel, which reports them.)
template <typename DT>
__global__ void __launch_bounds__(NT) tree_chunks_kernel(TreeShape ts, int level, int S, const DT* U,
                                                         const DT* W1, const DT* W2, const int* anchor,
                                                         const float* temp, const int* tokens,
                                                         const int8_t* plan, float4* scratch) {
  __shared__ df s_tab[DD_EXP_TAB];
  __shared__ float s_a[256];
  const int nidx = blockIdx.x / S, part = blockIdx.x % S;
  if (plan[nidx] != level) return;
  const int b = nidx / (ts.N + 1), node = nidx % (ts.N + 1) - 1;
  const float T = temp[b];
  const int x = node < 0 ? anchor[b] : tokens[(size_t)b * ts.N + node];
  if (x < 0 || x >= ts.V || !temp_ok(T)) return;
  if (threadIdx.x < DD_EXP_TAB) dd_exp_table_entry(s_tab, threadIdx.x);
  for (int i = threadIdx.x; i < ts.r; i += NT) s_a[i] = ldf(W1 + (size_t)x * ts.r + i);
  __syncthreads();
  const int NC = (ts.V + 31) / 32;
  const int per = (NC + S - 1) / S;
  const int c_lo = min(NC, part * per), c_hi = min(NC, c_lo + per);
  const DT* urow = U + ((size_t)b * ts.gamma + level) * ts.V;
  draft_row_chunks<DT>(ts, urow, W2, s_a, dd_recip(T), s_tab, scratch + (size_t)nidx * NC, c_lo, c_hi);
}

// One CTA per node slot; the nodes drafted at `level` draw their children from
// the chunk partials of tree_chunks_kernel.
template <typename DT>
__global__ void __launch_bounds__(NT) tree_draft_kernel(TreeShape ts, int level, const DT* U, const DT* W1,
                                                        const DT* W2, const int* anchor, const float* temp,
                                                        const int* parent, const uint8_t* mask,
                                                        const float* u_draft, int* tokens, float* q_tok,
                                                        const int8_t* plan, float4* scratch,
                                                        uint32_t* status) {
  __shared__ df s_tab[DD_EXP_TAB];
  __shared__ float shf[72];
  __shared__ float s_a[256];
  __shared__ int s_sel[2];
  __shared__ df s_pref;
  const int b = blockIdx.x / (ts.N + 1), node = (int)(blockIdx.x % (ts.N + 1)) - 1;
  const int* par = parent + (size_t)b * ts.N;
  const uint8_t* msk = mask + (size_t)b * ts.N;
  if (plan[blockIdx.x] != level) return;
  const float T = temp[b];
  const int x = node < 0 ? anchor[b] : tokens[(size_t)b * ts.N + node];
  if (x < 0 || x >= ts.V || !temp_ok(T)) {
    if (threadIdx.x == 0) {
      set_status(status, (x < 0 || x >= ts.V) ? SPEC_DEV_BAD_TOKEN : SPEC_DEV_BAD_TEMP);
      for (int s = node + 1; s < ts.N; ++s)
        if (par[s] == node && msk[s]) {
          tokens[(size_t)b * ts.N + s] = -1;
          q_tok[(size_t)b * ts.N + s] = NAN;
        }
    }
    return;
  }
  if (threadIdx.x < DD_EXP_TAB) dd_exp_table_entry(s_tab, threadIdx.x);
  for (int i = threadIdx.x; i < ts.r; i += NT) s_a[i] = ldf(W1 + (size_t)x * ts.r + i);
  __syncthreads();
  const int NC = (ts.V + 31) / 32;
  float4* chunks = scratch + (size_t)blockIdx.x * NC;
  const DT* urow = U + ((size_t)b * ts.gamma + level) * ts.V;
  const df invT = dd_recip(T);
  float mx = -INFINITY;
  for (int c = threadIdx.x; c < NC; c += NT) mx = fmaxf(mx, __ldcg(chunks + c).x);
  const float m = block_max(mx, shf);
  // chunk masses: per-thread contiguous ranges
  const int per = (NC + NT - 1) / NT;
  const int c0 = min(NC, (int)threadIdx.x * per), c1 = min(NC, c0 + per);
  df loc = {0.f, 0.f};
  for (int c = c0; c < c1; ++c) loc = dd_add(loc, chunk_mass(chunks, c, m, s_tab));
  df Z;
  const df ex = block_excl_scan_df(loc, &Z, shf);
  for (int s = node + 1; s < ts.N; ++s) {
    if (!(par[s] == node && msk[s])) continue;
    const df target = dd_mul_f(Z, u_draft[(size_t)b * ts.N + s]);
    if (threadIdx.x == 0) s_sel[0] = 0x7fffffff;
    __syncthreads();
    if (c0 < c1 && dd_le(ex, target) && !dd_le(dd_add(ex, loc), target)) {
      df run = ex;
      for (int c = c0; c < c1; ++c) {
        const df nx = dd_add(run, chunk_mass(chunks, c, m, s_tab));
        if (!dd_le(nx, target)) {
          s_sel[0] = c;                       // one thread holds the crossing
          s_pref = run;
          break;
        }
        run = nx;
      }
    }
    __syncthreads();
    int cs = s_sel[0];
    df pref = s_pref;
    if (cs == 0x7fffffff) {                   // rounding: the last chunk with mass
      cs = NC - 1;
      while (cs > 0 && !(__ldcg(chunks + cs).y > 0.f)) --cs;
      pref = dd_add(Z, dd_neg(chunk_mass(chunks, cs, m, s_tab)));
    }
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x, v = cs * 32 + lane;
      df w = {0.f, 0.f};
      if (v < ts.V) {
        const df l = dd_mul(dd_add_f(hp_bias<DT>(s_a, W2, ts.V, ts.r, v), ldf(urow + v)), invT);
        w = dd_exp(dd_add_f(l, -m), s_tab);
      }
      df inc = w;
      for (int d = 1; d < 32; d <<= 1) {
        const df o = shfl_up_df(inc, d);
        if (lane >= d) inc = dd_add(inc, o);
      }
      const df hi = dd_add(pref, inc);
      const uint32_t cl = __ballot_sync(0xffffffffu, w.hi > 0.f && !dd_le(hi, target));
      const uint32_t pos = __ballot_sync(0xffffffffu, w.hi > 0.f);
      const int t = cl ? __ffs(cl) - 1 : (pos ? 31 - __clz(pos) : 0);
      const float wh = __shfl_sync(0xffffffffu, w.hi, t), wl = __shfl_sync(0xffffffffu, w.lo, t);
      if (lane == 0) {
        tokens[(size_t)b * ts.N + s] = cs * 32 + t;
        q_tok[(size_t)b * ts.N + s] = (float)(dd_to_double(df{wh, wl}) / dd_to_double(Z));
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- verification
// Walk state of a request between levels: (node, depth, accepted, done).
// Level 0 starts at the root without reading it.

// Selected children of `node` (-1: the root).
__device__ __forceinline__ int tree_kids(const TreeShape& ts, const int* par, const uint8_t* msk, int node) {
  int nk = 0;
  for (int s = node + 1; s < ts.N; ++s) nk += (par[s] == node) & (msk[s] != 0);
  return nk;
}

// S CTAs per request: the draft logits row of the request's current node
// (U row of its depth + W1[x] W2, over T, in double-float), when the node has
// selected children; CTA part takes a contiguous share of the columns.
template <typename DT>
__global__ void __launch_bounds__(NT) tree_vrow_kernel(TreeShape ts, int level, int S, const DT* U,
                                                       const DT* W1, const DT* W2, const int* anchor,
                                                       const float* temp, const int* parent,
                                                       const uint8_t* mask, const int* tokens,
                                                       const int4* state, float2* scratch) {
  __shared__ float s_a[256];
  const int b = blockIdx.x / S, part = blockIdx.x % S;
  int node = -1, depth = 0;
  if (level > 0) {
    const int4 w = __ldcg(state + b);
    if (w.w) return;                         // the walk has ended
    node = w.x;
    depth = w.y;
  }
  const int* par = parent + (size_t)b * ts.N;
  const uint8_t* msk = mask + (size_t)b * ts.N;
  // (a root with a bad anchor or temperature, or bad slots, are reported by
  // the step kernel; the tokens of selected slots were checked at level 0)
  const float T = temp[b];
  const int x = node < 0 ? anchor[b] : tokens[(size_t)b * ts.N + node];
  if (x < 0 || x >= ts.V || !temp_ok(T) || tree_kids(ts, par, msk, node) == 0) return;
  for (int i = threadIdx.x; i < ts.r; i += NT) s_a[i] = ldf(W1 + (size_t)x * ts.r + i);
  __syncthreads();
  const df invT = dd_recip(T);
  const DT* urow = U + ((size_t)b * ts.gamma + depth) * ts.V;
  float2* lq = scratch + (size_t)b * 2 * ts.V + ts.V;
  const int per = (ts.V + S - 1) / S;
  const int v1 = min(ts.V, (part + 1) * per);
  for (int v = part * per + (int)threadIdx.x; v < v1; v += NT) {
    const df l = dd_mul(dd_add_f(hp_bias<DT>(s_a, W2, ts.V, ts.r, v), ldf(urow + v)), invT);
    lq[v] = make_float2(l.hi, l.lo);
  }
}

// One CTA of TV_THREADS per request: one step of the walk at its current
// node (its double-float passes over the vocabulary are the tree
// verification's bulk, so the CTA is four times the usual width).
constexpr int TV_THREADS = 1024;
template <typename DT>
__global__ void __launch_bounds__(TV_THREADS) tree_vstep_kernel(TreeShape ts, int level, const DT* target,
                                                        const int* anchor, const float* temp, const int* parent,
                                                        const uint8_t* mask, const int* tokens,
                                                        const float* u_accept, const float* u_final,
                                                        int* accept_len, int* out_tokens, int* path,
                                                        float2* scratch, int4* state, uint32_t* status) {
  __shared__ df s_tab[DD_EXP_TAB];
  __shared__ float shf[72];
  __shared__ int s_sel[2];
  __shared__ df s_izr[TREE_MAX_SLOTS];
  __shared__ int s_bad;
  const int b = blockIdx.x;
  const int* par = parent + (size_t)b * ts.N;
  const uint8_t* msk = mask + (size_t)b * ts.N;
  const int* tok = tokens + (size_t)b * ts.N;
  int* out = out_tokens + (size_t)b * (ts.gamma + 1);
  const float T = temp[b];
  int node = -1, depth = 0, n_acc = 0;
  if (level == 0) {
    if (threadIdx.x == 0) {
      int bad = 0;
      if (!temp_ok(T)) bad |= SPEC_DEV_BAD_TEMP;
      if (anchor[b] < 0 || anchor[b] >= ts.V) bad |= SPEC_DEV_BAD_TOKEN;
      for (int s = 0; s < ts.N; ++s) {
        if (par[s] < -1 || par[s] >= s) {
          bad |= SPEC_DEV_BAD_TREE;
          continue;
        }
        int d = 1;                              // depth: parents checked to precede
        for (int p = par[s]; p >= 0 && d <= ts.gamma; p = par[p]) {
          ++d;
          if (par[p] < -1 || par[p] >= p) break;  // flagged when slot p was checked
        }
        if (d > ts.gamma) bad |= SPEC_DEV_BAD_TREE;
        if (msk[s] && (tok[s] < 0 || tok[s] >= ts.V)) bad |= SPEC_DEV_BAD_TOKEN;
      }
      s_bad = bad;
      if (bad) {
        set_status(status, (uint32_t)bad);
        accept_len[b] = -1;
        for (int j = 0; j <= ts.gamma; ++j) out[j] = -1;
        for (int j = 0; j < ts.gamma; ++j) path[(size_t)b * ts.gamma + j] = -1;
        state[b] = make_int4(-1, 0, 0, 1);
      }
    }
    __syncthreads();
    if (s_bad) return;
  } else {
    const int4 w = __ldcg(state + b);
    if (w.w) return;
    node = w.x;
    depth = w.y;
    n_acc = w.z;
  }
  if (threadIdx.x < DD_EXP_TAB) dd_exp_table_entry(s_tab, threadIdx.x);
  __syncthreads();
  float2* lp = scratch + (size_t)b * 2 * ts.V;
  const float2* lq = lp + ts.V;                // this level's draft row (tree_vrow_kernel)
  const df invT = dd_recip(T);
  const int row = node < 0 ? 0 : 1 + node;
  row_logits<DT, TV_THREADS>(ts, target + ((size_t)b * (ts.N + 1) + row) * ts.V, nullptr, nullptr, invT, lp);
  const int nk = tree_kids(ts, par, msk, node);
  __syncthreads();
  float mp, mq = 0.f;
  df Zp, Zq = {1.f, 0.f};
  row_norm<TV_THREADS>(ts.V, lp, s_tab, shf, mp, Zp);
  if (nk > 0) row_norm<TV_THREADS>(ts.V, lq, s_tab, shf, mq, Zq);
  const df izp = dd_div(df{1.f, 0.f}, Zp), izq = dd_div(df{1.f, 0.f}, Zq);
  int nrej = 0, next = -1;
  for (int s = node + 1; s < ts.N && next < 0; ++s) {
    if (!(par[s] == node && msk[s])) continue;
    const int xs = tok[s];
    const df rx = resid_prob(lp, lq, xs, mp, izp, mq, izq, s_izr, nrej, s_tab);
    const df qx = row_prob(lq, xs, mq, izq, s_tab);
    // accept iff u < r(x) / q(x), i.e. u q(x) < r(x)
    const float u = u_accept[(size_t)b * ts.N + s];
    if (!dd_le(rx, dd_mul_f(qx, u))) {
      next = s;
      break;
    }
    // rejected: r <- normalize(max(0, r - q))
    df zs = {0.f, 0.f};
    for (int v = threadIdx.x; v < ts.V; v += TV_THREADS) {
      const df d = dd_add(resid_prob(lp, lq, v, mp, izp, mq, izq, s_izr, nrej, s_tab),
                          dd_neg(row_prob(lq, v, mq, izq, s_tab)));
      if (d.hi > 0.f) zs = dd_add(zs, d);
    }
    zs = tblock_sum_df<TV_THREADS>(zs, shf);
    if (threadIdx.x == 0) s_izr[nrej] = zs.hi > 0.f ? dd_div(df{1.f, 0.f}, zs) : df{0.f, 0.f};
    __syncthreads();
    ++nrej;
  }
  if (next >= 0) {
    if (threadIdx.x == 0) {
      out[n_acc] = tok[next];
      path[(size_t)b * ts.gamma + n_acc] = next;
      state[b] = make_int4(next, depth + 1, n_acc + 1, 0);
    }
    return;
  }
  // final token from r (the target row itself at a leaf)
  const df tgt = df{u_final[b], 0.f};            // r is normalised: target u
  const int ft = row_draw<TV_THREADS>(
      ts.V, tgt, [&](int v) { return resid_prob(lp, lq, v, mp, izp, mq, izq, s_izr, nrej, s_tab); }, shf,
      s_sel, nullptr);
  if (threadIdx.x == 0) {
    out[n_acc] = ft;
    for (int j = n_acc + 1; j <= ts.gamma; ++j) out[j] = -1;
    for (int j = n_acc; j < ts.gamma; ++j) path[(size_t)b * ts.gamma + j] = -1;
    accept_len[b] = n_acc;
    state[b] = make_int4(node, depth, n_acc, 1);
  }
}

// ---------------------------------------------------------------- launchers
cudaError_t launch_tree_select(int B, int N, int gamma, const int* parent, const float* conf, int n,
                               float* survival, uint8_t* mask, float* expected, uint32_t* status,
                               cudaStream_t st) {
  tree_select_kernel<<<B, NT, 0, st>>>(B, N, gamma, parent, conf, n, survival, mask, expected, status);
  return cudaGetLastError();
}

// Workspace of the tree calls: the draft's chunk partials [B][N+1][NC] and
// plan [B][N+1]; the verification's two rows per request [B][2][V] and walk
// states [B] (the draft's area is dead by then).
static size_t tree_plan_offset(const TreeShape& ts) {
  return ((size_t)ts.B * (ts.N + 1) * ((ts.V + 31) / 32) * 16 + 255) / 256 * 256;
}
static size_t tree_state_offset(const TreeShape& ts) {
  return ((size_t)ts.B * 2 * ts.V * 8 + 255) / 256 * 256;
}
size_t tree_workspace_bytes(const TreeShape& ts) {
  const size_t draft = tree_plan_offset(ts) + (size_t)ts.B * (ts.N + 1);
  const size_t verify = tree_state_offset(ts) + (size_t)ts.B * 16;
  return draft > verify ? draft : verify;
}

template <typename DT>
cudaError_t launch_tree_draft(const TreeShape& ts, const void* U, const void* W1, const void* W2,
                              const int* anchor, const float* temp, const int* parent, const uint8_t* mask,
                              const float* u_draft, int* tokens, float* q_tok, void* scratch,
                              uint32_t* status, cudaStream_t st) {
  int8_t* plan = reinterpret_cast<int8_t*>(static_cast<unsigned char*>(scratch) + tree_plan_offset(ts));
  tree_plan_kernel<<<ts.B, NT, 0, st>>>(ts, parent, mask, plan);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  constexpr int S = 16;                         // CTAs per drafted node
  for (int level = 0; level < ts.gamma; ++level) {
    tree_chunks_kernel<DT><<<ts.B * (ts.N + 1) * S, NT, 0, st>>>(ts, level, S, (const DT*)U, (const DT*)W1,
                                                                (const DT*)W2, anchor, temp, tokens, plan,
                                                                (float4*)scratch);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    tree_draft_kernel<DT><<<ts.B * (ts.N + 1), NT, 0, st>>>(
        ts, level, (const DT*)U, (const DT*)W1, (const DT*)W2, anchor, temp, parent, mask, u_draft, tokens,
        q_tok, plan, (float4*)scratch, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <typename DT>
cudaError_t launch_tree_verify(const TreeShape& ts, const void* target, const void* U, const void* W1,
                               const void* W2, const int* anchor, const float* temp, const int* parent,
                               const uint8_t* mask, const int* tokens, const float* u_accept,
                               const float* u_final, int* accept_len, int* out_tokens, int* path,
                               void* scratch, uint32_t* status, cudaStream_t st) {
  int4* state = reinterpret_cast<int4*>(static_cast<unsigned char*>(scratch) + tree_state_offset(ts));
  const int S = ts.B >= 2400 ? 1 : (2400 + ts.B - 1) / ts.B;  // about 2400 CTAs per row pass
  // a walk accepts at most gamma nodes, so gamma + 1 steps end every request
  for (int level = 0; level <= ts.gamma; ++level) {
    tree_vrow_kernel<DT><<<ts.B * S, NT, 0, st>>>(ts, level, S, (const DT*)U, (const DT*)W1, (const DT*)W2,
                                                  anchor, temp, parent, mask, tokens, state, (float2*)scratch);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    tree_vstep_kernel<DT><<<ts.B, TV_THREADS, 0, st>>>(ts, level, (const DT*)target, anchor, temp, parent, mask,
                                               tokens, u_accept, u_final, accept_len, out_tokens, path,
                                               (float2*)scratch, state, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

#define SPEC_INST(DT)                                                                                   \
  template cudaError_t launch_tree_draft<DT>(const TreeShape&, const void*, const void*, const void*,   \
                                             const int*, const float*, const int*, const uint8_t*,      \
                                             const float*, int*, float*, void*, uint32_t*, cudaStream_t); \
  template cudaError_t launch_tree_verify<DT>(const TreeShape&, const void*, const void*, const void*,  \
                                              const void*, const int*, const float*, const int*,        \
                                              const uint8_t*, const int*, const float*, const float*,   \
                                              int*, int*, int*, void*, uint32_t*, cudaStream_t);
SPEC_INST(float)
SPEC_INST(bf16)
#undef SPEC_INST

}  // namespace spec
