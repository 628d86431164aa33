// Draft side: one step k of DSpark's sequential stage with the Markov head
// ("[논문리뷰] DSpark ...", section 1.2: p_k(v | x_0, x_<k) = softmax(U_k + B_k),
// B(x_{k-1}, .) = W1[x_{k-1}] W2; sampled left to right), tempered by T_b.
//
//   draft_tile_kernel    grid (slices of BN columns) x (row tiles of BM requests).
//                        Gathers W1[x_{k-1}] rows, computes the bias tile, adds U_k,
//                        scales by 1/T and writes per (request, slice) the softmax
//                        partial (c, m, s, q2): c = max U over the slice, m = max of
//                        x = ((U-c)+bias)/T, s = sum exp(x-m), q2 = sum exp(x-m)^2.
//                        The full-vocabulary logits never leave the SM.
//   draft_sample_kernel  one CTA per request: merges the slice partials into the
//                        normaliser, finds the slice where the running mass crosses
//                        u * Z, recomputes that slice's BN weights and scans them for
//                        the token (smallest v with F(v) > u).  Decisions within the
//                        first pass's error band of a CDF breakpoint are queued for
//                        re-decision in extended precision (spec_refine.cu).
#include "spec_tc.cuh"
#include "spec_hp.cuh"

namespace spec {

// Tensor-memory context of a CTA: accumulator columns, MMA-completion
// mbarrier and the parity of its next phase.
struct TcCtx {
  uint32_t taddr;
  uint64_t* bar;
  uint32_t phase;
};

// One (request tile, slice) of draft step k.  PATH: 0 = SIMT fp32 FMAs,
// 1 = warp MMA (mma.sync), 2 = tcgen05 / TMEM (BM = 128; `tc` set up by the
// caller).  Returns false if the MMA did not complete within the bound.
// Tokens written by other CTAs of the same launch are read through L2.
template <typename DT, int BM, int PATH>
__device__ bool draft_tile_body(const Shape& sh, int k, int slice, int mtile, const DT* __restrict__ U,
                                const DT* __restrict__ W1, const DT* __restrict__ W2,
                                const int* __restrict__ anchor, const int* tokens,
                                const float* __restrict__ temp, const Ws& ws, uint32_t* status,
                                unsigned char* smem_raw, TcCtx* tc) {
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
      t = min(max(t, 0), sh.V - 1);          // bad tokens are reported by the sampler
      s_off[m] = ((size_t)b * sh.gamma + k) * sh.V;
    } else {
      s_off[m] = 0;
    }
    s_tok[m] = t;
  }
  DT* Us;
  float* stage;
  int su;
  if constexpr (PATH == 2) {
    static_assert(BM == TC_M, "tensor-memory path uses 128-row tiles");
    unsigned char* smem = align1k(smem_raw);
    const TcLayout lay(sh.r, false);
    bf16* As = reinterpret_cast<bf16*>(smem + lay.offA);
    bf16* Wsm = reinterpret_cast<bf16*>(smem + lay.offW);
    Us = reinterpret_cast<DT*>(smem + lay.offU);
    stage = reinterpret_cast<float*>(smem + lay.offStage);
    su = BN + 8;
    __syncthreads();
    tc_load_A(As, reinterpret_cast<const bf16*>(W1), s_tok, nrows, sh.r);
    tc_load_W2(Wsm, reinterpret_cast<const bf16*>(W2), sh.V, n0, sh.r);
    load_X_rows<DT>(Us, su, U, s_off, nrows, BM, sh.V, n0);
    cp_async_commit();
    cp_async_wait_all();
    fence_async_shared();
    tc_fence_before();
    __syncthreads();
    const bool ok = bias_tile_tc(As, Wsm, sh.r, tc->taddr, tc->bar, tc->phase, stage);
    if (!ok) {
      if (threadIdx.x == 0) set_status(status, SPEC_DEV_TIMEOUT);
      mbar_wait(tc->bar, tc->phase, 1u << 22);   // let an in-flight MMA drain
      tc->phase ^= 1u;
      return false;
    }
    tc->phase ^= 1u;
    __syncthreads();
  } else {
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

  // ---- epilogue: TPR threads per row, each COLS consecutive columns
  constexpr int TPR = NT / BM, COLS = BN / TPR;
  constexpr int SS = TileLayout<DT>::SS;
  const int m = threadIdx.x / TPR, part = threadIdx.x % TPR;
  const bool rowok = m < nrows;
  const int b = m0 + m;
  const float invT = rowok ? 1.0f / temp[b] : 1.0f;
  const int cbeg = part * COLS;
  const int cend = min(cbeg + COLS, sh.V - n0);   // valid columns of this thread
  const DT* urow = Us + (size_t)m * su;
  const float* brow = stage + m * SS;

  float c = -INFINITY;
  for (int i = cbeg; i < cend; ++i) c = fmaxf(c, tof(urow[i]));
  c = group_max<TPR>(c);
  float xm = -INFINITY;
  for (int i = cbeg; i < cend; ++i) xm = fmaxf(xm, fast_x(tof(urow[i]), c, brow[i], invT));
  xm = group_max<TPR>(xm);
  Kahan ks;
  float q2 = 0.f;
  for (int i = cbeg; i < cend; ++i) {
    float w = fast_w(fast_x(tof(urow[i]), c, brow[i], invT), xm);
    ks.add(w);
    q2 = fmaf(w, w, q2);
  }
  df s = group_sum_df<TPR>(ks.value());
  q2 = group_sum<TPR>(q2);
  if (rowok && part == 0)
    ws.dpart[(size_t)b * sh.NS + slice] = make_float4(c, xm, df_d(s) /*rounded*/, q2);
  return true;
}

// Weighted slice mass relative to the row's largest slice reference, in units
// of exp(reference logit):  f = exp((c - cM)/T + (m - mM)).
__device__ __forceinline__ float slice_factor(float4 p, float cM, float mM, float invT) {
  float a = __fadd_rn(__fmul_rn(__fsub_rn(p.x, cM), invT), __fsub_rn(p.y, mM));
  return expf(a);
}

// Draw token x_{k+1} of request b from its slice partials (one CTA).  Queues
// the draw on `counter` / ws.items when it lies inside the error band.
// `dsm` holds an r x BN slab.  Partials and tokens written by other CTAs of
// the same launch are read through L2.
template <typename DT>
__device__ void draft_sample_body(const Shape& sh, int k, int b, const DT* __restrict__ U,
                                  const DT* __restrict__ W1, const DT* __restrict__ W2,
                                  const int* __restrict__ anchor, const float* __restrict__ temp,
                                  const float* __restrict__ u_draft, int* tokens, float* q_tok,
                                  double* lse_q, float* diag, uint32_t* status, const Ws& ws,
                                  const Eps& eps, uint32_t* counter, unsigned char* dsm) {
  DT* slab = reinterpret_cast<DT*>(dsm);      // [r][BN] W2 slab of the crossing slice
  __shared__ float sh_f[72];
  __shared__ float s_a[256];
  __shared__ float s_part[2][BN];
  __shared__ int s_slice;
  __shared__ float s_pref[2];
  __shared__ float s_w[BN];

  __syncthreads();      // previous use of the shared buffers is finished
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
  const float invT = 1.0f / T;
  const float4* P = ws.dpart + (size_t)b * sh.NS;
  auto part = [&](int s) { return __ldcg(P + s); };

  // ---- reference slice: largest c/T + m (ties: any; only a shift)
  const int per = (sh.NS + NT - 1) / NT;
  const int s0 = threadIdx.x * per, s1 = min(s0 + per, sh.NS);
  float best = -INFINITY;
  int bidx = 0;
  for (int s = s0; s < s1; ++s) {
    float4 p = part(s);
    float key = fmaf(p.x, invT, p.y);
    if (key > best) { best = key; bidx = s; }
  }
  float bmax = block_max(best, sh_f);
  // lowest index attaining the max
  int cand = (best == bmax) ? bidx : 0x7fffffff;
  for (int m = 16; m; m >>= 1) cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, m));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) reinterpret_cast<int*>(sh_f)[threadIdx.x >> 5] = cand;
  __syncthreads();
  if (threadIdx.x == 0) {
    int c2 = 0x7fffffff;
    for (int w = 0; w < NT / 32; ++w) c2 = min(c2, reinterpret_cast<int*>(sh_f)[w]);
    s_slice = c2;
  }
  __syncthreads();
  const float4 PM = part(s_slice);
  const float cM = PM.x, mM = PM.y;
  __syncthreads();

  // ---- per-thread slice masses (double-float) and error-estimate sums
  df loc = {0.f, 0.f};
  float q2 = 0.f, m2 = 0.f;
  for (int s = s0; s < s1; ++s) {
    float4 p = part(s);
    float f = slice_factor(p, cM, mM, invT);
    float w = p.z * f;
    loc = df_addf(loc, w);
    q2 = fmaf(p.w * f, f, q2);
    m2 = fmaf(w, w, m2);
  }
  df Zdf;
  df excl = block_excl_scan_df(loc, &Zdf, sh_f);
  q2 = block_sum(q2, sh_f);
  m2 = block_sum(m2, sh_f);
  const double Z = df_d(Zdf);
  const float u = u_draft[ok];
  const df target = df_from_d((double)u * Z);

  // ---- crossing slice: first s with prefix_incl(s) > target
  if (threadIdx.x == 0) s_slice = 0x7fffffff;
  __syncthreads();
  int my_slice = -1;
  df my_pref = {0.f, 0.f};
  {
    df run = excl;
    df tneg = df_neg(target);
    if (df_d(df_add(excl, tneg)) <= 0.0 && df_d(df_add(df_add(excl, loc), tneg)) > 0.0) {
      for (int s = s0; s < s1; ++s) {
        float4 p = part(s);
        df nxt = df_addf(run, p.z * slice_factor(p, cM, mM, invT));
        if (df_d(df_add(nxt, tneg)) > 0.0) {
          my_slice = s;
          my_pref = run;
          atomicMin(&s_slice, s);
          break;
        }
        run = nxt;
      }
    }
  }
  __syncthreads();
  if (my_slice >= 0 && my_slice == s_slice) {
    s_pref[0] = my_pref.hi;
    s_pref[1] = my_pref.lo;
  }
  __syncthreads();
  bool fallback = false;
  if (s_slice == 0x7fffffff) {
    // rounding left the total at or below u*Z: last slice with mass
    fallback = true;
    if (threadIdx.x == 0) {
      int sl = sh.NS - 1;
      while (sl > 0 && !(part(sl).z > 0.f)) --sl;
      s_slice = sl;
    }
    __syncthreads();
    // prefix of everything before that slice
    df run = {0.f, 0.f};
    if (threadIdx.x == 0) {
      for (int s = 0; s < s_slice; ++s) {
        float4 p = part(s);
        run = df_addf(run, p.z * slice_factor(p, cM, mM, invT));
      }
      s_pref[0] = run.hi;
      s_pref[1] = run.lo;
    }
    __syncthreads();
  }
  const int sl = s_slice;
  const df pref = {s_pref[0], s_pref[1]};
  const float4 PS = part(sl);
  const float fS = slice_factor(PS, cM, mM, invT);

  // ---- recompute the slice's weights (bias by SIMT: two halves of k, W2 slab in smem)
  for (int i = threadIdx.x; i < sh.r; i += NT) s_a[i] = ldf(W1 + (size_t)prev * sh.r + i);
  const int n0 = sl * BN;
  stage_w2_slab<DT>(slab, W2, sh.V, 0, sh.r, n0, BN);
  {
    const int col = threadIdx.x % BN, half = threadIdx.x / BN;
    const int kh = sh.r / 2;
    float acc = 0.f;
    for (int i = half * kh; i < half * kh + kh; ++i) acc = fmaf(s_a[i], tof(slab[i * BN + col]), acc);
    s_part[half][col] = acc;
  }
  __syncthreads();
  float w = 0.f;
  if (threadIdx.x < BN) {
    const int v = n0 + threadIdx.x;
    if (v < sh.V) {
      float bias = __fadd_rn(s_part[0][threadIdx.x], s_part[1][threadIdx.x]);
      w = fast_w(fast_x(ldf(U + ok * sh.V + v), PS.x, bias, invT), PS.y);
    }
    s_w[threadIdx.x] = w;
  }
  __syncthreads();
  // in-slice target in slice units
  const double tin = (df_d(target) - df_d(pref)) / (double)fS;
  df wtot;
  df wex = block_excl_scan_df(df_make(threadIdx.x < BN ? w : 0.f), &wtot, sh_f);
  __shared__ int s_tok;
  __shared__ float s_lo[2], s_hi[2];
  if (threadIdx.x == 0) s_tok = 0x7fffffff;
  __syncthreads();
  double my_lo = 0.0, my_hi = 0.0;
  bool claim = false;
  if (threadIdx.x < BN && w > 0.f) {
    my_lo = df_d(wex);
    my_hi = df_d(df_addf(wex, w));
    if (my_lo <= tin && my_hi > tin) {
      claim = true;
      atomicMin(&s_tok, (int)threadIdx.x);
    }
  }
  __syncthreads();
  if (claim && (int)threadIdx.x == s_tok) {
    s_lo[0] = (float)(tin - my_lo);
    s_hi[0] = (float)(my_hi - tin);
  }
  __syncthreads();
  if (s_tok == 0x7fffffff) {
    fallback = true;
    if (threadIdx.x == 0) {
      int t = BN - 1;
      while (t > 0 && !(s_w[t] > 0.f)) --t;
      s_tok = t;
      s_lo[0] = 0.f;
      s_hi[0] = 0.f;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const int tok = n0 + s_tok;
    const double dmargin = fmin((double)s_lo[0], (double)s_hi[0]) * (double)fS / Z;
    const double qrow = sqrt((double)q2) / Z, mrow = sqrt((double)m2) / Z;
    const double band = (double)eps.scale * ((double)eps.elem * qrow + (double)eps.slice * mrow +
                                             (double)eps.abs_);
    const double lse = ((double)cM * (1.0 / (double)T) + (double)mM) + log(Z);
    tokens[ok] = tok;
    q_tok[ok] = (float)((double)s_w[s_tok] * (double)fS / Z);
    lse_q[ok] = lse;
    if (diag) {
      diag[ok * 4 + 0] = (float)((double)s_lo[0] * fS / Z);
      diag[ok * 4 + 1] = (float)((double)s_hi[0] * fS / Z);
      diag[ok * 4 + 2] = (float)band;
      diag[ok * 4 + 3] = (float)tok;
    }
    if (fallback || dmargin <= band) {
      uint32_t it = atomicAdd(counter, 1u);
      if ((int)it < ws.max_items) {
        HpItem h;
        h.b = b; h.j = k; h.kind = HP_DRAFT; h.prev = prev; h.u = u; h.fast_token = tok;
        h.shift_q = lse; h.shift_p = 0.0;
        ws.items[it] = h;
      } else {
        set_status(status, SPEC_DEV_OVERFLOW);
      }
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------- kernels
// One launch per step: tiles (grid = slices x request tiles).
template <typename DT, int BM, int PATH>
__global__ void __launch_bounds__(NT) draft_tile_kernel(Shape sh, int k, const DT* __restrict__ U,
                                                        const DT* __restrict__ W1,
                                                        const DT* __restrict__ W2,
                                                        const int* __restrict__ anchor,
                                                        const int* __restrict__ tokens,
                                                        const float* __restrict__ temp, Ws ws,
                                                        uint32_t* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ uint64_t s_bar;
  __shared__ uint32_t s_holder;
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) ws.ctrl[CTRL_ITEMS] = 0;
  TcCtx tc{0u, &s_bar, 0u};
  if constexpr (PATH == 2) {
    if (threadIdx.x == 0) mbar_init(&s_bar, 1);
    if (threadIdx.x < 32) tc_alloc(&s_holder, TC_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    tc.taddr = s_holder;
  }
  draft_tile_body<DT, BM, PATH>(sh, k, blockIdx.x, blockIdx.y, U, W1, W2, anchor, tokens, temp, ws,
                                status, smem_raw, &tc);
  if constexpr (PATH == 2) {
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) tc_dealloc(tc.taddr, TC_TMEM_COLS);
  }
}

// One launch per step: one CTA per request.
template <typename DT>
__global__ void __launch_bounds__(NT) draft_sample_kernel(
    Shape sh, int k, const DT* __restrict__ U, const DT* __restrict__ W1, const DT* __restrict__ W2,
    const int* __restrict__ anchor, const float* __restrict__ temp,
    const float* __restrict__ u_draft, int* tokens, float* q_tok, double* lse_q, float* diag,
    uint32_t* status, Ws ws, Eps eps) {
  extern __shared__ __align__(16) unsigned char dsm[];
  draft_sample_body<DT>(sh, k, blockIdx.x, U, W1, W2, anchor, temp, u_draft, tokens, q_tok, lse_q,
                        diag, status, ws, eps, ws.ctrl + CTRL_ITEMS, dsm);
}

struct DraftParams {
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
};

// The whole draft in one cooperative launch: for each step k, the tile phase
// (tiles strided over the CTAs), a grid barrier, the sampling phase (requests
// strided over the CTAs), a grid barrier, and -- only when that step queued
// near-boundary draws -- the two extended-precision phases, each followed by
// a grid barrier.  Tensor memory is allocated once per CTA.
template <typename DT, int BM, int PATH>
__global__ void __launch_bounds__(NT, 1) draft_persistent_kernel(DraftParams P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ uint64_t s_bar;
  __shared__ uint32_t s_holder;
  const Shape& sh = P.sh;
  const DT* U = (const DT*)P.U;
  const DT* W1 = (const DT*)P.W1;
  const DT* W2 = (const DT*)P.W2;
  uint32_t* ctrl = P.ws.ctrl;
  TcCtx tc{0u, &s_bar, 0u};
  if constexpr (PATH == 2) {
    if (threadIdx.x == 0) mbar_init(&s_bar, 1);
    if (threadIdx.x < 32) tc_alloc(&s_holder, TC_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    tc.taddr = s_holder;
  }
  uint32_t gen = threadIdx.x == 0 ? ld_acquire_gpu(ctrl + CTRL_BAR_GEN) : 0u;
  const HpRows R{P.U, P.U, P.W1, P.W2, P.temp};
  const int n_mt = (sh.B + BM - 1) / BM;
  const int n_tiles = sh.NS * n_mt;
  const uint32_t G = gridDim.x;
  for (int k = 0; k < sh.gamma; ++k) {
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += G)
      ok = draft_tile_body<DT, BM, PATH>(sh, k, t % sh.NS, t / sh.NS, U, W1, W2, P.anchor, P.tokens,
                                         P.temp, P.ws, P.status, smem_raw, &tc);
    if (!ok) {
      if (threadIdx.x == 0) atomicExch(ctrl + CTRL_ABORT, 1u);
      break;
    }
    if (!grid_sync(ctrl, G, gen, P.status)) break;
    for (int b = blockIdx.x; b < sh.B; b += G)
      draft_sample_body<DT>(sh, k, b, U, W1, W2, P.anchor, P.temp, P.u_draft, P.tokens, P.q_tok,
                            P.lse_q, P.diag, P.status, P.ws, P.eps, ctrl + CTRL_STEP0 + k,
                            smem_raw);
    if (!grid_sync(ctrl, G, gen, P.status)) break;
    const int n = min((int)__ldcg(ctrl + CTRL_STEP0 + k), P.ws.max_items);
    if (n > 0) {
      hp_sums_body<DT>(sh, R, P.ws, 0, n, smem_raw);
      if (!grid_sync(ctrl, G, gen, P.status)) break;
      hp_decide_body<DT>(sh, R, P.ws, n, P.tokens, P.q_tok, P.lse_q, nullptr, P.status, smem_raw);
      if (!grid_sync(ctrl, G, gen, P.status)) break;
    }
  }
  if constexpr (PATH == 2) {
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) tc_dealloc(tc.taddr, TC_TMEM_COLS);
  }
}

// ---------------------------------------------------------------- launchers
template <typename DT, int BM, int PATH>
static cudaError_t launch_tile(const Shape& sh, int k, const DT* U, const DT* W1, const DT* W2,
                               const int* anchor, const int* tokens, const float* temp, const Ws& ws,
                               uint32_t* status, cudaStream_t st) {
  const size_t smem = PATH == 2 ? TcLayout(sh.r, false).total : TileLayout<DT>(BM, sh.r, false).total;
  auto kern = draft_tile_kernel<DT, BM, PATH>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(sh.NS, (sh.B + BM - 1) / BM);
  kern<<<grid, NT, smem, st>>>(sh, k, U, W1, W2, anchor, tokens, temp, ws, status);
  return cudaGetLastError();
}

// path: 0 SIMT, 1 warp MMA, 2 tcgen05 (bf16 with r % 64 == 0 only; else warp MMA)
template <typename DT>
cudaError_t launch_draft_tile(const Shape& sh, int k, const void* U, const void* W1, const void* W2,
                              const int* anchor, const int* tokens, const float* temp, const Ws& ws,
                              int path, uint32_t* status, cudaStream_t st) {
  const DT* u = (const DT*)U;
  const DT* w1 = (const DT*)W1;
  const DT* w2 = (const DT*)W2;
  const int BM = sh.B <= 32 ? 32 : (sh.B <= 64 ? 64 : 128);
#define SPEC_TILE(BMV, P) launch_tile<DT, BMV, P>(sh, k, u, w1, w2, anchor, tokens, temp, ws, status, st)
  if (path == 0 || sizeof(DT) == 4) {
    if (BM == 32) return SPEC_TILE(32, 0);
    if (BM == 64) return SPEC_TILE(64, 0);
    return SPEC_TILE(128, 0);
  }
  if constexpr (sizeof(DT) == 2) {
    if (path == 2 && sh.r % 64 == 0) return SPEC_TILE(128, 2);
  }
  if (BM == 32) return SPEC_TILE(32, 1);
  if (BM == 64) return SPEC_TILE(64, 1);
  return SPEC_TILE(128, 1);
#undef SPEC_TILE
}

template <typename DT>
cudaError_t launch_draft_sample(const Shape& sh, int k, const void* U, const void* W1,
                                const void* W2, const int* anchor, const float* temp,
                                const float* u_draft, int* tokens, float* q_tok, double* lse_q,
                                float* diag, uint32_t* status, const Ws& ws, const Eps& eps,
                                cudaStream_t st) {
  const size_t smem = (size_t)sh.r * BN * sizeof(DT);
  cudaError_t e = cudaFuncSetAttribute(draft_sample_kernel<DT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  draft_sample_kernel<DT><<<sh.B, NT, smem, st>>>(sh, k, (const DT*)U, (const DT*)W1, (const DT*)W2,
                                               anchor, temp, u_draft, tokens, q_tok, lse_q, diag,
                                               status, ws, eps);
  return cudaGetLastError();
}

template <typename DT, int BM, int PATH>
static cudaError_t launch_persist(const DraftParams& P, int nsm, cudaStream_t st) {
  size_t smem = PATH == 2 ? TcLayout(P.sh.r, false).total : TileLayout<DT>(BM, P.sh.r, false).total;
  smem = smem > (size_t)P.sh.r * HPB * sizeof(DT) ? smem : (size_t)P.sh.r * HPB * sizeof(DT);
  auto kern = draft_persistent_kernel<DT, BM, PATH>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int n_tiles = P.sh.NS * ((P.sh.B + BM - 1) / BM);
  int G = nsm;                             // one CTA per SM (all must be co-resident)
  G = G < n_tiles ? G : n_tiles;
  G = G > P.sh.B ? G : (P.sh.B < nsm ? P.sh.B : nsm);
  G = G < 1 ? 1 : G;
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
                                    int nsm, cudaStream_t st) {
  DraftParams P{sh, U, W1, W2, anchor, temp, u_draft, tokens, q_tok, lse_q, diag, status, ws, eps};
  const int BM = sh.B <= 32 ? 32 : (sh.B <= 64 ? 64 : 128);
  if (path == 0 || sizeof(DT) == 4) {
    if (BM == 32) return launch_persist<DT, 32, 0>(P, nsm, st);
    if (BM == 64) return launch_persist<DT, 64, 0>(P, nsm, st);
    return launch_persist<DT, 128, 0>(P, nsm, st);
  }
  if constexpr (sizeof(DT) == 2) {
    if (path == 2 && sh.r % 64 == 0) return launch_persist<DT, 128, 2>(P, nsm, st);
  }
  if (BM == 32) return launch_persist<DT, 32, 1>(P, nsm, st);
  if (BM == 64) return launch_persist<DT, 64, 1>(P, nsm, st);
  return launch_persist<DT, 128, 1>(P, nsm, st);
}

template cudaError_t launch_draft_persistent<float>(const Shape&, const void*, const void*,
                                                    const void*, const int*, const float*,
                                                    const float*, int*, float*, double*, float*,
                                                    uint32_t*, const Ws&, const Eps&, int, int,
                                                    cudaStream_t);
template cudaError_t launch_draft_persistent<bf16>(const Shape&, const void*, const void*,
                                                   const void*, const int*, const float*,
                                                   const float*, int*, float*, double*, float*,
                                                   uint32_t*, const Ws&, const Eps&, int, int,
                                                   cudaStream_t);
template cudaError_t launch_draft_tile<float>(const Shape&, int, const void*, const void*,
                                              const void*, const int*, const int*, const float*,
                                              const Ws&, int, uint32_t*, cudaStream_t);
template cudaError_t launch_draft_tile<bf16>(const Shape&, int, const void*, const void*,
                                             const void*, const int*, const int*, const float*,
                                             const Ws&, int, uint32_t*, cudaStream_t);
template cudaError_t launch_draft_sample<float>(const Shape&, int, const void*, const void*,
                                                const void*, const int*, const float*, const float*,
                                                int*, float*, double*, float*, uint32_t*, const Ws&,
                                                const Eps&, cudaStream_t);
template cudaError_t launch_draft_sample<bf16>(const Shape&, int, const void*, const void*,
                                               const void*, const int*, const float*, const float*,
                                               int*, float*, double*, float*, uint32_t*, const Ws&,
                                               const Eps&, cudaStream_t);

}  // namespace spec
