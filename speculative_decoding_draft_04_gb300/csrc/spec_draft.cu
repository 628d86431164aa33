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

#include "spec_sample.cuh"
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

// ---------------------------------------------------------------- kernel
// The whole draft in one cooperative launch: for each step k, [the RNN head's
// gate phase and a grid barrier,] the tile phase (tiles strided over the CTAs,
// then the previous step's near-boundary draws re-decided by the CTAs as they
// finish their tiles), a grid barrier, the sampling phase (requests strided
// over the CTAs) and a grid barrier; then the last step's re-decisions and,
// if a re-decision changed a token, the steps after it again with their
// re-decisions in place.  Tensor memory is allocated once per CTA.
template <typename DT, int BM, int PATH, int HOOK>
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
  // HOOK_STALL (a test build): the first barrier expects one arrival more
  // than the grid has, so it can only end by its time limit
  auto gsync = [&]() {
    return grid_sync(ctrl, G, gen, P.status, (HOOK == HOOK_STALL && gen == 0u) ? 1u : 0u);
  };
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
      if (!gsync()) return false;
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
    if (!gsync()) return false;
    if (tr) tr[k * TRACE_SLOTS + 2] = globaltimer_ns();
    for (int b = blockIdx.x; b < sh.B; b += G)
      draft_sample_body<DT, HOOK>(sh, k, b, U, W1, W2, P.anchor, P.temp, P.u_draft, P.tokens,
                                  P.q_tok, P.lse_q, P.diag, P.status, P.ws, P.eps,
                                  ctrl + CTRL_STEP0 + k, P.ws.max_items, smem_raw);
    if (tr) tr[k * TRACE_SLOTS + 3] = globaltimer_ns();
    if (!gsync()) return false;
    if (tr) tr[k * TRACE_SLOTS + 4] = globaltimer_ns();
    const int n = min((int)__ldcg(ctrl + CTRL_STEP0 + k), P.ws.max_items);
    n_prev = deferred ? n : 0;
    if (!deferred && n > 0) {
      hp_sums_body<DT>(sh, R, P.ws, 0, n, smem_raw, true, P.tokens, P.q_tok, P.lse_q, P.status);
      if (tr) tr[k * TRACE_SLOTS + 5] = globaltimer_ns();
      if (!gsync()) return false;
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
    good = gsync();
  }
  if (good) {
    const uint32_t redo = __ldcg(ctrl + CTRL_REDO);
    const int k0 = sh.gamma - (int)redo + 1;            // first step to redo
    if (redo > 0 && k0 < sh.gamma) {
      if (blockIdx.x == 0 && threadIdx.x == 0)
        for (int k = k0; k < sh.gamma; ++k) ctrl[CTRL_STEP0 + k] = 0u;
      good = gsync();
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
template <typename DT, int BM, int PATH, int HOOK = HOOK_NONE>
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
  auto kern = draft_persistent_kernel<DT, BM, PATH, HOOK>;
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
// `hook` selects a test build (HOOK_PERTURB, HOOK_STALL), available on the
// fp32 path for batches of up to 32 requests and on the tensor-memory path;
// elsewhere a hook request fails with cudaErrorNotSupported.
template <typename DT>
cudaError_t launch_draft_persistent(const Shape& sh, const void* U, const void* W1, const void* W2,
                                    const int* anchor, const float* temp, const float* u_draft,
                                    int* tokens, float* q_tok, double* lse_q, float* diag,
                                    uint32_t* status, const Ws& ws, const Eps& eps, int path,
                                    int nsm, cudaStream_t st, const RnnParams* rnn, int hook) {
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
  if (hook != HOOK_NONE) {
    const bool tc = sizeof(DT) == 2 && path == 2 && sh.r % 64 == 0;
    if (!tc && (path == 0 || sizeof(DT) == 4) && BM == 32)
      return hook == HOOK_PERTURB ? launch_persist<DT, 32, 0, HOOK_PERTURB>(P, nsm, st)
                                  : launch_persist<DT, 32, 0, HOOK_STALL>(P, nsm, st);
    if constexpr (sizeof(DT) == 2) {
      if (tc) {
        cudaError_t e = encode_u_map(sh, U, &P.maps.u);
        if (e == cudaSuccess) e = encode_w2_map(sh, W2, &P.maps.w2);
        if (e != cudaSuccess) return e;
        return hook == HOOK_PERTURB ? launch_persist<DT, 128, 2, HOOK_PERTURB>(P, nsm, st)
                                    : launch_persist<DT, 128, 2, HOOK_STALL>(P, nsm, st);
      }
    }
    return cudaErrorNotSupported;
  }
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
                                                    cudaStream_t, const RnnParams*, int);
template cudaError_t launch_draft_persistent<bf16>(const Shape&, const void*, const void*,
                                                   const void*, const int*, const float*,
                                                   const float*, int*, float*, double*, float*,
                                                   uint32_t*, const Ws&, const Eps&, int, int,
                                                   cudaStream_t, const RnnParams*, int);

}  // namespace spec
