// Extended-precision re-decision of the verification's queued draws (the
// correction draw from normalize(max(0, p_n - q_n)) and the bonus draw from
// p_L, "Speculative Decoding Part 1", VESSL AI blog, section "수락 규칙") in
// one cooperative launch, with the vocabulary split across the CTAs instead
// of into (item, block) work units.
//
//   pass 0   every CTA walks its share of 32-column chunks (one warp per
//            chunk, lane = column) and computes, for each queued item, the
//            double-float target weight exp(t/T - lse_p) and, for a
//            correction draw, the draft weight exp((U + W1[x] W2)/T - lse_q)
//            with the transition bias as a compensated dot product (the
//            chunks' W2 columns staged in shared memory, eight chunks at a
//            time); per chunk the two sums, and the weights themselves for
//            the first ws.hpw_items items;
//   barrier
//   pass 1   every CTA sums the chunk sums of each correction item in the same
//            fixed order (so all hold the same normalisers), CTA 0 records
//            their reciprocals, and each CTA forms the residual
//            max(0, p/Z_p - q/Z_q) of its columns from the kept weights and
//            writes its chunk sums;
//   barrier
//   decide   one CTA per item finds the crossing chunk and scans it
//            (hp_decide_item, from the kept weights).
//
// The arithmetic of every weight is spec_hp.cuh's (double-float exponential,
// compensated sums), so the decisions agree with the float64 oracle except
// within about 1e-13 of a boundary.
#include "spec_hp.cuh"

namespace spec {

struct VrParams {
  Shape sh;
  HpRows R;
  Ws ws;
  int* out_tokens;
  uint32_t* status;
};

constexpr int VR_PIECE = 8;        // chunks per staged W2 piece (one per warp)

template <typename DT>
__global__ void __launch_bounds__(NT, 1) verify_redecide_kernel(const __grid_constant__ VrParams P) {
  extern __shared__ __align__(16) unsigned char dsm[];     // W2 piece (r x 256); the decisions' slab
  __shared__ HpShared S;
  __shared__ float s_a[16][256];                         // the correction items' W1 rows
  __shared__ HpItem s_it[16];
  __shared__ ItemCtx<DT> s_ctx[16];
  __shared__ df s_rc[16][2];                              // 1/Z_p, 1/Z_q per correction item
  const Shape& sh = P.sh;
  const Ws& ws = P.ws;
  uint32_t* ctrl = ws.ctrl;
  const int n = min((int)__ldcg(ctrl + CTRL_ITEMS), ws.max_items);
  if (n == 0) return;                                     // the common case: nothing queued
  const uint32_t G = gridDim.x;
  uint32_t gen = 0u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this CTA's chunks: [q0, q1) of NC, one warp per chunk at a time
  const int per = (sh.NC + (int)G - 1) / (int)G;
  const int q0 = min(sh.NC, (int)blockIdx.x * per), q1 = min(sh.NC, q0 + per);
  hp_table(S.tab);
  const int nk = min(n, ws.hpw_items);                    // items whose weights are kept

  // ---- pass 0: the CTA's chunks in pieces of 8 (one per warp), their W2
  // columns staged in shared memory by cp.async (one round trip per piece);
  // items in groups of 16 (their rows and contexts staged together)
  DT* w2s = reinterpret_cast<DT*>(dsm);                   // [r][HPB], the layout hp_bias_slab reads
  constexpr int PCOLS = VR_PIECE * CW;
  static_assert(PCOLS == HPB, "a staged piece is one extended-precision block wide");
  for (int p0 = q0; p0 < q1; p0 += VR_PIECE) {
    const int pc = min(VR_PIECE, q1 - p0);                 // chunks in this piece
    __syncthreads();                                       // the previous piece is consumed
    {
      constexpr int E = 16 / sizeof(DT);
      const int cpr = PCOLS / E;                           // 16-byte copies per W2 row
      for (int c = threadIdx.x; c < sh.r * cpr; c += NT) {
        const int i = c / cpr, qq = c - i * cpr;
        const int col = p0 * CW + qq * E;
        const bool valid = qq * E < pc * CW && col < sh.V;
        cp_async16(w2s + (size_t)i * PCOLS + qq * E, valid ? (const DT*)P.R.W2 + (size_t)i * sh.V + col
                                                           : (const DT*)P.R.W2, valid);
      }
      cp_async_commit();
    }
    for (int g0 = 0; g0 < n; g0 += 16) {
      const int cnt = min(16, n - g0);
      __syncthreads();
      if ((int)threadIdx.x < cnt) {
        s_it[threadIdx.x] = ldcg_item(ws.items + g0 + threadIdx.x);
        s_ctx[threadIdx.x] = item_ctx<DT>(sh, P.R, s_it[threadIdx.x]);
      }
      __syncthreads();
      for (int q = threadIdx.x; q < cnt * sh.r; q += NT) {
        const int i = q / sh.r, e = q - i * sh.r;
        const HpItem& it = s_it[i];
        s_a[i][e] = it.kind == HP_RESID ? ldf((const DT*)P.R.W1 + (size_t)it.prev * sh.r + e) : 0.f;
      }
      cp_async_wait_all();
      __syncthreads();
      if (warp < pc) {
        const int ch = p0 + warp;
        const int v = ch * CW + lane;
        const bool in = v < sh.V;
        for (int i = 0; i < cnt; ++i) {
          const HpItem& it = s_it[i];
          const ItemCtx<DT>& c = s_ctx[i];
          df ep = {0.f, 0.f}, eq = {0.f, 0.f};
          if (in) {
            ep = hp_wp_val<DT>(c, ldf(c.Trow + v), S.tab);
            // the bias in the same order and precision as every other
            // re-decision pass (hp_bias), from the staged columns
            if (it.kind == HP_RESID)
              eq = hp_wq_val<DT>(c, hp_bias_slab<DT>(s_a[i], w2s, sh.r, warp * CW + lane), ldf(c.Urow + v),
                                 S.tab);
            if (g0 + i < nk) ws.hpw[(size_t)(g0 + i) * sh.V + v] = make_float4(eq.hi, eq.lo, ep.hi, ep.lo);
          }
          const df A = warp_sum_df(ep);
          if (lane == 0) item_sums(ws, sh, g0 + i, 0)[ch] = make_float2(A.hi, A.lo);
          if (it.kind == HP_RESID) {
            const df Bq = warp_sum_df(eq);
            if (lane == 0) item_sums(ws, sh, g0 + i, 1)[ch] = make_float2(Bq.hi, Bq.lo);
          }
        }
      }
    }
  }
  if (!grid_sync(ctrl, G, gen, P.status)) return;

  // ---- pass 1: normalisers and residual chunk sums of the correction items
  bool any_resid = false;
  for (int g0 = 0; g0 < n; g0 += 16) {
    const int cnt = min(16, n - g0);
    __syncthreads();
    if ((int)threadIdx.x < cnt) {
      s_it[threadIdx.x] = ldcg_item(ws.items + g0 + threadIdx.x);
      s_ctx[threadIdx.x] = item_ctx<DT>(sh, P.R, s_it[threadIdx.x]);
    }
    __syncthreads();
    for (int i = 0; i < cnt; ++i) {
      if (s_it[i].kind != HP_RESID) continue;
      any_resid = true;
      // every CTA sums the same chunk sums in the same order
      const df izp = shared_recip(item_total(item_sums(ws, sh, g0 + i, 0), sh.NC, S.shf), &s_rc[i][0]);
      const df izq = shared_recip(item_total(item_sums(ws, sh, g0 + i, 1), sh.NC, S.shf), &s_rc[i][1]);
      if (blockIdx.x == 0 && threadIdx.x == 0) ws.hpnorm[g0 + i] = make_float4(izp.hi, izp.lo, izq.hi, izq.lo);
      const bool kept = g0 + i < nk;
      if (!kept && threadIdx.x < 64) {
        // (beyond the kept items the weights are recomputed column by column)
        for (int e = threadIdx.x; e < sh.r; e += 64)
          s_a[i][e] = ldf((const DT*)P.R.W1 + (size_t)s_it[i].prev * sh.r + e);
      }
      __syncthreads();
      for (int ch = q0 + warp; ch < q1; ch += NT / 32) {
        const int v = ch * CW + lane;
        df rr = {0.f, 0.f};
        if (v < sh.V) {
          df eq, ep;
          if (kept) {
            const float4 w4 = __ldcg(ws.hpw + (size_t)(g0 + i) * sh.V + v);
            eq = {w4.x, w4.y};
            ep = {w4.z, w4.w};
          } else {
            hp_weights<DT>(sh, P.R, s_it[i], s_ctx[i], s_a[i], S.tab, v, eq, ep);
          }
          rr = hp_resid(ep, eq, izp, izq);
        }
        const df C = warp_sum_df(rr);
        if (lane == 0) item_sums(ws, sh, g0 + i, 2)[ch] = make_float2(C.hi, C.lo);
      }
    }
  }
  // (every CTA reaches the same any_resid; without correction items the first
  // barrier already orders the decisions after every CTA's pass 0)
  if (any_resid && !grid_sync(ctrl, G, gen, P.status)) return;

  // ---- decisions
  for (int i = (int)blockIdx.x; i < n; i += (int)G)
    hp_decide_item<DT>(sh, P.R, ws, i, nullptr, nullptr, nullptr, P.out_tokens, P.status, S,
                       reinterpret_cast<DT*>(dsm), nullptr);
}

template <typename DT>
cudaError_t launch_verify_redecide(const Shape& sh, const HpRows& R, const Ws& ws, int* out_tokens,
                                   uint32_t* status, int nsm, cudaStream_t st) {
  VrParams P;
  P.sh = sh;
  P.R = R;
  P.ws = ws;
  P.out_tokens = out_tokens;
  P.status = status;
  const size_t smem = (size_t)sh.r * VR_PIECE * CW * sizeof(DT);   // (>= the decisions' r x CW slab)
  auto kern = verify_redecide_kernel<DT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  int G = nsm < sh.NC ? nsm : sh.NC;
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

template cudaError_t launch_verify_redecide<float>(const Shape&, const HpRows&, const Ws&, int*, uint32_t*, int,
                                                   cudaStream_t);
template cudaError_t launch_verify_redecide<bf16>(const Shape&, const HpRows&, const Ws&, int*, uint32_t*, int,
                                                  cudaStream_t);

}  // namespace spec
