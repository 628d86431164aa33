// Slice-resident draft: DSpark's sequential stage with the Markov head
// ("[논문리뷰] DSpark ...", section 1.2: p_k(v | x_0, x_<k) = softmax(U_k + B_k),
// B(x_{k-1}, .) = W1[x_{k-1}] W2, sampled left to right), tempered by T_b, for
// batches of up to 128 requests whose vocabulary splits into at most 8
// chunks of 32 columns per SM (V <= 256 x SMs: the H-Spec review's pruned
// 32000-entry vocabulary fits).
//
// One cooperative launch walks the gamma steps.  CTA c owns the vocabulary
// columns [32 K c, 32 K (c+1)) for the whole launch (K chunks of 32):
//
//   * its W2 columns (r x 32K bf16, the MN-major operand of the MMA in 64-column
//     atoms with 128-byte swizzle) are loaded by TMA once and stay in shared
//     memory for every step;
//   * the U_k rows of its columns arrive by TMA in 32-column chunks (8 KB for
//     128 requests, 64-byte swizzle).  The first chunks of step k+1 are loaded
//     during step k's sampling phase (U does not depend on the drawn tokens),
//     the rest prefetched into L2 then and loaded into the A operand's space
//     once the step's MMAs have read it;
//   * per step: the rows W1[x_{k-1}] (the A operand, K-major, 128-byte
//     swizzle) arrive by TMA from the A-row buffer the samplers filled (the
//     first step and a redo gather them by cp.async), one thread issues the
//     tcgen05 MMAs (M = 128 requests, one MMA of N = 32K columns per 16-row
//     step of K = r) into a TMEM accumulator, and all eight warps read it back
//     (tcgen05.ld) as two column
//     groups, thread = request row, reducing each 32-column chunk to its
//     partial (c, m, s, q2) with the same arithmetic as the tile-strided draft
//     kernel.  The transition bias never leaves the SM;
//   * grid barrier, then the sampling phase (one CTA per request, the shared
//     sampler of spec_sample.cuh), grid barrier.
//
// Draws within the first pass's error band are queued over all steps and
// re-decided in extended precision after the last step (spec_hp.cuh's
// method), in batches of ws.max_items: every CTA computes the items'
// double-float weights of its own columns from its resident W2 columns, then
// one CTA per item finds the crossing chunk and scans it.  A re-decision that
// changes a token sends every step after the earliest change through a redo
// with its re-decisions in place.  Every wait is bounded; a CTA that gives up raises the abort word,
// waits for its own copies and MMAs in flight, frees its tensor memory and
// returns.
#include <cstring>

#include "spec_sample.cuh"
#include "spec_tmap.cuh"

namespace spec {

constexpr int SL_CHUNK_BYTES = TC_M * CW * 2;   // one U chunk: 128 rows x 32 bf16
constexpr int SL_MAX_K = 8;                       // chunks per CTA (<= 256 accumulator columns)
constexpr int SL_MIN_RING = 3;                    // chunks with their own buffers
constexpr uint32_t SL_TMEM_COLS = 256;

// Shared-memory plan (offsets from a 1 KB aligned base): the resident W2
// atoms, the A tile, then `nring` chunk buffers.  U chunks c >= nring use the
// A tile's space (after the MMAs).  W2 + A is at least the r x 256 slab of the
// extended-precision pass, which reuses that space after the last step.
struct SlLayout {
  int natoms, nring;
  size_t offW, offA, offU, total;
  __host__ __device__ SlLayout(int r, int K) {
    natoms = (K * CW + 63) / 64;
    const size_t w = (size_t)natoms * r * 128;
    const size_t a = (size_t)(r / 64) * 16384;
    const size_t slab = (size_t)r * HPB * 2;
    offW = 0;
    offA = w;
    size_t wa = w + a;
    if (wa < slab) wa = slab;
    offU = (wa + 1023) & ~(size_t)1023;
    const int aslots = (int)(a / SL_CHUNK_BYTES);
    nring = K - aslots;
    if (nring < SL_MIN_RING) nring = SL_MIN_RING;
    if (nring > K) nring = K;
    total = offU + (size_t)nring * SL_CHUNK_BYTES + 1024;
  }
  __host__ __device__ size_t u_off(int c) const {
    return c < nring ? offU + (size_t)c * SL_CHUNK_BYTES : offA + (size_t)(c - nring) * SL_CHUNK_BYTES;
  }
};

// Barrier slots: the W2 load, the gathered A tile, the accumulator (two slots,
// both committed after the step's MMAs: the first chunks' epilogue waits on
// one, the A tile's reuse for U chunks on the other), the A tile by TMA, the U
// chunks.  Each completes once per tile phase (W2 once per load).
enum : int { SB_W2 = 0, SB_AFULL = 1, SB_ACC0 = 2, SB_ACC1 = 3, SB_ATMA = 4, SB_U0 = 5,
             SB_COUNT = SB_U0 + SL_MAX_K };
// Bits of the "armed" word: async operations issued and not yet waited for.
enum : uint32_t { ARM_W2 = 1u << 8, ARM_MMA = 1u << 9, ARM_A = 1u << 10 };

// 16-byte piece j (0..3) of row m of a 64-byte-swizzled [128][32] bf16 chunk.
__device__ __forceinline__ const unsigned char* sl_upiece(const unsigned char* ub, int m, int j) {
  return ub + m * 64 + ((j ^ ((m >> 1) & 3)) << 4);
}

// Warp-uniform bounded wait (every lane gets the same answer).
__device__ __forceinline__ bool sl_wait(uint64_t* bar, uint32_t parity, volatile int* fail) {
  const bool ok = tp_wait(bar, parity, fail);
  return __all_sync(0xffffffffu, ok);
}

template <int HOOK>
__global__ void __launch_bounds__(NT, 1) draft_slice_kernel(const __grid_constant__ DraftParams P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ uint64_t s_bar[SB_COUNT];
  __shared__ uint32_t s_holder;
  __shared__ uint32_t s_armed;
  __shared__ int s_tok[TC_M];
  __shared__ int s_fail;
  const Shape& sh = P.sh;
  const bf16* U = (const bf16*)P.U;
  const bf16* W1 = (const bf16*)P.W1;
  const bf16* W2 = (const bf16*)P.W2;
  uint32_t* ctrl = P.ws.ctrl;
  unsigned char* smem = align1k(smem_raw);
  const int K = P.slK;
  const SlLayout lay(sh.r, K);
  const int c0 = (int)blockIdx.x * K;               // first chunk of this CTA's columns
  const int kc = max(0, min(K, sh.NC - c0));        // chunks it owns
  const int n0 = c0 * CW;
  const int N = K * CW;                             // accumulator columns (<= 256)
  const int nring = min(lay.nring, kc);
  const uint32_t G = gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* fail = &s_fail;
  const HpRows R{P.U, P.U, P.W1, P.W2, P.temp};

  if (threadIdx.x == 0) {
    mbar_init(s_bar + SB_W2, 1);
    mbar_init(s_bar + SB_AFULL, NT);
    mbar_init(s_bar + SB_ACC0, 1);
    mbar_init(s_bar + SB_ACC1, 1);
    mbar_init(s_bar + SB_ATMA, 1);
    for (int c = 0; c < SL_MAX_K; ++c) mbar_init(s_bar + SB_U0 + c, 1);
    s_fail = 0;
    s_armed = 0u;
    tma_prefetch_map(&P.maps.u);
    tma_prefetch_map(&P.maps.w2);
    tma_prefetch_map(&P.maps.a);
  }
  if (warp == 0) tc_alloc(&s_holder, SL_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_holder;

  uint32_t gen = 0u;        // grid barriers passed (thread 0)
  uint32_t gi = 0u;         // tile phases run: the parity of the per-phase barriers
  uint32_t nw2 = 0u;        // W2 loads issued
  uint32_t ngath = 0u;      // A tiles gathered by cp.async (phases of SB_AFULL)
  uint32_t natma = 0u;      // A tiles loaded by TMA from the A-row buffer (phases of SB_ATMA)
  bool redo_mode = false;   // steps after a changed re-decision: A rows gathered from the tokens
  bool w2_ok = false;       // the W2 columns are resident
  int ring_step = -1;       // step whose first chunks are loaded or in flight (not yet consumed)
  unsigned long long* tr = (P.ws.trace && blockIdx.x == 0 && threadIdx.x == 0) ? P.ws.trace : nullptr;

  // HOOK_STALL (a test build): the first barrier expects one arrival more
  // than the grid has, so it can only end by its time limit
  auto gsync = [&]() {
    return grid_sync(ctrl, G, gen, P.status, (HOOK == HOOK_STALL && gen == 0u) ? 1u : 0u);
  };
  // first chunks of step k into their buffers, the rest prefetched into L2
  // (all threads call; thread 0 issues)
  auto issue_ring = [&](int k) {
    if (threadIdx.x == 0) {
      uint32_t arm = 0u;
      for (int c = 0; c < nring; ++c) {
        mbar_expect_tx(s_bar + SB_U0 + c, (uint32_t)SL_CHUNK_BYTES);
        tma_load_3d(smem + lay.u_off(c), &P.maps.u, n0 + c * CW, k, 0, s_bar + SB_U0 + c);
        arm |= 1u << c;
      }
      for (int c = nring; c < kc; ++c) tma_prefetch_3d(&P.maps.u, n0 + c * CW, k, 0);
      atomicOr(&s_armed, arm);
    }
    ring_step = k;
  };
  auto token = [&](int k, int m) -> int {
    if (m >= sh.B) return -1;
    const int t = (k == 0) ? P.anchor[m] : __ldcg(P.tokens + (size_t)m * sh.gamma + k - 1);
    return min(max(t, 0), sh.V - 1);          // bad tokens are reported by the sampler
  };

  // ---- tile phase of step k: partials of this CTA's chunks for every request
  auto tile_phase = [&](int k) -> bool {
    // trace (CTA 0): A requested, A and W2 landed, first chunk of each epilogue
    // group done, each group done (rows 2 MAX_GAMMA - 8 + k, if free)
    unsigned long long* tx = (P.ws.trace && blockIdx.x == 0 && (threadIdx.x & 127u) == 0u &&
                              MAX_GAMMA + sh.gamma <= 2 * MAX_GAMMA - 8 && k < 7)
                                 ? P.ws.trace + (2 * MAX_GAMMA - 8 + k) * TRACE_SLOTS
                                 : nullptr;
    fence_async_shared();        // earlier generic use of the buffers precedes the async proxy's
    __syncthreads();
    if (kc > 0) {
      const bool load_w2 = !w2_ok;
      if (threadIdx.x == 0 && load_w2) {
        const uint32_t ab = (uint32_t)(sh.r * 128);
        mbar_expect_tx(s_bar + SB_W2, ab * (uint32_t)lay.natoms);
        for (int a = 0; a < lay.natoms; ++a)
          tma_load_2d(smem + lay.offW + (size_t)a * ab, &P.maps.w2, n0 + 64 * a, 0, s_bar + SB_W2);
        atomicOr(&s_armed, ARM_W2);
      }
      if (load_w2) {
        ++nw2;
        w2_ok = true;
      }
      if (ring_step != k) issue_ring(k);
      // A operand: rows W1[x_{k-1}].  After the first step the samplers have
      // copied them into the A-row buffer, loaded here by TMA (4 boxes of 64
      // columns); the first step and the redo gather them by cp.async.
      const bool by_tma = k > 0 && !redo_mode;
      uint64_t* abar = by_tma ? s_bar + SB_ATMA : s_bar + SB_AFULL;
      const uint32_t apar = by_tma ? (natma & 1u) : (ngath & 1u);
      if (by_tma) {
        if (threadIdx.x == 0) {
          // the rows were written by other CTAs (generic proxy) before the grid barrier
          asm volatile("fence.proxy.async.global;\n" ::: "memory");
          mbar_expect_tx(abar, (uint32_t)(sh.r / 64) * 16384u);
          for (int a = 0; a < sh.r / 64; ++a)
            tma_load_2d(smem + lay.offA + (size_t)a * 16384, &P.maps.a, 64 * a, 0, abar);
          atomicOr(&s_armed, ARM_A);
        }
        ++natma;
      } else {
        for (int m = threadIdx.x; m < TC_M; m += NT) s_tok[m] = token(k, m);
        __syncthreads();
        if (tr) tr[k * TRACE_SLOTS + 6] = globaltimer_ns();
        tp_gather_a(smem + lay.offA, W1, s_tok, sh.r, (int)threadIdx.x, NT);
        if (tr) tr[k * TRACE_SLOTS + 7] = globaltimer_ns();
        fence_async_shared();
        mbar_arrive(abar);
        ++ngath;
      }
      const uint32_t par = gi & 1u;
      if (threadIdx.x == 0) {
        if (tx) tx[0] = globaltimer_ns();
        if (tp_wait(abar, apar, fail) && tp_wait(s_bar + SB_W2, (nw2 - 1u) & 1u, fail)) {
          if (tx) tx[1] = globaltimer_ns();
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + lay.offA), w0 = smem_u32(smem + lay.offW);
          const uint32_t ab = (uint32_t)(sh.r * 128);      // bytes of one 64-column W2 atom
          // one MMA of N = K x 32 columns per 16-row step of r (the A tile
          // is read once per step; the W2 atoms are LBO apart); both
          // accumulator barriers complete with it
          for (int kk = 0; kk < sh.r; kk += 16) {
            const uint64_t ad = tc_sdesc(a0 + (uint32_t)((kk >> 6) * 16384 + (kk & 63) * 2), 16, 1024);
            const uint64_t bd = tc_sdesc(w0 + (uint32_t)(kk * 128), ab, 1024);
            tc_mma(tmem, ad, bd, tc_idesc_n(N), kk > 0 ? 1u : 0u);
          }
          tc_commit(s_bar + SB_ACC0);
          tc_commit(s_bar + SB_ACC1);
          atomicOr(&s_armed, ARM_MMA);
        }
      }
      if (tr) tr[k * TRACE_SLOTS + 1] = globaltimer_ns();
      // epilogue: group grp takes chunks grp, grp + 2, ...; thread = request row
      const int grp = warp >> 2, q = warp & 3;
      const int m = 32 * q + lane;
      const bool rowok = m < sh.B;
      const float invT = rowok ? 1.0f / P.temp[m] : 1.0f;
      const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
      for (int c = grp; c < kc; c += 2) {
        if (c == nring && warp == 4 * grp) {
          // the A tile is read until the MMAs complete; then the step's
          // remaining chunks go into its space
          bool ok = sl_wait(s_bar + SB_ACC1, par, fail);
          if (ok && lane == 0) {
            uint32_t arm = 0u;
            for (int cc = nring; cc < kc; ++cc) {
              mbar_expect_tx(s_bar + SB_U0 + cc, (uint32_t)SL_CHUNK_BYTES);
              tma_load_3d(smem + lay.u_off(cc), &P.maps.u, n0 + cc * CW, k, 0, s_bar + SB_U0 + cc);
              arm |= 1u << cc;
            }
            atomicOr(&s_armed, arm);
          }
          __syncwarp();
          if (!ok) break;
        }
        if (!sl_wait(s_bar + (c < 4 ? SB_ACC0 : SB_ACC1), par, fail)) break;
        if (!sl_wait(s_bar + SB_U0 + c, par, fail)) break;
        tc_fence_after();
        float x[32];
        tc_ld32_issue(trow + (uint32_t)(32 * c), x);
        uint4 u[4];
        const unsigned char* ub = smem + lay.u_off(c);
#pragma unroll
        for (int j = 0; j < 4; ++j) u[j] = lds128(sl_upiece(ub, m, j));
        tc_wait_ld();
        const int nv = min(CW, sh.V - (n0 + c * CW));
        const float4 pv = nv >= CW ? chunk_partial<true>(u, x, CW, invT) : chunk_partial<false>(u, x, nv, invT);
        if (rowok) P.ws.dpart[(size_t)m * sh.NC + c0 + c] = pv;
        if (tx && threadIdx.x == 128u * grp && c == grp) tx[2 + grp] = globaltimer_ns();
      }
      if (tx && threadIdx.x == 128u * grp) tx[4 + grp] = globaltimer_ns();
    }
    tc_fence_before();
    __syncthreads();
    ring_step = -1;                              // this step's chunks are consumed
    if (*fail != 0) {
      // gi is left at this phase: the drain waits for its completions
      if (threadIdx.x == 0) set_status(P.status, SPEC_DEV_TIMEOUT);
      return false;
    }
    if (threadIdx.x == 0) s_armed = 0u;          // everything issued in this phase was waited for
    ++gi;
    return true;
  };

  // ---- sampling phase of step k (one CTA per request); first loads of step k+1
  auto sampling_phase = [&](int k) {
    fence_async_shared();
    __syncthreads();
    if (k + 1 < sh.gamma && kc > 0) issue_ring(k + 1);
    for (int b = blockIdx.x; b < sh.B; b += G)
      draft_sample_body<bf16, HOOK>(sh, k, b, U, W1, W2, P.anchor, P.temp, P.u_draft, P.tokens,
                                    P.q_tok, P.lse_q, P.diag, P.status, P.ws, P.eps,
                                    ctrl + CTRL_DITEMS, P.ws.item_cap, smem + lay.offA,
                                    (P.ws.trace && blockIdx.x == 0 && b == 0)
                                        ? P.ws.trace + (MAX_GAMMA + k) * TRACE_SLOTS : nullptr,
                                    redo_mode ? nullptr : reinterpret_cast<bf16*>(P.ws.abuf));
  };

  // ---- re-decision of the queued draws, ws.max_items at a time, on the
  // slice layout: each CTA computes the items' extended-precision weights of
  // its own columns from the W2 columns already in its shared memory (the
  // compensated dot products of spec_hp.cuh's method) and writes their
  // 32-column chunk sums; after a grid barrier one CTA per item finds the
  // crossing chunk, recomputes its 32 weights and scans them
  // (hp_decide_item).  W2 stays resident.
  __shared__ HpShared S_hp;
  auto redecide = [&](uint32_t* redo) -> bool {
    const int n = min((int)__ldcg(ctrl + CTRL_DITEMS), P.ws.item_cap);
    if (n == 0) return true;
    constexpr int SUB = 8;                                  // items whose rows are staged together
    // scratch in the A tile's space (free after a tile phase; at least r x 256
    // bytes): item records (<= 128 x 40 bytes), SUB factor rows, SUB contexts
    unsigned char* scratch = smem + lay.offA;
    HpItem* s_items = reinterpret_cast<HpItem*>(scratch);
    float* arows = reinterpret_cast<float*>(scratch + 8192);
    ItemCtx<bf16>* ictx = reinterpret_cast<ItemCtx<bf16>*>(scratch + 8192 + (size_t)SUB * sh.r * 4);
    hp_table(S_hp.tab);
    for (int base = 0; base < n; base += P.ws.max_items) {
      Ws wb = P.ws;
      wb.items = P.ws.items + base;
      const int nb = min(P.ws.max_items, n - base);
      if (kc > 0) {
        const int col = (int)threadIdx.x;        // this thread's column of the range
        const int v = n0 + col;
        const bool mine = col < kc * CW && v < sh.V;
        const int a = col >> 6, cc = col & 63;
        const unsigned char* wcol = smem + lay.offW + (size_t)a * sh.r * 128 + (cc & 7) * 2;
        __syncthreads();                         // the scratch space is free
        for (int i = threadIdx.x; i < nb; i += NT) s_items[i] = ldcg_item(wb.items + i);
        __syncthreads();
        for (int i0 = 0; i0 < nb; i0 += SUB) {
          const int cnt = min(SUB, nb - i0);
          // every item's factor row, context and this thread's logit, all loads at once
          for (int q = threadIdx.x; q < cnt * sh.r; q += NT) {
            const int i = q / sh.r, e = q - i * sh.r;
            arows[i * sh.r + e] = ldf(W1 + (size_t)s_items[i0 + i].prev * sh.r + e);
          }
          if ((int)threadIdx.x < cnt) ictx[threadIdx.x] = item_ctx<bf16>(sh, R, s_items[i0 + threadIdx.x]);
          float uq[SUB];
#pragma unroll
          for (int i = 0; i < SUB; ++i) {
            uq[i] = 0.f;
            if (i < cnt && mine) {
              const HpItem& it = s_items[i0 + i];
              uq[i] = ldf(U + ((size_t)it.b * sh.gamma + it.j) * sh.V + v);
            }
          }
          __syncthreads();
          if (tr && i0 == 0) tr[(2 * MAX_GAMMA - 1) * TRACE_SLOTS + 5] = globaltimer_ns();
#pragma unroll 1
          for (int i = 0; i < cnt; ++i) {
            df wq = {0.f, 0.f};
            if (mine) {
              const float* ar = arows + i * sh.r;
              DdSum k0, k1;
              for (int q0 = 0; q0 < sh.r; q0 += 8) {
                const unsigned char* rb = wcol + (size_t)q0 * 128;
#pragma unroll
                for (int j = 0; j < 8; j += 2) {
                  // row q0 + j of the swizzled atom: 16-byte chunk (cc / 8) ^ j
                  const float w0 = __bfloat162float(
                      *reinterpret_cast<const bf16*>(rb + j * 128 + (((cc >> 3) ^ j) << 4)));
                  const float w1 = __bfloat162float(
                      *reinterpret_cast<const bf16*>(rb + (j + 1) * 128 + (((cc >> 3) ^ (j + 1)) << 4)));
                  k0.add(__fmul_rn(ar[q0 + j], w0));   // bf16 x bf16 products are exact in fp32
                  k1.add(__fmul_rn(ar[q0 + j + 1], w1));
                }
              }
              wq = hp_wq_val<bf16>(ictx[i], dd_add(k0.value(), k1.value()), uq[i], S_hp.tab);
              // the first items keep their weights for the decision
              if (i0 + i < wb.hpw_items) wb.hpw[(size_t)(i0 + i) * sh.V + v] = make_float4(wq.hi, wq.lo, 0.f, 0.f);
            }
            const df csum = warp_sum_df(wq);
            if (lane == 0 && warp < kc)
              item_sums(wb, sh, i0 + i, 0)[c0 + warp] = make_float2(csum.hi, csum.lo);
          }
          if (tr && i0 == 0) tr[(2 * MAX_GAMMA - 1) * TRACE_SLOTS + 6] = globaltimer_ns();
          __syncthreads();                       // the staged rows are consumed
        }
      }
      if (tr) tr[(2 * MAX_GAMMA - 1) * TRACE_SLOTS + 1] = globaltimer_ns();
      if (!gsync()) return false;
      if (tr) tr[(2 * MAX_GAMMA - 1) * TRACE_SLOTS + 2] = globaltimer_ns();
      for (int i = (int)blockIdx.x; i < nb; i += (int)G)
        hp_decide_item<bf16>(sh, R, wb, i, P.tokens, P.q_tok, P.lse_q, nullptr, P.status, S_hp,
                             reinterpret_cast<bf16*>(smem + lay.offA), redo,
                             (P.ws.trace && i == 0 && MAX_GAMMA + sh.gamma <= 2 * MAX_GAMMA - 9)
                                 ? P.ws.trace + (2 * MAX_GAMMA - 9) * TRACE_SLOTS
                                 : nullptr);
      if (tr) tr[(2 * MAX_GAMMA - 1) * TRACE_SLOTS + 3] = globaltimer_ns();
      if (!gsync()) return false;
    }
    return true;
  };

  auto run_step = [&](int k) -> bool {
    if (tr) tr[k * TRACE_SLOTS + 0] = globaltimer_ns();
    if (!tile_phase(k)) return false;
    if (tr) tr[k * TRACE_SLOTS + 2] = globaltimer_ns();
    if (!gsync()) return false;
    if (tr) tr[k * TRACE_SLOTS + 3] = globaltimer_ns();
    sampling_phase(k);
    if (tr) tr[k * TRACE_SLOTS + 4] = globaltimer_ns();
    if (!gsync()) return false;
    if (tr) tr[k * TRACE_SLOTS + 5] = globaltimer_ns();
    return true;
  };

  if (kc > 0) issue_ring(0);
  bool good = true;
  for (int k = 0; k < sh.gamma && good; ++k) good = run_step(k);
  if (tr) tr[(2 * MAX_GAMMA - 1) * TRACE_SLOTS] = globaltimer_ns();
  if (good) good = redecide(ctrl + CTRL_REDO);
  if (tr) tr[(2 * MAX_GAMMA - 1) * TRACE_SLOTS + 4] = globaltimer_ns();
  if (good) {
    const uint32_t redo = __ldcg(ctrl + CTRL_REDO);
    const int k0 = sh.gamma - (int)redo + 1;            // first step to redo
    if (redo > 0 && k0 < sh.gamma) {
      redo_mode = true;
      for (int k = k0; k < sh.gamma && good; ++k) {
        if (blockIdx.x == 0 && threadIdx.x == 0) ctrl[CTRL_DITEMS] = 0u;
        good = run_step(k) && redecide(nullptr);
      }
    }
  }
  if (!good) {
    // leave: wait for this CTA's own copies and MMAs in flight (bounded)
    if (threadIdx.x == 0) atomicExch(ctrl + CTRL_ABORT, 1u);
    __syncthreads();
    if (threadIdx.x == 0) {
      const uint32_t a = s_armed;
      for (int c = 0; c < SL_MAX_K; ++c)
        if (a & (1u << c)) mbar_wait(s_bar + SB_U0 + c, gi & 1u, 1u << 20);
      if (a & ARM_W2) mbar_wait(s_bar + SB_W2, (nw2 - 1u) & 1u, 1u << 20);
      if (a & ARM_A) mbar_wait(s_bar + SB_ATMA, (natma - 1u) & 1u, 1u << 20);
      if (a & ARM_MMA) mbar_wait(s_bar + SB_ACC1, gi & 1u, 1u << 20);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tc_dealloc(tmem, SL_TMEM_COLS);
}

// ---------------------------------------------------------------- launcher
// Chunks per CTA when the slice-resident kernel applies to this shape on
// `nsm` SMs, else 0.
int slice_chunks(const Shape& sh, int nsm) {
  if (sh.rnn || sh.B > TC_M || sh.r % 64 != 0 || sh.r > 256 || nsm < 1) return 0;
  const int K = (sh.NC + nsm - 1) / nsm;
  if (K < 1 || K > SL_MAX_K) return 0;
  return K;
}

template <int HOOK>
static cudaError_t launch_slice(const DraftParams& P, int G, cudaStream_t st) {
  const SlLayout lay(P.sh.r, P.slK);
  const size_t smem = lay.total;
  auto kern = draft_slice_kernel<HOOK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cudaErrorNotSupported;
  }
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, smem);
  if (e != cudaSuccess || per_sm < 1) {
    cudaGetLastError();
    return cudaErrorNotSupported;
  }
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

// The whole draft in one cooperative launch of the slice-resident kernel (the
// control words must be zeroed).  cudaErrorNotSupported when the shape does
// not fit it (the caller then uses the tile-strided kernel).
cudaError_t launch_draft_slice(const Shape& sh, const void* U, const void* W1, const void* W2,
                               const int* anchor, const float* temp, const float* u_draft, int* tokens,
                               float* q_tok, double* lse_q, float* diag, uint32_t* status, const Ws& ws,
                               const Eps& eps, int nsm, cudaStream_t st, int hook) {
  const int K = slice_chunks(sh, nsm);
  if (K == 0) return cudaErrorNotSupported;
  DraftParams P;
  memset(&P, 0, sizeof(P));
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
  P.slK = K;
  cudaError_t e = encode_u_chunk_map(sh, U, &P.maps.u);
  if (e == cudaSuccess) e = encode_w2_map(sh, W2, &P.maps.w2);
  if (e == cudaSuccess) e = encode_abuf_map(sh.B, sh.r, ws.abuf, &P.maps.a);
  if (e != cudaSuccess) return e;
  const int tiles = (sh.NC + K - 1) / K;       // CTAs with columns
  int G = tiles > sh.B ? tiles : (sh.B < nsm ? sh.B : nsm);
  if (G > nsm) G = nsm;
  if (G < tiles) return cudaErrorNotSupported;
  if (hook == HOOK_PERTURB) return launch_slice<HOOK_PERTURB>(P, G, st);
  if (hook == HOOK_STALL) return launch_slice<HOOK_STALL>(P, G, st);
  return launch_slice<HOOK_NONE>(P, G, st);
}

}  // namespace spec
