// Slice-resident verification tiles: the alpha / residual sweep of the
// lossless acceptance step ("Speculative Decoding Part 1", VESSL AI blog,
// section "수락 규칙": alpha_j = sum_v min(p_j, q_j), residual max(0, p - q))
// for every packed draft row p = (b, j < L_b), with the draft distribution
// q_j rebuilt from U and the Markov bias W1[x_j] W2 (DSpark review, section
// 1.2), for shapes whose vocabulary splits into at most 8 chunks of 32
// columns per SM.
//
// CTA c owns the vocabulary columns [32 K c, 32 K (c+1)) (K chunks of 32, the
// same split as the slice-resident draft); its W2 columns (r x 32K bf16, the
// MN-major MMA operand, 64-column atoms with 128-byte swizzle) are loaded by
// TMA once and stay in shared memory.  It walks the packed rows in tiles of
// 128 (the count is read on the device):
//
//   warp 8       control: gathers the tile's rows W1[x_j] (or the RNN head's
//                factor rows) into the A operand (cp.async, K-major, 128-byte
//                swizzle) once the previous tile's MMAs have read it, then one
//                lane issues the MMAs (M = 128 rows, N = 32K in one group,
//                K = r) into one of two 256-column TMEM accumulators;
//   warps 0-7    epilogue, two column groups of four warps, thread = packed
//                row = TMEM lane: each 32-column chunk's bias from TMEM
//                (tcgen05.ld), the row's U and target values straight from
//                global memory (one chunk ahead), and the chunk's partial
//                (sum min(p, q), sum max(0, p - q), sum p^2, sum q^2) with the
//                arithmetic of the tile-strided kernel (spec_verify.cu), so the
//                final draw's recompute and error band stay consistent.
//
// The next tile's gather and MMAs overlap the current tile's epilogue.  Every
// wait is bounded; a wait that gives up sets SPEC_DEV_TIMEOUT and the kernel
// drains its own copies and MMAs before it frees its tensor memory.
#include <cstring>

#include "spec_tile_tc.cuh"
#include "spec_tmap.cuh"

namespace spec {

constexpr int VS_THREADS = 288;                  // 8 epilogue warps + 1 control warp
constexpr int VS_MAX_K = 8;
constexpr uint32_t VS_TMEM_COLS = 512;           // two accumulators of up to 256 columns

enum : int { VB_W2 = 0, VB_AFULL = 1, VB_AFREE = 2, VB_FULL0 = 3, VB_EMPTY0 = 5, VB_COUNT = 7 };

struct VsLayout {
  int natoms;
  size_t offW, offA, total;
  __host__ __device__ VsLayout(int r, int K) {
    natoms = (K * CW + 63) / 64;
    offW = 0;
    offA = (size_t)natoms * r * 128;
    total = offA + (size_t)(r / 64) * 16384 + 1024;
  }
};

struct VsParams {
  CUtensorMap w2;     // W2 as [r][V], box 64 x r, 128-byte swizzle
  Shape sh;
  const bf16* target;
  const bf16* U;
  const bf16* F;      // factor rows: W1 (Markov head) or the RNN head's a rows
  Ws ws;
  uint32_t* status;
  int K;              // chunks of CW columns per CTA
};

// The same first-pass expressions as the tile-strided verification epilogue.
constexpr float VS_LOG2E = 1.44269504f;
__device__ __forceinline__ float vs_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ df vs_fast_two_sum(float a, float b) {
  float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ df vs_mul_f_df(float c, df t) {
  float p = __fmul_rn(c, t.hi);
  float e = fmaf(c, t.hi, -p);
  e = fmaf(c, t.lo, e);
  return vs_fast_two_sum(p, e);
}
__device__ __forceinline__ float vs_norm_factor(float c, df invT, df nlse) {
  const df g = df_add(vs_mul_f_df(c, invT), nlse);
  return __fmul_rn(expf(g.hi), __fadd_rn(1.0f, g.lo));
}

// Named barrier over `n` threads that returns the OR of `v` over them, so
// every participant takes the same decision.
__device__ __forceinline__ bool named_bar_or(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Warp-uniform bounded wait.
__device__ __forceinline__ bool vs_wait(uint64_t* bar, uint32_t parity, volatile int* fail) {
  const bool ok = tp_wait(bar, parity, fail);
  return __all_sync(0xffffffffu, ok);
}

// 32 bf16 values (64 bytes) of a row from column v0; 16-byte pieces at or
// beyond V (V % 8 == 0) read as zeros.
__device__ __forceinline__ void vs_load_chunk(const bf16* row, int v0, int V, uint4 (&d)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    d[j] = (row && v0 + 8 * j < V) ? __ldg(reinterpret_cast<const uint4*>(row + v0 + 8 * j))
                                   : make_uint4(0u, 0u, 0u, 0u);
}

__global__ void __launch_bounds__(VS_THREADS, 1) verify_slice_kernel(const __grid_constant__ VsParams P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ uint64_t s_bar[VB_COUNT];
  __shared__ uint32_t s_holder;
  __shared__ int s_tok[2 * TC_M];                 // A rows' tokens of the current and next tile
  __shared__ int s_fail;
  const Shape& sh = P.sh;
  const Ws& ws = P.ws;
  unsigned char* smem = align1k(smem_raw);
  const int K = P.K;
  const VsLayout lay(sh.r, K);
  const int c0 = (int)blockIdx.x * K;
  const int kc = max(0, min(K, sh.NC - c0));
  const int n0 = c0 * CW;
  const int N = K * CW;                           // accumulator columns (<= 256)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* fail = &s_fail;
  const int Pk = (int)__ldcg(ws.ctrl + CTRL_NPACKED);
  const int ntiles = (Pk + TC_M - 1) / TC_M;
  // profiling stamps (SPEC_OPT_TRACE) of CTA 0, tiles < 8: control lane 0
  // [0] gather start, [1] A tile complete, [2] MMAs issued; epilogue thread 0
  // [3] accumulator ready, [4] tile done
  unsigned long long* vtr = (ws.trace && blockIdx.x == 0) ? ws.trace + 8 * TRACE_SLOTS : nullptr;

  if (threadIdx.x == 0) {
    mbar_init(s_bar + VB_W2, 1);
    mbar_init(s_bar + VB_AFULL, 256);
    mbar_init(s_bar + VB_AFREE, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_bar + VB_FULL0 + i, 1);
      mbar_init(s_bar + VB_EMPTY0 + i, 256);
    }
    s_fail = 0;
  }
  if (warp == 0) tc_alloc(&s_holder, VS_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_holder;

  if (kc > 0 && ntiles > 0) {
    if (warp == 8) {
      // ---------------------------------------------------------- control warp: MMAs
      const uint32_t ab = (uint32_t)(sh.r * 128);
      if (lane == 0) {
        tma_prefetch_map(&P.w2);
        mbar_expect_tx(s_bar + VB_W2, ab * (uint32_t)lay.natoms);
        for (int a = 0; a < lay.natoms; ++a)
          tma_load_2d(smem + lay.offW + (size_t)a * ab, &P.w2, n0 + 64 * a, 0, s_bar + VB_W2);
        int issued = 0;          // tiles whose MMAs were issued
        bool ok = tp_wait(s_bar + VB_W2, 0u, fail);
        const bool w2_seen = ok;
        for (int mt = 0; mt < ntiles && ok; ++mt) {
          const int buf = mt & 1;
          if (vtr && mt < 8) vtr[mt * TRACE_SLOTS + 0] = globaltimer_ns();
          ok = tp_wait(s_bar + VB_AFULL, (uint32_t)mt & 1u, fail);
          if (vtr && mt < 8) vtr[mt * TRACE_SLOTS + 1] = globaltimer_ns();
          if (ok && mt >= 2) ok = tp_wait(s_bar + VB_EMPTY0 + buf, (uint32_t)((mt >> 1) - 1) & 1u, fail);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + lay.offA), w0 = smem_u32(smem + lay.offW);
          const uint32_t d = tmem + (uint32_t)(buf * 256);
          // one MMA of N = K x 32 columns per 16-row step of r (the A tile is
          // read once per step; the W2 atoms are LBO apart)
          for (int kk = 0; kk < sh.r; kk += 16) {
            const uint64_t ad = tc_sdesc(a0 + (uint32_t)((kk >> 6) * 16384 + (kk & 63) * 2), 16, 1024);
            tc_mma(d, ad, tc_sdesc(w0 + (uint32_t)(kk * 128), ab, 1024), tc_idesc_n(N), kk > 0 ? 1u : 0u);
          }
          tc_commit(s_bar + VB_FULL0 + buf);
          issued = mt + 1;
          if (vtr && mt < 8) vtr[mt * TRACE_SLOTS + 2] = globaltimer_ns();
        }
        if (*fail) {
          // drain: the W2 copy and the last issued MMAs
          if (!w2_seen) mbar_wait(s_bar + VB_W2, 0u, 1u << 20);
          if (issued > 0) mbar_wait(s_bar + VB_FULL0 + ((issued - 1) & 1), (uint32_t)((issued - 1) >> 1) & 1u, 1u << 20);
        }
      }
      __syncwarp();
    } else {
      // ---------------------------------------------------------- epilogue warps
      // They also gather the A operand: tile mt + 1's rows are copied once tile
      // mt's MMAs are complete (its accumulator is ready), overlapping tile
      // mt's epilogue; the copies are waited for after the first chunk.
      const int tid = (int)threadIdx.x;                 // 0..255
      // Tile-local row i sits in TMEM lane (i % 4) * 32 + i / 4, so the rows of a
      // partial tile are spread evenly over the four lane quadrants (the warps
      // of the four sub-partitions).
      auto row_of_lane = [&](int mt, int m) -> int { return mt * TC_M + (m & 31) * 4 + (m >> 5); };
      auto token = [&](int mt, int m) -> int {
        const int p = row_of_lane(mt, m);
        return p < Pk ? min(max(__ldcg(ws.prevtok + p), 0), sh.NA - 1) : -1;
      };
      auto gather = [&](const int* tok) {
        const int lg = __ffs(sh.r / 8) - 1, cmask = sh.r / 8 - 1;
        unsigned char* As = smem + lay.offA;
        for (int c = tid; c < TC_M * (sh.r / 8); c += 256) {
          const int m = c >> lg, j = c & cmask;
          const int t = tok[m];
          const bool valid = t >= 0;
          cp_async16(As + (size_t)(j >> 3) * 16384 + m * 128 + (((j & 7) ^ (m & 7)) << 4),
                     valid ? P.F + (size_t)t * sh.r + j * 8 : P.F, valid);
        }
        cp_async_commit();
      };
      auto gather_done = [&]() {
        cp_async_wait_all();
        fence_async_shared();            // the rows are visible to the MMA's async proxy
        mbar_arrive(s_bar + VB_AFULL);
      };
      // L2 prefetch of a tile's row slices [n0, n0 + kc CW) of U (threads
      // 0..127) and of the target (128..255): one bulk prefetch per row and
      // tensor, a tile ahead of the epilogue's register loads
      const uint32_t pf_bytes = (uint32_t)(min(kc * CW, sh.V - n0) * (int)sizeof(bf16));
      auto pf_row = [&](int mt2) -> int2 {
        const int p = mt2 * TC_M + (tid & (TC_M - 1));
        return (mt2 < ntiles && p < Pk) ? __ldcg(ws.prow + p) : make_int2(-1, -1);
      };
      auto pf_issue = [&](int2 bj) {
        if (bj.x < 0) return;
        const bf16* row = tid < TC_M ? P.U + ((size_t)bj.x * sh.gamma + bj.y) * sh.V
                                     : P.target + ((size_t)bj.x * (sh.gamma + 1) + bj.y) * sh.V;
        bulk_prefetch_l2(row + n0, pf_bytes);
      };
      pf_issue(pf_row(0));
      int2 pf_next = pf_row(1);
      if (tid < TC_M) s_tok[tid] = token(0, tid);
      named_bar(1, 256);
      gather(s_tok);
      gather_done();
      const int grp = warp >> 2, q = warp & 3;
      const int m = 32 * q + lane;
      const uint32_t lanebase = tmem + ((uint32_t)(32 * q) << 16);
      for (int mt = 0; mt < ntiles; ++mt) {
        const int buf = mt & 1;
        const bool more = mt + 1 < ntiles;
        int* tok_next = s_tok + ((mt + 1) & 1) * TC_M;
        if (more && tid < TC_M) tok_next[tid] = token(mt + 1, tid);
        const int p = row_of_lane(mt, m);
        const bool rowok = p < Pk;
        float4 rc = make_float4(1.f, 0.f, 0.f, 0.f);
        float2 rp = make_float2(0.f, 0.f);
        const bf16* urow = nullptr;
        const bf16* trow = nullptr;
        if (rowok) {
          const int2 bj = ws.prow[p];
          rc = ws.rowc[p];
          rp = ws.rowp[(size_t)bj.x * (sh.gamma + 1) + bj.y];
          urow = P.U + ((size_t)bj.x * sh.gamma + bj.y) * sh.V;
          trow = P.target + ((size_t)bj.x * (sh.gamma + 1) + bj.y) * sh.V;
        }
        const float s2 = __fmul_rn(rc.x, VS_LOG2E);
        uint4 ua[4], ta[4];
        int c = grp;
        if (c < kc) {
          vs_load_chunk(urow, n0 + c * CW, sh.V, ua);
          vs_load_chunk(trow, n0 + c * CW, sh.V, ta);
        }
        const bool okw = vs_wait(s_bar + VB_FULL0 + buf, (uint32_t)(mt >> 1) & 1u, fail);
        // every epilogue thread is past tile mt's MMAs (the A tile is free), or
        // all of them stop together
        if (named_bar_or(1, 256, !okw || *fail != 0)) break;
        if (vtr && threadIdx.x == 0 && mt < 8) vtr[mt * TRACE_SLOTS + 3] = globaltimer_ns();
        tc_fence_after();
        if (more) gather(tok_next);
        pf_issue(pf_next);
        pf_next = pf_row(mt + 2);
        bool pending = more;
        if (!__any_sync(0xffffffffu, rowok)) c = kc;   // a warp without rows skips the chunks
        for (; c < kc; c += 2) {
          const int v0 = n0 + c * CW;
          uint4 un[4], tn[4];
          if (c + 2 < kc) {                      // the next chunk's values, in flight meanwhile
            vs_load_chunk(urow, v0 + 2 * CW, sh.V, un);
            vs_load_chunk(trow, v0 + 2 * CW, sh.V, tn);
          }
          float bias[32];
          tc_ld32_issue(lanebase + (uint32_t)(buf * 256 + 32 * c), bias);
          const int nval = rowok ? min(CW, sh.V - v0) : 0;
          // chunk references: the largest U and target of the valid columns
          float cU = -INFINITY, cT = -INFINITY;
          if (nval == CW) {
            __nv_bfloat162 mu = __float2bfloat162_rn(-INFINITY), mtt = mu;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const uint32_t wa[4] = {ua[g].x, ua[g].y, ua[g].z, ua[g].w};
              const uint32_t wt[4] = {ta[g].x, ta[g].y, ta[g].z, ta[g].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                mu = __hmax2(mu, *reinterpret_cast<const __nv_bfloat162*>(&wa[e]));
                mtt = __hmax2(mtt, *reinterpret_cast<const __nv_bfloat162*>(&wt[e]));
              }
            }
            cU = fmaxf(__low2float(mu), __high2float(mu));
            cT = fmaxf(__low2float(mtt), __high2float(mtt));
          } else {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const uint32_t wa[4] = {ua[g].x, ua[g].y, ua[g].z, ua[g].w};
              const uint32_t wt[4] = {ta[g].x, ta[g].y, ta[g].z, ta[g].w};
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (8 * g + e < nval) {
                  cU = fmaxf(cU, (e & 1) ? bf_hi(wa[e >> 1]) : bf_lo(wa[e >> 1]));
                  cT = fmaxf(cT, (e & 1) ? bf_hi(wt[e >> 1]) : bf_lo(wt[e >> 1]));
                }
            }
          }
          const float Fq = vs_norm_factor(cU, {rc.x, rc.y}, {rc.z, rc.w});
          const float Fp = vs_norm_factor(cT, {rc.x, rc.y}, {rp.x, rp.y});
          float al[2] = {0.f, 0.f}, p2[2] = {0.f, 0.f}, q2[2] = {0.f, 0.f};
          Kahan kr[2];
          tc_wait_ld();
          // the element terms (with the tile-strided kernel's rounding steps)
          auto term = [&](float uv, float tv, float bv, int e) {
            const float qv = __fmul_rn(vs_ex2(__fmul_rn(__fadd_rn(__fsub_rn(uv, cU), bv), s2)), Fq);
            const float pv = __fmul_rn(vs_ex2(__fmul_rn(__fsub_rn(tv, cT), s2)), Fp);
            al[e & 1] += fminf(pv, qv);
            kr[e & 1].add(fmaxf(0.f, __fsub_rn(pv, qv)));
            p2[e & 1] = fmaf(pv, pv, p2[e & 1]);
            q2[e & 1] = fmaf(qv, qv, q2[e & 1]);
          };
          if (nval == CW) {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const uint32_t wa[4] = {ua[g].x, ua[g].y, ua[g].z, ua[g].w};
              const uint32_t wt[4] = {ta[g].x, ta[g].y, ta[g].z, ta[g].w};
#pragma unroll
              for (int e = 0; e < 8; ++e)
                term((e & 1) ? bf_hi(wa[e >> 1]) : bf_lo(wa[e >> 1]),
                     (e & 1) ? bf_hi(wt[e >> 1]) : bf_lo(wt[e >> 1]), bias[8 * g + e], e);
            }
          } else {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const uint32_t wa[4] = {ua[g].x, ua[g].y, ua[g].z, ua[g].w};
              const uint32_t wt[4] = {ta[g].x, ta[g].y, ta[g].z, ta[g].w};
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (8 * g + e < nval)
                  term((e & 1) ? bf_hi(wa[e >> 1]) : bf_lo(wa[e >> 1]),
                       (e & 1) ? bf_hi(wt[e >> 1]) : bf_lo(wt[e >> 1]), bias[8 * g + e], e);
            }
          }
          if (nval > 0)
            ws.vpart[(size_t)p * sh.NSV + (v0 / VB)] =
                make_float4(al[0] + al[1], df_d(df_add(kr[0].value(), kr[1].value())), p2[0] + p2[1],
                            q2[0] + q2[1]);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            ua[j] = un[j];
            ta[j] = tn[j];
          }
          if (pending) {                         // the next tile's rows, after one chunk
            gather_done();
            pending = false;
          }
        }
        if (pending) gather_done();
        tc_fence_before();
        mbar_arrive(s_bar + VB_EMPTY0 + buf);
        if (vtr && threadIdx.x == 0 && mt < 8) vtr[mt * TRACE_SLOTS + 4] = globaltimer_ns();
      }
      cp_async_wait_all();                       // no copy of this thread is left in flight
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*fail && threadIdx.x == 0) set_status(P.status, SPEC_DEV_TIMEOUT);
  if (warp == 0) tc_dealloc(tmem, VS_TMEM_COLS);
}

// Chunks per CTA when the slice-resident verification applies, else 0.
int vslice_chunks(const Shape& sh, int nsm) {
  if (sh.r % 64 != 0 || sh.r > 256 || nsm < 1) return 0;
  const int K = (sh.NC + nsm - 1) / nsm;
  return (K >= 1 && K <= VS_MAX_K) ? K : 0;
}

// The verification tiles on the slice-resident kernel (cudaErrorNotSupported
// when the shape does not fit it).  F: W1 or the RNN head's factor rows.
cudaError_t launch_verify_slice(const Shape& sh, const bf16* target, const bf16* U, const bf16* F,
                                const bf16* W2, const Ws& ws, uint32_t* status, int nsm, cudaStream_t st) {
  const int K = vslice_chunks(sh, nsm);
  if (K == 0) return cudaErrorNotSupported;
  VsParams P;
  memset(&P, 0, sizeof(P));
  cudaError_t e = encode_w2_map(sh, W2, &P.w2);
  if (e != cudaSuccess) return e;
  P.sh = sh;
  P.target = target;
  P.U = U;
  P.F = F;
  P.ws = ws;
  P.status = status;
  P.K = K;
  const size_t smem = VsLayout(sh.r, K).total;
  e = cudaFuncSetAttribute(verify_slice_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cudaErrorNotSupported;
  }
  const int G = (sh.NC + K - 1) / K;
  verify_slice_kernel<<<G, VS_THREADS, smem, st>>>(P);
  return cudaGetLastError();
}

}  // namespace spec
