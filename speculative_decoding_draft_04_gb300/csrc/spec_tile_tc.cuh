// Warp-specialised tensor-memory tile engine for the rank-r bias tiles
// (bf16, r % 64 == 0) of the draft step (N = 128 columns per tile) and of the
// verification (N = 64).  A CTA walks its share of (row tile, slice of N
// vocabulary columns) tiles; the roles run concurrently and hand buffers to
// each other through shared-memory mbarriers:
//
//   warp 4             producer: one lane loads the W2 slice (r x N, read in
//                      place as the MN-major B operand, 128-byte swizzle) by
//                      TMA; the epilogue object loads the tile's logit rows
//                      (TMA for the draft's U_k, a cp.async row gather for the
//                      verification's packed U and target rows).
//   warps 6-7          gather the W1[x_{k-1}] rows of a request tile (the A
//                      operand, K-major, 128-byte swizzle) with cp.async, once
//                      per request tile, after the last MMA that read the old
//                      rows has completed (a barrier of its own, committed once
//                      per request tile: every waiter waits for each phase of
//                      the barriers it polls in turn, so a parity test is never
//                      two phases behind).
//   warp 5, one lane   issues the r/16 MMAs of a tile (M = 128, N = 128, K = 16)
//                      into one of two 128-column TMEM accumulators and commits
//                      them to the accumulator's "full" barrier and to the W2
//                      stage's "empty" barrier.
//   warps 0-3          epilogue, thread = tile row = TMEM lane: reads its row of
//   (and 8-11)         the accumulator (tcgen05.ld) and of the logit tile (shared
//                      memory) and reduces it to its partials without
//                      exchanging anything with other threads.  With EG = 2
//                      epilogue groups (a 384-thread CTA) the second group,
//                      warps 8-11 (same TMEM lanes: warp % 4), takes the other
//                      half of each tile's columns.
//
// Barrier phases are counted with running per-CTA counters (tiles, request
// tiles) that every thread advances identically, so the state carries over
// from one draft step to the next without re-initialising the barriers.
// Every wait is bounded; a wait that gives up raises a CTA-wide failure flag
// that makes every other wait return at once.
#pragma once

#include <cuda.h>

#include "spec_tc.cuh"

namespace spec {

constexpr uint32_t TP_TMEM_COLS = 256;         // two accumulators of up to 128 fp32 columns
constexpr int TP_XBYTES = 32768;               // logit rows of one tile: 128 x 128 bf16, or
                                               // 128 x 64 U rows + 128 x 64 target rows

// Barrier slots.
enum : int {
  TB_W2_FULL = 0,    // + stage (2)
  TB_W2_EMPTY = 2,   // + stage (2)
  TB_U_FULL = 4,     // + buffer (2): the tile's logit rows
  TB_U_EMPTY = 6,    // + buffer (2)
  TB_T_FULL = 8,     // + accumulator (2)
  TB_T_EMPTY = 10,   // + accumulator (2)
  TB_A_FULL = 12,
  TB_A_EMPTY = 13,   // committed after the last MMA of each request tile
  TB_COUNT = 14
};

// Shared-memory plan (offsets from a 1024-byte aligned base) for N-column
// tiles.
struct TpLayout {
  int nw;                                      // W2 stages (2 when they fit)
  size_t offA, offW, wbytes, offU, total;
  __host__ __device__ TpLayout(int r, int N) {
    const size_t a = (size_t)(r / 64) * 16384;
    wbytes = (size_t)(N / 64) * r * 128;
    nw = (a + 2 * wbytes + 2 * TP_XBYTES <= (size_t)208 * 1024) ? 2 : 1;
    offA = 0;
    offW = a;
    offU = offW + (size_t)nw * wbytes;
    total = offU + 2 * (size_t)TP_XBYTES + 1024;   // + slack for 1 KB alignment
  }
};

// Tensor maps of one call (encoded on the host, passed as a __grid_constant__
// kernel parameter).
struct TpMaps {
  CUtensorMap u;     // U viewed as [B][gamma][V], box 64 x 1 x 128, 128-byte swizzle
  CUtensorMap w2;    // W2 viewed as [r][V],       box 64 x r,       128-byte swizzle
  CUtensorMap a;     // slice-resident draft: its A-row buffer [rows][r], box 64 x 128
};

// Pipeline state of a CTA, identical in every thread.
struct TpState {
  uint32_t tmem;     // base of the 256 TMEM columns
  uint64_t* bar;     // TB_COUNT mbarriers
  int* fail;         // CTA-wide failure flag (shared)
  uint32_t gi;       // tiles processed so far by this CTA
  uint32_t ga;       // request tiles gathered so far
};

__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

// xfull_count: arrivals that complete a logit-row fill (1 for a TMA fill
// with its byte count, 32 for a cp.async gather by the producer warp);
// eg: epilogue groups of 128 threads.
__device__ __forceinline__ void tp_init(uint64_t* bar, uint32_t xfull_count, uint32_t eg = 1) {
  for (int s = 0; s < 2; ++s) {
    mbar_init(bar + TB_W2_FULL + s, 1);
    mbar_init(bar + TB_W2_EMPTY + s, 1);
    mbar_init(bar + TB_U_FULL + s, xfull_count);
    mbar_init(bar + TB_U_EMPTY + s, TC_M * eg);
    mbar_init(bar + TB_T_FULL + s, 1);
    mbar_init(bar + TB_T_EMPTY + s, TC_M * eg);
  }
  mbar_init(bar + TB_A_FULL, 64);
  mbar_init(bar + TB_A_EMPTY, 1);
}

// ---------------------------------------------------------------- primitives
// Bounded wait for the completion of the phase with parity `parity`: polls
// without blocking (mbarrier.test_wait), backs off, and gives up after
// TP_WAIT_NS of wall-clock time (the pipeline's stages take microseconds), or
// at once when another thread raised *fail.
constexpr unsigned long long TP_WAIT_NS = 100ull * 1000 * 1000;
__device__ __forceinline__ bool tp_test(uint32_t a, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(a), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ bool tp_wait(uint64_t* bar, uint32_t parity, volatile int* fail) {
  const uint32_t a = smem_u32(bar);
  for (int it = 0; it < 64; ++it)
    if (tp_test(a, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (tp_test(a, parity)) return true;
    if ((it & 15) == 15) {
      if (*fail) return false;
      if (globaltimer_ns() - t0 > TP_WAIT_NS) break;
    }
    __nanosleep(64);
  }
  *fail = 1;
  return false;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
// Arrive on `bar` once all of this thread's earlier cp.async copies are done
// (the arrival is one of the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// TMA tile loads into shared memory, completing on `bar` (bytes counted).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4}], [%5];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
// Prefetch a tile of a 3-D tensor map into L2 (no shared memory involved).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];\n" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}
// Contiguous bytes [p, p + bytes) into L2 by the bulk-copy engine (p 16-byte
// aligned, bytes a multiple of 16); no completion to wait for.
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ uint4 lds128(const unsigned char* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 16-byte chunk j (0..15) of row m of a 128-byte-swizzled [128][BN] bf16 tile
// stored as two 64-column boxes.
__device__ __forceinline__ const unsigned char* tp_uchunk(const unsigned char* ub, int m, int j) {
  return ub + (j >> 3) * (TC_M * 128) + m * 128 + (((j & 7) ^ (m & 7)) << 4);
}

// ---------------------------------------------------------------- the engine
// Tile list of this CTA: tiles t0 + i * stride, i < n; tile t is (row tile
// t / nsl, slice t % nsl) of N columns.  E supplies (all threads may call):
//   int  token(int mtile, int m)             W1 row of row m, -1 for none
//   void load_x(int mtile, int slice, unsigned char* xb, uint64_t* full, int lane,
//               int next_mtile, int next_slice)
//                                            fill the tile's logit rows (called by
//                                            the 32 lanes of the producer warp; the
//                                            next tile, -1 if none, may be prefetched)
//   void epilogue(int mtile, int slice, int m, const unsigned char* xb,
//                 uint32_t tmem_row, int grp) one row of one tile (grp: the
//                                            epilogue group, 0 when EG == 1)
// `s_tok` is a 128-entry shared array for the gatherers.  Returns false if a
// wait gave up (after draining what it started).
// Copy the TC_M rows W1[tok[m]] (r bf16 each, tok < 0: zero row) into the
// 128-byte-swizzled A tile with cp.async, thread q of `nt` taking 16-byte
// chunks q, q + nt, ...; waits for its own copies.  r / 8 is a power of two
// (r % 64 == 0 on this path).
__device__ __forceinline__ void tp_gather_a(unsigned char* As, const bf16* W1, const int* tok, int r,
                                            int q, int nt) {
  const int lg = __ffs(r / 8) - 1;            // log2(chunks per row)
  const int cmask = (r / 8) - 1;
  for (int c = q; c < TC_M * (r / 8); c += nt) {
    const int m = c >> lg, j = c & cmask;
    const int t = tok[m];
    const bool valid = t >= 0;
    const bf16* src = valid ? W1 + (size_t)t * r + j * 8 : W1;
    unsigned char* dst = As + (size_t)(j >> 3) * 16384 + m * 128 + (((j & 7) ^ (m & 7)) << 4);
    cp_async16(dst, src, valid);
  }
  cp_async_commit();
  cp_async_wait_all();
}

template <int N, class E, int EG = 1>
__device__ __forceinline__ bool tp_run(const E& e, const Shape& sh, const TpMaps& maps,
                                       const bf16* W1, int nsl, int t0, int stride, int n,
                                       unsigned char* smem_raw, TpState& st, int* s_tok,
                                       unsigned long long* ttr = nullptr) {
  static_assert(N == 64 || N == 128, "tile width");
  static_assert(EG == 1 || EG == 2, "epilogue groups");
  if (n <= 0) return true;
  unsigned char* smem = align1k(smem_raw);
  const TpLayout lay(sh.r, N);
  unsigned char* As = smem + lay.offA;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = sh.r;
  const uint32_t wbytes = (uint32_t)lay.wbytes;
  uint64_t* bar = st.bar;
  volatile int* fail = st.fail;
  auto mt_of = [&](int i) { return (t0 + i * stride) / nsl; };
  auto sl_of = [&](int i) { return (t0 + i * stride) % nsl; };

  // Earlier generic-proxy use of these buffers (sampling, re-decision phases)
  // is ordered before this phase's TMA and MMA accesses.
  fence_async_shared();
  __syncthreads();

  if (warp == 4) {
    if (lane == 0) tma_prefetch_map(&maps.w2);
    for (int i = 0; i < n && !*fail; ++i) {
      const uint32_t g = st.gi + i;
      const int n0 = sl_of(i) * N;
      if (lane == 0) {
        const int s = (int)(g % (uint32_t)lay.nw);
        const uint32_t f = g / (uint32_t)lay.nw;
        if (f == 0 || tp_wait(bar + TB_W2_EMPTY + s, (f - 1) & 1u, fail)) {
          unsigned char* wb = smem + lay.offW + (size_t)s * wbytes;
          mbar_expect_tx(bar + TB_W2_FULL + s, wbytes);
          for (int h = 0; h < N / 64; ++h)
            tma_load_2d(wb + h * r * 128, &maps.w2, n0 + 64 * h, 0, bar + TB_W2_FULL + s);
        }
      }
      __syncwarp();
      if (*fail) break;
      const int b = (int)(g & 1u);
      const uint32_t fu = g >> 1;
      if (fu >= 1 && !tp_wait(bar + TB_U_EMPTY + b, (fu - 1) & 1u, fail)) break;
      e.load_x(mt_of(i), sl_of(i), smem + lay.offU + (size_t)b * TP_XBYTES, bar + TB_U_FULL + b, lane,
               i + 1 < n ? mt_of(i + 1) : -1, i + 1 < n ? sl_of(i + 1) : -1);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      const uint32_t idesc = tc_idesc_n(N);
      const uint32_t a0 = smem_u32(As);
      uint32_t ga = st.ga;
      for (int i = 0; i < n; ++i) {
        const uint32_t g = st.gi + i;
        if (i == 0 || mt_of(i) != mt_of(i - 1)) {
          if (!tp_wait(bar + TB_A_FULL, ga & 1u, fail)) break;
          ++ga;
        }
        const int s = (int)(g % (uint32_t)lay.nw);
        if (!tp_wait(bar + TB_W2_FULL + s, (g / (uint32_t)lay.nw) & 1u, fail)) break;
        if (ttr && i == 0) ttr[2] = globaltimer_ns();
        const int b = (int)(g & 1u);
        if (g >= 2 && !tp_wait(bar + TB_T_EMPTY + b, ((g >> 1) - 1) & 1u, fail)) break;
        tc_fence_after();
        const uint32_t w0 = smem_u32(smem + lay.offW + (size_t)s * wbytes);
        const uint32_t d = st.tmem + (uint32_t)(b * N);
        for (int kk = 0; kk < r; kk += 16) {
          const uint64_t ad = tc_sdesc(a0 + (uint32_t)((kk >> 6) * 16384 + (kk & 63) * 2), 16, 1024);
          const uint64_t bd = tc_sdesc(w0 + (uint32_t)(kk * 128), (uint32_t)(r * 128), 1024);
          tc_mma(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar + TB_T_FULL + b);
        tc_commit(bar + TB_W2_EMPTY + s);
        if (ttr && i == 0) ttr[3] = globaltimer_ns();
        if (i == n - 1 || mt_of(i + 1) != mt_of(i)) tc_commit(bar + TB_A_EMPTY);
      }
    }
  } else if (warp == 6 || warp == 7) {
    // 64 gatherers copy the A tile's rows (16-byte chunks); for the first
    // request tile of the phase the 128 epilogue threads, idle until the first
    // accumulator is ready, copy with them (E::kHelpGather).  The two 192-thread
    // barriers of that first tile are always reached, also when a wait fails.
    const int q0 = threadIdx.x - 192;
    uint32_t ga = st.ga;
    for (int i = 0; i < n; ++i) {
      const bool helped = E::kHelpGather && i == 0;
      if (!helped && (*fail || (i > 0 && mt_of(i) == mt_of(i - 1)))) {
        if (*fail) break;
        continue;
      }
      // the last MMA that read the previous request tile's rows
      const bool okw = ga < 1 || tp_wait(bar + TB_A_EMPTY, (ga - 1) & 1u, fail);
      ++ga;
      const int mt = mt_of(i);
      if (okw)
        for (int m = q0; m < TC_M; m += 64) s_tok[m] = e.token(mt, m);
      if (helped) named_bar(2, 192); else named_bar(1, 64);
      if (ttr && q0 == 0 && i == 0) ttr[0] = globaltimer_ns();
      if (okw) tp_gather_a(As, W1, s_tok, r, helped ? 128 + q0 : q0, helped ? 192 : 64);
      if (ttr && q0 == 0 && i == 0) ttr[1] = globaltimer_ns();
      fence_async_shared();
      if (helped) named_bar(2, 192);          // the helpers' copies are in place too
      if (!okw) break;
      mbar_arrive(bar + TB_A_FULL);
      named_bar(1, 64);          // s_tok is free for the next request tile
    }
  } else {
    if constexpr (E::kHelpGather) {
      // help copy the phase's first A tile (the gatherers pass the tokens;
      // both barriers are reached by the gatherers in every case)
      named_bar(2, 192);
      if (!*fail) tp_gather_a(As, W1, s_tok, r, (int)threadIdx.x, 192);
      fence_async_shared();
      named_bar(2, 192);
    }
    // epilogue: thread = row
    const int m = threadIdx.x & (TC_M - 1);
    const int grp = warp >= 8 ? 1 : 0;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    for (int i = 0; i < n; ++i) {
      const uint32_t g = st.gi + i;
      const int b = (int)(g & 1u);
      if (!tp_wait(bar + TB_U_FULL + b, (g >> 1) & 1u, fail)) break;
      if (!tp_wait(bar + TB_T_FULL + b, (g >> 1) & 1u, fail)) break;
      if (ttr && threadIdx.x == 0 && i == 0) ttr[4] = globaltimer_ns();
      tc_fence_after();
      e.epilogue(mt_of(i), sl_of(i), m, smem + lay.offU + (size_t)b * TP_XBYTES,
                 st.tmem + lane_base + (uint32_t)(b * N), grp);
      if (ttr && threadIdx.x == 0) ttr[i == 0 ? 5 : 6] = globaltimer_ns();
      tc_fence_before();
      mbar_arrive(bar + TB_T_EMPTY + b);
      mbar_arrive(bar + TB_U_EMPTY + b);
    }
  }
  if (ttr && threadIdx.x == 0) ttr[7] = globaltimer_ns();
  // advance the running counters identically in every thread
  uint32_t segs = 0;
  for (int i = 0; i < n; ++i) segs += (i == 0 || mt_of(i) != mt_of(i - 1)) ? 1u : 0u;
  st.gi += (uint32_t)n;
  st.ga += segs;
  __syncwarp();
  __syncthreads();
  if (*fail) {
    // drain: the last accumulator's commit covers every MMA issued before it
    const uint32_t g = st.gi - 1;
    if (threadIdx.x == 0) mbar_wait(bar + TB_T_FULL + (g & 1u), (g >> 1) & 1u, 1u << 20);
    __syncthreads();
    return false;
  }
  return true;
}

}  // namespace spec
