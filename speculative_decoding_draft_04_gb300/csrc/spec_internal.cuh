// Internal device/host definitions shared by the kernels of libspec.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <math.h>

#include "../../include/spec.h"
#include "spec_df.cuh"

namespace spec {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------- geometry
constexpr int BN = 128;       // vocabulary columns per slice (one GEMM tile's N)
constexpr int CW = 32;        // vocabulary columns per draft partial (chunk)
constexpr int VB = 32;        // vocabulary columns per verification slice
constexpr int VT = 64;        // vocabulary columns per verification tensor-memory tile
constexpr int HPB = 256;      // columns per extended-precision block
constexpr int NT = 256;       // threads per CTA for every kernel
constexpr int MAX_GAMMA = 16;

struct Shape {
  int B, gamma, V, r, NS, NC, NSV, HB;   // NS = ceil(V / BN), NC = ceil(V / CW),
                                          // NSV = ceil(V / VB), HB = ceil(V / HPB)
  int rnn;     // 0: Markov head, factor rows W1[x_j]; 1: RNN head, factor rows [gamma][B]
  int NA;      // rows of the factor table: V (Markov) or gamma * B (RNN)
};

// Row of the transition-factor table for draft row j of request b: the Markov
// head's W1[x_j] (x_0 = the anchor) or the RNN head's a_j row of request b.
__device__ __forceinline__ int factor_row(const Shape& sh, int b, int j, int prev_token) {
  return sh.rnn ? j * sh.B + b : prev_token;
}

// A decision queued for re-decision in extended precision.
enum HpKind { HP_DRAFT = 0, HP_BONUS = 1, HP_RESID = 2 };
struct HpItem {
  int b, j, kind, prev;   // request, row, kind, previous token (draft rows)
  float u;                // the decision's uniform
  int fast_token;         // token chosen by the first pass
  double shift_q;         // first-pass logsumexp of the draft row
  double shift_p;         // first-pass logsumexp of the target row
};

// Control words at the start of the workspace.
//   CTRL_BAR_COUNT / CTRL_ABORT: grid barrier of the persistent draft kernels;
//   CTRL_DITEMS: draws queued by the slice-resident draft over all its steps
//   (ws.items, up to ws.item_cap); CTRL_HPNEXT: re-decision units handed out in the
//   draft's tile phases; CTRL_REDO: gamma - the earliest draft step whose
//   token a deferred re-decision changed (0: none); CTRL_STEP0 + k: queued
//   re-decisions of draft step k.
enum {
  CTRL_ITEMS = 0, CTRL_SLOW = 1, CTRL_NPACKED = 2, CTRL_BAR_COUNT = 3, CTRL_DITEMS = 4,
  CTRL_ABORT = 5, CTRL_HPNEXT = 6, CTRL_REDO = 7, CTRL_STEP0 = 8, CTRL_WORDS = 32
};

// Test builds of the draft kernels (never the default): HOOK_PERTURB makes
// queued draws write a wrong token first (the re-decision must correct it and
// trigger the redo); HOOK_STALL makes the first grid barrier wait for one
// arrival more than the grid has, so it can only end by its time limit.
enum { HOOK_NONE = 0, HOOK_PERTURB = 1, HOOK_STALL = 2 };

// Workspace views (host computes the offsets; see spec_abi.cu).
constexpr int TRACE_SLOTS = 8;   // timestamps per draft step (persistent kernel trace)
struct Ws {
  uint32_t* ctrl;       // [CTRL_WORDS]
  unsigned long long* trace;  // [2][MAX_GAMMA][TRACE_SLOTS] globaltimer ns, CTA 0: the
                              // draft's phases, then events inside its tile phase
  HpItem* items;        // [item_cap] queued decisions
  int max_items;        // decisions re-decided together (hpsum / hpcnt / hpnorm slots)
  int item_cap;         // entries of `items` (B * gamma: every draft draw of a cycle)
  float2* hpsum;        // [max_items][hp_cols][NC] chunk sums of the re-decided rows (hi, lo)
  int hp_cols;          // 3 (draft and verify) or 1 (draft only)
  uint32_t* hpcnt;      // [max_items] blocks summed so far (zeroed before the draft)
  float4* hpw;          // [hpw_items][V] residual items' weights (q hi, q lo, p hi, p lo),
                        // kept from the first sums pass for the residual pass
  int hpw_items;        // items with stored weights (0: none)
  float4* hpnorm;       // [max_items] residual items: 1/Z_p, 1/Z_q (double-floats), written
                        // once the first sums pass is complete
  // draft
  float4* dpart;        // [B][NC] draft partials per CW-column chunk: (c, m, s, q2)
  void* abuf;           // [min(B, 128)][r] storage type: the next draft step's A rows
                        // W1[x_k] (slice-resident draft kernel)
  // verify
  int* rowptr;          // [B+1]
  int2* prow;           // [B*gamma] packed (b, j), j < L_b
  int* prevtok;         // [B*gamma] x_j of each packed row
  int* vflags;          // [B] bit0 bad request, bits 8.. ratio flags
  double* lse_p;        // [B][gamma+1]
  float4* bpart;        // [B][NSV] bonus row (c, s, p2, 0)
  float4* vpart;        // [B*gamma][NSV] (alpha, resid, p2, q2)
  int* slow;            // [B]
  uint32_t* accbits;    // [B] first-pass ratio-test outcomes
  float4* rowc;         // [B*gamma] packed row: 1/T and -lse_q as double-float pairs
  float2* rowp;         // [B][gamma+1] -lse_p as a double-float pair
};

// Candidate trees: B requests of N slots, depth <= gamma.
struct TreeShape {
  int B, N, gamma, V, r;
};

// RNN head inputs and outputs of the draft (all null for the Markov head).
struct RnnParams {
  const void* Wr;        // [3r][2r] storage type
  const float* hproj;    // [B][gamma][3][r]
  void* arows;           // [gamma][B][r] storage type, out: the factor rows a_k
  void* state;           // [gamma+1][B][r] storage type, scratch: s_k of every step
};

// Inputs the extended-precision kernels read.
struct HpRows {
  const void* target;
  const void* U;
  const void* W1;
  const void* W2;
  const float* temp;
};

// Near-boundary band of a draw from a distribution with first-pass weights
// (units: probability).  The constants are calibrated: the largest first-pass
// errors measured against the float64 oracle over the seeded workloads, with
// a safety factor.
struct Eps {
  float elem;    // x sqrt(sum q^2): per-weight rounding of the first pass
  float slice;   // x sqrt(sum_slice mass^2): per-slice sums and factors
  float abs_;    // floor
  float ratio;   // relative band of a ratio test
  float norm;    // residual draws: error of the two row normalisers
  float scale;   // user multiplier (SPEC_OPT_EPS_SCALE)
};

// ---------------------------------------------------------------- loads
__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const bf16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float tof(float x) { return x; }
__device__ __forceinline__ float tof(bf16 x) { return __bfloat162float(x); }

// ---------------------------------------------------------------- first-pass logit
// x = ((U - c) + bias) * (1/T) with c a reference close to the largest U of
// the slice: for bf16 data U - c is exact, so the dominant entries carry
// only the rounding of a small number.  Explicit round-to-nearest intrinsics
// keep the compiler from fusing differently in different kernels, so a
// recomputation reproduces the same bits from the same bias.
__device__ __forceinline__ float fast_x(float Uv, float c, float bias, float invT) {
  return __fmul_rn(__fadd_rn(__fsub_rn(Uv, c), bias), invT);
}
__device__ __forceinline__ float fast_w(float x, float m) { return __expf(__fsub_rn(x, m)); }
__device__ __forceinline__ float fast_tx(float tv, float c, float invT) {
  return __fmul_rn(__fsub_rn(tv, c), invT);
}

// exp(g) for a double g, evaluated in single precision with the low part of g
// applied as a first-order correction (|g - float(g)| < 2^-24 |g|).
__device__ __forceinline__ float exp_split(double g) {
  float gh = (float)g;
  float gl = (float)(g - (double)gh);
  return expf(gh) * (1.0f + gl);
}

// ---------------------------------------------------------------- double-float
// (struct df and the host-portable operations are in spec_df.cuh)

__device__ __forceinline__ df df_make(float x) { return {x, 0.f}; }
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
__device__ __forceinline__ df df_add(df a, df b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  float hi = __fadd_rn(s, e);
  float lo = __fsub_rn(e, __fsub_rn(hi, s));
  return {hi, lo};
}
__device__ __forceinline__ df df_addf(df a, float b) { return df_add(a, df_make(b)); }
__device__ __forceinline__ df df_neg(df a) { return {-a.hi, -a.lo}; }
__device__ __forceinline__ double df_d(df a) { return (double)a.hi + (double)a.lo; }
__device__ __forceinline__ df df_from_d(double x) {
  float h = (float)x;
  return {h, (float)(x - (double)h)};
}
// a * f for a float f (error ~ 2^-46 relative)
__device__ __forceinline__ df df_mulf(df a, float f) {
  float p = __fmul_rn(a.hi, f);
  float e = fmaf(a.hi, f, -p);
  e = fmaf(a.lo, f, e);
  float hi = __fadd_rn(p, e);
  float lo = __fsub_rn(e, __fsub_rn(hi, p));
  return {hi, lo};
}
__device__ __forceinline__ df shfl_xor_df(df v, int m) {
  return {__shfl_xor_sync(0xffffffffu, v.hi, m), __shfl_xor_sync(0xffffffffu, v.lo, m)};
}
__device__ __forceinline__ df shfl_up_df(df v, int d) {
  return {__shfl_up_sync(0xffffffffu, v.hi, d), __shfl_up_sync(0xffffffffu, v.lo, d)};
}

// ---------------------------------------------------------------- block reductions (NT threads)
__device__ __forceinline__ float warp_max(float v) {
  for (int m = 16; m; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
  for (int m = 16; m; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}
__device__ __forceinline__ df warp_sum_df(df v) {
  for (int m = 16; m; m >>= 1) v = df_add(v, shfl_xor_df(v, m));
  return v;
}
// Results broadcast to all threads.  `sh` must hold >= 32 floats; calls are
// separated by __syncthreads inside.
__device__ __forceinline__ float block_max(float v, float* sh) {
  v = warp_max(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = (threadIdx.x < (NT >> 5)) ? sh[threadIdx.x] : -INFINITY;
  if (threadIdx.x < 32) r = warp_max(r);
  if (threadIdx.x == 0) sh[0] = r;
  __syncthreads();
  r = sh[0];
  __syncthreads();
  return r;
}
__device__ __forceinline__ float block_sum(float v, float* sh) {
  v = warp_sum(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = (threadIdx.x < (NT >> 5)) ? sh[threadIdx.x] : 0.f;
  if (threadIdx.x < 32) r = warp_sum(r);
  if (threadIdx.x == 0) sh[0] = r;
  __syncthreads();
  r = sh[0];
  __syncthreads();
  return r;
}
// Deterministic double-float sum over the block (fixed tree order).
__device__ __forceinline__ df block_sum_df(df v, float* sh) {
  v = warp_sum_df(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    sh[2 * (threadIdx.x >> 5)] = v.hi;
    sh[2 * (threadIdx.x >> 5) + 1] = v.lo;
  }
  __syncthreads();
  df r = {0.f, 0.f};
  if (threadIdx.x < (NT >> 5)) r = {sh[2 * threadIdx.x], sh[2 * threadIdx.x + 1]};
  if (threadIdx.x < 32) r = warp_sum_df(r);
  if (threadIdx.x == 0) { sh[0] = r.hi; sh[1] = r.lo; }
  __syncthreads();
  r = {sh[0], sh[1]};
  __syncthreads();
  return r;
}
// Exclusive prefix (double-float) of one value per thread in thread order;
// *total receives the block total.  `sh` holds >= 66 floats.
// Exclusive block scan of v with the block total, one barrier: warp scans by
// shuffles, then every thread adds the warp totals in warp order (so all hold
// the same total, and each warp's offset is a prefix of that same sum).  `sw`
// (NT / 32 entries) may be written again only after a later barrier.
__device__ __forceinline__ df block_scan1_df(df v, df* total, float2* sw) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  df inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const df o = shfl_up_df(inc, d);
    if (lane >= d) inc = df_add(inc, o);
  }
  if (lane == 31) sw[w] = make_float2(inc.hi, inc.lo);
  df within = shfl_up_df(inc, 1);
  if (lane == 0) within = {0.f, 0.f};
  __syncthreads();
  df off = {0.f, 0.f}, tot = {0.f, 0.f};
#pragma unroll
  for (int q = 0; q < NT / 32; ++q) {
    if (q == w) off = tot;
    const float2 t = sw[q];
    tot = df_add(tot, df{t.x, t.y});
  }
  *total = tot;
  return df_add(off, within);
}
// block_scan1_df with two fp32 block sums riding on the same barrier (every
// thread adds the warp sums in warp order, so all hold the same values).
__device__ __forceinline__ df block_scan1_df2(df v, df* total, float& a, float& c, float4* sw) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  df inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const df o = shfl_up_df(inc, d);
    if (lane >= d) inc = df_add(inc, o);
  }
#pragma unroll
  for (int m = 16; m; m >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, m);
    c += __shfl_xor_sync(0xffffffffu, c, m);
  }
  if (lane == 31) sw[w] = make_float4(inc.hi, inc.lo, a, c);
  df within = shfl_up_df(inc, 1);
  if (lane == 0) within = {0.f, 0.f};
  __syncthreads();
  df off = {0.f, 0.f}, tot = {0.f, 0.f};
  float ta = 0.f, tc = 0.f;
#pragma unroll
  for (int q = 0; q < NT / 32; ++q) {
    if (q == w) off = tot;
    const float4 t = sw[q];
    tot = df_add(tot, df{t.x, t.y});
    ta += t.z;
    tc += t.w;
  }
  a = ta;
  c = tc;
  *total = tot;
  return df_add(off, within);
}
__device__ __forceinline__ df block_excl_scan_df(df v, df* total, float* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  df inc = v;
  for (int d = 1; d < 32; d <<= 1) {
    df o = shfl_up_df(inc, d);
    if (lane >= d) inc = df_add(inc, o);
  }
  __syncthreads();
  if (lane == 31) { sh[2 * w] = inc.hi; sh[2 * w + 1] = inc.lo; }
  __syncthreads();
  if (w == 0) {
    df x = (lane < (NT >> 5)) ? df{sh[2 * lane], sh[2 * lane + 1]} : df{0.f, 0.f};
    df xi = x;
    for (int d = 1; d < 32; d <<= 1) {
      df o = shfl_up_df(xi, d);
      if (lane >= d) xi = df_add(xi, o);
    }
    // store exclusive warp offsets and the total
    df ex = shfl_up_df(xi, 1);
    if (lane == 0) ex = {0.f, 0.f};
    if (lane < (NT >> 5)) { sh[2 * lane] = ex.hi; sh[2 * lane + 1] = ex.lo; }
    if (lane == (NT >> 5) - 1) { sh[64] = xi.hi; sh[65] = xi.lo; }
  }
  __syncthreads();
  df off = {sh[2 * w], sh[2 * w + 1]};
  *total = {sh[64], sh[65]};
  df within = shfl_up_df(inc, 1);
  if (lane == 0) within = {0.f, 0.f};
  df ex = df_add(off, within);
  __syncthreads();
  return ex;
}


// sum_{i in [ib, ie)} a[i] * W2[i][v] with fp32 FMAs in i order.  W2 loads
// are issued 8 rows ahead of their use so the loop is not bound by the
// latency of one L2 round trip per row.  (ie - ib) % 8 == 0.
template <typename DT>
__device__ __forceinline__ float dot_col(const float* a, const DT* __restrict__ W2, int V, int ib,
                                         int ie, int v) {
  constexpr int UN = 8;
  float acc = 0.f;
  float cur[UN];
#pragma unroll
  for (int u = 0; u < UN; ++u) cur[u] = ib + u < ie ? ldf(W2 + (size_t)(ib + u) * V + v) : 0.f;
  for (int i0 = ib; i0 < ie; i0 += UN) {
    float nxt[UN];
    const bool more = i0 + UN < ie;
#pragma unroll
    for (int u = 0; u < UN; ++u) nxt[u] = more ? ldf(W2 + (size_t)(i0 + UN + u) * V + v) : 0.f;
#pragma unroll
    for (int u = 0; u < UN; ++u) acc = fmaf(a[i0 + u], cur[u], acc);
#pragma unroll
    for (int u = 0; u < UN; ++u) cur[u] = nxt[u];
  }
  return acc;
}

__device__ __forceinline__ void set_status(uint32_t* st, uint32_t bits) {
  if (st) atomicOr(st, bits);
}
__device__ __forceinline__ bool temp_ok(float T) { return isfinite(T) && T > 0.f; }

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Barrier across all CTAs of a cooperative launch (all co-resident).  Thread 0
// of each CTA adds 1 to a counter that only grows (zeroed before the launch)
// with a release, and waits with acquire loads until it reaches
// (barriers passed + 1) x CTAs: one atomic per CTA and no reset.  The CTA's
// other threads are ordered before the release by the __syncthreads.  Every
// wait is bounded: on timeout, or when another CTA has aborted, it sets
// SPEC_DEV_TIMEOUT / the abort word and returns false, and the caller leaves
// the kernel.  `gen` is thread 0's count of barriers passed (0 at kernel start).
// `extra` (test builds only) raises the count the barrier waits for.
__device__ __forceinline__ bool grid_sync(uint32_t* ctrl, uint32_t nblocks, uint32_t& gen,
                                          uint32_t* status, uint32_t extra = 0u) {
  __shared__ int s_gs_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const uint32_t target = (gen + 1) * nblocks + extra;
    uint32_t seen;
    asm volatile("atom.add.release.gpu.global.u32 %0, [%1], 1;\n"
                 : "=r"(seen) : "l"(ctrl + CTRL_BAR_COUNT) : "memory");
    seen += 1;
    // bounded by wall-clock time (1 s; a phase takes microseconds)
    uint32_t it = 0;
    unsigned long long t0 = 0;
    while (seen < target) {
      seen = ld_acquire_gpu(ctrl + CTRL_BAR_COUNT);
      if (seen >= target) break;
      ++it;
      if ((it & 7) == 0 && ld_acquire_gpu(ctrl + CTRL_ABORT) != 0u) { ok = 0; break; }
      if (it == 64) t0 = globaltimer_ns();
      if (it > 64) {
        if ((it & 63) == 0 && globaltimer_ns() - t0 > 1000ull * 1000 * 1000) {
          ok = 0;
          atomicExch(ctrl + CTRL_ABORT, 1u);
          set_status(status, SPEC_DEV_TIMEOUT);
          break;
        }
        __nanosleep(32);
      }
    }
    gen += 1;
    s_gs_ok = ok;
  }
  __syncthreads();
  return s_gs_ok != 0;
}

}  // namespace spec
