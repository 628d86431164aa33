// Extended-precision re-decision: shared device code (spec_refine.cu describes
// the method).  Every weight, sum and scan here is a double-float (spec_df.cuh)
// -- accurate to about 1e-13 relative, far below the first pass's error band
// -- so the path runs at the fp32 rate; fp64 appears only in a few per-item
// scalars.  Data written by other CTAs of the same launch (queued items, block
// sums) is read through L2 (ld.global.cg), so the bodies also serve the
// persistent draft kernel.
#pragma once

#include "spec_gemm.cuh"

namespace spec {

// HpItem is 40 bytes, so array elements are only 8-byte aligned: load it with
// 8-byte accesses.
static_assert(sizeof(HpItem) == 40 && alignof(HpItem) == 8, "HpItem layout");
__device__ __forceinline__ HpItem ldcg_item(const HpItem* p) {
  HpItem h;
  const int2* q = reinterpret_cast<const int2*>(p);
  const int2 a = __ldcg(q), b = __ldcg(q + 1), c = __ldcg(q + 2);
  h.b = a.x; h.j = a.y; h.kind = b.x; h.prev = b.y;
  h.u = __int_as_float(c.x);
  h.fast_token = c.y;
  h.shift_q = __ldcg(&p->shift_q);
  h.shift_p = __ldcg(&p->shift_p);
  return h;
}

// Per-item constants, identical in every thread.
template <typename DT>
struct ItemCtx {
  const DT* Urow;
  const DT* Trow;
  df invT;     // 1 / T_b
  df nsq;      // -shift_q (logsumexp of the draft row when known, else 0)
  df nsp;      // -shift_p (logsumexp of the target row)
};

template <typename DT>
__device__ __forceinline__ ItemCtx<DT> item_ctx(const Shape& sh, const HpRows& R, const HpItem& it) {
  ItemCtx<DT> c;
  c.Urow = (const DT*)R.U + ((size_t)it.b * sh.gamma + (it.kind == HP_BONUS ? 0 : it.j)) * sh.V;
  c.Trow = (const DT*)R.target + ((size_t)it.b * (sh.gamma + 1) + it.j) * sh.V;
  c.invT = dd_recip(R.temp[it.b]);
  c.nsq = dd_from_double(-it.shift_q);
  c.nsp = dd_from_double(-it.shift_p);
  return c;
}

// The same constants computed by thread 0 and shared (a CTA-wide call; the
// fp64 -> double-float conversions then cost one thread, not all).
template <typename DT>
__device__ __forceinline__ ItemCtx<DT> item_ctx_shared(const Shape& sh, const HpRows& R, const HpItem& it,
                                                       ItemCtx<DT>* slot) {
  if (threadIdx.x == 0) *slot = item_ctx<DT>(sh, R, it);
  __syncthreads();
  const ItemCtx<DT> c = *slot;
  __syncthreads();
  return c;
}

// Transition bias W1[x] . W2[:, v] as a double-float: four interleaved compensated
// chains over r (the products of bf16 operands are exact in fp32; fp32
// operands add each product's FMA remainder to a separate sum).  `a` holds
// W1[x] widened to float.  W2 is read straight from global memory, one column
// per thread (coalesced), one batch of 16 rows ahead.
template <typename DT>
__device__ __forceinline__ df hp_bias(const float* a, const DT* __restrict__ W2, int V, int r, int v) {
  constexpr int UN = 16;                        // r % 16 == 0
  DdSum k0, k1, k2, k3;
  float perr = 0.f;
  float cur[UN];
#pragma unroll
  for (int u = 0; u < UN; ++u) cur[u] = ldf(W2 + (size_t)u * V + v);
  for (int i0 = 0; i0 < r; i0 += UN) {
    float nxt[UN];
    const bool more = i0 + UN < r;
#pragma unroll
    for (int u = 0; u < UN; ++u) nxt[u] = more ? ldf(W2 + (size_t)(i0 + UN + u) * V + v) : 0.f;
#pragma unroll
    for (int u = 0; u < UN; u += 4) {
      const float p0 = __fmul_rn(a[i0 + u], cur[u]), p1 = __fmul_rn(a[i0 + u + 1], cur[u + 1]);
      const float p2 = __fmul_rn(a[i0 + u + 2], cur[u + 2]), p3 = __fmul_rn(a[i0 + u + 3], cur[u + 3]);
      if constexpr (sizeof(DT) == 4) {
        perr += fmaf(a[i0 + u], cur[u], -p0) + fmaf(a[i0 + u + 1], cur[u + 1], -p1) +
                fmaf(a[i0 + u + 2], cur[u + 2], -p2) + fmaf(a[i0 + u + 3], cur[u + 3], -p3);
      }
      k0.add(p0);
      k1.add(p1);
      k2.add(p2);
      k3.add(p3);
    }
#pragma unroll
    for (int u = 0; u < UN; ++u) cur[u] = nxt[u];
  }
  df s = dd_add(dd_add(k0.value(), k1.value()), dd_add(k2.value(), k3.value()));
  if constexpr (sizeof(DT) == 4) s = dd_add_f(s, perr);
  return s;
}
// The same bias with the r x HPB slab of W2 columns staged in shared memory
// (`col` = v's column in the slab); 16 slab rows are loaded per batch.
template <typename DT>
__device__ __forceinline__ df hp_bias_slab(const float* a, const DT* slab, int r, int col) {
  constexpr int UN = 16;
  DdSum k0, k1, k2, k3;
  float perr = 0.f;
  for (int i0 = 0; i0 < r; i0 += UN) {
    float w[UN];
#pragma unroll
    for (int u = 0; u < UN; ++u) w[u] = tof(slab[(size_t)(i0 + u) * HPB + col]);
#pragma unroll
    for (int u = 0; u < UN; u += 4) {
      const float p0 = __fmul_rn(a[i0 + u], w[u]), p1 = __fmul_rn(a[i0 + u + 1], w[u + 1]);
      const float p2 = __fmul_rn(a[i0 + u + 2], w[u + 2]), p3 = __fmul_rn(a[i0 + u + 3], w[u + 3]);
      if constexpr (sizeof(DT) == 4) {
        perr += fmaf(a[i0 + u], w[u], -p0) + fmaf(a[i0 + u + 1], w[u + 1], -p1) +
                fmaf(a[i0 + u + 2], w[u + 2], -p2) + fmaf(a[i0 + u + 3], w[u + 3], -p3);
      }
      k0.add(p0);
      k1.add(p1);
      k2.add(p2);
      k3.add(p3);
    }
  }
  df s = dd_add(dd_add(k0.value(), k1.value()), dd_add(k2.value(), k3.value()));
  if constexpr (sizeof(DT) == 4) s = dd_add_f(s, perr);
  return s;
}
// Two adjacent slab entries widened to float (4- or 8-byte aligned).
__device__ __forceinline__ void slab2(const bf16* p, float& x, float& y) {
  const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
  x = __uint_as_float(w << 16);
  y = __uint_as_float(w & 0xffff0000u);
}
__device__ __forceinline__ void slab2(const float* p, float& x, float& y) {
  const float2 w = *reinterpret_cast<const float2*>(p);
  x = w.x;
  y = w.y;
}

// Transition biases of all HPB columns of a block whose W2 columns are staged
// in `slab` (r x HPB), one per thread (a CTA-wide call).  Thread t of each
// half of the CTA takes columns 2(t mod NT/2) and 2(t mod NT/2) + 1 (one
// two-column load per row) over half of the r rows, with four compensated
// chains per column; the two halves meet in `xch` (HPB double-floats).  `a`
// is W1[x] widened to float, 16-byte aligned.  Thread t returns column t.
template <typename DT>
__device__ __forceinline__ df hp_bias_block(const float* a, const DT* slab, int r, df* xch) {
  constexpr int H = NT / 2;
  static_assert(2 * H == HPB, "two columns per thread cover a block");
  const int c0 = 2 * (threadIdx.x % H), half = threadIdx.x / H;
  const int rh = r / 2;                         // r % 16 == 0
  DdSum k0[4], k1[4];
  float e0 = 0.f, e1 = 0.f;
  for (int i = half * rh; i < (half + 1) * rh; i += 4) {
    const float4 av = *reinterpret_cast<const float4*>(a + i);
    const float aa[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float w0, w1;
      slab2(slab + (size_t)(i + u) * HPB + c0, w0, w1);
      const float p0 = __fmul_rn(aa[u], w0), p1 = __fmul_rn(aa[u], w1);
      if constexpr (sizeof(DT) == 4) {
        e0 += fmaf(aa[u], w0, -p0);
        e1 += fmaf(aa[u], w1, -p1);
      }
      k0[u].add(p0);
      k1[u].add(p1);
    }
  }
  df s0 = dd_add(dd_add(k0[0].value(), k0[1].value()), dd_add(k0[2].value(), k0[3].value()));
  df s1 = dd_add(dd_add(k1[0].value(), k1[1].value()), dd_add(k1[2].value(), k1[3].value()));
  if constexpr (sizeof(DT) == 4) {
    s0 = dd_add_f(s0, e0);
    s1 = dd_add_f(s1, e1);
  }
  __syncthreads();                              // xch may still be read by the caller's last use
  if (half == 1) {
    xch[c0] = s0;
    xch[c0 + 1] = s1;
  }
  __syncthreads();
  if (half == 0) {
    xch[c0] = dd_add(xch[c0], s0);
    xch[c0 + 1] = dd_add(xch[c0 + 1], s1);
  }
  __syncthreads();
  return xch[threadIdx.x];
}

// Issue the cp.async copies of a block's r x HPB W2 columns into `slab`
// (waited for by hp_block), so they overlap the item's own loads.
template <typename DT>
__device__ __forceinline__ void hp_issue_slab(DT* slab, const DT* W2, int V, int r, int c0) {
  constexpr int E = 16 / sizeof(DT);
  const int cpr = HPB / E;
  for (int c = threadIdx.x; c < r * cpr; c += NT) {
    const int i = c / cpr, q = c - i * cpr;
    const int n = c0 + q * E;
    const bool valid = n < V;
    cp_async16(slab + (size_t)i * HPB + q * E, valid ? W2 + (size_t)i * V + n : W2, valid);
  }
  cp_async_commit();
}

// Draft weight exp((U[v] + bias) / T - shift_q) and target weight
// exp(t[v] / T - shift_p), unnormalised unless the shifts are the row's
// logsumexp.
template <typename DT>
__device__ __forceinline__ df hp_wq(const ItemCtx<DT>& c, df bias, int v, const df* tab) {
  const df l = dd_add(dd_mul(dd_add_f(bias, ldf(c.Urow + v)), c.invT), c.nsq);
  return dd_exp(l, tab);
}
template <typename DT>
__device__ __forceinline__ df hp_wp(const ItemCtx<DT>& c, int v, const df* tab) {
  const df l = dd_add(dd_mul_f(c.invT, ldf(c.Trow + v)), c.nsp);
  return dd_exp(l, tab);
}
// The same weights from preloaded logits (uq = U[v], tp = target[v]).
template <typename DT>
__device__ __forceinline__ df hp_wq_val(const ItemCtx<DT>& c, df bias, float uq, const df* tab) {
  return dd_exp(dd_add(dd_mul(dd_add_f(bias, uq), c.invT), c.nsq), tab);
}
template <typename DT>
__device__ __forceinline__ df hp_wp_val(const ItemCtx<DT>& c, float tp, const df* tab) {
  return dd_exp(dd_add(dd_mul_f(c.invT, tp), c.nsp), tab);
}

// Both weights of entry v for an item (zero beyond V; eq is zero for a bonus
// item, ep for a draft item).
template <typename DT>
__device__ __forceinline__ void hp_weights(const Shape& sh, const HpRows& R, const HpItem& it,
                                           const ItemCtx<DT>& c, const float* a, const df* tab,
                                           int v, df& eq, df& ep) {
  eq = {0.f, 0.f};
  ep = {0.f, 0.f};
  if (v >= sh.V) return;
  if (it.kind != HP_BONUS) eq = hp_wq<DT>(c, hp_bias<DT>(a, (const DT*)R.W2, sh.V, sh.r, v), v, tab);
  if (it.kind != HP_DRAFT) ep = hp_wp<DT>(c, v, tab);
}
// Weights of entry v = blk * HPB + threadIdx.x of a block whose W2 columns
// are staged in `slab` (r x HPB).
template <typename DT>
__device__ __forceinline__ void hp_weights_slab(const Shape& sh, const HpItem& it,
                                                const ItemCtx<DT>& c, const float* a,
                                                const DT* slab, const df* tab, int v, df& eq,
                                                df& ep) {
  eq = {0.f, 0.f};
  ep = {0.f, 0.f};
  if (v >= sh.V) return;
  if (it.kind != HP_BONUS) eq = hp_wq<DT>(c, hp_bias_slab<DT>(a, slab, sh.r, v % HPB), v, tab);
  if (it.kind != HP_DRAFT) ep = hp_wp<DT>(c, v, tab);
}

// max(0, ep / Zp - eq / Zq) given the reciprocals
__device__ __forceinline__ df hp_resid(df ep, df eq, df izp, df izq) {
  const df d = dd_add(dd_mul(ep, izp), dd_neg(dd_mul(eq, izq)));
  return d.hi > 0.f ? d : df{0.f, 0.f};
}

__device__ __forceinline__ void hp_table(df* tab) {
  if (threadIdx.x < DD_EXP_TAB) dd_exp_table_entry(tab, threadIdx.x);
}

// Chunk sums of one item: column col (0: the item's own weights -- p for a
// verify item, q for a draft item; 1: q of a verify item; 2: the residual),
// NC double-floats of CW columns each.
__device__ __forceinline__ float2* item_sums(const Ws& ws, const Shape& sh, int item, int col) {
  return ws.hpsum + ((size_t)item * ws.hp_cols + col) * sh.NC;
}
__device__ __forceinline__ df ld_sum(const float2* p) {
  const float2 v = __ldcg(p);
  return {v.x, v.y};
}
// Sum of sums[q0, q1) in order; the loads are issued eight at a time so the
// loop waits on one L2 round trip per eight entries, not per entry.
__device__ __forceinline__ df range_sum(const float2* sums, int q0, int q1) {
  df s = {0.f, 0.f};
  for (int q = q0; q < q1; q += 8) {
    float2 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = q + i < q1 ? __ldcg(sums + q + i) : make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 8; ++i) s = dd_add(s, df{v[i].x, v[i].y});
  }
  return s;
}
// Contiguous share [q0, q1) of NC entries for this thread.
__device__ __forceinline__ void thread_range(int NC, int& q0, int& q1) {
  const int per = (NC + NT - 1) / NT;
  q0 = min(NC, (int)threadIdx.x * per);
  q1 = min(NC, q0 + per);
}
// Sum over an item's chunk sums (fixed order: per-thread ranges, then the
// block reduction).
__device__ __forceinline__ df item_total(const float2* sums, int NC, float* shf) {
  int q0, q1;
  thread_range(NC, q0, q1);
  return block_sum_df(range_sum(sums, q0, q1), shf);
}
// Reciprocal of a positive double-float, computed once (thread 0) and shared.
__device__ __forceinline__ df shared_recip(df z, df* slot) {
  if (threadIdx.x == 0) {
    // one Newton step on the fp32 reciprocal: 1/z ~ h (2 - z h)
    const float h = __frcp_rn(z.hi);
    const df e = dd_add_f(dd_neg(dd_mul_f(z, h)), 1.0f);      // 1 - z h
    *slot = dd_add_f(dd_mul_f(e, h), h);
  }
  __syncthreads();
  const df r = *slot;
  __syncthreads();
  return r;
}

// Shared state of the re-decision bodies.
struct HpShared {
  df tab[DD_EXP_TAB];
  float shf[72];
  alignas(16) float a[256];
  df part[NT / 32][CW];
  df rc[2];
  df pref;
  int sel;
  int last;
  ItemCtx<float> cf;
  ItemCtx<bf16> cb;
  template <typename DT>
  __device__ ItemCtx<DT>* ctx() {
    if constexpr (sizeof(DT) == 4) return &cf; else return &cb;
  }
};

// One block (HPB columns) of an item: the weights of its columns and, per
// warp, the sum over the warp's CW columns -- phase 0: columns 0 and 1 (1 only
// for verify items), phase 1: the residual (column 2) given the normalisers.
template <typename DT>
__device__ void hp_block(const Shape& sh, const HpRows& R, const Ws& ws, int phase, int item,
                         int blk, const HpItem& it, HpShared& S, DT* slab) {
  // the first hpw_items items keep their weights from phase 0 (the residual
  // pass and the re-decision read them); the slab copies were issued by the
  // caller in phase 0
  const bool keep = item < ws.hpw_items;
  const bool stored = keep && phase == 1;
  __syncthreads();
  if (it.kind != HP_BONUS && !stored)
    for (int i = threadIdx.x; i < sh.r; i += NT) S.a[i] = ldf((const DT*)R.W1 + (size_t)it.prev * sh.r + i);
  cp_async_wait_all();
  __syncthreads();
  df izp = {0.f, 0.f}, izq = {0.f, 0.f};
  if (phase == 1) {
    const float4 nz = __ldcg(ws.hpnorm + item);
    izp = {nz.x, nz.y};
    izq = {nz.z, nz.w};
  }
  const ItemCtx<DT> c = item_ctx_shared<DT>(sh, R, it, S.template ctx<DT>());
  const int v = blk * HPB + threadIdx.x;
  const bool in = v < sh.V;
  df eq = {0.f, 0.f}, ep = {0.f, 0.f};
  float4* wslot = keep && in ? ws.hpw + (size_t)item * sh.V + v : nullptr;
  if (stored) {
    if (wslot) {
      const float4 w4 = __ldcg(wslot);
      eq = {w4.x, w4.y};
      ep = {w4.z, w4.w};
    }
  } else {
    // logits first, so their loads overlap the bias sums
    const float uq = (in && it.kind != HP_BONUS) ? ldf(c.Urow + v) : 0.f;
    const float tp = (in && it.kind != HP_DRAFT) ? ldf(c.Trow + v) : 0.f;
    const df bias = it.kind != HP_BONUS ? hp_bias_block<DT>(S.a, slab, sh.r, &S.part[0][0])
                                        : df{0.f, 0.f};
    if (in) {
      if (it.kind != HP_BONUS) eq = hp_wq_val<DT>(c, bias, uq, S.tab);
      if (it.kind != HP_DRAFT) ep = hp_wp_val<DT>(c, tp, S.tab);
    }
    if (wslot) *wslot = make_float4(eq.hi, eq.lo, ep.hi, ep.lo);
  }
  const int chunk = v / CW;                      // = blk * (HPB / CW) + warp
  const bool store = (threadIdx.x & 31) == 0 && chunk < sh.NC;
  if (phase == 0) {
    const df A = warp_sum_df(it.kind == HP_DRAFT ? eq : ep);
    if (store) item_sums(ws, sh, item, 0)[chunk] = make_float2(A.hi, A.lo);
    if (it.kind != HP_DRAFT) {
      const df Bq = warp_sum_df(eq);
      if (store) item_sums(ws, sh, item, 1)[chunk] = make_float2(Bq.hi, Bq.lo);
    }
  } else {
    const df rr = (v < sh.V) ? hp_resid(ep, eq, izp, izq) : df{0.f, 0.f};
    const df C = warp_sum_df(rr);
    if (store) item_sums(ws, sh, item, 2)[chunk] = make_float2(C.hi, C.lo);
  }
}

// Re-decide one item from its chunk sums: find the chunk where the running
// mass crosses u * Z, recompute that chunk's CW weights (the r products of each
// column split over the NT/32 warps) and scan them; write the token (and for
// a draft item q(x) and the row's logsumexp).
template <typename DT>
__device__ void hp_decide_item(const Shape& sh, const HpRows& R, const Ws& ws, int item, int* tokens,
                               float* q_tok, double* lse_q, int* out_tokens, uint32_t* status,
                               HpShared& S, DT* slab, uint32_t* redo = nullptr,
                               unsigned long long* st = nullptr) {
  // (st: optional globaltimer stamps of thread 0 at the steps below)
  unsigned long long* ts = (st && threadIdx.x == 0) ? st : nullptr;
  if (ts) ts[0] = globaltimer_ns();
  const HpItem it = ldcg_item(ws.items + item);
  const bool resid = it.kind == HP_RESID;
  // the item's constants (thread 0) and normalisers, requested now: the
  // scan's barrier publishes the former, the latter are used after the scan
  if (threadIdx.x == 0) *S.template ctx<DT>() = item_ctx<DT>(sh, R, it);
  const float4 nz = resid ? __ldcg(ws.hpnorm + item) : make_float4(0.f, 0.f, 0.f, 0.f);
  if (threadIdx.x == 0) S.sel = 0x7fffffff;
  // one scan of the chunk sums gives both the normaliser (its total) and the
  // per-thread prefixes; per-thread contiguous ranges of chunks, the first
  // eight sums of each kept in registers for the crossing search
  int q0, q1;
  thread_range(sh.NC, q0, q1);
  const float2* sums = item_sums(ws, sh, item, resid ? 2 : 0);
  float2 sv[8];
  auto load_range = [&]() -> df {
#pragma unroll
    for (int i = 0; i < 8; ++i) sv[i] = q0 + i < q1 ? __ldcg(sums + q0 + i) : make_float2(0.f, 0.f);
    df acc = {0.f, 0.f};                         // (in index order, as the search adds)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = dd_add(acc, df{sv[i].x, sv[i].y});
    for (int q = q0 + 8; q < q1; q += 8) {
      float2 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = q + i < q1 ? __ldcg(sums + q + i) : make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = dd_add(acc, df{v[i].x, v[i].y});
    }
    return acc;
  };
  df loc = load_range();
  if (ts) ts[1] = globaltimer_ns();
  df Z;
  df ex = block_scan1_df(loc, &Z, reinterpret_cast<float2*>(S.shf));
  if (ts) ts[2] = globaltimer_ns();
  // residual with no mass: draw from p (a probability-zero event)
  const bool use_r = resid && Z.hi > 0.f;
  if (resid && !use_r) {
    sums = item_sums(ws, sh, item, 0);
    loc = load_range();
    __syncthreads();                            // S.shf is read by every thread
    ex = block_scan1_df(loc, &Z, reinterpret_cast<float2*>(S.shf));
  }
  const df target = dd_mul_f(Z, it.u);
  int mine = -1;
  df mypref = {0.f, 0.f};
  if (q0 < q1 && dd_le(ex, target) && !dd_le(dd_add(ex, loc), target)) {
    df run = ex;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (mine < 0 && q0 + i < q1) {
        const df nx = dd_add(run, df{sv[i].x, sv[i].y});
        if (!dd_le(nx, target)) {
          mine = q0 + i;
          mypref = run;
        } else {
          run = nx;
        }
      }
    }
    for (int q = q0 + 8; q < q1 && mine < 0; q += 8) {
      float2 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = q + i < q1 ? __ldcg(sums + q + i) : make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (mine < 0 && q + i < q1) {
          const df nx = dd_add(run, df{v[i].x, v[i].y});
          if (!dd_le(nx, target)) {
            mine = q + i;
            mypref = run;
          } else {
            run = nx;
          }
        }
      }
    }
    if (mine >= 0) atomicMin(&S.sel, mine);
  }
  __syncthreads();
  if (mine >= 0 && mine == S.sel) S.pref = mypref;
  __syncthreads();
  if (S.sel == 0x7fffffff) {
    // rounding left the total at or below u*Z: last chunk with mass
    if (threadIdx.x == 0) {
      int q = sh.NC - 1;
      while (q > 0 && !(ld_sum(sums + q).hi > 0.f)) --q;
      df run = {0.f, 0.f};
      for (int t = 0; t < q; ++t) run = dd_add(run, ld_sum(sums + t));
      S.sel = q;
      S.pref = run;
    }
    __syncthreads();
  }
  if (ts) ts[3] = globaltimer_ns();
  const int n0 = S.sel * CW;
  df izp = {0.f, 0.f}, izq = {0.f, 0.f};
  if (use_r) {
    izp = {nz.x, nz.y};
    izq = {nz.z, nz.w};
  }
  // ---- the chunk's weights: kept from phase 0 for the first hpw_items items,
  // else the biases recomputed (warp w sums rows [w r/8, (w+1) r/8) of column lane)
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool kept = item < ws.hpw_items;
  if (it.kind != HP_BONUS && !kept) {
    for (int i = threadIdx.x; i < sh.r; i += NT) S.a[i] = ldf((const DT*)R.W1 + (size_t)it.prev * sh.r + i);
    stage_w2_slab<DT>(slab, (const DT*)R.W2, sh.V, 0, sh.r, n0, CW);
    const int kw = sh.r / (NT / 32);             // r % 16 == 0
    DdSum acc;
    float perr = 0.f;
    for (int i = w * kw; i < (w + 1) * kw; ++i) {
      const float wv = tof(slab[(size_t)i * CW + lane]);
      const float p = __fmul_rn(S.a[i], wv);
      if constexpr (sizeof(DT) == 4) perr += fmaf(S.a[i], wv, -p);
      acc.add(p);
    }
    df part = acc.value();
    if constexpr (sizeof(DT) == 4) part = dd_add_f(part, perr);
    S.part[w][lane] = part;
  }
  __syncthreads();
  if (ts) ts[4] = globaltimer_ns();
  const ItemCtx<DT> c = *S.template ctx<DT>();     // (written before the scan's barrier)
  if (w == 0) {
    const int v = n0 + lane;
    df eq = {0.f, 0.f}, ep = {0.f, 0.f};
    if (v < sh.V && kept) {
      const float4 w4 = __ldcg(ws.hpw + (size_t)item * sh.V + v);
      eq = {w4.x, w4.y};
      ep = {w4.z, w4.w};
    } else if (v < sh.V) {
      if (it.kind != HP_BONUS) {
        df bias = S.part[0][lane];
        for (int g = 1; g < NT / 32; ++g) bias = dd_add(bias, S.part[g][lane]);
        eq = hp_wq<DT>(c, bias, v, S.tab);
      }
      if (it.kind != HP_DRAFT) ep = hp_wp<DT>(c, v, S.tab);
    }
    df val;
    if (it.kind == HP_DRAFT) val = eq;
    else if (use_r) val = (v < sh.V) ? hp_resid(ep, eq, izp, izq) : df{0.f, 0.f};
    else val = ep;
    // inclusive double-float scan across the warp
    df inc = val;
    for (int d = 1; d < 32; d <<= 1) {
      const df o = shfl_up_df(inc, d);
      if (lane >= d) inc = dd_add(inc, o);
    }
    const df hi = dd_add(S.pref, inc), lo = dd_add(hi, dd_neg(val));
    const bool positive = val.hi > 0.f;
    const uint32_t cl = __ballot_sync(0xffffffffu, positive && dd_le(lo, target) && !dd_le(hi, target));
    const uint32_t pos = __ballot_sync(0xffffffffu, positive);
    // no crossing: rounding left the total at u*Z -> last positive entry
    const int t = cl ? __ffs(cl) - 1 : (pos ? 31 - __clz(pos) : 0);
    const float vt = __shfl_sync(0xffffffffu, val.hi, t);
    if (lane == 0) {
      const int tok = n0 + t;
      if (it.kind == HP_DRAFT) {
        const size_t o = (size_t)it.b * sh.gamma + it.j;
        tokens[o] = tok;
        q_tok[o] = __fdiv_rn(vt, Z.hi);
        lse_q[o] = it.shift_q + dd_log(Z, S.tab);
      } else {
        out_tokens[(size_t)it.b * (sh.gamma + 1) + it.j] = tok;
      }
      if (status) {
        atomicAdd(status + 1, 1u);
        if (tok != it.fast_token) {
          atomicAdd(status + 2, 1u);
          // a draft token that changes invalidates that request's later steps
          if (redo && it.kind == HP_DRAFT) atomicMax(redo, (uint32_t)(sh.gamma - it.j));
        }
        atomicOr(status, (uint32_t)SPEC_DEV_REFINED);
      }
    }
  }
  if (ts) ts[5] = globaltimer_ns();
  __syncthreads();
  if (ts) ts[6] = globaltimer_ns();
}

// Block sums of the n queued items (phase 0: weights, phase 1: residuals of
// residual items) over (item, block of HPB columns) units.  With `fused`, the
// CTA that completes an item's last block of its final pass (phase 0 for draft
// and bonus items, phase 1 for residual items) re-decides the item at once;
// the per-item counters start at zero and are left at zero.  Units are strided
// over the CTAs, or -- when `next` is given -- taken one at a time from the
// counter *next (unit = *next - base; every CTA makes one last, failing take),
// so CTAs that arrive early take more.  A changed draft token raises *redo to
// gamma - step.
template <typename DT>
__device__ void hp_sums_body(const Shape& sh, const HpRows& R, const Ws& ws, int phase, int n,
                             unsigned char* dsm, bool fused = false, int* tokens = nullptr,
                             float* q_tok = nullptr, double* lse_q = nullptr,
                             uint32_t* status = nullptr, int* out_tokens = nullptr,
                             uint32_t* next = nullptr, uint32_t base = 0, uint32_t* redo = nullptr) {
  DT* slab = reinterpret_cast<DT*>(dsm);        // [r][HPB] W2 columns of one block
  __shared__ HpShared S;
  __shared__ uint32_t s_unit;
  hp_table(S.tab);
  __syncthreads();
  const int total = n * sh.HB;
  for (int w = blockIdx.x;; w += gridDim.x) {
    if (next) {
      __syncthreads();
      if (threadIdx.x == 0) s_unit = atomicAdd(next, 1u) - base;
      __syncthreads();
      w = (int)min(s_unit, (uint32_t)total);
    }
    if (w >= total) break;
    const int item = w / sh.HB, blk = w - item * sh.HB;
    if (phase == 0) {
      __syncthreads();                          // the previous unit is done with the slab
      hp_issue_slab<DT>(slab, (const DT*)R.W2, sh.V, sh.r, blk * HPB);
    }
    const HpItem it = ldcg_item(ws.items + item);
    if (phase == 1 && it.kind != HP_RESID) continue;
    if (phase == 1 && item >= ws.hpw_items) {  // no kept weights: recompute the block
      __syncthreads();
      hp_issue_slab<DT>(slab, (const DT*)R.W2, sh.V, sh.r, blk * HPB);
    }
    hp_block<DT>(sh, R, ws, phase, item, blk, it, S, slab);
    if (fused) {
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0) S.last = atomicAdd(ws.hpcnt + item, 1u) == (uint32_t)sh.HB - 1u;
      __syncthreads();
      if (S.last) {
        __threadfence();
        if (it.kind == HP_RESID && phase == 0) {
          // both normalisers are complete: their reciprocals serve every block
          // of the residual pass and the re-decision
          const df izp = shared_recip(item_total(item_sums(ws, sh, item, 0), sh.NC, S.shf), &S.rc[0]);
          const df izq = shared_recip(item_total(item_sums(ws, sh, item, 1), sh.NC, S.shf), &S.rc[1]);
          if (threadIdx.x == 0) ws.hpnorm[item] = make_float4(izp.hi, izp.lo, izq.hi, izq.lo);
        }
        if ((it.kind == HP_RESID) == (phase == 1))
          hp_decide_item<DT>(sh, R, ws, item, tokens, q_tok, lse_q, out_tokens, status, S, slab, redo);
        if (threadIdx.x == 0) ws.hpcnt[item] = 0u;
      }
    }
  }
}

}  // namespace spec
