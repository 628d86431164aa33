// Tile of the rank-r transition bias  bias[m][n] = sum_i A[m][i] * W2[i][n0+n]
// (DSpark review, section 1.2, "Markov head": B(x_{k-1}, .) = W1[x_{k-1}] W2,
// A's rows being gathered W1 rows), staged in shared memory as fp32.
#pragma once

#include "spec_internal.cuh"

namespace spec {

// ---------------------------------------------------------------- cp.async
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
// 16-byte global -> shared copy; zero-fills when !valid (src is then not read).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::); }

// Stage W2[i0:i0+KC][c0:c0+NC] into shared memory (row stride NC elements);
// columns >= V are zero.  c0 and NC multiples of 16 bytes' worth of elements.
template <typename DT>
__device__ __forceinline__ void stage_w2_slab(DT* dst, const DT* W2, int V, int i0, int KC, int c0,
                                              int NC) {
  constexpr int E = 16 / sizeof(DT);
  const int cpr = NC / E;
  for (int c = threadIdx.x; c < KC * cpr; c += NT) {
    const int i = c / cpr, q = c - i * cpr;
    const int n = c0 + q * E;
    const bool valid = n < V;
    cp_async16(dst + (size_t)i * NC + q * E, valid ? W2 + (size_t)(i0 + i) * V + n : W2, valid);
  }
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();
}
// The same copies, issued only (the caller waits with cp_async_wait_all and
// __syncthreads before reading the slab).
template <typename DT>
__device__ __forceinline__ void issue_w2_slab(DT* dst, const DT* W2, int V, int i0, int KC, int c0,
                                              int NC) {
  constexpr int E = 16 / sizeof(DT);
  const int cpr = NC / E;
  for (int c = threadIdx.x; c < KC * cpr; c += NT) {
    const int i = c / cpr, q = c - i * cpr;
    const int n = c0 + q * E;
    const bool valid = n < V;
    cp_async16(dst + (size_t)i * NC + q * E, valid ? W2 + (size_t)(i0 + i) * V + n : W2, valid);
  }
  cp_async_commit();
}

// ---------------------------------------------------------------- warp MMA
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- shared layout
// Element strides are padded by 16 bytes so ldmatrix rows fall in distinct banks.
template <typename DT>
struct TileLayout {
  static constexpr int PAD = 16 / sizeof(DT);
  static constexpr int SS = BN + 4;                  // stage stride (floats)
  int BM, r, sa, sw, su;
  size_t offA, offW, offStage, offU, offT, total;
  __host__ __device__ TileLayout(int BM_, int r_, bool with_target) : BM(BM_), r(r_) {
    sa = r + PAD;
    sw = BN + PAD;
    su = BN + PAD;
    size_t szA = (size_t)BM * sa * sizeof(DT);
    size_t szW = (size_t)r * sw * sizeof(DT);
    size_t szS = (size_t)BM * SS * sizeof(float);
    size_t region0 = szA + szW > szS ? szA + szW : szS;
    offA = 0;
    offW = szA;
    offStage = 0;                                    // aliases A and W2 after the MMA
    offU = (region0 + 15) & ~(size_t)15;
    size_t szU = (size_t)BM * su * sizeof(DT);
    offT = offU + szU;
    total = offT + (with_target ? szU : 0);
  }
};

// Issue the cp.async copies of one tile's operands.
//   A rows   : W1[rowtok(m)][0:r]           (rows m >= nrows are zero)
//   W2 tile  : W2[0:r][n0:n0+BN]            (columns >= V are zero)
//   X rows   : X[rowoff(m) + n0 : ... + BN] for each extra tensor
template <typename DT>
__device__ __forceinline__ void load_A_rows(DT* As, int sa, const DT* W1, const int* tok, int nrows,
                                            int BM, int r) {
  const int cpr = r * (int)sizeof(DT) / 16;          // 16-byte chunks per row
  for (int c = threadIdx.x; c < BM * cpr; c += NT) {
    int m = c / cpr, q = c - m * cpr;
    bool valid = m < nrows;
    const DT* src = valid ? W1 + (size_t)tok[m] * r + q * (16 / sizeof(DT)) : W1;
    cp_async16(As + (size_t)m * sa + q * (16 / sizeof(DT)), src, valid);
  }
}
template <typename DT>
__device__ __forceinline__ void load_W2_tile(DT* Ws, int sw, const DT* W2, int V, int n0, int r) {
  constexpr int E = 16 / sizeof(DT);
  constexpr int CPR = BN / E;
  for (int c = threadIdx.x; c < r * CPR; c += NT) {
    int i = c / CPR, q = c - i * CPR;
    int n = n0 + q * E;
    bool valid = n < V;
    const DT* src = valid ? W2 + (size_t)i * V + n : W2;
    cp_async16(Ws + (size_t)i * sw + q * E, src, valid);
  }
}
// rows of a [rows][V] view starting at element offsets rowoff[m]
template <typename DT>
__device__ __forceinline__ void load_X_rows(DT* Xs, int su, const DT* X, const size_t* rowoff,
                                            int nrows, int BM, int V, int n0) {
  constexpr int E = 16 / sizeof(DT);
  constexpr int CPR = BN / E;
  for (int c = threadIdx.x; c < BM * CPR; c += NT) {
    int m = c / CPR, q = c - m * CPR;
    int n = n0 + q * E;
    bool valid = m < nrows && n < V;
    const DT* src = valid ? X + rowoff[m] + n : X;
    cp_async16(Xs + (size_t)m * su + q * E, src, valid);
  }
}

// ---------------------------------------------------------------- bias tile, tensor path
// 8 warps as (BM/32) x (8/(BM/32)); each warp computes 32 rows x (BN*BM/256) columns
// with m16n8k16 bf16 MMAs accumulating in fp32 over k = 0..r-1 in order.
template <int BM>
__device__ __forceinline__ void bias_tile_mma(const bf16* As, int sa, const bf16* Ws, int sw,
                                              int r, float* stage) {
  constexpr int WARPS_M = BM / 32, WARPS_N = 8 / WARPS_M, WTN = BN / WARPS_N, N8 = WTN / 8;
  constexpr int SS = TileLayout<bf16>::SS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wm = warp % WARPS_M, wn = warp / WARPS_M;
  float acc[2][N8][4];
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int b = 0; b < N8; ++b)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.f;
  for (int kk = 0; kk < r; kk += 16) {
    uint32_t af[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
      ldmatrix_x4(af[mt], As + (size_t)(wm * 32 + mt * 16 + (lane & 15)) * sa + kk + (lane >> 4) * 8);
#pragma unroll
    for (int n2 = 0; n2 < N8 / 2; ++n2) {
      uint32_t bq[4];
      ldmatrix_x4_trans(bq, Ws + (size_t)(kk + (lane & 7) + ((lane >> 3) & 1) * 8) * sw + wn * WTN +
                                n2 * 16 + (lane >> 4) * 8);
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        mma_bf16_16816(acc[mt][2 * n2], af[mt], bq[0], bq[1]);
        mma_bf16_16816(acc[mt][2 * n2 + 1], af[mt], bq[2], bq[3]);
      }
    }
  }
  __syncthreads();   // all warps done reading A / W2 before the stage overwrites them
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < N8; ++nt) {
      int row = wm * 32 + mt * 16 + (lane >> 2);
      int col = wn * WTN + nt * 8 + (lane & 3) * 2;
      stage[row * SS + col] = acc[mt][nt][0];
      stage[row * SS + col + 1] = acc[mt][nt][1];
      stage[(row + 8) * SS + col] = acc[mt][nt][2];
      stage[(row + 8) * SS + col + 1] = acc[mt][nt][3];
    }
}

// ---------------------------------------------------------------- bias tile, SIMT path
// Thread t owns column t % BN and rows t / BN, t / BN + 2, ...; fp32 FMAs in k order.
template <typename DT, int BM>
__device__ __forceinline__ void bias_tile_simt(const DT* As, int sa, const DT* Ws, int sw, int r,
                                               float* stage) {
  constexpr int RPT = BM * BN / NT;        // rows per thread
  constexpr int SS = TileLayout<DT>::SS;
  const int col = threadIdx.x % BN, r0 = threadIdx.x / BN;
  float acc[RPT];
#pragma unroll
  for (int q = 0; q < RPT; ++q) acc[q] = 0.f;
  for (int i = 0; i < r; ++i) {
    float w = tof(Ws[(size_t)i * sw + col]);
#pragma unroll
    for (int q = 0; q < RPT; ++q) acc[q] = fmaf(tof(As[(size_t)(r0 + 2 * q) * sa + i]), w, acc[q]);
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < RPT; ++q) stage[(r0 + 2 * q) * SS + col] = acc[q];
}

template <typename DT, int BM, bool SIMT>
__device__ __forceinline__ void bias_tile(const DT* As, int sa, const DT* Ws, int sw, int r,
                                          float* stage) {
  if constexpr (SIMT || sizeof(DT) == 4) {
    bias_tile_simt<DT, BM>(As, sa, Ws, sw, r, stage);
  } else {
    bias_tile_mma<BM>(reinterpret_cast<const bf16*>(As), sa, reinterpret_cast<const bf16*>(Ws), sw,
                      r, stage);
  }
}

// ---------------------------------------------------------------- group helpers
// TPR consecutive lanes share one tile row in the epilogues.
template <int TPR>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int m = TPR / 2; m; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}
template <int TPR>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int m = TPR / 2; m; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}
template <int TPR>
__device__ __forceinline__ df group_sum_df(df v) {
#pragma unroll
  for (int m = TPR / 2; m; m >>= 1) v = df_add(v, shfl_xor_df(v, m));
  return v;
}

// Kahan-compensated running sum (non-negative terms)
struct Kahan {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    float y = __fsub_rn(x, c);
    float t = __fadd_rn(s, y);
    c = __fsub_rn(__fsub_rn(t, s), y);
    s = t;
  }
  __device__ __forceinline__ df value() const { return {s, -c}; }
};

}  // namespace spec
