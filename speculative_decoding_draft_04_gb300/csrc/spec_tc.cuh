// Fifth-generation tensor-core (tcgen05) path for the rank-r bias tile:
// D[128 x 128] (fp32, in tensor memory) = A[128 x r] * W2[r x 128], bf16 inputs.
//
//   A  = gathered W1 rows, K-major, 128-byte swizzle: r/64 "K atoms" of
//        128 rows x 128 bytes; 16-byte chunk c of row m sits at chunk c ^ (m % 8).
//   W2 = the [r][V] projection read in place (N contiguous: MN-major operand),
//        128-byte swizzle: two "MN atoms" of 64 columns, each r rows x 128 bytes,
//        chunk c of row k at chunk c ^ (k % 8).  Canonical MN-major layout:
//        8-row K groups 1024 bytes apart (SBO), MN atoms r*128 bytes apart (LBO).
//
// One thread issues r/16 MMAs (M=128, N=128, K=16 each) and commits them to an
// mbarrier; every wait on it is bounded and reports SPEC_DEV_TIMEOUT instead
// of hanging.  Every swizzle atom is 1024-byte aligned in shared memory.
#pragma once

#include "spec_gemm.cuh"

namespace spec {

constexpr int TC_M = 128, TC_N = BN;        // tile of one tcgen05 MMA group
constexpr uint32_t TC_TMEM_COLS = 128;      // fp32 accumulator columns

struct TcLayout {
  int r, ka;                      // K atoms of 64 elements
  size_t offA, offW, offStage, offU, offT, offBar, total;
  __host__ __device__ TcLayout(int r_, bool with_target) : r(r_) {
    ka = r / 64;
    offA = 0;                                           // ka * 16 KB
    offW = (size_t)ka * 16384;                          // 2 * r * 128 bytes
    size_t ab = offW + (size_t)2 * r * 128;
    size_t stage = (size_t)TC_M * TileLayout<bf16>::SS * 4;
    offStage = 0;                                       // aliases A/W2 after the MMA
    size_t region0 = ab > stage ? ab : stage;
    offU = (region0 + 1023) & ~(size_t)1023;
    size_t szU = (size_t)TC_M * (BN + 8) * sizeof(bf16);
    offT = offU + szU;
    offBar = offT + (with_target ? szU : 0);
    offBar = (offBar + 15) & ~(size_t)15;
    total = offBar + 16 + 1024;                         // + slack to align the base to 1 KB
  }
};

// Advance a shared-memory pointer to the next 1024-byte boundary of the
// shared window.
__device__ __forceinline__ unsigned char* align1k(unsigned char* p) {
  const uint32_t s = smem_u32(p);
  return p + ((1024u - (s & 1023u)) & 1023u);
}

// ---------------------------------------------------------------- operand loads
__device__ __forceinline__ void tc_load_A(bf16* As, const bf16* W1, const int* tok, int nrows, int r) {
  const int cpr = r / 8;                                 // 16-byte chunks per row
  for (int q = threadIdx.x; q < TC_M * cpr; q += NT) {
    const int m = q / cpr, j = q - m * cpr;
    const int a = j >> 3, c = j & 7;
    const bool valid = m < nrows;
    const bf16* src = valid ? W1 + (size_t)tok[m] * r + j * 8 : W1;
    unsigned char* dst = reinterpret_cast<unsigned char*>(As) + (size_t)a * 16384 + m * 128 +
                         ((c ^ (m & 7)) << 4);
    cp_async16(dst, src, valid);
  }
}
__device__ __forceinline__ void tc_load_W2(bf16* Ws, const bf16* W2, int V, int n0, int r) {
  for (int q = threadIdx.x; q < r * 16; q += NT) {
    const int k = q >> 4, j = q & 15;
    const int a = j >> 3, c = j & 7;
    const int n = n0 + j * 8;
    const bool valid = n < V;
    const bf16* src = valid ? W2 + (size_t)k * V + n : W2;
    unsigned char* dst = reinterpret_cast<unsigned char*>(Ws) + (size_t)a * r * 128 + k * 128 +
                         ((c ^ (k & 7)) << 4);
    cp_async16(dst, src, valid);
  }
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor: start, leading / stride byte offsets,
// descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t tc_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// Instruction descriptor, kind::f16: D fp32, A and B bf16, A K-major,
// B MN-major, M = 128, N = n (a multiple of 16 up to 256).
__device__ __forceinline__ uint32_t tc_idesc_n(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(TC_M >> 4) << 24);
}
__device__ __forceinline__ uint32_t tc_idesc() { return tc_idesc_n(TC_N); }

// ---------------------------------------------------------------- primitives
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::);
}
// Bounded wait for phase `parity` to complete; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t max_iter) {
  const uint32_t a = smem_u32(bar);
  for (uint32_t it = 0; it < max_iter; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(a), "r"(parity));
    if (done) return true;
    if (it > 64) __nanosleep(32);
  }
  return false;
}
__device__ __forceinline__ void tc_alloc(uint32_t* holder, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                   smem_u32(holder)),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::);
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols));
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::);
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::); }
__device__ __forceinline__ void fence_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::);
}
__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum));
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
          smem_u32(bar)));
}
// 32 consecutive fp32 columns of this thread's lane, without waiting: the
// registers are valid after tc_wait_ld().  The outputs are bound to the array
// elements as fp32 registers (a b32 destination accepts any 32-bit register),
// so the array stays in registers.
__device__ __forceinline__ void tc_ld32_issue(uint32_t taddr, float (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
        "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]),
        "=f"(v[14]), "=f"(v[15]), "=f"(v[16]), "=f"(v[17]), "=f"(v[18]), "=f"(v[19]), "=f"(v[20]),
        "=f"(v[21]), "=f"(v[22]), "=f"(v[23]), "=f"(v[24]), "=f"(v[25]), "=f"(v[26]), "=f"(v[27]),
        "=f"(v[28]), "=f"(v[29]), "=f"(v[30]), "=f"(v[31])
      : "r"(taddr));
}
// 8 consecutive fp32 columns of this thread's lane, without waiting.
__device__ __forceinline__ void tc_ld8_issue(uint32_t taddr, float (&v)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
                 "=f"(v[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
// 32 consecutive fp32 columns of this thread's lane
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::);
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------- the tile
// Preconditions: A and W2 staged (cp.async complete, fence.proxy.async issued,
// CTA synchronised), TMEM allocated at `taddr`, `bar` initialised and
// `parity` the phase this commit will complete.
// Writes the 128 x 128 fp32 tile to `stage` (row stride SS floats), which may
// alias A and W2.  Returns false (and leaves `stage` unspecified) if the MMA
// did not complete within the bound.
__device__ __forceinline__ bool bias_tile_tc(const bf16* As, const bf16* Ws, int r, uint32_t taddr,
                                             uint64_t* bar, uint32_t parity, float* stage) {
  constexpr int SS = TileLayout<bf16>::SS;
  if (threadIdx.x == 0) {
    tc_fence_after();
    const uint32_t a0 = smem_u32(As), w0 = smem_u32(Ws);
    const uint32_t idesc = tc_idesc();
    for (int kk = 0; kk < r; kk += 16) {
      const uint64_t ad = tc_sdesc(a0 + (uint32_t)((kk >> 6) * 16384 + (kk & 63) * 2), 16, 1024);
      const uint64_t bd = tc_sdesc(w0 + (uint32_t)(kk * 128), (uint32_t)(r * 128), 1024);
      tc_mma(taddr, ad, bd, idesc, kk > 0 ? 1u : 0u);
    }
    tc_commit(bar);
  }
  __syncwarp();
  const bool ok = mbar_wait(bar, parity, 1u << 22);
  tc_fence_after();
  // all threads must agree before the operands are overwritten
  const bool all_ok = __syncthreads_and(ok ? 1 : 0);
  if (!all_ok) return false;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = w & 3, half = w >> 2;
  const int row = 32 * q + lane;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    float v[32];
    tc_ld32(taddr + ((uint32_t)(32 * q) << 16) + (uint32_t)(64 * half + 32 * i), v);
#pragma unroll
    for (int c = 0; c < 32; ++c) stage[row * SS + 64 * half + 32 * i + c] = v[c];
  }
  tc_fence_before();
  return true;
}

}  // namespace spec
