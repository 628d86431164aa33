// Host side of the C ABI (include/spec.h): argument validation, workspace
// layout, launch sequencing on the caller's stream, options and per-stage
// event timing.  No device memory is ever allocated here.
#include <mutex>
#include <vector>

#include "spec_internal.cuh"

namespace spec {

// launchers (spec_draft.cu, spec_verify.cu, spec_refine.cu, spec_sched.cu)
template <typename DT>
cudaError_t launch_draft_persistent(const Shape&, const void*, const void*, const void*, const int*,
                                    const float*, const float*, int*, float*, double*, float*,
                                    uint32_t*, const Ws&, const Eps&, int, int, cudaStream_t,
                                    const RnnParams*, int);
cudaError_t launch_draft_slice(const Shape&, const void*, const void*, const void*, const int*,
                               const float*, const float*, int*, float*, double*, float*, uint32_t*,
                               const Ws&, const Eps&, int, cudaStream_t, int);
int slice_chunks(const Shape&, int);
cudaError_t launch_verify_slice(const Shape&, const bf16*, const bf16*, const bf16*, const bf16*, const Ws&,
                                uint32_t*, int, cudaStream_t);
int vslice_chunks(const Shape&, int);
template <typename DT>
cudaError_t launch_verify_redecide(const Shape&, const HpRows&, const Ws&, int*, uint32_t*, int, cudaStream_t);
cudaError_t launch_verify_prep(const Shape&, const int*, const float*, const int*, const double*,
                               const int*, const Ws&, uint32_t*, int*, int*, float*, float*,
                               cudaStream_t);
template <typename DT>
cudaError_t launch_target_stats(const Shape&, const void*, const float*, const int*, const Ws&,
                                cudaStream_t);
template <typename DT>
cudaError_t launch_verify_tile(const Shape&, const void*, const void*, const void*, const void*,
                               const Ws&, int, uint32_t*, cudaStream_t);
template <typename DT>
cudaError_t launch_verify_final(const Shape&, const void*, const void*, const void*, const void*,
                                const int*, const float*, const int*, const float*, const double*,
                                const int*, const float*, const float*, int*, int*, float*, float*,
                                float*, uint32_t*, const Ws&, const Eps&, cudaStream_t);
template <typename DT>
cudaError_t launch_hp_sums(const Shape&, const HpRows&, const Ws&, int, int*, uint32_t*, int, cudaStream_t);
template <typename DT>
cudaError_t launch_slow_verify(const Shape&, const HpRows&, const Ws&, const int*, const int*,
                               const double*, const int*, const float*, const float*, int*, int*,
                               uint32_t*, int, cudaStream_t);
template <typename DT>
cudaError_t launch_confidence(int, int, int, int, int, const void*, const void*, const float*,
                              const int*, const int*, float*, uint32_t*, cudaStream_t);
cudaError_t launch_schedule_rank(int, int, const float*, float*, int*, unsigned long long*, uint32_t*,
                                 cudaStream_t);
cudaError_t launch_schedule_select(int, int, const double*, int, const int*, const unsigned long long*,
                                   int*, long long*, double*, cudaStream_t);

cudaError_t launch_tree_select(int, int, int, const int*, const float*, int, float*, uint8_t*, float*,
                               uint32_t*, cudaStream_t);
size_t tree_workspace_bytes(const TreeShape&);
template <typename DT>
cudaError_t launch_tree_draft(const TreeShape&, const void*, const void*, const void*, const int*,
                              const float*, const int*, const uint8_t*, const float*, int*, float*, void*,
                              uint32_t*, cudaStream_t);
template <typename DT>
cudaError_t launch_tree_verify(const TreeShape&, const void*, const void*, const void*, const void*,
                               const int*, const float*, const int*, const uint8_t*, const int*,
                               const float*, const float*, int*, int*, int*, void*, uint32_t*,
                               cudaStream_t);

// ---------------------------------------------------------------- options
namespace {
std::mutex g_mu;
double g_eps_scale = 1.0;
bool g_force_simt = false;
int g_bias_path = 2;          // 1 warp MMA, 2 tcgen05 (see SPEC_OPT_BIAS_PATH)
bool g_trace = false;         // SPEC_OPT_TRACE
bool g_perturb = false;       // SPEC_OPT_PERTURB (test build of the draft kernels)
bool g_stall = false;         // SPEC_OPT_TEST_STALL (test build of the draft kernels)
int g_draft_kernel = 0;       // SPEC_OPT_DRAFT_KERNEL: 0 slice-resident where it fits, 1 tile-strided
int g_verify_kernel = 0;      // SPEC_OPT_VERIFY_KERNEL: 0 slice-resident tiles where they fit, 1 tile-strided

// Band constants (probability units) of the certified first-pass decisions.
// Largest first-pass margin error seen against the float64 oracle over C0-C4
// (about 4.3k draft and 1k final draws): 3.8e-8 absolute, at most
// 1.4e-7 x sqrt(sum q^2) and 1.1e-7 x sqrt(sum slice mass^2), and never more
// than 3.5% of the whole band the constants 7e-7 / 7e-7 / 1.5e-7 gave.  The
// halved constants keep the largest error under 7.1% of the band (a factor
// above 14); a wider band only sends more draws to the re-decision.
constexpr float EPS_ELEM = 3.5e-7f;
constexpr float EPS_SLICE = 3.5e-7f;
constexpr float EPS_ABS = 1.0e-9f;
constexpr float EPS_RATIO = 1.0e-6f;
constexpr float EPS_NORM = 7.5e-8f;

Eps current_eps() {
  std::lock_guard<std::mutex> lk(g_mu);
  Eps e;
  e.elem = EPS_ELEM;
  e.slice = EPS_SLICE;
  e.abs_ = EPS_ABS;
  e.ratio = EPS_RATIO;
  e.norm = EPS_NORM;
  e.scale = (float)g_eps_scale;
  return e;
}

// ---------------------------------------------------------------- profiling
enum Stage {
  ST_DRAFT_PERSISTENT, ST_DRAFT_SLICE, ST_VERIFY_PREP,
  ST_TARGET_STATS, ST_VERIFY_TILE, ST_VERIFY_SLICE, ST_VERIFY_FINAL, ST_SLOW_VERIFY, ST_VERIFY_HP_SUMS,
  ST_VERIFY_HP_RESID, ST_VERIFY_REDECIDE, ST_CONFIDENCE, ST_SCHED_RANK, ST_SCHED_SELECT, ST_TREE_SELECT,
  ST_TREE_DRAFT, ST_TREE_VERIFY, ST_COUNT
};
const char* kStageNames[ST_COUNT] = {
    "draft_persistent", "draft_slice", "verify_prep",
    "target_stats", "verify_tile", "verify_slice", "verify_final", "slow_verify", "verify_hp_sums",
    "verify_hp_resid", "verify_redecide", "confidence", "sched_rank", "sched_select", "tree_select",
    "tree_draft", "tree_verify"};
bool g_prof = false;
struct EvPair { cudaEvent_t a, b; int stage; };
std::vector<EvPair> g_pending;
std::vector<cudaEvent_t> g_pool;

cudaEvent_t get_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Records events around one launch when profiling is on.
struct ProfScope {
  cudaStream_t st;
  int stage;
  cudaEvent_t a = nullptr;
  bool on;
  ProfScope(cudaStream_t s, int sg) : st(s), stage(sg) {
    std::lock_guard<std::mutex> lk(g_mu);
    on = g_prof;
    if (on) {
      a = get_event();
      cudaEventRecord(a, st);
    }
  }
  ~ProfScope() {
    if (!on) return;
    std::lock_guard<std::mutex> lk(g_mu);
    cudaEvent_t b = get_event();
    cudaEventRecord(b, st);
    g_pending.push_back({a, b, stage});
  }
};

// SM count of the current device, cached per device ordinal: the cooperative
// draft sizes its grid from it, so a process that drives devices with
// different SM counts gets each device's own figure.  0 when the device
// cannot be queried (the launch then fails with SPEC_ECUDA).
constexpr int kMaxSmDevices = 64;
int g_num_sms[kMaxSmDevices] = {};
int num_sms() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev >= kMaxSmDevices) {
    int n = 0;
    return cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess ? n : 0;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_num_sms[dev] <= 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 0;
    g_num_sms[dev] = n;
  }
  return g_num_sms[dev];
}
int grid_for_refine() { return 2 * num_sms(); }

// ---------------------------------------------------------------- workspace
// Residual re-decisions whose weights are kept between their two passes.
constexpr int kHpwItems = 16;
struct Layout {
  size_t ctrl, trace, items, hpsum, hpcnt, hpw, hpnorm, rnnst, dpart, abuf, rowptr, prow, prevtok, vflags, lse_p,
      bpart, vpart, slow, accbits, rowc, rowp, total;
  int max_items, item_cap, hpw_items;
};

Layout layout(const Shape& sh) {
  Layout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = (off + bytes + 255) & ~(size_t)255;
    return o;
  };
  const size_t B = sh.B, g = sh.gamma;
  L.max_items = sh.B;
  L.item_cap = sh.B * sh.gamma;
  L.ctrl = take(CTRL_WORDS * sizeof(uint32_t));
  L.trace = take(2 * MAX_GAMMA * TRACE_SLOTS * sizeof(unsigned long long));
  L.items = take((size_t)L.item_cap * sizeof(HpItem));
  L.hpsum = take((size_t)L.max_items * 3 * sh.NC * sizeof(float2));
  L.hpcnt = take((size_t)L.max_items * sizeof(uint32_t));
  L.hpw_items = sh.B < kHpwItems ? sh.B : kHpwItems;
  L.hpw = take((size_t)L.hpw_items * sh.V * sizeof(float4));
  L.hpnorm = take((size_t)L.max_items * sizeof(float4));
  L.rnnst = take((size_t)(sh.gamma + 1) * sh.B * sh.r * sizeof(float));   // RNN head states
  L.dpart = take(B * sh.NC * sizeof(float4));
  L.abuf = take((size_t)(sh.B < 128 ? sh.B : 128) * sh.r * 4);
  L.rowptr = take((B + 1) * sizeof(int));
  L.prow = take(B * g * sizeof(int2));
  L.prevtok = take(B * g * sizeof(int));
  L.vflags = take(B * sizeof(int));
  L.lse_p = take(B * (g + 1) * sizeof(double));
  L.bpart = take(B * sh.NSV * sizeof(float4));
  L.vpart = take(B * g * sh.NSV * sizeof(float4));
  L.slow = take(B * sizeof(int));
  L.accbits = take(B * sizeof(uint32_t));
  L.rowc = take(B * g * sizeof(float4));
  L.rowp = take(B * (g + 1) * sizeof(float2));
  L.total = off;
  return L;
}

Ws views(const Layout& L, void* base) {
  unsigned char* p = static_cast<unsigned char*>(base);
  Ws w;
  w.ctrl = reinterpret_cast<uint32_t*>(p + L.ctrl);
  w.trace = nullptr;
  w.items = reinterpret_cast<HpItem*>(p + L.items);
  w.max_items = L.max_items;
  w.item_cap = L.item_cap;
  w.hpsum = reinterpret_cast<float2*>(p + L.hpsum);
  w.hp_cols = 3;
  w.hpcnt = reinterpret_cast<uint32_t*>(p + L.hpcnt);
  w.hpw = reinterpret_cast<float4*>(p + L.hpw);
  w.hpw_items = L.hpw_items;
  w.hpnorm = reinterpret_cast<float4*>(p + L.hpnorm);
  w.dpart = reinterpret_cast<float4*>(p + L.dpart);
  w.abuf = p + L.abuf;
  w.rowptr = reinterpret_cast<int*>(p + L.rowptr);
  w.prow = reinterpret_cast<int2*>(p + L.prow);
  w.prevtok = reinterpret_cast<int*>(p + L.prevtok);
  w.vflags = reinterpret_cast<int*>(p + L.vflags);
  w.lse_p = reinterpret_cast<double*>(p + L.lse_p);
  w.bpart = reinterpret_cast<float4*>(p + L.bpart);
  w.vpart = reinterpret_cast<float4*>(p + L.vpart);
  w.slow = reinterpret_cast<int*>(p + L.slow);
  w.accbits = reinterpret_cast<uint32_t*>(p + L.accbits);
  w.rowc = reinterpret_cast<float4*>(p + L.rowc);
  w.rowp = reinterpret_cast<float2*>(p + L.rowp);
  return w;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

int check_shape(int B, int gamma, int V, int r, int dtype) {
  if (B < 1 || B > 4096 || gamma < 1 || V < 16 || V >= (1 << 24) || r < 1) return SPEC_EINVAL;
  if (gamma > MAX_GAMMA) return SPEC_EUNSUPPORTED;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_EUNSUPPORTED;
  if (V % 8 != 0) return SPEC_EUNSUPPORTED;
  if (r % 16 != 0) return SPEC_EUNSUPPORTED;
  if (dtype == SPEC_BF16 && r > 256) return SPEC_EUNSUPPORTED;
  if (dtype == SPEC_F32 && r > 64) return SPEC_EUNSUPPORTED;
  return SPEC_OK;
}

Shape make_shape(int B, int gamma, int V, int r) {
  Shape s;
  s.B = B;
  s.gamma = gamma;
  s.V = V;
  s.r = r;
  s.NS = (V + BN - 1) / BN;
  s.NC = (V + CW - 1) / CW;
  s.NSV = (V + VB - 1) / VB;
  s.HB = (V + HPB - 1) / HPB;
  s.rnn = 0;
  s.NA = V;
  return s;
}

#define SPEC_TRY(x)                         \
  do {                                      \
    if ((x) != cudaSuccess) return SPEC_ECUDA; \
  } while (0)

// The whole draft: one cooperative launch (the control words are zeroed first
// on the same stream; the grid barrier counts on it).
// The slice-resident kernel (spec_draft_slice.cu) runs the Markov head on the
// tensor path when the shape fits it (B <= 128, V <= 256 columns per SM);
// otherwise, and for the RNN head, the tile-strided kernel (spec_draft.cu).
template <typename DT>
int launch_draft(const spec_draft_args* a, const Shape& sh, const Ws& ws, cudaStream_t st,
                 const RnnParams* rnn = nullptr) {
  int path, hook, kernel;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    path = g_force_simt ? 0 : g_bias_path;
    hook = g_perturb ? HOOK_PERTURB : (g_stall ? HOOK_STALL : HOOK_NONE);
    kernel = g_draft_kernel;
  }
  const int nsm = num_sms();
  if (nsm <= 0) return SPEC_ECUDA;
  SPEC_TRY(cudaMemsetAsync(a->dev_status, 0, 4 * sizeof(uint32_t), st));
  SPEC_TRY(cudaMemsetAsync(ws.ctrl, 0, CTRL_WORDS * sizeof(uint32_t), st));
  SPEC_TRY(cudaMemsetAsync(ws.hpcnt, 0, (size_t)ws.max_items * sizeof(uint32_t), st));
  const Eps eps = current_eps();
  if constexpr (sizeof(DT) == 2) {
    if (path == 2 && !rnn && kernel == 0 && slice_chunks(sh, nsm) > 0) {
      ProfScope p(st, ST_DRAFT_SLICE);
      const cudaError_t e = launch_draft_slice(sh, a->U, a->W1, a->W2, a->anchor, a->temperature,
                                               a->u_draft, a->draft_tokens, a->q_tok, a->lse_q, a->diag,
                                               a->dev_status, ws, eps, nsm, st, hook);
      if (e == cudaSuccess) return SPEC_OK;
      if (e != cudaErrorNotSupported) return SPEC_ECUDA;
    }
  }
  ProfScope p(st, ST_DRAFT_PERSISTENT);
  SPEC_TRY(launch_draft_persistent<DT>(sh, a->U, a->W1, a->W2, a->anchor, a->temperature, a->u_draft,
                                       a->draft_tokens, a->q_tok, a->lse_q, a->diag, a->dev_status,
                                       ws, eps, path, nsm, st, rnn, hook));
  return SPEC_OK;
}

template <typename DT>
int run_rnn_draft(const spec_rnn_draft_args* ra, cudaStream_t st) {
  const spec_draft_args* a = &ra->draft;
  Shape sh = make_shape(a->B, a->gamma, a->V, a->r);
  sh.rnn = 1;
  sh.NA = a->gamma * a->B;
  const Layout L = layout(sh);
  Ws ws = views(L, a->workspace);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_trace)
      ws.trace = reinterpret_cast<unsigned long long*>(static_cast<unsigned char*>(a->workspace) + L.trace);
  }
  RnnParams rp;
  rp.Wr = ra->Wr;
  rp.hproj = ra->hproj;
  rp.arows = ra->a_rows;
  rp.state = static_cast<unsigned char*>(a->workspace) + L.rnnst;
  return launch_draft<DT>(a, sh, ws, st, &rp);
}

template <typename DT>
int run_draft(const spec_draft_args* a, cudaStream_t st) {
  const Shape sh = make_shape(a->B, a->gamma, a->V, a->r);
  const Layout L = layout(sh);
  Ws ws = views(L, a->workspace);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_trace)
      ws.trace = reinterpret_cast<unsigned long long*>(static_cast<unsigned char*>(a->workspace) + L.trace);
  }
  return launch_draft<DT>(a, sh, ws, st);
}

template <typename DT>
int run_verify(const spec_verify_args* a, cudaStream_t st) {
  Shape sh = make_shape(a->B, a->gamma, a->V, a->r);
  if (a->a_rows) {                 // RNN head: factor rows from the draft
    sh.rnn = 1;
    sh.NA = a->gamma * a->B;
  }
  const void* F = a->a_rows ? a->a_rows : a->W1;
  const Layout L = layout(sh);
  Ws ws = views(L, a->workspace);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_trace)
      ws.trace = reinterpret_cast<unsigned long long*>(static_cast<unsigned char*>(a->workspace) + L.trace);
  }
  const Eps eps = current_eps();
  int path, vkernel;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    path = g_force_simt ? 0 : g_bias_path;
    vkernel = g_verify_kernel;
  }
  const int nsm = num_sms();
  const int grid = grid_for_refine();
  if (grid <= 0) return SPEC_ECUDA;
  HpRows R{a->target, a->U, F, a->W2, a->temperature};
  SPEC_TRY(cudaMemsetAsync(a->dev_status, 0, 4 * sizeof(uint32_t), st));
  {
    ProfScope p(st, ST_VERIFY_PREP);
    SPEC_TRY(launch_verify_prep(sh, a->anchor, a->temperature, a->draft_tokens, a->lse_q,
                                a->verify_len, ws, a->dev_status, a->accept_len, a->out_tokens,
                                a->alpha, a->p_tok, st));
  }
  {
    ProfScope p(st, ST_TARGET_STATS);
    SPEC_TRY(launch_target_stats<DT>(sh, a->target, a->temperature, a->verify_len, ws, st));
  }
  bool sliced = false;
  if constexpr (sizeof(DT) == 2) {
    if (path == 2 && vkernel == 0 && vslice_chunks(sh, nsm) > 0) {
      ProfScope p(st, ST_VERIFY_SLICE);
      const cudaError_t e = launch_verify_slice(sh, (const bf16*)a->target, (const bf16*)a->U, (const bf16*)F,
                                                (const bf16*)a->W2, ws, a->dev_status, nsm, st);
      if (e != cudaSuccess && e != cudaErrorNotSupported) return SPEC_ECUDA;
      sliced = e == cudaSuccess;
    }
  }
  if (!sliced) {
    ProfScope p(st, ST_VERIFY_TILE);
    SPEC_TRY(launch_verify_tile<DT>(sh, a->target, a->U, F, a->W2, ws, path, a->dev_status, st));
  }
  {
    ProfScope p(st, ST_VERIFY_FINAL);
    SPEC_TRY(launch_verify_final<DT>(sh, a->target, a->U, F, a->W2, a->anchor, a->temperature,
                                     a->draft_tokens, a->q_tok, a->lse_q, a->verify_len,
                                     a->u_accept, a->u_final, a->accept_len, a->out_tokens,
                                     a->alpha, a->p_tok, a->diag, a->dev_status, ws, eps, st));
  }
  {
    ProfScope p(st, ST_SLOW_VERIFY);
    SPEC_TRY(launch_slow_verify<DT>(sh, R, ws, a->anchor, a->draft_tokens, a->lse_q, a->verify_len,
                                    a->u_accept, a->u_final, a->accept_len, a->out_tokens,
                                    a->dev_status, grid, st));
  }
  if (vkernel == 0) {
    // one cooperative launch: the vocabulary split over the CTAs
    ProfScope p(st, ST_VERIFY_REDECIDE);
    SPEC_TRY(launch_verify_redecide<DT>(sh, R, ws, a->out_tokens, a->dev_status, nsm, st));
  } else {
    // (the work-unit passes of the tile-strided verification)
    {
      ProfScope p(st, ST_VERIFY_HP_SUMS);
      SPEC_TRY(launch_hp_sums<DT>(sh, R, ws, 0, a->out_tokens, a->dev_status, grid, st));
    }
    {
      ProfScope p(st, ST_VERIFY_HP_RESID);
      SPEC_TRY(launch_hp_sums<DT>(sh, R, ws, 1, a->out_tokens, a->dev_status, grid, st));
    }
  }
  return SPEC_OK;
}

// ---------------------------------------------------------------- static scratch
// Scratch of spec_markov_draft_static: only the regions the draft touches.
Layout draft_only_layout(const Shape& sh) {
  Layout L = {};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = (off + bytes + 255) & ~(size_t)255;
    return o;
  };
  L.max_items = sh.B;
  L.item_cap = sh.B * sh.gamma;
  L.ctrl = take(CTRL_WORDS * sizeof(uint32_t));
  L.items = take((size_t)L.item_cap * sizeof(HpItem));
  L.hpsum = take((size_t)L.max_items * sh.NC * sizeof(float2));
  L.hpcnt = take((size_t)L.max_items * sizeof(uint32_t));
  L.dpart = take((size_t)sh.B * sh.NC * sizeof(float4));
  L.abuf = take((size_t)(sh.B < 128 ? sh.B : 128) * sh.r * 4);
  L.total = off;
  return L;
}

Ws draft_only_views(const Layout& L, void* base) {
  unsigned char* p = static_cast<unsigned char*>(base);
  Ws w = {};
  w.ctrl = reinterpret_cast<uint32_t*>(p + L.ctrl);
  w.items = reinterpret_cast<HpItem*>(p + L.items);
  w.max_items = L.max_items;
  w.item_cap = L.item_cap;
  w.hpsum = reinterpret_cast<float2*>(p + L.hpsum);
  w.hp_cols = 1;
  w.hpcnt = reinterpret_cast<uint32_t*>(p + L.hpcnt);
  w.dpart = reinterpret_cast<float4*>(p + L.dpart);
  w.abuf = p + L.abuf;
  return w;
}

template <typename DT>
int run_draft_static(const spec_draft_args* a, void* scratch, cudaStream_t st) {
  const Shape sh = make_shape(a->B, a->gamma, a->V, a->r);
  return launch_draft<DT>(a, sh, draft_only_views(draft_only_layout(sh), scratch), st);
}

}  // namespace
}  // namespace spec

// The scratch area itself.  Host code must not use this symbol as a pointer:
// on the host it names a stand-in object, so its device address is obtained
// with cudaGetSymbolAddress once per device and passed to the kernels.
static __device__ __align__(256) unsigned char g_spec_static_scratch[SPEC_STATIC_SCRATCH_BYTES];

namespace spec {
namespace {
std::mutex g_static_mu;
constexpr int kMaxDevices = 64;
void* g_static_addr[kMaxDevices] = {};

// Device address of the scratch area on the current device (cached).
int static_scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ECUDA;
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_spec_static_scratch) != cudaSuccess || !p) return SPEC_ECUDA;
    g_static_addr[dev] = p;
  }
  *out = g_static_addr[dev];
  return SPEC_OK;
}
// Argument checks of spec_markov_draft / spec_verify (nothing enqueued).
int32_t check_draft_args(const spec_draft_args* a) {
  if (!a) return SPEC_EINVAL;
  int rc = check_shape(a->B, a->gamma, a->V, a->r, a->dtype);
  if (rc != SPEC_OK) return rc;
  if (!a->U || !a->W1 || !a->W2 || !a->anchor || !a->temperature || !a->u_draft ||
      !a->draft_tokens || !a->q_tok || !a->lse_q || !a->dev_status)
    return SPEC_EINVAL;
  if (!aligned(a->U, 16) || !aligned(a->W1, 16) || !aligned(a->W2, 16) || !aligned(a->anchor, 4) ||
      !aligned(a->temperature, 4) || !aligned(a->u_draft, 4) || !aligned(a->draft_tokens, 4) ||
      !aligned(a->q_tok, 4) || !aligned(a->lse_q, 8) || !aligned(a->dev_status, 4) ||
      (a->diag && !aligned(a->diag, 4)))
    return SPEC_EALIGN;
  const size_t need = layout(make_shape(a->B, a->gamma, a->V, a->r)).total;
  if (!a->workspace || a->workspace_bytes < need) return SPEC_EWORKSPACE;
  if (!aligned(a->workspace, 256)) return SPEC_EALIGN;
  return SPEC_OK;
}

int32_t check_verify_args(const spec_verify_args* a) {
  if (!a) return SPEC_EINVAL;
  int rc = check_shape(a->B, a->gamma, a->V, a->r, a->dtype);
  if (rc != SPEC_OK) return rc;
  if (!a->target || !a->U || !a->W1 || !a->W2 || !a->anchor || !a->temperature ||
      !a->draft_tokens || !a->q_tok || !a->lse_q || !a->verify_len || !a->u_accept ||
      !a->u_final || !a->accept_len || !a->out_tokens || !a->alpha || !a->dev_status)
    return SPEC_EINVAL;
  if (!aligned(a->target, 16) || !aligned(a->U, 16) || !aligned(a->W1, 16) || !aligned(a->W2, 16) ||
      !aligned(a->anchor, 4) || !aligned(a->temperature, 4) || !aligned(a->draft_tokens, 4) ||
      !aligned(a->q_tok, 4) || !aligned(a->lse_q, 8) || !aligned(a->verify_len, 4) ||
      !aligned(a->u_accept, 4) || !aligned(a->u_final, 4) || !aligned(a->accept_len, 4) ||
      !aligned(a->out_tokens, 4) || !aligned(a->alpha, 4) || !aligned(a->dev_status, 4) ||
      (a->p_tok && !aligned(a->p_tok, 4)) || (a->diag && !aligned(a->diag, 4)) ||
      (a->a_rows && !aligned(a->a_rows, 16)))
    return SPEC_EALIGN;
  const size_t need = layout(make_shape(a->B, a->gamma, a->V, a->r)).total;
  if (!a->workspace || a->workspace_bytes < need) return SPEC_EWORKSPACE;
  if (!aligned(a->workspace, 256)) return SPEC_EALIGN;
  return SPEC_OK;
}

}  // namespace
}  // namespace spec

using namespace spec;

extern "C" {

size_t spec_workspace_bytes(int32_t B, int32_t gamma, int32_t V, int32_t r, int32_t dtype) {
  if (check_shape(B, gamma, V, r, dtype) != SPEC_OK) return 0;
  return layout(make_shape(B, gamma, V, r)).total;
}

int32_t spec_markov_draft(const spec_draft_args* a, spec_stream_t stream) {
  const int32_t rc = check_draft_args(a);
  if (rc != SPEC_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return a->dtype == SPEC_BF16 ? run_draft<bf16>(a, st) : run_draft<float>(a, st);
}

int32_t spec_verify(const spec_verify_args* a, spec_stream_t stream) {
  const int32_t rc = check_verify_args(a);
  if (rc != SPEC_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return a->dtype == SPEC_BF16 ? run_verify<bf16>(a, st) : run_verify<float>(a, st);
}

int32_t spec_cycle_host(const spec_cycle_host_args* c, spec_stream_t stream) {
  if (!c) return SPEC_EINVAL;
  const spec_draft_args* d = &c->draft;
  const spec_verify_args* v = &c->verify;
  int32_t rc = check_draft_args(d);
  if (rc != SPEC_OK) return rc;
  rc = check_verify_args(v);
  if (rc != SPEC_OK) return rc;
  if (d->B != v->B || d->gamma != v->gamma || d->V != v->V || d->r != v->r || d->dtype != v->dtype ||
      d->U != v->U || d->W1 != v->W1 || d->W2 != v->W2 || d->anchor != v->anchor ||
      d->temperature != v->temperature || d->workspace != v->workspace ||
      d->draft_tokens != v->draft_tokens || d->q_tok != v->q_tok || d->lse_q != v->lse_q)
    return SPEC_EINVAL;
  if (!c->h_U || !c->h_target || !c->h_anchor || !c->h_temperature || !c->h_u_draft ||
      !c->h_verify_len || !c->h_u_accept || !c->h_u_final || !c->h_accept_len || !c->h_out_tokens)
    return SPEC_EINVAL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(c->copy_stream);
  const size_t es = d->dtype == SPEC_BF16 ? 2 : 4;
  const size_t B = (size_t)d->B, g = (size_t)d->gamma, V = (size_t)d->V;
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
  cudaEvent_t ev_in = nullptr, ev_t = nullptr;
  auto done = [&](int32_t r) {
    if (ev_in) cudaEventDestroy(ev_in);      // released once the recorded work completes
    if (ev_t) cudaEventDestroy(ev_t);
    return r;
  };
#define SPEC_CUDA_OR_FAIL(x) \
  do {                       \
    if ((x) != cudaSuccess) return done(SPEC_ECUDA); \
  } while (0)
  SPEC_CUDA_OR_FAIL(cudaMemcpyAsync((void*)d->U, c->h_U, B * g * V * es, h2d, st));
  SPEC_CUDA_OR_FAIL(cudaMemcpyAsync((void*)d->anchor, c->h_anchor, B * 4, h2d, st));
  SPEC_CUDA_OR_FAIL(cudaMemcpyAsync((void*)d->temperature, c->h_temperature, B * 4, h2d, st));
  SPEC_CUDA_OR_FAIL(cudaMemcpyAsync((void*)d->u_draft, c->h_u_draft, B * g * 4, h2d, st));
  SPEC_CUDA_OR_FAIL(cudaMemcpyAsync((void*)v->verify_len, c->h_verify_len, B * 4, h2d, st));
  SPEC_CUDA_OR_FAIL(cudaMemcpyAsync((void*)v->u_accept, c->h_u_accept, B * g * 4, h2d, st));
  SPEC_CUDA_OR_FAIL(cudaMemcpyAsync((void*)v->u_final, c->h_u_final, B * 4, h2d, st));
  const size_t tbytes = B * (g + 1) * V * es;
  if (cs) {
    SPEC_CUDA_OR_FAIL(cudaEventCreateWithFlags(&ev_in, cudaEventDisableTiming));
    SPEC_CUDA_OR_FAIL(cudaEventCreateWithFlags(&ev_t, cudaEventDisableTiming));
    SPEC_CUDA_OR_FAIL(cudaEventRecord(ev_in, st));
    SPEC_CUDA_OR_FAIL(cudaStreamWaitEvent(cs, ev_in, 0));
    SPEC_CUDA_OR_FAIL(cudaMemcpyAsync((void*)v->target, c->h_target, tbytes, h2d, cs));
    SPEC_CUDA_OR_FAIL(cudaEventRecord(ev_t, cs));
  } else {
    SPEC_CUDA_OR_FAIL(cudaMemcpyAsync((void*)v->target, c->h_target, tbytes, h2d, st));
  }
  rc = d->dtype == SPEC_BF16 ? run_draft<bf16>(d, st) : run_draft<float>(d, st);
  if (rc != SPEC_OK) return done(rc);
  if (cs) SPEC_CUDA_OR_FAIL(cudaStreamWaitEvent(st, ev_t, 0));
  rc = v->dtype == SPEC_BF16 ? run_verify<bf16>(v, st) : run_verify<float>(v, st);
  if (rc != SPEC_OK) return done(rc);
  SPEC_CUDA_OR_FAIL(cudaMemcpyAsync(c->h_accept_len, v->accept_len, B * 4, d2h, st));
  SPEC_CUDA_OR_FAIL(cudaMemcpyAsync(c->h_out_tokens, v->out_tokens, B * (g + 1) * 4, d2h, st));
  if (c->h_draft_tokens)
    SPEC_CUDA_OR_FAIL(cudaMemcpyAsync(c->h_draft_tokens, d->draft_tokens, B * g * 4, d2h, st));
  if (c->h_alpha) SPEC_CUDA_OR_FAIL(cudaMemcpyAsync(c->h_alpha, v->alpha, B * g * 4, d2h, st));
#undef SPEC_CUDA_OR_FAIL
  return done(SPEC_OK);
}

int32_t spec_rnn_draft(const spec_rnn_draft_args* ra, spec_stream_t stream) {
  if (!ra) return SPEC_EINVAL;
  const spec_draft_args* a = &ra->draft;
  int rc = check_shape(a->B, a->gamma, a->V, a->r, a->dtype);
  if (rc != SPEC_OK) return rc;
  if (!a->U || !a->W1 || !a->W2 || !a->anchor || !a->temperature || !a->u_draft ||
      !a->draft_tokens || !a->q_tok || !a->lse_q || !a->dev_status || !ra->Wr || !ra->hproj ||
      !ra->a_rows)
    return SPEC_EINVAL;
  if (!aligned(a->U, 16) || !aligned(a->W1, 16) || !aligned(a->W2, 16) || !aligned(a->anchor, 4) ||
      !aligned(a->temperature, 4) || !aligned(a->u_draft, 4) || !aligned(a->draft_tokens, 4) ||
      !aligned(a->q_tok, 4) || !aligned(a->lse_q, 8) || !aligned(a->dev_status, 4) ||
      (a->diag && !aligned(a->diag, 4)) || !aligned(ra->Wr, 16) || !aligned(ra->hproj, 16) ||
      !aligned(ra->a_rows, 16))
    return SPEC_EALIGN;
  const size_t need = layout(make_shape(a->B, a->gamma, a->V, a->r)).total;
  if (!a->workspace || a->workspace_bytes < need) return SPEC_EWORKSPACE;
  if (!aligned(a->workspace, 256)) return SPEC_EALIGN;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return a->dtype == SPEC_BF16 ? run_rnn_draft<bf16>(ra, st) : run_rnn_draft<float>(ra, st);
}

int32_t spec_markov_draft_static(const spec_draft_args* a, spec_stream_t stream) {
  if (!a) return SPEC_EINVAL;
  int rc = check_shape(a->B, a->gamma, a->V, a->r, a->dtype);
  if (rc != SPEC_OK) return rc;
  if (!a->U || !a->W1 || !a->W2 || !a->anchor || !a->temperature || !a->u_draft ||
      !a->draft_tokens || !a->q_tok || !a->lse_q || !a->dev_status)
    return SPEC_EINVAL;
  if (!aligned(a->U, 16) || !aligned(a->W1, 16) || !aligned(a->W2, 16) || !aligned(a->anchor, 4) ||
      !aligned(a->temperature, 4) || !aligned(a->u_draft, 4) || !aligned(a->draft_tokens, 4) ||
      !aligned(a->q_tok, 4) || !aligned(a->lse_q, 8) || !aligned(a->dev_status, 4) ||
      (a->diag && !aligned(a->diag, 4)))
    return SPEC_EALIGN;
  if (draft_only_layout(make_shape(a->B, a->gamma, a->V, a->r)).total > SPEC_STATIC_SCRATCH_BYTES)
    return SPEC_EWORKSPACE;
  void* scratch = nullptr;
  rc = static_scratch_address(&scratch);
  if (rc != SPEC_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return a->dtype == SPEC_BF16 ? run_draft_static<bf16>(a, scratch, st)
                               : run_draft_static<float>(a, scratch, st);
}

int32_t spec_confidence(const spec_confidence_args* a, spec_stream_t stream) {
  if (!a) return SPEC_EINVAL;
  if (a->R < 1 || a->R > 4096 || a->gamma < 1 || a->d < 8 || a->V < 1 || a->V >= (1 << 24) || a->r < 16)
    return SPEC_EINVAL;
  if (a->gamma > MAX_GAMMA || a->d % 8 != 0 || a->r % 16 != 0 || a->r > 256 ||
      (a->dtype != SPEC_F32 && a->dtype != SPEC_BF16))
    return SPEC_EUNSUPPORTED;
  if (!a->hidden || !a->W1 || !a->w || !a->anchor || !a->draft_tokens || !a->conf || !a->dev_status)
    return SPEC_EINVAL;
  if (!aligned(a->hidden, 16) || !aligned(a->W1, 16) || !aligned(a->w, 16) || !aligned(a->anchor, 4) ||
      !aligned(a->draft_tokens, 4) || !aligned(a->conf, 4) || !aligned(a->dev_status, 4))
    return SPEC_EALIGN;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  ProfScope p(st, ST_CONFIDENCE);
  const cudaError_t e =
      a->dtype == SPEC_BF16
          ? launch_confidence<bf16>(a->R, a->gamma, a->d, a->V, a->r, a->hidden, a->W1, a->w, a->anchor,
                                    a->draft_tokens, a->conf, a->dev_status, st)
          : launch_confidence<float>(a->R, a->gamma, a->d, a->V, a->r, a->hidden, a->W1, a->w, a->anchor,
                                     a->draft_tokens, a->conf, a->dev_status, st);
  return e == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

// Workspace of the scheduler: the candidates' ranks, then their tau
// increments in sorted order.
static size_t sched_rank_bytes(int R, int gamma) { return ((size_t)R * gamma * 4 + 255) & ~(size_t)255; }

size_t spec_schedule_workspace_bytes(int32_t R, int32_t gamma) {
  if (R < 1 || R > 4096 || gamma < 1 || gamma > MAX_GAMMA) return 0;
  return sched_rank_bytes(R, gamma) + (((size_t)R * gamma * 8 + 255) & ~(size_t)255);
}

int32_t spec_prefix_schedule(const spec_schedule_args* a, spec_stream_t stream) {
  if (!a) return SPEC_EINVAL;
  if (a->R < 1 || a->R > 4096 || a->gamma < 1 || a->sps_len <= a->R) return SPEC_EINVAL;
  if (a->gamma > MAX_GAMMA) return SPEC_EUNSUPPORTED;
  if (!a->conf || !a->sps || !a->survival || !a->verify_len || !a->totals || !a->theta || !a->dev_status)
    return SPEC_EINVAL;
  if (!aligned(a->conf, 4) || !aligned(a->sps, 8) || !aligned(a->survival, 4) ||
      !aligned(a->verify_len, 4) || !aligned(a->totals, 8) || !aligned(a->theta, 8) ||
      !aligned(a->dev_status, 4))
    return SPEC_EALIGN;
  const size_t need = spec_schedule_workspace_bytes(a->R, a->gamma);
  if (!a->workspace || a->workspace_bytes < need) return SPEC_EWORKSPACE;
  if (!aligned(a->workspace, 16)) return SPEC_EALIGN;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(a->workspace);
  int* rank = reinterpret_cast<int*>(ws);
  unsigned long long* su = reinterpret_cast<unsigned long long*>(ws + sched_rank_bytes(a->R, a->gamma));
  {
    ProfScope p(st, ST_SCHED_RANK);
    if (launch_schedule_rank(a->R, a->gamma, a->conf, a->survival, rank, su, a->dev_status, st) != cudaSuccess)
      return SPEC_ECUDA;
  }
  {
    ProfScope p(st, ST_SCHED_SELECT);
    if (launch_schedule_select(a->R, a->gamma, a->sps, a->sps_len, rank, su, a->verify_len,
                               reinterpret_cast<long long*>(a->totals), a->theta, st) != cudaSuccess)
      return SPEC_ECUDA;
  }
  return SPEC_OK;
}

// ---------------------------------------------------------------- trees
static int tree_check(int B, int N, int gamma, int V, int r, int dtype) {
  if (B < 1 || B > 4096 || N < 1 || gamma < 1 || V < 16 || V >= (1 << 24) || r < 1) return SPEC_EINVAL;
  if (N > 256 || gamma > MAX_GAMMA || r % 16 != 0 || r > 256 || V % 8 != 0 ||
      (dtype != SPEC_F32 && dtype != SPEC_BF16))
    return SPEC_EUNSUPPORTED;
  return SPEC_OK;
}

size_t spec_tree_workspace_bytes(int32_t B, int32_t N, int32_t V) {
  if (B < 1 || N < 1 || V < 16) return 0;
  return tree_workspace_bytes(TreeShape{B, N, 0, V, 0});
}

int32_t spec_tree_select(int32_t B, int32_t N, int32_t gamma, const int32_t* parent, const float* conf,
                         int32_t n, float* survival, uint8_t* mask, float* expected, uint32_t* dev_status,
                         spec_stream_t stream) {
  if (B < 1 || B > 4096 || N < 1 || gamma < 1 || n < 0 || !parent || !conf || !survival || !mask ||
      !dev_status)
    return SPEC_EINVAL;
  if (N > 256 || gamma > MAX_GAMMA) return SPEC_EUNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  ProfScope p(st, ST_TREE_SELECT);
  return launch_tree_select(B, N, gamma, parent, conf, n, survival, mask, expected, dev_status, st) ==
                 cudaSuccess
             ? SPEC_OK
             : SPEC_ECUDA;
}

int32_t spec_tree_draft(const spec_tree_draft_args* a, spec_stream_t stream) {
  if (!a) return SPEC_EINVAL;
  const int rc = tree_check(a->B, a->N, a->gamma, a->V, a->r, a->dtype);
  if (rc != SPEC_OK) return rc;
  if (!a->U || !a->W1 || !a->W2 || !a->anchor || !a->temperature || !a->parent || !a->mask ||
      !a->u_draft || !a->tokens || !a->q_tok || !a->dev_status)
    return SPEC_EINVAL;
  if (!aligned(a->U, 16) || !aligned(a->W1, 16) || !aligned(a->W2, 16)) return SPEC_EALIGN;
  if (!a->workspace || a->workspace_bytes < spec_tree_workspace_bytes(a->B, a->N, a->V))
    return SPEC_EWORKSPACE;
  if (!aligned(a->workspace, 16)) return SPEC_EALIGN;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const TreeShape ts{a->B, a->N, a->gamma, a->V, a->r};
  ProfScope p(st, ST_TREE_DRAFT);
  const cudaError_t e =
      a->dtype == SPEC_BF16
          ? launch_tree_draft<bf16>(ts, a->U, a->W1, a->W2, a->anchor, a->temperature, a->parent, a->mask,
                                    a->u_draft, a->tokens, a->q_tok, a->workspace, a->dev_status, st)
          : launch_tree_draft<float>(ts, a->U, a->W1, a->W2, a->anchor, a->temperature, a->parent, a->mask,
                                     a->u_draft, a->tokens, a->q_tok, a->workspace, a->dev_status, st);
  return e == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

int32_t spec_tree_verify(const spec_tree_verify_args* a, spec_stream_t stream) {
  if (!a) return SPEC_EINVAL;
  const int rc = tree_check(a->B, a->N, a->gamma, a->V, a->r, a->dtype);
  if (rc != SPEC_OK) return rc;
  if (!a->target || !a->U || !a->W1 || !a->W2 || !a->anchor || !a->temperature || !a->parent ||
      !a->mask || !a->tokens || !a->u_accept || !a->u_final || !a->accept_len || !a->out_tokens ||
      !a->path || !a->dev_status)
    return SPEC_EINVAL;
  if (!aligned(a->target, 16) || !aligned(a->U, 16) || !aligned(a->W1, 16) || !aligned(a->W2, 16))
    return SPEC_EALIGN;
  if (!a->workspace || a->workspace_bytes < spec_tree_workspace_bytes(a->B, a->N, a->V))
    return SPEC_EWORKSPACE;
  if (!aligned(a->workspace, 16)) return SPEC_EALIGN;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const TreeShape ts{a->B, a->N, a->gamma, a->V, a->r};
  ProfScope p(st, ST_TREE_VERIFY);
  const cudaError_t e =
      a->dtype == SPEC_BF16
          ? launch_tree_verify<bf16>(ts, a->target, a->U, a->W1, a->W2, a->anchor, a->temperature,
                                     a->parent, a->mask, a->tokens, a->u_accept, a->u_final, a->accept_len,
                                     a->out_tokens, a->path, a->workspace, a->dev_status, st)
          : launch_tree_verify<float>(ts, a->target, a->U, a->W1, a->W2, a->anchor, a->temperature,
                                      a->parent, a->mask, a->tokens, a->u_accept, a->u_final,
                                      a->accept_len, a->out_tokens, a->path, a->workspace, a->dev_status,
                                      st);
  return e == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

const char* spec_status_string(int32_t s) {
  switch (s) {
    case SPEC_OK: return "ok";
    case SPEC_EINVAL: return "invalid argument (NULL pointer or size out of range)";
    case SPEC_EUNSUPPORTED: return "unsupported shape or dtype";
    case SPEC_EALIGN: return "misaligned pointer";
    case SPEC_EWORKSPACE: return "workspace missing or too small";
    case SPEC_ECUDA: return "CUDA launch failed";
    default: return "unknown status";
  }
}

int32_t spec_set_option(int32_t key, double value) {
  std::lock_guard<std::mutex> lk(g_mu);
  switch (key) {
    case SPEC_OPT_EPS_SCALE:
      if (!(value >= 0.0)) return SPEC_EINVAL;
      g_eps_scale = value;
      return SPEC_OK;
    case SPEC_OPT_FORCE_SIMT:
      g_force_simt = value != 0.0;
      return SPEC_OK;
    case SPEC_OPT_BIAS_PATH:
      if (value != 1.0 && value != 2.0) return SPEC_EINVAL;
      g_bias_path = (int)value;
      return SPEC_OK;
    case SPEC_OPT_TRACE:
      g_trace = value != 0.0;
      return SPEC_OK;
    case SPEC_OPT_PERTURB:
      g_perturb = value != 0.0;
      return SPEC_OK;
    case SPEC_OPT_TEST_STALL:
      g_stall = value != 0.0;
      return SPEC_OK;
    case SPEC_OPT_DRAFT_KERNEL:
      if (value != 0.0 && value != 1.0) return SPEC_EINVAL;
      g_draft_kernel = (int)value;
      return SPEC_OK;
    case SPEC_OPT_VERIFY_KERNEL:
      if (value != 0.0 && value != 1.0) return SPEC_EINVAL;
      g_verify_kernel = (int)value;
      return SPEC_OK;
    default:
      return SPEC_EINVAL;
  }
}

int32_t spec_profile_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_prof = on != 0;
  return SPEC_OK;
}

int32_t spec_profile_read(double* ms, int32_t* launches, int32_t n) {
  std::vector<EvPair> pend;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    pend.swap(g_pending);
  }
  for (int i = 0; i < n; ++i) {
    if (ms) ms[i] = 0.0;
    if (launches) launches[i] = 0;
  }
  int rc = SPEC_OK;
  for (const EvPair& e : pend) {
    float t = 0.f;
    if (cudaEventSynchronize(e.b) != cudaSuccess || cudaEventElapsedTime(&t, e.a, e.b) != cudaSuccess)
      rc = SPEC_ECUDA;
    if (e.stage < n) {
      if (ms) ms[e.stage] += t;
      if (launches) launches[e.stage] += 1;
    }
  }
  std::lock_guard<std::mutex> lk(g_mu);
  for (const EvPair& e : pend) {
    g_pool.push_back(e.a);
    g_pool.push_back(e.b);
  }
  return rc;
}

const char* spec_stage_name(int32_t id) {
  if (id < 0 || id >= ST_COUNT) return "";
  return kStageNames[id];
}

int32_t spec_num_stages(void) { return ST_COUNT; }

}  // extern "C"
