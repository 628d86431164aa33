/*
 * spec.h -- C ABI of the GB300 sampling hot path of speculative decoding.
 *
 * Two calls make one speculative cycle:
 *
 *   spec_markov_draft  DSpark's sequential stage with the Markov head
 *                      ("[논문리뷰] DSpark: Confidence-Scheduled Speculative
 *                      Decoding with Semi-Autoregressive Generation", section
 *                      1.2 "Sequential stage", block factorisation and the
 *                      "Markov head" equation B(x_{k-1}, .) = W1[x_{k-1}] W2):
 *                      for k = 1..gamma, q_k = softmax((U_k + W1[x_{k-1}] W2)/T)
 *                      and x_k is drawn from q_k by inverse CDF.
 *
 *   spec_verify        lossless verification ("Speculative Decoding Part 1",
 *                      VESSL AI blog, section "알고리즘" and section "수락
 *                      규칙"): ratio tests u_j < p_j(x_{j+1}) / q_j(x_{j+1}) on
 *                      every position, first reject n, correction token from
 *                      normalize(max(0, p_n - q_n)) or bonus token from p_L, and
 *                      alpha_j = sum_v min(p_j(v), q_j(v)); each request stops
 *                      at its own verify length L_b (DSpark review, section
 *                      2.2: the scheduler's l_r in {0..gamma}).
 *
 * Notation: q = draft distribution, p = target distribution.  Row j of U
 * (0-based) is the draft logits of token x_{j+1}; row j of the target is the
 * target logits that test x_{j+1}; target row L_b gives the bonus token.
 * x_0 is the anchor.  The same temperature T_b divides the draft logits
 * (U + bias) and the target logits.
 *
 * Sampling convention: the token drawn from a distribution pi with a uniform
 * u is the smallest v (vocabulary order) with sum_{w<=v} pi(w) > u.  A ratio
 * test accepts iff u < p/q.
 *
 * Conventions for every call:
 *   - Tensor pointers are DEVICE pointers, row-major, 16-byte aligned, owned
 *     by the caller; the library never allocates device memory.  Scratch
 *     comes from the caller's workspace (spec_workspace_bytes()).
 *   - Work is enqueued on `stream` and the call returns at once; outputs are
 *     valid after the stream reaches that point.  The calls never
 *     synchronize, so they may be captured in a CUDA graph.
 *   - Host-detected errors (NULL pointer, unsupported shape or dtype,
 *     misalignment, workspace too small) return a negative spec_status and
 *     enqueue nothing.  A failed kernel launch returns SPEC_ECUDA.
 *   - Data-dependent errors are detected on the device and OR-ed into
 *     dev_status[0] (SPEC_DEV_* bits); the affected request's outputs are set
 *     to -1 / NaN.  Read dev_status after synchronizing.
 *   - Two calls may run concurrently only on distinct workspaces.
 *   - Supported: 1 <= gamma <= 16, 1 <= B <= 4096, 16 <= V < 2^24 with
 *     V % 8 == 0, r % 16 == 0 with r <= 256 (bf16) or r <= 64 (fp32).
 */
#ifndef SPEC_GB300_H
#define SPEC_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Identical to cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* spec_stream_t;

typedef enum {
  SPEC_OK = 0,
  SPEC_EINVAL = -1,        /* NULL pointer or a size out of range           */
  SPEC_EUNSUPPORTED = -2,  /* dtype / rank / gamma not supported             */
  SPEC_EALIGN = -3,        /* a pointer is not 16-byte aligned               */
  SPEC_EWORKSPACE = -4,    /* workspace NULL or smaller than required        */
  SPEC_ECUDA = -5          /* a CUDA launch or attribute call failed         */
} spec_status;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

/* Bits of dev_status[0].  dev_status is uint32_t[4]:
 *   [0] OR of the bits below
 *   [1] decisions re-decided in extended precision (near a boundary)
 *   [2] decisions whose token or outcome changed after re-deciding
 *   [3] requests verified on the extended-precision slow path (spec_verify);
 *       RNN head gate outputs recomputed in double-float (spec_rnn_draft)   */
enum {
  SPEC_DEV_BAD_TOKEN = 1,   /* anchor or draft token outside [0, V)          */
  SPEC_DEV_BAD_LEN = 2,     /* verify_len outside [0, gamma]                 */
  SPEC_DEV_BAD_TEMP = 4,    /* temperature not finite and > 0                */
  SPEC_DEV_TIMEOUT = 8,     /* a bounded device wait gave up                 */
  SPEC_DEV_REFINED = 16,    /* informational: at least one re-decision        */
  SPEC_DEV_OVERFLOW = 32,   /* more near-boundary decisions than list slots   */
  SPEC_DEV_BAD_CONF = 64,   /* a confidence logit not finite, or a confidence
                               outside [0, 1] given to the scheduler           */
  SPEC_DEV_BAD_TREE = 128   /* a tree slot whose parent does not precede it, or
                               deeper than gamma                                */
};

/* ---------------------------------------------------------------- draft */
typedef struct {
  int32_t B, gamma, V, r;
  int32_t dtype;              /* spec_dtype of U, W1, W2                        */
  const void* U;              /* [B][gamma][V] base draft logits U_1..U_gamma   */
  const void* W1;             /* [V][r]  Markov embedding (row lookup)          */
  const void* W2;             /* [r][V]  Markov logit projection                */
  const int32_t* anchor;      /* [B]     x_0                                    */
  const float* temperature;   /* [B]     T_b > 0                                */
  const float* u_draft;       /* [B][gamma] uniforms in (0,1); [b][k] draws x_{k+1} */
  int32_t* draft_tokens;      /* out [B][gamma]  x_1..x_gamma                   */
  float* q_tok;               /* out [B][gamma]  q_k(x_k)                       */
  double* lse_q;              /* out [B][gamma]  logsumexp_v((U_k(v)+B(v))/T)   */
  uint32_t* dev_status;       /* out uint32_t[4], zeroed by the call            */
  float* diag;                /* optional out [B][gamma][4]: first-pass margins
                                 u - F(x-1) and F(x) - u, the near-boundary band,
                                 first-pass token (before any re-decision)        */
  void* workspace;
  size_t workspace_bytes;
} spec_draft_args;

/* --------------------------------------------------------------- verify */
typedef struct {
  int32_t B, gamma, V, r;
  int32_t dtype;              /* spec_dtype of target, U, W1, W2                */
  const void* target;         /* [B][gamma+1][V] target logits                  */
  const void* U;              /* [B][gamma][V]   the draft's base logits        */
  const void* W1;             /* [V][r]                                         */
  const void* W2;             /* [r][V]                                         */
  const int32_t* anchor;      /* [B]                                            */
  const float* temperature;   /* [B]                                            */
  const int32_t* draft_tokens;/* [B][gamma] from spec_markov_draft              */
  const float* q_tok;         /* [B][gamma] from spec_markov_draft              */
  const double* lse_q;        /* [B][gamma] from spec_markov_draft              */
  const int32_t* verify_len;  /* [B] L_b in [0, gamma]; 0 = bonus token only    */
  const float* u_accept;      /* [B][gamma] ratio-test uniforms                 */
  const float* u_final;       /* [B] one uniform: correction OR bonus token     */
  int32_t* accept_len;        /* out [B]        n_b (tau = n_b + 1)             */
  int32_t* out_tokens;        /* out [B][gamma+1] x_1..x_n, correction/bonus, -1 */
  float* alpha;               /* out [B][gamma] sum_v min(p_j, q_j), j < L_b; NaN beyond */
  float* p_tok;               /* optional out [B][gamma] p_j(x_{j+1}), j < L_b; NaN beyond */
  uint32_t* dev_status;       /* out uint32_t[4], zeroed by the call            */
  const void* a_rows;         /* optional [gamma][B][r] (dtype): the draft head's
                                 factor rows a_j (spec_rnn_draft); NULL = the
                                 Markov head's W1[x_j]                          */
  float* diag;                /* optional out [B][4]: final draw's first-pass
                                 margins u - F(c-1), F(c) - u (in the normalised
                                 residual or bonus distribution), the band, and
                                 the first-pass token                            */
  void* workspace;
  size_t workspace_bytes;
} spec_verify_args;

/* Bytes of workspace either call needs for these sizes (0 if unsupported).
 * One workspace may serve both calls when they run in stream order.        */
size_t spec_workspace_bytes(int32_t B, int32_t gamma, int32_t V, int32_t r, int32_t dtype);

/* Draft gamma tokens per request.  Reads U, W1, W2, anchor, temperature,
 * u_draft; writes draft_tokens, q_tok, lse_q, dev_status (and diag).
 * The work is three cudaMemsetAsync (dev_status, the workspace's control
 * words and counters) and ONE cooperative kernel launch on `stream` with at
 * most one CTA per SM; it returns SPEC_ECUDA when the device cannot make the
 * CTAs co-resident.  Two kernels serve it: for bf16 with r % 64 == 0,
 * B <= 128 and V <= 256 x (SM count) (C1/C2-class shapes) the slice-resident
 * kernel, in which each CTA keeps the W2 columns of one vocabulary slice in
 * shared memory for all gamma steps; otherwise the tile-strided kernel.  Both
 * give the same results (see SPEC_OPT_DRAFT_KERNEL).  Its grid barriers are
 * bounded waits: a barrier that gives up sets SPEC_DEV_TIMEOUT and every CTA
 * returns.                                                                 */
int32_t spec_markov_draft(const spec_draft_args* args, spec_stream_t stream);

/* Verify one drafted block per request.  Writes accept_len, out_tokens,
 * alpha, dev_status (and p_tok, diag when non-NULL).                        */
int32_t spec_verify(const spec_verify_args* args, spec_stream_t stream);

/* ----------------------------------------- one cycle from host memory */
/* No counterpart on the pages: the end-to-end form of one speculative cycle
 * (spec_markov_draft, then spec_verify) for callers whose per-step inputs
 * arrive in host memory and who want the results there.
 *
 * The call enqueues, on `stream`: one cudaMemcpyAsync per input from its
 * host buffer into the device buffer that `draft` / `verify` name (U,
 * anchor, temperature, u_draft, verify_len, u_accept, u_final; target too
 * when copy_stream is NULL), the draft, the verification, and one
 * cudaMemcpyAsync per result back to host memory (accept_len, out_tokens;
 * draft_tokens and alpha when their host pointers are non-NULL).  With
 * copy_stream non-NULL the target logits, which only the verification
 * reads, are copied on copy_stream while the draft runs: that copy starts
 * after the other input copies on `stream` (so it neither races with the
 * previous call's verification nor shares the link with U's copy), and the
 * verification waits for it (two events, created and released by the call).
 * The host results are valid once `stream` has been synchronised.  Host
 * buffers should be page-locked (cudaHostAlloc, cudaHostRegister) for the
 * copies to be asynchronous.
 *
 * `draft` and `verify` must describe one cycle: the same B, gamma, V, r,
 * dtype, U, W1, W2, anchor, temperature and workspace, and verify's
 * draft_tokens, q_tok, lse_q equal to draft's outputs.  Every host pointer
 * except the two optional outputs must be non-NULL.  A violation, or any
 * error spec_markov_draft / spec_verify would return, is reported before
 * anything is enqueued; SPEC_ECUDA after a failed copy or launch (work
 * enqueued before it stays enqueued).                                      */
typedef struct {
  spec_draft_args draft;        /* device buffers of the draft (inputs filled by the call) */
  spec_verify_args verify;      /* device buffers of the verification             */
  const void* h_U;              /* host [B][gamma][V] (dtype)   -> draft.U          */
  const void* h_target;         /* host [B][gamma+1][V] (dtype) -> verify.target    */
  const int32_t* h_anchor;      /* host [B]                     -> draft.anchor     */
  const float* h_temperature;   /* host [B]                     -> draft.temperature */
  const float* h_u_draft;       /* host [B][gamma]              -> draft.u_draft    */
  const int32_t* h_verify_len;  /* host [B]                     -> verify.verify_len */
  const float* h_u_accept;      /* host [B][gamma]              -> verify.u_accept  */
  const float* h_u_final;       /* host [B]                     -> verify.u_final   */
  int32_t* h_accept_len;        /* host out [B]                 <- verify.accept_len */
  int32_t* h_out_tokens;        /* host out [B][gamma+1]        <- verify.out_tokens */
  int32_t* h_draft_tokens;      /* optional host out [B][gamma] <- draft.draft_tokens */
  float* h_alpha;               /* optional host out [B][gamma] <- verify.alpha     */
  spec_stream_t copy_stream;    /* optional second stream for the target copy (NULL: none) */
} spec_cycle_host_args;
int32_t spec_cycle_host(const spec_cycle_host_args* args, spec_stream_t stream);

/* ------------------------------------------------------------- RNN head */
/* DSpark's RNN head ("[논문리뷰] DSpark", section 1.2, "RNN head"): a state s_k
 * (s_0 = 0) carries the block's prefix; with z = [s_j; W1[x_j]; h_{j+1}] the
 * draft row j uses the factor a_j = tanh(W_o z) in place of the Markov head's
 * W1[x_j] (bias a_j W2) and updates s_{j+1} = sigma(W_g z) s_j +
 * (1 - sigma(W_g z)) tanh(W_c z).  The h block of z enters the gates linearly
 * and does not depend on drafted tokens: its three projections arrive as
 * hproj (formed with U by the parallel stage).  s and a are held in `dtype`
 * (each the exactly rounded value of the step's float64 result; the kernel
 * certifies every rounding or recomputes it in double-float).
 * Work: as spec_markov_draft (3 memsets + 1 cooperative launch), with one
 * more phase and grid barrier per step.  Writes a_rows, which spec_verify
 * takes to rebuild q.  Same limits as spec_markov_draft; Wr, hproj and
 * a_rows 16-byte aligned.                                                   */
typedef struct {
  spec_draft_args draft;      /* as for spec_markov_draft                       */
  const void* Wr;             /* [3r][2r] (dtype): rows g, c, o of the gates; columns
                                 act on s, then on W1[x]                         */
  const float* hproj;         /* [B][gamma][3][r]: (W_g^h h, W_c^h h, W_o^h h) of
                                 draft row j = h_{j+1}                           */
  void* a_rows;               /* out [gamma][B][r] (dtype)                      */
} spec_rnn_draft_args;
int32_t spec_rnn_draft(const spec_rnn_draft_args* args, spec_stream_t stream);

/* ------------------------------------------- draft without caller scratch */
/* No counterpart on the pages: this is a deployment convenience.
 *
 * Some callers cannot allocate device memory when they draft: code that runs
 * while another component is capturing the stream into a CUDA graph (an
 * allocation there would break or serialise the capture), services that
 * reserve their whole device-memory budget at start-up and forbid later
 * allocations, and plug-ins that receive only a stream from a host framework
 * that owns the allocator.  spec_markov_draft_static does the same work as
 * spec_markov_draft but ignores args->workspace / workspace_bytes and uses a
 * scratch area of SPEC_STATIC_SCRATCH_BYTES compiled into the library as
 * device memory.  It never calls cudaMalloc, cudaFree or any allocating
 * library routine.
 *
 *   - When the area is committed: the area belongs to the library's device
 *     code, so it is committed on a device when that code is loaded there.
 *     With lazy module loading (CUDA_MODULE_LOADING=LAZY, the default since
 *     CUDA 12) that is the first call of ANY spec_* entry point on that
 *     device (or this entry point's address look-up); with eager loading it
 *     is when the CUDA context is created.  Either way the device then holds
 *     the 32 MiB until the process exits.  Callers under a fixed memory
 *     budget should count it from their first library call on a device, and
 *     callers that capture streams should make that first library call
 *     before any capture begins.
 *
 *   - Size limit: the draft scratch is 128 + B*40 + B*ceil(V/32)*8 + B*4 +
 *     B*ceil(V/32)*16 bytes (each term rounded up to 256); larger problems
 *     are rejected with SPEC_EWORKSPACE before anything is enqueued.  All five
 *     named workloads fit (C4, the largest, needs about 24 MiB).
 *   - The first call of this entry point on a device looks up the area's
 *     device address with cudaGetSymbolAddress (with that device current)
 *     and caches it per device; make that first call before any stream
 *     capture too.
 *   - All calls in the process share the one area, and it keeps the previous
 *     call's contents (the call clears the words that must start at zero).
 *     Calls whose GPU work overlaps -- on different streams, or from
 *     different threads without ordering -- race on it: serialise them.
 */
#define SPEC_STATIC_SCRATCH_BYTES ((size_t)32 << 20)
int32_t spec_markov_draft_static(const spec_draft_args* args, spec_stream_t stream);

/* ------------------------------------- confidence head and prefix scheduler */
/* DSpark's confidence-scheduled verification ("[논문리뷰] DSpark", section 2.1
 * "Confidence Head" and section 2.2 "Hardware-Aware Prefix Scheduler").
 *
 * spec_confidence: c_{r,k} = sigmoid(w^T [h_k; W1[x_{k-1}]]) for every draft
 * row k = 1..gamma of every request r, x_0 the anchor.  Row k-1 (0-based) of
 * `hidden` is h_k, the backbone state that also produced U_k.  The dot
 * product and the logistic are evaluated in double-float and rounded once to
 * fp32 (the nearest float of the exact value, except within about 1e-13 of a
 * rounding midpoint).  One kernel launch.  A token outside [0, V) sets
 * SPEC_DEV_BAD_TOKEN and a logit that is not finite SPEC_DEV_BAD_CONF; that
 * row's confidence is NaN.  dev_status bits are OR-ed in and never cleared
 * by these two calls.
 * Requires 1 <= R <= 4096, 1 <= gamma <= 16, d >= 8 with d % 8 == 0,
 * 1 <= V < 2^24, r % 16 == 0 with 16 <= r <= 256, hidden / W1 / w 16-byte
 * aligned.                                                                  */
typedef struct {
  int32_t R, gamma, d, V, r;
  int32_t dtype;              /* spec_dtype of hidden and W1                    */
  const void* hidden;         /* [R][gamma][d] backbone hidden states h_1..h_gamma */
  const void* W1;             /* [V][r] Markov embedding (the draft's W1)       */
  const float* w;             /* [d + r] head weights: the h part, then the W1 part */
  const int32_t* anchor;      /* [R] x_0                                        */
  const int32_t* draft_tokens;/* [R][gamma] x_1..x_gamma (x_gamma is not read)   */
  float* conf;                /* out [R][gamma] c_1..c_gamma                    */
  uint32_t* dev_status;       /* uint32_t[4]; bits OR-ed into [0]               */
} spec_confidence_args;
int32_t spec_confidence(const spec_confidence_args* args, spec_stream_t stream);

/* spec_prefix_schedule: survival a_{r,j} = c_{r,1} ... c_{r,j} (fp32 products
 * left to right), then verify lengths l_r maximising Theta = tau * SPS(B),
 * B = sum_r (1 + l_r), tau = sum_r (1 + sum_{j<=l_r} a_{r,j}): the candidates
 * (r, j) are admitted in descending order of a (equal a: lower r, then lower
 * j) while Theta does not decrease; the first admission that would lower
 * Theta, or that would need SPS beyond the table, ends the search.
 * tau is accumulated in units of 2^-36 (each a rounded down) and Theta is
 * (tau units * 2^-36) * sps[B] in float64, so the decisions do not depend on
 * the order of summation.  A confidence outside [0, 1] or NaN counts as 0 and
 * sets SPEC_DEV_BAD_CONF.  Two kernel launches (ranking: one CTA per request;
 * selection: one CTA).
 * Outputs: survival [R][gamma]; verify_len [R] = l_r in [0, gamma] (the
 * spec_verify input of the same name); totals int64[4] = {B, tau in units of
 * 2^-36, admitted candidates, stop reason: 0 all admitted, 1 Theta would
 * decrease, 2 the cost table ends}; theta double[1] = Theta at the result.
 * sps: device float64[sps_len], SPS(B') for B' = 0..sps_len-1 (finite,
 * positive); sps_len must exceed R.  The workspace needs
 * spec_schedule_workspace_bytes(R, gamma) bytes, 16-byte aligned.
 * Requires 1 <= R <= 4096, 1 <= gamma <= 16.                                */
typedef struct {
  int32_t R, gamma;
  const float* conf;          /* [R][gamma] c_{r,j}                             */
  const double* sps;          /* [sps_len] steps per second at batch size B'     */
  int32_t sps_len;            /* > R                                            */
  float* survival;            /* out [R][gamma] a_{r,j}                         */
  int32_t* verify_len;        /* out [R] l_r                                    */
  int64_t* totals;            /* out [4] B, tau (2^-36 units), admitted, reason  */
  double* theta;              /* out [1]                                        */
  uint32_t* dev_status;       /* uint32_t[4]; bits OR-ed into [0]               */
  void* workspace;
  size_t workspace_bytes;
} spec_schedule_args;
size_t spec_schedule_workspace_bytes(int32_t R, int32_t gamma);
int32_t spec_prefix_schedule(const spec_schedule_args* args, spec_stream_t stream);

/* -------------------------------------------------------------- trees */
/* Tree drafting and verification ("Speculative Decoding Part 1", VESSL AI
 * blog, section "gamma 재배분: 체인 대신 트리"), the Markov head drafting every
 * node.  A request's candidate tree has N slots; parent[b][s] is -1 (the
 * root, the anchor x_0) or a slot < s; depth(s) = depth(parent) + 1 <= gamma.
 *
 * spec_tree_select: survival a_s = product of conf[b][.] from the root down
 * (fp32, left to right), then the top-n slots by a (ties: the shallower slot,
 * then the lower index) -- closed under prefixes.  mask[b][s] = 1 for the
 * chosen slots, survival[b][s] = a_s, expected[b] = sum of the chosen a
 * (optional).  A bad parent sets SPEC_DEV_BAD_TREE and selects nothing for
 * that request; a factor outside [0, 1] counts as 0 (SPEC_DEV_BAD_CONF).
 * One launch, one CTA per request.  1 <= N <= 256, 1 <= gamma <= 16.
 *
 * spec_tree_draft: every selected slot s at depth d + 1 whose parent node
 * holds token x (the anchor for the root) gets a token drawn by inverse CDF
 * with u_draft[b][s] from q = softmax((U[b][d] + W1[x] W2) / T_b); children
 * of one node are independent draws.  Unselected slots are left untouched.
 * One planning launch, then two launches per depth (each drafted node's
 * vocabulary split over 16 CTAs, then one CTA per node for its children's
 * draws), double-float arithmetic throughout.
 *
 * spec_tree_verify: walks each request's selected tree from the root.  At a
 * node with target row p (target[b][0] at the root, target[b][1 + s] at slot
 * s) and draft q, the selected children are tried in slot order: child c is
 * accepted iff u_accept[b][c] < r(x_c) / q(x_c), r starting at p and
 * replaced by normalize(max(0, r - q)) after each rejection (recursive
 * rejection sampling, for independently drawn children); the accepted child
 * becomes the next node; when none is accepted the final token is drawn from
 * r with u_final[b] (at a leaf r = p: the bonus token).  Outputs accept_len
 * (accepted nodes), out_tokens [B][gamma+1] (accepted tokens, final, -1) and
 * path [B][gamma] (accepted slots, -1).  gamma + 1 steps of two launches
 * (the current node's draft row over several CTAs per request, then one CTA
 * per request for the node's tests and draws), double-float arithmetic
 * throughout.
 *
 * Both draft and verify take the workspace spec_tree_workspace_bytes(B, N, V)
 * (16-byte aligned); dev_status bits are OR-ed in and never cleared.        */
int32_t spec_tree_select(int32_t B, int32_t N, int32_t gamma, const int32_t* parent, const float* conf,
                         int32_t n, float* survival, uint8_t* mask, float* expected,
                         uint32_t* dev_status, spec_stream_t stream);
typedef struct {
  int32_t B, N, gamma, V, r;
  int32_t dtype;              /* spec_dtype of U, W1, W2 (and target)            */
  const void* U;              /* [B][gamma][V]                                   */
  const void* W1;             /* [V][r]                                          */
  const void* W2;             /* [r][V]                                          */
  const int32_t* anchor;      /* [B]                                             */
  const float* temperature;   /* [B]                                             */
  const int32_t* parent;      /* [B][N]                                          */
  const uint8_t* mask;        /* [B][N] from spec_tree_select                    */
  const float* u_draft;       /* [B][N]                                          */
  int32_t* tokens;            /* out [B][N] (selected slots)                     */
  float* q_tok;               /* out [B][N] q(x_s) of each drawn token           */
  uint32_t* dev_status;
  void* workspace;
  size_t workspace_bytes;
} spec_tree_draft_args;
int32_t spec_tree_draft(const spec_tree_draft_args* args, spec_stream_t stream);
typedef struct {
  int32_t B, N, gamma, V, r;
  int32_t dtype;
  const void* target;         /* [B][N+1][V] target logits at the root and slots */
  const void* U;
  const void* W1;
  const void* W2;
  const int32_t* anchor;
  const float* temperature;
  const int32_t* parent;
  const uint8_t* mask;
  const int32_t* tokens;      /* [B][N] from spec_tree_draft                     */
  const float* u_accept;      /* [B][N]                                          */
  const float* u_final;       /* [B]                                             */
  int32_t* accept_len;        /* out [B]                                         */
  int32_t* out_tokens;        /* out [B][gamma+1]                                */
  int32_t* path;              /* out [B][gamma]                                  */
  uint32_t* dev_status;
  void* workspace;
  size_t workspace_bytes;
} spec_tree_verify_args;
int32_t spec_tree_verify(const spec_tree_verify_args* args, spec_stream_t stream);
size_t spec_tree_workspace_bytes(int32_t B, int32_t N, int32_t V);

/* ---------------------------------------------- operating-point report */
/* The analytic speed-up model of "Speculative Decoding Part 1: 도입 전에 확인해야
 * 할 것들" (VESSL AI blog), section "속도 향상을 결정하는 방정식" and the section on
 * the compute theorem, evaluated on the host (no GPU work).  With i.i.d.
 * acceptance probability alpha and draft cost ratio c = T_draft/(gamma T_target):
 * E[tau] = sum_{k<=gamma} alpha^k, S(gamma) = E[tau]/(c gamma + 1),
 * S <= min(1/c, 1/(1-alpha)), the stationarity condition
 * alpha^{gamma+1}(c - (c gamma + 1) ln alpha) = c, and the expected compute
 * ratio (gamma c_hat + gamma + 1)/E[tau].
 * Returns SPEC_EINVAL (nothing written) unless 0 <= alpha <= 1, c > 0,
 * c_hat >= 0, 1 <= gamma <= gamma_max <= 100000 and both pointers are set.  */
typedef struct {
  double alpha;              /* acceptance probability per position           */
  double c;                  /* draft cost ratio, > 0                          */
  double c_hat;              /* draft compute ratio (compute theorem), >= 0    */
  int32_t gamma;             /* draft length to evaluate                        */
  int32_t gamma_max;         /* search range 1..gamma_max for the best gamma    */
} spec_op_args;
typedef struct {
  double expected_tau;       /* E[tau] at gamma                                */
  double speedup;            /* S(gamma)                                       */
  double speedup_gamma1;     /* S(1) = (1 + alpha)/(c + 1)                     */
  double bound;              /* min(1/c, 1/(1 - alpha)); +inf terms dropped     */
  double gamma_continuous;   /* real root of the stationarity condition (0 if S
                                decreases from gamma = 0)                       */
  double speedup_star;       /* S(gamma_star)                                  */
  double compute_ratio;      /* expected compute relative to plain decoding    */
  int32_t gamma_star;        /* best integer gamma in 1..gamma_max (smallest on
                                ties)                                           */
  int32_t gains;             /* 1 if S(gamma) > 1                              */
} spec_op_result;
int32_t spec_operating_point(const spec_op_args* args, spec_op_result* out);

/* Measured acceptance statistics of one verification, on the device (no
 * counterpart formula beyond the report's inputs): out[0] = sum of alpha[b][j]
 * over j < L_b of valid requests, out[1] = the number of such positions,
 * out[2] = sum of (accept_len[b] + 1) over valid requests (accept_len >= 0),
 * out[3] = the number of valid requests.  alpha [B][gamma] and verify_len,
 * accept_len [B] are the spec_verify inputs/outputs (device pointers); out is
 * a device double[4], overwritten.  Enqueued on `stream`; SPEC_EINVAL for bad
 * sizes or NULL pointers.                                                    */
int32_t spec_acceptance_stats(int32_t B, int32_t gamma, const float* alpha,
                              const int32_t* verify_len, const int32_t* accept_len, double* out,
                              spec_stream_t stream);

/* Static text for a spec_status value. */
const char* spec_status_string(int32_t status);

/* ------------------------------------------------------ tuning / profiling */
/* Process-wide knobs (not thread-safe against concurrent calls):
 *   SPEC_OPT_EPS_SCALE   multiplies the near-boundary band (default 1.0)
 *   SPEC_OPT_FORCE_SIMT  1 = compute the bias with plain fp32 FMAs
 *   SPEC_OPT_BIAS_PATH   tensor path of the bf16 bias tiles: 1 = warp MMA,
 *                        2 = tcgen05 with the accumulator in tensor memory
 *                        (default; used when r % 64 == 0)
 *   SPEC_OPT_TRACE       1 = the persistent draft records globaltimer stamps
 *                        of its phase boundaries in the workspace (profiling)
 *   SPEC_OPT_PERTURB     1 = test hook: the draft runs a test build of its
 *                        kernel in which every draw queued for re-decision
 *                        first writes the next token instead of its own, so
 *                        the re-decision changes it and the draft's later
 *                        steps are redone (results unchanged)
 *   SPEC_OPT_TEST_STALL  1 = test hook: the draft runs a test build of its
 *                        kernel whose first grid barrier waits for one CTA
 *                        more than the grid has; the wait gives up after its
 *                        one-second limit, dev_status gets SPEC_DEV_TIMEOUT,
 *                        the outputs are left unspecified, and the kernel
 *                        returns with its copies drained and its tensor
 *                        memory freed (the CUDA context stays usable)
 *   SPEC_OPT_DRAFT_KERNEL  0 = the slice-resident draft kernel wherever the
 *                        shape fits it (default), 1 = always the tile-strided
 *                        draft kernel
 *   SPEC_OPT_VERIFY_KERNEL 0 = the slice-resident verification tiles wherever
 *                        the shape fits them (bf16, r % 64 == 0, V <= 256 x
 *                        SM count) and the re-decision of queued draws in one
 *                        cooperative launch (default); 1 = always the
 *                        tile-strided tiles and the two work-unit re-decision
 *                        passes
 * The two test hooks exist for the library's own tests; the default kernels
 * carry no trace of them.                                                   */
enum { SPEC_OPT_EPS_SCALE = 1, SPEC_OPT_FORCE_SIMT = 2, SPEC_OPT_BIAS_PATH = 3,
       SPEC_OPT_TRACE = 5, SPEC_OPT_PERTURB = 6, SPEC_OPT_TEST_STALL = 7,
       SPEC_OPT_DRAFT_KERNEL = 8, SPEC_OPT_VERIFY_KERNEL = 9 };   /* 4 is unused */
int32_t spec_set_option(int32_t key, double value);

/* Per-stage timing with CUDA events on the calls' streams.  enable(1)
 * starts recording, read() synchronizes the recorded events and returns, for
 * each stage id < n, the total milliseconds and launch count since the last
 * read (then clears them).  Stage names: spec_stage_name(id).              */
int32_t spec_profile_enable(int32_t on);
int32_t spec_profile_read(double* ms, int32_t* launches, int32_t n);
const char* spec_stage_name(int32_t id);
int32_t spec_num_stages(void);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_GB300_H */
