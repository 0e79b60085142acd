/*
 * hla.h -- C ABI of the GB300 (sm_103a) KDA + routed-MoE decode-step library.
 *
 * Sources the operations follow (by page title and section):
 *  [KIMI-WEBINAR]  "Kimi K3: From Day-0 Availability to Optimized Inference"
 *                  (webinar summary): KDA's fixed-size recurrent state; expert
 *                  weight streaming as the low-batch limit; speculative decoding
 *                  that stores drafted tokens' recurrent inputs and replays the
 *                  accepted portion from the last committed state; runtime
 *                  workspaces competing for memory.
 *  [VLLM-K3]       "Hyper-optimizing Kimi K3 in vLLM: Moving Fast and Responsibly",
 *                  Part 1 sec. 1 (small-matrix vs split-K projections, the KDA
 *                  decode kernel), sec. 2 (output projection + residual),
 *                  sec. 3 (router, routed and shared experts), sec. 4 (side-
 *                  stream prefetch of upcoming weights into L2).
 *  [K3-HF]         "Kimi-K3 release on HuggingFace", "Decoding the Model
 *                  Configuration": rms_norm_eps = 1e-6.
 *
 * The KDA update is the gated delta rule
 *     S_t = (I - beta_t k_t k_t^T) diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 *     o_t = S_t^T q_t,
 * S a d_k x d_v fp32 matrix per (sequence, head), alpha_t a per-key-channel
 * decay in (0,1) scaling the rows of S, beta_t a scalar per (token, head).
 *
 * Conventions for every entry point
 *  - Returns an hla_status (0 = HLA_OK).  Work is enqueued on `stream`
 *    (a cudaStream_t; NULL = the legacy default stream) and is asynchronous:
 *    no entry point synchronises the device or the stream.
 *  - Every pointer is a DEVICE pointer owned by the caller.  The library never
 *    allocates or frees device memory; operations that need scratch take a
 *    caller-owned workspace whose size comes from the matching
 *    *_workspace_size() query.  A workspace smaller than that returns
 *    HLA_ERR_WORKSPACE without launching anything.
 *  - Tensors are dense row-major with the shapes given; bf16 tensors hold raw
 *    bfloat16 bit patterns (hla_bf16).  Every tensor pointer must be 16-byte
 *    aligned (128-bit loads/stores); otherwise HLA_ERR_MISALIGNED.
 *  - Arguments are validated on the host before any launch; invalid ones return
 *    HLA_ERR_INVALID_ARG / HLA_ERR_UNSUPPORTED and leave all buffers untouched.
 *  - A failed launch returns HLA_ERR_CUDA (cudaGetLastError is consumed).
 *  - Entry points keep no state between calls apart from: the device status word
 *    (hla_device_status), the calling thread's last-variant string, the
 *    instrumentation counters, per-device cached attributes, per-thread and per-device events
 *    of the side-stream fork/join, the calling thread's open launch chain
 *    (hla_chain_begin), and the one scratch array shared by every
 *    skinny_proj_splitk_noalloc call.  Calls on different streams may run
 *    concurrently when their buffers do not overlap (skinny_proj_splitk_noalloc
 *    excepted: see there).
 *  - Projections of 32 or more tokens run on the tensor-core path, whose
 *    pipeline waits are bounded: a wait that gives up does not fail the launch
 *    but sets the device status word.  Every entry point that can reach that path
 *    (skinny_proj_splitk, skinny_proj_splitk_noalloc, skinny_proj_residual_rmsnorm,
 *    kda_qkvg_proj, moe_route_topk, moe_expert_forward, hla_decode_layer) can
 *    therefore return HLA_OK with invalid outputs; a caller that must know checks
 *    hla_device_status() after synchronising.
 *  - Results are deterministic: every reduction runs in a fixed order, so the
 *    same inputs give bit-identical outputs run to run.
 */
#ifndef HLA_H
#define HLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t hla_bf16;               /* bfloat16 bit pattern */
typedef struct CUstream_st *hla_stream;  /* identical to cudaStream_t */

enum hla_status {
    HLA_OK = 0,
    HLA_ERR_INVALID_ARG = 1,     /* null pointer, non-positive or inconsistent size */
    HLA_ERR_UNSUPPORTED = 2,     /* a shape outside what the kernels implement */
    HLA_ERR_MISALIGNED = 3,      /* a tensor pointer not 16-byte aligned */
    HLA_ERR_WORKSPACE = 4,       /* workspace null or smaller than the query returns */
    HLA_ERR_CUDA = 5,            /* a CUDA runtime call or launch failed */
    HLA_ERR_DEVICE_TIMEOUT = 6   /* a bounded device-side wait gave up */
};

enum hla_dtype { HLA_F32 = 0, HLA_BF16 = 1 };

enum hla_spec_phase { HLA_SPEC_VERIFY = 1, HLA_SPEC_REPLAY = 2, HLA_SPEC_BOTH = 3 };

/* Human-readable text for a status value (static storage). */
const char *hla_status_string(int status);

/* Name of the kernel variant the calling thread's most recent entry point
 * launched (e.g. "kda_recur<dk128,cw16,decode>"), for tests that must prove which
 * path ran.  Static/thread-local storage; "" before the first call. */
const char *hla_last_variant(void);

/* Library ABI version (major*100 + minor). */
int hla_version(void);

/* ---------------------------------------------------------------------------
 * Launch chains.  No counterpart on the source pages: a scheduling contract for callers that
 * queue several library calls back to back (a decode step: the layer, then the speculative
 * window's verify, accept and replay).
 * hla_chain_begin(stream) declares that the library calls this host thread makes on `stream`
 * until hla_chain_end() follow one another with nothing else queued on that stream between
 * them (no kernel, copy or event of the caller's).  Every kernel of those calls after the
 * chain's first is then launched as a programmatic dependent of the one before it: it may
 * start while its predecessor finishes, loads only data its predecessor does not write (static
 * weights, its own state) and waits for the predecessor before reading anything else.  Results
 * are bit-identical to plain launches.  What a kernel reads before its wait is the weights and
 * norm gains of its own call: inside a chain these must not be written by the call right before
 * it (weights are static in the decode loop).  Side streams are not part of the chain.  One chain
 * per host thread: a second hla_chain_begin, or hla_chain_end without one, returns
 * HLA_ERR_INVALID_ARG.  Every entry point that launches several kernels (hla_decode_layer,
 * kda_qkvg_proj, skinny_proj_splitk and its no-allocation form, skinny_proj_residual_rmsnorm,
 * moe_route_topk, moe_expert_forward) chains its own kernels at up to 32 tokens (the environment
 * variable HLA_PDL=0 / 1 turns that off / on at any size) and, inside a caller's chain on the same
 * stream, continues it.  Its first kernel follows whatever the caller queued before it.
 * -------------------------------------------------------------------------*/
int hla_chain_begin(hla_stream stream);
int hla_chain_end(void);

/* ---------------------------------------------------------------------------
 * KDA decode step.  [KIMI-WEBINAR] fixed-size recurrent state; [VLLM-K3]
 * Part 1 sec. 1, KDA decode kernel tuned to batch size and heads.
 *
 * One token per sequence: for every (b, h)
 *   S[slot(b), h] <- (I - beta k k^T) diag(alpha) S[slot(b), h] + beta k v^T
 *   o[b, h]       <- S[slot(b), h]^T q            (read from the updated state)
 *  B >= 1 sequences, H >= 1 heads, dk = dv in {64, 128}.
 *  S          fp32 [n_slots, H, dk, dv], updated in place.
 *  state_idx  int32 [B] slot of each sequence (distinct, < n_slots), or NULL
 *             for slot(b) = b.
 *  q, k       bf16 [B, H, dk]   (the kernels do not normalise them)
 *  v          bf16 [B, H, dv]
 *  alpha      fp32 [B, H, dk]   per-key-channel decay
 *  beta       fp32 [B, H]
 *  o          [B, H, dv], fp32 (o_dtype = HLA_F32) or bf16 (HLA_BF16).
 * -------------------------------------------------------------------------*/
int kda_decode_step(int B, int H, int dk, int dv, float *S, const int32_t *state_idx,
                    const hla_bf16 *q, const hla_bf16 *k, const hla_bf16 *v,
                    const float *alpha, const float *beta, void *o, int o_dtype,
                    hla_stream stream);

/* ---------------------------------------------------------------------------
 * Speculative window over T drafted tokens.  [KIMI-WEBINAR] speculative
 * decoding paragraphs: the target verifies drafted tokens; the drafted tokens'
 * recurrent inputs are kept; after acceptance only the accepted prefix is
 * replayed from the last committed state.
 *
 * The caller keeps the window's inputs (q, k, v, alpha, beta with a draft axis)
 * in its own buffers between the two phases.
 *  phase = HLA_SPEC_VERIFY: for every (b, h) apply the T tokens in order to a
 *          private on-chip copy of S[slot(b), h]; write o[b, t, h] for every t.
 *          S is read only and never written.  accepted_len is ignored.
 *  phase = HLA_SPEC_REPLAY: for every b with a = accepted_len[b] > 0, apply the
 *          first a tokens in order to S[slot(b), h] and store the result; for
 *          a = 0 the state is not touched at all.  o is ignored (may be NULL).
 *          accepted_len values are clamped to [0, T].
 *  phase = HLA_SPEC_BOTH returns HLA_ERR_UNSUPPORTED and launches nothing.  The
 *          accepted length of a window comes from the target's tokens, which the
 *          target model computes from the verify outputs of that same window, so
 *          a window's verify and its replay cannot share one call.  The one-pass
 *          form of a speculative step is kda_spec_replay_verify: the replay of the
 *          previous window's accepted prefix fused with the verify of the next.
 *  1 <= T <= 8; q, k [B, T, H, dk] bf16; v [B, T, H, dv] bf16;
 *  alpha [B, T, H, dk] fp32; beta [B, T, H] fp32; accepted_len int32 [B];
 *  o [B, T, H, dv] (o_dtype).  Other arguments as kda_decode_step.
 * Replaying all T tokens gives bit-identical state to T kda_decode_step calls
 * with the same inputs (same per-step arithmetic and reduction order).
 * -------------------------------------------------------------------------*/
int kda_spec_verify_replay(int phase, int B, int T, int H, int dk, int dv, float *S,
                           const int32_t *state_idx, const hla_bf16 *q, const hla_bf16 *k,
                           const hla_bf16 *v, const float *alpha, const float *beta,
                           const int32_t *accepted_len, void *o, int o_dtype,
                           hla_stream stream);

/* ---------------------------------------------------------------------------
 * Replay of the previous window fused with the verify of the next one.  [KIMI-WEBINAR]
 * speculative decoding: only the accepted portion of the last window is replayed from the
 * last committed state, and the next drafted window is verified from the new committed
 * state.  One pass over the state does both, so each (sequence, head) state is read once
 * and written once per speculative step instead of read twice.
 *  For every (b, h): from S[slot(b), h] apply the first a = accepted_prev[b] tokens of the
 *  previous window (clamped to [0, T_prev]); if a > 0 store the result as the committed state;
 *  then apply the T tokens of the new window to a private copy and write o[b, t, h] for every t
 *  (the new window is not committed).
 *  q_prev, k_prev [B, T_prev, H, dk] bf16, v_prev [B, T_prev, H, dv] bf16, alpha_prev fp32
 *  [B, T_prev, H, dk], beta_prev fp32 [B, T_prev, H]; accepted_prev int32 [B]; the new window
 *  q, k, v, alpha, beta with T in place of T_prev; o [B, T, H, dv] (o_dtype).
 *  1 <= T_prev, T <= 8.  Bit-identical to kda_spec_verify_replay(REPLAY) on the previous window
 *  followed by kda_spec_verify_replay(VERIFY) on the new one.
 * -------------------------------------------------------------------------*/
int kda_spec_replay_verify(int B, int T_prev, int T, int H, int dk, int dv, float *S,
                           const int32_t *state_idx, const hla_bf16 *q_prev, const hla_bf16 *k_prev,
                           const hla_bf16 *v_prev, const float *alpha_prev, const float *beta_prev,
                           const int32_t *accepted_prev, const hla_bf16 *q, const hla_bf16 *k,
                           const hla_bf16 *v, const float *alpha, const float *beta, void *o,
                           int o_dtype, hla_stream stream);

/* ---------------------------------------------------------------------------
 * Mixed batch: every sequence brings its own number of new tokens (one for a decoding
 * sequence, many for a prefill chunk).  [VLLM-K3] "What's Next": the decode path falls back
 * seamlessly for prefills and mixed batches.
 *  Sequence b owns the packed token rows cu_seqlens[b] .. cu_seqlens[b+1]-1; for every (b, h)
 *  those tokens are applied in order to S[slot(b), h] (gated delta rule, as kda_decode_step),
 *  o is written for every token, and the final state is stored.  A sequence with no tokens is
 *  not touched.
 *  cu_seqlens int32 [B + 1] (device, non-decreasing, cu_seqlens[0] = 0); q, k bf16 [N, H, dk];
 *  v bf16 [N, H, dv]; alpha fp32 [N, H, dk]; beta fp32 [N, H]; o [N, H, dv] (o_dtype), where
 *  N = cu_seqlens[B].  The tokens of one sequence are applied one after another with the state
 *  held on chip (the recurrent form); every step is bit-identical to kda_decode_step.
 * -------------------------------------------------------------------------*/
int kda_extend(int B, const int32_t *cu_seqlens, int H, int dk, int dv, float *S,
               const int32_t *state_idx, const hla_bf16 *q, const hla_bf16 *k, const hla_bf16 *v,
               const float *alpha, const float *beta, void *o, int o_dtype, hla_stream stream);

/* ---------------------------------------------------------------------------
 * Accepted-length bookkeeping.  [KIMI-WEBINAR] speculative decoding: greedy
 * acceptance of the drafted tokens the target agrees with.
 *  accepted_len[b]  = number of leading t with draft_ids[b,t] == target_ids[b,t]
 *  committed_len[b] += accepted_len[b]
 *  draft_ids, target_ids int32 [B, T] (1 <= T <= 64); accepted_len int32 [B] out;
 *  committed_len int32 [B] in/out.  Integer, bit-exact.
 * -------------------------------------------------------------------------*/
int spec_accept_prefix(int B, int T, const int32_t *draft_ids, const int32_t *target_ids,
                       int32_t *accepted_len, int32_t *committed_len, hla_stream stream);

/* ---------------------------------------------------------------------------
 * Skinny projection y = x W^T (+ residual).  [VLLM-K3] Part 1 sec. 1: small-
 * matrix kernel at batch 1-2, split-K (K divided across CTAs, then reduced)
 * above; sec. 2: the output projection feeds the residual add.
 *  x bf16 [M, K]; W bf16 [N, K]; residual bf16 [M, N] or NULL;
 *  y [M, N] fp32 or bf16 (y_dtype).  1 <= M <= 256, K % 32 == 0, N >= 1.
 *  split = number of K slices (0 = automatic by M, N, K).  split > 1 writes
 *  fp32 partials into the workspace and a second kernel sums them in increasing
 *  slice order, then adds the residual (fixed order: deterministic).
 *  Below 32 tokens, with N % 32 == 0 and every K slice at least 128 values long,
 *  persistent warps keep their weight loads running from one work item into the
 *  next (variant "xi"; HLA_DENSE_XITEM=0 runs one item per warp instead, with the
 *  same results bit for bit).
 * -------------------------------------------------------------------------*/
size_t skinny_proj_splitk_workspace_size(int M, int N, int K, int split);
int skinny_proj_splitk(int M, int N, int K, const hla_bf16 *x, const hla_bf16 *W,
                       const hla_bf16 *residual, void *y, int y_dtype, int split,
                       void *ws, size_t ws_bytes, hla_stream stream);

/* ---------------------------------------------------------------------------
 * Output projection + residual + the following RMSNorm in one pass over the result.
 * [KIMI-WEBINAR] fusing the residual addition and normalisation into the projection;
 * [VLLM-K3] Part 1 sec. 2 (the single-GPU part: projection, then the attention residual).
 *  r  = residual + x W^T            stored bf16 [M, N]   (residual bf16 [M, N] or NULL)
 *  xn = r * gamma / sqrt(mean(r^2) + eps)   over each row, stored bf16 [M, N]
 *  x bf16 [M, K]; W bf16 [N, K]; gamma bf16 [N]; K % 32 == 0, N % 8 == 0, 1 <= M <= 256.
 *  split as skinny_proj_splitk (0 = automatic; below 32 tokens the automatic split is at
 *  most 8, since the normalising pass reads every slice of each of its columns).  Bit-identical
 *  to skinny_proj_splitk (bf16 output) followed by hla_rmsnorm with the same split.  The
 *  workspace holds the fp32 split partials (at least one slice).
 * -------------------------------------------------------------------------*/
size_t skinny_proj_residual_rmsnorm_workspace_size(int M, int N, int K, int split);
int skinny_proj_residual_rmsnorm(int M, int N, int K, const hla_bf16 *x, const hla_bf16 *W,
                                 const hla_bf16 *residual, const hla_bf16 *gamma, float eps,
                                 hla_bf16 *r, hla_bf16 *xn, int split, void *ws, size_t ws_bytes,
                                 hla_stream stream);

/* ---------------------------------------------------------------------------
 * KDA input projection with its epilogue (decode layer).  [VLLM-K3] Part 1
 * sec. 1 (attention input projections) feeding the KDA decode kernel.
 *  z = x W^T, W bf16 [(3*dk + dv)*H + H, Hd] with row blocks
 *      [q (H*dk) | k (H*dk) | v (H*dv) | g (H*dk) | b (H)];
 *  q = z_q / ||z_q|| per head, k likewise (bf16 [M, H, dk]); v bf16 [M, H, dv];
 *  alpha = exp(-softplus(g)) fp32 [M, H, dk]; beta = sigmoid(b) fp32 [M, H].
 *  x bf16 [M, Hd], Hd % 32 == 0, 1 <= M <= 256, dk = dv in {64, 128}.
 * -------------------------------------------------------------------------*/
size_t kda_qkvg_proj_workspace_size(int M, int Hd, int H, int dk, int dv, int split);
int kda_qkvg_proj(int M, int Hd, int H, int dk, int dv, const hla_bf16 *x, const hla_bf16 *W,
                  hla_bf16 *q, hla_bf16 *k, hla_bf16 *v, float *alpha, float *beta,
                  int split, void *ws, size_t ws_bytes, hla_stream stream);

/* ---------------------------------------------------------------------------
 * RMSNorm.  [KIMI-WEBINAR] normalisation next to the residual adds; eps per
 * [K3-HF] (callers pass it).  y = x * gamma / sqrt(mean(x^2) + eps), fp32 math.
 *  x, y bf16 [M, Hd] (may alias); gamma bf16 [Hd]; Hd % 8 == 0.
 * -------------------------------------------------------------------------*/
int hla_rmsnorm(int M, int Hd, const hla_bf16 *x, const hla_bf16 *gamma, float eps,
                hla_bf16 *y, hla_stream stream);

/* ---------------------------------------------------------------------------
 * Router: fp32 logits x W_r^T, sigmoid scores, top-k.  [VLLM-K3] Part 1 sec. 3.
 *  Selection is on the fp32 logits (sigmoid is monotone), largest first, ties
 *  to the lower expert index; topk_idx lists the chosen experts by descending
 *  score; topk_w = sigmoid(logit) / sum over the chosen k.
 *  x bf16 [M, Hd]; W_r bf16 [E, Hd]; topk_idx int32 [M, k]; topk_w fp32 [M, k];
 *  logits fp32 [M, E] or NULL.  1 <= k <= 16, k <= E <= 1024, Hd % 32 == 0.
 * -------------------------------------------------------------------------*/
size_t moe_route_topk_workspace_size(int M, int Hd, int E);
int moe_route_topk(int M, int Hd, int E, int k, const hla_bf16 *x, const hla_bf16 *W_r,
                   int32_t *topk_idx, float *topk_w, float *logits, void *ws, size_t ws_bytes,
                   hla_stream stream);

/* ---------------------------------------------------------------------------
 * Routed + shared SwiGLU experts.  [KIMI-WEBINAR] expert weights streamed
 * through memory are the low-batch limit; [VLLM-K3] Part 1 sec. 3 (routed and
 * shared experts) and sec. 4 (L2 prefetch of upcoming weights on a side stream).
 *  y[m] = sum_j topk_w[m,j] * E_{topk_idx[m,j]}(x[m]) + sum_s E^shared_s(x[m])
 *         (+ residual[m]),  E(x) = W_down (SiLU(W_gate x) * (W_up x)).
 *  The slots are summed in fixed order (routed j = 0..k-1, then shared).
 *  x bf16 [M, Hd]; topk_idx int32 [M, k] (values in [0, E)); topk_w fp32 [M, k];
 *  W_gate, W_up bf16 [E, I, Hd]; W_down bf16 [E, Hd, I]; Ws_* the same with
 *  n_shared in place of E (NULL when n_shared = 0); residual bf16 [M, Hd] or
 *  NULL; y bf16 [M, Hd].  Hd % 32 == 0, I % 32 == 0, 1 <= M <= 256,
 *  1 <= k <= 16, E + n_shared <= 1024, 0 <= n_shared <= 16.
 *  Each active expert's weights are read once per call for all of its tokens.
 *  Persistent warps claim work items and keep their weight loads running from one
 *  item into the next when every K slice is long enough (variant flags "xgu" and
 *  "xdn"; HLA_MOE_XITEM=0 stops the loads at each item instead, with the same
 *  results bit for bit).
 *  prefetch_stream: NULL, or a second stream on which an L2 prefetch of the
 *  shared experts' weights runs while routing bookkeeping runs on `stream`;
 *  `stream` joins it before returning, so the call stays capturable as one
 *  graph branch.  Results are bit-identical with and without it.
 *  With HLA_SHARED_STREAM=1 in the environment the same stream instead runs
 *  the shared experts as dense SwiGLU products, concurrently with the routed
 *  experts (the shared expert does not depend on the routing: same page,
 *  Part 1 sec. 3); `stream` joins it before the final combine.  The shared
 *  experts' sums then run in another order, so results differ from the
 *  default placement in the last bits (within the MoE tolerance).
 * -------------------------------------------------------------------------*/
size_t moe_expert_forward_workspace_size(int M, int Hd, int I, int E, int k, int n_shared);
int moe_expert_forward(int M, int Hd, int I, int E, int k, int n_shared, const hla_bf16 *x,
                       const int32_t *topk_idx, const float *topk_w, const hla_bf16 *W_gate,
                       const hla_bf16 *W_up, const hla_bf16 *W_down, const hla_bf16 *Ws_gate,
                       const hla_bf16 *Ws_up, const hla_bf16 *Ws_down, const hla_bf16 *residual,
                       hla_bf16 *y, void *ws, size_t ws_bytes, hla_stream stream,
                       hla_stream prefetch_stream);

/* ---------------------------------------------------------------------------
 * L2 prefetch of a byte range of static weights.  [VLLM-K3] Part 1 sec. 4:
 * while a phase cannot use the memory bandwidth, a side-stream kernel pulls the
 * next operation's weights into cache.  Changes no data.  ptr 16-byte aligned.
 * -------------------------------------------------------------------------*/
int hla_l2_prefetch(const void *ptr, size_t bytes, hla_stream stream);

/* ---------------------------------------------------------------------------
 * One hybrid decode layer (executor over the entry points above).
 *  x -> RMSNorm -> kda_qkvg_proj -> kda_decode_step (S in place) ->
 *  o-projection + residual -> RMSNorm -> router -> routed + shared experts
 *  + residual -> y.  [VLLM-K3] Part 1 secs. 1-4; [KIMI-WEBINAR].
 * All pointers in hla_layer are device pointers to static weights.
 * -------------------------------------------------------------------------*/
typedef struct hla_layer {
    int hidden;            /* Hd */
    int heads;             /* H */
    int dk, dv;
    int n_experts, top_k, inter, n_shared;
    float eps;             /* RMSNorm epsilon */
    const hla_bf16 *gamma_attn, *gamma_moe;   /* [Hd] */
    const hla_bf16 *W_qkvgb;                  /* [(3*dk+dv)*H + H, Hd] */
    const hla_bf16 *W_o;                      /* [Hd, H*dv] */
    const hla_bf16 *W_router;                 /* [E, Hd] */
    const hla_bf16 *W_gate, *W_up, *W_down;   /* [E, I, Hd], [E, I, Hd], [E, Hd, I] */
    const hla_bf16 *Ws_gate, *Ws_up, *Ws_down;
} hla_layer;

/*  M sequences (one token each, 1 <= M <= 256); x, y bf16 [M, Hd] (distinct);
 *  S fp32 [n_slots, H, dk, dv] in place; state_idx as kda_decode_step.
 *  prefetch_stream as moe_expert_forward (NULL = no prefetch); with HLA_SHARED_STREAM=1
 *  the shared experts are forked onto it right after the second RMSNorm, before the router.
 *  All scratch is in ws (hla_decode_layer_workspace_size bytes, 16-byte aligned). */
size_t hla_decode_layer_workspace_size(const hla_layer *L, int M);
int hla_decode_layer(const hla_layer *L, int M, const hla_bf16 *x, float *S,
                     const int32_t *state_idx, hla_bf16 *y, void *ws, size_t ws_bytes,
                     hla_stream stream, hla_stream prefetch_stream);

/* Device pointers, inside a workspace last passed to hla_decode_layer with the same L and
 * M, of that call's routing decision: topk_idx int32 [M, top_k] and topk_w fp32 [M, top_k].
 * Valid until the workspace is reused.  Returns HLA_ERR_INVALID_ARG on bad arguments. */
int hla_decode_layer_routing(const hla_layer *L, int M, const void *ws, const int32_t **topk_idx,
                             const float **topk_w);

/* ---------------------------------------------------------------------------
 * skinny_proj_splitk without a workspace.  No counterpart on the source pages: this is
 * a convenience for callers that cannot allocate device memory when they run a
 * projection -- for example a server that fixes its whole device-memory budget at
 * start-up so that no request can later fail for lack of a workspace, a plugin whose
 * host application owns every allocation, or code on a path where a cudaMalloc would
 * stall the device.  It computes exactly what skinny_proj_splitk computes, with the same
 * arguments except the workspace, and allocates nothing: the split-K partials live in
 * one fixed device array of HLA_NOALLOC_SCRATCH_BYTES (16 MiB) inside the library, which
 * every GPU that loads the library keeps until the process exits.
 *  - The split is the one skinny_proj_splitk would use; when its partials
 *    (split x M x N x 4 bytes) do not fit the array the call returns HLA_ERR_WORKSPACE
 *    and launches nothing (pass a smaller split, e.g. 1, which needs no scratch).
 *  - Every call asks the runtime for the array's device address on the current device
 *    (a host-side lookup, so a device reset cannot leave a stale address behind).  The
 *    first call on a device may also load the library's device code there; make that
 *    first call before any stream capture.
 *  - At 32 or more tokens it runs on the tensor-core path: check hla_device_status()
 *    as the conventions above say.
 *  - All calls share the one array, so calls that can overlap on the GPU (different
 *    streams, or different host threads) race and give wrong results: serialise them.
 *    The array keeps the last call's partials; each call overwrites every partial it
 *    reads, so no clearing is needed.
 * -------------------------------------------------------------------------*/
#define HLA_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
int skinny_proj_splitk_noalloc(int M, int N, int K, const hla_bf16 *x, const hla_bf16 *W,
                               const hla_bf16 *residual, void *y, int y_dtype, int split,
                               hla_stream stream);

/* ---------------------------------------------------------------------------
 * Instrumentation (off by default; for profiling tools and benchmarks).
 * hla_launch_count: number of kernels this library has launched in the process.
 * hla_trace_enable: time every launch of one kernel family with a CUDA event pair
 *   recorded on the launching stream around it; kernel is one of "kda", "dense",
 *   "moe_gateup", "moe_down"; capacity = launches to keep (0 disables).  The events
 *   are created here, once, when tracing is enabled (not during stream capture).
 * hla_trace_read: wait for the recorded events, write up to max_n elapsed times
 *   (milliseconds) in launch order, return how many were recorded (<= capacity).
 * Not thread-safe; meant for one benchmarking thread.
 * -------------------------------------------------------------------------*/
unsigned long long hla_launch_count(void);
/* Reads and clears the device status word: 0, or HLA_ERR_DEVICE_TIMEOUT when a bounded
 * device-side wait (the tensor-core projection's pipeline barriers) gave up since the last
 * read.  Synchronous (copies 4 bytes from the device); HLA_ERR_CUDA if that copy fails. */
int hla_device_status(void);
/* Test hook for the failure path, with no counterpart on the source pages.  While on != 0,
 * every tensor-core projection launch makes one of its bounded device waits give up (block 0
 * waits 1 ms on a barrier that nothing arrives at) and records HLA_ERR_DEVICE_TIMEOUT, and
 * every block returns before it allocates tensor memory or issues a copy or an MMA; the
 * launch writes no output.  This lets a test check the status path without a real stall.
 * Takes effect for launches made after the call (a CUDA graph keeps what it captured);
 * process-wide, not thread-safe with concurrent launches.  Always returns HLA_OK. */
int hla_test_force_wait_timeout(int on);
int hla_trace_enable(const char *kernel, int capacity);
int hla_trace_read(float *ms_out, int max_n);

#ifdef __cplusplus
}
#endif

#endif /* HLA_H */
