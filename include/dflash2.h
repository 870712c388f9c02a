/*
 * dflash2.h -- C ABI of the DFlash 2 draft-block head for NVIDIA GB300 (sm_103a).
 *
 * The draft-block head turns a parallel drafter's per-position outputs into one
 * coherent draft block and verifies it ("DFlash 2: Keep Drafting Parallel",
 * Inco AI):
 *   dflash2_topk          top-16 candidates per block position
 *   dflash2_pair_scores   context gate + pairwise path-selector scores
 *   dflash2_pair_scores_proj  the same scores with A, B projected from E
 *   dflash2_walk          greedy or temperature-sampled walk over the scores
 *   dflash2_walk_viterbi  exact best path over the same scores
 *   dflash2_selector_eval Table 1's recall and acceptance-length evaluation
 *   dflash2_conv2tap      two-tap dynamic depthwise convolution
 *   dflash2_gemm_conv2tap the same conv fused into its producing GEMM
 *   dflash2_verify        block verification -> acceptance lengths
 *   dflash2_lmhead_topk   LM head GEMM with a streaming top-16 epilogue
 *   dflash2_lmhead_topk_gate  the same with the context gate folded in
 *
 * Conventions for every call
 *   - Pointers marked "device" are CUDA device pointers on the handle's device;
 *     "host" pointers are ordinary host memory.  The caller owns every buffer:
 *     the library never frees a pointer or keeps one past the call.  The only
 *     allocation the library makes is the handle's 4-byte error word, in
 *     dflash2_create; calls that need scratch take a caller workspace whose
 *     size a *_workspace query gives (dflash2_lmhead_topk_noalloc uses a fixed
 *     array inside the library instead).
 *   - The handle's device must be the calling thread's current device
 *     (cudaSetDevice); a compute call made while another device is current
 *     returns DFLASH2_ERR_INVALID_ARG before anything launches.
 *   - bf16 tensors are passed as `const uint16_t*` holding bf16 bit patterns.
 *   - Tensors are row-major and contiguous unless an explicit leading dimension
 *     (`ld`, in elements) is given.  bf16 base pointers must be 16-byte aligned
 *     and `ld` a multiple of 8; fp32/int32 pointers 4-byte aligned.
 *   - Token ids are int32; V must be < 2^31.  K (candidates per position) is 16.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  Outputs are valid once the stream reaches the call.
 *   - The return value is a dflash2_status.  Argument errors are detected on
 *     the host before anything is launched and leave outputs untouched.  No C++
 *     exception crosses this ABI.
 *   - Data-dependent errors found on the device (an out-of-range token id, a
 *     bounded wait that gave up) never fault: the kernel clamps the access,
 *     ORs a DFLASH2_DEVERR_* bit into the handle's device error word and
 *     continues; read it with dflash2_get_device_error().
 *   - A handle may be used from one host thread at a time.  Calls that share a
 *     handle but run on different streams only share the error word.
 */
#ifndef DFLASH2_H
#define DFLASH2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dflash2_handle dflash2_handle;

enum dflash2_status {
  DFLASH2_OK = 0,
  DFLASH2_ERR_INVALID_ARG = -1, /* null pointer, negative or inconsistent size      */
  DFLASH2_ERR_UNSUPPORTED = -2, /* k != 16, V < 16, d % 64 != 0, L > 64, ...         */
  DFLASH2_ERR_MISALIGNED = -3,  /* a pointer or leading dimension breaks alignment  */
  DFLASH2_ERR_CUDA = -4,        /* a CUDA runtime call or kernel launch failed      */
  DFLASH2_ERR_TIMEOUT = -5,     /* a bounded device wait gave up (see error word)   */
  DFLASH2_ERR_DEVICE = -6,      /* the device error word is non-zero                */
  DFLASH2_ERR_WORKSPACE = -7    /* the caller's workspace is too small              */
};

/* Bits of the device error word. */
#define DFLASH2_DEVERR_BAD_TOKEN 0x1u /* a token id outside [0, V) was clamped     */
#define DFLASH2_DEVERR_TIMEOUT 0x2u   /* a bounded wait (TMA / mbarrier) gave up  */
#define DFLASH2_DEVERR_BAD_SLOT 0x4u  /* a draft slot outside [0, 16) was clamped */

/* Library version: major * 10000 + minor * 100 + patch. */
int dflash2_version(void);

/* Human-readable name of a dflash2_status value (static storage). */
const char* dflash2_status_string(int status);

/*
 * Creates a handle bound to CUDA device `device`.  Allocates the 4-byte device
 * error word (the library's only allocation) and records the SM count.  Makes
 * `device` current on the calling thread.
 */
int dflash2_create(int device, dflash2_handle** out);

/* Frees the handle and its error word.  Synchronises the device first. */
int dflash2_destroy(dflash2_handle* h);

/* Number of SMs of the handle's device (host). */
int dflash2_num_sms(const dflash2_handle* h);

/*
 * Synchronises `stream`, copies the device error word to *bits (host) and, if
 * `clear` is non-zero, resets it to 0 (without `clear` a caller can poll the
 * word and leave its bits for another reader).
 */
int dflash2_get_device_error(dflash2_handle* h, void* stream, uint32_t* bits, int clear);

/*
 * Top-k candidates per row.  "A Lightweight Path Selector": DFlash 2 keeps the
 * top 16 candidates of the drafter's own logits U_t at every block position.
 *
 *   logits  device bf16 [rows, ld]; only columns [0, V) are read.
 *   vals    device fp32 [rows, k]  -- the candidates' logits (exact bf16 values)
 *   idx     device int32 [rows, k] -- their vocabulary ids
 * Order: value descending, ties by lowest id; -0 == +0; NaN ranks below -inf.
 * k must be 16; 16 <= V < 2^31; ld >= V, ld % 8 == 0; logits 16-byte aligned.
 * rows == 0 is a no-op.  No workspace: rows with few positions are split over a
 * thread-block cluster whose partial lists meet in distributed shared memory.
 */
int dflash2_topk(dflash2_handle* h, const uint16_t* logits, int64_t rows, int64_t V, int64_t ld,
                 int k, float* vals, int32_t* idx, void* stream);

/*
 * Context gate and pairwise path-selector scores.  "A Lightweight Path
 * Selector", score equation S_t(a,b) = U_t(b) + <A(a) (.) H(h_t), B(b)>:
 *
 *   H[b,t,:]   = sigmoid(W_H h[b,t,:] + b_H)                       (r = 256)
 *   S[b,t,i,j] = cand_val[b,t,j] + sum_q A[p_i,q] H[b,t,q] Bt[cand_idx[b,t,j],q]
 *   p_i = cand_idx[b,t-1,i] for t >= 1; p_i = last_verified[b] for t = 0, so the
 *   16 rows of S[b,0] are equal.
 *
 *   cand_idx, cand_val  device [B, L, 16] int32 / fp32 (dflash2_topk's output)
 *   last_verified       device int32 [B]
 *   hs                  device bf16 [B, L, d] drafter hidden states
 *   W_H                 device bf16 [256, d];  b_H device fp32 [256] or NULL (= 0)
 *   A, Bt               device bf16 [V, 256] predecessor / candidate embeddings
 *   gate                device fp32 [B, L, 256] output: H
 *   S                   device fp32 [B, L, 16, 16] output
 *   workspace           device scratch of at least dflash2_pair_scores_workspace(h, B,
 *                       L, d) bytes, 256-byte aligned: the gate contraction's fp32
 *                       split-K partials, rewritten by every call; calls that overlap
 *                       on the GPU must not share it.  The partials are summed in a
 *                       fixed order, so H has the same bits on every call.
 * Precision: the sum over q accumulates in fp32 on the tensor cores; each
 * product A[p_i,q] H[b,t,q] (an fp32 value) enters as its bf16 rounding plus the
 * bf16 rounding of the remainder, which carries it to about 2^-16 of its size.
 * d % 64 == 0, L <= 64.  Ids outside [0, V) are clamped and flagged.  A too-small
 * or NULL workspace returns DFLASH2_ERR_WORKSPACE.
 */
size_t dflash2_pair_scores_workspace(const dflash2_handle* h, int64_t B, int64_t L, int64_t d);
int dflash2_pair_scores(dflash2_handle* h, const int32_t* cand_idx, const float* cand_val,
                        const int32_t* last_verified, const uint16_t* hs, const uint16_t* W_H,
                        const float* b_H, const uint16_t* A, const uint16_t* Bt, int64_t B,
                        int64_t L, int64_t d, int64_t V, float* gate, float* S, void* workspace,
                        size_t ws_bytes, void* stream);

/*
 * Pair scores in projection form.  The score equation of "A Lightweight Path
 * Selector" matches 256-dimensional embeddings of the predecessor and the
 * candidate; here they are projections of the shared token embedding E,
 *   A(a) = W_A E(a),   B(b) = W_B E(b),
 * computed on the tensor cores (fp32 accumulation, not rounded) for exactly
 * the tokens of the step, then
 *   S[b,t,i,j] = cand_val[b,t,j] + sum_r A(pred_i)_r H[b,t,r] B(cand_j)_r
 * with the predecessors of dflash2_pair_scores.
 *   cand_idx, cand_val  device [B, L, 16] int32 / fp32
 *   last_verified       device int32 [B]
 *   gate                device fp32 [B, L, 256]: H, 16-byte aligned (e.g. the gate
 *                       output of dflash2_lmhead_topk_gate or dflash2_pair_scores)
 *   E                   device bf16 [V, d] shared token embedding
 *   W_A, W_B            device bf16 [256, d]
 *   P, P_bytes          device fp32 workspace of at least
 *                       dflash2_pair_scores_proj_workspace(h, B, L) bytes, 16-byte
 *                       aligned; on return it holds the projections, row
 *                       (b*L + t)*16 + j for candidate j of (b, t), then row
 *                       B*L*16 + b for last_verified[b]; each row is A (256) then B (256)
 *   S                   device fp32 [B, L, 16, 16] output
 * d % 64 == 0, L <= 64, B * L < 2^26.  Ids outside [0, V) are clamped and
 * flagged (DFLASH2_DEVERR_BAD_TOKEN).  A bounded wait that gives up raises
 * DFLASH2_DEVERR_TIMEOUT.
 */
size_t dflash2_pair_scores_proj_workspace(const dflash2_handle* h, int64_t B, int64_t L);
int dflash2_pair_scores_proj(dflash2_handle* h, const int32_t* cand_idx, const float* cand_val,
                             const int32_t* last_verified, const float* gate, const uint16_t* E,
                             const uint16_t* W_A, const uint16_t* W_B, int64_t B, int64_t L, int64_t d, int64_t V,
                             float* P, size_t P_bytes, float* S, void* stream);

/*
 * The walk over precomputed scores.  "A Lightweight Path Selector": from the
 * last verified token, greedy follows the best successor at each step and
 * sampling draws from the same scores.  Step t reads row 0 of S[b,0] at t = 0
 * and row draft_slot[b,t-1] afterwards.
 *   temperature <= 0: slot = lowest j maximising the row, a NaN score below
 *     every number (all NaN: slot 0); draft_q one-hot.
 *   temperature  > 0: every step in fp32 with correctly rounded operations:
 *     w_j = 2^((S_j - max S) * (log2(e) / T)) (Cody-Waite reduction and a
 *     degree-7 Taylor polynomial), Z summed in slot order, u = Philox4x32-10
 *     uniform of counter (b, t | 0 << 24, offset_lo, offset_hi), key (seed_lo,
 *     seed_hi), u = (x0 >> 8) * 2^-24; slot = smallest j with
 *     u Z < w_0 + ... + w_j; draft_q[b,t,j] = w_j / Z.  A row with no positive
 *     weight (every score NaN or -inf) takes the greedy slot, q one-hot there.
 *   S          device fp32 [B, L, 16, 16], 16-byte aligned (read with 16-byte loads)
 *   cand_idx   device int32 [B, L, 16]
 *   draft_tok  device int32 [B, L];  draft_slot device int32 [B, L]
 *   draft_q    device fp32 [B, L, 16] or NULL
 * Nothing in the walk waits on the device; draft_tok takes cand_idx as stored.
 */
int dflash2_walk(dflash2_handle* h, const float* S, const int32_t* cand_idx, int64_t B, int64_t L,
                 float temperature, uint64_t seed, uint64_t offset, int32_t* draft_tok,
                 int32_t* draft_slot, float* draft_q, void* stream);

/*
 * Exact best path over the same scores.  "A Lightweight Path Selector" calls
 * pairwise scoring the simplest selector and leaves more to explore; this walk
 * keeps the scores and replaces the myopic step by the max-sum path:
 *   slots j_0..j_{L-1} maximising S[b,0,0,j_0] + sum_{t>=1} S[b,t,j_{t-1},j_t],
 *   the sum formed left to right in fp32; ties keep the lowest predecessor,
 *   then the lowest final slot.
 *   S           device fp32 [B, L, 16, 16];  cand_idx device int32 [B, L, 16]
 *   draft_tok, draft_slot  device int32 [B, L]
 *   score       device fp32 [B] (the best path's score) or NULL
 * L <= 64.  Same layout, alignment and error rules as dflash2_walk.
 */
int dflash2_walk_viterbi(dflash2_handle* h, const float* S, const int32_t* cand_idx, int64_t B, int64_t L,
                         int32_t* draft_tok, int32_t* draft_slot, float* score, void* stream);

/*
 * Selector evaluation, Table 1 of "DFlash 2: Keep Drafting Parallel" ("The
 * Right Tokens Are Already There"): given the true tokens and the per-position
 * top-16 candidates (slot 0 = top-1), per sequence
 *   accept1[b]  = 1 + the number of leading positions whose top-1 is the true token,
 *   accept16[b] = 1 + the number of leading positions whose 16 candidates hold it
 *                 (an oracle selector that always picks the right candidate),
 * and per position counts[t] = (sequences whose earlier positions all hit under
 * the top-1 rule, how many of them hit at t, the same two under the top-16
 * rule), so Recall@1[t] = counts[t][1] / counts[t][0] and Recall@16[t] =
 * counts[t][3] / counts[t][2] are Table 1's conditional recalls.
 *   gt          device int32 [B, L];  cand_idx device int32 [B, L, 16]
 *   accept1, accept16  device int32 [B];  counts device int64 [L, 4] (overwritten)
 * L <= 64.  int32 pointers 4-byte aligned, counts 8-byte aligned.
 */
int dflash2_selector_eval(dflash2_handle* h, const int32_t* gt, const int32_t* cand_idx, int64_t B, int64_t L,
                          int32_t* accept1, int32_t* accept16, int64_t* counts, void* stream);

/*
 * Two-tap dynamic depthwise convolution.  "A Lightweight Local Convolution":
 * Conv_k(x)_t = k_{t,0} (.) x_t + k_{t,1} (.) x_{t-1}; each coefficient is a
 * learned base plus a correction from the current hidden state shared by every
 * 16 channels; position 0 reads the last verified token's representation.
 *   [c0; c1][b,t,:] = W_c h[b,t,:] (+ b_c)          W_c: [2d/16, d]
 *   y[b,t,ch] = (k0[ch] + c0[b,t,ch/16]) x[b,t,ch] + (k1[ch] + c1[b,t,ch/16]) xp[ch]
 *   xp = x[b,t-1,:] for t > 0, x_prev[b,:] for t = 0.
 *   x       device bf16 [B, L, d];  x_prev device bf16 [B, d]
 *   hs      device bf16 [B, L, d] or NULL (then h = x)
 *   k0, k1  device bf16 [d];  W_c device bf16 [2d/16, d];  b_c device fp32 [2d/16] or NULL
 *   y       device [B, L, d], fp32 if y_is_fp32 else bf16 (round to nearest even);
 *           must not overlap x, x_prev or hs.
 *   workspace  device scratch of at least dflash2_conv2tap_workspace(h, B, L, d)
 *              bytes, 256-byte aligned: the correction's fp32 split-K partials
 *              (a few per position and group), rewritten by every call; calls
 *              that overlap on the GPU must not share it.  The size depends on
 *              the device's SM count, hence the handle argument.
 * The correction is summed over its K splits in a fixed order, so a call gives
 * the same bits every time.  d % 64 == 0, L <= 64, B <= 65535.  A too-small or
 * NULL workspace returns DFLASH2_ERR_WORKSPACE.
 */
size_t dflash2_conv2tap_workspace(const dflash2_handle* h, int64_t B, int64_t L, int64_t d);
int dflash2_conv2tap(dflash2_handle* h, const uint16_t* x, const uint16_t* x_prev,
                     const uint16_t* hs, const uint16_t* k0, const uint16_t* k1,
                     const uint16_t* W_c, const float* b_c, int64_t B, int64_t L, int64_t d,
                     void* y, int y_is_fp32, void* workspace, size_t ws_bytes, void* stream);

/*
 * The two-tap conv fused into the GEMM that produces its input (the output
 * projection of a drafter sublayer; the conv sits before and after each
 * attention and feed-forward sublayer, "A Lightweight Local Convolution"), so
 * x never goes to memory:
 *   x[b,t,:] = A[b,t,:] W^T            (tensor cores, fp32, not rounded to bf16)
 *   [c0; c1][b,t,:] = W_c hs[b,t,:] (+ b_c)
 *   y[b,t,ch] = (k0[ch] + c0[b,t,ch/16]) x[b,t,ch] + (k1[ch] + c1[b,t,ch/16]) xp[ch]
 *   xp = x[b,t-1,:] for t > 0, x_prev[b,:] for t = 0.
 * The correction reads the given hidden state hs (a GEMM epilogue sees one
 * tile of x, never the whole row that W_c x would need).
 *   A       device bf16 [B, L, K];  W device bf16 [d, K]
 *   x_prev  device bf16 [B, d];  hs device bf16 [B, L, d]
 *   k0, k1, W_c, b_c  as dflash2_conv2tap
 *   c_work  device workspace of at least dflash2_gemm_conv2tap_workspace(h, B, L, d)
 *           bytes, 16-byte aligned; on return it starts with [c0; c1] ([B*L, 2d/16] fp32),
 *           followed by the kernel's per-row-tile counters
 *   y       device [B, L, d], fp32 if y_is_fp32 else bf16 (round to nearest even),
 *           16-byte aligned; must not overlap the inputs.
 * d % 64 == 0, K % 64 == 0, L <= 64.  A bounded wait that gives up raises
 * DFLASH2_DEVERR_TIMEOUT.
 */
size_t dflash2_gemm_conv2tap_workspace(const dflash2_handle* h, int64_t B, int64_t L, int64_t d);
int dflash2_gemm_conv2tap(dflash2_handle* h, const uint16_t* A, const uint16_t* W, const uint16_t* x_prev,
                          const uint16_t* hs, const uint16_t* k0, const uint16_t* k1, const uint16_t* W_c,
                          const float* b_c, int64_t B, int64_t L, int64_t K, int64_t d, float* c_work,
                          size_t c_bytes, void* y, int y_is_fp32, void* stream);

/*
 * Block verification against the target's logits.  "A Lightweight Path
 * Selector" (rejection sampling restores the exact target distribution) and
 * Table 1's note (the acceptance length includes the verifier's next token).
 *   temperature <= 0: a_t = argmax target[b,t,:] (lowest id on ties, NaN below
 *     -inf);  n = first t < L with draft_tok[b,t] != a_t (else L);
 *     out_tok[b] = draft_tok[b,0..n-1], a_n, then -1;  accept_len[b] = n + 1.
 *   temperature  > 0: speculative rejection sampling with p_t in exact fixed
 *     point: c = log2(e) / T (fp32), M = the row's largest non-NaN logit,
 *     W_v = floor(exp2_neg((l_v - M) c) 2^40) (the fp32 2^x of dflash2_walk),
 *     Z = sum_v W_v, p_t(v) = W_v / Z, an exact integer ratio whatever the
 *     order of the parallel sums.  With q = draft_q[b,t,draft_slot[b,t]]:
 *     accept t iff (u1 q) Z < W_x in fp64 (x = draft_tok[b,t]).  On the first
 *     rejection draw from R_v = max(0, W_v - sum_{j: cand_idx[b,t,j] = v} Q_j),
 *     Q_j = floor(min(draft_q[b,t,j], 1) Z), by inverse CDF in id order with the
 *     target floor(U2 R / 2^24), R = sum_v R_v (from W if R = 0); after L
 *     acceptances draw the bonus from W of row L the same way.  u1 = U1 2^-24
 *     and U2 are the 24-bit Philox integers of streams 1 and 2 at (b, t); a
 *     row with no finite logit (Z = 0) rejects and emits its arg-max.
 *   target      device bf16 [B, L+1, ld] (row (b,t) at (b*(L+1)+t)*ld)
 *   draft_tok, draft_slot  device int32 [B, L];  draft_q device fp32 [B, L, 16]
 *   cand_idx    device int32 [B, L, 16]
 *   accept_len  device int32 [B];  out_tok device int32 [B, L+1]
 *   workspace   device scratch of at least dflash2_verify_workspace(h, B, L, V)
 *               bytes, 256-byte aligned (counter words, per-row counters, maxima
 *               and sums, per-chunk sums), fully re-initialised by every call;
 *               calls that overlap on the GPU must not share it.
 * draft_q, draft_slot and cand_idx may be NULL when temperature <= 0, and every
 * draft argument may be NULL when L = 0 (only the bonus row is decided).
 * L <= 64, V <= 10,485,760 (DFLASH2_ERR_UNSUPPORTED beyond).  A too-small or
 * NULL workspace returns DFLASH2_ERR_WORKSPACE.  Out-of-range draft tokens,
 * slots and candidate ids are clamped (a draft token outside [0, V) weighs 0)
 * and flagged in the error word.
 */
size_t dflash2_verify_workspace(const dflash2_handle* h, int64_t B, int64_t L, int64_t V);
int dflash2_verify(dflash2_handle* h, const uint16_t* target, int64_t ld, const int32_t* draft_tok,
                   const int32_t* draft_slot, const float* draft_q, const int32_t* cand_idx,
                   int64_t B, int64_t L, int64_t V, float temperature, uint64_t seed,
                   uint64_t offset, int32_t* accept_len, int32_t* out_tok, void* workspace,
                   size_t ws_bytes, void* stream);

/*
 * Fused LM head + top-16: logits = hidden W^T are produced tile by tile on the
 * tensor cores (tcgen05, fp32 accumulation) and reduced to each row's top-16
 * on chip, so no logit reaches global memory (the head produces U_t, "DFlash's
 * own logit").
 *   hidden  device bf16 [M, d];  W device bf16 [V, d]
 *   vals    device fp32 [M, 16] (the fp32 logits);  idx device int32 [M, 16]
 *           (value descending, lowest id on ties)
 *   workspace  device scratch of at least dflash2_lmhead_topk_workspace(h, M, V, d)
 *              bytes, 256-byte aligned: per-CTA partial lists, fully rewritten
 *              by every call; calls that overlap on the GPU must not share it.
 * d % 64 == 0, V >= 16.  The workspace size depends on the device's SM count,
 * hence the handle argument (0 for a null handle or empty problem).
 */
size_t dflash2_lmhead_topk_workspace(const dflash2_handle* h, int64_t M, int64_t V, int64_t d);
int dflash2_lmhead_topk(dflash2_handle* h, const uint16_t* hidden, const uint16_t* W, int64_t M,
                        int64_t V, int64_t d, float* vals, int32_t* idx, void* workspace,
                        size_t ws_bytes, void* stream);

/*
 * Fused LM head + top-16 with the context gate folded in: W_H's 256 rows are
 * one more 256-row tile of the same GEMM (0.17% more products at V = 151936),
 * whose epilogue writes H = sigmoid(hidden W_H^T + b_H) instead of ranking.
 * vals and idx are those of dflash2_lmhead_topk on the same inputs.
 *   W_H   device bf16 [256, d];  b_H device fp32 [256] or NULL (= 0)
 *   gate  device fp32 [M, 256], 16-byte aligned
 * Other arguments, the workspace (dflash2_lmhead_topk_workspace covers both
 * forms) and the limits are those of dflash2_lmhead_topk.
 */
int dflash2_lmhead_topk_gate(dflash2_handle* h, const uint16_t* hidden, const uint16_t* W, const uint16_t* W_H,
                             const float* b_H, int64_t M, int64_t V, int64_t d, float* vals, int32_t* idx,
                             float* gate, void* workspace, size_t ws_bytes, void* stream);

/*
 * dflash2_lmhead_topk without a workspace argument, for callers that cannot
 * allocate device memory: code running inside an engine whose memory pool owns
 * every byte of the GPU, or a latency-critical serving loop where a cudaMalloc
 * or cudaFree (which may synchronise the device) is not acceptable.  The pages
 * have no counterpart of this call; it exists for those callers only.
 *
 * The partial lists go to a fixed scratch array of
 * DFLASH2_LMHEAD_NOALLOC_SCRATCH_BYTES bytes that the library declares as a
 * file-scope device variable: every GPU that loads the library holds it until
 * the process exits.  A problem whose partial lists exceed it (more than
 * DFLASH2_LMHEAD_NOALLOC_SCRATCH_BYTES / 128 row-runs; 1024 hidden rows fit on
 * any GPU with at most 256 SMs) is rejected with DFLASH2_ERR_WORKSPACE before
 * anything runs.  The call allocates nothing.
 *
 * The first call on a device looks up the scratch array's device address (with
 * that device made current for the lookup, then restored); make that first
 * call before any stream capture.  All calls share the one array and every
 * call rewrites the part it uses, so nothing needs clearing, but calls that
 * overlap on the GPU (different streams, or different handles of the same
 * device) race on it and must be serialised by the caller.  Arguments, output
 * layout and errors are otherwise those of dflash2_lmhead_topk.
 */
#define DFLASH2_LMHEAD_NOALLOC_SCRATCH_BYTES (4u << 20)
int dflash2_lmhead_topk_noalloc(dflash2_handle* h, const uint16_t* hidden, const uint16_t* W, int64_t M,
                                int64_t V, int64_t d, float* vals, int32_t* idx, void* stream);

/*
 * Self-test of failure detection, run without a GPU fault.  The pages have no
 * counterpart: every wait inside the library's kernels (an mbarrier that a TMA
 * copy or tensor-core commit completes, a word another CTA writes) is bounded,
 * and this call shows that a bound is kept.  It launches one kernel whose two
 * waits cannot be satisfied -- an mbarrier no thread arrives on, and
 * words[0] reaching 1, which no one writes -- each with limit `limit_ns`
 * (0 < limit_ns <= 2e9, the library's own limit).  Each wait gives up, ORs
 * DFLASH2_DEVERR_TIMEOUT into the error word, and the kernel returns normally,
 * leaving the context usable.
 *   words  device uint32 [2]: words[0] must hold 0 (the caller keeps it 0);
 *          words[1] receives bit 0 / bit 1 if the mbarrier / word wait was
 *          satisfied (never) and bit 2 when the kernel reached its end.
 */
int dflash2_selftest_wait_timeout(dflash2_handle* h, uint64_t limit_ns, uint32_t* words, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH2_H */
