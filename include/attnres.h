/*
 * attnres.h -- C ABI of the B300 (sm_103a) Attention Residuals (AttnRes) aggregation library.
 *
 * Before each sublayer l, every token replaces the fixed residual sum with softmax attention
 * over depth.  A static per-sublayer pseudo-query w_l scores each source v as
 * z = w_l . RMSNorm(v), and the sublayer input is h_l = sum_i softmax_i(z) v_i.
 * ("Attention Residuals" note on arXiv 2603.15031, §7 Full AttnRes; §8 Block AttnRes.)
 *
 * Block AttnRes sources of sublayer l in block n at position i: the embedding b_0, the
 * completed blocks b_1 .. b_{n-1}, and from i = 2 on the partial sum b_n^{i-1} (§8).
 * The library runs the two-phase schedule (§10; "Attention Residuals 阅读补充", section
 * "静态 Query 与两阶段计算"):
 *   phase 1  scores all S queries of a block against the completed sources in one pass and
 *            returns the normalised partial output plus (max, log-sum-exp);
 *   phase 2  runs sublayer by sublayer, merges the partial-sum source by online softmax and
 *            applies the sublayer's input RMSNorm in the same kernel.
 *
 * Conventions for every entry point
 *   - Memory: every pointer is caller-owned.  "device" pointers must point to memory of the
 *     current CUDA device; the library allocates nothing and keeps no state between calls.
 *   - Layout: a [T, d] tensor is T rows of d contiguous elements (row stride d).
 *   - dtype: ATTNRES_F32 stores float, ATTNRES_BF16 stores bfloat16 (round to nearest even);
 *     arithmetic is fp32 in both cases.  Statistics (m, lse, alpha) are always fp32.
 *   - Alignment: every device pointer must be 16-byte aligned and d a multiple of 8, so that
 *     every row starts on a 16-byte boundary; otherwise ATTNRES_ERR_MISALIGNED /
 *     ATTNRES_ERR_INVALID_ARG is returned and nothing is launched.
 *   - Asynchrony: work is queued on `stream` (a cudaStream_t passed as void*, NULL = legacy
 *     default stream).  No entry point synchronises.  Launch errors are reported as
 *     ATTNRES_ERR_CUDA (the CUDA error string is available from attnres_last_cuda_error()).
 *   - Errors: arguments are validated on the host before anything is launched; on any error
 *     no kernel runs and the outputs are untouched.  No exception crosses the ABI.
 *   - Aliasing: outputs must not overlap inputs, except where an entry point says so.
 */
#ifndef ATTNRES_H_
#define ATTNRES_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTNRES_OK = 0,
  ATTNRES_ERR_INVALID_ARG = 1,   /* null required pointer, non-positive size, bad enum     */
  ATTNRES_ERR_UNSUPPORTED = 2,   /* sizes beyond the limits below                          */
  ATTNRES_ERR_MISALIGNED = 3,    /* a device pointer or stride breaks 16-byte alignment    */
  ATTNRES_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed            */
  ATTNRES_ERR_TIMEOUT = 5        /* a kernel's bounded wait for its own copies gave up     */
} attnres_status;

typedef enum { ATTNRES_F32 = 0, ATTNRES_BF16 = 1 } attnres_dtype;

/*
 * Variant flags (bitwise or; 0 = the method as defined), the ablation variants of the report's
 * Table 4 ("Attention Residuals" note, result 4):
 *   ATTNRES_SIGMOID_WEIGHTS  alpha_i = sigmoid(z_i) = 1 / (1 + exp(-z_i)) for every source on
 *                            its own: no softmax competition, no sum-to-1.  h = sum_i alpha_i v_i.
 *                            Two-phase: phase 1 returns o = sum over its sources of
 *                            alpha_i b_i (unnormalised) and phase 2 adds the partial's term,
 *                            h = o + sigmoid(z_p) p; no log-sum-exp is involved.
 *   ATTNRES_NO_KEY_NORM      z_i = u . v_i: the key is the raw source (no RMS division, eps
 *                            unused); the key-norm gain goes with the norm, so u should carry
 *                            no gain (attnres_query_prep with gamma_key = NULL).
 * Any other bit returns ATTNRES_ERR_INVALID_ARG.
 */
#define ATTNRES_SIGMOID_WEIGHTS 0x1u
#define ATTNRES_NO_KEY_NORM 0x2u

/*
 * Storage flag of phase 1's output (not a variant of the method; accepted by attnres_phase1,
 * attnres_phase2_merge and attnres_phase2_merge_sources only, ATTNRES_ERR_INVALID_ARG
 * elsewhere):
 *   ATTNRES_O_F32            phase 1 writes o in fp32 whatever the I/O type, and phase 2 /
 *                            the grouped merge read o_l in fp32.  With bf16 I/O this removes
 *                            the one rounding between the phases: the two-phase result then
 *                            equals the direct softmax over all sources up to fp32 arithmetic
 *                            and the final bf16 store ("Attention Residuals" note §10: the
 *                            merge is exact).  It doubles o's bytes.  With ATTNRES_F32 I/O it
 *                            changes nothing.
 */
#define ATTNRES_O_F32 0x4u

/*
 * Depth-attention heads (`heads` argument; 1 = the method as defined), the multi-head variant
 * of Table 4 ("Attention Residuals" note, result 4: "Block, multi-head H = 16").  The pages
 * give no formula; the reading implemented here: the d features split into H contiguous slices
 * of dh = d / H, and head k is a complete aggregation on its slice (columns k*dh .. k*dh+dh-1):
 * the key RMS r_j,k is taken over the slice, the logit is u[slice] . b_j[slice] / r_j,k, and
 * the softmax (or sigmoid) over the sources runs per head.  The heads' outputs are
 * concatenated, and the sublayer's input RMSNorm normalises the whole d-vector.  Per-head
 * statistics gain a head index after the query (phase 1) or first (phase 2):
 * m, lse [S][H][T]; alpha [S][H][T][n].  Requires d % H == 0 and dh a multiple of 8.
 */
#define ATTNRES_MAX_HEADS 64

/* Limits (checked; larger values return ATTNRES_ERR_UNSUPPORTED). */
#define ATTNRES_MAX_SOURCES 64     /* sources per call (phase 1 and the full path)          */
#define ATTNRES_MAX_QUERIES 64     /* queries S per phase-1 call                             */
#define ATTNRES_MAX_D 16384        /* hidden size (a row stays in registers)               */

/* ABI version of this header; attnres_abi_version() returns the library's. */
#define ATTNRES_ABI_VERSION 9
int attnres_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* attnres_status_string(attnres_status status);

/* Message of the last CUDA error seen by this thread's calls ("" if none). */
const char* attnres_last_cuda_error(void);

/*
 * Device-side error poll.  The phase-1 kernels stage their tiles with asynchronous tensor
 * copies and wait for them on shared-memory barriers; every such wait is bounded.  A wait that gives
 * up (a copy that never lands) makes the kernel finish early with undefined outputs and counts
 * the event in a device word of the current device.  This call reads and clears that word:
 * ATTNRES_ERR_TIMEOUT if any wait gave up since the previous poll, ATTNRES_OK otherwise,
 * ATTNRES_ERR_CUDA if the word could not be read.  It synchronises with the device (it is a
 * diagnostic, not part of the hot path).
 */
attnres_status attnres_poll_device_errors(void);

/*
 * Self-test of the timeout path (a diagnostic, not part of the hot path): launches one small
 * kernel on `stream` whose bounded wait cannot succeed (an mbarrier that expects an arrival that
 * never comes).  It polls `polls` times (at most 2^20; 0 gives up at once), then counts the event
 * like any wait of the library that gives up, and returns; nothing hangs, nothing faults, and the
 * context stays usable.  After the kernel has run, attnres_poll_device_errors returns
 * ATTNRES_ERR_TIMEOUT (and clears the word).  Returns ATTNRES_ERR_INVALID_ARG for larger polls,
 * ATTNRES_ERR_CUDA if the launch fails.
 */
attnres_status attnres_selftest_wait_timeout(unsigned int polls, void* stream);

/*
 * Query preparation (row a0): u = w ⊙ gamma_key, row by row.
 * The key of a source is RMSNorm(v) = gamma_key ⊙ v / r(v) and the logit is w . RMSNorm(v)
 * ("Attention Residuals" §7; "Attention Residuals 阅读补充", RMSNorm definition), so
 * w . RMSNorm(v) = (w ⊙ gamma_key) . v / r(v).  The gain belongs to the target sublayer
 * (one query and one set of key-norm gains per sublayer), so the product is a per-sublayer
 * parameter: compute it once and pass u to the calls below.
 *   w            device, fp32 [rows, d]
 *   gamma_key    device, fp32 [rows, d], or NULL for all-ones gains (u = w)
 *   u_out        device, fp32 [rows, d]; may alias w (in place)
 *   u_split_out  device, bf16 [2 * rows, d], or NULL: rows 2r and 2r + 1 receive
 *                hi = bf16(u_r) and lo = bf16(u_r - hi) (round to nearest even), so that
 *                |u - hi - lo| <= 2^-16 |u|.  Phase 1 computes its logits on the tensor cores
 *                from this form (see attnres_phase1).  Must not overlap w or u_out.
 */
attnres_status attnres_query_prep(const float* w, const float* gamma_key, float* u_out,
                                  void* u_split_out, int rows, int d, void* stream);

/*
 * Phase 1 (rows a1-a4): the S queries of one block against the n completed sources,
 * one pass over the sources ("Attention Residuals" §10, step 1).
 * For every token t and query s, with r_j = sqrt(mean_k b_j[t,k]^2 + eps) and
 * z_j = u_s . b_j[t] / r_j:
 *     m[s,t]   = max_j z_j
 *     lse[s,t] = m + ln sum_j exp(z_j - m)
 *     o[s,t,:] = sum_j exp(z_j - lse) b_j[t,:]           (normalised partial output)
 *     alpha[s,t,j] = exp(z_j - lse)
 *   reps        device [n_src][T][d] (io dtype): source j, token t at
 *               reps + j*src_stride + t*d elements.  src_stride >= T*d, a multiple of 8.
 *   u           device fp32 [S, d]: the block's queries with key gains folded in
 *               (attnres_query_prep)
 *   u_split     device bf16 [2S, d] or NULL: the same queries split into hi/lo rows
 *               (attnres_query_prep's u_split_out for these S rows).  When it is given, the I/O
 *               type is bf16, 2 <= S <= 24 and n_src <= 64, the logit numerators u_s . b_j[t] are
 *               computed on the tensor cores as (hi + lo) . b_j[t] with fp32 accumulation;
 *               otherwise the CUDA cores compute them from u in fp32.  Both agree to fp32
 *               rounding plus the split's 2^-16 relative error in u.
 *   o_out       device [S][T][d] (io dtype; fp32 with ATTNRES_O_F32), required
 *   m_out, lse_out  device fp32 [S][T], each optional (NULL = not written); with
 *               ATTNRES_SIGMOID_WEIGHTS, o is the unnormalised sum and lse_out is not written
 *   alpha_out   device fp32 [S][T][n_src], optional
 *   flags       ATTNRES_SIGMOID_WEIGHTS | ATTNRES_NO_KEY_NORM | ATTNRES_O_F32 (see above),
 *               0 by default
 *   heads       depth-attention heads H (see above), 1 by default: m_out and lse_out are then
 *               [S][H][T] and alpha_out [S][H][T][n_src]; the tensor cores take H > 1 when
 *               d / H is a multiple of 64
 * Limits: 1 <= n_src <= 64, 1 <= S <= 64, and n_src <= 16 when S > 24 (the per-token tile
 * must fit one CTA); 1 <= heads <= 64; otherwise ATTNRES_ERR_UNSUPPORTED.
 * With S = 1 and the final pseudo-query this is also the final aggregation over
 * b_0 .. b_N (row a10).
 */
attnres_status attnres_phase1(const void* reps, int64_t src_stride, int n_src, int64_t T,
                              int d, attnres_dtype io, const float* u, const void* u_split,
                              int S, float eps, void* o_out, float* m_out, float* lse_out,
                              float* alpha_out, unsigned int flags, int heads, void* stream);

/*
 * Phase 2 merge (rows a5-a8): one sublayer l of the block ("Attention Residuals" §10,
 * step 2; "Attention Residuals 阅读补充", the merge of two partitions).
 * The partial-sum source is p = partial + v_prev (a missing term counts as zero), summed in
 * fp32 and used unrounded; with both NULL there is no partial source (first sublayer of the
 * block, b_n^0 = 0 is not a source).  With r = sqrt(mean p^2 + eps_key), z_p = u_l . p / r,
 * M = max(lse_l, z_p), a = exp(lse_l - M), c = exp(z_p - M):
 *     h = (a o_l + c p) / (a + c)            (h = o_l when there is no partial source)
 *     y = gamma_in ⊙ h / sqrt(mean h^2 + eps_in)
 *   o_l          device [T, d] (io dtype; fp32 with ATTNRES_O_F32): phase-1 output row block
 *                of this sublayer
 *   lse_l        device fp32 [T]; required when there is a partial source
 *   partial      device [T, d] (io dtype) or NULL: b_n^{i-2} (or b_n^{i-1} if v_prev is NULL)
 *   v_prev       device [T, d] (io dtype) or NULL: output of the previous sublayer
 *   partial_out  device [T, d] or NULL: receives p rounded to the io dtype (the fused
 *                partial-sum update b^{i-1} = b^{i-2} + v_{i-1}); may alias `partial`
 *   u_l          device fp32 [d]: query of sublayer l with its key gain folded in
 *   gamma_in     device fp32 [d] or NULL (all ones): input-norm gain of sublayer l
 *   h_out        device [T, d] or NULL;  y_out device [T, d], required
 *   alpha_p_out  device fp32 [T] or NULL: weight of the partial source, c / (a + c)
 *   flags        variant flags; with ATTNRES_SIGMOID_WEIGHTS h = o_l + sigmoid(z_p) p, lse_l is
 *                not read (may be NULL) and alpha_p_out receives sigmoid(z_p); ATTNRES_O_F32:
 *                o_l is fp32
 *   heads        depth-attention heads H: each head merges its slice with its own r, z_p and
 *                lse (lse_l and alpha_p_out are then [H][T]); y normalises the whole row
 */
attnres_status attnres_phase2_merge(const void* o_l, const float* lse_l, const void* partial,
                                    const void* v_prev, void* partial_out, int64_t T, int d,
                                    attnres_dtype io, const float* u_l, float eps_key,
                                    const float* gamma_in, float eps_in, void* h_out,
                                    void* y_out, float* alpha_p_out, unsigned int flags,
                                    int heads, void* stream);

/*
 * Partial-sum update / block close (rows a8-a9): out = partial + v, elementwise, rounded to
 * the io dtype ("Attention Residuals" §8: b_n^i = b_n^{i-1} + f_i(h_i); the closed partial
 * b_n^S becomes the next source).  `out` may alias `partial`.
 */
attnres_status attnres_partial_update(const void* partial, const void* v, void* out,
                                      int64_t T, int d, attnres_dtype io, void* stream);

/*
 * Direct (single-pass, not two-phase) aggregation of one sublayer over an explicit list of
 * sources: the plain Full AttnRes step ("Attention Residuals" §7), which is also the
 * comparison point of the two-phase path.  Computes the same h and y as phase 2 would over
 * the union of the sources.
 *   srcs        HOST array of n_src device pointers, each [T, d] (io dtype)
 *   u_l         device fp32 [d]; gamma_in device fp32 [d] or NULL
 *   h_out       device [T, d] or NULL; y_out device [T, d] or NULL (at least one required)
 *   alpha_out   device fp32 [T][n_src] or NULL
 *   flags       variant flags (sigmoid weights: h = sum_i sigmoid(z_i) v_i)
 *   heads       depth-attention heads H (alpha_out is then [H][T][n_src])
 * Limits: 1 <= n_src <= 64.
 */
attnres_status attnres_full_reference_path(const void* const* srcs, int n_src, int64_t T,
                                           int d, attnres_dtype io, const float* u_l,
                                           float eps_key, const float* gamma_in,
                                           float eps_in, void* h_out, void* y_out,
                                           float* alpha_out, unsigned int flags, int heads,
                                           void* stream);

/*
 * Phase 2 of Full AttnRes run by the grouped two-phase schedule ("Attention Residuals 阅读补充",
 * section "静态 Query 与两阶段计算": the layers fall into groups of S; phase 1
 * (attnres_phase1) scores a group's S queries against the history in one pass; phase 2 takes
 * the group's layers one by one and merges, by online softmax, the k representations the
 * group has produced so far).  For layer l with phase-1 result (o_l, lse_l) over the history A
 * and in-group sources B = srcs[0 .. k-1]:
 *     M = max(lse_l, max_{i in B} z_i)
 *     h = (e^{lse_l - M} o_l + sum_{i in B} e^{z_i - M} v_i) / (e^{lse_l - M} + sum_{i in B} e^{z_i - M})
 *     y = gamma_in ⊙ h / sqrt(mean h^2 + eps_in)
 * (k = 0 gives h = o_l.)  With ATTNRES_SIGMOID_WEIGHTS, h = o_l + sum_{i in B} sigmoid(z_i) v_i
 * and lse_l is not read.
 *   o_l, lse_l  device [T, d] (io dtype; fp32 with ATTNRES_O_F32) and fp32 [T]: phase 1's
 *               output row block of layer l
 *   srcs        HOST array of k device pointers, each [T, d] (io dtype); may be NULL when k = 0
 *   u_l, gamma_in, eps_key, eps_in: as for attnres_phase2_merge
 *   h_out, y_out  device [T, d] or NULL (at least one required)
 *   alpha_out   device fp32 [T][k] or NULL: weights of the in-group sources
 *   heads       depth-attention heads H: lse_l is [H][T] and alpha_out [H][T][k]
 * Limits: 0 <= k <= 64.
 */
attnres_status attnres_phase2_merge_sources(const void* o_l, const float* lse_l,
                                            const void* const* srcs, int k, int64_t T, int d,
                                            attnres_dtype io, const float* u_l, float eps_key,
                                            const float* gamma_in, float eps_in, void* h_out,
                                            void* y_out, float* alpha_out, unsigned int flags,
                                            int heads, void* stream);

/*
 * Backward of one sublayer's aggregation over an explicit source list (the direct form of
 * attnres_full_reference_path with its output y; softmax weights, key RMSNorm): the logit
 * gradient dL/dz_i = alpha_i g_h^T (v_i - h) ("Attention Residuals" note §7) and the RMSNorm
 * input gradient (1/r)(g' - yhat (yhat^T g') / d) with g' = gamma ⊙ g ("Attention Residuals
 * 阅读补充", section "梯度沿切向传播").  Given g_y = dL/dy:
 *     g_h  = gamma_in ⊙ g_y / r_h - h (sum_k gamma_in,k g_y,k h_k) / (d r_h^3)
 *     dz_i = alpha_i (g_h . v_i - g_h . h)
 *     dL/dv_i = alpha_i g_h + (dz_i / r_i) u - (dz_i z_i / (d r_i^2)) v_i
 *     du        += sum over tokens and sources of (dz_i / r_i) v_i
 *     dgamma_in += sum over tokens of g_y ⊙ h / r_h
 * u = w ⊙ gamma_key is the folded query; the parameter gradients follow elementwise:
 * dL/dw = gamma_key ⊙ du and dL/dgamma_key = w ⊙ du.  The forward quantities (r_i, z, alpha,
 * h, r_h) are recomputed from the sources.
 *   srcs        HOST array of n_src device pointers, each [T, d] (io dtype)
 *   u           device fp32 [d]; gamma_in device fp32 [d] or NULL (ones)
 *   g_y         device [T, d] (io dtype): dL/dy
 *   dsrcs       HOST array of n_src device pointers, each [T, d] (io dtype): receive dL/dv_i
 *   du          device fp32 [d]: the gradient is ADDED (zero it first for a fresh sum)
 *   dgamma_in   device fp32 [d] or NULL: added, like du
 * The sums over tokens are accumulated with atomic additions, so their last bits may vary
 * from run to run.  Single-head (softmax, key RMSNorm) only.  Limits: 1 <= n_src <= 16;
 * d <= 8192 (bf16) or 4096 (fp32).
 */
attnres_status attnres_backward(const void* const* srcs, int n_src, int64_t T, int d,
                                attnres_dtype io, const float* u, float eps_key,
                                const float* gamma_in, float eps_in, const void* g_y,
                                void* const* dsrcs, float* du, float* dgamma_in, void* stream);

/*
 * Backward of one whole block of Block AttnRes, structured by the two-phase schedule
 * ("Attention Residuals" note §8 and §10; the logit gradient of §7; "Attention Residuals
 * 阅读补充", section "梯度沿切向传播" for both RMSNorm gradients, and the Block AttnRes
 * training section: the inter-block attention is recomputed in the backward pass).
 * Forward of the block: sublayer i = 1 .. S reads the completed sources b_0 .. b_{n-1} and,
 * for i >= 2, the partial sum p_i = v_1 + ... + v_{i-1}; h_i is the depth softmax over those
 * sources (softmax weights, key RMSNorm, one head) and y_i = gamma_in,i ⊙ h_i / r(h_i).
 * Given g_i = dL/dy_i for every sublayer, this computes
 *     dL/db_j = sum over the block's sublayers of each one's gradient of b_j,
 *     dL/dv_k = sum_{i > k} dL/dp_i  (v_k enters the partial of every later sublayer),
 *     du_i    += sum over tokens of the query gradient of sublayer i (u = w ⊙ gamma_key; then
 *                dL/dw_i = gamma_key,i ⊙ du_i and dL/dgamma_key,i = w_i ⊙ du_i),
 *     dgamma_in,i += sum over tokens of g_i ⊙ h_i / r(h_i).
 * It recomputes phase 1 for the S queries in one pass over the n sources (o, lse and the
 * weights go to the workspace), then runs the merge backward of every sublayer per token, then
 * the sources' and the parameters' gradients; each source row is read three times and written
 * once per block, however many sublayers the block has.  The partial sums are re-formed in
 * fp32 from v.
 *   reps         device [n][T][d] (io dtype): source j at reps + j * src_stride elements
 *   v            device: v_k (k = 1 .. S-1) at v + (k - 1) * v_stride elements, [T, d] each;
 *                may be NULL when S == 1.  (v_S enters no sublayer input of the block.)
 *   u            device fp32 [S][d]: the block's folded queries (attnres_query_prep)
 *   u_split      device bf16 [2S][d] or NULL: their hi/lo split (tensor-core phase 1)
 *   gamma_in     device fp32 [S][d] or NULL (ones)
 *   g_y          device [S][T][d] (io dtype): dL/dy_i
 *   d_reps       device [n][T][d] (io dtype, contiguous): receives dL/db_j
 *   d_v          device: dL/dv_k at d_v + (k - 1) * dv_stride elements, k = 1 .. S-1; may be
 *                NULL when S == 1
 *   du           device fp32 [S][d]: the gradients are ADDED
 *   dgamma_in    device fp32 [S][d] or NULL: added, like du
 *   workspace    device, at least attnres_backward_block_workspace_size() bytes, 256-byte
 *                aligned; caller-owned scratch, overwritten by every call
 * The sums over tokens use atomic additions, so their last bits may vary from run to run.
 * Limits: 1 <= n_src <= 16, 1 <= S <= 24, d / (elements per 16 bytes) <= 1024 (bf16 d <= 8192,
 * fp32 d <= 4096); otherwise ATTNRES_ERR_UNSUPPORTED.  Strides are multiples of 8 elements.
 */
attnres_status attnres_backward_block_workspace_size(int n_src, int S, int64_t T, int d,
                                                     attnres_dtype io, uint64_t* bytes);
attnres_status attnres_backward_block(const void* reps, int64_t src_stride, int n_src,
                                      const void* v, int64_t v_stride, int S, int64_t T, int d,
                                      attnres_dtype io, const float* u, const void* u_split,
                                      float eps_key, const float* gamma_in, float eps_in,
                                      const void* g_y, void* d_reps, void* d_v,
                                      int64_t dv_stride, float* du, float* dgamma_in,
                                      void* workspace, uint64_t workspace_bytes, void* stream);

/*
 * The same block backward for callers that cannot allocate device memory while they run it:
 * code inside a framework whose allocator owns every device byte and hands out no extra buffer
 * during execution, or code on a latency-critical path that cannot afford cudaMalloc's
 * implicit synchronisation.  (The pages have no counterpart: this is a property of the
 * library, not of the method.)
 * Arguments and results are those of attnres_backward_block, without the workspace: the
 * scratch comes from a fixed array of ATTNRES_NOALLOC_SCRATCH_BYTES in this library's own
 * device memory, which every GPU that loads the library keeps until the process exits.  Nothing
 * is allocated by this call: no cudaMalloc, no cudaFree, no allocating library routine.
 *   - Size: if attnres_backward_block_workspace_size() for these sizes exceeds
 *     ATTNRES_NOALLOC_SCRATCH_BYTES (about 48 tokens at n = 9, S = 24, d = 7168), the call
 *     returns ATTNRES_ERR_UNSUPPORTED and nothing runs.
 *   - Set-up: the first call on a device, with that device current, looks up the array's device
 *     address (cudaGetSymbolAddress) and keeps it for later calls on that device; make that first
 *     call before any stream capture.
 *   - Sharing: every call uses the same array and leaves its contents behind.  Nothing in it
 *     needs to start at zero (each call writes every part before reading it), but calls whose
 *     work overlaps on the GPU (other streams, or other host threads) race on it: order them.
 */
#define ATTNRES_NOALLOC_SCRATCH_BYTES (64u << 20)
attnres_status attnres_backward_block_noalloc(const void* reps, int64_t src_stride, int n_src,
                                              const void* v, int64_t v_stride, int S, int64_t T,
                                              int d, attnres_dtype io, const float* u,
                                              const void* u_split, float eps_key,
                                              const float* gamma_in, float eps_in,
                                              const void* g_y, void* d_reps, void* d_v,
                                              int64_t dv_stride, float* du, float* dgamma_in,
                                              void* stream);

#ifdef __cplusplus
}
#endif
#endif /* ATTNRES_H_ */
