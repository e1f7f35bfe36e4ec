/*
 * kvq.h — C ABI of the rotated INT2 KV-cache library (libkvq.so), sm_103a.
 *
 * What the library computes
 * -------------------------
 * Quantise-on-append and split-K decode attention over a paged cache whose keys
 * and values are stored as 2-bit codes in a rotated basis.  The method is the
 * serving path described on "Output-Aware Rotation for INT2 KV-Cache
 * Quantization" (pith.science review of arXiv 2608.02691):
 *   - section "What carries the argument", mechanism (2): keys are centred by a
 *     per-channel mean, k -> k - mu, before rotation and quantisation; the shift
 *     adds one constant per query to every logit, so softmax is unchanged;
 *   - same section, mechanism (3) and "Core claim": the quantised path is
 *     rotation -> clipping -> grouping -> rounding, read back by
 *     dequantisation -> inverse rotation, with per-head orthogonal rotations that
 *     differ for keys and values (section "Assumptions & free parameters":
 *     "key rotation corrections A_K", "value rotation corrections A_V");
 *   - "Assumptions & free parameters": clipping ratios c_K = 0.96, c_V = 0.92;
 *   - "If this is right", third item, and the abstract: the paged KV-cache layout
 *     is kept and value-side rotations can be folded into W_V / W_O.
 * The pages do not fix the integer format.  This library fixes it: asymmetric
 * INT2, one group of 128 elements along head_dim per token, fp16 scale and zero
 * per group, 16-token pages.  That is 2 + 32/128 = 2.25 bits per element.
 *
 * The BF16 comparison cache (kvq_bf16_*) is this library's own speed reference:
 * plain attention over bf16 pages in the same page-table scheme.  "The KV cache
 * goes on a diet" (hangingcontext.com), section "Crush it to INT2", compares
 * INT2 decoding against a BF16 FlashDecoding-v2 kernel; no source of that kernel
 * is given, so the comparison point is written here.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *   - Every pointer argument named "device" is CUDA device memory owned by the
 *     caller.  The library never frees or retains it beyond the call.
 *   - `stream` is a cudaStream_t passed as void*.  NULL means the legacy default
 *     stream.  Every compute call is asynchronous on that stream.
 *   - The decode kernels are launched as programmatic dependents of the
 *     preceding work on the stream (CUDA programmatic dependent launch), so each
 *     can become resident before its predecessor ends; each reads its inputs only
 *     after waiting for that predecessor, so stream order holds for the caller's
 *     data.  A caller kernel that follows on the stream and is itself launched
 *     with the programmatic-serialisation attribute must execute
 *     griddepcontrol.wait (cudaGridDependencySynchronize) before reading `out`;
 *     ordinary launches, copies and host synchronisation need nothing.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - Return codes: KVQ_OK, or a KVQ_E* code below.  Argument errors are found on
 *     the host before anything is launched.  Data errors that only the device can
 *     see (a page id outside the pool, a position beyond the page table, a
 *     seq_len beyond the page table) set bits in the handle's device status word
 *     (kvq_get_status) and the offending token or page is skipped; the kernels
 *     never trap.  NaN / Inf inputs are not checked and propagate.
 *   - A handle is not thread-safe; calls on one handle must not overlap on the
 *     host.  Kernels of different handles may run concurrently.
 *   - A handle belongs to the device that was current when kvq_create ran.
 *     Calls that take a handle make that device current for their own work and
 *     give the caller's current device back before they return.
 *
 * Supported shapes: head_dim == 128, group == 128, page_size == 16,
 * num_heads / num_kv_heads in {1, 2, 4}, 1 <= num_kv_heads <= 64.  Other values
 * are rejected with KVQ_EINVAL.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------- */
#define KVQ_OK        0  /* success                                            */
#define KVQ_EINVAL    1  /* bad layout or argument (checked on the host)       */
#define KVQ_ENOSPACE  2  /* workspace smaller than kvq_workspace_bytes()       */
#define KVQ_ECUDA     3  /* a CUDA runtime call or kernel launch failed        */
#define KVQ_ENOTREADY 4  /* kvq_set_rotation() has not been called yet         */

/* ---- device status bits (kvq_get_status) -------------------------------- */
#define KVQ_STATUS_BAD_PAGE    1u  /* page id < 0 or >= num_pool_pages: skipped   */
#define KVQ_STATUS_BAD_POS     2u  /* position < 0 or >= max_pages*page_size      */
#define KVQ_STATUS_BAD_SEQLEN  4u  /* seq_len < 0 or > max_pages*page_size        */
#define KVQ_STATUS_BAD_SEQ     8u  /* seq_idx < 0 or >= batch                     */
#define KVQ_STATUS_TIMEOUT    16u  /* a bounded wait on a page copy gave up (2 s)  */

/* ---- layout flags -------------------------------------------------------- */
/* Decode returns the output in the rotated value basis (o_rot) instead of
 * o_rot * R_V^T.  This is the deployment form in which R_V is folded into
 * W_V / W_O ("If this is right", third item). */
#define KVQ_OUT_ROTATED 1u
/* The query passed to kvq_decode is already in the rotated key basis,
 * q_rot = q * R_K (the caller folded R_K into its query projection, after any
 * position encoding), so decode skips the query rotation.  Rejected by
 * kvq_decode_window (KVQ_EINVAL), whose BF16 tokens need the plain query. */
#define KVQ_Q_ROTATED 2u

typedef struct kvq_layout {
  int32_t num_heads;     /* H, query heads                                      */
  int32_t num_kv_heads;  /* Hkv, key/value heads; H % Hkv == 0 (GQA)            */
  int32_t head_dim;      /* D, must be 128                                      */
  int32_t group;         /* quantisation group along head_dim, must be 128      */
  int32_t page_size;     /* tokens per page, must be 16                         */
  float clip_k;          /* key clip ratio c_K, in (0, 1]; the pages use 0.96   */
  float clip_v;          /* value clip ratio c_V, in (0, 1]; the pages use 0.92 */
  float sm_scale;        /* softmax scale; <= 0 selects 1/sqrt(head_dim)        */
  uint32_t flags;        /* 0 or an OR of KVQ_OUT_ROTATED, KVQ_Q_ROTATED         */
} kvq_layout;

typedef struct kvq_handle kvq_handle;

/* ==========================================================================
 * INT2 page record — the byte layout of the paged cache.
 *
 * The pool is caller-owned device memory laid out as
 *     pool[num_pool_pages][num_kv_heads][KVQ_INT2_RECORD_BYTES].
 * One record holds 16 tokens of one KV head: the 2-bit codes of K and V and
 * their fp16 scale s and zero z.  Element d of token slot tau dequantises to
 *     x~ = code * s + z            (rotated and, for keys, centred basis).
 * The codes are stored in the order in which the decode kernel's tensor-core
 * fragments consume them, so that one 16-byte load per lane delivers a whole
 * page.  Below, tau in [0,16) is the token's slot in its page (position % 16),
 * d in [0,128) the element, and every word is a little-endian uint32.
 *
 * K codes, bytes [0, 512): 32 lanes x 16 bytes, lane L at byte 16*L, words
 * W[0..3].  For (tau, d):
 *     w = d >> 4,  r = d & 15,  h = r >> 3,  t = (r >> 1) & 3,  e = r & 1,
 *     L = 4*(tau & 7) + t,  word = 2*(tau >> 3) + h,  bit = 16*e + 2*w,
 *     code = (W[word] of lane L >> bit) & 3.
 * V codes, bytes [512, 1024): lane L at byte 512 + 16*L, words W[0..3].  For
 * (tau, d):
 *     m = d >> 4,  r = d & 15,  g = r & 7,  dh = r >> 3,
 *     t = (tau & 7) >> 1,  e = tau & 1,  th = tau >> 3,
 *     L = 4*g + t,  word = 2*th + dh,  bit = 16*e + 2*m,
 *     code = (W[word] of lane L >> bit) & 3.
 * Scale / zero, bytes [1024, 1152): eight 16-byte rows, row (tau & 7) at byte
 * 1024 + 16*(tau & 7).  Within a row, as fp16 little-endian:
 *     K: s at +4*(tau >> 3),     z at +4*(tau >> 3) + 2
 *     V: s at +8 + 4*(tau >> 3), z at +8 + 4*(tau >> 3) + 2
 * ========================================================================== */
#define KVQ_INT2_RECORD_BYTES 1152

/* ==========================================================================
 * BF16 page record (comparison cache): pool[num_pool_pages][num_kv_heads][8192].
 * Each element is one bf16 (2 bytes).  For (tau, d):
 *   K at byte 512*w + 16*L + 4*reg + 2*e with
 *     w = d >> 4, r = d & 15, h = r >> 3, t = (r >> 1) & 3, e = r & 1,
 *     L = 4*(tau & 7) + t, reg = (tau >> 3) + 2*h;
 *   V at byte 4096 + 512*m + 16*L + 4*reg + 2*e with
 *     m = d >> 4, r = d & 15, g = r & 7, dh = r >> 3,
 *     t = (tau & 7) >> 1, e = tau & 1, th = tau >> 3,
 *     L = 4*g + t, reg = 2*th + dh.
 * ========================================================================== */
#define KVQ_BF16_RECORD_BYTES 8192

/* ---- lifetime ------------------------------------------------------------ */

/* Validate `layout` on the host and create a handle.  On success *out owns a
 * small device allocation (status word) on the current CUDA device; the
 * rotation bank is allocated by kvq_set_rotation.  Returns KVQ_EINVAL for an
 * unsupported layout or NULL pointers (no CUDA call is made in that case). */
int kvq_create(const kvq_layout* layout, kvq_handle** out);

/* Free the handle and its device memory.  Synchronises the device first.
 * NULL is accepted and ignored. */
int kvq_destroy(kvq_handle* h);

/* Bytes of one INT2 page of all KV heads: num_kv_heads * 1152.  0 for NULL. */
size_t kvq_page_bytes(const kvq_handle* h);

/* Bytes of one BF16 comparison page of all KV heads: num_kv_heads * 8192. */
size_t kvq_bf16_page_bytes(const kvq_handle* h);

/* ---- rotation bank -------------------------------------------------------
 * Per-head orthogonal rotations and the key mean, the outputs of offline
 * calibration ("Core claim": per KV head and per layer, R = R0 exp(A - A^T);
 * "Assumptions & free parameters": mu and A_K, A_V are fitted on calibration
 * traces).  Calibration itself is not part of this library.
 *   R  : device fp32 [2][Hkv][D][D]; R[0] are the key rotations R_K, R[1] the
 *        value rotations R_V.  Row-vector convention: the rotated vector is
 *        r_i = sum_j x_j * R[j][i].
 *   mu : device fp32 [Hkv][D], the per-channel key mean.
 * The arrays are copied (stream-ordered) into the handle; the caller may free
 * them once the stream has passed this call.  May be called again to replace
 * the bank.  Orthogonality is not checked. */
int kvq_set_rotation(kvq_handle* h, const float* R, const float* mu, void* stream);

/* ---- quantise-on-append --------------------------------------------------
 * For each of n tokens i: take K[i][kv][:] and V[i][kv][:] for every KV head,
 * centre the key (k - mu), rotate key and value (R_K, R_V), clip, quantise to
 * INT2 with fp16 scale/zero and store the codes in the page record of position
 * positions[i] of sequence seq_idx[i]:
 *     page = page_table[seq_idx[i] * max_pages + positions[i] / 16],
 *     slot = positions[i] % 16.
 * The arithmetic is a fixed fp32 sequence, so the stored bytes are exactly
 * reproducible (per vector x of D elements, clip c):
 *     c_j  = (float)x_j - mu_j (keys) or (float)x_j (values)
 *     r_i  = fmaf chain: a = +0; for j = 0..D-1: a = fmaf(c_j, R[j][i], a)
 *     mx, mn = max_i r_i, min_i r_i
 *     s32 = (c*mx - c*mn) / 3   (each op rounded to fp32, IEEE division)
 *     s = fp16(s32), z = fp16(c*mn)  (round to nearest even)
 *     code_i = 0 if s == 0, else min(max(rint((r_i - z) / s), 0), 3)
 *              (fp32 subtract and divide, rint = round half to even)
 *   pool       : device, see the INT2 page record above.
 *   K, V       : device bf16 [n][Hkv][D].
 *   seq_idx    : device int32 [n], 0 <= seq_idx < batch.
 *   positions  : device int32 [n], 0 <= position < max_pages * 16.
 *   page_table : device int32 [batch][max_pages], entries in [0, num_pool_pages).
 * Two tokens of one call must not share (seq, position); if they do the result
 * is one of them, undefined which.  n == 0 is a no-op.  Returns KVQ_ENOTREADY
 * before kvq_set_rotation. */
int kvq_append(kvq_handle* h, void* pool, int num_pool_pages,
               const uint16_t* K, const uint16_t* V,
               const int32_t* seq_idx, const int32_t* positions, int n,
               const int32_t* page_table, int batch, int max_pages, void* stream);

/* ---- decode attention ----------------------------------------------------
 * Bytes of workspace kvq_decode needs for `batch` sequences and `num_splits`
 * splits (num_splits == 0: the automatic choice for that batch).  The
 * workspace holds the rotated queries and the split-K partials. */
size_t kvq_workspace_bytes(const kvq_handle* h, int batch, int num_splits);

/* One decode step for every sequence b in [0, batch):
 *     q_rot   = q[b][h] * R_K(kv)             (kv = h / (H / Hkv); q itself
 *                                               with KVQ_Q_ROTATED)
 *     logit_t = sm_scale * q_rot . k~_t        for positions t in [0, seq_lens[b])
 *     o_rot   = softmax(logit) . v~
 *     out     = o_rot * R_V(kv)^T              (o_rot if KVQ_OUT_ROTATED)
 * k~, v~ are the dequantised cache entries.  The mean term q . mu is the same
 * for every t and is left out (it does not change softmax).  Positions in
 * [0, seq_lens[b]) must have been appended.  seq_lens[b] == 0 gives out = 0.
 * The context is cut into page-aligned chunks whose partial softmax states are
 * merged with a log-sum-exp combine: num_splits chunks per (sequence, KV head)
 * when the batch's batch * num_splits chunks fit one wave of decode CTAs;
 * otherwise, with two or more sequences, those batch * num_splits chunks are
 * shared out over the sequences in proportion to their lengths (one chunk
 * size for the whole batch, so long and short sequences finish together; a
 * batch of equal lengths gets the same chunks either way).  The result does
 * not depend on the chunking beyond fp32 rounding.
 *   q          : device bf16 [batch][H][D].
 *   page_table : device int32 [batch][max_pages].
 *   seq_lens   : device int32 [batch].
 *   out        : device fp32 [batch][H][D].
 *   workspace  : device, >= kvq_workspace_bytes(h, batch, num_splits) bytes,
 *                256-byte aligned.  Contents on entry do not matter.
 *   num_splits : 0 = automatic, else 1..1024.
 * Returns KVQ_ENOSPACE if ws_bytes is too small. */
int kvq_decode(kvq_handle* h, const void* pool, int num_pool_pages,
               const uint16_t* q, const int32_t* page_table, int max_pages,
               const int32_t* seq_lens, int batch, float* out,
               void* workspace, size_t ws_bytes, int num_splits, void* stream);

/* ---- append and decode in one call ---------------------------------------------
 * The usual decode step: every sequence b with seq_lens[b] >= 1 gets one new
 * token, at position seq_lens[b] - 1, then attends over [0, seq_lens[b]).
 * Equal, byte for byte in the pool and bit for bit in out, to
 *     kvq_append(K_new[b], V_new[b] at (b, seq_lens[b] - 1) for each such b)
 *     kvq_decode(...same arguments...)
 * but the append and the query rotation run in one kernel, so a step is three
 * kernel launches instead of four.
 *   K_new, V_new : device bf16 [batch][Hkv][D], 4-byte aligned.
 *   pool         : written (the new tokens' slots) and read.
 *   other arguments, errors and status bits as for kvq_append / kvq_decode
 *   (a sequence whose new position has no valid page sets
 *   KVQ_STATUS_BAD_PAGE; its token is not stored). */
int kvq_append_decode(kvq_handle* h, void* pool, int num_pool_pages,
                      const uint16_t* K_new, const uint16_t* V_new, const uint16_t* q,
                      const int32_t* page_table, int max_pages, const int32_t* seq_lens,
                      int batch, float* out, void* workspace, size_t ws_bytes,
                      int num_splits, void* stream);

/* ---- decode with a BF16 sink + recent window ----------------------------------
 * The OptR setting ("Assumptions & free parameters" of the OptR page: a BF16
 * window of 64 sink and 256 recent tokens beside the INT2 cache).  For every
 * sequence b and query head h, with len = seq_lens[b], position t is a window
 * position if t < sink or t >= len - recent; the others are INT2 positions:
 *     logit_t = sm_scale * q . k_t                    window  (BF16 cache, plain q)
 *     logit_t = sm_scale * (q_rot . k~_t + q . mu)    INT2    (centring undone)
 *     value_t = v_t (window)  or  v~_t * R_V^T (INT2)
 *     out     = softmax(logit) . value               (out * R_V if KVQ_OUT_ROTATED)
 * One softmax spans both kinds; q . mu puts the INT2 logits on the scale of the
 * window ones.  sink = recent = 0 equals kvq_decode (up to that constant,
 * which softmax ignores); a window covering [0, len) equals kvq_bf16_decode.
 *   pool, page_table        : the INT2 cache, read at INT2 positions only.
 *   bf16_pool               : device, BF16 page records (kvq_bf16_append),
 *                             16-byte aligned, bf16_num_pool_pages pages.
 *   bf16_page_table         : device int32 [batch][max_pages] (same max_pages as
 *                             page_table); only entries of pages that hold a
 *                             window position are read, so a caller may keep
 *                             BF16 pages for the window alone.
 *   sink, recent            : >= 0, any values (not tied to the page size).
 *   workspace               : as for kvq_decode (kvq_workspace_bytes).
 * Other arguments, errors and status bits as for kvq_decode; a window page id
 * out of range sets KVQ_STATUS_BAD_PAGE and the page is skipped. */
int kvq_decode_window(kvq_handle* h, const void* pool, int num_pool_pages,
                      const void* bf16_pool, int bf16_num_pool_pages,
                      const int32_t* bf16_page_table, const uint16_t* q,
                      const int32_t* page_table, int max_pages, const int32_t* seq_lens,
                      int batch, int sink, int recent, float* out, void* workspace,
                      size_t ws_bytes, int num_splits, void* stream);

/* ---- append and window decode in one call -------------------------------------
 * The decode step of the windowed setting above: every sequence b with
 * seq_lens[b] >= 1 gets one new token at position seq_lens[b] - 1, stored in
 * both caches (the INT2 copy serves once the token leaves the window), then
 * attends as kvq_decode_window.  Equal, byte for byte in both pools and bit for
 * bit in out, to
 *     kvq_append(K_new[b], V_new[b] at (b, seq_lens[b] - 1) for each such b)
 *     kvq_bf16_append(the same tokens into bf16_pool through bf16_page_table)
 *     kvq_decode_window(...same arguments...)
 * in three kernel launches instead of five.
 *   K_new, V_new : device bf16 [batch][Hkv][D], 4-byte aligned.
 *   pool, bf16_pool : written (the new tokens' slots) and read.
 * Other arguments, errors and status bits as for those calls (a new position
 * without a valid INT2 or BF16 page sets KVQ_STATUS_BAD_PAGE; that copy of the
 * token is not stored). */
int kvq_append_decode_window(kvq_handle* h, void* pool, int num_pool_pages, void* bf16_pool,
                             int bf16_num_pool_pages, const int32_t* bf16_page_table,
                             const uint16_t* K_new, const uint16_t* V_new, const uint16_t* q,
                             const int32_t* page_table, int max_pages, const int32_t* seq_lens,
                             int batch, int sink, int recent, float* out, void* workspace,
                             size_t ws_bytes, int num_splits, void* stream);

/* ---- test export -----------------------------------------------------------
 * Dequantise positions [start, start+len) of sequence `seq` to fp32 in the
 * rotated (and, for keys, centred) basis: K_out[i][kv][d] = fmaf(code, s, z),
 * likewise V_out.  Both device fp32 [len][Hkv][D].  Either output may be NULL. */
int kvq_dequant(kvq_handle* h, const void* pool, int num_pool_pages,
                const int32_t* page_table, int max_pages, int seq, int start, int len,
                float* K_out, float* V_out, void* stream);

/* ---- BF16 comparison cache -------------------------------------------------
 * Same arguments as kvq_append / kvq_decode, over the BF16 page record.  The
 * keys and values are stored unchanged (no centring, no rotation, no
 * quantisation) and decode computes plain softmax attention with the unrotated
 * query; KVQ_OUT_ROTATED is ignored.  No rotation bank is needed. */
int kvq_bf16_append(kvq_handle* h, void* pool, int num_pool_pages,
                    const uint16_t* K, const uint16_t* V,
                    const int32_t* seq_idx, const int32_t* positions, int n,
                    const int32_t* page_table, int batch, int max_pages, void* stream);
size_t kvq_bf16_workspace_bytes(const kvq_handle* h, int batch, int num_splits);
int kvq_bf16_decode(kvq_handle* h, const void* pool, int num_pool_pages,
                    const uint16_t* q, const int32_t* page_table, int max_pages,
                    const int32_t* seq_lens, int batch, float* out,
                    void* workspace, size_t ws_bytes, int num_splits, void* stream);

/* ---- decode without a caller-supplied workspace ----------------------------
 * The paper has no counterpart: this is a convenience of this library.
 * kvq_decode needs a workspace that the caller allocates.  Callers that cannot
 * allocate one (an integration whose attention-op signature has no workspace
 * argument, or a serving process that reserves all device memory at start-up and
 * forbids allocation on the decode path) can call this instead.  It computes
 * exactly what kvq_decode computes, with its scratch taken from one fixed
 * 16 MiB array in device global memory that every GPU loading the library holds
 * until the process exits.  It calls no allocating routine.
 *   - Arguments as for kvq_decode, without workspace / ws_bytes.
 *   - num_splits == 0: the automatic choice, lowered until the scratch
 *     (kvq_workspace_bytes(h, batch, splits)) fits in 16 MiB.  An explicit
 *     num_splits whose scratch does not fit returns KVQ_ENOSPACE.
 *   - The first call on a device looks up the array's device address (with the
 *     handle's device made current); make that first call before any stream
 *     capture.
 *   - All calls share the one array and it keeps the last call's contents.
 *     Nothing in it needs to start at zero: each call writes every part it
 *     reads.  Calls whose kernels overlap on the GPU (other streams, other
 *     threads, other handles) race on it: order them on one stream. */
int kvq_decode_static(kvq_handle* h, const void* pool, int num_pool_pages,
                      const uint16_t* q, const int32_t* page_table, int max_pages,
                      const int32_t* seq_lens, int batch, float* out, int num_splits,
                      void* stream);

/* ---- OptR rotation calibration (off the decode path) ------------------------
 * Learns, per KV head, the rotations the cache uses: R = R0 exp(A - A^T), the
 * orthogonal correction of a base rotation R0 ("What carries the argument",
 * mechanism (1)), with Adam ("Assumptions & free parameters": 80 steps,
 * lambda_K = 1) through the whole quantised path with a straight-through
 * estimator for the rounding (mechanism (3)); keys first, then values:
 *   keys:   L_K = [ sum_h KL(p_h || p~_h) + lambda_K |sum_h (dp_h V) W_h^T|^2 ] / Nq
 *   values: L_V = [ |sum_h (p~_h dV) W_h^T|^2 ] / Nq,   p~ fixed at the calibrated keys,
 * summed over the last Nq query positions of a causal calibration chunk
 * (the referee report's Eqs. (14), (16); the OptR page's "Assumptions & free
 * parameters" puts the gradient on the final 64 query positions).  p is the attention with the exact keys, p~ with the keys
 * centred by mu, rotated, quantised by this library's INT2 quantiser (fp16
 * scale and zero), dequantised and rotated back; dV likewise for values.  The
 * straight-through backward replaces the rounding by the identity and
 * differentiates the clipping exactly.  A starts at 0; Adam beta1 0.9,
 * beta2 0.999, eps 1e-8 (readings: the pages give none of these).
 *   K, V       : device bf16 [Hkv][T][D] calibration keys / values (positions 0..T-1).
 *   Q          : device bf16 [Hkv][Nq][G][D] queries at positions T-Nq .. T-1.
 *   W_O        : device fp32 [Hkv][Dm][G*D], the KV head's slice of the output
 *                projection (head h's output o_h contributes o_h W_O[:, hD:(h+1)D]^T).
 *   R0         : device fp32 [2][Hkv][D][D] base rotations (keys, values).
 *   mu         : device fp32 [Hkv][D] key means.
 *   lr         : Adam step size (1e-3 is this library's default reading).
 *   sm_scale   : <= 0 selects 1/sqrt(D).
 *   R_out      : device fp32 [2][Hkv][D][D], the calibrated rotations, ready for
 *                kvq_set_rotation.
 *   history    : device fp32 [2][steps + 1][Hkv]: the loss before each Adam step
 *                and after the last one (keys, then values).
 *   workspace  : device, >= kvq_optr_workspace_bytes(...) bytes, 256-byte aligned.
 * The call returns when the calibration has finished (it synchronises `stream`
 * once per evaluation of an objective, to size the matrix exponential).  Shapes: 1 <= Hkv <= 64, 1 <= Nq <= T,
 * 1 <= G <= 8, Dm >= 1; D is 128. */
size_t kvq_optr_workspace_bytes(int num_kv_heads, int T, int Nq, int G, int Dm);
int kvq_optr_calibrate(int num_kv_heads, int T, int Nq, int G, int Dm,
                       const uint16_t* K, const uint16_t* V, const uint16_t* Q,
                       const float* W_O, const float* R0, const float* mu,
                       float clip_k, float clip_v, float lambda_k, float lr, int steps,
                       float sm_scale, float* R_out, float* history,
                       void* workspace, size_t ws_bytes, void* stream);

/* One evaluation of a calibration objective and its gradient, for callers that
 * drive their own optimiser (and for testing): which = 0, the key objective L_K
 * at R_K = R0_K exp(A_key - A_key^T); which = 1, the value objective L_V at
 * R_V = R0_V exp(A_value - A_value^T) with p~ taken at A_key.  A_key, A_value:
 * device fp32 [Hkv][D][D] (A_value may be NULL when which = 0).  loss: device
 * fp32 [Hkv]; grad: device fp32 [Hkv][D][D], d loss / dA (straight-through).
 * Other arguments as for kvq_optr_calibrate.  Returns when done. */
int kvq_optr_loss_grad(int num_kv_heads, int T, int Nq, int G, int Dm,
                       const uint16_t* K, const uint16_t* V, const uint16_t* Q,
                       const float* W_O, const float* R0, const float* mu,
                       float clip_k, float clip_v, float lambda_k, float sm_scale,
                       const float* A_key, const float* A_value, int which,
                       float* loss, float* grad, void* workspace, size_t ws_bytes,
                       void* stream);

/* ---- status and diagnostics ---------------------------------------------- */

/* Read and clear the handle's device status word (KVQ_STATUS_* bits).
 * Synchronises `stream`. */
int kvq_get_status(kvq_handle* h, uint32_t* bits, void* stream);

/* Self-test of the bounded waits: launches one CTA on `stream` whose thread
 * waits on a shared-memory mbarrier that nothing completes, bounded by
 * limit_us microseconds (1 ... 1,000,000) of the GPU's global timer, the same
 * wait every page copy uses (there bounded by two seconds).  The wait gives up
 * and sets KVQ_STATUS_TIMEOUT in the handle's status word; no copy is in
 * flight, so the context stays usable.  Asynchronous; read the bit with
 * kvq_get_status.  Lets a test check the give-up path without a fault. */
int kvq_selftest_wait_timeout(kvq_handle* h, int limit_us, void* stream);

/* The number of splits kvq_decode uses when num_splits == 0. */
int kvq_auto_splits(const kvq_handle* h, int batch, int max_pages);

/* Kernel timing: while enabled, each decode call (kvq_decode, kvq_decode_window,
 * kvq_decode_static, kvq_bf16_decode) records a CUDA event pair around its
 * split-K attention kernel only (not the query preparation, nor the
 * log-sum-exp combine, which are separate kernels).  kvq_profile_read
 * synchronises on the recorded events and returns the summed milliseconds and
 * the number of launches since the last enable, then clears the record. */
int kvq_profile_enable(kvq_handle* h, int enable);
int kvq_profile_read(kvq_handle* h, double* total_ms, int* launches);

/* A static description of a return code.  Never NULL. */
const char* kvq_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H_ */
