/*
 * specverify.h - C ABI of libspecverify.so, the batched lossless
 * speculative-decoding verify step for one GB300 GPU (sm_103a).
 *
 * Pages cited by title and section:
 *   [SD]  "Speculative decoding, the founding scheme" (hotelren.com/news/5905390)
 *   [SSD] "Self-speculative decoding with layer skip and KV reuse" (xdnf.cn/news/378309)
 *   [FS]  "FlashSpec speculative decoding in practice" (nzsm.cn/news/47291)
 *
 * Conventions for every call:
 *   - Pointers marked "device" must be CUDA device (or managed) memory on the
 *     current device; the caller owns every buffer.  The library never
 *     allocates and never frees.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on it and never synchronise the host,
 *     except sv_read_device_flags.
 *   - Arguments the host can check are checked before anything is launched;
 *     a non-OK status means nothing was enqueued.  sv_last_error() then gives
 *     a message (per host thread).
 *   - Problems only the device can see (a draft token outside [0, V), a bad
 *     k_b, non-finite logits, a bad temperature or uniform, a KV capacity
 *     overflow, a bounded wait that ran out) never trap: the affected
 *     sequence's outputs become n_accepted = 0 and out_tokens = -1, and a bit
 *     is set in the workspace's flag word (SV_FLAG_*), readable with
 *     sv_read_device_flags.
 *   - Each call runs on the calling thread's current device.  The kernels'
 *     launch attributes and the device's properties are set up by the first
 *     call on each device (ordinals 0..63; a call on a higher ordinal
 *     returns SV_ERR_CUDA), so one process may use several GPUs.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SV_OK = 0,
  SV_ERR_ARG = 1,          /* a pointer, size or scalar argument is invalid      */
  SV_ERR_SHAPE = 2,        /* B, K, V or a stride is out of the supported range  */
  SV_ERR_DTYPE = 3,        /* unknown dtype                                       */
  SV_ERR_CUDA = 4,         /* a CUDA runtime call failed (message has details)    */
  SV_ERR_WORKSPACE = 5,    /* workspace NULL, misaligned or smaller than needed   */
  SV_ERR_DEVICE_FLAG = 6,  /* sv_read_device_flags found a flag bit set           */
  SV_ERR_TIMEOUT = 7,      /* a bounded device wait ran out (SV_FLAG_TIMEOUT)     */
  SV_ERR_UNSUPPORTED = 8   /* valid request this build does not implement        */
} sv_status;

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

/* Per-row verify mode ([SSD §2.4]: greedy decoding is its own branch). */
enum { SV_SAMPLED = 0, SV_GREEDY = 1 };

/* Bits of the device flag word. */
enum {
  SV_FLAG_BAD_K = 1,           /* k_per_row[b] outside [0, K]                      */
  SV_FLAG_BAD_TOKEN = 2,       /* a tested draft token outside [0, V)              */
  SV_FLAG_NONFINITE = 4,       /* NaN or +inf in a row the rule needed, or a row
                                  that is -inf everywhere                           */
  SV_FLAG_BAD_TEMPERATURE = 8, /* temperature <= 0 or not finite on a sampled row  */
  SV_FLAG_BAD_UNIFORM = 16,    /* a consumed uniform outside [0, 1)                */
  SV_FLAG_BAD_MODE = 32,       /* mode[b] not SV_SAMPLED / SV_GREEDY               */
  SV_FLAG_CAPACITY = 64,       /* kv_commit: seq_len + n would pass capacity       */
  SV_FLAG_TIMEOUT = 128,       /* a bounded device wait ran out                    */
  SV_FLAG_BAD_N = 256          /* kv_commit: n_accepted outside [0, K] or above k_b */
};

/* Optional per-(sequence, position) diagnostics, float32 [B][K+1][SV_DIAG_FIELDS],
 * written only for the rows the call actually read (others untouched).  The
 * caller may pre-fill with NaN to tell them apart.  S values are
 * sum_v exp((z_v - m)/T); p, q are the processed probabilities of the draft
 * token; M the kept mass of top-p (1 without it). */
enum {
  SV_DIAG_M_T = 0,    /* target row max                                   */
  SV_DIAG_S_T = 1,    /* target normaliser                                */
  SV_DIAG_MASS_T = 2, /* target kept mass                                 */
  SV_DIAG_P_X = 3,    /* p'(x_i)                                          */
  SV_DIAG_M_D = 4,    /* draft row max                                    */
  SV_DIAG_S_D = 5,    /* draft normaliser                                 */
  SV_DIAG_MASS_D = 6, /* draft kept mass                                  */
  SV_DIAG_Q_X = 7,    /* q'(x_i)                                          */
  SV_DIAG_RATIO = 8,  /* p'(x_i) / q'(x_i) (0 if q' = 0)                  */
  SV_DIAG_ARGMAX = 9, /* greedy rows: target argmax (as float)            */
  SV_DIAG_S_W = 10,   /* at the cut: residual mass sum max(0, p' - q')    */
  SV_DIAG_FIELDS = 16
};

/* Library version (major*10000 + minor*100 + patch). */
int sv_version(void);

/* Bytes of device workspace sv_spec_verify, sv_kv_commit and
 * sv_lmhead_rmsnorm need for these sizes (V and dt are accepted for future
 * layouts; today the size depends on B and K only).  Returns 0 if the sizes
 * are out of range.  The workspace must be 256-byte aligned.  Its first four
 * bytes are the device flag word. */
size_t sv_workspace_size(int B, int K, int V, sv_dtype dt);

/*
 * sv_spec_verify - the verify step of one speculative round, batched.
 *
 * [SD §2.1-§2.2], [SSD §2.4, §4.3], [FS §2.3, §3.2, §5.4].  For every
 * sequence b with k = k_per_row[b] drafts x_0..x_{k-1}:
 *   sampled rows: p_i = softmax(z_target[b,i]/T_b), q_i = softmax(z_draft[b,i]/T_b),
 *     both truncated to top_p and renormalised when top_p < 1 (the same mask
 *     rule on both sides).  Position i is accepted iff u[b,i] < p_i(x_i)/q_i(x_i)
 *     (ratio 0 when q_i(x_i) = 0).  At the first rejection j the call draws
 *     y from norm(max(0, p_j - q_j)) (from p_j if that is all zero) with the
 *     single uniform u[b,K]; if all k are accepted it draws the bonus token
 *     y from p_k with u[b,K].  Draws are inverse-CDF in token-index order:
 *     y = min{v : C(v) > u * sum(w)}.
 *   greedy rows: a_i = argmax z_target[b,i] (lowest index on ties); accept
 *     while x_i == a_i; y = a_j at the first mismatch, or a_k as the bonus.
 *   Outputs: out_tokens[b] = x_0..x_{n-1}, y, then -1 up to K+1 entries;
 *   n_accepted[b] = n.  Rows after the first rejection do not affect the
 *   result and are not read.
 *
 *   target_logits   device, dtype, element (b,i,v) at
 *                   b*target_seq_stride + i*target_pos_stride + v, i in 0..K;
 *                   strides in elements, 0 selects the packed [B][K+1][V] layout.
 *   draft_logits    device, dtype, (b,i,v) at b*draft_seq_stride + i*draft_pos_stride + v,
 *                   i in 0..K-1; 0 strides select [B][K][V].  May be NULL only if
 *                   every row is greedy (mode non-NULL).
 *   dtype           SV_F32 or SV_BF16 (both logit tensors).
 *   B, K, V         sequences, max drafts (0 <= K <= 20), vocabulary (V >= 1);
 *                   B * (K + 1) <= 134217727 (each position is one cluster of
 *                   up to 16 CTAs and the grid holds at most 2^31 - 1).
 *   draft_tokens    device int32 [B][K]; only the first k_b of a row are read.
 *   k_per_row       device int32 [B] (each 0..K) or NULL for K everywhere.
 *   temperature     device float32 [B] (> 0 on sampled rows) or NULL for 1.0.
 *   top_p           (0, 1]; 1 disables the mask.
 *   uniforms        device float32 [B][K+1], values in [0, 1): column i < k_b
 *                   tests position i, column K is the resample / bonus draw.
 *   mode            device uint8 [B] of SV_SAMPLED / SV_GREEDY, or NULL for all
 *                   sampled.
 *   out_tokens      device int32 [B][K+1] (written).
 *   n_accepted      device int32 [B] (written).
 *   diag            device float32 [B][K+1][SV_DIAG_FIELDS] or NULL.
 *   workspace       device, >= sv_workspace_size(B, K, V, dtype) bytes, 256-B
 *                   aligned; contents need no initialisation; calls that share
 *                   a workspace must be ordered on one stream.
 * Outputs must not alias inputs.  Logit rows need not be 16-byte aligned
 * (the 16-byte-aligned body of a row is read with 16-byte asynchronous
 * copies, cp.async, and its ragged ends element by element).
 */
sv_status sv_spec_verify(const void* target_logits, int64_t target_seq_stride,
                         int64_t target_pos_stride, const void* draft_logits,
                         int64_t draft_seq_stride, int64_t draft_pos_stride, sv_dtype dtype,
                         int B, int K, int V, const int32_t* draft_tokens,
                         const int32_t* k_per_row, const float* temperature, float top_p,
                         const float* uniforms, const uint8_t* mode, int32_t* out_tokens,
                         int32_t* n_accepted, float* diag, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * sv_spec_verify_target_topp - sv_spec_verify with top-p applied to the target
 * rows only: the draft keeps its untruncated temperature softmax q in the
 * ratio p'(x)/q(x) and in the residual max(0, p' - q), the option
 * "Self-speculative decoding with layer skip and KV reuse" §3.4 prefers.  The
 * emitted tokens still follow the truncated target p'.  Same arguments,
 * layouts, ownership and errors as sv_spec_verify; with top_p = 1 the two
 * calls are identical.
 */
sv_status sv_spec_verify_target_topp(const void* target_logits, int64_t target_seq_stride,
                                     int64_t target_pos_stride, const void* draft_logits,
                                     int64_t draft_seq_stride, int64_t draft_pos_stride,
                                     sv_dtype dtype, int B, int K, int V,
                                     const int32_t* draft_tokens, const int32_t* k_per_row,
                                     const float* temperature, float top_p, const float* uniforms,
                                     const uint8_t* mode, int32_t* out_tokens, int32_t* n_accepted,
                                     float* diag, void* workspace, size_t workspace_bytes,
                                     void* stream);

/*
 * sv_spec_verify_noalloc - sv_spec_verify for callers that cannot allocate
 * device memory.  The pages describe no such call; it exists for embedders
 * such as plugins inside an inference server whose device memory is owned
 * and budgeted by the host framework, or real-time loops that must not take
 * the synchronisation a cudaMalloc implies, and that therefore have no
 * workspace to hand over.
 *
 * Same arguments, meaning and results as sv_spec_verify, minus the
 * workspace: the scratch lives in a 2 MiB array inside the library, present
 * on every GPU that loads it until the process exits.  The call allocates
 * nothing and frees nothing.
 *   - Limit: sv_workspace_size(B, K, V, dtype) must be <= 2 MiB (for example
 *     B <= 4096 with any K <= 20, B = 8192 with K <= 14, or B = 16384 with
 *     K <= 6); larger batches return SV_ERR_WORKSPACE without launching
 *     anything.
 *   - The first call on each device looks up that device's copy of the
 *     array (with the device current); make that first call before any
 *     stream capture.
 *   - All calls share the one array.  Each call clears what must start at
 *     zero, so calls ordered on one stream are independent; calls that can
 *     run at the same time on the GPU (other streams, other host threads)
 *     race on it and must be serialised by the caller.
 *   - The device flag word of these calls is not exposed (per-sequence
 *     errors still show as n_accepted = 0 and out_tokens = -1).
 */
sv_status sv_spec_verify_noalloc(const void* target_logits, int64_t target_seq_stride,
                                 int64_t target_pos_stride, const void* draft_logits,
                                 int64_t draft_seq_stride, int64_t draft_pos_stride,
                                 sv_dtype dtype, int B, int K, int V, const int32_t* draft_tokens,
                                 const int32_t* k_per_row, const float* temperature, float top_p,
                                 const float* uniforms, const uint8_t* mode, int32_t* out_tokens,
                                 int32_t* n_accepted, float* diag, void* stream);

/*
 * sv_kv_commit - roll each sequence's KV write pointer back to its accepted
 * length [SSD §3.3, §4.3; SD §4.3].  seq_lens[b] holds the length at the start
 * of the round (the drafts were written at seq_lens[b] .. seq_lens[b]+k_b-1);
 * afterwards it is seq_lens[b] + n_accepted[b], and cache entries at or past
 * it are stale.  The resampled / bonus token's KV is written next round.
 *   seq_lens    device int32 [B], read and written.
 *   n_accepted  device int32 [B] (e.g. from sv_spec_verify).
 *   capacity    device int32 [B] or NULL: a row whose new length would exceed
 *               capacity[b] is left unchanged and sets SV_FLAG_CAPACITY.
 *   k_per_row   device int32 [B] (the round's k_b) or NULL: with it, a row
 *               whose n_accepted exceeds k_b (more accepted than drafted) is
 *               left unchanged and sets SV_FLAG_BAD_N.
 *   K           if >= 0, n_accepted outside [0, K] leaves the row unchanged
 *               and sets SV_FLAG_BAD_N; if < 0 only n < 0 (and n > k_b when
 *               k_per_row is given) is rejected.  Without k_per_row, n in
 *               (k_b, K] of a ragged round cannot be told from a valid one.
 *   workspace   the verify workspace (its flag word is OR-ed, not cleared);
 *               at least 256 bytes.
 *   B           1 <= B <= 2^30, else SV_ERR_SHAPE.
 */
sv_status sv_kv_commit(int32_t* seq_lens, const int32_t* n_accepted, const int32_t* capacity,
                       const int32_t* k_per_row, int B, int K, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * sv_kv_commit_paged - sv_kv_commit for a paged KV cache ["Self-speculative
 * decoding with layer skip and KV reuse" §3.3, §4.5]: the write pointer moves
 * to seq_lens[b] + n_accepted[b] (= L'), pages 0 .. ceil(L'/page_size) - 1 of
 * the sequence stay, and every allocated page from index ceil(L'/page_size)
 * on is pushed on the free stack and its block-table entry set to -1.
 *   seq_lens      device int32 [B], read and written: the length at the start
 *                 of the round (the drafts were written at L .. L + k_b - 1).
 *   n_accepted    device int32 [B]; k_per_row device int32 [B] (the round's k).
 *   block_table   device int32 [B][max_pages], read and written: page ids,
 *                 -1 for none.
 *   free_pages    device int32 [free_capacity]: the free stack; released ids
 *                 are written at free_top onwards, in no fixed order.
 *   free_top      device int32 [1]: the stack's size, read and advanced.
 *   workspace     device, >= 16 bytes, 16-byte aligned: word 0 is the flag
 *                 word (OR-ed, not cleared; e.g. the verify workspace), words 1
 *                 and 2 are scratch.
 *   B, max_pages, page_size  1 <= B <= 2^30; lengths are int32 on the device,
 *                 so (max_pages + 1) * page_size must fit in int32; else
 *                 SV_ERR_SHAPE.
 * A sequence with n_accepted outside [0, k_b], or with L + k_b beyond its
 * table, is left unchanged and sets SV_FLAG_BAD_N.  If the call's releases
 * together would overflow the free stack, nothing changes and
 * SV_FLAG_CAPACITY is set.
 */
sv_status sv_kv_commit_paged(int32_t* seq_lens, const int32_t* n_accepted,
                             const int32_t* k_per_row, int32_t* block_table, int max_pages,
                             int page_size, int32_t* free_pages, int32_t* free_top,
                             int free_capacity, int B, void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * sv_dynk_init / sv_dynk_update - the dynamic draft length that feeds
 * k_per_row ["Self-speculative decoding with layer skip and KV reuse" §3.2,
 * §5.3]: each sequence's k follows its acceptance rate over the last 64
 * rounds in which it proposed drafts (tokens accepted / tokens proposed);
 * when that rate crosses above 0.85, k grows by one; when it crosses below
 * 0.7, it shrinks by one; k stays in [2, 8].  A crossing counts once, in the
 * round where the rate passes the threshold, and the tests are exact
 * (20*accepted > 17*proposed, 10*accepted < 7*proposed).
 *   state       device buffer of sv_dynk_state_size(B) bytes, 16-byte
 *               aligned, owned by the caller and kept between rounds;
 *               sv_dynk_init sets every k to k0 clamped to [2, 8] and empties
 *               the windows.
 *   n_accepted  device int32 [B]: the round's accepted lengths (e.g. from
 *               sv_spec_verify).
 *   k_used      device int32 [B]: the round's k_per_row (0: the sequence did
 *               not speculate; the round is not recorded).
 *   cap         device int32 [B] or NULL: bounds the next round's k (e.g. a
 *               context-length policy); the controller's own k is unchanged.
 *   k_next      device int32 [B]: min(k, cap), or 0 (no speculation) when
 *               that is below 2.
 *   workspace   a flag word (e.g. the verify workspace): a round with k_used
 *               outside [0, 255] or n_accepted outside [0, k_used] is not
 *               recorded and sets SV_FLAG_BAD_N.
 *   B           1 <= B <= 2^30 (sv_dynk_state_size returns 0 outside it, the
 *               other two SV_ERR_SHAPE).
 */
size_t sv_dynk_state_size(int B);
sv_status sv_dynk_init(void* state, int B, int k0, void* stream);
sv_status sv_dynk_update(void* state, int B, const int32_t* n_accepted, const int32_t* k_used,
                         const int32_t* cap, int32_t* k_next, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * sv_draft_sample - the draft side of a round: draw each sequence's k_b draft
 * tokens from its rows of draft logits [FS §3.2; SSD §3.2, §4.2].  Token i of
 * sequence b comes from row (b, i) with the processing sv_spec_verify applies
 * to its rows: the temperature softmax, top-p truncation with renormalisation
 * when top_p < 1, and the inverse CDF in index order with the uniform
 * uniforms[b*K + i] (the smallest v whose inclusive prefix of p' exceeds
 * u times the total); a greedy row (mode 1) takes the argmax, lowest index on
 * ties.  Rows are independent, so the call serves both a whole block of k
 * rows and one row per draft step (K = 1).
 *   draft_logits  device [B][K][V] of dtype; element strides per sequence and
 *                 per position as for sv_spec_verify (0 = dense).
 *   B, K, V       each >= 1, B * K <= 134217727 (one cluster per row).
 *   k_per_row     device int32 [B] in [0, K], or NULL (= K).
 *   temperature   device float32 [B] (> 0 for sampled rows), or NULL (= 1).
 *   top_p         in (0, 1].
 *   uniforms      device float32 [B][K] in [0, 1).
 *   mode          device uint8 [B] (0 sampled, 1 greedy), or NULL (= 0).
 *   out_tokens    device int32 [B][K]: the tokens; -1 at positions i >= k_b.
 *   workspace     device, >= sv_draft_sample_workspace_size() bytes, 256-byte
 *                 aligned; its first four bytes are the device flag word.
 * Per-position errors write -1 there and set SV_FLAG_NONFINITE (NaN, +inf or
 * an all -inf row) or SV_FLAG_BAD_UNIFORM; a bad k_b, mode or temperature
 * writes -1 at every position of the sequence and sets SV_FLAG_BAD_K /
 * _BAD_MODE / _BAD_TEMPERATURE.  Host-side argument errors return before any
 * launch.
 */
size_t sv_draft_sample_workspace_size(void);
sv_status sv_draft_sample(const void* draft_logits, int64_t seq_stride, int64_t pos_stride,
                          sv_dtype dtype, int B, int K, int V, const int32_t* k_per_row,
                          const float* temperature, float top_p, const float* uniforms,
                          const uint8_t* mode, int32_t* out_tokens, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Bytes of device workspace sv_lmhead_rmsnorm needs for M rows of width H
 * (the normalised, weighted bf16 copy of the hidden states); 0 if out of range. */
size_t sv_lmhead_workspace_size(int M, int H);

/*
 * sv_lmhead_rmsnorm - draft logits from layer-L hidden states through the
 * model's final RMSNorm and output head [SSD §3.1, §4.2]: the norm must not be
 * skipped when leaving at an intermediate layer.
 *   logits[m][n] = sum_k ( w[k] * h[m][k] / sqrt(mean_k h[m][k]^2 + eps) ) * W[k][n]
 *   hidden   device bf16 [M][H] row-major.
 *   norm_w   device bf16 [H].
 *   W        device bf16 [H][V] row-major (V contiguous).
 *   logits   device [M][V], out_dtype SV_BF16 or SV_F32.
 *   M, H, V  M >= 1; H % 64 == 0; V % 16 == 0 (tcgen05 tile and TMA rules).
 *   workspace   >= sv_lmhead_workspace_size(M, H) bytes, 256-byte aligned.
 * bf16 products, fp32 accumulation on the tensor cores.
 */
sv_status sv_lmhead_rmsnorm(const void* hidden, const void* norm_w, float eps, const void* W,
                            void* logits, sv_dtype out_dtype, int M, int H, int V,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * sv_read_device_flags - synchronise `stream` and copy the workspace's flag
 * word to *flags_host.  Returns SV_OK if it is 0, SV_ERR_TIMEOUT if
 * SV_FLAG_TIMEOUT is set, else SV_ERR_DEVICE_FLAG.
 */
sv_status sv_read_device_flags(const void* workspace, uint32_t* flags_host, void* stream);

/* Message for the last non-OK status returned on this host thread. */
const char* sv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
