/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact-attention library.
 *
 * The library computes exact scaled-dot-product attention,
 *
 *     x_ij = scale * <q_i, k_j> + b_ij        for j in J_i (the visible keys of row i)
 *     o_i  = sum_j exp(x_ij - m_i) v_j / l_i,  m_i = max_j x_ij,  l_i = sum_j exp(x_ij - m_i)
 *     lse_i = m_i + ln l_i
 *
 * tile by tile with the mergeable per-row state (m, l, u): a running maximum, the
 * exponential sum measured against it and the unnormalised value sum, both rescaled by
 * exp(m_old - m_new) when the maximum grows, and divided once per row at the end.
 *
 * Sources (page title, then section / step / figure):
 *   "How Does FlashAttention Preserve Global Softmax Across Tiles?"
 *       section 1  the operator, visible set J_i, fixed bias b_ij, d_k != d_v allowed,
 *                  scale independent of tile size;
 *       section 3  the state (m, l, u) and the merge of disjoint key subsets;
 *       section 5  tile loop, rows keep their own state, divide once at the end;
 *       section 6  global positions; causal masks align the two sequences' ends
 *                  ("bottom-right"); an entirely empty row returns zero; dropout is
 *                  disabled there, and a training backward must reproduce the forward's
 *                  mask and scaling (the keep mask of attn_fwd is therefore an input);
 *       section 7  the saved log-sum-exp L_i, and the backward that rebuilds the
 *                  probabilities from it (attn_bwd);
 *       section 8  decode (one query row, or a few, against a long key/value cache) split
 *                  over the keys, the partial states merged.
 *   "Flash attention and efficient attention: Visual walkthrough", Steps 4-5 (the three
 *       running numbers; re-basing a sum to a new maximum by one multiply).
 *   "Reducing Memory Traffic with Output Accumulation in FlashAttention", Figures 1-3
 *       (value-weighted sum first, both accumulators rescaled, one division).
 *
 * Conventions shared by every entry point:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; it must stay valid until
 *     the work queued on `stream` has finished.  The library keeps no pointer after a call
 *     returns and allocates no device memory.
 *   - All work is queued asynchronously on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) on the current CUDA device.
 *   - Arguments are checked on the host before anything is queued; a bad argument returns a
 *     non-zero attn_status_t and queues nothing.  attn_last_error() then describes it.
 *     No entry point throws or aborts.
 *   - Visible set J_i of query row i of batch entry b, with n_b = kv_lens[b] clamped to
 *     [0, Nk] (Nk when kv_lens is NULL):  j < n_b, and, when causal,
 *     j <= i + n_b - Nq (bottom-right alignment), and b_ij != -inf.
 *     Nothing stored at a masked position is ever used: NaN there cannot reach an output.
 *   - An empty row (J_i empty) gives o_i = +0.0 and lse_i = -inf, exactly.
 *   - Accumulation is fp32.  bf16 outputs are rounded to nearest even once, at the end.
 */
#ifndef ONLINE_SOFTMAX_FA2_GB300_ATTN_H
#define ONLINE_SOFTMAX_FA2_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *attn_stream_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,    /* null pointer, negative size, bad stride, bad scale */
    ATTN_ERR_UNSUPPORTED = 2,    /* valid, but this build has no kernel for it (e.g. head dim) */
    ATTN_ERR_MISALIGNED = 3,     /* a pointer or stride breaks the 16-byte rule of the path */
    ATTN_ERR_CUDA = 4,           /* a CUDA runtime call or a launch failed */
    ATTN_ERR_DEVICE_TIMEOUT = 5, /* a kernel gave up a bounded wait (see attn_device_error_flags) */
    ATTN_ERR_WORKSPACE = 6       /* the workspace is missing, misaligned or too small */
} attn_status_t;

typedef enum {
    ATTN_DTYPE_F32 = 0,   /* q, k, v, o are float32 */
    ATTN_DTYPE_BF16 = 1   /* q, k, v, o are bfloat16 */
} attn_dtype_t;

/*
 * Arguments of one attention forward.
 *
 *   q  [B, Nq, H, dk]   element (b, i, h, c) at q + b*q_stride[0] + i*q_stride[1]
 *                       + h*q_stride[2] + c          (strides in ELEMENTS; c contiguous)
 *   k  [B, Nk, H, dk]   same with k_stride;  v [B, Nk, H, dv] with v_stride
 *   o  [B, Nq, H, dv]   written, with o_stride
 *   lse [B, H, Nq]      fp32, contiguous, written; may be NULL
 *   bias                NULL, or fp32 b_ij of (b, h, i, j) at
 *                       bias + b*bias_stride[0] + h*bias_stride[1] + i*bias_stride[2] + j;
 *                       a stride of 0 broadcasts; -inf masks the position; bias is added
 *                       after scaling and is not scaled
 *   kv_lens             NULL, or device int32 [B]: keys j >= kv_lens[b] are padding
 *   causal              0: no causal mask; 1: bottom-right causal mask
 *   scale               multiplies <q_i, k_j>; the standard operator uses 1/sqrt(dk)
 *   block_k             float32 path only: key tile size 16, 32 or 64 (0 picks 64);
 *                       must be 0 for bfloat16
 *
 * bfloat16 path (tcgen05 tensor cores): dk in {64, 128, 192}, dv in {64, 128},
 *   scale > 0; q, k, v, o base pointers 16-byte aligned and their b, n, h strides non-zero
 *   multiples of 8 elements (16 bytes); bias 4-byte aligned (rows that are 16-byte aligned
 *   are read with 16-byte loads).
 * float32 path (exact fp32 SIMT): 1 <= dk, dv <= 256; any finite scale.
 *
 *   dropout_mask        NULL: no dropout.  Otherwise the keep mask of a training forward:
 *                       key j of row i of (b, h) is kept iff bit (j % 8) of byte
 *                       dropout_mask[b*s0 + h*s1 + i*s2 + j/8] is set (s = dropout_mask_stride,
 *                       in bytes; each row holds at least 16*ceil(Nk/128) bytes).  Kept
 *                       weights p_ij are scaled by 1 / (1 - dropout_p), dropped ones count 0
 *                       in o; the row sum and lse are those of the undropped softmax.  The
 *                       mask is an input so that a backward can reproduce it ("How Does
 *                       FlashAttention Preserve Global Softmax Across Tiles?", section 6,
 *                       disables dropout and asks exactly that of a training backward).
 *                       bfloat16: dk <= 128 only, the mask 16-byte aligned with strides that
 *                       are multiples of 16 bytes.  Not taken by attn_decode_splitkv, nor by
 *                       attn_bwd together with a bias (ATTN_ERR_UNSUPPORTED).
 *   dropout_p           in [0, 1) with a mask or with dropout_rng = 1; must be 0 otherwise.
 *   dropout_rng         0: the keep decisions come from dropout_mask (or there is no dropout).
 *                       1: they are drawn in-kernel, and no mask is read or stored anywhere:
 *                       the drop probability is quantised to p8 / 256, p8 = round(256 p) (at
 *                       most 255), and key j of row i of (b, h) is kept iff byte j % 16 of the
 *                       counter-based generator Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
 *                       "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11) at counter
 *                       (i, j / 16, b*H + h, dropout_offset mod 2^32) under key (dropout_seed
 *                       mod 2^32, dropout_seed div 2^32) -- its four output words in order,
 *                       each little-endian -- is at least p8; kept weights are scaled by
 *                       256 / (256 - p8).  dropout_mask must then be NULL.  attn_bwd given the
 *                       forward's (dropout_p, dropout_rng, dropout_seed, dropout_offset) draws
 *                       the same decisions.  Where a mask is not taken (see dropout_mask), the
 *                       in-kernel draw is not either.
 *   dropout_seed, dropout_offset  the generator's key and the fourth counter word (a fresh
 *                       offset per training step gives fresh decisions).
 */
typedef struct {
    int32_t dtype;           /* attn_dtype_t */
    int32_t causal;          /* 0 or 1 */
    int64_t B, H, Nq, Nk, dk, dv;
    const void *q;
    const void *k;
    const void *v;
    void *o;
    int64_t q_stride[3];     /* b, n, h */
    int64_t k_stride[3];
    int64_t v_stride[3];
    int64_t o_stride[3];
    float *lse;
    const float *bias;
    int64_t bias_stride[3];  /* b, h, i (j stride is 1) */
    const int32_t *kv_lens;
    float scale;
    int32_t block_k;
    const uint8_t *dropout_mask;
    int64_t dropout_mask_stride[3];  /* b, h, i (bytes) */
    float dropout_p;
    int32_t dropout_rng;             /* 0: keep bits from dropout_mask; 1: drawn in-kernel */
    uint64_t dropout_seed;
    uint64_t dropout_offset;
} attn_fwd_params_t;

/*
 * attn_fwd -- O and lse of exact attention for every (b, h, i).
 * ("How Does FlashAttention Preserve Global Softmax Across Tiles?", sections 1, 5, 6, 7.)
 * Queues one kernel.  Nq == 0 or B*H == 0 queues nothing and returns ATTN_OK.  Nk == 0 is
 * legal (every row is empty; k and v may then be NULL).
 */
attn_status_t attn_fwd(const attn_fwd_params_t *params, attn_stream_t stream);

/*
 * Size in bytes of the workspace attn_decode_splitkv needs for Nq query rows per sequence:
 * the per-split partial states, float32 [B, H, Nq, num_splits, 2 + dv] laid out
 * (m, l, u[0..dv)), where m is the maximum logit of the split (natural-log units),
 * l = sum exp(x_j - m) and u = sum exp(x_j - m) v_j over the keys of the split visible to
 * that row; an empty split is (-inf, 0, 0...).  Returns 0 for a negative or zero size.
 */
size_t attn_decode_workspace_bytes_rows(int64_t B, int64_t H, int64_t Nq, int64_t dv,
                                        int32_t num_splits);

/* attn_decode_workspace_bytes_rows with Nq = 1: float32 [B, H, num_splits, 2 + dv]. */
size_t attn_decode_workspace_bytes(int64_t B, int64_t H, int64_t dv, int32_t num_splits);

/*
 * attn_decode_splitkv -- a few query rows per (b, h) (1 <= params->Nq <= 8: one decode
 * step, or several tokens of one sequence at once) against a long key/value cache, the keys
 * of each sequence split into num_splits contiguous near-equal ranges of [0, n_b) (split s
 * covers [floor(s*n_b/S), floor((s+1)*n_b/S))).  Each key row of the cache is read once for
 * all Nq query rows.  params->causal applies the bottom-right mask of the conventions above
 * (row i sees keys j <= i + n_b - Nq), so the last row sees the whole sequence; a row that
 * sees no key is empty.
 * ("How Does FlashAttention Preserve Global Softmax Across Tiles?", section 8, decode;
 *  section 6, bottom-right alignment; section 3, merge.)
 * Queues two kernels on `stream`: the split kernel writes every partial state into
 * `workspace` (layout above), then the merge kernel writes o and lse exactly as attn_fwd
 * would.  The workspace is caller-owned device memory of at least
 * attn_decode_workspace_bytes_rows(B, H, Nq, dv, num_splits) bytes, 16-byte aligned; after
 * the call it holds the partial states.  Supported: bfloat16, dk == dv in {64, 128},
 * 1 <= num_splits <= 256.  Nq outside [1, 8] returns ATTN_ERR_INVALID_ARG.  The cache may
 * use any strides that keep each key row contiguous and 16-byte aligned (e.g. a [B, H, L, d]
 * cache passed with k_stride = {H*L*d, d, L*d}).
 */
attn_status_t attn_decode_splitkv(const attn_fwd_params_t *params, int32_t num_splits,
                                  void *workspace, size_t workspace_bytes,
                                  attn_stream_t stream);

/*
 * Size in bytes of the workspace attn_decode_splitkv_fused needs: the partial states exactly as
 * for attn_decode_splitkv (attn_decode_workspace_bytes_rows, rounded up to a multiple of 16),
 * then one 64-bit arrival counter per (b, h), [B, H].  Returns 0 for a negative or zero size.
 */
size_t attn_decode_fused_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t dv,
                                         int32_t num_splits);

/*
 * attn_decode_splitkv_fused -- attn_decode_splitkv in one kernel: the split kernel also does
 * the merge.  ("How Does FlashAttention Preserve Global Softmax Across Tiles?", section 8:
 * the extra partial round trip and merge launch of split-KV decode; section 3, the merge.)
 * Every split CTA writes its partial states, makes them visible device-wide and counts itself
 * on its (b, h)'s counter; the CTA that counts last merges the S states of every query row of
 * that (b, h) (the arithmetic of attn_merge_states) and writes o and lse.  No CTA waits for
 * another.  A counter holds (the call's own tag, count), with a fresh tag for every call, so
 * a count left by an earlier call, or any other contents, reads as zero.
 *   - Same arguments, checks and supported shapes as attn_decode_splitkv; same results, bit
 *     for bit (the same split kernel and the same merge arithmetic).
 *   - workspace: caller-owned device memory of at least attn_decode_fused_workspace_bytes(...)
 *     bytes, 16-byte aligned; its contents on entry do not matter.  After the call the
 *     partial-state part holds the partial states.
 *   - Calls that share a workspace and overlap on the GPU race on it: order them on a stream.
 *   - Bit 0 of the device error word is set if a count had to give up (4096 retries of its
 *     compare-and-swap; with S counting CTAs it retries at most S - 1 times).
 * Queues one kernel.
 */
attn_status_t attn_decode_splitkv_fused(const attn_fwd_params_t *params, int32_t num_splits,
                                        void *workspace, size_t workspace_bytes,
                                        attn_stream_t stream);

/*
 * attn_decode_splitkv_noalloc -- attn_decode_splitkv for callers that cannot allocate device
 * memory when they decode (a framework whose allocator owns the device memory, a plugin
 * handed only its inputs and outputs, a latency-bound loop where cudaMalloc would
 * synchronise the device).  The paper has no counterpart: the pages describe no such variant.
 *   - Same arguments, checks, kernels and results as attn_decode_splitkv, without the
 *     workspace: the partial states go to a device array built into the library, 32 MiB
 *     (B * H * Nq * num_splits * (2 + dv) * 4 bytes must fit; larger problems return
 *     ATTN_ERR_WORKSPACE and queue nothing).  Every device that loads the library holds that
 *     array until the process exits.  No device memory is allocated by any call.
 *   - Arguments are checked exactly as attn_decode_splitkv checks them, and before the size
 *     limit: a bad argument returns its own status, not ATTN_ERR_WORKSPACE.
 *   - The first call from a CUDA context looks up the array's device address (with the
 *     device current) and caches it per device, together with that context's unique id; a
 *     call from a new context (e.g. after cudaDeviceReset) looks it up again.
 *   - All calls share the one array.  Every call writes each partial state it reads, so
 *     nothing needs clearing, but calls whose work overlaps on the GPU (different streams,
 *     several host threads) race on it: order them on one stream.
 */
attn_status_t attn_decode_splitkv_noalloc(const attn_fwd_params_t *params, int32_t num_splits,
                                          attn_stream_t stream);

/*
 * attn_merge_states -- merge S partial states per (b, h) and finalise.
 * ("How Does FlashAttention Preserve Global Softmax Across Tiles?", section 3: put both
 *  maxima into the common maximum, scale l and u of each part by exp(m_s - m), add;
 *  empty parts are skipped.  "Flash attention and efficient attention: Visual
 *  walkthrough", Step 5.)
 *   partials  device fp32 [B, H, S, 2 + dv] as (m, l, u); a part with l == 0 is empty
 *   o         written: row (b, h) at o + b*o_stride[0] + h*o_stride[2] (o_stride[1] unused),
 *             element type o_dtype; u/l, or +0.0 when every part is empty
 *   lse       device fp32 [B, H] written: m + ln l, or -inf when every part is empty; may be
 *             NULL
 * Queues one kernel.
 */
attn_status_t attn_merge_states(const float *partials, int64_t B, int64_t H, int32_t num_splits,
                                int64_t dv, int32_t o_dtype, void *o, const int64_t o_stride[3],
                                float *lse, attn_stream_t stream);

/*
 * attn_fwd_partial -- the state (m, l, u) of every query row over one shard of the keys, for
 * attention split over the key axis (sequence parallelism across devices, or any split that
 * the caller merges later).  ("How Does FlashAttention Preserve Global Softmax Across
 * Tiles?", section 3: the state of a key subset and the merge of disjoint subsets; section 4:
 * every key in exactly one part; section 6: global positions.)
 *   params        as for attn_fwd, with k, v (and bias, if any) holding only the shard's keys:
 *                 params->Nk keys, local key j being global key key_offset + j.  params->o and
 *                 params->lse are not used (may be NULL).  kv_lens and the causal mask are in
 *                 global positions: key J of sequence b is visible to row i iff
 *                 J < min(kv_lens[b], Nk_total) and, when causal, J <= i + n_b - Nq.
 *   key_offset, Nk_total  the shard [key_offset, key_offset + Nk) of a sequence of Nk_total
 *                 keys (0 <= key_offset, key_offset + Nk <= Nk_total <= 2^31 - 1).
 *   partials      device fp32 [B, H, Nq, 2 + dv], 16-byte aligned, written: (m, l, u) with
 *                 l = sum exp(x_j - m) and u = sum exp(x_j - m) v_j over the shard's visible
 *                 keys, measured against the row's reference m (natural-log units): the largest
 *                 visible logit, or a value at most 8 ln 2 below it (the kernel moves its
 *                 reference only when a larger logit exceeds it by more than that; the merge
 *                 is the same for any common reference); (-inf, 0, 0...) for a row that sees
 *                 none of them.
 * Supported: bfloat16, dk == dv in {64, 128}, with or without a bias; no dropout.  Merging the
 * states of shards that cover each sequence's keys exactly once (attn_merge_states_rows)
 * gives attn_fwd's o and lse.  Queues one kernel.
 */
attn_status_t attn_fwd_partial(const attn_fwd_params_t *params, int64_t key_offset, int64_t Nk_total,
                               float *partials, attn_stream_t stream);

/*
 * attn_merge_states_rows -- attn_merge_states for Nq rows per (b, h) and any layout of the
 * parts: state s of row r = (b*H + h)*Nq + i is the 2 + dv floats (m, l, u) at
 * partials + r*row_stride + s*split_stride (strides in floats; 0, 0 mean the decode layout
 * [B, H, Nq, num_splits, 2 + dv]; states gathered from R devices as [R, B, H, Nq, 2 + dv]
 * take row_stride = 2 + dv, split_stride = B*H*Nq*(2 + dv)).  Writes o row (b, i, h) at
 * o + b*o_stride[0] + i*o_stride[1] + h*o_stride[2] (element type o_dtype) and lse [B, H, Nq]
 * (may be NULL); a row whose parts are all empty gets +0.0 and -inf.  1 <= num_splits <= 4096,
 * 1 <= dv <= 1024.  Queues one kernel.
 */
attn_status_t attn_merge_states_rows(const float *partials, int64_t B, int64_t H, int64_t Nq,
                                     int32_t num_splits, int64_t dv, int64_t row_stride,
                                     int64_t split_stride, int32_t o_dtype, void *o,
                                     const int64_t o_stride[3], float *lse, attn_stream_t stream);

/*
 * Arguments of one attention backward: the forward's arguments and outputs (fwd.o and
 * fwd.lse as the forward wrote them; fwd.lse is required), the upstream gradient of O, and
 * the three gradients to write.
 *   dout [B, Nq, H, dv]   bf16, with dout_stride (b, n, h; elements)
 *   dq   [B, Nq, H, dk]   bf16, written;  dk [B, Nk, H, dk], dv [B, Nk, H, dv] likewise
 */
typedef struct {
    attn_fwd_params_t fwd;
    const void *dout;
    int64_t dout_stride[3];
    void *dq;
    int64_t dq_stride[3];
    void *dk;
    int64_t dk_stride[3];
    void *dv;
    int64_t dv_stride[3];
} attn_bwd_params_t;

/*
 * Size in bytes of the workspace attn_bwd needs: an fp32 dQ accumulator [B, Nq, H, dk], the
 * fp32 row terms c_i [B, H, Nq], and lse_i * log2 e [B, H, Nq rounded up to a multiple of 128]
 * in fp32, each part starting on a 16-byte boundary.  Returns 0 for a negative or zero size.
 */
size_t attn_bwd_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t dk);

/*
 * attn_bwd -- gradients dQ, dK, dV of a loss through O = attention(Q, K, V) given the
 * upstream gradient G = dL/dO.
 * ("How Does FlashAttention Preserve Global Softmax Across Tiles?", section 7: the forward
 *  saves each row's log-sum-exp L_i and its output; the backward rebuilds the probabilities
 *  p_ij = exp(x_ij - L_i) tile by tile from Q, K, the fixed mask and bias, takes
 *  c_i = g_i . o_i, dS_ij = p_ij (g_i . v_j - c_i), and accumulates dV_j += p_ij g_i,
 *  dK_j += scale dS_ij q_i, dQ_i += scale dS_ij k_j.)
 * The mask, bias, kv_lens, causal and dropout settings must be the forward's: with a
 * dropout_mask in fwd (the forward's keep bits and dropout_p) the gradient reaching the
 * weights carries the mask and the 1 / (1 - p) scale, dV is formed from the kept, scaled
 * weights, and c_i = g_i . o_i already holds the dropout through o (without a bias only;
 * with one ATTN_ERR_UNSUPPORTED).  The bias is fixed: no gradient is formed for it.  An empty row (lse = -inf) passes no gradient, and a key that no
 * row sees gets dK = dV = 0.
 * Queues three kernels on `stream`: the row terms, the products (on the 5th-generation
 * tensor cores), and the conversion of dQ to bf16.  Supported: bfloat16, dk == dv in {64, 128}; every tensor
 * 16-byte aligned with strides that are multiples of 8 elements.  The workspace is
 * caller-owned device memory of at least attn_bwd_workspace_bytes(B, H, Nq, dk) bytes,
 * 16-byte aligned; its contents on entry do not matter.  dQ is accumulated with atomic
 * additions, so its rounding can differ from run to run in the last bits.
 */
attn_status_t attn_bwd(const attn_bwd_params_t *params, void *workspace, size_t workspace_bytes,
                       attn_stream_t stream);

/* Message describing the last non-OK status returned on the calling thread ("" if none). */
const char *attn_last_error(void);

/*
 * Device error word of the current device (synchronous: waits for the device to finish its
 * queued work first).  Bit 0: a kernel gave up a bounded wait on an mbarrier and returned
 * early (its outputs are then incomplete).  Bit 1: a kv_lens value was outside [0, Nk] and
 * was clamped.  clear != 0 resets the word to 0 after reading.  Returns ATTN_OK or
 * ATTN_ERR_CUDA.
 */
attn_status_t attn_device_error_flags(uint32_t *out, int32_t clear);

/* Library version, major*10000 + minor*100 + patch. */
int32_t attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ONLINE_SOFTMAX_FA2_GB300_ATTN_H */
