// attn_api.cu -- the C ABI: argument checks, dispatch to the kernels, error reporting.
//
// Every check happens here, on the host, before anything is queued; the launchers in the
// other translation units assume valid arguments.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "attn_internal.h"

namespace attn {

static thread_local char g_msg[512] = "";

attn_status_t fail(attn_status_t st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return st;
}

// The device error word: one per device, lives as long as the library is loaded.
__device__ uint32_t g_device_flags;

static constexpr int kMaxDevices = 64;
static uint32_t *g_flag_addr[kMaxDevices];
static int g_sm_count[kMaxDevices];
static std::mutex g_dev_mutex;

uint32_t *device_flags() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_flag_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_device_flags) != cudaSuccess) return nullptr;
        g_flag_addr[dev] = static_cast<uint32_t *>(ptr);
    }
    return g_flag_addr[dev];
}

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static attn_status_t check_strides(const char *name, const int64_t s[3]) {
    for (int i = 0; i < 3; ++i)
        if (s[i] < 0) return fail(ATTN_ERR_INVALID_ARG, "%s_stride[%d] = %lld is negative", name,
                                  i, (long long)s[i]);
    return ATTN_OK;
}

// Dropout of a training forward: a keep mask given, or the keep decisions drawn in-kernel.
static bool has_dropout(const attn_fwd_params_t *p) { return p->dropout_mask || p->dropout_rng == 1; }

// Checks shared by attn_fwd and attn_decode_splitkv.
static attn_status_t check_common(const attn_fwd_params_t *p) {
    if (!p) return fail(ATTN_ERR_INVALID_ARG, "params is NULL");
    if (p->dtype != ATTN_DTYPE_F32 && p->dtype != ATTN_DTYPE_BF16)
        return fail(ATTN_ERR_INVALID_ARG, "dtype %d is not ATTN_DTYPE_F32 or ATTN_DTYPE_BF16",
                    p->dtype);
    if (p->causal != 0 && p->causal != 1)
        return fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1 (got %d)", p->causal);
    if (p->B < 0 || p->H < 0 || p->Nq < 0 || p->Nk < 0)
        return fail(ATTN_ERR_INVALID_ARG, "negative size (B=%lld H=%lld Nq=%lld Nk=%lld)",
                    (long long)p->B, (long long)p->H, (long long)p->Nq, (long long)p->Nk);
    if (p->dk < 1 || p->dv < 1)
        return fail(ATTN_ERR_INVALID_ARG, "head dims must be >= 1 (dk=%lld dv=%lld)",
                    (long long)p->dk, (long long)p->dv);
    if (p->Nk > INT32_MAX || p->Nq > INT32_MAX)
        return fail(ATTN_ERR_UNSUPPORTED, "sequence lengths above 2^31-1 are not supported");
    if (!std::isfinite(p->scale)) return fail(ATTN_ERR_INVALID_ARG, "scale is not finite");
    attn_status_t st;
    if ((st = check_strides("q", p->q_stride)) || (st = check_strides("k", p->k_stride)) ||
        (st = check_strides("v", p->v_stride)) || (st = check_strides("o", p->o_stride)))
        return st;
    if (p->bias)
        for (int i = 0; i < 3; ++i)
            if (p->bias_stride[i] < 0)
                return fail(ATTN_ERR_INVALID_ARG, "bias_stride[%d] is negative", i);
    if (p->dropout_rng != 0 && p->dropout_rng != 1)
        return fail(ATTN_ERR_INVALID_ARG, "dropout_rng must be 0 or 1 (got %d)", p->dropout_rng);
    if (p->dropout_rng == 1 && p->dropout_mask)
        return fail(ATTN_ERR_INVALID_ARG, "dropout_rng = 1 draws the keep decisions: dropout_mask must be NULL");
    if (has_dropout(p)) {
        if (!(p->dropout_p >= 0.0f && p->dropout_p < 1.0f))
            return fail(ATTN_ERR_INVALID_ARG, "dropout_p must be in [0, 1) (got %g)", p->dropout_p);
        if (p->dropout_mask && (st = check_strides("dropout_mask", p->dropout_mask_stride))) return st;
    } else if (p->dropout_p != 0.0f) {
        return fail(ATTN_ERR_INVALID_ARG, "dropout_p = %g without a dropout_mask or dropout_rng", p->dropout_p);
    }
    if (p->B * p->H * p->Nq == 0) return ATTN_OK;
    if (!p->q || !p->o) return fail(ATTN_ERR_INVALID_ARG, "q or o is NULL");
    if (p->Nk > 0 && (!p->k || !p->v))
        return fail(ATTN_ERR_INVALID_ARG, "k or v is NULL while Nk = %lld", (long long)p->Nk);
    return ATTN_OK;
}

static bool stride_mult(const int64_t s[3], int64_t m) {
    return s[0] % m == 0 && s[1] % m == 0 && s[2] % m == 0;
}

}  // namespace attn

using namespace attn;

extern "C" attn_status_t attn_fwd(const attn_fwd_params_t *p, attn_stream_t stream) {
    g_msg[0] = 0;
    attn_status_t st = check_common(p);
    if (st) return st;
    if (p->B * p->H * p->Nq == 0) return ATTN_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (p->dtype == ATTN_DTYPE_F32) {
        if (p->dk > 256 || p->dv > 256)
            return fail(ATTN_ERR_UNSUPPORTED, "float32 path supports dk, dv <= 256 (dk=%lld dv=%lld)",
                        (long long)p->dk, (long long)p->dv);
        if (p->block_k != 0 && p->block_k != 16 && p->block_k != 32 && p->block_k != 64)
            return fail(ATTN_ERR_INVALID_ARG, "block_k must be 0, 16, 32 or 64 (got %d)",
                        p->block_k);
        return launch_fwd_f32(*p, s);
    }
    // bfloat16: tcgen05 tensor-core path
    if (p->dk != 64 && p->dk != 128 && p->dk != 192)
        return fail(ATTN_ERR_UNSUPPORTED, "bfloat16 path supports dk in {64, 128, 192} (got %lld)",
                    (long long)p->dk);
    if (p->dv != 64 && p->dv != 128)
        return fail(ATTN_ERR_UNSUPPORTED, "bfloat16 path supports dv in {64, 128} (got %lld)",
                    (long long)p->dv);
    if (!(p->scale > 0.0f))
        return fail(ATTN_ERR_UNSUPPORTED, "bfloat16 path needs scale > 0 (got %g)", p->scale);
    if (p->block_k != 0)
        return fail(ATTN_ERR_INVALID_ARG, "block_k must be 0 for bfloat16 (got %d)", p->block_k);
    if (!aligned16(p->q) || !aligned16(p->o) || (p->Nk > 0 && (!aligned16(p->k) || !aligned16(p->v))))
        return fail(ATTN_ERR_MISALIGNED, "q, k, v and o must be 16-byte aligned");
    if (!stride_mult(p->q_stride, 8) || !stride_mult(p->k_stride, 8) ||
        !stride_mult(p->v_stride, 8) || !stride_mult(p->o_stride, 8))
        return fail(ATTN_ERR_MISALIGNED, "bfloat16 strides must be multiples of 8 elements");
    if (p->bias && (reinterpret_cast<uintptr_t>(p->bias) & 3u))
        return fail(ATTN_ERR_MISALIGNED, "bias must be 4-byte aligned");
    if (has_dropout(p)) {
        if (p->dk > 128) return fail(ATTN_ERR_UNSUPPORTED, "bfloat16 dropout supports dk <= 128");
        if (p->dropout_mask && (!aligned16(p->dropout_mask) || !stride_mult(p->dropout_mask_stride, 16)))
            return fail(ATTN_ERR_MISALIGNED, "dropout_mask must be 16-byte aligned with strides that are multiples of 16 bytes");
    }
    return launch_fwd_bf16(*p, s);
}

extern "C" size_t attn_decode_workspace_bytes_rows(int64_t B, int64_t H, int64_t Nq, int64_t dv,
                                                   int32_t num_splits) {
    if (B < 0 || H < 0 || Nq < 1 || dv < 1 || num_splits < 1) return 0;
    return (size_t)B * (size_t)H * (size_t)Nq * (size_t)num_splits * (size_t)(2 + dv) * sizeof(float);
}

extern "C" size_t attn_decode_workspace_bytes(int64_t B, int64_t H, int64_t dv, int32_t num_splits) {
    return attn_decode_workspace_bytes_rows(B, H, 1, dv, num_splits);
}

namespace attn {

// Every check attn_decode_splitkv makes before it looks at the workspace, in the same order
// (the allocation-free entry point runs the same ones first).
attn_status_t check_decode_args(const attn_fwd_params_t *p, int32_t num_splits) {
    g_msg[0] = 0;
    attn_status_t st = check_common(p);
    if (st) return st;
    if (p->Nq < 1 || p->Nq > attn::kMaxDecodeRows)
        return fail(ATTN_ERR_INVALID_ARG, "decode needs 1 <= Nq <= %d (got %lld)", attn::kMaxDecodeRows,
                    (long long)p->Nq);
    if (num_splits < 1 || num_splits > 256)
        return fail(ATTN_ERR_INVALID_ARG, "num_splits must be in [1, 256] (got %d)", num_splits);
    if (p->dtype != ATTN_DTYPE_BF16)
        return fail(ATTN_ERR_UNSUPPORTED, "decode supports bfloat16 only");
    if (has_dropout(p)) return fail(ATTN_ERR_UNSUPPORTED, "decode takes no dropout");
    if (p->dk != p->dv || (p->dk != 64 && p->dk != 128))
        return fail(ATTN_ERR_UNSUPPORTED, "decode supports dk == dv in {64, 128} (dk=%lld dv=%lld)",
                    (long long)p->dk, (long long)p->dv);
    if (p->B * p->H == 0) return ATTN_OK;
    if (!aligned16(p->q) || !aligned16(p->o) || (p->Nk > 0 && (!aligned16(p->k) || !aligned16(p->v))))
        return fail(ATTN_ERR_MISALIGNED, "q, k, v and o must be 16-byte aligned");
    if (!stride_mult(p->q_stride, 8) || !stride_mult(p->k_stride, 8) ||
        !stride_mult(p->v_stride, 8) || !stride_mult(p->o_stride, 8))
        return fail(ATTN_ERR_MISALIGNED, "bfloat16 strides must be multiples of 8 elements");
    return ATTN_OK;
}

}  // namespace attn

extern "C" attn_status_t attn_decode_splitkv(const attn_fwd_params_t *p, int32_t num_splits,
                                             void *workspace, size_t workspace_bytes,
                                             attn_stream_t stream) {
    attn_status_t st = check_decode_args(p, num_splits);
    if (st) return st;
    if (p->B * p->H == 0) return ATTN_OK;
    size_t need = attn_decode_workspace_bytes_rows(p->B, p->H, p->Nq, p->dv, num_splits);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need)
        return fail(ATTN_ERR_WORKSPACE, "workspace must be 16-byte aligned and hold %zu bytes (got %zu)",
                    need, workspace_bytes);
    float *part = static_cast<float *>(workspace);
    st = launch_decode_split(*p, num_splits, part, nullptr, reinterpret_cast<cudaStream_t>(stream));
    if (st) return st;
    return launch_merge(part, p->B, p->H, p->Nq, num_splits, p->dv, p->dtype, p->o, p->o_stride, p->lse,
                        reinterpret_cast<cudaStream_t>(stream));
}

// Partial states (as for attn_decode_splitkv, rounded up to 16 bytes), then B * H counters.
static size_t fused_counters_offset(int64_t B, int64_t H, int64_t Nq, int64_t dv, int32_t num_splits) {
    return (attn_decode_workspace_bytes_rows(B, H, Nq, dv, num_splits) + 15) & ~(size_t)15;
}

extern "C" size_t attn_decode_fused_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t dv,
                                                    int32_t num_splits) {
    if (B < 0 || H < 0 || Nq < 1 || dv < 1 || num_splits < 1) return 0;
    return fused_counters_offset(B, H, Nq, dv, num_splits) + (size_t)B * (size_t)H * sizeof(uint64_t);
}

extern "C" attn_status_t attn_decode_splitkv_fused(const attn_fwd_params_t *p, int32_t num_splits,
                                                   void *workspace, size_t workspace_bytes,
                                                   attn_stream_t stream) {
    attn_status_t st = check_decode_args(p, num_splits);
    if (st) return st;
    if (p->B * p->H == 0) return ATTN_OK;
    const size_t need = attn_decode_fused_workspace_bytes(p->B, p->H, p->Nq, p->dv, num_splits);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need)
        return fail(ATTN_ERR_WORKSPACE, "workspace must be 16-byte aligned and hold %zu bytes (got %zu)",
                    need, workspace_bytes);
    float *part = static_cast<float *>(workspace);
    auto *counters = reinterpret_cast<unsigned long long *>(
        static_cast<char *>(workspace) + fused_counters_offset(p->B, p->H, p->Nq, p->dv, num_splits));
    return launch_decode_split(*p, num_splits, part, counters, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" attn_status_t attn_merge_states(const float *partials, int64_t B, int64_t H,
                                           int32_t num_splits, int64_t dv, int32_t o_dtype,
                                           void *o, const int64_t o_stride[3], float *lse,
                                           attn_stream_t stream) {
    g_msg[0] = 0;
    if (B < 0 || H < 0) return fail(ATTN_ERR_INVALID_ARG, "negative B or H");
    if (num_splits < 1 || num_splits > 4096)
        return fail(ATTN_ERR_INVALID_ARG, "num_splits must be in [1, 4096] (got %d)", num_splits);
    if (dv < 1 || dv > 1024) return fail(ATTN_ERR_UNSUPPORTED, "dv must be in [1, 1024]");
    if (o_dtype != ATTN_DTYPE_F32 && o_dtype != ATTN_DTYPE_BF16)
        return fail(ATTN_ERR_INVALID_ARG, "bad o_dtype %d", o_dtype);
    if (B * H == 0) return ATTN_OK;
    if (!partials || !o || !o_stride) return fail(ATTN_ERR_INVALID_ARG, "partials, o or o_stride is NULL");
    for (int i = 0; i < 3; ++i)
        if (o_stride[i] < 0) return fail(ATTN_ERR_INVALID_ARG, "o_stride[%d] is negative", i);
    return launch_merge(partials, B, H, 1, num_splits, dv, o_dtype, o, o_stride, lse,
                        reinterpret_cast<cudaStream_t>(stream));
}

extern "C" attn_status_t attn_fwd_partial(const attn_fwd_params_t *p, int64_t key_offset, int64_t Nk_total,
                                          float *partials, attn_stream_t stream) {
    g_msg[0] = 0;
    if (!p) return fail(ATTN_ERR_INVALID_ARG, "params is NULL");
    attn_fwd_params_t c = *p;  // o is not written: stand partials in for it in the shared checks
    if (!c.o) c.o = partials;
    attn_status_t st = check_common(&c);
    if (st) return st;
    if (p->dtype != ATTN_DTYPE_BF16) return fail(ATTN_ERR_UNSUPPORTED, "partial states support bfloat16 only");
    if (p->dk != p->dv || (p->dk != 64 && p->dk != 128))
        return fail(ATTN_ERR_UNSUPPORTED, "partial states support dk == dv in {64, 128} (dk=%lld dv=%lld)",
                    (long long)p->dk, (long long)p->dv);
    if (has_dropout(p)) return fail(ATTN_ERR_UNSUPPORTED, "partial states take no dropout");
    if (p->block_k != 0) return fail(ATTN_ERR_INVALID_ARG, "block_k must be 0 for bfloat16 (got %d)", p->block_k);
    if (!(p->scale > 0.0f)) return fail(ATTN_ERR_UNSUPPORTED, "bfloat16 path needs scale > 0 (got %g)", p->scale);
    if (key_offset < 0 || Nk_total < key_offset + p->Nk || Nk_total > INT32_MAX)
        return fail(ATTN_ERR_INVALID_ARG,
                    "the shard [key_offset, key_offset + Nk) = [%lld, %lld) must lie in [0, Nk_total = %lld)",
                    (long long)key_offset, (long long)(key_offset + p->Nk), (long long)Nk_total);
    if (p->B * p->H * p->Nq == 0) return ATTN_OK;
    if (!partials || !aligned16(partials)) return fail(ATTN_ERR_MISALIGNED, "partials must be 16-byte aligned");
    if (!aligned16(p->q) || (p->Nk > 0 && (!aligned16(p->k) || !aligned16(p->v))))
        return fail(ATTN_ERR_MISALIGNED, "q, k and v must be 16-byte aligned");
    if (!stride_mult(p->q_stride, 8) || !stride_mult(p->k_stride, 8) || !stride_mult(p->v_stride, 8))
        return fail(ATTN_ERR_MISALIGNED, "bfloat16 strides must be multiples of 8 elements");
    if (p->bias && (reinterpret_cast<uintptr_t>(p->bias) & 3u))
        return fail(ATTN_ERR_MISALIGNED, "bias must be 4-byte aligned");
    return launch_fwd_bf16_partial(*p, key_offset, Nk_total, partials, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" attn_status_t attn_merge_states_rows(const float *partials, int64_t B, int64_t H, int64_t Nq,
                                                int32_t num_splits, int64_t dv, int64_t row_stride,
                                                int64_t split_stride, int32_t o_dtype, void *o,
                                                const int64_t o_stride[3], float *lse, attn_stream_t stream) {
    g_msg[0] = 0;
    if (B < 0 || H < 0 || Nq < 0) return fail(ATTN_ERR_INVALID_ARG, "negative B, H or Nq");
    if (num_splits < 1 || num_splits > 4096)
        return fail(ATTN_ERR_INVALID_ARG, "num_splits must be in [1, 4096] (got %d)", num_splits);
    if (dv < 1 || dv > 1024) return fail(ATTN_ERR_UNSUPPORTED, "dv must be in [1, 1024]");
    if (row_stride < 0 || split_stride < 0) return fail(ATTN_ERR_INVALID_ARG, "negative state stride");
    if (o_dtype != ATTN_DTYPE_F32 && o_dtype != ATTN_DTYPE_BF16)
        return fail(ATTN_ERR_INVALID_ARG, "bad o_dtype %d", o_dtype);
    if (B * H * Nq == 0) return ATTN_OK;
    if (!partials || !o || !o_stride) return fail(ATTN_ERR_INVALID_ARG, "partials, o or o_stride is NULL");
    for (int i = 0; i < 3; ++i)
        if (o_stride[i] < 0) return fail(ATTN_ERR_INVALID_ARG, "o_stride[%d] is negative", i);
    // the zero strides stand for the decode layout inside launch_merge: spell them out here
    const int64_t rs = row_stride ? row_stride : (int64_t)num_splits * (2 + dv);
    const int64_t ss = split_stride ? split_stride : 2 + dv;
    return launch_merge(partials, B, H, Nq, num_splits, dv, o_dtype, o, o_stride, lse,
                        reinterpret_cast<cudaStream_t>(stream), rs, ss);
}

// dQ accumulator [B, Nq, H, dk], c_i [B, H, Nq], and lse * log2 e [B, H, Nq rounded up to 128]
// (whole 128-row tiles of it are copied with one bulk copy each), each 16-byte aligned.
static size_t bwd_ws_parts(int64_t B, int64_t H, int64_t Nq, int64_t dk, size_t *off_c, size_t *off_l) {
    auto up16 = [](size_t x) { return (x + 15) & ~(size_t)15; };
    const size_t acc = (size_t)B * (size_t)H * (size_t)Nq * (size_t)dk * sizeof(float);
    const size_t rows = (size_t)B * (size_t)H * (size_t)Nq * sizeof(float);
    const size_t padded = (size_t)B * (size_t)H * (size_t)((Nq + 127) / 128 * 128) * sizeof(float);
    *off_c = up16(acc);
    *off_l = *off_c + up16(rows);
    return *off_l + padded;
}

extern "C" size_t attn_bwd_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t dk) {
    if (B < 0 || H < 0 || Nq < 0 || dk < 1) return 0;
    size_t oc, ol;
    return bwd_ws_parts(B, H, Nq, dk, &oc, &ol);
}

extern "C" attn_status_t attn_bwd(const attn_bwd_params_t *p, void *workspace, size_t workspace_bytes,
                                  attn_stream_t stream) {
    g_msg[0] = 0;
    if (!p) return fail(ATTN_ERR_INVALID_ARG, "params is NULL");
    const attn_fwd_params_t *f = &p->fwd;
    attn_status_t st = check_common(f);
    if (st) return st;
    if (f->dtype != ATTN_DTYPE_BF16) return fail(ATTN_ERR_UNSUPPORTED, "backward supports bfloat16 only");
    if (has_dropout(f)) {  // the backward of a dropout forward runs on the tcgen05 kernel
        if (f->bias)
            return fail(ATTN_ERR_UNSUPPORTED, "the backward of a dropout forward takes no bias");
        if (f->dropout_mask && (!aligned16(f->dropout_mask) || !stride_mult(f->dropout_mask_stride, 16)))
            return fail(ATTN_ERR_MISALIGNED, "dropout_mask must be 16-byte aligned with strides that are multiples of 16 bytes");
    }
    if (f->dk != f->dv || (f->dk != 64 && f->dk != 128))
        return fail(ATTN_ERR_UNSUPPORTED, "backward supports dk == dv in {64, 128} (dk=%lld dv=%lld)",
                    (long long)f->dk, (long long)f->dv);
    if ((st = check_strides("dout", p->dout_stride)) || (st = check_strides("dq", p->dq_stride)) ||
        (st = check_strides("dk", p->dk_stride)) || (st = check_strides("dv", p->dv_stride)))
        return st;
    if (f->B * f->H * (f->Nq + f->Nk) == 0) return ATTN_OK;
    if (f->Nq > 0 && (!f->lse || !p->dout || !p->dq))
        return fail(ATTN_ERR_INVALID_ARG, "lse, dout and dq are required (lse as the forward wrote it)");
    if (f->Nk > 0 && (!p->dk || !p->dv)) return fail(ATTN_ERR_INVALID_ARG, "dk or dv is NULL");
    if (f->Nk > 0 && f->Nq > 0 && (!f->k || !f->v)) return fail(ATTN_ERR_INVALID_ARG, "k or v is NULL");
    const void *ptrs[] = {f->q, f->k, f->v, f->o, p->dout, p->dq, p->dk, p->dv, f->lse};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return fail(ATTN_ERR_MISALIGNED, "every tensor must be 16-byte aligned");
    if (!stride_mult(f->q_stride, 8) || !stride_mult(f->k_stride, 8) || !stride_mult(f->v_stride, 8) ||
        !stride_mult(f->o_stride, 8) || !stride_mult(p->dout_stride, 8) || !stride_mult(p->dq_stride, 8) ||
        !stride_mult(p->dk_stride, 8) || !stride_mult(p->dv_stride, 8))
        return fail(ATTN_ERR_MISALIGNED, "bfloat16 strides must be multiples of 8 elements");
    if (f->B * f->Nq * f->H * (f->dk / 8) > INT32_MAX)
        return fail(ATTN_ERR_UNSUPPORTED, "backward supports B * Nq * H * dk / 8 < 2^31");
    const size_t need = attn_bwd_workspace_bytes(f->B, f->H, f->Nq, f->dk);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need)
        return fail(ATTN_ERR_WORKSPACE, "workspace must be 16-byte aligned and hold %zu bytes (got %zu)", need,
                    workspace_bytes);
    size_t off_c, off_l;
    bwd_ws_parts(f->B, f->H, f->Nq, f->dk, &off_c, &off_l);
    float *dq_acc = static_cast<float *>(workspace);
    float *crow = reinterpret_cast<float *>(static_cast<char *>(workspace) + off_c);
    float *lrow = reinterpret_cast<float *>(static_cast<char *>(workspace) + off_l);
    return launch_bwd(*p, dq_acc, crow, lrow, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" const char *attn_last_error(void) { return g_msg; }

extern "C" attn_status_t attn_device_error_flags(uint32_t *out, int32_t clear) {
    g_msg[0] = 0;
    if (!out) return fail(ATTN_ERR_INVALID_ARG, "out is NULL");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaDeviceSynchronize: %s", cudaGetErrorString(e));
    e = cudaMemcpyFromSymbol(out, g_device_flags, sizeof(uint32_t));
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "reading the error word: %s", cudaGetErrorString(e));
    if (clear) {
        uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_device_flags, &zero, sizeof(uint32_t));
        if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "clearing the error word: %s", cudaGetErrorString(e));
    }
    return ATTN_OK;
}

extern "C" int32_t attn_version(void) { return 100; }
