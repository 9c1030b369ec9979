// attn_internal.h -- host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/attn.h"

namespace attn {

// Error bits of the device error word (see attn_device_error_flags).
enum : uint32_t { kFlagWaitTimeout = 1u, kFlagKvLenClamped = 2u };

// Records a message for attn_last_error() and returns `st`.
attn_status_t fail(attn_status_t st, const char *fmt, ...);

// Device address of the device error word of the current device (nullptr on failure).
uint32_t *device_flags();

// Launchers.  Arguments have been validated by the caller (attn_api.cu).
attn_status_t launch_fwd_f32(const attn_fwd_params_t &p, cudaStream_t s);
attn_status_t launch_fwd_bf16(const attn_fwd_params_t &p, cudaStream_t s);
// The forward over one shard of the keys (local key j = global key key_offset + j of Nk_total),
// writing each row's state (m, l, u) to partials [B, H, Nq, 2 + dv] (fwd_bf16_sm103.cu).
attn_status_t launch_fwd_bf16_partial(const attn_fwd_params_t &p, int64_t key_offset, int64_t Nk_total,
                                      float *partials, cudaStream_t s);
// counters: NULL for the split kernel alone (the merge is a second launch); otherwise the
// per-(b, h) arrival counters of the fused merge (any contents on entry).
attn_status_t launch_decode_split(const attn_fwd_params_t &p, int num_splits, float *partials,
                                  unsigned long long *counters, cudaStream_t s);
// State s of row r = (b*H + h)*Nq + i at partials + r*row_stride + s*split_stride (floats);
// zero strides mean the decode layout [B, H, Nq, S, 2 + dv].
attn_status_t launch_merge(const float *partials, int64_t B, int64_t H, int64_t Nq, int num_splits,
                           int64_t dv, int o_dtype, void *o, const int64_t o_stride[3],
                           float *lse, cudaStream_t s, int64_t row_stride = 0, int64_t split_stride = 0);

// Largest number of query rows per sequence the split-KV decode takes.
constexpr int kMaxDecodeRows = 8;

// The argument checks of attn_decode_splitkv that precede its workspace check (clears the
// last error message first).
attn_status_t check_decode_args(const attn_fwd_params_t *p, int32_t num_splits);

attn_status_t launch_bwd(const attn_bwd_params_t &p, float *dq_acc, float *crow, float *lrow, cudaStream_t s);

// 4-D TMA map over a bf16 [B, N, H, d] tensor with element strides s (b, n, h); box 64 x 128,
// 128-byte swizzle (fwd_bf16_sm103.cu).
attn_status_t encode(CUtensorMap *m, const void *ptr, int64_t B, int64_t N, int64_t H, int64_t d,
                     const int64_t s[3], const char *name);

// The backward's products on the tcgen05 tensor cores (bwd_tc_sm103.cu; dk == dv in {64, 128});
// dq_acc, crow and lrow (lse * log2 e, rows padded to a multiple of 128) as for launch_bwd,
// already filled by the prep kernel.
attn_status_t launch_bwd_tc(const attn_bwd_params_t &p, float *dq_acc, const float *crow, const float *lrow,
                            cudaStream_t s);

// Number of SMs of the current device (cached per device).
int sm_count();

// In-kernel dropout draws (dropout_rng = 1): the drop probability quantised to p8 / 256 with
// p8 = round(256 p), at most 255 (see include/attn.h).
inline uint32_t dropout_p8(float p) {
    const double x = (double)p * 256.0 + 0.5;
    const uint32_t q = x <= 0.0 ? 0u : (uint32_t)x;
    return q > 255u ? 255u : q;
}

// Launches kern as a programmatic dependent of the previous kernel in the stream: its CTAs
// may be scheduled once every CTA of that kernel has executed griddepcontrol.launch_dependents
// (or exited), so its launch and set-up overlap that kernel's tail.  A kernel launched this
// way executes griddepcontrol.wait before it reads or writes global memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace attn
