// bwd.cu -- attention backward: dQ, dK, dV of a loss through O, for bf16 inputs with fp32
// accumulation.
//
// "How Does FlashAttention Preserve Global Softmax Across Tiles?", section 7: the forward
// keeps each row's log-sum-exp L_i and its output; the backward rebuilds the probabilities
// tile by tile from Q, K, the fixed mask and bias, and L_i (p_ij = exp(x_ij - L_i)), takes the
// softmax Jacobian's row reduction as c_i = g_i . o_i (g_i the upstream gradient of row i),
// forms the gradient of the scaled logits dS_ij = p_ij (g_i . v_j - c_i), accumulates
// dV_j += p_ij g_i, dK_j += scale dS_ij q_i, dQ_i += scale dS_ij k_j, and discards the tile.
// The bias is fixed (no gradient is formed for it); an empty row passes no gradient.
//
// Three kernels on the caller's stream:
//   bwd_prep_kernel   c_i = g_i . o_i per row (fp32, into the workspace), lse_i * log2 e per
//                     row, and a zeroed fp32 dQ accumulator row;
//   bwd_tc_kernel     (bwd_tc_sm103.cu) the five products on the tensor cores, one CTA per
//                     128-key block, for dk == dv in {64, 128}, with or without a bias and
//                     dropout;
//   bwd_dq_kernel     dQ accumulator -> bf16.
// Masking is the forward's: key j of sequence b is visible to row i iff j < n_b, and when
// causal j <= i + n_b - Nq, and the bias there is not -inf.
#include <cmath>
#include <mutex>

#include <cuda_bf16.h>

#include "attn_internal.h"
#include "sm100_ptx.cuh"

namespace attn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct BwdArgs {
    int B, H, Nq, Nk, causal;
    float scale, scale_log2;
    const __nv_bfloat16 *q, *k, *v, *o, *g;
    long long qs0, qs1, qs2, ks0, ks1, ks2, vs0, vs1, vs2, os0, os1, os2, gs0, gs1, gs2;
    const float *lse;  // [B, H, Nq]
    const float *bias;
    long long bs0, bs1, bs2;
    const int *kv_lens;
    float *dq_acc;  // [B, Nq, H, D] fp32
    float *crow;    // [B, H, Nq] fp32: c_i = g_i . o_i
    float *lrow;    // [B, H, Nq rounded up to 128] fp32: lse_i * log2 e
    __nv_bfloat16 *dq, *dk, *dv;
    long long dqs0, dqs1, dqs2, dks0, dks1, dks2, dvs0, dvs1, dvs2;
    uint32_t *flags;
};

// c_i = g_i . o_i and a zeroed dQ accumulator row; D/8 lanes per row (b * Nq + i) * H + h,
// each with 16-byte loads of o and g
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(BwdArgs a) {
    ptx::launch_dependents();  // the products kernel may start its own loads meanwhile
    constexpr int LPR = D / 8;  // lanes per row
    const int rows = a.B * a.Nq * a.H;
    const int row = (blockIdx.x * 256 + threadIdx.x) / LPR, sub = threadIdx.x % LPR;
    const bool live = row < rows;
    float acc = 0.f;
    if (live) {
        const int h = row % a.H, bi = row / a.H, i = bi % a.Nq, b = bi / a.Nq;
        const uint4 ov = *reinterpret_cast<const uint4 *>(a.o + b * a.os0 + (long long)i * a.os1 + h * a.os2 + 8 * sub);
        const uint4 gv = *reinterpret_cast<const uint4 *>(a.g + b * a.gs0 + (long long)i * a.gs1 + h * a.gs2 + 8 * sub);
        const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ow[w]));
            const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&gw[w]));
            acc = fmaf(of.x, gf.x, fmaf(of.y, gf.y, acc));
        }
        float4 *dqa = reinterpret_cast<float4 *>(a.dq_acc + (long long)row * D + 8 * sub);
        dqa[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        dqa[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (live && sub == 0) {
        const int h = row % a.H, bi = row / a.H, i = bi % a.Nq, b = bi / a.Nq;
        a.crow[((long long)b * a.H + h) * a.Nq + i] = acc;
        const int nq_pad = (a.Nq + 127) / 128 * 128;
        a.lrow[((long long)b * a.H + h) * nq_pad + i] = a.lse[((long long)b * a.H + h) * a.Nq + i] * kLog2e;
    }
}

// dQ accumulator (fp32 [B, Nq, H, D]) -> bf16 dQ with the caller's strides; 8 values per
// thread (two 16-byte loads, one 16-byte store)
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_kernel(BwdArgs a) {
    ptx::grid_dep_wait();  // the accumulator is complete once the products kernel is
    const int rows = a.B * a.Nq * a.H;
    const int x = blockIdx.x * 256 + threadIdx.x, row = x / (D / 8), c = 8 * (x % (D / 8));
    if (row >= rows) return;
    const int h = row % a.H, bi = row / a.H, i = bi % a.Nq, b = bi / a.Nq;
    const float4 *src = reinterpret_cast<const float4 *>(a.dq_acc + (long long)row * D + c);
    const float4 f0 = src[0], f1 = src[1];
    *reinterpret_cast<uint4 *>(a.dq + b * a.dqs0 + (long long)i * a.dqs1 + h * a.dqs2 + c) =
        make_uint4(ptx::pack_bf16x2(f0.x, f0.y), ptx::pack_bf16x2(f0.z, f0.w), ptx::pack_bf16x2(f1.x, f1.y),
                   ptx::pack_bf16x2(f1.z, f1.w));
}

// Prep, then the products (the tcgen05 kernel), then the dQ conversion.  A failed tcgen05
// launch reports through attn_last_error and returns cudaErrorLaunchFailure here.
template <int D>
cudaError_t launch_all(const BwdArgs &a, const attn_bwd_params_t &p, cudaStream_t st) {
    const long long rows = (long long)a.B * a.Nq * a.H;
    const unsigned row_blocks = (unsigned)((rows * (D / 8) + 255) / 256);
    if (rows > 0) {
        bwd_prep_kernel<D><<<row_blocks, 256, 0, st>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if ((long long)a.B * a.H * a.Nk > 0 &&
        launch_bwd_tc(p, a.dq_acc, a.crow, a.lrow, st) != ATTN_OK)
        return cudaErrorLaunchFailure;
    if (rows > 0) {
        // launched with programmatic stream serialization: its CTAs may be scheduled while the
        // products kernel drains, and wait there for it to complete
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(row_blocks);
        cfg.blockDim = dim3(256);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, bwd_dq_kernel<D>, a);
    }
    return cudaSuccess;
}

}  // namespace

attn_status_t launch_bwd(const attn_bwd_params_t &p, float *dq_acc, float *crow, float *lrow, cudaStream_t st) {
    const attn_fwd_params_t &f = p.fwd;
    BwdArgs a;
    a.B = (int)f.B; a.H = (int)f.H; a.Nq = (int)f.Nq; a.Nk = (int)f.Nk; a.causal = f.causal;
    a.scale = f.scale; a.scale_log2 = f.scale * kLog2e;
    a.q = static_cast<const __nv_bfloat16 *>(f.q);
    a.k = static_cast<const __nv_bfloat16 *>(f.k);
    a.v = static_cast<const __nv_bfloat16 *>(f.v);
    a.o = static_cast<const __nv_bfloat16 *>(f.o);
    a.g = static_cast<const __nv_bfloat16 *>(p.dout);
    a.qs0 = f.q_stride[0]; a.qs1 = f.q_stride[1]; a.qs2 = f.q_stride[2];
    a.ks0 = f.k_stride[0]; a.ks1 = f.k_stride[1]; a.ks2 = f.k_stride[2];
    a.vs0 = f.v_stride[0]; a.vs1 = f.v_stride[1]; a.vs2 = f.v_stride[2];
    a.os0 = f.o_stride[0]; a.os1 = f.o_stride[1]; a.os2 = f.o_stride[2];
    a.gs0 = p.dout_stride[0]; a.gs1 = p.dout_stride[1]; a.gs2 = p.dout_stride[2];
    a.lse = f.lse;
    a.bias = f.bias; a.bs0 = f.bias_stride[0]; a.bs1 = f.bias_stride[1]; a.bs2 = f.bias_stride[2];
    a.kv_lens = f.kv_lens;
    a.dq_acc = dq_acc; a.crow = crow; a.lrow = lrow;
    a.dq = static_cast<__nv_bfloat16 *>(p.dq);
    a.dk = static_cast<__nv_bfloat16 *>(p.dk);
    a.dv = static_cast<__nv_bfloat16 *>(p.dv);
    a.dqs0 = p.dq_stride[0]; a.dqs1 = p.dq_stride[1]; a.dqs2 = p.dq_stride[2];
    a.dks0 = p.dk_stride[0]; a.dks1 = p.dk_stride[1]; a.dks2 = p.dk_stride[2];
    a.dvs0 = p.dv_stride[0]; a.dvs1 = p.dv_stride[1]; a.dvs2 = p.dv_stride[2];
    a.flags = device_flags();
    if (!a.flags) return fail(ATTN_ERR_CUDA, "could not resolve the device error word");
    if (f.B > 65535 || f.H > 65535) return fail(ATTN_ERR_UNSUPPORTED, "backward supports B, H <= 65535");
    const cudaError_t e = f.dk == 64 ? launch_all<64>(a, p, st) : launch_all<128>(a, p, st);
    if (e == cudaErrorLaunchFailure && attn_last_error()[0]) return ATTN_ERR_CUDA;  // message set by the tcgen05 launcher
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "backward launch: %s", cudaGetErrorString(e));
    return ATTN_OK;
}

}  // namespace attn
