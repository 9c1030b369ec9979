// fwd_f32.cu -- exact float32 attention forward on the SIMT cores.
//
// The float32 operator needs 1e-5 agreement with float64, which TF32 tensor cores cannot
// give, so this path stays on FFMA.  It follows the tile loop of "How Does FlashAttention
// Preserve Global Softmax Across Tiles?", section 5: a CTA keeps a tile of BQ = 16 query
// rows, streams key/value tiles of BK (16, 32 or 64) keys through shared memory, and every
// row keeps its own state (m, l, u) -- the running maximum, the exponential sum against it
// and the unnormalised value sum -- rescaling both l and u by exp(m_old - m_new) when the
// maximum grows and dividing once at the end.  A row whose tile holds no visible key skips
// the update (section 6), and a row with no visible key at all returns o = 0, lse = -inf.
//
// Layout of work: grid (ceil(Nq/16), H, B), 128 threads = 4 warps, 4 query rows per warp.
// For a row, lane t scores keys t and t + 32 of the tile; warp shuffles give the tile
// maximum and the tile's exponential sum; the value update gives each lane dv/32 columns.
#include <cfloat>
#include <cmath>

#include "attn_internal.h"
#include "dropout_rng.cuh"

namespace attn {
namespace {

constexpr int kBQ = 16;
constexpr int kThreads = 128;
constexpr int kRowsPerWarp = kBQ / (kThreads / 32);
constexpr int kMaxD = 256;

struct F32Args {
    int B, H, Nq, Nk, dk, dv, causal;
    float scale;
    const float *q, *k, *v;
    float *o, *lse;
    long long qs0, qs1, qs2, ks0, ks1, ks2, vs0, vs1, vs2, os0, os1, os2;
    const float *bias;
    long long bs0, bs1, bs2;
    const int *kv_lens;
    uint32_t *flags;
    const uint8_t *dmask;  // dropout keep bits (bit j % 8 of byte j / 8 of a row), or null
    long long dms0, dms1, dms2;
    float inv_keep;        // 1 / (1 - dropout_p), the realised p for in-kernel draws
    int rng;               // keep decisions drawn in-kernel (dropout_rng.cuh)
    uint32_t seed_lo, seed_hi, offset, p8x4;
};

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <int BK>
__global__ void __launch_bounds__(kThreads) fwd_f32_kernel(F32Args a) {
    extern __shared__ float smem[];
    const int dk = a.dk, dv = a.dv, ldk = dk + 1;
    float *Qs = smem;                    // [kBQ][dk]
    float *Ks = Qs + kBQ * dk;           // [BK][dk + 1]  (padded: lanes read distinct banks)
    float *Vs = Ks + BK * ldk;           // [BK][dv]
    float *Ps = Vs + BK * dv;            // [4 warps][BK]

    const int b = blockIdx.z, h = blockIdx.y, q0 = blockIdx.x * kBQ;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    int n = a.Nk;  // this sequence's key length, clamped to [0, Nk]
    if (a.kv_lens) {
        int raw = a.kv_lens[b];
        n = min(max(raw, 0), a.Nk);
        if (raw != n && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
            atomicOr(a.flags, kFlagKvLenClamped);
    }
    const int shift = n - a.Nq;  // bottom-right causal: key j visible to row i iff j <= i + shift

    for (int t = threadIdx.x; t < kBQ * dk; t += kThreads) {
        int r = t / dk, c = t % dk;
        int i = q0 + r;
        Qs[t] = i < a.Nq ? a.q[b * a.qs0 + (long long)i * a.qs1 + h * a.qs2 + c] : 0.f;
    }

    // keys this CTA can see at all: [0, kv_end)
    int kv_end = n;
    if (a.causal) kv_end = min(n, max(0, min(q0 + kBQ, a.Nq) - 1 + shift + 1));

    constexpr int kCols = kMaxD / 32;
    float acc[kRowsPerWarp][kCols];
    float m_run[kRowsPerWarp], l_run[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        m_run[r] = -INFINITY;
        l_run[r] = 0.f;
#pragma unroll
        for (int c = 0; c < kCols; ++c) acc[r][c] = 0.f;
    }

    for (int j0 = 0; j0 < kv_end; j0 += BK) {
        __syncthreads();  // previous tile fully consumed
        for (int t = threadIdx.x; t < BK * dk; t += kThreads) {
            int jj = t / dk, c = t % dk, j = j0 + jj;
            Ks[jj * ldk + c] = j < kv_end ? a.k[b * a.ks0 + (long long)j * a.ks1 + h * a.ks2 + c] : 0.f;
        }
        for (int t = threadIdx.x; t < BK * dv; t += kThreads) {
            int jj = t / dv, c = t % dv, j = j0 + jj;
            Vs[t] = j < kv_end ? a.v[b * a.vs0 + (long long)j * a.vs1 + h * a.vs2 + c] : 0.f;
        }
        __syncthreads();

#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const int rr = warp * kRowsPerWarp + r, i = q0 + rr;
            if (i >= a.Nq) continue;  // warp-uniform
            // logits of this lane's keys (masked ones are -inf and never read further)
            float x[BK / 32 > 0 ? BK / 32 : 1];
            bool vis[BK / 32 > 0 ? BK / 32 : 1];
            float tmax = -INFINITY;
#pragma unroll
            for (int u = 0; u < (BK + 31) / 32; ++u) {
                const int jj = lane + 32 * u, j = j0 + jj;
                bool ok = jj < BK && j < n && (!a.causal || j <= i + shift);
                float s = -INFINITY;
                if (ok) {
                    float dot = 0.f;
                    for (int c = 0; c < dk; ++c) dot = fmaf(Qs[rr * dk + c], Ks[jj * ldk + c], dot);
                    s = a.scale * dot;
                    if (a.bias) {
                        float bj = a.bias[b * a.bs0 + h * a.bs1 + (long long)i * a.bs2 + j];
                        if (bj == -INFINITY) ok = false;
                        else s += bj;
                    }
                    if (!ok) s = -INFINITY;
                }
                x[u] = s;
                vis[u] = ok;
                tmax = fmaxf(tmax, s);
            }
            tmax = warp_max(tmax);
            if (tmax == -INFINITY) continue;  // no visible key of this tile: state unchanged
            float m_new, alpha;
            if (m_run[r] == -INFINITY) {  // first update: the old state has no mass
                m_new = tmax;
                alpha = 0.f;
            } else {
                m_new = fmaxf(m_run[r], tmax);
                alpha = expf(m_run[r] - m_new);
            }
            float psum = 0.f;
#pragma unroll
            for (int u = 0; u < (BK + 31) / 32; ++u) {
                const int jj = lane + 32 * u;
                float p = vis[u] ? expf(x[u] - m_new) : 0.f;
                psum += p;  // the row sum keeps the undropped weight
                if (a.dmask && vis[u]) {  // dropout: kept weights scaled, dropped ones 0 in o
                    const int j = j0 + jj;
                    const uint8_t bits = a.dmask[b * a.dms0 + h * a.dms1 + (long long)i * a.dms2 + (j >> 3)];
                    p = ((bits >> (j & 7)) & 1u) ? p * a.inv_keep : 0.f;
                } else if (a.rng && vis[u]) {  // the same, drawn in-kernel (one draw per 16 keys)
                    const int j = j0 + jj;
                    const uint32_t bits = rng::keep16((uint32_t)i, (uint32_t)(j >> 4), (uint32_t)(b * a.H + h), a.offset,
                                                      a.seed_lo, a.seed_hi, a.p8x4);
                    p = ((bits >> (j & 15)) & 1u) ? p * a.inv_keep : 0.f;
                }
                if (jj < BK) Ps[warp * BK + jj] = p;
            }
            psum = warp_sum(psum);
            l_run[r] = alpha * l_run[r] + psum;
            m_run[r] = m_new;
            __syncwarp();
#pragma unroll
            for (int cc = 0; cc < kCols; ++cc) {
                const int c = lane + 32 * cc;
                if (c < dv) {
                    float s = alpha * acc[r][cc];
                    for (int jj = 0; jj < BK; ++jj) s = fmaf(Ps[warp * BK + jj], Vs[jj * dv + c], s);
                    acc[r][cc] = s;
                }
            }
            __syncwarp();
        }
    }

    // divide once; empty rows give +0.0 and lse = -inf
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int i = q0 + warp * kRowsPerWarp + r;
        if (i >= a.Nq) continue;
        const bool empty = !(l_run[r] > 0.f);
        const float inv = empty ? 0.f : 1.f / l_run[r];
        float *orow = a.o + b * a.os0 + (long long)i * a.os1 + h * a.os2;
#pragma unroll
        for (int cc = 0; cc < kCols; ++cc) {
            const int c = lane + 32 * cc;
            if (c < dv) orow[c] = empty ? 0.f : acc[r][cc] * inv;
        }
        if (a.lse && lane == 0)
            a.lse[((long long)b * a.H + h) * a.Nq + i] = empty ? -INFINITY : m_run[r] + logf(l_run[r]);
    }
}

template <int BK>
attn_status_t launch_bk(const F32Args &a, dim3 grid, cudaStream_t s) {
    size_t smem = sizeof(float) * ((size_t)kBQ * a.dk + (size_t)BK * (a.dk + 1) + (size_t)BK * a.dv +
                                   (size_t)(kThreads / 32) * BK);
    cudaError_t e = cudaFuncSetAttribute(fwd_f32_kernel<BK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    fwd_f32_kernel<BK><<<grid, kThreads, smem, s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "fwd_f32 launch: %s", cudaGetErrorString(e));
    return ATTN_OK;
}

}  // namespace

attn_status_t launch_fwd_f32(const attn_fwd_params_t &p, cudaStream_t s) {
    F32Args a;
    a.B = (int)p.B; a.H = (int)p.H; a.Nq = (int)p.Nq; a.Nk = (int)p.Nk;
    a.dk = (int)p.dk; a.dv = (int)p.dv; a.causal = p.causal; a.scale = p.scale;
    a.q = static_cast<const float *>(p.q); a.k = static_cast<const float *>(p.k);
    a.v = static_cast<const float *>(p.v); a.o = static_cast<float *>(p.o); a.lse = p.lse;
    a.qs0 = p.q_stride[0]; a.qs1 = p.q_stride[1]; a.qs2 = p.q_stride[2];
    a.ks0 = p.k_stride[0]; a.ks1 = p.k_stride[1]; a.ks2 = p.k_stride[2];
    a.vs0 = p.v_stride[0]; a.vs1 = p.v_stride[1]; a.vs2 = p.v_stride[2];
    a.os0 = p.o_stride[0]; a.os1 = p.o_stride[1]; a.os2 = p.o_stride[2];
    a.bias = p.bias;
    a.bs0 = p.bias_stride[0]; a.bs1 = p.bias_stride[1]; a.bs2 = p.bias_stride[2];
    a.kv_lens = p.kv_lens;
    a.dmask = p.dropout_mask;
    a.dms0 = p.dropout_mask_stride[0]; a.dms1 = p.dropout_mask_stride[1]; a.dms2 = p.dropout_mask_stride[2];
    a.rng = p.dropout_rng == 1;
    const uint32_t p8 = dropout_p8(p.dropout_p);
    a.seed_lo = (uint32_t)(p.dropout_seed & 0xffffffffu);
    a.seed_hi = (uint32_t)(p.dropout_seed >> 32);
    a.offset = (uint32_t)(p.dropout_offset & 0xffffffffu);
    a.p8x4 = p8 * 0x01010101u;
    a.inv_keep = a.rng ? (float)(256.0 / (256.0 - (double)p8))
                       : p.dropout_mask ? (float)(1.0 / (1.0 - (double)p.dropout_p)) : 1.f;
    a.flags = device_flags();
    if (!a.flags) return fail(ATTN_ERR_CUDA, "could not resolve the device error word");
    if (p.B > 65535 || p.H > 65535)
        return fail(ATTN_ERR_UNSUPPORTED, "float32 path supports B, H <= 65535");
    dim3 grid((unsigned)((p.Nq + kBQ - 1) / kBQ), (unsigned)p.H, (unsigned)p.B);
    switch (p.block_k) {
        case 16: return launch_bk<16>(a, grid, s);
        case 32: return launch_bk<32>(a, grid, s);
        default: return launch_bk<64>(a, grid, s);
    }
}

}  // namespace attn
