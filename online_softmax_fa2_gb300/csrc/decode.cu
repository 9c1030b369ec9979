// decode.cu -- split-KV decode and the merge of partial (m, l, u) states.
//
// "How Does FlashAttention Preserve Global Softmax Across Tiles?", section 8: decode has one
// query row against a long key/value cache, so the work is reading the cache.  The keys of
// each sequence are split into S contiguous ranges; each range gives a partial state
// (m, l, u) (section 3), and the partial states are merged by putting both maxima into the
// common maximum and scaling l and u of each part by exp(m_s - m) before adding (section 3;
// "Flash attention and efficient attention: Visual walkthrough", Step 5).  Empty parts are
// skipped; a row whose parts are all empty gives o = +0.0, lse = -inf (section 6).
//
// Split kernel: grid (S, H, B), 128 threads.  The cache is read once, with 16-byte loads:
// a group of D/8 lanes holds one key row (each lane 8 bf16 of K and 8 of V), so a warp
// reads 32/(D/8) key rows per load instruction, coalesced.  Each group runs the online
// update over its keys (key lo + g + t*G of the split for t = 0, 1, ..., G groups per CTA,
// 4 keys in flight per group), with the logits kept in base-2 units (x * log2 e) so that one ex2
// gives each exponential.  The G group states are then merged in shared memory and the
// split's state is written in natural-log units.
#include <cmath>
#include <mutex>

#include <cuda_bf16.h>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct DecArgs {
    int B, H, Nk, S, Nq, causal;
    float scale_log2;
    const __nv_bfloat16 *q, *k, *v;
    long long qs0, qs1, qs2, ks0, ks1, ks2, vs0, vs1, vs2;
    const float *bias;
    long long bs0, bs1, bs2;
    const int *kv_lens;
    float *part;  // [B, H, Nq, S, 2 + D]
    uint32_t *flags;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float f[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        f[2 * t] = __uint_as_float(w[t] << 16);
        f[2 * t + 1] = __uint_as_float(w[t] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// R: query rows handled per CTA (Nq <= R; rows Nq..R-1 are padding and do nothing).  Every
// key row is read once for all R query rows.
template <int D, int R>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(DecArgs a) {
    constexpr int LPK = D / 8;            // lanes per key row
    constexpr int G = kThreads / LPK;     // key groups per CTA
    constexpr int U = R <= 2 ? 4 : 2;     // keys in flight per group
    __shared__ float sm_m[R][G], sm_l[R][G];
    __shared__ float sm_u[R][G][D + 1];

    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int g = threadIdx.x / LPK, sub = threadIdx.x % LPK, c0 = sub * 8;
    const int nq = a.Nq;

    int n = a.Nk;
    if (a.kv_lens) {
        int raw = a.kv_lens[b];
        n = min(max(raw, 0), a.Nk);
        if (raw != n && threadIdx.x == 0 && s == 0 && h == 0) atomicOr(a.flags, kFlagKvLenClamped);
    }
    const int lo = (int)(((long long)s * n) / a.S), hi = (int)(((long long)(s + 1) * n) / a.S);

    // row r sees keys j < vis[r]: j < n, and, when causal, j <= r + n - Nq (the sequences'
    // ends aligned, "bottom-right"); a row with vis <= 0 sees no key
    int vis[R];
    float qf[R][8];
    const float *bias_row[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        vis[r] = r < nq ? (a.causal ? min(n, max(0, r + n - nq + 1)) : n) : 0;
        bias_row[r] = (a.bias && r < nq) ? a.bias + b * a.bs0 + h * a.bs1 + r * a.bs2 : nullptr;
        if (r < nq) {
            bf16x8_to_f32(*reinterpret_cast<const uint4 *>(a.q + b * a.qs0 + r * a.qs1 + h * a.qs2 + c0), qf[r]);
#pragma unroll
            for (int t = 0; t < 8; ++t) qf[r][t] *= a.scale_log2;
        } else {
#pragma unroll
            for (int t = 0; t < 8; ++t) qf[r][t] = 0.f;
        }
    }

    const __nv_bfloat16 *kb = a.k + b * a.ks0 + h * a.ks2 + c0;
    const __nv_bfloat16 *vb = a.v + b * a.vs0 + h * a.vs2 + c0;

    float m[R], l[R], u[R][8];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int t = 0; t < 8; ++t) u[r][t] = 0.f;
    }

    // Every thread runs the same iterations (the shuffles below need the whole warp);
    // key base + w*G + g belongs to group g.
    for (int base = lo; base < hi; base += G * U) {
        uint4 kr[U], vr[U];
#pragma unroll
        for (int w = 0; w < U; ++w) {
            const int j = base + w * G + g;
            kr[w] = make_uint4(0u, 0u, 0u, 0u);
            vr[w] = kr[w];
            if (j < hi) {
                kr[w] = ld_stream(kb + (long long)j * a.ks1);
                vr[w] = ld_stream(vb + (long long)j * a.vs1);
            }
        }
        float x[R][U];
#pragma unroll
        for (int w = 0; w < U; ++w) {
            float kf[8];
            bf16x8_to_f32(kr[w], kf);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float d = 0.f;
#pragma unroll
                for (int t = 0; t < 8; ++t) d = fmaf(qf[r][t], kf[t], d);
                x[r][w] = d;
            }
        }
#pragma unroll
        for (int w = 0; w < U; ++w) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
#pragma unroll
                for (int o = LPK / 2; o > 0; o >>= 1) x[r][w] += __shfl_xor_sync(0xffffffffu, x[r][w], o);
            }
        }
#pragma unroll
        for (int w = 0; w < U; ++w) {
            const int j = base + w * G + g;
            if (j >= hi) break;  // uniform across the group
            float vf[8];
            bf16x8_to_f32(vr[w], vf);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (j >= vis[r]) continue;  // masked (or a padding row); uniform across the group
                float xs = x[r][w];
                if (bias_row[r]) {
                    const float bj = bias_row[r][j];
                    if (bj == -INFINITY) continue;  // masked key
                    xs = fmaf(bj, kLog2e, xs);
                }
                const float m_new = fmaxf(m[r], xs);
                const float alpha = (m[r] == -INFINITY) ? 0.f : ex2(m[r] - m_new);
                const float p = ex2(xs - m_new);
                l[r] = fmaf(alpha, l[r], p);
#pragma unroll
                for (int t = 0; t < 8; ++t) u[r][t] = fmaf(alpha, u[r][t], p * vf[t]);
                m[r] = m_new;
            }
        }
    }

#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (sub == 0) {
            sm_m[r][g] = m[r];
            sm_l[r][g] = l[r];
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) sm_u[r][g][c0 + t] = u[r][t];
    }
    __syncthreads();

    // merge the G group states of each row; thread c owns column c
    for (int r = 0; r < nq; ++r) {
        float M = -INFINITY;
#pragma unroll
        for (int gg = 0; gg < G; ++gg)
            if (sm_l[r][gg] > 0.f) M = fmaxf(M, sm_m[r][gg]);
        float *out = a.part + ((((long long)b * a.H + h) * nq + r) * a.S + s) * (2 + D);
        if (M == -INFINITY) {  // empty split
            for (int c = threadIdx.x; c < D; c += kThreads) out[2 + c] = 0.f;
            if (threadIdx.x == 0) {
                out[0] = -INFINITY;
                out[1] = 0.f;
            }
            continue;
        }
        float L = 0.f;
#pragma unroll
        for (int gg = 0; gg < G; ++gg)
            if (sm_l[r][gg] > 0.f) L = fmaf(ex2(sm_m[r][gg] - M), sm_l[r][gg], L);
        for (int c = threadIdx.x; c < D; c += kThreads) {
            float acc = 0.f;
#pragma unroll
            for (int gg = 0; gg < G; ++gg)
                if (sm_l[r][gg] > 0.f) acc = fmaf(ex2(sm_m[r][gg] - M), sm_u[r][gg][c], acc);
            out[2 + c] = acc;
        }
        if (threadIdx.x == 0) {
            out[0] = M * kLn2;  // back to natural-log units: exp(x - m) == 2^(x*log2e - M)
            out[1] = L;
        }
    }
}

// Merge: one CTA per (b, h, query row i) -- partial-state row (b*H + h)*Nq + i; thread t owns
// columns t, t + 128, ...
template <typename OutT>
__global__ void __launch_bounds__(kThreads) merge_kernel(const float *part, int H, int Nq, int S, int dv,
                                                           OutT *o, long long os0, long long os1,
                                                           long long os2, float *lse) {
    const long long row = blockIdx.x;
    const int i = (int)(row % Nq), bh = (int)(row / Nq), b = bh / H, h = bh % H;
    const float *st = part + row * S * (2 + dv);
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) {
        const float l = st[s * (2 + dv) + 1];
        if (l > 0.f) M = fmaxf(M, st[s * (2 + dv)]);
    }
    OutT *orow = o + b * os0 + i * os1 + h * os2;
    if (M == -INFINITY) {
        for (int c = threadIdx.x; c < dv; c += blockDim.x) orow[c] = OutT(0.f);
        if (lse && threadIdx.x == 0) lse[row] = -INFINITY;
        return;
    }
    float L = 0.f;
    for (int s = 0; s < S; ++s) {
        const float l = st[s * (2 + dv) + 1];
        if (l > 0.f) L = fmaf(expf(st[s * (2 + dv)] - M), l, L);
    }
    const float inv = 1.f / L;
    for (int c = threadIdx.x; c < dv; c += blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s < S; ++s) {
            const float *x = st + s * (2 + dv);
            if (x[1] > 0.f) acc = fmaf(expf(x[0] - M), x[2 + c], acc);
        }
        orow[c] = OutT(acc * inv);
    }
    if (lse && threadIdx.x == 0) lse[row] = M + logf(L);
}

}  // namespace

attn_status_t launch_decode_split(const attn_fwd_params_t &p, int num_splits, float *partials,
                                  cudaStream_t st) {
    DecArgs a;
    a.B = (int)p.B; a.H = (int)p.H; a.Nk = (int)p.Nk; a.S = num_splits;
    a.Nq = (int)p.Nq; a.causal = p.causal;
    a.scale_log2 = p.scale * kLog2e;
    a.q = static_cast<const __nv_bfloat16 *>(p.q);
    a.k = static_cast<const __nv_bfloat16 *>(p.k);
    a.v = static_cast<const __nv_bfloat16 *>(p.v);
    a.qs0 = p.q_stride[0]; a.qs1 = p.q_stride[1]; a.qs2 = p.q_stride[2];
    a.ks0 = p.k_stride[0]; a.ks1 = p.k_stride[1]; a.ks2 = p.k_stride[2];
    a.vs0 = p.v_stride[0]; a.vs1 = p.v_stride[1]; a.vs2 = p.v_stride[2];
    a.bias = p.bias; a.bs0 = p.bias_stride[0]; a.bs1 = p.bias_stride[1]; a.bs2 = p.bias_stride[2];
    a.kv_lens = p.kv_lens; a.part = partials;
    a.flags = device_flags();
    if (!a.flags) return fail(ATTN_ERR_CUDA, "could not resolve the device error word");
    if (p.B > 65535 || p.H > 65535) return fail(ATTN_ERR_UNSUPPORTED, "decode supports B, H <= 65535");
    if (p.Nq < 1 || p.Nq > kMaxDecodeRows)
        return fail(ATTN_ERR_UNSUPPORTED, "decode supports 1 <= Nq <= %d (got %lld)", kMaxDecodeRows,
                    (long long)p.Nq);
    dim3 grid((unsigned)num_splits, (unsigned)p.H, (unsigned)p.B);
#define ATTN_DECODE_LAUNCH(D_)                                                                 \
    if (p.Nq == 1) decode_split_kernel<D_, 1><<<grid, kThreads, 0, st>>>(a);                 \
    else if (p.Nq == 2) decode_split_kernel<D_, 2><<<grid, kThreads, 0, st>>>(a);            \
    else if (p.Nq <= 4) decode_split_kernel<D_, 4><<<grid, kThreads, 0, st>>>(a);            \
    else decode_split_kernel<D_, 8><<<grid, kThreads, 0, st>>>(a);
    if (p.dk == 64) {
        ATTN_DECODE_LAUNCH(64)
    } else {
        ATTN_DECODE_LAUNCH(128)
    }
#undef ATTN_DECODE_LAUNCH
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "decode split launch: %s", cudaGetErrorString(e));
    return ATTN_OK;
}

attn_status_t launch_merge(const float *partials, int64_t B, int64_t H, int64_t Nq, int num_splits,
                           int64_t dv, int o_dtype, void *o, const int64_t o_stride[3], float *lse,
                           cudaStream_t st) {
    if (B * H * Nq > 0x7fffffffLL) return fail(ATTN_ERR_UNSUPPORTED, "B*H*Nq too large");
    dim3 grid((unsigned)(B * H * Nq));
    if (o_dtype == ATTN_DTYPE_BF16)
        merge_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(partials, (int)H, (int)Nq, num_splits, (int)dv,
                                                               static_cast<__nv_bfloat16 *>(o), o_stride[0],
                                                               o_stride[1], o_stride[2], lse);
    else
        merge_kernel<float><<<grid, kThreads, 0, st>>>(partials, (int)H, (int)Nq, num_splits, (int)dv,
                                                       static_cast<float *>(o), o_stride[0], o_stride[1],
                                                       o_stride[2], lse);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "merge launch: %s", cudaGetErrorString(e));
    return ATTN_OK;
}

}  // namespace attn

// ---------------------------------------------------------------------------------------
// Allocation-free decode.
//
// Some callers cannot allocate device memory at the moment they decode: a host framework
// whose caching allocator already owns the device memory and forbids side allocations, a
// plugin that is handed only its input and output buffers, or a latency-bound serving loop
// in which cudaMalloc/cudaFree would synchronise the device.  For them the split kernel's
// partial states live in one statically allocated device array of this file, sized for up to
// kNoAllocScratchBytes; every device that loads the library holds this array until the
// process exits.  The kernels, the arguments checks and the results are those of
// attn_decode_splitkv: this entry point only supplies the workspace.
namespace attn {
namespace {

constexpr size_t kNoAllocScratchBytes = 32u << 20;  // 32 MiB of partial states

static __device__ __align__(256) float g_decode_scratch[kNoAllocScratchBytes / sizeof(float)];

// Host code cannot use g_decode_scratch's name as a device address, so the address is looked
// up once per device (with that device current) and cached.
void *g_scratch_addr[64];
std::mutex g_scratch_mutex;

attn_status_t noalloc_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(ATTN_ERR_UNSUPPORTED, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
        if (e != cudaSuccess)
            return fail(ATTN_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return ATTN_OK;
}

}  // namespace
}  // namespace attn

extern "C" attn_status_t attn_decode_splitkv_noalloc(const attn_fwd_params_t *p, int32_t num_splits,
                                                     attn_stream_t stream) {
    using namespace attn;
    if (p && num_splits >= 1) {
        const size_t need = attn_decode_workspace_bytes_rows(p->B, p->H, p->Nq, p->dv, num_splits);
        if (need > kNoAllocScratchBytes)
            return fail(ATTN_ERR_WORKSPACE,
                        "allocation-free decode needs %zu bytes of partial states for B=%lld H=%lld "
                        "Nq=%lld dv=%lld num_splits=%d; its built-in scratch holds %zu",
                        need, (long long)p->B, (long long)p->H, (long long)p->Nq, (long long)p->dv, num_splits,
                        kNoAllocScratchBytes);
    }
    void *scratch = nullptr;
    attn_status_t st = noalloc_scratch(&scratch);
    if (st) return st;
    return attn_decode_splitkv(p, num_splits, scratch, kNoAllocScratchBytes, stream);
}
