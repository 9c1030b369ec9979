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
// Three kernels on the caller's stream (with dk == dv == 128 and no bias the products run in
// bwd_tc_sm103.cu's tcgen05 kernel instead of bwd_main_kernel):
//   bwd_prep_kernel   c_i = g_i . o_i per row (fp32, into the workspace) and a zeroed fp32 dQ
//                     accumulator row;
//   bwd_main_kernel   one CTA per (64-key block, h, b), four warps, warp w owning keys
//                     16w..16w+15 of the block.  Query tiles of 32 rows stream through
//                     shared memory (Q, the upstream gradient G, L and c; double-buffered
//                     cp.async copies, rows padded so that ldmatrix is free of bank
//                     conflicts).  Per tile, on the tensor cores (mma.sync m16n8k16, bf16 in,
//                     fp32 accumulate):
//                       S^T = K_w Q^T and dP^T = V_w G^T           (16 keys x 32 rows)
//                       P^T, dS^T elementwise in registers (mask, bias, L, c)
//                       dV_w += P^T G and dK_w += dS^T Q            (P^T and dS^T are the
//                                        accumulator fragments of S^T and dP^T, reused as A)
//                       dS^T -> shared memory; dQ (32 rows x d/4 of the head dimension per
//                       warp) = dS K over the block's 64 keys, added to the fp32
//                       accumulator with vector reductions;
//                     dK (times scale) and dV of the block's keys are written once at the end;
//   bwd_dq_kernel     dQ accumulator -> bf16.
// Masking is the forward's: key j of sequence b is visible to row i iff j < n_b, and when
// causal j <= i + n_b - Nq, and the bias there is not -inf.  Keys past n_b are zero-filled in
// shared memory, so nothing stored there reaches a product.
#include <cmath>
#include <mutex>

#include <cuda_bf16.h>

#include "attn_internal.h"
#include "sm100_ptx.cuh"
#include "warp_mma.cuh"

namespace attn {
namespace {

using namespace wmma16;

constexpr int kBwdThreads = 128;
constexpr int kKB = 64;  // keys per CTA, 16 per warp
constexpr int kQT = 32;  // query rows per tile
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

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ int seq_n(const BwdArgs &a, int b, bool report) {
    if (!a.kv_lens) return a.Nk;
    const int raw = a.kv_lens[b];
    const int n = min(max(raw, 0), a.Nk);
    if (raw != n && report) atomicOr(a.flags, kFlagKvLenClamped);
    return n;
}

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

template <int D>
struct BwdLayout {
    static constexpr int kRB = 2 * D + 16;     // padded bf16 row of K, V, Q or G (bytes)
    static constexpr int kKVBytes = kKB * kRB;  // the K (or V) block
    static constexpr int kTBytes = kQT * kRB;   // one Q (or G) tile
    static constexpr int kSB = 2 * kQT + 16;    // padded row of dS^T: 32 rows bf16 (bytes)
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kKVBytes;
    static constexpr int kOffQ = 2 * kKVBytes;         // two stages
    static constexpr int kOffG = kOffQ + 2 * kTBytes;  // two stages
    static constexpr int kOffL = kOffG + 2 * kTBytes;  // L, two stages of kQT floats
    static constexpr int kOffC = kOffL + 2 * kQT * 4;  // c, likewise
    static constexpr int kOffS = kOffC + 2 * kQT * 4;  // dS^T [kKB keys][kQT rows]
    static constexpr int kBytes = kOffS + kKB * kSB;
};

template <int D, bool kBias>
__global__ void __launch_bounds__(kBwdThreads) bwd_main_kernel(BwdArgs a) {
    using L = BwdLayout<D>;
    constexpr int NK = D / 16;   // 16-wide steps of the head dimension
    constexpr int ND = D / 8;    // 8-wide tiles of the head dimension
    constexpr int NQ = D / 32;   // 8-wide tiles of dQ per warp (a quarter of the head dimension)
    extern __shared__ __align__(128) uint8_t sm[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int mi = lane >> 3, r8 = lane & 7;  // ldmatrix: the matrix and row this lane addresses
    const int kb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int n = seq_n(a, b, threadIdx.x == 0 && kb == 0 && h == 0);
    const int shift = n - a.Nq;  // causal: key j visible to row i iff j <= i + shift
    const int j0 = kb * kKB, jw = j0 + 16 * warp;
    // query tiles holding a row that sees a key of this block
    const int i_first = a.causal ? max(0, j0 - shift) : 0;
    const bool any = j0 < n && i_first < a.Nq;
    const int t_first = i_first / kQT, t_end = any ? (a.Nq + kQT - 1) / kQT : t_first;

    float dk_acc[ND][4], dv_acc[ND][4];
#pragma unroll
    for (int nd = 0; nd < ND; ++nd)
#pragma unroll
        for (int e = 0; e < 4; ++e) dk_acc[nd][e] = dv_acc[nd][e] = 0.f;

    if (t_first < t_end) {
        const __nv_bfloat16 *kg = a.k + b * a.ks0 + h * a.ks2, *vg = a.v + b * a.vs0 + h * a.vs2;
        const __nv_bfloat16 *qg = a.q + b * a.qs0 + h * a.qs2, *gg = a.g + b * a.gs0 + h * a.gs2;
        const float *lg = a.lse + ((long long)b * a.H + h) * a.Nq, *cg = a.crow + ((long long)b * a.H + h) * a.Nq;
        // the K and V block (keys >= n zero-filled); they join the first tile's copy group
        for (int c = threadIdx.x; c < kKB * (D / 8); c += kBwdThreads) {
            const int key = c / (D / 8), ch = c % (D / 8), j = j0 + key;
            const bool in = j < n;
            const long long jj = in ? j : j0;  // j0 < n here: a valid row even when nothing is copied
            cp_async16(smem_addr(sm + L::kOffK + key * L::kRB + ch * 16), kg + jj * a.ks1 + ch * 8, in ? 16u : 0u);
            cp_async16(smem_addr(sm + L::kOffV + key * L::kRB + ch * 16), vg + jj * a.vs1 + ch * 8, in ? 16u : 0u);
        }
        auto issue_tile = [&](int tt, int st) {
            const int i0 = tt * kQT;
            for (int c = threadIdx.x; c < kQT * (D / 8); c += kBwdThreads) {
                const int row = c / (D / 8), ch = c % (D / 8), i = i0 + row;
                const bool in = i < a.Nq;
                const long long ii = in ? i : i0;
                cp_async16(smem_addr(sm + L::kOffQ + st * L::kTBytes + row * L::kRB + ch * 16), qg + ii * a.qs1 + ch * 8,
                           in ? 16u : 0u);
                cp_async16(smem_addr(sm + L::kOffG + st * L::kTBytes + row * L::kRB + ch * 16), gg + ii * a.gs1 + ch * 8,
                           in ? 16u : 0u);
            }
            if (threadIdx.x < kQT) {
                const int i = i0 + threadIdx.x;
                const bool in = i < a.Nq;
                const long long ii = in ? i : i0;
                cp_async4(smem_addr(sm + L::kOffL + (st * kQT + threadIdx.x) * 4), lg + ii, in ? 4u : 0u);
                cp_async4(smem_addr(sm + L::kOffC + (st * kQT + threadIdx.x) * 4), cg + ii, in ? 4u : 0u);
            }
            cp_async_commit();
        };
        issue_tile(t_first, 0);
        int st = 0;
        for (int tt = t_first; tt < t_end; ++tt, st ^= 1) {
            if (tt + 1 < t_end) issue_tile(tt + 1, st ^ 1);
            else cp_async_commit();
            cp_async_wait<1>();
            __syncthreads();
            const uint32_t sK = smem_addr(sm + L::kOffK), sV = smem_addr(sm + L::kOffV);
            const uint32_t sQ = smem_addr(sm + L::kOffQ + st * L::kTBytes);
            const uint32_t sG = smem_addr(sm + L::kOffG + st * L::kTBytes);
            const float *sL = reinterpret_cast<const float *>(sm + L::kOffL) + st * kQT;
            const float *sC = reinterpret_cast<const float *>(sm + L::kOffC) + st * kQT;
            const int i0 = tt * kQT;

            // S^T = K_w Q^T and dP^T = V_w G^T: 16 keys x 32 rows, four 8-row tiles each
            float sc[4][4], dp[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[nt][e] = dp[nt][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < NK; ++kk) {
                // A (rows = keys, k = dims): matrices (keys +0, +8) x (dims +0, +8), keys fastest
                const uint32_t aoff = (16 * warp + (mi & 1) * 8 + r8) * L::kRB + (16 * kk + (mi >> 1) * 8) * 2;
                uint32_t ka[4], va[4];
                ldsm_x4(sK + aoff, ka);
                ldsm_x4(sV + aoff, va);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    // B (k = dims, n = rows): matrices (rows +0, +8) x (dims +0, +8), dims fastest
                    const uint32_t boff = (16 * half + (mi >> 1) * 8 + r8) * L::kRB + (16 * kk + (mi & 1) * 8) * 2;
                    uint32_t qb[4], gb[4];
                    ldsm_x4(sQ + boff, qb);
                    ldsm_x4(sG + boff, gb);
                    mma_16816(sc[2 * half], ka[0], ka[1], ka[2], ka[3], qb[0], qb[1]);
                    mma_16816(sc[2 * half + 1], ka[0], ka[1], ka[2], ka[3], qb[2], qb[3]);
                    mma_16816(dp[2 * half], va[0], va[1], va[2], va[3], gb[0], gb[1]);
                    mma_16816(dp[2 * half + 1], va[0], va[1], va[2], va[3], gb[2], gb[3]);
                }
            }
            // P^T and dS^T: element e of tile nt is key jw + g + 8 (e >> 1), row i0 + 8 nt + 2t + (e & 1)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = jw + g + 8 * (e >> 1), il = 8 * nt + 2 * t + (e & 1), i = i0 + il;
                    bool vis = j < n && i < a.Nq && (!a.causal || j <= i + shift);
                    float x = sc[nt][e] * a.scale_log2;
                    if (kBias && vis) {
                        const float bb = a.bias[b * a.bs0 + h * a.bs1 + (long long)i * a.bs2 + j];
                        vis = bb != -INFINITY;
                        x = fmaf(bb, kLog2e, x);
                    }
                    const float p = vis ? ex2f(x - sL[il] * kLog2e) : 0.f;
                    sc[nt][e] = p;
                    dp[nt][e] = p * (dp[nt][e] - sC[il]);
                }
            }
            // dV_w += P^T G and dK_w += dS^T Q: M = 16 keys, K = 32 rows in two steps, N = D
#pragma unroll
            for (int kq = 0; kq < 2; ++kq) {
                const uint32_t pa0 = pack_bf16(sc[2 * kq][0], sc[2 * kq][1]), pa1 = pack_bf16(sc[2 * kq][2], sc[2 * kq][3]);
                const uint32_t pa2 = pack_bf16(sc[2 * kq + 1][0], sc[2 * kq + 1][1]);
                const uint32_t pa3 = pack_bf16(sc[2 * kq + 1][2], sc[2 * kq + 1][3]);
                const uint32_t sa0 = pack_bf16(dp[2 * kq][0], dp[2 * kq][1]), sa1 = pack_bf16(dp[2 * kq][2], dp[2 * kq][3]);
                const uint32_t sa2 = pack_bf16(dp[2 * kq + 1][0], dp[2 * kq + 1][1]);
                const uint32_t sa3 = pack_bf16(dp[2 * kq + 1][2], dp[2 * kq + 1][3]);
#pragma unroll
                for (int nd2 = 0; nd2 < ND / 2; ++nd2) {
                    // B (k = rows, n = dims) by transposing [row][dim]: (rows +0, +8) x (dims +0, +8), rows fastest
                    const uint32_t toff = (16 * kq + (mi & 1) * 8 + r8) * L::kRB + (16 * nd2 + (mi >> 1) * 8) * 2;
                    uint32_t gbv[4], qbv[4];
                    ldsm_x4_trans(sG + toff, gbv);
                    ldsm_x4_trans(sQ + toff, qbv);
                    mma_16816(dv_acc[2 * nd2], pa0, pa1, pa2, pa3, gbv[0], gbv[1]);
                    mma_16816(dv_acc[2 * nd2 + 1], pa0, pa1, pa2, pa3, gbv[2], gbv[3]);
                    mma_16816(dk_acc[2 * nd2], sa0, sa1, sa2, sa3, qbv[0], qbv[1]);
                    mma_16816(dk_acc[2 * nd2 + 1], sa0, sa1, sa2, sa3, qbv[2], qbv[3]);
                }
            }
            // dS^T (bf16) into shared memory as [key][row]
            uint8_t *sS = sm + L::kOffS;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
                    *reinterpret_cast<uint32_t *>(sS + (16 * warp + g + 8 * hh) * L::kSB + (8 * nt + 2 * t) * 2) =
                        pack_bf16(dp[nt][2 * hh], dp[nt][2 * hh + 1]);
            __syncthreads();

            // dQ of the tile's 32 rows, this warp's quarter of the head dimension, over the
            // block's 64 keys: M = 32 rows in two tiles, K = 64 keys in four steps
            float dqa[2][NQ][4];
#pragma unroll
            for (int mq = 0; mq < 2; ++mq)
#pragma unroll
                for (int nd = 0; nd < NQ; ++nd)
#pragma unroll
                    for (int e = 0; e < 4; ++e) dqa[mq][nd][e] = 0.f;
            const int dn0 = warp * (D / 4);
            const uint32_t sSa = smem_addr(sS);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint32_t da[2][4];
#pragma unroll
                for (int mq = 0; mq < 2; ++mq) {
                    // A (rows = query rows, k = keys) by transposing [key][row]: (keys +0, +8) x (rows +0, +8), rows fastest
                    const uint32_t soff = (16 * kk + (mi >> 1) * 8 + r8) * L::kSB + (16 * mq + (mi & 1) * 8) * 2;
                    ldsm_x4_trans(sSa + soff, da[mq]);
                }
#pragma unroll
                for (int nd2 = 0; nd2 < NQ / 2; ++nd2) {
                    // B (k = keys, n = dims) by transposing [key][dim]: (keys +0, +8) x (dims +0, +8), keys fastest
                    const uint32_t koff = (16 * kk + (mi & 1) * 8 + r8) * L::kRB + (dn0 + 16 * nd2 + (mi >> 1) * 8) * 2;
                    uint32_t kbv[4];
                    ldsm_x4_trans(sK + koff, kbv);
#pragma unroll
                    for (int mq = 0; mq < 2; ++mq) {
                        mma_16816(dqa[mq][2 * nd2], da[mq][0], da[mq][1], da[mq][2], da[mq][3], kbv[0], kbv[1]);
                        mma_16816(dqa[mq][2 * nd2 + 1], da[mq][0], da[mq][1], da[mq][2], da[mq][3], kbv[2], kbv[3]);
                    }
                }
            }
#pragma unroll
            for (int mq = 0; mq < 2; ++mq)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int i = i0 + 16 * mq + g + 8 * hh;
                    if (i >= a.Nq) continue;
                    float *dst = a.dq_acc + (((long long)b * a.Nq + i) * a.H + h) * D + dn0 + 2 * t;
#pragma unroll
                    for (int nd = 0; nd < NQ; ++nd)
                        red_add_v2(dst + 8 * nd, a.scale * dqa[mq][nd][2 * hh], a.scale * dqa[mq][nd][2 * hh + 1]);
                }
            __syncthreads();  // dS^T and this stage are free for the next tile
        }
        cp_async_wait<0>();
    }

    // dK (times scale) and dV of this warp's keys; a key no row sees gets zeros
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int j = jw + g + 8 * hh;
        if (j >= a.Nk) continue;
        __nv_bfloat16 *dkr = a.dk + b * a.dks0 + (long long)j * a.dks1 + h * a.dks2 + 2 * t;
        __nv_bfloat16 *dvr = a.dv + b * a.dvs0 + (long long)j * a.dvs1 + h * a.dvs2 + 2 * t;
#pragma unroll
        for (int nd = 0; nd < ND; ++nd) {
            *reinterpret_cast<uint32_t *>(dkr + 8 * nd) =
                pack_bf16(a.scale * dk_acc[nd][2 * hh], a.scale * dk_acc[nd][2 * hh + 1]);
            *reinterpret_cast<uint32_t *>(dvr + 8 * nd) = pack_bf16(dv_acc[nd][2 * hh], dv_acc[nd][2 * hh + 1]);
        }
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
        make_uint4(pack_bf16(f0.x, f0.y), pack_bf16(f0.z, f0.w), pack_bf16(f1.x, f1.y), pack_bf16(f1.z, f1.w));
}

template <int D, bool kBias>
cudaError_t launch_main(const BwdArgs &a, cudaStream_t st) {
    const int smem = BwdLayout<D>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(bwd_main_kernel<D, kBias>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((a.Nk + kKB - 1) / kKB), (unsigned)a.H, (unsigned)a.B);
    bwd_main_kernel<D, kBias><<<grid, kBwdThreads, smem, st>>>(a);
    return cudaGetLastError();
}

// Prep, then the products (the tcgen05 kernel for d = 128 without a bias, the warp-level
// kernel otherwise), then the dQ conversion.  A failed tcgen05 launch reports through
// attn_last_error and returns cudaErrorLaunchFailure here.
template <int D>
cudaError_t launch_all(const BwdArgs &a, const attn_bwd_params_t &p, cudaStream_t st) {
    const long long rows = (long long)a.B * a.Nq * a.H;
    const unsigned row_blocks = (unsigned)((rows * (D / 8) + 255) / 256);
    if (rows > 0) {
        bwd_prep_kernel<D><<<row_blocks, 256, 0, st>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if ((long long)a.B * a.H * a.Nk > 0) {
        if (D == 128 && !a.bias) {
            if (launch_bwd_tc(p, a.dq_acc, a.crow, a.lrow, st) != ATTN_OK) return cudaErrorLaunchFailure;
        } else {
            cudaError_t e = a.bias ? launch_main<D, true>(a, st) : launch_main<D, false>(a, st);
            if (e != cudaSuccess) return e;
        }
    }
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
