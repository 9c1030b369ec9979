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
// Several query rows of one sequence (2 <= Nq <= 8, bottom-right causal optional) share one
// pass over the cache: see decode_rows_mma_kernel below.  Partial states are laid out
// [B, H, Nq, S, 2 + D]; the merge kernel takes one (b, h, row) per CTA.
//
// Fused merge (attn_decode_splitkv_fused): every split CTA of a (b, h) writes its states and
// counts itself on that (b, h)'s counter with a release; the CTA that counts last reads all S
// states from L2, merges them as the merge kernel does, and writes o and lse.  No CTA waits for another, so one launch does the whole step.  A
// counter word holds (tag of the call, count): each call has a tag of its own, and a count
// stored under another tag (an earlier call, or whatever the workspace held) reads as zero,
// so the workspace needs no clearing.
//
// Split kernel (one row): grid (S, H, B), 128 threads.  The cache is read once, with 16-byte loads:
// a group of D/8 lanes holds one key row (each lane 8 bf16 of K and 8 of V), so a warp
// reads 32/(D/8) key rows per load instruction, coalesced.  Each group runs the online
// update over its keys (key lo + g + t*G of the split for t = 0, 1, ..., G groups per CTA,
// 4 keys in flight per group), with the logits kept in base-2 units (x * log2 e) so that one ex2
// gives each exponential.  The G group states are then merged in shared memory and the
// split's state is written in natural-log units.
#include <atomic>
#include <chrono>
#include <cmath>
#include <mutex>

#include <cuda_bf16.h>

#include "attn_internal.h"
#include "sm100_ptx.cuh"
#include "warp_mma.cuh"

namespace attn {
namespace {

using namespace wmma16;

// Tags of fused decode calls: 48 bits, distinct for every call of the process, never 0; the
// sequence starts from the clock so that it does not repeat an earlier process's.
unsigned long long next_decode_tag() {
    static std::atomic<unsigned long long> next{
        (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count() * 2654435761ull};
    for (;;) {
        const unsigned long long t = next.fetch_add(1) & 0xffffffffffffull;
        if (t) return t;
    }
}

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
    // fused merge only: per-(b, h) arrival counters (tag << 16 | count), the call's tag, outputs
    unsigned long long *counters;
    unsigned long long tag;
    __nv_bfloat16 *o;
    long long os0, os1, os2;
    float *lse;
};

// Merges the S partial states st, st + ss, st + 2 ss, ... ((m, l, u[0..dv)) each, l == 0:
// empty) into one output row and its lse (+0.0 and -inf when every part is empty).  One warp: the common maximum M is
// reduced over the lanes; then, 32 parts at a time, each lane forms one part's weight
// exp(m_s - M) (0 for an empty part), and the weights are passed round by shuffles while every
// lane sums weight * u_s over its columns (lane, lane + 32, ... of a block of 256 columns).
// The states are read from L2 (ld.global.cg), so states that other CTAs wrote during this
// launch are seen once their writers' fences have been observed.
template <typename OutT>
__device__ __forceinline__ void merge_row(const float *st, int S, long long ss, int dv, OutT *orow,
                                          float *lse_out) {
    const int lane = threadIdx.x & 31;
    const long long ld = ss;
    float M = -INFINITY;
    for (int s = lane; s < S; s += 32)
        if (__ldcg(st + s * ld + 1) > 0.f) M = fmaxf(M, __ldcg(st + s * ld));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (M == -INFINITY) {
        for (int c = lane; c < dv; c += 32) orow[c] = OutT(0.f);
        if (lse_out && lane == 0) *lse_out = -INFINITY;
        return;
    }
    float lsum = 0.f;
    for (int s = lane; s < S; s += 32) {
        const float l = __ldcg(st + s * ld + 1);
        if (l > 0.f) lsum = fmaf(expf(__ldcg(st + s * ld) - M), l, lsum);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    const float inv = 1.f / lsum;
    for (int c0 = 0; c0 < dv; c0 += 256) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int s0 = 0; s0 < S; s0 += 32) {
            const int s = s0 + lane;
            float w = 0.f;
            if (s < S && __ldcg(st + s * ld + 1) > 0.f) w = expf(__ldcg(st + s * ld) - M);
            const int n = min(32, S - s0);
            for (int i = 0; i < n; ++i) {
                const float wi = __shfl_sync(0xffffffffu, w, i);
                if (wi == 0.f) continue;  // uniform across the warp
                const float *u = st + (s0 + i) * ld + 2 + c0 + lane;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    if (c0 + lane + 32 * k < dv) acc[k] = fmaf(wi, __ldcg(u + 32 * k), acc[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (c0 + lane + 32 * k < dv) orow[c0 + lane + 32 * k] = OutT(acc[k] * inv);
    }
    if (lse_out && lane == 0) *lse_out = M + logf(lsum);
}

// Fused merge: once every thread's states are written, warp 0 alone stays (the other warps
// leave, freeing their slots); its lane 0 makes the CTA's states visible device-wide and counts
// the CTA on its (b, h) counter, and the warp of the last of the S CTAs merges every row of
// (b, h).  The count is a compare-and-swap on (tag << 16 | count): it retries only when
// another split of the same (b, h) counted in between (at most S - 1 times), and gives up,
// reporting through the error word, after 4096.
template <int D>
__device__ __forceinline__ void fused_tail(const DecArgs &a, int b, int h) {
    __syncthreads();  // the CTA's states are written (ordered before lane 0's fence below)
    if (threadIdx.x >= 32) return;
    int last = 0;
    if (threadIdx.x == 0) {
        __threadfence();  // release: the states, visible device-wide before the count
        unsigned long long *cnt = a.counters + (long long)b * a.H + h;
        unsigned long long seen = *reinterpret_cast<volatile unsigned long long *>(cnt), mine = 0;
        for (int tries = 0;; ++tries) {
            mine = ((seen >> 16) == a.tag ? (seen & 0xffffull) : 0ull) + 1ull;
            const unsigned long long prev = atomicCAS(cnt, seen, (a.tag << 16) | mine);
            if (prev == seen) break;
            seen = prev;
            if (tries >= 4096) {
                atomicOr(a.flags, kFlagWaitTimeout);
                mine = 0;
                break;
            }
        }
        last = (mine == (unsigned long long)a.S);
        if (last) __threadfence();  // acquire: the other splits' states, observed through their counts
    }
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    for (int r = 0; r < a.Nq; ++r) {
        const long long row = ((long long)b * a.H + h) * a.Nq + r;
        merge_row<__nv_bfloat16>(a.part + row * a.S * (2 + D), a.S, 2 + D, D,
                                 a.o + b * a.os0 + r * a.os1 + h * a.os2, a.lse ? a.lse + row : nullptr);
    }
}

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

// One query row (Nq == 1; with one row the bottom-right causal mask hides no key).
template <int D, bool kFuse>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(DecArgs a) {
    constexpr int LPK = D / 8;            // lanes per key row
    constexpr int G = kThreads / LPK;     // key groups per CTA
    constexpr int U = 4;                  // keys in flight per group
    __shared__ float sm_m[G], sm_l[G];
    __shared__ float sm_u[G][D + 1];

    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int g = threadIdx.x / LPK, sub = threadIdx.x % LPK, c0 = sub * 8;
    // launched as a programmatic dependent: global memory only after the previous kernel
    ptx::grid_dep_wait();
    ptx::launch_dependents();

    int n = a.Nk;
    if (a.kv_lens) {
        int raw = a.kv_lens[b];
        n = min(max(raw, 0), a.Nk);
        if (raw != n && threadIdx.x == 0 && s == 0 && h == 0) atomicOr(a.flags, kFlagKvLenClamped);
    }
    const int lo = (int)(((long long)s * n) / a.S), hi = (int)(((long long)(s + 1) * n) / a.S);

    float qf[8];
    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(a.q + b * a.qs0 + h * a.qs2 + c0), qf);
#pragma unroll
    for (int t = 0; t < 8; ++t) qf[t] *= a.scale_log2;

    const __nv_bfloat16 *kb = a.k + b * a.ks0 + h * a.ks2 + c0;
    const __nv_bfloat16 *vb = a.v + b * a.vs0 + h * a.vs2 + c0;
    const float *bias_row = a.bias ? a.bias + b * a.bs0 + h * a.bs1 : nullptr;

    float m = -INFINITY, l = 0.f, u[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) u[t] = 0.f;

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
        float x[U];
#pragma unroll
        for (int w = 0; w < U; ++w) {
            float kf[8];
            bf16x8_to_f32(kr[w], kf);
            float d = 0.f;
#pragma unroll
            for (int t = 0; t < 8; ++t) d = fmaf(qf[t], kf[t], d);
            x[w] = d;
        }
#pragma unroll
        for (int w = 0; w < U; ++w) {
#pragma unroll
            for (int o = LPK / 2; o > 0; o >>= 1) x[w] += __shfl_xor_sync(0xffffffffu, x[w], o);
        }
#pragma unroll
        for (int w = 0; w < U; ++w) {
            const int j = base + w * G + g;
            if (j >= hi) break;  // uniform across the group
            float xs = x[w];
            if (bias_row) {
                float bj = bias_row[j];
                if (bj == -INFINITY) continue;  // masked key
                xs = fmaf(bj, kLog2e, xs);
            }
            float m_new = fmaxf(m, xs);
            float alpha = (m == -INFINITY) ? 0.f : ex2(m - m_new);
            float p = ex2(xs - m_new);
            float vf[8];
            bf16x8_to_f32(vr[w], vf);
            l = fmaf(alpha, l, p);
#pragma unroll
            for (int t = 0; t < 8; ++t) u[t] = fmaf(alpha, u[t], p * vf[t]);
            m = m_new;
        }
    }

    if (sub == 0) {
        sm_m[g] = m;
        sm_l[g] = l;
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) sm_u[g][c0 + t] = u[t];
    __syncthreads();

    // merge the G group states; thread c owns column c
    float M = -INFINITY;
#pragma unroll
    for (int gg = 0; gg < G; ++gg)
        if (sm_l[gg] > 0.f) M = fmaxf(M, sm_m[gg]);
    float *out = a.part + (((long long)b * a.H + h) * a.S + s) * (2 + D);
    if (M == -INFINITY) {  // empty split
        for (int c = threadIdx.x; c < D; c += kThreads) out[2 + c] = 0.f;
        if (threadIdx.x == 0) {
            out[0] = -INFINITY;
            out[1] = 0.f;
        }
    } else {
        float L = 0.f;
#pragma unroll
        for (int gg = 0; gg < G; ++gg)
            if (sm_l[gg] > 0.f) L = fmaf(ex2(sm_m[gg] - M), sm_l[gg], L);
        for (int c = threadIdx.x; c < D; c += kThreads) {
            float acc = 0.f;
#pragma unroll
            for (int gg = 0; gg < G; ++gg)
                if (sm_l[gg] > 0.f) acc = fmaf(ex2(sm_m[gg] - M), sm_u[gg][c], acc);
            out[2 + c] = acc;
        }
        if (threadIdx.x == 0) {
            out[0] = M * kLn2;  // back to natural-log units: exp(x - m) == 2^(x*log2e - M)
            out[1] = L;
        }
    }
    if constexpr (kFuse) fused_tail<D>(a, b, h);
}

// ---------------------------------------------------------------- several query rows (Nq >= 2)
//
// With 2 to 8 query rows per sequence the per-key work grows with the rows while the bytes
// read stay those of one row, so the scores and the value sums go to the tensor cores
// (mma.sync m16n8k16, bf16 inputs, fp32 accumulation; the products are 16 keys by at most 8
// rows, far below what tcgen05 tiles are for).  Each warp owns one split of one (b, h): CTA x
// of the grid holds splits 4x .. 4x + 3.  The warp walks its split's 16-key tiles, copied into
// its own shared memory with cp.async (double-buffered, rows padded to 16 B past 2*D so that
// ldmatrix reads are free of bank conflicts; keys past the split are zero-filled, so nothing
// stored past kv_len reaches a product):
//   S = Q K^T     M = 16 query rows (rows >= Nq are zero), N = 8 keys, K = 16 dims per step;
//                 the K operand comes from ldmatrix on the [key][dim] tile;
//   O^T += V^T P^T  M = 16 dims, N = 8 query rows, K = 16 keys; V^T comes from ldmatrix.trans,
//                 and P^T is the S accumulator itself: the fragment a thread holds of S (row
//                 g, keys 2t, 2t+1 of each 8-key half) is the fragment it must supply of P^T.
// The online update runs per query row on the four lanes that hold it (row max over their
// eight scores and two shuffles); the row's rescale factor reaches the lanes holding that row
// of O^T by a shuffle.  At the end the warp writes its split's state of each row straight
// from its fragments, as the one-row kernel writes its split's: no state is merged across warps.

constexpr int kRowsKT = 16;  // keys per warp tile
constexpr int kRowsWarps = kThreads / 32;

template <int D>
struct RowsLayout {
    static constexpr int kRowBytes = 2 * D + 16;               // padded key row
    static constexpr int kTileBytes = kRowsKT * kRowBytes;     // one K or V tile
    static constexpr int kBytes = kRowsWarps * 2 * 2 * kTileBytes;  // [warp][stage][K, V]
};

// The fused merge for a warp that owns a whole split: lane 0 counts the split as done on the
// (b, h) counter (tagged as in fused_tail); the warp whose count completes the S splits merges
// every row.  Bounded like fused_tail.
template <int D>
__device__ __forceinline__ void fused_tail_warp(const DecArgs &a, int b, int h) {
    __syncwarp();  // this warp's states are written (ordered before lane 0's fence below)
    const int lane = threadIdx.x & 31;
    int last = 0;
    if (lane == 0) {
        __threadfence();  // release: the states, visible device-wide before the count
        unsigned long long *cnt = a.counters + (long long)b * a.H + h;
        unsigned long long seen = *reinterpret_cast<volatile unsigned long long *>(cnt), mine = 0;
        for (int tries = 0;; ++tries) {
            mine = ((seen >> 16) == a.tag ? (seen & 0xffffull) : 0ull) + 1ull;
            const unsigned long long prev = atomicCAS(cnt, seen, (a.tag << 16) | mine);
            if (prev == seen) break;
            seen = prev;
            if (tries >= 4096) {
                atomicOr(a.flags, kFlagWaitTimeout);
                mine = 0;
                break;
            }
        }
        last = (mine == (unsigned long long)a.S);
        if (last) __threadfence();  // acquire: the other splits' states, observed through their counts
    }
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    for (int r = 0; r < a.Nq; ++r) {
        const long long row = ((long long)b * a.H + h) * a.Nq + r;
        merge_row<__nv_bfloat16>(a.part + row * a.S * (2 + D), a.S, 2 + D, D,
                                 a.o + b * a.os0 + r * a.os1 + h * a.os2, a.lse ? a.lse + row : nullptr);
    }
}

template <int D, bool kFuse>
__global__ void __launch_bounds__(kThreads) decode_rows_mma_kernel(DecArgs a) {
    using L = RowsLayout<D>;
    constexpr int NK = D / 16;  // k-steps of S = Q K^T; 16-dim tiles of O^T
    extern __shared__ __align__(128) uint8_t dsm[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int s = blockIdx.x * kRowsWarps + warp, h = blockIdx.y, b = blockIdx.z;
    const int nq = a.Nq;
    // launched as a programmatic dependent: global memory only after the previous kernel
    ptx::grid_dep_wait();
    ptx::launch_dependents();
    if (s >= a.S) return;  // the last CTA's warps past the split count (no CTA-wide barrier below)

    int n = a.Nk;
    if (a.kv_lens) {
        int raw = a.kv_lens[b];
        n = min(max(raw, 0), a.Nk);
        if (raw != n && lane == 0 && s == 0 && h == 0) atomicOr(a.flags, kFlagKvLenClamped);
    }
    const int lo = (int)(((long long)s * n) / a.S), hi = (int)(((long long)(s + 1) * n) / a.S);

    // this lane's softmax row is g (keys < vis_g visible); its rows of O^T are 2t and 2t + 1
    const int vis_g = g < nq ? (a.causal ? min(n, max(0, g + n - nq + 1)) : n) : 0;
    const float *bias_g = (a.bias && g < nq) ? a.bias + b * a.bs0 + h * a.bs1 + g * a.bs2 : nullptr;
    uint32_t qa[NK][2];  // A fragments of Q: row g, dims 16 kk + 2t (+1) and + 8 (+9)
#pragma unroll
    for (int kk = 0; kk < NK; ++kk) {
        qa[kk][0] = qa[kk][1] = 0u;
        if (g < nq) {
            const __nv_bfloat16 *qr = a.q + b * a.qs0 + g * a.qs1 + h * a.qs2 + 16 * kk + 2 * t;
            qa[kk][0] = *reinterpret_cast<const uint32_t *>(qr);
            qa[kk][1] = *reinterpret_cast<const uint32_t *>(qr + 8);
        }
    }
    float m_g = -INFINITY, l_g = 0.f;  // row g's reference and this lane's share of its sum
    float o[NK][4];
#pragma unroll
    for (int mt = 0; mt < NK; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    const __nv_bfloat16 *kb = a.k + b * a.ks0 + h * a.ks2;
    const __nv_bfloat16 *vb = a.v + b * a.vs0 + h * a.vs2;
    uint8_t *wsm = dsm + warp * 4 * L::kTileBytes;
    const int ntiles = (hi - lo + kRowsKT - 1) / kRowsKT;
    // tile T of the split into stage st: 16 keys x D dims of K and of V, 16 B per copy
    auto issue = [&](int T, int st) {
        uint8_t *sK = wsm + (2 * st) * L::kTileBytes, *sV = sK + L::kTileBytes;
        const int j0 = lo + T * kRowsKT;
#pragma unroll
        for (int i = 0; i < kRowsKT * (D / 8) / 32; ++i) {
            const int c = lane + 32 * i, key = c / (D / 8), ch = c % (D / 8);
            const int j = j0 + key;
            const bool in = j < hi;
            const long long jj = in ? j : lo;  // a valid address even when nothing is copied
            cp_async16(smem_addr(sK + key * L::kRowBytes + ch * 16), kb + jj * a.ks1 + ch * 8, in ? 16u : 0u);
            cp_async16(smem_addr(sV + key * L::kRowBytes + ch * 16), vb + jj * a.vs1 + ch * 8, in ? 16u : 0u);
        }
        cp_async_commit();
    };
    const int mi = lane >> 3, mr = lane & 7;  // ldmatrix: matrix and row this lane addresses
    int st = 0;
    if (ntiles > 0) issue(0, 0);
    else cp_async_commit();
    for (int T = 0; T < ntiles; ++T, st ^= 1) {
        if (T + 1 < ntiles) issue(T + 1, st ^ 1);
        else cp_async_commit();
        cp_async_wait<1>();
        __syncwarp();
        const uint8_t *sK = wsm + (2 * st) * L::kTileBytes, *sV = sK + L::kTileBytes;
        // matrices (keys 0-7 | 8-15) x (dims +0-7 | +8-15); this lane's row address
        const uint32_t rowoff = ((mi >> 1) * 8 + mr) * L::kRowBytes + (mi & 1) * 16;

        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < NK; ++kk) {
            uint32_t kf[4];
            ldsm_x4(smem_addr(sK) + rowoff + kk * 32, kf);
            mma_16816(sc[0], qa[kk][0], 0u, qa[kk][1], 0u, kf[0], kf[1]);
            mma_16816(sc[1], qa[kk][0], 0u, qa[kk][1], 0u, kf[2], kf[3]);
        }
        // row g's scores: keys j0 + 2t, + 1 (first half), j0 + 8 + 2t, + 1 (second half)
        const int j0 = lo + T * kRowsKT;
        float x[4] = {sc[0][0], sc[0][1], sc[1][0], sc[1][1]};
        float tm = -INFINITY;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int j = j0 + (e >> 1) * 8 + 2 * t + (e & 1);
            float xs = x[e] * a.scale_log2;
            if (j >= hi || j >= vis_g) xs = -INFINITY;
            else if (bias_g) {
                const float bj = bias_g[j];
                xs = (bj == -INFINITY) ? -INFINITY : fmaf(bj, kLog2e, xs);
            }
            x[e] = xs;
            tm = fmaxf(tm, xs);
        }
        tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 1));
        tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 2));
        const float m_new = fmaxf(m_g, tm);
        const float alpha = (m_g == -INFINITY) ? 0.f : ex2(m_g - m_new);
        float p[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) p[e] = (m_new == -INFINITY) ? 0.f : ex2(x[e] - m_new);
        l_g = fmaf(alpha, l_g, (p[0] + p[1]) + (p[2] + p[3]));
        m_g = m_new;
        // rows 2t and 2t + 1 of O^T take the factors of those rows (held by lanes 8t, 8t + 4)
        const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * t);
        const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * t + 4);
        const uint32_t pb0 = pack_bf16(p[0], p[1]), pb1 = pack_bf16(p[2], p[3]);
#pragma unroll
        for (int mt = 0; mt < NK; ++mt) {
            o[mt][0] *= a0;
            o[mt][1] *= a1;
            o[mt][2] *= a0;
            o[mt][3] *= a1;
            uint32_t vf[4];
            ldsm_x4_trans(smem_addr(sV) + rowoff + mt * 32, vf);
            mma_16816(o[mt], vf[0], vf[1], vf[2], vf[3], pb0, pb1);
        }
        __syncwarp();  // every lane is done with this stage before it is refilled
    }
    cp_async_wait<0>();
    l_g += __shfl_xor_sync(0xffffffffu, l_g, 1);
    l_g += __shfl_xor_sync(0xffffffffu, l_g, 2);

    // the split's state of each row: (m, l) from the lanes that own the row (t == 0), u from the
    // fragments of O^T (lane (g, t) holds dims 16 mt + g (+ 8) of rows 2t and 2t + 1); a row
    // that saw no key of the split gets (-inf, 0, 0)
    float *part_b = a.part + (((long long)b * a.H + h) * nq) * a.S * (2 + D);
    auto state = [&](int r) { return part_b + ((long long)r * a.S + s) * (2 + D); };
    if (t == 0 && g < nq) {
        float *out = state(g);
        out[0] = l_g > 0.f ? m_g * kLn2 : -INFINITY;
        out[1] = l_g;
    }
#pragma unroll
    for (int mt = 0; mt < NK; ++mt) {
        if (2 * t < nq) {
            float *r0 = state(2 * t) + 2 + 16 * mt + g;
            r0[0] = o[mt][0];
            r0[8] = o[mt][2];
        }
        if (2 * t + 1 < nq) {
            float *r1 = state(2 * t + 1) + 2 + 16 * mt + g;
            r1[0] = o[mt][1];
            r1[8] = o[mt][3];
        }
    }
    if constexpr (kFuse) fused_tail_warp<D>(a, b, h);
}

// Merge: one warp per (b, h, query row i) -- row r = (b*H + h)*Nq + i, whose state s sits at
// part + r * rs + s * ss -- four rows per CTA.
template <typename OutT>
__global__ void __launch_bounds__(kThreads) merge_kernel(const float *part, long long rows, int H, int Nq, int S,
                                                           long long rs, long long ss, int dv, OutT *o,
                                                           long long os0, long long os1, long long os2,
                                                           float *lse) {
    ptx::grid_dep_wait();  // the partial states come from the kernel before this one
    ptx::launch_dependents();
    const long long row = (long long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int i = (int)(row % Nq), bh = (int)(row / Nq), b = bh / H, h = bh % H;
    merge_row<OutT>(part + row * rs, S, ss, dv, o + b * os0 + i * os1 + h * os2, lse ? lse + row : nullptr);
}

template <int D, bool kFuse>
cudaError_t launch_rows(const DecArgs &a, dim3 grid, cudaStream_t st) {
    const int smem = RowsLayout<D>::kBytes;
    cudaError_t e =
        cudaFuncSetAttribute(decode_rows_mma_kernel<D, kFuse>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_rows_mma_kernel<D, kFuse>, grid, dim3(kThreads), smem, st, a);
}

}  // namespace

attn_status_t launch_decode_split(const attn_fwd_params_t &p, int num_splits, float *partials,
                                  unsigned long long *counters, cudaStream_t st) {
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
    a.counters = counters;
    a.tag = counters ? next_decode_tag() : 0ull;
    a.o = static_cast<__nv_bfloat16 *>(p.o);
    a.os0 = p.o_stride[0]; a.os1 = p.o_stride[1]; a.os2 = p.o_stride[2];
    a.lse = p.lse;
    a.flags = device_flags();
    if (!a.flags) return fail(ATTN_ERR_CUDA, "could not resolve the device error word");
    if (p.B > 65535 || p.H > 65535) return fail(ATTN_ERR_UNSUPPORTED, "decode supports B, H <= 65535");
    if (p.Nq < 1 || p.Nq > kMaxDecodeRows)
        return fail(ATTN_ERR_UNSUPPORTED, "decode supports 1 <= Nq <= %d (got %lld)", kMaxDecodeRows,
                    (long long)p.Nq);
    dim3 grid((unsigned)num_splits, (unsigned)p.H, (unsigned)p.B);
    cudaError_t e = cudaSuccess;
    const bool fuse = counters != nullptr;
    if (p.Nq == 1) {
        auto kern = p.dk == 64 ? (fuse ? decode_split_kernel<64, true> : decode_split_kernel<64, false>)
                               : (fuse ? decode_split_kernel<128, true> : decode_split_kernel<128, false>);
        e = launch_pdl(kern, grid, dim3(kThreads), 0, st, a);
    } else {
        // several rows: one warp per split, kRowsWarps splits per CTA
        const dim3 rgrid((unsigned)((num_splits + kRowsWarps - 1) / kRowsWarps), (unsigned)p.H, (unsigned)p.B);
        if (p.dk == 64) e = fuse ? launch_rows<64, true>(a, rgrid, st) : launch_rows<64, false>(a, rgrid, st);
        else e = fuse ? launch_rows<128, true>(a, rgrid, st) : launch_rows<128, false>(a, rgrid, st);
    }
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "decode rows launch: %s", cudaGetErrorString(e));
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "decode split launch: %s", cudaGetErrorString(e));
    return ATTN_OK;
}

attn_status_t launch_merge(const float *partials, int64_t B, int64_t H, int64_t Nq, int num_splits,
                           int64_t dv, int o_dtype, void *o, const int64_t o_stride[3], float *lse,
                           cudaStream_t st, int64_t row_stride, int64_t split_stride) {
    const long long rows = (long long)B * H * Nq;
    const long long rs = row_stride ? row_stride : (long long)num_splits * (2 + dv);
    const long long ss = split_stride ? split_stride : 2 + dv;
    if (rows > 0x7fffffffLL) return fail(ATTN_ERR_UNSUPPORTED, "B*H*Nq too large");
    dim3 grid((unsigned)((rows + kThreads / 32 - 1) / (kThreads / 32)));
    const cudaError_t e =
        o_dtype == ATTN_DTYPE_BF16
            ? launch_pdl(merge_kernel<__nv_bfloat16>, grid, dim3(kThreads), 0, st, partials, rows, (int)H, (int)Nq,
                         num_splits, rs, ss, (int)dv, static_cast<__nv_bfloat16 *>(o), o_stride[0], o_stride[1],
                         o_stride[2], lse)
            : launch_pdl(merge_kernel<float>, grid, dim3(kThreads), 0, st, partials, rows, (int)H, (int)Nq,
                         num_splits, rs, ss, (int)dv, static_cast<float *>(o), o_stride[0], o_stride[1],
                         o_stride[2], lse);
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

// Host code cannot use g_decode_scratch's name as a device address: the address is looked up
// (cudaGetSymbolAddress, with the device current) the first time a CUDA context calls this
// entry point, and cached per device together with that context's unique id.  A later call
// from another context on the same device -- for instance after cudaDeviceReset replaced the
// primary context -- finds a different id and looks the address up again.
struct ScratchSlot {
    unsigned long long ctx_id;
    void *ptr;
};
ScratchSlot g_scratch_slot[64];
std::mutex g_scratch_mutex;

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

bool driver_fn(const char *name, void **fn) {
    cudaDriverEntryPointQueryResult q;
    return cudaGetDriverEntryPointByVersion(name, fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
           q == cudaDriverEntryPointSuccess && *fn;
}

// Unique id of the calling thread's current context, or 0 when there is none yet.
attn_status_t current_ctx_id(unsigned long long *id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    if (!get_current || !get_id) {
        void *a = nullptr, *b = nullptr;
        if (!driver_fn("cuCtxGetCurrent", &a) || !driver_fn("cuCtxGetId", &b))
            return fail(ATTN_ERR_CUDA, "cuCtxGetCurrent / cuCtxGetId are not available");
        get_current = reinterpret_cast<CtxGetCurrentFn>(a);
        get_id = reinterpret_cast<CtxGetIdFn>(b);
    }
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuCtxGetCurrent failed");
    *id = 0;
    if (ctx && get_id(ctx, id) != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuCtxGetId failed");
    return ATTN_OK;
}

attn_status_t noalloc_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(ATTN_ERR_UNSUPPORTED, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    unsigned long long id = 0;
    attn_status_t st = current_ctx_id(&id);
    if (st) return st;
    ScratchSlot &slot = g_scratch_slot[dev];
    if (!slot.ptr || id == 0 || slot.ctx_id != id) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
        if (e != cudaSuccess)
            return fail(ATTN_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        if ((st = current_ctx_id(&id))) return st;  // the lookup may have made the context current
        slot.ptr = ptr;
        slot.ctx_id = id;
    }
    *out = slot.ptr;
    return ATTN_OK;
}

}  // namespace
}  // namespace attn

extern "C" attn_status_t attn_decode_splitkv_noalloc(const attn_fwd_params_t *p, int32_t num_splits,
                                                     attn_stream_t stream) {
    using namespace attn;
    // the workspace entry point's own checks first, so that a bad argument is reported as such
    attn_status_t st = check_decode_args(p, num_splits);
    if (st) return st;
    const size_t need = attn_decode_workspace_bytes_rows(p->B, p->H, p->Nq, p->dv, num_splits);
    if (need > kNoAllocScratchBytes)
        return fail(ATTN_ERR_WORKSPACE,
                    "allocation-free decode needs %zu bytes of partial states for B=%lld H=%lld "
                    "Nq=%lld dv=%lld num_splits=%d; its built-in scratch holds %zu",
                    need, (long long)p->B, (long long)p->H, (long long)p->Nq, (long long)p->dv, num_splits,
                    kNoAllocScratchBytes);
    if (p->B * p->H == 0) return ATTN_OK;
    void *scratch = nullptr;
    if ((st = noalloc_scratch(&scratch))) return st;
    return attn_decode_splitkv(p, num_splits, scratch, kNoAllocScratchBytes, stream);
}
