// fwd_bf16_common.cuh -- pieces shared by the two bf16 prefill kernels (one 128-row query tile
// per CTA, and two tiles per CTA): arguments, tile constants, and the per-row softmax steps
// that run on one thread per query row (the row's TMEM lane).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <cmath>

#include "attn_internal.h"
#include "dropout_rng.cuh"
#include "sm100_ptx.cuh"

namespace attn {
namespace bf16fwd {

constexpr int BQ = 128;                 // query rows per tile (= MMA M = TMEM lanes)
constexpr int BK = 128;                 // keys per tile (= N of S = Q K^T, = K of O += P V)
constexpr int kPanelBytes = 128 * 128;  // 128 rows x 64 bf16 (128 bytes), 128B-swizzled
constexpr int kSmemMax = 232448;        // 227 KB of dynamic shared memory per CTA
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// A row keeps its reference maximum until a tile's maximum exceeds it by more than 8 in
// base-2 units (a factor 256): rescaling is exact for any reference shared by l and u, and
// exponentials <= 256 stay far from fp32/bf16 overflow.
constexpr float kRescaleThreshold = 8.0f;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // every mbarrier wait gives up after 1 s

struct Args {
    int B, H, Nq, Nk, causal, n_items;
    float scale_log2;
    __nv_bfloat16 *o;
    long long os0, os1, os2;
    float *lse;
    const float *bias;
    long long bs0, bs1, bs2;
    const int *kv_lens;
    uint32_t *flags;
    // division by B * H and by H as a multiply-high and two shifts (fill_divisors)
    uint32_t div_bhn_m, div_h_m;
    int div_bhn_s, div_h_s;  // first shift | second shift << 8
};

// The multiply-high division of Granlund and Montgomery ("Division by invariant integers using
// multiplication", PLDI 1994, section 4), exact for every 32-bit dividend: for a divisor d >= 1
// with l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1 and n / d = (t + ((n - t) >> s1)) >> s2
// where t = umulhi(m, n), s1 = min(l, 1), s2 = max(l - 1, 0).
inline void fast_div_params(uint32_t d, uint32_t &m, int &s) {
    int l = 0;
    while (l < 32 && (1ull << l) < d) ++l;
    m = (uint32_t)(((1ull << 32) * ((1ull << l) - d)) / d) + 1;
    s = (l < 1 ? l : 1) | ((l > 1 ? l - 1 : 0) << 8);
}
inline void fill_divisors(Args &a) {
    fast_div_params((uint32_t)(a.B * a.H), a.div_bhn_m, a.div_bhn_s);
    fast_div_params((uint32_t)a.H, a.div_h_m, a.div_h_s);
}
__device__ __forceinline__ uint32_t div_fast(uint32_t n, uint32_t m, int s) {
    const uint32_t t = __umulhi(m, n);
    return (t + ((n - t) >> (s & 255))) >> (s >> 8);
}

// Options beyond the plain operator, in a kernel argument of their own so that the kernels
// that use none keep their argument block (and their register allocation):
//   dropout of a training forward: keep bits (bit j % 8 of byte j / 8 of a row), or null;
//   a forward over one shard of the keys (partial states): local key j is global key
//   key_off + j of a sequence of Nk_tot keys, and part receives each row's (m, l, u).
struct DropArgs {
    const uint8_t *dmask;
    long long dms0, dms1, dms2;
    float inv_keep;  // 1 / (1 - dropout_p), the realised p for in-kernel draws
    int key_off, Nk_tot;
    float *part;
    // in-kernel draws (rng != 0): Philox4x32-10 under key (seed_lo, seed_hi), fourth counter
    // word offset, byte threshold p8 in each byte of p8x4 (dropout_rng.cuh)
    int rng;
    uint32_t seed_lo, seed_hi, offset, p8x4;
};

// The DropArgs fields of a forward's dropout settings (mask or in-kernel draws).
inline void fill_dropout(DropArgs &dr, const attn_fwd_params_t &p) {
    dr.dmask = p.dropout_mask;
    dr.dms0 = p.dropout_mask_stride[0];
    dr.dms1 = p.dropout_mask_stride[1];
    dr.dms2 = p.dropout_mask_stride[2];
    dr.rng = p.dropout_rng == 1;
    const uint32_t p8 = dropout_p8(p.dropout_p);
    dr.seed_lo = (uint32_t)(p.dropout_seed & 0xffffffffu);
    dr.seed_hi = (uint32_t)(p.dropout_seed >> 32);
    dr.offset = (uint32_t)(p.dropout_offset & 0xffffffffu);
    dr.p8x4 = p8 * 0x01010101u;
    dr.inv_keep = dr.rng ? (float)(256.0 / (256.0 - (double)p8))
                         : p.dropout_mask ? (float)(1.0 / (1.0 - (double)p.dropout_p)) : 1.f;
}

// Key length of sequence b, clamped to [0, Nk] (a clamp is reported once per sequence); Nk is
// the whole sequence's key count (a.Nk unless the kernel computes over one shard).
__device__ __forceinline__ int seq_len(const Args &a, int b, bool report, int Nk) {
    if (!a.kv_lens) return Nk;
    const int raw = a.kv_lens[b];
    const int n = min(max(raw, 0), Nk);
    if (raw != n && report) atomicOr(a.flags, kFlagKvLenClamped);
    return n;
}
__device__ __forceinline__ int seq_len(const Args &a, int b, bool report) { return seq_len(a, b, report, a.Nk); }

// Number of 128-key tiles a query tile starting at row r0 must visit: keys past the last
// visible key of its last row are never loaded (causal: key j visible to row i iff
// j <= i + n - Nq, i.e. the sequences' ends aligned).
__device__ __forceinline__ int kv_tiles(const Args &a, int r0, int n) {
    if (r0 >= a.Nq) return 0;
    int kv_end = n;
    if (a.causal) kv_end = min(n, max(0, min(r0 + BQ, a.Nq) + n - a.Nq));
    return (kv_end + BK - 1) / BK;
}

// The same in a shard's own key numbering: keys j < n are within the sequence and, under the
// causal mask, key j is visible to row i iff j <= i + shift.
__device__ __forceinline__ int kv_tiles_shard(const Args &a, int r0, int n, int shift) {
    if (r0 >= a.Nq) return 0;
    int kv_end = n;
    if (a.causal) kv_end = min(n, max(0, min(r0 + BQ, a.Nq) + shift));
    return (kv_end + BK - 1) / BK;
}

// The row of S held in TMEM columns [col, col + BK) of this thread's lane.
__device__ __forceinline__ void load_s_row(uint32_t taddr, float (&x)[BK]) {
    uint32_t raw[BK];
#pragma unroll
    for (int cc = 0; cc < BK / 32; ++cc)
        ptx::tmem_ld32(taddr + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&raw[cc * 32]));
    ptx::tmem_ld_wait();
#pragma unroll
    for (int cc = 0; cc < BK / 32; ++cc)
        ptx::reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&raw[cc * 32]));
#pragma unroll
    for (int k = 0; k < BK; ++k) x[k] = __uint_as_float(raw[k]);
}

// Bias of this row for keys [kv0, kv0 + BK) in base-2 units (b * log2 e), written into xb;
// keys >= n (masked in any case) read as 0 and are never loaded.  The loads have no consumer
// until load_s_row_bias, so a call placed right after a tile's P is stored keeps them in
// flight while the thread waits for the next S.
__device__ __forceinline__ void load_bias(const float *bias_row, bool bias_vec, int kv0, int n,
                                          float (&xb)[BK]) {
    if (!bias_row) {
#pragma unroll
        for (int k = 0; k < BK; ++k) xb[k] = 0.f;
        return;
    }
    if (bias_vec && kv0 + BK <= n) {
#pragma unroll
        for (int k4 = 0; k4 < BK / 4; ++k4) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(bias_row + kv0) + k4);
            xb[4 * k4 + 0] = v.x * kLog2e;
            xb[4 * k4 + 1] = v.y * kLog2e;
            xb[4 * k4 + 2] = v.z * kLog2e;
            xb[4 * k4 + 3] = v.w * kLog2e;
        }
    } else {
#pragma unroll
        for (int k = 0; k < BK; ++k) xb[k] = (kv0 + k < n) ? __ldg(bias_row + kv0 + k) * kLog2e : 0.f;
    }
}

// Row r of a 32-key bias panel staged in shared memory by TMA (128 rows x 128 bytes, 128-byte
// swizzle: 16-byte chunk c of row r at chunk c ^ (r & 7)), in base-2 units, into keys
// [32 p, 32 p + 32) of xb.  Eight consecutive rows read eight different bank groups.
__device__ __forceinline__ void read_bias_panel(const uint8_t *panel, int r, int p, float (&xb)[BK]) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float4 v = *reinterpret_cast<const float4 *>(panel + r * 128 + ((c ^ (r & 7)) * 16));
        xb[p * 32 + 4 * c + 0] = v.x * kLog2e;
        xb[p * 32 + 4 * c + 1] = v.y * kLog2e;
        xb[p * 32 + 4 * c + 2] = v.z * kLog2e;
        xb[p * 32 + 4 * c + 3] = v.w * kLog2e;
    }
}

// x = S * c + xb in place: the row of S from TMEM columns [taddr, taddr + BK), 32 columns at a
// time (so that S and the bias never need 256 registers at once).
__device__ __forceinline__ void load_s_row_bias(uint32_t taddr, float c, float (&xb)[BK]) {
#pragma unroll
    for (int cc = 0; cc < BK / 32; ++cc) {
        uint32_t t[32];
        ptx::tmem_ld32(taddr + cc * 32, t);
        ptx::tmem_ld_wait();
        ptx::reg_fence(t);
#pragma unroll
        for (int k = 0; k < 32; ++k) xb[cc * 32 + k] = fmaf(__uint_as_float(t[k]), c, xb[cc * 32 + k]);
    }
}

// Masks keys >= lim (a select: whatever is stored at a masked position, NaN included, is
// dropped here) and returns the tile maximum in base-2 units (-inf when no key of the tile is
// visible).  With a bias, x already holds base-2 logits; without one, x is raw S and the
// scale is applied to the maximum only (c > 0) and later inside the exponent.
template <bool kBias>
__device__ __forceinline__ float tile_logits(float (&x)[BK], float c, int kv0, bool need_mask,
                                             int lim) {
    if (need_mask) {
#pragma unroll
        for (int k = 0; k < BK; ++k)
            if (kv0 + k >= lim) x[k] = -INFINITY;
    }
    float m8[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) m8[t] = x[t];
#pragma unroll
    for (int k = 8; k < BK; ++k) m8[k & 7] = fmaxf(m8[k & 7], x[k]);
    float mt = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                     fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
    if (!kBias) mt *= c;
    return mt;
}

// The reference maximum of a row: the first visible key sets it
// (the old state has no mass, so nothing is rescaled); afterwards it moves only when the tile
// maximum exceeds it by more than kRescaleThreshold, and then alpha = 2^(m_old - m_new).
__device__ __forceinline__ float update_max(float mt, float &m_run, bool &rescale) {
    rescale = false;
    if (mt == -INFINITY) return 1.f;
    if (m_run == -INFINITY) {
        m_run = mt;
        return 1.f;
    }
    if (mt > m_run + kRescaleThreshold) {
        const float alpha = ptx::ex2(m_run - mt);
        m_run = mt;
        rescale = true;
        return alpha;
    }
    return 1.f;
}

// p = 2^(x - m) in place (half a packed FFMA + one ex2 per element); returns the row's
// tile mass.
template <bool kBias>
__device__ __forceinline__ float tile_exp(float (&x)[BK], float c, float m_run) {
    const float mref = (m_run == -INFINITY) ? 0.f : m_run;
    const float cc = kBias ? 1.f : c;
    float s8[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) s8[t] = 0.f;
    // two elements per packed f32x2 FMA and add: half the FP32 instructions of the softmax
#pragma unroll
    for (int k = 0; k < BK; k += 2) {
        ptx::fma2(x[k], x[k + 1], x[k], x[k + 1], cc, cc, -mref, -mref);
        x[k] = ptx::ex2(x[k]);
        x[k + 1] = ptx::ex2(x[k + 1]);
        ptx::add2(s8[k & 7], s8[(k & 7) + 1], s8[k & 7], s8[(k & 7) + 1], x[k], x[k + 1]);
    }
    return ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
}

// P rounded to bf16, packed two per 32-bit TMEM column (lower key in the low half), into the
// columns [taddr, taddr + BK/2) that held S.
__device__ __forceinline__ void store_p(uint32_t taddr, const float (&x)[BK]) {
#pragma unroll
    for (int cc = 0; cc < BK / 64; ++cc) {
        uint32_t pk[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) pk[t] = ptx::pack_bf16x2(x[cc * 64 + 2 * t], x[cc * 64 + 2 * t + 1]);
        ptx::tmem_st32(taddr + cc * 32, pk);
    }
    ptx::tmem_st_wait();
}

// u <- alpha * u for this lane's DV accumulator columns at taddr.
template <int DV>
__device__ __forceinline__ void scale_o(uint32_t taddr, float alpha) {
#pragma unroll
    for (int cc = 0; cc < DV / 32; ++cc) {
        uint32_t ov[32];
        ptx::tmem_ld32(taddr + cc * 32, ov);
        ptx::tmem_ld_wait();
        ptx::reg_fence(ov);
#pragma unroll
        for (int t = 0; t < 32; ++t) ov[t] = __float_as_uint(__uint_as_float(ov[t]) * alpha);
        ptx::tmem_st32(taddr + cc * 32, ov);
    }
    ptx::tmem_st_wait();
}

// Divide once: o = g u / l rounded to bf16 into orow (skipped when orow is null: a row past
// Nq), lse = (m + log2 l) * ln 2; g = 1, or 1 / (1 - p) for a dropout forward whose kept
// weights entered u unscaled.  An empty row (l == 0) gives +0.0 and -inf.  Warp-collective.
template <int DV>
__device__ __forceinline__ void write_row(uint32_t taddr, float l_run, float m_run,
                                          __nv_bfloat16 *orow, float *lse_out, float gain = 1.f) {
    const bool empty = !(l_run > 0.f);
    const float inv = empty ? 0.f : gain / l_run;
    uint4 *o4 = reinterpret_cast<uint4 *>(orow);
#pragma unroll
    for (int cc = 0; cc < DV / 32; ++cc) {
        uint32_t ov[32];
        ptx::tmem_ld32(taddr + cc * 32, ov);
        ptx::tmem_ld_wait();
        ptx::reg_fence(ov);
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 16; ++t)
            pk[t] = empty ? 0u
                          : ptx::pack_bf16x2(__uint_as_float(ov[2 * t]) * inv,
                                             __uint_as_float(ov[2 * t + 1]) * inv);
        if (o4) {
#pragma unroll
            for (int t = 0; t < 4; ++t)
                o4[cc * 4 + t] = make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
        }
    }
    if (lse_out) *lse_out = empty ? -INFINITY : (m_run + log2f(l_run)) * kLn2;
}

// As write_row, but the bf16 row goes into a shared-memory staging tile laid out like a TMA
// box of 128 rows x 64 columns per panel with the 128-byte swizzle (16-byte chunk c of row r
// at chunk c ^ (r & 7)), for a bulk-tensor store; row r's eight chunks fall in eight
// different bank groups, so a warp's writes do not conflict.
template <int DV>
__device__ __forceinline__ void stage_row(uint32_t taddr, float l_run, float m_run, uint8_t *stage,
                                          int r, float *lse_out, float gain = 1.f) {
    const bool empty = !(l_run > 0.f);
    const float inv = empty ? 0.f : gain / l_run;
#pragma unroll
    for (int cc = 0; cc < DV / 32; ++cc) {
        uint32_t ov[32];
        ptx::tmem_ld32(taddr + cc * 32, ov);
        ptx::tmem_ld_wait();
        ptx::reg_fence(ov);
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 16; ++t)
            pk[t] = empty ? 0u
                          : ptx::pack_bf16x2(__uint_as_float(ov[2 * t]) * inv,
                                             __uint_as_float(ov[2 * t + 1]) * inv);
        // columns [32 cc, 32 cc + 32) = panel cc / 2, chunks 4 (cc % 2) .. 4 (cc % 2) + 3
        uint8_t *row = stage + (cc / 2) * kPanelBytes + r * 128;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int chunk = (cc % 2) * 4 + t;
            *reinterpret_cast<uint4 *>(row + ((chunk ^ (r & 7)) * 16)) =
                make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
        }
    }
    if (lse_out) *lse_out = empty ? -INFINITY : (m_run + log2f(l_run)) * kLn2;
}

// The row's state over the keys it saw, to st[0 .. 2 + DV) (skipped when st is null: a row
// past Nq): m in natural-log units (the base-2 reference m_run times ln 2), the exponential
// sum l and the unnormalised value sum u, both measured against that reference; (-inf, 0, 0)
// for a row that saw no key.  st is 8-byte aligned; floats are stored in pairs.  Warp-collective.
template <int DV>
__device__ __forceinline__ void write_state(uint32_t taddr, float l_run, float m_run, float *st) {
    const bool empty = !(l_run > 0.f);
    float2 *s2 = reinterpret_cast<float2 *>(st);
    if (st) s2[0] = empty ? make_float2(-INFINITY, 0.f) : make_float2(m_run * kLn2, l_run);
#pragma unroll
    for (int cc = 0; cc < DV / 32; ++cc) {
        uint32_t ov[32];
        ptx::tmem_ld32(taddr + cc * 32, ov);
        ptx::tmem_ld_wait();
        ptx::reg_fence(ov);
        if (st) {
#pragma unroll
            for (int t = 0; t < 16; ++t)
                s2[1 + cc * 16 + t] = empty ? make_float2(0.f, 0.f)
                                            : make_float2(__uint_as_float(ov[2 * t]), __uint_as_float(ov[2 * t + 1]));
        }
    }
}

// The state of a row that sees no key of the kernel's: (-inf, 0, 0).
template <int DV>
__device__ __forceinline__ void write_empty_state(float *st) {
    float2 *s2 = reinterpret_cast<float2 *>(st);
    s2[0] = make_float2(-INFINITY, 0.f);
#pragma unroll
    for (int c = 0; c < DV / 2; ++c) s2[1 + c] = make_float2(0.f, 0.f);
}

// A row that sees no key at all: o = +0.0, lse = -inf (no TMEM involved).
template <int DV>
__device__ __forceinline__ void write_empty_row(__nv_bfloat16 *orow, float *lse_out) {
    uint4 *o4 = reinterpret_cast<uint4 *>(orow);
#pragma unroll
    for (int c = 0; c < DV / 8; ++c) o4[c] = make_uint4(0u, 0u, 0u, 0u);
    if (lse_out) *lse_out = -INFINITY;
}

// Zero value row `row` (all DV columns) of a V tile in shared memory.  In the 128-byte
// swizzled layout a row's 16-byte chunks are permuted only within that row's 128 bytes, so
// clearing the row's bytes in every 64-column panel clears exactly that key.
template <int DV>
__device__ __forceinline__ void zero_v_row(uint8_t *sV, int row) {
#pragma unroll
    for (int p = 0; p < DV / 64; ++p) {
        uint4 *dst = reinterpret_cast<uint4 *>(sV + p * kPanelBytes + row * 128);
#pragma unroll
        for (int t = 0; t < 8; ++t) dst[t] = make_uint4(0u, 0u, 0u, 0u);
    }
}

}  // namespace bf16fwd

// Launches the two-tile kernel (dk <= 128); defined in fwd_bf16_pair_sm103.cu.
attn_status_t launch_fwd_bf16_pair(const CUtensorMap &mq, const CUtensorMap &mk,
                                   const CUtensorMap &mv, const CUtensorMap &mo,
                                   const bf16fwd::Args &a, const bf16fwd::DropArgs &dr, int dk, int dv, bool bias,
                                   cudaStream_t s);

}  // namespace attn
