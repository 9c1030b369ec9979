// fwd_bf16_sm103.cu -- fused bf16 attention forward on the 5th-generation tensor cores.
//
// One CTA computes one 128-row query tile of one (b, h) ("How Does FlashAttention Preserve
// Global Softmax Across Tiles?", section 5: a tile of queries keeps its own per-row state
// while key/value tiles stream past; section 8: query-block parallelism).  Work items are
// numbered longest first (the last query tiles of a causal problem see the most keys), and
// the hardware hands them to SMs as SMs free up.
//
// Roles (256 threads):
//   warp 0      TMA producer: Q once, then K and V tiles into two shared-memory rings
//               (128-byte swizzled panels of 64 columns, the layout the tensor cores read).
//               A K slot is released as soon as S = Q K^T has read it and a V slot when
//               O += P V has, so loads run several tiles ahead of the tensor cores.
//   warp 1      tensor-core issuer (one thread): S_j = Q K_j^T into tensor memory (TMEM),
//               into one of three buffers so S_{j+1} is computed while the softmax works on
//               S_j, then O += P_j V_j with P_j read from TMEM.  A buffer is reused only after
//               the P V product that read it has completed (a tcgen05.commit per buffer), so
//               the next S never overwrites a P still being read.  Owns the TMEM allocation.
//   warps 4-7   softmax: thread t owns query row t (TMEM lane t), so row maxima and row sums
//               need no shuffles.  Per key tile: load the row of S from TMEM, scale (and add
//               the bias), mask in global positions, take the new maximum, form
//               p = exp(x - m) with one ex2 per element, add to l, round P to bf16 into the
//               TMEM columns S_j occupied, and signal the issuer.  At the end: o = u / l once,
//               lse = m + ln l, empty rows o = +0.0 and lse = -inf.
//
// The (m, l, u) update follows "Reducing Memory Traffic with Output Accumulation in
// FlashAttention" ("Rescaling Both Accumulators When the Maximum Increases"): when the
// maximum grows, both l and the accumulator u (here the O columns in TMEM) are multiplied by
// exp(m_old - m_new).  Rescaling is exact for any reference point shared by l and u, so a
// row keeps its reference until the tile maximum exceeds it by more than 2^8 (then the
// exponentials stay <= 256, far from fp32/bf16 overflow); rows therefore rescale O only a few
// times in a whole pass instead of at every tile.
//
// Masking (section 6): key j of sequence b is visible to row i iff j < n_b and, when causal,
// j <= i + n_b - Nq; a bias of -inf masks too.  Tiles past the last visible key are never
// loaded.  Masked logits are selected to -inf (never multiplied), so NaN stored at a masked
// position cannot reach the output; value rows past n_b inside the last tile are zeroed in
// shared memory before the P V product (0 * NaN would otherwise be NaN).
//
// Every mbarrier wait is bounded (1 s of wall time): on expiry the thread raises a CTA-wide
// abort flag and the device error word, every role leaves its loop, in-flight copies and
// tensor-core work are waited for (again bounded), TMEM is freed and the CTA exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "fwd_bf16_common.cuh"

namespace attn {
namespace {

using namespace bf16fwd;

constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr int kSBufs = 3;          // S/P buffers: TMEM columns [0,128), [128,256), [256,384)
constexpr uint32_t kTmemO = 384;   // O accumulator columns [384, 384 + dv)
constexpr int kMaxStages = 4;

// kTmaBias: the bias streams through shared memory as 32-key panels (128 rows x 32 keys fp32,
// 128-byte swizzled), four per key tile, in a ring of four filled by a producer of its own:
// a panel is refilled as soon as the softmax has read it.
constexpr int kBiasPanels = 4;
constexpr int kBiasBytes = kBiasPanels * kPanelBytes;

struct Ctrl {
    uint64_t q_full;
    uint64_t k_full[kMaxStages], k_empty[kMaxStages], v_full[kMaxStages], v_empty[kMaxStages];
    uint64_t s_full[kSBufs], p_full[kSBufs], pv_done[kSBufs];
    uint64_t o_done;     // one completion per P V product (O rescale waits on PV_{j-1})
    uint64_t o_final;    // completes once, after the last P V product
    uint64_t o_staged;   // every row of the output tile written to its shared-memory stage
    uint64_t b_full[kBiasPanels], b_empty[kBiasPanels];  // the bias panel ring
    uint64_t final_mma;
    uint32_t tmem_base;
    int abort;
};


template <int DK, int DV, bool kTmaBias = false>
struct Layout {
    static constexpr int kQBytes = (DK / 64) * kPanelBytes;
    static constexpr int kKBytes = (DK / 64) * kPanelBytes;
    static constexpr int kVBytes = (DV / 64) * kPanelBytes;
    static constexpr int kFixed = kQBytes + (kTmaBias ? kBiasBytes : 0) + 2048;
    static constexpr bool fits(int ks, int vs) { return kFixed + ks * kKBytes + vs * kVBytes <= kSmemMax; }
    // the deepest K and V rings that fit next to Q (and the bias panels); a V tile waits for
    // the P V product two tiles back, so V gets the second stage first
    static constexpr int kKStages = fits(4, 4) ? 4 : fits(3, 3) ? 3 : fits(2, 3) ? 2 : fits(2, 2) ? 2 : 1;
    static constexpr int kVStages = fits(4, 4) ? 4 : fits(3, 3) ? 3 : fits(2, 3) ? 3 : fits(2, 2) ? 2
                                  : fits(1, 2) ? 2 : 1;
    static constexpr int kKOff = kQBytes;                       // K ring
    static constexpr int kVOff = kQBytes + kKStages * kKBytes;  // V ring
    static constexpr int kBOff = kVOff + kVStages * kVBytes;    // bias panels
    static constexpr int kDataBytes = kBOff + (kTmaBias ? kBiasBytes : 0);
    static constexpr int kBytes = kDataBytes + (int)sizeof(Ctrl) + 1024;  // + alignment slack
    static_assert(kBytes <= kSmemMax, "shared memory budget");
};

// With per-sequence key lengths the work of a query tile depends on its sequence, so for up to
// 32 sequences the CTAs take the sequences in order of decreasing length (ties by index), the
// longest work first.  Warp-collective: lane t holds sequence t's length, counts the lanes
// ahead of it, and the sequence of rank R is the lane whose count is R.
__device__ __forceinline__ int batch_by_rank(const Args &a, int R) {
    const int lane = threadIdx.x & 31;
    const int len = lane < a.B ? seq_len(a, lane, false) : -1;
    int rank = 0;
#pragma unroll
    for (int o = 0; o < 32; ++o) {
        const int lo = __shfl_sync(0xffffffffu, len, o);
        rank += (lo > len) || (lo == len && o < lane);
    }
    return __ffs(__ballot_sync(0xffffffffu, lane < a.B && rank == R)) - 1;
}

template <int DK, int DV, bool kBias, bool kTmaBias>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_o, const Args a) {
    static_assert(kBias || !kTmaBias, "a staged bias needs a bias");
    using L = Layout<DK, DV, kTmaBias>;
    constexpr int KS = L::kKStages, VS = L::kVStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t *sQ = smem;
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem + L::kDataBytes);
    volatile int *abort = &ctrl->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // launched as a programmatic dependent of the previous kernel in the stream: nothing in
    // global memory is read before that kernel has completed
    ptx::grid_dep_wait();
    // work items longest first: later query tiles (causal ones see more keys) first, or, with
    // per-sequence key lengths, longer sequences first
    int qt, b, h;
    if (a.kv_lens && a.B <= 32) {
        const int per_b = a.H * a.n_items;
        const int rem = (int)(blockIdx.x % per_b);
        qt = a.n_items - 1 - rem / a.H;
        h = rem % a.H;
        b = batch_by_rank(a, (int)(blockIdx.x / per_b));
    } else {
        const int bhn = a.B * a.H;
        qt = a.n_items - 1 - (int)(blockIdx.x / bhn);
        const int bh = (int)(blockIdx.x % bhn);
        b = bh / a.H;
        h = bh % a.H;
    }
    const int q0 = qt * BQ;

    const int n = seq_len(a, b, threadIdx.x == 0 && qt == 0 && h == 0);
    const int shift = n - a.Nq;  // causal: key j visible to row i iff j <= i + shift
    const int n_tiles = kv_tiles(a, q0, n);

    if (n_tiles == 0) {  // every row of this tile is empty: o = +0.0, lse = -inf
        if (warp >= 4) {
            const int i = q0 + (int)threadIdx.x - 128;
            if (i < a.Nq)
                write_empty_row<DV>(a.o + b * a.os0 + (long long)i * a.os1 + h * a.os2,
                                    a.lse ? a.lse + ((long long)b * a.H + h) * a.Nq + i : nullptr);
        }
        return;
    }

    if (threadIdx.x == 0) {
        ptx::mbar_init(&ctrl->q_full, 1);
        for (int s = 0; s < KS; ++s) {
            ptx::mbar_init(&ctrl->k_full[s], 1);
            ptx::mbar_init(&ctrl->k_empty[s], 1);
        }
        for (int s = 0; s < VS; ++s) {
            ptx::mbar_init(&ctrl->v_full[s], 1);
            ptx::mbar_init(&ctrl->v_empty[s], 1);
        }
        for (int s = 0; s < kSBufs; ++s) {
            ptx::mbar_init(&ctrl->s_full[s], 1);
            ptx::mbar_init(&ctrl->p_full[s], 128);
            ptx::mbar_init(&ctrl->pv_done[s], 1);
        }
        ptx::mbar_init(&ctrl->o_done, 1);
        ptx::mbar_init(&ctrl->o_final, 1);
        ptx::mbar_init(&ctrl->o_staged, 128);
        for (int s = 0; s < kBiasPanels; ++s) {
            ptx::mbar_init(&ctrl->b_full[s], 1);
            ptx::mbar_init(&ctrl->b_empty[s], 128);
        }
        ptx::mbar_init(&ctrl->final_mma, 1);
        ctrl->abort = 0;
        ptx::fence_mbar_init();
    }
    if (threadIdx.x == 0) {
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
        ptx::prefetch_tmap(&tm_o);
        if (kTmaBias) ptx::prefetch_tmap(&tm_b);
        // this thread produces Q and K: both start loading before the tensor-memory
        // allocation and the block barrier
        ptx::mbar_arrive_expect_tx(&ctrl->q_full, L::kQBytes);
#pragma unroll
        for (int p = 0; p < DK / 64; ++p)
            ptx::tma_load_4d(sQ + p * kPanelBytes, &tm_q, &ctrl->q_full, p * 64, q0, h, b);
        ptx::mbar_arrive_expect_tx(&ctrl->k_full[0], L::kKBytes);
#pragma unroll
        for (int p = 0; p < DK / 64; ++p)
            ptx::tma_load_4d(smem + L::kKOff + p * kPanelBytes, &tm_k, &ctrl->k_full[0], p * 64, 0, h, b);
    }
    if (warp == 1) {
        ptx::tmem_alloc(&ctrl->tmem_base, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    // the next kernel in the stream may be scheduled once every CTA of this grid has started
    ptx::launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer: Q, K
        if (lane == 0) {
            int last_k = 0;  // last tile whose copy was issued (Q and K_0: issued above)
            for (int j = 1; j < n_tiles; ++j) {
                const int st = j % KS;
                if (j >= KS && !ptx::mbar_wait(&ctrl->k_empty[st], ((j / KS) - 1) & 1, abort, a.flags,
                                               kFlagWaitTimeout, kWaitLimitNs))
                    break;
                uint8_t *sK = smem + L::kKOff + st * L::kKBytes;
                ptx::mbar_arrive_expect_tx(&ctrl->k_full[st], L::kKBytes);
#pragma unroll
                for (int p = 0; p < DK / 64; ++p)
                    ptx::tma_load_4d(sK + p * kPanelBytes, &tm_k, &ctrl->k_full[st], p * 64, j * BK, h, b);
                last_k = j;
            }
            if (*abort) {  // let copies still in flight land before the CTA exits
                ptx::mbar_wait_quiet(&ctrl->q_full, 0, kWaitLimitNs);
                for (int j = max(0, last_k - KS + 1); j <= last_k; ++j)
                    ptx::mbar_wait_quiet(&ctrl->k_full[j % KS], (j / KS) & 1, kWaitLimitNs);
            }
        }
    } else if (warp == 3) {
        // ------------------------------------------------------------ TMA producer: V
        // (a thread of its own, so that a V tile waiting for its slot never holds up K)
        if (lane == 0) {
            int last_v = -1;
            for (int j = 0; j < n_tiles; ++j) {
                const int st = j % VS;
                if (j >= VS && !ptx::mbar_wait(&ctrl->v_empty[st], ((j / VS) - 1) & 1, abort, a.flags,
                                               kFlagWaitTimeout, kWaitLimitNs))
                    break;
                uint8_t *sV = smem + L::kVOff + st * L::kVBytes;
                ptx::mbar_arrive_expect_tx(&ctrl->v_full[st], L::kVBytes);
#pragma unroll
                for (int p = 0; p < DV / 64; ++p)
                    ptx::tma_load_4d(sV + p * kPanelBytes, &tm_v, &ctrl->v_full[st], p * 64, j * BK, h, b);
                last_v = j;
            }
            if (*abort)
                for (int j = max(0, last_v - VS + 1); j <= last_v; ++j)
                    ptx::mbar_wait_quiet(&ctrl->v_full[j % VS], (j / VS) & 1, kWaitLimitNs);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ tensor-core issuer
        if (lane == 0) {
            constexpr uint32_t kIdS = ptx::idesc_bf16_f32(BQ, BK, false);
            constexpr uint32_t kIdO = ptx::idesc_bf16_f32(BQ, DV, true);
            const uint32_t q_addr = ptx::smem_u32(sQ);
            bool ok = ptx::mbar_wait(&ctrl->q_full, 0, abort, a.flags, kFlagWaitTimeout, kWaitLimitNs);
            auto issue_s = [&](int j) -> bool {
                const int st = j % KS, buf = j % kSBufs;
                // buffer reuse: the P V product of tile j - 3 (which read this buffer) is done
                if (j >= kSBufs &&
                    !ptx::mbar_wait(&ctrl->pv_done[buf], ((j / kSBufs) - 1) & 1, abort, a.flags,
                                    kFlagWaitTimeout, kWaitLimitNs))
                    return false;
                if (!ptx::mbar_wait(&ctrl->k_full[st], (j / KS) & 1, abort, a.flags,
                                    kFlagWaitTimeout, kWaitLimitNs))
                    return false;
                ptx::tc_fence_after();
                const uint32_t k_addr = ptx::smem_u32(smem + L::kKOff + st * L::kKBytes);
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint32_t off = (kk / 4) * kPanelBytes + (kk % 4) * 32;
                    ptx::mma_ss(tmem + buf * BK, ptx::sdesc_sw128(q_addr + off, 16, 1024),
                                ptx::sdesc_sw128(k_addr + off, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
                }
                ptx::mma_commit(&ctrl->s_full[buf]);
                ptx::mma_commit(&ctrl->k_empty[st]);
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int j = 0; ok && j < n_tiles; ++j) {
                if (j + 1 < n_tiles && !issue_s(j + 1)) break;
                const int st = j % VS, buf = j % kSBufs;
                if (!ptx::mbar_wait(&ctrl->p_full[buf], (j / kSBufs) & 1, abort, a.flags,
                                    kFlagWaitTimeout, kWaitLimitNs))
                    break;
                if (!ptx::mbar_wait(&ctrl->v_full[st], (j / VS) & 1, abort, a.flags,
                                    kFlagWaitTimeout, kWaitLimitNs))
                    break;
                ptx::tc_fence_after();
                const uint32_t v_addr = ptx::smem_u32(smem + L::kVOff + st * L::kVBytes);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    // P: bf16 pairs packed in TMEM columns (8 columns per 16 keys);
                    // V: MN-major (dv contiguous), 8-key groups 1024 B apart, 64-column
                    // panels kPanelBytes apart.
                    ptx::mma_ts(tmem + kTmemO, tmem + buf * BK + kk * 8,
                                ptx::sdesc_sw128(v_addr + kk * 16 * 128, kPanelBytes, 1024), kIdO,
                                (j > 0 || kk > 0) ? 1u : 0u);
                }
                ptx::mma_commit(&ctrl->o_done);
                ptx::mma_commit(&ctrl->pv_done[buf]);
                ptx::mma_commit(&ctrl->v_empty[st]);
                if (j == n_tiles - 1) ptx::mma_commit(&ctrl->o_final);
            }
            // all tensor-core work of this CTA done before TMEM is released
            ptx::mma_commit(&ctrl->final_mma);
            if (!ptx::mbar_wait_quiet(&ctrl->final_mma, 0, kWaitLimitNs)) atomicOr(a.flags, kFlagWaitTimeout);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ bias producer
        if (kTmaBias && lane == 0) {
            // panel q of the key tiles (32 keys each, four per tile) into ring slot q % 6, as
            // soon as the softmax has read what the slot held
            const int n_panels = 4 * n_tiles;
            int last = -1;
            for (int q = 0; q < n_panels; ++q) {
                const int sl = q % kBiasPanels;
                if (q >= kBiasPanels && !ptx::mbar_wait(&ctrl->b_empty[sl], ((q / kBiasPanels) - 1) & 1, abort,
                                                        a.flags, kFlagWaitTimeout, kWaitLimitNs))
                    break;
                ptx::mbar_arrive_expect_tx(&ctrl->b_full[sl], kPanelBytes);
                ptx::tma_load_4d(smem + L::kBOff + sl * kPanelBytes, &tm_b, &ctrl->b_full[sl],
                                 (q >> 2) * BK + 32 * (q & 3), q0, h, b);
                last = q;
            }
            if (*abort)  // let copies still in flight land before the CTA exits
                for (int q = max(0, last - kBiasPanels + 1); q <= last; ++q)
                    ptx::mbar_wait_quiet(&ctrl->b_full[q % kBiasPanels], (q / kBiasPanels) & 1, kWaitLimitNs);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax warpgroup
        const int r = (int)threadIdx.x - 128;  // row in tile == TMEM lane
        const int i = q0 + r;
        const uint32_t lane_addr = tmem + ((uint32_t)((warp - 4) * 32) << 16);
        const float c = a.scale_log2;
        const float *bias_row = nullptr;
        if (kBias && i < a.Nq) bias_row = a.bias + b * a.bs0 + h * a.bs1 + (long long)i * a.bs2;
        const bool bias_vec = (reinterpret_cast<uintptr_t>(bias_row) & 15u) == 0;  // float4 loads
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        // every lane waits; the warp goes on only if all lanes succeeded (tcgen05.ld/st and
        // the vote below are warp-collective, so the lanes must not part ways)
        auto wait_warp = [&](uint64_t *bar, uint32_t parity) -> bool {
            const bool w = ptx::mbar_wait(bar, parity, abort, a.flags, kFlagWaitTimeout, kWaitLimitNs);
            return __all_sync(0xffffffffu, w);
        };

        float x[BK];  // with a bias: the next tile's bias, loaded ahead
        if (kBias && !kTmaBias) load_bias(bias_row, bias_vec, 0, n, x);
        for (int j = 0; j < n_tiles; ++j) {
            const int buf = j % kSBufs, kv0 = j * BK;
            if (kTmaBias) {  // this tile's bias row from its four staged panels, freeing each
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const int q = 4 * j + p, sl = q % kBiasPanels;
                    if (!wait_warp(&ctrl->b_full[sl], (q / kBiasPanels) & 1)) {
                        ok = false;
                        break;
                    }
                    read_bias_panel(smem + L::kBOff + sl * kPanelBytes, r, p, x);
                    ptx::mbar_arrive(&ctrl->b_empty[sl]);
                }
                if (!ok) break;
            }
            if (!wait_warp(&ctrl->s_full[buf], (j / kSBufs) & 1)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            if (kBias) load_s_row_bias(lane_addr + buf * BK, c, x);
            else load_s_row(lane_addr + buf * BK, x);
            const bool need_mask = (kv0 + BK > n) || (a.causal && kv0 + BK - 1 > q0 + shift);
            const int lim = a.causal ? min(n, i + shift + 1) : n;  // keys < lim visible
            const float mt = tile_logits<kBias>(x, c, kv0, need_mask, lim);
            bool rescale;
            const float alpha = update_max(mt, m_run, rescale);
            const float lsum = tile_exp<kBias>(x, c, m_run);
            l_run = fmaf(alpha, l_run, lsum);

            // u <- alpha * u: rescale this warp's O rows once PV_{j-1} has landed.  (The
            // commit behind s_full for S_j covers PV_{j-2}, so o_done is in phase j-1 or j
            // here and its parity is unambiguous.)
            if (__any_sync(0xffffffffu, rescale)) {
                if (!wait_warp(&ctrl->o_done, (j - 1) & 1)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                scale_o<DV>(lane_addr + kTmemO, alpha);
            }

            // value rows past n inside this tile (still in bounds) may hold anything: zero them
            if (kv0 + BK > n && n < a.Nk) {
                const int st = j % VS;
                if (!wait_warp(&ctrl->v_full[st], (j / VS) & 1)) {
                    ok = false;
                    break;
                }
                if (kv0 + r >= n && kv0 + r < a.Nk) zero_v_row<DV>(smem + L::kVOff + st * L::kVBytes, r);
                ptx::fence_proxy_async_smem();
            }

            // P (bf16) into the TMEM columns that held S_j
            store_p(lane_addr + buf * BK, x);
            ptx::tc_fence_before();
            ptx::mbar_arrive(&ctrl->p_full[buf]);
            if (kBias && !kTmaBias && j + 1 < n_tiles) load_bias(bias_row, bias_vec, kv0 + BK, n, x);
        }

        // epilogue: o = u / l once, lse = m + ln l; empty rows o = +0.0, lse = -inf.  The rows
        // go into Q's shared memory (its last reader, the last S product, completed before
        // o_final) in the swizzled box layout, and one thread stores the tile with TMA (rows
        // past Nq are not written) once every row is staged
        if (ok && wait_warp(&ctrl->o_final, 0)) {
            ptx::tc_fence_after();
            stage_row<DV>(lane_addr + kTmemO, l_run, m_run, sQ, r,
                          (a.lse && i < a.Nq) ? a.lse + ((long long)b * a.H + h) * a.Nq + i : nullptr);
            ptx::tc_fence_before();
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&ctrl->o_staged);
            if (r == 0 && ptx::mbar_wait(&ctrl->o_staged, 0, abort, a.flags, kFlagWaitTimeout, kWaitLimitNs)) {
#pragma unroll
                for (int p = 0; p < DV / 64; ++p) ptx::tma_store_4d(&tm_o, sQ + p * kPanelBytes, p * 64, q0, h, b);
                ptx::bulk_commit();
                ptx::bulk_wait_read();
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------- host side

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 4-D map over a [B, N, H, d] bf16 tensor with element strides s (b, n, h); box 64 x 128.
attn_status_t encode(CUtensorMap *m, const void *ptr, int64_t B, int64_t N, int64_t H, int64_t d,
                     const int64_t s[3], const char *name) {
    auto enc = get_encoder();
    if (!enc) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    auto bstride = [](int64_t st, int64_t size) -> cuuint64_t {
        return size <= 1 ? 16u : (cuuint64_t)(st * 2);  // stride of a size-1 dim is unused
    };
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[3] = {bstride(s[1], N), bstride(s[2], H), bstride(s[0], B)};
    cuuint32_t box[4] = {64, 128, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ATTN_ERR_INVALID_ARG, "TMA descriptor for %s rejected (CUresult %d)", name, (int)r);
    return ATTN_OK;
}

namespace {

// 4-D map over the fp32 bias [B, H, Nq, Nk] (key stride 1, element strides bs: b, h, i);
// box 32 keys x 128 rows, 128-byte swizzle.  Returns false when the bias does not meet the
// TMA rules (16-byte aligned base, strides that are non-zero multiples of 16 bytes).
bool encode_bias(CUtensorMap *m, const attn_fwd_params_t &p) {
    auto enc = get_encoder();
    if (!enc || (reinterpret_cast<uintptr_t>(p.bias) & 15u)) return false;
    const int64_t sizes[3] = {p.B, p.H, p.Nq};
    for (int t = 0; t < 3; ++t)
        if (sizes[t] > 1 && (p.bias_stride[t] <= 0 || p.bias_stride[t] % 4)) return false;
    auto bstride = [](int64_t st, int64_t size) -> cuuint64_t {
        return size <= 1 ? 16u : (cuuint64_t)(st * 4);
    };
    cuuint64_t dims[4] = {(cuuint64_t)p.Nk, (cuuint64_t)p.Nq, (cuuint64_t)p.H, (cuuint64_t)p.B};
    cuuint64_t strides[3] = {bstride(p.bias_stride[2], p.Nq), bstride(p.bias_stride[1], p.H),
                             bstride(p.bias_stride[0], p.B)};
    cuuint32_t box[4] = {32, 128, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(p.bias), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DK, int DV, bool kBias, bool kTmaBias>
attn_status_t launch_t(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                       const CUtensorMap &mb, const CUtensorMap &mo, const Args &a, unsigned grid,
                       cudaStream_t s) {
    int smem = Layout<DK, DV, kTmaBias>::kBytes;
    if (smem < 116 * 1024) smem = 116 * 1024;  // one CTA per SM: it owns all 512 TMEM columns
    auto kern = fwd_bf16_kernel<DK, DV, kBias, kTmaBias>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    e = launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, mq, mk, mv, mb, mo, a);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "fwd_bf16 launch: %s", cudaGetErrorString(e));
    return ATTN_OK;
}

template <bool kBias, bool kTmaBias>
attn_status_t dispatch(int dk, int dv, const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                       const CUtensorMap &mb, const CUtensorMap &mo, const Args &a, unsigned grid,
                       cudaStream_t s) {
    if (dk == 192 && dv == 128) return launch_t<192, 128, kBias, kTmaBias>(mq, mk, mv, mb, mo, a, grid, s);
    if (dk == 192 && dv == 64) return launch_t<192, 64, kBias, kTmaBias>(mq, mk, mv, mb, mo, a, grid, s);
    if constexpr (kTmaBias) {  // dk <= 128 with a staged bias (the output tile fits in Q's buffer)
        if (dk == 128 && dv == 128) return launch_t<128, 128, true, true>(mq, mk, mv, mb, mo, a, grid, s);
        if (dk == 128 && dv == 64) return launch_t<128, 64, true, true>(mq, mk, mv, mb, mo, a, grid, s);
        if (dk == 64 && dv == 64) return launch_t<64, 64, true, true>(mq, mk, mv, mb, mo, a, grid, s);
    }
    return fail(ATTN_ERR_UNSUPPORTED, "no one-tile bf16 kernel for dk=%d dv=%d", dk, dv);
}

}  // namespace

attn_status_t launch_fwd_bf16(const attn_fwd_params_t &p, cudaStream_t s) {
    for (int t = 0; t < 3; ++t) {
        if ((p.q_stride[t] == 0 && (t == 0 ? p.B : t == 1 ? p.Nq : p.H) > 1) ||
            (p.Nk > 0 && ((p.k_stride[t] == 0 || p.v_stride[t] == 0) && (t == 0 ? p.B : t == 1 ? p.Nk : p.H) > 1)))
            return fail(ATTN_ERR_UNSUPPORTED, "bfloat16 path needs non-zero q/k/v strides");
    }
    CUtensorMap mq, mk, mv;
    attn_status_t st = encode(&mq, p.q, p.B, p.Nq, p.H, p.dk, p.q_stride, "q");
    if (st) return st;
    if (p.Nk > 0) {
        if ((st = encode(&mk, p.k, p.B, p.Nk, p.H, p.dk, p.k_stride, "k"))) return st;
        if ((st = encode(&mv, p.v, p.B, p.Nk, p.H, p.dv, p.v_stride, "v"))) return st;
    } else {
        mk = mq;  // never read: with no keys every tile is empty
        mv = mq;
    }
    // dk <= 128: two query tiles per CTA; dk = 192: one (two would not fit in shared memory).
    // With a bias that TMA can stage (and no dropout), dk >= dv <= 128 also takes the one-tile
    // kernel: its bias streams through shared memory in panels, which the two-tile kernel has
    // no room for (it reads each row's bias into registers)
    CUtensorMap mb = mq;  // read only by kernels that stage the bias
    const bool staged_bias = p.bias && p.Nk > 0 && encode_bias(&mb, p);
    const bool drop = p.dropout_mask || p.dropout_rng == 1;
    const bool pair = p.dk <= 128 && !(staged_bias && !drop && p.dk >= p.dv);
    Args a;
    a.B = (int)p.B; a.H = (int)p.H; a.Nq = (int)p.Nq; a.Nk = (int)p.Nk; a.causal = p.causal;
    a.n_items = (int)((p.Nq + (pair ? 2 * BQ : BQ) - 1) / (pair ? 2 * BQ : BQ));
    fill_divisors(a);
    a.scale_log2 = p.scale * kLog2e;
    a.o = static_cast<__nv_bfloat16 *>(p.o);
    a.os0 = p.o_stride[0]; a.os1 = p.o_stride[1]; a.os2 = p.o_stride[2];
    a.lse = p.lse;
    a.bias = p.bias; a.bs0 = p.bias_stride[0]; a.bs1 = p.bias_stride[1]; a.bs2 = p.bias_stride[2];
    a.kv_lens = p.kv_lens;
    DropArgs dr{};
    fill_dropout(dr, p);
    dr.key_off = 0;
    dr.Nk_tot = (int)p.Nk;
    dr.part = nullptr;
    a.flags = device_flags();
    if (!a.flags) return fail(ATTN_ERR_CUDA, "could not resolve the device error word");
    CUtensorMap mo;
    if ((st = encode(&mo, p.o, p.B, p.Nq, p.H, p.dv, p.o_stride, "o"))) return st;
    if (pair) return launch_fwd_bf16_pair(mq, mk, mv, mo, a, dr, (int)p.dk, (int)p.dv, p.bias != nullptr, s);
    if (dr.dmask || dr.rng) return fail(ATTN_ERR_UNSUPPORTED, "dropout with dk = %lld is not built", (long long)p.dk);
    const long long grid = (long long)a.n_items * p.B * p.H;
    if (grid > 0x7fffffffLL) return fail(ATTN_ERR_UNSUPPORTED, "too many query tiles");
    if (staged_bias) return dispatch<true, true>((int)p.dk, (int)p.dv, mq, mk, mv, mb, mo, a, (unsigned)grid, s);
    if (p.bias) return dispatch<true, false>((int)p.dk, (int)p.dv, mq, mk, mv, mb, mo, a, (unsigned)grid, s);
    return dispatch<false, false>((int)p.dk, (int)p.dv, mq, mk, mv, mb, mo, a, (unsigned)grid, s);
}

attn_status_t launch_fwd_bf16_partial(const attn_fwd_params_t &p, int64_t key_offset, int64_t Nk_total,
                                      float *partials, cudaStream_t s) {
    for (int t = 0; t < 3; ++t) {
        if ((p.q_stride[t] == 0 && (t == 0 ? p.B : t == 1 ? p.Nq : p.H) > 1) ||
            (p.Nk > 0 && ((p.k_stride[t] == 0 || p.v_stride[t] == 0) && (t == 0 ? p.B : t == 1 ? p.Nk : p.H) > 1)))
            return fail(ATTN_ERR_UNSUPPORTED, "bfloat16 path needs non-zero q/k/v strides");
    }
    CUtensorMap mq, mk, mv;
    attn_status_t st = encode(&mq, p.q, p.B, p.Nq, p.H, p.dk, p.q_stride, "q");
    if (st) return st;
    if (p.Nk > 0) {
        if ((st = encode(&mk, p.k, p.B, p.Nk, p.H, p.dk, p.k_stride, "k"))) return st;
        if ((st = encode(&mv, p.v, p.B, p.Nk, p.H, p.dv, p.v_stride, "v"))) return st;
    } else {
        mk = mq;  // never read: with no keys every tile is empty
        mv = mq;
    }
    Args a;
    a.B = (int)p.B; a.H = (int)p.H; a.Nq = (int)p.Nq; a.Nk = (int)p.Nk; a.causal = p.causal;
    a.n_items = (int)((p.Nq + 2 * BQ - 1) / (2 * BQ));
    fill_divisors(a);
    a.scale_log2 = p.scale * kLog2e;
    a.o = nullptr;
    a.os0 = a.os1 = a.os2 = 0;
    a.lse = nullptr;
    a.bias = p.bias; a.bs0 = p.bias_stride[0]; a.bs1 = p.bias_stride[1]; a.bs2 = p.bias_stride[2];
    a.kv_lens = p.kv_lens;
    DropArgs dr{};
    dr.inv_keep = 1.f;
    dr.key_off = (int)key_offset;
    dr.Nk_tot = (int)Nk_total;
    dr.part = partials;
    a.flags = device_flags();
    if (!a.flags) return fail(ATTN_ERR_CUDA, "could not resolve the device error word");
    // the output map is never used by the partial-state kernel
    return launch_fwd_bf16_pair(mq, mk, mv, mq, a, dr, (int)p.dk, (int)p.dv, p.bias != nullptr, s);
}

}  // namespace attn
