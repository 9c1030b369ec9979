// fwd_bf16_pair_sm103.cu -- bf16 attention forward, two 128-row query tiles per CTA.
//
// A CTA owns 256 consecutive query rows of one (b, h): tile A (rows q0..q0+127) and tile B
// (rows q0+128..q0+255).  Every K and V tile brought into shared memory serves both query
// tiles, which halves the key/value traffic per FLOP against one tile per CTA, and the two
// tiles' softmax warpgroups take turns with the tensor cores: while one warpgroup turns its
// S into P, the tensor cores compute the other tile's products ("How Does FlashAttention
// Preserve Global Softmax Across Tiles?", section 5: every query row keeps its own state;
// section 8: query-block parallelism).  Work items are numbered longest first.
//
// Roles (384 threads = 3 warpgroups):
//   warp 0       TMA producer: Q_A and Q_B once, then K and V tiles into two rings.
//   warp 1       tensor-core issuer (one thread); owns the 512 TMEM columns:
//                  S_A/P_A [0,128)  S_B/P_B [128,256)  O_A [256,384)  O_B [384,512).
//                Per key tile j: O_A += P_A V_j, then S_A(j+1) = Q_A K_{j+1}^T into the
//                same columns (tcgen05.mma operations from one thread execute in issue
//                order, so the product reads P_A before the next S overwrites it); then B.
//   warps 4-7    softmax of tile A, one thread per query row (its TMEM lane).
//   warps 8-11   softmax of tile B.
// The commit behind S_X(j+1) covers P_X(j) V_j, so a softmax thread that sees S_X(j+1) may
// rescale O_X directly: no product is writing it.
//
// The per-row steps (mask, maximum, exponentials, rescale, one division at the end) are those
// of fwd_bf16_common.cuh; masking and the empty-row policy are as in the one-tile kernel.
#include "fwd_bf16_common.cuh"

namespace attn {
namespace {

using namespace bf16fwd;

constexpr int kThreads = 384;
// Registers: launched at 168 per thread (384 x 168 = 64512); the load/issue warpgroup gives
// most of its share to the two softmax warpgroups: 128 x 56 + 256 x 224 = 64512.
constexpr uint32_t kRegsIssue = 56, kRegsSoftmax = 224;
static_assert(128 * kRegsIssue + 256 * kRegsSoftmax <= kThreads * 168, "register split");
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxStages = 4;

struct Ctrl {
    uint64_t q_full;
    uint64_t k_full[kMaxStages], k_empty[kMaxStages], v_full[kMaxStages], v_empty[kMaxStages];
    uint64_t s_full[2], p_full[2], o_final[2], o_staged[2];
    uint64_t final_mma;
    uint32_t tmem_base;
    int abort;
};

template <int DK, int DV>
struct Layout {
    static constexpr int kQBytes = (DK / 64) * kPanelBytes;  // one query tile
    static constexpr int kKBytes = (DK / 64) * kPanelBytes;
    static constexpr int kVBytes = (DV / 64) * kPanelBytes;
    static constexpr int kFixed = 2 * kQBytes + (int)sizeof(Ctrl) + 1024;
    // as many K stages as fit with 2 V stages (at most 4), then V stages likewise
    static constexpr int kKStages =
        (kFixed + 4 * kKBytes + 2 * kVBytes <= kSmemMax) ? 4
        : (kFixed + 3 * kKBytes + 2 * kVBytes <= kSmemMax) ? 3 : 2;
    static constexpr int kVStages =
        (kFixed + kKStages * kKBytes + 4 * kVBytes <= kSmemMax) ? 4
        : (kFixed + kKStages * kKBytes + 3 * kVBytes <= kSmemMax) ? 3 : 2;
    static constexpr int kKOff = 2 * kQBytes;
    static constexpr int kVOff = kKOff + kKStages * kKBytes;
    static constexpr int kDataBytes = kVOff + kVStages * kVBytes;
    static constexpr int kBytes = kDataBytes + (int)sizeof(Ctrl) + 1024;
    static_assert(kBytes <= kSmemMax, "shared memory budget");
};

template <int DK, int DV, bool kBias>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_o, const Args a) {
    using L = Layout<DK, DV>;
    constexpr int KS = L::kKStages, VS = L::kVStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem + L::kDataBytes);
    volatile int *abort = &ctrl->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bhn = a.B * a.H;
    const int item = a.n_items - 1 - (int)(blockIdx.x / bhn);  // longest first
    const int bh = (int)(blockIdx.x % bhn), b = bh / a.H, h = bh % a.H;
    const int q0 = item * 2 * BQ;
    const int n = seq_len(a, b, threadIdx.x == 0 && item == 0 && h == 0);
    const int shift = n - a.Nq;
    const int nA = kv_tiles(a, q0, n), nB = kv_tiles(a, q0 + BQ, n);
    const int nmax = max(nA, nB);

    // softmax thread's row (warps 4..11) and tile
    const int X = (warp >= 8) ? 1 : 0;
    const int r = (int)threadIdx.x - 128 - X * BQ;
    const int i = q0 + X * BQ + r;
    const int nX = X ? nB : nA;

    if (nmax == 0) {  // every row of both tiles is empty
        if (warp >= 4 && i < a.Nq)
            write_empty_row<DV>(a.o + b * a.os0 + (long long)i * a.os1 + h * a.os2,
                                a.lse ? a.lse + ((long long)b * a.H + h) * a.Nq + i : nullptr);
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
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(&ctrl->s_full[t], 1);
            ptx::mbar_init(&ctrl->p_full[t], BQ);
            ptx::mbar_init(&ctrl->o_final[t], 1);
            ptx::mbar_init(&ctrl->o_staged[t], BQ);
        }
        ptx::mbar_init(&ctrl->final_mma, 1);
        ctrl->abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
        ptx::prefetch_tmap(&tm_o);
    }
    if (warp == 1) {
        ptx::tmem_alloc(&ctrl->tmem_base, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;

    if (warp < 4) {
      ptx::regs_dec<kRegsIssue>();
      if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(&ctrl->q_full, 2 * L::kQBytes);
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int p = 0; p < DK / 64; ++p)
                    ptx::tma_load_4d(smem + t * L::kQBytes + p * kPanelBytes, &tm_q, &ctrl->q_full,
                                     p * 64, q0 + t * BQ, h, b);
            int last_k = -1, last_v = -1;
            for (int j = 0; j < nmax; ++j) {
                const int ks = j % KS, vs = j % VS;
                if (j >= KS && !ptx::mbar_wait(&ctrl->k_empty[ks], ((j / KS) - 1) & 1, abort,
                                               a.flags, kFlagWaitTimeout, kWaitLimitNs))
                    break;
                uint8_t *sK = smem + L::kKOff + ks * L::kKBytes;
                ptx::mbar_arrive_expect_tx(&ctrl->k_full[ks], L::kKBytes);
#pragma unroll
                for (int p = 0; p < DK / 64; ++p)
                    ptx::tma_load_4d(sK + p * kPanelBytes, &tm_k, &ctrl->k_full[ks], p * 64, j * BK, h, b);
                last_k = j;
                if (j >= VS && !ptx::mbar_wait(&ctrl->v_empty[vs], ((j / VS) - 1) & 1, abort,
                                               a.flags, kFlagWaitTimeout, kWaitLimitNs))
                    break;
                uint8_t *sV = smem + L::kVOff + vs * L::kVBytes;
                ptx::mbar_arrive_expect_tx(&ctrl->v_full[vs], L::kVBytes);
#pragma unroll
                for (int p = 0; p < DV / 64; ++p)
                    ptx::tma_load_4d(sV + p * kPanelBytes, &tm_v, &ctrl->v_full[vs], p * 64, j * BK, h, b);
                last_v = j;
            }
            if (*abort) {  // let copies still in flight land before the CTA exits
                ptx::mbar_wait_quiet(&ctrl->q_full, 0, kWaitLimitNs);
                for (int j = max(0, last_k - KS + 1); j <= last_k; ++j)
                    ptx::mbar_wait_quiet(&ctrl->k_full[j % KS], (j / KS) & 1, kWaitLimitNs);
                for (int j = max(0, last_v - VS + 1); j <= last_v; ++j)
                    ptx::mbar_wait_quiet(&ctrl->v_full[j % VS], (j / VS) & 1, kWaitLimitNs);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ tensor-core issuer
        if (lane == 0) {
            constexpr uint32_t kIdS = ptx::idesc_bf16_f32(BQ, BK, false);
            constexpr uint32_t kIdO = ptx::idesc_bf16_f32(BQ, DV, true);
            const uint32_t q_addr = ptx::smem_u32(smem);
            auto wait = [&](uint64_t *bar, uint32_t parity) {
                return ptx::mbar_wait(bar, parity, abort, a.flags, kFlagWaitTimeout, kWaitLimitNs);
            };
            // S_t(j) = Q_t K_j^T into TMEM columns [t*128, t*128 + 128)
            auto issue_s = [&](int t, int j) -> bool {
                const int ks = j % KS;
                if (!wait(&ctrl->k_full[ks], (j / KS) & 1)) return false;
                ptx::tc_fence_after();
                const uint32_t k_addr = ptx::smem_u32(smem + L::kKOff + ks * L::kKBytes);
                const uint32_t qa = q_addr + t * L::kQBytes;
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint32_t off = (kk / 4) * kPanelBytes + (kk % 4) * 32;
                    ptx::mma_ss(tmem + t * BQ, ptx::sdesc_sw128(qa + off, 16, 1024),
                                ptx::sdesc_sw128(k_addr + off, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
                }
                ptx::mma_commit(&ctrl->s_full[t]);
                return true;
            };
            bool ok = wait(&ctrl->q_full, 0);
            if (ok && nA > 0) ok = issue_s(0, 0);
            if (ok && nB > 0) ok = issue_s(1, 0);
            if (ok) ptx::mma_commit(&ctrl->k_empty[0]);
            for (int j = 0; ok && j < nmax; ++j) {
                const int vs = j % VS;
                for (int t = 0; ok && t < 2; ++t) {
                    const int nt = t ? nB : nA;
                    if (j >= nt) continue;
                    if (!wait(&ctrl->p_full[t], j & 1) || !wait(&ctrl->v_full[vs], (j / VS) & 1)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t v_addr = ptx::smem_u32(smem + L::kVOff + vs * L::kVBytes);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        ptx::mma_ts(tmem + 2 * BQ + t * BQ, tmem + t * BQ + kk * 8,
                                    ptx::sdesc_sw128(v_addr + kk * 16 * 128, kPanelBytes, 1024), kIdO,
                                    (j > 0 || kk > 0) ? 1u : 0u);
                    if (j == nt - 1) ptx::mma_commit(&ctrl->o_final[t]);
                    // S_t(j+1) overwrites the columns P_t(j) occupies: tcgen05.mma operations
                    // issued by one thread execute in issue order, so the product just issued
                    // has read P_t(j) before S_t(j+1) is written; and the commit behind
                    // s_full[t] covers that product, so O_t is complete when the softmax sees
                    // S_t(j+1).
                    if (j + 1 < nt && !issue_s(t, j + 1)) {
                        ok = false;
                        break;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(&ctrl->v_empty[vs]);
                if (j + 1 < nmax) ptx::mma_commit(&ctrl->k_empty[(j + 1) % KS]);
            }
            ptx::mma_commit(&ctrl->final_mma);
            if (!ptx::mbar_wait_quiet(&ctrl->final_mma, 0, kWaitLimitNs)) atomicOr(a.flags, kFlagWaitTimeout);
        }
      }
    } else {
        ptx::regs_inc<kRegsSoftmax>();
        // ------------------------------------------------------------ softmax warpgroups
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t s_col = X * BQ, o_col = 2 * BQ + X * BQ;
        const int r0 = q0 + X * BQ;
        const float c = a.scale_log2;
        const float *bias_row = nullptr;
        if (kBias && i < a.Nq) bias_row = a.bias + b * a.bs0 + h * a.bs1 + (long long)i * a.bs2;
        const bool bias_vec = (reinterpret_cast<uintptr_t>(bias_row) & 15u) == 0;
        __nv_bfloat16 *orow = (i < a.Nq) ? a.o + b * a.os0 + (long long)i * a.os1 + h * a.os2 : nullptr;
        float *lse_out = (a.lse && i < a.Nq) ? a.lse + ((long long)b * a.H + h) * a.Nq + i : nullptr;
        auto wait_warp = [&](uint64_t *bar, uint32_t parity) -> bool {
            const bool w = ptx::mbar_wait(bar, parity, abort, a.flags, kFlagWaitTimeout, kWaitLimitNs);
            return __all_sync(0xffffffffu, w);
        };
        if (nX == 0) {
            if (orow) write_empty_row<DV>(orow, lse_out);
        } else {
            float m_run = -INFINITY, l_run = 0.f;
            bool ok = true;
            const int lim = a.causal ? min(n, i + shift + 1) : n;  // keys < lim are visible
            float x[BK];  // with a bias: the next tile's bias, loaded ahead
            if (kBias) load_bias(bias_row, bias_vec, 0, n, x);
            for (int j = 0; j < nX; ++j) {
                const int kv0 = j * BK;
                if (!wait_warp(&ctrl->s_full[X], j & 1)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                if (kBias) load_s_row_bias(lane_addr + s_col, c, x);
                else load_s_row(lane_addr + s_col, x);
                const bool need_mask = (kv0 + BK > n) || (a.causal && kv0 + BK - 1 > r0 + shift);
                const float mt = tile_logits<kBias>(x, c, kv0, need_mask, lim);
                bool rescale;
                const float alpha = update_max(mt, m_run, rescale);
                const float lsum = tile_exp<kBias>(x, c, m_run);
                l_run = fmaf(alpha, l_run, lsum);
                if (__any_sync(0xffffffffu, rescale)) scale_o<DV>(lane_addr + o_col, alpha);
                // value rows past n inside this tile may hold anything: the warpgroup of the
                // first tile that uses V_j zeroes them before its product reads V_j
                if (kv0 + BK > n && n < a.Nk && (X == 0 || j >= nA)) {
                    if (!wait_warp(&ctrl->v_full[j % VS], (j / VS) & 1)) {
                        ok = false;
                        break;
                    }
                    if (kv0 + r >= n && kv0 + r < a.Nk)
                        zero_v_row<DV>(smem + L::kVOff + (j % VS) * L::kVBytes, r);
                    ptx::fence_proxy_async_smem();
                }
                store_p(lane_addr + s_col, x);
                ptx::tc_fence_before();
                ptx::mbar_arrive(&ctrl->p_full[X]);
                if (kBias && j + 1 < nX) load_bias(bias_row, bias_vec, kv0 + BK, n, x);
            }
            if (ok && wait_warp(&ctrl->o_final[X], 0)) {
                ptx::tc_fence_after();
                if constexpr (DV <= DK) {
                    // divide once, stage the bf16 tile in Q_X's shared memory (its last reader,
                    // S_X of the last key tile, completed before o_final) and store it with TMA
                    uint8_t *stage = smem + X * L::kQBytes;
                    stage_row<DV>(lane_addr + o_col, l_run, m_run, stage, r, lse_out);
                    ptx::fence_proxy_async_smem();
                    ptx::mbar_arrive(&ctrl->o_staged[X]);
                    // one thread stores the tile once all 128 rows are staged (a bounded wait:
                    // a warp that gave up earlier never arrives, and the store is then skipped)
                    if (r == 0 && ptx::mbar_wait(&ctrl->o_staged[X], 0, abort, a.flags,
                                                 kFlagWaitTimeout, kWaitLimitNs)) {
#pragma unroll
                        for (int p = 0; p < DV / 64; ++p)
                            ptx::tma_store_4d(&tm_o, stage + p * kPanelBytes, p * 64, r0, h, b);
                        ptx::bulk_commit();
                        ptx::bulk_wait_read();
                    }
                } else {
                    write_row<DV>(lane_addr + o_col, l_run, m_run, orow, lse_out);
                }
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

template <int DK, int DV, bool kBias>
attn_status_t launch_t(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                       const CUtensorMap &mo, const Args &a, cudaStream_t s) {
    const int smem = Layout<DK, DV>::kBytes;
    auto kern = fwd_bf16_pair_kernel<DK, DV, kBias>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    const long long grid = (long long)a.n_items * a.B * a.H;
    if (grid > 0x7fffffffLL) return fail(ATTN_ERR_UNSUPPORTED, "too many query tiles");
    kern<<<(unsigned)grid, kThreads, smem, s>>>(mq, mk, mv, mo, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "fwd_bf16_pair launch: %s", cudaGetErrorString(e));
    return ATTN_OK;
}

}  // namespace

attn_status_t launch_fwd_bf16_pair(const CUtensorMap &mq, const CUtensorMap &mk,
                                   const CUtensorMap &mv, const CUtensorMap &mo,
                                   const bf16fwd::Args &a, int dk, int dv, bool bias,
                                   cudaStream_t s) {
#define ATTN_PAIR_CASE(DK_, DV_)                                                              \
    if (dk == DK_ && dv == DV_)                                                                \
        return bias ? launch_t<DK_, DV_, true>(mq, mk, mv, mo, a, s)                           \
                    : launch_t<DK_, DV_, false>(mq, mk, mv, mo, a, s);
    ATTN_PAIR_CASE(128, 128)
    ATTN_PAIR_CASE(64, 64)
    ATTN_PAIR_CASE(128, 64)
    ATTN_PAIR_CASE(64, 128)
#undef ATTN_PAIR_CASE
    return fail(ATTN_ERR_UNSUPPORTED, "no two-tile bf16 kernel for dk=%d dv=%d", dk, dv);
}

}  // namespace attn
