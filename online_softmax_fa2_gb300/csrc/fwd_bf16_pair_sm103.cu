// fwd_bf16_pair_sm103.cu -- bf16 attention forward, two 128-row query tiles per CTA.
//
// A work item is 256 consecutive query rows of one (b, h): tile A (rows q0..q0+127) and tile
// B (rows q0+128..q0+255).  Every K and V tile brought into shared memory serves both query
// tiles, which halves the key/value traffic per FLOP against one tile per item, and the two
// tiles' softmax warpgroups take turns with the tensor cores: while one warpgroup turns its
// S into P, the tensor cores compute the other tile's products ("How Does FlashAttention
// Preserve Global Softmax Across Tiles?", section 5: every query row keeps its own state;
// section 8: query-block parallelism).
//
// The kernel is persistent: one CTA per SM walks a fixed list of items, numbered longest
// first and dealt out in rows taken in alternating direction.  Barrier phases run on from one
// item to the next, so the next item's Q and first K/V tiles load, and its first S products
// run, while the softmax warpgroups are still writing the previous item's rows.
//
// Roles (384 threads = 3 warpgroups):
//   warp 0       TMA producer: per item Q_A and Q_B, then K and V tiles into two rings.
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
    uint64_t q_full[2], q_empty[2];
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
    // tile A's output is staged in a buffer of its own, so that Q_A is released by its last
    // S product alone and the next item's Q_A loads while the item's last key tiles run
    static constexpr int kStageBytes = kVBytes;
    static constexpr int kFixed = 2 * kQBytes + kStageBytes + (int)sizeof(Ctrl) + 1024;
    // as many K stages as fit with 2 V stages (at most 4), then V stages likewise
    static constexpr int kKStages =
        (kFixed + 4 * kKBytes + 2 * kVBytes <= kSmemMax) ? 4
        : (kFixed + 3 * kKBytes + 2 * kVBytes <= kSmemMax) ? 3 : 2;
    static constexpr int kVStages =
        (kFixed + kKStages * kKBytes + 4 * kVBytes <= kSmemMax) ? 4
        : (kFixed + kKStages * kKBytes + 3 * kVBytes <= kSmemMax) ? 3 : 2;
    static constexpr int kKOff = 2 * kQBytes;
    static constexpr int kVOff = kKOff + kKStages * kKBytes;
    static constexpr int kStageOff = kVOff + kVStages * kVBytes;
    static constexpr int kDataBytes = kStageOff + kStageBytes;
    static constexpr int kBytes = kDataBytes + (int)sizeof(Ctrl) + 1024;
    static_assert(kBytes <= kSmemMax, "shared memory budget");
};

// Work item k (0 <= k < B * H * n_items, numbered longest first) -> (b, h, 256-row block).
// n and shift are in the kernel's own key numbering (a shard's, for partial states): keys
// j < n lie within the sequence, and under the causal mask key j is visible to row i iff
// j <= i + shift.
struct Item {
    int b, h, q0, n, shift, nA, nB, nmax;
};

template <bool kShard = false>
__device__ __forceinline__ Item decode_item(const Args &a, const DropArgs &dr, int k, bool report) {
    Item it;
    // k / (B H) and bh / H by multiply-high (every role decodes at every item boundary)
    const int kq = (int)div_fast((uint32_t)k, a.div_bhn_m, a.div_bhn_s);
    const int blk = a.n_items - 1 - kq;  // later query blocks see more keys: first
    const int bh = k - kq * (a.B * a.H);
    it.b = (int)div_fast((uint32_t)bh, a.div_h_m, a.div_h_s);
    it.h = bh - it.b * a.H;
    it.q0 = blk * 2 * BQ;
    if constexpr (kShard) {
        const int len = seq_len(a, it.b, report && blk == 0 && it.h == 0, dr.Nk_tot);  // the whole sequence's
        it.n = min(max(len - dr.key_off, 0), a.Nk);
        it.shift = len - a.Nq - dr.key_off;
    } else {  // the whole sequence: no offset
        const int len = seq_len(a, it.b, report && blk == 0 && it.h == 0);
        it.n = len;
        it.shift = len - a.Nq;
    }
    it.nA = kv_tiles_shard(a, it.q0, it.n, it.shift);
    it.nB = kv_tiles_shard(a, it.q0 + BQ, it.n, it.shift);
    it.nmax = max(it.nA, it.nB);
    return it;
}

// The r-th item of CTA c among G resident CTAs: rows of G consecutive items of the
// longest-first list, taken in alternating direction (c, then G-1-c, ...), so that each CTA's
// total is close to the mean.
__device__ __forceinline__ int item_index(int r, int c, int G) {
    return r * G + ((r & 1) ? G - 1 - c : c);
}

// The first item after the r-th of CTA c that has a key tile (nmax = 0 if none is left).
template <bool kShard>
__device__ __forceinline__ Item next_item(const Args &a, const DropArgs &dr, int r, int c, int G, int total) {
    for (int k = item_index(++r, c, G); k < total; k = item_index(++r, c, G)) {
        const Item it = decode_item<kShard>(a, dr, k, false);
        if (it.nmax > 0) return it;
    }
    Item none{};
    return none;
}

// Dropout (training forward): store_p with the row's 128 keep bits for the key tile applied as
// P is rounded and packed (bit t of word w = key 32w + t of the tile; dropped weights 0, kept
// ones as they are: the 1 / (1 - dropout_p) of the kept ones is applied once, to the row's
// output, in the epilogue).  The bits are needed only while the row's values are already
// leaving registers, which keeps the softmax threads from spilling.
__device__ __forceinline__ void store_p_keep(uint32_t taddr, const float (&x)[BK], const uint4 &keep) {
    const uint32_t w[4] = {keep.x, keep.y, keep.z, keep.w};
#pragma unroll
    for (int cc = 0; cc < BK / 64; ++cc) {
        uint32_t pk[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            const int k = cc * 64 + 2 * t;
            const float lo = ((w[k >> 5] >> (k & 31)) & 1u) ? x[k] : 0.f;
            const float hi = ((w[(k + 1) >> 5] >> ((k + 1) & 31)) & 1u) ? x[k + 1] : 0.f;
            pk[t] = ptx::pack_bf16x2(lo, hi);
        }
        ptx::tmem_st32(taddr + cc * 32, pk);
    }
    ptx::tmem_st_wait();
}

__device__ __forceinline__ uint4 ld_keep(const uint8_t *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// The next tile's keep bits are prefetched into L1 and loaded only where they are applied, so
// that no register holds them through the softmax.
__device__ __forceinline__ void prefetch_keep(const uint8_t *p) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// kPartial: write each row's state (m, l, u) over the kernel's keys to dr.part ([B, H, Nq,
// 2 + DV] fp32; m the row's reference in natural-log units, l and u measured against it;
// (-inf, 0, 0) for a row that sees no key) instead of o and lse.
// kDrop: 0 no dropout, 1 keep bits from a mask, 2 keep bits drawn in-kernel (separate
// instantiations, so that neither path holds the other's state in registers).
template <int DK, int DV, bool kBias, int kDrop, bool kPartial>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_o, const Args a, const DropArgs dr) {
    using L = Layout<DK, DV>;
    constexpr int KS = L::kKStages, VS = L::kVStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem + L::kDataBytes);
    volatile int *abort = &ctrl->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = a.B * a.H * a.n_items;
    const int G = (int)gridDim.x, cta = (int)blockIdx.x;

    bool pre_q = false, pre_k = false;  // loads thread 0 issued ahead of the block barrier
    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(&ctrl->q_full[t], 1);
            ptx::mbar_init(&ctrl->q_empty[t], 1);  // released by the item's last S_t
            ptx::mbar_init(&ctrl->o_staged[t], BQ);
            ptx::mbar_init(&ctrl->s_full[t], 1);
            ptx::mbar_init(&ctrl->p_full[t], BQ);
            ptx::mbar_init(&ctrl->o_final[t], 1);
        }
        for (int s = 0; s < KS; ++s) {
            ptx::mbar_init(&ctrl->k_full[s], 1);
            ptx::mbar_init(&ctrl->k_empty[s], 1);
        }
        for (int s = 0; s < VS; ++s) {
            ptx::mbar_init(&ctrl->v_full[s], 1);
            ptx::mbar_init(&ctrl->v_empty[s], 1);
        }
        ptx::mbar_init(&ctrl->final_mma, 1);
        ctrl->abort = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
        ptx::prefetch_tmap(&tm_o);
        // launched as a programmatic dependent of the previous kernel in the stream: nothing
        // in global memory is read before that kernel has completed
        ptx::grid_dep_wait();
        // this thread is the producer: the first item's Q_A and K_0 start loading before the
        // tensor-memory allocation and the block barrier
        const Item it = next_item<kPartial>(a, dr, -1, cta, G, total);
        if (it.nmax > 0) {
            if (it.nA > 0) {
                ptx::mbar_arrive_expect_tx(&ctrl->q_full[0], L::kQBytes);
#pragma unroll
                for (int p = 0; p < DK / 64; ++p)
                    ptx::tma_load_4d(smem + p * kPanelBytes, &tm_q, &ctrl->q_full[0], p * 64, it.q0, it.h,
                                     it.b);
                pre_q = true;
            }
            ptx::mbar_arrive_expect_tx(&ctrl->k_full[0], L::kKBytes);
#pragma unroll
            for (int p = 0; p < DK / 64; ++p)
                ptx::tma_load_4d(smem + L::kKOff + p * kPanelBytes, &tm_k, &ctrl->k_full[0], p * 64, 0, it.h,
                                 it.b);
            pre_k = true;
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc(&ctrl->tmem_base, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::grid_dep_wait();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    // the next kernel in the stream may be scheduled onto SMs as this grid's CTAs finish: its
    // set-up then overlaps this grid's tail (it reads global memory only after this grid
    // has completed)
    ptx::launch_dependents();

    // Barrier phases run on from one item to the next: g counts key tiles (K/V ring slots),
    // and per query tile, Q loads, S/P hand-offs and finished items are counted likewise.
    if (warp < 4) {
      ptx::regs_dec<kRegsIssue>();
      if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int g = 0, nqA = pre_q ? 1 : 0, nqB = 0, last_k = pre_k ? 0 : -1, last_v = -1;
            // Q_t of the next item, once the previous item's last S_t has read the buffer
            auto load_q = [&](int t, int &nq, const Item &it) -> bool {
                if (nq > 0 && !ptx::mbar_wait(&ctrl->q_empty[t], (nq - 1) & 1, abort, a.flags,
                                              kFlagWaitTimeout, kWaitLimitNs))
                    return false;
                ptx::mbar_arrive_expect_tx(&ctrl->q_full[t], L::kQBytes);
#pragma unroll
                for (int p = 0; p < DK / 64; ++p)
                    ptx::tma_load_4d(smem + t * L::kQBytes + p * kPanelBytes, &tm_q, &ctrl->q_full[t],
                                     p * 64, it.q0 + t * BQ, it.h, it.b);
                ++nq;
                return true;
            };
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int k = item_index(r, cta, G);
                if (k >= total) break;
                const Item it = decode_item<kPartial>(a, dr, k, false);
                if (it.nmax == 0) continue;
                // Q_A, K_0, Q_B, V_0, K_1, ...: S_A(0) needs only the first two
                if (it.nA > 0 && !(g == 0 && pre_q) && !load_q(0, nqA, it)) break;
                for (int j = 0; ok && j < it.nmax; ++j) {
                    const int gj = g + j, ks = gj % KS, vs = gj % VS;
                    if (!(gj == 0 && pre_k)) {
                        if (gj >= KS && !ptx::mbar_wait(&ctrl->k_empty[ks], ((gj / KS) - 1) & 1, abort,
                                                        a.flags, kFlagWaitTimeout, kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        uint8_t *sK = smem + L::kKOff + ks * L::kKBytes;
                        ptx::mbar_arrive_expect_tx(&ctrl->k_full[ks], L::kKBytes);
#pragma unroll
                        for (int p = 0; p < DK / 64; ++p)
                            ptx::tma_load_4d(sK + p * kPanelBytes, &tm_k, &ctrl->k_full[ks], p * 64, j * BK,
                                             it.h, it.b);
                        last_k = gj;
                    }
                    if (j == 0 && it.nB > 0 && !load_q(1, nqB, it)) {
                        ok = false;
                        break;
                    }
                    if (gj >= VS && !ptx::mbar_wait(&ctrl->v_empty[vs], ((gj / VS) - 1) & 1, abort,
                                                    a.flags, kFlagWaitTimeout, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sV = smem + L::kVOff + vs * L::kVBytes;
                    ptx::mbar_arrive_expect_tx(&ctrl->v_full[vs], L::kVBytes);
#pragma unroll
                    for (int p = 0; p < DV / 64; ++p)
                        ptx::tma_load_4d(sV + p * kPanelBytes, &tm_v, &ctrl->v_full[vs], p * 64, j * BK,
                                         it.h, it.b);
                    last_v = gj;
                }
                g += it.nmax;
            }
            if (*abort) {  // let copies still in flight land before the CTA exits
                if (nqA > 0) ptx::mbar_wait_quiet(&ctrl->q_full[0], (nqA - 1) & 1, kWaitLimitNs);
                if (nqB > 0) ptx::mbar_wait_quiet(&ctrl->q_full[1], (nqB - 1) & 1, kWaitLimitNs);
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
            // The tensor cores' queue holds little more than one product, so whatever this
            // thread does between two groups of products leaves them idle for about as long.
            // It therefore keeps everything ready: ring slots and barrier parities advance by
            // one step per key tile (no division), and shared-memory descriptors are kept as
            // their 32-bit low words (ptx::mma_ss_lo), stepped by adds.
            const uint32_t q_lo = ptx::sdesc_lo(ptx::smem_u32(smem), 16);  // Q_A; K-major: LBO 16 B
            // K slot s: q_lo + kKLo + s * kKStep; V slot s (MN-major, LBO = one panel): likewise
            constexpr uint32_t kKLo = L::kKOff >> 4, kKStep = L::kKBytes >> 4, kVStep = L::kVBytes >> 4;
            constexpr uint32_t kVLo = (L::kVOff >> 4) + (((uint32_t)kPanelBytes >> 4) << 16) - (1u << 16);
            auto wait = [&](uint64_t *bar, uint32_t parity) {
                return ptx::mbar_wait(bar, parity, abort, a.flags, kFlagWaitTimeout, kWaitLimitNs);
            };
            // S_t = Q_t K^T into TMEM columns [t*128, t*128 + 128), K in ring slot ks
            // (the bases are hidden from the optimiser so that the per-step operands are formed by
            // one add each instead of being hoisted out of the loops into registers)
            auto s_products = [&](int t, int ks) {
                uint32_t ql = q_lo, tm = tmem;
                ptx::opaque(ql);
                ptx::opaque(tm);
                const uint32_t qt = ql + t * (L::kQBytes >> 4), kt = ql + kKLo + ks * kKStep;
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint32_t off = ((kk / 4) * kPanelBytes + (kk % 4) * 32) >> 4;
                    ptx::mma_ss_lo(tm + t * BQ, qt + off, kt + off, kIdS, kk > 0 ? 1u : 0u);
                }
                ptx::mma_commit(&ctrl->s_full[t]);
            };
            // O_t (+)= P_t V, P_t from TMEM columns [t*128, t*128 + 64), V in ring slot vs
            auto pv_products = [&](int t, int vs, bool first) {
                uint32_t ql = q_lo, tm = tmem;
                ptx::opaque(ql);
                ptx::opaque(tm);
                const uint32_t vt = ql + kVLo + vs * kVStep;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    ptx::mma_ts_lo(tm + 2 * BQ + t * BQ, tm + t * BQ + kk * 8, vt + ((kk * 16 * 128) >> 4), kIdO,
                                   (!first || kk > 0) ? 1u : 0u);
            };
            // ring slots of the next K tile and of the current V tile; barrier parities as bits:
            // 0 K full, 1 V full, 2/3 Q_A/Q_B full, 4/5 P_A/P_B handed over
            int ks = 0, vs = 0;
            uint32_t ph = 0;
            auto par = [&](int bit) -> uint32_t { return (ph >> bit) & 1u; };
            auto flip = [&](int bit) { ph ^= 1u << bit; };
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int k = item_index(r, cta, G);
                if (k >= total) break;
                const Item it = decode_item<kPartial>(a, dr, k, false);
                if (it.nmax == 0) continue;
                const int nA = it.nA, nB = it.nB, nmax = it.nmax;
                // first S of each tile: the previous item's last P V product of that tile, issued
                // earlier, reads its P from these columns first (issue order)
                if (!wait(&ctrl->k_full[ks], par(0))) break;
                if (nA > 0) {
                    if (!wait(&ctrl->q_full[0], par(2))) break;
                    flip(2);
                    ptx::tc_fence_after();
                    s_products(0, ks);
                    if (nA == 1) ptx::mma_commit(&ctrl->q_empty[0]);
                }
                if (nB > 0) {
                    if (!wait(&ctrl->q_full[1], par(3))) break;
                    flip(3);
                    ptx::tc_fence_after();
                    s_products(1, ks);
                    if (nB == 1) ptx::mma_commit(&ctrl->q_empty[1]);
                }
                ptx::mma_commit(&ctrl->k_empty[ks]);
                if (++ks == KS) { ks = 0; flip(0); }
                for (int j = 0; j < nmax; ++j) {
                    // O_t += P_t V_j, then S_t(j+1) into the columns P_t(j) occupies:
                    // tcgen05.mma operations issued by one thread execute in issue order, so
                    // the product has read P_t(j) before S_t(j+1) is written; and the commit
                    // behind s_full[t] covers that product, so O_t is complete when the
                    // softmax sees S_t(j+1).
                    const bool more = j + 1 < nmax;
                    if (!wait(&ctrl->v_full[vs], par(1)) || (more && !wait(&ctrl->k_full[ks], par(0)))) {
                        ok = false;
                        break;
                    }
                    if (j < nA) {
                        if (!wait(&ctrl->p_full[0], par(4))) { ok = false; break; }
                        flip(4);
                        ptx::tc_fence_after();
                        pv_products(0, vs, j == 0);
                        if (j == nA - 1) ptx::mma_commit(&ctrl->o_final[0]);
                        if (j + 1 < nA) {
                            s_products(0, ks);
                            if (j + 2 == nA) ptx::mma_commit(&ctrl->q_empty[0]);
                        }
                    }
                    if (j < nB) {
                        if (!wait(&ctrl->p_full[1], par(5))) { ok = false; break; }
                        flip(5);
                        ptx::tc_fence_after();
                        pv_products(1, vs, j == 0);
                        if (j == nB - 1) ptx::mma_commit(&ctrl->o_final[1]);
                        if (j + 1 < nB) {
                            s_products(1, ks);
                            if (j + 2 == nB) ptx::mma_commit(&ctrl->q_empty[1]);
                        }
                    }
                    // the last V slot of the item is released by tile B's epilogue, which stages
                    // its output there
                    if (more) {
                        ptx::mma_commit(&ctrl->v_empty[vs]);
                        ptx::mma_commit(&ctrl->k_empty[ks]);
                        if (++ks == KS) { ks = 0; flip(0); }
                    }
                    if (++vs == VS) { vs = 0; flip(1); }
                }
            }
            ptx::mma_commit(&ctrl->final_mma);
            if (!ptx::mbar_wait_quiet(&ctrl->final_mma, 0, kWaitLimitNs)) atomicOr(a.flags, kFlagWaitTimeout);
        }
      }
    } else {
        ptx::regs_inc<kRegsSoftmax>();
        // ------------------------------------------------------------ softmax warpgroups
        const int X = (warp >= 8) ? 1 : 0;              // query tile of this warpgroup
        const int r = (int)threadIdx.x - 128 - X * BQ;  // row in the tile == TMEM lane
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t s_col = X * BQ, o_col = 2 * BQ + X * BQ;
        const float c = a.scale_log2;
        auto wait_warp = [&](uint64_t *bar, uint32_t parity) -> bool {
            const bool w = ptx::mbar_wait(bar, parity, abort, a.flags, kFlagWaitTimeout, kWaitLimitNs);
            return __all_sync(0xffffffffu, w);
        };
        int g = 0, u = 0, nfin = 0;
        bool ok = true;
        for (int rr = 0; ok; ++rr) {
            const int k = item_index(rr, cta, G);
            if (k >= total) break;
            const Item it = decode_item<kPartial>(a, dr, k, threadIdx.x == 128);
            const int nX = X ? it.nB : it.nA;
            const int r0 = it.q0 + X * BQ, i = r0 + r;
            // this row's output and log-sum-exp (null past Nq)
            auto out_row = [&]() -> __nv_bfloat16 * {
                return (i < a.Nq) ? a.o + it.b * a.os0 + (long long)i * a.os1 + it.h * a.os2 : nullptr;
            };
            auto out_lse = [&]() -> float * {
                return (a.lse && i < a.Nq) ? a.lse + ((long long)it.b * a.H + it.h) * a.Nq + i : nullptr;
            };
            if (nX == 0) {  // no key visible to any row of this tile
                if (i < a.Nq) {
                    if constexpr (kPartial) write_empty_state<DV>(dr.part + (((long long)it.b * a.H + it.h) * a.Nq + i) * (2 + DV));
                    else write_empty_row<DV>(out_row(), out_lse());
                }
                g += it.nmax;
                continue;
            }
            const int shift = it.shift;
            const float *bias_row = nullptr;
            if (kBias && i < a.Nq) bias_row = a.bias + it.b * a.bs0 + it.h * a.bs1 + (long long)i * a.bs2;
            const bool bias_vec = (reinterpret_cast<uintptr_t>(bias_row) & 15u) == 0;
            const int lim = a.causal ? min(it.n, i + shift + 1) : it.n;  // keys < lim are visible
            float m_run = -INFINITY, l_run = 0.f;
            float x[BK];  // with a bias: the next tile's bias, loaded ahead
            if (kBias) load_bias(bias_row, bias_vec, 0, it.n, x);
            // dropout: this row's keep bits, 16 bytes per key tile, the next tile's loaded ahead
            // from the mask, or drawn in-kernel while the thread waits for the next S
            const uint8_t *keep_row = nullptr;
            uint4 keep = make_uint4(0u, 0u, 0u, 0u);
            const uint32_t bh = (uint32_t)(it.b * a.H + it.h);
            if constexpr (kDrop == 2) {
                if (i < a.Nq) keep = rng::keep128((uint32_t)i, 0u, bh, dr.offset, dr.seed_lo, dr.seed_hi, dr.p8x4);
            } else if constexpr (kDrop == 1) {
                if (i < a.Nq) {
                    keep_row = dr.dmask + it.b * dr.dms0 + it.h * dr.dms1 + (long long)i * dr.dms2;
                    prefetch_keep(keep_row);
                }
            }
            for (int j = 0; j < nX; ++j) {
                const int kv0 = j * BK, gj = g + j;
                if (!wait_warp(&ctrl->s_full[X], (u + j) & 1)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                if (kBias) load_s_row_bias(lane_addr + s_col, c, x);
                else load_s_row(lane_addr + s_col, x);
                const bool need_mask = (kv0 + BK > it.n) || (a.causal && kv0 + BK - 1 > r0 + shift);
                const float mt = tile_logits<kBias>(x, c, kv0, need_mask, lim);
                bool rescale;
                const float alpha = update_max(mt, m_run, rescale);
                const float lsum = tile_exp<kBias>(x, c, m_run);
                l_run = fmaf(alpha, l_run, lsum);

                if (__any_sync(0xffffffffu, rescale)) scale_o<DV>(lane_addr + o_col, alpha);
                // value rows past n inside this tile may hold anything: the warpgroup of the
                // first query tile that uses V_j zeroes them before its product reads V_j
                if (kv0 + BK > it.n && it.n < a.Nk && (X == 0 || j >= it.nA)) {
                    if (!wait_warp(&ctrl->v_full[gj % VS], (gj / VS) & 1)) {
                        ok = false;
                        break;
                    }
                    if (kv0 + r >= it.n && kv0 + r < a.Nk)
                        zero_v_row<DV>(smem + L::kVOff + (gj % VS) * L::kVBytes, r);
                    ptx::fence_proxy_async_smem();
                }
                // dropout: the row sum above kept the undropped weights; P drops them
                if constexpr (kDrop == 1) {
                    store_p_keep(lane_addr + s_col, x,
                                 keep_row ? ld_keep(keep_row + j * (BK / 8)) : make_uint4(0u, 0u, 0u, 0u));
                } else if constexpr (kDrop == 2) {
                    store_p_keep(lane_addr + s_col, x, keep);
                } else {
                    store_p(lane_addr + s_col, x);
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(&ctrl->p_full[X]);
                if (kBias && j + 1 < nX) load_bias(bias_row, bias_vec, kv0 + BK, it.n, x);
                if constexpr (kDrop == 1) {
                    if (keep_row && j + 1 < nX) prefetch_keep(keep_row + (j + 1) * (BK / 8));
                } else if constexpr (kDrop == 2) {
                    if (i < a.Nq && j + 1 < nX)
                        keep = rng::keep128((uint32_t)i, (uint32_t)(kv0 + BK), bh, dr.offset, dr.seed_lo, dr.seed_hi,
                                            dr.p8x4);
                }
            }
            if (!ok || !wait_warp(&ctrl->o_final[X], nfin & 1)) break;
            ptx::tc_fence_after();
            if constexpr (kPartial) {
                // the row's state goes straight to global memory; the buffers the staged store
                // would have released are released here
                write_state<DV>(lane_addr + o_col, l_run, m_run,
                                i < a.Nq ? dr.part + (((long long)it.b * a.H + it.h) * a.Nq + i) * (2 + DV)
                                         : nullptr);
                ptx::tc_fence_before();
                if (r == 0) {
                    if (X) ptx::mbar_arrive(&ctrl->v_empty[(g + it.nmax - 1) % VS]);
                }
                g += it.nmax;
                u += nX;
                ++nfin;
                continue;
            }
            // divide once and store the row; the next item's first P V product overwrites O_X
            // only after this thread's next P hand-off, which follows these TMEM loads
            // Each tile's rows go through shared memory in the swizzled box layout, and one
            // thread stores the tile with TMA.  Tile A stages in a buffer of its own (Q_A has
            // been released by its last S product, so the next item's Q_A is already loading).
            // Tile B finishes last (it sees at least as many key tiles as tile A) and stages in
            // the item's last V slot, whose products have all completed, so that the next
            // item's Q_B can load meanwhile; the store releases that slot.
            {
                const int sl = (g + it.nmax - 1) % VS;
                uint8_t *stage = X ? smem + L::kVOff + sl * L::kVBytes : smem + L::kStageOff;
                stage_row<DV>(lane_addr + o_col, l_run, m_run, stage, r, out_lse(), kDrop != 0 ? dr.inv_keep : 1.f);
                ptx::tc_fence_before();
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive(&ctrl->o_staged[X]);
                if (r == 0) {
                    if (ptx::mbar_wait(&ctrl->o_staged[X], nfin & 1, abort, a.flags, kFlagWaitTimeout,
                                       kWaitLimitNs)) {
#pragma unroll
                        for (int p = 0; p < DV / 64; ++p)
                            ptx::tma_store_4d(&tm_o, stage + p * kPanelBytes, p * 64, r0, it.h, it.b);
                        ptx::bulk_commit();
                        ptx::bulk_wait_read();
                    }
                    if (X) ptx::mbar_arrive(&ctrl->v_empty[sl]);
                }
            }
            g += it.nmax;
            u += nX;
            ++nfin;
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

template <int DK, int DV, bool kBias, int kDrop, bool kPartial = false>
attn_status_t launch_t(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                       const CUtensorMap &mo, const Args &a, const DropArgs &dr, cudaStream_t s) {
    const int smem = Layout<DK, DV>::kBytes;
    auto kern = fwd_bf16_pair_kernel<DK, DV, kBias, kDrop, kPartial>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    const long long total = (long long)a.n_items * a.B * a.H;
    if (total > 0x7fffffffLL) return fail(ATTN_ERR_UNSUPPORTED, "too many query tiles");
    // persistent: one CTA per SM (each holds most of the shared memory and all of TMEM)
    const int sms = sm_count();
    if (sms <= 0) return fail(ATTN_ERR_CUDA, "could not read the SM count");
    const unsigned grid = (unsigned)(total < sms ? total : sms);
    e = launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, mq, mk, mv, mo, a, dr);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "fwd_bf16_pair launch: %s", cudaGetErrorString(e));
    return ATTN_OK;
}

}  // namespace

attn_status_t launch_fwd_bf16_pair(const CUtensorMap &mq, const CUtensorMap &mk,
                                   const CUtensorMap &mv, const CUtensorMap &mo,
                                   const bf16fwd::Args &a, const bf16fwd::DropArgs &dr, int dk, int dv, bool bias,
                                   cudaStream_t s) {
    if (dr.part) {  // partial states: dk == dv in {64, 128}, no dropout (checked by the caller)
        if (dk == 128 && dv == 128)
            return bias ? launch_t<128, 128, true, 0, true>(mq, mk, mv, mo, a, dr, s)
                        : launch_t<128, 128, false, 0, true>(mq, mk, mv, mo, a, dr, s);
        if (dk == 64 && dv == 64)
            return bias ? launch_t<64, 64, true, 0, true>(mq, mk, mv, mo, a, dr, s)
                        : launch_t<64, 64, false, 0, true>(mq, mk, mv, mo, a, dr, s);
        return fail(ATTN_ERR_UNSUPPORTED, "partial states need dk == dv in {64, 128} (dk=%d dv=%d)", dk, dv);
    }
#define ATTN_PAIR_CASE(DK_, DV_)                                                              \
    if (dk == DK_ && dv == DV_) {                                                              \
        if (dr.rng)                                                                            \
            return bias ? launch_t<DK_, DV_, true, 2>(mq, mk, mv, mo, a, dr, s)                    \
                        : launch_t<DK_, DV_, false, 2>(mq, mk, mv, mo, a, dr, s);                  \
        if (dr.dmask)                                                                          \
            return bias ? launch_t<DK_, DV_, true, 1>(mq, mk, mv, mo, a, dr, s)                    \
                        : launch_t<DK_, DV_, false, 1>(mq, mk, mv, mo, a, dr, s);                  \
        return bias ? launch_t<DK_, DV_, true, 0>(mq, mk, mv, mo, a, dr, s)                        \
                    : launch_t<DK_, DV_, false, 0>(mq, mk, mv, mo, a, dr, s);                      \
    }
    ATTN_PAIR_CASE(128, 128)
    ATTN_PAIR_CASE(64, 64)
    ATTN_PAIR_CASE(128, 64)
    ATTN_PAIR_CASE(64, 128)
#undef ATTN_PAIR_CASE
    return fail(ATTN_ERR_UNSUPPORTED, "no two-tile bf16 kernel for dk=%d dv=%d", dk, dv);
}

}  // namespace attn
