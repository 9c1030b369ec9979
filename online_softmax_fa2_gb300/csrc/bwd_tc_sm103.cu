// bwd_tc_sm103.cu -- attention backward for dk == dv in {64, 128} on the 5th-generation tensor
// cores.
//
// The same gradients as bwd.cu ("How Does FlashAttention Preserve Global Softmax Across
// Tiles?", section 7: rebuild p_ij = exp(x_ij - L_i), c_i = g_i . o_i, dS_ij = p_ij (g_i . v_j -
// c_i); dV_j += p_ij g_i, dK_j += scale dS_ij q_i, dQ_i += scale dS_ij k_j), with 128 x 128 tiles
// whose five products run as tcgen05.mma into tensor memory.  One CTA owns a block of 128 keys
// of one (b, h) and walks the query tiles of 128 rows that see any of its keys:
//
//   TMEM (512 columns)   S^T / P^T [0, 128)   dP^T / dS^T [128, 256)   dV [256, 384)   dK [384, 512)
//                        Each tile is handled as two halves of 64 query rows with barriers of
//                        their own (half h: S^T columns [64h, 64h + 64), dP^T [128 + 64h, ...)), so
//                        that P^T and dS^T of one half are formed while the tensor cores run the
//                        products of the other.  dQ^T of a half goes into that half's dP^T columns
//                        once dK has read its dS^T there.
//   S^T  = K Q^T         A = K, B = Q   (both [row][dim] in shared memory, K-major)
//   dP^T = V G^T         A = V, B = G   (G: the upstream gradient dL/dO)
//   P^T, dS^T            one thread per key (TMEM lane): mask, exp(x - L), (dP - c); P^T and
//                        dS^T go back into TMEM as bf16, dS^T also into shared memory
//   dV  += P^T G         A = P^T from TMEM, B = G read MN-major (as V in the forward's P V)
//   dK  += dS^T Q        A = dS^T from TMEM, B = Q read MN-major
//   dQ^T = K^T dS^T      A = K read MN-major, B = the [key][row] copy of dS^T read MN-major
//                        (transposed so that a TMEM lane is one head dimension: a warp's
//                        reduction of one row into dQ is then a single 128-byte line)
//
// Roles (384 threads): warp 0 loads K and V once and Q, G per tile with TMA; warp 1 issues the
// products (one thread); warps 4-7 form P^T and dS^T and, at the end, write dK (times scale)
// and dV; warps 8-11 read each tile's dQ^T from TMEM (one thread per head dimension), turn
// blocks of 4 rows x 4 dimensions around among 4 lanes, and add scale * dQ to the fp32
// accumulator with 16-byte reductions (a warp instruction covers 4 whole 128-byte rows).
//
// The grid is (H, B, key blocks), so that with a causal mask the blocks that see the most query
// tiles are dispatched first.  The kernel is launched with programmatic stream serialization:
// its CTAs may set up and load K, V, Q and G while the prep kernel drains, and wait for it only
// where they touch its outputs (lse * log2 e, c, the zeroed dQ accumulator).  With dropout
// (kDrop) the forward's keep mask scales the gradient reaching P.  Every mbarrier wait is
// bounded as in the forward kernels.
#include "fwd_bf16_common.cuh"

namespace attn {
namespace {

using namespace bf16fwd;

constexpr int kTcThreads = 384;
constexpr int kTile = 2 * kPanelBytes;  // 128 rows x 128 bf16: two 64-column 128B-swizzled panels
// K, V, then Q and G in two stages each, then the [key][row] copy of dS^T
constexpr int kOffK = 0, kOffV = kTile, kOffQ = 2 * kTile, kOffG = 4 * kTile, kOffS = 6 * kTile;
constexpr int kOffL = 7 * kTile;         // lse * log2 e of the tile's 128 rows, two stages
constexpr int kOffCtrl = kOffL + 2 * 512;
constexpr int kHalf = BQ / 2;  // query rows of a half tile

struct TcArgs {
    int B, H, Nq, Nk, causal;
    float scale, scale_log2;
    const float *crow;  // [B, H, Nq]
    const float *lrow;  // [B, H, nq_pad]: lse * log2 e, rows padded to a multiple of 128
    int nq_pad;
    const int *kv_lens;
    const float *bias;  // [B, H, Nq, Nk] with element strides bs0, bs1, bs2 (key stride 1), or null
    long long bs0, bs1, bs2;
    int bias_pf;        // bias rows 16-byte aligned: the producer prefetches them into L2
    float *dq_acc;  // [B, Nq, H, D]
    __nv_bfloat16 *dk, *dv;
    long long dks0, dks1, dks2, dvs0, dvs1, dvs2;
    uint32_t *flags;
};

struct TcCtrl {
    // q_full, q_empty: per stage; s_full .. ds_free: per half tile
    uint64_t kv_full, q_full[2], q_empty[2], s_full[2], p_ready[2], dq_full[2], dq_free[2], ds_free[2], kv_final;
    uint32_t tmem_base;
    int abort;
};

constexpr int kSmemBytes = kOffCtrl + (int)sizeof(TcCtrl) + 1024;
static_assert(kSmemBytes <= kSmemMax, "shared memory budget");

// kind::f16 instruction descriptor with bf16 A and B, fp32 D, A and B K-major or MN-major
// (bit 15: A MN-major, bit 16: B MN-major)
__host__ __device__ constexpr uint32_t idesc_ab(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// 1-D bulk copy global -> shared of `bytes` (multiple of 16, both addresses 16-byte aligned),
// completion counted on `bar`
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     ptx::smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(ptx::smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

}  // namespace
namespace ptx {
// (d0, d1) = (a0 * b0, a1 * b1) in one packed instruction
__device__ __forceinline__ void mul2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
}  // namespace ptx
namespace {

// A read-only load that the compiler keeps where it is written (so that a batch of them is in
// flight before the values are used)
__device__ __forceinline__ float ld_nc_f32(const float *p) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// L2 prefetch of `bytes` (a multiple of 16) from a 16-byte aligned address
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void red_add_v4(float *addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// 4 x 4 transpose among the lanes 4g .. 4g + 3 of a warp: on entry lane 4g + t holds x[s] =
// M[s][t]; on exit it holds x[s] = M[t][s].  Two butterfly stages, each swapping the lane bit
// with the index bit of the same weight (two shuffles per stage).
__device__ __forceinline__ void transpose4(float (&x)[4], int lane) {
#pragma unroll
    for (int bit = 1; bit <= 2; bit <<= 1) {
        const bool hi = lane & bit;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            // the pair (lo, lo + bit) of indices that this stage exchanges
            const int lo = bit == 1 ? 2 * j : j;
            const float send = hi ? x[lo] : x[lo + bit];
            const float got = __shfl_xor_sync(0xffffffffu, send, bit);
            if (hi) x[lo] = got;
            else x[lo + bit] = got;
        }
    }
}

// kDrop: the forward ran with dropout; `dr` holds its keep bits (bit j % 8 of byte j / 8 of a
// row) and 1 / (1 - p).  The gradient reaching P then carries the mask and its scale: the
// stored P^T (for dV) is z p / (1 - p), and dS = p (z dP / (1 - p) - c).
//
// D is the head dimension (dk = dv = D, 64 or 128).  With D = 64 only the first 64-column
// panel of Q, V and G is loaded and the products over the head dimension take half the
// steps; K's second panel is filled with zeros by the copy (its columns lie past the tensor),
// so that dQ^T = K^T dS^T keeps M = 128 and its rows 64 .. 127 come out zero.
//
// kBias: the forward's bias is added to the logits before the exponential.  The transform
// thread of key j reads b_ij of the 32 rows of a chunk before it waits for the chunk's S^T
// (for each row the warp's 32 keys are one 128-byte line).
template <bool kDrop, int D, bool kBias>
__global__ void __launch_bounds__(kTcThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                  const TcArgs a, const bf16fwd::DropArgs dr) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    TcCtrl *ctrl = reinterpret_cast<TcCtrl *>(smem + kOffCtrl);
    volatile int *abort = &ctrl->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // key block slowest: CTAs are dispatched in order of their linear index, so with a causal
    // mask (block kb sees the query tiles from about kb on) the longest blocks of every head
    // start first and the short ones fill the tail
    const int h = blockIdx.x, b = blockIdx.y, kb = blockIdx.z;

    int n = a.Nk;
    if (a.kv_lens) {
        const int raw = a.kv_lens[b];
        n = min(max(raw, 0), a.Nk);
        if (raw != n && threadIdx.x == 0 && kb == 0 && h == 0) atomicOr(a.flags, kFlagKvLenClamped);
    }
    const int shift = n - a.Nq;  // causal: key j visible to row i iff j <= i + shift
    const int j0 = kb * BK;
    const int i_first = a.causal ? max(0, j0 - shift) : 0;
    const bool any = j0 < n && i_first < a.Nq;
    const int t_first = i_first / BQ, t_end = any ? (a.Nq + BQ - 1) / BQ : t_first;

    // the dQ conversion queued after this kernel may be scheduled (it waits for completion)
    ptx::launch_dependents();
    if (!any) {  // no row sees a key of this block: dK = dV = 0
        if (warp >= 4 && warp < 8) {
            const int j = j0 + (int)threadIdx.x - 128;
            if (j < a.Nk) {
                uint4 *dkr = reinterpret_cast<uint4 *>(a.dk + b * a.dks0 + (long long)j * a.dks1 + h * a.dks2);
                uint4 *dvr = reinterpret_cast<uint4 *>(a.dv + b * a.dvs0 + (long long)j * a.dvs1 + h * a.dvs2);
                for (int c = 0; c < D / 8; ++c) dkr[c] = dvr[c] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        return;
    }

    if (threadIdx.x == 0) {
        ptx::mbar_init(&ctrl->kv_full, 1);
        for (int st = 0; st < 2; ++st) {
            ptx::mbar_init(&ctrl->q_full[st], 1);
            ptx::mbar_init(&ctrl->q_empty[st], 1);
        }
        for (int hh = 0; hh < 2; ++hh) {
            ptx::mbar_init(&ctrl->s_full[hh], 1);
            ptx::mbar_init(&ctrl->p_ready[hh], 128);
            ptx::mbar_init(&ctrl->dq_full[hh], 1);
            ptx::mbar_init(&ctrl->dq_free[hh], 128);
            ptx::mbar_init(&ctrl->ds_free[hh], 1);
        }
        ptx::mbar_init(&ctrl->kv_final, 1);
        ctrl->abort = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
        ptx::prefetch_tmap(&tm_g);
        // K in two panels always (with D = 64 the second is zero-filled), V, Q and G in D / 64
        ptx::mbar_arrive_expect_tx(&ctrl->kv_full, (2 + D / 64) * kPanelBytes);
        for (int p = 0; p < 2; ++p)
            ptx::tma_load_4d(smem + kOffK + p * kPanelBytes, &tm_k, &ctrl->kv_full, p * 64, j0, h, b);
        for (int p = 0; p < D / 64; ++p)
            ptx::tma_load_4d(smem + kOffV + p * kPanelBytes, &tm_v, &ctrl->kv_full, p * 64, j0, h, b);
        ptx::mbar_arrive_expect_tx(&ctrl->q_full[0], 2 * (D / 64) * kPanelBytes + 512);
        for (int p = 0; p < D / 64; ++p) {
            ptx::tma_load_4d(smem + kOffQ + p * kPanelBytes, &tm_q, &ctrl->q_full[0], p * 64, t_first * BQ, h, b);
            ptx::tma_load_4d(smem + kOffG + p * kPanelBytes, &tm_g, &ctrl->q_full[0], p * 64, t_first * BQ, h, b);
        }
        // lse * log2 e, the row terms c and the zeroed dQ accumulator come from the prep kernel,
        // which this launch may overlap: every role that touches them waits for it first
        ptx::grid_dep_wait();
        bulk_load(smem + kOffL, a.lrow + ((long long)b * a.H + h) * a.nq_pad + t_first * BQ, 512, &ctrl->q_full[0]);
    }
    if (warp == 1) {
        ptx::tmem_alloc(&ctrl->tmem_base, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    auto wait = [&](uint64_t *bar, uint32_t parity) {
        return ptx::mbar_wait(bar, parity, abort, a.flags, kFlagWaitTimeout, kWaitLimitNs);
    };
    const int ntiles = t_end - t_first;
    // the bias rows of query tile t over this block's keys into L2 (ahead of the transform's loads)
    auto prefetch_bias = [&](int t) {
        if constexpr (kBias) {
            if (!a.bias_pf) return;
            const uint32_t bytes = (uint32_t)((min(a.Nk, j0 + BK) - j0) * 4) & ~15u;
            if (bytes == 0) return;
            const float *base = a.bias + b * a.bs0 + h * a.bs1 + j0;
            for (int i = t * BQ; i < min(a.Nq, t * BQ + BQ); ++i) prefetch_l2(base + (long long)i * a.bs2, bytes);
        }
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int loaded = 1;
            prefetch_bias(t_first);
            // tile k into stage k & 1, once the products of tile k - 2 have read that stage
            for (int k = 1; k < ntiles; ++k) {
                const int st = k & 1;
                if (k >= 2 && !wait(&ctrl->q_empty[st], ((k >> 1) - 1) & 1)) break;
                const int i0 = (t_first + k) * BQ;
                prefetch_bias(t_first + k);
                ptx::mbar_arrive_expect_tx(&ctrl->q_full[st], 2 * (D / 64) * kPanelBytes + 512);
                bulk_load(smem + kOffL + st * 512, a.lrow + ((long long)b * a.H + h) * a.nq_pad + i0, 512,
                          &ctrl->q_full[st]);
                for (int p = 0; p < D / 64; ++p) {
                    ptx::tma_load_4d(smem + kOffQ + st * kTile + p * kPanelBytes, &tm_q, &ctrl->q_full[st], p * 64, i0,
                                     h, b);
                    ptx::tma_load_4d(smem + kOffG + st * kTile + p * kPanelBytes, &tm_g, &ctrl->q_full[st], p * 64, i0,
                                     h, b);
                }
                ++loaded;
            }
            if (*abort) {  // copies in flight land before the CTA exits
                ptx::mbar_wait_quiet(&ctrl->kv_full, 0, kWaitLimitNs);
                for (int k = max(0, loaded - 2); k < loaded; ++k)
                    ptx::mbar_wait_quiet(&ctrl->q_full[k & 1], (k >> 1) & 1, kWaitLimitNs);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ tensor-core issuer
        if (lane == 0) {
            constexpr uint32_t kIdS = idesc_ab(BK, kHalf, false, false);  // S^T, dP^T of a half
            constexpr uint32_t kIdKV = idesc_ab(BK, D, false, true);      // dV, dK: A from TMEM, B MN-major
            constexpr uint32_t kIdQ = idesc_ab(128, kHalf, true, true);   // dQ^T: A and B MN-major
            const uint32_t sK = ptx::smem_u32(smem + kOffK), sV = ptx::smem_u32(smem + kOffV);
            const uint32_t sS = ptx::smem_u32(smem + kOffS);
            // K-major operands: 16-dim steps are 32 bytes apart inside a 64-column panel
            const uint64_t kd = ptx::sdesc_sw128(sK, 16, 1024), vd = ptx::sdesc_sw128(sV, 16, 1024);
            // MN-major operands: 16-row steps are 16 rows x 128 bytes apart; the two 64-wide
            // panels of the N (or M) dimension are kPanelBytes apart
            const uint64_t km = ptx::sdesc_sw128(sK, kPanelBytes, 1024);
            // S^T and dP^T of half hh of tile k (Q, G in stage k & 1); dP^T overwrites the
            // previous tile's dQ^T of this half, so it waits until that has been read
            auto s_dp = [&](int k, int hh) -> bool {
                const uint32_t off_q = kOffQ + (k & 1) * kTile + hh * kHalf * 128;
                const uint32_t off_g = kOffG + (k & 1) * kTile + hh * kHalf * 128;
                const uint64_t qd = ptx::sdesc_sw128(ptx::smem_u32(smem + off_q), 16, 1024);
                const uint64_t gd = ptx::sdesc_sw128(ptx::smem_u32(smem + off_g), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk / 4) * kPanelBytes + (kk % 4) * 32) >> 4;
                    ptx::mma_ss(tmem + hh * kHalf, kd + off, qd + off, kIdS, kk > 0 ? 1u : 0u);
                }
                if (k > 0 && !wait(&ctrl->dq_free[hh], (k - 1) & 1)) return false;
                ptx::tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk / 4) * kPanelBytes + (kk % 4) * 32) >> 4;
                    ptx::mma_ss(tmem + 128 + hh * kHalf, vd + off, gd + off, kIdS, kk > 0 ? 1u : 0u);
                }
                ptx::mma_commit(&ctrl->s_full[hh]);
                return true;
            };
            // dV += P^T G, dK += dS^T Q over the half's 64 rows, then its dQ^T = K^T dS^T
            auto grads = [&](int k, int hh) {
                const uint32_t sQ = ptx::smem_u32(smem + kOffQ + (k & 1) * kTile);
                const uint32_t sG = ptx::smem_u32(smem + kOffG + (k & 1) * kTile);
                const uint64_t gm = ptx::sdesc_sw128(sG, kPanelBytes, 1024);
                const uint64_t qm = ptx::sdesc_sw128(sQ, kPanelBytes, 1024);
                const uint64_t sm_ = ptx::sdesc_sw128(sS + hh * kPanelBytes, kPanelBytes, 1024);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {  // P^T bf16 pairs: 8 columns per 16 rows
                    const uint32_t row_off = ((hh * kHalf + kk * 16) * 128) >> 4;
                    ptx::mma_ts(tmem + 256, tmem + hh * kHalf + kk * 8, gm + row_off, kIdKV,
                                (k > 0 || hh > 0 || kk > 0) ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t row_off = ((hh * kHalf + kk * 16) * 128) >> 4;
                    ptx::mma_ts(tmem + 384, tmem + 128 + hh * kHalf + kk * 8, qm + row_off, kIdKV,
                                (k > 0 || hh > 0 || kk > 0) ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // into the columns the half's dS^T occupied
                    ptx::mma_ss(tmem + 128 + hh * kHalf, km + ((kk * 16 * 128) >> 4), sm_ + ((kk * 16 * 128) >> 4),
                                kIdQ, kk > 0 ? 1u : 0u);
                ptx::mma_commit(&ctrl->dq_full[hh]);
                ptx::mma_commit(&ctrl->ds_free[hh]);
            };
            bool ok = wait(&ctrl->kv_full, 0) && wait(&ctrl->q_full[0], 0);
            if (ok) {
                ptx::tc_fence_after();
                ok = s_dp(0, 0) && s_dp(0, 1);
            }
            for (int k = 0; ok && k < ntiles; ++k) {
                const bool more = k + 1 < ntiles;
                // half 0 of tile k, then S^T and dP^T of half 0 of tile k + 1 while the
                // transform works on half 1
                if (!wait(&ctrl->p_ready[0], k & 1)) break;
                ptx::tc_fence_after();
                grads(k, 0);
                if (more) {
                    if (!wait(&ctrl->q_full[(k + 1) & 1], ((k + 1) >> 1) & 1)) break;
                    ptx::tc_fence_after();
                    if (!s_dp(k + 1, 0)) break;
                }
                if (!wait(&ctrl->p_ready[1], k & 1)) break;
                ptx::tc_fence_after();
                grads(k, 1);
                ptx::mma_commit(&ctrl->q_empty[k & 1]);  // the last reads of stage k & 1
                if (more && !s_dp(k + 1, 1)) break;
            }
            ptx::mma_commit(&ctrl->kv_final);
            if (!ptx::mbar_wait_quiet(&ctrl->kv_final, 0, kWaitLimitNs)) atomicOr(a.flags, kFlagWaitTimeout);
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ P^T and dS^T (one key each)
        const int r = (int)threadIdx.x - 128;  // key in the block == TMEM lane
        const int j = j0 + r;
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        auto wait_warp = [&](uint64_t *bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, wait(bar, parity));
        };
        bool ok = wait_warp(&ctrl->kv_full, 0);
        if (ok && j >= n) {  // K rows past the sequence may hold anything: zero them for dQ^T = K^T dS^T
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                uint4 *dst = reinterpret_cast<uint4 *>(smem + kOffK + p * kPanelBytes + r * 128);
#pragma unroll
                for (int t = 0; t < 8; ++t) dst[t] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::grid_dep_wait();
        const float *c_bh = a.crow + ((long long)b * a.H + h) * a.Nq;
        for (int k = 0; ok && k < ntiles; ++k) {
            const int i0 = (t_first + k) * BQ;
            // c of the tile's rows, lane t holding rows 32c + t: loaded before the wait for S^T
            float Cq[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int it = i0 + 32 * c + lane;
                Cq[c] = it < a.Nq ? __ldg(c_bh + it) : 0.f;
            }
            // dropout: lane t holds, for rows 32c + t, the keep bits of this warp's 32 keys (from
            // the forward's mask, or drawn in-kernel as the forward drew them)
            uint32_t Zq[4];
            if constexpr (kDrop) {
                const int jw = j0 + 32 * (warp & 3);
                if (dr.rng) {
                    // row it sees keys < vis (its sequence's keys, and under the causal mask
                    // keys <= it + shift): groups of 16 keys past them are not drawn
                    const uint32_t bh = (uint32_t)(b * a.H + h), g0 = (uint32_t)(jw >> 4);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int it = i0 + 32 * c + lane;
                        const int vis = (a.causal ? min(n, it + shift + 1) : n) - jw;
                        uint32_t z = 0u;
                        if (it < a.Nq && vis > 0) {
                            z = rng::keep16((uint32_t)it, g0, bh, dr.offset, dr.seed_lo, dr.seed_hi, dr.p8x4);
                            if (vis > 16)
                                z |= rng::keep16((uint32_t)it, g0 + 1, bh, dr.offset, dr.seed_lo, dr.seed_hi, dr.p8x4)
                                     << 16;
                        }
                        Zq[c] = z;
                    }
                } else {
                    const uint8_t *zb = dr.dmask + b * dr.dms0 + h * dr.dms1 + jw / 8;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int it = i0 + 32 * c + lane;
                        Zq[c] = it < a.Nq ? __ldg(reinterpret_cast<const uint32_t *>(zb + (long long)it * dr.dms2)) : 0u;
                    }
                }
            }
            // bias: the 32 rows of chunk c at this thread's key, issued one chunk ahead of use
            // (rows and keys past the ends read row Nq - 1 / key Nk - 1; those weights are
            // selected away)
            float bv[kBias ? 32 : 1];
            auto load_bias = [&](int c) {
                if constexpr (kBias) {
                    const float *bcol = a.bias + b * a.bs0 + h * a.bs1 + min(j, a.Nk - 1);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        bv[e] = ld_nc_f32(bcol + (long long)min(i0 + 32 * c + e, a.Nq - 1) * a.bs2);
                }
            };
            for (int hh = 0; ok && hh < 2; ++hh) {
            load_bias(2 * hh);  // in flight during the wait for S^T
            // s_full implies the tile's copies are done; waiting on their barrier as well makes
            // the copied L visible to these threads
            if (!wait_warp(&ctrl->s_full[hh], k & 1) || !wait_warp(&ctrl->q_full[k & 1], (k >> 1) & 1) ||
                (k > 0 && !wait_warp(&ctrl->ds_free[hh], (k - 1) & 1))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
#pragma unroll 1
            for (int c = 2 * hh; c < 2 * hh + 2; ++c) {  // rows 32c .. 32c + 31 of the tile
                // c of row 32c + e is lane e's Cq[c]; L comes from the copy in shared memory (one
                // broadcast read)
                const float Ct = Cq[c];
                uint32_t Zt = 0u;
                if constexpr (kDrop) Zt = Zq[c];
                const float *Ls = reinterpret_cast<const float *>(smem + kOffL + (k & 1) * 512) + 32 * c;
                uint32_t sv[32], dv[32];
                ptx::tmem_ld32(lane_addr + 32 * c, sv);
                ptx::tmem_ld32(lane_addr + 128 + 32 * c, dv);
                ptx::tmem_ld_wait();
                ptx::reg_fence(sv);
                ptx::reg_fence(dv);
                uint32_t pp[16], dp[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float2 L2 = *reinterpret_cast<const float2 *>(Ls + e);
                    const float C0 = __shfl_sync(0xffffffffu, Ct, e), C1 = __shfl_sync(0xffffffffu, Ct, e + 1);
                    float x0, x1, g0, g1;
                    ptx::fma2(x0, x1, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), a.scale_log2, a.scale_log2,
                              -L2.x, -L2.y);
                    if constexpr (kBias) ptx::fma2(x0, x1, bv[e], bv[e + 1], kLog2e, kLog2e, x0, x1);
                    float zs0 = 1.f, zs1 = 1.f;  // z / (1 - p) of rows e, e + 1 for this key
                    if constexpr (kDrop) {
                        const uint32_t w0 = __shfl_sync(0xffffffffu, Zt, e), w1 = __shfl_sync(0xffffffffu, Zt, e + 1);
                        zs0 = ((w0 >> lane) & 1u) ? dr.inv_keep : 0.f;
                        zs1 = ((w1 >> lane) & 1u) ? dr.inv_keep : 0.f;
                        ptx::fma2(g0, g1, __uint_as_float(dv[e]), __uint_as_float(dv[e + 1]), zs0, zs1, -C0, -C1);
                    } else {
                        ptx::add2(g0, g1, __uint_as_float(dv[e]), __uint_as_float(dv[e + 1]), -C0, -C1);
                    }
                    const int i = i0 + 32 * c + e;
                    // visibility of rows i and i + 1 (selects, not products: anything stored past
                    // the sequence, NaN included, is dropped)
                    bool v0 = j < n && i < a.Nq && (!a.causal || j <= i + shift);
                    bool v1 = j < n && i + 1 < a.Nq && (!a.causal || j <= i + 1 + shift);
                    if constexpr (kBias) {  // a -inf bias masks the key (a row it empties has L = -inf)
                        v0 = v0 && bv[e] != -INFINITY;
                        v1 = v1 && bv[e + 1] != -INFINITY;
                    }
                    const float p0 = v0 ? ptx::ex2(x0) : 0.f, p1 = v1 ? ptx::ex2(x1) : 0.f;
                    float d0, d1;
                    ptx::mul2(d0, d1, p0, p1, g0, g1);
                    if constexpr (kDrop) {  // P^T for dV: the kept, scaled weights
                        float q0, q1;
                        ptx::mul2(q0, q1, p0, p1, zs0, zs1);
                        pp[e / 2] = ptx::pack_bf16x2(q0, q1);
                    } else {
                        pp[e / 2] = ptx::pack_bf16x2(p0, p1);
                    }
                    dp[e / 2] = ptx::pack_bf16x2(v0 ? d0 : 0.f, v1 ? d1 : 0.f);
                }
                if (c == 2 * hh) load_bias(c + 1);  // the next chunk's, while this one is stored
                // P^T and dS^T of the half packed into the first 32 of its S^T and dP^T columns
                // (all read by now: chunk 2hh + 1 packs over chunk 2hh)
                tmem_st16(lane_addr + 32 * hh + 16 * c, pp);
                tmem_st16(lane_addr + 128 + 32 * hh + 16 * c, dp);
                // dS^T into shared memory as [key][row]: rows 32c.. are 16-byte chunks
                // 4 (c % 2) .. + 3 of panel c / 2, 128-byte swizzled like a TMA box
                uint8_t *row = smem + kOffS + (c / 2) * kPanelBytes + r * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int chunk = (c % 2) * 4 + q;
                    *reinterpret_cast<uint4 *>(row + ((chunk ^ (r & 7)) * 16)) =
                        make_uint4(dp[4 * q], dp[4 * q + 1], dp[4 * q + 2], dp[4 * q + 3]);
                }
            }
            ptx::tmem_st_wait();
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&ctrl->p_ready[hh]);
            }
        }
        // dK (times scale) and dV of this key
        if (ok && wait_warp(&ctrl->kv_final, 0)) {
            ptx::tc_fence_after();
            __nv_bfloat16 *dkr = a.dk + b * a.dks0 + (long long)j * a.dks1 + h * a.dks2;
            __nv_bfloat16 *dvr = a.dv + b * a.dvs0 + (long long)j * a.dvs1 + h * a.dvs2;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t kv[32], vv[32];
                ptx::tmem_ld32(lane_addr + 384 + 32 * c, kv);
                ptx::tmem_ld32(lane_addr + 256 + 32 * c, vv);
                ptx::tmem_ld_wait();
                ptx::reg_fence(kv);
                ptx::reg_fence(vv);
                if (j < a.Nk) {
                    const bool seen = j < n;  // a key past the sequence gets +0.0 exactly
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t pk[4], pv[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            pk[t] = ptx::pack_bf16x2(a.scale * __uint_as_float(kv[8 * q + 2 * t]),
                                                     a.scale * __uint_as_float(kv[8 * q + 2 * t + 1]));
                            pv[t] = ptx::pack_bf16x2(__uint_as_float(vv[8 * q + 2 * t]), __uint_as_float(vv[8 * q + 2 * t + 1]));
                        }
                        *reinterpret_cast<uint4 *>(dkr + 32 * c + 8 * q) =
                            seen ? make_uint4(pk[0], pk[1], pk[2], pk[3]) : make_uint4(0u, 0u, 0u, 0u);
                        *reinterpret_cast<uint4 *>(dvr + 32 * c + 8 * q) =
                            seen ? make_uint4(pv[0], pv[1], pv[2], pv[3]) : make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
        }
    } else if (warp >= 8) {
        // ------------------------------------------------------------ dQ^T (one head dimension each)
        const int d = (int)threadIdx.x - 256;
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const long long row_stride = (long long)a.H * D;
        ptx::grid_dep_wait();
        bool ok = true;
        for (int k = 0; ok && k < ntiles; ++k) {
            for (int hh = 0; hh < 2; ++hh) {
                const bool w = ptx::mbar_wait(&ctrl->dq_full[hh], k & 1, abort, a.flags, kFlagWaitTimeout, kWaitLimitNs);
                if (!__all_sync(0xffffffffu, w)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const int i0 = (t_first + k) * BQ + hh * kHalf, rows = min(kHalf, a.Nq - i0);
                float *dst = a.dq_acc + (((long long)b * a.Nq + i0) * a.H + h) * D + (d & ~3);
                // the half's 64 rows of this dimension into registers first, so the columns are
                // free for the next tile's dP^T before the reductions are issued
                uint32_t qv[2][32];
#pragma unroll
                for (int c = 0; c < 2; ++c) ptx::tmem_ld32(lane_addr + 128 + hh * kHalf + 32 * c, qv[c]);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 2; ++c) ptx::reg_fence(qv[c]);
                ptx::tc_fence_before();
                ptx::mbar_arrive(&ctrl->dq_free[hh]);
                // rows 4m .. 4m + 3 of the half: after the transpose lane 4g + s holds dimensions
                // 4g .. 4g + 3 (of this warp's 32) of row 4m + s
#pragma unroll
                for (int m = 0; m < kHalf / 4; ++m) {
                    float x[4];
#pragma unroll
                    for (int t = 0; t < 4; ++t) x[t] = a.scale * __uint_as_float(qv[m / 8][4 * (m % 8) + t]);
                    transpose4(x, lane);
                    const int row = 4 * m + (lane & 3);
                    if (d < D && row < rows) red_add_v4(dst + row * row_stride, x[0], x[1], x[2], x[3]);
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

}  // namespace

attn_status_t launch_bwd_tc(const attn_bwd_params_t &p, float *dq_acc, const float *crow, const float *lrow,
                            cudaStream_t s) {
    const attn_fwd_params_t &f = p.fwd;
    CUtensorMap mq, mk, mv, mg;
    attn_status_t st;
    if (f.dk != f.dv || (f.dk != 64 && f.dk != 128))
        return fail(ATTN_ERR_UNSUPPORTED, "the tcgen05 backward supports dk == dv in {64, 128}");
    if ((st = encode(&mq, f.q, f.B, f.Nq, f.H, f.dk, f.q_stride, "q")) ||
        (st = encode(&mk, f.k, f.B, f.Nk, f.H, f.dk, f.k_stride, "k")) ||
        (st = encode(&mv, f.v, f.B, f.Nk, f.H, f.dv, f.v_stride, "v")) ||
        (st = encode(&mg, p.dout, f.B, f.Nq, f.H, f.dv, p.dout_stride, "dout")))
        return st;
    TcArgs a;
    a.B = (int)f.B; a.H = (int)f.H; a.Nq = (int)f.Nq; a.Nk = (int)f.Nk; a.causal = f.causal;
    a.scale = f.scale; a.scale_log2 = f.scale * kLog2e;
    a.crow = crow; a.lrow = lrow; a.nq_pad = (int)((f.Nq + 127) / 128 * 128);
    a.kv_lens = f.kv_lens; a.dq_acc = dq_acc;
    a.bias = f.bias;
    a.bs0 = f.bias_stride[0]; a.bs1 = f.bias_stride[1]; a.bs2 = f.bias_stride[2];
    {
        const int64_t sizes[3] = {f.B, f.H, f.Nq};
        bool pf = f.bias && (reinterpret_cast<uintptr_t>(f.bias) & 15u) == 0;
        for (int t = 0; t < 3; ++t) pf = pf && (sizes[t] <= 1 || f.bias_stride[t] % 4 == 0);
        a.bias_pf = pf ? 1 : 0;
    }
    a.dk = static_cast<__nv_bfloat16 *>(p.dk);
    a.dv = static_cast<__nv_bfloat16 *>(p.dv);
    a.dks0 = p.dk_stride[0]; a.dks1 = p.dk_stride[1]; a.dks2 = p.dk_stride[2];
    a.dvs0 = p.dv_stride[0]; a.dvs1 = p.dv_stride[1]; a.dvs2 = p.dv_stride[2];
    a.flags = device_flags();
    if (!a.flags) return fail(ATTN_ERR_CUDA, "could not resolve the device error word");
    bf16fwd::DropArgs dr{};
    fill_dropout(dr, f);
    const bool drop = dr.dmask || dr.rng;
    if (drop && f.bias) return fail(ATTN_ERR_UNSUPPORTED, "the backward of a dropout forward takes no bias");
    auto kernel = f.dk == 64 ? (drop     ? bwd_tc_kernel<true, 64, false>
                                : f.bias ? bwd_tc_kernel<false, 64, true>
                                         : bwd_tc_kernel<false, 64, false>)
                             : (drop     ? bwd_tc_kernel<true, 128, false>
                                : f.bias ? bwd_tc_kernel<false, 128, true>
                                         : bwd_tc_kernel<false, 128, false>);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    if ((f.Nk + BK - 1) / BK > 65535 || f.B > 65535)
        return fail(ATTN_ERR_UNSUPPORTED, "backward supports B <= 65535 and Nk <= %d", 65535 * BK);
    // programmatic stream serialization: CTAs may start (TMEM, barriers, the K, V, Q, dO
    // copies) while the prep kernel drains
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)f.H, (unsigned)f.B, (unsigned)((f.Nk + BK - 1) / BK));
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, mq, mk, mv, mg, a, dr);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "backward (tcgen05) launch: %s", cudaGetErrorString(e));
    return ATTN_OK;
}

}  // namespace attn
