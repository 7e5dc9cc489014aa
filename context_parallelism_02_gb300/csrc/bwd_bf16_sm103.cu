// bwd_bf16_sm103.cu -- ring-attention backward for sm_103a tensor cores.
//
// The pages state only that context parallelism leaves the gradients equal to
// single-device training ("Sequence and Context Parallelism", "What it does
// not change") and that activations are kept for the backward pass ("Sequence
// Parallelism in LLMs", "The Activation Memory Wall"); they give no backward
// algorithm.  This file computes the textbook gradient of attention with the
// saved lse, over the same (rank, ring step, tile) schedule as the forward:
//   P = exp(scale * q k^T - lse)   (masked by global positions)
//   Delta_i = rowsum(dO_i * out_i)
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - Delta)
//   dQ = scale * dS K,  dK = scale * dS^T Q
//
// Three launches:
//   bwd_delta  -- Delta (fp32) into the caller's workspace (HBM-bound).
//   bwd_dq     -- query-stationary: per 128-row query tile, walk the KV tiles
//                 of every ring step (as the forward does), S = Q K^T and
//                 dP = dO V^T into tensor memory, dS in bf16 back into tensor
//                 memory, dQ += dS K accumulated in tensor memory.
//   bwd_dkdv   -- key-stationary: per 128-key tile, walk the query tiles of
//                 every rank that holds it at some ring step, S^T = K Q^T and
//                 dP^T = V dO^T into tensor memory, P^T and dS^T in bf16 back
//                 into tensor memory, dV += P^T dO and dK += dS^T Q.
// Splitting dQ from dK/dV recomputes S and dP once more (7 tile MMAs per
// visible tile pair instead of 5) but needs no atomics: every output element
// is written once, and the result is deterministic.
//
// Roles of both tensor-core kernels (384 threads, three warpgroups): warp 0
// TMA producer (dQ: K tiles; warp 3 loads Q, dO and V), MMA issuers that run
// converged with one elected lane issuing (dQ: warps 1 and 2; dK/dV: warps 1,
// 2 and 3), warps 4-7 and 8-11 the elementwise gradient (dQ: the two
// 64-column halves of one 128x128 tile; dK/dV: one warpgroup per half-step
// buffer), one thread per tensor-memory lane.  Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "cp_common.cuh"
#include "kernels.h"
#include "tc_helpers.cuh"
#include "tmem_io.cuh"

namespace cp {

namespace {

using namespace tc;

constexpr int T = 128;             // tile rows (queries or keys)
constexpr int NTHREADS = 384;
constexpr int REGS_CTRL = 88;
constexpr int REGS_GRAD = 208;
static_assert(128 * REGS_CTRL + 256 * REGS_GRAD <= NTHREADS * 168, "register split exceeds the launch budget");
constexpr float LOG2E = 1.4426950408889634f;

template <int D>
struct Tile {
    static constexpr int BOXES = D / 64;
    static constexpr int BOX = 128 * 128;
    static constexpr int BYTES = BOXES * BOX;
};

// Unrolled issue sequences (compile-time offsets added to base descriptors
// inside the MMA asm): the MMA threads share their SM sub-partitions with busy
// gradient warps, so they spend as few instructions per MMA as possible.

// D/16 MMAs M=128, K=16, A and B K-major; A in 128-row boxes (16 KB), B in
// boxes of BOXB bytes (16 KB for 128 rows, 8 KB for 64)
template <int KK, int D, int BOXB>
__device__ __forceinline__ void ss_seq(uint32_t tD, uint64_t dA, uint64_t dB, uint32_t id)
{
    if constexpr (KK < D / 16) {
        constexpr uint32_t oa = (uint32_t)(((KK >> 2) * 16384 + (KK & 3) * 32) >> 4);
        constexpr uint32_t ob = (uint32_t)(((KK >> 2) * BOXB + (KK & 3) * 32) >> 4);
        mma_ss_off<oa, ob>(tD, dA, dB, id, KK > 0 ? 1u : 0u);
        ss_seq<KK + 1, D, BOXB>(tD, dA, dB, id);
    }
}

// D/16 MMAs M=128, K=16: A (bf16 pairs, 8 columns per 16 elements) from tensor
// memory, B K-major in 128-row boxes (16 KB)
template <int KK, int D>
__device__ __forceinline__ void ts_k_seq(uint32_t tD, uint32_t tA, uint64_t dB, uint32_t id)
{
    if constexpr (KK < D / 16) {
        constexpr uint32_t ob = (uint32_t)(((KK >> 2) * 16384 + (KK & 3) * 32) >> 4);
        mma_ts_off<ob>(tD, tA + (uint32_t)(KK * 8), dB, id, KK > 0 ? 1u : 0u);
        ts_k_seq<KK + 1, D>(tD, tA, dB, id);
    }
}

// NK MMAs M=128, N=D, K=16: A (bf16 pairs) from tensor memory, B MN-major
// (k-steps of 16 rows, 2048 B); A columns relative to tA: 8 KK (MAP 0), or
// 32 (KK/2) + 8 (KK%2) (MAP 1: two runs of 16 columns, 32 apart).
// acc0 = accumulate flag of the first MMA.
template <int KK, int NK, int MAP>
__device__ __forceinline__ void ts_mn_seq(uint32_t tD, uint32_t tA, uint64_t dB, uint32_t id,
                                          uint32_t acc0)
{
    if constexpr (KK < NK) {
        constexpr uint32_t acol = MAP == 0 ? (uint32_t)(KK * 8) : (uint32_t)(32 * (KK >> 1) + 8 * (KK & 1));
        constexpr uint32_t ob = (uint32_t)((KK * 2048) >> 4);
        mma_ts_off<ob>(tD, tA + acol, dB, id, KK == 0 ? acc0 : 1u);
        ts_mn_seq<KK + 1, NK, MAP>(tD, tA, dB, id, acc0);
    }
}

// ----------------------------------------------------------------------------- Delta

__global__ void __launch_bounds__(256) bwd_delta_kernel(const __nv_bfloat16 *__restrict__ out,
                                                        const __nv_bfloat16 *__restrict__ dout,
                                                        float *__restrict__ delta, int S, int Hq,
                                                        int D, int64_t rows)
{
    // one warp per (b, s, h) row, rows in BSHD order
    const int lane = threadIdx.x & 31;
    const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r = wid; r < rows; r += nw) {
        const __nv_bfloat16 *o = out + r * D;
        const __nv_bfloat16 *g = dout + r * D;
        float acc = 0.f;
        for (int d = lane * 4; d < D; d += 128) {
            const uint2 ov = *reinterpret_cast<const uint2 *>(o + d);
            const uint2 gv = *reinterpret_cast<const uint2 *>(g + d);
            const __nv_bfloat162 *o2 = reinterpret_cast<const __nv_bfloat162 *>(&ov);
            const __nv_bfloat162 *g2 = reinterpret_cast<const __nv_bfloat162 *>(&gv);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float2 a = __bfloat1622float2(o2[e]);
                const float2 b = __bfloat1622float2(g2[e]);
                acc = fmaf(a.x, b.x, acc);
                acc = fmaf(a.y, b.y, acc);
            }
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) {
            const int64_t h = r % Hq;
            const int64_t bs = r / Hq;   // b * S + s
            const int64_t b = bs / S, s = bs % S;
            delta[(b * Hq + h) * S + s] = acc;
        }
    }
}

// ----------------------------------------------------------------------------- dQ
//
// Query-stationary.  Tensor memory (columns): S [0,128), dP [128,256), the dQ
// accumulator [256, 256+D), dS in bf16 pairs [256+D, 320+D), the block's dO
// rows in bf16 pairs [320+D, 320+3D/2).  Shared memory holds the Q tile, four
// K stages and two V stages.  S = Q K^T reads both operands from shared
// memory; dP = dO V^T and dQ += dS K read their A operands from tensor memory
// (dO written there once by the gradient warps, dS on every tile), which
// halves the shared-memory reads of the dP MMAs.
//
// S(j) and dP(j) have their own barriers both ways, so S(j+1) is issued as
// soon as the gradient warps have read S(j) and runs while they read dP(j)
// and compute; dQ(j) comes last.  K_j is read by S(j) and by dQ(j); with the
// MMA order S(j+1), dP(j+1), dQ(j) the load of K(j+4) into the stage of K(j)
// has three tile groups of MMAs to land.

constexpr int Q_KST = 4;
enum {
    Q_QTM = 0,                   // Q tile landed
    Q_DOFULL = 1,                // dO rows in tensor memory (8 arrivals: the gradient warps)
    Q_KFULL = 2,                 // Q_KST stages
    Q_KEMPTY = 2 + Q_KST,        // Q_KST stages; commits after S(j) and after dQ(j)
    Q_VFULL = 2 + 2 * Q_KST,     // 2 stages
    Q_VEMPTY = 4 + 2 * Q_KST,    // 2 stages
    Q_SDONE = 6 + 2 * Q_KST,     // S(j) complete
    Q_PDONE = 7 + 2 * Q_KST,     // dP(j) complete
    Q_SFREE = 8 + 2 * Q_KST,     // S(j) read by the gradient warps (8 arrivals)
    Q_PFREE = 9 + 2 * Q_KST,     // dP(j) read (8 arrivals)
    Q_DS = 10 + 2 * Q_KST,       // dS(j) written (8 arrivals)
    Q_DSFREE = 11 + 2 * Q_KST,   // dQ(j) complete: the dS columns may be rewritten
    Q_FIN = 12 + 2 * Q_KST,
    Q_DRAIN = 13 + 2 * Q_KST,    // one commit per issuer (2)
    Q_NBAR = 14 + 2 * Q_KST
};

template <int D>
struct DqCfg {
    static constexpr int TB = Tile<D>::BYTES;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = TB;                    // Q_KST stages
    static constexpr int OFF_V = (1 + Q_KST) * TB;      // 2 stages
    static constexpr int OFF_BAR = (3 + Q_KST) * TB;
    static constexpr int OFF_MISC = OFF_BAR + 8 * Q_NBAR;
    static constexpr int NEED = OFF_MISC + 16;
    static constexpr int SMEM = NEED > 120 * 1024 ? NEED : 120 * 1024;
    static_assert(SMEM <= 232448, "dQ kernel shared memory");
    static constexpr uint32_t TM_S = 0, TM_P = 128, TM_DQ = 256, TM_DS = 256 + D, TM_DO = 320 + D;
    static_assert(TM_DO + D / 2 <= 512, "dQ kernel tensor memory");
};

// stage index and phase parity of a ring of NS buffers, advanced once per use
template <int NS>
struct Ring {
    int st = 0, ph = 0;
    __device__ __forceinline__ void next()
    {
        if (++st == NS) {
            st = 0;
            ph ^= 1;
        }
    }
};

struct BwdArgs {
    int B, Hq, Hkv, S, D, N, causal, layout;
    float scale;
    int upc;            // query units (128 rows) per chunk
    int tpc;            // key tiles per chunk
    unsigned *err;
    uint64_t limit_ns;   // pipeline waits
    uint64_t drain_ns;   // waits that drain copies and MMAs before exit
};

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                  const BwdArgs a, const float *__restrict__ lse,
                  const float *__restrict__ delta, __nv_bfloat16 *__restrict__ dq,
                  const __nv_bfloat16 *__restrict__ dout)
{
    using C = DqCfg<D>;
    constexpr int TB = C::TB;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_u32(smem_raw);
    if (base & 1023u) {   // the 128B-swizzled tiles need 1 KB alignment
        if (threadIdx.x == 0) atomicCAS(a.err, 0u, ERRW_SMEM_ALIGN);
        return;
    }
    const uint32_t sQ = base + C::OFF_Q, sK = base + C::OFF_K,
                   sV = base + C::OFF_V, bar0 = base + C::OFF_BAR;
#define BAR(i) (bar0 + 8u * (uint32_t)(i))
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem_raw + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem_raw + C::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Geom g = make_geom(a.S, a.N, a.layout, a.causal);
    const Unit w = decode_unit_grouped(g, a.B, a.Hq, a.upc, T, blockIdx.x);
    const int kvh = w.h / (a.Hq / a.Hkv);
    const int n = KvIter<T>::count(g, w.r, w.qmax);
    // extents of the tensor maps' (rank, row) dimensions, for the debug-bounds build
    const int map_r = striped(g) ? g.N : 1, map_rows = a.S / map_r;

    if (threadIdx.x == 0) {
        mbar_init(BAR(Q_QTM), 1);
        mbar_init(BAR(Q_DOFULL), 8);
        for (int i = 0; i < Q_KST; ++i) {
            mbar_init(BAR(Q_KFULL + i), 1);
            mbar_init(BAR(Q_KEMPTY + i), 2);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(BAR(Q_VFULL + i), 1);
            mbar_init(BAR(Q_VEMPTY + i), 1);
        }
        mbar_init(BAR(Q_SDONE), 1);
        mbar_init(BAR(Q_PDONE), 1);
        mbar_init(BAR(Q_SFREE), 8);
        mbar_init(BAR(Q_PFREE), 8);
        mbar_init(BAR(Q_DS), 8);
        mbar_init(BAR(Q_DSFREE), 1);
        mbar_init(BAR(Q_FIN), 1);
        mbar_init(BAR(Q_DRAIN), 2);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         smem_u32(tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl wc{a.err, abort_flag, a.limit_ns};

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_CTRL));
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------------------ K producer
            const uint64_t pol_kv = policy_evict_last();
            KvIter<T> it;
            it.begin(g, w.r, w.qmax);
            int nk = 0;
            Ring<Q_KST> kr;
            for (int j = 0; j < n; ++j, it.next(), kr.next()) {
                if (j >= Q_KST && !wait1(BAR(Q_KEMPTY + kr.st), kr.ph ^ 1, wc)) break;
                mbar_arrive_expect_tx(BAR(Q_KFULL + kr.st), TB);
                const int kmr = dbg_coord(a.err, it.mrank(), map_r), kmw = dbg_coord(a.err, it.mrow(), map_rows);
                for (int bx = 0; bx < D / 64; ++bx)
                    tma_load5(sK + kr.st * TB + bx * 16384, &tmK, BAR(Q_KFULL + kr.st), bx * 64, kvh,
                              kmr, kmw, w.b, pol_kv);
                ++nk;
            }
            {
                // wait (bounded) for the copies still in flight before the block
                // exits: always, since a consumer may give up after the last copy
                // was issued (after a normal run these phases are complete)
                volatile int no_abort = 0;
                WaitCtl dc{a.err, &no_abort, a.drain_ns};
                for (int j = nk > Q_KST ? nk - Q_KST : 0; j < nk; ++j)
                    wait1(BAR(Q_KFULL + j % Q_KST), (j / Q_KST) & 1, dc);
            }
        } else if (warp == 3 && lane == 0) {
            // ------------------------------------------------------------ dO and V producer
            const uint64_t pol_q = policy_evict_first(), pol_kv = policy_evict_last();
            const int qmr = dbg_coord(a.err, slot_mrank(g, w.q0), map_r);
            const int qmw = dbg_coord(a.err, slot_mrow(g, w.q0), map_rows);
            mbar_arrive_expect_tx(BAR(Q_QTM), TB);
            for (int bx = 0; bx < D / 64; ++bx)
                tma_load5(sQ + bx * 16384, &tmQ, BAR(Q_QTM), bx * 64, w.h, qmr, qmw, w.b, pol_q);
            KvIter<T> it;
            it.begin(g, w.r, w.qmax);
            int nv = 0;
            for (int j = 0; j < n; ++j, it.next()) {
                const int sv = j & 1;
                if (j >= 2 && !wait1(BAR(Q_VEMPTY + sv), ((j >> 1) - 1) & 1, wc)) break;
                mbar_arrive_expect_tx(BAR(Q_VFULL + sv), TB);
                const int vmr = dbg_coord(a.err, it.mrank(), map_r), vmw = dbg_coord(a.err, it.mrow(), map_rows);
                for (int bx = 0; bx < D / 64; ++bx)
                    tma_load5(sV + sv * TB + bx * 16384, &tmV, BAR(Q_VFULL + sv), bx * 64, kvh,
                              vmr, vmw, w.b, pol_kv);
                ++nv;
            }
            {
                volatile int no_abort = 0;
                WaitCtl dc{a.err, &no_abort, a.drain_ns};
                wait1(BAR(Q_QTM), 0, dc);
                for (int j = nv > 2 ? nv - 2 : 0; j < nv; ++j) wait1(BAR(Q_VFULL + (j & 1)), (j >> 1) & 1, dc);
            }
        } else if (warp == 1 || warp == 2) {
            // ------------------------------------------------------------ MMA issuers
            // warp 1: S = Q K^T (A = Q from tensor memory) and dP = dO V^T;
            // warp 2: dQ += dS K.  Each warp runs converged (warp-collective
            // waits), so its operands stay warp-uniform, and one elected lane
            // issues the MMAs and their commits.
            constexpr uint32_t idSP = idesc_bf16(128, T, false);     // K-major A and B
            constexpr uint32_t idDQ = idesc_bf16(128, D, true);      // B = K MN-major
            const uint32_t tS = tmem + C::TM_S, tP = tmem + C::TM_P, tDQ = tmem + C::TM_DQ,
                           tDS = tmem + C::TM_DS, tDO = tmem + C::TM_DO;
            const bool leader = elect_one();
            bool ok = true;
            if (warp == 1) {
                const uint64_t dQd = sdesc(sQ, 16, 1024);
                const uint64_t dK0 = sdesc(sK, 16, 1024), dV0 = sdesc(sV, 16, 1024);
                ok = waitw(BAR(Q_QTM), 0, wc) && waitw(BAR(Q_DOFULL), 0, wc);
                Ring<Q_KST> kr;
                for (int j = 0; ok && j < n; ++j, kr.next()) {
                    const int sv = j & 1;
                    if ((j > 0 && !waitw(BAR(Q_SFREE), (j - 1) & 1, wc)) ||
                        !waitw(BAR(Q_KFULL + kr.st), kr.ph, wc))
                        break;
                    const uint64_t dK = dK0 + (uint64_t)(kr.st * (TB >> 4));
                    if (leader) {
                        tc_fence_after();
                        ss_seq<0, D, 16384>(tS, dQd, dK, idSP);
                        mma_commit(BAR(Q_SDONE));
                        mma_commit(BAR(Q_KEMPTY + kr.st));
                    }
                    __syncwarp();
                    if ((j > 0 && !waitw(BAR(Q_PFREE), (j - 1) & 1, wc)) ||
                        !waitw(BAR(Q_VFULL + sv), (j >> 1) & 1, wc))
                        break;
                    const uint64_t dV = dV0 + (uint64_t)(sv * (TB >> 4));
                    if (leader) {
                        tc_fence_after();
                        ts_k_seq<0, D>(tP, tDO, dV, idSP);   // A = dO from tensor memory
                        mma_commit(BAR(Q_PDONE));
                        mma_commit(BAR(Q_VEMPTY + sv));
                    }
                    __syncwarp();
                }
            } else {
                const uint64_t dKmn0 = sdesc(sK, 16384, 1024);
                Ring<Q_KST> kr;
                for (int j = 0; ok && j < n; ++j, kr.next()) {
                    if (!waitw(BAR(Q_DS), j & 1, wc) || !waitw(BAR(Q_KFULL + kr.st), kr.ph, wc))
                        break;
                    const uint64_t dK = dKmn0 + (uint64_t)(kr.st * (TB >> 4));
                    const uint32_t acc0 = j > 0 ? 1u : 0u;
                    if (leader) {
                        tc_fence_after();
                        ts_mn_seq<0, T / 16, 0>(tDQ, tDS, dK, idDQ, acc0);
                        mma_commit(BAR(Q_KEMPTY + kr.st));
                        mma_commit(BAR(Q_DSFREE));
                        if (j + 1 == n) mma_commit(BAR(Q_FIN));
                    }
                    __syncwarp();
                }
            }
            if (leader) mma_commit(BAR(Q_DRAIN));
            __syncwarp();
            volatile int no_abort = 0;
            WaitCtl dc{a.err, &no_abort, a.drain_ns};
            waitw(BAR(Q_DRAIN), 0, dc);
        }
        __syncwarp();
        tc_fence_before();
        asm volatile("barrier.sync 1, %0;" ::"n"(NTHREADS) : "memory");
        if (warp == 0) {
            tc_fence_after();
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
        }
        return;
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_GRAD));
        // ------------------------------------------------------------ dS = P (dP - Delta)
        const int half = (warp - 4) >> 2;             // columns [64*half, 64*half+64)
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + C::TM_S + 64u * half;
        const uint32_t tP = tmem + lane_off + C::TM_P + 64u * half;
        const uint32_t tDQ = tmem + lane_off + C::TM_DQ;
        const uint32_t tDS = tmem + lane_off + C::TM_DS + 32u * half;
        const int qpos = w.q0 + row;                  // slot
        const bool valid = qpos < w.cend;
        const int qp = dbg_coord(a.err, valid ? slot_pos(g, qpos) : 0, a.S);   // global position
        const float sl2 = a.scale * LOG2E;
        float lse2 = 0.f, dlt = 0.f;
        if (valid) {
            lse2 = lse[((int64_t)w.b * a.Hq + w.h) * a.S + qp] * LOG2E;
            dlt = delta[((int64_t)w.b * a.Hq + w.h) * a.S + qp];
        }
        {
            // this half's D/2 elements of the row's dO, as D/4 bf16 pairs, into the
            // A operand of dP = dO V^T (rows past the unit's chunk are zero; their
            // results are never stored)
            uint32_t dv4[D / 4];
            if (valid) {
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    dout + (((int64_t)w.b * a.S + qp) * a.Hq + w.h) * D + (D / 2) * half);
#pragma unroll
                for (int i = 0; i < D / 16; ++i) {
                    const uint4 x = src[i];
                    dv4[4 * i] = x.x;
                    dv4[4 * i + 1] = x.y;
                    dv4[4 * i + 2] = x.z;
                    dv4[4 * i + 3] = x.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < D / 4; ++i) dv4[i] = 0u;
            }
            const uint32_t tDO = tmem + lane_off + C::TM_DO + (uint32_t)(D / 4) * half;
            if constexpr (D == 128)
                tmem_st_x32(tDO, dv4);
            else
                tmem_st_x16(tDO, dv4);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(Q_DOFULL));
        }
        bool ok = true;
        KvIter<T> it;
        it.begin(g, w.r, w.qmax);
        for (int j = 0; j < n; ++j, it.next()) {
            const int ks = it.start(), kl = it.len();
            int lim = kl;                              // visible columns [0, lim) of the tile
            if (a.causal) {
                const int c = qpos - ks + 1 + it.shift;
                lim = c < lim ? c : lim;
            }
            lim -= 64 * half;                          // in this half's local columns
            if (!waitw(BAR(Q_SDONE), j & 1, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[64];
            tmem_ld_x64(tS, sr);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(Q_SFREE));   // S(j+1) may be issued
            // P = exp2(S sl2 - lse2); the per-element mask only where some row of
            // the warp does not see the whole half tile
            const bool full = __all_sync(0xffffffffu, lim >= 64);
            float p[64];
#pragma unroll
            for (int e = 0; e < 64; e += 2) {
                ffma2(p[e], p[e + 1], __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]), sl2, -lse2);
                p[e] = ex2(p[e]);
                p[e + 1] = ex2(p[e + 1]);
            }
            if (!full) {
#pragma unroll
                for (int e = 0; e < 64; ++e) p[e] = e < lim ? p[e] : 0.f;
            }
            if (!waitw(BAR(Q_PDONE), j & 1, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t pr[64];
            tmem_ld_x64(tP, pr);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(Q_PFREE));   // dP(j+1) may be issued
            // dS = P (dP - Delta)
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                float t0, t1;
                fadd2v(t0, t1, __uint_as_float(pr[2 * e]), __uint_as_float(pr[2 * e + 1]), -dlt, -dlt);
                fmul2v(t0, t1, t0, t1, p[2 * e], p[2 * e + 1]);
                pk[e] = pack_bf16(t0, t1);
            }
            // dS(j) may be written once dQ(j-1) has read dS(j-1)
            if (j > 0 && !waitw(BAR(Q_DSFREE), (j - 1) & 1, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            tmem_st_x32(tDS, pk);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(Q_DS));
        }
        if (ok && waitw(BAR(Q_FIN), 0, wc)) {
            tc_fence_after();
            // each half writes D/2 columns of dQ = scale * acc
            constexpr int HD = D / 2;
            __nv_bfloat16 *orow = dq + (((int64_t)w.b * a.S + qp) * a.Hq + w.h) * D + HD * half;
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t o[32];
                tmem_ld_x32(tDQ + HD * half + 32u * c, o);
                if (valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * c);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        uint4 pkt;
                        pkt.x = pack_bf16(__uint_as_float(o[8 * v4 + 0]) * a.scale, __uint_as_float(o[8 * v4 + 1]) * a.scale);
                        pkt.y = pack_bf16(__uint_as_float(o[8 * v4 + 2]) * a.scale, __uint_as_float(o[8 * v4 + 3]) * a.scale);
                        pkt.z = pack_bf16(__uint_as_float(o[8 * v4 + 4]) * a.scale, __uint_as_float(o[8 * v4 + 5]) * a.scale);
                        pkt.w = pack_bf16(__uint_as_float(o[8 * v4 + 6]) * a.scale, __uint_as_float(o[8 * v4 + 7]) * a.scale);
                        dst[v4] = pkt;
                    }
                }
            }
        }
        __syncwarp();
        tc_fence_before();
        asm volatile("barrier.sync 1, %0;" ::"n"(NTHREADS) : "memory");
        return;
    }
#undef BAR
}

// ----------------------------------------------------------------------------- dK, dV
//
// Key-stationary, in half tiles of 64 queries: for each query tile the block
// visits (QIter order), two half steps s.  Per half step: S^T = K Q_s^T and
// dP^T = V dO_s^T (M=128 keys, N=64) into tensor-memory buffer s%2; gradient
// warpgroup s%2 turns them into P^T and dS^T (bf16 pairs, written over the
// first half of the columns it read); then dV += P^T dO_s and dK += dS^T Q_s
// (N=D, K=64).  With two buffers and one warpgroup per buffer, the MMAs of
// step s+1 run while warpgroup s%2 works on step s.  S^T and dP^T have
// barriers of their own: S^T(s+2) is issued into buffer s%2 once dV(s) has
// read P^T(s) out of the S^T columns, dP^T(s+2) once dK(s) has read dS^T(s)
// out of the dP^T columns (commit barriers, since the MMA groups come from
// different issuing warps), and the gradient warps turn S^T into P^T before
// they wait for dP^T.  A buffer's serial chain is then P^T -> dV -> S^T of
// the step after next, without the dS^T and dK stages.
// Each gradient thread handles all 64 columns of its steps, so it moves them
// with two 64-column tensor-memory loads and two 32-column stores.
//
// Tensor memory (columns): buffer x at 128x: S^T [0,64), dP^T [64,128);
// dV [256, 256+D), dK [256+D, 256+2D).  Shared memory: K and V (128 rows),
// K_QST half stages of (Q_s, dO_s) 64-row tiles, and their lse / Delta.

constexpr int K_QST = 5;
enum {
    K_KVFULL = 0,
    K_QFULL = 1,                  // K_QST half stages
    K_QEMPTY = 1 + K_QST,         // K_QST half stages
    K_S = 1 + 2 * K_QST,          // 2 buffers: S^T complete
    K_PW = 3 + 2 * K_QST,         // 2 buffers: P^T written (4 arrivals: one warpgroup)
    K_SFREE = 5 + 2 * K_QST,      // 2 buffers: dV(s) complete, the S^T columns may be rewritten
    K_FIN = 7 + 2 * K_QST,
    K_DRAIN = 8 + 2 * K_QST,      // one commit per issuing warp (3)
    K_DSW = 9 + 2 * K_QST,        // 2 buffers: dS^T written (4 arrivals)
    K_DP = 11 + 2 * K_QST,        // 2 buffers: dP^T complete
    K_DPFREE = 13 + 2 * K_QST,    // 2 buffers: dK(s) complete, the dP^T columns may be rewritten
    K_NBAR = 15 + 2 * K_QST
};

template <int D>
struct DkvCfg {
    static constexpr int TB = Tile<D>::BYTES;            // 128 rows
    static constexpr int HB = TB / 2;                    // 64 rows
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = TB;
    static constexpr int OFF_Q = 2 * TB;                 // K_QST stages of (Q_s, dO_s)
    static constexpr int STAGE = 2 * HB;
    static constexpr int OFF_STAT = OFF_Q + K_QST * STAGE;   // K_QST x (lse2[64], delta[64]) fp32
    static constexpr int OFF_BAR = OFF_STAT + K_QST * 2 * 64 * 4;
    static constexpr int OFF_MISC = OFF_BAR + 8 * K_NBAR;
    static constexpr int NEED = OFF_MISC + 16;
    static constexpr int SMEM = NEED > 120 * 1024 ? NEED : 120 * 1024;
    static_assert(SMEM <= 232448, "dK/dV kernel shared memory");
    static constexpr uint32_t TM_DV = 256, TM_DK = 256 + D;
    static_assert(TM_DK + D <= 512, "dK/dV kernel tensor memory");
};

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQh, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDOh,
                    const BwdArgs a, const float *__restrict__ lse, const float *__restrict__ delta,
                    __nv_bfloat16 *__restrict__ dk, __nv_bfloat16 *__restrict__ dv)
{
    using C = DkvCfg<D>;
    constexpr int TB = C::TB, HB = C::HB;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_u32(smem_raw);
    if (base & 1023u) {   // the 128B-swizzled tiles need 1 KB alignment
        if (threadIdx.x == 0) atomicCAS(a.err, 0u, ERRW_SMEM_ALIGN);
        return;
    }
    const uint32_t sK = base + C::OFF_K, sV = base + C::OFF_V, sQ = base + C::OFF_Q,
                   bar0 = base + C::OFF_BAR;
    float *stat = reinterpret_cast<float *>(smem_raw + C::OFF_STAT);   // [stage][lse2 | delta][64]
#define BAR(i) (bar0 + 8u * (uint32_t)(i))
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem_raw + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem_raw + C::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Geom g = make_geom(a.S, a.N, a.layout, a.causal);
    const KvUnit w = decode_kv_unit<T>(g, a.B, a.Hkv, a.tpc, blockIdx.x);
    const int grp = a.Hq / a.Hkv;
    // extents of the tensor maps' (rank, row) dimensions, for the debug-bounds build
    const int map_r = striped(g) ? g.N : 1, map_rows = a.S / map_r;
    const int ns = 2 * QIter<T>::count(g, w.src, w.ks, grp);   // half steps

    if (threadIdx.x == 0) {
        mbar_init(BAR(K_KVFULL), 1);
        for (int i = 0; i < K_QST; ++i) {
            mbar_init(BAR(K_QFULL + i), 1);
            mbar_init(BAR(K_QEMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(BAR(K_S + i), 1);
            mbar_init(BAR(K_DP + i), 1);
            mbar_init(BAR(K_PW + i), 4);
            mbar_init(BAR(K_DSW + i), 4);
            mbar_init(BAR(K_SFREE + i), 1);
            mbar_init(BAR(K_DPFREE + i), 1);
        }
        mbar_init(BAR(K_FIN), 1);
        mbar_init(BAR(K_DRAIN), 3);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         smem_u32(tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl wc{a.err, abort_flag, a.limit_ns};

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_CTRL));
        if (warp == 0) {
            // ------------------------------------------------------------ producer (whole warp)
            const uint64_t pol_kv = policy_evict_first(), pol_q = policy_evict_last();
            if (lane == 0) {
                const int kmr = dbg_coord(a.err, slot_mrank(g, w.ks), map_r);
                const int kmw = dbg_coord(a.err, slot_mrow(g, w.ks), map_rows);
                mbar_arrive_expect_tx(BAR(K_KVFULL), 2 * TB);
                for (int bx = 0; bx < D / 64; ++bx) {
                    tma_load5(sK + bx * 16384, &tmK, BAR(K_KVFULL), bx * 64, w.g, kmr, kmw, w.b, pol_kv);
                    tma_load5(sV + bx * 16384, &tmV, BAR(K_KVFULL), bx * 64, w.g, kmr, kmw, w.b, pol_kv);
                }
            }
            QIter<T> it;
            it.begin(g, w.src, w.ks, w.g * grp, grp);
            int issued = 0;
            Ring<K_QST> qr;
            for (int s = 0; s < ns; ++s, qr.next()) {
                if (s >= K_QST && !waitw(BAR(K_QEMPTY + qr.st), qr.ph ^ 1, wc)) break;
                const int hs = s & 1;
                const int qa = it.start() + 64 * hs, ql = it.len() - 64 * hs, h = it.head();
                // map coordinates; the second half-tile may start past the end of
                // the map (a short last tile): the copy then reads the fill value
                const int qr_rank = dbg_coord(a.err, it.mrank(), map_r);
                const int qr_row = dbg_coord(a.err, it.mrow(), map_rows) + 64 * hs;
                // per-row statistics of the half tile, negated: -lse (log2 units), -Delta
                float *ls = stat + qr.st * 128, *dl = ls + 64;
                for (int e = lane; e < 64; e += 32) {
                    float l2 = 0.f, dd = 0.f;
                    if (e < ql) {
                        const int64_t off =
                            ((int64_t)w.b * a.Hq + h) * a.S + dbg_coord(a.err, slot_pos(g, qa + e), a.S);
                        l2 = -lse[off] * LOG2E;
                        dd = -delta[off];
                    }
                    ls[e] = l2;
                    dl[e] = dd;
                }
                __syncwarp();
                if (lane == 0) {
                    const uint32_t sq = sQ + qr.st * C::STAGE;
                    mbar_arrive_expect_tx(BAR(K_QFULL + qr.st), 2 * HB);
                    for (int bx = 0; bx < D / 64; ++bx) {
                        tma_load5(sq + bx * 8192, &tmQh, BAR(K_QFULL + qr.st), bx * 64, h, qr_rank,
                                  qr_row, w.b, pol_q);
                        tma_load5(sq + HB + bx * 8192, &tmDOh, BAR(K_QFULL + qr.st), bx * 64, h, qr_rank,
                                  qr_row, w.b, pol_q);
                    }
                }
                __syncwarp();
                issued = s + 1;
                if (hs) it.next();
            }
            if (lane == 0) {
                // wait (bounded) for the copies still in flight before the block
                // exits: always, since a consumer may give up after the last copy
                // was issued (after a normal run these phases are complete)
                volatile int no_abort = 0;
                WaitCtl dc{a.err, &no_abort, a.drain_ns};
                wait1(BAR(K_KVFULL), 0, dc);
                for (int s = issued > K_QST ? issued - K_QST : 0; s < issued; ++s)
                    wait1(BAR(K_QFULL + s % K_QST), (s / K_QST) & 1, dc);
            }
        } else {
            // ------------------------------------------------------------ MMA issuers
            // Three issuing warps, so that a wait of one never leaves the tensor
            // pipe without work from the others: warp 2 issues S^T(s) into buffer
            // s%2 once dV(s-2) has read P^T(s-2) out of those columns, warp 3
            // dP^T(s) once dK(s-2) has read dS^T(s-2), and warp 1 dV(s) and dK(s)
            // once the gradient warpgroup has written P^T(s) and dS^T(s).  Each
            // warp runs converged (warp-collective waits), so its operands stay
            // warp-uniform, and one elected lane issues the MMAs and commits.
            const bool leader = elect_one();
            bool ok = waitw(BAR(K_KVFULL), 0, wc);
            if (warp >= 2) {
                constexpr uint32_t idSP = idesc_bf16(128, 64, false);   // N = 64 queries
                // warp 2: S^T = K Q_s^T; warp 3: dP^T = V dO_s^T
                const bool dp = warp == 3;
                const uint64_t dA = sdesc(dp ? sV : sK, 16, 1024);
                const uint64_t dQ0 = sdesc(sQ, 16, 1024) + (dp ? (uint64_t)(HB >> 4) : 0);   // Q_s / dO_s K-major
                const int b_free = dp ? K_DPFREE : K_SFREE, b_done = dp ? K_DP : K_S;
                const uint32_t col = dp ? 64u : 0u;
                Ring<K_QST> rs;
                for (int s = 0; ok && s < ns; ++s, rs.next()) {
                    if ((s >= 2 && !waitw(BAR(b_free + (s & 1)), ((s >> 1) - 1) & 1, wc)) ||
                        !waitw(BAR(K_QFULL + rs.st), rs.ph, wc))
                        break;
                    const uint32_t tb = tmem + 128u * (uint32_t)(s & 1) + col;
                    const uint64_t so = (uint64_t)(rs.st * (C::STAGE >> 4));
                    if (leader) {
                        tc_fence_after();
                        ss_seq<0, D, 8192>(tb, dA, dQ0 + so, idSP);
                        mma_commit(BAR(b_done + (s & 1)));
                    }
                    __syncwarp();
                }
            } else {
                constexpr uint32_t idKV = idesc_bf16(128, D, true);     // dV, dK: B MN-major
                const uint64_t dQmn0 = sdesc(sQ, 8192, 1024);          // Q_s, dO_s MN-major
                const uint32_t tDV = tmem + C::TM_DV, tDK = tmem + C::TM_DK;
                Ring<K_QST> rs;
                for (int s = 0; ok && s < ns; ++s, rs.next()) {
                    if (!waitw(BAR(K_PW + (s & 1)), (s >> 1) & 1, wc)) break;
                    const uint32_t tb = tmem + 128u * (uint32_t)(s & 1);
                    const uint64_t so = (uint64_t)(rs.st * (C::STAGE >> 4));
                    const uint32_t acc0 = s > 0 ? 1u : 0u;
                    // dV += P^T dO_s as soon as P^T is written, while the gradient
                    // warps compute dS^T; then dK += dS^T Q_s (K = 64 queries: 4 MMAs each)
                    if (leader) {
                        tc_fence_after();
                        ts_mn_seq<0, 4, 0>(tDV, tb, dQmn0 + so + (uint64_t)(HB >> 4), idKV, acc0);
                        mma_commit(BAR(K_SFREE + (s & 1)));
                    }
                    __syncwarp();
                    if (!waitw(BAR(K_DSW + (s & 1)), (s >> 1) & 1, wc)) break;
                    if (leader) {
                        tc_fence_after();
                        ts_mn_seq<0, 4, 0>(tDK, tb + 64u, dQmn0 + so, idKV, acc0);
                        // S^T(s) and dP^T(s) completed before the gradient warps read
                        // them, so the stage is free once dV/dK(s) complete
                        mma_commit(BAR(K_QEMPTY + rs.st));
                        mma_commit(BAR(K_DPFREE + (s & 1)));
                    }
                    __syncwarp();
                }
                if (leader) mma_commit(BAR(K_FIN));
                __syncwarp();
            }
            if (leader) mma_commit(BAR(K_DRAIN));
            __syncwarp();
            volatile int no_abort = 0;
            WaitCtl dc{a.err, &no_abort, a.drain_ns};
            waitw(BAR(K_DRAIN), 0, dc);
        }
        __syncwarp();
        tc_fence_before();
        asm volatile("barrier.sync 1, %0;" ::"n"(NTHREADS) : "memory");
        if (warp == 0) {
            tc_fence_after();
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
        }
        return;
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_GRAD));
        // ------------------------------------------------------------ P^T, dS^T
        const int half = (warp - 4) >> 2;           // warpgroup: half steps s with s % 2 == half
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;        // key row of the tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tb = tmem + lane_off + 128u * (uint32_t)half;
        const int kpos = w.ks + row;
        const float sl2 = a.scale * LOG2E;
        bool ok = true;
        QIter<T> it;
        it.begin(g, w.src, w.ks, w.g * grp, grp);
        Ring<K_QST> qr;
        if (half) qr.next();
        for (int i = 0; 2 * i + half < ns; ++i, it.next(), qr.next(), qr.next()) {
            const int qa = it.start() + 64 * half, ql = it.len() - 64 * half, sh = it.shift;
            if (!waitw(BAR(K_S + half), i & 1, wc) || !waitw(BAR(K_QFULL + qr.st), qr.ph, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[64], pr[64];
            tmem_ld_x64(tb, sr);
            // visible query columns c: c < ql and (not causal or qa + c >= kpos)
            const int lo = a.causal ? kpos - sh - qa : 0;
            const float4 *ls4 = reinterpret_cast<const float4 *>(stat + qr.st * 128);   // -lse2
            const float4 *dl4 = ls4 + 16;                                               // -Delta
            // most tiles are visible to the whole warp: no per-element mask there
            const bool full = __all_sync(0xffffffffu, lo <= 0 && ql >= 64);
            // P^T (fp32, kept in place of S^T for dS^T) and its bf16 pairs, stored
            // at once so that their registers are free for dS^T
            {
                uint32_t pp[32];
#pragma unroll
                for (int e4 = 0; e4 < 16; ++e4) {
                    const float4 l = ls4[e4];
                    const int c = 4 * e4;
                    float p0, p1, p2, p3;
                    ffma2v(p0, p1, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]), sl2, sl2, l.x, l.y);
                    ffma2v(p2, p3, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]), sl2, sl2, l.z, l.w);
                    p0 = ex2(p0);
                    p1 = ex2(p1);
                    p2 = ex2(p2);
                    p3 = ex2(p3);
                    if (!full) {
                        p0 = (c >= lo && c < ql) ? p0 : 0.f;
                        p1 = (c + 1 >= lo && c + 1 < ql) ? p1 : 0.f;
                        p2 = (c + 2 >= lo && c + 2 < ql) ? p2 : 0.f;
                        p3 = (c + 3 >= lo && c + 3 < ql) ? p3 : 0.f;
                    }
                    sr[c] = __float_as_uint(p0);
                    sr[c + 1] = __float_as_uint(p1);
                    sr[c + 2] = __float_as_uint(p2);
                    sr[c + 3] = __float_as_uint(p3);
                    pp[2 * e4] = pack_bf16(p0, p1);
                    pp[2 * e4 + 1] = pack_bf16(p2, p3);
                }
                tmem_st_x32(tb, pp);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(K_PW + half));   // dV(s) may start
            }
            if (!waitw(BAR(K_DP + half), i & 1, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            tmem_ld_x64(tb + 64u, pr);
            {
                // dS^T = P^T (dP^T - Delta)
                uint32_t dd[32];
#pragma unroll
                for (int e4 = 0; e4 < 16; ++e4) {
                    const float4 d = dl4[e4];
                    const int c = 4 * e4;
                    float t0, t1, t2, t3;
                    fadd2v(t0, t1, __uint_as_float(pr[c]), __uint_as_float(pr[c + 1]), d.x, d.y);
                    fadd2v(t2, t3, __uint_as_float(pr[c + 2]), __uint_as_float(pr[c + 3]), d.z, d.w);
                    fmul2v(t0, t1, t0, t1, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
                    fmul2v(t2, t3, t2, t3, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
                    dd[2 * e4] = pack_bf16(t0, t1);
                    dd[2 * e4 + 1] = pack_bf16(t2, t3);
                }
                tmem_st_x32(tb + 64u, dd);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(K_DSW + half));
        }
        if (ok && waitw(BAR(K_FIN), 0, wc)) {
            tc_fence_after();
            // half 0 writes dV, half 1 writes dK (times scale)
            const bool valid = row < w.kl;
            const float f = half ? a.scale : 1.f;
            const uint32_t tAcc = tmem + lane_off + (half ? C::TM_DK : C::TM_DV);
            __nv_bfloat16 *orow =
                (half ? dk : dv) + (((int64_t)w.b * a.S + dbg_coord(a.err, valid ? slot_pos(g, kpos) : 0, a.S)) * a.Hkv + w.g) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld_x32(tAcc + 32u * c, o);
                if (valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * c);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        uint4 pkt;
                        pkt.x = pack_bf16(__uint_as_float(o[8 * v4 + 0]) * f, __uint_as_float(o[8 * v4 + 1]) * f);
                        pkt.y = pack_bf16(__uint_as_float(o[8 * v4 + 2]) * f, __uint_as_float(o[8 * v4 + 3]) * f);
                        pkt.z = pack_bf16(__uint_as_float(o[8 * v4 + 4]) * f, __uint_as_float(o[8 * v4 + 5]) * f);
                        pkt.w = pack_bf16(__uint_as_float(o[8 * v4 + 6]) * f, __uint_as_float(o[8 * v4 + 7]) * f);
                        dst[v4] = pkt;
                    }
                }
            }
        }
        __syncwarp();
        tc_fence_before();
        asm volatile("barrier.sync 1, %0;" ::"n"(NTHREADS) : "memory");
        return;
    }
#undef BAR
}

template <int D>
int launch_bwd_d(const BwdPtrs &p, BwdArgs a, cudaStream_t st)
{
    CUtensorMap mk, mv, mdo, mq, mq64, mdo64;
    const int R = a.layout == CP_LAYOUT_STRIPED ? a.N : 1;
    if (!make_map(&mk, p.k, a.B, a.S, a.Hkv, D, 128, R) || !make_map(&mv, p.v, a.B, a.S, a.Hkv, D, 128, R) ||
        !make_map(&mdo, p.dout, a.B, a.S, a.Hq, D, 128, R) || !make_map(&mq, p.q, a.B, a.S, a.Hq, D, 128, R) ||
        !make_map(&mq64, p.q, a.B, a.S, a.Hq, D, 64, R) || !make_map(&mdo64, p.dout, a.B, a.S, a.Hq, D, 64, R))
        return CP_ECUDA;
    static bool attr_done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CP_ECUDA;
    if (dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 DqCfg<D>::SMEM) != cudaSuccess ||
            cudaFuncSetAttribute(bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 DkvCfg<D>::SMEM) != cudaSuccess)
            return CP_ECUDA;
        attr_done[dev] = true;
    }
    const Geom g = make_geom(a.S, a.N, a.layout, a.causal);
    float *delta = static_cast<float *>(p.workspace);

    // Delta = rowsum(dO * out)
    const int64_t rows = (int64_t)a.B * a.S * a.Hq;
    int64_t blocks = (rows + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    bwd_delta_kernel<<<(unsigned)blocks, 256, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(p.out), static_cast<const __nv_bfloat16 *>(p.dout), delta,
        a.S, a.Hq, D, rows);
    if (cudaGetLastError() != cudaSuccess) return CP_ECUDA;

    a.upc = (g.clen + T - 1) / T;
    a.tpc = (g.clen + T - 1) / T;
    const int64_t qunits = (int64_t)g.N * g.cpr * a.upc * a.B * a.Hq;
    const int64_t kunits = (int64_t)g.N * g.cpr * a.tpc * a.B * a.Hkv;
    if (qunits > 0x7fffffffLL || kunits > 0x7fffffffLL) return CP_EUNSUPPORTED;
    bwd_dq_kernel<D><<<(unsigned)qunits, NTHREADS, DqCfg<D>::SMEM, st>>>(
        mq, mk, mv, mdo, a, p.lse, delta,
        static_cast<__nv_bfloat16 *>(p.dq), static_cast<const __nv_bfloat16 *>(p.dout));
    if (cudaGetLastError() != cudaSuccess) return CP_ECUDA;
    bwd_dkdv_kernel<D><<<(unsigned)kunits, NTHREADS, DkvCfg<D>::SMEM, st>>>(
        mq64, mk, mv, mdo64, a, p.lse, delta, static_cast<__nv_bfloat16 *>(p.dk),
        static_cast<__nv_bfloat16 *>(p.dv));
    return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ECUDA;
}

}  // namespace

size_t bwd_workspace_bytes(int B, int Hq, int64_t S)
{
    // Delta: B*Hq*S fp32, rounded up to 256 bytes
    const size_t b = (size_t)B * (size_t)Hq * (size_t)S * 4u;
    return (b + 255u) & ~(size_t)255u;
}

int launch_bwd_bf16(const BwdPtrs &p, const FwdArgs &f, cudaStream_t st)
{
    BwdArgs a;
    a.B = f.B;
    a.Hq = f.Hq;
    a.Hkv = f.Hkv;
    a.S = f.S;
    a.D = f.D;
    a.N = f.N;
    a.causal = f.causal;
    a.layout = f.layout;
    a.scale = f.scale;
    a.upc = a.tpc = 0;
    a.err = f.err;
    a.limit_ns = f.limit_ns;
    a.drain_ns = f.drain_ns;
    if (f.D == 64) return launch_bwd_d<64>(p, a, st);
    if (f.D == 128) return launch_bwd_d<128>(p, a, st);
    return CP_EUNSUPPORTED;
}

}  // namespace cp
