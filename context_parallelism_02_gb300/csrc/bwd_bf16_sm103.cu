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
// TMA producer, warp 1 MMA issuer, warps 2-3 idle, warps 4-7 and 8-11 the two
// halves (64 columns each) of the elementwise gradient of one 128x128 tile, one
// thread per tensor-memory lane.  Every wait is bounded.
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
constexpr int REGS_CTRL = 56;
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
// inside the MMA asm): the MMA thread shares its SM sub-partition with busy
// gradient warps, so it must spend as few instructions per MMA as possible.

// D/16 MMAs M=128, N=128, K=16, A and B K-major (128-row boxes of 16 KB)
template <int KK, int D>
__device__ __forceinline__ void ss_seq(uint32_t tD, uint64_t dA, uint64_t dB, uint32_t id)
{
    if constexpr (KK < D / 16) {
        constexpr uint32_t o = (uint32_t)(((KK >> 2) * 16384 + (KK & 3) * 32) >> 4);
        mma_ss_off<o, o>(tD, dA, dB, id, KK > 0 ? 1u : 0u);
        ss_seq<KK + 1, D>(tD, dA, dB, id);
    }
}

// 8 MMAs M=128, N=D, K=16: A (bf16 pairs) from tensor memory -- columns
// [0,32) and [64,96) relative to tA, or [0,64) if CONTIG -- and B MN-major;
// acc0 = accumulate flag of the first
template <int KK, bool CONTIG = false>
__device__ __forceinline__ void ts_seq(uint32_t tD, uint32_t tA, uint64_t dB, uint32_t id,
                                       uint32_t acc0)
{
    if constexpr (KK < T / 16) {
        constexpr uint32_t acol =
            (CONTIG || KK < 4) ? (uint32_t)(KK * 8) : (uint32_t)(64 + (KK - 4) * 8);
        constexpr uint32_t ob = (uint32_t)((KK * 16 * 128) >> 4);
        mma_ts_off<ob>(tD, tA + acol, dB, id, KK == 0 ? acc0 : 1u);
        ts_seq<KK + 1, CONTIG>(tD, tA, dB, id, acc0);
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

enum {
    Q_QFULL = 0,
    Q_KFULL = 1,
    Q_KEMPTY = 3,
    Q_VFULL = 5,
    Q_VEMPTY = 7,
    Q_SDP = 9,
    Q_DS = 10,       // one arrival per gradient warp (8): dS(j) written
    Q_FIN = 11,
    Q_DRAIN = 12,    // one commit per issuer (2)
    Q_SDPFREE = 13,  // one arrival per gradient warp (8): S(j), dP(j) read
    Q_DSFREE = 14,   // dQ(j) complete: the dS columns may be rewritten
    Q_NBAR = 15
};

template <int D>
struct DqCfg {
    static constexpr int TB = Tile<D>::BYTES;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_DO = TB;
    static constexpr int OFF_K = 2 * TB;     // 2 stages
    static constexpr int OFF_V = 4 * TB;     // 2 stages
    static constexpr int OFF_BAR = 6 * TB;
    static constexpr int OFF_MISC = OFF_BAR + 8 * Q_NBAR;
    static constexpr int NEED = OFF_MISC + 16 + 1024;
    static constexpr int SMEM = NEED > 120 * 1024 ? NEED : 120 * 1024;
};

struct BwdArgs {
    int B, Hq, Hkv, S, D, N, causal, layout;
    float scale;
    int upc;            // query units (128 rows) per chunk
    int tpc;            // key tiles per chunk
    unsigned *err;
    uint64_t limit_ns;
};

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                  const BwdArgs a, const float *__restrict__ lse, const float *__restrict__ delta,
                  __nv_bfloat16 *__restrict__ dq)
{
    using C = DqCfg<D>;
    constexpr int TB = C::TB;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sQ = base + C::OFF_Q, sDO = base + C::OFF_DO, sK = base + C::OFF_K,
                   sV = base + C::OFF_V, bar0 = base + C::OFF_BAR;
#define BAR(i) (bar0 + 8u * (uint32_t)(i))
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + C::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Geom g = make_geom(a.S, a.N, a.layout, a.causal);
    const Unit w = decode_unit(g, a.B, a.Hq, 0, a.N, a.upc, T, blockIdx.x);
    const int kvh = w.h / (a.Hq / a.Hkv);
    const int n = KvIter<T>::count(g, w.r, w.qmax);

    if (threadIdx.x == 0) {
        mbar_init(BAR(Q_QFULL), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(BAR(Q_KFULL + i), 1);
            mbar_init(BAR(Q_KEMPTY + i), 2);   // K_j: read by S(j) and by dQ(j)
            mbar_init(BAR(Q_VFULL + i), 1);
            mbar_init(BAR(Q_VEMPTY + i), 1);
        }
        mbar_init(BAR(Q_SDP), 1);
        mbar_init(BAR(Q_DS), 8);
        mbar_init(BAR(Q_FIN), 1);
        mbar_init(BAR(Q_DRAIN), 2);
        mbar_init(BAR(Q_SDPFREE), 8);
        mbar_init(BAR(Q_DSFREE), 1);
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
            // ------------------------------------------------------------ producer
            const uint64_t pol_q = policy_evict_first(), pol_kv = policy_evict_last();
            mbar_arrive_expect_tx(BAR(Q_QFULL), 2 * TB);
            for (int bx = 0; bx < D / 64; ++bx) {
                tma_load4(sQ + bx * 16384, &tmQ, BAR(Q_QFULL), bx * 64, w.h, w.q0, w.b, pol_q);
                tma_load4(sDO + bx * 16384, &tmDO, BAR(Q_QFULL), bx * 64, w.h, w.q0, w.b, pol_q);
            }
            KvIter<T> it;
            it.begin(g, w.r, w.qmax);
            int nk = 0, nv = 0;
            for (int j = 0; j < n; ++j, it.next()) {
                const int st = j & 1, row = it.start();
                if (j >= 2 && !wait1(BAR(Q_KEMPTY + st), ((j >> 1) - 1) & 1, wc)) break;
                mbar_arrive_expect_tx(BAR(Q_KFULL + st), TB);
                for (int bx = 0; bx < D / 64; ++bx)
                    tma_load4(sK + st * TB + bx * 16384, &tmK, BAR(Q_KFULL + st), bx * 64, kvh, row,
                              w.b, pol_kv);
                ++nk;
                if (j >= 2 && !wait1(BAR(Q_VEMPTY + st), ((j >> 1) - 1) & 1, wc)) break;
                mbar_arrive_expect_tx(BAR(Q_VFULL + st), TB);
                for (int bx = 0; bx < D / 64; ++bx)
                    tma_load4(sV + st * TB + bx * 16384, &tmV, BAR(Q_VFULL + st), bx * 64, kvh, row,
                              w.b, pol_kv);
                ++nv;
            }
            if (*abort_flag) {
                volatile int no_abort = 0;
                WaitCtl dc{a.err, &no_abort, a.limit_ns};
                wait1(BAR(Q_QFULL), 0, dc);
                for (int j = nk > 2 ? nk - 2 : 0; j < nk; ++j) wait1(BAR(Q_KFULL + (j & 1)), (j >> 1) & 1, dc);
                for (int j = nv > 2 ? nv - 2 : 0; j < nv; ++j) wait1(BAR(Q_VFULL + (j & 1)), (j >> 1) & 1, dc);
            }
        } else if ((warp == 1 || warp == 2) && lane == 0) {
            // ------------------------------------------------------------ MMA issuers
            // warp 1 issues S = Q K^T and dP = dO V^T as soon as the gradient warps
            // have read the previous ones; warp 2 issues dQ += dS K.  dS has its
            // own tensor-memory columns, so the two streams only meet through
            // the gradient warps' barriers.
            constexpr uint32_t idSP = idesc_bf16(128, T, false);      // S, dP: K-major A and B
            constexpr uint32_t idDQ = idesc_bf16(128, D, true);       // dQ: B = K MN-major
            const uint32_t tS = tmem, tP = tmem + 128u, tQ = tmem + 256u, tDS = tmem + 384u;
            bool ok = true;
            if (warp == 1) {
                const uint64_t dQd = sdesc(sQ, 16, 1024), dDOd = sdesc(sDO, 16, 1024);
                const uint64_t dK0 = sdesc(sK, 16, 1024), dV0 = sdesc(sV, 16, 1024);
                ok = wait1(BAR(Q_QFULL), 0, wc);
                for (int j = 0; ok && j < n; ++j) {
                    const int st = j & 1;
                    if (j > 0 && !wait1(BAR(Q_SDPFREE), (j - 1) & 1, wc)) break;
                    if (!wait1(BAR(Q_KFULL + st), (j >> 1) & 1, wc) ||
                        !wait1(BAR(Q_VFULL + st), (j >> 1) & 1, wc))
                        break;
                    tc_fence_after();
                    const uint64_t so = (uint64_t)(st * (TB >> 4));
                    ss_seq<0, D>(tS, dQd, dK0 + so, idSP);
                    ss_seq<0, D>(tP, dDOd, dV0 + so, idSP);
                    mma_commit(BAR(Q_SDP));
                    mma_commit(BAR(Q_VEMPTY + st));
                    mma_commit(BAR(Q_KEMPTY + st));
                }
            } else {
                const uint64_t dKmn0 = sdesc(sK, 16384, 1024);
                for (int j = 0; ok && j < n; ++j) {
                    const int st = j & 1;
                    if (!wait1(BAR(Q_DS), j & 1, wc) || !wait1(BAR(Q_KFULL + st), (j >> 1) & 1, wc))
                        break;
                    tc_fence_after();
                    // dQ += dS K_j, dS (bf16 pairs) in columns [384, 448)
                    ts_seq<0, true>(tQ, tDS, dKmn0 + (uint64_t)(st * (TB >> 4)), idDQ, j > 0 ? 1u : 0u);
                    mma_commit(BAR(Q_KEMPTY + st));
                    mma_commit(BAR(Q_DSFREE));
                    if (j + 1 == n) mma_commit(BAR(Q_FIN));
                }
            }
            mma_commit(BAR(Q_DRAIN));
            volatile int no_abort = 0;
            WaitCtl dc{a.err, &no_abort, a.limit_ns};
            wait1(BAR(Q_DRAIN), 0, dc);
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
        const uint32_t tS = tmem + lane_off + 64u * half;
        const uint32_t tP = tmem + lane_off + 128u + 64u * half;
        const uint32_t tQ = tmem + lane_off + 256u;
        const uint32_t tDS = tmem + lane_off + 384u + 32u * half;
        const int qpos = w.q0 + row;
        const bool valid = qpos < w.cend;
        const float sl2 = a.scale * LOG2E;
        float lse2 = 0.f, dlt = 0.f;
        if (valid) {
            lse2 = lse[((int64_t)w.b * a.Hq + w.h) * a.S + qpos] * LOG2E;
            dlt = delta[((int64_t)w.b * a.Hq + w.h) * a.S + qpos];
        }
        bool ok = true;
        KvIter<T> it;
        it.begin(g, w.r, w.qmax);
        for (int j = 0; j < n; ++j, it.next()) {
            if (!waitw(BAR(Q_SDP), j & 1, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[64], pr[64];
            tmem_ld_x64(tS, sr);
            tmem_ld_x64(tP, pr);
            // S(j) and dP(j) may now be overwritten by the next tile's MMAs
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(Q_SDPFREE));
            const int ks = it.start(), kl = it.len();
            int lim = kl;                              // visible columns [0, lim) of the tile
            if (a.causal) {
                const int c = qpos - ks + 1;
                lim = c < lim ? c : lim;
            }
            lim -= 64 * half;                          // in this half's local columns
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                float d0 = 0.f, d1 = 0.f;
                const float p0 = ex2(fmaf(__uint_as_float(sr[2 * e]), sl2, -lse2));
                const float p1 = ex2(fmaf(__uint_as_float(sr[2 * e + 1]), sl2, -lse2));
                if (2 * e < lim) d0 = p0 * (__uint_as_float(pr[2 * e]) - dlt);
                if (2 * e + 1 < lim) d1 = p1 * (__uint_as_float(pr[2 * e + 1]) - dlt);
                pk[e] = pack_bf16(d0, d1);
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
            __nv_bfloat16 *orow = dq + (((int64_t)w.b * a.S + qpos) * a.Hq + w.h) * D + HD * half;
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t o[32];
                tmem_ld_x32(tQ + HD * half + 32u * c, o);
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

enum {
    K_KVFULL = 0,
    K_QFULL = 1,    // 2 stages
    K_QEMPTY = 3,   // 2 stages
    K_SDP = 5,
    K_PDS = 6,
    K_FIN = 7,
    K_DRAIN = 8,
    K_NBAR = 9
};

template <int D>
struct DkvCfg {
    static constexpr int TB = Tile<D>::BYTES;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = TB;
    static constexpr int OFF_Q = 2 * TB;      // 2 stages
    static constexpr int OFF_DO = 4 * TB;     // 2 stages
    static constexpr int OFF_STAT = 6 * TB;   // 2 stages x (lse2[128], delta[128]) fp32
    static constexpr int OFF_BAR = OFF_STAT + 2 * 2 * 128 * 4;
    static constexpr int OFF_MISC = OFF_BAR + 8 * K_NBAR;
    static constexpr int NEED = OFF_MISC + 16 + 1024;
    static constexpr int SMEM = NEED > 120 * 1024 ? NEED : 120 * 1024;
};

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const BwdArgs a, const float *__restrict__ lse, const float *__restrict__ delta,
                    __nv_bfloat16 *__restrict__ dk, __nv_bfloat16 *__restrict__ dv)
{
    using C = DkvCfg<D>;
    constexpr int TB = C::TB;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sK = base + C::OFF_K, sV = base + C::OFF_V, sQ = base + C::OFF_Q,
                   sDO = base + C::OFF_DO, bar0 = base + C::OFF_BAR;
    float *stat = reinterpret_cast<float *>(gbase + C::OFF_STAT);   // [stage][lse2 | delta][128]
#define BAR(i) (bar0 + 8u * (uint32_t)(i))
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + C::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Geom g = make_geom(a.S, a.N, a.layout, a.causal);
    const KvUnit w = decode_kv_unit<T>(g, a.B, a.Hkv, a.tpc, blockIdx.x);
    const int grp = a.Hq / a.Hkv;
    const int n = QIter<T>::count(g, w.src, w.ks, grp);

    if (threadIdx.x == 0) {
        mbar_init(BAR(K_KVFULL), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(BAR(K_QFULL + i), 1);
            mbar_init(BAR(K_QEMPTY + i), 1);
        }
        mbar_init(BAR(K_SDP), 1);
        mbar_init(BAR(K_PDS), 8);
        mbar_init(BAR(K_FIN), 1);
        mbar_init(BAR(K_DRAIN), 1);
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
                mbar_arrive_expect_tx(BAR(K_KVFULL), 2 * TB);
                for (int bx = 0; bx < D / 64; ++bx) {
                    tma_load4(sK + bx * 16384, &tmK, BAR(K_KVFULL), bx * 64, w.g, w.ks, w.b, pol_kv);
                    tma_load4(sV + bx * 16384, &tmV, BAR(K_KVFULL), bx * 64, w.g, w.ks, w.b, pol_kv);
                }
            }
            QIter<T> it;
            it.begin(g, w.src, w.ks, w.g * grp, grp);
            int issued = 0;
            for (int i = 0; i < n; ++i, it.next()) {
                const int st = i & 1;
                if (i >= 2 && !waitw(BAR(K_QEMPTY + st), ((i >> 1) - 1) & 1, wc)) break;
                const int qa = it.start(), ql = it.len(), h = it.head();
                // per-row statistics of the query tile: lse (log2 units) and Delta
                float *ls = stat + st * 256, *dl = ls + 128;
                for (int e = lane; e < 128; e += 32) {
                    float l2 = 0.f, dd = 0.f;
                    if (e < ql) {
                        const int64_t off = ((int64_t)w.b * a.Hq + h) * a.S + qa + e;
                        l2 = lse[off] * LOG2E;
                        dd = delta[off];
                    }
                    ls[e] = l2;
                    dl[e] = dd;
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_expect_tx(BAR(K_QFULL + st), 2 * TB);
                    for (int bx = 0; bx < D / 64; ++bx) {
                        tma_load4(sQ + st * TB + bx * 16384, &tmQ, BAR(K_QFULL + st), bx * 64, h, qa,
                                  w.b, pol_q);
                        tma_load4(sDO + st * TB + bx * 16384, &tmDO, BAR(K_QFULL + st), bx * 64, h,
                                  qa, w.b, pol_q);
                    }
                }
                __syncwarp();
                issued = i + 1;
            }
            if (lane == 0 && *abort_flag) {
                volatile int no_abort = 0;
                WaitCtl dc{a.err, &no_abort, a.limit_ns};
                wait1(BAR(K_KVFULL), 0, dc);
                for (int i = issued > 2 ? issued - 2 : 0; i < issued; ++i)
                    wait1(BAR(K_QFULL + (i & 1)), (i >> 1) & 1, dc);
            }
        } else if (warp == 1 && lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            constexpr uint32_t idSP = idesc_bf16(128, T, false);    // S^T, dP^T
            constexpr uint32_t idKV = idesc_bf16(128, D, true);     // dV, dK: B MN-major
            const uint32_t tS = tmem, tP = tmem + 128u, tV = tmem + 256u, tK = tmem + 384u;
            const uint64_t dKd = sdesc(sK, 16, 1024), dVd = sdesc(sV, 16, 1024);
            const uint64_t dQ0 = sdesc(sQ, 16, 1024), dDO0 = sdesc(sDO, 16, 1024);
            const uint64_t dQmn0 = sdesc(sQ, 16384, 1024), dDOmn0 = sdesc(sDO, 16384, 1024);
            bool ok = wait1(BAR(K_KVFULL), 0, wc);
            for (int i = 0; ok && i < n; ++i) {
                const int st = i & 1;
                if (!wait1(BAR(K_QFULL + st), (i >> 1) & 1, wc)) break;
                tc_fence_after();
                const uint64_t so = (uint64_t)(st * (TB >> 4));
                ss_seq<0, D>(tS, dKd, dQ0 + so, idSP);
                ss_seq<0, D>(tP, dVd, dDO0 + so, idSP);
                mma_commit(BAR(K_SDP));
                if (!wait1(BAR(K_PDS), i & 1, wc)) break;
                tc_fence_after();
                ts_seq<0>(tV, tS, dDOmn0 + (uint64_t)(st * (TB >> 4)), idKV, i > 0 ? 1u : 0u);
                ts_seq<0>(tK, tP, dQmn0 + (uint64_t)(st * (TB >> 4)), idKV, i > 0 ? 1u : 0u);
                mma_commit(BAR(K_QEMPTY + st));
            }
            mma_commit(BAR(K_FIN));
            mma_commit(BAR(K_DRAIN));
            volatile int no_abort = 0;
            WaitCtl dc{a.err, &no_abort, a.limit_ns};
            wait1(BAR(K_DRAIN), 0, dc);
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
        const int half = (warp - 4) >> 2;           // query columns [64*half, 64*half+64)
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;        // key row of the tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + 64u * half;
        const uint32_t tP = tmem + lane_off + 128u + 64u * half;
        const int kpos = w.ks + row;
        const float sl2 = a.scale * LOG2E;
        bool ok = true;
        QIter<T> it;
        it.begin(g, w.src, w.ks, w.g * grp, grp);
        for (int i = 0; i < n; ++i, it.next()) {
            const int st = i & 1;
            if (!waitw(BAR(K_SDP), i & 1, wc) || !waitw(BAR(K_QFULL + st), (i >> 1) & 1, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[64], pr[64];
            tmem_ld_x64(tS, sr);
            tmem_ld_x64(tP, pr);
            const int qa = it.start(), ql = it.len();
            // visible query columns c of this tile: c < ql and (not causal or qa + c >= kpos)
            int lo = 0;
            if (a.causal) lo = kpos - qa;
            lo -= 64 * half;
            const int hi = ql - 64 * half;
            const float *ls = stat + st * 256 + 64 * half, *dl = ls + 128;
            uint32_t pp[32], dd[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int c0 = 2 * e, c1 = 2 * e + 1;
                const float p0 = ex2(fmaf(__uint_as_float(sr[c0]), sl2, -ls[c0]));
                const float p1 = ex2(fmaf(__uint_as_float(sr[c1]), sl2, -ls[c1]));
                const bool v0 = c0 >= lo && c0 < hi, v1 = c1 >= lo && c1 < hi;
                const float q0 = v0 ? p0 : 0.f, q1 = v1 ? p1 : 0.f;
                pp[e] = pack_bf16(q0, q1);
                dd[e] = pack_bf16(q0 * (__uint_as_float(pr[c0]) - dl[c0]),
                                  q1 * (__uint_as_float(pr[c1]) - dl[c1]));
            }
            tmem_st_x32(tS, pp);
            tmem_st_x32(tP, dd);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(K_PDS));
        }
        if (ok && waitw(BAR(K_FIN), 0, wc)) {
            tc_fence_after();
            // half 0 writes dV, half 1 writes dK (times scale)
            const bool valid = row < w.kl;
            const float f = half ? a.scale : 1.f;
            const uint32_t tAcc = tmem + lane_off + (half ? 384u : 256u);
            __nv_bfloat16 *orow = (half ? dk : dv) + (((int64_t)w.b * a.S + kpos) * a.Hkv + w.g) * D;
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
    CUtensorMap mq, mk, mv, mdo;
    if (!make_map(&mq, p.q, a.B, a.S, a.Hq, D) || !make_map(&mk, p.k, a.B, a.S, a.Hkv, D) ||
        !make_map(&mv, p.v, a.B, a.S, a.Hkv, D) || !make_map(&mdo, p.dout, a.B, a.S, a.Hq, D))
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
        mq, mk, mv, mdo, a, p.lse, delta, static_cast<__nv_bfloat16 *>(p.dq));
    if (cudaGetLastError() != cudaSuccess) return CP_ECUDA;
    bwd_dkdv_kernel<D><<<(unsigned)kunits, NTHREADS, DkvCfg<D>::SMEM, st>>>(
        mq, mk, mv, mdo, a, p.lse, delta, static_cast<__nv_bfloat16 *>(p.dk),
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
    if (f.D == 64) return launch_bwd_d<64>(p, a, st);
    if (f.D == 128) return launch_bwd_d<128>(p, a, st);
    return CP_EUNSUPPORTED;
}

}  // namespace cp
