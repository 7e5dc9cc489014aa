// fwd_bf16_sm103.cu -- the bf16 flash_block kernel of the ring forward, for
// sm_103a tensor cores (tcgen05 + tensor memory + TMA).
//
// What it computes: for the queries of one virtual rank, the N ring steps of
// "Context Parallelism" (ring sketch: flash_block(q, k, v, out, m, lse,
// source) with source = (rank - step) mod world), each step attending to the
// KV shard of the source rank under the global-position causal mask of
// "Causal Masking and Load Balancing", with the running (O, m, l) folded by
// the online-softmax rescaling of "Sequence Parallelism in LLMs",
// "Algorithmic Mechanics".  The fold runs across steps without leaving the
// SM: O lives in tensor memory from the first KV tile of step 0 to the last
// tile of step N-1.
//
// Work unit: two 128-row query tiles (Q0, Q1) of one chunk and one
// (batch, query head); both share every K/V tile.  Units are launched in
// descending query position, which under a causal mask is descending work.
//
// Roles (384 threads, three warpgroups):
//   warp 0      TMA producer: Q0/Q1 once, then K_j and V_j into 2-deep rings;
//               also allocates / frees the 512 tensor-memory columns.
//   warp 1      MMA issuer (one thread): S_i = Q_i K_j^T (SS, both K-major,
//               128B-swizzled) and O_i += P_i V_j (P from tensor memory, V
//               MN-major), commits to mbarriers.
//   warps 2-3   idle (they only complete warpgroup 0)
//   warps 4-7   softmax of Q0, warps 8-11 softmax of Q1: one thread per query
//               row, reads its S row from tensor memory, masks partial tiles,
//               keeps (m, l), writes P (bf16) back over S, rescales its O row
//               only when the running max grew by more than 2^8, and writes
//               out / lse at the end.
// Issue order of the MMA thread per KV tile j:
//   PV_0(j), S_0(j+1), PV_1(j), S_1(j+1)
// so a completed S_i(j+1) also guarantees PV_i(j) finished: the softmax warps
// may then rescale O_i and overwrite P_i without another barrier.
//
// Tensor memory columns: S0/P0 [0,128), S1/P1 [128,256), O0 [256,256+D),
// O1 [384,384+D).
//
// Every wait is bounded (cp_common.cuh); on time-out the block records
// CP_ETIMEOUT, drains its copies and MMAs, frees tensor memory and exits.
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

constexpr int QT = 128;          // query rows per tile
constexpr int KT = 128;          // keys per KV tile
constexpr int KST = 2;           // K ring depth
constexpr int VST = 2;           // V ring depth
constexpr int NTHREADS = 384;
// Register split (setmaxnreg): the block launches at 168 registers per thread
// (64512 in total); warpgroup 0 (producer, MMA issuer, two idle warps) drops to
// 56 and the two softmax warpgroups rise to 208: 128*56 + 256*208 = 60416.
constexpr int REGS_CTRL = 56;
constexpr int REGS_SOFTMAX = 208;
static_assert(true, "");
constexpr float RESCALE_LOG2 = 8.0f;   // rescale O only when the max grows by > 2^8

enum {
    B_Q = 0,
    B_KFULL = 1,
    B_KEMPTY = B_KFULL + KST,
    B_VFULL = B_KEMPTY + KST,
    B_VEMPTY = B_VFULL + VST,
    B_SFULL = B_VEMPTY + VST,
    B_PFULL = B_SFULL + 2,
    B_OFIN = B_PFULL + 2,
    B_DRAIN = B_OFIN + 2,
    NBAR = B_DRAIN + 1
};

template <int D>
struct Cfg {
    static constexpr int BOXES = D / 64;        // 64-element (128-byte) column boxes per tile
    static constexpr int BOX = 128 * 128;       // bytes of one box: 128 rows x 128 bytes
    static constexpr int TILE = BOXES * BOX;    // bytes of one 128-row bf16 tile
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + 2 * TILE;
    static constexpr int OFF_V = OFF_K + KST * TILE;
    static constexpr int OFF_BAR = OFF_V + VST * TILE;
    static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;
    // + slack to align the base to 1 KB; at least 120 KB so that one block
    // owns the SM and its 512 tensor-memory columns
    static constexpr int SMEM_NEED = OFF_MISC + 16 + 1024;
    static constexpr int SMEM = SMEM_NEED > 120 * 1024 ? SMEM_NEED : 120 * 1024;
};

// --- the kernel ------------------------------------------------------------------

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdArgs a, const float sl2,
                    __nv_bfloat16 *__restrict__ out, float *__restrict__ lse)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t sQ = base + C::OFF_Q, sK = base + C::OFF_K, sV = base + C::OFF_V;
    const uint32_t bar0 = base + C::OFF_BAR;
#define BAR(i) (bar0 + 8u * (uint32_t)(i))
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + C::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Geom g = make_geom(a.S, a.N, a.layout, a.causal);
    const Unit w = decode_unit(g, a.B, a.Hq, a.rank_lo, a.rank_hi, a.upc, 2 * QT, blockIdx.x);
    const int kvh = w.h / (a.Hq / a.Hkv);
    const int n = KvIter<KT>::count(g, w.r, w.qmax);

    if (threadIdx.x == 0) {
        mbar_init(BAR(B_Q), 1);
        for (int i = 0; i < KST; ++i) {
            mbar_init(BAR(B_KFULL + i), 1);
            mbar_init(BAR(B_KEMPTY + i), 1);
        }
        for (int i = 0; i < VST; ++i) {
            mbar_init(BAR(B_VFULL + i), 1);
            mbar_init(BAR(B_VEMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(BAR(B_SFULL + i), 1);
            mbar_init(BAR(B_PFULL + i), 128);
            mbar_init(BAR(B_OFIN + i), 1);
        }
        mbar_init(BAR(B_DRAIN), 1);
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
            // ------------------------------------------------------------ producer
            if (lane == 0) {
                const uint64_t pol_q = policy_evict_first(), pol_kv = policy_evict_last();
                mbar_arrive_expect_tx(BAR(B_Q), 2 * C::TILE);
                for (int qi = 0; qi < 2; ++qi)
                    for (int bx = 0; bx < C::BOXES; ++bx)
                        tma_load4(sQ + qi * C::TILE + bx * C::BOX, &tmQ, BAR(B_Q), bx * 64, w.h,
                                  w.q0 + qi * QT, w.b, pol_q);
                KvIter<KT> it;
                it.begin(g, w.r, w.qmax);
                int issued = 0;
                for (int j = 0; j < n; ++j, it.next()) {
                    const int sk = j % KST, sv = j % VST;
                    const int row = it.start();
                    if (j >= KST && !wait1(BAR(B_KEMPTY + sk), ((j / KST) - 1) & 1, wc)) break;
                    mbar_arrive_expect_tx(BAR(B_KFULL + sk), C::TILE);
                    for (int bx = 0; bx < C::BOXES; ++bx)
                        tma_load4(sK + sk * C::TILE + bx * C::BOX, &tmK, BAR(B_KFULL + sk), bx * 64,
                                  kvh, row, w.b, pol_kv);
                    if (j >= VST && !wait1(BAR(B_VEMPTY + sv), ((j / VST) - 1) & 1, wc)) {
                        issued = -(j + 1);   // K_j issued, V_j not
                        break;
                    }
                    mbar_arrive_expect_tx(BAR(B_VFULL + sv), C::TILE);
                    for (int bx = 0; bx < C::BOXES; ++bx)
                        tma_load4(sV + sv * C::TILE + bx * C::BOX, &tmV, BAR(B_VFULL + sv), bx * 64,
                                  kvh, row, w.b, pol_kv);
                    issued = j + 1;
                }
                // Drain: wait (bounded) for the copies still in flight so none lands
                // after the block exits.  In a normal run these have all completed.
                if (*abort_flag) {
                    const int nk = issued < 0 ? -issued : issued;
                    const int nv = issued < 0 ? -issued - 1 : issued;
                    WaitCtl dc{a.err, abort_flag, a.limit_ns};
                    volatile int no_abort = 0;
                    dc.abort = &no_abort;
                    mbar_try_wait(BAR(B_Q), 0) || wait1(BAR(B_Q), 0, dc);
                    for (int j = (nk > KST ? nk - KST : 0); j < nk; ++j)
                        wait1(BAR(B_KFULL + j % KST), (j / KST) & 1, dc);
                    for (int j = (nv > VST ? nv - VST : 0); j < nv; ++j)
                        wait1(BAR(B_VFULL + j % VST), (j / VST) & 1, dc);
                }
            }
        } else if (warp == 1) {
            // ------------------------------------------------------------ MMA issuer
            if (lane == 0) {
                constexpr uint32_t idS = idesc_bf16(128, KT, false);
                constexpr uint32_t idO = idesc_bf16(128, D, true);
                // S_i / P_i at columns 128*i, O_i at 256 + 128*i
                auto issue_S = [&](int qi, int sk) {
                    const uint32_t tS = tmem + 128u * qi;
    #pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (uint32_t)((kk >> 2) * C::BOX + (kk & 3) * 32);
                        const uint64_t ad = sdesc(sQ + qi * C::TILE + off, 16, 1024);
                        const uint64_t bd = sdesc(sK + sk * C::TILE + off, 16, 1024);
                        mma_ss(tS, ad, bd, idS, kk > 0 ? 1u : 0u);
                    }
                };
                auto issue_PV = [&](int qi, int sv, bool acc) {
                    const uint32_t tS = tmem + 128u * qi, tO = tmem + 256u + 128u * qi;
    #pragma unroll
                    for (int kk = 0; kk < KT / 16; ++kk) {
                        const uint64_t bd = sdesc(sV + sv * C::TILE + kk * 16 * 128, C::BOX, 1024);
                        mma_ts(tO, tS + (uint32_t)(kk * 8), bd, idO, (acc || kk > 0) ? 1u : 0u);
                    }
                };
                bool ok = wait1(BAR(B_Q), 0, wc) && wait1(BAR(B_KFULL + 0), 0, wc);
                if (ok) {
                    tc_fence_after();
                    issue_S(0, 0);
                    mma_commit(BAR(B_SFULL + 0));
                    issue_S(1, 0);
                    mma_commit(BAR(B_SFULL + 1));
                    mma_commit(BAR(B_KEMPTY + 0));
                }
                for (int j = 0; ok && j < n; ++j) {
                    const int sv = j % VST;
                    const bool has_next = (j + 1) < n;
                    const int sk = (j + 1) % KST;
                    if (!wait1(BAR(B_VFULL + sv), (j / VST) & 1, wc)) break;
                    if (has_next && !wait1(BAR(B_KFULL + sk), ((j + 1) / KST) & 1, wc)) break;
                    for (int qi = 0; qi < 2; ++qi) {
                        if (!wait1(BAR(B_PFULL + qi), j & 1, wc)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_PV(qi, sv, j > 0);
                        if (qi == 1) mma_commit(BAR(B_VEMPTY + sv));
                        if (has_next) {
                            issue_S(qi, sk);
                            mma_commit(BAR(B_SFULL + qi));
                            if (qi == 1) mma_commit(BAR(B_KEMPTY + sk));
                        } else {
                            mma_commit(BAR(B_OFIN + qi));
                        }
                    }
                }
                // all MMAs of this block are complete once the drain barrier fires
                mma_commit(BAR(B_DRAIN));
                WaitCtl dc{a.err, abort_flag, a.limit_ns};
                volatile int no_abort = 0;
                dc.abort = &no_abort;
                wait1(BAR(B_DRAIN), 0, dc);
            }
        }
        // end of warpgroup 0: wait for every role, then warp 0 frees tensor memory
        __syncwarp();
        tc_fence_before();
        asm volatile("barrier.sync 1, %0;" ::"n"(NTHREADS) : "memory");
        if (warp == 0) {
            tc_fence_after();
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
        }
        return;
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_SOFTMAX));
        // ------------------------------------------------------------ softmax
        const int qi = (warp - 4) >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + (qi ? 128u : 0u);
        const uint32_t tO = tmem + lane_off + (qi ? 384u : 256u);
        const int qfirst = w.q0 + qi * QT;
        const int qpos = qfirst + row;
        const float NEG_INF = -INFINITY;
        float m_run = NEG_INF, l_run = 0.f;
        bool ok = true;

        KvIter<KT> it;
        it.begin(g, w.r, w.qmax);
        for (int j = 0; j < n; ++j, it.next()) {
            if (!waitw(BAR(B_SFULL + qi), j & 1, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[128];
            tmem_ld_x128(tS, sr);
            float *s = reinterpret_cast<float *>(sr);
            const int ks = it.start();
            const int kl = it.len();
            if (kl < KT || (a.causal && ks + kl - 1 > qfirst)) {
                // partial tile: columns [0, lim) are visible to this row
                int lim = kl;
                if (a.causal) {
                    const int c = qpos - ks + 1;
                    lim = c < lim ? c : lim;
                }
#pragma unroll
                for (int c = 0; c < KT; ++c)
                    if (c >= lim) s[c] = NEG_INF;
            }
            float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
            for (int c = 4; c < KT; c += 4) {
                mx0 = fmaxf(mx0, s[c]);
                mx1 = fmaxf(mx1, s[c + 1]);
                mx2 = fmaxf(mx2, s[c + 2]);
                mx3 = fmaxf(mx3, s[c + 3]);
            }
            const float mt = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
            const float mn = fmaxf(m_run, mt);
            const bool need = mn > m_run + RESCALE_LOG2;
            if (__any_sync(0xffffffffu, need)) {
                const float f = need ? ex2(m_run - mn) : 1.f;
                if (j > 0) {
                    // O_i holds PV_i(0..j-1) (complete: S_i(j) was committed after it)
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld_x32(tO + 32u * c, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                        tmem_st_x32(tO + 32u * c, o);
                    }
                }
                if (need) {
                    l_run *= f;
                    m_run = mn;
                }
            }
            const float mu = (m_run == NEG_INF) ? 0.f : m_run;
            float l0 = 0.f, l1 = 0.f;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float p0 = ex2(fmaf(s[32 * qq + 2 * e], sl2, -mu));
                    const float p1 = ex2(fmaf(s[32 * qq + 2 * e + 1], sl2, -mu));
                    l0 += p0;
                    l1 += p1;
                    pk[e] = pack_bf16(p0, p1);
                }
                tmem_st_x16(tS + 16u * qq, pk);
            }
            tmem_wait_st();
            l_run += l0 + l1;
            tc_fence_before();
            mbar_arrive(BAR(B_PFULL + qi));
        }
        if (ok && waitw(BAR(B_OFIN + qi), 0, wc)) {
            tc_fence_after();
            const bool valid = qpos < w.cend;
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            __nv_bfloat16 *orow = out + (((int64_t)w.b * a.S + qpos) * a.Hq + w.h) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld_x32(tO + 32u * c, o);
                if (valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * c);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        uint4 pkt;
                        pkt.x = pack_bf16(__uint_as_float(o[8 * v4 + 0]) * inv, __uint_as_float(o[8 * v4 + 1]) * inv);
                        pkt.y = pack_bf16(__uint_as_float(o[8 * v4 + 2]) * inv, __uint_as_float(o[8 * v4 + 3]) * inv);
                        pkt.z = pack_bf16(__uint_as_float(o[8 * v4 + 4]) * inv, __uint_as_float(o[8 * v4 + 5]) * inv);
                        pkt.w = pack_bf16(__uint_as_float(o[8 * v4 + 6]) * inv, __uint_as_float(o[8 * v4 + 7]) * inv);
                        dst[v4] = pkt;
                    }
                }
            }
            if (valid)
                lse[((int64_t)w.b * a.Hq + w.h) * a.S + qpos] =
                    l_run > 0.f ? (m_run + lg2(l_run)) * 0.69314718055994531f : NEG_INF;
        }
        __syncwarp();
        tc_fence_before();
        asm volatile("barrier.sync 1, %0;" ::"n"(NTHREADS) : "memory");
        return;
    }
#undef BAR
}

// --- host side -----------------------------------------------------------------

template <int D>
int launch_d(const void *q, const void *k, const void *v, void *out, float *lse, FwdArgs a,
             cudaStream_t st)
{
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, q, a.B, a.S, a.Hq, D) || !make_map(&mk, k, a.B, a.S, a.Hkv, D) ||
        !make_map(&mv, v, a.B, a.S, a.Hkv, D))
        return CP_ECUDA;
    static bool attr_done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CP_ECUDA;
    if (dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(fwd_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg<D>::SMEM) != cudaSuccess)
            return CP_ECUDA;
        attr_done[dev] = true;
    }
    const Geom g = make_geom(a.S, a.N, a.layout, a.causal);
    a.upc = (g.clen + 2 * QT - 1) / (2 * QT);
    const int64_t units = (int64_t)num_selected_chunks(g, a.rank_lo, a.rank_hi) * a.upc * a.B * a.Hq;
    if (units == 0) return CP_OK;
    if (units > 0x7fffffffLL) return CP_EUNSUPPORTED;
    const float sl2 = a.scale * 1.4426950408889634f;
    fwd_bf16_kernel<D><<<(unsigned)units, NTHREADS, Cfg<D>::SMEM, st>>>(
        mq, mk, mv, a, sl2, reinterpret_cast<__nv_bfloat16 *>(out), lse);
    return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ECUDA;
}

}  // namespace

int launch_fwd_bf16(const void *q, const void *k, const void *v, void *out, float *lse,
                    FwdArgs a, cudaStream_t st)
{
    if (a.D == 64) return launch_d<64>(q, k, v, out, lse, a, st);
    if (a.D == 128) return launch_d<128>(q, k, v, out, lse, a, st);
    return CP_EUNSUPPORTED;
}

}  // namespace cp
