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
// Work unit: one 128-row query tile of one chunk and one (batch, query head),
// walking 256-key tiles (S = Q K^T as M=128, N=256 MMAs).  Every tile carries a
// fixed cost beyond its MMAs (about 0.3 us of S read-back, row-max exchange,
// barrier round trips and MMA completion), so the largest tile that fits the
// 512 tensor-memory columns beside P and O amortises it best: 192- and 128-key
// tiles with more buffering of V, S and P measured slower.  Units are numbered
// in descending query position, which under a causal mask is descending work.
//
// Modes (template parameter): the ring over global-order tensors; split-KV
// partials (a unit's walk cut into pieces, each written in fp32 for a merge
// kernel); and one ring step on shard-local buffers (flash_block_step),
// merged into a running (out, lse) state.  A launch either runs one block
// per work item, or (PERSIST, few items per SM) one block per SM taking its
// items in turn, with every barrier phase a running count across items.
//
// Roles (384 threads, three warpgroups):
//   warp 0      TMA producer (one thread): Q once per unit (the next unit's
//               Q before the current unit's last V); K tiles (256 rows) into
//               a 2-deep ring one tile ahead; V tiles as two 128-row halves;
//               warp 0 also allocates and frees the 512 tensor-memory columns.
//   warp 1      issues S = Q K^T, warp 2 issues O += P V: each runs converged
//               (warp-collective waits) and one elected lane issues.
//   warp 3      idle (it completes warpgroup 0 for the register split).
//   warps 4-7   softmax of key columns [0,128), warps 8-11 of [128,256):
//               one thread per query row.  The halves exchange row maxima
//               through shared memory (an mbarrier per tile, bounded wait),
//               so both keep the same running max.
// Tensor memory columns: S [0,256) fp32, P [256,384) bf16 pairs,
// O [384,384+D) fp32.  P has its own columns, so S(j+1) is issued as soon as
// the softmax has read S(j) and PV(j) once P(j) is written, which keeps the
// tensor pipe busy while the softmax computes exponentials.  The
// softmax writes P(j+1) and rescales O only after the commit of PV(j).  O is
// rescaled only when the running max grows by more than 2^8 (exact: the same
// stale max is used for P and l).
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

constexpr int QT = 128;          // query rows per unit
constexpr int KT = 256;          // keys per KV tile
constexpr int NTHREADS = 384;
// Register split (setmaxnreg): the block launches at 168 registers per thread
// (64512 in total); warpgroup 0 drops to 64 and the two softmax warpgroups
// rise to 208: 128*64 + 256*208 = 61440.  (At 56 the persistent control
// warps spilled.)
constexpr int REGS_CTRL = 64;
constexpr int REGS_SOFTMAX = 208;
static_assert(128 * REGS_CTRL + 256 * REGS_SOFTMAX <= NTHREADS * 168, "register split exceeds the launch budget");
constexpr float RESCALE_LOG2 = 8.0f;   // rescale O only when the max grows by > 2^8

enum {
    B_Q = 0,
    B_KFULL = 1,     // 2 K stages
    B_KEMPTY = 3,
    B_VFULL = 5,     // 2 V halves
    B_VEMPTY = 7,
    B_SFULL = 9,
    B_SFREE = 10,    // one arrival per softmax warp (8): S(j) read
    B_PFULL = 11,    // one arrival per softmax warp (8): P(j) written
    B_PFREE = 12,    // PV(j) complete
    B_OFIN = 13,
    B_DRAIN = 14,
    B_MX = 15,       // one arrival per softmax warp (8): row maxima / sums published
    B_QEMPTY = 16,   // a unit's S MMAs complete: the Q buffer may be reloaded
    NBAR = 17
};

template <int D>
struct Cfg {
    static constexpr int QBYTES = QT * D * 2;          // Q tile: D/64 boxes of 128 rows
    static constexpr int KBYTES = KT * D * 2;          // K stage: D/64 boxes of 256 rows
    static constexpr int KBOX = KT * 128;              // bytes of one 256-row box
    static constexpr int VBYTES = 128 * D * 2;         // V half: D/64 boxes of 128 rows
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + QBYTES;
    static constexpr int OFF_V = OFF_K + 2 * KBYTES;
    static constexpr int OFF_PM = OFF_V + 2 * VBYTES;  // row-max exchange: [2][2][128] fp32
    static constexpr int OFF_BAR = OFF_PM + 2 * 2 * 128 * 4;
    static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;
    static constexpr int SMEM_NEED = OFF_MISC + 16;
    // at least 120 KB so that one block owns the SM and its 512 TMEM columns
    static constexpr int SMEM = SMEM_NEED > 120 * 1024 ? SMEM_NEED : 120 * 1024;
    static_assert(SMEM <= 232448, "shared memory budget");
};

// --- unrolled issue sequences -----------------------------------------------------

// S = Q K^T: D/16 MMAs of M=128, N=256, K=16 (both operands K-major, 128B swizzle)
template <int KK, int D>
__device__ __forceinline__ void issue_s_seq(uint32_t tS, uint64_t dQ, uint64_t dK, uint32_t id)
{
    if constexpr (KK < D / 16) {
        constexpr uint32_t oq = (uint32_t)(((KK >> 2) * 16384 + (KK & 3) * 32) >> 4);
        constexpr uint32_t ok = (uint32_t)(((KK >> 2) * Cfg<D>::KBOX + (KK & 3) * 32) >> 4);
        mma_ss_off<oq, ok>(tS, dQ, dK, id, KK > 0 ? 1u : 0u);
        issue_s_seq<KK + 1, D>(tS, dQ, dK, id);
    }
}

// O += P V for one 128-key half: 8 MMAs of M=128, N=D, K=16 (P from tensor
// memory, V MN-major).  acc0 is the accumulate flag of the first one.
template <int K8, int HH>
__device__ __forceinline__ void issue_pv_seq(uint32_t tO, uint32_t tP, uint64_t dV, uint32_t id,
                                             uint32_t acc0)
{
    if constexpr (K8 < 8) {
        constexpr uint32_t ov = (uint32_t)((K8 * 16 * 128) >> 4);
        mma_ts_off<ov>(tO, tP + (uint32_t)((8 * HH + K8) * 8), dV, id, K8 == 0 ? acc0 : 1u);
        issue_pv_seq<K8 + 1, HH>(tO, tP, dV, id, acc0);
    }
}

// --- the kernel ------------------------------------------------------------------

// Modes:
//   MODE_RING   the whole ring over global-order q, k, v; out bf16, lse fp32.
//   MODE_SPLIT  the block runs split `sp` of its unit's walk (tiles [j0, j0 + n)
//               of the n_all tiles, cut into so.n nearly equal pieces) and
//               writes the normalised partial (out, lse) of those keys, in fp32,
//               to so.out / so.lse at the row index of the output row:
//               [sp][B][S][Hq][D] and [sp][B][S][Hq].
//   MODE_STEP   one ring step of one rank on shard-local buffers (the
//               flash_block of the ring sketch): q is the rank's shard, k and v
//               the block of the source rank, each in its local row order; the
//               block's result is merged into the running state (stp.out_acc,
//               stp.lse_acc) with the log-sum-exp form of the online-softmax
//               rescaling, and optionally written rounded to bf16.
enum { MODE_RING = 0, MODE_SPLIT = 1, MODE_STEP = 2 };

// PERSIST: the block runs several work items in turn (fewer blocks than
// items); otherwise it runs item blockIdx.x alone and its item loops run once,
// so every running count below folds to the per-unit index.
template <int D, int MODE, bool PERSIST>
__global__ void __launch_bounds__(NTHREADS, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdArgs a, const float sl2,
                    __nv_bfloat16 *__restrict__ out, float *__restrict__ lse, const SplitOut so,
                    const StepOut stp)
{
    constexpr bool SPLIT = MODE == MODE_SPLIT;
    constexpr bool STEP = MODE == MODE_STEP;
    using C = Cfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_u32(smem_raw);
    if (base & 1023u) {   // the 128B-swizzled tiles need 1 KB alignment
        if (threadIdx.x == 0) atomicCAS(a.err, 0u, ERRW_SMEM_ALIGN);
        return;
    }
    uint8_t *gbase = smem_raw;
    const uint32_t sQ = base + C::OFF_Q, sK = base + C::OFF_K, sV = base + C::OFF_V;
    float *pm = reinterpret_cast<float *>(gbase + C::OFF_PM);
    const uint32_t bar0 = base + C::OFF_BAR;
#define BAR(i) (bar0 + 8u * (uint32_t)(i))
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + C::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Geom g = make_geom(a.S, a.N, a.layout, a.causal);
    const int C_loc = g.clen * g.cpr;   // rows of one shard (MODE_STEP buffers)
    // extents of the tensor maps' (rank, row) dimensions, for the debug-bounds build
    const int map_r = (!STEP && striped(g)) ? g.N : 1;
    const int map_rows = STEP ? C_loc : a.S / map_r;
    // Work items: the launch's units (times the splits).  Split index slowest:
    // the blocks in flight run the same split of consecutive units, which walk
    // the same key tiles (as in an unsplit launch) and share them in L2;
    // adjacent splits of one unit would walk disjoint key ranges and stream
    // them from DRAM.
    const int nunits = a.n_units;
    const int n_items = nunits * (SPLIT ? so.n : 1);

    // The block runs items item_of(0), item_of(1), ...: rounds of gridDim.x
    // items, alternately forwards and backwards over the longest-first
    // numbering, so the blocks' totals stay close.  With one block per item
    // (gridDim.x == n_items) the block runs item blockIdx.x alone.
    auto item_of = [&](int it) -> int {
        if (!PERSIST) return it == 0 ? (int)blockIdx.x : n_items;
        const int64_t G = gridDim.x, c = blockIdx.x;
        const int64_t item = it * G + ((it & 1) ? G - 1 - c : c);
        return item < n_items ? (int)item : n_items;
    };
    struct Item {
        Unit w;
        int sp, j0, n, kvh;
    };
    auto decode = [&](int item) -> Item {
        Item x;
        x.sp = SPLIT ? item / nunits : 0;
        const int ublk = SPLIT ? item - x.sp * nunits : item;
        x.w = a.head_grouped ? decode_unit_grouped(g, a.B, a.Hq, a.upc, QT, ublk)
                             : decode_unit(g, a.B, a.Hq, a.rank_lo, a.rank_hi, a.upc, QT, ublk);
        x.kvh = x.w.h / (a.Hq / a.Hkv);
        const int n_all = STEP ? KvIter<KT>::count(g, x.w.r, x.w.qmax, stp.step_k, stp.step_k + 1)
                               : KvIter<KT>::count(g, x.w.r, x.w.qmax);
        x.j0 = SPLIT ? (int)((int64_t)n_all * x.sp / so.n) : 0;
        x.n = SPLIT ? (int)((int64_t)n_all * (x.sp + 1) / so.n) - x.j0 : n_all;
        return x;
    };
    // The block's next item with at least one key tile, from item_of(it) on:
    // advances it and returns false once the block's items are used up.
    auto next_busy = [&](int &it, Item &x) -> bool {
        for (;; ++it) {
            if (!PERSIST && it > 0) return false;
            const int item = item_of(it);
            if (item >= n_items) return false;
            x = decode(item);
            if (x.n > 0) return true;
        }
    };

    if (threadIdx.x == 0) {
        mbar_init(BAR(B_Q), 1);
        mbar_init(BAR(B_QEMPTY), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(BAR(B_KFULL + i), 1);
            mbar_init(BAR(B_KEMPTY + i), 1);
            mbar_init(BAR(B_VFULL + i), 1);
            mbar_init(BAR(B_VEMPTY + i), 1);
        }
        mbar_init(BAR(B_SFULL), 1);
        mbar_init(BAR(B_SFREE), 8);
        mbar_init(BAR(B_PFULL), 8);
        mbar_init(BAR(B_PFREE), 1);
        mbar_init(BAR(B_OFIN), 1);
        mbar_init(BAR(B_DRAIN), 2);
        mbar_init(BAR(B_MX), 8);
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

    // Phases run on across the block's items: every barrier's phase index is a
    // running count (Q loads, K/V tiles, S and PV tiles, units, exchanges).
    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_CTRL));
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------------------ producer
            const uint64_t pol_q = policy_evict_first(), pol_kv = policy_evict_last();
            int nq = 0, nk = 0, nv = 0;   // Q loads, K tiles, V halves issued so far
            // Q of item y into the single Q buffer, once the previous unit's S
            // MMAs are done with it
            auto load_q = [&](const Item &y) -> bool {
                if (nq > 0 && !wait1(BAR(B_QEMPTY), (nq - 1) & 1, wc)) return false;
                mbar_arrive_expect_tx(BAR(B_Q), C::QBYTES);
                // map coordinates (rank, row) of the unit's first query
                const int qmr = dbg_coord(a.err, STEP ? 0 : slot_mrank(g, y.w.q0), map_r);
                const int qmw = dbg_coord(a.err, STEP ? slot_lrow(g, y.w.r, y.w.q0) : slot_mrow(g, y.w.q0), map_rows);
                const int qh = dbg_coord(a.err, y.w.h, a.Hq), qb = dbg_coord(a.err, y.w.b, a.B);
                for (int bx = 0; bx < D / 64; ++bx)
                    tma_load5(sQ + bx * 16384, &tmQ, BAR(B_Q), bx * 64, qh, qmr, qmw, qb, pol_q);
                ++nq;
                return true;
            };
            // Items with keys only, decoded one ahead while the current one loads;
            // the next unit's Q goes out between the current unit's last K and
            // last V (its S MMAs are done by then), so that the next unit's first
            // S can run while the softmax warps finish this unit's epilogue.
            int it = 0;
            Item x;
            bool have = next_busy(it, x);
            bool ok = !have || load_q(x);
            while (ok && have) {
                int it2 = it + 1;
                Item y = x;
                // K runs one tile ahead of V; the V loads reuse the K tile starts
                KvIter<KT> itk;
                if (STEP)
                    itk.begin_steps(g, x.w.r, x.w.qmax, stp.step_k, stp.step_k + 1);
                else
                    itk.begin(g, x.w.r, x.w.qmax);
                if (SPLIT) itk.skip(x.j0);
                int kr_cur = 0, kw_cur = 0, kr_next = 0, kw_next = 0;   // map coordinates (rank, row)
                const int kvh = dbg_coord(a.err, x.kvh, a.Hkv), qb = dbg_coord(a.err, x.w.b, a.B);
                auto load_k = [&]() -> bool {   // the next K tile, global index nk
                    const int st = nk & 1;
                    if (nk >= 2 && !wait1(BAR(B_KEMPTY + st), ((nk >> 1) - 1) & 1, wc)) return false;
                    mbar_arrive_expect_tx(BAR(B_KFULL + st), C::KBYTES);
                    kr_next = dbg_coord(a.err, STEP ? 0 : itk.mrank(), map_r);
                    kw_next = dbg_coord(a.err, STEP ? itk.lrow() : itk.mrow(), map_rows);
                    for (int bx = 0; bx < D / 64; ++bx)
                        tma_load5(sK + st * C::KBYTES + bx * C::KBOX, &tmK, BAR(B_KFULL + st), bx * 64,
                                  kvh, kr_next, kw_next, qb, pol_kv);
                    itk.next();
                    ++nk;
                    return true;
                };
                ok = load_k();
                const bool have2 = PERSIST && next_busy(it2, y);
                for (int j = 0; ok && j < x.n; ++j) {
                    kr_cur = kr_next;
                    kw_cur = kw_next;
                    // global index of tile j: nv / 2 (V halves are issued tile by tile)
                    const int t = nv >> 1;
                    if ((j + 1 < x.n && !load_k()) || (j + 1 == x.n && have2 && !load_q(y))) {
                        ok = false;
                        break;
                    }
                    for (int hh = 0; hh < 2; ++hh) {
                        if (t >= 1 && !wait1(BAR(B_VEMPTY + hh), (t - 1) & 1, wc)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(BAR(B_VFULL + hh), C::VBYTES);
                        for (int bx = 0; bx < D / 64; ++bx)
                            tma_load5(sV + hh * C::VBYTES + bx * 16384, &tmV, BAR(B_VFULL + hh), bx * 64,
                                      kvh, kr_cur, kw_cur + 128 * hh, qb, pol_kv);
                        ++nv;
                    }
                }
                x = y;
                it = it2;
                have = have2;
            }
            {
                // Drain: wait (bounded) for the copies still in flight -- always,
                // since a consumer may give up after this thread has issued its last
                // copy.  Each wait is on the last phase its barrier was armed for, so
                // after a normal run every one of them is already complete.
                volatile int no_abort = 0;
                WaitCtl dc{a.err, &no_abort, a.drain_ns};
                if (nq > 0) wait1(BAR(B_Q), (nq - 1) & 1, dc);
                for (int j = nk > 2 ? nk - 2 : 0; j < nk; ++j) wait1(BAR(B_KFULL + (j & 1)), (j >> 1) & 1, dc);
                for (int h = nv > 2 ? nv - 2 : 0; h < nv; ++h) wait1(BAR(B_VFULL + (h & 1)), (h >> 1) & 1, dc);
            }
        } else if (warp == 1 || warp == 2) {
            // ------------------------------------------------------------ MMA issuers
            // Two issuing warps on different SM sub-partitions: warp 1 issues
            // S = Q K^T, warp 2 issues O += P V.  They touch disjoint tensor-memory
            // columns (S vs P and O); every dependency between them goes through
            // the softmax barriers (S_FREE, P_FULL, P_FREE).  Splitting halves the
            // issue work each one competes for against two busy softmax warps, and
            // a wait of one issuer never holds back the other.  Each warp runs
            // converged (warp-collective waits), so its operands stay warp-uniform,
            // and one elected lane issues the MMAs and their commits.
            constexpr uint32_t idS = idesc_bf16(128, KT, false);
            constexpr uint32_t idO = idesc_bf16(128, D, true);
            const uint32_t tS = tmem, tP = tmem + 256u, tO = tmem + 384u;
            const bool leader = elect_one();
            bool ok = true;
            int nq = 0, nt = 0;   // units started, tiles issued so far
            if (warp == 1) {
                const uint64_t dQ = sdesc(sQ, 16, 1024);
                const uint64_t dK0 = sdesc(sK, 16, 1024);
                for (int it = 0; ok && (PERSIST || it == 0); ++it) {
                    const int item = item_of(it);
                    if (item >= n_items) break;
                    const int n = decode(item).n;
                    if (n == 0) continue;
                    if (!waitw(BAR(B_Q), nq & 1, wc)) break;
                    for (int j = 0; j < n; ++j, ++nt) {
                        const int st = nt & 1;
                        if ((nt > 0 && !waitw(BAR(B_SFREE), (nt - 1) & 1, wc)) ||
                            !waitw(BAR(B_KFULL + st), (nt >> 1) & 1, wc)) {
                            ok = false;
                            break;
                        }
                        const uint64_t dK = dK0 + (uint64_t)(st * (C::KBYTES >> 4));
                        if (leader) {
                            tc_fence_after();
                            issue_s_seq<0, D>(tS, dQ, dK, idS);
                            mma_commit(BAR(B_SFULL));
                            mma_commit(BAR(B_KEMPTY + st));
                        }
                        __syncwarp();
                    }
                    if (!ok) break;
                    // Q may be reloaded once the unit's S MMAs have completed
                    if (leader) mma_commit(BAR(B_QEMPTY));
                    __syncwarp();
                    ++nq;
                }
            } else {
                const uint64_t dV0 = sdesc(sV, 16384, 1024);
                const uint64_t dV1 = dV0 + (uint64_t)(C::VBYTES >> 4);
                for (int it = 0; ok && (PERSIST || it == 0); ++it) {
                    const int item = item_of(it);
                    if (item >= n_items) break;
                    const int n = decode(item).n;
                    for (int j = 0; j < n; ++j, ++nt) {
                        // P(nt) written: every softmax warp has also finished reading
                        // the previous unit's O, which the first PV of this unit
                        // (accumulate 0) overwrites
                        if (!waitw(BAR(B_PFULL), nt & 1, wc) || !waitw(BAR(B_VFULL + 0), nt & 1, wc)) {
                            ok = false;
                            break;
                        }
                        const uint32_t acc0 = j > 0 ? 1u : 0u;
                        if (leader) {
                            tc_fence_after();
                            issue_pv_seq<0, 0>(tO, tP, dV0, idO, acc0);
                            mma_commit(BAR(B_VEMPTY + 0));
                        }
                        __syncwarp();
                        if (!waitw(BAR(B_VFULL + 1), nt & 1, wc)) {
                            ok = false;
                            break;
                        }
                        if (leader) {
                            tc_fence_after();
                            issue_pv_seq<0, 1>(tO, tP, dV1, idO, 1u);
                            mma_commit(BAR(B_VEMPTY + 1));
                            mma_commit(BAR(B_PFREE));
                            if (j + 1 == n) mma_commit(BAR(B_OFIN));
                        }
                        __syncwarp();
                    }
                }
            }
            // all MMAs of this warp are complete once the drain barrier (two
            // arrivals: one commit per issuer) fires
            if (leader) mma_commit(BAR(B_DRAIN));
            __syncwarp();
            volatile int no_abort = 0;
            WaitCtl dc{a.err, &no_abort, a.drain_ns};
            waitw(BAR(B_DRAIN), 0, dc);
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
        const int half = (warp - 4) >> 2;            // key columns [128*half, 128*half+128)
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + 128u * half;
        const uint32_t tP = tmem + lane_off + 256u + 64u * half;
        const uint32_t tO = tmem + lane_off + 384u + (uint32_t)(D / 2) * half;
        const float NEG_INF = -INFINITY;
        bool ok = true;
        int nu = 0, nt = 0, nx = 0;   // units finished, tiles done, row-max exchanges so far

        // Every item, empty ones included, decoded one ahead: the next one is
        // decoded while this unit's last PV completes.
        Item xn;
        bool have = item_of(0) < n_items;
        if (have) xn = decode(item_of(0));
        auto advance = [&](int it) {
            const int nxt = item_of(it + 1);
            have = PERSIST && nxt < n_items;
            if (have) xn = decode(nxt);
        };
        for (int it = 0; ok && have; ++it) {
            const Item x = xn;
            const Unit &w = x.w;
            const int n = x.n;
            const int qpos = w.q0 + row;
            const bool valid = qpos < w.cend;
            if (n == 0) {
                // A split or step with no key for the unit: this thread writes its
                // row's half.  Split: the merge identity (out 0, lse -inf).  Step:
                // merging changes nothing (out_final, if asked for, is the state
                // rounded); a first step writes the empty state (out 0, lse -inf).
                if constexpr (SPLIT) {
                    if (valid) {
                        const int64_t prow = (((int64_t)x.sp * a.B + w.b) * a.S + slot_pos(g, qpos)) * a.Hq + w.h;
                        float4 *dst = reinterpret_cast<float4 *>(so.out + prow * D + (D / 2) * half);
#pragma unroll
                        for (int c4 = 0; c4 < D / 8; ++c4) dst[c4] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (half == 0) so.lse[prow] = NEG_INF;
                    }
                } else if constexpr (STEP) {
                    if (valid) {
                        const int lr = dbg_coord(a.err, slot_lrow(g, w.r, qpos), C_loc);
                        const int64_t srow = ((int64_t)w.b * C_loc + lr) * a.Hq + w.h;
                        float4 *acc = reinterpret_cast<float4 *>(stp.out_acc + srow * D + (D / 2) * half);
                        uint4 *fin = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(stp.out_final) +
                                                               srow * D + (D / 2) * half);
#pragma unroll
                        for (int c8 = 0; c8 < D / 16; ++c8) {
                            float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
                            if (stp.accumulate) {
                                x0 = acc[2 * c8];
                                x1 = acc[2 * c8 + 1];
                            } else {
                                acc[2 * c8] = x0;
                                acc[2 * c8 + 1] = x1;
                            }
                            if (stp.out_final)
                                fin[c8] = make_uint4(pack_bf16(x0.x, x0.y), pack_bf16(x0.z, x0.w),
                                                     pack_bf16(x1.x, x1.y), pack_bf16(x1.z, x1.w));
                        }
                        if (!stp.accumulate && half == 0)
                            stp.lse_acc[((int64_t)w.b * a.Hq + w.h) * C_loc + lr] = NEG_INF;
                    }
                }
                advance(it);
                continue;
            }
            float m_run = NEG_INF, l_run = 0.f;      // l_run: this half's share of the row sum

            KvIter<KT> kit;
            if (STEP)
                kit.begin_steps(g, w.r, w.qmax, stp.step_k, stp.step_k + 1);
            else
                kit.begin(g, w.r, w.qmax);
            if (SPLIT) kit.skip(x.j0);
            for (int j = 0; j < n; ++j, ++nt, ++nx, kit.next()) {
                if (!waitw(BAR(B_SFULL), nt & 1, wc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sr[128];
                tmem_ld_x128(tS, sr);
                // S may now be overwritten: one arrival per warp (per-thread
                // arrivals would serialise 256 atomics on one shared-memory word)
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(B_SFREE));
                float *s = reinterpret_cast<float *>(sr);
                const int ks = kit.start();
                const int kl = kit.len();
                if (kl < KT || (a.causal && ks + kl - 1 > w.q0 + kit.shift)) {
                    // partial tile: key columns [0, lim) of the 256 are visible to this row
                    int lim = kl;
                    if (a.causal) {
                        const int c = qpos - ks + 1 + kit.shift;
                        lim = c < lim ? c : lim;
                    }
                    lim -= 128 * half;
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c >= lim) s[c] = NEG_INF;
                }
                // row max over this half: four independent 3-input max chains
                float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
                for (int c = 4; c < 124; c += 8) {
                    mx0 = fmax3(mx0, s[c], s[c + 1]);
                    mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
                    mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
                    mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
                }
                mx0 = fmax3(mx0, s[124], s[125]);
                mx1 = fmax3(mx1, s[126], s[127]);
                mx0 = fmax3(mx0, mx2, mx3);
                // Publish this half's row maximum (double-buffered by exchange
                // parity; the barrier's phase completes once all 256 threads
                // published theirs).
                float *pmj = pm + (nx & 1) * 256;
                const float mloc = fmaxf(mx0, mx1) * sl2;
                pmj[half * 128 + row] = fmaxf(mx0, mx1);
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(B_MX));
                // The exponentials use the running max m_run as long as this half's own
                // maximum stays within 2^8 of it (P <= 2^8, no overflow), so the exchange
                // is off the critical path; the combined max is checked afterwards and,
                // in the rare case it grew by more than 2^8, P is scaled down to the new
                // max.  The first visible tile (m_run = -inf) and a half whose own max
                // jumped take the exchanged max first.
                const bool early = __any_sync(0xffffffffu, mloc > m_run + RESCALE_LOG2);
                float mt = NEG_INF;
                if (early) {
                    if (!waitw(BAR(B_MX), nx & 1, wc)) {
                        ok = false;
                        break;
                    }
                    mt = fmaxf(pmj[0 * 128 + row], pmj[1 * 128 + row]) * sl2;
                }
                float mn = fmaxf(m_run, mt);
                bool need = mn > m_run + RESCALE_LOG2;
                float f = need ? ex2(m_run - mn) : 1.f;    // ex2(-inf) = 0 on the first tile
                if (need) m_run = mn;
                const float mu = (m_run == NEG_INF) ? 0.f : m_run;
                // P = exp2(s*sl2 - mu), packed to bf16 as it is produced
                float l0 = 0.f, l1 = 0.f;
                uint32_t pk0[32], pk1[32];
#pragma unroll
                for (int c = 0; c < 128; c += 2) {
                    float x0, x1;
                    ffma2(x0, x1, s[c], s[c + 1], sl2, -mu);
                    const float p0 = ex2(x0), p1 = ex2(x1);
                    const uint32_t pk = pack_bf16(p0, p1);
                    fadd2(l0, l1, p0, p1);
                    if (c < 64) pk0[c / 2] = pk;
                    else pk1[(c - 64) / 2] = pk;
                }
                if (!early) {
                    if (!waitw(BAR(B_MX), nx & 1, wc)) {
                        ok = false;
                        break;
                    }
                    mt = fmaxf(pmj[0 * 128 + row], pmj[1 * 128 + row]) * sl2;
                    mn = fmaxf(m_run, mt);
                    need = mn > m_run + RESCALE_LOG2;
                    if (__any_sync(0xffffffffu, need)) {
                        // the other half raised the max (rare): rescale this tile's P and sum
                        f = need ? ex2(m_run - mn) : 1.f;
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            pk0[e] = pack_bf16(__uint_as_float(pk0[e] << 16) * f, __uint_as_float(pk0[e] & 0xffff0000u) * f);
                            pk1[e] = pack_bf16(__uint_as_float(pk1[e] << 16) * f, __uint_as_float(pk1[e] & 0xffff0000u) * f);
                        }
                        l0 *= f;
                        l1 *= f;
                        if (need) m_run = mn;
                    }
                }
                // P may be written, and O rescaled, once the previous PV has
                // completed (the previous unit's last one for j = 0)
                if (nt > 0 && !waitw(BAR(B_PFREE), (nt - 1) & 1, wc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) {
                        uint32_t o[32];
                        tmem_ld_x32(tO + 32u * c, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                        tmem_st_x32(tO + 32u * c, o);
                    }
                }
                l_run = l_run * f + (l0 + l1);
                tmem_st_x32(tP, pk0);
                tmem_st_x32(tP + 32u, pk1);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(B_PFULL));
            }
            advance(it);
            if (!ok || !waitw(BAR(B_OFIN), nu & 1, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // MODE_STEP: the running lse of the row, read by both halves before
            // the exchange below (half 0 overwrites it only after the exchange)
            float prev2 = NEG_INF;
            int64_t srow = 0;
            if constexpr (STEP) {
                srow = ((int64_t)w.b * C_loc + dbg_coord(a.err, slot_lrow(g, w.r, valid ? qpos : w.q0), C_loc)) *
                           a.Hq + w.h;
                if (valid && stp.accumulate)
                    prev2 = stp.lse_acc[((int64_t)w.b * a.Hq + w.h) * C_loc + slot_lrow(g, w.r, qpos)] *
                            1.4426950408889634f;
            }
            // total row sum: this half's share plus the other's (exchange nx;
            // buffer nx&1 was last read before the arrivals of exchange nx-1)
            float *pmn = pm + (nx & 1) * 256;
            pmn[half * 128 + row] = l_run;
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_MX));
            if (!waitw(BAR(B_MX), nx & 1, wc)) {
                ok = false;
                break;
            }
            ++nx;
            const float l_tot = pmn[row] + pmn[128 + row];
            const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
            const int qp = slot_pos(g, qpos);   // global position of the row
            if constexpr (STEP) {
                // merge the block (O / l, lse_blk) into the state (out_acc, lse):
                // lse_new = ln(e^lse + e^lse_blk), out_new = e^(lse - lse_new) out_acc
                // + e^(lse_blk - lse_new) O / l, in base 2; an empty side has
                // weight 0, both empty leave (0, -inf)
                const float blk2 = l_tot > 0.f ? m_run + lg2(l_tot) : NEG_INF;
                const float mx = fmaxf(prev2, blk2);
                float wa = 0.f, wb = 0.f, new2 = NEG_INF;
                if (mx != NEG_INF) {
                    const float ea = ex2(prev2 - mx), eb = ex2(blk2 - mx);   // ex2(-inf) = 0
                    const float rs = 1.f / (ea + eb);
                    new2 = mx + lg2(ea + eb);
                    wa = ea * rs;
                    wb = eb * rs * inv;
                }
                // a row that sees no key of this block keeps its state untouched
                // (weights 1 and 0 give back its out exactly; its lse is not rewritten)
                const bool keep = stp.accumulate && blk2 == NEG_INF;
                if (keep) {
                    wa = 1.f;
                    wb = 0.f;
                }
                float *orow = stp.out_acc + srow * D + (D / 2) * half;
                __nv_bfloat16 *frow = static_cast<__nv_bfloat16 *>(stp.out_final) + srow * D + (D / 2) * half;
                // this half of the row: one tensor-memory load
                uint32_t o[D / 2];
                if constexpr (D == 128)
                    tmem_ld_x64(tO, o);
                else
                    tmem_ld_x32(tO, o);
                const bool a32 = ((reinterpret_cast<uintptr_t>(stp.out_acc) |
                                   reinterpret_cast<uintptr_t>(stp.out_final)) & 31) == 0;
                if (a32) {
                    // The state in pieces of 32 columns (128 bytes of fp32), read and
                    // written regrouped so that every load and store instruction of
                    // the warp covers whole pieces (rows lie Hq*D elements apart);
                    // out_final's half-row is written the same way.
                    uint32_t fk[D / 4];
#pragma unroll
                    for (int pc = 0; pc < D / 64; ++pc) {
                        uint32_t pv[32], r[32];
                        if (stp.accumulate) {
                            load_warp_rows<32>(orow + 32 * pc, valid, pv, lane);
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e) pv[e] = 0u;
                        }
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            r[e] = __float_as_uint(wa * __uint_as_float(pv[e]) + wb * __uint_as_float(o[32 * pc + e]));
                        store_warp_rows<32>(orow + 32 * pc, valid, r, lane);
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            fk[16 * pc + e] = pack_bf16(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
                    }
                    if (stp.out_final) store_warp_rows<D / 4>(frow, valid, fk, lane);
                } else if (valid) {
                    // every lane reads and writes its own row, 16 bytes at a time
#pragma unroll
                    for (int c16 = 0; c16 < D / 32; ++c16) {   // D/2 columns
                        float pv[16], r[16];
                        float *src = orow + 16 * c16;
                        if (stp.accumulate) {
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                const float4 t = reinterpret_cast<const float4 *>(src)[q4];
                                pv[4 * q4] = t.x;
                                pv[4 * q4 + 1] = t.y;
                                pv[4 * q4 + 2] = t.z;
                                pv[4 * q4 + 3] = t.w;
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; ++e) pv[e] = 0.f;
                        }
#pragma unroll
                        for (int e = 0; e < 16; ++e) r[e] = wa * pv[e] + wb * __uint_as_float(o[16 * c16 + e]);
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
                            reinterpret_cast<float4 *>(src)[q4] =
                                make_float4(r[4 * q4], r[4 * q4 + 1], r[4 * q4 + 2], r[4 * q4 + 3]);
                        if (stp.out_final) {
                            uint32_t pk[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) pk[e] = pack_bf16(r[2 * e], r[2 * e + 1]);
                            uint4 *fdst = reinterpret_cast<uint4 *>(frow + 16 * c16);
                            fdst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                            fdst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                        }
                    }
                }
                if (valid && !keep && half == 0)
                    stp.lse_acc[((int64_t)w.b * a.Hq + w.h) * C_loc + slot_lrow(g, w.r, qpos)] =
                        new2 == NEG_INF ? NEG_INF : new2 * 0.69314718055994531f;
            } else if constexpr (SPLIT) {
                const int64_t prow =
                    (((int64_t)x.sp * a.B + w.b) * a.S + dbg_coord(a.err, valid ? qp : 0, a.S)) * a.Hq + w.h;
                float *orow = so.out + prow * D + (D / 2) * half;
                // this half of the row: one tensor-memory load; with 32-byte aligned
                // partials written in pieces of 32 columns (128 bytes), regrouped so
                // that every store instruction of the warp covers whole pieces,
                // else every lane writes its own row in 16-byte pieces
                uint32_t o[D / 2];
                if constexpr (D == 128)
                    tmem_ld_x64(tO, o);
                else
                    tmem_ld_x32(tO, o);
#pragma unroll
                for (int e = 0; e < D / 2; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * inv);
                if ((reinterpret_cast<uintptr_t>(so.out) & 31) == 0) {
#pragma unroll
                    for (int pc = 0; pc < D / 64; ++pc)
                        store_warp_rows<32>(orow + 32 * pc, valid, *reinterpret_cast<const uint32_t(*)[32]>(o + 32 * pc),
                                            lane);
                } else if (valid) {
#pragma unroll
                    for (int v4 = 0; v4 < D / 8; ++v4)   // D/2 columns, 4 per store
                        reinterpret_cast<float4 *>(orow)[v4] =
                            make_float4(__uint_as_float(o[4 * v4]), __uint_as_float(o[4 * v4 + 1]),
                                        __uint_as_float(o[4 * v4 + 2]), __uint_as_float(o[4 * v4 + 3]));
                }
                if (valid && half == 0)
                    so.lse[prow] = l_tot > 0.f ? (m_run + lg2(l_tot)) * 0.69314718055994531f : NEG_INF;
            } else {
                __nv_bfloat16 *orow =
                    out + (((int64_t)w.b * a.S + dbg_coord(a.err, valid ? qp : 0, a.S)) * a.Hq + w.h) * D + (D / 2) * half;
                // this half of the row: one tensor-memory load, rounded to bf16
                uint32_t o[D / 2];
                if constexpr (D == 128)
                    tmem_ld_x64(tO, o);
                else
                    tmem_ld_x32(tO, o);
                uint32_t pk[D / 4];
#pragma unroll
                for (int e = 0; e < D / 4; ++e)
                    pk[e] = pack_bf16(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
                // Rows lie Hq*D elements apart.  With a 32-byte aligned output the
                // warp regroups its half-rows so that each store instruction writes
                // whole ones (store_warp_rows); otherwise every lane writes its own
                // row in 16-byte pieces.
                if ((reinterpret_cast<uintptr_t>(out) & 31) == 0) {
                    store_warp_rows<D / 4>(orow, valid, pk, lane);
                } else if (valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow);
#pragma unroll
                    for (int v4 = 0; v4 < D / 16; ++v4)   // D/2 columns, 8 per store
                        dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                }
                if (valid && half == 0)
                    lse[((int64_t)w.b * a.Hq + w.h) * a.S + qp] =
                        l_tot > 0.f ? (m_run + lg2(l_tot)) * 0.69314718055994531f : NEG_INF;
            }
            ++nu;
        }
        __syncwarp();
        tc_fence_before();
        asm volatile("barrier.sync 1, %0;" ::"n"(NTHREADS) : "memory");
        return;
    }
#undef BAR
}

// --- host side -----------------------------------------------------------------

template <int D, int MODE>
int launch_d(const void *q, const void *k, const void *v, void *out, float *lse, FwdArgs a,
             const SplitOut &so, const StepOut &stp, cudaStream_t st)
{
    CUtensorMap mq, mk, mv;
    const Geom g = make_geom(a.S, a.N, a.layout, a.causal);
    if (MODE == MODE_STEP) {
        // shard-local buffers: [B][S/N][H][D] in the shards' local row order
        const int64_t C = (int64_t)g.clen * g.cpr;
        if (!make_map(&mq, q, a.B, C, a.Hq, D, 128, 1) || !make_map(&mk, k, a.B, C, a.Hkv, D, KT, 1) ||
            !make_map(&mv, v, a.B, C, a.Hkv, D, 128, 1))
            return CP_ECUDA;
    } else {
        const int R = a.layout == CP_LAYOUT_STRIPED ? a.N : 1;
        if (!make_map(&mq, q, a.B, a.S, a.Hq, D, 128, R) || !make_map(&mk, k, a.B, a.S, a.Hkv, D, KT, R) ||
            !make_map(&mv, v, a.B, a.S, a.Hkv, D, 128, R))
            return CP_ECUDA;
    }
    static bool attr_done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CP_ECUDA;
    if (dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(fwd_bf16_kernel<D, MODE, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg<D>::SMEM) != cudaSuccess ||
            cudaFuncSetAttribute(fwd_bf16_kernel<D, MODE, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg<D>::SMEM) != cudaSuccess)
            return CP_ECUDA;
        attr_done[dev] = true;
    }
    a.upc = (g.clen + QT - 1) / QT;
    // Unit order.  Blocks start in launch order on the SM that frees first, so
    // numbering units longest first (heads fastest, descending position) is a
    // longest-processing-time schedule.  But then the blocks in flight touch
    // every head's K/V at once; when those exceed what L2 can keep
    // (S = 131072: 512 MB), every query tile re-reads its K/V from DRAM, so a
    // launch over all ranks numbers each (batch, head) contiguously instead
    // (blocks in flight share one or two heads' K/V).  Up to 96 MB of K/V
    // (of the 129 MB L2) the longest-first order was measured to cost no DRAM
    // time and shortens the tail (S = 16384 and 20480, 67 and 84 MB of K/V:
    // 16-19 % faster than the grouped order).
    const int64_t kv_bytes = 2ll * a.B * a.S * a.Hkv * D * 2;
    a.head_grouped = (MODE != MODE_STEP && a.rank_lo == 0 && a.rank_hi == a.N &&
                      kv_bytes > 96ll * 1024 * 1024) ? 1 : 0;
    const int64_t units = (int64_t)num_selected_chunks(g, a.rank_lo, a.rank_hi) * a.upc * a.B * a.Hq;
    if (units == 0) return CP_OK;
    const int64_t items = units * (MODE == MODE_SPLIT ? so.n : 1);
    if (items > 0x7fffffffLL) return CP_EUNSUPPORTED;
    a.n_units = (int)units;
    // One block per item while there are many items per SM: the hardware then
    // hands blocks out longest first as SMs free up.  With few items per SM the
    // fixed cost of a block (barrier set-up, tensor-memory allocation, the Q load
    // and the pipeline fill before the first PV, the epilogue) weighs, so one
    // persistent block per SM runs several items, loading the next unit's Q
    // while the previous one finishes.  Its static assignment (alternating
    // rounds over the numbering) balances only a longest-first numbering, so a
    // head-grouped launch keeps one block per item and the hardware's dynamic
    // dispatch.  (A split launch already spreads long rows over blocks; it
    // keeps one block per item too.)
    int64_t blocks = items;
    const int64_t sms = sm_count();
    if (MODE != MODE_SPLIT && !a.head_grouped && items <= 16 * sms && items > sms) blocks = sms;
    const int cap = fwd_grid_limit();   // test hook: the grid, overriding the rule above
    if (cap > 0) blocks = items < cap ? items : cap;
    const float sl2 = a.scale * 1.4426950408889634f;
    if (blocks < items)
        fwd_bf16_kernel<D, MODE, true><<<(unsigned)blocks, NTHREADS, Cfg<D>::SMEM, st>>>(
            mq, mk, mv, a, sl2, reinterpret_cast<__nv_bfloat16 *>(out), lse, so, stp);
    else
        fwd_bf16_kernel<D, MODE, false><<<(unsigned)blocks, NTHREADS, Cfg<D>::SMEM, st>>>(
            mq, mk, mv, a, sl2, reinterpret_cast<__nv_bfloat16 *>(out), lse, so, stp);
    return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ECUDA;
}

}  // namespace

int launch_fwd_bf16(const void *q, const void *k, const void *v, void *out, float *lse,
                    FwdArgs a, cudaStream_t st)
{
    const SplitOut none{1, nullptr, nullptr};
    const StepOut nostep{0, 0, nullptr, nullptr, nullptr};
    if (a.D == 64) return launch_d<64, MODE_RING>(q, k, v, out, lse, a, none, nostep, st);
    if (a.D == 128) return launch_d<128, MODE_RING>(q, k, v, out, lse, a, none, nostep, st);
    return CP_EUNSUPPORTED;
}

int launch_fwd_bf16_split(const void *q, const void *k, const void *v, FwdArgs a,
                          const SplitOut &so, cudaStream_t st)
{
    if (so.n < 1 || !so.out || !so.lse) return CP_EINVAL;
    const StepOut nostep{0, 0, nullptr, nullptr, nullptr};
    if (a.D == 64) return launch_d<64, MODE_SPLIT>(q, k, v, nullptr, nullptr, a, so, nostep, st);
    if (a.D == 128) return launch_d<128, MODE_SPLIT>(q, k, v, nullptr, nullptr, a, so, nostep, st);
    return CP_EUNSUPPORTED;
}

int launch_fwd_bf16_step(const void *q, const void *k, const void *v, FwdArgs a,
                         const StepOut &stp, cudaStream_t st)
{
    if (!stp.out_acc || !stp.lse_acc || a.rank_hi != a.rank_lo + 1) return CP_EINVAL;
    const SplitOut none{1, nullptr, nullptr};
    if (a.D == 64) return launch_d<64, MODE_STEP>(q, k, v, nullptr, nullptr, a, none, stp, st);
    if (a.D == 128) return launch_d<128, MODE_STEP>(q, k, v, nullptr, nullptr, a, none, stp, st);
    return CP_EUNSUPPORTED;
}

}  // namespace cp
