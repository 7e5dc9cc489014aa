// cp_common.cuh -- sequence sharding, ring schedule and tile classifier shared
// by the host entry points and the device kernels of libcp, plus the small
// device helpers every kernel uses (bounded mbarrier waits, error word).
//
// Sharding ("Sequence Parallelism in LLMs: Megatron-SP, Ulysses,
// RingAttention", "Algorithmic Mechanics" step 1; "Context Parallelism",
// "The causal imbalance"): the sequence is cut into chunks of equal length.
// Contiguous: N chunks, rank r holds chunk r.  Zigzag: 2N chunks, rank r holds
// chunks r and 2N-1-r (chunk r first in its local order).  Striped ("Causal
// Masking and Load Balancing", striped partitioning): token p goes to rank
// p mod N, so rank r holds positions r, r+N, r+2N, ... in that order.
//
// Slots: every layout numbers the rows of the ranks' shards 0..S-1, chunk by
// chunk (chunk ch covers slots [ch*clen, (ch+1)*clen)).  For contiguous and
// zigzag a slot is its global position.  For striped, chunk r is rank r's
// whole shard and slot r*clen + t is position r + N t.  The kernels tile
// slots; the causal test "key position <= query position" between a query
// chunk of rank r and a key chunk of rank src reads, in slots,
//   key slot <= query slot + diag_shift(r, src),
// with diag_shift = 0 for contiguous and zigzag and (src-r)*clen - [src > r]
// for striped (key row t_k of src is visible to query row t_q of r iff
// t_k <= t_q - [src > r]).
//
// Ring schedule ("Algorithmic Mechanics" step 2; the ring sketch of "Context
// Parallelism"): at step k = 0..N-1 rank r holds the KV shard of rank
// (r - k) mod N and the causal mask is taken from that shard's global
// positions ("Causal Masking and Load Balancing": key j visible to query i
// iff j <= i).
//
// Tile classifier: a KV tile of the held shard whose first key lies after the
// last query of the unit is fully masked and is never visited; a tile that
// crosses the diagonal (or is cut short by the chunk end) is "partial" and is
// masked element by element; every other tile is fully visible.
#pragma once

#include <stdint.h>

#include "cp.h"

#if defined(__CUDACC__)
#define CP_HD __host__ __device__ __forceinline__
#else
#define CP_HD inline
#endif

namespace cp {

// Error word values (per device, read and cleared by cp_get_error).
constexpr unsigned ERRW_TIMEOUT = 1u;       // a bounded wait ran out
constexpr unsigned ERRW_SMEM_ALIGN = 2u;    // dynamic shared memory not 1 KB aligned
constexpr unsigned ERRW_BOUNDS = 3u;        // debug-bounds build: tile coordinate out of range

// All positions are int32: the library rejects S > INT32_MAX, and 32-bit
// index arithmetic keeps the kernels free of 64-bit division routines.
struct Geom {
    int S;
    int N;
    int layout;
    int causal;
    int clen;       // chunk length: S/N (contiguous) or S/(2N) (zigzag)
    int cpr;        // chunks per rank: 1 or 2
};

CP_HD Geom make_geom(int S, int N, int layout, int causal)
{
    Geom g;
    g.S = S;
    g.N = N;
    g.layout = layout;
    g.causal = causal;
    g.cpr = (layout == CP_LAYOUT_ZIGZAG) ? 2 : 1;
    g.clen = S / (N * g.cpr);
    return g;
}

CP_HD bool striped(const Geom &g) { return g.layout == CP_LAYOUT_STRIPED; }

// Global position of slot u.
CP_HD int slot_pos(const Geom &g, int u)
{
    if (!striped(g)) return u;
    const int r = u / g.clen;
    return r + g.N * (u - r * g.clen);
}

// Causal diagonal between query rank r and key rank src, in slots.
CP_HD int diag_shift(const Geom &g, int r, int src)
{
    if (!striped(g) || !g.causal) return 0;
    return (src - r) * g.clen - (src > r ? 1 : 0);
}

// Coordinates of slot u in the tensor maps (rank, row): a striped shard is
// read with a row stride of N positions, every other layout as one block.
CP_HD int slot_mrank(const Geom &g, int u) { return striped(g) ? u / g.clen : 0; }
CP_HD int slot_mrow(const Geom &g, int u) { return striped(g) ? u - (u / g.clen) * g.clen : u; }

// i-th chunk (0 or 1) held by rank r.
CP_HD int rank_chunk(const Geom &g, int r, int i)
{
    return (g.layout == CP_LAYOUT_ZIGZAG && i == 1) ? 2 * g.N - 1 - r : r;
}

// Rank holding chunk ch.
CP_HD int chunk_rank(const Geom &g, int ch)
{
    return (g.layout == CP_LAYOUT_ZIGZAG && ch >= g.N) ? 2 * g.N - 1 - ch : ch;
}

// Global position of local row t of rank r.
CP_HD int shard_pos(const Geom &g, int r, int t)
{
    if (striped(g)) return r + g.N * t;
    int i = t / g.clen;
    return rank_chunk(g, r, i) * g.clen + (t - i * g.clen);
}

CP_HD int ring_source(int N, int r, int k)
{
    int s = (r - k) % N;
    return s < 0 ? s + N : s;
}

// Row of slot u in the local order of rank r's shard (u must be held by r):
// the shard's first chunk is local rows [0, clen), its second (zigzag)
// [clen, 2 clen).  A shard-local call (flash_block_step) addresses its q, k
// and v buffers this way.
CP_HD int slot_lrow(const Geom &g, int r, int u)
{
    const int ch = u / g.clen;
    return (ch == r ? 0 : g.clen) + (u - ch * g.clen);
}

// Chunks of the ranks [lo, hi), listed by descending global position.  With a
// causal mask a query's work grows with its position, so walking units in this
// order hands out the longest work first.
CP_HD int num_selected_chunks(const Geom &g, int lo, int hi) { return (hi - lo) * g.cpr; }

CP_HD int selected_chunk(const Geom &g, int lo, int hi, int idx)
{
    int nr = hi - lo;
    if (g.layout == CP_LAYOUT_ZIGZAG)
        return idx < nr ? 2 * g.N - 1 - lo - idx : hi - 1 - (idx - nr);
    return hi - 1 - idx;
}

// Number of TILE-key tiles of chunk [cstart, cstart+clen) that a unit whose
// last query slot is qmax must visit (qmax already moved by diag_shift).
template <int TILE>
CP_HD int tiles_needed(const Geom &g, int cstart, int qmax)
{
    int ntiles = (g.clen + TILE - 1) / TILE;
    if (!g.causal) return ntiles;
    if (qmax < cstart) return 0;
    int n = (qmax - cstart) / TILE + 1;
    return n < ntiles ? n : ntiles;
}

// Walks the KV tiles a unit of queries (held by rank r, last query qmax)
// visits, in ring order: steps k = 0..N-1, the source's chunks in local order,
// tiles in increasing position.
template <int TILE>
struct KvIter {
    Geom g;
    int r, qmax;
    int k, ci, kend;    // ring steps [.., kend) are walked
    int t, nt, cstart, cend;
    int src, shift;     // rank holding the current chunk; diag_shift(r, src)

    // the whole ring: steps 0..N-1
    CP_HD void begin(const Geom &g_, int r_, int qmax_) { begin_steps(g_, r_, qmax_, 0, g_.N); }
    // ring steps [k0, k1) only (k1 = k0 + 1: the one block a shard-local step holds)
    CP_HD void begin_steps(const Geom &g_, int r_, int qmax_, int k0, int k1)
    {
        g = g_;
        r = r_;
        qmax = qmax_;
        k = k0;
        kend = k1;
        ci = -1;
        t = nt = cstart = cend = src = shift = 0;
        advance_chunk();
    }
    CP_HD bool advance_chunk()
    {
        for (;;) {
            ++ci;
            if (ci >= g.cpr) {
                ci = 0;
                ++k;
            }
            if (k >= kend) return false;
            src = ring_source(g.N, r, k);
            shift = diag_shift(g, r, src);
            int ch = rank_chunk(g, src, ci);
            cstart = ch * g.clen;
            cend = cstart + g.clen;
            nt = tiles_needed<TILE>(g, cstart, qmax + shift);
            t = 0;
            if (nt > 0) return true;
        }
    }
    CP_HD bool valid() const { return k < kend; }
    CP_HD int start() const { return cstart + t * TILE; }
    // tensor-map coordinates of the tile's first key
    CP_HD int mrank() const { return striped(g) ? src : 0; }
    CP_HD int mrow() const { return striped(g) ? t * TILE : start(); }
    // row of the tile's first key in the source's shard-local buffer
    CP_HD int lrow() const { return ci * g.clen + t * TILE; }
    CP_HD int len() const
    {
        int l = cend - start();
        return l < TILE ? l : TILE;
    }
    CP_HD void next()
    {
        if (++t >= nt) advance_chunk();
    }
    // Advance m tiles (whole chunks at a time where possible).
    CP_HD void skip(int m)
    {
        while (m > 0 && valid()) {
            const int take = nt - t < m ? nt - t : m;
            t += take;
            m -= take;
            if (t >= nt) advance_chunk();
        }
    }
    // Total tiles of the walk over ring steps [k0, k1) (closed form per chunk;
    // the whole ring in closed form, see ring_count).
    CP_HD static int count(const Geom &g, int r, int qmax, int k0 = 0, int k1 = -1)
    {
        if (k1 < 0) k1 = g.N;
        if (k0 == 0 && k1 == g.N) return ring_count(g, r, qmax);
        int n = 0;
        for (int k = k0; k < k1; ++k) {
            int src = ring_source(g.N, r, k);
            for (int ci = 0; ci < g.cpr; ++ci)
                n += tiles_needed<TILE>(g, rank_chunk(g, src, ci) * g.clen,
                                        qmax + diag_shift(g, r, src));
        }
        return n;
    }
    // The whole ring (steps 0..N-1) holds every chunk of the sequence exactly
    // once, so the per-step sum collapses.  Contiguous and zigzag (no diagonal
    // shift): the chunks below the one holding qmax are visible in full, that
    // chunk up to qmax, the chunks above it not at all.  Striped: the chunk of
    // source src shows its local rows up to t - [src > r], t the local row of
    // qmax, for the r + 1 sources src <= r and the N - 1 - r sources above.
    CP_HD static int ring_count(const Geom &g, int r, int qmax)
    {
        const int ntiles = (g.clen + TILE - 1) / TILE;
        if (!g.causal) return g.N * g.cpr * ntiles;
        if (!striped(g)) {
            const int cq = qmax / g.clen;
            const int part = (qmax - cq * g.clen) / TILE + 1;
            return cq * ntiles + (part < ntiles ? part : ntiles);
        }
        const int t = qmax - r * g.clen;
        int lo = t / TILE + 1, hi = t >= 1 ? (t - 1) / TILE + 1 : 0;
        lo = lo < ntiles ? lo : ntiles;
        hi = hi < ntiles ? hi : ntiles;
        return (r + 1) * lo + (g.N - 1 - r) * hi;
    }
};

// A unit of work: `qrows` consecutive query rows of one chunk, for one
// (batch, query head).  Units are numbered heads fastest, then batch, then by
// descending position.
struct Unit {
    int b, h, r;
    int q0;     // first query slot
    int cend;   // end of the unit's chunk (rows at or past it are not stored)
    int qmax;   // last valid query slot
};

// Chunk cu (in selected_chunk order) and position index pu of the i-th of the
// nch * upc units of one (batch, head), numbered longest first: contiguous and
// zigzag chunk by chunk (a unit's work grows with its chunk's position, and
// within a chunk with its own), striped position by position over the chunks
// (every rank's chunk has the same work profile, which grows with the local
// position).
CP_HD void unit_chunk_pos(const Geom &g, int nch, int upc, int i, int &cu, int &pu)
{
    if (striped(g)) {
        cu = i % nch;
        pu = i / nch;
    } else {
        pu = i % upc;
        cu = i / upc;
    }
}

CP_HD Unit decode_unit(const Geom &g, int B, int Hq, int lo, int hi, int upc, int qrows, int u)
{
    Unit w;
    w.h = u % Hq;
    int rest = u / Hq;
    w.b = rest % B;
    rest /= B;
    int cu, pu;
    unit_chunk_pos(g, num_selected_chunks(g, lo, hi), upc, rest, cu, pu);
    int ch = selected_chunk(g, lo, hi, cu);
    w.r = chunk_rank(g, ch);
    int cstart = ch * g.clen;
    w.cend = cstart + g.clen;
    w.q0 = cstart + (upc - 1 - pu) * qrows;
    int last = w.q0 + qrows;
    if (last > w.cend) last = w.cend;
    w.qmax = last - 1;
    return w;
}

// The same units numbered with each (batch, head) contiguous: all query tiles
// of one head (by descending position) before the next head.  Blocks that run
// together then stream the KV tiles of one or two heads, which stay in L2.
CP_HD Unit decode_unit_grouped(const Geom &g, int B, int Hq, int upc, int qrows, int u)
{
    const int nch = num_selected_chunks(g, 0, g.N);
    Unit w;
    int cu, pu;
    unit_chunk_pos(g, nch, upc, u % (nch * upc), cu, pu);
    const int rest = u / (nch * upc);
    w.h = rest % Hq;
    w.b = rest / Hq;
    const int ch = selected_chunk(g, 0, g.N, cu);
    w.r = chunk_rank(g, ch);
    const int cstart = ch * g.clen;
    w.cend = cstart + g.clen;
    w.q0 = cstart + (upc - 1 - pu) * qrows;
    int last = w.q0 + qrows;
    if (last > w.cend) last = w.cend;
    w.qmax = last - 1;
    return w;
}

// ---------------------------------------------------------------------------
// Backward: key-stationary walk.  A KV tile of the shard of rank src receives
// gradient from the queries of every rank r that holds it at some ring step,
// r = (src + k) mod N for k = 0..N-1 (the same (rank, step) pairs the forward
// visits), and from every query head of its GQA group.

// Units of KV tiles: tiles by ascending position (under a causal mask early
// keys receive the most work), then kv head, then batch -- each (batch, kv
// head) contiguous, so that blocks running together read the same queries.
struct KvUnit {
    int b, g;       // batch, kv head
    int src;        // rank holding the tile's chunk
    int ks;         // first key
    int kl;         // valid keys in the tile
    int kcend;      // end of the tile's chunk
};

template <int TILE>
CP_HD KvUnit decode_kv_unit(const Geom &g, int B, int Hkv, int tpc, int u)
{
    KvUnit w;
    const int nch = g.N * g.cpr;
    const int t = u % tpc;
    int rest = u / tpc;
    const int ch = rest % nch;
    rest /= nch;
    w.g = rest % Hkv;
    w.b = rest / Hkv;
    (void)B;
    w.src = chunk_rank(g, ch);
    const int cstart = ch * g.clen;
    w.kcend = cstart + g.clen;
    w.ks = cstart + t * TILE;
    const int l = w.kcend - w.ks;
    w.kl = l < TILE ? l : TILE;
    return w;
}

// Number of TILE-row query tiles of chunk [cstart, cend) that see key slot ks
// (already moved by -diag_shift), and the first of them.
template <int TILE>
CP_HD int qtiles_seeing(const Geom &g, int cstart, int ks, int &t0)
{
    const int ntiles = (g.clen + TILE - 1) / TILE;
    t0 = 0;
    if (!g.causal) return ntiles;
    if (cstart + g.clen - 1 < ks) return 0;
    if (ks - cstart > TILE - 1) t0 = (ks - cstart) / TILE;
    return ntiles - t0;
}

// Walks the query tiles (head, ring step, chunk, tile) that see a KV tile.
template <int TILE>
struct QIter {
    Geom g;
    int src, ks, h0, grp;
    int hh, k, ci, t, t0, nt, cstart, cend;
    int r, shift;       // rank of the current query chunk; diag_shift(r, src)

    CP_HD void begin(const Geom &g_, int src_, int ks_, int h0_, int grp_)
    {
        g = g_;
        src = src_;
        ks = ks_;
        h0 = h0_;
        grp = grp_;
        hh = 0;
        k = 0;
        ci = -1;
        t = nt = t0 = cstart = cend = r = shift = 0;
        advance_chunk();
    }
    CP_HD bool advance_chunk()
    {
        for (;;) {
            ++ci;
            if (ci >= g.cpr) {
                ci = 0;
                ++k;
                if (k >= g.N) {
                    k = 0;
                    ++hh;
                }
            }
            if (hh >= grp) return false;
            r = (src + k) % g.N;
            shift = diag_shift(g, r, src);
            const int ch = rank_chunk(g, r, ci);
            cstart = ch * g.clen;
            cend = cstart + g.clen;
            nt = qtiles_seeing<TILE>(g, cstart, ks - shift, t0);
            t = 0;
            if (nt > 0) return true;
        }
    }
    CP_HD bool valid() const { return hh < grp; }
    CP_HD int head() const { return h0 + hh; }
    CP_HD int start() const { return cstart + (t0 + t) * TILE; }
    // tensor-map coordinates of the tile's first query
    CP_HD int mrank() const { return striped(g) ? r : 0; }
    CP_HD int mrow() const { return striped(g) ? (t0 + t) * TILE : start(); }
    CP_HD int len() const
    {
        const int l = cend - start();
        return l < TILE ? l : TILE;
    }
    CP_HD void next()
    {
        if (++t >= nt) advance_chunk();
    }
    CP_HD static int count(const Geom &g, int src, int ks, int grp)
    {
        int n = 0;
        for (int k = 0; k < g.N; ++k) {
            const int r = (src + k) % g.N;
            for (int ci = 0; ci < g.cpr; ++ci) {
                int t0;
                n += qtiles_seeing<TILE>(g, rank_chunk(g, r, ci) * g.clen,
                                         ks - diag_shift(g, r, src), t0);
            }
        }
        return n * grp;
    }
};

}  // namespace cp

#if defined(__CUDACC__)
namespace cp {

// ---------------------------------------------------------------------------
// Device helpers.

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the same phase (no suspension inside the instruction).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounds below this are the failure-path test hook's: the slow paths then poll
// with the non-blocking test, so that a wait cannot be satisfied inside one
// long suspension and the bound is what decides.
constexpr uint64_t SHORT_WAIT_NS = 1000;

// Debug-bounds build (compiled with -DCP_DEBUG_BOUNDS): a tile coordinate or
// row index outside [0, hi) is recorded in the error word (CP_EBOUNDS) and
// replaced by 0, so the access itself stays in bounds; no trap.  In the
// normal build this is the identity.
__device__ __forceinline__ int dbg_coord(unsigned *err, int v, int hi)
{
#ifdef CP_DEBUG_BOUNDS
    if (v < 0 || v >= hi) {
        atomicCAS(err, 0u, ERRW_BOUNDS);
        return 0;
    }
#else
    (void)err;
    (void)hi;
#endif
    return v;
}

// Shared state of the bounded waits of one block.
struct WaitCtl {
    unsigned *err;          // device error word
    volatile int *abort;    // block-wide "give up" flag in shared memory
    uint64_t limit_ns;      // how long one wait may take
};

__device__ __forceinline__ void raise_timeout(const WaitCtl &w)
{
    *w.abort = 1;
    atomicCAS(w.err, 0u, ERRW_TIMEOUT);
}

// Slow paths of the waits below: spin with try_wait, check the clock and the
// block's abort flag every few rounds.  Kept out of line so that the fast path
// costs no registers.
static __device__ __forceinline__ bool wait1_slow(uint32_t bar, uint32_t parity, WaitCtl w)
{
    uint64_t t0 = globaltimer();
    const bool poll = w.limit_ns < SHORT_WAIT_NS;
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if (*w.abort) return false;
        if (globaltimer() - t0 > w.limit_ns) {
            raise_timeout(w);
            return false;
        }
    }
}

static __device__ __forceinline__ bool waitw_slow(uint32_t bar, uint32_t parity, WaitCtl w)
{
    const unsigned FULL = 0xffffffffu;
    uint64_t t0 = globaltimer();
    const bool poll = w.limit_ns < SHORT_WAIT_NS;
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (__all_sync(FULL, poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)))
                return true;
        int give_up = 0;
        if ((threadIdx.x & 31) == 0) {
            if (*w.abort) give_up = 1;
            else if (globaltimer() - t0 > w.limit_ns) {
                raise_timeout(w);
                give_up = 1;
            }
        }
        if (__shfl_sync(FULL, give_up, 0)) return false;
    }
}

// First probe of a wait: try_wait, which may suspend inside the instruction
// until the phase completes; under a failure-path test bound (below
// SHORT_WAIT_NS) the non-blocking test, so that a phase still pending at the
// first probe always reaches the bound check.
__device__ __forceinline__ bool mbar_probe(uint32_t bar, uint32_t parity, const WaitCtl &w)
{
    return w.limit_ns >= SHORT_WAIT_NS ? mbar_try_wait(bar, parity) : mbar_test_wait(bar, parity);
}

// Single-thread bounded wait on phase `parity` of an mbarrier.  Returns false
// when the limit ran out (the error word is set) or another thread gave up.
__device__ __forceinline__ bool wait1(uint32_t bar, uint32_t parity, const WaitCtl &w)
{
    if (mbar_probe(bar, parity, w)) return true;
    return wait1_slow(bar, parity, w);
}

// Warp-collective bounded wait: every lane observes the phase, and the
// outcome is the same on all lanes (so .sync.aligned instructions that follow
// never diverge).
__device__ __forceinline__ bool waitw(uint32_t bar, uint32_t parity, const WaitCtl &w)
{
    if (__all_sync(0xffffffffu, mbar_probe(bar, parity, w))) return true;
    return waitw_slow(bar, parity, w);
}

}  // namespace cp
#endif
