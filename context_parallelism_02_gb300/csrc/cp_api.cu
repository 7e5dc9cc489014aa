// cp_api.cu -- the extern "C" entry points of libcp (declared in cp.h):
// argument checking, dispatch to the kernels, and the per-device error word.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "cp.h"
#include "cp_common.cuh"
#include "kernels.h"

namespace cp {

// Per-device error word: a kernel whose bounded wait runs out writes a code
// here (first writer wins); cp_get_error reads and clears it.
__device__ unsigned g_err_word;

namespace {

constexpr int MAX_DEV = 64;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;   // 2 s per device-side wait

// Bound of the pipeline waits of kernels launched from now on; 0 selects
// WAIT_LIMIT_NS.  Only the cp_debug_set_wait_limit test hook changes it.
std::atomic<uint64_t> g_pipeline_limit_ns{0};

// Largest grid of the forward kernel; 0: no limit.  Only the
// cp_debug_set_grid_limit test hook changes it.
std::atomic<int> g_fwd_grid_limit{0};

uint64_t pipeline_limit_ns()
{
    const uint64_t v = g_pipeline_limit_ns.load(std::memory_order_relaxed);
    return v ? v : WAIT_LIMIT_NS;
}

unsigned *err_ptr()
{
    static unsigned *ptrs[MAX_DEV] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEV) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<unsigned *>(p);
    }
    return ptrs[dev];
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// An NVTX range named after the entry point, open for the host-side part of
// the call (argument checks and launches), so that a profiler's timeline
// attributes the kernels that follow to the call that queued them.  With no
// tool attached a push or pop costs a few nanoseconds.
struct NvtxScope {
    explicit NvtxScope(const char *name) { nvtxRangePushA(name); }
    ~NvtxScope() { nvtxRangePop(); }
    NvtxScope(const NvtxScope &) = delete;
    NvtxScope &operator=(const NvtxScope &) = delete;
};

int check_shard(int64_t S, int N, int layout)
{
    if (N < 1 || S < 0 || S > 0x7fffffffLL) return CP_EINVAL;
    if (layout != CP_LAYOUT_CONTIGUOUS && layout != CP_LAYOUT_ZIGZAG && layout != CP_LAYOUT_STRIPED)
        return CP_EINVAL;
    if (S % N) return CP_EINVAL;
    if (layout == CP_LAYOUT_ZIGZAG && S % (2 * (int64_t)N)) return CP_EINVAL;
    return CP_OK;
}

// sum over queries i in [qa, qb) of |{j in [ks, ks+L) : j <= i}|, in closed form
int64_t visible_pairs(int64_t qa, int64_t qb, int64_t ks, int64_t L)
{
    int64_t sum = 0;
    // queries that see a strict prefix of the tile: ks <= i <= ks+L-2, count i-ks+1
    const int64_t lo = qa > ks ? qa : ks;
    const int64_t hi = (qb - 1) < (ks + L - 2) ? (qb - 1) : (ks + L - 2);
    if (lo <= hi) {
        const int64_t x1 = lo - ks + 1, x2 = hi - ks + 1;
        sum += (x1 + x2) * (x2 - x1 + 1) / 2;
    }
    // queries that see the whole tile: i >= ks+L-1
    const int64_t full_lo = qa > (ks + L - 1) ? qa : (ks + L - 1);
    if (qb > full_lo) sum += L * (qb - full_lo);
    return sum;
}

// Argument checks shared by the forward entry points (no CUDA call); fills a
// except a.err.  Returns CP_OK, an error code, or 1 for an empty problem
// (nothing to launch).
int prepare_fwd(const void *q, const void *k, const void *v, const void *out, const float *lse,
                int B, int Hq, int Hkv, int64_t S, int D, int N, int causal, int layout, int dtype,
                float scale, int rank_lo, int rank_hi, FwdArgs &a)
{
    if (B < 0 || Hq < 1 || Hkv < 1 || (causal != 0 && causal != 1)) return CP_EINVAL;
    int rc = check_shard(S, N, layout);
    if (rc) return rc;
    if (Hq % Hkv) return CP_EINVAL;
    if (rank_lo < 0 || rank_hi > N || rank_lo >= rank_hi) return CP_EINVAL;
    if (dtype != CP_F32 && dtype != CP_BF16) return CP_EUNSUPPORTED;
    if (D != 64 && D != 128) return CP_EUNSUPPORTED;
    if (B == 0 || S == 0) return 1;
    if (!q || !k || !v || !out || !lse) return CP_EINVAL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || ((uintptr_t)lse & 3u))
        return CP_EINVAL;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.S = (int)S;
    a.D = D;
    a.N = N;
    a.causal = causal;
    a.layout = layout;
    a.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
    a.rank_lo = rank_lo;
    a.rank_hi = rank_hi;
    a.upc = 0;
    a.head_grouped = 0;
    a.n_units = 0;
    a.err = nullptr;
    a.limit_ns = pipeline_limit_ns();
    a.drain_ns = WAIT_LIMIT_NS;
    return CP_OK;
}

int fwd_common(const void *q, const void *k, const void *v, void *out, float *lse, int B, int Hq,
               int Hkv, int64_t S, int D, int N, int causal, int layout, int dtype, float scale,
               int rank_lo, int rank_hi, void *stream)
{
    FwdArgs a;
    const int rc = prepare_fwd(q, k, v, out, lse, B, Hq, Hkv, S, D, N, causal, layout, dtype, scale,
                               rank_lo, rank_hi, a);
    if (rc) return rc == 1 ? CP_OK : rc;
    a.err = err_ptr();
    if (!a.err) return CP_ECUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dtype == CP_F32)
        return launch_fwd_f32(static_cast<const float *>(q), static_cast<const float *>(k),
                              static_cast<const float *>(v), static_cast<float *>(out), lse, a, st);
    return launch_fwd_bf16(q, k, v, out, lse, a, st);
}

// Bytes of a split forward's partials: n (D + 1) fp32 per (batch, position,
// head), rounded up to 256; 0 if that overflows.
size_t split_workspace_bytes(int B, int Hq, int64_t S, int D, int n)
{
    const unsigned __int128 b = (unsigned __int128)n * (unsigned)B * (uint64_t)S * (unsigned)Hq *
                                (unsigned)(D + 1) * 4u;
    if (b > ((unsigned __int128)1 << 62)) return 0;
    return (size_t)((b + 255) / 256 * 256);
}

}  // namespace

unsigned *device_error_word() { return err_ptr(); }

uint64_t device_wait_limit_ns() { return pipeline_limit_ns(); }

uint64_t device_drain_limit_ns() { return WAIT_LIMIT_NS; }

int fwd_grid_limit() { return g_fwd_grid_limit.load(std::memory_order_relaxed); }

int sm_count()
{
    static int counts[MAX_DEV] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEV) return 148;
    if (!counts[dev]) {
        int c = 0;
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c < 1)
            c = 148;
        counts[dev] = c;
    }
    return counts[dev];
}

}  // namespace cp

using namespace cp;

extern "C" {

int cp_shard_map(int64_t S, int N, int layout, int32_t *pos_host)
{
    if (!pos_host) return CP_EINVAL;
    int rc = check_shard(S, N, layout);
    if (rc) return rc;
    if (S == 0) return CP_OK;
    const Geom g = make_geom((int)S, N, layout, 1);
    const int L = (int)(S / N);
    for (int r = 0; r < N; ++r)
        for (int t = 0; t < L; ++t) pos_host[(int64_t)r * L + t] = shard_pos(g, r, t);
    return CP_OK;
}

int cp_schedule_pairs(int64_t S, int N, int layout, int causal, int64_t *pairs_host,
                      int64_t *tiles_host)
{
    if (!pairs_host) return CP_EINVAL;
    int rc = check_shard(S, N, layout);
    if (rc) return rc;
    for (int i = 0; i < N * N; ++i) {
        pairs_host[i] = 0;
        if (tiles_host) tiles_host[i] = 0;
    }
    if (S == 0) return CP_OK;
    // Walk the units and KV tiles of the bf16 kernel (one 128-row query tile
    // per unit, 256-key KV tiles) and count what each query tile covers.
    constexpr int QROWS = 128, T = 256;
    const Geom g = make_geom((int)S, N, layout, causal);
    const int upc = (g.clen + QROWS - 1) / QROWS;
    const int units = num_selected_chunks(g, 0, N) * upc;
    for (int u = 0; u < units; ++u) {
        const Unit w = decode_unit(g, 1, 1, 0, N, upc, QROWS, u);
        KvIter<T> it;
        it.begin(g, w.r, w.qmax);
        for (; it.valid(); it.next()) {
            const int64_t ks = it.start(), ke = ks + it.len();   // keys [ks, ke)
            for (int qi = 0; qi < QROWS / 128; ++qi) {
                const int64_t qa = w.q0 + (int64_t)qi * 128;
                int64_t qb = qa + 128;                         // queries [qa, qb)
                if (qb > w.cend) qb = w.cend;
                if (qa >= qb) continue;
                // in slots the causal diagonal moves by it.shift (striped)
                const int64_t p = causal ? visible_pairs(qa, qb, ks - it.shift, ke - ks)
                                         : (qb - qa) * (ke - ks);
                pairs_host[w.r * N + it.k] += p;
                if (tiles_host) tiles_host[w.r * N + it.k] += 1;
            }
        }
    }
    return CP_OK;
}

int ring_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                  int Hq, int Hkv, int64_t S, int D, int N, int causal, int layout, int dtype,
                  float scale, void *stream)
{
    NvtxScope nvtx_("ring_attn_fwd");
    return fwd_common(q, k, v, out, lse, B, Hq, Hkv, S, D, N, causal, layout, dtype, scale, 0, N,
                      stream);
}

int ring_attn_fwd_rank(const void *q, const void *k, const void *v, void *out, float *lse,
                       int B, int Hq, int Hkv, int64_t S, int D, int N, int causal, int layout,
                       int dtype, float scale, int rank_lo, int rank_hi, void *stream)
{
    NvtxScope nvtx_("ring_attn_fwd_rank");
    return fwd_common(q, k, v, out, lse, B, Hq, Hkv, S, D, N, causal, layout, dtype, scale,
                      rank_lo, rank_hi, stream);
}

int flash_block_step(const void *q, const void *k, const void *v, float *out_acc, float *lse_acc,
                     void *out_final, int B, int Hq, int Hkv, int64_t S, int D, int N, int rank,
                     int source, int causal, int layout, int dtype, float scale, int accumulate,
                     void *stream)
{
    NvtxScope nvtx_("flash_block_step");
    if (N < 1 || rank < 0 || rank >= N || source < 0 || source >= N) return CP_EINVAL;
    if (accumulate != 0 && accumulate != 1) return CP_EINVAL;
    FwdArgs a;
    const int rc = prepare_fwd(q, k, v, out_acc, lse_acc, B, Hq, Hkv, S, D, N, causal, layout,
                               dtype, scale, rank, rank + 1, a);
    if (rc) return rc == 1 ? CP_OK : rc;
    if (out_final && !aligned16(out_final)) return CP_EINVAL;
    a.err = err_ptr();
    if (!a.err) return CP_ECUDA;
    StepOut so;
    so.step_k = ((rank - source) % N + N) % N;
    so.accumulate = accumulate;
    so.out_acc = out_acc;
    so.lse_acc = lse_acc;
    so.out_final = out_final;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dtype == CP_F32)
        return launch_fwd_f32_step(static_cast<const float *>(q), static_cast<const float *>(k),
                                   static_cast<const float *>(v), a, so, st);
    return launch_fwd_bf16_step(q, k, v, a, so, st);
}

size_t ring_attn_fwd_split_workspace(int B, int Hq, int64_t S, int D, int n_split)
{
    if (B < 0 || Hq < 0 || S < 0 || S > 0x7fffffffLL || (D != 64 && D != 128) || n_split < 1 ||
        n_split > CP_MAX_SPLIT)
        return 0;
    return split_workspace_bytes(B, Hq, S, D, n_split);
}

int cp_fwd_split_count(int B, int Hq, int64_t S, int D, int N, int causal, int layout, int rank_lo,
                       int rank_hi, int num_sms)
{
    if (B < 1 || Hq < 1 || (causal != 0 && causal != 1) || num_sms < 1) return CP_EINVAL;
    int rc = check_shard(S, N, layout);
    if (rc) return rc;
    if (S == 0) return CP_EINVAL;
    if (rank_lo < 0 || rank_hi > N || rank_lo >= rank_hi) return CP_EINVAL;
    if (D != 64 && D != 128) return CP_EUNSUPPORTED;
    return fwd_split_choose(B, Hq, (int)S, D, N, causal, layout, rank_lo, rank_hi, num_sms, 32);
}

int ring_attn_fwd_split(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                        int Hq, int Hkv, int64_t S, int D, int N, int causal, int layout, int dtype,
                        float scale, int rank_lo, int rank_hi, int n_split, void *workspace,
                        size_t ws_bytes, void *stream)
{
    NvtxScope nvtx_("ring_attn_fwd_split");
    if (n_split < 1 || n_split > CP_MAX_SPLIT) return CP_EINVAL;
    FwdArgs a;
    const int rc = prepare_fwd(q, k, v, out, lse, B, Hq, Hkv, S, D, N, causal, layout, dtype, scale,
                               rank_lo, rank_hi, a);
    if (rc < 0) return rc;
    if (dtype != CP_BF16) return CP_EUNSUPPORTED;
    if (rc == 1) return CP_OK;
    const size_t need = split_workspace_bytes(B, Hq, S, D, n_split);
    if (n_split > 1 && (!workspace || !aligned16(workspace) || need == 0 || ws_bytes < need))
        return CP_EINVAL;
    a.err = err_ptr();
    if (!a.err) return CP_ECUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (n_split == 1) return launch_fwd_bf16(q, k, v, out, lse, a, st);
    SplitOut so;
    so.n = n_split;
    so.out = static_cast<float *>(workspace);
    so.lse = so.out + (int64_t)n_split * B * S * Hq * D;
    int r = launch_fwd_bf16_split(q, k, v, a, so, st);
    if (r) return r;
    return launch_fwd_split_combine(a, so, out, lse, st);
}

size_t ring_attn_bwd_workspace(int B, int Hq, int64_t S)
{
    if (B < 0 || Hq < 0 || S < 0) return 0;
    return bwd_workspace_bytes(B, Hq, S);
}

int ring_attn_bwd(const void *q, const void *k, const void *v, const void *out, const float *lse,
                  const void *dout, void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int64_t S,
                  int D, int N, int causal, int layout, int dtype, float scale, void *workspace,
                  size_t ws_bytes, void *stream)
{
    NvtxScope nvtx_("ring_attn_bwd");
    if (B < 0 || Hq < 1 || Hkv < 1 || (causal != 0 && causal != 1)) return CP_EINVAL;
    int rc = check_shard(S, N, layout);
    if (rc) return rc;
    if (Hq % Hkv) return CP_EINVAL;
    if (dtype != CP_BF16 && dtype != CP_F32) return CP_EUNSUPPORTED;
    if (D != 64 && D != 128) return CP_EUNSUPPORTED;
    if (B == 0 || S == 0) return CP_OK;
    if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv || !workspace) return CP_EINVAL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace) ||
        ((uintptr_t)lse & 3u))
        return CP_EINVAL;
    if (ws_bytes < bwd_workspace_bytes(B, Hq, S)) return CP_EINVAL;
    FwdArgs a;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.S = (int)S;
    a.D = D;
    a.N = N;
    a.causal = causal;
    a.layout = layout;
    a.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
    a.rank_lo = 0;
    a.rank_hi = N;
    a.upc = 0;
    a.head_grouped = 0;
    a.n_units = 0;
    a.err = err_ptr();
    a.limit_ns = pipeline_limit_ns();
    a.drain_ns = WAIT_LIMIT_NS;
    if (!a.err) return CP_ECUDA;
    BwdPtrs p{q, k, v, out, lse, dout, dq, dk, dv, workspace};
    if (dtype == CP_F32) return launch_bwd_f32(p, a, static_cast<cudaStream_t>(stream));
    return launch_bwd_bf16(p, a, static_cast<cudaStream_t>(stream));
}

int lse_merge(const float *out_a, const float *lse_a, const float *out_b, const float *lse_b,
              float *out, float *lse, int64_t rows, int D, void *stream)
{
    NvtxScope nvtx_("lse_merge");
    if (rows < 0 || D < 4 || D % 4) return CP_EINVAL;
    if (rows == 0) return CP_OK;
    if (!out_a || !lse_a || !out_b || !lse_b || !out || !lse) return CP_EINVAL;
    if (!aligned16(out_a) || !aligned16(out_b) || !aligned16(out)) return CP_EINVAL;
    if (((uintptr_t)lse_a | (uintptr_t)lse_b | (uintptr_t)lse) & 3u) return CP_EINVAL;
    return launch_lse_merge(out_a, lse_a, out_b, lse_b, out, lse, rows, D,
                            static_cast<cudaStream_t>(stream));
}

int lse_merge_n(const float *out_parts, const float *lse_parts, int n, int64_t rows, int D,
                float *out, float *lse, void *stream)
{
    NvtxScope nvtx_("lse_merge_n");
    if (n < 1 || rows < 0 || D < 4 || D % 4) return CP_EINVAL;
    if (rows > INT64_MAX / D / n) return CP_EINVAL;
    if (rows == 0) return CP_OK;
    if (!out_parts || !lse_parts || !out || !lse) return CP_EINVAL;
    if (!aligned16(out_parts) || !aligned16(out)) return CP_EINVAL;
    if (((uintptr_t)lse_parts | (uintptr_t)lse) & 3u) return CP_EINVAL;
    return launch_lse_merge_n(out_parts, lse_parts, n, rows, D, out, lse,
                              static_cast<cudaStream_t>(stream));
}

size_t usp_attn_fwd_workspace(int Hq, int Hkv, int64_t S, int D, int dtype)
{
    if (Hq < 1 || Hkv < 1 || S < 0 || D < 1 || (dtype != CP_F32 && dtype != CP_BF16)) return 0;
    const size_t elem = dtype == CP_BF16 ? 2 : 4;
    // one batch at a time: q and out (Hq heads), k and v (Hkv heads), head-group-major
    const size_t b = (size_t)(2 * Hq + 2 * Hkv) * (size_t)S * (size_t)D * elem;
    return (b + 255u) & ~(size_t)255u;
}

int usp_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse, int B, int Hq,
                 int Hkv, int64_t S, int D, int n_ulysses, int n_ring, int causal, int layout,
                 int dtype, float scale, void *workspace, size_t ws_bytes, void *stream)
{
    NvtxScope nvtx_("usp_attn_fwd");
    if (n_ulysses < 1 || n_ring < 1 || B < 0 || Hq < 1 || Hkv < 1) return CP_EINVAL;
    if (Hq % Hkv) return CP_EINVAL;
    int rc = check_shard(S, n_ring, layout);
    if (rc) return rc;
    rc = check_shard(S, n_ulysses, CP_LAYOUT_CONTIGUOUS);
    if (rc) return rc;
    if (Hq % n_ulysses || Hkv % n_ulysses) return CP_EHEADS;   // P <= H_KV per Ulysses group
    if (dtype != CP_F32 && dtype != CP_BF16) return CP_EUNSUPPORTED;
    if (D != 64 && D != 128) return CP_EUNSUPPORTED;
    if (B == 0 || S == 0) return CP_OK;
    if (!q || !k || !v || !out || !lse || !workspace) return CP_EINVAL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(workspace) ||
        ((uintptr_t)lse & 3u))
        return CP_EINVAL;
    if (ws_bytes < usp_attn_fwd_workspace(Hq, Hkv, S, D, dtype)) return CP_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t elem = dtype == CP_BF16 ? 2 : 4;
    const int hq = Hq / n_ulysses, hkv = Hkv / n_ulysses;
    const int64_t rowq = S * Hq * D * elem, rowkv = S * Hkv * D * elem;   // bytes per batch
    char *ws = static_cast<char *>(workspace);
    char *yq = ws, *yk = yq + rowq, *yv = yk + rowkv, *yo = yv + rowkv;
    for (int b = 0; b < B; ++b) {
        // Ulysses all-to-all (seq -> head): batch b's [S][H][D] is the stack of
        // n_ulysses sequence shards; each group u receives the whole sequence
        // for heads [u H/n_ulysses, (u+1) H/n_ulysses)
        const char *qb = static_cast<const char *>(q) + b * rowq;
        const char *kb = static_cast<const char *>(k) + b * rowkv;
        const char *vb = static_cast<const char *>(v) + b * rowkv;
        if ((rc = launch_ulysses(qb, yq, 1, (int)S, Hq, D, n_ulysses, CP_LAYOUT_CONTIGUOUS, (int)elem, 1, st)) ||
            (rc = launch_ulysses(kb, yk, 1, (int)S, Hkv, D, n_ulysses, CP_LAYOUT_CONTIGUOUS, (int)elem, 1, st)) ||
            (rc = launch_ulysses(vb, yv, 1, (int)S, Hkv, D, n_ulysses, CP_LAYOUT_CONTIGUOUS, (int)elem, 1, st)))
            return rc;
        // ring attention within every head group over n_ring virtual ranks;
        // the group's lse rows [b][u H/n_ulysses ...][S] are contiguous in lse
        for (int u = 0; u < n_ulysses; ++u) {
            rc = fwd_common(yq + u * S * hq * D * elem, yk + u * S * hkv * D * elem,
                            yv + u * S * hkv * D * elem, yo + u * S * hq * D * elem,
                            lse + ((int64_t)b * Hq + (int64_t)u * hq) * S, 1, hq, hkv, S, D, n_ring,
                            causal, layout, dtype, scale, 0, n_ring, stream);
            if (rc) return rc;
        }
        // the second all-to-all (head -> seq) puts out back in BSHD order
        if ((rc = launch_ulysses(yo, static_cast<char *>(out) + b * rowq, 1, (int)S, Hq, D, n_ulysses,
                                 CP_LAYOUT_CONTIGUOUS, (int)elem, 0, st)))
            return rc;
    }
    return CP_OK;
}

static int ulysses_common(const void *src, void *dst, int B, int64_t S, int H, int D, int N,
                          int layout, int elem_bytes, int to_head, void *stream)
{
    if (B < 0 || H < 1 || D < 1) return CP_EINVAL;
    if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8) return CP_EINVAL;
    int rc = check_shard(S, N, layout);
    if (rc) return rc;
    if (H % N) return CP_EHEADS;
    if (B == 0 || S == 0) return CP_OK;
    if (!src || !dst) return CP_EINVAL;
    return launch_ulysses(src, dst, B, (int)S, H, D, N, layout, elem_bytes, to_head,
                          static_cast<cudaStream_t>(stream));
}

int ulysses_seq_to_head(const void *x, void *y, int B, int64_t S, int H, int D, int N,
                        int layout, int elem_bytes, void *stream)
{
    NvtxScope nvtx_("ulysses_seq_to_head");
    return ulysses_common(x, y, B, S, H, D, N, layout, elem_bytes, 1, stream);
}

int ulysses_head_to_seq(const void *y, void *x, int B, int64_t S, int H, int D, int N,
                        int layout, int elem_bytes, void *stream)
{
    NvtxScope nvtx_("ulysses_head_to_seq");
    return ulysses_common(y, x, B, S, H, D, N, layout, elem_bytes, 0, stream);
}

int cp_get_error(void *stream)
{
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return CP_ECUDA;
    unsigned w = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&w, g_err_word, sizeof(w)) != cudaSuccess) return CP_ECUDA;
    if (w && cudaMemcpyToSymbol(g_err_word, &zero, sizeof(zero)) != cudaSuccess) return CP_ECUDA;
    if (w == ERRW_TIMEOUT) return CP_ETIMEOUT;
    if (w == ERRW_SMEM_ALIGN) return CP_ESMEM;
    if (w == ERRW_BOUNDS) return CP_EBOUNDS;
    return w ? CP_ECUDA : CP_OK;
}

const char *cp_strerror(int code)
{
    switch (code) {
    case CP_OK: return "ok";
    case CP_EINVAL: return "invalid argument (null pointer, size, divisibility or alignment)";
    case CP_EHEADS: return "head count not divisible by the number of ranks (P <= H ceiling)";
    case CP_EUNSUPPORTED: return "unsupported dtype, head dimension or shape";
    case CP_ECUDA: return "CUDA runtime or launch failure";
    case CP_ETIMEOUT: return "a device-side bounded wait ran out; outputs are undefined";
    case CP_ESMEM: return "a kernel's dynamic shared memory was not 1 KB aligned; it returned without work";
    case CP_EBOUNDS:
        return "debug-bounds build: a kernel met an out-of-range tile coordinate and skipped it";
    default: return "unknown status code";
    }
}

int cp_debug_set_wait_limit(uint64_t limit_ns)
{
    if (limit_ns > WAIT_LIMIT_NS) return CP_EINVAL;
    g_pipeline_limit_ns.store(limit_ns, std::memory_order_relaxed);
    return CP_OK;
}

int cp_debug_set_grid_limit(int max_blocks)
{
    if (max_blocks < 0) return CP_EINVAL;
    g_fwd_grid_limit.store(max_blocks, std::memory_order_relaxed);
    return CP_OK;
}

int cp_debug_wait_timeout(uint64_t limit_ns, void *stream)
{
    if (limit_ns < 1000ull) limit_ns = 1000ull;
    if (limit_ns > 5000000000ull) limit_ns = 5000000000ull;
    unsigned *e = err_ptr();
    if (!e) return CP_ECUDA;
    return launch_debug_wait(e, limit_ns, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
