// ulysses.cu -- the DeepSpeed-Ulysses relayouts as one local permutation.
//
// "Sequence Parallelism in LLMs", "DeepSpeed Ulysses": the first all-to-all
// turns every rank's [Batch, S/P, H, D] sequence shard into [Batch, S, H/P, D]
// (all tokens, one group of H/P heads); the second turns it back.  With all N
// ranks' buffers on one device the pair of collectives is a pure permutation:
//   x[r][b][t][g*H/N + hh][:]  <->  y[g][b][pos(r, t)][hh][:]
// where pos is the layout's shard map (contiguous, zigzag or striped), so that each head
// group sees the sequence in global order.
//
// The unit of copying is a run of H/N heads x D elements, contiguous on both
// sides.  Runs are numbered in the order of the side that is read, so reads
// are fully sequential, in vectors of 16 bytes when sizes and pointers allow.
// Runs of at least 8 vectors go through the group kernel, which resolves a
// run's destination once per warp and group; shorter runs through a kernel
// that resolves it per vector.  HBM-bound: bytes moved = 2 x tensor bytes.
#include <cuda_runtime.h>

#include "cp_common.cuh"
#include "kernels.h"

namespace cp {

namespace {

struct UlyArgs {
    Geom g;
    int B;
    int64_t L;          // rows per rank shard, S / N
    int64_t run_vecs;   // vectors per run
    int64_t total;      // vectors in the tensor
};

// rank and local row of global position s
__device__ __forceinline__ void locate(const Geom &g, int s, int &r, int &t)
{
    if (striped(g)) {
        r = s % g.N;
        t = s / g.N;
        return;
    }
    const int ch = s / g.clen;
    r = chunk_rank(g, ch);
    const int within = s - ch * g.clen;
    t = (g.layout == CP_LAYOUT_ZIGZAG && ch >= g.N) ? g.clen + within : within;
}

// Destination run of source run `run` (I: 32- or 64-bit index arithmetic).
template <bool TO_HEAD, typename I>
__device__ __forceinline__ I dest_run(const UlyArgs &u, I run)
{
    const I N = (I)u.g.N, B = (I)u.B, L = (I)u.L, S = (I)u.g.S;
    if (TO_HEAD) {
        // read side x: run = ((r*B + b)*L + t)*N + g
        const I gi = run % N;
        I rest = run / N;
        const I t = rest % L;
        rest /= L;
        const I b = rest % B;
        const I r = rest / B;
        const I s = (I)shard_pos(u.g, (int)r, (int)t);
        return (gi * B + b) * S + s;
    }
    // read side y: run = (g*B + b)*S + s
    const I s = run % S;
    I rest = run / S;
    const I b = rest % B;
    const I gi = rest / B;
    int r, t;
    locate(u.g, (int)s, r, t);
    return (((I)r * B + b) * L + (I)t) * N + gi;
}

// Each thread moves UNROLL vectors, blockDim apart (coalesced), with all loads
// issued before the stores so that several requests per thread are in flight.
template <typename V, bool TO_HEAD, typename I>
__global__ void __launch_bounds__(256) ulysses_kernel(const V *__restrict__ src, V *__restrict__ dst,
                                                      UlyArgs u)
{
    constexpr int UNROLL = 4;
    const I total = (I)u.total, rv = (I)u.run_vecs;
    const I step = (I)gridDim.x * blockDim.x * UNROLL;
    for (I v0 = (I)blockIdx.x * blockDim.x * UNROLL + threadIdx.x; v0 < total; v0 += step) {
        V val[UNROLL];
#pragma unroll
        for (int i = 0; i < UNROLL; ++i) {
            const I v = v0 + (I)i * blockDim.x;
            if (v < total) val[i] = src[v];
        }
#pragma unroll
        for (int i = 0; i < UNROLL; ++i) {
            const I v = v0 + (I)i * blockDim.x;
            if (v < total) {
                const I run = v / rv;
                dst[dest_run<TO_HEAD, I>(u, run) * rv + (v - run * rv)] = val[i];
            }
        }
    }
}

// Each warp moves groups of 256 consecutive source vectors (8 per lane, 32
// apart: coalesced, all loads before the stores).  The destination of a run
// is computed once per group, by the lane that owns the run, and handed to
// the lanes that store into it by a warp shuffle; a lane's run and offset
// advance by additions from its first vector.  With at least 8 vectors per
// run a group spans at most 32 runs (one per lane).
template <typename V, bool TO_HEAD, typename I>
__global__ void __launch_bounds__(256) ulysses_group_kernel(const V *__restrict__ src,
                                                            V *__restrict__ dst, UlyArgs u)
{
    constexpr int VPL = 8, GV = 32 * VPL;
    const int lane = threadIdx.x & 31;
    const I total = (I)u.total;
    const I rv = (I)u.run_vecs;
    const I nrun = total / rv;
    const I wid = ((I)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const I nw = ((I)gridDim.x * blockDim.x) >> 5;
    for (I g0 = wid * GV; g0 < total; g0 += nw * GV) {
        V val[VPL];
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const I v = g0 + (I)(lane + 32 * k);
            if (v < total) val[k] = src[v];
        }
        const I r0 = g0 / rv;                        // first run of the group
        const I rj = r0 + (I)lane;                   // the run this lane resolves
        const I dj = rj < nrun ? dest_run<TO_HEAD, I>(u, rj) : (I)0;
        const I first = g0 - r0 * rv + (I)lane;      // offset of this lane's first vector from run r0
        int q = (int)(first / rv);
        I rem = first - (I)q * rv;
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const I d = __shfl_sync(0xffffffffu, dj, q);
            const I v = g0 + (I)(lane + 32 * k);
            if (v < total) dst[d * rv + rem] = val[k];
            rem += 32;
            while (rem >= rv) {
                rem -= rv;
                ++q;
            }
        }
    }
}

template <typename V>
int launch_v(const void *src, void *dst, const UlyArgs &u, int to_head, cudaStream_t st)
{
    if (u.run_vecs >= 8) {
        int64_t blocks = (u.total + 2047) / 2048;    // 8 warps x 256 vectors per block
        const int64_t cap = (int64_t)sm_count() * 8;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) return CP_OK;
        const bool small = u.total < 0x7fffffffLL - 4096 && (int64_t)u.B * u.g.S * u.g.N < 0x7fffffffLL;
        const V *s = (const V *)src;
        V *d = (V *)dst;
        if (small) {
            if (to_head) ulysses_group_kernel<V, true, uint32_t><<<(unsigned)blocks, 256, 0, st>>>(s, d, u);
            else ulysses_group_kernel<V, false, uint32_t><<<(unsigned)blocks, 256, 0, st>>>(s, d, u);
        } else {
            if (to_head) ulysses_group_kernel<V, true, int64_t><<<(unsigned)blocks, 256, 0, st>>>(s, d, u);
            else ulysses_group_kernel<V, false, int64_t><<<(unsigned)blocks, 256, 0, st>>>(s, d, u);
        }
        return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ECUDA;
    }
    int64_t blocks = (u.total + 1023) / 1024;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) return CP_OK;
    const bool small = u.total < 0x7fffffffLL && (int64_t)u.B * u.g.S * u.g.N < 0x7fffffffLL;
    const V *s = (const V *)src;
    V *d = (V *)dst;
    if (small) {
        if (to_head) ulysses_kernel<V, true, uint32_t><<<(unsigned)blocks, 256, 0, st>>>(s, d, u);
        else ulysses_kernel<V, false, uint32_t><<<(unsigned)blocks, 256, 0, st>>>(s, d, u);
    } else {
        if (to_head) ulysses_kernel<V, true, int64_t><<<(unsigned)blocks, 256, 0, st>>>(s, d, u);
        else ulysses_kernel<V, false, int64_t><<<(unsigned)blocks, 256, 0, st>>>(s, d, u);
    }
    return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ECUDA;
}

}  // namespace

int launch_ulysses(const void *src, void *dst, int B, int S, int H, int D, int N, int layout,
                   int elem_bytes, int to_head, cudaStream_t st)
{
    UlyArgs u;
    u.g = make_geom(S, N, layout, 0);
    u.B = B;
    u.L = S / N;
    const int64_t run_bytes = (int64_t)(H / N) * D * elem_bytes;
    const uintptr_t al = (uintptr_t)src | (uintptr_t)dst | (uintptr_t)run_bytes;
    int vb = 16;
    while (vb > 1 && (al % vb)) vb >>= 1;
    u.run_vecs = run_bytes / vb;
    u.total = (int64_t)B * S * H * D * elem_bytes / vb;
    switch (vb) {
    case 16: return launch_v<uint4>(src, dst, u, to_head, st);
    case 8: return launch_v<uint2>(src, dst, u, to_head, st);
    case 4: return launch_v<uint32_t>(src, dst, u, to_head, st);
    case 2: return launch_v<uint16_t>(src, dst, u, to_head, st);
    default: return launch_v<uint8_t>(src, dst, u, to_head, st);
    }
}

}  // namespace cp
