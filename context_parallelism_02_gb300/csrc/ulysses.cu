// ulysses.cu -- the DeepSpeed-Ulysses relayouts as one local permutation.
//
// "Sequence Parallelism in LLMs", "DeepSpeed Ulysses": the first all-to-all
// turns every rank's [Batch, S/P, H, D] sequence shard into [Batch, S, H/P, D]
// (all tokens, one group of H/P heads); the second turns it back.  With all N
// ranks' buffers on one device the pair of collectives is a pure permutation:
//   x[r][b][t][g*H/N + hh][:]  <->  y[g][b][pos(r, t)][hh][:]
// where pos is the layout's shard map (contiguous or zigzag), so that each head
// group sees the sequence in global order.
//
// The unit of copying is a run of H/N heads x D elements, contiguous on both
// sides.  Runs are numbered in the order of the side that is read, so reads
// are fully sequential; each thread moves one vector (16 bytes when sizes and
// pointers allow) per iteration.  HBM-bound: bytes moved = 2 x tensor bytes.
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
    const int ch = s / g.clen;
    r = chunk_rank(g, ch);
    const int within = s - ch * g.clen;
    t = (g.layout == CP_LAYOUT_ZIGZAG && ch >= g.N) ? g.clen + within : within;
}

template <typename V, bool TO_HEAD>
__global__ void __launch_bounds__(256) ulysses_kernel(const V *__restrict__ src, V *__restrict__ dst,
                                                      UlyArgs u)
{
    const int N = u.g.N;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < u.total; v += stride) {
        const int64_t run = v / u.run_vecs;
        const int64_t e = v - run * u.run_vecs;
        int64_t other;
        if (TO_HEAD) {
            // read side x: run = ((r*B + b)*L + t)*N + g
            const int gi = (int)(run % N);
            int64_t rest = run / N;
            const int t = (int)(rest % u.L);
            rest /= u.L;
            const int b = (int)(rest % u.B);
            const int r = (int)(rest / u.B);
            const int s = shard_pos(u.g, r, t);
            other = (((int64_t)gi * u.B + b) * u.g.S + s);
        } else {
            // read side y: run = (g*B + b)*S + s
            const int s = (int)(run % u.g.S);
            int64_t rest = run / u.g.S;
            const int b = (int)(rest % u.B);
            const int gi = (int)(rest / u.B);
            int r, t;
            locate(u.g, s, r, t);
            other = ((((int64_t)r * u.B + b) * u.L + t) * N + gi);
        }
        dst[other * u.run_vecs + e] = src[v];
    }
}

template <typename V>
int launch_v(const void *src, void *dst, const UlyArgs &u, int to_head, cudaStream_t st)
{
    int64_t blocks = (u.total + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) return CP_OK;
    if (to_head)
        ulysses_kernel<V, true><<<(unsigned)blocks, 256, 0, st>>>((const V *)src, (V *)dst, u);
    else
        ulysses_kernel<V, false><<<(unsigned)blocks, 256, 0, st>>>((const V *)src, (V *)dst, u);
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
