// lse_merge.cu -- merge two (or n) normalised partial attention results.
//
// "Sequence Parallelism in LLMs", "Algorithmic Mechanics" (online softmax
// rescaling): with each partial carried as (out_x, lse_x) = (O, m + ln l),
// m = max(lse_a, lse_b), w_x = e^(lse_x - m) / (e^(lse_a - m) + e^(lse_b - m)),
// out = w_a out_a + w_b out_b and lse = m + ln(e^(lse_a - m) + e^(lse_b - m)).
// An empty partial (lse = -inf) gets weight 0; two empty partials give
// (0, -inf).
//
// HBM-bound: per row it reads 2 rows of D floats + 2 lse and writes one row +
// one lse.  One warp per row, 16-byte vectors, two rows in flight per warp,
// grid sized to fill every SM.
#include <cuda_runtime.h>
#include <math.h>

#include "cp_common.cuh"
#include "kernels.h"

namespace cp {

namespace {

struct Weights {
    float wa, wb, lse;
};

__device__ __forceinline__ Weights merge_weights(float la, float lb)
{
    Weights r;
    const float m = fmaxf(la, lb);
    if (m == -INFINITY) {
        r.wa = r.wb = 0.f;
        r.lse = -INFINITY;
        return r;
    }
    const float ea = expf(la - m), eb = expf(lb - m);
    const float s = ea + eb;
    r.wa = ea / s;
    r.wb = eb / s;
    r.lse = m + logf(s);
    return r;
}

__device__ __forceinline__ float4 axpby(float wa, float4 a, float wb, float4 b)
{
    return make_float4(fmaf(wa, a.x, wb * b.x), fmaf(wa, a.y, wb * b.y), fmaf(wa, a.z, wb * b.z),
                       fmaf(wa, a.w, wb * b.w));
}

__global__ void __launch_bounds__(256) lse_merge_kernel(const float4 *xa,
                                                        const float *la,
                                                        const float4 *xb,
                                                        const float *lb, float4 *xo, float *lo,
                                                        int64_t rows, int d4)
{
    const int lane = threadIdx.x & 31;
    const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r0 = 2 * wid; r0 < rows; r0 += 2 * nw) {
        const int64_t r1 = r0 + 1;
        const bool two = r1 < rows;
        const float a0 = la[r0], b0 = lb[r0];
        const float a1 = two ? la[r1] : -INFINITY, b1 = two ? lb[r1] : -INFINITY;
        for (int i = lane; i < d4; i += 32) {
            const float4 va0 = xa[r0 * d4 + i], vb0 = xb[r0 * d4 + i];
            float4 va1, vb1;
            if (two) {
                va1 = xa[r1 * d4 + i];
                vb1 = xb[r1 * d4 + i];
            }
            const Weights w0 = merge_weights(a0, b0);
            xo[r0 * d4 + i] = axpby(w0.wa, va0, w0.wb, vb0);
            if (two) {
                const Weights w1 = merge_weights(a1, b1);
                xo[r1 * d4 + i] = axpby(w1.wa, va1, w1.wb, vb1);
            }
        }
        // every lane has read la/lb of both rows before lane 0 overwrites them
        __syncwarp();
        if (lane == 0) {
            lo[r0] = merge_weights(a0, b0).lse;
            if (two) lo[r1] = merge_weights(a1, b1).lse;
        }
    }
}

// n-way merge: lse = m + ln sum_i e^(lse_i - m), out = sum_i e^(lse_i - lse) out_i
// with m = max_i lse_i.  One warp per row; every lane reads the n lse values
// of the row (a broadcast load) and keeps its own column vectors, so out may
// alias the first partial.  Partials are read four at a time to keep loads in
// flight.
__global__ void __launch_bounds__(256) lse_merge_n_kernel(const float4 *xs, const float *ls, int n,
                                                          int64_t rows, int d4, float4 *xo, float *lo)
{
    const int lane = threadIdx.x & 31;
    const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t pstride = rows * d4;   // float4s per partial
    for (int64_t r = wid; r < rows; r += nw) {
        float m = -INFINITY;
        for (int i = 0; i < n; ++i) m = fmaxf(m, ls[(int64_t)i * rows + r]);
        float l = 0.f;
        if (m != -INFINITY)
            for (int i = 0; i < n; ++i) l += expf(ls[(int64_t)i * rows + r] - m);
        const float inv = m == -INFINITY ? 0.f : 1.f / l;
        for (int c = lane; c < d4; c += 32) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 *x = xs + r * d4 + c;
            int i = 0;
            if (m != -INFINITY) {
                for (; i + 4 <= n; i += 4) {
                    float4 v[4];
                    float w[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        v[u] = x[(int64_t)(i + u) * pstride];
                        w[u] = expf(ls[(int64_t)(i + u) * rows + r] - m) * inv;
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        acc.x = fmaf(w[u], v[u].x, acc.x);
                        acc.y = fmaf(w[u], v[u].y, acc.y);
                        acc.z = fmaf(w[u], v[u].z, acc.z);
                        acc.w = fmaf(w[u], v[u].w, acc.w);
                    }
                }
                for (; i < n; ++i) {
                    const float4 v = x[(int64_t)i * pstride];
                    const float w = expf(ls[(int64_t)i * rows + r] - m) * inv;
                    acc.x = fmaf(w, v.x, acc.x);
                    acc.y = fmaf(w, v.y, acc.y);
                    acc.z = fmaf(w, v.z, acc.z);
                    acc.w = fmaf(w, v.w, acc.w);
                }
            }
            xo[r * d4 + c] = acc;
        }
        // every lane has read the row's lse values before lane 0 overwrites one
        __syncwarp();
        if (lane == 0) lo[r] = m == -INFINITY ? -INFINITY : m + logf(l);
    }
}

__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int off = 16; off; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
    return x;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int off = 16; off; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// n <= 32: lane i holds partial i's weight (one exp per partial and row),
// RPW rows per warp, the column vectors of up to 4 partials of every row in
// flight before their weights are applied (4 rows for small n, where a row
// alone moves too few bytes to cover the memory latency).
template <int RPW>
__global__ void __launch_bounds__(256) lse_merge_n32_kernel(const float4 *xs, const float *ls, int n,
                                                            int64_t rows, int d4, float4 *xo, float *lo)
{
    const int lane = threadIdx.x & 31;
    const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t pstride = rows * d4;   // float4s per partial
    for (int64_t r0 = RPW * wid; r0 < rows; r0 += RPW * nw) {
        float m[RPW], sum[RPW];
        // the column loop runs the same number of times on every lane (the
        // weight shuffles below need the whole warp); lanes past d4 only idle
        for (int c0 = 0; c0 < d4; c0 += 32) {
            const int c = c0 + lane;
            const bool act = c < d4;
            const float4 *x0 = xs + r0 * d4 + c;
            // the first four partials' columns are requested before the
            // weights, so that both memory latencies overlap
            float4 v[RPW][4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int j = 0; j < RPW; ++j) {
                    v[j][u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (act && u < n && r0 + j < rows) v[j][u] = x0[(int64_t)u * pstride + j * d4];
                }
            float w[RPW];
#pragma unroll
            for (int j = 0; j < RPW; ++j) {
                const bool in = lane < n && r0 + j < rows;
                const float a = in ? ls[(int64_t)lane * rows + r0 + j] : -INFINITY;
                m[j] = warp_max(a);
                const float e = m[j] == -INFINITY ? 0.f : expf(a - m[j]);
                sum[j] = warp_sum(e);
                w[j] = sum[j] > 0.f ? e / sum[j] : 0.f;
            }
            float4 acc[RPW];
#pragma unroll
            for (int j = 0; j < RPW; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int i = 0; i < n; i += 4) {
                if (i > 0) {
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int j = 0; j < RPW; ++j) {
                            v[j][u] = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (act && i + u < n && r0 + j < rows)
                                v[j][u] = x0[(int64_t)(i + u) * pstride + j * d4];
                        }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int j = 0; j < RPW; ++j) {
                        const float q = __shfl_sync(0xffffffffu, w[j], (i + u) & 31);
                        if (i + u < n) {
                            acc[j].x = fmaf(q, v[j][u].x, acc[j].x);
                            acc[j].y = fmaf(q, v[j][u].y, acc[j].y);
                            acc[j].z = fmaf(q, v[j][u].z, acc[j].z);
                            acc[j].w = fmaf(q, v[j][u].w, acc[j].w);
                        }
                    }
            }
            if (act) {
#pragma unroll
                for (int j = 0; j < RPW; ++j)
                    if (r0 + j < rows) xo[(r0 + j) * d4 + c] = acc[j];
            }
        }
        // every lane has read the rows' lse values before lane 0 overwrites them
        __syncwarp();
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < RPW; ++j)
                if (r0 + j < rows) lo[r0 + j] = m[j] == -INFINITY ? -INFINITY : m[j] + logf(sum[j]);
        }
    }
}

}  // namespace

int launch_lse_merge_n(const float *out_parts, const float *lse_parts, int n, int64_t rows, int D,
                       float *out, float *lse, cudaStream_t st)
{
    if (rows == 0) return CP_OK;
    if (n == 2)   // the two-way kernel keeps more bytes in flight per warp
        return launch_lse_merge(out_parts, lse_parts, out_parts + rows * D, lse_parts + rows, out, lse,
                                rows, D, st);
    const int64_t cap = (int64_t)sm_count() * 8;
    if (n <= 32) {
        const int rpw = n <= 4 ? 4 : 2;
        int64_t blocks = ((rows + rpw - 1) / rpw + 7) / 8;
        if (blocks > cap) blocks = cap;
        const float4 *xs = reinterpret_cast<const float4 *>(out_parts);
        float4 *xo = reinterpret_cast<float4 *>(out);
        if (rpw == 4)
            lse_merge_n32_kernel<4><<<(unsigned)blocks, 256, 0, st>>>(xs, lse_parts, n, rows, D / 4, xo, lse);
        else
            lse_merge_n32_kernel<2><<<(unsigned)blocks, 256, 0, st>>>(xs, lse_parts, n, rows, D / 4, xo, lse);
        return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ECUDA;
    }
    int64_t blocks = (rows + 7) / 8;
    if (blocks > cap) blocks = cap;
    lse_merge_n_kernel<<<(unsigned)blocks, 256, 0, st>>>(
        reinterpret_cast<const float4 *>(out_parts), lse_parts, n, rows, D / 4,
        reinterpret_cast<float4 *>(out), lse);
    return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ECUDA;
}

int launch_lse_merge(const float *out_a, const float *lse_a, const float *out_b,
                     const float *lse_b, float *out, float *lse, int64_t rows, int D,
                     cudaStream_t st)
{
    if (rows == 0) return CP_OK;
    const int64_t warps_needed = (rows + 1) / 2;
    int64_t blocks = (warps_needed + 7) / 8;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    lse_merge_kernel<<<(unsigned)blocks, 256, 0, st>>>(
        reinterpret_cast<const float4 *>(out_a), lse_a, reinterpret_cast<const float4 *>(out_b),
        lse_b, reinterpret_cast<float4 *>(out), lse, rows, D / 4);
    return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ECUDA;
}

}  // namespace cp
