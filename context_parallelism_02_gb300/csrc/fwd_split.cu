// fwd_split.cu -- split-KV forward: the merge of the per-split partials, and
// the host-side choice of the number of splits.
//
// A unit of the forward (one 128-row query tile of one (batch, head)) walks
// the KV tiles of its N ring steps.  When the launch has few units, or a few
// very long ones (one rank's queries of a long sequence, one or two heads),
// the blocks of the last wave leave SMs idle.  The split forward cuts every
// walk into n consecutive pieces, runs each piece as its own block, and
// merges the n normalised partials of every row with the log-sum-exp
// combination of "Sequence Parallelism in LLMs", "Algorithmic Mechanics"
// (online softmax rescaling; lse = m + ln l):
//   lse = ln sum_i e^lse_i,   out = sum_i e^(lse_i - lse) out_i.
// The pieces cover disjoint key sets, so the merge is exact up to rounding.
// A piece with no visible key carries lse = -inf and drops out.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include <functional>
#include <queue>
#include <vector>

#include "cp_common.cuh"
#include "kernels.h"

namespace cp {

namespace {

// One group of D/4 lanes per output row, one float4 of each partial per lane.
// Rows are numbered (batch, selected slot, head): the heads of one position
// are adjacent rows of out and of the partials.
template <int D>
__global__ void __launch_bounds__(256) split_combine_kernel(const float4 *__restrict__ po,
                                                            const float *__restrict__ pl, int ns,
                                                            int64_t pstride, Geom g, int Hq, int lo,
                                                            int hi, int64_t rows,
                                                            __nv_bfloat16 *__restrict__ out,
                                                            float *__restrict__ lse)
{
    constexpr int LPR = D / 4;      // lanes per row
    constexpr int RPW = 32 / LPR;   // rows per warp
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR, c = lane - sub * LPR;
    const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t nsel = (int64_t)num_selected_chunks(g, lo, hi) * g.clen;   // slots per batch
    for (int64_t r = wid * RPW + sub; r < rows; r += nw * RPW) {
        const int h = (int)(r % Hq);
        const int64_t rest = r / Hq;
        const int ts = (int)(rest % nsel);
        const int b = (int)(rest / nsel);
        const int cu = ts / g.clen;
        const int slot = selected_chunk(g, lo, hi, cu) * g.clen + (ts - cu * g.clen);
        const int qp = slot_pos(g, slot);
        const int64_t orow = ((int64_t)b * g.S + qp) * Hq + h;   // row of out and of every partial
        float m = -INFINITY;
        for (int i = 0; i < ns; ++i) m = fmaxf(m, pl[i * pstride + orow]);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float sum = 0.f;
        if (m != -INFINITY) {
#pragma unroll 4
            for (int i = 0; i < ns; ++i) {
                const float li = pl[i * pstride + orow];
                const float4 x = po[(i * pstride + orow) * LPR + c];
                const float e = li == -INFINITY ? 0.f : expf(li - m);
                sum += e;
                acc.x = fmaf(e, x.x, acc.x);
                acc.y = fmaf(e, x.y, acc.y);
                acc.z = fmaf(e, x.z, acc.z);
                acc.w = fmaf(e, x.w, acc.w);
            }
            const float inv = 1.f / sum;
            acc.x *= inv;
            acc.y *= inv;
            acc.z *= inv;
            acc.w *= inv;
        }
        const __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x, acc.y);
        const __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t *>(&lo2);
        pk.y = *reinterpret_cast<const uint32_t *>(&hi2);
        reinterpret_cast<uint2 *>(out + orow * D)[c] = pk;
        if (c == 0) lse[((int64_t)b * Hq + h) * g.S + qp] = m == -INFINITY ? -INFINITY : m + logf(sum);
    }
}

// Cost model of the split choice, in units of one 128 x 256 tile of the
// forward kernel (about 2,700 SM cycles, ~1.45 us at D = 128; a D = 64 tile
// has the same softmax work and half the MMA work).  The fixed cost of a
// block (launch, barrier set-up, tensor-memory allocation, the first Q/K
// loads and the unoverlapped first tile, the epilogue) was fitted to timed
// launches of 1 to 16 splits on a GB300: about 10 tiles (~15 us).
constexpr double BLOCK_OVERHEAD_TILES = 10.0;
constexpr double EMPTY_BLOCK_TILES = 1.0;      // an empty split: launch + the identity rows
constexpr double MIN_GAIN = 0.97;              // more splits only if at least 3 % cheaper
constexpr double COMBINE_LAUNCH_TILES = 4.0;
constexpr double HBM_BYTES_PER_S = 6.5e12;

}  // namespace

int launch_fwd_split_combine(const FwdArgs &a, const SplitOut &so, void *out, float *lse,
                             cudaStream_t st)
{
    const Geom g = make_geom(a.S, a.N, a.layout, a.causal);
    const int64_t rows = (int64_t)a.B * num_selected_chunks(g, a.rank_lo, a.rank_hi) * g.clen * a.Hq;
    if (rows == 0) return CP_OK;
    const int64_t pstride = (int64_t)a.B * a.S * a.Hq;
    const int rpw = 32 / (a.D / 4);
    int64_t blocks = (rows + 8 * rpw - 1) / (8 * rpw);
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    const float4 *po = reinterpret_cast<const float4 *>(so.out);
    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(out);
    if (a.D == 128)
        split_combine_kernel<128><<<(unsigned)blocks, 256, 0, st>>>(po, so.lse, so.n, pstride, g, a.Hq,
                                                                    a.rank_lo, a.rank_hi, rows, o, lse);
    else if (a.D == 64)
        split_combine_kernel<64><<<(unsigned)blocks, 256, 0, st>>>(po, so.lse, so.n, pstride, g, a.Hq,
                                                                   a.rank_lo, a.rank_hi, rows, o, lse);
    else
        return CP_EUNSUPPORTED;
    return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ECUDA;
}

// Pick the number of splits: simulate the block dispatcher (blocks start in
// launch order on the SM that frees first, one block per SM) for each
// candidate count, add the merge pass, and keep the cheapest, preferring
// fewer splits unless more are at least 3 % cheaper.
int fwd_split_choose(int B, int Hq, int S, int D, int N, int causal, int layout, int rank_lo,
                     int rank_hi, int num_sms, int max_split)
{
    if (B < 1 || Hq < 1 || S < 1 || N < 1 || num_sms < 1 || max_split < 1) return 1;
    const Geom g = make_geom(S, N, layout, causal);
    const int upc = (g.clen + 127) / 128;
    const int nch = num_selected_chunks(g, rank_lo, rank_hi);
    const bool grouped = rank_lo == 0 && rank_hi == N;
    const int64_t units = (int64_t)nch * upc * B * Hq;
    // no split is a candidate (too many blocks already): skip the simulation
    if (max_split < 2 || units * 2 > 64LL * num_sms) return 1;
    std::vector<int> tiles((size_t)nch * upc);
    for (int cu = 0; cu < nch; ++cu) {
        const int ch = selected_chunk(g, rank_lo, rank_hi, cu);
        const int cstart = ch * g.clen, cend = cstart + g.clen;
        for (int pu = 0; pu < upc; ++pu) {
            const int q0 = cstart + (upc - 1 - pu) * 128;
            const int last = q0 + 128 < cend ? q0 + 128 : cend;
            tiles[(size_t)cu * upc + pu] = KvIter<256>::count(g, chunk_rank(g, ch), last - 1);
        }
    }
    const int64_t rows = (int64_t)B * nch * g.clen * Hq;
    const double tile_s = D == 128 ? 1.45e-6 : 1.1e-6;
    static const int cand[] = {1, 2, 3, 4, 5, 6, 8, 10, 12, 16, 20, 24, 32};
    double best = 0.0;
    int best_n = 1;
    for (int ns : cand) {
        if (ns > max_split) break;
        if (ns > 1 && units * ns > 64LL * num_sms) break;
        std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
        for (int i = 0; i < num_sms; ++i) free_at.push(0.0);
        double makespan = 0.0;
        for (int sp = 0; sp < ns; ++sp)   // blocks in launch order: split index slowest
            for (int64_t u = 0; u < units; ++u) {
                int cu, pu;
                unit_chunk_pos(g, nch, upc, (int)(grouped ? u % ((int64_t)nch * upc) : u / ((int64_t)B * Hq)), cu,
                               pu);
                const int64_t n = tiles[(size_t)(cu * upc + pu)];
                const int64_t len = n * (sp + 1) / ns - n * sp / ns;
                const double t =
                    free_at.top() + (len > 0 ? BLOCK_OVERHEAD_TILES + (double)len : EMPTY_BLOCK_TILES);
                free_at.pop();
                free_at.push(t);
                if (t > makespan) makespan = t;
            }
        double cost = makespan;
        if (ns > 1) {
            const double bytes = (double)rows * ((double)ns * (4.0 * D + 4.0) + 2.0 * D + 4.0);
            cost += COMBINE_LAUNCH_TILES + bytes / HBM_BYTES_PER_S / tile_s;
        }
        if (ns == 1 || cost < MIN_GAIN * best) {
            best = cost;
            best_n = ns;
        }
    }
    return best_n;
}

}  // namespace cp
