// fwd_f32.cu -- fp32 ring-attention forward on the CUDA cores (fp64 arithmetic).
//
// The fp32 path has to agree with an fp64 reference to ~1e-5 even with
// logits of several tens (q scaled by 8), which rules out the tf32
// tensor-core kinds and also plain fp32 dot products: a logit near 30 carries
// an fp32 rounding error of ~2e-6, which a near one-hot softmax passes
// straight into the output.  So this kernel reads and writes fp32 but forms
// scores, the running max and sum, and the output accumulator in fp64 on the
// CUDA cores.  It is the precision path, not the fast path.  It walks exactly the ring schedule
// of the bf16 kernel ("Algorithmic Mechanics": step k uses the KV shard of
// rank (i-k) mod P; flash_block of the "Context Parallelism" ring sketch) with
// 16-row query units and 32-key KV tiles, and folds every tile into the
// running (O, m, l) with the online-softmax rescaling equations of
// "Algorithmic Mechanics".
//
// STEP: one ring step of one rank on shard-local buffers (flash_block_step):
// q is the rank's shard and k, v the source's block, in local row order; the
// block's (out, lse) is merged into the running fp32 state in fp64.
#include <cuda_runtime.h>
#include <math.h>

#include "cp_common.cuh"
#include "kernels.h"

namespace cp {

namespace {

constexpr int QR = 16;      // query rows per unit
constexpr int TK = 32;      // keys per KV tile
constexpr int WARPS = 8;
constexpr int ROWS_PER_WARP = QR / WARPS;

template <int D, bool STEP>
__global__ void __launch_bounds__(WARPS * 32) fwd_f32_kernel(const float *__restrict__ q,
                                                             const float *__restrict__ k,
                                                             const float *__restrict__ v,
                                                             float *__restrict__ out,
                                                             float *__restrict__ lse,
                                                             FwdArgs a, const StepOut stp)
{
    constexpr int DPL = D / 32;   // output elements per lane
    __shared__ float Qs[QR][D];
    __shared__ float Ks[TK][D + 1];
    __shared__ float Vs[TK][D];

    const Geom g = make_geom(a.S, a.N, a.layout, a.causal);
    const Unit w = decode_unit(g, a.B, a.Hq, a.rank_lo, a.rank_hi, a.upc, QR, blockIdx.x);
    const int grp = a.Hq / a.Hkv;
    const int kvh = w.h / grp;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C_loc = g.clen * g.cpr;   // rows of one shard (STEP buffers)

    // load the query rows of the unit (rows past the chunk end are zero)
    for (int i = threadIdx.x; i < QR * D; i += blockDim.x) {
        int rr = i / D, d = i % D;
        int pos = w.q0 + rr;   // slot; its global position is slot_pos
        const int64_t row = STEP ? (int64_t)w.b * C_loc + slot_lrow(g, w.r, pos)
                                 : (int64_t)w.b * a.S + slot_pos(g, pos);
        Qs[rr][d] = (pos < w.cend) ? q[(row * a.Hq + w.h) * D + d] : 0.f;
    }

    double o[ROWS_PER_WARP][DPL];
    double m[ROWS_PER_WARP], l[ROWS_PER_WARP];
#pragma unroll
    for (int i = 0; i < ROWS_PER_WARP; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.0;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[i][e] = 0.0;
    }
    const double scale = (double)a.scale;

    KvIter<TK> it;
    if (STEP)
        it.begin_steps(g, w.r, w.qmax, stp.step_k, stp.step_k + 1);
    else
        it.begin(g, w.r, w.qmax);
    for (; it.valid(); it.next()) {
        const int ks = it.start();
        const int kl = it.len();
        __syncthreads();
        for (int i = threadIdx.x; i < TK * D; i += blockDim.x) {
            int j = i / D, d = i % D;
            float kv = 0.f, vv = 0.f;
            if (j < kl) {
                const int64_t row = STEP ? (int64_t)w.b * C_loc + it.lrow() + j
                                         : (int64_t)w.b * a.S + slot_pos(g, ks + j);
                int64_t off = (row * a.Hkv + kvh) * D + d;
                kv = k[off];
                vv = v[off];
            }
            Ks[j][d] = kv;
            Vs[j][d] = vv;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < ROWS_PER_WARP; ++i) {
            const int rr = warp * ROWS_PER_WARP + i;
            const int qpos = w.q0 + rr;
            // lane j scores key j
            double s = 0.0;
#pragma unroll 8
            for (int d = 0; d < D; ++d) s = fma((double)Qs[rr][d], (double)Ks[lane][d], s);
            s *= scale;
            const bool vis = lane < kl && (!a.causal || ks + lane <= qpos + it.shift);
            if (!vis) s = -INFINITY;
            double mt = s;
#pragma unroll
            for (int off = 16; off; off >>= 1) mt = fmax(mt, __shfl_xor_sync(0xffffffffu, mt, off));
            const double mn = fmax(m[i], mt);
            if (mn == -INFINITY) continue;   // nothing visible yet: state unchanged
            const double alpha = exp(m[i] - mn);
            const double p = vis ? exp(s - mn) : 0.0;
            double ps = p;
#pragma unroll
            for (int off = 16; off; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
            l[i] = l[i] * alpha + ps;
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[i][e] *= alpha;
#pragma unroll 4
            for (int j = 0; j < TK; ++j) {
                const double pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
                for (int e = 0; e < DPL; ++e) o[i][e] = fma(pj, (double)Vs[j][lane + 32 * e], o[i][e]);
            }
            m[i] = mn;
        }
    }

#pragma unroll
    for (int i = 0; i < ROWS_PER_WARP; ++i) {
        const int rr = warp * ROWS_PER_WARP + i;
        const int qpos = w.q0 + rr;
        if (qpos >= w.cend) continue;
        const double inv = l[i] > 0.0 ? 1.0 / l[i] : 0.0;
        if constexpr (STEP) {
            // merge (o / l, m + ln l) into the state: lse_new = ln(e^lse + e^lse_blk),
            // out_new = e^(lse - lse_new) out + e^(lse_blk - lse_new) o / l
            const int64_t srow = ((int64_t)w.b * C_loc + slot_lrow(g, w.r, qpos)) * a.Hq + w.h;
            float *lp = stp.lse_acc + ((int64_t)w.b * a.Hq + w.h) * C_loc + slot_lrow(g, w.r, qpos);
            double prev = -INFINITY;
            if (stp.accumulate) prev = __shfl_sync(0xffffffffu, lane == 0 ? (double)*lp : 0.0, 0);
            const double blk = l[i] > 0.0 ? m[i] + log(l[i]) : -INFINITY;
            const double mx = fmax(prev, blk);
            double wa = 0.0, wb = 0.0, lnew = -INFINITY;
            if (mx != -INFINITY) {
                const double ea = exp(prev - mx), eb = exp(blk - mx);
                lnew = mx + log(ea + eb);
                wa = ea / (ea + eb);
                wb = eb / (ea + eb) * inv;
            }
            float *orow = stp.out_acc + srow * D;
            float *frow = static_cast<float *>(stp.out_final);
#pragma unroll
            for (int e = 0; e < DPL; ++e) {
                const double pv = stp.accumulate ? (double)orow[lane + 32 * e] : 0.0;
                const float r = (float)(wa * pv + wb * o[i][e]);
                orow[lane + 32 * e] = r;
                if (frow) frow[srow * D + lane + 32 * e] = r;
            }
            if (lane == 0) *lp = (float)lnew;
            continue;
        }
        const int qp = slot_pos(g, qpos);
        float *orow = out + (((int64_t)w.b * a.S + qp) * a.Hq + w.h) * D;
#pragma unroll
        for (int e = 0; e < DPL; ++e) orow[lane + 32 * e] = (float)(o[i][e] * inv);
        if (lane == 0)
            lse[((int64_t)w.b * a.Hq + w.h) * a.S + qp] =
                l[i] > 0.0 ? (float)(m[i] + log(l[i])) : -INFINITY;
    }
}

}  // namespace

int launch_fwd_f32(const float *q, const float *k, const float *v, float *out, float *lse,
                   FwdArgs a, cudaStream_t st)
{
    const Geom g = make_geom(a.S, a.N, a.layout, a.causal);
    a.upc = (g.clen + QR - 1) / QR;
    const int64_t units = (int64_t)num_selected_chunks(g, a.rank_lo, a.rank_hi) * a.upc * a.B * a.Hq;
    if (units == 0) return CP_OK;
    if (units > 0x7fffffffLL) return CP_EUNSUPPORTED;
    dim3 grid((unsigned)units), block(WARPS * 32);
    const StepOut nostep{0, 0, nullptr, nullptr, nullptr};
    if (a.D == 64)
        fwd_f32_kernel<64, false><<<grid, block, 0, st>>>(q, k, v, out, lse, a, nostep);
    else
        fwd_f32_kernel<128, false><<<grid, block, 0, st>>>(q, k, v, out, lse, a, nostep);
    return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ECUDA;
}

int launch_fwd_f32_step(const float *q, const float *k, const float *v, FwdArgs a,
                        const StepOut &stp, cudaStream_t st)
{
    if (!stp.out_acc || !stp.lse_acc || a.rank_hi != a.rank_lo + 1) return CP_EINVAL;
    const Geom g = make_geom(a.S, a.N, a.layout, a.causal);
    a.upc = (g.clen + QR - 1) / QR;
    const int64_t units = (int64_t)num_selected_chunks(g, a.rank_lo, a.rank_hi) * a.upc * a.B * a.Hq;
    if (units == 0) return CP_OK;
    if (units > 0x7fffffffLL) return CP_EUNSUPPORTED;
    dim3 grid((unsigned)units), block(WARPS * 32);
    if (a.D == 64)
        fwd_f32_kernel<64, true><<<grid, block, 0, st>>>(q, k, v, nullptr, nullptr, a, stp);
    else
        fwd_f32_kernel<128, true><<<grid, block, 0, st>>>(q, k, v, nullptr, nullptr, a, stp);
    return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ECUDA;
}

}  // namespace cp
