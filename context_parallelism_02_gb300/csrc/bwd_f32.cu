// bwd_f32.cu -- fp32 ring-attention backward on the FMA pipes (precision path).
//
// The same textbook gradient as the bf16 tensor-core kernels (the pages give
// no backward algorithm; "Sequence and Context Parallelism", "What it does not
// change", states only that the gradients equal single-device training):
//   P = exp(scale * q k^T - lse)   (masked by global positions)
//   Delta_i = rowsum(dO_i * out_i)
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - Delta)
//   dQ = scale * dS K,  dK = scale * dS^T Q
// Inputs and outputs are fp32; every score, exponential, dot product and
// accumulator is fp64 (as in the fp32 forward), so the result is the exact
// gradient up to the fp32 rounding of the inputs and outputs.  Delta is
// formed in fp64 by each kernel from out and dO, so the fp32 path leaves the
// caller's workspace untouched.
//
// Two kernels, no atomics (every output element is written once):
//   dQ   -- query-stationary: 8 query rows per block (one per warp), walking
//           the KV tiles of the ring schedule (32 keys, one per lane).
//   dK/dV -- key-stationary: 8 keys per block (one per warp), walking the
//           query tiles (32 queries, one per lane) of every (rank, step,
//           head of the GQA group) that sees them.
// Each warp first scores its row against the 32 rows of the tile (one per
// lane), then switches to one output column per lane to accumulate.
#include <cuda_runtime.h>
#include <math.h>

#include "cp_common.cuh"
#include "kernels.h"

namespace cp {

namespace {

constexpr int WARPS = 8;
constexpr int QR = 8;      // dQ kernel: query rows per block
constexpr int TK = 32;     // dQ kernel: keys per KV tile
constexpr int KR = 8;      // dK/dV kernel: key rows per block
constexpr int TQ = 32;     // dK/dV kernel: queries per query tile

struct F32Args {
    int B, Hq, Hkv, S, N, causal, layout;
    double scale;
    int upc;    // query units (QR rows) per chunk
    int tpc;    // key units (KR rows) per chunk
};

__device__ __forceinline__ double warp_sum(double x)
{
#pragma unroll
    for (int off = 16; off; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

template <int D>
__global__ void __launch_bounds__(WARPS * 32)
    bwd_f32_dq_kernel(const float *__restrict__ q, const float *__restrict__ k,
                      const float *__restrict__ v, const float *__restrict__ out,
                      const float *__restrict__ dout, const float *__restrict__ lse,
                      float *__restrict__ dq, F32Args a)
{
    constexpr int DPL = D / 32;   // columns per lane (d = lane + 32 e)
    __shared__ float Ks[TK][D + 1];
    __shared__ float Vs[TK][D + 1];
    __shared__ float Qs[QR][D];
    __shared__ float DOs[QR][D];
    __shared__ double dss[QR][TK];

    const Geom g = make_geom(a.S, a.N, a.layout, a.causal);
    const Unit w = decode_unit(g, a.B, a.Hq, 0, a.N, a.upc, QR, blockIdx.x);
    const int kvh = w.h / (a.Hq / a.Hkv);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = warp;
    const int qpos = w.q0 + row;              // slot
    const int qp = slot_pos(g, qpos);         // global position
    const bool valid = qpos < w.cend;

    // the warp's query row, and Delta = rowsum(dO * out) in fp64
    double dlt = 0.0;
    const int64_t roff = (((int64_t)w.b * a.S + qp) * a.Hq + w.h) * D;
#pragma unroll
    for (int e = 0; e < DPL; ++e) {
        const int d = lane + 32 * e;
        float qv = 0.f, gv = 0.f, ov = 0.f;
        if (valid) {
            qv = q[roff + d];
            gv = dout[roff + d];
            ov = out[roff + d];
        }
        Qs[row][d] = qv;
        DOs[row][d] = gv;
        dlt = fma((double)gv, (double)ov, dlt);
    }
    dlt = warp_sum(dlt);
    const double lse_i = valid ? (double)lse[((int64_t)w.b * a.Hq + w.h) * a.S + qp] : 0.0;

    double acc[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] = 0.0;

    KvIter<TK> it;
    it.begin(g, w.r, w.qmax);
    for (; it.valid(); it.next()) {
        const int ks = it.start(), kl = it.len();
        __syncthreads();
        for (int i = threadIdx.x; i < TK * D; i += blockDim.x) {
            const int j = i / D, d = i % D;
            float kv = 0.f, vv = 0.f;
            if (j < kl) {
                const int64_t off = (((int64_t)w.b * a.S + slot_pos(g, ks + j)) * a.Hkv + kvh) * D + d;
                kv = k[off];
                vv = v[off];
            }
            Ks[j][d] = kv;
            Vs[j][d] = vv;
        }
        __syncthreads();
        // lane j: dS of (row, key j)
        double ds = 0.0;
        if (valid && lane < kl && (!a.causal || ks + lane <= qpos + it.shift)) {
            double s = 0.0, dp = 0.0;
#pragma unroll 8
            for (int d = 0; d < D; ++d) {
                s = fma((double)Qs[row][d], (double)Ks[lane][d], s);
                dp = fma((double)DOs[row][d], (double)Vs[lane][d], dp);
            }
            const double p = exp(s * a.scale - lse_i);
            ds = p * (dp - dlt);
        }
        dss[row][lane] = ds;
        __syncwarp();
        // lane d: dQ += dS K
#pragma unroll 4
        for (int j = 0; j < TK; ++j) {
            const double dsj = dss[row][j];
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[e] = fma(dsj, (double)Ks[j][lane + 32 * e], acc[e]);
        }
        __syncwarp();
    }
    if (valid) {
#pragma unroll
        for (int e = 0; e < DPL; ++e) dq[roff + lane + 32 * e] = (float)(acc[e] * a.scale);
    }
}

template <int D>
__global__ void __launch_bounds__(WARPS * 32)
    bwd_f32_dkdv_kernel(const float *__restrict__ q, const float *__restrict__ k,
                        const float *__restrict__ v, const float *__restrict__ out,
                        const float *__restrict__ dout, const float *__restrict__ lse,
                        float *__restrict__ dk, float *__restrict__ dv, F32Args a)
{
    constexpr int DPL = D / 32;
    constexpr int RPW = TQ / WARPS;   // query rows each warp loads
    __shared__ float Qs[TQ][D + 1];
    __shared__ float DOs[TQ][D + 1];
    __shared__ float Ks[KR][D];
    __shared__ float Vs[KR][D];
    __shared__ double lses[TQ], dlts[TQ];
    __shared__ double pvs[KR][TQ], dss[KR][TQ];

    const Geom g = make_geom(a.S, a.N, a.layout, a.causal);
    const KvUnit w = decode_kv_unit<KR>(g, a.B, a.Hkv, a.tpc, blockIdx.x);
    const int grp = a.Hq / a.Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = warp;                 // the warp's key row
    const int kpos = w.ks + j;   // slot
    const bool kvalid = j < w.kl;
    const int64_t koff = (((int64_t)w.b * a.S + slot_pos(g, kpos)) * a.Hkv + w.g) * D;
#pragma unroll
    for (int e = 0; e < DPL; ++e) {
        const int d = lane + 32 * e;
        Ks[j][d] = kvalid ? k[koff + d] : 0.f;
        Vs[j][d] = kvalid ? v[koff + d] : 0.f;
    }
    double adk[DPL], adv[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) adk[e] = adv[e] = 0.0;

    QIter<TQ> it;
    it.begin(g, w.src, w.ks, w.g * grp, grp);
    for (; it.valid(); it.next()) {
        const int qa = it.start(), ql = it.len(), h = it.head();
        __syncthreads();
        // rows c of the query tile: q, dO, lse, Delta (fp64)
        for (int rr = 0; rr < RPW; ++rr) {
            const int c = warp * RPW + rr;
            const bool cv = c < ql;
            const int qc = cv ? slot_pos(g, qa + c) : 0;
            const int64_t off = (((int64_t)w.b * a.S + qc) * a.Hq + h) * D;
            double dl = 0.0;
#pragma unroll
            for (int e = 0; e < DPL; ++e) {
                const int d = lane + 32 * e;
                float qv = 0.f, gv = 0.f, ov = 0.f;
                if (cv) {
                    qv = q[off + d];
                    gv = dout[off + d];
                    ov = out[off + d];
                }
                Qs[c][d] = qv;
                DOs[c][d] = gv;
                dl = fma((double)gv, (double)ov, dl);
            }
            dl = warp_sum(dl);
            if (lane == 0) {
                dlts[c] = dl;
                lses[c] = cv ? (double)lse[((int64_t)w.b * a.Hq + h) * a.S + qc] : 0.0;
            }
        }
        __syncthreads();
        // lane c: P and dS of (query c, key j)
        double p = 0.0, ds = 0.0;
        if (kvalid && lane < ql && (!a.causal || qa + lane >= kpos - it.shift)) {
            double s = 0.0, dp = 0.0;
#pragma unroll 8
            for (int d = 0; d < D; ++d) {
                s = fma((double)Qs[lane][d], (double)Ks[j][d], s);
                dp = fma((double)DOs[lane][d], (double)Vs[j][d], dp);
            }
            p = exp(s * a.scale - lses[lane]);
            ds = p * (dp - dlts[lane]);
        }
        pvs[j][lane] = p;
        dss[j][lane] = ds;
        __syncwarp();
        // lane d: dV += P^T dO, dK += dS^T Q
#pragma unroll 4
        for (int c = 0; c < TQ; ++c) {
            const double pc = pvs[j][c], dc = dss[j][c];
#pragma unroll
            for (int e = 0; e < DPL; ++e) {
                adv[e] = fma(pc, (double)DOs[c][lane + 32 * e], adv[e]);
                adk[e] = fma(dc, (double)Qs[c][lane + 32 * e], adk[e]);
            }
        }
        __syncwarp();
    }
    if (kvalid) {
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
            dk[koff + lane + 32 * e] = (float)(adk[e] * a.scale);
            dv[koff + lane + 32 * e] = (float)adv[e];
        }
    }
}

template <int D>
int launch_d(const BwdPtrs &p, const F32Args &a, cudaStream_t st)
{
    const Geom g = make_geom(a.S, a.N, a.layout, a.causal);
    const int64_t qunits = (int64_t)num_selected_chunks(g, 0, a.N) * a.upc * a.B * a.Hq;
    const int64_t kunits = (int64_t)g.N * g.cpr * a.tpc * a.B * a.Hkv;
    if (qunits > 0x7fffffffLL || kunits > 0x7fffffffLL) return CP_EUNSUPPORTED;
    const float *q = static_cast<const float *>(p.q), *k = static_cast<const float *>(p.k),
                *v = static_cast<const float *>(p.v), *o = static_cast<const float *>(p.out),
                *g_ = static_cast<const float *>(p.dout);
    if (qunits > 0)
        bwd_f32_dq_kernel<D><<<(unsigned)qunits, WARPS * 32, 0, st>>>(q, k, v, o, g_, p.lse,
                                                                      static_cast<float *>(p.dq), a);
    if (cudaGetLastError() != cudaSuccess) return CP_ECUDA;
    if (kunits > 0)
        bwd_f32_dkdv_kernel<D><<<(unsigned)kunits, WARPS * 32, 0, st>>>(
            q, k, v, o, g_, p.lse, static_cast<float *>(p.dk), static_cast<float *>(p.dv), a);
    return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ECUDA;
}

}  // namespace

int launch_bwd_f32(const BwdPtrs &p, const FwdArgs &f, cudaStream_t st)
{
    F32Args a;
    a.B = f.B;
    a.Hq = f.Hq;
    a.Hkv = f.Hkv;
    a.S = f.S;
    a.N = f.N;
    a.causal = f.causal;
    a.layout = f.layout;
    a.scale = (double)f.scale;
    const Geom g = make_geom(f.S, f.N, f.layout, f.causal);
    a.upc = (g.clen + QR - 1) / QR;
    a.tpc = (g.clen + KR - 1) / KR;
    if (f.D == 64) return launch_d<64>(p, a, st);
    if (f.D == 128) return launch_d<128>(p, a, st);
    return CP_EUNSUPPORTED;
}

}  // namespace cp
