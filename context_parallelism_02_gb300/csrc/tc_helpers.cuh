// tc_helpers.cuh -- inline-PTX building blocks of the sm_103a tensor-core
// kernels: shared-memory matrix descriptors, tcgen05 MMA / commit / fences,
// TMA tile loads with L2 cache hints, 32-byte global loads and stores (and the
// warp-regrouped row loads / stores built on them), MUFU ex2 / lg2, packed fp32
// arithmetic, bf16 packing, and the host-side tensor-map encoder for BSHD bf16
// tensors.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace cp {
namespace tc {

// --- descriptors --------------------------------------------------------------

// Shared-memory matrix descriptor, 128-byte swizzle (layout code 2),
// descriptor version 1 (bits 46-47) as sm_100-class tensor cores require.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulate, bf16 A and B,
// A and B K-major or MN-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major, bool a_mn_major = false)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                       uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// SS / TS MMAs whose descriptors are a base descriptor plus a compile-time
// offset (16-byte units), added inside the asm so that an unrolled issue
// sequence keeps only the base descriptors in registers.
template <uint32_t OFFA, uint32_t OFFB>
__device__ __forceinline__ void mma_ss_off(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                           uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
        "add.s64 da, %1, %5;\n\tadd.s64 db, %2, %6;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc), "n"(OFFA), "n"(OFFB)
        : "memory");
}

template <uint32_t OFFB>
__device__ __forceinline__ void mma_ts_off(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                           uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
        "add.s64 db, %2, %5;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc), "n"(OFFB)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// One lane of a converged warp (elect.sync: the lowest active lane).  A warp
// that runs its control flow converged keeps its MMA operands (descriptors,
// tensor-memory addresses, loop counters) warp-uniform, and only the elected
// lane issues.
__device__ __forceinline__ bool elect_one()
{
    uint32_t pred;
    asm volatile(
        "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// One 32-byte global store (eight 32-bit words); the address must be 32-byte
// aligned.  A lane writes a whole sector, half the store instructions of
// 16-byte stores.
__device__ __forceinline__ void st_global_v8(void *p, const uint32_t (&v)[8])
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]), "r"(v[1]),
                 "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

// Writes one piece of NW 32-bit words (64 or 128 bytes: bf16 pairs or fp32) per lane,
// lane t's piece in its own row (rows anywhere in memory, pieces 32-byte
// aligned), so that every store instruction covers whole pieces.  A lane storing
// its own piece would make each instruction touch 32 lines; here lanes in groups
// of G = NW/8 swap 32-byte chunks over shuffles, and lane j of a group then
// stores chunk j of each of the group's G pieces, one piece per instruction.
// Every lane of the warp calls it; pieces with ok == false are not written.
template <int NW>
__device__ __forceinline__ void store_warp_rows(void *piece, bool ok, const uint32_t (&pk)[NW], int lane)
{
    constexpr int G = NW / 8;
    static_assert(G == 2 || G == 4, "pieces of 64 or 128 bytes");
    const int j = lane & (G - 1), gb = lane & ~(G - 1);
    // rv[k]: chunk j of the piece of lane gb + (j ^ k); in exchange k this lane
    // sends its chunk j ^ k, the one that lane wants
    uint32_t rv[G][8];
#pragma unroll
    for (int k = 0; k < G; ++k) {
        const int c = j ^ k;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            uint32_t v = pk[e];
#pragma unroll
            for (int cc = 1; cc < G; ++cc) v = c == cc ? pk[8 * cc + e] : v;
            rv[k][e] = k == 0 ? v : __shfl_xor_sync(0xffffffffu, v, k);
        }
    }
#pragma unroll
    for (int m = 0; m < G; ++m) {   // instruction m: the piece of lane gb + m
        const int k = j ^ m;
        uint32_t d[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            uint32_t v = rv[0][e];
#pragma unroll
            for (int kk = 1; kk < G; ++kk) v = k == kk ? rv[kk][e] : v;
            d[e] = v;
        }
        const int src = gb + m;
        const bool rok = __shfl_sync(0xffffffffu, ok ? 1 : 0, src) != 0;
        uint8_t *rp = reinterpret_cast<uint8_t *>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(piece), src));
        if (rok) st_global_v8(rp + 32 * j, d);
    }
}

// Eight 32-bit words from global memory in one 32-byte access (32-byte aligned).
__device__ __forceinline__ void ld_global_v8u(const void *p, uint32_t (&v)[8])
{
    asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "l"(p)
                 : "memory");
}

// The load counterpart of store_warp_rows: lane t receives the NW words of its
// own piece, and every load instruction of the warp covers whole pieces.  Lane j
// of a group of G = NW/8 lanes loads chunk j of each of the group's G pieces,
// one piece per instruction; the chunks then go to their pieces' lanes over
// shuffles.  Every lane of the warp calls it; pieces with ok == false are not
// read (their words come back 0).
template <int NW>
__device__ __forceinline__ void load_warp_rows(const void *piece, bool ok, uint32_t (&pk)[NW], int lane)
{
    constexpr int G = NW / 8;
    static_assert(G == 2 || G == 4, "pieces of 64 or 128 bytes");
    const int j = lane & (G - 1), gb = lane & ~(G - 1);
    uint32_t ld[G][8];   // ld[m]: chunk j of the piece of lane gb + m
#pragma unroll
    for (int m = 0; m < G; ++m) {
        const int src = gb + m;
        const bool rok = __shfl_sync(0xffffffffu, ok ? 1 : 0, src) != 0;
        const uint8_t *rp = reinterpret_cast<const uint8_t *>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(piece), src));
        if (rok) {
            ld_global_v8u(rp + 32 * j, ld[m]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) ld[m][e] = 0u;
        }
    }
#pragma unroll
    for (int e = 0; e < NW; ++e) pk[e] = 0u;
    // exchange k: this lane sends chunk j of the piece of lane gb + (j ^ k), which
    // that lane wants, and receives chunk j ^ k of its own piece
#pragma unroll
    for (int k = 0; k < G; ++k) {
        const int c = j ^ k;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            uint32_t v = ld[0][e];
#pragma unroll
            for (int mm = 1; mm < G; ++mm) v = c == mm ? ld[mm][e] : v;
            const uint32_t r = k == 0 ? v : __shfl_xor_sync(0xffffffffu, v, k);
#pragma unroll
            for (int cc = 0; cc < G; ++cc) pk[8 * cc + e] = c == cc ? r : pk[8 * cc + e];
        }
    }
}

// Eight fp32 values from / to global memory in one 32-byte access (32-byte
// aligned addresses only).
__device__ __forceinline__ void ld_global_v8f(const float *p, float *r)
{
    asm volatile("ld.global.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]), "=f"(r[7])
                 : "l"(p));
}
__device__ __forceinline__ void st_global_v8f(float *p, const float *r)
{
    asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(r[0]), "f"(r[1]),
                 "f"(r[2]), "f"(r[3]), "f"(r[4]), "f"(r[5]), "f"(r[6]), "f"(r[7])
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tma_load4(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                          int c0, int c1, int c2, int c3, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
        "l"((uint64_t)map), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load5(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                          int c0, int c1, int c2, int c3, int c4, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(dst),
        "l"((uint64_t)map), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// (d0, d1) = (a0*b + c, a1*b + c) on the paired fp32 pipe
__device__ __forceinline__ void ffma2(float &d0, float &d1, float a0, float a1, float b, float c)
{
    uint64_t A, B, C, R;
    asm("mov.b64 %0, {%1, %2};" : "=l"(A) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(B) : "f"(b), "f"(b));
    asm("mov.b64 %0, {%1, %2};" : "=l"(C) : "f"(c), "f"(c));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(R) : "l"(A), "l"(B), "l"(C));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(R));
}

// (s0, s1) += (a0, a1) on the paired fp32 pipe
__device__ __forceinline__ void fadd2(float &s0, float &s1, float a0, float a1)
{
    uint64_t S, A, R;
    asm("mov.b64 %0, {%1, %2};" : "=l"(S) : "f"(s0), "f"(s1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(A) : "f"(a0), "f"(a1));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(R) : "l"(S), "l"(A));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(s0), "=f"(s1) : "l"(R));
}

// (d0, d1) = (a0*b0 + c0, a1*b1 + c1) on the paired fp32 pipe
__device__ __forceinline__ void ffma2v(float &d0, float &d1, float a0, float a1, float b0, float b1,
                                       float c0, float c1)
{
    uint64_t A, B, C, R;
    asm("mov.b64 %0, {%1, %2};" : "=l"(A) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(B) : "f"(b0), "f"(b1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(C) : "f"(c0), "f"(c1));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(R) : "l"(A), "l"(B), "l"(C));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(R));
}

// (d0, d1) = (a0 + b0, a1 + b1) on the paired fp32 pipe
__device__ __forceinline__ void fadd2v(float &d0, float &d1, float a0, float a1, float b0, float b1)
{
    uint64_t A, B, R;
    asm("mov.b64 %0, {%1, %2};" : "=l"(A) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(B) : "f"(b0), "f"(b1));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(R) : "l"(A), "l"(B));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(R));
}

// (d0, d1) = (a0 * b0, a1 * b1) on the paired fp32 pipe
__device__ __forceinline__ void fmul2v(float &d0, float &d1, float a0, float a1, float b0, float b1)
{
    uint64_t A, B, R;
    asm("mov.b64 %0, {%1, %2};" : "=l"(A) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(B) : "f"(b0), "f"(b1));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(R) : "l"(A), "l"(B));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(R));
}

// two floats -> bf16x2 (round to nearest even), `lo` in the low half
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// --- host side ---------------------------------------------------------------

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                              const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                              const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeFn get_encode()
{
    static EncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(p);
    });
    return fn;
}

// [B][S][H][D] bf16 viewed as [B][S/R][R][H][D]; box = 64 columns x box_rows
// rows of one (b, r, h), 128B swizzle.  R = N reads one rank of the striped
// layout (consecutive rows N positions apart); R = 1 is the plain layout.
// Coordinates (innermost first): column, head, r, row, batch.
inline bool make_map(CUtensorMap *m, const void *ptr, int B, int64_t S, int H, int D,
                     int box_rows = 128, int R = 1)
{
    EncodeFn enc = get_encode();
    if (!enc || R < 1 || S % R) return false;
    cuuint64_t dims[5] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)R, (cuuint64_t)(S / R),
                          (cuuint64_t)B};
    cuuint64_t strides[4] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)R * H * D * 2,
                             (cuuint64_t)S * H * D * 2};
    cuuint32_t box[5] = {64, 1, 1, (cuuint32_t)box_rows, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(ptr), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc
}  // namespace cp
