// bwd_noalloc.cu -- ring_attn_bwd for callers that cannot allocate device
// memory.
//
// Who needs this: code that runs where cudaMalloc is not an option -- for
// example a plugin or extension that may only use the buffers its host
// framework hands it, a caller working inside a memory pool or allocator it
// does not own, or a process with a fixed memory budget decided up front.
// ring_attn_bwd asks such callers for a scratch buffer they have no way to
// obtain.  ring_attn_bwd_noalloc takes the same inputs and outputs but keeps
// its scratch (the per-row Delta = rowsum(dout * out), fp32) in a fixed
// array compiled into the library, so it allocates nothing.
//
// The array below is a static device variable: every GPU that loads the
// library holds it (16 MiB) until the process exits.  Host code cannot use
// the array's name as a device address -- on the host it names a host-side
// stand-in -- so the first call on each device looks up the real device
// address with cudaGetSymbolAddress (with that device current) and caches
// it.  That first call therefore does one runtime query; make it before any
// stream capture.  All calls on a device share the one array: two calls whose
// kernels overlap on the GPU (different streams, no ordering between them)
// race on it.  Nothing in the array needs to start at zero: the Delta kernel
// writes every entry it later reads, so stale contents from an earlier call
// are harmless.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "cp.h"
#include "kernels.h"

namespace cp {

namespace {

// Scratch for Delta: CP_BWD_NOALLOC_MAX_ROWS fp32 rows (B * Hq * S <= 4 Mi).
static __device__ __align__(256) float g_bwd_scratch[CP_BWD_NOALLOC_MAX_ROWS];

constexpr int MAX_DEV = 64;

// Device address of g_bwd_scratch on the current device, looked up once per
// device; nullptr if the lookup failed.
float *scratch_ptr()
{
    static float *ptrs[MAX_DEV] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEV) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!ptrs[dev]) {
        float *p = nullptr;
        if (cudaGetSymbolAddress((void **)&p, g_bwd_scratch) != cudaSuccess) return nullptr;
        ptrs[dev] = p;
    }
    return ptrs[dev];
}

bool al16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

int noalloc_impl(const void *q, const void *k, const void *v, const void *out, const float *lse,
                 const void *dout, void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int64_t S,
                 int D, int N, int causal, int layout, int dtype, float scale, void *stream)
{
    if (B < 0 || Hq < 1 || Hkv < 1 || N < 1 || S < 0 || S > 0x7fffffffLL) return CP_EINVAL;
    if (causal != 0 && causal != 1) return CP_EINVAL;
    if (layout != CP_LAYOUT_CONTIGUOUS && layout != CP_LAYOUT_ZIGZAG && layout != CP_LAYOUT_STRIPED)
        return CP_EINVAL;
    if (S % N || (layout == CP_LAYOUT_ZIGZAG && S % (2 * (int64_t)N))) return CP_EINVAL;
    if (Hq % Hkv) return CP_EINVAL;
    if (dtype != CP_BF16) return CP_EUNSUPPORTED;
    if (D != 64 && D != 128) return CP_EUNSUPPORTED;
    // the fixed scratch holds one fp32 Delta per (batch, query head, position)
    if ((int64_t)B * Hq * S > (int64_t)CP_BWD_NOALLOC_MAX_ROWS) return CP_EINVAL;
    if (B == 0 || S == 0) return CP_OK;
    if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv) return CP_EINVAL;
    if (!al16(q) || !al16(k) || !al16(v) || !al16(out) || !al16(dout) || !al16(dq) || !al16(dk) ||
        !al16(dv) || ((uintptr_t)lse & 3u))
        return CP_EINVAL;
    float *scratch = scratch_ptr();
    unsigned *err = device_error_word();
    if (!scratch || !err) return CP_ECUDA;
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
    a.err = err;
    a.limit_ns = device_wait_limit_ns();
    a.drain_ns = device_drain_limit_ns();
    BwdPtrs p{q, k, v, out, lse, dout, dq, dk, dv, scratch};
    return launch_bwd_bf16(p, a, static_cast<cudaStream_t>(stream));
}

}  // namespace

}  // namespace cp

using namespace cp;

extern "C" int ring_attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *out,
                                     const float *lse, const void *dout, void *dq, void *dk,
                                     void *dv, int B, int Hq, int Hkv, int64_t S, int D, int N,
                                     int causal, int layout, int dtype, float scale, void *stream)
{
    nvtxRangePushA("ring_attn_bwd_noalloc");
    const int rc = noalloc_impl(q, k, v, out, lse, dout, dq, dk, dv, B, Hq, Hkv, S, D, N, causal,
                                layout, dtype, scale, stream);
    nvtxRangePop();
    return rc;
}
