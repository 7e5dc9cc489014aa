// kernels.h -- launchers shared between the C-ABI entry points (cp_api.cu)
// and the kernel translation units.  Internal to libcp.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace cp {

struct FwdArgs {
    int B, Hq, Hkv;
    int S;                // sequence length (<= INT32_MAX)
    int D, N, causal, layout;
    float scale;          // softmax scale
    int rank_lo, rank_hi; // virtual ranks whose queries are computed
    int upc;              // query units per chunk (set by the launcher)
    int head_grouped;     // units numbered with each (batch, head) contiguous (set by the launcher)
    int n_units;          // query units of the launch (set by the launcher)
    unsigned *err;        // device error word
    uint64_t limit_ns;    // bound of every pipeline wait
    uint64_t drain_ns;    // bound of the waits that drain copies and MMAs before exit
};

// Partial results of a split forward (fp32, normalised): n splits of every
// unit's key walk; out [n][B][S][Hq][D], lse [n][B][S][Hq].
struct SplitOut {
    int n;
    float *out;
    float *lse;
};

// State of a shard-local ring step (flash_block_step): the queries of rank
// a.rank_lo (a.rank_hi = a.rank_lo + 1) in that rank's local row order,
// against the KV block it holds at ring step step_k, merged into the running
// (out_acc, lse_acc).  C = S / N rows per shard.
struct StepOut {
    int step_k;        // source rank = (rank - step_k) mod N
    int accumulate;    // 0: the state is overwritten with this block's result
    float *out_acc;    // [B][C][Hq][D] fp32, normalised output so far
    float *lse_acc;    // [B][Hq][C] fp32, natural log
    void *out_final;   // [B][C][Hq][D] in the input dtype (merged result), or null
};

int launch_fwd_f32(const float *q, const float *k, const float *v, float *out, float *lse,
                   FwdArgs a, cudaStream_t st);
int launch_fwd_f32_step(const float *q, const float *k, const float *v, FwdArgs a,
                        const StepOut &so, cudaStream_t st);
int launch_fwd_bf16_step(const void *q, const void *k, const void *v, FwdArgs a,
                         const StepOut &so, cudaStream_t st);
int launch_fwd_bf16(const void *q, const void *k, const void *v, void *out, float *lse,
                    FwdArgs a, cudaStream_t st);
int launch_fwd_bf16_split(const void *q, const void *k, const void *v, FwdArgs a,
                          const SplitOut &so, cudaStream_t st);
// Merge the so.n partials of the rows of ranks [a.rank_lo, a.rank_hi) into
// out (bf16, [B][S][Hq][D]) and lse ([B][Hq][S]).
int launch_fwd_split_combine(const FwdArgs &a, const SplitOut &so, void *out, float *lse,
                             cudaStream_t st);
// Number of splits for a split forward of these sizes on num_sms SMs (host;
// 1 when splitting does not pay), at most max_split.
int fwd_split_choose(int B, int Hq, int S, int D, int N, int causal, int layout, int rank_lo,
                     int rank_hi, int num_sms, int max_split);
int launch_lse_merge_n(const float *out_parts, const float *lse_parts, int n, int64_t rows, int D,
                       float *out, float *lse, cudaStream_t st);
int launch_lse_merge(const float *out_a, const float *lse_a, const float *out_b,
                     const float *lse_b, float *out, float *lse, int64_t rows, int D,
                     cudaStream_t st);
int launch_ulysses(const void *src, void *dst, int B, int S, int H, int D, int N, int layout,
                   int elem_bytes, int to_head, cudaStream_t st);
int launch_debug_wait(unsigned *err, uint64_t limit_ns, cudaStream_t st);

struct BwdPtrs {
    const void *q, *k, *v, *out;
    const float *lse;
    const void *dout;
    void *dq, *dk, *dv;
    void *workspace;   // Delta, bwd_workspace_bytes() bytes
};
int launch_bwd_bf16(const BwdPtrs &p, const FwdArgs &a, cudaStream_t st);
// fp32 inputs/outputs, fp64 arithmetic; does not touch p.workspace
int launch_bwd_f32(const BwdPtrs &p, const FwdArgs &a, cudaStream_t st);
size_t bwd_workspace_bytes(int B, int Hq, int64_t S);

// Number of SMs of the current device (cached per device).
int sm_count();

// Device address of the current device's error word (set up once per device),
// the bound of the pipeline waits (2 s unless a test shortened it with
// cp_debug_set_wait_limit) and the bound of the drain waits (always 2 s).
unsigned *device_error_word();
uint64_t device_wait_limit_ns();
uint64_t device_drain_limit_ns();

// Test hook: largest grid of the forward kernel (0: no limit), so that tests
// can make every block run many work items.
int fwd_grid_limit();

}  // namespace cp
