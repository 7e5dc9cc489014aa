/*
 * cp.h -- C ABI of libcp: exact ring / context-parallel attention on one
 * GB300 (sm_103a), with the N ranks of the ring emulated on the device.
 *
 * The operation is the ring attention of
 *   - "Sequence Parallelism in LLMs: Megatron-SP, Ulysses, RingAttention"
 *     (llms.blog), section "RingAttention and Blockwise Context Parallelism":
 *     "Algorithmic Mechanics" (partitioning, ring iteration, online softmax
 *     rescaling) and "Causal Masking and Load Balancing";
 *   - "Context Parallelism" (aiwiki), sections "Ring attention" and "The
 *     causal imbalance", and its ring sketch ring_attention(q, k, v, group)
 *     calling flash_block(q, k, v, out, m, lse, source);
 * which the pages state is exact: the result equals single-device attention
 * ("Sequence and Context Parallelism" (praveentn.live), "What it does not
 * change").
 *
 * Conventions shared by every call
 *   - Tensors are BSHD in GLOBAL token order: q and out [B][S][Hq][D],
 *     k and v [B][S][Hkv][D] (innermost D contiguous, no padding);
 *     lse is [B][Hq][S] fp32, natural log.
 *   - Query head h reads kv head h / (Hq / Hkv) (contiguous GQA groups).
 *   - causal: key j is visible to query i iff j <= i, in global positions.
 *   - layout: CP_LAYOUT_CONTIGUOUS splits S into N shards of S/N tokens;
 *     CP_LAYOUT_ZIGZAG splits S into 2N chunks and gives rank r chunks r and
 *     2N-1-r (local row order: chunk r first; S % 2N == 0);
 *     CP_LAYOUT_STRIPED gives token p to rank p mod N ("Sequence Parallelism
 *     in LLMs", "Causal Masking and Load Balancing", striped partitioning;
 *     local row t of rank r is position r + N t).  S % N == 0 for all three.
 *   - Ring schedule: rank r at step k = 0..N-1 uses the KV shard of rank
 *     (r - k) mod N; N compute steps (step 0 is the local block).
 *   - Device pointers are caller-owned device memory (the library keeps no
 *     reference after the call returns).  They must be 16-byte aligned.
 *   - stream is a cudaStream_t (NULL = legacy default stream).  Compute calls
 *     are asynchronous on it and return after the launch.
 *   - The library allocates no device memory (its only device state is a
 *     per-device error word and the fixed scratch of ring_attn_bwd_noalloc,
 *     both compiled in).  It reports device-side failures (a bounded wait that
 *     timed out, a misaligned shared-memory base, and in the debug-bounds
 *     build an out-of-range tile coordinate) through the error word, read by
 *     cp_get_error().
 *   - Return value: CP_OK or a negative CP_E* code; never an exception.
 */
#ifndef CP_H_
#define CP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define CP_OK 0
#define CP_EINVAL (-1)        /* null pointer, bad size, divisibility, misalignment */
#define CP_EHEADS (-2)        /* Ulysses: H not divisible by N (P <= H ceiling) */
#define CP_EUNSUPPORTED (-3)  /* dtype / head dim / shape combination not built */
#define CP_ECUDA (-4)         /* a CUDA runtime call or launch failed */
#define CP_ETIMEOUT (-5)      /* a device-side bounded wait ran out (cp_get_error) */
#define CP_ESMEM (-6)         /* a kernel's dynamic shared memory base was not 1 KB aligned
                                 (cp_get_error); the kernel returned without work */
#define CP_EBOUNDS (-7)       /* debug-bounds build only: an out-of-range tile coordinate was
                                 met and skipped (cp_get_error) */

/* sequence layouts */
#define CP_LAYOUT_CONTIGUOUS 0
#define CP_LAYOUT_ZIGZAG 1
#define CP_LAYOUT_STRIPED 2

/* element types of q, k, v, out (lse is always fp32) */
#define CP_F32 0
#define CP_BF16 1

/*
 * cp_shard_map -- global position of every local row of every rank.
 * "Algorithmic Mechanics", step 1 (contiguous: rank i holds block i of size
 * s/P) and "The causal imbalance" (zigzag: 2N chunks, rank i holds chunks i
 * and 2N-1-i).
 *   pos_host: HOST array of N*(S/N) int32, written as pos[r*(S/N) + t].
 * Errors: CP_EINVAL if pos_host is NULL, N < 1, S % N (contiguous),
 * S % (2N) (zigzag), S/N > INT32_MAX or an unknown layout.  Host only.
 */
int cp_shard_map(int64_t S, int N, int layout, int32_t *pos_host);

/*
 * cp_schedule_pairs -- walk the exact tile schedule that ring_attn_fwd
 * executes and count, per (rank r, ring step k), the masked-in
 * (query, key) pairs it covers and the (128-query x 256-key) tile pairs it
 * runs.
 * "Causal Masking and Load Balancing": under a causal mask contiguous
 * sharding is imbalanced; zigzag equalises the masked-in work per rank.
 *   pairs_host: HOST int64 [N*N], pairs[r*N + k];
 *   tiles_host: HOST int64 [N*N] executed tile pairs, or NULL.
 * Errors: CP_EINVAL as for cp_shard_map.  Host only.
 */
int cp_schedule_pairs(int64_t S, int N, int layout, int causal, int64_t *pairs_host,
                      int64_t *tiles_host);

/*
 * ring_attn_fwd -- exact attention as ring attention computes it, N virtual
 * ranks emulated in one launch.  Each rank's queries run N flash_block steps
 * against the KV shard held at that step ("Context Parallelism", ring
 * sketch: source = (rank - step) mod world), masked by global positions of
 * that source ("Causal Masking and Load Balancing"), with the running
 * (out, m, l) folded by online-softmax rescaling ("Algorithmic Mechanics").
 * Fully masked (128-query x 256-key) tile pairs are skipped, so executed
 * work tracks the masked-in work.
 *   q [B][S][Hq][D], k, v [B][S][Hkv][D]: device, dtype CP_F32 or CP_BF16.
 *   out [B][S][Hq][D]: same dtype (bf16 rounded to nearest even).
 *   lse [B][Hq][S]: fp32, lse_i = ln sum_j exp(scale * q_i.k_j).
 *   out and lse may be device memory or page-locked host memory that the
 *   device addresses directly (pinned, unified addressing): the kernels write
 *   them with ordinary stores, so the result lands in host memory without a
 *   separate copy.  q, k and v must be device memory.
 *   D in {64, 128}; Hq % Hkv == 0; scale <= 0 selects 1/sqrt(D).
 *   CP_BF16 runs tcgen05 tensor-core kernels (bf16 operands, fp32
 *   accumulation); CP_F32 runs the precision path: fp32 inputs and outputs,
 *   with scores, the running max and sum and the output accumulated in fp64
 *   on the CUDA cores.
 * Errors: CP_EINVAL (null pointer, misalignment, B/Hq/Hkv/S/N < 1, S % N,
 * S % 2N for zigzag, Hq % Hkv), CP_EUNSUPPORTED (D or dtype), CP_ECUDA.
 */
int ring_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                  int Hq, int Hkv, int64_t S, int D, int N, int causal, int layout, int dtype,
                  float scale, void *stream);

/*
 * ring_attn_fwd_rank -- the same computation restricted to the queries held
 * by virtual ranks [rank_lo, rank_hi): rows of other ranks in out and lse are
 * left untouched.  Used to time each rank's share of the ring (the causal
 * imbalance of "The causal imbalance").  Arguments and errors as
 * ring_attn_fwd, plus CP_EINVAL unless 0 <= rank_lo < rank_hi <= N.
 */
int ring_attn_fwd_rank(const void *q, const void *k, const void *v, void *out, float *lse,
                       int B, int Hq, int Hkv, int64_t S, int D, int N, int causal, int layout,
                       int dtype, float scale, int rank_lo, int rank_hi, void *stream);

/*
 * flash_block_step -- one step of a real ring, on shard-local buffers: the
 * flash_block(q, k, v, out, m, lse, source) call of the ring sketch in
 * "Context Parallelism" ("Ring attention"), i.e. step k of "Algorithmic
 * Mechanics" for one device.  The queries of `rank` attend to the KV block of
 * `source` (the block held at ring step k = (rank - source) mod N), under the
 * causal mask of the global positions of both shards ("Causal Masking and
 * Load Balancing"), and the block's result is folded into the running state
 * with the online-softmax rescaling written in log-sum-exp form:
 *   lse_new = ln(e^lse_acc + e^lse_blk),
 *   out_new = e^(lse_acc - lse_new) out_acc + e^(lse_blk - lse_new) out_blk.
 * A ring runs N such steps per device, source = (rank - k) mod N for
 * k = 0..N-1, while the KV block moves to rank + 1 (the caller's transfer).
 * C = S / N is the shard length; every buffer is in the rank's (or the
 * source's) local row order of cp_shard_map:
 *   q [B][C][Hq][D]: the queries of `rank`; k, v [B][C][Hkv][D]: the block
 *   of `source`; dtype CP_BF16 or CP_F32 (device).
 *   out_acc [B][C][Hq][D] fp32 and lse_acc [B][Hq][C] fp32 (natural log):
 *   the running normalised state, read and written (device).  accumulate = 0
 *   overwrites it with this block's result (the first step; rows that see no
 *   key of the block get out 0, lse -inf), accumulate = 1 merges into it.
 *   The empty state (out 0, lse -inf) is the merge identity.
 *   out_final: NULL, or [B][C][Hq][D] in the input dtype: the merged output
 *   rounded to it (bf16: nearest even), e.g. on the last step.  For CP_F32 it
 *   may alias out_acc.
 *   S, N, layout, causal: the global sequence and its sharding (as for
 *   ring_attn_fwd); rank, source in [0, N).  scale <= 0 selects 1/sqrt(D).
 * Rows of the state that see no key of the block are left unchanged
 * (accumulate = 1).  CP_BF16 runs the tcgen05 flash_block kernel (fp32
 * accumulation); CP_F32 the precision path (fp64 arithmetic).
 * Errors: as ring_attn_fwd, plus CP_EINVAL for rank, source or accumulate
 * out of range and a misaligned out_final.
 */
int flash_block_step(const void *q, const void *k, const void *v, float *out_acc, float *lse_acc,
                     void *out_final, int B, int Hq, int Hkv, int64_t S, int D, int N, int rank,
                     int source, int causal, int layout, int dtype, float scale, int accumulate,
                     void *stream);

/* Largest n_split ring_attn_fwd_split accepts. */
#define CP_MAX_SPLIT 64

/*
 * ring_attn_fwd_split -- ring_attn_fwd_rank with every query tile's key walk
 * (its N ring steps, in ring order) cut into n_split consecutive pieces, each
 * run by its own thread block, and the pieces merged by log-sum-exp
 * ("Algorithmic Mechanics", online softmax rescaling with lse = m + ln l:
 * lse = ln sum_i e^lse_i, out = sum_i e^(lse_i - lse) out_i).  The pieces
 * cover disjoint keys, so the result is the same attention, up to rounding.
 * It spreads long query rows over more SMs when a launch has few or uneven
 * query tiles (one rank's queries, few heads).
 *   q, k, v, out, lse, B..scale, rank_lo, rank_hi: as ring_attn_fwd_rank;
 *   dtype CP_BF16 only.
 *   n_split: 1..CP_MAX_SPLIT; 1 runs ring_attn_fwd_rank (workspace unused).
 *   workspace: device, at least ring_attn_fwd_split_workspace(B, Hq, S, D,
 *   n_split) bytes, 16-byte aligned, caller-owned scratch (the fp32 partials);
 *   its contents on entry do not matter.  Two launches on stream: the split
 *   kernel, then the merge.
 * Errors: as ring_attn_fwd_rank, plus CP_EINVAL (n_split out of range, null,
 * misaligned or too small workspace) and CP_EUNSUPPORTED for CP_F32.
 */
int ring_attn_fwd_split(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                        int Hq, int Hkv, int64_t S, int D, int N, int causal, int layout, int dtype,
                        float scale, int rank_lo, int rank_hi, int n_split, void *workspace,
                        size_t ws_bytes, void *stream);

/* ring_attn_fwd_split_workspace -- bytes ring_attn_fwd_split needs:
 * n_split B S Hq (D + 1) 4, rounded up to 256; 0 for bad sizes.  Host only. */
size_t ring_attn_fwd_split_workspace(int B, int Hq, int64_t S, int D, int n_split);

/*
 * cp_fwd_split_count -- a number of splits for ring_attn_fwd_split on a
 * device with num_sms SMs: the count (at most 32) that minimises the
 * estimated time of a simulated dispatch of the blocks (launch order, one
 * block per SM, cost = tiles walked + a fixed per-block overhead) plus the
 * merge's HBM traffic; 1 when splitting does not pay.  Host only.
 * Returns >= 1, or CP_EINVAL / CP_EUNSUPPORTED for arguments that
 * ring_attn_fwd_split would reject (B, Hq, S, N, layout, rank range, D,
 * num_sms < 1).
 */
int cp_fwd_split_count(int B, int Hq, int64_t S, int D, int N, int causal, int layout, int rank_lo,
                       int rank_hi, int num_sms);

/*
 * lse_merge -- merge two normalised partial attention results over disjoint
 * key sets ("Algorithmic Mechanics", online softmax rescaling, written with
 * lse = m + ln l):  lse = ln(e^lse_a + e^lse_b),
 * out = e^(lse_a - lse) out_a + e^(lse_b - lse) out_b.  An empty partial has
 * lse = -inf and drops out; both empty gives (0, -inf).
 *   out_a, out_b, out: device fp32 [rows][D]; lse_a, lse_b, lse: device fp32
 *   [rows].  out may alias out_a or out_b, lse may alias lse_a or lse_b.
 *   D % 4 == 0, rows >= 0 (rows == 0 is a no-op).
 * Errors: CP_EINVAL (null pointer, misalignment, D), CP_ECUDA.
 */
int lse_merge(const float *out_a, const float *lse_a, const float *out_b, const float *lse_b,
              float *out, float *lse, int64_t rows, int D, void *stream);

/*
 * lse_merge_n -- merge n normalised partial results over disjoint key sets in
 * one pass: the log-sum-exp combination of lse_merge ("Algorithmic
 * Mechanics") taken over all n at once,
 *   lse = ln sum_i e^lse_i,  out = sum_i e^(lse_i - lse) out_i,
 * e.g. the N per-step partials of one rank, or partials of a query row split
 * across blocks.  Partials with lse = -inf drop out; all empty gives (0, -inf).
 *   out_parts: device fp32 [n][rows][D]; lse_parts: device fp32 [n][rows];
 *   out [rows][D], lse [rows]: device fp32.  out may alias one partial of
 *   out_parts and lse one row set of lse_parts.
 *   n >= 1, D % 4 == 0, rows >= 0 (rows == 0 is a no-op); HBM traffic is
 *   (n + 1) (D + 1) 4 bytes per row.
 * Errors: CP_EINVAL (null pointer, misalignment, n, D, size overflow), CP_ECUDA.
 */
int lse_merge_n(const float *out_parts, const float *lse_parts, int n, int64_t rows, int D,
                float *out, float *lse, void *stream);

/*
 * ulysses_seq_to_head / ulysses_head_to_seq -- the two all-to-all relayouts
 * of DeepSpeed-Ulysses done as one local permutation over all N ranks'
 * buffers ("Sequence Parallelism in LLMs", "DeepSpeed Ulysses": [Batch, S/P,
 * H, D] -> [Batch, S, H/P, D] and back).
 *   x: rank-major stack of the N sequence shards, [N][B][S/N][H][D], rank r's
 *      rows in the order of the sequence layout (cp_shard_map);
 *   y: rank-major stack of the N head groups, [N][B][S][H/N][D]: rank g holds
 *      heads [g*H/N, (g+1)*H/N) over the full sequence in global order.
 *   elem_bytes in {1, 2, 4, 8}; pure byte copies (bit exact).
 * Errors: CP_EHEADS if H % N != 0 (the head-count ceiling P <= H of
 * "Communication Cost and Constraints"), CP_EINVAL (null pointer, S % N,
 * S % 2N for zigzag, sizes), CP_ECUDA.
 */
int ulysses_seq_to_head(const void *x, void *y, int B, int64_t S, int H, int D, int N,
                        int layout, int elem_bytes, void *stream);
int ulysses_head_to_seq(const void *y, void *x, int B, int64_t S, int H, int D, int N,
                        int layout, int elem_bytes, void *stream);

/*
 * usp_attn_fwd -- Unified Sequence Parallelism ("Sequence Parallelism in LLMs",
 * "Unified Sequence Parallelism (USP / 2D SP)"): a 2-D grid of n_ulysses x
 * n_ring virtual ranks.  The Ulysses dimension splits the heads with the
 * all-to-all of "DeepSpeed Ulysses"; the ring dimension circulates K/V blocks
 * as ring_attn_fwd does.  On one device, per batch: the seq->head relayout
 * (ulysses_seq_to_head over n_ulysses contiguous shards) gives every Ulysses
 * group u the whole sequence for heads [u H/n_ulysses, (u+1) H/n_ulysses);
 * ring attention runs in each group over n_ring virtual ranks with the given
 * layout; the head->seq relayout returns out to BSHD order.  The result is
 * attention over all keys, as for ring_attn_fwd.
 *   q, k, v, out, lse, causal, layout, dtype, scale: as ring_attn_fwd.
 *   n_ulysses >= 1 must divide Hq and Hkv (the Ulysses head ceiling
 *   P <= H_KV: CP_EHEADS otherwise) and S; n_ring >= 1 with the layout's
 *   divisibility of S.
 *   workspace: device, at least usp_attn_fwd_workspace(Hq, Hkv, S, D, dtype)
 *   bytes, 16-byte aligned, caller-owned scratch (the head-group copies of one
 *   batch); its contents on entry do not matter.
 * Errors: as ring_attn_fwd, plus CP_EHEADS, and CP_EINVAL for a null or too
 * small workspace.
 */
int usp_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse, int B, int Hq,
                 int Hkv, int64_t S, int D, int n_ulysses, int n_ring, int causal, int layout,
                 int dtype, float scale, void *workspace, size_t ws_bytes, void *stream);

/* usp_attn_fwd_workspace -- bytes of scratch usp_attn_fwd needs:
 * (2 Hq + 2 Hkv) S D element bytes, rounded up to 256; 0 for bad sizes.  Host only. */
size_t usp_attn_fwd_workspace(int Hq, int Hkv, int64_t S, int D, int dtype);

/*
 * ring_attn_bwd -- gradients of L = sum(dout * out) for the ring forward
 * above.  The pages state that context parallelism leaves the gradients equal
 * to single-device training ("Sequence and Context Parallelism", "What it
 * does not change") and give no backward algorithm; this is the textbook
 * attention gradient with the saved lse, walked over the same (rank, ring
 * step, tile) schedule as the forward:
 *   P = exp(scale q.k - lse), Delta = rowsum(dout * out), dS = P (dout.v - Delta),
 *   dq = scale dS k, dk = scale dS^T q, dv = P^T dout.
 *   q, out, dout, dq [B][S][Hq][D]; k, v, dk, dv [B][S][Hkv][D]: device,
 *   bf16 (dtype CP_BF16: tensor cores, fp32 accumulation) or fp32 (CP_F32:
 *   the precision path, fp64 arithmetic on the CUDA cores).
 *   lse [B][Hq][S] fp32: the forward's lse (natural log).
 *   workspace: device, at least ring_attn_bwd_workspace(B, Hq, S) bytes,
 *   16-byte aligned, caller-owned scratch (Delta, bf16 path; the fp32 path
 *   forms Delta in fp64 itself and leaves it untouched); its contents on
 *   entry do not matter and are overwritten.
 *   Every output element is written exactly once (no atomics): the result is
 *   deterministic.  D in {64, 128}.
 * Errors: CP_EINVAL (as ring_attn_fwd, plus a null or too small workspace),
 * CP_EUNSUPPORTED (dtype or D), CP_ECUDA.
 */
int ring_attn_bwd(const void *q, const void *k, const void *v, const void *out, const float *lse,
                  const void *dout, void *dq, void *dk, void *dv, int B, int Hq, int Hkv,
                  int64_t S, int D, int N, int causal, int layout, int dtype, float scale,
                  void *workspace, size_t ws_bytes, void *stream);

/* ring_attn_bwd_workspace -- bytes of scratch ring_attn_bwd needs
 * (B*Hq*S fp32, rounded up to 256 bytes); 0 for negative sizes.  Host only. */
size_t ring_attn_bwd_workspace(int B, int Hq, int64_t S);

/*
 * ring_attn_bwd_noalloc -- ring_attn_bwd for callers that cannot allocate
 * device memory.  The pages have no counterpart: this exists for code that
 * may only use buffers handed to it (a plugin inside another framework, a
 * caller bound to a memory pool or a fixed budget) and so has no way to
 * provide ring_attn_bwd's workspace.  Same arguments, layouts and results as
 * ring_attn_bwd with dtype CP_BF16 (the only dtype it takes), minus the
 * workspace: the scratch (one fp32 per
 * (batch, query head, position)) lives in a 16 MiB array compiled into the
 * library, which every GPU that loads the library keeps until the process
 * exits.  The call allocates nothing.
 *   Limit: B * Hq * S <= CP_BWD_NOALLOC_MAX_ROWS, else CP_EINVAL (nothing is
 *   launched).
 *   The first call on a device looks up the array's device address (one
 *   runtime query, with that device current); make it before any stream
 *   capture.  All calls on a device share the array: calls whose kernels
 *   overlap on the GPU race.  Nothing in it needs clearing between calls.
 * Errors: as ring_attn_bwd, plus CP_EINVAL for sizes beyond the limit.
 */
#define CP_BWD_NOALLOC_MAX_ROWS (4 * 1024 * 1024)
int ring_attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *out,
                          const float *lse, const void *dout, void *dq, void *dk, void *dv,
                          int B, int Hq, int Hkv, int64_t S, int D, int N, int causal, int layout,
                          int dtype, float scale, void *stream);

/*
 * cp_get_error -- synchronise `stream`, then read and clear the calling
 * device's error word.  Returns CP_OK, CP_ETIMEOUT (a kernel's bounded wait
 * ran out and the kernel returned early; its outputs are undefined),
 * CP_ESMEM (a kernel found its dynamic shared memory misaligned and returned
 * without work), CP_EBOUNDS (debug-bounds build only) or CP_ECUDA (the
 * synchronisation itself failed).  The first failure recorded since the last
 * read wins.
 */
int cp_get_error(void *stream);

/* cp_strerror -- static description of a status code. */
const char *cp_strerror(int code);

/*
 * cp_debug_wait_timeout -- test hook for the failure path: launches one
 * block that waits on a shared-memory barrier nobody arrives at, with a
 * wait limit of limit_ns nanoseconds (clamped to [1e3, 5e9]).  The wait runs
 * out, the kernel records CP_ETIMEOUT in the error word and returns; the
 * context stays usable.  Errors: CP_ECUDA.
 */
int cp_debug_wait_timeout(uint64_t limit_ns, void *stream);

/*
 * cp_debug_set_wait_limit -- test hook for the failure path of the pipelined
 * tensor-core kernels (forward in every mode, the two backward kernels): the
 * bound, in nanoseconds, of their pipeline waits for every launch made
 * afterwards in this process; 0 restores the default (2 s).  The waits that
 * drain a block's copies and MMAs before it exits keep the 2 s bound.  With
 * a bound of a few nanoseconds the first wait that is not already satisfied
 * runs out: the block records CP_ETIMEOUT, drains, frees its tensor memory
 * and exits, and the context stays usable.  Process-wide; not for use while
 * other threads launch work.  Errors: CP_EINVAL above 2e9.  Host only.
 */
int cp_debug_set_wait_limit(uint64_t limit_ns);

/*
 * cp_debug_set_grid_limit -- test hook: the tensor-core forward (ring, split
 * and step modes) launches min(work items, max_blocks) thread blocks from now
 * on in this process, each running its share of the items in turn (0 restores
 * the default grid: one block per item, or, for ring and step launches with
 * at most 16 items per SM, one block per SM).  Results do not depend on the grid: every item is
 * computed the same way whichever block runs it.  Process-wide; not for use
 * while other threads launch work.  Errors: CP_EINVAL for max_blocks < 0.
 * Host only.
 */
int cp_debug_set_grid_limit(int max_blocks);

#ifdef __cplusplus
}
#endif

#endif /* CP_H_ */
