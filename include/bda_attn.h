/*
 * bda_attn.h -- C ABI of libbda_attn.so: forward and backward block-causal and
 * staircase attention over packed variable-length bf16 Q/K/V with GQA, for
 * NVIDIA B300 (sm_103a).
 *
 * The operation (sources):
 *   - ORL announcement thread (24vids.com mirror), highlight 3: block attention
 *     for diffusion LMs, redesigned as a *block-causal* kernel.  A sequence is
 *     cut into blocks of `block_size` tokens; a query sees every key of its own
 *     block (bidirectionally) and every key of all earlier blocks.
 *   - Same thread, Insight 3, and ORL paper card (thelatestinai.com), Figure 3
 *     caption: training replays packed, load-balanced trajectories with a
 *     *staircase* kernel.  After a clean prefix of P tokens sit copies of the
 *     active block (each `block_size` tokens, one per denoising step); each copy
 *     sees the prefix and itself only; prefix rows are block-causal within the
 *     prefix.
 *   - Plain softmax attention otherwise (the thread measures it against
 *     FlashAttention): O = softmax(scale * Q K^T + mask) V, with the natural-log
 *     log-sum-exp of each row (LSE) kept for the backward pass.
 * Where the sources are silent the library reads them as follows:
 *   - a sequence with fewer queries than keys (a decode step) aligns its
 *     queries with the last keys: query i sits at key position i + Lk - Lq;
 *   - GQA: query head h uses KV head h / (hq / hkv);
 *   - LSE is natural-log, fp32.
 *
 * Layouts (row-major, "THD" packing, head_dim contiguous):
 *   q, o, dout, dq : bf16 [total_q][hq][head_dim]
 *   k, v, dk, dv   : bf16 [total_k][hkv][head_dim]
 *   lse            : fp32 [hq][total_q]
 *   sequence s owns query rows [cu_seqlens_q[s], cu_seqlens_q[s+1]) and key rows
 *   [cu_seqlens_k[s], cu_seqlens_k[s+1]).
 *
 * Conventions:
 *   - Every tensor pointer is a DEVICE pointer, 16-byte aligned; the caller
 *     owns all memory.  The library allocates no device memory: scratch lives
 *     in a caller-provided workspace of bda_attn_workspace_size() bytes.
 *   - cu_seqlens_* and prefix_len are HOST arrays, read during the call only.
 *   - All compute calls are asynchronous on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).  bda_attn_plan must precede fwd/bwd on the
 *     same stream with the same problem, mask and workspace.
 *   - Errors are status codes; nothing aborts.  Argument errors are found on
 *     the host before anything is launched.  A device-side wait that runs out
 *     of time (it never should) records BDA_ERR_DEVICE_TIMEOUT in the
 *     workspace; bda_attn_check_status() reads it.
 *   - Thread safety: stateless apart from the workspace; calls on distinct
 *     workspaces may run concurrently.
 *   - Supported: bf16; head_dim 64 or 128; hq % hkv == 0; block_size >= 1;
 *     staircase needs cu_seqlens_q == cu_seqlens_k and
 *     (len - prefix_len) % block_size == 0 with 0 <= prefix_len <= len.
 */
#ifndef BDA_ATTN_H
#define BDA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *bda_stream_t;

typedef enum {
  BDA_OK = 0,
  BDA_ERR_INVALID_ARG = 1,    /* bad pointer, size, layout or descriptor */
  BDA_ERR_UNSUPPORTED = 2,    /* valid but not implemented (e.g. head_dim 96) */
  BDA_ERR_WORKSPACE = 3,      /* workspace or host plan buffer too small */
  BDA_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed */
  BDA_ERR_DEVICE_TIMEOUT = 5  /* a kernel's bounded wait ran out (reported after the fact) */
} bda_status;

typedef enum {
  BDA_MASK_BLOCK_CAUSAL = 0,
  BDA_MASK_STAIRCASE = 1,
  /* Several active blocks per trajectory (the "irregular trajectories" the
   * announcement thread's Insight 3 replays with the staircase kernel):
   * after the clean prefix [0, P) -- block-causal in blocks of B -- come
   * groups of copies, one group per active block, in order; group g holds
   * group_copies[g] copies of B tokens, and each of its copies sees the
   * clean keys [0, group_visible[g]) (the prompt and the clean blocks before
   * its block) and itself only.  STAIRCASE is one group with visible = P.
   * The compute calls take the groups in block order: along a sequence, the
   * visible counts of its non-empty groups must not decrease (a layout out
   * of that order is counted by bda_attn_count_pairs but the other calls
   * return BDA_ERR_UNSUPPORTED for it). */
  BDA_MASK_STAIRCASE_MULTI = 2
} bda_mask_kind;

/* Mask descriptor.  The mask is never materialised: kernels evaluate it from
 * block indices (see the file comment for its definition). */
typedef struct {
  int32_t kind;                   /* bda_mask_kind */
  int32_t block_size;             /* B >= 1; staircase copies are B tokens long */
  const int32_t *prefix_len_host; /* staircase kinds: [nseq] prefix lengths (host); else NULL */
  /* STAIRCASE_MULTI only (else NULL): sequence s owns groups
   * [group_offsets_host[s], group_offsets_host[s+1]) of group_copies_host /
   * group_visible_host; sum of its copies * B == its length - P, and
   * 0 <= visible <= P. */
  const int32_t *group_offsets_host; /* [nseq+1], starts at 0, non-decreasing */
  const int32_t *group_copies_host;  /* copies per group, >= 0 */
  const int32_t *group_visible_host; /* clean keys each group's copies see */
} bda_mask_desc;

/* Problem shape.  softmax_scale <= 0 selects 1/sqrt(head_dim). */
typedef struct {
  int32_t nseq;
  int32_t hq;
  int32_t hkv;
  int32_t head_dim;
  float softmax_scale;
  const int32_t *cu_seqlens_q_host; /* [nseq+1], cu[0] == 0, non-decreasing */
  const int32_t *cu_seqlens_k_host; /* [nseq+1] */
} bda_problem;

/* Bytes of the host plan buffer bda_attn_plan fills (0 on invalid input). */
size_t bda_attn_plan_size(const bda_problem *prob, const bda_mask_desc *mask);

/* Bytes of device workspace for fwd (with_bwd = 0) or fwd+bwd (with_bwd = 1):
 * the plan, a status word, the split forward's partial results (problems
 * that fill few SMs), and for the backward D = rowsum(dO*O) fp32
 * [hq][total_q] plus an fp32 dQ accumulator [total_q][hq][head_dim].
 * 0 on invalid input. */
size_t bda_attn_workspace_size(const bda_problem *prob, const bda_mask_desc *mask, int with_bwd);

/* Tile planner (host).  Cuts every sequence into 128-row query tiles (query
 * tokens x the query heads of one KV group) and 128-key tiles, classifies each
 * (query tile, key tile) pair as FULL, PARTIAL or EMPTY from the block indices,
 * drops EMPTY pairs, and orders the work units longest-first so a grid of
 * CTAs balances unequal packed sequences ("packed compute-balanced training",
 * ORL announcement thread, Insight 3; "packed and load-balanced", ORL paper
 * card, Figure 3 caption).  Fills host_plan (caller-owned, plan_size bytes;
 * pinned memory keeps the copy asynchronous) and enqueues its copy into the
 * workspace on `stream`; host_plan must stay unchanged until that copy has
 * run.  Also clears the workspace status word. */
bda_status bda_attn_plan(const bda_problem *prob, const bda_mask_desc *mask, void *host_plan,
                         size_t host_plan_bytes, void *ws, size_t ws_bytes, bda_stream_t stream);

/* The host half of bda_attn_plan: fills host_plan and touches no device or
 * CUDA state (plans can be built ahead of time on any CPU thread; copying
 * the plan_size bytes to the start of the workspace is then the caller's
 * job).  BDA_ERR_WORKSPACE if host_plan_bytes < bda_attn_plan_size(). */
bda_status bda_attn_plan_host(const bda_problem *prob, const bda_mask_desc *mask, void *host_plan,
                              size_t host_plan_bytes);

/* Forward: o = softmax(scale * q k^T + mask) v and lse (natural log, fp32).
 * Rows of o/lse outside every sequence are not written.  A problem whose
 * query tiles fill few SMs (fewer than 74 tiles x head groups, e.g. a decode
 * step) runs the split forward: each query tile's key tiles are cut into
 * chunks, one CTA per chunk and head group, and a second kernel merges the
 * chunks' partial results (kept in the workspace); larger problems run the
 * persistent forward. */
bda_status bda_attn_fwd(const bda_problem *prob, const bda_mask_desc *mask, const void *q,
                        const void *k, const void *v, void *o, float *lse, void *ws,
                        size_t ws_bytes, bda_stream_t stream);

/* Forward with an FP8 KV cache (the decode engine of the ORL paper card runs
 * its NVFP4 configurations with an FP8 KV cache, Table 11 caption).  k8, v8:
 * e4m3 codes (OCP FP8 E4M3: bias 7, largest finite 448), one byte each,
 * layout [total_k][hkv][head_dim]; k_scale, v_scale: DEVICE fp32 [hkv]
 * dequantisation scales, K = k8 * k_scale[h], V = v8 * v_scale[h].  Computes
 * the attention of bda_attn_fwd over those K and V: the codes are expanded
 * exactly to bf16 in shared memory and the scales applied in fp32, so only
 * the KV bytes read from HBM change.  Same plan and workspace as
 * bda_attn_fwd (bda_attn_plan first); runs the split forward kernel for
 * every problem size. */
bda_status bda_attn_fwd_fp8kv(const bda_problem *prob, const bda_mask_desc *mask, const void *q,
                              const void *k8, const void *v8, const float *k_scale,
                              const float *v_scale, void *o, float *lse, void *ws, size_t ws_bytes,
                              bda_stream_t stream);

/* FP8 KV-cache quantisation (same source as bda_attn_fwd_fp8kv): x8 =
 * e4m3(x / scale[h]) for bf16 x [rows][heads][head_dim] (DEVICE), bytes out
 * in the same layout; the quotient is the IEEE fp32 division, rounded to
 * the nearest e4m3 value with ties to even and saturated to +-448 (NaN stays
 * NaN).  scale: DEVICE fp32 [heads].  head_dim 64 or 128; x and x8 16-byte
 * aligned. */
bda_status bda_kv_quantize_fp8(const void *x, void *x8, const float *scale, long long rows,
                               int heads, int head_dim, bda_stream_t stream);

/* Per-head dequantisation scales for bda_kv_quantize_fp8: scale[h] =
 * max |x[., h, .]| / 448 (1 for a head that is all zero), so the largest
 * value maps to the largest e4m3 code.  scale: DEVICE fp32 [heads],
 * heads <= 4096. */
bda_status bda_kv_fp8_scales(const void *x, float *scale, long long rows, int heads, int head_dim,
                             bda_stream_t stream);

/* Backward of sum(o * dout): dq, dk, dv (bf16, same layouts as q, k, v);
 * dk/dv sum over the query heads that share a KV head.  Needs o and lse from
 * bda_attn_fwd with the same inputs, and a workspace sized with with_bwd = 1.
 * Runs the three stages below in order. */
bda_status bda_attn_bwd(const bda_problem *prob, const bda_mask_desc *mask, const void *q,
                        const void *k, const void *v, const void *o, const float *lse,
                        const void *dout, void *dq, void *dk, void *dv, void *ws,
                        size_t ws_bytes, bda_stream_t stream);

/* Backward stage 1: D[h][t] = sum_c dout[t][h][c] * o[t][h][c] (fp32) into the
 * workspace, and zero the workspace's fp32 dQ accumulator. */
bda_status bda_attn_bwd_preprocess(const bda_problem *prob, const bda_mask_desc *mask,
                                   const void *o, const void *dout, void *ws, size_t ws_bytes,
                                   bda_stream_t stream);

/* Backward stage 2: per 128-key tile and KV head, recompute P^T and dP^T and
 * accumulate dk, dv (written as bf16) and the fp32 dQ accumulator. */
bda_status bda_attn_bwd_dkdv(const bda_problem *prob, const bda_mask_desc *mask, const void *q,
                             const void *k, const void *v, const float *lse, const void *dout,
                             void *dk, void *dv, void *ws, size_t ws_bytes, bda_stream_t stream);

/* Backward stage 3: dq = bf16(scale * dQ accumulator). */
bda_status bda_attn_bwd_dq_convert(const bda_problem *prob, const bda_mask_desc *mask, void *dq,
                                   void *ws, size_t ws_bytes, bda_stream_t stream);

/* Number of allowed (query, key) pairs per query head, summed over the
 * sequences (useful-work count; masked pairs excluded).  -1 on invalid input. */
long long bda_attn_count_pairs(const bda_problem *prob, const bda_mask_desc *mask);

/* Synchronises `stream`, reads the workspace status word, clears it, and
 * returns BDA_ERR_DEVICE_TIMEOUT if a kernel recorded a timeout, or
 * BDA_ERR_UNSUPPORTED if a kernel found its shared memory misaligned (the
 * kernels then return without computing; never expected on sm_103a). */
bda_status bda_attn_check_status(void *ws, size_t ws_bytes, bda_stream_t stream);

/* Forward without a workspace.  The paper has no counterpart: this entry
 * exists for callers that cannot allocate device memory where they run
 * attention -- e.g. a plugin inside an engine that owns all device memory
 * through its own pool, or a decode loop that must not risk the device-wide
 * synchronisation an allocation can cause.  Same arguments and results as
 * bda_attn_fwd, minus the workspace: the tile plan and the status word live
 * in a 1 MiB array compiled into the library (every GPU that loads the
 * library holds it until the process exits).  Each call builds the forward
 * plan on the host and writes it into the array through the parameters of a
 * small copy kernel on `stream` (no host-to-device memcpy: the call does not
 * wait for the stream's earlier work), then launches the forward.  Allocates
 * nothing (no cudaMalloc/cudaFree, no library allocator).
 *   - BDA_ERR_WORKSPACE if the forward plan needs more than the 1 MiB array
 *     (about 16 thousand query tiles of 128 rows); use bda_attn_fwd with a
 *     workspace then.
 *   - The first call on a device looks the array's device address up
 *     (cudaGetSymbolAddress, with that device current).
 *   - BDA_ERR_UNSUPPORTED if `stream` is being captured into a CUDA graph:
 *     a captured call would replay this call's plan over an array that
 *     later calls overwrite.
 *   - Every call overwrites the shared array; calls whose GPU work overlaps
 *     (other streams, other host threads) race on it and must be serialised
 *     by the caller. */
bda_status bda_attn_fwd_noalloc(const bda_problem *prob, const bda_mask_desc *mask, const void *q,
                                const void *k, const void *v, void *o, float *lse,
                                bda_stream_t stream);

/* Status of the most recent bda_attn_fwd_noalloc on the current device
 * (no counterpart on the pages; the same role as bda_attn_check_status for
 * the no-alloc array): synchronises `stream`, reads the array's status word,
 * clears it, and returns BDA_ERR_DEVICE_TIMEOUT or BDA_ERR_UNSUPPORTED as
 * bda_attn_check_status does.  Call it after the forward whose status is
 * wanted and before the next no-alloc call (which resets the word).
 * Allocates nothing; refuses a stream under capture. */
bda_status bda_attn_fwd_noalloc_check_status(bda_stream_t stream);

/* Failure-detection testing hook (no counterpart on the pages).  Arms a
 * one-shot fault for the next launch of `stage` in this process (1 = the
 * forward kernel, of bda_attn_fwd or bda_attn_fwd_noalloc; 2 = the backward
 * dK/dV kernel): CTA 0 of that launch leaves its first Q load un-issued,
 * waits timeout_ns (1 us .. 1 s) for it, records BDA_ERR_DEVICE_TIMEOUT in
 * the status word, lets its in-flight copies and MMAs land, frees its TMEM
 * and returns.  Nothing faults and no wait is unbounded; the outputs of that
 * launch are unspecified.  stage 0 disarms.  BDA_ERR_INVALID_ARG otherwise.
 * Never armed unless called. */
bda_status bda_testing_arm_wait_timeout(int stage, unsigned long long timeout_ns);

/* Testing hook (no counterpart on the pages): which forward kernel
 * bda_attn_fwd runs -- 0 as the plan says (default), 1 always the
 * persistent kernel, 2 always the split kernel.  Both compute the same
 * result; tests use this to check each on every problem shape.
 * BDA_ERR_INVALID_ARG for other values. */
bda_status bda_testing_force_forward_kernel(int which);

const char *bda_status_string(bda_status s);

/* Text of the CUDA error behind the most recent BDA_ERR_CUDA returned on the
 * calling thread ("" if none).  The string stays valid until the next call
 * on that thread. */
const char *bda_last_cuda_error(void);

#ifdef __cplusplus
}
#endif
#endif /* BDA_ATTN_H */
