/*
 * thd_attn.h -- C ABI of libthdattn.so: causal softmax attention over packed
 * variable-length THD tensors, decomposed the way P2P (ring) context
 * parallelism decomposes it, with every CP rank emulated on one GPU.
 *
 * Sources (web pages), cited by page and section:
 *   [P1] TransformerEngine issue #2208, "thd format is not supported with
 *        hierarchical CP implementation yet" (traceback through
 *        AttnFuncWithCPAndKVP2P; maintainer reply on P2P vs A2A).
 *   [P2] TransformerEngine issue #3487, "THD P2P context-parallel regression
 *        when padded cu_seqlens are value-equal but not object-identical"
 *        ("Describe the bug", "Steps/Code to reproduce bug",
 *        "Expected behavior").
 *   [P3] "Hybrid / Hierarchical Context Parallel Skill" ("Contraintes
 *        requises": seq_length % (2 * context_parallel_size) == 0;
 *        "Pitfalls" item 5).
 *
 * Conventions for every entry point
 *   - THD layout: tensor [T, H, D] is row-major and contiguous, token-major:
 *     element (t, h, d) at ((t * H) + h) * D + d.  bf16 tensors are passed
 *     as `void*` to 2-byte IEEE bfloat16 storage.
 *   - cu_seqlens (int32, B+1 entries, cu[0] == 0) are exclusive prefix sums of
 *     the VALID lengths L_b.  cu_seqlens_padded (int32, B+1, may be NULL) are
 *     the buffer offsets: sequence b's valid tokens sit at rows
 *     [pad[b], pad[b] + L_b) and rows [pad[b] + L_b, pad[b+1]) are pad.
 *     NULL means no padding (pad = cu).
 *   - Each padded length P_b must be divisible by 2 * cp_size [P3
 *     "Contraintes requises"]; chunk length cb = P_b / (2 cp_size); emulated
 *     rank r owns chunks r and 2 cp_size - 1 - r.
 *   - All pointers are DEVICE pointers owned by the caller; the library never
 *     allocates device memory and never synchronises the host.  All work is
 *     enqueued on `stream` (a cudaStream_t; NULL = legacy default stream).
 *   - Return value: a host-side status (THD_OK or THD_ERR_*) for argument
 *     errors found without reading device memory, and launch failures.
 *   - Metadata errors can only be seen on the device (cu_seqlens live in
 *     device memory).  The first kernel of each call writes `*dev_status`
 *     (int32, device): 0 when the metadata is valid, else a THD_DEV_*
 *     code; every later kernel of the call reads it and returns without
 *     touching the outputs when it is nonzero.  Read it after the stream has
 *     synchronised.  Kernels that give up a bounded wait write
 *     THD_ERR_TIMEOUT there.
 *   - Workspace: caller-provided device memory of at least
 *     thd_workspace_size(...) bytes, 256-byte aligned; its contents need not be
 *     initialised and are not meaningful after the call.
 *   - Nothing is captured across calls except read-only state (driver entry
 *     points, per-device attributes); calls are safe to capture in a CUDA
 *     graph as long as the pointers stay valid.
 */
#ifndef THD_ATTN_H
#define THD_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* thd_stream_t; /* identical to cudaStream_t */

#if defined(__GNUC__)
#define THD_API __attribute__((visibility("default")))
#else
#define THD_API
#endif

/* host-side status codes */
#define THD_OK 0
#define THD_ERR_INVALID_ARG 1 /* null pointer, bad size, misaligned pointer */
#define THD_ERR_UNSUPPORTED 2 /* head_dim not 64/128, unsupported mode */
#define THD_ERR_CUDA 3        /* a CUDA call or launch failed */
#define THD_ERR_TIMEOUT 4     /* (device) a bounded wait gave up */
#define THD_ERR_WORKSPACE 5   /* workspace too small or misaligned */

/* device-side status codes written to *dev_status */
#define THD_DEV_ERR_NONZERO_START 101  /* cu_seqlens[0] or padded[0] != 0 */
#define THD_DEV_ERR_NOT_MONOTONE 102   /* negative length */
#define THD_DEV_ERR_VALID_GT_PAD 103   /* L_b > P_b */
#define THD_DEV_ERR_NOT_DIVISIBLE 104  /* P_b % (2 cp_size) != 0 */
#define THD_DEV_ERR_EXCEEDS_BUF 105    /* pad[B] larger than the buffer rows */
#define THD_DEV_ERR_CAUSAL_LENGTHS 106 /* top-left causal with q and kv lengths differing */
#define THD_DEV_ERR_CAPACITY 107       /* internal schedule capacity exceeded */

/* Kernel identifiers for the profiling hook. */
#define THD_KERNEL_PLAN 1
#define THD_KERNEL_FWD 2
#define THD_KERNEL_BWD_PREP 3
#define THD_KERNEL_BWD 4
#define THD_KERNEL_BWD_DQ 5
#define THD_KERNEL_LSE_MERGE 6
#define THD_KERNEL_TAIL_ZERO 7
#define THD_KERNEL_PARTITION 8
#define THD_KERNEL_A2A 9

/* mask modes (the `causal` argument of the attention entry points) */
#define THD_CAUSAL_NONE 0
#define THD_CAUSAL_TOP_LEFT 1
#define THD_CAUSAL_BOTTOM_RIGHT 2

/* thd_cp_a2a directions */
#define THD_A2A_TO_GROUPS 0 /* shards -> per-member head groups (the all-to-all in front of attention) */
#define THD_A2A_TO_SHARDS 1 /* per-member head groups -> shards (the all-to-all behind it) */

/* Human-readable text for any status above (host or device). Never NULL. */
THD_API const char* thd_status_string(int status);

/* Library ABI version (major * 100 + minor). */
THD_API int thd_version(void);

/*
 * Bytes of workspace thd_attn_fwd (for_bwd = 0) or thd_attn_bwd (for_bwd = 1)
 * needs for these sizes.  T_q / T_kv are the buffer rows of q and k/v.
 * Returns 0 for invalid sizes.
 */
THD_API size_t thd_workspace_size(int B, int64_t T_q, int64_t T_kv, int Hq, int Hkv, int D, int cp_size, int for_bwd);

/*
 * thd_cp_partition -- per-rank cu_seqlens for THD + P2P context parallelism,
 * for every emulated rank in ONE launch.
 *
 * [P2 "Describe the bug"] names the helper get_cu_seqlens_on_cp_rank, which
 * the padded path calls once per ring step; [P3 "Contraintes requises"]
 * fixes the 2*cp_size split.  For rank r and sequence b, with
 * cb = P_b / (2 cp_size):
 *     v1 = clamp(L_b - r cb, 0, cb)                (valid rows of chunk r)
 *     v2 = clamp(L_b - (2 cp_size - 1 - r) cb, 0, cb)
 *     cu_rank[r][b+1]        = cu_rank[r][b] + v1 + v2
 *     cu_rank_padded[r][b]   = pad[b] / cp_size
 *     cu_rank_half[r][0][b+1] = cu_rank_half[r][0][b] + v1
 *     cu_rank_half[r][1][b+1] = cu_rank_half[r][1][b] + v2
 *     token_map[r * (T / cp_size) + p] = global padded row of rank-local row p
 *       (rank-local rows of sequence b: chunk r then chunk 2cp-1-r), T = pad[B].
 * Arguments:
 *   cu_seqlens [B+1], cu_seqlens_padded [B+1] or NULL: device int32.
 *   pad_between_seqs: -1 decide from VALUES (padded iff some entry differs,
 *     never by pointer identity [P2 "Expected behavior"]), 0 ignore the
 *     padded array, 1 use it.
 *   cu_rank, cu_rank_padded: [cp_size][B+1] int32; cu_rank_half
 *     [cp_size][2][B+1] int32; token_map [token_map_capacity] int32.  Any
 *     output may be NULL (not written).  token_map needs capacity >= pad[B]
 *     (else THD_DEV_ERR_EXCEEDS_BUF).
 *   dev_status: device int32, always written.
 * Bit-exact (integer).
 */
THD_API int thd_cp_partition(const int32_t* cu_seqlens, const int32_t* cu_seqlens_padded, int B, int cp_size,
                     int pad_between_seqs, int32_t* cu_rank, int32_t* cu_rank_padded, int32_t* cu_rank_half,
                     int32_t* token_map, int64_t token_map_capacity, int32_t* dev_status, thd_stream_t stream);

/*
 * thd_attn_fwd -- O = softmax(scale q k^T + mask) v per sequence and head,
 * and lse = logsumexp of the masked scaled scores (natural log).
 *
 * Decomposition [P1 traceback: AttnFuncWithCPAndKVP2P; P3 "Contraintes
 * requises"]: work is split per emulated rank r (local query rows = chunk r
 * then chunk 2cp-1-r of each sequence) and ring step i, where rank r
 * holds the KV of rank s = (r - i) mod cp_size; per-step partials are merged
 * on chip by online-softmax (log-sum-exp) correction.  The merged result
 * equals plain attention.  Query and key sequences are chunked separately
 * (P_q / 2cp and P_kv / 2cp rows).
 *
 * Masks (`causal`; the pages train causal self-attention, the top-left mask
 * with equal lengths; the other two are the plainest completions):
 *   THD_CAUSAL_NONE (0): every valid key.
 *   THD_CAUSAL_TOP_LEFT (1): query i sees key j iff j <= i; needs equal q
 *     and kv valid and padded lengths per sequence (else the device status
 *     THD_DEV_ERR_CAUSAL_LENGTHS).
 *   THD_CAUSAL_BOTTOM_RIGHT (2): j <= i + L_kv - L_q, the last query aligned
 *     with the last key (a query block at the end of its keys); equal to
 *     top-left when the lengths agree.  With L_q > L_kv the first L_q - L_kv
 *     queries see no key: o = 0, lse = -inf (and zero gradients).
 *
 *   q   [T_q, Hq, D] bf16;  k, v [T_kv, Hkv, D] bf16 (Hq % Hkv == 0; query
 *       head h reads kv head h / (Hq/Hkv)).  16-byte aligned.
 *   o   [T_q, Hq, D] bf16 output; lse [Hq, T_q] fp32 output.  Rows that hold
 *       no valid token (pad rows and rows [pad_q[B], T_q)) get o = 0 and
 *       lse = -inf.
 *   D: 64 or 128.  causal: 0, 1 or 2 as above.  softmax_scale > 0.
 *   cp_size >= 1: the emulated CP degree.  pad_between_seqs as in
 *   thd_cp_partition (decided per side from values when -1).
 *   Pad rows inside tiles are read: they must hold finite values.
 */
THD_API int thd_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu_seqlens_q,
                 const int32_t* cu_seqlens_kv, const int32_t* cu_seqlens_q_padded,
                 const int32_t* cu_seqlens_kv_padded, int B, int64_t T_q, int64_t T_kv, int Hq, int Hkv, int D,
                 int causal, float softmax_scale, int cp_size, int pad_between_seqs, void* workspace,
                 size_t workspace_bytes, int32_t* dev_status, thd_stream_t stream);

/*
 * thd_attn_fwd_step -- the partial of ONE ring step, materialised: for every
 * emulated rank r, the attention of its local queries against the KV it
 * holds at step `step` (rank s = (r - step) mod cp_size), written in fp32 at
 * the queries' global rows:
 *   o_part [T_q, Hq, D] fp32, lse_part [Hq, T_q] fp32 (natural log).
 * Rows that get no contribution at this step get o = 0, lse = -inf.  Merging
 * the cp_size step partials with thd_lse_merge gives thd_attn_fwd's result
 * (the ring with communication replaced by reads of rank s's rows).
 * Other arguments as thd_attn_fwd.
 */
THD_API int thd_attn_fwd_step(const void* q, const void* k, const void* v, float* o_part, float* lse_part,
                      const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, const int32_t* cu_seqlens_q_padded,
                      const int32_t* cu_seqlens_kv_padded, int B, int64_t T_q, int64_t T_kv, int Hq, int Hkv,
                      int D, int causal, float softmax_scale, int cp_size, int pad_between_seqs, int step,
                      void* workspace, size_t workspace_bytes, int32_t* dev_status, thd_stream_t stream);

/*
 * thd_attn_fwd_step_bf16 -- thd_attn_fwd_step with the step's partial output
 * in bf16, the precision the ring keeps its per-step outputs in when they are
 * materialised [P1 traceback: AttnFuncWithCPAndKVP2P.forward, per-step
 * outputs corrected into the running output]:
 *   o_part [T_q, Hq, D] bf16 (16-byte aligned), lse_part [Hq, T_q] fp32.
 * Same rows, masks and -inf/0 conventions as thd_attn_fwd_step; merge the
 * steps with thd_lse_merge_bf16 into an fp32 accumulator.
 */
THD_API int thd_attn_fwd_step_bf16(const void* q, const void* k, const void* v, void* o_part, float* lse_part,
                                   const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                                   const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded, int B,
                                   int64_t T_q, int64_t T_kv, int Hq, int Hkv, int D, int causal,
                                   float softmax_scale, int cp_size, int pad_between_seqs, int step,
                                   void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                   thd_stream_t stream);

/*
 * thd_attn_fwd_noalloc -- thd_attn_fwd for callers that cannot allocate device
 * memory where they call the library.  The pages have no counterpart to
 * this entry point; it exists for deployment.  Examples of such callers: a
 * plug-in that only receives input and output pointers from a host framework
 * whose own pool allocator owns the device memory; a serving loop with a
 * fixed, pre-planned memory budget; code that must not call cudaMalloc,
 * which can synchronise the device and is not allowed inside stream capture.
 *
 * Same arguments and results as thd_attn_fwd, minus the workspace: the
 * scratch lives in a static device array of THD_NOALLOC_SCRATCH_BYTES (1 MiB)
 * inside the library, which every GPU that loads the library keeps until the
 * process exits.  The entry point calls no cudaMalloc/cudaFree and no
 * allocating library routine.
 *   - Limit: returns THD_ERR_WORKSPACE, launching nothing, when
 *     thd_workspace_size(B, T_q, T_kv, Hq, Hkv, D, cp_size, 0) exceeds
 *     THD_NOALLOC_SCRATCH_BYTES (about T_q / 128 + cp_size * B < 65000 schedule
 *     entries, e.g. up to ~8M tokens for a few sequences).
 *   - Set-up: the first call on each device looks up the array's device
 *     address (cudaGetSymbolAddress) with that device current; make that first
 *     call before any stream capture.
 *   - Sharing: every call on a device uses the same array, which keeps the
 *     last call's contents (nothing in it needs clearing; each call rewrites
 *     what it reads).  Calls whose kernels overlap on the GPU (different
 *     streams, or host threads without ordering) race on it: serialise them.
 */
#define THD_NOALLOC_SCRATCH_BYTES (1 << 20)
THD_API int thd_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                 const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                                 const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded, int B,
                                 int64_t T_q, int64_t T_kv, int Hq, int Hkv, int D, int causal, float softmax_scale,
                                 int cp_size, int pad_between_seqs, int32_t* dev_status, thd_stream_t stream);

/*
 * thd_attn_bwd -- gradients of thd_attn_fwd w.r.t. q, k, v.
 * [P2 "Steps/Code to reproduce bug"] runs forward/backward on this layout.
 *   q, k, v, o (forward output), dout: bf16 as in thd_attn_fwd; lse [Hq, T_q]
 *   fp32 from thd_attn_fwd.
 *   dq [dq_rows, Hq, D], dk/dv [dkv_rows, Hkv, D] bf16 outputs, with
 *   dq_rows >= T_q and dkv_rows >= T_kv.  Every row without a valid token,
 *   including the slack rows [pad[B], rows), is written with 0 (the THD
 *   gradient tail-zero of [P2 "Describe the bug"], done on the device with
 *   no extra launch and no work when there is no slack).
 * dK/dV of each kv head sum over its query-head group.  Two passes: a
 * key-stationary kernel for dK/dV and a query-stationary kernel for dQ (it
 * recomputes S and dP for its query tile); every output element is summed in
 * a fixed order, so dQ, dK and dV are bit-reproducible across runs.
 * Launches: the planner (both schedules in one launch), the Delta
 * preprocess, dQ, dK/dV.
 */
THD_API int thd_attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                 void* dq, void* dk, void* dv, int64_t dq_rows, int64_t dkv_rows, const int32_t* cu_seqlens_q,
                 const int32_t* cu_seqlens_kv, const int32_t* cu_seqlens_q_padded,
                 const int32_t* cu_seqlens_kv_padded, int B, int64_t T_q, int64_t T_kv, int Hq, int Hkv, int D,
                 int causal, float softmax_scale, int cp_size, int pad_between_seqs, void* workspace,
                 size_t workspace_bytes, int32_t* dev_status, thd_stream_t stream);

/*
 * thd_lse_merge -- in place: (o_acc, lse_acc) <- merge((o_acc, lse_acc),
 * (o_part, lse_part)), the ring's per-step output correction
 * [P1 traceback].  Per (t, h), with a = lse_acc, b = lse_part:
 *     lse = max(a, b) + log1p(exp(-|a - b|))
 *     o   = exp(a - lse) o_acc + exp(b - lse) o_part
 * A side with lse = -inf contributes nothing; both -inf give (0, -inf).
 *   o_acc, o_part [T, H, D] fp32; lse_acc, lse_part [H, T] fp32; 16-byte
 *   aligned.  D a multiple of 4.  H at most 16384 (else THD_ERR_UNSUPPORTED).
 */
THD_API int thd_lse_merge(float* o_acc, float* lse_acc, const float* o_part, const float* lse_part, int64_t T, int H,
                  int D, thd_stream_t stream);

/*
 * thd_lse_merge_bf16 -- thd_lse_merge with the incoming partial o_part in
 * bf16 ([T, H, D], 8-byte aligned; thd_attn_fwd_step_bf16's output); the
 * accumulator (o_acc fp32, lse_acc) and lse_part are as in thd_lse_merge.
 */
THD_API int thd_lse_merge_bf16(float* o_acc, float* lse_acc, const void* o_part, const float* lse_part, int64_t T,
                               int H, int D, thd_stream_t stream);

/*
 * thd_grad_tail_zero -- zero gradient rows past the last padded endpoint:
 * rows [cu_seqlens_q_padded[B], dq_rows) of dq and [cu_seqlens_kv_padded[B],
 * dkv_rows) of dk and dv (bf16, [rows, H, D]).  [P2 "Describe the bug"]:
 * the THD tail-zero; [P2 "Expected behavior"]: no work when the valid
 * endpoint equals the buffer end.  The endpoint is read ON THE DEVICE (no
 * host sync, graph-safe); when the caller already knows there is no tail
 * (host_knows_no_tail = 1) nothing is launched.  Any of dq/dk/dv may be NULL.
 * An endpoint outside [0, rows] is invalid metadata: that buffer is left
 * untouched (no write ever falls outside [0, rows) of a buffer).
 */
THD_API int thd_grad_tail_zero(void* dq, void* dk, void* dv, int64_t dq_rows, int64_t dkv_rows, int Hq, int Hkv, int D,
                       const int32_t* cu_seqlens_q_padded, const int32_t* cu_seqlens_kv_padded, int B,
                       int host_knows_no_tail, thd_stream_t stream);

/*
 * ---- Ulysses (A2A) and hierarchical a2a+p2p context parallelism, emulated ----
 *
 * [P1, the maintainer's reply]: A2A (Ulysses) exchanges heads for sequence
 * and THD had no A2A path; [P3]: hierarchical CP runs A2A inside groups of
 * a2a_size ranks and the P2P ring across cp_size / a2a_size groups, with
 * prod(sizes) == cp_size.  Layouts (the pages print none; plainest reading):
 *   shards [cp_size][T/cp_size, H, D] bf16: CP rank r's THD shard, its rows
 *     in load-balanced order -- chunk r then chunk 2cp-1-r of every sequence,
 *     chunk = P_b / (2 cp_size) rows -- the rows thd_cp_partition's token map
 *     lists for rank r;
 *   groups [a2a_size][T, H/a2a_size, D] bf16: member i of the A2A groups
 *     holds heads [i H/a2a, (i+1) H/a2a) of every token at its global padded
 *     row.  Groups are runs of a2a_size consecutive ranks, so group j holds
 *     exactly p2p rank j's rows of the 2 * (cp/a2a) split.
 * a2a_size == cp_size is pure Ulysses; a2a_size == 1 is the plain P2P ring.
 * T is the global row count (shard stride T/cp_size rows, T % cp_size == 0);
 * rows past cu_seqlens_padded[B] are not moved.
 */

/*
 * thd_cp_a2a -- move one tensor between the two layouts, every rank and
 * group in one launch.  direction THD_A2A_TO_GROUPS reads shards from src
 * and writes groups to dst; THD_A2A_TO_SHARDS the reverse.
 *   src, dst: device bf16, 16-byte aligned, not overlapping.
 *   cu_seqlens_padded: device int32 [B+1]; checked on the device (starts at
 *     0, monotone, every P_b divisible by 2*cp_size, pad[B] <= T), else a
 *     THD_DEV_ERR_* code in *dev_status and nothing written.
 *   H % a2a_size == 0, cp_size % a2a_size == 0, D a multiple of 8.
 * Bit-exact (a permutation of rows).  Launches: the planner (checks only)
 * and the copy kernel.
 */
THD_API int thd_cp_a2a(const void* src, void* dst, const int32_t* cu_seqlens_padded, int B, int64_t T, int H, int D,
                       int cp_size, int a2a_size, int direction, int32_t* dev_status, thd_stream_t stream);

/*
 * Bytes of workspace thd_attn_fwd_a2a (for_bwd = 0) or thd_attn_bwd_a2a
 * (for_bwd = 1) needs: global-order copies of the moved tensors plus the
 * attention workspace.  Returns 0 for unsupported sizes.
 */
THD_API size_t thd_a2a_workspace_size(int B, int64_t T, int Hq, int Hkv, int D, int cp_size, int a2a_size,
                                      int for_bwd);

/*
 * thd_attn_fwd_a2a -- attention through the emulated A2A / hierarchical
 * decomposition: q, k, v shards -> the members' buffers (one launch); every
 * member runs the fused P2P ring of p2p = cp_size / a2a_size ranks over its
 * heads; O -> shards.  On one GPU the members' buffers are the head slices
 * of one tensor in global row order (the a2a_size = 1 layout of thd_cp_a2a),
 * so a single thd_attn_fwd launch with cp_size = p2p serves every member;
 * its work items are per head, so a member's result depends on its own
 * slice alone.  Equal to unsplit attention (tested).
 *   q [cp][T/cp, Hq, D], k, v [cp][T/cp, Hkv, D], o [cp][T/cp, Hq, D]: shards.
 *   lse: fp32 [Hq, T] in global row order (members' heads stacked).
 *   cu_seqlens, cu_seqlens_padded: device int32 [B+1], self-attention (the
 *     same for q and kv); the padded offsets define the shards.
 *   Hq, Hkv divisible by a2a_size; D 64 or 128.
 * Launches: 5 (checks, move in, planner, forward, move out).  Workspace:
 * thd_a2a_workspace_size(.., 0).
 */
THD_API int thd_attn_fwd_a2a(const void* q, const void* k, const void* v, void* o, float* lse,
                             const int32_t* cu_seqlens, const int32_t* cu_seqlens_padded, int B, int64_t T, int Hq,
                             int Hkv, int D, int causal, float softmax_scale, int cp_size, int a2a_size,
                             void* workspace, size_t workspace_bytes, int32_t* dev_status, thd_stream_t stream);

/*
 * thd_attn_bwd_a2a -- gradients through the same decomposition: q, k, v, o,
 * dO shards -> the members' buffers (one launch); the thd_attn_bwd path with
 * cp_size = p2p for every member at once; dQ, dK, dV -> shards (one launch).
 *   Shards as in thd_attn_fwd_a2a; lse [Hq, T] as it returns it; dq
 *   [cp][T/cp, Hq, D], dk, dv [cp][T/cp, Hkv, D].  Rows of each shard past
 *   cu_seqlens_padded[B] / cp_size are not written.
 * Launches: 7 (checks, move in, the four of thd_attn_bwd, move out).
 * Workspace: thd_a2a_workspace_size(.., 1).
 * Bit-reproducible.
 */
THD_API int thd_attn_bwd_a2a(const void* q, const void* k, const void* v, const void* o, const float* lse,
                             const void* dout, void* dq, void* dk, void* dv, const int32_t* cu_seqlens,
                             const int32_t* cu_seqlens_padded, int B, int64_t T, int Hq, int Hkv, int D, int causal,
                             float softmax_scale, int cp_size, int a2a_size, void* workspace, size_t workspace_bytes,
                             int32_t* dev_status, thd_stream_t stream);

/*
 * Profiling hook (not needed for normal use): while enabled for `kernel_id`
 * (a THD_KERNEL_* value), every launch of that kernel is bracketed by a pair
 * of CUDA events recorded on its stream, up to `max_records` launches.
 * thd_profile_read synchronises those events and returns the durations in
 * milliseconds (oldest first) and their number.  kernel_id 0 disables.
 */
THD_API int thd_profile_enable(int kernel_id, int max_records);
THD_API int thd_profile_read(float* ms_out, int max_out, int* count_out);

/* Number of kernels this library has launched in this process. */
THD_API uint64_t thd_launch_count(void);

/*
 * Test hook for the failure path (not for normal use): the NEXT launch of
 * kernel_id (THD_KERNEL_FWD, THD_KERNEL_BWD or THD_KERNEL_BWD_DQ) runs no
 * work: every thread waits on a barrier that nothing completes, the bounded
 * wait gives up after its limit (2 s), each CTA frees its tensor memory and
 * the call's *dev_status reads THD_ERR_TIMEOUT.  That call's outputs are not
 * written.  The device stays usable for the next call.  kernel_id 0 disarms.
 * One-shot and process-wide.
 */
THD_API int thd_test_arm_stall(int kernel_id);

/*
 * Test hook (not for normal use): the forward has two kernels with the same
 * results up to rounding order -- one that runs a single work item per CTA
 * at a time (used when sequences average at least 16384 tokens) and one
 * with two items in flight per CTA (used otherwise).  which =
 * THD_FWD_KERNEL_SINGLE or THD_FWD_KERNEL_DUAL makes every later forward
 * call (fused or one-step) use that kernel, so tests can run both on any
 * workload; 0 restores the automatic choice.  Process-wide.  Returns
 * THD_ERR_INVALID_ARG for any other value.
 */
#define THD_FWD_KERNEL_SINGLE 1
#define THD_FWD_KERNEL_DUAL 2
THD_API int thd_test_select_fwd_kernel(int which);

#ifdef __cplusplus
}
#endif

#endif /* THD_ATTN_H */
