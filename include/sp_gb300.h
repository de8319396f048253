/*
 * sp_gb300.h -- C ABI of the GB300 (sm_103a) blockwise-attention library.
 *
 * One data-parallel hot path, simulated on one GPU:
 *
 *   1. The Ulysses sequence-shard <-> head-shard redistribution, which on one
 *      device is a layout permutation ("Ulysses SP: entrenar modelos con
 *      millones de tokens", section "Cómo funciona Ulysses Sequence
 *      Parallelism (SP)"; "DeepSpeed-Ulysses", section "Method":
 *      (N/P, d) -> (N, d/P)).
 *   2. Exact softmax attention computed blockwise over P key/value blocks in
 *      ring order, partial results combined by the cumulative (online)
 *      softmax ("Ring Attention", section "Cómo funciona la atención en
 *      anillo"), with the causal mask derived from O(n) position_ids
 *      ("Ulysses SPで100万トークン学習", section 3).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor argument is a DEVICE pointer to a dense, row-major
 *   (C-contiguous) buffer owned by the caller.  The library never allocates,
 *   frees or retains device memory, and keeps no pointer after returning.
 * - All work is enqueued on `stream` (NULL = legacy default stream) and runs
 *   asynchronously; the call returns once the kernels are launched.
 * - Arguments are validated on the host BEFORE anything is launched; a
 *   rejected call returns an SP_ERR_* status and enqueues nothing.
 * - A CUDA error when configuring or launching a kernel returns SP_ERR_CUDA
 *   (the CUDA error itself is left for cudaGetLastError()).
 * - Outputs must not overlap inputs.
 * - Sizes are element counts; B, S, H*, d, P must be >= 1 unless stated.
 *
 * Layouts (innermost dimension last):
 *   sequence-sharded  x     [B][S][H][d]        (P shards = P slices of S)
 *   head-sharded      y     [P][B][S][H/P][d]   (y[r] = what rank r holds)
 *   q                       [B][S][Hq][d]
 *   k, v                    [B][S][Hkv][d]      (GQA: q head h uses kv head
 *                                                h / (Hq/Hkv))
 *   position_ids            [B][S] int32
 *   out                     [B][S][Hq][d]
 *   lse                     [B][Hq][S] float32, natural log of
 *                           sum_j exp(scale * q.k_j) over the allowed keys
 */
#ifndef SP_GB300_H
#define SP_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; declared here so that this header
 * does not need the CUDA headers. */
typedef struct CUstream_st* sp_stream_t;

typedef enum sp_status {
  SP_OK = 0,
  SP_ERR_INVALID_ARG = 1,     /* bad pointer, size, divisibility or enum   */
  SP_ERR_UNSUPPORTED = 2,     /* valid request the library does not support */
  SP_ERR_WORKSPACE = 3,       /* workspace NULL/too small/misaligned        */
  SP_ERR_CUDA = 4,            /* CUDA runtime/driver error at launch        */
  SP_ERR_DEVICE_TIMEOUT = 5   /* a kernel gave up waiting on a barrier      */
} sp_status;

typedef enum sp_dtype {
  SP_BF16 = 0,   /* bfloat16 storage; float32 accumulation                */
  SP_F32 = 1     /* float32 storage and arithmetic                         */
} sp_dtype;

typedef enum sp_block_order {
  /* block p = tokens [p*S/P, (p+1)*S/P): the sequence sharding of the
   * Ulysses pages (GPU i holds tokens [i*n/P, (i+1)*n/P)). */
  SP_ORDER_CONTIGUOUS = 0,
  /* block p = tokens {t : t mod P == p}: Striped Attention ("Ring
   * Attention", "Cómo funciona la atención en anillo": each device's tokens
   * spread uniformly over the sequence; stripe width 1). */
  SP_ORDER_STRIPED = 1
} sp_block_order;

/* Human-readable name of a status code (static string, never NULL). */
const char* sp_status_string(sp_status status);

/* ------------------------------------------------------------------------
 * Ulysses redistribution as a permutation (bit-exact copy).
 *
 * sp_ulysses_seq_to_head: y[r][b][t][hl][:] = x[b][t][r*(H/P) + hl][:]
 *   x: [B][S][H][d], y: [P][B][S][H/P][d], element type `dtype`.
 *   This is what the first all-to-all of a Ulysses attention layer delivers:
 *   rank r ends up with every position of head group r (heads
 *   r*H/P .. (r+1)*H/P - 1, contiguous groups).
 * sp_ulysses_head_to_seq: the inverse (the second all-to-all):
 *   x[b][t][r*(H/P) + hl][:] = y[r][b][t][hl][:].
 *
 * Errors: SP_ERR_INVALID_ARG if a pointer is NULL, a size < 1, S % P != 0
 * (the pages require the sequence length to be divisible by sp_size) or
 * H % P != 0 (Ulysses needs num_heads >= sp_size, in equal groups).
 * ------------------------------------------------------------------------ */
sp_status sp_ulysses_seq_to_head(const void* x, void* y, int B, int S, int H, int d, int P,
                                 sp_dtype dtype, sp_stream_t stream);
sp_status sp_ulysses_head_to_seq(const void* y, void* x, int B, int S, int H, int d, int P,
                                 sp_dtype dtype, sp_stream_t stream);

/* The permutations have two kernels with the same results: a TMA-staged
 * copy (chunks gathered and scattered through shared memory by tensor-map
 * and bulk copies) and a vector copy (16-byte loads and stores by every
 * thread).  The TMA-staged one runs when a launch reads at least
 * `min_bytes` (default 128 MiB) and its rules hold (chunks of 256 B .. 8 KiB,
 * a multiple of 16 B; every pointer 16-byte aligned); below that its longer
 * request latency costs more than it gains.  Sets the threshold for the
 * whole process (0: TMA-staged whenever the rules hold) and returns the
 * previous value.  No counterpart on the pages (a tuning choice). */
size_t sp_permute_set_bulk_min_bytes(size_t min_bytes);

/* Error word of the TMA-staged permutation kernel (one per GPU, process
 * wide): that kernel stages chunks through shared memory with bulk copies and
 * waits on barriers with a bounded wait; a wait that runs out of time (which
 * does not happen in a correct run) records 1 here and its CTA returns early,
 * leaving the output undefined.  Writes the word to *code (must not be NULL)
 * and clears it.  Synchronous (a copy from device memory on the current
 * device).  Returns SP_OK when the word was 0, SP_ERR_DEVICE_TIMEOUT when it
 * was set, SP_ERR_CUDA or SP_ERR_INVALID_ARG.  No counterpart on the pages
 * (they name no failure detection for the kernels). */
sp_status sp_get_permute_error(int* code);

/* sp_ulysses_seq_to_head for the q, k and v of one layer in a single launch:
 * q [B][S][Hq][d] -> yq [P][B][S][Hq/P][d], k, v [B][S][Hkv][d] ->
 * yk, yv [P][B][S][Hkv/P][d].  Same results and errors as three
 * sp_ulysses_seq_to_head calls (also SP_ERR_INVALID_ARG if Hkv % P != 0). */
sp_status sp_ulysses_seq_to_head_qkv(const void* q, const void* k, const void* v, void* yq,
                                     void* yk, void* yv, int B, int S, int Hq, int Hkv, int d,
                                     int P, sp_dtype dtype, sp_stream_t stream);

/* ------------------------------------------------------------------------
 * Document starts from position_ids (the O(n) causal-mask carrier,
 * "Ulysses SPで100万トークン学習", section 3).
 *
 * A document starts at token 0 and at every t with
 * position_ids[b][t] != position_ids[b][t-1] + 1.  doc_start[b][t] = the
 * first token of t's document.  Query t may attend key j iff
 * doc_start[b][t] <= j <= t, which is "same document and j <= t".
 *
 * position_ids: [B][S] int32 (device); doc_start: [B][S] int32 (device).
 * workspace: device scratch of sp_segment_starts_workspace_bytes(B, S)
 * bytes, 256-byte aligned.
 * Errors: SP_ERR_INVALID_ARG (NULL pointer, size < 1),
 * SP_ERR_WORKSPACE (workspace NULL, misaligned or too small).
 * ------------------------------------------------------------------------ */
size_t sp_segment_starts_workspace_bytes(int B, int S);
sp_status sp_segment_starts(const int32_t* position_ids, int32_t* doc_start, int B, int S,
                            void* workspace, size_t workspace_bytes, sp_stream_t stream);

/* ------------------------------------------------------------------------
 * Blockwise (ring) attention, forward.
 *
 * The sequence is cut into P blocks (`order`).  For every query block i the
 * key/value blocks are visited in ring order j = (i - s) mod P,
 * s = 0 .. P-1 ("Ring Attention", "Cómo funciona la atención en anillo"),
 * and merged by the online softmax: a running max m, a running sum of
 * exponentiated scores l and a running weighted-value sum O, rescaled by
 * exp(m_old - m_new) when the max grows and divided at the end.  The
 * result is exact softmax attention (up to rounding):
 *
 *   out[b][t][h][:] = sum_{j allowed} softmax_j(scale * q[b][t][h] . k[b][j][h/g]) v[b][j][h/g][:]
 *   lse[b][h][t]    = log sum_{j allowed} exp(scale * q[b][t][h] . k[b][j][h/g])
 *
 * with g = Hq / Hkv.  allowed(t, j): every j when position_ids == NULL;
 * otherwise doc_start(t) <= j <= t (same document, causal), see
 * sp_segment_starts.
 *
 * q [B][S][Hq][d], k/v [B][S][Hkv][d], out [B][S][Hq][d] in `dtype`;
 * lse [B][Hq][S] float32 (may be NULL if not wanted).
 * scale <= 0 selects 1/sqrt(d).
 * Supported: SP_BF16 with d == 128 (tcgen05 tensor cores, fp32
 * accumulation, P rounded to bf16 before the PV product, out rounded to
 * nearest-even bf16); SP_F32 with 1 <= d <= 256 (fp32 FFMA throughout).
 * A row with no allowed key (only possible with the step variant below)
 * gets out = 0 and lse = -inf.
 *
 * workspace: device scratch of at least
 * sp_blockwise_attn_workspace_bytes(B, S, position_ids != NULL) bytes,
 * 256-byte aligned; it holds the device error word, the persistent kernel's
 * work counter (both reset by the call) and the doc_start array, so calls
 * that may run concurrently (different streams) need separate workspaces.
 * Its contents need not be initialised.  A non-causal bf16 call given
 * sp_blockwise_attn_split_workspace_bytes(...) bytes (about 21 MiB more) may
 * also split the items of its last, partly filled wave of CTAs into pieces
 * whose fp32 partial results are merged by their log-sum-exp (the ring's
 * partial combine), so that the last wave fills the GPU; the result is the
 * same up to rounding.
 *
 * Errors: SP_ERR_INVALID_ARG (NULL q/k/v/out, size < 1, S % P != 0,
 * Hq % Hkv != 0, bad order or dtype), SP_ERR_UNSUPPORTED (d outside the
 * supported set), SP_ERR_WORKSPACE, SP_ERR_CUDA.  Device-side barrier
 * timeouts (which do not occur in a correct run) are reported afterwards
 * by sp_get_device_error.
 * ------------------------------------------------------------------------ */
size_t sp_blockwise_attn_workspace_bytes(int B, int S, int causal);
size_t sp_blockwise_attn_split_workspace_bytes(int B, int S, int causal);
sp_status sp_blockwise_attn_fwd(const void* q, const void* k, const void* v,
                                const int32_t* position_ids, int B, int S, int Hq, int Hkv, int d,
                                int P, sp_block_order order, float scale, sp_dtype dtype, void* out,
                                float* lse, void* workspace, size_t workspace_bytes,
                                sp_stream_t stream);

/* One ring step only: every query block i attends key/value block
 * j = (i - step) mod P and nothing else.  This is the partial result device
 * i holds after ring step `step`; sp_attn_merge_partials over
 * step = 0 .. P-1 reproduces sp_blockwise_attn_fwd.  Same arguments,
 * layouts and errors as sp_blockwise_attn_fwd, plus 0 <= step < P.  Rows
 * with no allowed key in that block get out = 0, lse = -inf. */
sp_status sp_blockwise_attn_step(const void* q, const void* k, const void* v,
                                 const int32_t* position_ids, int B, int S, int Hq, int Hkv, int d,
                                 int P, sp_block_order order, int step, float scale, sp_dtype dtype,
                                 void* out, float* lse, void* workspace, size_t workspace_bytes,
                                 sp_stream_t stream);

/* ------------------------------------------------------------------------
 * Per-device forms: what ONE device of a real ring computes from the blocks
 * it holds ("Ring Attention", "Cómo funciona la atención en anillo": device i
 * keeps query block i and at step s works on the key/value block
 * j = (i - s) mod P that the ring has brought it).  The tensors hold single
 * blocks, rows in block order (row u of block p is token p*S/P + u
 * contiguous, u*P + p striped):
 *   q_blk, out_blk: [B][S/P][Hq][d]   query block i and its partial result
 *   k_blk, v_blk:   [B][S/P][Hkv][d]  key/value block j
 *   lse_blk:        [B][Hq][S/P] fp32 (may be NULL)
 * position_ids is the whole sequence's [B][S] (every device holds it: the
 * mask needs global token indices and document starts; NULL = non-causal).
 * Rows with no allowed key in block j get out = 0, lse = -inf (merging them
 * with sp_attn_merge_partials gives them weight 0).  The workspace is the
 * one sp_blockwise_attn_workspace_bytes(B, S, causal) sizes.  Errors as for
 * sp_blockwise_attn_fwd, plus SP_ERR_INVALID_ARG unless 0 <= i, j < P.
 *
 * sp_ring_block_step: query block i against key/value block j only.
 * sp_attn_merge_partials over the P steps of device i gives block i's rows
 * of sp_blockwise_attn_fwd.
 */
sp_status sp_ring_block_step(const void* q_blk, const void* k_blk, const void* v_blk,
                             const int32_t* position_ids, int B, int S, int Hq, int Hkv, int d,
                             int P, sp_block_order order, int i, int j, float scale,
                             sp_dtype dtype, void* out_blk, float* lse_blk, void* workspace,
                             size_t workspace_bytes, sp_stream_t stream);

/* sp_ring_block_step_accumulate: sp_ring_block_step folded into a running
 * result, the step a device of the ring repeats ("Ring Attention", "Cómo
 * funciona la atención en anillo": each arriving block's partial is combined
 * with what the device has so far by the cumulative softmax).  On entry
 * out_blk / lse_blk (lse_blk required) hold the running result of the steps
 * so far; on return they hold it merged with pair (i, j)'s partial:
 *   lse' = log(exp(lse) + exp(lse_ij)),
 *   out' = exp(lse - lse') * out + exp(lse_ij - lse') * out_ij
 * where out_ij is the partial before rounding to bf16.  A row whose running
 * lse is -inf takes the partial alone and its running out is not read (it
 * may hold anything); rows with no allowed key in block j keep their values
 * bit for bit.  Running lse values must be finite or -inf.  Contiguous blocks
 * under the causal mask with j > i add nothing, and the call returns SP_OK
 * without a launch.  The result equals sp_ring_block_step into a temporary
 * followed by sp_attn_merge_partials of the two, up to one bf16 rounding of
 * the partial.  SP_ERR_UNSUPPORTED unless dtype is SP_BF16 (d = 128); other
 * arguments and errors as for sp_ring_block_step. */
sp_status sp_ring_block_step_accumulate(const void* q_blk, const void* k_blk, const void* v_blk,
                                        const int32_t* position_ids, int B, int S, int Hq,
                                        int Hkv, int d, int P, sp_block_order order, int i, int j,
                                        float scale, sp_dtype dtype, void* out_blk,
                                        float* lse_blk, void* workspace, size_t workspace_bytes,
                                        sp_stream_t stream);

/* Query block i against the whole sequence, visited in ring order: what a
 * device computes once K and V have been all-gathered instead of passed
 * around the ring ("Ulysses序列并行技术详解：ms-swift如何降低长序列显存占用":
 * K and V reach every rank through all-gathers).  k, v: [B][S][Hkv][d] (the
 * whole sequence); q_blk, out_blk, lse_blk as above.  Equals block i's rows
 * of sp_blockwise_attn_fwd. */
sp_status sp_query_block_attn_fwd(const void* q_blk, const void* k, const void* v,
                                  const int32_t* position_ids, int B, int S, int Hq, int Hkv,
                                  int d, int P, sp_block_order order, int i, float scale,
                                  sp_dtype dtype, void* out_blk, float* lse_blk, void* workspace,
                                  size_t workspace_bytes, sp_stream_t stream);

/* ------------------------------------------------------------------------
 * Ulysses + Ring hybrid, for fewer heads than devices.
 *
 * Ulysses needs num_heads >= sp_size ("Ulysses SP: entrenar modelos con
 * millones de tokens", "Comparación práctica: Ulysses vs Ring Attention");
 * "Ulysses SPで100万トークン学習" section 6 points to a Ulysses + Ring hybrid
 * when GQA/MQA leaves too few heads.  With P = P_u * P_r simulated devices:
 *   1. sp_ulysses_seq_to_head of q, k, v with P_u head groups;
 *   2. blockwise ring attention with P_r blocks inside every head group
 *      (batch P_u * B; every group uses the same B rows of position_ids);
 *   3. sp_ulysses_head_to_seq of the output.
 * q [B][S][Hq][d], k/v [B][S][Hkv][d], out [B][S][Hq][d] (sequence-sharded
 * layout in and out); lse (may be NULL) in the head-sharded layout
 * [P_u][B][Hq/P_u][S] float32 -- what each Ulysses group holds.
 * Requires S % P_u == 0, S % P_r == 0, Hq % P_u == 0, Hkv % P_u == 0,
 * Hq % Hkv == 0 (SP_ERR_INVALID_ARG otherwise); the dtype/d support of
 * sp_blockwise_attn_fwd.  workspace: at least
 * sp_ulysses_ring_attn_workspace_bytes(...) bytes, 256-byte aligned (it holds
 * the head-sharded copies of q, k, v and of the output, and the attention
 * workspace).
 * ------------------------------------------------------------------------ */
size_t sp_ulysses_ring_attn_workspace_bytes(int B, int S, int Hq, int Hkv, int d, int causal,
                                            sp_dtype dtype);
sp_status sp_ulysses_ring_attn_fwd(const void* q, const void* k, const void* v,
                                   const int32_t* position_ids, int B, int S, int Hq, int Hkv,
                                   int d, int P_u, int P_r, sp_block_order order, float scale,
                                   sp_dtype dtype, void* out, float* lse, void* workspace,
                                   size_t workspace_bytes, sp_stream_t stream);

/* sp_blockwise_attn_fwd without a workspace argument, for callers that
 * cannot allocate device memory (code that must not call cudaMalloc, such as
 * a host callback or a plugin hook, or a framework whose allocator only hands
 * out the caller's own tensors).  The pages describe no such variant: it has
 * no counterpart there.
 *
 * Same arguments, layouts, results and errors as sp_blockwise_attn_fwd,
 * minus workspace / workspace_bytes.  The workspace is a fixed 5 MiB array
 * with static storage on the device, held by every GPU that loads the
 * library until the process exits.  Any non-causal call fits; a causal call
 * needs sp_blockwise_attn_workspace_bytes(B, S, 1) <= 5 MiB, which holds for
 * every B*S <= 1,048,576 tokens; larger requests return SP_ERR_WORKSPACE and
 * launch nothing.  Allocates nothing (no cudaMalloc / cudaFree, no
 * allocating library call).
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before capturing the stream into a CUDA graph.  All calls on a device share
 * the array, which keeps the last call's contents (each call clears its error
 * word and rewrites doc_start in full): calls whose kernels overlap on the
 * GPU race on it.  The device error word of this variant cannot be read
 * back. */
sp_status sp_blockwise_attn_fwd_noalloc(const void* q, const void* k, const void* v,
                                        const int32_t* position_ids, int B, int S, int Hq,
                                        int Hkv, int d, int P, sp_block_order order, float scale,
                                        sp_dtype dtype, void* out, float* lse, sp_stream_t stream);

/* ------------------------------------------------------------------------
 * Blockwise attention, backward (the pages train with sequence parallelism;
 * these are the derivatives of the forward above).
 *
 *   P  = exp(scale * Q K^T - lse)  on the allowed pairs (lse from the forward)
 *   dV = P^T dO
 *   dS = P * (dO V^T - D),  D_t = sum_c dO[t][c] * O[t][c]
 *   dQ = scale * dS K,   dK = scale * dS^T Q      (GQA: summed over the group)
 *
 * q, out, dout, dq [B][S][Hq][d]; k, v, dk, dv [B][S][Hkv][d] in `dtype`;
 * lse [B][Hq][S] float32 as written by sp_blockwise_attn_fwd for the same q,
 * k, v, position_ids and scale.  dQ visits the key/value blocks in ring order
 * j = (i - s) mod P; dK/dV visit the query blocks in the order block j meets
 * them on the ring, i = (j + s) mod P.  float32 accumulation; bf16 outputs
 * rounded to nearest-even.  Supported: SP_BF16 with d == 128 (tensor cores:
 * P and dS are rounded to bf16 before they enter the dV, dQ and dK products;
 * every tensor pointer 16-byte aligned, else SP_ERR_INVALID_ARG), SP_F32
 * with d <= 256 (CUDA cores, float32 throughout).  workspace:
 * sp_blockwise_attn_bwd_workspace_bytes(B, S, Hq, P, position_ids != NULL)
 * bytes, 256-byte aligned (it includes a float32 dQ accumulator of
 * B * Hq * P * Lbp * 128 floats, Lbp = S/P rounded up to a multiple of 128,
 * used by the bf16 path when dQ is accumulated by reductions, see
 * sp_set_bwd_dq_reduction).  Errors as for sp_blockwise_attn_fwd.
 * ------------------------------------------------------------------------ */
size_t sp_blockwise_attn_bwd_workspace_bytes(int B, int S, int Hq, int P, int causal);

/* How the bf16 backward forms dQ, for the whole process; returns the
 * previous setting.
 *   on != 0 (default): one kernel per 128-key tile multiplies S^T and dP^T
 *     once and forms dV, dK and each (query tile, key tile) piece of dQ; the
 *     pieces are added into the workspace's float32 accumulator by vector
 *     reductions in whatever order the tiles finish, then scaled and rounded
 *     to bf16.  10 d FLOPs per allowed (query, key) pair; dq is reproducible
 *     to float32 rounding of the sum, not bit for bit.
 *   on == 0: two kernels (dQ query-stationary, dK/dV key-stationary) that
 *     each multiply S and dP; 14 d FLOPs per pair; bit-reproducible.
 * dk and dv are bit-reproducible in both forms.  No counterpart on
 * the pages (an implementation choice). */
int sp_set_bwd_dq_reduction(int on);
sp_status sp_blockwise_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                                const void* dout, const float* lse, const int32_t* position_ids,
                                int B, int S, int Hq, int Hkv, int d, int P, sp_block_order order,
                                float scale, sp_dtype dtype, void* dq, void* dk, void* dv,
                                void* workspace, size_t workspace_bytes, sp_stream_t stream);

/* ------------------------------------------------------------------------
 * Backward of one ring step on one device (the device that holds query
 * block i, with key/value block j received from its ring neighbour; "Ring
 * Attention", "Cómo funciona la atención en anillo" -- the pages train with
 * it, "Ulysses SP: entrenar modelos con millones de tokens").  Adds block
 * pair (i, j)'s part of the gradients of the whole-sequence attention:
 *
 *   P   = exp(scale * Q_i K_j^T - lse_i)  on the allowed pairs (lse_i: the
 *         forward's log-sum-exp of block i's rows over ALL key blocks)
 *   D_i = rowsum(dout_i * out_i)           (out_i: the forward's output)
 *   dS  = P * (dout_i V_j^T - D_i)
 *   dq_acc += scale * dS K_j,  dk_acc += scale * dS^T Q_i,  dv_acc += P^T dout_i
 *   (GQA: the query heads of a group add into their key/value head)
 *
 * Summed over j (for dq_acc) or over i (for dk_acc, dv_acc) these are the
 * whole-sequence gradients, so a ring that passes K_j, V_j together with
 * their dk/dv accumulators visits every pair once.
 *
 * q_blk, out_blk, dout_blk [B][S/P][Hq][d] (block i's rows in local order:
 * local row u holds token u*P + i striped, i*S/P + u contiguous); k_blk,
 * v_blk [B][S/P][Hkv][d] (block j); lse_blk [B][Hq][S/P] float32;
 * position_ids [B][S] of the whole sequence or NULL (non-causal).
 * dq_acc [B][S/P][Hq][d], dk_acc, dv_acc [B][S/P][Hkv][d]: float32
 * accumulators, read and written (the caller zeroes them before the first
 * step); the pieces of one call (dq: one per key tile; dk, dv: one per
 * query head of the group) are added in no fixed order, so results are
 * reproducible to float32 rounding.  Supported: SP_BF16 with d == 128
 * (tensor cores; P and dS rounded to bf16 before the products, float32
 * accumulation), else
 * SP_ERR_UNSUPPORTED; tensor pointers 16-byte aligned.  workspace:
 * sp_ring_block_step_bwd_workspace_bytes(B, S, Hq, P, position_ids != NULL)
 * bytes, 256-byte aligned.  Errors as for sp_blockwise_attn_bwd, and
 * SP_ERR_INVALID_ARG for i or j outside [0, P).  Contiguous blocks under the
 * causal mask with j > i have no allowed pair: the call returns SP_OK
 * without a launch and the accumulators keep their values.
 * ------------------------------------------------------------------------ */
size_t sp_ring_block_step_bwd_workspace_bytes(int B, int S, int Hq, int P, int causal);
sp_status sp_ring_block_step_bwd(const void* q_blk, const void* k_blk, const void* v_blk,
                                 const void* out_blk, const void* dout_blk, const float* lse_blk,
                                 const int32_t* position_ids, int B, int S, int Hq, int Hkv,
                                 int d, int P, sp_block_order order, int i, int j, float scale,
                                 sp_dtype dtype, float* dq_acc, float* dk_acc, float* dv_acc,
                                 void* workspace, size_t workspace_bytes, sp_stream_t stream);

/* ------------------------------------------------------------------------
 * Merge of per-block partial results (the cross-device combine of ring
 * attention, "Ring Attention", "Cómo funciona la atención en anillo").
 *
 *   lse[b][h][t] = log sum_p exp(lses[p][b][h][t])
 *   out[b][t][h][:] = sum_p exp(lses[p][b][h][t] - lse[b][h][t]) * outs[p][b][t][h][:]
 *
 * outs [P][B][S][H][d] in `dtype`, lses [P][B][H][S] float32 (device);
 * out [B][S][H][d] in `dtype`, lse [B][H][S] float32 (may be NULL).
 * A partial with lse = -inf has weight 0; if all are -inf, out = 0 and
 * lse = -inf.  Arithmetic in float32; bf16 output rounded to nearest-even.
 * Errors: SP_ERR_INVALID_ARG (NULL pointer, size < 1, bad dtype).
 * ------------------------------------------------------------------------ */
sp_status sp_attn_merge_partials(const void* outs, const float* lses, int P, int B, int S, int H,
                                 int d, sp_dtype dtype, void* out, float* lse, sp_stream_t stream);

/* Waits for `stream`, then reads the device error word that the attention
 * kernels of the last calls using `workspace` left there (0 = no error;
 * otherwise a barrier wait ran out of time and that kernel returned early,
 * its output undefined).  Writes the raw word to *code when code != NULL and
 * clears it.  Returns SP_OK, SP_ERR_DEVICE_TIMEOUT or SP_ERR_CUDA. */
sp_status sp_get_device_error(void* workspace, int* code, sp_stream_t stream);

/* Check of the device-side failure path: launches one thread that waits, with
 * the same bounded wait the attention kernel uses, on a barrier that nothing
 * ever completes, limited to timeout_us microseconds (1 .. 1e6).  The kernel
 * then records its timeout code in the workspace error word and returns, so
 * sp_get_device_error(workspace, ...) reports SP_ERR_DEVICE_TIMEOUT and the
 * context stays usable.  workspace: >= 256 bytes, 256-byte aligned.  No
 * counterpart on the pages (they name no failure detection for the kernel). */
sp_status sp_check_barrier_timeout(void* workspace, int timeout_us, sp_stream_t stream);

/* Number of kernels the last successful call on this host thread enqueued
 * (lets a caller count device launches without a profiler). */
int sp_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SP_GB300_H */
