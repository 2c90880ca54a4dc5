/*
 * dma.h - causal + document-masked grouped-query attention for one
 * context-parallel rank, on NVIDIA GB300 (sm_103a).
 *
 * The problem (as the Llama 3 infrastructure pages state it):
 *   - "The Llama 3 Herd of Models - part 3/16", section 3.3.2, "Context
 *     parallelism for long sequences": the sequence is cut into 2*CP equal
 *     chunks, rank i holds chunks i and 2*CP-1-i; K and V are all-gathered
 *     and attention is computed for the local queries against the full K/V,
 *     under the full causal mask; K/V are small thanks to GQA.
 *   - "Paper notes: The Llama 3 Herd of Models", "Two architectural
 *     choices": GQA with 8 key-value heads; document masking keeps attention
 *     inside a document.
 *   - review of "Scaling Llama 3 Training with Efficient Parallelism
 *     Strategies", section "Context Parallelism (CP)": every CP rank receives
 *     the whole sequence's document information to build its mask.
 *   - "Training Infrastructure and Systems", "FlashAttention: never write the
 *     score matrix" ("Online softmax", "Tiling"): the blocked forward keeps a
 *     running max and sum, writes O and per-row statistics, and the backward
 *     recomputes the scores.
 *
 * Query at global position p may attend key k iff doc_start(p) <= k <= p.
 * Query head h uses K/V head h / (n_heads / n_kv_heads) (contiguous groups).
 *
 * Tensor layouts (all row-major, contiguous, device memory):
 *   q, dout, dq    : [batch][2*C][n_heads][head_dim]   bf16, this rank's rows
 *                    in local order: chunk cp_rank first, then chunk
 *                    2*cp_size-1-cp_rank (C = seq_len / (2*cp_size)).
 *   o              : same layout, fp32 (see dma_attn_fwd).
 *   k, v           : [batch][seq_len][n_kv_heads][head_dim] bf16, the full
 *                    gathered sequence in natural position order.
 *   lse            : [batch][n_heads][2*C] fp32, natural log of the sum of
 *                    exp of the scaled, masked logits of each query row.
 *   dk, dv         : [batch][seq_len][n_kv_heads][head_dim] fp32: this rank's
 *                    partial gradients (only its own query rows contribute);
 *                    summing them over all ranks gives the full gradients.
 *                    Every element is written (zeros where no local query
 *                    attends).
 *   cu_doc_lens    : int32 [n_docs + 1] cumulative document offsets over the
 *                    flattened batch*seq_len token stream: cu[0] = 0,
 *                    strictly increasing, cu[n_docs] = batch*seq_len, and
 *                    every sample boundary b*seq_len present.
 *
 * Ownership: every device buffer (tensors, cu_doc_lens, the plan workspace)
 * belongs to the caller.  The library never allocates device memory.  The
 * plan handle itself is a small host object created by dma_plan and freed by
 * dma_plan_destroy; it points into the caller's workspace, which must stay
 * valid (and untouched) until the plan is destroyed.
 *
 * Streams: every call is asynchronous on `stream` (a cudaStream_t; NULL is
 * the legacy default stream).  Nothing synchronizes except dma_plan_check and
 * dma_debug_wait_probe.  A plan's workspace also holds scratch the kernels
 * share (Delta, the fp16 copy of V, the work counters from which the forward
 * and dK/dV kernels take their work items), so the calls made on one plan
 * must not overlap on the GPU: issue them on one stream (or order them with
 * events).  Different plans may run concurrently.
 *
 * Errors: arguments the host can check are rejected before any launch with
 * DMA_ERR_INVALID_ARG / DMA_ERR_UNSUPPORTED / DMA_ERR_WORKSPACE.  Problems only
 * the device can see (malformed cu_doc_lens, an expired bounded wait) are
 * recorded in a status word in the workspace and returned by dma_plan_check;
 * kernels launched on a plan whose status is set do no work.  No call aborts
 * or traps.
 */
#ifndef DMA_H_
#define DMA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DMA_OK = 0,
  DMA_ERR_INVALID_ARG = 1, /* null pointer, negative size, rank out of range */
  DMA_ERR_BAD_DOCS = 2,    /* cu_doc_lens violates its contract (device) */
  DMA_ERR_UNSUPPORTED = 3, /* shape outside the supported set, or not sm_103 */
  DMA_ERR_CUDA = 4,        /* a CUDA runtime / driver call failed */
  DMA_ERR_TIMEOUT = 5,     /* a bounded device-side wait expired */
  DMA_ERR_WORKSPACE = 6,   /* workspace too small or misaligned */
  /* Not an error: the results were computed, but finite v values beyond the
   * fp16 range (|v| > 65504) were saturated at +-65504 in the forward's fp16
   * copy of v, so o and lse of the rows that attend them are inexact.
   * Reported by dma_plan_check (and the no-alloc forward's status_dev) only
   * when no error occurred. */
  DMA_WARN_V_SATURATED = 7
} dma_status;

/* bf16 values are passed as raw 16-bit patterns. */
typedef uint16_t dma_bf16;

/* Tile classes (one byte per pair of query tile and key tile). */
enum { DMA_TILE_SKIP = 0, DMA_TILE_FULL = 1, DMA_TILE_PARTIAL = 2 };

typedef struct dma_plan_s* dma_plan_t;

/*
 * Bytes of device workspace dma_plan needs for this shape (256-byte aligned
 * base required).  Returns 0 for an unsupported or invalid shape.
 * max_docs is accepted for interface stability and does not change the size.
 * The last part of the layout is the backward's pool of fp32 partial dK, dV
 * for cut query lists: 2 x kv_pool_slots x 128 x n_kv_heads x head_dim x 4
 * bytes (kv_pool_slots: max(batch * n_ktiles, min(ceil(512 / n_kv_heads),
 * what the lists could use)); see dma_plan_view).  The allocation-free
 * forward needs only the part before it.
 */
size_t dma_plan_workspace_bytes(int batch, int seq_len, int cp_size,
                                int n_heads, int n_kv_heads, int head_dim,
                                int max_docs);

/*
 * Build the rank's plan: the context-parallel query-position map (part 3/16,
 * 3.3.2: chunks i and 2*CP-1-i), the document start of every local query,
 * the rank-major chunk order, and the classification of every pair of query
 * tile and key tile as skip / full / partial with its row and column lists.
 *
 * Supported shapes: cp_size >= 1; 0 <= cp_rank < cp_size; batch >= 0
 * (batch 0 builds an empty plan whose calls do nothing); seq_len divisible
 * by 2*cp_size with chunk C = seq_len/(2*cp_size) a multiple of 64;
 * g = n_heads/n_kv_heads in {1,2,4,8,16} with C a multiple of 128/g;
 * head_dim in {64, 128}.  A query tile is 128 rows = 128/g positions x g
 * heads of one K/V group; a key tile is 128 positions.
 *
 * softmax_scale <= 0 selects 1/sqrt(head_dim).
 * cu_doc_lens (device) is read only by kernels this call enqueues; it may be
 * freed once they complete.  The returned handle is valid on success only.
 * Device: the current CUDA device must be compute capability 10.3.
 */
dma_status dma_plan(const int32_t* cu_doc_lens, int n_docs, int batch,
                    int seq_len, int cp_size, int cp_rank, int n_heads,
                    int n_kv_heads, int head_dim, float softmax_scale,
                    void* workspace, size_t workspace_bytes, void* stream,
                    dma_plan_t* out);

/*
 * Forward: o = softmax(scale * q k^T + mask) v and the row log-sum-exp.
 * Two launches: an fp16 copy of v into the plan workspace, then the attention
 * kernel, in which pairs of tiles
 * classified skip issue no work.  The probabilities enter the P V product in
 * fp16 and o is written in fp32: a bf16 o could not hold a 1e-2 absolute
 * error bound once |o| >= 4 (half a bf16 ulp there is 0.0156), which rows that
 * see only a few keys of a short document reach.
 * The fp16 copy keeps NaN and +-Inf as they are (they reach o as they would
 * in bf16 arithmetic); finite values beyond +-65504 saturate there, which the
 * plan's status then reports as DMA_WARN_V_SATURATED.
 */
dma_status dma_attn_fwd(dma_plan_t plan, const dma_bf16* q, const dma_bf16* k,
                        const dma_bf16* v, float* o, float* lse,
                        void* stream);

/*
 * Backward: dq (bf16), and this rank's partial dk, dv (fp32), given the
 * forward's o and lse and the upstream gradient dout.  The backward
 * recomputes the scores ("Training Infrastructure and Systems",
 * "FlashAttention: never write the score matrix", "Tiling"); dk and dv are
 * kept in fp32 ("The Llama 3 Herd of Models - part 3/16", 3.3.2, "Numerical
 * stability").  Two launches (three when the key tiles' query lists are
 * split, see below): a query-stationary dQ kernel that also computes
 * Delta = rowsum(dout * o) into the plan workspace, then a key-stationary
 * dK/dV kernel reduced over the group's query heads.  dk and dv are fully
 * overwritten.
 */
dma_status dma_attn_bwd(dma_plan_t plan, const dma_bf16* q, const dma_bf16* k,
                        const dma_bf16* v, const float* o, const float* lse,
                        const dma_bf16* dout, dma_bf16* dq, float* dk,
                        float* dv, void* stream);

/*
 * The launches of the backward, callable one by one (in stream order):
 *   dma_attn_bwd_dq_delta: dq (bf16) and Delta = rowsum(dout * o) into the
 *                       plan workspace, in one kernel; what dma_attn_bwd runs.
 *   dma_attn_bwd_delta: Delta alone (a pass over o and dout of its own).
 *   dma_attn_bwd_dq   : dq from the Delta already in the workspace.
 *   dma_attn_bwd_dkdv : dk, dv (fp32, fully overwritten) from q, k, v, lse,
 *                       dout and the workspace's Delta, in one kernel.  The
 *                       query lists of key tiles that the plan cut into
 *                       segments (see kv_slices in dma_plan_view) leave fp32
 *                       partials in the workspace, which the same kernel
 *                       adds into dk, dv in segment order (the same on
 *                       every run).
 * Delta must be in place (dq_delta or delta) before dq or dkdv runs.
 */
dma_status dma_attn_bwd_dq_delta(dma_plan_t plan, const dma_bf16* q, const dma_bf16* k,
                                 const dma_bf16* v, const float* o, const float* lse,
                                 const dma_bf16* dout, dma_bf16* dq, void* stream);
dma_status dma_attn_bwd_delta(dma_plan_t plan, const float* o, const dma_bf16* dout,
                              void* stream);
dma_status dma_attn_bwd_dkdv(dma_plan_t plan, const dma_bf16* q, const dma_bf16* k,
                             const dma_bf16* v, const float* lse, const dma_bf16* dout,
                             float* dk, float* dv, void* stream);
dma_status dma_attn_bwd_dq(dma_plan_t plan, const dma_bf16* q, const dma_bf16* k,
                           const dma_bf16* v, const float* lse, const dma_bf16* dout,
                           dma_bf16* dq, void* stream);

/* Synchronize `stream` and return the plan's device status: DMA_ERR_BAD_DOCS
 * or DMA_ERR_TIMEOUT if the device recorded an error, else
 * DMA_WARN_V_SATURATED if a forward saturated v values, else DMA_OK; or
 * DMA_ERR_CUDA if the read-back itself failed. */
dma_status dma_plan_check(dma_plan_t plan, void* stream);

/* Free the host handle (the caller's workspace is untouched). NULL is ok. */
dma_status dma_plan_destroy(dma_plan_t plan);

/* Static, human-readable name of a status code. */
const char* dma_status_str(dma_status s);

/*
 * Cut this rank's rows out of a full-sequence tensor, and put them back:
 *   full  : [batch][seq_len][H][elem_bytes-sized elements x row_elems]
 *   local : [batch][2*C][...] in the plan's local order.
 * row_bytes = bytes of one position (H * head_dim * element size).
 * Bit-exact copies; used to emulate the sharding on one device.
 */
dma_status dma_cp_gather(dma_plan_t plan, const void* full, void* local,
                         size_t row_bytes, void* stream);
dma_status dma_cp_scatter(dma_plan_t plan, const void* local, void* full,
                          size_t row_bytes, void* stream);

/*
 * Chunk-order copies for a real context-parallel exchange ("The Llama 3 Herd
 * of Models - part 3/16", 3.3.2: K and V are all-gathered across the CP
 * ranks before attention; "Numerical stability": the gradients are
 * reduce-scattered in FP32).  An all-gather of every rank's local rows (its
 * chunks r and 2*CP-1-r, in the local order of the plan) lands rank-major:
 *   gathered : [cp_size][batch][2*C][row_bytes]   (C = seq_len / (2*cp_size))
 * while the kernels read K and V in natural sequence order:
 *   full     : [batch][seq_len][row_bytes]
 * dma_cp_unpermute copies gathered -> full (after the all-gather of K, V);
 * dma_cp_permute copies full -> gathered (before the reduce-scatter of a
 * rank's partial dK, dV, so that block r of the result is rank r's rows).
 * Plain device pointers, no plan needed; bit-exact; asynchronous on stream.
 * Errors: DMA_ERR_INVALID_ARG for null pointers, row_bytes == 0 or seq_len
 * not divisible by 2*cp_size.
 */
dma_status dma_cp_unpermute(const void* gathered, void* full, int batch, int seq_len,
                            int cp_size, size_t row_bytes, void* stream);
dma_status dma_cp_permute(const void* full, void* gathered, int batch, int seq_len,
                          int cp_size, size_t row_bytes, void* stream);

/*
 * Read-only view of the plan's device arrays (for tests and tools).
 * All pointers are device pointers into the caller's workspace.
 *   qpos      int32 [2C]             global position of each local row
 *   doc_lo    int32 [batch][2C]      first position of that row's document
 *   chunk_order int32 [2*cp_size]    rank-major chunk order
 *   tile_class uint8 [batch][n_qtiles][n_ktiles]
 *   row_ptr   int32 [batch*n_qtiles + 1], row_idx int32 [nnz]:
 *             ascending non-skip key tiles of each query tile; bit 31 set
 *             when the pair is partial.
 *   col_ptr   int32 [batch*n_ktiles + 1], col_idx int32 [nnz]: the same by
 *             key tile (query-tile indices, bit 31 = partial).
 *   fwd_order int32 [batch*n_qtiles]: query tiles (b*n_qtiles + t) by
 *             non-increasing list length, ties by index.
 *   bwd_order int32 [batch*n_ktiles]: key tiles likewise.
 *   kv_slices int32 [n_kv_slices][8]: the dK/dV work list in launch order.
 *             Per slice: key tile (b*n_ktiles + kt), first entry in col_idx,
 *             length, segment, split-unit index (-1 when the tile's list is
 *             not cut), pool slot (-1 for segment 0 and uncut lists), 0, 0.
 *             The planner cuts the lists longer than a length L into
 *             ceil(n / L) contiguous segments when its bound on the greedy
 *             makespan over n_sms SMs says one SM would otherwise run long
 *             after the others; slices are ordered by non-increasing length.
 *   kv_splits int32 [n_kv_splits][4]: per cut list: key tile, pool slot of
 *             segment 1, segments, 0.
 *   counts    int32 [2]: n_kv_slices, n_kv_splits (device-written).
 *   n_sms, kv_pool_slots: SMs the plan balances over; slots of the pool of
 *             fp32 partial dK, dV (segments 1.. of cut lists) in the workspace.
 */
typedef struct {
  int batch, seq_len, cp_size, cp_rank, n_heads, n_kv_heads, head_dim;
  int chunk, local_len, group, q_tile_positions, n_qtiles, n_ktiles;
  float softmax_scale;
  const int32_t* qpos;
  const int32_t* doc_lo;
  const int32_t* chunk_order;
  const uint8_t* tile_class;
  const int32_t* row_ptr;
  const int32_t* row_idx;
  const int32_t* col_ptr;
  const int32_t* col_idx;
  const int32_t* fwd_order;
  const int32_t* bwd_order;
  const uint32_t* status;
  const int32_t* kv_slices;
  const int32_t* kv_splits;
  const int32_t* counts;
  int n_sms, kv_pool_slots;
} dma_plan_view;

dma_status dma_plan_get_view(dma_plan_t plan, dma_plan_view* out);

/*
 * Bounded device waits: every spin on a barrier gives up after this many
 * nanoseconds, records DMA_ERR_TIMEOUT in the status word, drains its own
 * copies, frees its tensor memory and returns.  Default 2e9 (2 s); the
 * environment variable DMA_WAIT_TIMEOUT_NS overrides the default at dma_plan.
 */
dma_status dma_plan_set_wait_timeout(dma_plan_t plan, uint64_t timeout_ns);

/*
 * Test hook for the failure path: launch one block that waits, bounded by
 * timeout_ns, on a shared-memory barrier nothing will ever arrive on.  It
 * writes DMA_ERR_TIMEOUT into *status_dev (device uint32) when the wait
 * expires.  Synchronizes `stream`, and returns the recorded status (or
 * DMA_ERR_CUDA).  Nothing faults or hangs: the kernel returns after the limit.
 */
dma_status dma_debug_wait_probe(uint64_t timeout_ns, uint32_t* status_dev,
                                void* stream);

/*
 * Allocation-free forward (the pages have no counterpart: this is a
 * convenience of this library).  For callers that may not allocate device
 * memory at all -- code that must not grow or step outside a fixed memory
 * pool, or hosts that forbid cudaMalloc -- and so cannot provide the plan
 * workspace the other entry points need.  It does what dma_plan followed by
 * dma_attn_fwd does, with all scratch (the plan and the fp16 copy of v) in a
 * 64 MiB array compiled into the library; the caller passes only inputs and
 * outputs.
 *   - Every GPU that loads the library holds the 64 MiB until the process
 *     exits.  Shapes whose scratch exceeds it return DMA_ERR_WORKSPACE (the
 *     scratch is dma_plan_workspace_bytes less the backward's pool of
 *     partials described there).
 *   - The first call on a device looks up the array's device address with
 *     that device current; make that first call outside any stream capture.
 *     Only a successful lookup is kept (a failed one returns DMA_ERR_CUDA and
 *     is tried again by the next call).
 *   - All calls share the one array: calls whose work overlaps on the GPU
 *     (different streams, or different host threads) race and corrupt each
 *     other; serialize them (one stream is enough).
 *   - status_dev (optional, device uint32) receives the plan's status
 *     (DMA_OK, DMA_ERR_BAD_DOCS, DMA_ERR_TIMEOUT or DMA_WARN_V_SATURATED, as
 *     dma_plan_check would return it) in stream order; on a
 *     malformed cu_doc_lens, o and lse are left unwritten.
 *   - It calls no allocator: no cudaMalloc, no cudaFree, no host heap.
 */
dma_status dma_attn_fwd_noalloc(const int32_t* cu_doc_lens, int n_docs, int batch,
                                int seq_len, int cp_size, int cp_rank, int n_heads,
                                int n_kv_heads, int head_dim, float softmax_scale,
                                const dma_bf16* q, const dma_bf16* k,
                                const dma_bf16* v, float* o, float* lse,
                                uint32_t* status_dev, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DMA_H_ */
