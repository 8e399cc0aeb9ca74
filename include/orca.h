/*
 * orca.h -- C ABI of liborca.so: one GPU, one process.
 *
 * Orca-style serving of a decoder-only GPT: an iteration-level scheduler hands
 * the engine one iteration at a time; the engine runs that iteration over an
 * arbitrary mix of initiation (prompt) and increment (one-token) requests with
 * selective batching, and returns one greedy next token per request.
 *
 * Sources (page title, section):
 *   [houmin]      garden.houmin.site "Orca" notes: 3.1.1 iteration-level
 *                 scheduling (workflow steps 1-5), 3.1.2 selective batching.
 *   [0h-n0]       "論文解説: Orca — Iteration-Level Scheduling..." : Selective
 *                 Batching, scheduler algorithm, implementation notes.
 *   [arcsin2]     "ORCA: A Distributed Serving System for Transformer-Based
 *                 Generative Models" notes: 3.2 selective batching, 4.1
 *                 architecture (engine master sends request ids, token indices
 *                 and initiation/increment state), 4.2 scheduling algorithm.
 *   [ultralytics] "Continuous Batching" glossary: limits on sequences and
 *                 tokens per step.
 *
 * Conventions for every function below:
 *   - Return value: ORCA_OK (0) on success, a negative ORCA_ERR_* otherwise.
 *     Nothing throws across the ABI.  orca_strerror() names a code.
 *   - Host arrays passed in are owned by the caller and only read during the
 *     call.  Device pointers passed in are owned by the caller and must stay
 *     valid for as long as the callee documents.
 *   - All device work is issued on the CUDA stream given at engine creation.
 *   - The library is not thread-safe: one thread drives one engine.
 */
#ifndef ORCA_H_
#define ORCA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------------ */
/* status codes                                                              */
/* ------------------------------------------------------------------------ */
#define ORCA_OK 0
#define ORCA_ERR_INVALID (-1)     /* bad argument or inconsistent batch descriptor */
#define ORCA_ERR_KV_FULL (-2)     /* no free contiguous K/V range of that size      */
#define ORCA_ERR_CUDA (-3)        /* a CUDA runtime / driver call failed            */
#define ORCA_ERR_DEVICE_FLAG (-4) /* a kernel recorded an error (bad index, expired */
                                  /* bounded wait); the engine stays usable         */
#define ORCA_ERR_NOT_FOUND (-5)   /* unknown request id                             */
#define ORCA_ERR_OOM (-6)         /* host or device allocation failed               */
#define ORCA_ERR_LIMIT (-7)       /* sizes exceed the fixed scratch of an           */
                                  /* allocation-free entry point                    */

#define ORCA_DTYPE_FP32 0 /* every tensor fp32; SIMT FFMA kernels              */
#define ORCA_DTYPE_BF16 1 /* matrices, embeddings, K/V, GEMM operands in bf16; */
                          /* fp32 accumulation, statistics and residual stream */

const char *orca_strerror(int code);

/* ------------------------------------------------------------------------ */
/* model and engine                                                          */
/* ------------------------------------------------------------------------ */
/* Decoder shape and engine limits.  head_dim = hidden / n_heads must be 16, 32,
 * 64 or 128.  For bf16, hidden, 3*hidden and ffn must be multiples of 64. */
typedef struct orca_model_config {
    int32_t n_layers, hidden, n_heads, ffn, vocab, max_pos;
    int32_t dtype;      /* ORCA_DTYPE_* */
    int32_t max_tokens; /* per-iteration budget on sum(n_input), the flattened rows */
    int32_t max_batch;  /* requests per iteration */
    int64_t kv_slots;   /* K/V pool size in tokens (all layers share the index) */
    int32_t pack_weights; /* bf16 only: 1 = keep an engine-owned copy of w_qkv, w_o, w_1, w_2 and
                             of tok_emb (as LM head) repacked tile-contiguous for streaming
                             (see orca_pack_weight); 0 = read the caller's matrices directly */
} orca_model_config;

/* Per-layer weights: device pointers, borrowed by the engine and read on every
 * iteration, so they must outlive it (with pack_weights the four matrices are
 * copied at creation and need not).  Matrices are row-major
 * [out, in] in the model dtype; vectors are fp32.
 *   w_qkv [3H, H] (rows 0..H-1 produce q, H..2H-1 k, 2H..3H-1 v; head j is the
 *   j-th group of head_dim rows of each), w_o [H, H], w_1 [F, H], w_2 [H, F]. */
typedef struct orca_layer_weights {
    const void *w_qkv, *w_o, *w_1, *w_2;
    const float *b_qkv, *b_o, *b_1, *b_2;
    const float *ln1_g, *ln1_b, *ln2_g, *ln2_b;
} orca_layer_weights;

/* tok_emb [V, H] is also the (tied) LM head; pos_emb [max_pos, H].  `layers`
 * is a HOST array of n_layers entries, read during orca_engine_create only. */
typedef struct orca_weights {
    const void *tok_emb, *pos_emb;
    const float *lnf_g, *lnf_b;
    const orca_layer_weights *layers;
} orca_weights;

typedef struct orca_engine orca_engine;

/* Create an engine.  Allocates, once, the K/V pool of kv_slots tokens for every
 * layer ([0h-n0] implementation notes: reserve all K/V memory at start-up, no
 * per-request device allocation) and the activation buffers for max_tokens
 * rows.  `stream` is a cudaStream_t (NULL = legacy default stream).
 * Errors: INVALID (shape), OOM, CUDA. */
int orca_engine_create(const orca_model_config *cfg, const orca_weights *w, void *stream, orca_engine **out);
int orca_engine_destroy(orca_engine *eng);

/* ------------------------------------------------------------------------ */
/* K/V reservation ([0h-n0] scheduler algorithm: reserve a request's maximum  */
/* length when it is admitted; [houmin] 3.1.1: free it when it finishes)      */
/* ------------------------------------------------------------------------ */
/* Reserve n_tokens contiguous slots for request_id: first fit at the lowest
 * free offset.  *out_offset = first slot.  Errors: KV_FULL (nothing changed),
 * INVALID (n_tokens <= 0 or id already holds a reservation). */
int orca_kv_alloc(orca_engine *eng, int64_t request_id, int32_t n_tokens, int64_t *out_offset);
/* Release the reservation of request_id (merged with free neighbours).
 * Errors: NOT_FOUND. */
int orca_kv_free(orca_engine *eng, int64_t request_id);

/* Layout of the K/V pool, for callers that load a pre-existing context.
 * Element (layer l, K=0/V=1, head h, slot s, component c) is at
 *   base + ((((l*2 + kv)*n_heads + h)*kv_slots + s)*head_dim + c)
 * elements of elem_bytes each.  The pointer is owned by the engine. */
typedef struct orca_kv_layout {
    void *base;
    int64_t kv_slots;
    int32_t n_layers, n_heads, head_dim, elem_bytes;
} orca_kv_layout;
int orca_kv_layout_get(orca_engine *eng, orca_kv_layout *out);

/* ------------------------------------------------------------------------ */
/* one iteration                                                             */
/* ------------------------------------------------------------------------ */
/* Batch descriptor ([arcsin2] 4.1: request ids, token indices and the
 * initiation/increment state per request).  All arrays are HOST memory, n_req
 * entries unless noted.  Request i owns rows off[i] .. off[i]+n_input[i]-1 of
 * the flattened [sum(n_input), H] activation, off = exclusive prefix sum.
 *   phase[i]    0 = initiation (ctx_len must be 0), 1 = increment (ctx_len > 0);
 *               [houmin] 3.1.2: the phase is whether K/V exists for it.
 *   n_input[i]  rows this iteration (the prompt length, or 1).
 *   ctx_len[i]  tokens already cached; row j sits at position ctx_len[i] + j.
 *   kv_offset[i] the offset orca_kv_alloc returned for request_id[i];
 *               ctx_len[i] + n_input[i] must not exceed that reservation.
 *   tokens      sum(n_input) input ids, request by request.  A value >= 0 is a
 *               token id (< vocab).  A value t < 0 refers to the token this
 *               engine returned for request j = -1 - t of the previous
 *               iteration (feedback without a host round trip).
 * Every request id appears at most once. */
typedef struct orca_batch {
    int32_t n_req;
    const int64_t *request_id;
    const int32_t *phase;
    const int32_t *n_input;
    const int32_t *ctx_len;
    const int64_t *kv_offset;
    const int32_t *tokens;
} orca_batch;

/* Run one iteration ([houmin] 3.1.1 workflow steps 2-4; [houmin] 3.1.2 /
 * [0h-n0] Selective Batching): embed the flattened rows, run every layer with
 * the token-wise operations on [sum L, H] and attention split per request
 * (causal within the request's new rows, over its own cached K/V; this
 * iteration's K/V are appended first), then LayerNorm each request's last row,
 * apply the tied LM head and take the greedy argmax (lowest id on ties).
 * out_next_tokens: HOST array of n_req entries.  Synchronous: returns after the
 * tokens are on the host.  Errors: INVALID (descriptor), CUDA, DEVICE_FLAG. */
int orca_run_iteration(orca_engine *eng, const orca_batch *batch, int32_t *out_next_tokens);

/* Pre-planned iterations, for a caller that keeps descriptors resident on the
 * device and runs several iterations without a host round trip.
 * orca_plan_build validates `batch` exactly like orca_run_iteration and packs
 * it into `host_buf` (int32 words; needs orca_plan_words() words).  The caller
 * copies those words to device memory (16-byte aligned) and later calls
 * orca_run_planned with both copies; iterations must run in the order their
 * plans were built.  orca_run_planned is asynchronous on the engine stream;
 * dev_out_next (device, n_req int32, may be NULL) receives the next tokens.
 * orca_engine_sync waits for the stream and reports DEVICE_FLAG errors. */
int64_t orca_plan_words(const orca_engine *eng, const orca_batch *batch);
int orca_plan_build(orca_engine *eng, const orca_batch *batch, int32_t *host_buf, int64_t cap_words);
int orca_run_planned(orca_engine *eng, const int32_t *host_plan, const int32_t *dev_plan, int32_t *dev_out_next);
int orca_engine_sync(orca_engine *eng);

/* The same iteration as a conventional padded + masked batch ([houmin] 3.1.2
 * "问题" and [arcsin2] 3.2: batching needs tensors of one shape, so requests
 * of different lengths are padded and masked; [0h-n0] "Request-Level vs
 * Iteration-Level Scheduling": the baseline Orca is compared with).  The
 * descriptor is the same; the engine runs every request with Lq = max
 * n_input rows -- its own rows, then pad rows of token 0 at the positions
 * that follow, whose K/V land inside its reservation (ctx_len + Lq must fit
 * it and max_pos) and are overwritten by its next real row -- and, when Lq =
 * 1, every request's attention covers the batch's longest key range
 * Lk = max(ctx_len) + 1, its keys past ctx_len[i] masked.  The next token of
 * request i comes from its last real row, so the results equal those of the
 * selective batch; only the work differs (Lq * n_req rows must fit
 * max_tokens).  A request-level scheduler keeps finished members in their
 * batch as single-row requests on token 0, whose tokens it ignores.
 * Errors and synchrony as orca_run_iteration / orca_plan_build. */
int orca_run_iteration_padded(orca_engine *eng, const orca_batch *batch, int32_t *out_next_tokens);
int64_t orca_plan_words_padded(const orca_engine *eng, const orca_batch *batch);
int orca_plan_build_padded(orca_engine *eng, const orca_batch *batch, int32_t *host_buf, int64_t cap_words);

/* Parity/debug read-back of the last iteration: the final-LayerNorm output of
 * each request's last row (n_req x hidden floats) and the logits (n_req x vocab
 * floats), copied to HOST memory.  n = number of floats the buffer holds. */
int orca_get_last_hidden(orca_engine *eng, float *host_out, int64_t n);
int orca_get_last_logits(orca_engine *eng, float *host_out, int64_t n);

/* Engine counters: kernel launches issued since creation, iterations run. */
typedef struct orca_engine_stats {
    int64_t launches, iterations;
} orca_engine_stats;
int orca_engine_stats_get(orca_engine *eng, orca_engine_stats *out);

/* Per-kernel timing on the engine stream.  When enabled, every launch of one
 * sampled layer per iteration (layer = iteration index mod n_layers) and the
 * LM head are bracketed by CUDA events.  orca_engine_timing_read syncs and
 * returns up to `cap` records (oldest first) and clears them. */
typedef struct orca_kernel_time {
    int32_t kind;     /* ORCA_K_* */
    int32_t layer;    /* -1 for per-iteration kernels */
    float ms;         /* event-to-event time on the stream */
    double bytes;     /* algorithmic bytes moved (weights + activations + K/V) */
    double flops;     /* algorithmic flops */
} orca_kernel_time;
#define ORCA_K_EMBED 0
#define ORCA_K_LN 1
#define ORCA_K_GEMM_QKV 2
#define ORCA_K_KV_APPEND 3
#define ORCA_K_ATTN_DECODE 4
#define ORCA_K_ATTN_PREFILL 5
#define ORCA_K_GEMM_O 6
#define ORCA_K_GEMM_FFN1 7
#define ORCA_K_GEMM_FFN2 8
#define ORCA_K_LM_HEAD 9
#define ORCA_K_ARGMAX 10
#define ORCA_K_FINAL_LN 11
int orca_engine_timing(orca_engine *eng, int32_t enable);
int orca_engine_timing_read(orca_engine *eng, orca_kernel_time *out, int32_t cap, int32_t *n_out);

/* Failure-detection test hook (the pages describe no such facility).  Launches,
 * on the engine stream, a kernel whose one thread waits on a barrier that
 * nothing completes, with the same bounded wait every pipelined kernel uses
 * but a limit of limit_ns nanoseconds (1 ns .. 10 s).  The wait gives up,
 * records an expired wait in the engine's device error word and the kernel
 * returns; the next orca_engine_sync (or orca_run_iteration) reports
 * ORCA_ERR_DEVICE_FLAG, clears the word and the engine stays usable.
 * Asynchronous.  Errors: INVALID (limit out of range), CUDA. */
int orca_debug_expire_wait(orca_engine *eng, int64_t limit_ns);

/* Host-side fault injection: when the process environment holds
 * ORCA_FAULT=kv_alloc:N at the creation of an engine or of a scheduler without
 * an engine, the N-th K/V reservation of that object's pool fails as if the
 * pool were full (ORCA_ERR_KV_FULL; a scheduler then stops admitting for that
 * iteration, as the [0h-n0] scheduler algorithm does when K/V runs out). */

/* ------------------------------------------------------------------------ */
/* operator entry points (device pointers; used by the kernel parity tests)  */
/* ------------------------------------------------------------------------ */
/* y[t, f] = sum_k x[t, k] * w[f, k]  (+ bias[f]) (GeLU if gelu) ; then
 *   resid != NULL : out_f32[t, f] = resid[t, f] + y   (resid may equal out_f32)
 *   else          : out_f32 or out_bf16 (exactly one non-NULL) = y.
 * dtype BF16: x, w bf16 (tcgen05 tensor cores, fp32 accumulation; k % 64 == 0);
 * dtype FP32: x, w fp32 (SIMT FFMA).  Rows of out have stride ld_out.
 * With 129 or more rows and at least one 128-feature output tile per SM the
 * bf16 path runs the stream-K kernel (units of 64-wide K blocks spread evenly
 * over every SM, cut tiles finished by whichever piece arrives last, in a
 * fixed CTA order, so results are reproducible run to run).
 * Asynchronous on the engine's stream (uses the engine's stream-K workspace
 * and arrival counters, so calls on one engine must not overlap);
 * orca_engine_sync waits and reports device-side errors.
 * Tuning overrides, read once per process from the environment:
 * ORCA_GEMM_SK (1 = stream-K whenever the workspace allows, -1 = never),
 * ORCA_GEMM_STAGES (ring depth cap), ORCA_GEMM_SPLITS (split-K ways where the
 * caller completes partials; orca_run_iteration only).
 * Errors: INVALID (shape / pointer combination), CUDA. */
int orca_op_linear(orca_engine *eng, int32_t dtype, const void *x, const void *w, int32_t w_packed, int32_t m_tok,
                   int32_t n_out, int32_t k, const float *bias, int32_t gelu, const float *resid, float *out_f32,
                   void *out_bf16, int32_t ld_out);

/* Repack a bf16 weight w [n_out, k] (k % 64 == 0) for streaming: tiles of 128
 * rows x 64 columns, tile (ft, kb) stored contiguously at element offset
 * (ft * k/64 + kb) * 8192 in exactly the 128-byte-swizzled layout the tensor
 * cores read from shared memory, rows past n_out zero.  `out` (device) must
 * hold orca_packed_weight_elems(n_out, k) bf16 elements.  Asynchronous on the
 * engine stream.  A packed weight is passed to orca_op_linear with w_packed = 1. */
int64_t orca_packed_weight_elems(int32_t n_out, int32_t k);
int orca_pack_weight(orca_engine *eng, const void *w, int32_t n_out, int32_t k, void *out);

/* Attention of one layer for a batch of requests (the kernels of
 * orca_run_iteration), on device data.  Layout as inside an iteration:
 *   qkv      [sum(n_input), 3*hidden] rows of the batch, request by request;
 *            only the q columns [0, hidden) are read (dtype elements).
 *   kv_layer one layer of a K/V pool: [K|V][n_heads][kv_slots][head_dim]; the
 *            rows of this iteration must already be in it.
 *   out      [sum(n_input), hidden].
 * n_input, ctx_len, kv_offset: HOST arrays of n_req entries.  Row j of
 * request i sits at position ctx_len[i] + j and attends to keys 0 ..
 * ctx_len[i] + j of slots kv_offset[i] ... ([houmin] 3.1.2: attention runs per
 * request).  Requests with one row take the split-K decode kernel, others the
 * prefill kernel.  n_req <= max_batch of the engine; asynchronous on the
 * engine stream, using the engine's scratch.  Errors: INVALID, CUDA. */
int orca_op_attention(orca_engine *eng, int32_t dtype, const void *qkv, const void *kv_layer, int64_t kv_slots,
                      int32_t n_heads, int32_t head_dim, int32_t n_req, const int32_t *n_input,
                      const int32_t *ctx_len, const int64_t *kv_offset, void *out);

/* Allocation-free decode attention.  The Orca paper has no counterpart to this
 * entry point: it exists for callers that cannot allocate device memory at
 * call time -- for
 * example code running inside a memory-constrained host process that has
 * handed all device memory to its own allocator, or a runtime that forbids
 * cudaMalloc on its serving thread -- and so cannot create an engine.  It runs
 * the same split-K decode kernel as orca_op_attention for requests that have
 * exactly one input row each (increment phase), with the kernel's scratch
 * (plan tables, per-(request, head) arrival counters, split-K partials) in a
 * fixed device array of about 16.5 MiB inside this library.  Every GPU that loads the
 * library holds that array until the process exits.
 *   qkv [n_req, 3*hidden], kv_layer [K|V][n_heads][kv_slots][head_dim],
 *   out [n_req, hidden]: device pointers, owned by the caller.
 *   ctx_len, kv_offset: HOST arrays of n_req entries; request i attends to
 *   slots kv_offset[i] .. kv_offset[i] + ctx_len[i] (ctx_len[i] + 1 keys).
 *   stream: cudaStream_t (NULL = legacy default stream).
 * Limits: n_req <= 256, n_heads <= 128, head_dim in {16, 32, 64, 128}, and the
 * split-K partials (work items x n_heads x (head_dim + 2) floats, a work item
 * being 64 to 512 keys of one request) within 4 Mi floats; beyond them the call
 * returns ORCA_ERR_LIMIT and does nothing.
 * It calls no cudaMalloc, cudaFree or other allocating routine.  The first call
 * on a device looks up the array's device address (once per device, with that
 * device current).  The host tables are copied from pageable memory, which
 * waits for the stream's earlier work.
 * Every call shares the one array and it keeps the last call's contents (the
 * counters are cleared at each call): calls that overlap on the GPU -- on
 * different streams, or from different threads -- race and must not be made.
 * Device-side wait timeouts are not reported by this entry point.
 * Errors: INVALID (arguments), LIMIT (sizes), CUDA. */
int orca_attention_decode_noalloc(int32_t dtype, const void *qkv, const void *kv_layer, int64_t kv_slots,
                                  int32_t n_heads, int32_t head_dim, int32_t n_req, const int32_t *ctx_len,
                                  const int64_t *kv_offset, void *out, void *stream);

/* ------------------------------------------------------------------------ */
/* iteration-level scheduler ([houmin] 3.1.1, [0h-n0] scheduler algorithm,    */
/* [arcsin2] 4.2)                                                            */
/* ------------------------------------------------------------------------ */
/* Request pool + FCFS selection under max_batch, max_tokens (rows per
 * iteration) and the K/V pool.  Candidates are ordered by (arrival, id); the
 * batch is the longest prefix of that order that fits; a waiting request that
 * does not fit (including a failed K/V reservation) stops admission.  After an
 * iteration every selected request gets its token; a request is done after
 * out_len tokens and its K/V is freed at once.
 * mode 1 = request-level baseline: a batch is formed only when the previous
 * one has completely finished; its K/V is freed when it completes.
 * chunked_prefill (mode 0 only): a request still in its prompt whose remaining
 * prompt exceeds what is left of the iteration's max_tokens takes exactly what
 * is left (>= 1 token) and admission stops there; its prompt runs in chunks
 * over consecutive iterations, each with the tokens processed so far as
 * context (phase 1, n_input > 1), and only the iteration that processes its
 * last prompt token yields a token (the engine's output for an earlier chunk
 * is ignored).  Prompts longer than max_tokens become admissible.  The pages
 * describe no chunking (a later system's idea); this is the plainest reading. */
typedef struct orca_sched_config {
    int32_t max_batch, max_tokens;
    int64_t kv_slots;      /* used only when no engine is attached */
    int32_t kv_reserve;    /* tokens reserved per request; 0 = prompt + out_len */
    int32_t mode;          /* 0 iteration-level, 1 request-level */
    int32_t token_feedback;/* 1: increment inputs are emitted as references to
                              the previous iteration's outputs (see orca_batch) */
    int32_t chunked_prefill; /* 0 or 1 (see above) */
    int32_t n_workers;     /* batches that may be open at once ([houmin] 3.1.3
                              pipelining); 0 or 1 = one; > 1 needs mode 0 and
                              token_feedback 0 */
} orca_sched_config;

typedef struct orca_sched orca_sched;

/* `eng` may be NULL: the scheduler then keeps its own host-side K/V pool of
 * cfg->kv_slots tokens (same placement rule), which needs no GPU. */
int orca_sched_create(const orca_sched_config *cfg, orca_engine *eng, orca_sched **out);
int orca_sched_destroy(orca_sched *s);

/* Add a request.  prompt: HOST array.  arrival is on the iteration clock.
 * ctx0 > 0 enters a request whose first ctx0 tokens are already cached: its
 * K/V is reserved now (out_kv_offset, may be NULL) and prompt holds exactly its
 * one pending input token.  Errors: INVALID (does not fit its reservation or
 * the token budget), KV_FULL (ctx0 > 0 only). */
int orca_sched_submit(orca_sched *s, int64_t id, double arrival, const int32_t *prompt, int32_t prompt_len,
                      int32_t out_len, int32_t ctx0, int64_t *out_kv_offset);

/* Turn token feedback on or off from the next iteration on.  References are
 * only emitted to iterations that ran while feedback was on, so a caller may
 * schedule some iterations on the host only (feedback off) and then hand the
 * following ones to the engine. */
int orca_sched_set_token_feedback(orca_sched *s, int32_t enable);

/* Select the batch for the current iteration.  *status = 1 and *out filled
 * (arrays owned by the scheduler, valid until the next call) when there is
 * work; *status = 0 for an idle tick (the clock advanced, no batch); *status
 * = 2 when every request has finished; *status = 3 when nothing can be
 * selected until an open batch completes.  A selected batch stays open until
 * orca_sched_complete; with n_workers > 1 up to n_workers batches may be open
 * ([houmin] 3.1.3: while one batch runs the next is scheduled), and a request
 * in an open batch is never selected again before it completes, so open
 * batches are disjoint.  The clock advances at each selection and idle tick.
 * Errors: INVALID when n_workers batches are already open. */
int orca_sched_next(orca_sched *s, orca_batch *out, int32_t *status);

/* Report the next tokens (HOST, one per request) of the OLDEST open batch;
 * retires its finished requests. */
int orca_sched_complete(orca_sched *s, const int32_t *next_tokens);

/* Cancel a waiting or running request between iterations ([houmin] 3.1.1: a
 * request that leaves the pool has its memory freed at once): it never runs
 * again, its K/V reservation is freed immediately (also in request-level
 * mode), its tokens so far stay readable (state 3), and a request-level batch
 * whose remaining members are all done completes at once.
 * Errors: NOT_FOUND (unknown id), INVALID (the request is in an open batch,
 * finished, or already cancelled). */
int orca_sched_cancel(orca_sched *s, int64_t id);

typedef struct orca_sched_stats {
    int64_t clock;            /* iteration clock */
    int64_t iterations;       /* engine iterations issued */
    int64_t generated;        /* tokens generated */
    int64_t finished, waiting, running;
    int64_t kv_reserved;      /* tokens currently reserved */
    int64_t cancelled;
} orca_sched_stats;
int orca_sched_stats_get(orca_sched *s, orca_sched_stats *out);

/* Per-request record.  admitted_at / finished_at are iteration-clock values
 * (-1 = not yet; a request entered with ctx0 > 0 is admitted at -1). */
typedef struct orca_request_info {
    int64_t id, kv_offset;
    int32_t state; /* 0 waiting, 1 running, 2 finished, 3 cancelled */
    int32_t ctx_len, n_generated;
    int64_t admitted_at, finished_at;
} orca_request_info;
int orca_sched_request_get(orca_sched *s, int64_t id, orca_request_info *out);
/* Generated tokens of a request (HOST buffer of cap entries). */
int orca_sched_request_tokens(orca_sched *s, int64_t id, int32_t *out, int32_t cap, int32_t *n_out);

/* Serve loop: keep up to n_workers batches selected, run the oldest with
 * orca_run_iteration and complete it, until every request has finished or
 * max_iterations engine iterations ran.  The engine is the one the scheduler
 * was created with. */
int orca_sched_run(orca_sched *s, int64_t max_iterations);

#ifdef __cplusplus
}
#endif
#endif /* ORCA_H_ */
