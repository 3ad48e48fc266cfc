/*
 * rwkv7.h -- C ABI of the GB300 (sm_103a) RWKV-7 batched decode library.
 *
 * The library runs the batched single-token decode step of an RWKV-7 language
 * model over a pool of per-sequence state slots, as the continuous-batching
 * worker of the RWKV-Runner Albatross article does ("连续批处理Worker 主循环":
 * forward_seq_batch over the organised slot batch, then penalties and
 * sample_next_tokens_batch), with prefill kept apart from decode as in the
 * RWKV-Server article ("RWKV 批量推理中 Prefill 的正确打开方式", §五: prefill
 * prompt[:-1], then decode from prompt[-1]).
 *
 * Conventions for every entry point:
 *  - Return value: RWKV7_OK (0) or a negative RWKV7_E* code; rwkv7_last_error()
 *    then returns a text description (valid until the next call on the ctx).
 *  - Ownership: the library owns the weights, the slot pool (recurrent states,
 *    occurrence counts, sampling parameters) and its scratch memory, all in
 *    device memory it allocates in rwkv7_create / rwkv7_set_weight.  Pointers
 *    named d_* are caller-owned DEVICE pointers; h_* / host_* are caller-owned
 *    HOST pointers.  Nothing is retained after a call returns except inside the
 *    ctx.
 *  - Execution: calls taking device pointers are asynchronous and ordered on the
 *    ctx's CUDA stream (the one given to rwkv7_create, or the legacy default
 *    stream if NULL).  Errors found on the device (an out-of-range or repeated
 *    slot, an out-of-range token) are latched in a device word and reported by
 *    the next rwkv7_synchronize() as RWKV7_EINVAL; the kernels never access
 *    memory out of bounds because of them.  Calls taking host pointers
 *    synchronize the stream before they return.
 *  - Not thread-safe: one ctx is used by one host thread at a time.
 */
#ifndef RWKV7_H
#define RWKV7_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define RWKV7_API __attribute__((visibility("default")))
#else
#define RWKV7_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define RWKV7_OK 0
#define RWKV7_EINVAL (-1)   /* bad argument: null pointer, size, slot or token out of range */
#define RWKV7_ESHAPE (-2)   /* weight name unknown or its size does not match the config */
#define RWKV7_ENOMEM (-3)   /* device or host allocation failed */
#define RWKV7_ECUDA (-4)    /* a CUDA runtime/driver call failed */
#define RWKV7_ETIMEOUT (-5) /* a bounded wait inside a kernel gave up */
#define RWKV7_ESTATE (-6)   /* call out of order (e.g. decode before every weight is set) */

#define RWKV7_MAX_STEP_BATCH 256 /* slots per fused step; larger B is split into sub-steps */

typedef struct rwkv7_ctx rwkv7_ctx;

/* Model shape and pool size.  head_size must be 64; d_model a multiple of 64;
 * d_ffn a multiple of 64; lora_* multiples of 8; n_slots >= 1. */
typedef struct {
    int32_t n_layer, d_model, head_size, d_ffn, vocab;
    int32_t lora_w, lora_a, lora_v, lora_g;
    int32_t n_slots;
} rwkv7_config;

/* Per-slot sampling parameters (defaults of the Albatross adapter: temperature 1,
 * top_p 0.3, top_k 0 (off), frequency 1, penalty_decay 0.996, presence 0).
 * greedy != 0 (or temperature <= 0) takes the argmax of the raw logits (lowest
 * index on ties) and leaves the occurrence counts untouched. */
typedef struct {
    float temperature, top_p;
    int32_t top_k;
    float presence, frequency, penalty_decay;
    uint64_t seed;
    int32_t greedy;
} rwkv7_sampling;

/* Create a context on the current CUDA device; allocates the slot pool and
 * scratch.  cuda_stream: a cudaStream_t (may be NULL). */
RWKV7_API int rwkv7_create(const rwkv7_config *cfg, void *cuda_stream, rwkv7_ctx **out);

/* As rwkv7_create, with the weight format of the projection matrices:
 * weight_bits 16 (fp16, as rwkv7_create) or 8 -- the int8 weight variant, in
 * which every matrix the step streams (r, k, v, output, LoRA, channel-mix key
 * and value, head; not the embedding) is int8 values q [out, in] with one fp16
 * scale per output row, W = q * scale, set with rwkv7_set_weight_i8; the other
 * tensors stay fp16.  The roadmap of the RWKV-Runner Albatross article lists
 * int8 weights among the engine's next steps; the scale per row is this
 * library's choice.  An int8 context runs the tensor-core modes 0 and 1 only.
 * Returns RWKV7_EINVAL for another weight_bits. */
RWKV7_API int rwkv7_create_ex(const rwkv7_config *cfg, int32_t weight_bits, void *cuda_stream, rwkv7_ctx **out);

/* 16 or 8 (see rwkv7_create_ex); 0 for NULL. */
RWKV7_API int32_t rwkv7_weight_bits(const rwkv7_ctx *ctx);

/* Device allocator hook.  A context created after this call takes every
 * device allocation of its lifetime (weights, slot pool, scratch) from
 * alloc(user, bytes, &ptr) -- which returns 0 and a 256-byte aligned device
 * pointer on success, anything else on failure -- and hands each back to
 * release(user, ptr) in rwkv7_destroy, so a serving process can place the
 * library's memory in its own pool.  Both NULL restores cudaMalloc / cudaFree;
 * only one NULL returns RWKV7_EINVAL.  A refused allocation makes the creating
 * call return RWKV7_ENOMEM with the ctx still destroyable.  Process-wide;
 * contexts already created keep the allocator they were created with. */
typedef int (*rwkv7_alloc_fn)(void *user, size_t bytes, void **d_ptr);
typedef void (*rwkv7_free_fn)(void *user, void *d_ptr);
RWKV7_API int rwkv7_set_device_allocator(rwkv7_alloc_fn alloc, rwkv7_free_fn release, void *user);

/* Free everything the ctx owns (synchronizes its stream first).  NULL is a no-op. */
RWKV7_API void rwkv7_destroy(rwkv7_ctx *ctx);

RWKV7_API const char *rwkv7_last_error(const rwkv7_ctx *ctx);

/* Copy one named fp16 tensor from host memory into the device weights.  Names
 * and [out, in] shapes follow the weight-file convention (e.g. "emb" [V, d],
 * "blocks.3.att.key" [d, d], "blocks.3.ffn.value" [d, d_ffn]).  bytes must be
 * the tensor's exact size.  Synchronous. */
RWKV7_API int rwkv7_set_weight(rwkv7_ctx *ctx, const char *name, const void *host_f16, size_t bytes);

/* Int8 context only: copy one named matrix given as host int8 values q
 * [out][in] (q_bytes = out * in) and fp16 row scales [out] (scale_bytes =
 * 2 * out).  RWKV7_ESHAPE for a name that is not an int8 matrix of this
 * context or for wrong sizes; rwkv7_set_weight refuses these names in an int8
 * context.  Synchronous. */
RWKV7_API int rwkv7_set_weight_i8(rwkv7_ctx *ctx, const char *name, const int8_t *host_q, size_t q_bytes,
                                  const void *host_scale_f16, size_t scale_bytes);

/* Read every tensor from an RWKV7W01 weight file (text header, 256-byte aligned
 * fp16 data) and set it.  Synchronous. */
RWKV7_API int rwkv7_load_weights(rwkv7_ctx *ctx, const char *path);

/* Slot pool (RWKV-Runner Albatross article, "策略语法与参数解析": the worker
 * keeps real_state_size = batch_size state slots, one per active sequence, and
 * swaps slots when it reorganises the batch; here slots are addressed by index,
 * so reorganising needs no copies).  Slots run from 0 to n_slots - 1; an index
 * outside that range returns RWKV7_EINVAL.  Stream-ordered. */
RWKV7_API int rwkv7_slot_reset(rwkv7_ctx *ctx, int32_t slot);            /* zero state, occurrence counts, draw counter */
RWKV7_API int rwkv7_slot_swap(rwkv7_ctx *ctx, int32_t a, int32_t b);     /* exchange everything two slots hold */
/* dst := src (recurrent and shift states; dst's occurrence counts and draw
 * counter restart).  The article's roadmap ("边界与后续路线") names a prefix
 * state cache, first as an in-memory LRU; this copy is its building block. */
RWKV7_API int rwkv7_slot_copy(rwkv7_ctx *ctx, int32_t src, int32_t dst);
/* Per-slot sampling parameters, kept in the pool (the Albatross worker holds
 * per-slot temperature / top_p / top_k / penalty tensors pre-allocated on the
 * device, "连续批处理Worker 主循环"; its adapter's defaults are listed with
 * rwkv7_sampling).  Copied from host memory; stream-ordered. */
RWKV7_API int rwkv7_slot_set_sampling(rwkv7_ctx *ctx, int32_t slot, const rwkv7_sampling *params);

/* Checkpoint of one slot's recurrent state -- the per-sequence state tuple
 * (shift_state, wkv_state) that the RWKV-Server article's prefill hands to the
 * model ("RWKV 批量推理中 Prefill 的正确打开方式", §五, the prefill method of
 * task.py) -- as fp32 wkv [L][H][64][64], then fp32 token-shift states of the
 * time mix [L][d] and of the channel mix [L][d].  host_buf is a caller-owned
 * HOST buffer of exactly rwkv7_slot_state_bytes() bytes (RWKV7_EINVAL
 * otherwise).  Both calls synchronize the ctx stream. */
RWKV7_API size_t rwkv7_slot_state_bytes(const rwkv7_ctx *ctx);
RWKV7_API int rwkv7_slot_get_state(rwkv7_ctx *ctx, int32_t slot, void *host_buf, size_t bytes);
RWKV7_API int rwkv7_slot_set_state(rwkv7_ctx *ctx, int32_t slot, const void *host_buf, size_t bytes);

/* Consume T tokens (device int32 [T]) into one slot.  If d_logits_out is not
 * NULL it receives the fp32 logits [V] after the last token.  The tokens are
 * processed in chunks of RWKV7_MAX_STEP_BATCH counted from the first one, so
 * splitting a prompt into calls at multiples of that size gives bit-identical
 * states (the prefix-state cache relies on this). */
RWKV7_API int rwkv7_prefill_seq(rwkv7_ctx *ctx, int32_t slot, const int32_t *d_tokens, int32_t T,
                      float *d_logits_out);

/* One decode step of B slots -- the Albatross worker's per-round
 * forward_seq_batch over the organised slot batch followed by its penalties and
 * sample_next_tokens_batch (RWKV-Runner article, "连续批处理Worker 主循环"), the
 * B > 1, T = 1 path of the RWKV-Server article ("RWKV 批量推理中 Prefill 的正确打开方式",
 * §三): slot d_slots[b] consumes token d_tokens[b] (device int32 [B] each;
 * slots distinct, 1 <= B <= n_slots; B > 256 runs as consecutive fused steps).
 * Writes fp32 logits [B][V] to d_logits_out if not NULL, and if d_next_out is
 * not NULL samples the next token of every slot with its sampling parameters
 * (updating its occurrence counts and draw counter) into d_next_out [B].
 * Returns RWKV7_EINVAL for null inputs or B out of range, RWKV7_ESTATE before
 * every weight is set; bad slot or token values are latched on the device and
 * reported by rwkv7_synchronize.  Asynchronous on the ctx stream. */
RWKV7_API int rwkv7_decode_step(rwkv7_ctx *ctx, const int32_t *d_slots, const int32_t *d_tokens,
                      int32_t B, float *d_logits_out, int32_t *d_next_out);

/* Same step with host buffers (h_logits_out / h_next_out may be NULL): copies
 * the inputs in, runs the step and copies the results out; synchronous.  Slots
 * and tokens are checked on the host before anything is launched. */
RWKV7_API int rwkv7_decode_step_host(rwkv7_ctx *ctx, const int32_t *h_slots, const int32_t *h_tokens,
                           int32_t B, float *h_logits_out, int32_t *h_next_out);

/* Sample one token per slot from caller logits (device fp32 [B][V], row b for
 * slot d_slots[b]) with the slots' sampling parameters -- the worker's batched
 * sample_next_tokens_batch with per-slot top_k / top_p / temperature and the
 * presence / frequency penalties applied first (RWKV-Runner article,
 * "连续批处理Worker 主循环"; defaults from "适配器Runner 与异步引擎之间的桥").
 * Updates the slots' occurrence counts and draw counters; writes d_next_out
 * [B].  RWKV7_EINVAL for null pointers or B out of range.  Asynchronous. */
RWKV7_API int rwkv7_sample_batch(rwkv7_ctx *ctx, const int32_t *d_slots, const float *d_logits,
                       int32_t B, int32_t *d_next_out);

/* Largest B * V that rwkv7_sample_rows_static accepts: 4,194,304 fp32 elements
 * (16 MiB), e.g. 64 rows of a 65,536-token vocabulary. */
#define RWKV7_SAMPLE_STATIC_MAX_ELEMS (1 << 22)

/* Allocation-free variant of rwkv7_sample_batch.  The articles describe no counterpart:
 * it is a library convenience for callers that must not allocate device memory
 * while they sample -- a serving process that has already handed all of HBM to
 * its own arena (so cudaMalloc would fail), or a loop that cannot afford the
 * device-wide synchronisation that cudaMalloc / cudaFree may cause, stalling
 * the decode stream of every other batch.  It needs no rwkv7_ctx (whose
 * creation allocates a whole slot pool): the caller owns every input and
 * output, and the sampler's penalised-logit scratch lives in a fixed 16 MiB
 * array of the library's device code, which the CUDA runtime reserves on every
 * device that loads the library and keeps until the process exits.  The call
 * makes no cudaMalloc / cudaFree and calls no allocating library routine.
 *
 * It runs the same kernel, with the same arithmetic, as rwkv7_sample_batch, so
 * given equal logits, parameters, occurrence counts and draw counters both
 * return the same tokens.
 *
 *  d_logits    device fp32 [B][V], row b = the logits of batch row b
 *  d_rows      device int32 [B]: row b samples with per-sequence entry d_rows[b]
 *              of the three arrays below (distinct within one call; an index
 *              outside [0, n_rows) sets flag 1 in *d_err and gives token 0)
 *  B, V        1 <= B, 1 <= V, B * V <= RWKV7_SAMPLE_STATIC_MAX_ELEMS; larger
 *              batches are rejected (RWKV7_EINVAL) and must be split by the caller
 *  n_rows      entries in each per-sequence array
 *  d_occ       device fp32 [n_rows][V] occurrence counts, read and updated
 *  d_params    device rwkv7_sampling [n_rows] (8-byte aligned), read only
 *  d_ndraw     device uint64 [n_rows] draw counters (8-byte aligned), read and
 *              incremented once per sampled (non-greedy) row
 *  d_next_out  device int32 [B], the sampled tokens
 *  d_err       device uint32 word; flags are OR-ed into it (1 = row index out of
 *              range, 16 = no token could be kept); the caller clears it
 *  cuda_stream the cudaStream_t to launch on (NULL = legacy default stream)
 *              -- it and every pointer above must belong to the CURRENT device
 *              (the one whose scratch address the call uses)
 *  err_msg     if not NULL, receives a static text describing a host-side error
 *              ("" on success); valid until the next call from the same thread
 *
 * Set-up: the first call on each device (with that device current) looks up the
 * scratch array's device address and sets the kernel's shared-memory limit;
 * make that first call before any stream capture on that device.
 * Scratch contents: nothing in it has to start at zero -- each call writes
 * every element it later reads -- and it keeps the last call's values.  All
 * calls on a device share the one array, so two calls whose kernels overlap on
 * the GPU (different streams, or different host threads without ordering)
 * race on it and may return wrong tokens; order them on one stream.
 * Asynchronous on cuda_stream; returns RWKV7_OK, RWKV7_EINVAL (null pointer,
 * misaligned array, bad or too large size) or RWKV7_ECUDA. */
RWKV7_API int rwkv7_sample_rows_static(const float *d_logits, const int32_t *d_rows, int32_t B, int32_t V,
                                       int32_t n_rows, float *d_occ, const rwkv7_sampling *d_params,
                                       uint64_t *d_ndraw, int32_t *d_next_out, uint32_t *d_err,
                                       void *cuda_stream, const char **err_msg);

/* Wait for the ctx's stream and report device-side errors latched since the
 * last call (RWKV7_EINVAL for bad slots/tokens, RWKV7_ETIMEOUT for a bounded
 * wait that gave up).  Clears the latched error. */
RWKV7_API int rwkv7_synchronize(rwkv7_ctx *ctx);

/* Test hook: OR `flags` (bits of the device error word: 1 bad slot, 2 bad
 * token, 4 repeated slot, 8 a bounded in-kernel wait gave up, 16 sampler
 * found no token) into the ctx's device error word, as a kernel would latch
 * it, so that the error path of rwkv7_synchronize can be exercised without
 * making any kernel fail.  Synchronizes the ctx stream. */
RWKV7_API int rwkv7_debug_latch_error(rwkv7_ctx *ctx, uint32_t flags);

/* Select the decode implementation: 0 = tensor-core kernels with CUDA-graph
 * replay (default), 1 = the same kernels launched directly, 2 = CUDA-core
 * (SIMT) projection kernels launched directly (a slow cross-check; fp16
 * weights only).  RWKV7_EINVAL for another value. */
RWKV7_API int rwkv7_set_mode(rwkv7_ctx *ctx, int32_t mode);

/* The ctx's own device I/O buffers for a fused step (capacity min(n_slots, 256)
 * rows): passing these pointers to rwkv7_decode_step skips its staging copies. */
RWKV7_API int rwkv7_get_io_buffers(rwkv7_ctx *ctx, int32_t **d_slots, int32_t **d_tokens, float **d_logits,
                         int32_t **d_next);

/* Sparse channel mix (RWKV-Server article, "RWKV 批量推理中 Prefill 的正确打开方式"
 * §三: cmix_sparse_one / cmix_sparse_rows skip the value rows whose ReLU^2
 * input is zero): the value projection reads only the 64-row blocks of the
 * value matrix whose hidden block is nonzero for some slot of the step.  This
 * returns, since the previous call (or rwkv7_create), the number of such
 * nonzero blocks and the number of blocks considered (layers x d_ffn/64 per
 * step or prefill chunk), then resets both.  Synchronous. */
RWKV7_API int rwkv7_ffn_union_stats(rwkv7_ctx *ctx, uint64_t *nonzero_blocks, uint64_t *blocks);

/* Kernel classes of rwkv7_profile_step, in output order. */
#define RWKV7_PROF_EMBED 0       /* embedding + LayerNorm 0 (+ slot/token checks) */
#define RWKV7_PROF_LN_MIX 1      /* LayerNorm + token-shift mixes (time and channel mix) */
#define RWKV7_PROF_GEMM_PROJ 2   /* r, k, v and LoRA-down projections */
#define RWKV7_PROF_GEMM_LORA 3   /* LoRA-up projections with decay / gate epilogues */
#define RWKV7_PROF_WKV 4         /* state update + GroupNorm + bonus + output gate */
#define RWKV7_PROF_GEMM_OUT 5    /* output projection + residual */
#define RWKV7_PROF_GEMM_KEY 6    /* channel-mix key + ReLU^2 */
#define RWKV7_PROF_GEMM_VALUE 7  /* channel-mix value (nonzero blocks) + residual */
#define RWKV7_PROF_LN_OUT 8      /* final LayerNorm */
#define RWKV7_PROF_GEMM_HEAD 9   /* head projection to fp32 logits */
#define RWKV7_PROF_SAMPLER 10    /* penalties + sampling */
#define RWKV7_PROF_LORA_FIN 11   /* LoRA-down split sums + tanh / sigmoid to fp16 hidden */
#define RWKV7_PROF_GEMM_FFN 12   /* channel-mix key + ReLU^2 and value + residual in one launch */
#define RWKV7_PROF_CLASSES 13

/* Run one step of B <= min(n_slots, 256) slots with every kernel launched
 * directly (no graph, no dependent-launch overlap) and bracketed by CUDA events
 * on the ctx stream; ms_out[n_classes] receives each class's summed device
 * time and launches_out[n_classes] its launch count.  Synchronous.  The step
 * updates the slots' states like rwkv7_decode_step (logits stay internal). */
RWKV7_API int rwkv7_profile_step(rwkv7_ctx *ctx, const int32_t *d_slots, const int32_t *d_tokens,
                                 int32_t B, int32_t with_sampling, float *ms_out,
                                 int32_t *launches_out, int32_t n_classes);

/* In-graph timeline of one decode step of B <= min(n_slots, 256) slots (with
 * logits, and with sampling if with_sampling != 0), for measurement: the step
 * runs as the same CUDA graph the decode path replays (mode 0; mode 1 launches
 * it directly), every kernel stamping the GPU's global nanosecond timer.  For
 * launch i (in launch order) host_times[4*i .. 4*i+3] receive the earliest CTA
 * start, the earliest and the latest return of a CTA from its wait for the
 * preceding kernel, and the latest CTA end; host_classes[i] its
 * RWKV7_PROF_* class; *n_launches the number of launches (at most
 * max_launches).  The end of launch i minus the end of launch i - 1 is the time
 * that launch adds to the step.  The step is a real step: the slots' states
 * advance.  Synchronous; RWKV7_EINVAL for bad arguments or mode 2. */
RWKV7_API int rwkv7_step_timeline(rwkv7_ctx *ctx, const int32_t *d_slots, const int32_t *d_tokens, int32_t B,
                                  int32_t with_sampling, uint64_t *host_times, int32_t *host_classes,
                                  int32_t max_launches, int32_t *n_launches);

/* Number of kernels one decode step of B slots launches (with / without
 * sampling), for launch accounting.  It depends on B: batches wider than
 * 256 slots run as several fused steps, and where the LoRA-down tiles are k-split
 * a batch wider than half the SMs runs r, k, v and the two LoRA stages as
 * three launches instead of one (with the same results). */
RWKV7_API int32_t rwkv7_step_kernel_count(const rwkv7_ctx *ctx, int32_t B, int32_t with_sampling);

#ifdef __cplusplus
}
#endif
#endif /* RWKV7_H */
