/*
 * llm.h - C ABI of the GB300 batch-1 quantized decode engine (libllm.so).
 *
 * The engine runs the autoregressive decode step of a dense Qwen2/Qwen3-style
 * grouped-query-attention decoder whose seven per-layer projections (q, k, v,
 * o, gate, up, down) hold weight-only quantized codes, on one GPU, replaying
 * the whole step from one CUDA graph.
 *
 * Sources for the operation (page titles and sections):
 *   - "How To Construct Your Personal LLM Runtime From Scratch": §3 (model
 *     dims, GQA 7:1, 16-token bf16/fp16 KV pages, symmetric INT4 group-128
 *     with one scale per group per output row), §4 (packed weight file that is
 *     refused on a wrong magic or layout id), §6 (scalars live in device memory
 *     so a captured graph stays valid as the context grows), §7 (ValueShuffle
 *     nibble order, INT4 decode contract).
 *   - "Bare-Metal LLM Inference on NVIDIA H100", "Architectural Blueprint" and
 *     "Challenge 2" (one graph per step instead of ~280 eager launches).
 *   - "FlashQwen", stages 5-8 (greedy argmax on the GPU returning one int,
 *     single-token decode from a CUDA graph, flash-decoding split-K attention
 *     with a combine pass, INT8 weights with one scale per output row) and the
 *     in-chat /reset command (the KV cache persists until reset).
 *
 * Conventions for every call:
 *   - Return value: LLM_OK (0) or a negative LLM_ERR_* code; nothing throws
 *     across this boundary.  llm_status_str() names a code.
 *   - "device" pointers are CUDA device addresses on the current device;
 *     "host" pointers are ordinary CPU memory.
 *   - Calls on one handle are not thread-safe; use one handle per thread.
 */
#ifndef QD_LLM_H
#define QD_LLM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define LLM_OK 0
#define LLM_ERR_ARG (-1)          /* null/misaligned pointer, unsupported shape or value     */
#define LLM_ERR_LAYOUT (-2)       /* layout_id does not match weight_format (refused load)    */
#define LLM_ERR_CONTEXT_FULL (-3) /* the step would write position >= max_context            */
#define LLM_ERR_CUDA (-4)         /* a CUDA runtime call failed (allocation, launch, copy)    */
#define LLM_ERR_TIMEOUT (-5)      /* a bounded device-side wait gave up (sticky error word)   */
#define LLM_ERR_DEVICE (-6)       /* a device-side check failed (sticky error word)           */
#define LLM_ERR_STATE (-7)        /* call out of order (e.g. llm_logits before any step)      */
#define LLM_ERR_FORMAT (-8)       /* not a model file: wrong magic, version, checksum or size  */
#define LLM_ERR_IO (-9)           /* a model file could not be opened, read or written        */

/* ---- weight formats and packed layouts -------------------------------- */
/* INT4, symmetric, zero point 0, group 128 along K, one bfloat16 scale per
 * (output row, group).  Codes are two's-complement nibbles in [-8, 7].       */
#define LLM_FMT_INT4_G128 1
/* INT8, symmetric, one fp32 scale per output row, codes in [-127, 127].      */
#define LLM_FMT_INT8_ROW 2

/* Layout 1 ("ValueShuffle", the pages' lane map): uint32 words [N][K/8],
 * row-major and K-contiguous; logical code k = 8w + i of a row sits in word w
 * at bit shift {0,16,4,20,8,24,12,28}[i] (even lanes in the low half-word,
 * odd lanes in the high half-word).  Scales: bfloat16 [N][K/128] row-major.
 * llm_pack_int4_g128() writes this layout.                                   */
#define LLM_LAYOUT_INT4_VALUESHUFFLE 1
/* Layout 2: int8 codes [N][K] in natural byte order, row-major; scales fp32 [N]. */
#define LLM_LAYOUT_INT8_ROW 2

/* ---- configuration ----------------------------------------------------- */
typedef struct llm_config {
    int32_t n_layers;   /* decoder layers L                                    */
    int32_t hidden;     /* residual width h (multiple of 128)                  */
    int32_t n_q_heads;  /* query heads Hq                                      */
    int32_t n_kv_heads; /* key/value heads Hkv; Hq % Hkv == 0, Hq/Hkv <= 8      */
    int32_t head_dim;   /* d: 64 or 128                                        */
    int32_t mlp;        /* SwiGLU width F (multiple of 128)                    */
    int32_t vocab;      /* V (multiple of 64)                                  */
    float rms_eps;      /* RMSNorm epsilon                                     */
    float rope_base;    /* RoPE base; theta_i = base^(-2i/d), pairs (i, i+d/2) */
    int32_t qkv_bias;   /* 1: q/k/v projections add a bf16 bias                */
    int32_t qk_norm;    /* 1: per-head RMSNorm of q and k before RoPE (Qwen3)  */
    int32_t tied_lm_head; /* 1: the LM head is the bf16 embedding matrix       */
    int32_t weight_format; /* LLM_FMT_*                                        */
    int32_t layout_id;     /* LLM_LAYOUT_*; must match weight_format           */
    int32_t max_context;   /* KV capacity in tokens (>= 1)                     */
    int32_t page_tokens;   /* tokens per KV page; must be 16                   */
} llm_config;

/* Per-layer weights, all DEVICE pointers, 16-byte aligned, borrowed: the
 * caller keeps them alive and unchanged until llm_destroy().
 *   w*: packed codes in the config's layout; shapes [N][K] with
 *       q: [Hq*d][h], k,v: [Hkv*d][h], o: [h][Hq*d], gate,up: [F][h], down: [h][F]
 *   s*: scales in the config's layout (bf16 [N][K/128] or fp32 [N])
 *   b*: bf16 bias [N] (only read when qkv_bias), else may be NULL
 *   attn_norm, mlp_norm: bf16 [h]; q_norm, k_norm: bf16 [d] (only when qk_norm) */
typedef struct llm_layer_weights {
    const void *wq, *sq, *bq;
    const void *wk, *sk, *bk;
    const void *wv, *sv, *bv;
    const void *wo, *so;
    const void *wg, *sg;
    const void *wu, *su;
    const void *wd, *sd;
    const void *attn_norm, *mlp_norm;
    const void *q_norm, *k_norm;
} llm_layer_weights;

/* Model-level weights (DEVICE pointers, borrowed) plus a HOST array of layers
 * that is copied during llm_create().
 *   embed:      bf16 [V][h]
 *   final_norm: bf16 [h]
 *   lm_head:    bf16 [V][h] (INT4 models, untied); int8 [V][h] with lm_scale
 *               fp32 [V] (INT8 models); ignored when tied_lm_head           */
typedef struct llm_weights {
    const void *embed;
    const void *final_norm;
    const void *lm_head;
    const void *lm_scale;
    const llm_layer_weights *layers;
} llm_weights;

typedef struct llm_t llm_t; /* opaque; owned by the library */

/* Validate the configuration and weights, allocate the paged KV cache (one
 * pool for K and one for V, [L][pages][Hkv][16][d] bf16, sharing one page
 * table), the workspace and the RoPE table, and capture the decode step into
 * one CUDA graph on `cuda_stream` (a cudaStream_t, or NULL for a stream the
 * engine creates).  On success *out owns everything; on error *out is NULL
 * and nothing leaks.  Errors: LLM_ERR_ARG, LLM_ERR_LAYOUT, LLM_ERR_CUDA.     */
int llm_create(const llm_config *cfg, const llm_weights *weights, void *cuda_stream,
               llm_t **out);

/* Run the prompt tokens[0..n-1] (HOST array) at positions seq_len..seq_len+n-1,
 * filling the KV cache, and return the greedy next token in *first_token
 * (HOST).  Blocks until done.  Prompts of 2 or more tokens run as one batch
 * on the tensor cores (llm_set_prefill_batched); the first such call
 * allocates the batch workspace (up to 1024 rows of residual, GEMM-operand,
 * QKV and SwiGLU activations; the GEMMs read the packed weight codes and
 * dequantize them in shared memory, so no weight copy is made).  Errors:
 * LLM_ERR_ARG (n <= 0, token out of range), LLM_ERR_CONTEXT_FULL,
 * LLM_ERR_CUDA, LLM_ERR_TIMEOUT (a bounded wait inside a GEMM ran out),
 * LLM_ERR_DEVICE (a device-side check failed).                              */
int llm_prefill(llm_t *h, const int32_t *tokens, int32_t n, int32_t *first_token);

/* One decode step by graph replay.  The step consumes `forced_input` when it
 * is >= 0 (teacher forcing), else the token the previous step emitted, writes
 * its K/V at position seq_len, and returns the greedy argmax in *out_token
 * (HOST).  Blocks until done.  Errors: LLM_ERR_ARG, LLM_ERR_CONTEXT_FULL
 * (checked before any launch), LLM_ERR_STATE (no previous token), LLM_ERR_CUDA,
 * LLM_ERR_TIMEOUT (a bounded device-side wait ran out: the step's outputs are
 * undefined and the sticky error word stays set until llm_reset),
 * LLM_ERR_DEVICE (a device-side check failed, same rule).                    */
int llm_decode_step(llm_t *h, int32_t forced_input, int32_t *out_token);

/* Enqueue n greedy decode steps (graph replays) on the engine's stream and
 * return without waiting; each step feeds the previous step's argmax.  The
 * emitted tokens stay on the device (llm_sync() then llm_last_token()).     */
int llm_decode_enqueue(llm_t *h, int32_t n);

/* Wait for enqueued work; reports a sticky device error if one was raised.  */
int llm_sync(llm_t *h);

/* Token emitted by the most recent completed step (HOST out).               */
int llm_last_token(llm_t *h, int32_t *token);

/* Copy the fp32 logits [vocab] of the most recent step to host_out.         */
int llm_logits(llm_t *h, float *host_out, int32_t vocab);

/* Number of tokens in the KV cache (the next step's position).              */
int llm_seq_len(llm_t *h, int32_t *seq_len);

/* Forget the sequence: seq_len = 0.  Keeps every allocation and the graph.  */
int llm_reset(llm_t *h);

/* Shorten the sequence to seq_len tokens (0 <= seq_len <= current length);
 * the next step writes position seq_len.  Stream-ordered and asynchronous:
 * it does not wait for enqueued steps.  The last emitted token stays the
 * next input.  Errors: LLM_ERR_ARG, LLM_ERR_CUDA.                           */
int llm_truncate(llm_t *h, int32_t seq_len);

/* Per-region timing of one decode step ("How To Construct Your Personal LLM
 * Runtime From Scratch", §6: the per-token ITL breakdown by region).  Runs
 * one step, advancing the sequence like a greedy step, and writes the
 * duration in ms of region i to kernel_ms[i] (HOST, capacity cap).  Order:
 * for each layer {qkv, attention, o_proj, gate_up, down}, then lm_head;
 * *n_kernels = 5 * n_layers + 1 (with a fused kernel, the first of its
 * regions holds it and the others read 0).  With the persistent step kernel a region is
 * the time between phase starts as seen by CTA 0 (device clock, waits for
 * other CTAs included); with the kernel chain it is one kernel, launched one
 * by one with a CUDA event between neighbours.  Blocks until done.          */
int llm_profile_step(llm_t *h, float *kernel_ms, int32_t cap, int32_t *n_kernels);

/* In-graph timeline of the kernel chain ("How To Construct Your Personal LLM
 * Runtime From Scratch", §6: where the token's time goes, kernel gaps
 * included).  Captures n_steps consecutive greedy steps into one graph whose
 * every launch records, on the device's global timer (ns), the time its last
 * CTA finished, runs it once (advancing the sequence by n_steps, like
 * llm_decode_enqueue) and writes stamps[i * n + j] = finish time of launch j
 * of step i (HOST, capacity cap >= n_steps * (5 * n_layers + 2)); *n_per_step
 * = n, the launches per step.  The launches overlap exactly as in normal
 * replay (programmatic dependent launch included), so stamps[i][j] -
 * stamps[i][j - 1] is launch j's share of the step period and the shares of a
 * step sum to its period.  Blocks until done.  Errors: LLM_ERR_ARG (persistent
 * step on, cap too small), LLM_ERR_STATE (no token to feed),
 * LLM_ERR_CONTEXT_FULL, LLM_ERR_CUDA.                                       */
int llm_timeline_steps(llm_t *h, int32_t n_steps, uint64_t *stamps, int32_t cap, int32_t *n_per_step);

/* ---- Multi-sequence decode ------------------------------------------------
 * Up to 8 sequences decoding together on one GPU ("Systems Foundations for
 * LLMs", PagedAttention and its block manager): one K/V pool of 16-token pages
 * shared by all sequences, a page table per sequence filled on demand from a
 * free list (page 0 is reserved), and steps in which every weight is read once
 * for all the sequences taking part (their linear layers run as skinny GEMMs on
 * the tensor cores, mma.sync with bf16 operands and fp32 accumulation; attention
 * runs per sequence through its own page table).  Each step is one CUDA graph
 * replay.  Weights: as for llm_create (borrowed, same layouts). */
typedef struct llm_batch_t llm_batch_t; /* opaque; owned by the library */

/* max_seqs: sequence slots (1..8); n_pages: pages in the shared pool including
 * the reserved one (0 = max_seqs * ceil(max_context / 16) + 1).  Validation and
 * errors as for llm_create. */
int llm_batch_create(const llm_config *cfg, const llm_weights *weights, int32_t max_seqs, int32_t n_pages,
                     void *cuda_stream, llm_batch_t **out);
void llm_batch_destroy(llm_batch_t *h);

/* A new, empty sequence in a free slot -> *seq.  LLM_ERR_STATE: all slots hold one. */
int llm_batch_add(llm_batch_t *h, int32_t *seq);

/* End a sequence: its pages go back to the free list, its slot becomes free.  */
int llm_batch_release(llm_batch_t *h, int32_t seq);

/* One decode step for the n sequences seqs[0..n-1] (distinct, live): each
 * consumes inputs[i] when inputs is non-NULL and inputs[i] >= 0, else the token
 * its previous step emitted; each writes its K/V at its current length (a new
 * page is taken from the free list whenever the length crosses a page
 * boundary) and emits its greedy argmax into out_tokens[i] (HOST; may be NULL).
 * The other slots keep their caches and lengths.  Blocks until done.  Errors:
 * LLM_ERR_ARG, LLM_ERR_STATE (a sequence with nothing to feed),
 * LLM_ERR_CONTEXT_FULL (a sequence at max_context, or the free list cannot
 * cover the step: checked before any work), LLM_ERR_CUDA, LLM_ERR_DEVICE /
 * LLM_ERR_TIMEOUT (a device-side check of a sequence in the step).          */
int llm_batch_step(llm_batch_t *h, const int32_t *seqs, const int32_t *inputs, int32_t n, int32_t *out_tokens);

/* Feed a prompt to one sequence, token by token through the batched step (the
 * other sequences do not move); *first_token = the greedy token after it.    */
int llm_batch_prefill(llm_batch_t *h, int32_t seq, const int32_t *tokens, int32_t n, int32_t *first_token);

/* fp32 logits [vocab] of the sequence's last step (HOST).                    */
int llm_batch_logits(llm_batch_t *h, int32_t seq, float *host_out, int32_t vocab);

/* A sequence's length, its physical pages in logical order (HOST, capacity
 * cap; may be NULL), their count, and the pages left on the free list.       */
int llm_batch_seq_info(llm_batch_t *h, int32_t seq, int32_t *len, int32_t *pages, int32_t cap,
                       int32_t *n_pages, int32_t *free_pages);

/* Test hook: the order in which the free list hands out pages 1..n_pages-1
 * (order[0] first); only while no slot holds a sequence.                     */
int llm_batch_set_page_order(llm_batch_t *h, const int32_t *order, int32_t n);

/* Test hook: the K and V pools ([L][n_pages][Hkv][16][d] bf16, device).       */
int llm_batch_debug_kv(llm_batch_t *h, void **k_pool, void **v_pool, int32_t *n_pages);

/* Free everything the handle owns (not the caller's weights).  NULL is a no-op. */
void llm_destroy(llm_t *h);

/* Static string naming a status code. */
const char *llm_status_str(int status);

/* Identity of the build: the first 16 hex digits of a SHA-256 over the
 * library's sources, these headers and its compile flags (no counterpart in
 * the source pages; the Python package refuses a library whose id does not
 * match the sources next to it).  Static string, never NULL.                 */
const char *llm_build_id(void);

/* Test and benchmark hook: DEVICE pointers to the KV pools ([L][pages][Hkv][16][d]
 * bf16) and the page table (int32 [pages], logical page -> physical page,
 * identity after create) so a caller can fill or shuffle them, and the number
 * of pages.  When set_len >= 0 the sequence length becomes set_len (the caller
 * promises positions 0..set_len-1 hold valid K/V).  Any out-param may be NULL. */
int llm_debug_kv(llm_t *h, void **k_pool, void **v_pool, int32_t **page_table,
                 int32_t *n_pages, int32_t set_len);

/* Execution mode for llm_decode_step / llm_prefill: 1 = replay the captured
 * graph (default), 0 = launch the same kernels one by one (eager), for timing
 * the difference.                                                           */
int llm_set_graph_mode(llm_t *h, int32_t use_graph);

/* 1: the whole step is one persistent kernel, one CTA per SM, weights
 * streamed by TMA through a shared-memory ring, the phases of a layer ordered
 * by device counters (available where the model's shapes fit it).  0
 * (default): the step is a chain of 5 * n_layers + 1 kernels.  Re-captures the graph; waits for enqueued work
 * first.  Errors: LLM_ERR_ARG (null handle, or 1 for a model outside the
 * persistent kernel's shapes), LLM_ERR_CUDA.                                */
int llm_set_persistent(llm_t *h, int32_t on);

/* 1: the MLP block of a layer -- RMSNorm, gate/up, SiLU * mul
 * and down ("从头开始手写一个Qwen的Naive CUDA Kernel推理引擎(一)", "SwiGLU") --
 * runs as one kernel in which every CTA multiplies its slice of the hidden
 * units by the matching columns of W_down (repacked by llm_create into an
 * engine-owned copy, mlp * hidden / 2 bytes per layer for INT4) and adds the
 * partial sums into a residual buffer with integer reductions in L2 (64-bit
 * fixed point, 2^-32 units: exact, so results do not depend on the order of
 * the CTAs; |values| must stay below 2^31).  Shapes: hidden % 256 == 0,
 * hidden <= 4096, mlp % 128 == 0.  On by default where it fits and hidden <=
 * 2048 (measured faster there); 0: the block is two GEMV kernels (gate/up,
 * then down).
 * With int8 activations (llm_set_act_int8) the two kernels always run.
 * Re-captures the graph.  Errors: LLM_ERR_ARG (null handle, or 1 for shapes
 * the kernel does not take), LLM_ERR_CUDA.                                  */
int llm_set_fused_mlp(llm_t *h, int32_t on);

/* o_proj folded into the decode attention: where the attention runs as one
 * cluster per KV head (INT4 weights, head_dim 128), that cluster multiplies
 * its heads' outputs by its columns of W_o (copied into shared memory while
 * the cluster merges its split-K partials) and adds each row's partial sum
 * into an engine-owned buffer with 64-bit fixed-point reductions in L2
 * (2^-32 units, exact, independent of the order of the CTAs); the gate/up
 * GEMV adds that buffer to the residual before its RMSNorm and the down GEMV
 * folds it into the residual and zeroes it.  The o_proj kernel is then not
 * launched.  1: on; 0 (default): o_proj as its own GEMV.  Not with the fused
 * MLP block, the fused QKV + attention kernel or int8 activations (those
 * steps keep the o_proj GEMV).  Re-captures the graph.  Errors: LLM_ERR_ARG
 * (null handle, or 1 where the attention plan or shapes do not allow it),
 * LLM_ERR_CUDA.                                                             */
int llm_set_o_fold(llm_t *h, int32_t on);
/* The current llm_set_o_fold setting in *on (1 or 0).  LLM_ERR_ARG on null.  */
int llm_get_o_fold(llm_t *h, int32_t *on);

/* Launch kinds of a decode step, in launch order (the step as last captured):
 * writes kinds[i] for each launch (HOST, capacity cap) and *n = launches; 0
 * for the persistent kernel.  Kinds: */
#define LLM_KIND_QKV 0
#define LLM_KIND_ATTENTION 1
#define LLM_KIND_O_PROJ 2
#define LLM_KIND_GATE_UP 3
#define LLM_KIND_DOWN 4
#define LLM_KIND_LM_HEAD 5
#define LLM_KIND_SAMPLER 6
#define LLM_KIND_QKV_ATTENTION 7
#define LLM_KIND_MLP 8
int llm_step_kinds(llm_t *h, int32_t *kinds, int32_t cap, int32_t *n);

/* L2 staging of weights ahead of the kernel that reads them: kernels of the
 * chain issue bulk L2 prefetches (cp.async.bulk.prefetch.L2, by the TMA
 * engine) of a later kernel's weights at their start, so that HBM streams
 * while the latency-bound kernels of the attention block run.  Flags (OR):
 * 1 = QKV prefetches the layer's gate/up weights, 2 = gate/up prefetches the
 * layer's down weights, 4 = down prefetches the next layer's QKV and o_proj
 * codes, 8 = QKV prefetches the layer's o_proj weights (without 1),
 * 16 = o_proj prefetches the layer's gate/up weights; 0 = off.  Results are
 * unchanged (prefetches only move data into L2).  Re-captures the graph.
 * Errors: LLM_ERR_ARG (null handle, flags outside 0..31), LLM_ERR_CUDA.      */
int llm_set_l2_prefetch(llm_t *h, int32_t flags);

/* Test hook of the persistent kernel's failure path: its phase-counter waits
 * expect `extra_arrivals` (0 or 1) arrivals more than any step delivers and
 * give up after counter_wait_ns (1 us .. 1 s; default 1 s).  With 1, every
 * step run as the persistent kernel ends by that bounded wait: the kernel
 * records the timeout in the sticky error word, stops issuing copies, waits
 * (with the normal 1 s bound) for the copies it has in flight, and returns;
 * llm_decode_step then returns LLM_ERR_TIMEOUT, and llm_reset makes the engine
 * usable again.  No GPU fault or hang is involved.  Re-captures the graph when
 * the persistent kernel is on.  Errors: LLM_ERR_ARG (null handle, a model
 * outside the persistent kernel's shapes, values out of range), LLM_ERR_CUDA. */
int llm_debug_step_wait(llm_t *h, int32_t extra_arrivals, int64_t counter_wait_ns);

/* Prefill mode for prompts of 2 or more tokens.  1 (default where the model's
 * shapes allow it): the prompt runs as a batch -- per layer RMSNorm, weight
 * matrices dequantized to fp16 and multiplied on the tcgen05 tensor cores
 * (fp32 accumulate), causal attention over the paged cache, and the LM head on
 * the last row only ("Bare-Metal LLM Inference on NVIDIA H100": prefill is a
 * compute-bound GEMM phase).  0: the prompt is fed through the decode step one
 * token at a time.  Both give the same cache and first token within the
 * acceptance tolerance.  Errors: LLM_ERR_ARG (null handle, or 1 for a model
 * whose shapes the batched path does not take: (Hq + 2 Hkv) d and hidden must
 * be multiples of 128, mlp of 64).                                          */
int llm_set_prefill_batched(llm_t *h, int32_t on);

/* 1 (default): consecutive kernels of the step are launched with programmatic
 * dependent launch (a kernel's CTAs may start before the previous kernel ends,
 * issue their first weight copies and wait for it on the device); 0: plain
 * stream order.  Re-captures the graph; waits for enqueued work first.
 * Errors: LLM_ERR_ARG, LLM_ERR_CUDA.                                         */
int llm_set_pdl(llm_t *h, int32_t use_pdl);

/* 1 (where the model fits it: head_dim 128, no per-head q/k norms, one 16-CTA
 * cluster per KV head resident at once, context up to 8K tokens): the QKV
 * projection and the attention of a layer run as one kernel -- the
 * cluster of a KV head computes the group's projection rows, exchanges them
 * through distributed shared memory and attends over its pages, whose copies
 * started before the projection.  The step is then 4 * n_layers + 1 kernels;
 * llm_profile_step reports the fused kernel in each layer's QKV entry and 0 in
 * its attention entry.  0 (default; the fused kernel measured slower at the 7B
 * shape): separate QKV and attention kernels.  Results agree
 * within rounding (the projection's K parts are summed in another order).
 * Re-captures the graph; waits for enqueued work first.  Errors: LLM_ERR_ARG
 * (null handle, or 1 for a model outside the fused kernel), LLM_ERR_CUDA.    */
int llm_set_fused_attention(llm_t *h, int32_t on);

/* 1: the o_proj, gate/up and down GEMVs of the decode step (INT4 models) run
 * on activations quantized to int8 per group of 128 inside each GEMV's
 * staging (scale = absmax / 127, round half to even) with __dp4a products
 * ("How To Construct Your Personal LLM Runtime From Scratch", §7, Path A;
 * llm_op_gemv_int4_a8 gives the exact definition).  The QKV projection,
 * the LM head and the batched prefill keep their activations.  0 (default):
 * fp16 activations.  The logits change by the activation rounding (within
 * the acceptance tolerance on the test models).  Not with the persistent
 * step.  Re-captures the graph; waits for enqueued work first.  Errors:
 * LLM_ERR_ARG (null handle, INT8 model, persistent step, or shapes outside
 * the GEMV), LLM_ERR_CUDA.                                                  */
int llm_set_act_int8(llm_t *h, int32_t on);

/* How each step (and the batched prefill) picks the next token.  temperature
 * <= 0 (default): greedy argmax, lowest index on ties ("FlashQwen", "Stage 5 -
 * GPU argmax for greedy").  Otherwise sampling on the GPU ("FlashQwen" run
 * options --temperature / --top-k / --top-p, Qwen's recommended 0.6 / 20 /
 * 0.95; naive Qwen engine, "Sampler"): the top_k largest logits (lowest index
 * on ties), weights exp((l - l_max) / temperature), the smallest prefix of
 * them in decreasing order whose weight reaches top_p of their sum, and the
 * first token of that prefix whose running weight exceeds u times the
 * prefix's weight, with u uniform in [0, 1) from SplitMix64 started at
 * mix(seed), draw number = the position whose logits are sampled (so a step
 * at a given position draws the same u after llm_reset or llm_truncate).
 * One extra kernel after the LM head; llm_profile_step counts it in the LM
 * head's entry.  1 <= top_k <= min(vocab, 1024), 0 < top_p <= 1.  Not with
 * the persistent step.  Re-captures the graph; waits for enqueued work first.
 * Errors: LLM_ERR_ARG, LLM_ERR_CUDA.                                          */
int llm_set_sampling(llm_t *h, float temperature, int32_t top_k, float top_p, uint64_t seed);

/* ---- offline packer (host memory, no GPU needed) ----------------------- */

/* Pack logical INT4 codes (int8 [N][K], values in [-8, 7], K % 128 == 0) into
 * layout LLM_LAYOUT_INT4_VALUESHUFFLE words [N][K/8].  Returns LLM_ERR_ARG on
 * a null pointer, a bad shape or a code outside [-8, 7].                     */
int llm_pack_int4_g128(const int8_t *codes, int64_t N, int64_t K, uint32_t *words);

/* Layout LLM_LAYOUT_INT8_ROW keeps codes in natural order: this copies and
 * checks the range [-127, 127].                                              */
int llm_pack_int8_row(const int8_t *codes, int64_t N, int64_t K, int8_t *out);

/* ---- quantizers (host memory, no GPU needed) --------------------------- */

/* Symmetric INT4, zero point 0, group 128 along K ("How To Construct Your
 * Personal LLM Runtime From Scratch", §3): for each (row, group) the scale is
 * absmax / 7 in fp32, stored as bfloat16 (round to nearest even); each code is
 * the fp32 quotient w / scale (the stored scale) rounded half to even and
 * clamped to [-8, 7]; an all-zero group gets scale 0 and codes 0.
 * w: fp32 [N][K] (HOST), K % 128 == 0; codes: int8 [N][K]; scales: bf16 bits
 * [N][K/128].  Returns LLM_ERR_ARG on a null pointer, a bad shape or a
 * non-finite weight.  Feed the codes to llm_pack_int4_g128().               */
int llm_quantize_int4_g128(const float *w, int64_t N, int64_t K, int8_t *codes, uint16_t *scales);

/* Symmetric INT8 with one fp32 scale per output row ("FlashQwen", Stage 8):
 * scale = absmax / 127 in fp32; code = w / scale rounded half to even,
 * clamped to [-127, 127]; a zero row gets scale 0 and codes 0.
 * w: fp32 [N][K] (HOST); codes: int8 [N][K]; scales: fp32 [N].             */
int llm_quantize_int8_row(const float *w, int64_t N, int64_t K, int8_t *codes, float *scales);

/* ---- model file ---------------------------------------------------------- */
/* One binary file holds a packed model ("How To Construct Your Personal LLM
 * Runtime From Scratch", §3-§4: one mmap-able file, a 256-byte header opening
 * with an 8-byte magic, payloads on 128-byte boundaries, refused on a wrong
 * magic or layout id before any weight is uploaded):
 *   bytes 0-7 the magic "QDECODEW"; 8-11 version 1; 12-15 header size 256;
 *   16-79 the llm_config (16 little-endian 4-byte fields in declaration
 *   order); 80-87 payload offset 256; 88-95 payload bytes; 96-103 FNV-1a 64
 *   of bytes 0-95; zeros to byte 256.  Then each tensor on the next 128-byte
 *   boundary, in this order, with the sizes llm_create() documents: embed,
 *   final_norm, [lm_head (bf16, INT4 models; int8, INT8 models), [lm_scale
 *   (INT8 models)]] unless tied_lm_head, then per layer wq sq [bq] wk sk [bk]
 *   wv sv [bv] wo so wg sg wu su wd sd attn_norm mlp_norm [q_norm k_norm]
 *   (brackets: only with qkv_bias, resp. qk_norm).  Padding bytes are zero. */

/* Size in bytes of the file for this configuration.  Errors: LLM_ERR_ARG.   */
int llm_model_file_bytes(const llm_config *cfg, int64_t *bytes);

/* Write the model to `path` (created or truncated).  host_weights: the same
 * fields as for llm_create() but HOST pointers, in the config's packed layout
 * (llm_pack_int4_g128 / llm_pack_int8_row output and their scales); read
 * only during the call.  Errors: LLM_ERR_ARG (null or missing tensor, bad
 * shape), LLM_ERR_LAYOUT (layout_id does not match weight_format), LLM_ERR_IO. */
int llm_model_file_write(const char *path, const llm_config *cfg, const llm_weights *host_weights);

/* Read and check a file's header into *cfg_out (no weights are read).
 * Errors: LLM_ERR_IO (cannot open), LLM_ERR_FORMAT (wrong magic, version or
 * checksum, impossible shape, size that does not match the configuration or
 * a truncated file), LLM_ERR_LAYOUT (layout_id does not match the format).  */
int llm_model_file_read_config(const char *path, llm_config *cfg_out);

/* Check the file as llm_model_file_read_config() does, copy its payload to
 * one device allocation (read in 64 MB chunks), and llm_create() an engine
 * on those weights; the handle owns the allocation and llm_destroy() frees
 * it.  max_context > 0 replaces the file's max_context; 0 keeps it.  On error
 * *out is NULL and nothing leaks.  Errors: those of
 * llm_model_file_read_config(), LLM_ERR_CUDA, and those of llm_create().    */
int llm_create_from_file(const char *path, int32_t max_context, void *cuda_stream, llm_t **out);

#ifdef __cplusplus
}
#endif
#endif /* QD_LLM_H */
