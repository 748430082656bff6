/*
 * gpt.h — C ABI of the persistent GPT training-step library (libgpt.so).
 *
 * One call of gpt_train_step runs one full training step of a GPT language
 * model — token/position embedding, pre-LN transformer blocks (causal
 * multi-head attention, GELU MLP), final LayerNorm, LM head, mean softmax
 * cross-entropy, the backward pass and an AdamW update of every parameter — as
 * ONE persistent CUDA kernel launch.  Inside that launch resident thread blocks
 * claim tasks (GEMM tiles, attention blocks, row blocks, optimizer chunks) from
 * a ticket counter and order dependent tasks with release/acquire completion
 * counters, so the host launches nothing between the operations of a step.
 *
 * Sources of the method (web pages; cited by title and section):
 *  - "Open Flapping Airplanes" experiment record (A100 reproduction), section
 *    "What ran": one persistent kernel whose resident blocks repeatedly take
 *    tasks from a scheduler; the training role runs "forward pass, backward
 *    pass, and weight updates" of a 12-layer, width-768, 12-head GPT on 8 x 512
 *    tokens a step with AdamW from seeded initial weights.  Section "A longer
 *    run exposed a scheduler overflow": a task budget computed as a 32-bit
 *    product wrapped; every counter here is 64-bit.
 *  - "How one persistent kernel runs three jobs" (review): training claims
 *    tasks through ticket counters; completed phases publish their writes with
 *    a memory fence before incrementing counters, dependents use acquire reads
 *    and wait; forward releases backward without host launches.
 *  - "Coppelius training on the RTX 3090": loss = mean cross-entropy over the
 *    step's rows (figure "Loss"); per-invocation exit status, error notifier and
 *    finite-loss check (section "Channel health"); checkpoints (section
 *    "Checkpoint lineage").
 *
 * Conventions for every function:
 *  - Return 0 on success or a negative GPT_ERR_* code; gpt_last_error() gives
 *    the text of the handle's last error.  No C++ exception crosses the ABI.
 *  - A handle is not thread-safe: one host thread at a time.
 *  - "device" pointers are CUDA device addresses on the handle's device;
 *    "host" pointers are ordinary host memory (pageable or pinned).  The caller
 *    owns every buffer it passes; the library never frees or retains them past
 *    the call.
 *  - Flat parameter-sized vectors use the canonical order: wte [V,C], wpe [T,C],
 *    then per layer ln1_g, ln1_b, w_qkv [3C,C], b_qkv [3C], w_o [C,C], b_o [C],
 *    ln2_g, ln2_b, w_1 [F,C], b_1 [F], w_2 [C,F], b_2 [C]; then lnf_g, lnf_b,
 *    w_lm [V,C] (biases present only when the config enables them).  Matrices
 *    are row-major [out_features, in_features]; y = x W^T + b.
 */
#ifndef GPT_H_
#define GPT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define GPT_OK               0
#define GPT_ERR_INVALID_ARG (-1)  /* bad config, pointer, size or index            */
#define GPT_ERR_CUDA        (-2)  /* a CUDA runtime/driver call failed              */
#define GPT_ERR_OOM         (-3)  /* device or host allocation failed               */
#define GPT_ERR_TIMEOUT     (-4)  /* a device wait gave up; the handle is poisoned  */
#define GPT_ERR_NONFINITE   (-5)  /* the step's loss is NaN or infinite             */
#define GPT_ERR_BAD_TOKEN   (-6)  /* a token or target id outside [0, vocab)        */
#define GPT_ERR_POISONED    (-7)  /* an earlier timeout left the handle unusable    */
#define GPT_ERR_UNSUPPORTED (-8)  /* shape not supported by the compiled kernels    */

/* Arithmetic of a handle. */
#define GPT_DTYPE_FP32 0  /* every tensor and every operation in fp32 (SIMT)          */
#define GPT_DTYPE_BF16 1  /* bf16 GEMM/attention operands and stored activations,
                             fp32 accumulation, statistics, residual stream, grads,
                             master weights and AdamW moments                       */

/*
 * Model and optimizer configuration.  Architecture: "What ran" (model shape);
 * the choices the pages leave open are fields here with these defaults:
 * linear_bias 1 (biases on QKV, attention-out and both MLP linears; never on
 * the LM head), ln_bias 1, tie_embeddings 0 (the only value supported),
 * gelu_tanh 1 (tanh approximation; 0 = erf form), eps 1e-8, ln_eps 1e-5,
 * wd_on_1d 0 (weight decay on 2-D tensors only), constant learning rate.
 * Limits: d_model a multiple of 64 and <= 1024, d_mlp a multiple of 64,
 * head_dim = d_model / n_head <= 128, seq_len <= 1024, batch*seq_len <= 8192;
 * for GPT_DTYPE_BF16 also head_dim == 64, seq_len a multiple of 128, vocab a
 * multiple of 64 and batch*seq_len a multiple of 128.
 */
typedef struct gpt_config {
  int32_t n_layer, d_model, n_head, d_mlp, vocab, seq_len, batch;
  int32_t dtype;             /* GPT_DTYPE_FP32 or GPT_DTYPE_BF16                    */
  int32_t linear_bias, ln_bias, tie_embeddings, gelu_tanh;
  float   lr, beta1, beta2, eps, weight_decay, ln_eps;
  int32_t wd_on_1d;
  uint32_t wait_timeout_ms;  /* bound of every in-kernel wait; 0 = default 2000 ms  */
  int32_t deterministic;     /* accepted for compatibility: every reduction of this
                                library has a fixed order, so steps are always
                                bitwise repeatable                                  */
  /* Model variant of the RTX 3090 page's 57.7M model (bf16 only; "Coppelius
   * training on the RTX 3090": RoPE on q/k, gated-GELU FFN, tied embedding):
   *   rope: rotate pairs (2i, 2i+1) of every head's q and k by t * 10000^(-2i/64)
   *     at position t; no learned position table;
   *   gated_mlp: the first MLP matrix is w_gu [2F, C] (rows 2f, 2f+1 = gate and
   *     up of feature f), the MLP output GELU(gate) * up (needs linear_bias 0);
   *   tie_embeddings (above): the LM head is wte.                               */
  int32_t rope, gated_mlp;
} gpt_config;

typedef struct gpt gpt;  /* opaque handle; owns every device buffer it allocates */

/* Fills *cfg with the defaults above for the 162M model (12L/768/12H, F 3072,
 * V 50304, T 512, B 8, bf16, lr 6e-4, betas 0.9/0.95, wd 0.1). */
void gpt_default_config(gpt_config* cfg);

/* Bytes of device memory a handle with this config needs (its arena). 0 on an
 * invalid config. */
size_t gpt_arena_bytes(const gpt_config* cfg);

/* Host-only: number of parameters of a model with this config (the length of
 * every flat parameter-sized vector; "What ran" prints the 162M model's count).
 * 0 on an invalid config.  Needs no GPU. */
size_t gpt_param_count(const gpt_config* cfg);

/*
 * Creates a handle on the current CUDA device.  Weights are initialised on the
 * host from `seed` ("What ran": seeded initial weights; "Reproduce the run":
 * initial weights generated on the CPU): matrices and embeddings N(0, 0.02)
 * drawn from SplitMix64 + Box-Muller per the specification in the package's
 * inputs module, biases and LayerNorm biases 0, LayerNorm gains 1; AdamW
 * moments 0, step count 0.
 *   cuda_stream: cudaStream_t the handle launches on (NULL = legacy default).
 *   arena/arena_bytes: optional caller-owned device allocation of at least
 *     gpt_arena_bytes(cfg) bytes, 256-byte aligned, that must outlive the
 *     handle; NULL/0 = the library allocates (and frees) its own.
 *   out: receives the handle; unchanged on failure.
 * Errors: INVALID_ARG (bad config, NULL out, arena too small or misaligned),
 * UNSUPPORTED, OOM, CUDA.
 */
int gpt_create(const gpt_config* cfg, uint64_t seed, void* cuda_stream,
               void* arena, size_t arena_bytes, gpt** out);

/*
 * One training step: forward, backward and AdamW, as one persistent kernel
 * launch on the handle's stream; returns after the step completed (the call
 * synchronises the stream).
 *   tokens, targets: DEVICE int32 [batch, seq_len], row-major, ids in
 *     [0, vocab); targets[b,t] is the id that should follow tokens[b,t].
 *   loss: HOST float*, receives the mean cross-entropy of this step's forward
 *     pass (before the update).  May be NULL.
 * Errors: INVALID_ARG (NULL tokens/targets), BAD_TOKEN, NONFINITE, TIMEOUT
 * (handle poisoned), POISONED, CUDA.  On BAD_TOKEN (out-of-range ids are
 * clamped for the computation) and NONFINITE the launch still runs to its
 * end, but every AdamW task sees the flag and skips its update: parameters,
 * moments and the step count are left as they were before the call.
 */
int gpt_train_step(gpt* h, const int32_t* tokens, const int32_t* targets, float* loss);

/*
 * Same step with HOST token/target buffers: the call copies them to the
 * handle's device staging buffers on its stream, runs the step and reads the
 * loss back.  tokens/targets: HOST int32 [batch, seq_len].
 */
int gpt_train_step_host(gpt* h, const int32_t* tokens, const int32_t* targets, float* loss);

/*
 * Learning-rate schedule of a multi-step call.  The record mentions a 4,000-step
 * learning-rate schedule without giving its form ("Open Flapping Airplanes"
 * record, section "Reproducibility needs inputs and an environment record"); the
 * reading implemented is linear warmup then cosine decay:
 *   kind GPT_LR_CONSTANT: every update uses cfg.lr;
 *   kind GPT_LR_WARMUP_COSINE: update t (1-based count of applied updates) uses
 *     lr_max * t / warmup_steps              for t <= warmup_steps,
 *     lr_min + (lr_max - lr_min) (1 + cos(pi (t - warmup_steps) /
 *                                   (total_steps - warmup_steps))) / 2   up to total_steps,
 *     lr_min                                 after total_steps.
 */
enum { GPT_LR_CONSTANT = 0, GPT_LR_WARMUP_COSINE = 1 };
typedef struct {
  int32_t kind;
  int32_t warmup_steps;  /* >= 0 */
  int64_t total_steps;   /* > warmup_steps */
  float lr_max, lr_min;  /* lr_max >= lr_min >= 0 */
} gpt_lr_schedule;

/*
 * Host-only: the rate sched gives update number step (>= 1); base_lr is used
 * for GPT_LR_CONSTANT.  Returns a negative value for an invalid schedule.
 */
float gpt_lr_at(const gpt_lr_schedule* sched, float base_lr, int64_t step);

/*
 * k training steps in one call ("K steps per launch": the "Open Flapping
 * Airplanes" record times its whole run inside one kernel interval, section
 * "Measured results"): step j reads DEVICE tokens + j*batch*seq_len and targets
 * + j*batch*seq_len (int32 [k, batch, seq_len], row-major, caller-owned, valid
 * until the call returns) and updates with the rate sched gives its update
 * number (NULL: cfg.lr).  Up to 256 steps run inside ONE launch of the
 * persistent kernel: after each step every block passes a grid barrier (a
 * device counter, bounded wait) and starts the next step with the next epoch,
 * its rate and bias corrections taken from a device table the call uploads
 * first; each step writes its loss and status into a device ring that the host
 * reads once per launch.  Longer calls use one launch per 256 steps.
 * losses: HOST float[k] (may be NULL) receives every step's pre-update loss.
 * Errors as gpt_train_step; on BAD_TOKEN or NONFINITE at step j the steps
 * before j are applied, step j and every later step of the call leave
 * parameters, moments and the step count unchanged (their losses are still
 * computed and returned), and gpt_last_error names j.
 */
int gpt_train_steps(gpt* h, const int32_t* tokens, const int32_t* targets, int32_t k,
                    const gpt_lr_schedule* sched, float* losses);

/* Number of parameters (length of every flat parameter-sized vector): the
 * count "What ran" prints for its model (162,417,408; this library's 162M model
 * keeps linear and LayerNorm biases and has 162,716,160).  0 for a NULL handle. */
size_t gpt_num_params(const gpt* h);

/* Number of tensors in the canonical order (the model of "What ran": token and
 * position embeddings, per layer two LayerNorms, QKV, attention-out and two MLP
 * linears, the final LayerNorm and the LM head).  0 for a NULL handle. */
int gpt_num_tensors(const gpt* h);

/*
 * Describes tensor i of the canonical order: *name (static storage of the
 * handle), shape[0..1] (shape[1] = 1 for vectors) and *offset (element offset
 * in the flat vector).  Any output pointer may be NULL.  INVALID_ARG if i is
 * out of range.
 */
int gpt_tensor_info(const gpt* h, int i, const char** name, int64_t shape[2], size_t* offset);

/* Copies the fp32 master parameters to HOST dst[0..n), n == gpt_num_params:
 * the parameter half of a checkpoint ("Coppelius training on the RTX 3090",
 * section "Checkpoint lineage": each invocation resumes the checkpoint the one
 * before wrote).  Synchronises the handle's stream.  INVALID_ARG for a NULL
 * handle or dst or a wrong n; CUDA if the copy fails. */
int gpt_get_params(gpt* h, float* dst, size_t n);

/* Overwrites the fp32 master parameters (and the bf16 copies the kernels read)
 * from HOST src[0..n), n == gpt_num_params: resuming a checkpoint ("Checkpoint
 * lineage", as above).  Optimizer state is unchanged.  The values are not
 * checked: a non-finite parameter makes the next step's loss non-finite, and
 * that step returns NONFINITE without updating anything.  INVALID_ARG for a
 * NULL handle or src or a wrong n; CUDA if the copy fails. */
int gpt_set_params(gpt* h, const float* src, size_t n);

/* Copies the gradient computed by the last step (fp32, canonical order) to
 * HOST dst[0..n), n == gpt_num_params ("Coppelius training on the RTX 3090",
 * section "Optimizer internals": the last step's embedding gradient is
 * inspected after each invocation; here every tensor's is available, for
 * parity checks).  Also valid after a BAD_TOKEN or NONFINITE step.  INVALID_ARG
 * for a NULL handle or dst or a wrong n; CUDA if the copy fails. */
int gpt_get_grads(gpt* h, float* dst, size_t n);

/* AdamW state: first and second moments (HOST float[gpt_num_params] each,
 * either may be NULL) and the number of updates applied so far (bias
 * correction of the next update uses step + 1).  The optimizer half of a
 * checkpoint ("Checkpoint lineage"; "Optimizer internals": AdamW's first moment
 * after each invocation).  INVALID_ARG for a NULL handle, a NULL step pointer
 * (get) or a negative step (set); CUDA if a copy fails. */
int gpt_get_opt_state(gpt* h, float* m, float* v, int64_t* step);
int gpt_set_opt_state(gpt* h, const float* m, const float* v, int64_t step);

/*
 * Test hook: gpt_debug_skip_release(h, k) makes the next step's task number k
 * (ticket order) skip its completion release, so that its dependents' bounded
 * waits expire and the step returns GPT_ERR_TIMEOUT without hanging; -1 turns
 * it off.  After such a timeout gpt_reset() clears the poisoned state.
 */
int gpt_debug_skip_release(gpt* h, int64_t task_index);

/* Clears counters, the ticket and the error word after a timeout; parameters
 * and optimizer state are kept. */
int gpt_reset(gpt* h);

/*
 * Serving partition: greedy generation (batch 1) from the live weights on a
 * reserved set of blocks of the persistent kernel, next to the training step
 * ("Open Flapping Airplanes" record, section "What ran": 17 of the A100's SMs
 * serve "autoregressive text generation from the changing model"; "How one
 * persistent kernel runs three jobs": static block roles, serving claims tasks
 * through its own ticket counter, one token releases the next).  A decode step
 * takes the token at position s (the prompt, then the generated ones) through
 * the model with the keys and values of positions < s kept in an fp32 cache,
 * and the next token is the argmax of its logits (the smallest id among equal
 * logits); activations are fp32, weights the bf16 copy that training updates.
 * bf16 model with learned positions, a GELU MLP and an untied LM head only
 * (UNSUPPORTED otherwise).  The step's ticket and every counter are 64-bit ("A
 * longer run exposed a scheduler overflow": a task budget of 4,194,304 x 2,225
 * wrapped at 32 bits); first_step starts the session's counters as if that many
 * steps had run before (a boundary test of the budget), 0 normally.
 *
 * gpt_serve_begin: HOST prompt[n_prompt] (ids in [0, vocab)), max_new >= 1 new
 *   tokens, n_prompt + max_new <= seq_len; `blocks` (1 .. grid-1) blocks serve
 *   during every later training launch, each of which runs up to
 *   tokens_per_step decode steps per training step (0: serve only in
 *   gpt_serve_run).  Allocates the session's device state (about 2 x layers x
 *   seq_len x d_model fp32 of cache); an earlier session is ended first.
 *   Errors: INVALID_ARG, BAD_TOKEN, UNSUPPORTED, OOM, CUDA.
 * gpt_serve_run: a launch in which only the serving blocks work (no training
 *   step, no epoch consumed) for up to max_steps decode steps; kernel_ms (HOST,
 *   may be NULL) receives its device time.  Errors: INVALID_ARG, POISONED,
 *   TIMEOUT, CUDA.
 * gpt_serve_tokens: the tokens generated so far (*n of them; the first
 *   min(*n, cap) are copied to HOST dst, which may be NULL).
 * gpt_serve_end: frees the session (no-op without one).
 */
int gpt_serve_begin(gpt* h, const int32_t* prompt, int32_t n_prompt, int32_t max_new, int32_t blocks,
                    int32_t tokens_per_step, int64_t first_step);
int gpt_serve_run(gpt* h, int32_t max_steps, float* kernel_ms);
int gpt_serve_tokens(gpt* h, int32_t* dst, int32_t cap, int32_t* n);
int gpt_serve_end(gpt* h);

/*
 * Measurement hook (per-phase timing, after the per-family table of
 * "Coppelius training on the RTX 3090", section "Where a step's time goes"):
 * runs the operations op_first .. op_first + op_count - 1 of the handle's step
 * graph (the order gpt_graph_describe reports for this config and this GPU's SM
 * count) as their own launch of the persistent kernel, `reps` times back to
 * back, on whatever the arena holds (run a step first so the activations are
 * real).  Their tasks keep the step's ticket order and their dependencies on
 * each other; dependencies on operations outside the range are dropped.
 * Operations that update in place act again: the cross-entropy rewrites the
 * logits buffer (which after a step holds the logit gradients), AdamW updates
 * the parameters and moments with the next update's bias correction (the update
 * count is not advanced).  tokens, targets: DEVICE int32 [batch, seq_len], as
 * gpt_train_step.  kernel_ms (HOST, may be NULL): mean device time of one
 * launch, from CUDA events on the handle's stream around each launch.
 * Errors: INVALID_ARG (range, reps outside 1..1000), POISONED, OOM (its small
 * task/counter buffer), CUDA, TIMEOUT (a wait inside the range gave up; the
 * handle is not poisoned).
 */
int gpt_run_ops(gpt* h, int32_t op_first, int32_t op_count, const int32_t* tokens, const int32_t* targets,
                int32_t reps, float* kernel_ms);

/* Size of the step's task graph: number of tasks, and the grid (resident
 * blocks) the persistent kernel is launched with.  Any pointer may be NULL. */
int gpt_graph_info(const gpt* h, int64_t* n_tasks, int32_t* grid, int32_t* block);

/*
 * In-kernel trace (observability, after the pages' per-launch device
 * timestamps: "Coppelius training on the RTX 3090", section "Where a step's
 * time goes").  gpt_trace_enable(h, 1) allocates a device buffer of 32 bytes
 * per task; every later step records, per task (ticket order), four uint64:
 * claim time, start time (after its dependency waits), end time (after its
 * release), all %globaltimer nanoseconds, and the SM id (low 32 bits) and
 * block index (high 32 bits) that ran it.
 * gpt_get_trace copies the last step's record to HOST dst[0..4*n_tasks); with
 * n = 4*n_tasks + 8*grid it also copies, per block, the last wait each GEMM
 * role entered (scheduler, TMA producer, MMA issuer, four epilogue warps) as
 * kind << 56 | (run-local task count mod 2^24) << 32 | task, and an eighth word
 * holding the block's number of GEMM runs << 32 | the last run's first task; the
 * kinds numbered 1..11 as: scheduler dependency wait, scheduler queue-slot
 * wait, producer queue wait, producer stage wait, MMA queue wait, MMA
 * accumulator wait, MMA stage wait, epilogue queue wait, epilogue tile,
 * epilogue group sync, role finished.  gpt_trace_enable(h, 0) frees the buffer.
 */
int gpt_trace_enable(gpt* h, int32_t on);
int gpt_get_trace(gpt* h, uint64_t* dst, size_t n);

/* Device time of the last step's kernel launch in milliseconds, from CUDA
 * events the library records on the handle's stream around the launch (after
 * gpt_train_steps: around its last launch, which ran up to 256 steps). */
int gpt_last_kernel_ms(const gpt* h, float* ms);

/* Text of the handle's last error ("" if none): the error notifier of
 * "Coppelius training on the RTX 3090", section "Channel health" (each
 * invocation's exit status, error notifier and finite-loss check).  h may be
 * NULL: the last error of gpt_create or of a handle-less call (test hooks,
 * gpt_train_step_static) in this process.  The string stays valid until the
 * next call on the same handle. */
const char* gpt_last_error(const gpt* h);

/* Releases every resource of the handle.  gpt_destroy(NULL) is a no-op. */
void gpt_destroy(gpt* h);

/*
 * 64-bit task budget of a workload that runs `iterations` rounds of
 * `tasks_per_iteration` tasks ("A longer run exposed a scheduler overflow":
 * the 32-bit product 4,194,304 x 2,225 wrapped).  Returns the product, or -1
 * if it does not fit in int64.
 */
int64_t gpt_task_budget(int64_t iterations, int64_t tasks_per_iteration);

/*
 * Host-only: fills HOST dst[0..n) (n == the parameter count of cfg) with the
 * seeded initial weights gpt_create(cfg, seed) would start from.  Needs no GPU.
 */
int gpt_init_params_host(const gpt_config* cfg, uint64_t seed, float* dst, size_t n);

/* One task of the step's graph as gpt_graph_describe reports it. */
typedef struct gpt_task_info {
  int32_t op;            /* operation the task belongs to                         */
  int32_t idx;           /* index of the task within its operation               */
  int32_t sig;           /* completion counter the task increments when done     */
  int32_t sig2;          /* op-level counter it also increments (-1: none)      */
  int32_t nwait;         /* number of dependency ranges (<= 3)                    */
  int32_t wait_first[3]; /* first counter of each range (-1 unused)               */
  int32_t wait_count[3]; /* counters in each range                                */
  int32_t wait_need[3];  /* per-step count each counter of the range must reach  */
} gpt_task_info;

/*
 * Host-only: builds the step's task graph for cfg (as if on a GPU with num_sms
 * SMs; <= 0 means 152, a GB300) without device memory, and reports it: *n_tasks tasks in
 * ticket order (the first max_tasks copied to HOST tasks[], may be NULL) and
 * *n_ops operations (type and task count of the first max_ops into HOST
 * op_types[] / op_tasks[], and into op_dims[6*i .. 6*i+5]: for GEMM
 * operations M, N, K and the tile width (zeros otherwise), then the op's first
 * completion counter and its number of counters (one per 128-row block of the
 * token dimension for ops with token-major output on the bf16 path plus one
 * op-level counter that every task of the op also increments, else 1);
 * each may be NULL).  Tasks are reported in ticket order.  Operation types are the kernel's
 * OpType values (0 embed, 1 LN forward, 2 GEMM, 3 attention forward, 4 cross-
 * entropy, 5 loss, 6 LN backward, 7 column sum, 8 attention backward,
 * 9 token-embedding backward, 10 position-embedding backward, 11 AdamW,
 * 12 attention-backward pre-pass, 13 attention dK/dV, 14 attention dQ,
 * 15 token sort).
 */
int gpt_graph_describe(const gpt_config* cfg, int32_t num_sms, int64_t* n_tasks, int32_t* n_ops,
                       gpt_task_info* tasks, int64_t max_tasks, int32_t* op_types, int32_t* op_tasks,
                       int32_t* op_dims, int32_t max_ops);

/*
 * Training step that allocates nothing (the pages have no counterpart: this is
 * an addition of this library).  It is for callers that cannot allocate device
 * memory: runtimes whose device memory is owned by a pool allocator that
 * allows no side allocations (a cudaMalloc next to the pool would break its
 * reservation or fragment it), and embedded or real-time hosts that must not
 * allocate after start-up (an allocation can block the calling thread for an
 * unbounded time).  The same persistent kernel runs the same task graph as
 * gpt_train_step, with GPT_DTYPE_FP32 arithmetic; every piece of scratch
 * (gradients, activations, the task graph, counters, error words) lives in one
 * 16 MiB file-scope device array that every GPU which loads libgpt.so holds
 * until the process exits.  No cudaMalloc, cudaFree, pinned or library
 * allocation is made; the task list is built in ordinary host heap memory and
 * copied into the array from pageable memory.
 *   cfg: GPT_DTYPE_FP32 only; models whose scratch exceeds 16 MiB (the tiny
 *     configuration needs about 5.6 MiB) are rejected with GPT_ERR_INVALID_ARG
 *     and a message giving the size they need, before anything is written to
 *     the array.
 *   params, m, v: DEVICE fp32 [gpt_param_count(cfg)] in the canonical order:
 *     the parameters and AdamW moments, read and updated in place.  The library
 *     cannot check their length: shorter buffers are read and written past
 *     their end.
 *   step: AdamW updates applied so far (bias correction uses step + 1); on
 *     GPT_OK the caller counts one more.
 *   tokens, targets: DEVICE int32 [batch, seq_len]; loss: HOST float*, may be
 *     NULL.  Runs on cuda_stream; the call copies the graph from host memory,
 *     writes the activation pads, launches the kernel and synchronises the
 *     stream before it returns.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * Every call sets the kernel's shared-memory limit (cudaFuncSetAttribute).
 * Every call shares the one array: it rewrites the graph and the pads and zeroes
 * the counters, the ticket and the error words before its launch, so calls whose
 * work overlaps on the GPU (other threads, other streams) race and must not be
 * made.  Errors as gpt_train_step (BAD_TOKEN / NONFINITE leave params, m, v as
 * they were), plus UNSUPPORTED for bf16; text via gpt_last_error(NULL).
 */
int gpt_train_step_static(const gpt_config* cfg, float* params, float* m, float* v, int64_t step,
                          const int32_t* tokens, const int32_t* targets, float* loss, void* cuda_stream);

/*
 * Test hook: one GEMM C[M,N] = sum_k A(m,k) B(n,k), fp32 output, run as a
 * one-task graph of the same persistent kernel (SIMT fp32 path for
 * GPT_DTYPE_FP32, tcgen05/TMA path for GPT_DTYPE_BF16).  A, B, C are DEVICE
 * pointers; A(m,k) = A[m*lda + k] (a_mn = 0, K-major) or A[k*lda + m] (a_mn = 1,
 * MN-major), likewise B with ldb/b_mn; C[m*ldc + n], or with ksplit > 1 split s
 * writes its partial sum to C + s*M*ldc.  Runs on cuda_stream and synchronises.
 * bf16 requires K % (64 ksplit) == 0, N % 64 == 0, lda and ldb multiples of 8.
 * kernel_ms: HOST float*, receives the kernel's device time (CUDA events
 * around the launch); may be NULL.
 * Errors: INVALID_ARG, UNSUPPORTED, OOM, CUDA, TIMEOUT; text via
 * gpt_last_error(NULL).
 */
int gpt_test_gemm(int32_t dtype, int32_t M, int32_t N, int32_t K, const void* A, int64_t lda, int32_t a_mn,
                  const void* B, int64_t ldb, int32_t b_mn, float* C, int64_t ldc, int32_t ksplit,
                  void* cuda_stream, float* kernel_ms);

/*
 * Test hook: one bf16 tensor-core GEMM as in gpt_test_gemm (A, B bf16, same
 * layouts), followed by one of the fused epilogues the training step uses on
 * the accumulator acc[m, n] (fp32):
 *   epi 0  store:         out bf16 [M, ldo] = acc + bias
 *   epi 1  residual add:  out fp32 [M, ldo] = src fp32 [M, lds] + acc + bias
 *   epi 2  GELU:          out bf16 = GELU'(acc + bias), out2 bf16 [M, ldo2] = GELU(acc + bias)
 *   epi 4  GELU backward: out bf16 = acc * src bf16 [M, lds]  (src: a stored GELU')
 * GELU is the tanh form when gelu_tanh != 0, else the erf form (the step's
 * MLP activation).  bias fp32 [N] or NULL (ignored by epi 4).  All pointers DEVICE; out may alias src (epi 1).
 * Requires K % 64 == 0, N % 64 == 0, lda, ldb % 8 == 0, ldo, ldo2, lds % 4 == 0.
 * kernel_ms (HOST, may be NULL) receives the launch's device time.  Errors:
 * INVALID_ARG, UNSUPPORTED, OOM, CUDA, TIMEOUT; text via gpt_last_error(NULL).
 */
int gpt_test_gemm_epilogue(int32_t M, int32_t N, int32_t K, const void* A, int64_t lda, int32_t a_mn,
                           const void* B, int64_t ldb, int32_t b_mn, int32_t epi, int32_t gelu_tanh, void* out,
                           int64_t ldo, void* out2, int64_t ldo2, const float* bias, const void* src, int64_t lds,
                           void* cuda_stream, float* kernel_ms);

/*
 * Test hook: causal multi-head attention forward and backward as a graph of
 * the persistent kernel's attention tasks.  DEVICE buffers, token-major rows
 * n = b*T + t: qkv [B*T, 3*H*d] (q | k | v, head h at columns h*d), o
 * [B*T, H*d] output, lse float [B, H, T] output (natural-log LSE of the
 * scaled scores), dout [B*T, H*d] input gradient of o, dqkv [B*T, 3*H*d]
 * output, scratch float workspace of at least B*H*T floats (bf16) or
 * B*H*2*T*d floats (fp32).  Element type bf16 (GPT_DTYPE_BF16: tensor cores,
 * d == 64, T % 128 == 0) or fp32 (GPT_DTYPE_FP32: SIMT).  Scale 1/sqrt(d).
 */
int gpt_test_attention(int32_t dtype, int32_t B, int32_t T, int32_t H, int32_t d, const void* qkv, void* o,
                       float* lse, const void* dout, void* dqkv, float* scratch, void* cuda_stream);

#ifdef __cplusplus
}
#endif
#endif /* GPT_H_ */
