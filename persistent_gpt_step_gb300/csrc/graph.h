// graph.h — task-graph descriptors shared by the host graph builder and the
// persistent kernel.  Plain structs of device pointers and sizes.
//
// The step is a list of tasks in a topological (ticket) order.  A task names an
// operation (an "op": one GEMM, one LayerNorm, the attention of one layer ...)
// and its tile / block index within that op.  Every op owns 64-bit completion
// counters: one per 128-row block of the token dimension for ops whose output
// is token-major, else one.  A task may wait for up to kMaxWaits ranges of
// counters to reach epoch * need (need = the producer's tasks per counter),
// then runs, then adds 1 to its own counter with release semantics.
// Dependencies only point to earlier tickets, so with every block resident the
// graph cannot deadlock
// ("How one persistent kernel runs three jobs": ticket counters, release
// fences before the counter increments, acquire waits by dependents).
#pragma once
#include <stdint.h>

namespace pgs {

constexpr int kMaxWaits = 3;
// tile shapes shared by the host graph builder and the kernels
constexpr int kSimtTile = 64;             // SIMT GEMM: 64 x 64 tiles
constexpr int kTcBM = 128;                // tensor-core GEMM: 128-row tiles
constexpr int kTcBK = 64;                 // one 128-byte swizzle row of bf16
constexpr int kTcStages = 4;
constexpr int kTcStageA = kTcBM * kTcBK * 2;          // 16 KB
constexpr int kTcStageB = 256 * kTcBK * 2;            // 32 KB (BN <= 256)
constexpr int kTcStageBytes = kTcStageA + kTcStageB;  // 48 KB
constexpr int kTcSmemBytes = kTcStages * kTcStageBytes;
constexpr int kEpiStageBytes = 32 * 64 * 4;            // per epilogue warp: 32 rows x 64 fp32
constexpr int kTmemCols = 512;            // two fp32 accumulators of up to 128 x 256
constexpr int kAdamSub = 4096;            // AdamW: parameters per bulk-copied sub-chunk
constexpr int kAdamStages = 3;            // AdamW: staging buffers (sub-chunks in flight + 1)
constexpr int kAdamStageBytes = kAdamSub * (4 * 4 + 2);  // p, g, m, v fp32 + bf16 copy
constexpr int kThreads = 256;     // threads of every persistent block
constexpr int kWarps = kThreads / 32;

enum OpType : int32_t {
  OP_EMBED = 0,      // x0 = wte[tok] + wpe[t]                       tasks: row blocks
  OP_LN_FWD,         // y = LN(x); mean, rstd                        tasks: row blocks
  OP_GEMM,           // C = A . B^T (+ epilogue)                     tasks: tiles
  OP_ATTN_FWD,       // causal softmax(q k^T / sqrt d) v, LSE        tasks: (b, h, q block)
  OP_CE,             // per-row loss; logits -> dlogits in place     tasks: row blocks
  OP_LOSS,           // mean of the row losses                       tasks: 1
  OP_LN_BWD,         // dres_out = dres_in + LN'(dy); dg/db partials tasks: row blocks
  OP_COLSUM,         // dst[c] = sum_r src[r, c] (fixed order)        tasks: column chunks
  OP_ATTN_BWD,       // dq, dk, dv of the causal attention           tasks: (b, h)
  OP_EMBED_BWD_WTE,  // dwte[v] = sum_{n: tok[n] = v} dx0[n]         tasks: vocab blocks
  OP_EMBED_BWD_WPE,  // dwpe[t] = sum_b dx0[b, t]                    tasks: position blocks
  OP_ADAMW,          // AdamW on a contiguous parameter range        tasks: chunks
  OP_ATTN_BWD_PRE,   // D = rowsum(dO * O) per head (tensor-core path) tasks: 64-row blocks
  OP_ATTN_BWD_KV,    // dK, dV of the causal attention               tasks: (b, h, 128 keys)
  OP_ATTN_BWD_Q,     // dQ of the causal attention                   tasks: (b, h, 128 queries)
  OP_TOKEN_SORT,     // (token, position) pairs sorted by token      tasks: 1
  OP_NOP,            // scheduler test: no work                      tasks: any
  OP_NUM_TYPES
};

enum Epilogue : int32_t {
  EPI_STORE = 0,     // out(act)  = acc (+ bias)
  EPI_RESID,         // out(f32)  = resid(f32) + acc (+ bias)
  EPI_GELU,          // out(act)  = GELU'(acc + bias) ; out2(act) = GELU(acc + bias)
  EPI_F32,           // out(f32)  = acc                   (dX partials, weight gradients)
  EPI_GELU_BWD,      // out(act)  = acc * aux(act)        (aux: the GELU' the forward stored)
  EPI_STORE_ROPE,    // out(act)  = acc (+ bias), q and k columns rotated (rotary embedding; see rope below)
  EPI_GEGLU,         // gated MLP up: columns (2f, 2f+1) = (gate, up) of feature f;
                     // out(act) [., 2N/2] = acc (kept for the backward), out2(act) [., N/2] = GELU(gate) * up
  EPI_GEGLU_BWD,     // gated MLP: acc = dh [., F]; aux(act) = stored (gate, up) [., 2F];
                     // out(act) [., 2F] = (dh * up * GELU'(gate), dh * GELU(gate)) per feature
};

struct GemmArgs {
  int32_t M, N, K;          // C[M, N] = sum_k A(m, k) B(n, k)
  int32_t BM, BN, BK;       // tile shape of one task
  int32_t tiles_n, ksplit;  // tasks = tiles_m * tiles_n * ksplit
  int32_t m_fastest;        // task order: 1 = M tiles vary fastest (B tile reused by consecutive tasks)
  // element access for the SIMT path: A(m,k) = A[m*sam + k*sak], B(n,k) = B[n*sbn + k*sbk]
  const void* A; int64_t sam, sak;
  const void* B; int64_t sbn, sbk;
  // tensor-core path: tensor-map indices and operand majorness (1 = MN-major)
  int32_t a_map, b_map, a_mn, b_mn;
  // output tensor map for the TMA-store epilogue (EPI_STORE / EPI_F32): 32 x 32
  // boxes of out, rows split * M + m; -1 = the epilogue stores with generic stores
  int32_t c_map;
  // EPI_STORE_ROPE (the QKV projection with rotary embedding): columns < 2 N / 3 (q and
  // k) rotate pair (2i, 2i+1) of each 64-wide head by the angle of row m's
  // position m mod rope_T: rope[(m mod rope_T) * 32 + i] = (cos, sin); null = none
  const float2* rope;
  int32_t rope_T;
  int32_t epi;
  void* out;  int64_t ldo;   // with ksplit > 1 split s writes out + s * split_stride
  int64_t split_stride;
  void* out2; int64_t ldo2;
  const float* bias;         // [N] or null
  const float* resid; int64_t ldr;
  const void* aux; int64_t ldaux;
  // weight gradient with the bias gradient folded in (EPI_F32): columns
  // n >= n_real come from a padded operand whose column n_real is all ones, so
  // column n_real of the product is the bias gradient, written to bias_grad[m];
  // the other padded columns are dropped.  n_real = N when there is none.
  int32_t n_real;
  float* bias_grad;
};

struct LnFwdArgs {
  const float* x; const float* g; const float* b;  // b may be null
  void* y; float* mean; float* rstd;
  int32_t rows, C, rows_per_task;
  float eps;
  int32_t ldy;      // row pitch of y (>= C)
  float* copy;      // may be null: x is also copied here (pitch C), the residual
                    // GEMM's output, which its epilogue then adds its product into
};

struct LnBwdArgs {
  const float* dy; int32_t dy_splits; int64_t dy_split_stride;  // dy = sum of splits
  const float* x; const float* mean; const float* rstd; const float* g;
  const float* dres_in;       // may be null
  float* dres_out; void* dres_act;
  float* dg_part; float* db_part;   // [tasks, C]; db_part may be null
  int32_t rows, C, rows_per_task;
  int32_t staged;   // bf16 path: the task's rows of dy, x, dres_in are bulk-copied into shared memory
};

struct AttnArgs {
  const void* qkv;  // act [B*T, 3C]: q | k | v, head h at columns h*d
  void* o;          // act [B*T, C]
  float* lse;       // [B, H, T]
  const void* dout; // act [B*T, C]   (backward)
  void* dqkv;       // act [B*T, 3C]  (backward)
  float* scratch;   // SIMT backward: dK/dV accumulators; tensor-core path: D [B, H, T]
  int32_t B, T, H, d, C, q_block;
  float scale;
  int32_t ld_o;     // row pitch of o (>= C)
  const float2* rope;  // rotary embedding (cos, sin) [T][d/2]: the backward rotates dq, dk back; null = none
  // tensor-core path: tensor maps (indices into KParams::tmaps) of qkv [B*T, 3C] and
  // dout [B*T, C], 64-column x 128-row boxes with the 128-byte swizzle; -1 = none
  int32_t qkv_map, do_map;
};

struct CeArgs {
  void* logits;              // act [N, V], overwritten by dlogits
  float* row_loss;           // [N]
  int32_t N, V, rows_per_task;
  int32_t staged;            // bf16: two whole rows fit in shared memory (bulk-copied)
};

struct LossArgs {
  const float* row_loss; float* loss; int32_t N;
};

struct ColsumArgs {
  const void* src; int32_t src_f32; int64_t ld;
  int32_t rows, cols, cols_per_task;
  float* dst;
};

struct EmbedArgs {
  const float* wte; const float* wpe; float* x0;
  const float* dx0; float* dwte; float* dwpe;
  int32_t N, B, T, C, V, rows_per_task;
  int32_t* sorted_tok; int32_t* sorted_pos;   // token ids in increasing order, stable
  int32_t* block_start;  // [V / rows_per_task + 1]: first sorted entry of each vocabulary block
  int32_t accumulate;    // token-embedding backward: add into dwte (tied LM head wrote it first)
};

struct AdamArgs {
  float* p; const float* g; float* m; float* v; uint16_t* shadow;  // shadow may be null
  int64_t n; int64_t chunk;
  float decay;   // 1 = apply weight decay
};

struct OpDesc {
  int32_t type;
  int32_t ntasks;
  union {
    GemmArgs gemm;
    LnFwdArgs lnf;
    LnBwdArgs lnb;
    AttnArgs attn;
    CeArgs ce;
    LossArgs loss;
    ColsumArgs colsum;
    EmbedArgs emb;
    AdamArgs adam;
  };
};

// A task waits until counters[first .. first+count) each reach epoch * need.
struct WaitSpec {
  int32_t first, count;
  uint32_t need;
};

struct TaskDesc {
  int32_t op;
  int32_t idx;                     // task index within its op
  int32_t sig;                     // counter this task adds 1 to when done
  int32_t sig2;                    // op-level counter also added to (-1: none)
  int32_t nwait;
  WaitSpec wait[kMaxWaits];
  int32_t pad[2];
};

// Soft error bits (the step runs to its end, AdamW skips its update).
constexpr uint32_t kSoftBadToken = 1u;
constexpr uint32_t kSoftNonFinite = 2u;
// Fatal error codes (blocks drain and exit).
constexpr uint32_t kFatalTimeout = 1u;
constexpr uint32_t kFatalMbarTimeout = 2u;

// ---- serving partition: greedy generation from the live weights --------------
// A reserved set of blocks runs one decode step per token: embedding, per layer
// LayerNorm, QKV (q kept, k and v appended to the cache), attention over the
// cache, attention-out (+ residual), LayerNorm, MLP up (+ GELU), MLP down (+
// residual), final LayerNorm, LM head in 64-row slices (each slice keeps its
// best logit), argmax.  The ops of a step form a chain; a step's embedding waits
// for the previous step's argmax ("one token releases the next").  Activations
// are fp32, weights the bf16 copy the training step keeps current.
enum ServeOpType : int32_t { SV_EMBED = 0, SV_LN, SV_GEMV, SV_ATTN, SV_ARGMAX };
enum ServeEpi : int32_t { SE_STORE = 0, SE_QKV, SE_RESID, SE_GELU, SE_LOGITS };
constexpr int kServeRows = 64;  // output rows of a GEMV task

struct ServeOp {
  int32_t type, ntasks, epi, K, N;
  const uint16_t* W;          // SV_GEMV: bf16 [N, K] (row-major, y = W x + b)
  const float* bias;          // [N] or null
  const float* in;            // [K] input vector (SV_LN, SV_GEMV, SV_ATTN: q)
  float* out;                 // output vector (SE_RESID: the residual stream, added to)
  float* kc; float* vc;       // SE_QKV / SV_ATTN: this layer's key and value cache [T, C] fp32
  const float* g; const float* b;  // SV_LN gain and bias (b may be null)
};

struct ServeParams {
  const ServeOp* ops; int32_t nops;
  const int32_t* task_op; const int32_t* task_idx;  // [P]: op and index of task k of a step
  int32_t P;                     // tasks per step
  unsigned long long* counters;  // [nops]: tasks of each op completed, over all steps
  unsigned long long* ticket;    // next serving ticket: step (ticket / P) - base, task ticket % P
  unsigned long long base;       // steps completed before this session started (counters start at base x ntasks)
  int64_t limit;                 // this launch serves steps < limit (the host restores the ticket per launch)
  int32_t* seq;                  // [T]: the prompt, then the generated tokens
  int32_t n_prompt;
  int32_t C, H, T, V;
  float ln_eps;
  int32_t gelu_tanh;
  const float* wte; const float* wpe;   // fp32 master embeddings (the training step keeps them current)
  float* part_max; int32_t* part_idx;   // [n_slices]: best logit of each LM-head slice and its id
  int32_t n_slices;
};

struct KParams {
  const TaskDesc* tasks; int64_t ntasks;
  const OpDesc* ops;
  unsigned long long* counters;
  unsigned long long* tickets;     // [2]: ticket counter of even / odd launches (this one: epoch & 1)
  unsigned long long epoch;        // 1-based step number of this launch
  uint32_t* err;                   // [0] fatal code, [1] soft bits, [2] task of a fatal error, [3] counter
  uint64_t timeout_ns;
  int64_t skip_release;            // test hook: this task skips its release (-1 = none)
  const void* tmaps;               // CUtensorMap[] (tensor-core path)
  const int32_t* tokens; const int32_t* targets;
  float lr, beta1, beta2, eps, wd, bc1, bc2;
  unsigned long long* trace;       // optional [ntasks][4]: claim, start, end (globaltimer ns), SM id
  float* loss_out;                 // multi-step launches: the loss ring, one slot per step (else null)
  uint32_t* status_out;            // ... and the status ring (the soft error bits after the loss)
  // K steps in one launch: step s (0-based) has epoch epoch + s, reads tokens and
  // targets + s * tok_stride, updates with step_hyper[3 s .. 3 s + 2] = (lr, bc1, bc2)
  // (null: the fields above), and writes loss_out[s], status_out[s].  Between two
  // steps every training block passes a grid barrier on grid_bar, which every
  // training block adds 1 to after each step (after step s of this launch it
  // holds bar_base + (s + 1) * the number of training blocks).
  int32_t nsteps;                  // <= 1: one step
  int64_t tok_stride;
  const float* step_hyper;
  unsigned long long* grid_bar;    // null: no step barrier (one-step launches of test graphs)
  // serving partition: blocks >= train_blocks serve (greedy generation) instead of
  // training; the grid barrier counts the training blocks only
  const ServeParams* serve;        // null: every block trains
  int32_t train_blocks;
  unsigned long long bar_base;     // grid-barrier arrivals before this launch (each step adds train_blocks)
};

}  // namespace pgs
