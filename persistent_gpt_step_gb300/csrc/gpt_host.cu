// gpt_host.cu — host side of libgpt.so: configuration, parameter table, the
// device arena, seeded initialisation, the task-graph builder, TMA tensor maps,
// the per-step launch of the persistent kernel and the C ABI of gpt.h.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <queue>
#include <string>
#include <thread>
#include <vector>

#include "../../include/gpt.h"
#include "graph.h"
#include "launch.h"

using namespace pgs;

namespace {

thread_local std::string g_create_error;

// ----------------------------------------------------------------------------
// Seeded initial weights: SplitMix64 (Steele, Lea, Flood 2014) + Box-Muller.
// Specification (shared with the test-side generator, implemented twice):
//   out(s, n) = mix(s + (n + 1) * 0x9E3779B97F4A7C15); key_t = out(seed, t);
//   u1 = (out(key_t, 2e) >> 11) 2^-53, u2 = (out(key_t, 2e+1) >> 11) 2^-53;
//   w = fp32(0.02 * sqrt(-2 ln(1 - u1)) cos(2 pi u2)).
// ----------------------------------------------------------------------------
inline uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}
inline uint64_t sm64_out(uint64_t state, uint64_t n) {
  return sm64_mix(state + (n + 1) * 0x9E3779B97F4A7C15ULL);
}
void normal_fill(float* dst, size_t n, uint64_t seed, uint64_t tensor_index) {
  const uint64_t key = sm64_out(seed, tensor_index);
  const double two_pi = 2.0 * 3.141592653589793;
  auto work = [&](size_t lo, size_t hi) {
    for (size_t e = lo; e < hi; ++e) {
      const double u1 = (double)(sm64_out(key, 2 * e) >> 11) * 0x1p-53;
      const double u2 = (double)(sm64_out(key, 2 * e + 1) >> 11) * 0x1p-53;
      const double z = std::sqrt(-2.0 * std::log(1.0 - u1)) * std::cos(two_pi * u2);
      dst[e] = (float)(0.02 * z);
    }
  };
  const size_t nth = n < (1u << 16) ? 1 : std::max(1u, std::min(32u, std::thread::hardware_concurrency()));
  if (nth == 1) { work(0, n); return; }
  std::vector<std::thread> th;
  for (size_t i = 0; i < nth; ++i) th.emplace_back(work, n * i / nth, n * (i + 1) / nth);
  for (auto& t : th) t.join();
}

inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40);  // NaN stays NaN
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

// ----------------------------------------------------------------------------
// Parameter table (canonical order, see gpt.h)
// ----------------------------------------------------------------------------
enum InitKind { INIT_NORMAL, INIT_ZEROS, INIT_ONES };
struct TensorInfo {
  std::string name;
  int64_t rows, cols;  // cols = 1 for vectors
  int ndim;
  size_t offset;
  InitKind init;
};

struct TensorIds {  // indices into the table, per layer
  int ln1_g, ln1_b, w_qkv, b_qkv, w_o, b_o, ln2_g, ln2_b, w_1, b_1, w_2, b_2;
};

struct Dims {
  int L, C, H, d, F, V, T, B, N;
};

}  // namespace

// ----------------------------------------------------------------------------
// The handle
// ----------------------------------------------------------------------------
constexpr int kStepRing = 256;  // steps of a multi-step call between host reads of the loss ring

struct gpt {
  gpt_config cfg;
  Dims D;
  int device = 0, num_sms = 0;
  cudaStream_t stream = nullptr;
  std::vector<TensorInfo> tensors;
  std::vector<TensorIds> lid;
  int t_wte = 0, t_wpe = 0, t_lnf_g = 0, t_lnf_b = -1, t_wlm = 0;
  size_t nparams = 0;

  // device memory
  uint8_t* arena = nullptr;
  size_t arena_bytes = 0;
  bool own_arena = false;
  uint8_t* meta = nullptr;  // tasks, ops, tensor maps, counters, error words, staging
  size_t meta_bytes = 0;

  // arena views
  float *params = nullptr, *grads = nullptr, *m = nullptr, *v = nullptr;
  uint16_t* shadow = nullptr;
  float* loss_dev = nullptr;

  // graph
  std::vector<OpDesc> ops;
  std::vector<TaskDesc> tasks;
  std::vector<std::vector<uint8_t>> tmaps;  // 128-byte CUtensorMaps
  TaskDesc* d_tasks = nullptr;
  OpDesc* d_ops = nullptr;
  void* d_tmaps = nullptr;
  unsigned long long* d_counters = nullptr;
  unsigned long long* d_ticket = nullptr;
  uint32_t* d_err = nullptr;
  int32_t* d_tok_stage = nullptr;

  // launch
  const void* kernel = nullptr;
  int grid = 0;
  size_t smem_bytes = 0;
  uint64_t launches = 0;     // completed launches since the last reset
  int64_t opt_step = 0;      // AdamW updates applied
  int64_t skip_release = -1;
  bool poisoned = false;
  bool describe_only = false;  // build the graph without device memory or tensor maps
  int n_counters = 0;          // completion counters of the graph
  std::vector<int> op_ctr0, op_nblk;  // first counter and counter count of each op

  cudaEvent_t ev0 = nullptr, ev1 = nullptr;  // bracket the kernel of the last step
  float last_kernel_ms = 0.f;
  unsigned long long* d_trace = nullptr;  // optional per-task timestamps (gpt_trace_enable)
  unsigned long long bar_count = 0;       // grid-barrier arrivals so far (reset with the counters)
  // serving session (gpt_serve_begin): device state in serve_mem, ServeParams at d_serve
  struct Serve {
    bool active = false;
    int32_t blocks = 0, n_prompt = 0, n_new = 0, per_step = 0;
    int64_t steps_total = 0, steps_done = 0;
    unsigned long long base = 0;
    int32_t P = 0;
    uint8_t* mem = nullptr;
    ServeParams* d_params = nullptr;
    ServeParams host{};  // the device copy's contents (limit and ticket are refreshed per launch)
  } serve;
  // host staging (pinned) for the per-step status
  struct Status {
    uint32_t err[4];
    float loss;
    uint32_t pad[3];
    float ring_loss[kStepRing];        // multi-step calls: per-step losses ...
    uint32_t ring_status[kStepRing];   // ... and soft error bits, read back once per chunk
    float ring_hyper[3 * kStepRing];   // ... and the (lr, bc1, bc2) table uploaded before the launch
  };
  float* d_loss_ring = nullptr;        // device rings of kStepRing slots (in the metadata allocation)
  uint32_t* d_status_ring = nullptr;
  float* d_step_hyper = nullptr;       // multi-step launch: (lr, bc1, bc2) of each step, kStepRing x 3
  unsigned long long* d_grid_bar = nullptr;  // grid barrier between the steps of a launch
  Status* h_status = nullptr;
  std::string err;
};

namespace {

int fail(gpt* h, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (h) h->err = buf; else g_create_error = buf;
  return code;
}

#define CUDA_TRY(h, call)                                                                    \
  do {                                                                                       \
    cudaError_t e_ = (call);                                                                 \
    if (e_ != cudaSuccess)                                                                   \
      return fail((h), GPT_ERR_CUDA, "%s failed: %s", #call, cudaGetErrorString(e_));        \
  } while (0)

bool is_bf16(const gpt_config& c) { return c.dtype == GPT_DTYPE_BF16; }

int validate(const gpt_config& c, std::string* why) {
  auto bad = [&](const char* s) { *why = s; return GPT_ERR_INVALID_ARG; };
  if (c.n_layer < 1 || c.d_model < 1 || c.n_head < 1 || c.d_mlp < 1 || c.vocab < 2 || c.seq_len < 1 ||
      c.batch < 1)
    return bad("every size must be positive (vocab >= 2)");
  if (c.dtype != GPT_DTYPE_FP32 && c.dtype != GPT_DTYPE_BF16) return bad("dtype must be 0 (fp32) or 1 (bf16)");
  if ((c.tie_embeddings || c.rope || c.gated_mlp) && !is_bf16(c)) {
    *why = "rotary embedding, the gated MLP and tied embeddings are built for the bf16 path only";
    return GPT_ERR_UNSUPPORTED;
  }
  if (c.gated_mlp && c.linear_bias) { *why = "the gated MLP has no linear biases (linear_bias 0)"; return GPT_ERR_UNSUPPORTED; }
  if (c.d_model % c.n_head) return bad("d_model must be a multiple of n_head");
  const int hd = c.d_model / c.n_head;
  if (c.d_model % 64 || c.d_model > 1024) { *why = "d_model must be a multiple of 64 and <= 1024"; return GPT_ERR_UNSUPPORTED; }
  if (c.d_mlp % 64) { *why = "d_mlp must be a multiple of 64"; return GPT_ERR_UNSUPPORTED; }
  if (hd > 128) { *why = "head_dim must be <= 128"; return GPT_ERR_UNSUPPORTED; }
  if (c.seq_len > 1024) { *why = "seq_len must be <= 1024"; return GPT_ERR_UNSUPPORTED; }
  if ((int64_t)c.batch * c.seq_len > 8192) { *why = "batch * seq_len must be <= 8192"; return GPT_ERR_UNSUPPORTED; }
  if (is_bf16(c)) {
    if (((int64_t)c.batch * c.seq_len) % 128) { *why = "bf16: batch * seq_len must be a multiple of 128"; return GPT_ERR_UNSUPPORTED; }
    if (c.vocab % 64) { *why = "bf16: vocab must be a multiple of 64"; return GPT_ERR_UNSUPPORTED; }
    if (hd != 64) { *why = "bf16: head_dim must be 64"; return GPT_ERR_UNSUPPORTED; }
    if (c.seq_len % 128) { *why = "bf16: seq_len must be a multiple of 128"; return GPT_ERR_UNSUPPORTED; }
  }
  if (!(c.lr >= 0.f) || !(c.beta1 >= 0.f && c.beta1 < 1.f) || !(c.beta2 >= 0.f && c.beta2 < 1.f) ||
      !(c.eps > 0.f) || !(c.ln_eps > 0.f) || !(c.weight_decay >= 0.f))
    return bad("bad optimizer / LayerNorm constants");
  return GPT_OK;
}

void build_table(gpt* h) {
  const gpt_config& c = h->cfg;
  const int64_t C = c.d_model, F = c.d_mlp, V = c.vocab, T = c.seq_len;
  auto add = [&](const std::string& name, int64_t r, int64_t cc, int nd, InitKind k) {
    TensorInfo t{name, r, cc, nd, h->nparams, k};
    h->nparams += (size_t)(r * cc);
    h->tensors.push_back(t);
    return (int)h->tensors.size() - 1;
  };
  h->t_wte = add("wte", V, C, 2, INIT_NORMAL);
  h->t_wpe = c.rope ? -1 : add("wpe", T, C, 2, INIT_NORMAL);
  for (int l = 0; l < c.n_layer; ++l) {
    const std::string p = "h" + std::to_string(l) + ".";
    TensorIds id{};
    id.ln1_g = add(p + "ln1_g", C, 1, 1, INIT_ONES);
    id.ln1_b = c.ln_bias ? add(p + "ln1_b", C, 1, 1, INIT_ZEROS) : -1;
    id.w_qkv = add(p + "w_qkv", 3 * C, C, 2, INIT_NORMAL);
    id.b_qkv = c.linear_bias ? add(p + "b_qkv", 3 * C, 1, 1, INIT_ZEROS) : -1;
    id.w_o = add(p + "w_o", C, C, 2, INIT_NORMAL);
    id.b_o = c.linear_bias ? add(p + "b_o", C, 1, 1, INIT_ZEROS) : -1;
    id.ln2_g = add(p + "ln2_g", C, 1, 1, INIT_ONES);
    id.ln2_b = c.ln_bias ? add(p + "ln2_b", C, 1, 1, INIT_ZEROS) : -1;
    id.w_1 = c.gated_mlp ? add(p + "w_gu", 2 * F, C, 2, INIT_NORMAL) : add(p + "w_1", F, C, 2, INIT_NORMAL);
    id.b_1 = c.linear_bias ? add(p + "b_1", F, 1, 1, INIT_ZEROS) : -1;
    id.w_2 = add(p + "w_2", C, F, 2, INIT_NORMAL);
    id.b_2 = c.linear_bias ? add(p + "b_2", C, 1, 1, INIT_ZEROS) : -1;
    h->lid.push_back(id);
  }
  h->t_lnf_g = add("lnf_g", C, 1, 1, INIT_ONES);
  h->t_lnf_b = c.ln_bias ? add("lnf_b", C, 1, 1, INIT_ZEROS) : -1;
  h->t_wlm = c.tie_embeddings ? h->t_wte : add("w_lm", V, C, 2, INIT_NORMAL);
}

// ----------------------------------------------------------------------------
// Arena layout: every buffer 256-byte aligned.  Per-layer activations are kept
// for the backward pass; every buffer has a single writer per step.
// ----------------------------------------------------------------------------
struct Bump {
  size_t off = 0;
  size_t take(size_t bytes) {
    off = (off + 255) & ~(size_t)255;
    size_t r = off;
    off += bytes;
    return r;
  }
};

struct Layout {
  size_t ldc, ldf;  // row pitch (elements) of the padded C- and F-wide activations
  size_t params, grads, m, v, shadow;
  std::vector<size_t> x, xm, ln1, ln1_mu, ln1_rs, qkv, atto, lse, ln2, ln2_mu, ln2_rs, dgelu, gact;
  size_t lnf, lnf_mu, lnf_rs, logits, row_loss, loss;
  size_t daf;
  std::vector<size_t> dx, dx_act, dxm, dxm_act, dh, da2, dO, dqkv, da1, att_scr;
  std::vector<size_t> ln1_gp, ln1_bp, ln2_gp, ln2_bp;
  size_t lnf_gp, lnf_bp;
  size_t sorted_tok, sorted_pos, block_start;
  size_t rope;  // rotary embedding (cos, sin) [T][32] fp32 pairs (rope configs)
  size_t total;
};

constexpr int kRowsLn = 32;       // rows per LayerNorm task
constexpr int kRowsCe = 4;        // rows per cross-entropy task

// The bf16 cross-entropy stages two whole rows of logits in shared memory when
// they fit beside the GEMM pipeline's footprint (it reuses that space).
bool ce_staged(const gpt_config& c) {
  const size_t row = ((size_t)c.vocab * 2 + 127) & ~(size_t)127;
  return c.dtype == GPT_DTYPE_BF16 && c.vocab % 8 == 0 && 2 * row + 64 <= (size_t)kTcSmemBytes + 4 * kEpiStageBytes;
}
constexpr int kRowsEmb = 32;      // rows per embedding task
constexpr int kVocabRows = 64;    // vocabulary rows per embedding-backward task
constexpr int kColsColsum = 64;   // columns per column-sum task
constexpr int64_t kAdamChunk = 65536;

int ln_tasks(int N) { return (N + kRowsLn - 1) / kRowsLn; }

// Rows per LayerNorm-backward task.  On the bf16 path (C = 128 NV, NV <= 8) a
// task stages its rows of `arrays` fp32 [rows, C] inputs in shared memory (dy
// and its split-K partials, x, the incoming residual gradient): 16 rows when
// they fit beside nothing else (the GEMM ring's space), else 8; otherwise the
// register path with kRowsLn rows.
int ln_bwd_rows(const gpt_config& c, int arrays) {
  if (c.dtype != GPT_DTYPE_BF16 || c.d_model % 128 || c.d_model > 1024) return kRowsLn;
  const size_t budget = (size_t)kTcSmemBytes + 4 * kEpiStageBytes;
  for (int rows : {16, 8})
    if ((size_t)arrays * rows * c.d_model * 4 <= budget) return rows;
  return kRowsLn;
}
bool ln_bwd_staged(const gpt_config& c, int arrays) { return ln_bwd_rows(c, arrays) != kRowsLn; }
// arrays a LayerNorm backward reads: a layer's (dy, x, dres_in); the final one's (dy splits, x)
int ln_bwd_arrays_layer() { return 3; }
int ln_bwd_arrays_final(int lm_ksplit) { return lm_ksplit + 1; }

// own_state = false: the caller owns the parameters and AdamW moments (the
// allocation-free step), so the arena holds no regions for them.
Layout make_layout(const gpt_config& c, size_t nparams, int lm_ksplit, bool own_state = true) {
  Layout Lo;
  Bump b;
  const size_t N = (size_t)c.batch * c.seq_len, C = c.d_model, F = c.d_mlp, V = c.vocab;
  const size_t act = is_bf16(c) ? 2 : 4;
  const int L = c.n_layer;
  const size_t BHT = (size_t)c.batch * c.n_head * c.seq_len;
  // gain / bias partials: one row per LayerNorm-backward task
  const size_t nrb = (N + ln_bwd_rows(c, ln_bwd_arrays_layer()) - 1) / ln_bwd_rows(c, ln_bwd_arrays_layer());
  const size_t nrb_f = (N + ln_bwd_rows(c, ln_bwd_arrays_final(lm_ksplit)) - 1) /
                       ln_bwd_rows(c, ln_bwd_arrays_final(lm_ksplit));
  // activations a weight-gradient GEMM reads as its second operand carry a
  // 64-column pad whose first column is 1 (bias gradients come out of the GEMM)
  const size_t pad = c.linear_bias ? 64 : 0;
  Lo.ldc = C + pad;
  Lo.ldf = F + pad;
  Lo.params = own_state ? b.take(nparams * 4) : 0;
  Lo.grads = b.take(nparams * 4);
  Lo.m = own_state ? b.take(nparams * 4) : 0;
  Lo.v = own_state ? b.take(nparams * 4) : 0;
  Lo.shadow = is_bf16(c) ? b.take(nparams * 2) : 0;
  for (int l = 0; l <= L; ++l) Lo.x.push_back(b.take(N * C * 4));
  for (int l = 0; l < L; ++l) {
    Lo.xm.push_back(b.take(N * C * 4));
    Lo.ln1.push_back(b.take(N * Lo.ldc * act));
    Lo.ln1_mu.push_back(b.take(N * 4));
    Lo.ln1_rs.push_back(b.take(N * 4));
    Lo.qkv.push_back(b.take(N * 3 * C * act));
    Lo.atto.push_back(b.take(N * Lo.ldc * act));
    Lo.lse.push_back(b.take(BHT * 4));
    Lo.ln2.push_back(b.take(N * Lo.ldc * act));
    Lo.ln2_mu.push_back(b.take(N * 4));
    Lo.ln2_rs.push_back(b.take(N * 4));
    // GELU'(pre-activation), or for the gated MLP the (gate, up) pairs [N, 2F], for the backward
    Lo.dgelu.push_back(b.take(N * F * (c.gated_mlp ? 2 : 1) * act));
    Lo.gact.push_back(b.take(N * Lo.ldf * act));
  }
  Lo.lnf = b.take(N * C * act);
  Lo.lnf_mu = b.take(N * 4);
  Lo.lnf_rs = b.take(N * 4);
  Lo.logits = b.take(N * V * act);
  Lo.row_loss = b.take(N * 4);
  Lo.loss = b.take(256);
  Lo.daf = b.take((size_t)lm_ksplit * N * C * 4);
  for (int l = 0; l <= L; ++l) {
    Lo.dx.push_back(b.take(N * C * 4));
    Lo.dx_act.push_back(b.take(N * C * act));
  }
  for (int l = 0; l < L; ++l) {
    Lo.dxm.push_back(b.take(N * C * 4));
    Lo.dxm_act.push_back(b.take(N * C * act));
    Lo.dh.push_back(b.take(N * F * (c.gated_mlp ? 2 : 1) * act));
    Lo.da2.push_back(b.take(N * C * 4));
    Lo.dO.push_back(b.take(N * C * act));
    Lo.dqkv.push_back(b.take(N * 3 * C * act));
    Lo.da1.push_back(b.take(N * C * 4));
    Lo.att_scr.push_back(b.take((size_t)c.batch * c.n_head * 2 * c.seq_len * (C / c.n_head) * 4));
    Lo.ln1_gp.push_back(b.take(nrb * C * 4));
    Lo.ln1_bp.push_back(b.take(nrb * C * 4));
    Lo.ln2_gp.push_back(b.take(nrb * C * 4));
    Lo.ln2_bp.push_back(b.take(nrb * C * 4));
  }
  Lo.lnf_gp = b.take(nrb_f * C * 4);
  Lo.lnf_bp = b.take(nrb_f * C * 4);
  Lo.rope = c.rope ? b.take((size_t)c.seq_len * 32 * 8) : 0;
  Lo.sorted_tok = b.take(N * 4);
  Lo.sorted_pos = b.take(N * 4);
  Lo.block_start = b.take((V / 64 + 2) * 4);
  Lo.total = (b.off + 255) & ~(size_t)255;
  return Lo;
}

// ----------------------------------------------------------------------------
// TMA tensor maps (driver entry point fetched through the runtime)
// ----------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  }
  return fn;
}

// 2-D bf16 tensor [outer][inner] (row pitch ld elements); box = 64 x box_outer, 128-byte swizzle.
int make_tmap(gpt* h, const void* base, int64_t inner, int64_t outer, int64_t ld, int box_outer) {
  if (h->describe_only) {
    h->tmaps.push_back(std::vector<uint8_t>(128, 0));
    return (int)h->tmaps.size() - 1;
  }
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return -1;
  std::vector<uint8_t> buf(128, 0);
  CUtensorMap* m = reinterpret_cast<CUtensorMap*>(buf.data());
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return -1;
  h->tmaps.push_back(buf);
  return (int)h->tmaps.size() - 1;
}

// Output map of a GEMM's TMA-store epilogue: rows x cols of bf16 (64-byte
// swizzle) or fp32 (128-byte swizzle), 32 x 32 boxes (one epilogue warp's rows,
// one 32-column group).  -1 when the output does not meet the TMA rules (16-byte
// aligned base and row pitch); the epilogue then stores with generic stores.
int make_tmap_out(gpt* h, void* base, bool f32, int64_t cols, int64_t rows, int64_t ld) {
  const int64_t es = f32 ? 4 : 2;
  if (((uintptr_t)base & 15) || (ld * es) % 16 || cols < 1 || rows < 1) return -1;
  if (h->describe_only) {
    h->tmaps.push_back(std::vector<uint8_t>(128, 0));
    return (int)h->tmaps.size() - 1;
  }
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return -1;
  std::vector<uint8_t> buf(128, 0);
  CUtensorMap* m = reinterpret_cast<CUtensorMap*>(buf.data());
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * es)};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return -1;
  h->tmaps.push_back(buf);
  return (int)h->tmaps.size() - 1;
}

// Gives a tensor-core GEMM op the output map of the TMA-store epilogue where it
// has one (bf16 store or fp32 store; with a K split the splits' outputs must be
// stacked row blocks of whole 128-row tiles; a residual GEMM without a separate
// residual operand adds into its output, which already holds the residual).
void set_out_map(gpt* h, OpDesc& op) {
  if (op.type != OP_GEMM) return;  // (the arguments are a union: only a GEMM op has c_map)
  GemmArgs& g = op.gemm;
  g.c_map = -1;
  if (!is_bf16(h->cfg) || !g.out) return;
  if (g.epi == EPI_RESID && !g.resid) {
    g.c_map = make_tmap_out(h, g.out, true, g.N, g.M, g.ldo);
  } else if (g.epi == EPI_STORE || g.epi == EPI_STORE_ROPE) {
    g.c_map = make_tmap_out(h, g.out, false, g.N, g.M, g.ldo);
  } else if (g.epi == EPI_F32) {
    if (g.ksplit > 1 && (g.M % kTcBM || g.split_stride != (int64_t)g.M * g.ldo)) return;
    g.c_map = make_tmap_out(h, g.out, true, g.n_real, (int64_t)g.M * g.ksplit, g.ldo);
  }
}

// ----------------------------------------------------------------------------
// Graph builder
// ----------------------------------------------------------------------------
// Host copy of the kernel's GEMM tile order (split-major, then M- or N-fastest).
void gemm_coords_host(const GemmArgs& g, int idx, int& tm, int& tn, int& split) {
  const int tiles_m = (g.M + g.BM - 1) / g.BM;
  const int per_split = tiles_m * g.tiles_n;
  split = idx / per_split;
  const int r = idx - split * per_split;
  if (g.m_fastest) { tm = r % tiles_m; tn = r / tiles_m; }
  else { tn = r % g.tiles_n; tm = r / g.tiles_n; }
}

// Builds the task list op by op.  On the tensor-core path every op whose output
// is token-major gets one completion counter per kRowBlock rows, and a task of
// such an op waits only for the row blocks it reads (the same rows, or for
// attention the prefix / suffix of its sequence); weight-gradient GEMMs, column
// sums, the loss, embedding gradients and AdamW read every row and wait for
// whole ops.  finish() then re-orders the tickets by list scheduling.
constexpr int kRowBlock = 128;

struct Builder {
  gpt* h;
  struct OpInfo {
    int ctr0, nblk, per_block;
    int op_ctr, ntasks;  // op-level counter (blocks > 1), counts every task
  };
  std::vector<OpInfo> info;
  std::vector<double> cost;  // estimated microseconds per task (ticket order of construction)
  int nctr = 0;

  // block of task i of op o, the row-block range [lo, hi] it reads (lo < 0: all
  // rows), and its estimated time
  void shape(const OpDesc& o, int i, int& blk, int& lo, int& hi, double& us) const {
    const Dims& D = h->D;
    const bool rowed = is_bf16(h->cfg);
    const double bw = 40e3;     // bytes per microsecond one SM streams
    blk = 0; lo = -1; hi = -1;
    us = 1.0;
    auto rows_task = [&](int rows_per_task, double bytes_per_row) {
      if (rowed) { blk = i * rows_per_task / kRowBlock; lo = hi = blk; }
      us = 1.0 + rows_per_task * bytes_per_row / bw;
    };
    const int nqb = D.T / 128;
    switch (o.type) {
      case OP_EMBED: rows_task(o.emb.rows_per_task, 12.0 * D.C); break;
      case OP_LN_FWD: rows_task(o.lnf.rows_per_task, 6.0 * D.C); break;
      case OP_LN_BWD:  // 18C bytes a row; the register path streams at half the rate (traced)
        rows_task(o.lnb.rows_per_task, (o.lnb.staged ? 18.0 : 36.0) * D.C);
        break;
      case OP_CE: rows_task(o.ce.rows_per_task, 6.0 * D.V); break;
      case OP_ATTN_BWD_PRE: rows_task(64, 4.0 * D.C); break;
      case OP_GEMM: {
        const GemmArgs& g = o.gemm;
        int tm, tn, sp;
        gemm_coords_host(g, i, tm, tn, sp);
        const double k = (double)g.K / g.ksplit;
        // traced in the 162M step: a tile costs ~6 us beyond its MMA work at ~7 TFLOP/s
        // per SM (loads in flight, epilogue, release), the GELU epilogue ~6 us more
        us = 6.0 + 2.0 * g.BM * g.BN * k / 7e6 + (g.epi == EPI_GELU ? 6.0 : 0.0);
        if (rowed && !g.a_mn && g.M == D.N) { blk = tm; lo = hi = tm; }  // token-major output rows
      } break;
      case OP_ATTN_FWD:
      case OP_ATTN_BWD_Q:
        if (rowed) {
          const int qb = nqb - 1 - i % nqb, b = i / (nqb * D.H);
          blk = (b * D.T + qb * 128) / kRowBlock;
          lo = o.type == OP_ATTN_FWD ? b * D.T / kRowBlock : blk;
          hi = blk;
          // (scaled to traced task times; the forward's fixed part is underestimated, which
          // measured better in the list order than costs fitted to the trace)
          us = 1.0 + (o.type == OP_ATTN_FWD ? 4.0 : 6.0) * 128.0 * (qb * 128 + 128) * D.d / 1.25e6;
        } else {
          us = 1.0 + 4.0 * D.T * D.T * D.d / 1e5;
        }
        break;
      case OP_ATTN_BWD_KV:
        if (rowed) {
          const int kb = i % nqb, b = i / (nqb * D.H);
          blk = (b * D.T + kb * 128) / kRowBlock;
          lo = blk;
          hi = (b * D.T + D.T) / kRowBlock - 1;
          us = 1.0 + 8.0 * 128.0 * (D.T - kb * 128) * D.d / 1.25e6;
        }
        break;
      case OP_ATTN_BWD: us = 1.0 + 12.0 * D.T * D.T * D.d / 1e5; break;
      case OP_COLSUM: us = 1.0 + (double)o.colsum.rows * o.colsum.cols_per_task * 4.0 / bw; break;
      case OP_ADAMW: us = 1.0 + std::min<double>(o.adam.chunk, (double)o.adam.n) * 30.0 / bw; break;
      case OP_EMBED_BWD_WTE: us = 2.0 + o.emb.rows_per_task * 4.0 * D.C / bw; break;
      case OP_TOKEN_SORT: us = 5.0 + D.N / 8.0; break;
      case OP_EMBED_BWD_WPE: us = 1.0 + o.emb.rows_per_task * 4.0 * D.C * D.B / bw; break;
      default: break;
    }
  }

  int add(const OpDesc& op_in, std::initializer_list<int> deps) {
    const int id = (int)h->ops.size();
    OpDesc op = op_in;
    set_out_map(h, op);
    h->ops.push_back(op);
    int dl[kMaxWaits], nd = 0;
    for (int d : deps) {
      if (d < 0) continue;
      bool dup = false;
      for (int i = 0; i < nd; ++i) dup |= dl[i] == d;
      if (!dup) dl[nd++] = d;
    }
    // block structure of this op
    int nblk = 1;
    if (is_bf16(h->cfg)) {
      int b, lo, hi;
      double us;
      for (int i = 0; i < op.ntasks; ++i) {
        shape(op, i, b, lo, hi, us);
        nblk = std::max(nblk, b + 1);
      }
    }
    OpInfo oi{nctr, nblk, 0, nblk > 1 ? nctr + nblk : nctr, op.ntasks};
    std::vector<int> per(nblk, 0);
    for (int i = 0; i < op.ntasks; ++i) {
      TaskDesc t{};
      int b, lo, hi;
      double us;
      shape(op, i, b, lo, hi, us);
      t.op = id;
      t.idx = i;
      t.sig = nctr + b;
      t.sig2 = nblk > 1 ? nctr + nblk : -1;
      per[b]++;
      t.nwait = nd;
      for (int w = 0; w < nd; ++w) {
        const OpInfo& pi = info[dl[w]];
        if (pi.nblk == 1 || lo < 0) {
          t.wait[w] = WaitSpec{pi.op_ctr, 1, (uint32_t)pi.ntasks};  // whole op: one counter
        } else {
          t.wait[w] = WaitSpec{pi.ctr0 + lo, hi - lo + 1, (uint32_t)pi.per_block};
        }
      }
      h->tasks.push_back(t);
      cost.push_back(us);
    }
    for (int b = 0; b < nblk; ++b)
      if (per[b] != per[0]) {
        fprintf(stderr, "libgpt: op %d has uneven row blocks\n", id);
        std::abort();
      }
    oi.per_block = per[0];
    info.push_back(oi);
    nctr += nblk > 1 ? nblk + 1 : 1;
    return id;
  }

  // Ticket order by list scheduling: simulate the graph on `workers` blocks with
  // the cost model, always starting the ready task with the longest remaining
  // path (bottom level) first; the start order becomes the ticket order.  A task
  // starts only after every task it waits for has finished, so dependencies
  // still point to earlier tickets.
  void finish(int workers) {
    const int T = (int)h->tasks.size();
    std::vector<int> remaining(nctr, 0);
    std::vector<std::vector<int>> waiters(nctr);
    std::vector<int> unmet(T, 0);
    for (int t = 0; t < T; ++t) {
      const TaskDesc& d = h->tasks[t];
      remaining[d.sig]++;
      if (d.sig2 >= 0) remaining[d.sig2]++;
      for (int w = 0; w < d.nwait; ++w)
        for (int c = 0; c < d.wait[w].count; ++c) {
          waiters[d.wait[w].first + c].push_back(t);
          unmet[t]++;
        }
    }
    // bottom levels, in reverse construction order (a topological order)
    std::vector<double> bl(T, 0.0), blc(nctr, 0.0);
    for (int t = T - 1; t >= 0; --t) {
      const TaskDesc& d = h->tasks[t];
      bl[t] = cost[t] + std::max(blc[d.sig], d.sig2 >= 0 ? blc[d.sig2] : 0.0);
      for (int w = 0; w < d.nwait; ++w)
        for (int c = 0; c < d.wait[w].count; ++c) {
          double& x = blc[d.wait[w].first + c];
          x = std::max(x, bl[t]);
        }
    }
    // priority = bottom level (critical path first).  Measured on the 162M step,
    // raising the priority of tasks that have waited long (to pull AdamW and
    // column sums forward into the backward) only made the step slower.
    auto cmp = [&](int a, int b) { return bl[a] < bl[b] || (bl[a] == bl[b] && a > b); };
    std::priority_queue<int, std::vector<int>, decltype(cmp)> ready(cmp);
    double now = 0.0;
    auto make_ready = [&](int t) { ready.push(t); };
    for (int t = 0; t < T; ++t)
      if (unmet[t] == 0) make_ready(t);
    typedef std::pair<double, int> Ev;
    std::priority_queue<Ev, std::vector<Ev>, std::greater<Ev>> running;
    std::vector<int> order;
    order.reserve(T);
    int idle = std::max(1, workers);
    while ((int)order.size() < T) {
      while (idle > 0 && !ready.empty()) {
        const int t = ready.top();
        ready.pop();
        order.push_back(t);
        running.push(Ev(now + cost[t], t));
        --idle;
      }
      if (running.empty()) break;  // cannot happen for a valid graph
      const Ev e = running.top();
      running.pop();
      now = e.first;
      ++idle;
      for (const int c : {h->tasks[e.second].sig, h->tasks[e.second].sig2}) {
        if (c < 0) continue;
        if (--remaining[c] == 0)
          for (int w : waiters[c])
            if (--unmet[w] == 0) make_ready(w);
      }
    }
    if ((int)order.size() != T) {
      fprintf(stderr, "libgpt: task graph has a cycle\n");
      std::abort();
    }
    std::vector<TaskDesc> sorted(T);
    for (int i = 0; i < T; ++i) sorted[i] = h->tasks[order[i]];
    h->tasks.swap(sorted);
    h->n_counters = nctr;
    h->op_ctr0.clear();
    h->op_nblk.clear();
    for (const OpInfo& oi : info) {
      h->op_ctr0.push_back(oi.ctr0);
      h->op_nblk.push_back(oi.nblk > 1 ? oi.nblk + 1 : 1);  // block counters + the op counter
    }
  }
};

// One GEMM operand: element (mn, k) of a row-major 2-D tensor with row pitch ld;
// K-major = stored [mn][k], MN-major = stored [k][mn].
struct Operand {
  const void* p;
  int64_t ld;
  bool mn_major;
};

int pick_bn(int M, int N, int num_sms, bool weight_grad) {
  // Weight-gradient GEMMs (both operands MN-major, K = tokens) run beside the
  // input-gradient chain of the backward, so what they cost is SM time, not a
  // wave of their own: 256-wide tiles do about twice the work per SM-second of
  // 128-wide ones there (traced in the 162M step).
  if (weight_grad && N >= 256 && N % 64 == 0) return 256;
  // otherwise prefer wide tiles, but not at the price of badly filled waves
  const int tm = (M + kTcBM - 1) / kTcBM;
  int best = 64;
  double best_eff = -1;
  for (int bn : {256, 128, 64}) {
    if (N % 64) continue;
    const int tiles = tm * ((N + bn - 1) / bn);
    const int waves = (tiles + num_sms - 1) / num_sms;
    double eff = (double)tiles / ((double)waves * num_sms) * (bn == 256 ? 1.0 : bn == 128 ? 0.92 : 0.75);
    eff *= (double)N / ((double)((N + bn - 1) / bn) * bn);  // ragged last tile
    if (eff > best_eff + 1e-9) { best_eff = eff; best = bn; }
  }
  return best;
}

int gemm_op(gpt* h, OpDesc* op, int M, int N, int K, Operand A, Operand B, int epi, int ksplit) {
  GemmArgs& g = op->gemm;
  std::memset(op, 0, sizeof(OpDesc));
  op->type = OP_GEMM;
  g.M = M; g.N = N; g.K = K;
  g.A = A.p; g.B = B.p;
  g.sam = A.mn_major ? 1 : A.ld; g.sak = A.mn_major ? A.ld : 1;
  g.sbn = B.mn_major ? 1 : B.ld; g.sbk = B.mn_major ? B.ld : 1;
  g.a_mn = A.mn_major; g.b_mn = B.mn_major;
  g.epi = epi;
  g.ksplit = ksplit;
  g.n_real = N;
  g.bias_grad = nullptr;
  g.a_map = g.b_map = g.c_map = -1;
  if (is_bf16(h->cfg)) {
    g.BM = kTcBM;
    g.BN = pick_bn(M, N, h->num_sms, A.mn_major && B.mn_major && epi == EPI_F32);
    g.BK = kTcBK;
    g.a_map = A.mn_major ? make_tmap(h, A.p, M, K, A.ld, 64) : make_tmap(h, A.p, K, M, A.ld, kTcBM);
    g.b_map = B.mn_major ? make_tmap(h, B.p, N, K, B.ld, 64) : make_tmap(h, B.p, K, N, B.ld, g.BN);
    if (g.a_map < 0 || g.b_map < 0) return fail(h, GPT_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  } else {
    g.BM = kSimtTile; g.BN = kSimtTile; g.BK = 16;
  }
  g.tiles_n = (N + g.BN - 1) / g.BN;
  g.m_fastest = N > M ? 1 : 0;  // consecutive tasks share the tile of the larger operand
  const int tiles_m = (M + g.BM - 1) / g.BM;
  op->ntasks = tiles_m * g.tiles_n * ksplit;
  return GPT_OK;
}

OpDesc blank(int type, int ntasks) {
  OpDesc o;
  std::memset(&o, 0, sizeof o);
  o.type = type;
  o.ntasks = ntasks;
  return o;
}

int build_graph(gpt* h, const Layout& Lo, int lm_ksplit) {
  const gpt_config& c = h->cfg;
  const Dims& D = h->D;
  uint8_t* A = h->arena;
  auto F32 = [&](size_t off) { return reinterpret_cast<float*>(A + off); };
  auto ACT = [&](size_t off) { return reinterpret_cast<void*>(A + off); };
  const bool bf = is_bf16(c);
  // weights as GEMM operands: bf16 copies on the tensor-core path, fp32 master otherwise
  auto W = [&](int t) -> const void* {
    const size_t off = h->tensors[t].offset;
    return bf ? (const void*)(h->shadow + off) : (const void*)(h->params + off);
  };
  auto P = [&](int t) -> float* { return t < 0 ? nullptr : h->params + h->tensors[t].offset; };
  auto G = [&](int t) -> float* { return t < 0 ? nullptr : h->grads + h->tensors[t].offset; };
  Builder bld{h};
  const int N = D.N, C = D.C, F = D.F, V = D.V, L = D.L;
  const int LDC = (int)Lo.ldc, LDF = (int)Lo.ldf;  // padded pitches (bias-gradient column)
  const bool gated = c.gated_mlp != 0, tied = c.tie_embeddings != 0;
  const int F2 = gated ? 2 * F : F;  // rows of the first MLP matrix (gate and up interleaved)
  const float2* rope_cs = c.rope ? reinterpret_cast<const float2*>(A + Lo.rope) : nullptr;
  int rc;

  // ---------------- forward ----------------
  OpDesc o = blank(OP_EMBED, (N + kRowsEmb - 1) / kRowsEmb);
  o.emb = EmbedArgs{P(h->t_wte), P(h->t_wpe), F32(Lo.x[0]), nullptr, nullptr, nullptr,
                    N, D.B, D.T, C, V, kRowsEmb, nullptr, nullptr, nullptr};
  int prev = bld.add(o, {});
  std::vector<int> op_ln1(L), op_qkv(L), op_attn(L), op_atto(L), op_ln2(L), op_up(L), op_down(L);
  std::vector<int> qkv_maps(L, -1);
  const int qblock = D.T <= 512 ? 64 : 32;
  for (int l = 0; l < L; ++l) {
    const TensorIds& id = h->lid[l];
    // bf16 path: LayerNorm also copies its input (the residual stream) into the
    // next residual GEMM's output, and that GEMM's epilogue adds its product in
    o = blank(OP_LN_FWD, ln_tasks(N));
    o.lnf = LnFwdArgs{F32(Lo.x[l]), P(id.ln1_g), P(id.ln1_b), ACT(Lo.ln1[l]), F32(Lo.ln1_mu[l]),
                      F32(Lo.ln1_rs[l]), N, C, kRowsLn, c.ln_eps, LDC, bf ? F32(Lo.xm[l]) : nullptr};
    op_ln1[l] = bld.add(o, {prev});
    // qkv = ln1 . Wqkv^T + b
    if ((rc = gemm_op(h, &o, N, 3 * C, C, {ACT(Lo.ln1[l]), LDC, false}, {W(id.w_qkv), C, false},
                      rope_cs ? EPI_STORE_ROPE : EPI_STORE, 1)))
      return rc;
    o.gemm.out = ACT(Lo.qkv[l]); o.gemm.ldo = 3 * C; o.gemm.bias = P(id.b_qkv);
    o.gemm.rope = rope_cs; o.gemm.rope_T = D.T;
    op_qkv[l] = bld.add(o, {op_ln1[l]});
    o = blank(OP_ATTN_FWD, bf ? D.B * D.H * (D.T / 128) : D.B * D.H * ((D.T + qblock - 1) / qblock));
    o.attn = AttnArgs{ACT(Lo.qkv[l]), ACT(Lo.atto[l]), F32(Lo.lse[l]), nullptr, nullptr, nullptr,
                      D.B, D.T, D.H, D.d, C, qblock, 1.0f / std::sqrt((float)D.d), LDC, nullptr, -1, -1};
    if (bf) {  // the attention tasks' TMA boxes: one head (64 columns) of 128 tokens
      o.attn.qkv_map = qkv_maps[l] = make_tmap(h, Lo.qkv[l] + A, 3 * C, N, 3 * C, 128);
      if (qkv_maps[l] < 0) return fail(h, GPT_ERR_CUDA, "cuTensorMapEncodeTiled failed (qkv)");
    }
    op_attn[l] = bld.add(o, {op_qkv[l]});
    // xm = x + o . Wo^T + b
    if ((rc = gemm_op(h, &o, N, C, C, {ACT(Lo.atto[l]), LDC, false}, {W(id.w_o), C, false}, EPI_RESID, 1)))
      return rc;
    o.gemm.out = F32(Lo.xm[l]); o.gemm.ldo = C; o.gemm.bias = P(id.b_o);
    o.gemm.resid = bf ? nullptr : F32(Lo.x[l]); o.gemm.ldr = C;
    op_atto[l] = bld.add(o, {op_attn[l]});
    if (bf && h->ops[op_atto[l]].gemm.c_map < 0) return fail(h, GPT_ERR_CUDA, "cuTensorMapEncodeTiled failed (residual)");
    o = blank(OP_LN_FWD, ln_tasks(N));
    o.lnf = LnFwdArgs{F32(Lo.xm[l]), P(id.ln2_g), P(id.ln2_b), ACT(Lo.ln2[l]), F32(Lo.ln2_mu[l]),
                      F32(Lo.ln2_rs[l]), N, C, kRowsLn, c.ln_eps, LDC, bf ? F32(Lo.x[l + 1]) : nullptr};
    op_ln2[l] = bld.add(o, {op_atto[l]});
    // h = ln2 . W1^T + b1 ; g = GELU(h)
    // gated: [gate, up] pairs kept for the backward, GELU(gate) * up to the next GEMM
    if ((rc = gemm_op(h, &o, N, F2, C, {ACT(Lo.ln2[l]), LDC, false}, {W(id.w_1), C, false},
                      gated ? EPI_GEGLU : EPI_GELU, 1)))
      return rc;
    o.gemm.out = ACT(Lo.dgelu[l]); o.gemm.ldo = F2; o.gemm.out2 = ACT(Lo.gact[l]); o.gemm.ldo2 = LDF;
    o.gemm.bias = P(id.b_1);
    op_up[l] = bld.add(o, {op_ln2[l]});
    // x_{l+1} = xm + g . W2^T + b2
    if ((rc = gemm_op(h, &o, N, C, F, {ACT(Lo.gact[l]), LDF, false}, {W(id.w_2), F, false}, EPI_RESID, 1)))
      return rc;
    o.gemm.out = F32(Lo.x[l + 1]); o.gemm.ldo = C; o.gemm.bias = P(id.b_2);
    o.gemm.resid = bf ? nullptr : F32(Lo.xm[l]); o.gemm.ldr = C;
    op_down[l] = prev = bld.add(o, {op_up[l]});
    if (bf && h->ops[op_down[l]].gemm.c_map < 0) return fail(h, GPT_ERR_CUDA, "cuTensorMapEncodeTiled failed (residual)");
  }
  o = blank(OP_LN_FWD, ln_tasks(N));
  o.lnf = LnFwdArgs{F32(Lo.x[L]), P(h->t_lnf_g), P(h->t_lnf_b), ACT(Lo.lnf), F32(Lo.lnf_mu), F32(Lo.lnf_rs),
                    N, C, kRowsLn, c.ln_eps, C};
  const int op_lnf = bld.add(o, {prev});
  // logits = lnf . Wlm^T
  if ((rc = gemm_op(h, &o, N, V, C, {ACT(Lo.lnf), C, false}, {W(h->t_wlm), C, false}, EPI_STORE, 1))) return rc;
  o.gemm.out = ACT(Lo.logits); o.gemm.ldo = V;
  const int op_lm = bld.add(o, {op_lnf});
  o = blank(OP_CE, (N + kRowsCe - 1) / kRowsCe);
  o.ce = CeArgs{ACT(Lo.logits), F32(Lo.row_loss), N, V, kRowsCe, ce_staged(c) ? 1 : 0};
  const int op_ce = bld.add(o, {op_lm});
  o = blank(OP_LOSS, 1);
  o.loss = LossArgs{F32(Lo.row_loss), F32(Lo.loss), N};
  const int op_loss = bld.add(o, {op_ce});

  // ---------------- backward ----------------
  auto adam = [&](int t, std::initializer_list<int> deps) {
    const TensorInfo& ti = h->tensors[t];
    const int64_t n = ti.rows * ti.cols;
    OpDesc a = blank(OP_ADAMW, (int)((n + kAdamChunk - 1) / kAdamChunk));
    a.adam = AdamArgs{h->params + ti.offset, h->grads + ti.offset, h->m + ti.offset, h->v + ti.offset,
                      bf ? h->shadow + ti.offset : nullptr, n, kAdamChunk,
                      (ti.ndim == 2 || c.wd_on_1d) ? 1.0f : 0.0f};
    // the gradient producers depend (through the backward) on every cross-entropy
    // row, whose task flags a non-finite loss, so AdamW sees that flag and the
    // bad-token flag without waiting for the loss reduction
    std::vector<int> dl(deps);
    if (dl.size() == 1) bld.add(a, {dl[0]});
    else bld.add(a, {dl[0], dl[1]});
  };
  auto colsum = [&](const void* src, bool f32, int64_t ld, int rows, int cols, float* dst, int dep,
                    int dep2 = -1) {
    OpDesc s = blank(OP_COLSUM, (cols + kColsColsum - 1) / kColsColsum);
    s.colsum = ColsumArgs{src, f32 ? 1 : 0, ld, rows, cols, kColsColsum, dst};
    return bld.add(s, {dep, dep2});
  };
  // LM head: daf = dz . Wlm ; dWlm = dz^T . lnf
  if ((rc = gemm_op(h, &o, N, C, V, {ACT(Lo.logits), V, false}, {W(h->t_wlm), C, true}, EPI_F32, lm_ksplit)))
    return rc;
  o.gemm.out = F32(Lo.daf); o.gemm.ldo = C; o.gemm.split_stride = (int64_t)N * C;
  const int op_lm_dx = bld.add(o, {op_ce});
  if ((rc = gemm_op(h, &o, V, C, N, {ACT(Lo.logits), V, true}, {ACT(Lo.lnf), C, true}, EPI_F32, 1))) return rc;
  o.gemm.out = G(h->t_wlm); o.gemm.ldo = C;
  const int op_lm_dw = bld.add(o, {op_ce});
  if (!tied) adam(h->t_wlm, {op_lm_dw, op_lm_dx});  // tied: wte's update follows the embedding gradient
  // final LayerNorm backward
  const int rows_f = ln_bwd_rows(c, ln_bwd_arrays_final(lm_ksplit));
  const int nrb_f = (N + rows_f - 1) / rows_f;
  o = blank(OP_LN_BWD, nrb_f);
  o.lnb = LnBwdArgs{F32(Lo.daf), lm_ksplit, (int64_t)N * C, F32(Lo.x[L]), F32(Lo.lnf_mu), F32(Lo.lnf_rs),
                    P(h->t_lnf_g), nullptr, F32(Lo.dx[L]), ACT(Lo.dx_act[L]), F32(Lo.lnf_gp),
                    h->t_lnf_b >= 0 ? F32(Lo.lnf_bp) : nullptr, N, C, rows_f,
                    ln_bwd_staged(c, ln_bwd_arrays_final(lm_ksplit)) ? 1 : 0};
  int op_dres = bld.add(o, {op_lm_dx});
  const int rows_l = ln_bwd_rows(c, ln_bwd_arrays_layer());
  const int nrb = (N + rows_l - 1) / rows_l;
  const int staged_l = ln_bwd_staged(c, ln_bwd_arrays_layer()) ? 1 : 0;
  {
    const int r1 = colsum(F32(Lo.lnf_gp), true, C, nrb_f, C, G(h->t_lnf_g), op_dres);
    adam(h->t_lnf_g, {r1});
    if (h->t_lnf_b >= 0) {
      const int r2 = colsum(F32(Lo.lnf_bp), true, C, nrb_f, C, G(h->t_lnf_b), op_dres);
      adam(h->t_lnf_b, {r2});
    }
  }
  for (int l = L - 1; l >= 0; --l) {
    const TensorIds& id = h->lid[l];
    // MLP down: dg = dx . W2 (then * GELU'(h)) ; dW2 = dx^T . g ; db2 = dx^T . 1
    // (gated: dh becomes the (gate, up) gradient pairs [N, 2F] from the stored pairs)
    if ((rc = gemm_op(h, &o, N, F, C, {ACT(Lo.dx_act[l + 1]), C, false}, {W(id.w_2), F, true},
                      gated ? EPI_GEGLU_BWD : EPI_GELU_BWD, 1)))
      return rc;
    o.gemm.out = ACT(Lo.dh[l]); o.gemm.ldo = F2; o.gemm.aux = ACT(Lo.dgelu[l]); o.gemm.ldaux = F2;
    const int op_down_dx = bld.add(o, {op_dres});
    // [dW2 | db2] = dx^T . [g | 1]
    if ((rc = gemm_op(h, &o, C, LDF, N, {ACT(Lo.dx_act[l + 1]), C, true}, {ACT(Lo.gact[l]), LDF, true}, EPI_F32, 1)))
      return rc;
    o.gemm.out = G(id.w_2); o.gemm.ldo = F; o.gemm.n_real = F; o.gemm.bias_grad = G(id.b_2);
    const int op_down_dw = bld.add(o, {op_dres});
    if (id.b_2 >= 0) adam(id.b_2, {op_down_dw});
    adam(id.w_2, {op_down_dw, op_down_dx});
    // MLP up: da2 = dh . W1 ; dW1 = dh^T . ln2 ; db1 = dh^T . 1
    if ((rc = gemm_op(h, &o, N, C, F2, {ACT(Lo.dh[l]), F2, false}, {W(id.w_1), C, true}, EPI_F32, 1))) return rc;
    o.gemm.out = F32(Lo.da2[l]); o.gemm.ldo = C;
    const int op_up_dx = bld.add(o, {op_down_dx});
    // [dW1 | db1] = dh^T . [ln2 | 1]
    if ((rc = gemm_op(h, &o, F2, LDC, N, {ACT(Lo.dh[l]), F2, true}, {ACT(Lo.ln2[l]), LDC, true}, EPI_F32, 1)))
      return rc;
    o.gemm.out = G(id.w_1); o.gemm.ldo = C; o.gemm.n_real = C; o.gemm.bias_grad = G(id.b_1);
    const int op_up_dw = bld.add(o, {op_down_dx});
    if (id.b_1 >= 0) adam(id.b_1, {op_up_dw});
    adam(id.w_1, {op_up_dw, op_up_dx});
    // LN2 backward: dxm = dx + LN2'(da2)
    o = blank(OP_LN_BWD, nrb);
    o.lnb = LnBwdArgs{F32(Lo.da2[l]), 1, 0, F32(Lo.xm[l]), F32(Lo.ln2_mu[l]), F32(Lo.ln2_rs[l]), P(id.ln2_g),
                      F32(Lo.dx[l + 1]), F32(Lo.dxm[l]), ACT(Lo.dxm_act[l]), F32(Lo.ln2_gp[l]),
                      id.ln2_b >= 0 ? F32(Lo.ln2_bp[l]) : nullptr, N, C, rows_l, staged_l};
    const int op_ln2b = bld.add(o, {op_up_dx, op_dres});
    adam(id.ln2_g, {colsum(F32(Lo.ln2_gp[l]), true, C, nrb, C, G(id.ln2_g), op_ln2b)});
    if (id.ln2_b >= 0) adam(id.ln2_b, {colsum(F32(Lo.ln2_bp[l]), true, C, nrb, C, G(id.ln2_b), op_ln2b)});
    // attention out: dO = dxm . Wo ; dWo = dxm^T . o ; dbo = dxm^T . 1
    if ((rc = gemm_op(h, &o, N, C, C, {ACT(Lo.dxm_act[l]), C, false}, {W(id.w_o), C, true}, EPI_STORE, 1)))
      return rc;
    o.gemm.out = ACT(Lo.dO[l]); o.gemm.ldo = C;
    const int op_atto_dx = bld.add(o, {op_ln2b});
    // [dWo | dbo] = dxm^T . [o | 1]
    if ((rc = gemm_op(h, &o, C, LDC, N, {ACT(Lo.dxm_act[l]), C, true}, {ACT(Lo.atto[l]), LDC, true}, EPI_F32, 1)))
      return rc;
    o.gemm.out = G(id.w_o); o.gemm.ldo = C; o.gemm.n_real = C; o.gemm.bias_grad = G(id.b_o);
    const int op_atto_dw = bld.add(o, {op_ln2b});
    if (id.b_o >= 0) adam(id.b_o, {op_atto_dw});
    adam(id.w_o, {op_atto_dw, op_atto_dx});
    // attention backward -> dqkv
    AttnArgs att{ACT(Lo.qkv[l]), ACT(Lo.atto[l]), F32(Lo.lse[l]), ACT(Lo.dO[l]), ACT(Lo.dqkv[l]),
                 F32(Lo.att_scr[l]), D.B, D.T, D.H, D.d, C, qblock, 1.0f / std::sqrt((float)D.d), LDC,
                 rope_cs, -1, -1};
    if (bf) {
      att.qkv_map = qkv_maps[l];
      att.do_map = make_tmap(h, Lo.dO[l] + A, C, N, C, 128);
      if (att.do_map < 0) return fail(h, GPT_ERR_CUDA, "cuTensorMapEncodeTiled failed (dO)");
    }
    int op_attb, op_attb2 = -1;
    if (bf) {
      o = blank(OP_ATTN_BWD_PRE, N / 64);
      o.attn = att;
      const int op_pre = bld.add(o, {op_atto_dx});
      o = blank(OP_ATTN_BWD_KV, D.B * D.H * (D.T / 128));
      o.attn = att;
      op_attb = bld.add(o, {op_pre});
      o = blank(OP_ATTN_BWD_Q, D.B * D.H * (D.T / 128));
      o.attn = att;
      op_attb2 = bld.add(o, {op_pre});
    } else {
      o = blank(OP_ATTN_BWD, D.B * D.H);
      o.attn = att;
      op_attb = bld.add(o, {op_atto_dx});
    }
    // QKV: da1 = dqkv . Wqkv ; dWqkv = dqkv^T . ln1 ; dbqkv = dqkv^T . 1
    if ((rc = gemm_op(h, &o, N, C, 3 * C, {ACT(Lo.dqkv[l]), 3 * C, false}, {W(id.w_qkv), C, true}, EPI_F32, 1)))
      return rc;
    o.gemm.out = F32(Lo.da1[l]); o.gemm.ldo = C;
    const int op_qkv_dx = bld.add(o, {op_attb, op_attb2});
    // [dWqkv | dbqkv] = dqkv^T . [ln1 | 1]
    if ((rc = gemm_op(h, &o, 3 * C, LDC, N, {ACT(Lo.dqkv[l]), 3 * C, true}, {ACT(Lo.ln1[l]), LDC, true}, EPI_F32,
                      1)))
      return rc;
    o.gemm.out = G(id.w_qkv); o.gemm.ldo = C; o.gemm.n_real = C; o.gemm.bias_grad = G(id.b_qkv);
    const int op_qkv_dw = bld.add(o, {op_attb, op_attb2});
    if (id.b_qkv >= 0) adam(id.b_qkv, {op_qkv_dw});
    adam(id.w_qkv, {op_qkv_dw, op_qkv_dx});
    // LN1 backward: dx_l = dxm + LN1'(da1)
    o = blank(OP_LN_BWD, nrb);
    o.lnb = LnBwdArgs{F32(Lo.da1[l]), 1, 0, F32(Lo.x[l]), F32(Lo.ln1_mu[l]), F32(Lo.ln1_rs[l]), P(id.ln1_g),
                      F32(Lo.dxm[l]), F32(Lo.dx[l]), ACT(Lo.dx_act[l]), F32(Lo.ln1_gp[l]),
                      id.ln1_b >= 0 ? F32(Lo.ln1_bp[l]) : nullptr, N, C, rows_l, staged_l};
    op_dres = bld.add(o, {op_qkv_dx, op_ln2b});
    adam(id.ln1_g, {colsum(F32(Lo.ln1_gp[l]), true, C, nrb, C, G(id.ln1_g), op_dres)});
    if (id.ln1_b >= 0) adam(id.ln1_b, {colsum(F32(Lo.ln1_bp[l]), true, C, nrb, C, G(id.ln1_b), op_dres)});
  }
  // embeddings: sort (token, position) pairs, then one task per block of vocabulary rows
  int32_t* stok = reinterpret_cast<int32_t*>(A + Lo.sorted_tok);
  int32_t* spos = reinterpret_cast<int32_t*>(A + Lo.sorted_pos);
  int32_t* bstart = reinterpret_cast<int32_t*>(A + Lo.block_start);
  o = blank(OP_TOKEN_SORT, 1);
  o.emb = EmbedArgs{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, N, D.B, D.T, C, V, kVocabRows,
                    stok, spos, bstart};
  const int op_sort = bld.add(o, {});
  o = blank(OP_EMBED_BWD_WTE, (V + kVocabRows - 1) / kVocabRows);
  o.emb = EmbedArgs{nullptr, nullptr, nullptr, F32(Lo.dx[0]), G(h->t_wte), G(h->t_wpe), N, D.B, D.T, C, V,
                    kVocabRows, stok, spos, bstart, tied ? 1 : 0};
  // tied: the LM head's weight gradient is written first, the scatter adds to it
  const int op_wte = bld.add(o, {op_dres, op_sort, tied ? op_lm_dw : -1});
  adam(h->t_wte, {op_wte});
  if (h->t_wpe >= 0) {
    o = blank(OP_EMBED_BWD_WPE, (D.T + kRowsEmb - 1) / kRowsEmb);
    o.emb = EmbedArgs{nullptr, nullptr, nullptr, F32(Lo.dx[0]), G(h->t_wte), G(h->t_wpe), N, D.B, D.T, C, V,
                      kRowsEmb, nullptr, nullptr, nullptr};
    const int op_wpe = bld.add(o, {op_dres});
    adam(h->t_wpe, {op_wpe});
  }
  bld.finish(h->num_sms > 0 ? h->num_sms : 152);
  (void)op_lm; (void)op_qkv; (void)op_attn; (void)op_atto; (void)op_ln2; (void)op_up; (void)op_down;
  return GPT_OK;
}

size_t smem_needed(const gpt* h) {
  const Dims& D = h->D;
  const int qblock = D.T <= 512 ? 64 : 32;
  size_t s = 0;
  s = std::max(s, (size_t)(2 * 16 * (kSimtTile + 4) * 4));                     // SIMT GEMM
  s = std::max(s, (size_t)(2 * kWarps * D.C * 4));                             // LN backward partials
  s = std::max(s, (size_t)D.N * 16 + 256 * 4);                                 // token sort
  s = std::max(s, (size_t)(D.N + 3) / 4 * 16 + (size_t)kWarps * D.C * 4);      // embedding backward (wte)
  s = std::max(s, (size_t)(qblock * D.d + 64 * (D.d + 1) + qblock * D.T) * 4); // attention forward
  s = std::max(s, (size_t)(2 * qblock * D.d + 64 * (D.d + 1) + qblock * D.T + qblock) * 4);  // backward
  s = std::max(s, (size_t)kThreads * 4);
  s = std::max(s, (size_t)kAdamStages * kAdamStageBytes);          // AdamW staging
  if (is_bf16(h->cfg)) s = std::max(s, (size_t)kTcSmemBytes + 4 * kEpiStageBytes);
  return s + 1024;  // 1024-byte alignment slack
}

// Writes the 64-column pad of every activation a weight-gradient GEMM reads as
// its second operand: column 0 of the pad = 1 (so the GEMM also produces the
// bias gradient), the rest 0.  Nothing else writes these columns.
int init_bias_pads(gpt* h, const Layout& Lo) {
  const Dims& D = h->D;
  if (Lo.ldc == (size_t)D.C) return GPT_OK;
  const bool bf = is_bf16(h->cfg);
  const size_t es = bf ? 2 : 4, padc = 64;
  std::vector<uint8_t> pad(D.N * padc * es, 0);
  for (int r = 0; r < D.N; ++r) {
    if (bf) { const uint16_t one = 0x3F80; std::memcpy(&pad[(size_t)r * padc * es], &one, 2); }
    else { const float one = 1.0f; std::memcpy(&pad[(size_t)r * padc * es], &one, 4); }
  }
  auto put = [&](size_t off, size_t width, size_t ld) {
    return cudaMemcpy2DAsync(h->arena + off + width * es, ld * es, pad.data(), padc * es, padc * es, D.N,
                             cudaMemcpyHostToDevice, h->stream);
  };
  for (int l = 0; l < D.L; ++l) {
    CUDA_TRY(h, put(Lo.ln1[l], D.C, Lo.ldc));
    CUDA_TRY(h, put(Lo.ln2[l], D.C, Lo.ldc));
    CUDA_TRY(h, put(Lo.atto[l], D.C, Lo.ldc));
    CUDA_TRY(h, put(Lo.gact[l], D.F, Lo.ldf));
  }
  CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  return GPT_OK;
}

int fill_shadow_and_upload(gpt* h, const float* host_params) {
  CUDA_TRY(h, cudaMemcpyAsync(h->params, host_params, h->nparams * 4, cudaMemcpyHostToDevice, h->stream));
  if (is_bf16(h->cfg)) {
    std::vector<uint16_t> sh(h->nparams);
    for (size_t i = 0; i < h->nparams; ++i) sh[i] = f32_to_bf16_rne(host_params[i]);
    CUDA_TRY(h, cudaMemcpyAsync(h->shadow, sh.data(), h->nparams * 2, cudaMemcpyHostToDevice, h->stream));
    CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  } else {
    CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  }
  return GPT_OK;
}

int reset_counters(gpt* h) {
  const size_t nctr = (size_t)h->n_counters;
  CUDA_TRY(h, cudaMemsetAsync(h->d_counters, 0, nctr * sizeof(unsigned long long), h->stream));
  CUDA_TRY(h, cudaMemsetAsync(h->d_ticket, 0, 2 * sizeof(unsigned long long), h->stream));
  CUDA_TRY(h, cudaMemsetAsync(h->d_err, 0, 4 * sizeof(uint32_t), h->stream));
  if (h->d_grid_bar) CUDA_TRY(h, cudaMemsetAsync(h->d_grid_bar, 0, sizeof(unsigned long long), h->stream));
  CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  h->launches = 0;
  h->bar_count = 0;
  h->poisoned = false;
  return GPT_OK;
}

// Queues one launch of the step kernel on the handle's stream (no
// synchronisation): epoch = launch number, lr and the bias corrections of update
// number t; loss_out / status_out: ring slots of a multi-step call (or null).
KParams step_params(gpt* h, const int32_t* tokens, const int32_t* targets, unsigned long long epoch, float lr,
                    int64_t t) {
  KParams kp;
  std::memset(&kp, 0, sizeof kp);
  kp.tasks = h->d_tasks;
  kp.ntasks = (int64_t)h->tasks.size();
  kp.ops = h->d_ops;
  kp.counters = h->d_counters;
  kp.tickets = h->d_ticket;
  kp.epoch = epoch;
  kp.err = h->d_err;
  kp.timeout_ns = (uint64_t)(h->cfg.wait_timeout_ms ? h->cfg.wait_timeout_ms : 2000) * 1000000ull;
  kp.skip_release = h->skip_release;
  kp.tmaps = h->d_tmaps;
  kp.tokens = tokens;
  kp.targets = targets;
  kp.nsteps = 1;
  kp.tok_stride = (int64_t)h->D.N;
  kp.grid_bar = h->d_grid_bar;
  kp.trace = h->d_trace;
  kp.lr = lr; kp.beta1 = h->cfg.beta1; kp.beta2 = h->cfg.beta2; kp.eps = h->cfg.eps;
  kp.wd = h->cfg.weight_decay;
  kp.bc1 = (float)(1.0 - std::pow((double)h->cfg.beta1, (double)t));
  kp.bc2 = (float)(1.0 - std::pow((double)h->cfg.beta2, (double)t));
  return kp;
}

// Serving blocks of an active session for a launch that trains `steps` steps
// (0: a serving-only launch): the session's step limit for this launch and its
// ticket are written to the device, and the training blocks' count is set.
int serve_prepare(gpt* h, KParams& kp, int64_t steps_budget) {
  gpt::Serve& sv = h->serve;
  if (!sv.active || sv.steps_done >= sv.steps_total || steps_budget <= 0) return GPT_OK;
  const int64_t limit = std::min<int64_t>(sv.steps_total, sv.steps_done + steps_budget);
  sv.host.limit = limit;
  const unsigned long long ticket = (sv.base + (unsigned long long)sv.steps_done) * (unsigned long long)sv.P;
  CUDA_TRY(h, cudaMemcpyAsync(sv.d_params, &sv.host, sizeof(ServeParams), cudaMemcpyHostToDevice, h->stream));
  CUDA_TRY(h, cudaMemcpyAsync(sv.host.ticket, &ticket, sizeof ticket, cudaMemcpyHostToDevice, h->stream));
  kp.serve = sv.d_params;
  kp.train_blocks = h->grid - sv.blocks;
  return GPT_OK;
}

int launch_kernel(gpt* h, KParams& kp) {
  if (kp.grid_bar) kp.bar_base = h->bar_count;
  int32_t gelu_tanh = h->cfg.gelu_tanh;
  void* args[2] = {&kp, &gelu_tanh};
  cudaError_t e = cudaLaunchCooperativeKernel(h->kernel, dim3(h->grid), dim3(kThreads), args, h->smem_bytes,
                                              h->stream);
  if (e != cudaSuccess) return fail(h, GPT_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
  if (kp.grid_bar && kp.ntasks > 0)  // every training block arrives once per step
    h->bar_count += (unsigned long long)(kp.nsteps > 1 ? kp.nsteps : 1) *
                    (unsigned long long)(kp.serve ? kp.train_blocks : h->grid);
  if (kp.serve) h->serve.steps_done = h->serve.host.limit;  // every step below the limit completes in the launch
  return GPT_OK;
}

int enqueue_step(gpt* h, const int32_t* tokens, const int32_t* targets, unsigned long long epoch, float lr,
                 int64_t t, float* loss_out, uint32_t* status_out) {
  KParams kp = step_params(h, tokens, targets, epoch, lr, t);
  kp.loss_out = loss_out;
  kp.status_out = status_out;
  h->skip_release = -1;
  const int rc = serve_prepare(h, kp, h->serve.per_step);
  if (rc != GPT_OK) return rc;
  return launch_kernel(h, kp);
}

int launch_step(gpt* h, const int32_t* tokens, const int32_t* targets, float* loss) {
  if (h->poisoned) return fail(h, GPT_ERR_POISONED, "handle poisoned by an earlier timeout; call gpt_reset");
  if (h->ev0) CUDA_TRY(h, cudaEventRecord(h->ev0, h->stream));
  int rc = enqueue_step(h, tokens, targets, h->launches + 1, h->cfg.lr, h->opt_step + 1, nullptr, nullptr);
  if (rc != GPT_OK) return rc;
  if (h->ev1) CUDA_TRY(h, cudaEventRecord(h->ev1, h->stream));
  CUDA_TRY(h, cudaMemcpyAsync(h->h_status->err, h->d_err, 4 * sizeof(uint32_t), cudaMemcpyDeviceToHost, h->stream));
  CUDA_TRY(h, cudaMemcpyAsync(&h->h_status->loss, h->loss_dev, sizeof(float), cudaMemcpyDeviceToHost, h->stream));
  CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  if (h->ev0 && h->ev1) cudaEventElapsedTime(&h->last_kernel_ms, h->ev0, h->ev1);
  const uint32_t fatal = h->h_status->err[0], soft = h->h_status->err[1];
  if (fatal) {
    h->poisoned = true;
    return fail(h, GPT_ERR_TIMEOUT, "device wait timed out (code %u, task %u, counter/barrier %u)", fatal,
                h->h_status->err[2], h->h_status->err[3]);
  }
  h->launches++;
  if (loss) *loss = h->h_status->loss;
  if (soft) {
    CUDA_TRY(h, cudaMemsetAsync(h->d_err + 1, 0, sizeof(uint32_t), h->stream));
    CUDA_TRY(h, cudaStreamSynchronize(h->stream));
    if (soft & kSoftBadToken) return fail(h, GPT_ERR_BAD_TOKEN, "token or target id outside [0, vocab)");
    return fail(h, GPT_ERR_NONFINITE, "non-finite loss %g", (double)h->h_status->loss);
  }
  h->opt_step++;
  h->err.clear();
  return GPT_OK;
}

bool schedule_ok(const gpt_lr_schedule* s) {
  if (!s) return true;
  if (s->kind == GPT_LR_CONSTANT) return true;
  if (s->kind != GPT_LR_WARMUP_COSINE) return false;
  return s->warmup_steps >= 0 && s->total_steps > s->warmup_steps && std::isfinite(s->lr_max) &&
         std::isfinite(s->lr_min) && s->lr_min >= 0.f && s->lr_max >= s->lr_min;
}

double schedule_lr(const gpt_lr_schedule* s, double base_lr, int64_t t) {
  if (!s || s->kind == GPT_LR_CONSTANT) return base_lr;
  if (s->warmup_steps > 0 && t <= s->warmup_steps) return (double)s->lr_max * (double)t / s->warmup_steps;
  if (t >= s->total_steps) return s->lr_min;
  const double frac = (double)(t - s->warmup_steps) / (double)(s->total_steps - s->warmup_steps);
  return s->lr_min + 0.5 * ((double)s->lr_max - s->lr_min) * (1.0 + std::cos(M_PI * frac));
}

// k steps, queued in chunks of kStepRing launches with one host read per chunk.
int train_steps(gpt* h, const int32_t* tokens, const int32_t* targets, int32_t k, const gpt_lr_schedule* sched,
                float* losses) {
  if (h->poisoned) return fail(h, GPT_ERR_POISONED, "handle poisoned by an earlier timeout; call gpt_reset");
  const int64_t n = (int64_t)h->D.N;
  for (int32_t j0 = 0; j0 < k; j0 += kStepRing) {
    const int32_t kc = std::min<int32_t>(kStepRing, k - j0);
    // the chunk's kc steps run inside ONE launch of the persistent kernel: step j has
    // epoch launches + 1 + j, its rate and bias corrections come from this table
    for (int32_t j = 0; j < kc; ++j) {
      const int64_t t = h->opt_step + 1 + j;
      h->h_status->ring_hyper[3 * j] = (float)schedule_lr(sched, h->cfg.lr, t);
      h->h_status->ring_hyper[3 * j + 1] = (float)(1.0 - std::pow((double)h->cfg.beta1, (double)t));
      h->h_status->ring_hyper[3 * j + 2] = (float)(1.0 - std::pow((double)h->cfg.beta2, (double)t));
    }
    CUDA_TRY(h, cudaMemcpyAsync(h->d_step_hyper, h->h_status->ring_hyper, 3 * kc * sizeof(float),
                                cudaMemcpyHostToDevice, h->stream));
    if (h->ev0) CUDA_TRY(h, cudaEventRecord(h->ev0, h->stream));
    {
      KParams kp = step_params(h, tokens + j0 * n, targets + j0 * n, h->launches + 1, h->cfg.lr, h->opt_step + 1);
      kp.nsteps = kc;
      kp.step_hyper = h->d_step_hyper;
      kp.loss_out = h->d_loss_ring;
      kp.status_out = h->d_status_ring;
      h->skip_release = -1;
      int rc = serve_prepare(h, kp, (int64_t)h->serve.per_step * kc);
      if (rc == GPT_OK) rc = launch_kernel(h, kp);
      if (rc != GPT_OK) {
        cudaStreamSynchronize(h->stream);
        h->poisoned = true;
        return rc;
      }
    }
    if (h->ev1) CUDA_TRY(h, cudaEventRecord(h->ev1, h->stream));
    CUDA_TRY(h, cudaMemcpyAsync(h->h_status->err, h->d_err, 4 * sizeof(uint32_t), cudaMemcpyDeviceToHost,
                                h->stream));
    CUDA_TRY(h, cudaMemcpyAsync(h->h_status->ring_loss, h->d_loss_ring, kc * sizeof(float),
                                cudaMemcpyDeviceToHost, h->stream));
    CUDA_TRY(h, cudaMemcpyAsync(h->h_status->ring_status, h->d_status_ring, kc * sizeof(uint32_t),
                                cudaMemcpyDeviceToHost, h->stream));
    CUDA_TRY(h, cudaStreamSynchronize(h->stream));
    if (h->ev0 && h->ev1) cudaEventElapsedTime(&h->last_kernel_ms, h->ev0, h->ev1);
    const uint32_t fatal = h->h_status->err[0];
    if (fatal) {
      h->poisoned = true;
      return fail(h, GPT_ERR_TIMEOUT, "device wait timed out in steps %d..%d of the call (code %u, task %u, "
                  "counter/barrier %u)", j0, j0 + kc - 1, fatal, h->h_status->err[2], h->h_status->err[3]);
    }
    h->launches += kc;
    if (losses) std::memcpy(losses + j0, h->h_status->ring_loss, kc * sizeof(float));
    int32_t good = kc;
    for (int32_t j = 0; j < kc; ++j)
      if (h->h_status->ring_status[j]) { good = j; break; }
    h->opt_step += good;
    if (good < kc) {  // the soft flag stayed raised for the rest of the chunk: no later update applied
      const uint32_t soft = h->h_status->ring_status[good];
      CUDA_TRY(h, cudaMemsetAsync(h->d_err + 1, 0, sizeof(uint32_t), h->stream));
      CUDA_TRY(h, cudaStreamSynchronize(h->stream));
      if (soft & kSoftBadToken)
        return fail(h, GPT_ERR_BAD_TOKEN, "token or target id outside [0, vocab) at step %d of the call",
                    j0 + good);
      return fail(h, GPT_ERR_NONFINITE, "non-finite loss %g at step %d of the call",
                  (double)h->h_status->ring_loss[good], j0 + good);
    }
  }
  h->err.clear();
  return GPT_OK;
}

}  // namespace

// ============================================================================
// C ABI
// ============================================================================
extern "C" {

void gpt_default_config(gpt_config* c) {
  if (!c) return;
  std::memset(c, 0, sizeof *c);
  c->n_layer = 12; c->d_model = 768; c->n_head = 12; c->d_mlp = 3072; c->vocab = 50304;
  c->seq_len = 512; c->batch = 8; c->dtype = GPT_DTYPE_BF16;
  c->linear_bias = 1; c->ln_bias = 1; c->tie_embeddings = 0; c->gelu_tanh = 1;
  c->lr = 6e-4f; c->beta1 = 0.9f; c->beta2 = 0.95f; c->eps = 1e-8f; c->weight_decay = 0.1f; c->ln_eps = 1e-5f;
  c->wd_on_1d = 0; c->wait_timeout_ms = 2000; c->deterministic = 1;
}

static int lm_ksplit_for(const gpt_config& c, int num_sms) {
  if (!is_bf16(c)) return 1;
  // The vocabulary-long reduction of the LM-head input gradient (which the
  // whole backward waits for) is split into the largest number of whole
  // k-block ranges, at most 8, whose tiles still fit in two waves: for the
  // 162M step 3 splits (288 tiles) measured 7.92 ms against 8.01 with 2 and
  // 7.95 with 6.
  const int N = c.batch * c.seq_len;
  const int tiles = (N / kTcBM) * ((c.d_model + 255) / 256);
  const int kblocks = c.vocab / kTcBK;
  int ks = 1;
  for (int k = 2; k <= 8; ++k)
    if (kblocks % k == 0 && tiles * k <= 2 * num_sms) ks = k;
  return ks;
}

size_t gpt_arena_bytes(const gpt_config* cfg) {
  if (!cfg) return 0;
  std::string why;
  if (validate(*cfg, &why) != GPT_OK) return 0;
  gpt tmp;
  tmp.cfg = *cfg;
  build_table(&tmp);
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return make_layout(*cfg, tmp.nparams, lm_ksplit_for(*cfg, sms)).total;
}

size_t gpt_param_count(const gpt_config* cfg) {
  if (!cfg) return 0;
  std::string why;
  if (validate(*cfg, &why) != GPT_OK) return 0;
  gpt tmp;
  tmp.cfg = *cfg;
  build_table(&tmp);
  return tmp.nparams;
}

int gpt_create(const gpt_config* cfg, uint64_t seed, void* cuda_stream, void* arena, size_t arena_bytes, gpt** out) {
  g_create_error.clear();
  if (!cfg || !out) return fail(nullptr, GPT_ERR_INVALID_ARG, "cfg and out must be non-NULL");
  std::string why;
  int rc = validate(*cfg, &why);
  if (rc != GPT_OK) return fail(nullptr, rc, "invalid config: %s", why.c_str());
  gpt* h = new (std::nothrow) gpt();
  if (!h) return fail(nullptr, GPT_ERR_OOM, "host allocation failed");
  h->cfg = *cfg;
  if (!h->cfg.wait_timeout_ms) h->cfg.wait_timeout_ms = 2000;
  const gpt_config& c = h->cfg;
  h->D = Dims{c.n_layer, c.d_model, c.n_head, c.d_model / c.n_head, c.d_mlp, c.vocab, c.seq_len, c.batch,
              c.batch * c.seq_len};
  h->stream = (cudaStream_t)cuda_stream;
  auto bail = [&](int code) {
    std::string msg = h->err;
    gpt_destroy(h);
    g_create_error = msg;
    return code;
  };
  if (cudaGetDevice(&h->device) != cudaSuccess) { fail(h, GPT_ERR_CUDA, "no CUDA device"); return bail(GPT_ERR_CUDA); }
  cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  int cc_major = 0, cc_minor = 0;
  cudaDeviceGetAttribute(&cc_major, cudaDevAttrComputeCapabilityMajor, h->device);
  cudaDeviceGetAttribute(&cc_minor, cudaDevAttrComputeCapabilityMinor, h->device);
  if (cc_major != 10 || cc_minor != 3) {
    fail(h, GPT_ERR_UNSUPPORTED, "compiled for sm_103a; device is sm_%d%d", cc_major, cc_minor);
    return bail(GPT_ERR_UNSUPPORTED);
  }
  build_table(h);
  const int lm_ks = lm_ksplit_for(c, h->num_sms);
  const Layout Lo = make_layout(c, h->nparams, lm_ks);
  // arena
  if (arena) {
    if (arena_bytes < Lo.total || (reinterpret_cast<uintptr_t>(arena) & 255)) {
      fail(h, GPT_ERR_INVALID_ARG, "arena must be 256-byte aligned and >= %zu bytes", Lo.total);
      return bail(GPT_ERR_INVALID_ARG);
    }
    h->arena = static_cast<uint8_t*>(arena);
  } else {
    if (cudaMalloc(&h->arena, Lo.total) != cudaSuccess) {
      cudaGetLastError();
      fail(h, GPT_ERR_OOM, "cudaMalloc of %zu arena bytes failed", Lo.total);
      return bail(GPT_ERR_OOM);
    }
    h->own_arena = true;
  }
  h->arena_bytes = Lo.total;
  h->params = reinterpret_cast<float*>(h->arena + Lo.params);
  h->grads = reinterpret_cast<float*>(h->arena + Lo.grads);
  h->m = reinterpret_cast<float*>(h->arena + Lo.m);
  h->v = reinterpret_cast<float*>(h->arena + Lo.v);
  h->shadow = is_bf16(c) ? reinterpret_cast<uint16_t*>(h->arena + Lo.shadow) : nullptr;
  h->loss_dev = reinterpret_cast<float*>(h->arena + Lo.loss);
  // graph
  rc = build_graph(h, Lo, lm_ks);
  if (rc != GPT_OK) return bail(rc);
  // metadata allocation: tasks | ops | tensor maps | counters | ticket | err | token staging
  Bump mb;
  const size_t o_tasks = mb.take(h->tasks.size() * sizeof(TaskDesc));
  const size_t o_ops = mb.take(h->ops.size() * sizeof(OpDesc));
  const size_t o_maps = mb.take(std::max<size_t>(1, h->tmaps.size()) * 128);
  const size_t o_ctr = mb.take((size_t)h->n_counters * sizeof(unsigned long long));
  const size_t o_tic = mb.take(2 * sizeof(unsigned long long));
  const size_t o_err = mb.take(4 * sizeof(uint32_t));
  const size_t o_tok = mb.take(2 * (size_t)h->D.N * sizeof(int32_t));
  const size_t o_ring = mb.take((size_t)kStepRing * (sizeof(float) + sizeof(uint32_t)));
  const size_t o_hyper = mb.take((size_t)kStepRing * 3 * sizeof(float));
  const size_t o_bar = mb.take(sizeof(unsigned long long));
  h->meta_bytes = mb.off;
  if (cudaMalloc(&h->meta, h->meta_bytes) != cudaSuccess) {
    cudaGetLastError();
    fail(h, GPT_ERR_OOM, "cudaMalloc of graph metadata failed");
    return bail(GPT_ERR_OOM);
  }
  h->d_tasks = reinterpret_cast<TaskDesc*>(h->meta + o_tasks);
  h->d_ops = reinterpret_cast<OpDesc*>(h->meta + o_ops);
  h->d_tmaps = h->meta + o_maps;
  h->d_counters = reinterpret_cast<unsigned long long*>(h->meta + o_ctr);
  h->d_ticket = reinterpret_cast<unsigned long long*>(h->meta + o_tic);
  h->d_err = reinterpret_cast<uint32_t*>(h->meta + o_err);
  h->d_tok_stage = reinterpret_cast<int32_t*>(h->meta + o_tok);
  h->d_loss_ring = reinterpret_cast<float*>(h->meta + o_ring);
  h->d_status_ring = reinterpret_cast<uint32_t*>(h->meta + o_ring + (size_t)kStepRing * sizeof(float));
  h->d_step_hyper = reinterpret_cast<float*>(h->meta + o_hyper);
  h->d_grid_bar = reinterpret_cast<unsigned long long*>(h->meta + o_bar);
  if (cudaMallocHost(&h->h_status, sizeof(gpt::Status)) != cudaSuccess) {
    cudaGetLastError();
    fail(h, GPT_ERR_OOM, "pinned host allocation failed");
    return bail(GPT_ERR_OOM);
  }
#define CREATE_TRY(call)                                                                       \
  do {                                                                                         \
    cudaError_t e_ = (call);                                                                   \
    if (e_ != cudaSuccess) {                                                                   \
      fail(h, GPT_ERR_CUDA, "%s failed: %s", #call, cudaGetErrorString(e_));                   \
      return bail(GPT_ERR_CUDA);                                                               \
    }                                                                                          \
  } while (0)
  CREATE_TRY(cudaMemcpyAsync(h->d_tasks, h->tasks.data(), h->tasks.size() * sizeof(TaskDesc),
                             cudaMemcpyHostToDevice, h->stream));
  CREATE_TRY(cudaMemcpyAsync(h->d_ops, h->ops.data(), h->ops.size() * sizeof(OpDesc), cudaMemcpyHostToDevice,
                             h->stream));
  for (size_t i = 0; i < h->tmaps.size(); ++i)
    CREATE_TRY(cudaMemcpyAsync(static_cast<uint8_t*>(h->d_tmaps) + 128 * i, h->tmaps[i].data(), 128,
                               cudaMemcpyHostToDevice, h->stream));
  // seeded initial weights on the host; m = v = 0; grads = 0
  {
    std::vector<float> hp(h->nparams);
    for (size_t t = 0; t < h->tensors.size(); ++t) {
      const TensorInfo& ti = h->tensors[t];
      const size_t n = (size_t)(ti.rows * ti.cols);
      float* dst = hp.data() + ti.offset;
      if (ti.init == INIT_NORMAL) normal_fill(dst, n, seed, t);
      else std::fill(dst, dst + n, ti.init == INIT_ONES ? 1.0f : 0.0f);
    }
    rc = fill_shadow_and_upload(h, hp.data());
    if (rc != GPT_OK) return bail(rc);
  }
  if (init_bias_pads(h, Lo) != GPT_OK) return bail(GPT_ERR_CUDA);
  if (c.rope) {  // rotary embedding table: (cos, sin) of t * 10000^(-2i/64), computed in double
    std::vector<float> cs((size_t)c.seq_len * 64);
    for (int t = 0; t < c.seq_len; ++t)
      for (int i = 0; i < 32; ++i) {
        const double th = (double)t * std::pow(10000.0, -2.0 * i / 64.0);
        cs[(size_t)t * 64 + 2 * i] = (float)std::cos(th);
        cs[(size_t)t * 64 + 2 * i + 1] = (float)std::sin(th);
      }
    CREATE_TRY(cudaMemcpyAsync(h->arena + Lo.rope, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice, h->stream));
    CREATE_TRY(cudaStreamSynchronize(h->stream));
  }
  CREATE_TRY(cudaMemsetAsync(h->grads, 0, h->nparams * 4, h->stream));
  CREATE_TRY(cudaMemsetAsync(h->m, 0, h->nparams * 4, h->stream));
  CREATE_TRY(cudaMemsetAsync(h->v, 0, h->nparams * 4, h->stream));
  // kernel + grid: every block must be resident (cooperative launch checks it)
  h->kernel = !is_bf16(c) ? step_kernel_fp32()
              : (c.rope || c.gated_mlp || c.tie_embeddings) ? step_kernel_bf16_ext() : step_kernel_bf16();
  h->smem_bytes = smem_needed(h);
  CREATE_TRY(cudaFuncSetAttribute(h->kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)h->smem_bytes));
  int per_sm = 0;
  CREATE_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, h->kernel, kThreads, h->smem_bytes));
  if (per_sm < 1) {
    fail(h, GPT_ERR_UNSUPPORTED, "kernel does not fit on an SM (%zu bytes shared memory)", h->smem_bytes);
    return bail(GPT_ERR_UNSUPPORTED);
  }
  h->grid = h->num_sms * std::min(per_sm, 1);
  CREATE_TRY(cudaEventCreate(&h->ev0));
  CREATE_TRY(cudaEventCreate(&h->ev1));
  if (reset_counters(h) != GPT_OK) return bail(GPT_ERR_CUDA);
#undef CREATE_TRY
  *out = h;
  return GPT_OK;
}

int gpt_train_step(gpt* h, const int32_t* tokens, const int32_t* targets, float* loss) {
  if (!h) return GPT_ERR_INVALID_ARG;
  if (!tokens || !targets) return fail(h, GPT_ERR_INVALID_ARG, "tokens and targets must be device pointers");
  return launch_step(h, tokens, targets, loss);
}

int gpt_train_step_host(gpt* h, const int32_t* tokens, const int32_t* targets, float* loss) {
  if (!h) return GPT_ERR_INVALID_ARG;
  if (!tokens || !targets) return fail(h, GPT_ERR_INVALID_ARG, "tokens and targets must be host pointers");
  const size_t n = (size_t)h->D.N;
  CUDA_TRY(h, cudaMemcpyAsync(h->d_tok_stage, tokens, n * 4, cudaMemcpyHostToDevice, h->stream));
  CUDA_TRY(h, cudaMemcpyAsync(h->d_tok_stage + n, targets, n * 4, cudaMemcpyHostToDevice, h->stream));
  return launch_step(h, h->d_tok_stage, h->d_tok_stage + n, loss);
}

float gpt_lr_at(const gpt_lr_schedule* sched, float base_lr, int64_t step) {
  if (!schedule_ok(sched) || step < 1) return -1.0f;
  return (float)schedule_lr(sched, base_lr, step);
}

int gpt_train_steps(gpt* h, const int32_t* tokens, const int32_t* targets, int32_t k,
                    const gpt_lr_schedule* sched, float* losses) {
  if (!h) return GPT_ERR_INVALID_ARG;
  if (!tokens || !targets || k < 1) return fail(h, GPT_ERR_INVALID_ARG, "tokens/targets must be device pointers, k >= 1");
  if (!schedule_ok(sched)) return fail(h, GPT_ERR_INVALID_ARG, "invalid learning-rate schedule");
  return train_steps(h, tokens, targets, k, sched, losses);
}

size_t gpt_num_params(const gpt* h) { return h ? h->nparams : 0; }
int gpt_num_tensors(const gpt* h) { return h ? (int)h->tensors.size() : 0; }

int gpt_tensor_info(const gpt* h, int i, const char** name, int64_t shape[2], size_t* offset) {
  if (!h || i < 0 || i >= (int)h->tensors.size()) return GPT_ERR_INVALID_ARG;
  const TensorInfo& t = h->tensors[i];
  if (name) *name = t.name.c_str();
  if (shape) { shape[0] = t.rows; shape[1] = t.cols; }
  if (offset) *offset = t.offset;
  return GPT_OK;
}

static int copy_out(gpt* h, float* dst, const float* src, size_t n) {
  if (!h || !dst) return GPT_ERR_INVALID_ARG;
  if (n != h->nparams) return fail(h, GPT_ERR_INVALID_ARG, "n must equal gpt_num_params (%zu)", h->nparams);
  CUDA_TRY(h, cudaMemcpyAsync(dst, src, n * 4, cudaMemcpyDeviceToHost, h->stream));
  CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  return GPT_OK;
}

int gpt_get_params(gpt* h, float* dst, size_t n) { return h ? copy_out(h, dst, h->params, n) : GPT_ERR_INVALID_ARG; }
int gpt_get_grads(gpt* h, float* dst, size_t n) { return h ? copy_out(h, dst, h->grads, n) : GPT_ERR_INVALID_ARG; }

int gpt_set_params(gpt* h, const float* src, size_t n) {
  if (!h || !src) return GPT_ERR_INVALID_ARG;
  if (n != h->nparams) return fail(h, GPT_ERR_INVALID_ARG, "n must equal gpt_num_params (%zu)", h->nparams);
  return fill_shadow_and_upload(h, src);
}

int gpt_get_opt_state(gpt* h, float* m, float* v, int64_t* step) {
  if (!h) return GPT_ERR_INVALID_ARG;
  if (m) CUDA_TRY(h, cudaMemcpyAsync(m, h->m, h->nparams * 4, cudaMemcpyDeviceToHost, h->stream));
  if (v) CUDA_TRY(h, cudaMemcpyAsync(v, h->v, h->nparams * 4, cudaMemcpyDeviceToHost, h->stream));
  CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  if (step) *step = h->opt_step;
  return GPT_OK;
}

int gpt_set_opt_state(gpt* h, const float* m, const float* v, int64_t step) {
  if (!h || step < 0) return GPT_ERR_INVALID_ARG;
  if (m) CUDA_TRY(h, cudaMemcpyAsync(h->m, m, h->nparams * 4, cudaMemcpyHostToDevice, h->stream));
  if (v) CUDA_TRY(h, cudaMemcpyAsync(h->v, v, h->nparams * 4, cudaMemcpyHostToDevice, h->stream));
  CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  h->opt_step = step;
  return GPT_OK;
}

int gpt_serve_end(gpt* h) {
  if (!h) return GPT_ERR_INVALID_ARG;
  if (h->serve.mem) {
    cudaStreamSynchronize(h->stream);
    cudaFree(h->serve.mem);
  }
  h->serve = gpt::Serve{};
  return GPT_OK;
}

int gpt_serve_begin(gpt* h, const int32_t* prompt, int32_t n_prompt, int32_t max_new, int32_t blocks,
                    int32_t tokens_per_step, int64_t first_step) {
  if (!h) return GPT_ERR_INVALID_ARG;
  const gpt_config& c = h->cfg;
  const Dims& D = h->D;
  if (!is_bf16(c) || c.rope || c.gated_mlp || c.tie_embeddings)
    return fail(h, GPT_ERR_UNSUPPORTED, "serving runs the bf16 model with learned positions, a GELU MLP and an "
                "untied LM head");
  if (!prompt || n_prompt < 1 || max_new < 1 || (int64_t)n_prompt + max_new > D.T || blocks < 1 ||
      blocks >= h->grid || tokens_per_step < 0 || first_step < 0 || first_step > ((int64_t)1 << 40))
    return fail(h, GPT_ERR_INVALID_ARG, "need a prompt of >= 1 token, max_new >= 1, n_prompt + max_new <= %d, "
                "1 <= blocks < %d, tokens_per_step >= 0, 0 <= first_step <= 2^40", D.T, h->grid);
  for (int32_t i = 0; i < n_prompt; ++i)
    if (prompt[i] < 0 || prompt[i] >= D.V) return fail(h, GPT_ERR_BAD_TOKEN, "prompt token %d outside [0, vocab)", i);
  gpt_serve_end(h);
  gpt::Serve& sv = h->serve;
  const int C = D.C, F = D.F, L = D.L, T = D.T, V = D.V;
  const int n_slices = (V + kServeRows - 1) / kServeRows;
  // ops of one step, in chain order
  std::vector<ServeOp> ops;
  Bump mb;
  const size_t o_kv = mb.take((size_t)L * 2 * T * C * 4);
  const size_t o_x = mb.take((size_t)C * 4), o_a = mb.take((size_t)C * 4), o_q = mb.take((size_t)C * 4);
  const size_t o_o = mb.take((size_t)C * 4), o_h = mb.take((size_t)F * 4);
  const size_t o_pm = mb.take((size_t)n_slices * 4), o_pi = mb.take((size_t)n_slices * 4);
  const size_t o_seq = mb.take((size_t)T * 4);
  const size_t o_tic = mb.take(8);
  const int nops = 1 + 7 * L + 3;
  const size_t o_ctr = mb.take((size_t)nops * 8);
  const size_t o_ops = mb.take((size_t)nops * sizeof(ServeOp));
  const size_t o_par = mb.take(sizeof(ServeParams));
  // tasks per step
  int P = 0;
  std::vector<int32_t> task_op, task_idx;
  const size_t o_task = mb.take((size_t)(1 + L * (2 + 3 * C / kServeRows + D.H + C / kServeRows + F / kServeRows +
                                                 C / kServeRows) + 2 + n_slices + 8) * 8);
  if (cudaMalloc(&sv.mem, mb.off) != cudaSuccess) {
    cudaGetLastError();
    sv.mem = nullptr;
    return fail(h, GPT_ERR_OOM, "cudaMalloc of %zu serving bytes failed", mb.off);
  }
  uint8_t* M = sv.mem;
  auto F32 = [&](size_t off) { return reinterpret_cast<float*>(M + off); };
  float* kv = F32(o_kv);
  auto Wt = [&](int t) { return t < 0 ? nullptr : h->shadow + h->tensors[t].offset; };
  auto Pt = [&](int t) { return t < 0 ? (const float*)nullptr : (const float*)(h->params + h->tensors[t].offset); };
  auto add = [&](int type, int ntasks, int epi, int K, int N, const uint16_t* W, const float* bias, const float* in,
                 float* out, float* kc, float* vc, const float* g, const float* b) {
    ServeOp o{type, ntasks, epi, K, N, W, bias, in, out, kc, vc, g, b};
    for (int i = 0; i < ntasks; ++i) {
      task_op.push_back((int32_t)ops.size());
      task_idx.push_back(i);
    }
    ops.push_back(o);
  };
  auto rows = [](int N) { return (N + kServeRows - 1) / kServeRows; };
  add(SV_EMBED, 1, SE_STORE, 0, C, nullptr, nullptr, nullptr, F32(o_x), nullptr, nullptr, nullptr, nullptr);
  for (int l = 0; l < L; ++l) {
    const TensorIds& id = h->lid[l];
    float* kc = kv + (size_t)l * 2 * T * C;
    float* vc = kc + (size_t)T * C;
    add(SV_LN, 1, SE_STORE, 0, C, nullptr, nullptr, F32(o_x), F32(o_a), nullptr, nullptr, Pt(id.ln1_g), Pt(id.ln1_b));
    add(SV_GEMV, rows(3 * C), SE_QKV, C, 3 * C, Wt(id.w_qkv), Pt(id.b_qkv), F32(o_a), F32(o_q), kc, vc, nullptr,
        nullptr);
    add(SV_ATTN, D.H, SE_STORE, 0, C, nullptr, nullptr, F32(o_q), F32(o_o), kc, vc, nullptr, nullptr);
    add(SV_GEMV, rows(C), SE_RESID, C, C, Wt(id.w_o), Pt(id.b_o), F32(o_o), F32(o_x), nullptr, nullptr, nullptr,
        nullptr);
    add(SV_LN, 1, SE_STORE, 0, C, nullptr, nullptr, F32(o_x), F32(o_a), nullptr, nullptr, Pt(id.ln2_g), Pt(id.ln2_b));
    add(SV_GEMV, rows(F), SE_GELU, C, F, Wt(id.w_1), Pt(id.b_1), F32(o_a), F32(o_h), nullptr, nullptr, nullptr,
        nullptr);
    add(SV_GEMV, rows(C), SE_RESID, F, C, Wt(id.w_2), Pt(id.b_2), F32(o_h), F32(o_x), nullptr, nullptr, nullptr,
        nullptr);
  }
  add(SV_LN, 1, SE_STORE, 0, C, nullptr, nullptr, F32(o_x), F32(o_a), nullptr, nullptr, Pt(h->t_lnf_g),
      Pt(h->t_lnf_b));
  add(SV_GEMV, n_slices, SE_LOGITS, C, V, Wt(h->t_wlm), nullptr, F32(o_a), nullptr, nullptr, nullptr, nullptr,
      nullptr);
  add(SV_ARGMAX, 1, SE_STORE, 0, 0, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr);
  P = (int)task_op.size();
  if ((int)ops.size() != nops || (size_t)P * 8 > mb.off - o_task) {
    gpt_serve_end(h);
    return fail(h, GPT_ERR_UNSUPPORTED, "serving graph size mismatch");
  }
  ServeParams& sp = sv.host;
  std::memset(&sp, 0, sizeof sp);
  sp.ops = reinterpret_cast<const ServeOp*>(M + o_ops);
  sp.nops = nops;
  sp.task_op = reinterpret_cast<const int32_t*>(M + o_task);
  sp.task_idx = reinterpret_cast<const int32_t*>(M + o_task) + P;
  sp.P = P;
  sp.counters = reinterpret_cast<unsigned long long*>(M + o_ctr);
  sp.ticket = reinterpret_cast<unsigned long long*>(M + o_tic);
  sp.base = (unsigned long long)first_step;
  sp.limit = 0;
  sp.seq = reinterpret_cast<int32_t*>(M + o_seq);
  sp.n_prompt = n_prompt;
  sp.C = C; sp.H = D.H; sp.T = T; sp.V = V;
  sp.ln_eps = c.ln_eps;
  sp.gelu_tanh = c.gelu_tanh;
  sp.wte = Pt(h->t_wte);
  sp.wpe = Pt(h->t_wpe);
  sp.part_max = F32(o_pm);
  sp.part_idx = reinterpret_cast<int32_t*>(M + o_pi);
  sp.n_slices = n_slices;
  // counters as if first_step steps had completed: op o at first_step x its tasks
  std::vector<unsigned long long> ctr(nops);
  for (int o = 0; o < nops; ++o) ctr[o] = (unsigned long long)first_step * (unsigned long long)ops[o].ntasks;
  std::vector<int32_t> seq(T, 0);
  std::memcpy(seq.data(), prompt, (size_t)n_prompt * 4);
  std::vector<int32_t> tasks(task_op);
  tasks.insert(tasks.end(), task_idx.begin(), task_idx.end());
  sv.d_params = reinterpret_cast<ServeParams*>(M + o_par);
  cudaError_t e = cudaMemsetAsync(M, 0, mb.off, h->stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(M + o_ops, ops.data(), ops.size() * sizeof(ServeOp), cudaMemcpyHostToDevice, h->stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(M + o_task, tasks.data(), tasks.size() * 4, cudaMemcpyHostToDevice, h->stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(M + o_ctr, ctr.data(), ctr.size() * 8, cudaMemcpyHostToDevice, h->stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(M + o_seq, seq.data(), seq.size() * 4, cudaMemcpyHostToDevice, h->stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(sv.d_params, &sp, sizeof sp, cudaMemcpyHostToDevice, h->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
  if (e != cudaSuccess) {
    gpt_serve_end(h);
    return fail(h, GPT_ERR_CUDA, "serving set-up failed: %s", cudaGetErrorString(e));
  }
  sv.active = true;
  sv.blocks = blocks;
  sv.n_prompt = n_prompt;
  sv.n_new = max_new;
  sv.per_step = tokens_per_step;
  sv.steps_total = (int64_t)n_prompt - 1 + max_new;
  sv.steps_done = 0;
  sv.base = (unsigned long long)first_step;
  sv.P = P;
  return GPT_OK;
}

int gpt_serve_run(gpt* h, int32_t max_steps, float* kernel_ms) {
  if (!h) return GPT_ERR_INVALID_ARG;
  if (!h->serve.active) return fail(h, GPT_ERR_INVALID_ARG, "no serving session (gpt_serve_begin)");
  if (max_steps < 1) return fail(h, GPT_ERR_INVALID_ARG, "max_steps must be >= 1");
  if (h->poisoned) return fail(h, GPT_ERR_POISONED, "handle poisoned by an earlier timeout; call gpt_reset");
  if (h->serve.steps_done >= h->serve.steps_total) return GPT_OK;
  // a launch whose training blocks have no task: only the serving blocks work, and no
  // training epoch, ticket or grid-barrier arrival is consumed
  KParams kp = step_params(h, h->d_tok_stage, h->d_tok_stage, h->launches + 1, h->cfg.lr, h->opt_step + 1);
  kp.ntasks = 0;
  kp.grid_bar = nullptr;
  kp.trace = nullptr;
  kp.skip_release = -1;
  int rc = serve_prepare(h, kp, max_steps);
  if (rc != GPT_OK) return rc;
  if (h->ev0) CUDA_TRY(h, cudaEventRecord(h->ev0, h->stream));
  rc = launch_kernel(h, kp);
  if (rc != GPT_OK) return rc;
  if (h->ev1) CUDA_TRY(h, cudaEventRecord(h->ev1, h->stream));
  uint32_t err[4] = {0, 0, 0, 0};
  CUDA_TRY(h, cudaMemcpyAsync(err, h->d_err, sizeof err, cudaMemcpyDeviceToHost, h->stream));
  CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  if (h->ev0 && h->ev1) cudaEventElapsedTime(&h->last_kernel_ms, h->ev0, h->ev1);
  if (kernel_ms) *kernel_ms = h->last_kernel_ms;
  if (err[0]) {
    h->poisoned = true;
    return fail(h, GPT_ERR_TIMEOUT, "serving wait timed out (code %u, task %u, counter %u)", err[0], err[2], err[3]);
  }
  return GPT_OK;
}

int gpt_serve_tokens(gpt* h, int32_t* dst, int32_t cap, int32_t* n) {
  if (!h || !n) return GPT_ERR_INVALID_ARG;
  if (!h->serve.active) return fail(h, GPT_ERR_INVALID_ARG, "no serving session (gpt_serve_begin)");
  const gpt::Serve& sv = h->serve;
  const int64_t produced = std::max<int64_t>(0, sv.steps_done + 1 - sv.n_prompt);
  *n = (int32_t)produced;
  if (dst && produced > 0) {
    const int32_t m = (int32_t)std::min<int64_t>(produced, cap);
    CUDA_TRY(h, cudaMemcpyAsync(dst, sv.host.seq + sv.n_prompt, (size_t)m * 4, cudaMemcpyDeviceToHost, h->stream));
    CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  }
  return GPT_OK;
}

int gpt_run_ops(gpt* h, int32_t op_first, int32_t op_count, const int32_t* tokens, const int32_t* targets,
                int32_t reps, float* kernel_ms) {
  if (!h) return GPT_ERR_INVALID_ARG;
  const int nops = (int)h->ops.size();
  if (!tokens || !targets || op_first < 0 || op_count < 1 || reps < 1 || reps > 1000 ||
      (int64_t)op_first + op_count > nops)
    return fail(h, GPT_ERR_INVALID_ARG, "need device tokens/targets, 0 <= op_first, op_first + op_count <= %d, "
                "1 <= reps <= 1000", nops);
  if (h->poisoned) return fail(h, GPT_ERR_POISONED, "handle poisoned by an earlier timeout; call gpt_reset");
  // the range's tasks in the step's ticket order; the range owns the contiguous
  // counters [c_lo, c_hi), and waits on counters outside it are dropped (those
  // producers' outputs are taken as the arena holds them)
  const int last = op_first + op_count - 1;
  const int c_lo = h->op_ctr0[op_first], c_hi = h->op_ctr0[last] + h->op_nblk[last];
  std::vector<TaskDesc> sub;
  for (const TaskDesc& t : h->tasks) {
    if (t.op < op_first || t.op > last) continue;
    TaskDesc u = t;
    u.nwait = 0;
    for (int w = 0; w < t.nwait; ++w)
      if (t.wait[w].first >= c_lo && t.wait[w].first < c_hi) u.wait[u.nwait++] = t.wait[w];
    sub.push_back(u);
  }
  Bump mb;
  const size_t o_tasks = mb.take(sub.size() * sizeof(TaskDesc));
  const size_t o_ctr = mb.take((size_t)h->n_counters * sizeof(unsigned long long));
  const size_t o_tic = mb.take(2 * sizeof(unsigned long long));
  const size_t o_err = mb.take(4 * sizeof(uint32_t));
  uint8_t* d = nullptr;
  if (cudaMalloc(&d, mb.off) != cudaSuccess) {
    cudaGetLastError();
    return fail(h, GPT_ERR_OOM, "cudaMalloc of %zu bytes failed", mb.off);
  }
  std::vector<cudaEvent_t> ev(2 * (size_t)reps, nullptr);
  int rc = GPT_OK;
  uint32_t err[4] = {0, 0, 0, 0};
  do {
    if (cudaMemcpyAsync(d + o_tasks, sub.data(), sub.size() * sizeof(TaskDesc), cudaMemcpyHostToDevice, h->stream) ||
        cudaMemsetAsync(d + o_ctr, 0, mb.off - o_ctr, h->stream)) {
      rc = fail(h, GPT_ERR_CUDA, "set-up copies failed");
      break;
    }
    for (auto& e : ev)
      if (cudaEventCreate(&e) != cudaSuccess) rc = fail(h, GPT_ERR_CUDA, "cudaEventCreate failed");
    if (rc != GPT_OK) break;
    for (int r = 0; r < reps && rc == GPT_OK; ++r) {
      // epochs 1..reps on counters that start at zero: no reset between launches
      KParams kp = step_params(h, tokens, targets, (unsigned long long)r + 1, h->cfg.lr, h->opt_step + 1);
      kp.tasks = reinterpret_cast<const TaskDesc*>(d + o_tasks);
      kp.ntasks = (int64_t)sub.size();
      kp.counters = reinterpret_cast<unsigned long long*>(d + o_ctr);
      kp.tickets = reinterpret_cast<unsigned long long*>(d + o_tic);
      kp.err = reinterpret_cast<uint32_t*>(d + o_err);
      kp.skip_release = -1;
      kp.trace = nullptr;
      kp.grid_bar = nullptr;  // the handle's step barrier counts the handle's own steps only
      cudaEventRecord(ev[2 * r], h->stream);
      rc = launch_kernel(h, kp);
      cudaEventRecord(ev[2 * r + 1], h->stream);
    }
    if (cudaMemcpyAsync(err, d + o_err, sizeof err, cudaMemcpyDeviceToHost, h->stream) ||
        cudaStreamSynchronize(h->stream))
      rc = fail(h, GPT_ERR_CUDA, "run of the op range failed");
  } while (0);
  if (rc == GPT_OK && err[0])
    rc = fail(h, GPT_ERR_TIMEOUT, "a wait timed out in the op range (code %u, task %u, counter %u)", err[0], err[2],
              err[3]);
  if (rc == GPT_OK && kernel_ms) {
    double sum = 0.0;
    for (int r = 0; r < reps; ++r) {
      float ms = 0.f;
      cudaEventElapsedTime(&ms, ev[2 * r], ev[2 * r + 1]);
      sum += ms;
    }
    *kernel_ms = (float)(sum / reps);
  }
  for (auto& e : ev)
    if (e) cudaEventDestroy(e);
  cudaStreamSynchronize(h->stream);
  cudaFree(d);
  return rc;
}

int gpt_debug_skip_release(gpt* h, int64_t task_index) {
  if (!h || task_index < -1 || task_index >= (int64_t)h->tasks.size()) return GPT_ERR_INVALID_ARG;
  h->skip_release = task_index;
  return GPT_OK;
}

int gpt_reset(gpt* h) {
  if (!h) return GPT_ERR_INVALID_ARG;
  return reset_counters(h);
}

int gpt_graph_info(const gpt* h, int64_t* n_tasks, int32_t* grid, int32_t* block) {
  if (!h) return GPT_ERR_INVALID_ARG;
  if (n_tasks) *n_tasks = (int64_t)h->tasks.size();
  if (grid) *grid = h->grid;
  if (block) *block = kThreads;
  return GPT_OK;
}

int gpt_trace_enable(gpt* h, int32_t on) {
  if (!h) return GPT_ERR_INVALID_ARG;
  if (on && !h->d_trace) {
    const size_t bytes = (h->tasks.size() * 4 + (size_t)h->grid * 8) * sizeof(unsigned long long);
    if (cudaMalloc(&h->d_trace, bytes) != cudaSuccess) {
      cudaGetLastError();
      h->d_trace = nullptr;
      return fail(h, GPT_ERR_OOM, "cudaMalloc of the trace buffer failed");
    }
    CUDA_TRY(h, cudaMemsetAsync(h->d_trace, 0, bytes, h->stream));
    CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  } else if (!on && h->d_trace) {
    cudaStreamSynchronize(h->stream);
    cudaFree(h->d_trace);
    h->d_trace = nullptr;
  }
  return GPT_OK;
}

int gpt_get_trace(gpt* h, uint64_t* dst, size_t n) {
  if (!h || !dst) return GPT_ERR_INVALID_ARG;
  if (!h->d_trace) return fail(h, GPT_ERR_INVALID_ARG, "tracing is off (gpt_trace_enable)");
  if (n != h->tasks.size() * 4 && n != h->tasks.size() * 4 + (size_t)h->grid * 8)
    return fail(h, GPT_ERR_INVALID_ARG, "n must be 4 * n_tasks (+ 8 * grid for the GEMM role states)");
  CUDA_TRY(h, cudaMemcpyAsync(dst, h->d_trace, n * 8, cudaMemcpyDeviceToHost, h->stream));
  CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  return GPT_OK;
}

int gpt_last_kernel_ms(const gpt* h, float* ms) {
  if (!h || !ms) return GPT_ERR_INVALID_ARG;
  *ms = h->last_kernel_ms;
  return GPT_OK;
}

const char* gpt_last_error(const gpt* h) { return h ? h->err.c_str() : g_create_error.c_str(); }

void gpt_destroy(gpt* h) {
  if (!h) return;
  if (h->stream || h->meta || h->arena) cudaStreamSynchronize(h->stream);
  if (h->meta) cudaFree(h->meta);
  if (h->own_arena && h->arena) cudaFree(h->arena);
  if (h->h_status) cudaFreeHost(h->h_status);
  if (h->d_trace) cudaFree(h->d_trace);
  if (h->serve.mem) cudaFree(h->serve.mem);
  if (h->ev0) cudaEventDestroy(h->ev0);
  if (h->ev1) cudaEventDestroy(h->ev1);
  delete h;
}

// Runs the ops/tasks already built in h once (test hooks): graph metadata in a
// temporary allocation, one launch of the persistent kernel, then freed.
static int run_test_graph(gpt& h, int32_t dtype) {
  Bump mb;
  const size_t o_tasks = mb.take(h.tasks.size() * sizeof(TaskDesc));
  const size_t o_ops = mb.take(h.ops.size() * sizeof(OpDesc));
  const size_t o_maps = mb.take(std::max<size_t>(1, h.tmaps.size()) * 128);
  const size_t o_ctr = mb.take((size_t)h.n_counters * sizeof(unsigned long long));
  const size_t o_tic = mb.take(2 * sizeof(unsigned long long));
  const size_t o_err = mb.take(4 * sizeof(uint32_t));
  const size_t o_loss = mb.take(sizeof(float));
  h.meta_bytes = mb.off;
  if (cudaMalloc(&h.meta, h.meta_bytes) != cudaSuccess) {
    cudaGetLastError();
    h.meta = nullptr;
    return fail(nullptr, GPT_ERR_OOM, "cudaMalloc failed");
  }
  h.d_tasks = reinterpret_cast<TaskDesc*>(h.meta + o_tasks);
  h.d_ops = reinterpret_cast<OpDesc*>(h.meta + o_ops);
  h.d_tmaps = h.meta + o_maps;
  h.d_counters = reinterpret_cast<unsigned long long*>(h.meta + o_ctr);
  h.d_ticket = reinterpret_cast<unsigned long long*>(h.meta + o_tic);
  h.d_err = reinterpret_cast<uint32_t*>(h.meta + o_err);
  h.loss_dev = reinterpret_cast<float*>(h.meta + o_loss);
  int result = GPT_OK;
  do {
    if (cudaMallocHost(&h.h_status, sizeof(gpt::Status)) != cudaSuccess) { result = GPT_ERR_OOM; break; }
    if (cudaMemcpyAsync(h.d_tasks, h.tasks.data(), h.tasks.size() * sizeof(TaskDesc), cudaMemcpyHostToDevice,
                        h.stream) ||
        cudaMemcpyAsync(h.d_ops, h.ops.data(), h.ops.size() * sizeof(OpDesc), cudaMemcpyHostToDevice, h.stream)) {
      result = GPT_ERR_CUDA;
      break;
    }
    bool bad = false;
    for (size_t i = 0; i < h.tmaps.size(); ++i)
      bad |= cudaMemcpyAsync(static_cast<uint8_t*>(h.d_tmaps) + 128 * i, h.tmaps[i].data(), 128,
                             cudaMemcpyHostToDevice, h.stream) != cudaSuccess;
    if (bad) { result = GPT_ERR_CUDA; break; }
    h.kernel = dtype == GPT_DTYPE_BF16 ? step_kernel_bf16() : step_kernel_fp32();
    h.smem_bytes = dtype == GPT_DTYPE_BF16 ? (size_t)kTcSmemBytes + 4 * kEpiStageBytes + 1024 : smem_needed(&h);
    if (cudaFuncSetAttribute(h.kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)h.smem_bytes)) {
      result = GPT_ERR_CUDA;
      break;
    }
    h.grid = h.num_sms;
    if (reset_counters(&h) != GPT_OK) { result = GPT_ERR_CUDA; break; }
    result = launch_step(&h, reinterpret_cast<const int32_t*>(h.meta), reinterpret_cast<const int32_t*>(h.meta),
                         nullptr);
  } while (0);
  if (result != GPT_OK) g_create_error = h.err.empty() ? std::string("test graph failed") : h.err;
  cudaStreamSynchronize(h.stream);
  cudaFree(h.meta);
  h.meta = nullptr;
  if (h.h_status) cudaFreeHost(h.h_status);
  h.h_status = nullptr;
  return result;
}

int gpt_test_gemm(int32_t dtype, int32_t M, int32_t N, int32_t K, const void* A, int64_t lda, int32_t a_mn,
                  const void* B, int64_t ldb, int32_t b_mn, float* C, int64_t ldc, int32_t ksplit,
                  void* cuda_stream, float* kernel_ms) {
  g_create_error.clear();
  if (!A || !B || !C || M < 1 || N < 1 || K < 1 || ksplit < 1 || (dtype != GPT_DTYPE_FP32 && dtype != GPT_DTYPE_BF16))
    return fail(nullptr, GPT_ERR_INVALID_ARG, "bad GEMM test arguments");
  if (dtype == GPT_DTYPE_BF16 && (K % (kTcBK * ksplit) || N % 64 || lda % 8 || ldb % 8 || ldc % 4))
    return fail(nullptr, GPT_ERR_UNSUPPORTED, "bf16 GEMM test: K %% (64 ksplit), N %% 64, lda/ldb %% 8 must be 0");
  gpt h;
  gpt_default_config(&h.cfg);
  h.cfg.dtype = dtype;
  h.stream = (cudaStream_t)cuda_stream;
  cudaGetDevice(&h.device);
  cudaDeviceGetAttribute(&h.num_sms, cudaDevAttrMultiProcessorCount, h.device);
  h.D = Dims{1, 64, 1, 64, 64, 64, 1, 1, 1};
  OpDesc o;
  int rc = gemm_op(&h, &o, M, N, K, {A, lda, a_mn != 0}, {B, ldb, b_mn != 0}, EPI_F32, ksplit);
  if (rc != GPT_OK) { g_create_error = h.err; return rc; }
  o.gemm.out = C; o.gemm.ldo = ldc; o.gemm.split_stride = (int64_t)M * ldc;
  Builder bld{&h};
  bld.add(o, {});
  bld.finish(h.num_sms);
  if (kernel_ms) {
    cudaEventCreate(&h.ev0);
    cudaEventCreate(&h.ev1);
  }
  rc = run_test_graph(h, dtype);
  if (kernel_ms) {
    *kernel_ms = h.last_kernel_ms;
    cudaEventDestroy(h.ev0);
    cudaEventDestroy(h.ev1);
    h.ev0 = h.ev1 = nullptr;
  }
  return rc;
}

int gpt_test_gemm_epilogue(int32_t M, int32_t N, int32_t K, const void* A, int64_t lda, int32_t a_mn,
                           const void* B, int64_t ldb, int32_t b_mn, int32_t epi, int32_t gelu_tanh, void* out,
                           int64_t ldo, void* out2, int64_t ldo2, const float* bias, const void* src, int64_t lds,
                           void* cuda_stream, float* kernel_ms) {
  g_create_error.clear();
  if (!A || !B || !out || M < 1 || N < 1 || K < 1 || ldo < N)
    return fail(nullptr, GPT_ERR_INVALID_ARG, "bad GEMM epilogue test arguments");
  if (epi != EPI_STORE && epi != EPI_RESID && epi != EPI_GELU && epi != EPI_GELU_BWD)
    return fail(nullptr, GPT_ERR_INVALID_ARG, "epi must be 0 (store), 1 (residual), 2 (GELU) or 4 (GELU backward)");
  if ((epi == EPI_GELU && (!out2 || ldo2 < N || ldo2 % 4)) || ((epi == EPI_RESID || epi == EPI_GELU_BWD) &&
                                                              (!src || lds < N || lds % 4)))
    return fail(nullptr, GPT_ERR_INVALID_ARG, "missing or misaligned second output / source operand");
  if (K % kTcBK || N % 64 || lda % 8 || ldb % 8 || ldo % 4)
    return fail(nullptr, GPT_ERR_UNSUPPORTED, "GEMM epilogue test: K %% 64, N %% 64, lda/ldb %% 8, ldo %% 4 must be 0");
  gpt h;
  gpt_default_config(&h.cfg);
  h.cfg.dtype = GPT_DTYPE_BF16;
  h.cfg.gelu_tanh = gelu_tanh;
  h.stream = (cudaStream_t)cuda_stream;
  cudaGetDevice(&h.device);
  cudaDeviceGetAttribute(&h.num_sms, cudaDevAttrMultiProcessorCount, h.device);
  h.D = Dims{1, 64, 1, 64, 64, 64, 1, 1, 1};
  OpDesc o;
  int rc = gemm_op(&h, &o, M, N, K, {A, lda, a_mn != 0}, {B, ldb, b_mn != 0}, epi, 1);
  if (rc != GPT_OK) { g_create_error = h.err; return rc; }
  o.gemm.out = out; o.gemm.ldo = ldo;
  o.gemm.out2 = out2; o.gemm.ldo2 = ldo2;
  o.gemm.bias = epi == EPI_GELU_BWD ? nullptr : bias;
  if (epi == EPI_RESID) {  // the output holds the residual first; the epilogue adds into it
    if (cudaMemcpy2DAsync(out, (size_t)ldo * 4, src, (size_t)lds * 4, (size_t)N * 4, (size_t)M,
                          cudaMemcpyDeviceToDevice, h.stream) != cudaSuccess)
      return fail(nullptr, GPT_ERR_CUDA, "residual copy failed");
    o.gemm.resid = nullptr;
  }
  if (epi == EPI_GELU_BWD) { o.gemm.aux = src; o.gemm.ldaux = lds; }
  Builder bld{&h};
  const int op_id = bld.add(o, {});
  if (epi == EPI_RESID && h.ops[op_id].gemm.c_map < 0)
    return fail(nullptr, GPT_ERR_UNSUPPORTED, "residual epilogue: output not TMA-addressable (16-byte aligned base)");
  bld.finish(h.num_sms);
  if (kernel_ms) {
    cudaEventCreate(&h.ev0);
    cudaEventCreate(&h.ev1);
  }
  rc = run_test_graph(h, GPT_DTYPE_BF16);
  if (kernel_ms) {
    *kernel_ms = h.last_kernel_ms;
    cudaEventDestroy(h.ev0);
    cudaEventDestroy(h.ev1);
    h.ev0 = h.ev1 = nullptr;
  }
  return rc;
}

int gpt_test_attention(int32_t dtype, int32_t B, int32_t T, int32_t H, int32_t d, const void* qkv, void* o,
                       float* lse, const void* dout, void* dqkv, float* scratch, void* cuda_stream) {
  g_create_error.clear();
  if (!qkv || !o || !lse || !dout || !dqkv || !scratch || B < 1 || T < 1 || H < 1 || d < 1 ||
      (dtype != GPT_DTYPE_FP32 && dtype != GPT_DTYPE_BF16))
    return fail(nullptr, GPT_ERR_INVALID_ARG, "bad attention test arguments");
  if (dtype == GPT_DTYPE_BF16 && (d != 64 || T % 128))
    return fail(nullptr, GPT_ERR_UNSUPPORTED, "bf16 attention needs head_dim 64 and T %% 128 == 0");
  if (dtype == GPT_DTYPE_FP32 && (T > 1024 || d > 128))
    return fail(nullptr, GPT_ERR_UNSUPPORTED, "fp32 attention needs T <= 1024 and head_dim <= 128");
  gpt h;
  gpt_default_config(&h.cfg);
  h.cfg.dtype = dtype;
  h.cfg.n_head = H; h.cfg.d_model = H * d; h.cfg.seq_len = T; h.cfg.batch = B;
  h.stream = (cudaStream_t)cuda_stream;
  cudaGetDevice(&h.device);
  cudaDeviceGetAttribute(&h.num_sms, cudaDevAttrMultiProcessorCount, h.device);
  h.D = Dims{1, H * d, H, d, 64, 64, T, B, B * T};
  const int qblock = T <= 512 ? 64 : 32;
  AttnArgs att{qkv, o, lse, dout, dqkv, scratch, B, T, H, d, H * d, qblock, 1.0f / std::sqrt((float)d),
               H * d, nullptr, -1, -1};
  if (dtype == GPT_DTYPE_BF16) {  // TMA boxes of one head (64 columns) x 128 tokens
    att.qkv_map = make_tmap(&h, qkv, 3 * H * d, (int64_t)B * T, 3 * H * d, 128);
    att.do_map = make_tmap(&h, dout, H * d, (int64_t)B * T, H * d, 128);
    if (att.qkv_map < 0 || att.do_map < 0) return fail(nullptr, GPT_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  }
  Builder bld{&h};
  OpDesc op = blank(OP_ATTN_FWD, dtype == GPT_DTYPE_BF16 ? B * H * (T / 128) : B * H * ((T + qblock - 1) / qblock));
  op.attn = att;
  const int f = bld.add(op, {});
  if (dtype == GPT_DTYPE_BF16) {
    op = blank(OP_ATTN_BWD_PRE, (B * T + 63) / 64);
    op.attn = att;
    const int pre = bld.add(op, {f});
    op = blank(OP_ATTN_BWD_KV, B * H * (T / 128));
    op.attn = att;
    bld.add(op, {pre});
    op = blank(OP_ATTN_BWD_Q, B * H * (T / 128));
    op.attn = att;
    bld.add(op, {pre});
  } else {
    op = blank(OP_ATTN_BWD, B * H);
    op.attn = att;
    bld.add(op, {f});
  }
  bld.finish(h.num_sms);
  return run_test_graph(h, dtype);
}

int gpt_init_params_host(const gpt_config* cfg, uint64_t seed, float* dst, size_t n) {
  if (!cfg || !dst) return fail(nullptr, GPT_ERR_INVALID_ARG, "cfg and dst must be non-NULL");
  std::string why;
  int rc = validate(*cfg, &why);
  if (rc != GPT_OK) return fail(nullptr, rc, "invalid config: %s", why.c_str());
  gpt h;
  h.cfg = *cfg;
  build_table(&h);
  if (n != h.nparams) return fail(nullptr, GPT_ERR_INVALID_ARG, "n must be %zu", h.nparams);
  for (size_t t = 0; t < h.tensors.size(); ++t) {
    const TensorInfo& ti = h.tensors[t];
    const size_t cnt = (size_t)(ti.rows * ti.cols);
    float* d = dst + ti.offset;
    if (ti.init == INIT_NORMAL) normal_fill(d, cnt, seed, t);
    else std::fill(d, d + cnt, ti.init == INIT_ONES ? 1.0f : 0.0f);
  }
  return GPT_OK;
}

int gpt_graph_describe(const gpt_config* cfg, int32_t num_sms, int64_t* n_tasks, int32_t* n_ops,
                       gpt_task_info* tasks, int64_t max_tasks, int32_t* op_types, int32_t* op_tasks,
                       int32_t* op_dims, int32_t max_ops) {
  if (!cfg || !n_tasks || !n_ops) return fail(nullptr, GPT_ERR_INVALID_ARG, "NULL argument");
  std::string why;
  int rc = validate(*cfg, &why);
  if (rc != GPT_OK) return fail(nullptr, rc, "invalid config: %s", why.c_str());
  gpt h;
  h.cfg = *cfg;
  h.describe_only = true;
  h.num_sms = num_sms > 0 ? num_sms : 152;
  h.D = Dims{cfg->n_layer, cfg->d_model, cfg->n_head, cfg->d_model / cfg->n_head, cfg->d_mlp, cfg->vocab,
             cfg->seq_len, cfg->batch, cfg->batch * cfg->seq_len};
  build_table(&h);
  const int ks = lm_ksplit_for(*cfg, h.num_sms);
  const Layout Lo = make_layout(*cfg, h.nparams, ks);
  h.params = h.grads = h.m = h.v = nullptr;  // addresses are never dereferenced here
  rc = build_graph(&h, Lo, ks);
  if (rc != GPT_OK) { g_create_error = h.err; return rc; }
  *n_tasks = (int64_t)h.tasks.size();
  *n_ops = (int32_t)h.ops.size();
  if (tasks)
    for (int64_t i = 0; i < std::min<int64_t>(max_tasks, (int64_t)h.tasks.size()); ++i) {
      const TaskDesc& t = h.tasks[i];
      tasks[i].op = t.op;
      tasks[i].idx = t.idx;
      tasks[i].sig = t.sig;
      tasks[i].sig2 = t.sig2;
      tasks[i].nwait = t.nwait;
      for (int w = 0; w < 3; ++w) {
        tasks[i].wait_first[w] = w < t.nwait ? t.wait[w].first : -1;
        tasks[i].wait_count[w] = w < t.nwait ? t.wait[w].count : 0;
        tasks[i].wait_need[w] = w < t.nwait ? (int32_t)t.wait[w].need : 0;
      }
    }
  for (int32_t i = 0; i < std::min<int32_t>(max_ops, (int32_t)h.ops.size()); ++i) {
    if (op_types) op_types[i] = h.ops[i].type;
    if (op_tasks) op_tasks[i] = h.ops[i].ntasks;
    if (op_dims) {
      const bool g = h.ops[i].type == OP_GEMM;
      const GemmArgs& a = h.ops[i].gemm;
      const int32_t v[6] = {g ? a.M : 0, g ? a.N : 0, g ? a.K : 0, g ? a.BN : 0, h.op_ctr0[i], h.op_nblk[i]};
      for (int k = 0; k < 6; ++k) op_dims[6 * i + k] = v[k];
    }
  }
  return GPT_OK;
}

int64_t gpt_task_budget(int64_t iterations, int64_t tasks_per_iteration) {
  if (iterations < 0 || tasks_per_iteration < 0) return -1;
  if (tasks_per_iteration != 0 && iterations > INT64_MAX / tasks_per_iteration) return -1;
  return iterations * tasks_per_iteration;
}

}  // extern "C"

// ============================================================================
// Training step without any allocation.
//
// For callers that cannot allocate device memory themselves or through us:
// runtimes whose memory is owned by a pool allocator that forbids side
// allocations, and embedded or real-time hosts that must not allocate after
// start-up (an allocation can block for an unbounded time).  The step's scratch (gradients,
// activations, the task graph, counters and error words) lives in one
// file-scope device array; the caller passes parameters, AdamW moments, tokens
// and targets.  Only the fp32 arithmetic is offered (the bf16 path would have to
// rebuild its bf16 weight copy inside the array on every call), and only models
// whose scratch fits in kStaticScratchBytes.
// ============================================================================
namespace {

constexpr size_t kStaticScratchBytes = (size_t)16 << 20;  // 16 MiB on every GPU that loads libgpt.so
constexpr int kStaticMaxDevices = 64;

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
uint8_t* g_static_ptr[kStaticMaxDevices] = {};

// Device address of g_static_scratch on the current device (looked up once per
// device; the host-side name of the array is not a device address).
int static_scratch_address(int device, uint8_t** out) {
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[device]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p)
      return fail(nullptr, GPT_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed: %s",
                  cudaGetErrorString(e));
    g_static_ptr[device] = static_cast<uint8_t*>(p);
  }
  *out = g_static_ptr[device];
  return GPT_OK;
}

}  // namespace

extern "C" int gpt_train_step_static(const gpt_config* cfg, float* params, float* m, float* v, int64_t step,
                                     const int32_t* tokens, const int32_t* targets, float* loss,
                                     void* cuda_stream) {
  g_create_error.clear();
  if (!cfg || !params || !m || !v || !tokens || !targets || step < 0)
    return fail(nullptr, GPT_ERR_INVALID_ARG, "cfg, params, m, v, tokens, targets must be non-NULL; step >= 0");
  std::string why;
  int rc = validate(*cfg, &why);
  if (rc != GPT_OK) return fail(nullptr, rc, "invalid config: %s", why.c_str());
  if (cfg->dtype != GPT_DTYPE_FP32)
    return fail(nullptr, GPT_ERR_UNSUPPORTED, "gpt_train_step_static supports GPT_DTYPE_FP32 only");
  gpt h;
  h.cfg = *cfg;
  if (!h.cfg.wait_timeout_ms) h.cfg.wait_timeout_ms = 2000;
  h.D = Dims{cfg->n_layer, cfg->d_model, cfg->n_head, cfg->d_model / cfg->n_head, cfg->d_mlp, cfg->vocab,
             cfg->seq_len, cfg->batch, cfg->batch * cfg->seq_len};
  h.stream = (cudaStream_t)cuda_stream;
  if (cudaGetDevice(&h.device) != cudaSuccess) return fail(nullptr, GPT_ERR_CUDA, "no CUDA device");
  if (h.device < 0 || h.device >= kStaticMaxDevices)
    return fail(nullptr, GPT_ERR_UNSUPPORTED, "device ordinal %d >= %d", h.device, kStaticMaxDevices);
  cudaDeviceGetAttribute(&h.num_sms, cudaDevAttrMultiProcessorCount, h.device);
  build_table(&h);
  const int lm_ks = lm_ksplit_for(h.cfg, h.num_sms);
  const Layout Lo = make_layout(h.cfg, h.nparams, lm_ks, /*own_state=*/false);
  uint8_t* scratch = nullptr;
  rc = static_scratch_address(h.device, &scratch);
  if (rc != GPT_OK) return rc;
  // scratch: the arena layout without parameter and moment regions (the
  // caller's buffers take their place), then the graph and the sync words
  h.arena = scratch;
  h.params = params;
  h.m = m;
  h.v = v;
  h.grads = reinterpret_cast<float*>(scratch + Lo.grads);
  h.loss_dev = reinterpret_cast<float*>(scratch + Lo.loss);
  rc = build_graph(&h, Lo, lm_ks);
  if (rc != GPT_OK) { g_create_error = h.err; return rc; }
  Bump mb;
  mb.off = Lo.total;
  const size_t o_tasks = mb.take(h.tasks.size() * sizeof(TaskDesc));
  const size_t o_ops = mb.take(h.ops.size() * sizeof(OpDesc));
  const size_t o_ctr = mb.take((size_t)h.n_counters * sizeof(unsigned long long));
  const size_t o_tic = mb.take(2 * sizeof(unsigned long long));
  const size_t o_err = mb.take(4 * sizeof(uint32_t));
  // the whole footprint is checked before anything is written to the array
  if (mb.off > kStaticScratchBytes)
    return fail(nullptr, GPT_ERR_INVALID_ARG,
                "gpt_train_step_static: this model needs %zu bytes of scratch, above the %zu-byte static maximum",
                mb.off, kStaticScratchBytes);
  if (init_bias_pads(&h, Lo) != GPT_OK) {
    g_create_error = h.err;
    return GPT_ERR_CUDA;
  }
  h.d_tasks = reinterpret_cast<TaskDesc*>(scratch + o_tasks);
  h.d_ops = reinterpret_cast<OpDesc*>(scratch + o_ops);
  h.d_counters = reinterpret_cast<unsigned long long*>(scratch + o_ctr);
  h.d_ticket = reinterpret_cast<unsigned long long*>(scratch + o_tic);
  h.d_err = reinterpret_cast<uint32_t*>(scratch + o_err);
  gpt::Status status{};
  h.h_status = &status;  // pageable host memory: no pinned allocation
  h.opt_step = step;
  h.launches = 0;
  h.kernel = step_kernel_fp32();
  h.smem_bytes = smem_needed(&h);
  int per_sm = 0;
  cudaError_t e = cudaFuncSetAttribute(h.kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)h.smem_bytes);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, h.kernel, kThreads, h.smem_bytes);
  if (e == cudaSuccess && per_sm < 1) e = cudaErrorInvalidConfiguration;
  if (e == cudaSuccess) {
    h.grid = h.num_sms;
    // the array keeps the previous call's contents: the graph is rewritten and
    // every counter, the ticket and the error words restart from zero
    e = cudaMemcpyAsync(h.d_tasks, h.tasks.data(), h.tasks.size() * sizeof(TaskDesc), cudaMemcpyHostToDevice,
                        h.stream);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h.d_ops, h.ops.data(), h.ops.size() * sizeof(OpDesc), cudaMemcpyHostToDevice, h.stream);
    if (e == cudaSuccess)
      e = cudaMemsetAsync(scratch + o_ctr, 0, mb.off - o_ctr, h.stream);
  }
  if (e != cudaSuccess) {
    h.h_status = nullptr;
    return fail(nullptr, GPT_ERR_CUDA, "gpt_train_step_static set-up failed: %s", cudaGetErrorString(e));
  }
  rc = launch_step(&h, tokens, targets, loss);
  if (rc != GPT_OK) g_create_error = h.err;
  h.h_status = nullptr;
  return rc;
}
