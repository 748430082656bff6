// serve.cuh — the serving partition of the persistent kernel: greedy
// autoregressive generation (batch 1) from the live weights on a reserved set of
// blocks, running in the same launch as the training step ("Open Flapping
// Airplanes" record, section "What ran": SM roles, serving does "autoregressive
// text generation from the changing model"; "How one persistent kernel runs
// three jobs": blocks take static roles, serving claims tasks through its own
// ticket counter, "one token releases the next").
//
// A step of the decode processes the token at position s (the prompt, then the
// generated ones) with the layers' keys and values of positions < s in an fp32
// cache, and writes the argmax of the next-token logits at position s + 1 (once
// the prompt is consumed).  Every counter and ticket is 64-bit: the task budget
// of a long session (steps x tasks per step) does not wrap ("A longer run
// exposed a scheduler overflow").
#pragma once
#include "device.cuh"
#include "tc_gemm.cuh"

namespace pgs {

__device__ __forceinline__ float block_sum(float v, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) s += red[w];  // fixed order: every thread gets the same sum
  return s;
}

// x = wte[token] + wpe[position]
__device__ inline void serve_embed(const ServeParams& sp, const ServeOp& op, int64_t s) {
  int tok = sp.seq[s];
  tok = tok < 0 ? 0 : (tok >= sp.V ? sp.V - 1 : tok);
  for (int c = threadIdx.x; c < sp.C; c += kThreads)
    op.out[c] = sp.wte[(int64_t)tok * sp.C + c] + sp.wpe[s * sp.C + c];
}

// out = LN(in) (biased variance, eps), one row of C
__device__ inline void serve_ln(const ServeParams& sp, const ServeOp& op, float* red) {
  float acc = 0.f;
  for (int c = threadIdx.x; c < sp.C; c += kThreads) acc += op.in[c];
  const float mean = block_sum(acc, red) / (float)sp.C;
  acc = 0.f;
  for (int c = threadIdx.x; c < sp.C; c += kThreads) {
    const float d = op.in[c] - mean;
    acc += d * d;
  }
  const float rstd = rsqrtf(block_sum(acc, red) / (float)sp.C + sp.ln_eps);
  for (int c = threadIdx.x; c < sp.C; c += kThreads) {
    float y = (op.in[c] - mean) * rstd * op.g[c];
    if (op.b) y += op.b[c];
    op.out[c] = y;
  }
}

// Rows [64 idx, 64 idx + 64) of y = W in + b with the op's epilogue.  The input
// vector is staged in shared memory; each warp reduces 8 rows, its lanes
// reading 16-byte chunks (8 bf16) of a row, so a warp reads whole 512-byte spans.
// The loads of all 8 rows over a 768-wide slice of K are issued before any is
// reduced: one memory latency per slice instead of one per row.
__device__ inline void serve_gemv(const ServeParams& sp, const ServeOp& op, int idx, int64_t s, float* sx,
                                  float* red) {
  constexpr int kR = kServeRows / kWarps;  // rows of a warp
  constexpr int kU = 3;                    // 16-byte chunks of a row per lane per slice (3 x 32 x 8 = 768)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int k = threadIdx.x; k < op.K; k += kThreads) sx[k] = op.in[k];
  __syncthreads();
  const int r0 = idx * kServeRows + warp * kR;
  const int nch = op.K / 8;  // 16-byte chunks of a row
  float acc[kR];
#pragma unroll
  for (int i = 0; i < kR; ++i) acc[i] = 0.f;
  for (int c0 = 0; c0 < nch; c0 += kU * 32) {
    uint4 u[kR][kU];
#pragma unroll
    for (int i = 0; i < kR; ++i)
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int c = c0 + j * 32 + lane;
        u[i][j] = (r0 + i < op.N && c < nch)
                      ? reinterpret_cast<const uint4*>(op.W + (int64_t)(r0 + i) * op.K)[c]
                      : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const int c = c0 + j * 32 + lane;
      if (c >= nch) break;
      const float4 x0 = *reinterpret_cast<const float4*>(sx + 8 * c);
      const float4 x1 = *reinterpret_cast<const float4*>(sx + 8 * c + 4);
#pragma unroll
      for (int i = 0; i < kR; ++i) {
        const __nv_bfloat162* hh = reinterpret_cast<const __nv_bfloat162*>(&u[i][j]);
        const float2 a0 = __bfloat1622float2(hh[0]), a1 = __bfloat1622float2(hh[1]);
        const float2 a2 = __bfloat1622float2(hh[2]), a3 = __bfloat1622float2(hh[3]);
        acc[i] += a0.x * x0.x + a0.y * x0.y + a1.x * x0.z + a1.y * x0.w + a2.x * x1.x + a2.y * x1.y + a3.x * x1.z +
                  a3.y * x1.w;
      }
    }
  }
  float best = -INFINITY;
  int best_i = 0x7fffffff;
#pragma unroll
  for (int i = 0; i < kR; ++i) {
    const int r = r0 + i;
    const float sum = warp_sum(acc[i]);
    if (r < op.N && lane == 0) {
      const float y = sum + (op.bias ? op.bias[r] : 0.f);
      switch (op.epi) {
        case SE_QKV:  // q | k | v: k and v are this position's cache rows
          if (r < sp.C) op.out[r] = y;
          else if (r < 2 * sp.C) op.kc[s * sp.C + (r - sp.C)] = y;
          else op.vc[s * sp.C + (r - 2 * sp.C)] = y;
          break;
        case SE_RESID: op.out[r] += y; break;
        case SE_GELU: op.out[r] = gelu_f(y, sp.gelu_tanh != 0); break;
        case SE_LOGITS:
          if (y > best || (y == best && r < best_i)) { best = y; best_i = r; }
          break;
        default: op.out[r] = y; break;
      }
    }
  }
  if (op.epi == SE_LOGITS) {  // the slice's best logit (smallest id among equal logits)
    __syncthreads();
    float* rv = red;
    int* ri = reinterpret_cast<int*>(red + kWarps);
    if (lane == 0) { rv[warp] = best; ri[warp] = best_i; }
    __syncthreads();
    if (threadIdx.x == 0) {
      float bv = rv[0];
      int bi = ri[0];
      for (int w = 1; w < kWarps; ++w)
        if (rv[w] > bv || (rv[w] == bv && ri[w] < bi)) { bv = rv[w]; bi = ri[w]; }
      sp.part_max[idx] = bv;
      sp.part_idx[idx] = bi;
    }
  }
}

// One head of causal attention for the query at position s over the cached
// keys and values of positions 0..s: softmax(q k_j / sqrt(d)) v (d = 64).
// Scores: one thread per key, its key row loaded whole (16 x 16 bytes in
// flight).  Output: warp w accumulates p_j v_j over the keys j = w mod 8, a lane
// holding two of the 64 columns, the loads of four keys in flight; the warps'
// partial rows are added in warp order.
__device__ inline void serve_attn(const ServeParams& sp, const ServeOp& op, int h, int64_t s, float* sm,
                                  float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int d = 64;
  const float scale = 0.125f;  // 1 / sqrt(64)
  float* sq = sm;              // [64] the query
  float* sc = sm + 64;         // [T] scores, then probabilities
  float* po = sc + sp.T;       // [kWarps][64] partial outputs
  const int n = (int)s + 1;
  if (threadIdx.x < d) sq[threadIdx.x] = op.in[h * d + threadIdx.x];
  __syncthreads();
  float m = -INFINITY;
  for (int j = threadIdx.x; j < n; j += kThreads) {
    const float4* kr = reinterpret_cast<const float4*>(op.kc + (int64_t)j * sp.C + h * d);
    float4 kv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) kv[i] = kr[i];
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      acc += kv[i].x * sq[4 * i] + kv[i].y * sq[4 * i + 1] + kv[i].z * sq[4 * i + 2] + kv[i].w * sq[4 * i + 3];
    sc[j] = acc * scale;
    m = fmaxf(m, acc * scale);
  }
  m = warp_max(m);
  if (lane == 0) red[warp] = m;
  __syncthreads();
  m = red[0];
  for (int w = 1; w < kWarps; ++w) m = fmaxf(m, red[w]);
  __syncthreads();
  float acc = 0.f;
  for (int j = threadIdx.x; j < n; j += kThreads) {
    const float p = expf(sc[j] - m);
    sc[j] = p;
    acc += p;
  }
  const float l = block_sum(acc, red);  // (its barrier also orders the probabilities before their use)
  float2 o = make_float2(0.f, 0.f);
  const float* vb = op.vc + h * d + 2 * lane;
  int j = warp;
  for (; j + 3 * kWarps < n; j += 4 * kWarps) {
    float2 v4[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v4[u] = *reinterpret_cast<const float2*>(vb + (int64_t)(j + u * kWarps) * sp.C);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float p = sc[j + u * kWarps];
      o.x += p * v4[u].x;
      o.y += p * v4[u].y;
    }
  }
  for (; j < n; j += kWarps) {
    const float2 v = *reinterpret_cast<const float2*>(vb + (int64_t)j * sp.C);
    const float p = sc[j];
    o.x += p * v.x;
    o.y += p * v.y;
  }
  po[warp * 64 + 2 * lane] = o.x;
  po[warp * 64 + 2 * lane + 1] = o.y;
  __syncthreads();
  if (threadIdx.x < d) {
    float r = 0.f;
    for (int w = 0; w < kWarps; ++w) r += po[w * 64 + threadIdx.x];
    op.out[h * d + threadIdx.x] = r / l;
  }
}

// The next token: the best of the LM-head slices (smallest id among equal logits).
__device__ inline void serve_argmax(const ServeParams& sp, int64_t s, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int i = threadIdx.x; i < sp.n_slices; i += kThreads) {
    const float v = sp.part_max[i];
    const int id = sp.part_idx[i];
    if (v > bv || (v == bv && id < bi)) { bv = v; bi = id; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
    if (v2 > bv || (v2 == bv && i2 < bi)) { bv = v2; bi = i2; }
  }
  int* ri = reinterpret_cast<int*>(red + kWarps);
  if (lane == 0) { red[warp] = bv; ri[warp] = bi; }
  __syncthreads();
  if (threadIdx.x == 0) {
    float v = red[0];
    int id = ri[0];
    for (int w = 1; w < kWarps; ++w)
      if (red[w] > v || (red[w] == v && ri[w] < id)) { v = red[w]; id = ri[w]; }
    if (s + 1 >= sp.n_prompt && s + 1 < sp.T) sp.seq[s + 1] = id;  // inside the prompt the next token is given
  }
}

// The serving loop of a block with a serving role: claim a ticket, wait for the
// producer op of the same step (a step's first op waits for the previous step's
// argmax), run the task, publish it.  Ends when a claimed ticket lies beyond this
// launch's step limit (or another block recorded a fatal error).
__device__ inline void serve_loop(const KParams& kp, uint8_t* smem, int64_t* sh_task, int32_t* sh_ok) {
  const ServeParams& sp = *kp.serve;
  float* red = reinterpret_cast<float*>(smem);         // [2 kWarps] reductions
  float* sm = reinterpret_cast<float*>(smem + 256);    // staged vectors / attention scores
  for (;;) {
    if (threadIdx.x == 0) {
      int ok = 0;
      int64_t t = -1;
      if (ld_volatile_u32(&kp.err[0]) == 0u) {
        t = (int64_t)atomicAdd(sp.ticket, 1ull);
        const int64_t s = t / sp.P - (int64_t)sp.base;
        if (s < sp.limit) {
          const int k = (int)(t % sp.P);
          const int o = sp.task_op[k];
          // producer: the previous op of this step, or the previous step's argmax
          const int src = o > 0 ? o - 1 : sp.nops - 1;
          const unsigned long long step = sp.base + (unsigned long long)s;
          const unsigned long long target =
              o > 0 ? (step + 1ull) * (unsigned long long)sp.ops[src].ntasks : step * (unsigned long long)sp.ops[src].ntasks;
          ok = 1;
          const unsigned long long* c = sp.counters + src;
          if (ld_acquire_u64(c) < target) {
            const uint64_t t0 = globaltimer_ns();
            ok = 0;
            for (uint64_t it = 0; it < kp.timeout_ns / 30 + 1024; ++it) {
              __nanosleep(64);
              if (ld_acquire_u64(c) >= target) { ok = 1; break; }
              if ((it & 15) == 15) {
                if (ld_volatile_u32(&kp.err[0]) != 0u) break;
                if (globaltimer_ns() - t0 > kp.timeout_ns) { set_fatal(kp, kFatalTimeout, (uint32_t)k, 0xFFFFFFFEu); break; }
              }
            }
          }
        }
      }
      *sh_task = t;
      *sh_ok = ok;
    }
    __syncthreads();
    const int64_t t = *reinterpret_cast<volatile int64_t*>(sh_task);
    if (!*reinterpret_cast<volatile int32_t*>(sh_ok)) break;
    const int64_t s = t / sp.P - (int64_t)sp.base;
    const int k = (int)(t % sp.P);
    const ServeOp& op = sp.ops[sp.task_op[k]];
    const int idx = sp.task_idx[k];
    switch (op.type) {
      case SV_EMBED: serve_embed(sp, op, s); break;
      case SV_LN: serve_ln(sp, op, red); break;
      case SV_GEMV: serve_gemv(sp, op, idx, s, sm, red); break;
      case SV_ATTN: serve_attn(sp, op, idx, s, sm, red); break;
      case SV_ARGMAX: serve_argmax(sp, s, red); break;
      default: break;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      red_release_add_u64(sp.counters + sp.task_op[k], 1ull);
    }
  }
}

}  // namespace pgs
