// device.cuh — device primitives of the persistent kernel: memory-ordering
// operations on the completion counters, bounded waits, error reporting and
// element conversions.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "graph.h"

namespace pgs {

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t* p) {
  return *(volatile const uint32_t*)p;
}

// Orders this thread's generic-proxy global accesses with later async-proxy
// (TMA) accesses: used by producers after their stores and by consumers after
// their acquire, before tensor-core operand loads of data other blocks wrote.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Block-wide barrier in its non-aligned PTX form, for the end of a GEMM run,
// where lane 0 of warps 0-2 leaves a long single-thread role loop while the
// other lanes have long arrived: the non-aligned form counts every thread on
// its own and does not rely on the warp having reconverged.  Everywhere else
// the aligned __syncthreads() is used (it keeps more registers free).
__device__ __forceinline__ void cta_sync() { asm volatile("barrier.sync 0;" ::: "memory"); }

// Step of a multi-step launch that this block is running (0 for a one-step
// launch).  Thread 0 writes it at the start of each step, before a block
// barrier; every task body reads the step's epoch, inputs, rates and ring
// slots through the helpers below.
static __shared__ int32_t g_step;

__device__ __forceinline__ unsigned long long step_epoch(const KParams& kp) {
  return kp.epoch + (unsigned long long)g_step;
}
__device__ __forceinline__ const int32_t* step_tokens(const KParams& kp) {
  return kp.tokens + (int64_t)g_step * kp.tok_stride;
}
__device__ __forceinline__ const int32_t* step_targets(const KParams& kp) {
  return kp.targets + (int64_t)g_step * kp.tok_stride;
}
__device__ __forceinline__ float step_lr(const KParams& kp) { return kp.step_hyper ? kp.step_hyper[3 * g_step] : kp.lr; }
__device__ __forceinline__ float step_bc1(const KParams& kp) {
  return kp.step_hyper ? kp.step_hyper[3 * g_step + 1] : kp.bc1;
}
__device__ __forceinline__ float step_bc2(const KParams& kp) {
  return kp.step_hyper ? kp.step_hyper[3 * g_step + 2] : kp.bc2;
}

__device__ __forceinline__ void set_fatal(const KParams& kp, uint32_t code, uint32_t task,
                                          uint32_t ctr) {
  if (atomicCAS(&kp.err[0], 0u, code) == 0u) {
    kp.err[2] = task;
    kp.err[3] = ctr;
  }
}

__device__ __forceinline__ void set_soft(const KParams& kp, uint32_t bits) {
  atomicOr(&kp.err[1], bits);
}

// Spins (one thread) until counters[ctr] >= target.  Gives up after the
// handle's timeout (globaltimer) or an iteration cap, whichever comes first,
// recording a fatal error; also gives up when another block recorded one.
__device__ __forceinline__ bool wait_counter(const KParams& kp, int32_t ctr,
                                             unsigned long long target, uint32_t task) {
  const unsigned long long* p = kp.counters + ctr;
  if (ld_acquire_u64(p) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  // ~30 ns minimum per iteration (acquire load + sleep) bounds the count too.
  const uint64_t max_iters = kp.timeout_ns / 30 + 1024;
  uint32_t sleep = 32;
  for (uint64_t it = 0; it < max_iters; ++it) {
    __nanosleep(sleep);
    if (sleep < 256) sleep <<= 1;
    if (ld_acquire_u64(p) >= target) return true;
    if ((it & 15) == 15) {
      if (ld_volatile_u32(&kp.err[0]) != 0u) return false;
      if (globaltimer_ns() - t0 > kp.timeout_ns) break;
    }
  }
  set_fatal(kp, kFatalTimeout, task, (uint32_t)ctr);
  return false;
}

// Waits (one thread) for every dependency range of task t.
__device__ __forceinline__ bool task_ready(const KParams& kp, int64_t t) {
  const TaskDesc& d = kp.tasks[t];
  for (int w = 0; w < d.nwait; ++w) {
    const WaitSpec ws = d.wait[w];
    const unsigned long long target = step_epoch(kp) * (unsigned long long)ws.need;
    for (int c = 0; c < ws.count; ++c)
      if (!wait_counter(kp, ws.first + c, target, (uint32_t)t)) return false;
  }
  return true;
}

// Claims the next ticket (one thread): the index of a task in kp.tasks, or
// kp.ntasks when the graph is exhausted or a fatal error was recorded.  Tickets
// are a 64-bit counter per launch parity; the previous launch zeroed this one.
__device__ __forceinline__ int64_t claim_task(const KParams& kp) {
  if (ld_volatile_u32(&kp.err[0]) != 0u) return kp.ntasks;
  const int64_t t = (int64_t)atomicAdd(kp.tickets + (step_epoch(kp) & 1ull), 1ull);
  return t < kp.ntasks ? t : kp.ntasks;
}

// ---- element conversions (act_t = float or __nv_bfloat16) -------------------
template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One AdamW step of one parameter (decoupled weight decay first):
// p *= decay; m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2;
// p -= lr (m / bc1) / (sqrt(v / bc2) + eps).  Shared by the AdamW task and the
// fused weight-gradient epilogue so both produce the same bits.
struct AdamHyper {
  float lr, b1, b2, ib1, ib2, rbc1, rbc2, eps;
};
__device__ __forceinline__ AdamHyper adam_hyper(const KParams& kp) {
  return AdamHyper{step_lr(kp), kp.beta1, kp.beta2, 1.0f - kp.beta1, 1.0f - kp.beta2, 1.0f / step_bc1(kp),
                   1.0f / step_bc2(kp), kp.eps};
}
__device__ __forceinline__ void adamw_elem(const AdamHyper& hp, float decay, float g, float& p, float& m,
                                           float& v) {
  p *= decay;
  m = hp.b1 * m + hp.ib1 * g;
  v = hp.b2 * v + hp.ib2 * g * g;
  const float mh = m * hp.rbc1, vh = v * hp.rbc2;
  p -= hp.lr * mh / (sqrtf(vh) + hp.eps);
}

// GELU, tanh form 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) or erf form.
__device__ __forceinline__ float gelu_f(float x, bool tanh_form) {
  if (tanh_form) {
    const float k0 = 0.7978845608028654f;
    return 0.5f * x * (1.0f + tanhf(k0 * (x + 0.044715f * x * x * x)));
  }
  return 0.5f * x * (1.0f + erff(x * 0.7071067811865476f));
}
__device__ __forceinline__ float gelu_grad_f(float x, bool tanh_form) {
  if (tanh_form) {
    const float k0 = 0.7978845608028654f;
    float t = tanhf(k0 * (x + 0.044715f * x * x * x));
    return 0.5f * (1.0f + t) + 0.5f * x * (1.0f - t * t) * k0 * (1.0f + 3.0f * 0.044715f * x * x);
  }
  return 0.5f * (1.0f + erff(x * 0.7071067811865476f)) +
         x * expf(-0.5f * x * x) * 0.3989422804014327f;
}

}  // namespace pgs
