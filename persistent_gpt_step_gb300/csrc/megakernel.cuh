// megakernel.cuh — the persistent training-step kernel.
//
// Every resident block loops: claim the next ticket (64-bit atomic), read that
// task's descriptor, wait (acquire, bounded) until its producers' completion
// counters reach epoch * need, run the task body with all its threads, then
// publish its writes (fence + release add on its op's counter).  The host
// launches this kernel once per training step; nothing else runs in between
// ("How one persistent kernel runs three jobs": ticket counters, fenced
// publication, acquire waits; "Open Flapping Airplanes" record, "What ran":
// resident blocks repeatedly take tasks from the scheduler).
#pragma once
#include "device.cuh"
#include "tasks_rows.cuh"
#include "tasks_simt.cuh"
#include "tc_gemm.cuh"
#include "attn_tc.cuh"

namespace pgs {

struct KernelShared {
  uint64_t bars[2 * kTcStages + 1];
  uint32_t tmem_base;
  int32_t ok;
  int64_t task;
};

template <typename act_t, bool kTC>
__global__ void __launch_bounds__(kThreads, 1) gpt_step_kernel(const __grid_constant__ KParams kp,
                                                               int32_t gelu_tanh) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ KernelShared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5;
  TcState st = {0u, 0u, 0u, 0u, 0u};
  if constexpr (kTC) {
    if (threadIdx.x == 0) {
      for (int i = 0; i < kTcStages; ++i) {
        mbar_init(smem_u32(&sh.bars[i]), 1);               // full: producer arrive + tx bytes
        mbar_init(smem_u32(&sh.bars[kTcStages + i]), 1);   // empty: one MMA commit
      }
      mbar_init(smem_u32(&sh.bars[2 * kTcStages]), 1);     // accumulator ready
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) tmem_alloc(smem_u32(&sh.tmem_base), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  for (;;) {
    if (threadIdx.x == 0) {
      int64_t t = kp.ntasks;
      int ok = 0;
      if (ld_volatile_u32(&kp.err[0]) == 0u) {
        t = (int64_t)(atomicAdd(kp.ticket, 1ull) - kp.ticket_base);
        if (t < kp.ntasks) {
          ok = 1;
          const uint64_t t_claim = kp.trace ? globaltimer_ns() : 0;
          const TaskDesc& d = kp.tasks[t];
          for (int w = 0; w < d.nwait && ok; ++w)
            ok = wait_counter(kp, d.wait_ctr[w], kp.epoch * (unsigned long long)d.wait_need[w],
                              (uint32_t)t);
          if (kp.trace) {
            uint32_t smid;
            asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
            kp.trace[4 * t + 0] = t_claim;
            kp.trace[4 * t + 1] = globaltimer_ns();
            kp.trace[4 * t + 3] = smid;
          }
        }
      }
      sh.task = t;
      sh.ok = ok;
    }
    __syncthreads();
    const int64_t t = sh.task;
    if (!sh.ok || t >= kp.ntasks) break;
    const TaskDesc& d = kp.tasks[t];
    const OpDesc& op = kp.ops[d.op];
    const int idx = d.idx;
    switch (op.type) {
      case OP_EMBED: task_embed<act_t>(kp, op.emb, idx); break;
      case OP_LN_FWD: task_ln_fwd<act_t>(op.lnf, idx); break;
      case OP_GEMM:
        if constexpr (kTC) {
          if (threadIdx.x == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncthreads();
          task_gemm_tc(kp, op.gemm, idx, smem, sh.bars, sh.tmem_base, st, gelu_tanh != 0);
        } else {
          task_gemm_simt<act_t>(op.gemm, idx, reinterpret_cast<float*>(smem), gelu_tanh != 0);
        }
        break;
      case OP_ATTN_FWD:
        if constexpr (kTC) task_attn_fwd_tc(op.attn, idx, smem);
        else task_attn_fwd_simt<act_t>(op.attn, idx, reinterpret_cast<float*>(smem));
        break;
      case OP_ATTN_BWD_PRE:
        if constexpr (kTC) task_attn_bwd_pre(op.attn, idx);
        break;
      case OP_ATTN_BWD_KV:
        if constexpr (kTC) task_attn_bwd_kv_tc(op.attn, idx, smem);
        break;
      case OP_ATTN_BWD_Q:
        if constexpr (kTC) task_attn_bwd_q_tc(op.attn, idx, smem);
        break;
      case OP_CE:
        if constexpr (kTC) {
          if ((op.ce.V & 7) == 0) task_ce_bf16_vec(kp, op.ce, idx);
          else task_ce<act_t>(kp, op.ce, idx);
        } else {
          task_ce<act_t>(kp, op.ce, idx);
        }
        break;
      case OP_LOSS: task_loss(kp, op.loss, reinterpret_cast<float*>(smem)); break;
      case OP_LN_BWD: task_ln_bwd<act_t>(op.lnb, idx, reinterpret_cast<float*>(smem)); break;
      case OP_COLSUM: task_colsum<act_t>(op.colsum, idx, reinterpret_cast<float*>(smem)); break;
      case OP_ATTN_BWD: task_attn_bwd_simt<act_t>(op.attn, idx, reinterpret_cast<float*>(smem)); break;
      case OP_EMBED_BWD_WTE: task_embed_bwd_wte(kp, op.emb, idx, reinterpret_cast<int*>(smem)); break;
      case OP_EMBED_BWD_WPE: task_embed_bwd_wpe(op.emb, idx); break;
      case OP_ADAMW: task_adamw(kp, op.adam, idx); break;
      default: break;
    }
    __syncthreads();
    if (threadIdx.x == 0 && t != kp.skip_release) {
      __threadfence();
      fence_proxy_async_global();
      red_release_add_u64(kp.counters + d.op, 1ull);
    }
    if (threadIdx.x == 0 && kp.trace) kp.trace[4 * t + 2] = globaltimer_ns();
  }

  if constexpr (kTC) {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(sh.tmem_base, kTmemCols);
  }
}

}  // namespace pgs
