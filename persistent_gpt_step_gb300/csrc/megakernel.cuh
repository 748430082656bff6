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
#include "serve.cuh"

namespace pgs {

struct KernelShared {
  GemmShared gemm;
  AttnShared att;
  uint64_t adam_bars[kAdamStages];
  uint32_t adam_iter;
  uint32_t tmem_base;
  int32_t ok;
  int32_t step_ok;   // the grid barrier after a step of a multi-step launch passed
  int64_t task;
};

// kExt: the rotary-embedding / gated-MLP model variant (its extra epilogues
// and the rotation in the attention backward are compiled into this instance only).
template <typename act_t, bool kTC, bool kExt = false>
__global__ void __launch_bounds__(kThreads, 1) gpt_step_kernel(const __grid_constant__ KParams kp,
                                                               int32_t gelu_tanh) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ KernelShared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5;
  TcState st = {0u, 0u, 0u, 0u, 0u, 0u};
  if (threadIdx.x == 0) {
    for (int i = 0; i < kAdamStages; ++i) mbar_init(smem_u32(&sh.adam_bars[i]), 1);
    sh.adam_iter = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if constexpr (kTC) {
    if (threadIdx.x == 0) {
      for (int i = 0; i < kTcStages; ++i) {
        mbar_init(smem_u32(&sh.gemm.stage_full[i]), 1);   // producer arrive + tx bytes
        mbar_init(smem_u32(&sh.gemm.stage_empty[i]), 1);  // one MMA commit
      }
      for (int i = 0; i < kQSlots; ++i) {
        mbar_init(smem_u32(&sh.gemm.q_full[i]), 1);     // scheduler publishes a queue entry
        mbar_init(smem_u32(&sh.gemm.q_empty[i]), 3);    // producer, MMA and releaser are done with it
        mbar_init(smem_u32(&sh.gemm.tile_done[i]), 4);  // each epilogue warp finished the slot's tile
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(smem_u32(&sh.gemm.acc_full[i]), 1);   // MMA commit: accumulator complete
        mbar_init(smem_u32(&sh.gemm.acc_empty[i]), 4);  // each epilogue warp drained it
      }
      sh.gemm.prod_claim = 0;
      for (int i = 0; i < AB_NUM; ++i) {
        mbar_init(smem_u32(&sh.att.bar[i]), 1);  // one arrival: a TMA expect-tx or a tcgen05 commit
        sh.att.use[i] = 0;
      }
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncwarp();  // tcgen05.alloc is warp-aligned
    if (warp == 0) tmem_alloc(smem_u32(&sh.tmem_base), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  const bool serving = kp.serve != nullptr && (int)blockIdx.x >= kp.train_blocks;
  if (serving) serve_loop(kp, smem, &sh.task, &sh.ok);  // a serving role for the whole launch
  const unsigned long long nbar = kp.serve ? (unsigned long long)kp.train_blocks : (unsigned long long)gridDim.x;
  const int nsteps = serving || kp.ntasks == 0 ? 0 : (kp.nsteps > 1 ? kp.nsteps : 1);
  for (int step = 0; step < nsteps; ++step) {
  if (threadIdx.x == 0) {
    g_step = step;
    // the ticket of the next step (or launch): its last user, the previous step, has
    // ended on every block (grid barrier below, or the end of the previous launch)
    if (blockIdx.x == 0) kp.tickets[(kp.epoch + (unsigned long long)step + 1ull) & 1ull] = 0ull;
  }
  __syncthreads();
  int64_t pending = -1;  // ticket claimed by a GEMM run, dependencies not yet waited
  for (;;) {
    if (threadIdx.x == 0) {
      int64_t t = kp.ntasks;
      int ok = 0;
      if (ld_volatile_u32(&kp.err[0]) == 0u) {
        t = pending >= 0 ? pending : claim_task(kp);
        if (t < kp.ntasks) {
          ok = 1;
          const uint64_t t_claim = kp.trace ? globaltimer_ns() : 0;
          ok = task_ready(kp, t);
          // this thread issues the bulk / tensor copies of row and attention tasks:
          // order the producers' writes it has acquired before those async-proxy reads
          fence_proxy_async_global();
          if (kp.trace) {
            uint32_t smid;
            asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
            kp.trace[4 * t + 0] = t_claim;
            kp.trace[4 * t + 1] = globaltimer_ns();
            kp.trace[4 * t + 3] = smid | ((unsigned long long)blockIdx.x << 32);
          }
        }
      }
      sh.task = t;
      sh.ok = ok;
    }
    __syncthreads();
    const int64_t t = *reinterpret_cast<volatile int64_t*>(&sh.task);  // read once (thread 0 rewrites it next round)
    if (!*reinterpret_cast<volatile int32_t*>(&sh.ok) || t >= kp.ntasks) break;
    pending = -1;
    const TaskDesc& d = kp.tasks[t];
    const OpDesc& op = kp.ops[d.op];
    const int idx = d.idx;
    if constexpr (kTC) {
      if (op.type == OP_GEMM) {
        pending = gemm_run<kExt>(kp, t, sh.gemm, smem, sh.tmem_base, st, gelu_tanh != 0);
        continue;  // the run released its tasks
      }
    }
    switch (op.type) {
      case OP_EMBED: { const EmbedArgs a = op.emb; task_embed<act_t>(kp, a, idx); } break;
      case OP_LN_FWD: { const LnFwdArgs a = op.lnf; task_ln_fwd<act_t>(a, idx); } break;
      case OP_GEMM:
        if constexpr (!kTC) {
          const GemmArgs a = op.gemm;
          task_gemm_simt<act_t>(a, idx, reinterpret_cast<float*>(smem), gelu_tanh != 0);
        }
        break;
      case OP_ATTN_FWD:
        {
          const AttnArgs a = op.attn;
          if constexpr (kTC) task_attn_fwd_tc(kp, a, idx, smem, sh.att, sh.tmem_base);
          else task_attn_fwd_simt<act_t>(a, idx, reinterpret_cast<float*>(smem));
        }
        break;
      case OP_ATTN_BWD_PRE:
        if constexpr (kTC) { const AttnArgs a = op.attn; task_attn_bwd_pre(a, idx); }
        break;
      case OP_ATTN_BWD_KV:
        if constexpr (kTC) { const AttnArgs a = op.attn; task_attn_bwd_kv_tc<kExt>(kp, a, idx, smem, sh.att, sh.tmem_base); }
        break;
      case OP_ATTN_BWD_Q:
        if constexpr (kTC) { const AttnArgs a = op.attn; task_attn_bwd_q_tc<kExt>(kp, a, idx, smem, sh.att, sh.tmem_base); }
        break;
      case OP_CE:
        {
          const CeArgs a = op.ce;
          if constexpr (kTC) {
            if (a.staged) task_ce_bf16_staged(kp, a, idx, smem, sh.adam_bars, &sh.adam_iter);
            else if ((a.V & 7) == 0) task_ce_bf16_vec(kp, a, idx);
            else task_ce<act_t>(kp, a, idx);
          } else {
            task_ce<act_t>(kp, a, idx);
          }
        }
        break;
      case OP_LOSS: { const LossArgs a = op.loss; task_loss(kp, a, reinterpret_cast<float*>(smem)); } break;
      case OP_LN_BWD: {
        const LnBwdArgs a = op.lnb;
        if (kTC && a.staged) task_ln_bwd_staged_any<act_t>(kp, a, idx, smem, sh.adam_bars, &sh.adam_iter);
        else task_ln_bwd<act_t>(a, idx, reinterpret_cast<float*>(smem));
      } break;
      case OP_COLSUM: { const ColsumArgs a = op.colsum; task_colsum<act_t>(a, idx, reinterpret_cast<float*>(smem)); } break;
      case OP_ATTN_BWD: { const AttnArgs a = op.attn; task_attn_bwd_simt<act_t>(a, idx, reinterpret_cast<float*>(smem)); } break;
      case OP_EMBED_BWD_WTE: { const EmbedArgs a = op.emb; task_embed_bwd_wte(kp, a, idx, reinterpret_cast<int*>(smem)); } break;
      case OP_EMBED_BWD_WPE: { const EmbedArgs a = op.emb; task_embed_bwd_wpe(a, idx); } break;
      case OP_TOKEN_SORT: { const EmbedArgs a = op.emb; task_token_sort(kp, a, reinterpret_cast<int*>(smem)); } break;
      case OP_ADAMW: {
        const AdamArgs a = op.adam;
        task_adamw(kp, a, idx, smem, sh.adam_bars, &sh.adam_iter);
      } break;
      default: break;
    }
    __syncthreads();
    if (threadIdx.x == 0 && t != kp.skip_release) {
      __threadfence();
      fence_proxy_async_global();
      red_release_add_u64(kp.counters + d.sig, 1ull);
      if (d.sig2 >= 0) red_release_add_u64(kp.counters + d.sig2, 1ull);
    }
    if (threadIdx.x == 0 && kp.trace) kp.trace[4 * t + 2] = globaltimer_ns();
  }
  // End of this block's share of the step: its AdamW bulk stores complete and are
  // published, and the block arrives at the grid barrier (after step s of the
  // launch it holds bar_base + (s + 1) x the training blocks).  Between two steps
  // of the launch every training block waits there, so the next step reads the
  // updated weights.
  if (threadIdx.x == 0) {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    if (kp.grid_bar) {
      fence_proxy_async_global();
      __threadfence();
      red_release_add_u64(kp.grid_bar, 1ull);
    }
  }
  if (step + 1 < nsteps) {
    if (threadIdx.x == 0) {
      const unsigned long long target = kp.bar_base + (unsigned long long)(step + 1) * nbar;
      int ok = 1;
      if (ld_volatile_u32(&kp.err[0]) == 0u) {
        const uint64_t t0 = globaltimer_ns();
        const uint64_t max_iters = kp.timeout_ns / 30 + 1024;
        ok = 0;
        for (uint64_t it = 0; it < max_iters; ++it) {
          if (ld_acquire_u64(kp.grid_bar) >= target) { ok = 1; break; }
          __nanosleep(128);
          if ((it & 15) == 15) {
            if (ld_volatile_u32(&kp.err[0]) != 0u) break;
            if (globaltimer_ns() - t0 > kp.timeout_ns) { set_fatal(kp, kFatalTimeout, 0xFFFFFFFFu, 0xFFFFFFFFu); break; }
          }
        }
        fence_proxy_async_global();  // later tensor copies read the other blocks' updates
      }
      sh.step_ok = ok && ld_volatile_u32(&kp.err[0]) == 0u;
    }
    __syncthreads();
    if (!*reinterpret_cast<volatile int32_t*>(&sh.step_ok)) break;  // every thread reads the same word
  }
  }  // steps

  if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  if constexpr (kTC) {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    __syncwarp();
    if (warp == 0) tmem_dealloc(sh.tmem_base, kTmemCols);
  }
}

}  // namespace pgs
