// tc_gemm.cuh — bf16 GEMM task on the 5th-generation tensor cores (sm_103a):
// TMA (cp.async.bulk.tensor, 128-byte swizzle) stages A and B tiles through a
// multi-stage shared-memory ring guarded by mbarriers; one thread issues
// tcgen05.mma (kind::f16, bf16 x bf16 -> fp32) into a TMEM accumulator; the
// block's eight warps read the accumulator back with tcgen05.ld and run the
// fused epilogue (bias, residual add, GELU, GELU', fp32 or bf16 stores).
//
// Operand majorness comes from the UMMA descriptors, not from transposes:
//   forward       C = X  W^T   A = X  [M,K] K-major,   B = W [N,K] K-major
//   input grad    C = dY W     A = dY [M,K] K-major,   B = W [K,N] MN-major
//   weight grad   C = dY^T X   A = dY [K,M] MN-major,  B = X [K,N] MN-major
#pragma once
#include "device.cuh"

namespace pgs {

struct TcState {          // pipeline state carried by the block across GEMM tasks
  uint32_t prod_stage, prod_phase;   // producer thread
  uint32_t mma_stage, mma_phase;     // MMA thread
  uint32_t acc_phase;                // every thread
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// ---- mbarrier -------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on an mbarrier phase; on expiry records a fatal error.
__device__ __forceinline__ bool mbar_wait(const KParams& kp, uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  const uint64_t max_iters = kp.timeout_ns / 20 + 1024;
  for (uint64_t it = 0; it < max_iters; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 63) {
      if (ld_volatile_u32(&kp.err[0]) != 0u) return false;
      if (globaltimer_ns() - t0 > kp.timeout_ns) break;
    }
  }
  set_fatal(kp, kFatalMbarTimeout, 0xffffffffu, bar);
  return false;
}

// ---- TMA -------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int32_t c0, int32_t c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(tmap), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// ---- tcgen05 -----------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on `bar` when every tcgen05 operation this thread issued so far completes.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// 32 lanes x 32 bits, 16 consecutive columns: thread i gets row (lane base + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15},"
      " [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (>> 4), fixed version 1 at bit 46, 128-byte swizzle (2) at bits 61-63.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
         ((uint64_t)(sbo >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, majorness, N, M.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---- epilogue on 16 consecutive columns of one row ------------------------------------
__device__ __forceinline__ void store_bf16x16(__nv_bfloat16* dst, const float* v) {
  uint4 u0, u1;
  __nv_bfloat162* h0 = reinterpret_cast<__nv_bfloat162*>(&u0);
  __nv_bfloat162* h1 = reinterpret_cast<__nv_bfloat162*>(&u1);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h0[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    h1[i] = __floats2bfloat162_rn(v[8 + 2 * i], v[8 + 2 * i + 1]);
  }
  reinterpret_cast<uint4*>(dst)[0] = u0;
  reinterpret_cast<uint4*>(dst)[1] = u1;
}

__device__ __forceinline__ void epilogue16(const GemmArgs& g, int split, int m, int n, float* v,
                                           bool gelu_tanh) {
  if (g.bias && g.epi != EPI_F32 && g.epi != EPI_GELU_BWD) {
    const float4* b4 = reinterpret_cast<const float4*>(g.bias + n);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float4 b = b4[i];
      v[4 * i] += b.x; v[4 * i + 1] += b.y; v[4 * i + 2] += b.z; v[4 * i + 3] += b.w;
    }
  }
  switch (g.epi) {
    case EPI_STORE:
      store_bf16x16(reinterpret_cast<__nv_bfloat16*>(g.out) + (int64_t)m * g.ldo + n, v);
      break;
    case EPI_RESID: {
      const float4* r4 = reinterpret_cast<const float4*>(g.resid + (int64_t)m * g.ldr + n);
      float4* o4 = reinterpret_cast<float4*>(reinterpret_cast<float*>(g.out) + (int64_t)m * g.ldo + n);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float4 r = r4[i];
        o4[i] = make_float4(r.x + v[4 * i], r.y + v[4 * i + 1], r.z + v[4 * i + 2], r.w + v[4 * i + 3]);
      }
    } break;
    case EPI_GELU: {
      store_bf16x16(reinterpret_cast<__nv_bfloat16*>(g.out) + (int64_t)m * g.ldo + n, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = gelu_f(v[i], gelu_tanh);
      store_bf16x16(reinterpret_cast<__nv_bfloat16*>(g.out2) + (int64_t)m * g.ldo2 + n, v);
    } break;
    case EPI_F32: {
      float4* o4 = reinterpret_cast<float4*>(reinterpret_cast<float*>(g.out) + split * g.split_stride +
                                             (int64_t)m * g.ldo + n);
#pragma unroll
      for (int i = 0; i < 4; ++i) o4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } break;
    case EPI_GELU_BWD: {
      const uint4* h4 = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(g.aux) +
                                                       (int64_t)m * g.ldaux + n);
      uint4 hu[2] = {h4[0], h4[1]};
      const __nv_bfloat16* hb = reinterpret_cast<const __nv_bfloat16*>(hu);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] *= gelu_grad_f(__bfloat162float(hb[i]), gelu_tanh);
      store_bf16x16(reinterpret_cast<__nv_bfloat16*>(g.out) + (int64_t)m * g.ldo + n, v);
    } break;
  }
}

// ---- the GEMM task -----------------------------------------------------------------------
// smem_tiles: 1024-byte aligned ring of kTcStages stages; bars: full[S], empty[S], acc.
__device__ inline void task_gemm_tc(const KParams& kp, const GemmArgs& g, int idx, uint8_t* smem_tiles,
                             uint64_t* bars, uint32_t tmem_base, TcState& st, bool gelu_tanh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles_m = (g.M + kTcBM - 1) / kTcBM;
  const int tn = idx % g.tiles_n;
  const int tm = (idx / g.tiles_n) % tiles_m;
  const int split = idx / (g.tiles_n * tiles_m);
  const int BN = g.BN;
  const int kchunk = (g.K + g.ksplit - 1) / g.ksplit;  // multiple of kTcBK (host checks)
  const int k0 = split * kchunk;
  const int nkb = (min(g.K, k0 + kchunk) - k0 + kTcBK - 1) / kTcBK;
  const int m0 = tm * kTcBM, n0 = tn * BN;
  const uint8_t* maps = reinterpret_cast<const uint8_t*>(kp.tmaps);  // 128-byte CUtensorMaps
  const void* amap = maps + 128 * g.a_map;
  const void* bmap = maps + 128 * g.b_map;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kTcStages),
                 accb = smem_u32(bars + 2 * kTcStages);
  const uint32_t tiles0 = smem_u32(smem_tiles);
  const uint32_t bytes = kTcStageA + (uint32_t)BN * kTcBK * 2;

  if (warp == 0 && lane == 0) {
    // ---- producer: TMA loads of A and B k-blocks into the ring ----
    fence_proxy_async_global();  // operands written by other blocks' generic stores
    for (int kb = 0; kb < nkb; ++kb) {
      if (!mbar_wait(kp, empty0 + 8 * st.prod_stage, st.prod_phase ^ 1u)) break;
      const uint32_t full = full0 + 8 * st.prod_stage;
      mbar_arrive_expect_tx(full, bytes);
      const uint32_t sa = tiles0 + st.prod_stage * kTcStageBytes;
      const uint32_t sb = sa + kTcStageA;
      const int kk = k0 + kb * kTcBK;
      if (!g.a_mn) {
        tma_load_2d(sa, amap, kk, m0, full);
      } else {
        tma_load_2d(sa, amap, m0, kk, full);
        tma_load_2d(sa + 8192, amap, m0 + 64, kk, full);
      }
      if (!g.b_mn) {
        tma_load_2d(sb, bmap, kk, n0, full);
      } else {
        for (int j = 0; j < BN / 64; ++j) tma_load_2d(sb + 8192 * j, bmap, n0 + 64 * j, kk, full);
      }
      if (++st.prod_stage == kTcStages) { st.prod_stage = 0; st.prod_phase ^= 1u; }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----
    const uint32_t idesc = idesc_bf16(kTcBM, BN, g.a_mn, g.b_mn);
    for (int kb = 0; kb < nkb; ++kb) {
      if (!mbar_wait(kp, full0 + 8 * st.mma_stage, st.mma_phase)) break;
      tc_fence_after();
      const uint32_t sa = tiles0 + st.mma_stage * kTcStageBytes;
      const uint32_t sb = sa + kTcStageA;
#pragma unroll
      for (int k = 0; k < kTcBK / 16; ++k) {
        const uint64_t ad = g.a_mn ? smem_desc_sw128(sa + k * 2048, 8192, 1024)
                                   : smem_desc_sw128(sa + k * 32, 16, 1024);
        const uint64_t bd = g.b_mn ? smem_desc_sw128(sb + k * 2048, 8192, 1024)
                                   : smem_desc_sw128(sb + k * 32, 16, 1024);
        tc_mma(tmem_base, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
      }
      tc_commit(empty0 + 8 * st.mma_stage);  // frees the stage once these MMAs have read it
      if (++st.mma_stage == kTcStages) { st.mma_stage = 0; st.mma_phase ^= 1u; }
    }
    tc_commit(accb);  // accumulator complete
  }
  __syncwarp();

  // ---- epilogue: all 8 warps; warp w reads TMEM lanes 32 (w % 4).., column half w / 4 ----
  const bool ok = mbar_wait(kp, accb, st.acc_phase);
  st.acc_phase ^= 1u;
  tc_fence_after();
  if (ok) {
    const int q = warp & 3, half = warp >> 2;
    const int row = m0 + q * 32 + lane;
    const int cbeg = half * (BN / 2), cend = cbeg + BN / 2;
    for (int c = cbeg; c < cend; c += 16) {
      float v[16];
      tmem_ld16(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)c, v);
      const int n = n0 + c;
      if (row < g.M && n < g.N) epilogue16(g, split, row, n, v, gelu_tanh);
    }
  }
  tc_fence_before();
}

}  // namespace pgs
