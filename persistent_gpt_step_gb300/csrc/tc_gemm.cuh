// tc_gemm.cuh — bf16 GEMM task on the 5th-generation tensor cores (sm_103a):
// TMA (cp.async.bulk.tensor, 128-byte swizzle) stages A and B tiles through a
// multi-stage shared-memory ring guarded by mbarriers; one thread issues
// tcgen05.mma (kind::f16, bf16 x bf16 -> fp32) into one of two TMEM
// accumulators; four epilogue warps read the other back with tcgen05.ld and run
// the fused epilogue (bias, residual add, GELU, GELU', fp32 or bf16 stores — the
// plain stores as bulk tensor copies of 32 x 32 boxes, the residual add as a bulk
// tensor reduction into the output, which already holds the residual stream).
//
// Operand majorness comes from the UMMA descriptors, not from transposes:
//   forward       C = X  W^T   A = X  [M,K] K-major,   B = W [N,K] K-major
//   input grad    C = dY W     A = dY [M,K] K-major,   B = W [K,N] MN-major
//   weight grad   C = dY^T X   A = dY [K,M] MN-major,  B = X [K,N] MN-major
#pragma once
#include "device.cuh"
#include "tasks_simt.cuh"

namespace pgs {

// Pipeline state a block carries across its GEMM runs for the whole launch.
// Each role thread keeps its own copy and advances only its own fields; the
// queue, tile-done and accumulator mbarriers are initialised once per launch
// and these counts give every wait its slot and phase parity.
struct TcState {
  uint32_t prod_stage, prod_phase;   // producer thread: operand stage ring
  uint32_t mma_stage, mma_phase;     // MMA thread: operand stage ring
  uint32_t q_seq;                    // queue entries published (scheduler) / taken (consumers)
  uint32_t acc_seq;                  // accumulators filled (MMA) / drained (epilogue)
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
  // the thread may sleep up to 1 us in the instruction until the phase completes
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(1000u)
      : "memory");
  return ok != 0;
}
// Bounded wait on an mbarrier phase; on expiry records a fatal error in err
// (the KParams error words: [0] code, [2] task, [3] counter).
__device__ __forceinline__ bool mbar_wait_e(uint32_t* err, uint64_t timeout_ns, uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  const uint64_t max_iters = timeout_ns / 20 + 1024;
  for (uint64_t it = 0; it < max_iters; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 63) {
      if (ld_volatile_u32(&err[0]) != 0u) return false;
      if (globaltimer_ns() - t0 > timeout_ns) break;
    }
  }
  if (atomicCAS(&err[0], 0u, kFatalMbarTimeout) == 0u) {
    err[2] = 0x80000000u | (threadIdx.x << 16) | blockIdx.x;  // which block and thread gave up
    err[3] = bar;
  }
  return false;
}
__device__ __forceinline__ bool mbar_wait(const KParams& kp, uint32_t bar, uint32_t parity) {
  return mbar_wait_e(kp.err, kp.timeout_ns, bar, parity);
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

// Stores a 32 x 32 box from shared memory (bulk async-group of this thread).
__device__ __forceinline__ void tma_store_2d(const void* tmap, int32_t c0, int32_t c1, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(tmap), "r"(c0),
               "r"(c1), "r"(src)
               : "memory");
}
// Adds a 32 x 32 fp32 box from shared memory into global memory (element-wise,
// performed at L2; bulk async-group of this thread).
__device__ __forceinline__ void tma_reduce_add_2d(const void* tmap, int32_t c0, int32_t c1, uint32_t src) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   tmap),
               "r"(c0), "r"(c1), "r"(src)
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
// Issue-only variant: the registers are valid after tmem_ld_wait16 on them.
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15},"
      " [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// Waits for this thread's outstanding tcgen05.ld; the register operands tie
// every later use of r to the wait, so no use is scheduled before it.
__device__ __forceinline__ void tmem_ld_wait16(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
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

// ---- epilogue on 64 consecutive columns of one row ------------------------------------
// GELU on the bf16 path uses the SFU tanh (tanh.approx.f32, relative error about
// 2^-11), below the bf16 rounding of the stored result.
__device__ __forceinline__ float tanh_sfu(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// GELU and its derivative at x together (one tanh for both in the tanh form):
// GELU(x) = 0.5 x (1 + t), GELU'(x) = 0.5 (1 + t) + 0.5 x (1 - t^2) k0 (1 + 3 c x^2),
// t = tanh(k0 (x + c x^3)), k0 = sqrt(2/pi), c = 0.044715; erf form otherwise.
__device__ __forceinline__ void gelu_pair_bf(float x, bool tanh_form, float& g, float& dg) {
  if (!tanh_form) {
    g = gelu_f(x, false);
    dg = gelu_grad_f(x, false);
    return;
  }
  // k0 (x + c x^3) = x (k0 + c k0 x^2); k0 (1 + 3 c x^2) = k0 + 3 c k0 x^2 (constants folded)
  const float k0 = 0.7978845608028654f, ck0 = 0.044715f * 0.7978845608028654f;
  const float x2 = x * x;
  const float t = tanh_sfu(x * fmaf(ck0, x2, k0));
  const float h = 0.5f * x;
  g = fmaf(h, t, h);
  dg = fmaf(h * fmaf(-t, t, 1.0f), fmaf(3.0f * ck0, x2, k0), fmaf(0.5f, t, 0.5f));
}

// Two-wide fp32 arithmetic (fma / mul / add .rn.f32x2, sm_100 and later): one
// instruction for two independent lanes, each rounded as the scalar operation is.
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%6, %7};\n"
      " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 f2_add(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
// The tanh-form GELU pair of two inputs with the two-wide instructions; the same
// roundings as gelu_pair_bf (1 - t^2 and k0 + 3 c k0 x^2 are formed negated, which
// is exact), so the results are bitwise those of two scalar calls.
__device__ __forceinline__ void gelu_pair_tanh2(float2 x, float2& g, float2& dg) {
  constexpr float k0 = 0.7978845608028654f, ck0 = 0.044715f * 0.7978845608028654f;
  const float2 x2 = f2_mul(x, x);
  const float2 arg = f2_mul(x, f2_fma(make_float2(ck0, ck0), x2, make_float2(k0, k0)));
  const float2 t = make_float2(tanh_sfu(arg.x), tanh_sfu(arg.y));
  const float2 h = f2_mul(make_float2(0.5f, 0.5f), x);
  g = f2_fma(h, t, h);
  const float2 p = f2_fma(make_float2(0.5f, 0.5f), t, make_float2(0.5f, 0.5f));
  const float2 nq = f2_fma(make_float2(-3.0f * ck0, -3.0f * ck0), x2, make_float2(-k0, -k0));  // -(k0 + 3 c k0 x^2)
  const float2 w = f2_mul(h, f2_fma(t, t, make_float2(-1.0f, -1.0f)));                        // -h (1 - t^2)
  dg = f2_fma(w, nq, p);
}

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

// One epilogue warp's part of a tile: TMEM lane quarter (32 rows from row0),
// all BN columns, in 32-column groups.  The accumulators go TMEM -> registers
// -> a per-warp 32 x 32 fp32 staging tile in shared memory (16-byte chunks
// XOR-swizzled by row) -> back to registers in a row-contiguous layout: thread
// u owns columns 4 (u mod 8) .. +3 of rows 4i + u / 8, so bias, GELU and
// the stores touch whole 64- or 128-byte row segments.
//
// An epilogue that reads a second operand (the stored GELU derivative, the
// gated MLP's pairs) issues all 8 of a group's loads at once: the first group's
// before waiting for the accumulator (they land while the MMAs still run), each
// next group's before the current one is processed, so a tile pays about one
// memory latency instead of one per few rows.  Returns false when the wait for
// the accumulator (acc_bar, parity) timed out or another block failed.
template <int EPI>
struct EpiSrc {
  using T = uint2;  // EPI_GELU_BWD: four bf16 GELU derivatives
};
template <>
struct EpiSrc<EPI_GEGLU_BWD> {
  using T = uint4;  // the (gate, up) bf16 pairs of four features
};

template <int EPI>
__device__ __forceinline__ void epi_load_src(typename EpiSrc<EPI>::T* dst, const void* src, int64_t lds, int M,
                                             int r0, int col) {
  using T = typename EpiSrc<EPI>::T;
  constexpr int64_t es = 2;                                  // element bytes of the source (bf16)
  constexpr int64_t cw = EPI == EPI_GEGLU_BWD ? 2 : 1;       // source columns per output column
  const T* p = reinterpret_cast<const T*>(reinterpret_cast<const char*>(src) + ((int64_t)r0 * lds + cw * col) * es);
  const int64_t step = 4 * lds * es / (int64_t)sizeof(T);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (r0 + 4 * i < M) dst[i] = p[i * step];
}

template <int EPI>
static __device__ __noinline__ bool epi_tile(const int M, const int N, const int BN, const int row0, const int n0,
                                             const uint32_t tbase, uint8_t* stage, void* const out,
                                             const int64_t ldo, void* const out2, const int64_t ldo2,
                                             const float* const bias, const void* const src, const int64_t lds,
                                             const bool gelu_tanh, const int n_real, float* const bias_grad,
                                             const uint32_t acc_bar, const uint32_t acc_parity, uint32_t* const err,
                                             const uint64_t timeout_ns, const void* const cmap, const int crow0) {
  constexpr bool kSrc = EPI == EPI_GELU_BWD || EPI == EPI_GEGLU_BWD;
  using SrcT = typename EpiSrc<EPI>::T;
  const int lane = threadIdx.x & 31;
  const int cu = 4 * (lane & 7);     // this thread's first column within the group
  const int rq = lane >> 3;          // first row (of 4)
  const int r0 = row0 + rq;
  const int cend = min(BN, N - n0);  // N is a multiple of 64
  // The second operand (the stored GELU derivative, the gated pairs) is staged
  // with cp.async, each thread's own eight pieces in the upper half of the warp's
  // staging area ([slot][row i][lane]): two 2 KB slots, two column groups ahead,
  // for the 8-byte derivative pieces; one 4 KB slot, one group ahead, for the
  // 16-byte pairs.  No registers are held while the copies are in flight.
  constexpr int kPiece = (int)sizeof(SrcT);
  constexpr int kSlots = EPI == EPI_GELU_BWD ? 2 : 1;
  constexpr uint32_t kSlotBytes = 8u * 32u * (uint32_t)kPiece;
  constexpr int64_t kCw = EPI == EPI_GEGLU_BWD ? 2 : 1;  // source columns per output column
  const uint32_t aslot = smem_u32(stage) + 4096u;
  auto async_src = [&](int c, uint32_t slot) {
    const int col = n0 + c + cu;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = r0 + 4 * i;
      const char* g = r < M ? reinterpret_cast<const char*>(src) + ((int64_t)r * lds + kCw * col) * 2
                            : reinterpret_cast<const char*>(src);
      asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;" ::"r"(aslot + slot * kSlotBytes +
                                                                         (uint32_t)(i * 32 + lane) * (uint32_t)kPiece),
                   "l"(g), "n"(kPiece), "r"(r < M ? kPiece : 0)
                   : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  if constexpr (kSrc) {
    async_src(0, 0u);
    if (kSlots == 2 && 32 < cend) async_src(32, 1u);
  }
  const bool acc_ok = mbar_wait_e(err, timeout_ns, acc_bar, acc_parity);
  __syncwarp();  // lanes leave the poll loop separately; tcgen05.ld below is warp-aligned
  if (!acc_ok) return false;
  tc_fence_after();
  if constexpr (EPI == EPI_STORE || EPI == EPI_STORE_ROPE || EPI == EPI_F32 || EPI == EPI_RESID) {
    if (cmap) {
      // TMA-store path: each lane holds its own row's 32 columns, writes them
      // (bias added and rounded to bf16, or fp32) into a swizzled 32 x 32 box in
      // the warp's staging area (two boxes, alternating), and lane 0 stores the
      // box with one bulk tensor copy — one pass through shared memory and no
      // per-row global stores.  The residual epilogue (its output already holds
      // the residual stream, copied there by the LayerNorm that read it) adds the
      // box (accumulator + bias, fp32) into the output with a bulk tensor
      // reduction instead: out = residual + (acc + bias), one rounding, as the
      // row path computes it.
      const uint32_t sbase = smem_u32(stage);
      int gi = 0;
      for (int c = 0; c < cend; c += 32, ++gi) {
        const int n = n0 + c;
        uint32_t r[2][16];
        tmem_ld16_issue(tbase + (uint32_t)c, r[0]);
        tmem_ld16_issue(tbase + (uint32_t)(c + 16), r[1]);
        tmem_ld_wait16(r[0]);
        tmem_ld_wait16(r[1]);
        if constexpr (EPI == EPI_F32) {
          if (n >= n_real) {  // the padded columns: the first is the bias gradient, the rest are dropped
            if (n == n_real && bias_grad && row0 + lane < M) bias_grad[row0 + lane] = __uint_as_float(r[0][0]);
            continue;
          }
        }
        const uint32_t buf = sbase + (uint32_t)(gi & 1) * 4096u;
        if (gi >= 2 && lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncwarp();  // the box written two groups ago has been read by its store
        if constexpr (EPI == EPI_F32) {
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)  // 128-byte rows, 16-byte chunk ch at ch ^ (row mod 8)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(buf + lane * 128 + ((ch ^ (lane & 7)) << 4)),
                         "r"(r[ch >> 2][4 * (ch & 3)]), "r"(r[ch >> 2][4 * (ch & 3) + 1]),
                         "r"(r[ch >> 2][4 * (ch & 3) + 2]), "r"(r[ch >> 2][4 * (ch & 3) + 3])
                         : "memory");
        } else if constexpr (EPI == EPI_RESID) {
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {  // the same 128-byte swizzled rows, bias added
            float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
            if (bias) b = reinterpret_cast<const float4*>(bias + n)[ch];
            const uint32_t* x = &r[ch >> 2][4 * (ch & 3)];
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(buf + lane * 128 + ((ch ^ (lane & 7)) << 4)),
                         "f"(__uint_as_float(x[0]) + b.x), "f"(__uint_as_float(x[1]) + b.y),
                         "f"(__uint_as_float(x[2]) + b.z), "f"(__uint_as_float(x[3]) + b.w)
                         : "memory");
          }
        } else {
          uint32_t w[16];
          // rotary embedding of q and k (src: the (cos, sin) table of period lds)
          const float2* cs = (EPI == EPI_STORE_ROPE && n < 2 * (N / 3))
                                 ? reinterpret_cast<const float2*>(src) + (int64_t)((row0 + lane) % (int)lds) * 32 +
                                       ((n & 63) >> 1)
                                 : nullptr;
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
            if (bias) b = reinterpret_cast<const float4*>(bias + n)[q4];
            const uint32_t* x = &r[q4 >> 2][4 * (q4 & 3)];
            float y0 = __uint_as_float(x[0]) + b.x, y1 = __uint_as_float(x[1]) + b.y;
            float y2 = __uint_as_float(x[2]) + b.z, y3 = __uint_as_float(x[3]) + b.w;
            if (cs) {
              const float2 c0 = cs[2 * q4], c1 = cs[2 * q4 + 1];
              const float t0 = y0 * c0.x - y1 * c0.y, t1 = y0 * c0.y + y1 * c0.x;
              const float t2 = y2 * c1.x - y3 * c1.y, t3 = y2 * c1.y + y3 * c1.x;
              y0 = t0; y1 = t1; y2 = t2; y3 = t3;
            }
            __nv_bfloat162 lo = __floats2bfloat162_rn(y0, y1);
            __nv_bfloat162 hi = __floats2bfloat162_rn(y2, y3);
            w[2 * q4] = *reinterpret_cast<uint32_t*>(&lo);
            w[2 * q4 + 1] = *reinterpret_cast<uint32_t*>(&hi);
          }
#pragma unroll
          for (int ch = 0; ch < 4; ++ch)  // 64-byte rows, 16-byte chunk ch at ch ^ ((row / 2) mod 4)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                         ::"r"(buf + lane * 64 + ((ch ^ ((lane >> 1) & 3)) << 4)), "r"(w[4 * ch]),
                         "r"(w[4 * ch + 1]), "r"(w[4 * ch + 2]), "r"(w[4 * ch + 3])
                         : "memory");
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic smem writes -> the bulk copy
        __syncwarp();
        if (lane == 0) {
          if constexpr (EPI == EPI_RESID) tma_reduce_add_2d(cmap, n, crow0, buf);
          else tma_store_2d(cmap, n, crow0, buf);
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
      }
      if (lane == 0) {  // the tile's stores are complete before the warp reports it done
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        fence_proxy_async_global();
      }
      __syncwarp();
      return true;
    }
  }
  if constexpr (EPI == EPI_RESID) {
    return false;  // the residual epilogue has only the reduction path
  } else {
  for (int c = 0; c < cend; c += 32) {
    const int n = n0 + c;
    {
      uint32_t r[2][16];
      tmem_ld16_issue(tbase + (uint32_t)c, r[0]);
      tmem_ld16_issue(tbase + (uint32_t)(c + 16), r[1]);
      tmem_ld_wait16(r[0]);
      tmem_ld_wait16(r[1]);
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int ch = 4 * j + h;  // 16-byte chunk of this thread's row
          *reinterpret_cast<uint4*>(stage + lane * 128 + ((ch ^ (lane & 7)) << 4)) =
              make_uint4(r[j][4 * h], r[j][4 * h + 1], r[j][4 * h + 2], r[j][4 * h + 3]);
        }
      __syncwarp();
    }
    SrcT cur[kSrc ? 8 : 1];
    if constexpr (kSrc) {
      const uint32_t slot = kSlots == 2 ? ((uint32_t)(c >> 5) & 1u) : 0u;
      if (kSlots == 2 && c + 32 < cend) asm volatile("cp.async.wait_group 1;" ::: "memory");  // this group landed
      else asm volatile("cp.async.wait_group 0;" ::: "memory");
      const uint32_t sp = aslot + slot * kSlotBytes + (uint32_t)lane * (uint32_t)kPiece;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t ad = sp + (uint32_t)(i * 32 * kPiece);
        if constexpr (kPiece == 8) {
          uint2 v;
          asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(ad) : "memory");
          cur[i] = *reinterpret_cast<SrcT*>(&v);
        } else {
          uint4 v;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(ad)
                       : "memory");
          cur[i] = *reinterpret_cast<SrcT*>(&v);
        }
      }
      // refill the slot just read (by this thread alone)
      if (kSlots == 2 && c + 64 < cend) async_src(c + 64, slot);
      if (kSlots == 1 && c + 32 < cend) async_src(c + 32, 0u);
    }
    const int col = n + cu;
    float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
    if (EPI != EPI_F32 && EPI != EPI_GELU_BWD && EPI != EPI_GEGLU_BWD && bias)
      b = *reinterpret_cast<const float4*>(bias + col);
    // the thread's 8 rows are read from the staging tile before any of them is
    // processed: the global stores below may alias the staging pointer as far as
    // the compiler knows, so reads interleaved with them would run one row at a
    // time; read first, the 32 values' arithmetic chains are independent
    float4 vr[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rl = rq + 4 * i;
      vr[i] = *reinterpret_cast<const float4*>(stage + rl * 128 + (((lane & 7) ^ (rl & 7)) << 4));
    }
    auto row = [&](const int i) {
      const int rl = rq + 4 * i;
      const int m = row0 + rl;
      float4 v = vr[i];
      v.x += b.x; v.y += b.y; v.z += b.z; v.w += b.w;
      if constexpr (EPI == EPI_STORE || EPI == EPI_STORE_ROPE) {
        if constexpr (EPI == EPI_STORE_ROPE) {
          if (n < 2 * (N / 3)) {  // rotary embedding of q and k (src: the (cos, sin) table, lds: its period)
            const float2* cs =
                reinterpret_cast<const float2*>(src) + (int64_t)(m % (int)lds) * 32 + ((col & 63) >> 1);
            const float2 c0 = cs[0], c1 = cs[1];
            v = make_float4(v.x * c0.x - v.y * c0.y, v.x * c0.y + v.y * c0.x, v.z * c1.x - v.w * c1.y,
                            v.z * c1.y + v.w * c1.x);
          }
        }
        __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + (int64_t)m * ldo + col) =
            make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
      } else if constexpr (EPI == EPI_GELU) {  // out = GELU'(v) for the backward, out2 = GELU(v)
        float g[4], dg[4];
        if (gelu_tanh) {
          float2 g01, d01, g23, d23;
          gelu_pair_tanh2(make_float2(v.x, v.y), g01, d01);
          gelu_pair_tanh2(make_float2(v.z, v.w), g23, d23);
          g[0] = g01.x; g[1] = g01.y; g[2] = g23.x; g[3] = g23.y;
          dg[0] = d01.x; dg[1] = d01.y; dg[2] = d23.x; dg[3] = d23.y;
        } else {
          gelu_pair_bf(v.x, false, g[0], dg[0]);
          gelu_pair_bf(v.y, false, g[1], dg[1]);
          gelu_pair_bf(v.z, false, g[2], dg[2]);
          gelu_pair_bf(v.w, false, g[3], dg[3]);
        }
        __nv_bfloat162 lo = __floats2bfloat162_rn(dg[0], dg[1]), hi = __floats2bfloat162_rn(dg[2], dg[3]);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + (int64_t)m * ldo + col) =
            make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
        lo = __floats2bfloat162_rn(g[0], g[1]);
        hi = __floats2bfloat162_rn(g[2], g[3]);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out2) + (int64_t)m * ldo2 + col) =
            make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
      } else if constexpr (EPI == EPI_F32) {
        if (n >= n_real) {  // the padded columns: the first is the bias gradient
          if (n == n_real && cu == 0 && bias_grad) bias_grad[m] = v.x;
        } else {
          *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + (int64_t)m * ldo + col) = v;
        }
      } else if constexpr (EPI == EPI_GEGLU) {  // out = (gate, up) kept; out2 = GELU(gate) * up
        __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + (int64_t)m * ldo + col) =
            make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
        float g0, g1, d0, d1;
        gelu_pair_bf(v.x, gelu_tanh, g0, d0);
        gelu_pair_bf(v.z, gelu_tanh, g1, d1);
        (void)d0; (void)d1;
        __nv_bfloat162 hv = __floats2bfloat162_rn(g0 * v.y, g1 * v.w);
        *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(out2) + (int64_t)m * ldo2 + (col >> 1)) = hv;
      } else if constexpr (EPI == EPI_GEGLU_BWD) {  // v = dh of features col..col+3
        const uint4 gu = cur[i];
        const uint32_t w[4] = {gu.x, gu.y, gu.z, gu.w};
        const float dh[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[j]));  // (gate, up)
          float g, dg;
          gelu_pair_bf(a.x, gelu_tanh, g, dg);
          __nv_bfloat162 t = __floats2bfloat162_rn(dh[j] * a.y * dg, dh[j] * g);
          o[j] = *reinterpret_cast<uint32_t*>(&t);
        }
        *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out) + (int64_t)m * ldo + 2 * col) =
            make_uint4(o[0], o[1], o[2], o[3]);
      } else if constexpr (EPI == EPI_GELU_BWD) {
        const uint2 hv = cur[i];  // GELU'(pre-activation), stored by the forward
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hv.x));
        const float2 e = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hv.y));
        __nv_bfloat162 lo = __floats2bfloat162_rn(v.x * a.x, v.y * a.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(v.z * e.x, v.w * e.y);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + (int64_t)m * ldo + col) =
            make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
      }
    };
    if (row0 + 32 <= M) {  // every row of this warp exists: no per-row branch
#pragma unroll
      for (int i = 0; i < 8; ++i) row(i);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (row0 + rq + 4 * i < M) row(i);
    }
  }
  return true;
  }
}

// Waits for the tile's accumulator and runs its epilogue (false: the wait failed).
// kExt: the kernel of the rotary / gated-MLP model variant, which alone carries
// those epilogues (the plain model's kernel keeps its register allocation).
template <bool kExt>
__device__ __forceinline__ bool epilogue_tile(const KParams& kp, const GemmArgs& g, int split, int row0, int n0,
                                              uint32_t tbase, uint8_t* stage, bool gelu_tanh, uint32_t acc_bar,
                                              uint32_t acc_parity) {
  const void* const cmap = g.c_map >= 0 ? reinterpret_cast<const uint8_t*>(kp.tmaps) + 128 * g.c_map : nullptr;
  const int crow0 = row0 + split * g.M;
  switch (g.epi) {
    case EPI_STORE:
      return epi_tile<EPI_STORE>(g.M, g.N, g.BN, row0, n0, tbase, stage, g.out, g.ldo, nullptr, 0, g.bias, nullptr,
                                 0, gelu_tanh, g.N, nullptr, acc_bar, acc_parity, kp.err, kp.timeout_ns, cmap, crow0);
    case EPI_STORE_ROPE:  // second operand: the rotary table and its period
      if constexpr (kExt)
        return epi_tile<EPI_STORE_ROPE>(g.M, g.N, g.BN, row0, n0, tbase, stage, g.out, g.ldo, nullptr, 0, g.bias,
                                        g.rope, g.rope_T, gelu_tanh, g.N, nullptr, acc_bar, acc_parity, kp.err,
                                        kp.timeout_ns, cmap, crow0);
      return false;
    case EPI_GEGLU:
      if constexpr (kExt)
        return epi_tile<EPI_GEGLU>(g.M, g.N, g.BN, row0, n0, tbase, stage, g.out, g.ldo, g.out2, g.ldo2, g.bias,
                                   nullptr, 0, gelu_tanh, g.N, nullptr, acc_bar, acc_parity, kp.err, kp.timeout_ns,
                                   nullptr, crow0);
      return false;
    case EPI_GEGLU_BWD:
      if constexpr (kExt)
        return epi_tile<EPI_GEGLU_BWD>(g.M, g.N, g.BN, row0, n0, tbase, stage, g.out, g.ldo, nullptr, 0, nullptr,
                                       g.aux, g.ldaux, gelu_tanh, g.N, nullptr, acc_bar, acc_parity, kp.err,
                                       kp.timeout_ns, nullptr, crow0);
      return false;
    case EPI_RESID:
      return epi_tile<EPI_RESID>(g.M, g.N, g.BN, row0, n0, tbase, stage, g.out, g.ldo, nullptr, 0, g.bias, g.resid,
                                 g.ldr, gelu_tanh, g.N, nullptr, acc_bar, acc_parity, kp.err, kp.timeout_ns, cmap, crow0);
    case EPI_GELU:
      return epi_tile<EPI_GELU>(g.M, g.N, g.BN, row0, n0, tbase, stage, g.out, g.ldo, g.out2, g.ldo2, g.bias,
                                nullptr, 0, gelu_tanh, g.N, nullptr, acc_bar, acc_parity, kp.err, kp.timeout_ns, cmap, crow0);
    case EPI_F32:
      return epi_tile<EPI_F32>(g.M, g.N, g.BN, row0, n0, tbase, stage,
                               reinterpret_cast<float*>(g.out) + split * g.split_stride, g.ldo, nullptr, 0, nullptr,
                               nullptr, 0, gelu_tanh, g.n_real, g.bias_grad, acc_bar, acc_parity, kp.err,
                               kp.timeout_ns, cmap, crow0);
    default:
      return epi_tile<EPI_GELU_BWD>(g.M, g.N, g.BN, row0, n0, tbase, stage, g.out, g.ldo, nullptr, 0, nullptr, g.aux,
                                    g.ldaux, gelu_tanh, g.N, nullptr, acc_bar, acc_parity, kp.err, kp.timeout_ns, cmap, crow0);
  }
}

// ---- GEMM runs: warp-specialised pipeline over consecutive GEMM tasks ---------------
//
// While a block's current task is a GEMM, its warps split into roles that each
// loop over the same sequence of GEMM tasks:
//   warp 2         scheduler: lane 0 claims the next ticket once a queue slot
//                  is free and the producer has issued three quarters of the
//                  current tile's k-blocks (a ticket held but not started is work
//                  no other block can take), waits for its dependencies, and the
//                  warp copies the op's arguments into the slot in shared memory;
//   warp 0 lane 0  TMA producer: k-blocks of A and B into the stage ring;
//   warp 1 lane 0  MMA issuer: tcgen05.mma into one of two TMEM accumulators;
//   warps 4..7     epilogue: TMEM -> registers -> fused epilogue -> global,
//                  each warp on its own 32 rows, without waiting for the others;
//   warp 3 lane 0  releaser: once the four epilogue warps are done with a tile,
//                  publishes it (proxy fence + release add) and frees its slot.
// Tile i+1's loads and MMAs therefore overlap tile i's epilogue, and no
// epilogue warp waits for a release to drain its stores.  The run ends when the
// scheduler claims a task that is not a GEMM (or the graph ends); that ticket
// goes back to the main loop, dependencies not yet waited.
constexpr int kQSlots = 2;

struct GemmShared {
  uint64_t stage_full[kTcStages], stage_empty[kTcStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t q_full[kQSlots], q_empty[kQSlots];
  uint64_t tile_done[kQSlots];  // the four epilogue warps finished the slot's tile
  int64_t q_task[kQSlots];
  int32_t q_idx[kQSlots], q_sig[kQSlots], q_sig2[kQSlots];
  GemmArgs q_args[kQSlots];     // the op's arguments, read by every role from here
  int64_t next;
  uint32_t prod_claim;          // queue entries for which the producer has passed the claim point
};

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// The queue slots are rewritten by the scheduler once the producer, the MMA
// issuer and the releaser have signalled "slot empty" (the releaser does so only
// after the epilogue warps finished the slot's tile).  A role reads the slot's
// task word exactly once; volatile accesses keep the compiler from re-reading it
// later (a plain load may legally be repeated under register pressure).
__device__ __forceinline__ int64_t q_read(const int64_t* slot) { return *reinterpret_cast<const volatile int64_t*>(slot); }
__device__ __forceinline__ void q_write(int64_t* slot, int64_t v) { *reinterpret_cast<volatile int64_t*>(slot) = v; }

// With tracing on, each GEMM role keeps its current wait in a per-block record
// after the per-task trace (8 words per block: scheduler, producer, MMA, the four
// epilogue warps, spare): kind << 56 | (i mod 2^24) << 32 | task.  After a failed
// step the host reads where every block's pipeline stopped.
enum RoleWait : uint32_t {
  RW_SCHED_READY = 1, RW_SCHED_QEMPTY, RW_PROD_QFULL, RW_PROD_STAGE, RW_MMA_QFULL, RW_MMA_ACC, RW_MMA_STAGE,
  RW_EPI_QFULL, RW_EPI_TILE, RW_EPI_DONE, RW_DONE
};
__device__ __forceinline__ void role_note(const KParams& kp, int role, uint32_t kind, uint32_t i, int64_t t) {
  if (kp.trace)
    kp.trace[4 * kp.ntasks + 8 * blockIdx.x + role] =
        ((unsigned long long)kind << 56) | ((unsigned long long)(i & 0xffffffu) << 32) | (uint32_t)t;
}

// Queue position of entry seq: its slot and the phase parity of that slot's use.
__device__ __forceinline__ uint32_t q_slot(uint32_t seq) { return seq % kQSlots; }
__device__ __forceinline__ uint32_t q_parity(uint32_t seq) { return (seq / kQSlots) & 1u; }

// The epilogue warps' part of a GEMM run (warps 4..7 read TMEM lane quarters
// 0..3): for each queue entry, wait for the tile's accumulator, run the fused
// epilogue on the warp's 32 rows, hand the accumulator back to the MMA issuer
// and tell the releaser the warp is done.  Out of line, so the live state
// around the epilogue calls is this loop's alone (the epilogue bodies keep their
// registers).  Returns the updated queue and accumulator sequence counts.
template <bool kExt>
static __device__ __noinline__ uint2 epilogue_role(const KParams* const kpp, GemmShared& gs, const uint32_t tmem_base,
                                                   uint8_t* const smem_tiles, uint32_t q_seq, uint32_t acc_seq,
                                                   const bool gelu_tanh) {
  const KParams kp = *kpp;  // a value copy: fields stay in registers across asm memory clobbers
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t q_full0 = smem_u32(&gs.q_full[0]), done0 = smem_u32(&gs.tile_done[0]);
  const uint32_t acc_full0 = smem_u32(&gs.acc_full[0]), acc_empty0 = smem_u32(&gs.acc_empty[0]);
  const int q = warp & 3;
  for (uint32_t i = 0;; ++i) {
    const uint32_t seq = q_seq, slot = q_slot(seq);
    if (lane == 0) role_note(kp, 3 + q, RW_EPI_QFULL, i, -1);
    if (!mbar_wait(kp, q_full0 + 8 * slot, q_parity(seq))) break;
    const int64_t t = q_read(&gs.q_task[slot]);
    ++q_seq;
    if (t < 0) {
      // every use of a slot completes one tile-done phase, the run's last
      // (non-GEMM) entry included, so the phase parities follow the queue's
      __syncwarp();
      if (lane == 0) mbar_arrive(done0 + 8 * slot);
      break;
    }
    const uint32_t acc = acc_seq, buf = acc & 1;
    ++acc_seq;
    const GemmArgs& g = gs.q_args[slot];  // valid until the releaser frees the slot, after this tile
    int tm, tn, split;
    gemm_coords(g, gs.q_idx[slot], tm, tn, split);
    if (lane == 0) role_note(kp, 3 + q, RW_EPI_TILE, i, t);
    const bool ok = epilogue_tile<kExt>(kp, g, split, tm * kTcBM + q * 32, tn * g.BN,
                                  tmem_base + ((uint32_t)(q * 32) << 16) + buf * 256,
                                  smem_tiles + kTcSmemBytes + (warp - 4) * kEpiStageBytes, gelu_tanh,
                                  acc_full0 + 8 * buf, (acc >> 1) & 1);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(acc_empty0 + 8 * buf);
      mbar_arrive(done0 + 8 * slot);  // release (CTA scope): this warp's stores precede it
      role_note(kp, 3 + q, RW_EPI_DONE, i, t);
    }
    if (!ok) break;
  }
  return make_uint2(q_seq, acc_seq);
}

// Scheduler role (warp 2): claims tickets ahead and fills the queue.
static __device__ __noinline__ TcState scheduler_role(const KParams* const kpp, GemmShared& gs,
                                                 uint8_t* const smem_tiles, const uint32_t tmem_base, TcState st,
                                                 const int64_t t_first) {
  const KParams kp = *kpp;  // a value copy: fields stay in registers across asm memory clobbers
  const int lane = threadIdx.x & 31;
  (void)lane;
  const uint32_t q_full0 = smem_u32(&gs.q_full[0]), q_empty0 = smem_u32(&gs.q_empty[0]);
  const uint32_t done0 = smem_u32(&gs.tile_done[0]);
  const uint32_t acc_full0 = smem_u32(&gs.acc_full[0]), acc_empty0 = smem_u32(&gs.acc_empty[0]);
  const uint32_t full0 = smem_u32(&gs.stage_full[0]), empty0 = smem_u32(&gs.stage_empty[0]);
  const uint32_t tiles0 = smem_u32(smem_tiles);
  const uint8_t* maps = reinterpret_cast<const uint8_t*>(kp.tmaps);  // 128-byte CUtensorMaps
  (void)q_full0; (void)q_empty0; (void)done0; (void)acc_full0; (void)acc_empty0; (void)full0; (void)empty0;
  (void)tiles0; (void)maps; (void)tmem_base; (void)t_first;
  // ---- scheduler: publishes t_first, then claims ahead.  Lane 0 claims and
  // waits; the whole warp copies the op's arguments into the slot (one 8-byte
  // word per lane, so no thread holds the whole struct in registers). ----
  static_assert(sizeof(GemmArgs) % 8 == 0 && sizeof(GemmArgs) <= 32 * 8, "GemmArgs copy");
  for (uint32_t i = 0;; ++i) {
    int64_t t = t_first;
    int gemm = 1, stop = 0;
    uint32_t slot = 0;
    if (lane == 0) {
      const uint32_t seq = st.q_seq;
      slot = q_slot(seq);
      role_note(kp, 0, RW_SCHED_QEMPTY, i, t);
      if (seq >= kQSlots && !mbar_wait(kp, q_empty0 + 8 * slot, q_parity(seq) ^ 1u)) {
        gs.next = kp.ntasks;
        stop = 1;
      }
      if (!stop && i > 0) {  // claim only once the slot is free: no ticket is held longer than needed
        // ... and the producer has issued three quarters of the previous entry's k-blocks
        const uint64_t t0 = globaltimer_ns();
        while (*reinterpret_cast<volatile uint32_t*>(&gs.prod_claim) < st.q_seq) {
          __nanosleep(64);  // leave the issue slots to the epilogue warp of this sub-partition
          if (globaltimer_ns() - t0 > kp.timeout_ns) break;  // no error: claiming late is only slower
        }
        t = kp.ntasks;
        gemm = 0;
        if (ld_volatile_u32(&kp.err[0]) == 0u) {
          t = claim_task(kp);
          if (t < kp.ntasks && kp.ops[kp.tasks[t].op].type == OP_GEMM) {
            const uint64_t t_claim = kp.trace ? globaltimer_ns() : 0;
            role_note(kp, 0, RW_SCHED_READY, i, t);
            gemm = task_ready(kp, t) ? 1 : 0;
            if (!gemm) t = kp.ntasks;  // a wait failed: stop the run, the main loop drains
            else if (kp.trace) {
              kp.trace[4 * t + 0] = t_claim;
              kp.trace[4 * t + 1] = globaltimer_ns();
              uint32_t smid;
              asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
              kp.trace[4 * t + 3] = smid | ((unsigned long long)blockIdx.x << 32);
            }
          }
        }
      }
    }
    __syncwarp();
    stop = __shfl_sync(0xffffffffu, stop, 0);
    if (stop) break;
    gemm = __shfl_sync(0xffffffffu, gemm, 0);
    t = __shfl_sync(0xffffffffu, t, 0);
    slot = __shfl_sync(0xffffffffu, slot, 0);
    if (gemm) {
      const TaskDesc& d = kp.tasks[t];
      if (lane < (int)(sizeof(GemmArgs) / 8))
        reinterpret_cast<uint64_t*>(&gs.q_args[slot])[lane] =
            reinterpret_cast<const uint64_t*>(&kp.ops[d.op].gemm)[lane];
      if (lane == 0) {
        gs.q_idx[slot] = d.idx;
        gs.q_sig[slot] = d.sig;
        gs.q_sig2[slot] = d.sig2;
      }
    }
    __syncwarp();  // every lane's copy precedes lane 0's arrival
    if (lane == 0) {
      q_write(&gs.q_task[slot], gemm ? t : -2 - t);
      mbar_arrive(q_full0 + 8 * slot);  // release: the slot's contents precede the arrival
      ++st.q_seq;
      if (!gemm) gs.next = t;
    }
    if (!gemm) break;
  }
  return st;
}

// TMA producer role (warp 0 lane 0): streams each tile's k-blocks of A and B.
static __device__ __forceinline__ TcState producer_role(const KParams* const kpp, GemmShared& gs,
                                                 uint8_t* const smem_tiles, const uint32_t tmem_base, TcState st,
                                                 const int64_t t_first) {
  const KParams kp = *kpp;  // a value copy: fields stay in registers across asm memory clobbers
  const int lane = threadIdx.x & 31;
  (void)lane;
  const uint32_t q_full0 = smem_u32(&gs.q_full[0]), q_empty0 = smem_u32(&gs.q_empty[0]);
  const uint32_t done0 = smem_u32(&gs.tile_done[0]);
  const uint32_t acc_full0 = smem_u32(&gs.acc_full[0]), acc_empty0 = smem_u32(&gs.acc_empty[0]);
  const uint32_t full0 = smem_u32(&gs.stage_full[0]), empty0 = smem_u32(&gs.stage_empty[0]);
  const uint32_t tiles0 = smem_u32(smem_tiles);
  const uint8_t* maps = reinterpret_cast<const uint8_t*>(kp.tmaps);  // 128-byte CUtensorMaps
  (void)q_full0; (void)q_empty0; (void)done0; (void)acc_full0; (void)acc_empty0; (void)full0; (void)empty0;
  (void)tiles0; (void)maps; (void)tmem_base; (void)t_first;
  if (lane == 0) {
    // ---- TMA producer ----
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // smem last written by generic stores
    for (uint32_t i = 0;; ++i) {
      const uint32_t seq = st.q_seq, slot = q_slot(seq);
      role_note(kp, 1, RW_PROD_QFULL, i, -1);
      if (!mbar_wait(kp, q_full0 + 8 * slot, q_parity(seq))) break;
      const int64_t t = q_read(&gs.q_task[slot]);
      ++st.q_seq;
      if (t < 0) {
        mbar_arrive(q_empty0 + 8 * slot);
        break;
      }
      const GemmArgs& g = gs.q_args[slot];
      int tm, tn, split;
      gemm_coords(g, gs.q_idx[slot], tm, tn, split);
      const int kchunk = (g.K + g.ksplit - 1) / g.ksplit;
      const int k0 = split * kchunk;
      const int nkb = (min(g.K, k0 + kchunk) - k0 + kTcBK - 1) / kTcBK;
      const int m0 = tm * kTcBM, n0 = tn * g.BN;
      const void* amap = maps + 128 * g.a_map;
      const void* bmap = maps + 128 * g.b_map;
      const uint32_t bytes = kTcStageA + (uint32_t)g.BN * kTcBK * 2;
      const int a_mn = g.a_mn, b_mn = g.b_mn, bn64 = g.BN / 64;
      mbar_arrive(q_empty0 + 8 * slot);  // everything needed is in registers now
      role_note(kp, 1, RW_PROD_STAGE, i, t);
      fence_proxy_async_global();  // operands written by other blocks' generic stores
      bool ok = true;
      for (int kb = 0; kb < nkb && ok; ++kb) {
        if (kb == (3 * nkb) / 4) *reinterpret_cast<volatile uint32_t*>(&gs.prod_claim) = st.q_seq;
        ok = mbar_wait(kp, empty0 + 8 * st.prod_stage, st.prod_phase ^ 1u);
        if (!ok) break;
        const uint32_t full = full0 + 8 * st.prod_stage;
        mbar_arrive_expect_tx(full, bytes);
        const uint32_t sa = tiles0 + st.prod_stage * kTcStageBytes;
        const uint32_t sb = sa + kTcStageA;
        const int kk = k0 + kb * kTcBK;
        if (!a_mn) {
          tma_load_2d(sa, amap, kk, m0, full);
        } else {
          tma_load_2d(sa, amap, m0, kk, full);
          tma_load_2d(sa + 8192, amap, m0 + 64, kk, full);
        }
        if (!b_mn) {
          tma_load_2d(sb, bmap, kk, n0, full);
        } else {
          for (int j = 0; j < bn64; ++j) tma_load_2d(sb + 8192 * j, bmap, n0 + 64 * j, kk, full);
        }
        if (++st.prod_stage == kTcStages) { st.prod_stage = 0; st.prod_phase ^= 1u; }
      }
      if (!ok) break;
    }
  }
  return st;
}

// MMA issuer role (warp 1 lane 0): one tcgen05.mma chain per tile.
static __device__ __forceinline__ TcState mma_role(const KParams* const kpp, GemmShared& gs,
                                                 uint8_t* const smem_tiles, const uint32_t tmem_base, TcState st,
                                                 const int64_t t_first) {
  const KParams kp = *kpp;  // a value copy: fields stay in registers across asm memory clobbers
  const int lane = threadIdx.x & 31;
  (void)lane;
  const uint32_t q_full0 = smem_u32(&gs.q_full[0]), q_empty0 = smem_u32(&gs.q_empty[0]);
  const uint32_t done0 = smem_u32(&gs.tile_done[0]);
  const uint32_t acc_full0 = smem_u32(&gs.acc_full[0]), acc_empty0 = smem_u32(&gs.acc_empty[0]);
  const uint32_t full0 = smem_u32(&gs.stage_full[0]), empty0 = smem_u32(&gs.stage_empty[0]);
  const uint32_t tiles0 = smem_u32(smem_tiles);
  const uint8_t* maps = reinterpret_cast<const uint8_t*>(kp.tmaps);  // 128-byte CUtensorMaps
  (void)q_full0; (void)q_empty0; (void)done0; (void)acc_full0; (void)acc_empty0; (void)full0; (void)empty0;
  (void)tiles0; (void)maps; (void)tmem_base; (void)t_first;
  if (lane == 0) {
    // ---- MMA issuer ----
    for (uint32_t i = 0;; ++i) {
      const uint32_t seq = st.q_seq, slot = q_slot(seq);
      role_note(kp, 2, RW_MMA_QFULL, i, -1);
      if (!mbar_wait(kp, q_full0 + 8 * slot, q_parity(seq))) break;
      const int64_t t = q_read(&gs.q_task[slot]);
      ++st.q_seq;
      if (t < 0) {
        mbar_arrive(q_empty0 + 8 * slot);
        break;
      }
      const GemmArgs& g = gs.q_args[slot];
      int tm, tn, split;
      gemm_coords(g, gs.q_idx[slot], tm, tn, split);
      const int kchunk = (g.K + g.ksplit - 1) / g.ksplit;
      const int k0 = split * kchunk;
      const int nkb = (min(g.K, k0 + kchunk) - k0 + kTcBK - 1) / kTcBK;
      const uint32_t idesc = idesc_bf16(kTcBM, g.BN, g.a_mn, g.b_mn);
      const int a_mn = g.a_mn, b_mn = g.b_mn;
      mbar_arrive(q_empty0 + 8 * slot);
      role_note(kp, 2, RW_MMA_ACC, i, t);
      const uint32_t acc = st.acc_seq, buf = acc & 1;
      if (acc >= 2 && !mbar_wait(kp, acc_empty0 + 8 * buf, ((acc >> 1) - 1) & 1)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * 256;
      bool ok = true;
      role_note(kp, 2, RW_MMA_STAGE, i, t);
      for (int kb = 0; kb < nkb; ++kb) {
        ok = mbar_wait(kp, full0 + 8 * st.mma_stage, st.mma_phase);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sa = tiles0 + st.mma_stage * kTcStageBytes;
        const uint32_t sb = sa + kTcStageA;
#pragma unroll
        for (int k = 0; k < kTcBK / 16; ++k) {
          const uint64_t ad = a_mn ? smem_desc_sw128(sa + k * 2048, 8192, 1024)
                                   : smem_desc_sw128(sa + k * 32, 16, 1024);
          const uint64_t bd = b_mn ? smem_desc_sw128(sb + k * 2048, 8192, 1024)
                                   : smem_desc_sw128(sb + k * 32, 16, 1024);
          tc_mma(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit(empty0 + 8 * st.mma_stage);  // frees the stage once these MMAs have read it
        if (++st.mma_stage == kTcStages) { st.mma_stage = 0; st.mma_phase ^= 1u; }
      }
      if (!ok) break;
      tc_commit(acc_full0 + 8 * buf);  // accumulator complete
      ++st.acc_seq;
    }
  }
  return st;
}

// Releaser role (warp 3 lane 0): publishes each finished tile and frees its slot.
static __device__ __noinline__ TcState releaser_role(const KParams* const kpp, GemmShared& gs,
                                                 uint8_t* const smem_tiles, const uint32_t tmem_base, TcState st,
                                                 const int64_t t_first) {
  const KParams kp = *kpp;  // a value copy: fields stay in registers across asm memory clobbers
  const int lane = threadIdx.x & 31;
  (void)lane;
  const uint32_t q_full0 = smem_u32(&gs.q_full[0]), q_empty0 = smem_u32(&gs.q_empty[0]);
  const uint32_t done0 = smem_u32(&gs.tile_done[0]);
  const uint32_t acc_full0 = smem_u32(&gs.acc_full[0]), acc_empty0 = smem_u32(&gs.acc_empty[0]);
  const uint32_t full0 = smem_u32(&gs.stage_full[0]), empty0 = smem_u32(&gs.stage_empty[0]);
  const uint32_t tiles0 = smem_u32(smem_tiles);
  const uint8_t* maps = reinterpret_cast<const uint8_t*>(kp.tmaps);  // 128-byte CUtensorMaps
  (void)q_full0; (void)q_empty0; (void)done0; (void)acc_full0; (void)acc_empty0; (void)full0; (void)empty0;
  (void)tiles0; (void)maps; (void)tmem_base; (void)t_first;
  if (lane == 0) {
    // ---- releaser: publishes finished tiles in order and frees their slots ----
    for (uint32_t i = 0;; ++i) {
      const uint32_t seq = st.q_seq, slot = q_slot(seq);
      if (!mbar_wait(kp, q_full0 + 8 * slot, q_parity(seq))) break;
      const int64_t t = q_read(&gs.q_task[slot]);
      ++st.q_seq;
      if (t < 0) {  // the epilogue warps' arrivals for this entry complete before the run ends
        mbar_arrive(q_empty0 + 8 * slot);
        break;
      }
      if (!mbar_wait(kp, done0 + 8 * slot, q_parity(seq))) break;
      if (t != kp.skip_release) {
        // the four warps' stores precede their arrivals, which this thread has
        // acquired; the release add makes them visible at gpu scope (and the
        // proxy fence to the consumers' TMA loads)
        fence_proxy_async_global();
        red_release_add_u64(kp.counters + gs.q_sig[slot], 1ull);
        if (gs.q_sig2[slot] >= 0) red_release_add_u64(kp.counters + gs.q_sig2[slot], 1ull);
      }
      if (kp.trace) kp.trace[4 * t + 2] = globaltimer_ns();
      mbar_arrive(q_empty0 + 8 * slot);
    }
  }
  return st;
}

// Runs GEMM tasks starting with t_first (claimed, dependencies satisfied) and
// returns the next claimed ticket (not a GEMM, or >= ntasks).  Every role runs
// out of line, so each role loop is register-allocated on its own and not
// together with the rest of the persistent kernel.
template <bool kExt>
__device__ inline int64_t gemm_run(const KParams& kp, int64_t t_first, GemmShared& gs, uint8_t* smem_tiles,
                                   uint32_t tmem_base, TcState& st, bool gelu_tanh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (kp.trace && threadIdx.x == 0) {  // spare role word: runs so far on this block and this run's first task
    unsigned long long* w = kp.trace + 4 * kp.ntasks + 8 * blockIdx.x + 7;
    *w = ((((*w >> 32) & 0xffffffull) + 1) << 32) | (uint32_t)t_first;
  }
  if (warp == 2) {
    st = scheduler_role(&kp, gs, smem_tiles, tmem_base, st, t_first);
  } else if (warp == 0) {
    st = producer_role(&kp, gs, smem_tiles, tmem_base, st, t_first);
  } else if (warp == 1) {
    st = mma_role(&kp, gs, smem_tiles, tmem_base, st, t_first);
  } else if (warp >= 4) {
    const uint2 seqs = epilogue_role<kExt>(&kp, gs, tmem_base, smem_tiles, st.q_seq, st.acc_seq, gelu_tanh);
    st.q_seq = seqs.x;
    st.acc_seq = seqs.y;
  } else {
    st = releaser_role(&kp, gs, smem_tiles, tmem_base, st, t_first);
  }
  if (lane == 0 && warp != 3 && ld_volatile_u32(&kp.err[0]) == 0u)  // a failed role keeps its last wait
    role_note(kp, warp < 3 ? (warp == 2 ? 0 : warp + 1) : 3 + (warp & 3), RW_DONE, 0, -1);
  __syncwarp();
  cta_sync();
  return gs.next;
}

}  // namespace pgs
