// attn_tc.cuh — causal flash attention on tensor cores (bf16 operands, fp32
// accumulation), forward and backward, as tasks of the persistent kernel.
//
// Head dimension 64, sequence length a multiple of 128.  Tiles move global ->
// shared with cp.async into 128-byte rows whose 16-byte chunks are XOR-swizzled
// by (row mod 8), so ldmatrix reads are bank-conflict free.  Products use
// mma.sync m16n8k16 (bf16 x bf16 -> fp32); the softmax runs on the accumulator
// fragments in registers with the running-max ("online") rescaling, in base 2.
//
//   forward, task (b, h, 128 queries):  S = q k^T * scale, causal mask,
//       running max m and sum l per row, O = sum_j exp(S - m) v / l,
//       LSE = m + ln l (natural log) saved for the backward pass.
//   backward pre-pass, task (64 rows):  D_i = sum_c dO_ic O_ic per head.
//   backward dK/dV, task (b, h, 128 keys): for every query block at or after
//       the keys: P^T = exp(S^T - LSE), dV += P^T dO, dP^T = V dO^T,
//       dS^T = P^T (dP^T - D) * scale, dK += dS^T Q.
//   backward dQ, task (b, h, 128 queries): for every key block up to the
//       diagonal: P, dP = dO V^T, dS = P (dP - D) * scale, dQ += dS K.
// dQ and dK/dV are separate tasks (recomputing P) so every output has exactly
// one writer and the step stays deterministic (no atomics).
#pragma once
#include "device.cuh"
#include "tasks_rows.cuh"
#include "tc_gemm.cuh"

namespace pgs {

constexpr int kAttQ = 128;   // query rows per forward / dQ task (8 warps x 16)
constexpr int kAttK = 128;   // key rows per dK/dV task (8 warps x 16)
constexpr int kAttSub = 64;  // rows of the streamed blocks

__device__ __forceinline__ void cp_async16(uint32_t smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// d += a (16x16, row) * b (16x8, col)
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// byte offset of 16-byte chunk `ch` (0..7) of row r in a swizzled [rows][64] bf16 tile
__device__ __forceinline__ uint32_t swz(int r, int ch) { return (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4)); }

// rows x 64 bf16 tile from global (row pitch ld elements) into a swizzled smem tile
__device__ __forceinline__ void tile_load_async(uint32_t s, const __nv_bfloat16* g, int64_t ld, int rows) {
  for (int e = threadIdx.x; e < rows * 8; e += kThreads) {
    const int r = e >> 3, ch = e & 7;
    cp_async16(s + swz(r, ch), g + (int64_t)r * ld + ch * 8);
  }
}

// A fragments (16 rows from r0, 64 columns = 4 k-steps) of a swizzled tile
__device__ __forceinline__ void load_a_frags(uint32_t s, int r0, uint32_t (*f)[4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) ldsm_x4(s + swz(r0 + (lane & 15), kk * 2 + (lane >> 4)), f[kk]);
}

// acc[8][4] (16 x 64) += A (16 x 64, k = 64 columns of the A fragments) * B^T
// with B stored [n][k] (64 n-rows x 64 k) in a swizzled tile.
__device__ __forceinline__ void mma_abt(float (*acc)[4], const uint32_t (*af)[4], uint32_t sb) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      uint32_t b[4];
      ldsm_x4(sb + swz(np * 16 + (lane & 7) + ((lane >> 4) << 3), kk * 2 + ((lane >> 3) & 1)), b);
      mma16816(acc[2 * np], af[kk], b[0], b[1]);
      mma16816(acc[2 * np + 1], af[kk], b[2], b[3]);
    }
}

// Packs a 16 x 64 fp32 accumulator tile into bf16 A fragments (4 k-steps of 16).
__device__ __forceinline__ void pack_a(const float (*p)[4], uint32_t (*pa)[4]) {
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    pa[t][0] = pack_bf16x2(p[2 * t][0], p[2 * t][1]);
    pa[t][1] = pack_bf16x2(p[2 * t][2], p[2 * t][3]);
    pa[t][2] = pack_bf16x2(p[2 * t + 1][0], p[2 * t + 1][1]);
    pa[t][3] = pack_bf16x2(p[2 * t + 1][2], p[2 * t + 1][3]);
  }
}

// acc[8][4] (16 x 64) += A (16 x 64, packed bf16 fragments, k = 64) * B
// with B stored [k][n] (64 k-rows x 64 n) in a swizzled tile.
__device__ __forceinline__ void mma_pb(float (*acc)[4], const uint32_t (*pa)[4], uint32_t sb) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      uint32_t b[4];
      ldsm_x4_t(sb + swz(t * 16 + (lane & 7) + (((lane >> 3) & 1) << 3), np * 2 + (lane >> 4)), b);
      mma16816(acc[2 * np], pa[t], b[0], b[1]);
      mma16816(acc[2 * np + 1], pa[t], b[2], b[3]);
    }
  }
}

// Packs the pair (x0, x1) of head dimensions (c, c+1) at position t into bf16,
// rotated back by the rotary angle (the gradient of a rotated q or k w.r.t. the
// projection before the rotation) when kRope.
template <bool kRope>
__device__ __forceinline__ uint32_t pack_unrotate(const float2* rope, int t, int c, float x0, float x1) {
  if constexpr (kRope) {
    const float2 cs = rope[t * 32 + (c >> 1)];
    const float y0 = x0 * cs.x + x1 * cs.y, y1 = x1 * cs.x - x0 * cs.y;
    x0 = y0;
    x1 = y1;
  }
  return pack_bf16x2(x0, x1);
}

__device__ __forceinline__ void zero_acc(float (*acc)[4]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
}

// ---- forward ----------------------------------------------------------------
__device__ inline void task_attn_fwd_tc(const AttnArgs& a, int idx, uint8_t* smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = a.T / kAttQ;
  const int qb = nqb - 1 - idx % nqb;  // longest blocks are claimed first
  const int h = (idx / nqb) % a.H, b = idx / (nqb * a.H);
  const int q0 = qb * kAttQ;
  const int64_t ld = 3 * (int64_t)a.C;
  const __nv_bfloat16* base = reinterpret_cast<const __nv_bfloat16*>(a.qkv) + (int64_t)b * a.T * ld + h * 64;
  const uint32_t sQ = smem_u32(smem), sK = sQ + kAttQ * 128, sV = sK + 2 * kAttSub * 128;
  tile_load_async(sQ, base + (int64_t)q0 * ld, ld, kAttQ);
  tile_load_async(sK, base + a.C, ld, kAttSub);
  tile_load_async(sV, base + 2 * a.C, ld, kAttSub);
  cp_async_commit();
  const int nkv = (q0 + kAttQ) / kAttSub;
  const float sl2 = a.scale * 1.4426950408889634f;
  const int row0 = q0 + warp * 16;
  const int ra = row0 + (lane >> 2), rb = ra + 8;  // this thread's two query rows
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[8][4];
  zero_acc(o);
  uint32_t qf[4][4];
  for (int j = 0; j < nkv; ++j) {
    if (j + 1 < nkv) {
      const int nb = (j + 1) & 1;
      tile_load_async(sK + nb * kAttSub * 128, base + a.C + (int64_t)(j + 1) * kAttSub * ld, ld, kAttSub);
      tile_load_async(sV + nb * kAttSub * 128, base + 2 * a.C + (int64_t)(j + 1) * kAttSub * ld, ld, kAttSub);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (j == 0) load_a_frags(sQ, warp * 16, qf);
    const int k0 = j * kAttSub;
    if (k0 <= row0 + 15) {
      const uint32_t kb = sK + (j & 1) * kAttSub * 128, vb = sV + (j & 1) * kAttSub * 128;
      float s[8][4];
      zero_acc(s);
      mma_abt(s, qf, kb);
      float mx0 = m0, mx1 = m1;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int c = k0 + nt * 8 + 2 * (lane & 3);
        s[nt][0] = c <= ra ? s[nt][0] * sl2 : -INFINITY;
        s[nt][1] = c + 1 <= ra ? s[nt][1] * sl2 : -INFINITY;
        s[nt][2] = c <= rb ? s[nt][2] * sl2 : -INFINITY;
        s[nt][3] = c + 1 <= rb ? s[nt][3] * sl2 : -INFINITY;
        mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float al0 = exp2f(m0 - mx0), al1 = exp2f(m1 - mx1);
      m0 = mx0;
      m1 = mx1;
      l0 *= al0;
      l1 *= al1;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        o[nt][0] *= al0; o[nt][1] *= al0; o[nt][2] *= al1; o[nt][3] *= al1;
        s[nt][0] = exp2f(s[nt][0] - mx0);
        s[nt][1] = exp2f(s[nt][1] - mx0);
        s[nt][2] = exp2f(s[nt][2] - mx1);
        s[nt][3] = exp2f(s[nt][3] - mx1);
        l0 += s[nt][0] + s[nt][1];
        l1 += s[nt][2] + s[nt][3];
      }
      uint32_t pa[4][4];
      pack_a(s, pa);
      mma_pb(o, pa, vb);
    }
    __syncthreads();
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float i0 = 1.0f / l0, i1 = 1.0f / l1;
  __nv_bfloat16* O = reinterpret_cast<__nv_bfloat16*>(a.o) + (int64_t)b * a.T * a.ld_o + h * 64;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const int c = nt * 8 + 2 * (lane & 3);
    *reinterpret_cast<uint32_t*>(O + (int64_t)ra * a.ld_o + c) = pack_bf16x2(o[nt][0] * i0, o[nt][1] * i0);
    *reinterpret_cast<uint32_t*>(O + (int64_t)rb * a.ld_o + c) = pack_bf16x2(o[nt][2] * i1, o[nt][3] * i1);
  }
  if ((lane & 3) == 0) {
    float* L = a.lse + ((int64_t)b * a.H + h) * a.T;
    const float ln2 = 0.6931471805599453f;
    L[ra] = (m0 + log2f(l0)) * ln2;
    L[rb] = (m1 + log2f(l1)) * ln2;
  }
}

// ---- backward pre-pass: D = rowsum(dO * O) per (row, head) --------------------
__device__ inline void task_attn_bwd_pre(const AttnArgs& a, int idx) {
  // D[b, h, t] = sum_d dO[t, h d] O[t, h d]: 8 lanes per head (8 elements each),
  // four heads per warp-wide pass.  A warp loads two rows' dO and O (every
  // head) before reducing either, so its eight rows cost four memory latencies
  // instead of one per row and head group.  Heads beyond 16 take a second round.
  constexpr int kRG = 2, kHG = 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.B * a.T;
  const int r0 = idx * kAttSub, r1 = min(r0 + kAttSub, N);
  const int sub = lane & 7;
  const __nv_bfloat16* dO = reinterpret_cast<const __nv_bfloat16*>(a.dout);
  const __nv_bfloat16* O = reinterpret_cast<const __nv_bfloat16*>(a.o);
  for (int rb = r0 + warp; rb < r1; rb += kRG * kWarps) {
    for (int hb = 0; hb < a.H; hb += 4 * kHG) {
      uint4 u[kRG][kHG], v[kRG][kHG];
#pragma unroll
      for (int i = 0; i < kRG; ++i) {
        const int r = rb + i * kWarps;
#pragma unroll
        for (int j = 0; j < kHG; ++j) {
          const int h = hb + 4 * j + (lane >> 3);
          if (r < r1 && h < a.H) {
            u[i][j] = *reinterpret_cast<const uint4*>(dO + (int64_t)r * a.C + h * 64 + sub * 8);
            v[i][j] = *reinterpret_cast<const uint4*>(O + (int64_t)r * a.ld_o + h * 64 + sub * 8);
          } else {
            u[i][j] = make_uint4(0u, 0u, 0u, 0u);
            v[i][j] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kRG; ++i) {
        const int r = rb + i * kWarps;
#pragma unroll
        for (int j = 0; j < kHG; ++j) {
          const int h = hb + 4 * j + (lane >> 3);
          if (hb + 4 * j >= a.H) break;  // warp-uniform
          float fu[8], fv[8];
          bf16x8_to_f(u[i][j], fu);
          bf16x8_to_f(v[i][j], fv);
          float s = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) s += fu[e] * fv[e];
          s += __shfl_xor_sync(0xffffffffu, s, 1);
          s += __shfl_xor_sync(0xffffffffu, s, 2);
          s += __shfl_xor_sync(0xffffffffu, s, 4);
          if (sub == 0 && h < a.H && r < r1) {
            const int b = r / a.T, t = r % a.T;
            a.scratch[((int64_t)b * a.H + h) * a.T + t] = s;
          }
        }
      }
    }
  }
}

// ---- backward dK/dV -------------------------------------------------------------
template <bool kRope>
__device__ inline void task_attn_bwd_kv_tc(const AttnArgs& a, int idx, uint8_t* smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = a.T / kAttK;
  const int kb = idx % nkb;  // earliest keys see the most queries: claimed first
  const int h = (idx / nkb) % a.H, b = idx / (nkb * a.H);
  const int k0 = kb * kAttK;
  const int64_t ld = 3 * (int64_t)a.C;
  const __nv_bfloat16* base = reinterpret_cast<const __nv_bfloat16*>(a.qkv) + (int64_t)b * a.T * ld + h * 64;
  const __nv_bfloat16* dOb = reinterpret_cast<const __nv_bfloat16*>(a.dout) + (int64_t)b * a.T * a.C + h * 64;
  const float* L = a.lse + ((int64_t)b * a.H + h) * a.T;
  const float* Dv = a.scratch + ((int64_t)b * a.H + h) * a.T;
  const uint32_t sK = smem_u32(smem), sV = sK + kAttK * 128, sQ = sV + kAttK * 128,
                 sO = sQ + 2 * kAttSub * 128;
  float* sL = reinterpret_cast<float*>(smem + (sO - sK) + 2 * kAttSub * 128);  // [2][64] LSE, [2][64] D
  tile_load_async(sK, base + a.C + (int64_t)k0 * ld, ld, kAttK);
  tile_load_async(sV, base + 2 * a.C + (int64_t)k0 * ld, ld, kAttK);
  const int i_first = k0 / kAttSub, nq = a.T / kAttSub;
  auto load_q = [&](int i, int buf) {
    tile_load_async(sQ + buf * kAttSub * 128, base + (int64_t)i * kAttSub * ld, ld, kAttSub);
    tile_load_async(sO + buf * kAttSub * 128, dOb + (int64_t)i * kAttSub * a.C, a.C, kAttSub);
    for (int e = threadIdx.x; e < 2 * kAttSub; e += kThreads) {
      const int which = e / kAttSub, r = e % kAttSub;
      sL[(which * 2 + buf) * kAttSub + r] = which == 0 ? L[i * kAttSub + r] : Dv[i * kAttSub + r];
    }
  };
  load_q(i_first, 0);
  cp_async_commit();
  const float sl2 = a.scale * 1.4426950408889634f;
  const float log2e = 1.4426950408889634f;
  const int key0 = k0 + warp * 16;
  const int ka = key0 + (lane >> 2), kbr = ka + 8;  // this thread's two key rows
  float dk[8][4], dv[8][4];
  zero_acc(dk);
  zero_acc(dv);
  for (int i = i_first; i < nq; ++i) {
    const int buf = (i - i_first) & 1;
    if (i + 1 < nq) {
      load_q(i + 1, buf ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const int qi0 = i * kAttSub;
    if (qi0 + kAttSub - 1 >= key0) {
      const uint32_t qb_s = sQ + buf * kAttSub * 128, ob_s = sO + buf * kAttSub * 128;
      const float* lseb = sL + (0 * 2 + buf) * kAttSub;
      const float* Db = sL + (1 * 2 + buf) * kAttSub;
      float p[8][4], dp[8][4];
      uint32_t af[4][4];           // A fragments reloaded from shared memory (register budget)
      load_a_frags(sK, warp * 16, af);
      zero_acc(p);
      mma_abt(p, af, qb_s);        // S^T = K Q^T
      load_a_frags(sV, warp * 16, af);
      zero_acc(dp);
      mma_abt(dp, af, ob_s);       // dP^T = V dO^T
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int cq = nt * 8 + 2 * (lane & 3);  // query column within the block
        const float l0 = lseb[cq] * log2e, l1 = lseb[cq + 1] * log2e;
        const float d0 = Db[cq], d1 = Db[cq + 1];
        const int q = qi0 + cq;
        p[nt][0] = q >= ka ? exp2f(p[nt][0] * sl2 - l0) : 0.f;
        p[nt][1] = q + 1 >= ka ? exp2f(p[nt][1] * sl2 - l1) : 0.f;
        p[nt][2] = q >= kbr ? exp2f(p[nt][2] * sl2 - l0) : 0.f;
        p[nt][3] = q + 1 >= kbr ? exp2f(p[nt][3] * sl2 - l1) : 0.f;
        dp[nt][0] = p[nt][0] * (dp[nt][0] - d0) * a.scale;
        dp[nt][1] = p[nt][1] * (dp[nt][1] - d1) * a.scale;
        dp[nt][2] = p[nt][2] * (dp[nt][2] - d0) * a.scale;
        dp[nt][3] = p[nt][3] * (dp[nt][3] - d1) * a.scale;
      }
      uint32_t pa[4][4], pd[4][4];  // P^T and dS^T as bf16 fragments (the fp32 tiles die here)
      pack_a(p, pa);
      pack_a(dp, pd);
      mma_pb(dv, pa, ob_s);  // dV += P^T dO
      mma_pb(dk, pd, qb_s);  // dK += dS^T Q
    }
    __syncthreads();
  }
  __nv_bfloat16* dq = reinterpret_cast<__nv_bfloat16*>(a.dqkv) + (int64_t)b * a.T * ld + h * 64;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const int c = nt * 8 + 2 * (lane & 3);
    *reinterpret_cast<uint32_t*>(dq + (int64_t)ka * ld + a.C + c) = pack_unrotate<kRope>(a.rope, ka, c, dk[nt][0], dk[nt][1]);
    *reinterpret_cast<uint32_t*>(dq + (int64_t)kbr * ld + a.C + c) = pack_unrotate<kRope>(a.rope, kbr, c, dk[nt][2], dk[nt][3]);
    *reinterpret_cast<uint32_t*>(dq + (int64_t)ka * ld + 2 * a.C + c) = pack_bf16x2(dv[nt][0], dv[nt][1]);
    *reinterpret_cast<uint32_t*>(dq + (int64_t)kbr * ld + 2 * a.C + c) = pack_bf16x2(dv[nt][2], dv[nt][3]);
  }
}

// ---- backward dQ ------------------------------------------------------------------
template <bool kRope>
__device__ inline void task_attn_bwd_q_tc(const AttnArgs& a, int idx, uint8_t* smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = a.T / kAttQ;
  const int qb = nqb - 1 - idx % nqb;
  const int h = (idx / nqb) % a.H, b = idx / (nqb * a.H);
  const int q0 = qb * kAttQ;
  const int64_t ld = 3 * (int64_t)a.C;
  const __nv_bfloat16* base = reinterpret_cast<const __nv_bfloat16*>(a.qkv) + (int64_t)b * a.T * ld + h * 64;
  const __nv_bfloat16* dOb = reinterpret_cast<const __nv_bfloat16*>(a.dout) + (int64_t)b * a.T * a.C + h * 64;
  const uint32_t sQ = smem_u32(smem), sO = sQ + kAttQ * 128, sK = sO + kAttQ * 128,
                 sV = sK + 2 * kAttSub * 128;
  tile_load_async(sQ, base + (int64_t)q0 * ld, ld, kAttQ);
  tile_load_async(sO, dOb + (int64_t)q0 * a.C, a.C, kAttQ);
  tile_load_async(sK, base + a.C, ld, kAttSub);
  tile_load_async(sV, base + 2 * a.C, ld, kAttSub);
  cp_async_commit();
  const int nkv = (q0 + kAttQ) / kAttSub;
  const float sl2 = a.scale * 1.4426950408889634f;
  const float log2e = 1.4426950408889634f;
  const int row0 = q0 + warp * 16;
  const int ra = row0 + (lane >> 2), rb = ra + 8;
  const float* L = a.lse + ((int64_t)b * a.H + h) * a.T;
  const float* Dv = a.scratch + ((int64_t)b * a.H + h) * a.T;
  const float la = L[ra] * log2e, lb = L[rb] * log2e, da = Dv[ra], db = Dv[rb];
  float dq[8][4];
  zero_acc(dq);
  uint32_t qf[4][4], of[4][4];
  for (int j = 0; j < nkv; ++j) {
    if (j + 1 < nkv) {
      const int nb = (j + 1) & 1;
      tile_load_async(sK + nb * kAttSub * 128, base + a.C + (int64_t)(j + 1) * kAttSub * ld, ld, kAttSub);
      tile_load_async(sV + nb * kAttSub * 128, base + 2 * a.C + (int64_t)(j + 1) * kAttSub * ld, ld, kAttSub);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (j == 0) {
      load_a_frags(sQ, warp * 16, qf);
      load_a_frags(sO, warp * 16, of);
    }
    const int k0 = j * kAttSub;
    if (k0 <= row0 + 15) {
      const uint32_t kb = sK + (j & 1) * kAttSub * 128, vb = sV + (j & 1) * kAttSub * 128;
      float p[8][4], dp[8][4];
      zero_acc(p);
      mma_abt(p, qf, kb);   // S = Q K^T
      zero_acc(dp);
      mma_abt(dp, of, vb);  // dP = dO V^T
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int c = k0 + nt * 8 + 2 * (lane & 3);
        p[nt][0] = c <= ra ? exp2f(p[nt][0] * sl2 - la) : 0.f;
        p[nt][1] = c + 1 <= ra ? exp2f(p[nt][1] * sl2 - la) : 0.f;
        p[nt][2] = c <= rb ? exp2f(p[nt][2] * sl2 - lb) : 0.f;
        p[nt][3] = c + 1 <= rb ? exp2f(p[nt][3] * sl2 - lb) : 0.f;
        p[nt][0] *= (dp[nt][0] - da) * a.scale;
        p[nt][1] *= (dp[nt][1] - da) * a.scale;
        p[nt][2] *= (dp[nt][2] - db) * a.scale;
        p[nt][3] *= (dp[nt][3] - db) * a.scale;
      }
      uint32_t pa[4][4];
      pack_a(p, pa);
      mma_pb(dq, pa, kb);  // dQ += dS K
    }
    __syncthreads();
  }
  __nv_bfloat16* dqp = reinterpret_cast<__nv_bfloat16*>(a.dqkv) + (int64_t)b * a.T * ld + h * 64;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const int c = nt * 8 + 2 * (lane & 3);
    *reinterpret_cast<uint32_t*>(dqp + (int64_t)ra * ld + c) = pack_unrotate<kRope>(a.rope, ra, c, dq[nt][0], dq[nt][1]);
    *reinterpret_cast<uint32_t*>(dqp + (int64_t)rb * ld + c) = pack_unrotate<kRope>(a.rope, rb, c, dq[nt][2], dq[nt][3]);
  }
}

}  // namespace pgs
