// attn_tc.cuh — causal flash attention on the 5th-generation tensor cores
// (tcgen05, sm_103a), forward and backward, as tasks of the persistent kernel.
//
// Head dimension 64, sequence length a multiple of 128.  Every operand tile is a
// 128-row x 64-column bf16 block (one head of 128 tokens) that TMA copies from
// the [tokens, 3C] qkv buffer (or the [tokens, C] output gradient) into shared
// memory with the 128-byte swizzle; the products run as tcgen05.mma (kind::f16,
// M = 128) issued by one thread, with fp32 accumulators in tensor memory
// (TMEM), and the softmax reads them back with tcgen05.ld: each of the 8 warps
// owns 32 rows (its TMEM lane quarter) and one half of the columns, one row per
// thread.  Probabilities and score gradients go back to shared memory as bf16
// in the K-major swizzled layout the next product reads.
//
//   forward, task (b, h, 128 queries), key blocks j = 0 .. diagonal:
//       S_j = Q K_j^T (TMEM, two buffers: S_{j+1} is computed while S_j is
//       reduced), running row max m and sum l in registers (base 2), P_j =
//       exp2(S_j * scale * log2 e - m) (the SFU's approximate 2^x) to shared
//       memory, O_j = P_j V_j into one of two TMEM buffers; the thread adds O_j
//       to its 32 output columns, rescaled by exp2(m_old - m_new), while the
//       next block's probabilities are formed.
//       O = sum / l, LSE = ln 2 (m + log2 l) saved for the backward pass.
//   backward pre-pass, task (64 rows):  D_i = sum_c dO_ic O_ic per head.
//   backward dK/dV, task (b, h, 128 keys), query blocks i at or after the keys:
//       S^T = K Q_i^T and dP^T = V dO_i^T (TMEM), P^T = exp2(S^T scale log2 e -
//       LSE log2 e), dS^T = P^T (dP^T - D) scale, then dV += P^T dO_i and
//       dK += dS^T Q_i accumulate in TMEM across the query blocks.
//   backward dQ, task (b, h, 128 queries), key blocks up to the diagonal:
//       S = Q K_j^T, dP = dO V_j^T, dS = P (dP - D) scale, dQ += dS K_j in TMEM.
// dQ and dK/dV are separate tasks (recomputing P) so every output has exactly
// one writer and the step stays deterministic (no atomics).
//
// Algorithm: the online-softmax attention of Dao et al. ("FlashAttention",
// 2022) in the forward and its recomputation-based backward; the method's
// pages name the families (attention-forward, attention-key, attention-query:
// "Coppelius training on the RTX 3090", section "Where a step's time goes").
#pragma once
#include "device.cuh"
#include "tasks_rows.cuh"
#include "tc_gemm.cuh"

namespace pgs {

constexpr int kAttBlk = 128;                 // rows of every attention tile (queries or keys)
constexpr uint32_t kAttTile = kAttBlk * 128;  // bytes of a 128 x 64 bf16 tile
constexpr int kAttPreRows = 64;               // token rows of a backward pre-pass task

// mbarriers of the attention tasks (initialised once per launch, phases counted
// in use[]): Q (or K/V of a dK/dV task) loaded; the streamed pair of tiles of
// stage 0..3 loaded; scores of buffer 0/1 complete; products of buffer 0/1 complete.
//
// The streamed pairs (K_j, V_j, or Q_i, dO_i) go through a ring of kAttStages
// stages (three in the dK/dV task, whose two resident tiles leave less room):
// at 512 tokens every block of a task is requested when the task starts, and a
// stage is refilled as soon as the product that last read it is known complete,
// which the threads wait for anyway, so no thread ever blocks on a refill.
constexpr int kAttStages = 4, kAttStagesKV = 3;
enum AttBar : int { AB_FIXED = 0, AB_LD0 = 1, AB_S0 = AB_LD0 + kAttStages, AB_O0 = AB_S0 + 2, AB_NUM = AB_O0 + 2 };

struct AttnShared {
  uint64_t bar[AB_NUM];
  uint32_t use[AB_NUM];          // phases of each barrier completed so far in this launch
};

// Small per-task arrays in the dynamic shared memory, above every task's tiles
// (at most 13 tiles = 208 KB): values exchanged between the two column halves
// of a row, and the dK/dV task's LSE (base 2) and D of a query block, two buffers.
constexpr uint32_t kAttScratchOff = 13 * kAttTile;
struct AttnScratch {
  float red[2][kAttBlk];
  float ld[2][2][kAttBlk];
};
static_assert(kAttScratchOff + sizeof(AttnScratch) <= (uint32_t)(kTcSmemBytes + 4 * kEpiStageBytes),
              "attention scratch beyond the dynamic shared memory");

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
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

// 32 lanes x 32 consecutive fp32 columns of TMEM (thread i: lane base + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Row `row` of a 128-row K-major bf16 operand tile in the 128-byte swizzled
// layout: 32 values (columns 32 q .. 32 q + 31 of the 64 the tile holds) as four
// 16-byte chunks; chunk c of a row lives at (c ^ (row mod 8)) * 16.
__device__ __forceinline__ void st_row32_sw128(uint32_t tile, int row, int q, const float* v) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int ch = 4 * q + c;
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(tile + row * 128 + ((ch ^ (row & 7)) << 4)),
                 "r"(pack_bf16x2(v[8 * c], v[8 * c + 1])), "r"(pack_bf16x2(v[8 * c + 2], v[8 * c + 3])),
                 "r"(pack_bf16x2(v[8 * c + 4], v[8 * c + 5])), "r"(pack_bf16x2(v[8 * c + 6], v[8 * c + 7]))
                 : "memory");
  }
}

// Descriptors of the operand tiles: K-major (rows = M or N, 64 K-values in a
// 128-byte row; k-step kk of 16 advances 32 bytes inside the row, a second
// 64-wide K atom lies kAttTile further) and MN-major (rows = K, 64 N-values in a
// 128-byte row; k-step kk advances 16 rows = 2048 bytes).
__device__ __forceinline__ uint64_t att_desc_k(uint32_t tile, int kk) {
  return smem_desc_sw128(tile + (uint32_t)(kk >> 2) * kAttTile + (uint32_t)(kk & 3) * 32u, 16, 1024);
}
__device__ __forceinline__ uint64_t att_desc_mn(uint32_t tile, int kk) {
  return smem_desc_sw128(tile + (uint32_t)kk * 2048u, 8192, 1024);
}
// d (+)= A B^T over K = 16 nk: A K-major [128, K], B K-major [N, K]
__device__ __forceinline__ void att_mma_kk(uint32_t d, uint32_t a, uint32_t b, int nk, uint32_t idesc, bool acc) {
#pragma unroll 1
  for (int kk = 0; kk < nk; ++kk) tc_mma(d, att_desc_k(a, kk), att_desc_k(b, kk), idesc, (acc || kk > 0) ? 1u : 0u);
}
// d (+)= A B over K = 16 nk: A K-major [128, K], B MN-major [K, N]
__device__ __forceinline__ void att_mma_kmn(uint32_t d, uint32_t a, uint32_t b, int nk, uint32_t idesc, bool acc) {
#pragma unroll 1
  for (int kk = 0; kk < nk; ++kk) tc_mma(d, att_desc_k(a, kk), att_desc_mn(b, kk), idesc, (acc || kk > 0) ? 1u : 0u);
}

// Phase bookkeeping: use u (from 0, counted over the launch) of barrier b has parity u & 1.
struct AttPhases {
  uint32_t use[AB_NUM];
  __device__ __forceinline__ void load(const AttnShared& as) {
#pragma unroll
    for (int i = 0; i < AB_NUM; ++i) use[i] = *reinterpret_cast<const volatile uint32_t*>(&as.use[i]);
  }
  // parity of the k-th use of barrier b in this task
  __device__ __forceinline__ uint32_t par(int b, int k) const { return (use[b] + (uint32_t)k) & 1u; }
};

// Number of j in [0, n) with j mod m == b (0 <= b < m, n >= 0).
__device__ __forceinline__ uint32_t n_mod(int n, int b, int m) { return (uint32_t)((n - b + m - 1) / m); }

// Bounded wait of every calling thread; a failure is recorded in the error words
// and later waits return at once, so every thread keeps the same control flow.
__device__ __forceinline__ void att_wait(const KParams& kp, uint32_t bar, uint32_t parity) {
  (void)mbar_wait(kp, bar, parity);
}

// Pair barrier of the two warps that share a TMEM lane quarter (column halves).
__device__ __forceinline__ void pair_sync(int quarter) {
  asm volatile("bar.sync %0, 64;" ::"r"(1 + quarter) : "memory");
}

// ---- forward ----------------------------------------------------------------
__device__ inline void task_attn_fwd_tc(const KParams& kp, const AttnArgs& a, int idx, uint8_t* smem,
                                        AttnShared& as, uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int nqb = a.T / kAttBlk;
  const int qb = nqb - 1 - idx % nqb;  // longest blocks are claimed first
  const int h = (idx / nqb) % a.H, b = idx / (nqb * a.H);
  const int q0 = qb * kAttBlk, nkb = qb + 1, row0 = b * a.T;
  const void* map = reinterpret_cast<const uint8_t*>(kp.tmaps) + 128 * a.qkv_map;
  // tiles: Q | K stages 0..3 | V stages 0..3 | P buffers 0, 1 (two tiles each)
  const uint32_t sQ = smem_u32(smem), sK = sQ + kAttTile, sV = sK + kAttStages * kAttTile,
                 sP = sV + kAttStages * kAttTile;
  const uint32_t bar0 = smem_u32(&as.bar[0]);
  AttnScratch& sc = *reinterpret_cast<AttnScratch*>(smem + kAttScratchOff);
  AttPhases ph;
  ph.load(as);
  // One thread of three different warps each: the copies, the score products, the
  // value products.  Issuing a product takes its thread about as long as the tensor
  // pipe needs for the products queued before it, so the issue work is spread over
  // warps that otherwise do the same share of the softmax.
  const bool leader = threadIdx.x == 0, s_issuer = threadIdx.x == 32, o_issuer = threadIdx.x == 64;
  const int r = quarter * 32 + lane;                        // this thread's query row (TMEM lane)
  const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
  const uint32_t id_s = idesc_bf16(128, 128, 0, 0), id_o = idesc_bf16(128, 64, 0, 1);
  auto load_kv = [&](int j) {  // leader: K_j and V_j into stage j mod kAttStages
    const int st = j % kAttStages;
    const uint32_t bar = bar0 + 8 * (AB_LD0 + st);
    mbar_arrive_expect_tx(bar, 2 * kAttTile);
    tma_load_2d(sK + st * kAttTile, map, a.C + h * 64, row0 + j * kAttBlk, bar);
    tma_load_2d(sV + st * kAttTile, map, 2 * a.C + h * 64, row0 + j * kAttBlk, bar);
  };
  auto issue_s = [&](int j) {  // s_issuer: S_j = Q K_j^T into TMEM columns 128 (j & 1)
    const int buf = j & 1, st = j % kAttStages;
    att_wait(kp, bar0 + 8 * (AB_LD0 + st), ph.par(AB_LD0 + st, j / kAttStages));
    tc_fence_after();
    att_mma_kk(tmem + 128u * buf, sQ, sK + st * kAttTile, 4, id_s, false);
    tc_commit(bar0 + 8 * (AB_S0 + buf));
  };
  if (leader) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // earlier generic writes of this memory
    mbar_arrive_expect_tx(bar0 + 8 * AB_FIXED, kAttTile);
    tma_load_2d(sQ, map, h * 64, row0 + q0, bar0 + 8 * AB_FIXED);
    for (int j = 0; j < min(kAttStages, nkb); ++j) load_kv(j);
  }
  if (s_issuer) {
    att_wait(kp, bar0 + 8 * AB_FIXED, ph.par(AB_FIXED, 0));
    issue_s(0);
  }
  __syncwarp();
  const float sl2 = a.scale * 1.4426950408889634f;
  float o[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) o[i] = 0.f;
  float m_run = -INFINITY, l_run = 0.f, alpha_pend = 0.f;
  for (int j = 0; j < nkb; ++j) {
    const int buf = j & 1;
    if (s_issuer && j + 1 < nkb) issue_s(j + 1);  // its buffer was last read before the previous block barrier
    __syncwarp();
    att_wait(kp, bar0 + 8 * (AB_S0 + buf), ph.par(AB_S0 + buf, j >> 1));
    __syncwarp();
    tc_fence_after();
    float s[64];
    tmem_ld32(trow + 128u * buf + 64u * half, s);
    tmem_ld32(trow + 128u * buf + 64u * half + 32u, s + 32);
    const bool diag = j == nkb - 1;
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < 64; i += 2) {  // the scale two columns per instruction
      const float2 v = f2_mul(make_float2(s[i], s[i + 1]), make_float2(sl2, sl2));
      s[i] = (diag && half * 64 + i > r) ? -INFINITY : v.x;
      s[i + 1] = (diag && half * 64 + i + 1 > r) ? -INFINITY : v.y;
      mx = fmaxf(mx, s[i]);
      mx = fmaxf(mx, s[i + 1]);
    }
    sc.red[half][r] = mx;
    pair_sync(quarter);
    const float m_new = fmaxf(m_run, fmaxf(sc.red[0][r], sc.red[1][r]));
    const float alpha = ex2_sfu(m_run - m_new);
    float ls = 0.f;
#pragma unroll
    for (int i = 0; i < 64; i += 2) {
      const float2 d = f2_add(make_float2(s[i], s[i + 1]), make_float2(-m_new, -m_new));
      s[i] = ex2_sfu(d.x);
      s[i + 1] = ex2_sfu(d.y);
      ls += s[i];
      ls += s[i + 1];
    }
    l_run = l_run * alpha + ls;
    m_run = m_new;
    // P_j (bf16) into buffer buf: its previous reader (the product of block j - 2) completed
    // before the partial of block j - 2 was added to o in the previous iteration
    const uint32_t pt = sP + (uint32_t)buf * 2u * kAttTile + (uint32_t)half * kAttTile;
    st_row32_sw128(pt, r, 0, s);
    st_row32_sw128(pt, r, 1, s + 32);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic smem writes -> tensor core reads
    tc_fence_before();
    __syncthreads();
    if (o_issuer) {
      tc_fence_after();
      att_mma_kmn(tmem + 256u + 64u * buf, pt - (uint32_t)half * kAttTile, sV + (j % kAttStages) * kAttTile, 8,
                  id_o, false);
      tc_commit(bar0 + 8 * (AB_O0 + buf));
    }
    __syncwarp();
    if (j >= 1) {  // add the partial of block j - 1, rescaled from its running max to this one
      const int pb = (j - 1) & 1;
      att_wait(kp, bar0 + 8 * (AB_O0 + pb), ph.par(AB_O0 + pb, (j - 1) >> 1));
      // K_{j-1} and V_{j-1} are no longer read (every earlier product is complete): refill their stage
      if (leader && j - 1 + kAttStages < nkb) load_kv(j - 1 + kAttStages);
      __syncwarp();
      tc_fence_after();
      float part[32];
      tmem_ld32(trow + 256u + 64u * pb + 32u * half, part);
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = o[i] * alpha_pend + part[i];
    }
    alpha_pend = alpha;
  }
  {
    const int pb = (nkb - 1) & 1;
    att_wait(kp, bar0 + 8 * (AB_O0 + pb), ph.par(AB_O0 + pb, (nkb - 1) >> 1));
    __syncwarp();
    tc_fence_after();
    float part[32];
    tmem_ld32(trow + 256u + 64u * pb + 32u * half, part);
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] = o[i] * alpha_pend + part[i];
  }
  sc.red[half][r] = l_run;  // every earlier read of red[] came before the last block barrier
  pair_sync(quarter);
  const float L = sc.red[0][r] + sc.red[1][r];
  const float inv = 1.0f / L;
  uint4* O = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.o) + (int64_t)(row0 + q0 + r) * a.ld_o +
                                      h * 64 + half * 32);
#pragma unroll
  for (int c = 0; c < 4; ++c)
    O[c] = make_uint4(pack_bf16x2(o[8 * c] * inv, o[8 * c + 1] * inv), pack_bf16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                      pack_bf16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv), pack_bf16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
  if (half == 0) a.lse[((int64_t)b * a.H + h) * a.T + q0 + r] = (m_run + log2f(L)) * 0.6931471805599453f;
  tc_fence_before();
  __syncthreads();  // every TMEM read and red[] use of this task is done
  if (leader) {
    as.use[AB_FIXED] = ph.use[AB_FIXED] + 1u;
#pragma unroll
    for (int st = 0; st < kAttStages; ++st) as.use[AB_LD0 + st] = ph.use[AB_LD0 + st] + n_mod(nkb, st, kAttStages);
#pragma unroll
    for (int bb = 0; bb < 2; ++bb) {
      as.use[AB_S0 + bb] = ph.use[AB_S0 + bb] + n_mod(nkb, bb, 2);
      as.use[AB_O0 + bb] = ph.use[AB_O0 + bb] + n_mod(nkb, bb, 2);
    }
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
  const int r0 = idx * kAttPreRows, r1 = min(r0 + kAttPreRows, N);
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
__device__ inline void task_attn_bwd_kv_tc(const KParams& kp, const AttnArgs& a, int idx, uint8_t* smem,
                                           AttnShared& as, uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int nkb = a.T / kAttBlk;
  const int kb = idx % nkb;  // earliest keys see the most queries: claimed first
  const int h = (idx / nkb) % a.H, b = idx / (nkb * a.H);
  const int k0 = kb * kAttBlk, row0 = b * a.T, nq = nkb - kb;  // query blocks kb .. nkb - 1
  const void* qmap = reinterpret_cast<const uint8_t*>(kp.tmaps) + 128 * a.qkv_map;
  const void* dmap = reinterpret_cast<const uint8_t*>(kp.tmaps) + 128 * a.do_map;
  // tiles: K | V | Q stages 0..2 | dO stages 0..2 | P^T (two tiles) | dS^T (two tiles)
  const uint32_t sK = smem_u32(smem), sV = sK + kAttTile, sQ = sK + 2 * kAttTile,
                 sO = sQ + kAttStagesKV * kAttTile, sPt = sO + kAttStagesKV * kAttTile, sDs = sPt + 2 * kAttTile;
  const uint32_t bar0 = smem_u32(&as.bar[0]);
  AttnScratch& sc = *reinterpret_cast<AttnScratch*>(smem + kAttScratchOff);
  AttPhases ph;
  ph.load(as);
  // the copies, and each of the four products, issued by one thread of a different warp
  const bool leader = threadIdx.x == 0, st_issuer = threadIdx.x == 32, dpt_issuer = threadIdx.x == 64,
             dv_issuer = threadIdx.x == 96, dk_issuer = threadIdx.x == 160;
  const int r = quarter * 32 + lane;  // this thread's key row (TMEM lane)
  const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
  const uint32_t id_s = idesc_bf16(128, 128, 0, 0), id_o = idesc_bf16(128, 64, 0, 1);
  const float* Lg = a.lse + ((int64_t)b * a.H + h) * a.T;
  const float* Dg = a.scratch + ((int64_t)b * a.H + h) * a.T;
  const float log2e = 1.4426950408889634f, sl2 = a.scale * log2e;
  auto load_qo = [&](int it) {  // leader: Q and dO of query block kb + it into stage it mod kAttStagesKV
    const int st = it % kAttStagesKV, i = kb + it;
    const uint32_t bar = bar0 + 8 * (AB_LD0 + st);
    mbar_arrive_expect_tx(bar, 2 * kAttTile);
    tma_load_2d(sQ + st * kAttTile, qmap, h * 64, row0 + i * kAttBlk, bar);
    tma_load_2d(sO + st * kAttTile, dmap, h * 64, row0 + i * kAttBlk, bar);
  };
  auto stage_ld = [&](int it) {  // all threads: -LSE (base 2) and -D of query block kb + it
    const int i = kb + it, c = threadIdx.x & (kAttBlk - 1), w = threadIdx.x >> 7;
    const float v = w == 0 ? Lg[i * kAttBlk + c] * log2e : Dg[i * kAttBlk + c];
    sc.ld[it & 1][w][c] = -v;
  };
  if (leader) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive_expect_tx(bar0 + 8 * AB_FIXED, 2 * kAttTile);
    tma_load_2d(sK, qmap, a.C + h * 64, row0 + k0, bar0 + 8 * AB_FIXED);
    tma_load_2d(sV, qmap, 2 * a.C + h * 64, row0 + k0, bar0 + 8 * AB_FIXED);
    for (int it = 0; it < min(kAttStagesKV, nq); ++it) load_qo(it);
  }
  __syncwarp();
  stage_ld(0);
  __syncthreads();
  for (int it = 0; it < nq; ++it) {
    const int buf = it & 1, st = it % kAttStagesKV;
    // S^T = K Q_i^T and dP^T = V dO_i^T (their TMEM columns were read before the last block barrier)
    if (st_issuer || dpt_issuer) {
      if (it == 0) att_wait(kp, bar0 + 8 * AB_FIXED, ph.par(AB_FIXED, 0));
      att_wait(kp, bar0 + 8 * (AB_LD0 + st), ph.par(AB_LD0 + st, it / kAttStagesKV));
      tc_fence_after();
      if (st_issuer) att_mma_kk(tmem, sK, sQ + st * kAttTile, 4, id_s, false);
      else att_mma_kk(tmem + 128u, sV, sO + st * kAttTile, 4, id_s, false);
      tc_commit(bar0 + 8 * (AB_S0 + (st_issuer ? 0 : 1)));
    }
    __syncwarp();
    if (it + 1 < nq) stage_ld(it + 1);  // read after this block's barrier; its buffer was last read before the previous one
    att_wait(kp, bar0 + 8 * AB_S0, ph.par(AB_S0, it));
    att_wait(kp, bar0 + 8 * (AB_S0 + 1), ph.par(AB_S0 + 1, it));
    if (it >= 1) {  // the previous products no longer read P^T, dS^T, nor Q_{i-1}, dO_{i-1}: refill that stage
      att_wait(kp, bar0 + 8 * AB_O0, ph.par(AB_O0, it - 1));
      att_wait(kp, bar0 + 8 * (AB_O0 + 1), ph.par(AB_O0 + 1, it - 1));
      if (leader && it - 1 + kAttStagesKV < nq) load_qo(it - 1 + kAttStagesKV);
    }
    __syncwarp();
    tc_fence_after();
    const bool diag = it == 0;  // the key block's own query block: queries before a key are masked
    const float4* nlse2 = reinterpret_cast<const float4*>(sc.ld[buf][0]);  // -LSE log2 e per query column
    const float4* ndd = reinterpret_cast<const float4*>(sc.ld[buf][1]);    // -D per query column
    const float2 sl2v = make_float2(sl2, sl2), scv = make_float2(a.scale, a.scale);
#pragma unroll 1
    for (int q = 0; q < 2; ++q) {  // 32 query columns at a time
      float s[32], dp[32];
      const int c0 = half * 64 + q * 32;
      tmem_ld32(trow + (uint32_t)c0, s);
      tmem_ld32(trow + 128u + (uint32_t)c0, dp);
      // two columns per instruction: p = 2^(s sl2 - lse2), ds = p (dp - D) scale
#pragma unroll
      for (int e4 = 0; e4 < 8; ++e4) {
        const float4 nl = nlse2[(c0 >> 2) + e4], nd = ndd[(c0 >> 2) + e4];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int e = 4 * e4 + 2 * k, c = c0 + e;
          const float2 arg = f2_fma(make_float2(s[e], s[e + 1]), sl2v, k ? make_float2(nl.z, nl.w) : make_float2(nl.x, nl.y));
          const float2 p = make_float2((diag && c < r) ? 0.f : ex2_sfu(arg.x), (diag && c + 1 < r) ? 0.f : ex2_sfu(arg.y));
          const float2 t = f2_add(make_float2(dp[e], dp[e + 1]), k ? make_float2(nd.z, nd.w) : make_float2(nd.x, nd.y));
          const float2 ds = f2_mul(f2_mul(p, t), scv);
          s[e] = p.x; s[e + 1] = p.y;
          dp[e] = ds.x; dp[e + 1] = ds.y;
        }
      }
      st_row32_sw128(sPt + (uint32_t)half * kAttTile, r, q, s);
      st_row32_sw128(sDs + (uint32_t)half * kAttTile, r, q, dp);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    if (dv_issuer || dk_issuer) {  // dV += P^T dO_i, dK += dS^T Q_i
      tc_fence_after();
      if (dv_issuer) att_mma_kmn(tmem + 256u, sPt, sO + st * kAttTile, 8, id_o, it > 0);
      else att_mma_kmn(tmem + 320u, sDs, sQ + st * kAttTile, 8, id_o, it > 0);
      tc_commit(bar0 + 8 * (AB_O0 + (dv_issuer ? 0 : 1)));
    }
    __syncwarp();
  }
  att_wait(kp, bar0 + 8 * AB_O0, ph.par(AB_O0, nq - 1));
  att_wait(kp, bar0 + 8 * (AB_O0 + 1), ph.par(AB_O0 + 1, nq - 1));
  __syncwarp();
  tc_fence_after();
  const int64_t ld = 3 * (int64_t)a.C;
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.dqkv) + (int64_t)(row0 + k0 + r) * ld + h * 64 + half * 32;
  {
    float v[32];
    tmem_ld32(trow + 256u + 32u * half, v);  // dV
    uint4* dst = reinterpret_cast<uint4*>(out + 2 * a.C);
#pragma unroll
    for (int c = 0; c < 4; ++c)
      dst[c] = make_uint4(pack_bf16x2(v[8 * c], v[8 * c + 1]), pack_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                          pack_bf16x2(v[8 * c + 4], v[8 * c + 5]), pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
    tmem_ld32(trow + 320u + 32u * half, v);  // dK (rotated back to the projection's frame with rotary embedding)
    const int t = k0 + r;
    uint32_t w[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) w[e] = pack_unrotate<kRope>(a.rope, t, half * 32 + 2 * e, v[2 * e], v[2 * e + 1]);
    dst = reinterpret_cast<uint4*>(out + a.C);
#pragma unroll
    for (int c = 0; c < 4; ++c) dst[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
  }
  tc_fence_before();
  __syncthreads();
  if (leader) {
    as.use[AB_FIXED] = ph.use[AB_FIXED] + 1u;
#pragma unroll
    for (int st = 0; st < kAttStagesKV; ++st) as.use[AB_LD0 + st] = ph.use[AB_LD0 + st] + n_mod(nq, st, kAttStagesKV);
#pragma unroll
    for (int bb = 0; bb < 2; ++bb) {
      as.use[AB_S0 + bb] = ph.use[AB_S0 + bb] + (uint32_t)nq;
      as.use[AB_O0 + bb] = ph.use[AB_O0 + bb] + (uint32_t)nq;
    }
  }
}

// ---- backward dQ ------------------------------------------------------------------
template <bool kRope>
__device__ inline void task_attn_bwd_q_tc(const KParams& kp, const AttnArgs& a, int idx, uint8_t* smem,
                                          AttnShared& as, uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int nqb = a.T / kAttBlk;
  const int qb = nqb - 1 - idx % nqb;
  const int h = (idx / nqb) % a.H, b = idx / (nqb * a.H);
  const int q0 = qb * kAttBlk, row0 = b * a.T, nkb = qb + 1;
  const void* qmap = reinterpret_cast<const uint8_t*>(kp.tmaps) + 128 * a.qkv_map;
  const void* dmap = reinterpret_cast<const uint8_t*>(kp.tmaps) + 128 * a.do_map;
  // tiles: Q | dO | K stages 0..3 | V stages 0..3 | dS (two tiles)
  const uint32_t sQ = smem_u32(smem), sO = sQ + kAttTile, sK = sQ + 2 * kAttTile, sV = sK + kAttStages * kAttTile,
                 sDs = sV + kAttStages * kAttTile;
  const uint32_t bar0 = smem_u32(&as.bar[0]);
  AttPhases ph;
  ph.load(as);
  // the copies, and each of the three products, issued by one thread of a different warp
  const bool leader = threadIdx.x == 0, s_issuer = threadIdx.x == 32, dp_issuer = threadIdx.x == 64,
             dq_issuer = threadIdx.x == 96;
  const int r = quarter * 32 + lane;  // this thread's query row (TMEM lane)
  const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
  const uint32_t id_s = idesc_bf16(128, 128, 0, 0), id_o = idesc_bf16(128, 64, 0, 1);
  const float log2e = 1.4426950408889634f, sl2 = a.scale * log2e;
  const float lse2 = a.lse[((int64_t)b * a.H + h) * a.T + q0 + r] * log2e;
  const float dd = a.scratch[((int64_t)b * a.H + h) * a.T + q0 + r];
  auto load_kv = [&](int j) {  // leader: K_j and V_j into stage j mod kAttStages
    const int st = j % kAttStages;
    const uint32_t bar = bar0 + 8 * (AB_LD0 + st);
    mbar_arrive_expect_tx(bar, 2 * kAttTile);
    tma_load_2d(sK + st * kAttTile, qmap, a.C + h * 64, row0 + j * kAttBlk, bar);
    tma_load_2d(sV + st * kAttTile, qmap, 2 * a.C + h * 64, row0 + j * kAttBlk, bar);
  };
  if (leader) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive_expect_tx(bar0 + 8 * AB_FIXED, 2 * kAttTile);
    tma_load_2d(sQ, qmap, h * 64, row0 + q0, bar0 + 8 * AB_FIXED);
    tma_load_2d(sO, dmap, h * 64, row0 + q0, bar0 + 8 * AB_FIXED);
    for (int j = 0; j < min(kAttStages, nkb); ++j) load_kv(j);
  }
  __syncwarp();
  for (int j = 0; j < nkb; ++j) {
    const int st = j % kAttStages;
    // S = Q K_j^T, dP = dO V_j^T (their TMEM columns were read before the last block barrier)
    if (s_issuer || dp_issuer) {
      if (j == 0) att_wait(kp, bar0 + 8 * AB_FIXED, ph.par(AB_FIXED, 0));
      att_wait(kp, bar0 + 8 * (AB_LD0 + st), ph.par(AB_LD0 + st, j / kAttStages));
      tc_fence_after();
      if (s_issuer) att_mma_kk(tmem, sQ, sK + st * kAttTile, 4, id_s, false);
      else att_mma_kk(tmem + 128u, sO, sV + st * kAttTile, 4, id_s, false);
      tc_commit(bar0 + 8 * (AB_S0 + (s_issuer ? 0 : 1)));
    }
    __syncwarp();
    att_wait(kp, bar0 + 8 * AB_S0, ph.par(AB_S0, j));
    att_wait(kp, bar0 + 8 * (AB_S0 + 1), ph.par(AB_S0 + 1, j));
    if (j >= 1) {  // the previous product no longer reads dS, nor K_{j-1}, V_{j-1}: refill that stage
      att_wait(kp, bar0 + 8 * AB_O0, ph.par(AB_O0, j - 1));
      if (leader && j - 1 + kAttStages < nkb) load_kv(j - 1 + kAttStages);
    }
    __syncwarp();
    tc_fence_after();
    const bool diag = j == nkb - 1;  // keys after a query are masked
#pragma unroll 1
    for (int q = 0; q < 2; ++q) {
      float s[32], dp[32];
      const int c0 = half * 64 + q * 32;
      tmem_ld32(trow + (uint32_t)c0, s);
      tmem_ld32(trow + 128u + (uint32_t)c0, dp);
#pragma unroll
      for (int e = 0; e < 32; e += 2) {  // two columns per instruction
        const int c = c0 + e;
        const float2 arg = f2_fma(make_float2(s[e], s[e + 1]), make_float2(sl2, sl2), make_float2(-lse2, -lse2));
        const float2 p = make_float2((diag && c > r) ? 0.f : ex2_sfu(arg.x), (diag && c + 1 > r) ? 0.f : ex2_sfu(arg.y));
        const float2 t = f2_add(make_float2(dp[e], dp[e + 1]), make_float2(-dd, -dd));
        const float2 ds = f2_mul(f2_mul(p, t), make_float2(a.scale, a.scale));
        dp[e] = ds.x; dp[e + 1] = ds.y;
      }
      st_row32_sw128(sDs + (uint32_t)half * kAttTile, r, q, dp);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    if (dq_issuer) {  // dQ += dS K_j
      tc_fence_after();
      att_mma_kmn(tmem + 256u, sDs, sK + st * kAttTile, 8, id_o, j > 0);
      tc_commit(bar0 + 8 * AB_O0);
    }
    __syncwarp();
  }
  att_wait(kp, bar0 + 8 * AB_O0, ph.par(AB_O0, nkb - 1));
  __syncwarp();
  tc_fence_after();
  {
    float v[32];
    tmem_ld32(trow + 256u + 32u * half, v);
    const int t = q0 + r;
    uint32_t w[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) w[e] = pack_unrotate<kRope>(a.rope, t, half * 32 + 2 * e, v[2 * e], v[2 * e + 1]);
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.dqkv) +
                                          (int64_t)(row0 + t) * 3 * a.C + h * 64 + half * 32);
#pragma unroll
    for (int c = 0; c < 4; ++c) dst[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
  }
  tc_fence_before();
  __syncthreads();
  if (leader) {
    as.use[AB_FIXED] = ph.use[AB_FIXED] + 1u;
#pragma unroll
    for (int st = 0; st < kAttStages; ++st) as.use[AB_LD0 + st] = ph.use[AB_LD0 + st] + n_mod(nkb, st, kAttStages);
    as.use[AB_S0] = ph.use[AB_S0] + (uint32_t)nkb;
    as.use[AB_S0 + 1] = ph.use[AB_S0 + 1] + (uint32_t)nkb;
    as.use[AB_O0] = ph.use[AB_O0] + (uint32_t)nkb;
  }
}

}  // namespace pgs
