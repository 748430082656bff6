// tasks_simt.cuh — CUDA-core (SIMT, fp32 arithmetic) bodies of the dense tasks:
// a tiled GEMM with the fused epilogues, and causal attention forward/backward.
// These carry the fp32 configuration bit for bit in fp32 (no TF32).
#pragma once
#include "device.cuh"

namespace pgs {

// Tile of GEMM task idx: split-major, then M- or N-fastest as the host chose.
__device__ __forceinline__ void gemm_coords(const GemmArgs& g, int idx, int& tm, int& tn, int& split) {
  const int tiles_m = (g.M + g.BM - 1) / g.BM;
  const int per_split = tiles_m * g.tiles_n;
  split = idx / per_split;
  const int r = idx - split * per_split;
  if (g.m_fastest) { tm = r % tiles_m; tn = r / tiles_m; }
  else { tn = r % g.tiles_n; tm = r / g.tiles_n; }
}

// ---- GEMM epilogue, one element ----------------------------------------------
template <typename act_t>
__device__ __forceinline__ void epilogue_one(const GemmArgs& g, int split, int m, int n, float acc,
                                             bool gelu_tanh) {
  switch (g.epi) {
    case EPI_STORE: {
      if (g.bias) acc += g.bias[n];
      reinterpret_cast<act_t*>(g.out)[(int64_t)m * g.ldo + n] = from_f<act_t>(acc);
    } break;
    case EPI_RESID: {
      if (g.bias) acc += g.bias[n];
      reinterpret_cast<float*>(g.out)[(int64_t)m * g.ldo + n] = g.resid[(int64_t)m * g.ldr + n] + acc;
    } break;
    case EPI_GELU: {
      if (g.bias) acc += g.bias[n];
      reinterpret_cast<act_t*>(g.out)[(int64_t)m * g.ldo + n] = from_f<act_t>(gelu_grad_f(acc, gelu_tanh));
      reinterpret_cast<act_t*>(g.out2)[(int64_t)m * g.ldo2 + n] = from_f<act_t>(gelu_f(acc, gelu_tanh));
    } break;
    case EPI_F32: {
      if (n >= g.n_real) {  // padded columns: the first one is the bias gradient
        if (n == g.n_real && g.bias_grad) g.bias_grad[m] = acc;
        break;
      }
      reinterpret_cast<float*>(g.out)[split * g.split_stride + (int64_t)m * g.ldo + n] = acc;
    } break;
    case EPI_GELU_BWD: {
      const float dg = to_f<act_t>(reinterpret_cast<const act_t*>(g.aux)[(int64_t)m * g.ldaux + n]);
      reinterpret_cast<act_t*>(g.out)[(int64_t)m * g.ldo + n] = from_f<act_t>(acc * dg);
    } break;
  }
}

// ---- SIMT GEMM: 64 x 64 tile, BK 16, 4 x 4 outputs per thread ----------------
constexpr int kSimtBM = kSimtTile, kSimtBN = kSimtTile, kSimtBK = 16;

template <typename act_t>
__device__ inline void task_gemm_simt(const GemmArgs& g, int idx, float* smem, bool gelu_tanh) {
  int tm, tn, split;
  gemm_coords(g, idx, tm, tn, split);
  const int kchunk = (g.K + g.ksplit - 1) / g.ksplit;
  const int k0 = split * kchunk, k1 = min(g.K, k0 + kchunk);
  const int m0 = tm * kSimtBM, n0 = tn * kSimtBN;
  float* As = smem;                                // [BK][BM + 4]
  float* Bs = smem + kSimtBK * (kSimtBM + 4);      // [BK][BN + 4]
  const act_t* A = reinterpret_cast<const act_t*>(g.A);
  const act_t* B = reinterpret_cast<const act_t*>(g.B);
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int kk = k0; kk < k1; kk += kSimtBK) {
    // cooperative loads: 64 x 16 elements per operand, 4 per thread
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int li = threadIdx.x + e * kThreads;  // 0..1023
      // choose the loop order that walks the contiguous dimension across threads
      int r, k;
      if (g.sak == 1) { k = li % kSimtBK; r = li / kSimtBK; } else { r = li % kSimtBM; k = li / kSimtBM; }
      const int gm = m0 + r, gk = kk + k;
      As[k * (kSimtBM + 4) + r] =
          (gm < g.M && gk < k1) ? to_f<act_t>(A[(int64_t)gm * g.sam + (int64_t)gk * g.sak]) : 0.f;
      if (g.sbk == 1) { k = li % kSimtBK; r = li / kSimtBK; } else { r = li % kSimtBN; k = li / kSimtBN; }
      const int gn = n0 + r, gk2 = kk + k;
      Bs[k * (kSimtBN + 4) + r] =
          (gn < g.N && gk2 < k1) ? to_f<act_t>(B[(int64_t)gn * g.sbn + (int64_t)gk2 * g.sbk]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kSimtBK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[k * (kSimtBM + 4) + ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[k * (kSimtBN + 4) + tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
      if (m < g.M && n < g.N) epilogue_one<act_t>(g, split, m, n, acc[i][j], gelu_tanh);
    }
}

// ---- SIMT causal attention ---------------------------------------------------
// qkv row n = b*T + t holds q | k | v; head h occupies columns h*d .. h*d+d-1.
template <typename act_t>
__device__ __forceinline__ float qkv_at(const AttnArgs& a, int b, int t, int part, int h, int c) {
  const act_t* p = reinterpret_cast<const act_t*>(a.qkv);
  return to_f<act_t>(p[((int64_t)b * a.T + t) * (3 * a.C) + part * a.C + h * a.d + c]);
}

// Scores of query rows q0..q0+rows-1 against keys 0..kv_len-1 into S[QB][T]
// (masked entries = -inf).  Q rows are staged in Qs[QB][d].
template <typename act_t>
__device__ inline void attn_scores(const AttnArgs& a, int b, int h, int q0, int rows, int kv_len,
                            float* Qs, float* Ks, float* S) {
  const int QB = a.q_block, d = a.d;
  for (int e = threadIdx.x; e < QB * d; e += kThreads) {
    const int i = e / d, c = e % d;
    Qs[e] = i < rows ? qkv_at<act_t>(a, b, q0 + i, 0, h, c) : 0.f;
  }
  for (int j0 = 0; j0 < kv_len; j0 += 64) {
    __syncthreads();
    for (int e = threadIdx.x; e < 64 * d; e += kThreads) {
      const int jj = e / d, c = e % d;
      Ks[jj * (d + 1) + c] = (j0 + jj < kv_len) ? qkv_at<act_t>(a, b, j0 + jj, 1, h, c) : 0.f;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < QB * 64; e += kThreads) {
      const int i = e / 64, jj = e % 64, j = j0 + jj;
      if (i < rows && j < kv_len) {
        float s = 0.f;
        for (int c = 0; c < d; ++c) s = fmaf(Qs[i * d + c], Ks[jj * (d + 1) + c], s);
        S[i * a.T + j] = (j > q0 + i) ? -INFINITY : s * a.scale;
      }
    }
  }
  __syncthreads();
}

template <typename act_t>
__device__ inline void task_attn_fwd_simt(const AttnArgs& a, int idx, float* smem) {
  const int nqb = (a.T + a.q_block - 1) / a.q_block;
  const int qb = idx % nqb, h = (idx / nqb) % a.H, b = idx / (nqb * a.H);
  const int QB = a.q_block, d = a.d;
  const int q0 = qb * QB, rows = min(QB, a.T - q0), kv_len = q0 + rows;
  float* Qs = smem;                 // [QB][d]
  float* Ks = Qs + QB * d;          // [64][d+1]
  float* S = Ks + 64 * (d + 1);     // [QB][T]
  attn_scores<act_t>(a, b, h, q0, rows, kv_len, Qs, Ks, S);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = warp; i < rows; i += kWarps) {
    const int last = q0 + i;  // keys 0..last are visible
    float m = -INFINITY;
    for (int j = lane; j <= last; j += 32) m = fmaxf(m, S[i * a.T + j]);
    m = warp_max(m);
    float s = 0.f;
    for (int j = lane; j <= last; j += 32) {
      const float e = expf(S[i * a.T + j] - m);
      S[i * a.T + j] = e;
      s += e;
    }
    s = warp_sum(s);
    const float inv = 1.0f / s;
    for (int j = lane; j < kv_len; j += 32) S[i * a.T + j] = j <= last ? S[i * a.T + j] * inv : 0.f;
    if (lane == 0) a.lse[((int64_t)b * a.H + h) * a.T + q0 + i] = m + logf(s);
  }
  __syncthreads();
  act_t* O = reinterpret_cast<act_t*>(a.o);
  for (int e = threadIdx.x; e < rows * d; e += kThreads) {
    const int i = e / d, c = e % d;
    float acc = 0.f;
    for (int j = 0; j <= q0 + i; ++j) acc = fmaf(S[i * a.T + j], qkv_at<act_t>(a, b, j, 2, h, c), acc);
    O[((int64_t)b * a.T + q0 + i) * a.ld_o + h * d + c] = from_f<act_t>(acc);
  }
}

// Backward of one (batch, head): for every query block, P is recomputed from
// the saved LSE; D_i = sum_c dO_ic O_ic; dV += P^T dO; dS = P (dO V^T - D) scale;
// dQ = dS K; dK += dS^T Q.  dK/dV accumulate in this task's private fp32 scratch.
template <typename act_t>
__device__ inline void task_attn_bwd_simt(const AttnArgs& a, int idx, float* smem) {
  const int h = idx % a.H, b = idx / a.H;
  const int QB = a.q_block, d = a.d, T = a.T;
  float* dK = a.scratch + (int64_t)idx * 2 * T * d;
  float* dV = dK + (int64_t)T * d;
  for (int e = threadIdx.x; e < 2 * T * d; e += kThreads) dK[e] = 0.f;
  float* Qs = smem;                 // [QB][d]
  float* Ks = Qs + QB * d;          // [64][d+1]
  float* S = Ks + 64 * (d + 1);     // [QB][T]
  float* dOs = S + QB * T;          // [QB][d]
  float* Ds = dOs + QB * d;         // [QB]
  const act_t* dO = reinterpret_cast<const act_t*>(a.dout);
  const act_t* Oa = reinterpret_cast<const act_t*>(a.o);
  act_t* dqkv = reinterpret_cast<act_t*>(a.dqkv);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = (T + QB - 1) / QB;
  for (int qb = 0; qb < nqb; ++qb) {
    const int q0 = qb * QB, rows = min(QB, T - q0), kv_len = q0 + rows;
    __syncthreads();
    attn_scores<act_t>(a, b, h, q0, rows, kv_len, Qs, Ks, S);
    for (int e = threadIdx.x; e < QB * d; e += kThreads) {
      const int i = e / d, c = e % d;
      dOs[e] = i < rows ? to_f<act_t>(dO[((int64_t)b * T + q0 + i) * a.C + h * d + c]) : 0.f;
    }
    for (int i = warp; i < rows; i += kWarps) {
      const float lse = a.lse[((int64_t)b * a.H + h) * T + q0 + i];
      for (int j = lane; j < kv_len; j += 32)
        S[i * T + j] = j <= q0 + i ? expf(S[i * T + j] - lse) : 0.f;
      float s = 0.f;
      for (int c = lane; c < d; c += 32)
        s += to_f<act_t>(dO[((int64_t)b * T + q0 + i) * a.C + h * d + c]) *
             to_f<act_t>(Oa[((int64_t)b * T + q0 + i) * a.ld_o + h * d + c]);
      s = warp_sum(s);
      if (lane == 0) Ds[i] = s;
    }
    __syncthreads();
    // dV[j] += sum_i P[i, j] dO[i]
    for (int e = threadIdx.x; e < kv_len * d; e += kThreads) {
      const int j = e / d, c = e % d;
      float acc = 0.f;
      for (int i = max(0, j - q0); i < rows; ++i) acc = fmaf(S[i * T + j], dOs[i * d + c], acc);
      dV[(int64_t)j * d + c] += acc;
    }
    __syncthreads();
    // dS = P (dP - D) scale, with dP[i, j] = dO_i . v_j  (in place over P)
    for (int e = threadIdx.x; e < rows * kv_len; e += kThreads) {
      const int i = e / kv_len, j = e % kv_len;
      if (j <= q0 + i) {
        float dp = 0.f;
        for (int c = 0; c < d; ++c) dp = fmaf(dOs[i * d + c], qkv_at<act_t>(a, b, j, 2, h, c), dp);
        S[i * T + j] = S[i * T + j] * (dp - Ds[i]) * a.scale;
      }
    }
    __syncthreads();
    // dQ[i] = sum_j dS[i, j] k_j
    for (int e = threadIdx.x; e < rows * d; e += kThreads) {
      const int i = e / d, c = e % d;
      float acc = 0.f;
      for (int j = 0; j <= q0 + i; ++j) acc = fmaf(S[i * T + j], qkv_at<act_t>(a, b, j, 1, h, c), acc);
      dqkv[((int64_t)b * T + q0 + i) * (3 * a.C) + h * d + c] = from_f<act_t>(acc);
    }
    // dK[j] += sum_i dS[i, j] q_i
    for (int e = threadIdx.x; e < kv_len * d; e += kThreads) {
      const int j = e / d, c = e % d;
      float acc = 0.f;
      for (int i = max(0, j - q0); i < rows; ++i) acc = fmaf(S[i * T + j], Qs[i * d + c], acc);
      dK[(int64_t)j * d + c] += acc;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < T * d; e += kThreads) {
    const int j = e / d, c = e % d;
    dqkv[((int64_t)b * T + j) * (3 * a.C) + a.C + h * d + c] = from_f<act_t>(dK[e]);
    dqkv[((int64_t)b * T + j) * (3 * a.C) + 2 * a.C + h * d + c] = from_f<act_t>(dV[e]);
  }
}

}  // namespace pgs
