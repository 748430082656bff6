// tasks_rows.cuh — row-parallel and elementwise task bodies of the persistent
// kernel: embedding, LayerNorm forward/backward, softmax cross-entropy with its
// gradient, the loss reduction, column sums, embedding backward and AdamW.
// Every body is executed by all kThreads threads of one block and uses a fixed
// summation order, so a step is bitwise repeatable.
#pragma once
#include "device.cuh"
#include "tc_gemm.cuh"

namespace pgs {

// ---- 1-D bulk copies (async proxy) between global and shared memory ----
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }


// x0[n] = wte[tok[n]] + wpe[n mod T]  (token + learned position embedding).
template <typename act_t>
__device__ inline void task_embed(const KParams& kp, const EmbedArgs& a, int idx) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = idx * a.rows_per_task, r1 = min(r0 + a.rows_per_task, a.N);
  for (int r = r0 + warp; r < r1; r += kWarps) {
    int tok = step_tokens(kp)[r];
    if (tok < 0 || tok >= a.V) {
      if (lane == 0) set_soft(kp, kSoftBadToken);
      tok = tok < 0 ? 0 : a.V - 1;
    }
    const float4* we = reinterpret_cast<const float4*>(a.wte + (int64_t)tok * a.C);
    float4* xo = reinterpret_cast<float4*>(a.x0 + (int64_t)r * a.C);
    if (a.wpe) {
      const float4* pe = reinterpret_cast<const float4*>(a.wpe + (int64_t)(r % a.T) * a.C);
      for (int c = lane; c < a.C / 4; c += 32) {
        float4 u = we[c], w = pe[c];
        xo[c] = make_float4(u.x + w.x, u.y + w.y, u.z + w.z, u.w + w.w);
      }
    } else {  // rotary position embedding instead of a learned position table
      for (int c = lane; c < a.C / 4; c += 32) xo[c] = we[c];
    }
  }
}

// LayerNorm forward, one warp per row.  mean = sum x / C,
// var = sum (x - mean)^2 / C (biased), y = (x - mean) rstd g + b.
// NV > 0: C = 128 NV, lane holds float4 number lane + 32 i in registers;
// NV = 0: any C (multiple of 32), three passes over the row (L1-resident).
template <typename act_t>
__device__ __forceinline__ void store4(act_t* p, float a, float b, float c, float d);
template <>
__device__ __forceinline__ void store4<float>(float* p, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, float a, float b, float c, float d) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&lo);
  u.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = u;
}

template <typename act_t, int NV>
__device__ __forceinline__ void ln_fwd_rows(const LnFwdArgs& a, int r0, int r1) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  act_t* y = reinterpret_cast<act_t*>(a.y);
  const float invC = 1.0f / (float)a.C;
  if constexpr (NV > 0) {
    // g and b are the same for every row; the next row's x is loaded while
    // this one is reduced and written, so a warp waits about once per task.
    float4 g[NV], bb[NV], nv[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int c = 4 * (lane + 32 * i);
      g[i] = *reinterpret_cast<const float4*>(a.g + c);
      bb[i] = a.b ? *reinterpret_cast<const float4*>(a.b + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    int r = r0 + warp;
    if (r < r1) {
#pragma unroll
      for (int i = 0; i < NV; ++i) nv[i] = reinterpret_cast<const float4*>(a.x + (int64_t)r * a.C)[lane + 32 * i];
    }
    for (; r < r1; r += kWarps) {
      float4 v[NV];
#pragma unroll
      for (int i = 0; i < NV; ++i) v[i] = nv[i];
      if (r + kWarps < r1) {
#pragma unroll
        for (int i = 0; i < NV; ++i)
          nv[i] = reinterpret_cast<const float4*>(a.x + (int64_t)(r + kWarps) * a.C)[lane + 32 * i];
      }
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < NV; ++i) s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
      const float mean = warp_sum(s) * invC;
      float q = 0.f;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const float d0 = v[i].x - mean, d1 = v[i].y - mean, d2 = v[i].z - mean, d3 = v[i].w - mean;
        q += (d0 * d0 + d1 * d1) + (d2 * d2 + d3 * d3);
      }
      const float rstd = rsqrtf(warp_sum(q) * invC + a.eps);
      act_t* yr = y + (int64_t)r * a.ldy;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int c = 4 * (lane + 32 * i);
        store4<act_t>(yr + c, (v[i].x - mean) * rstd * g[i].x + bb[i].x, (v[i].y - mean) * rstd * g[i].y + bb[i].y,
                      (v[i].z - mean) * rstd * g[i].z + bb[i].z, (v[i].w - mean) * rstd * g[i].w + bb[i].w);
      }
      if (a.copy) {
#pragma unroll
        for (int i = 0; i < NV; ++i) reinterpret_cast<float4*>(a.copy + (int64_t)r * a.C)[lane + 32 * i] = v[i];
      }
      if (lane == 0) { a.mean[r] = mean; a.rstd[r] = rstd; }
    }
  } else {
    for (int r = r0 + warp; r < r1; r += kWarps) {
      const float* x = a.x + (int64_t)r * a.C;
      act_t* yr = y + (int64_t)r * a.ldy;
      float s = 0.f;
      for (int c = lane; c < a.C; c += 32) s += x[c];
      const float mean = warp_sum(s) * invC;
      float q = 0.f;
      for (int c = lane; c < a.C; c += 32) { const float d = x[c] - mean; q += d * d; }
      const float rstd = rsqrtf(warp_sum(q) * invC + a.eps);
      for (int c = lane; c < a.C; c += 32) {
        float o = (x[c] - mean) * rstd * a.g[c];
        if (a.b) o += a.b[c];
        yr[c] = from_f<act_t>(o);
        if (a.copy) a.copy[(int64_t)r * a.C + c] = x[c];
      }
      if (lane == 0) { a.mean[r] = mean; a.rstd[r] = rstd; }
    }
  }
}

template <typename act_t>
__device__ inline void task_ln_fwd(const LnFwdArgs& a, int idx) {
  const int r0 = idx * a.rows_per_task, r1 = min(r0 + a.rows_per_task, a.rows);
  switch ((a.C & 127) ? 0 : a.C >> 7) {
    case 2: ln_fwd_rows<act_t, 2>(a, r0, r1); break;
    case 4: ln_fwd_rows<act_t, 4>(a, r0, r1); break;
    case 6: ln_fwd_rows<act_t, 6>(a, r0, r1); break;
    case 8: ln_fwd_rows<act_t, 8>(a, r0, r1); break;
    default: ln_fwd_rows<act_t, 0>(a, r0, r1); break;
  }
}

// LayerNorm backward for a block of rows:
//   dxhat = dy g; dx = rstd (dxhat - mean(dxhat) - xhat mean(dxhat xhat));
//   dres_out = dres_in + dx (fp32 and act copies);
//   dg_part[task] = sum_rows dy xhat, db_part[task] = sum_rows dy.
// Warp w adds its rows' dy xhat and dy, in row order, into its own shared-memory
// rows; the warps' rows are then added in warp order (fixed summation order).
template <typename act_t, int NV>
__device__ __forceinline__ void ln_bwd_load(const LnBwdArgs& a, int r, int lane, float4* dy, float4* xv, float4* din,
                                            float& mean, float& rstd) {
  mean = a.mean[r];
  rstd = a.rstd[r];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int64_t c = (int64_t)r * a.C + 4 * (lane + 32 * i);
    dy[i] = *reinterpret_cast<const float4*>(a.dy + c);
    xv[i] = *reinterpret_cast<const float4*>(a.x + c);
    din[i] = a.dres_in ? *reinterpret_cast<const float4*>(a.dres_in + c) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int sp = 1; sp < a.dy_splits; ++sp) {  // split-K partials of dy (final LayerNorm only)
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const float4 e = *reinterpret_cast<const float4*>(a.dy + sp * a.dy_split_stride + (int64_t)r * a.C +
                                                        4 * (lane + 32 * i));
      dy[i].x += e.x; dy[i].y += e.y; dy[i].z += e.z; dy[i].w += e.w;
    }
  }
}

template <typename act_t, int NV>
__device__ __forceinline__ void ln_bwd_rows(const LnBwdArgs& a, int r0, int r1, float* sg, float* sb) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  act_t* dact = reinterpret_cast<act_t*>(a.dres_act);
  const float invC = 1.0f / (float)a.C;
  float* wg = sg + warp * a.C;
  float* wb = sb + warp * a.C;
  if constexpr (NV > 0) {
    // dy, x and the incoming residual gradient of a row are loaded together, and
    // (for C <= 768, where the registers allow) those of the warp's next row
    // while this one is reduced and written: about one memory latency per task.
    constexpr bool kPrefetch = NV <= 6;
    float4 ndy[NV], nx[NV], ndin[NV];
    float nmean = 0.f, nrstd = 0.f;
    int r = r0 + warp;
    if (kPrefetch && r < r1) ln_bwd_load<act_t, NV>(a, r, lane, ndy, nx, ndin, nmean, nrstd);
    for (; r < r1; r += kWarps) {
      float4 dy[NV], xh[NV], din[NV];
      float mean, rstd;
      if constexpr (kPrefetch) {
        mean = nmean;
        rstd = nrstd;
#pragma unroll
        for (int i = 0; i < NV; ++i) { dy[i] = ndy[i]; xh[i] = nx[i]; din[i] = ndin[i]; }
        if (r + kWarps < r1) ln_bwd_load<act_t, NV>(a, r + kWarps, lane, ndy, nx, ndin, nmean, nrstd);
      } else {
        ln_bwd_load<act_t, NV>(a, r, lane, dy, xh, din, mean, rstd);
      }
      float4 g[NV];
#pragma unroll
      for (int i = 0; i < NV; ++i) g[i] = *reinterpret_cast<const float4*>(a.g + 4 * (lane + 32 * i));
      float s1 = 0.f, s2 = 0.f;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int c = 4 * (lane + 32 * i);
        const float4 d = dy[i];
        xh[i] = make_float4((xh[i].x - mean) * rstd, (xh[i].y - mean) * rstd, (xh[i].z - mean) * rstd,
                            (xh[i].w - mean) * rstd);
        const float a0 = d.x * g[i].x, a1 = d.y * g[i].y, a2 = d.z * g[i].z, a3 = d.w * g[i].w;
        s1 += (a0 + a1) + (a2 + a3);
        s2 += (a0 * xh[i].x + a1 * xh[i].y) + (a2 * xh[i].z + a3 * xh[i].w);
        float4 pg = *reinterpret_cast<float4*>(wg + c);
        pg.x += d.x * xh[i].x; pg.y += d.y * xh[i].y; pg.z += d.z * xh[i].z; pg.w += d.w * xh[i].w;
        *reinterpret_cast<float4*>(wg + c) = pg;
        float4 pb = *reinterpret_cast<float4*>(wb + c);
        pb.x += d.x; pb.y += d.y; pb.z += d.z; pb.w += d.w;
        *reinterpret_cast<float4*>(wb + c) = pb;
      }
      s1 = warp_sum(s1) * invC;
      s2 = warp_sum(s2) * invC;
      float* out = a.dres_out + (int64_t)r * a.C;
      act_t* oa = dact + (int64_t)r * a.C;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int c = 4 * (lane + 32 * i);
        const float4 o = make_float4(rstd * (dy[i].x * g[i].x - s1 - xh[i].x * s2) + din[i].x,
                                     rstd * (dy[i].y * g[i].y - s1 - xh[i].y * s2) + din[i].y,
                                     rstd * (dy[i].z * g[i].z - s1 - xh[i].z * s2) + din[i].z,
                                     rstd * (dy[i].w * g[i].w - s1 - xh[i].w * s2) + din[i].w);
        *reinterpret_cast<float4*>(out + c) = o;
        store4<act_t>(oa + c, o.x, o.y, o.z, o.w);
      }
    }
  } else {
    for (int r = r0 + warp; r < r1; r += kWarps) {
      const float mean = a.mean[r], rstd = a.rstd[r];
      const float* x = a.x + (int64_t)r * a.C;
      float* out = a.dres_out + (int64_t)r * a.C;
      const float* din = a.dres_in ? a.dres_in + (int64_t)r * a.C : nullptr;
      act_t* oa = dact + (int64_t)r * a.C;
      float s1 = 0.f, s2 = 0.f;
      for (int c = lane; c < a.C; c += 32) {
        float d = 0.f;
        for (int sp = 0; sp < a.dy_splits; ++sp) d += a.dy[sp * a.dy_split_stride + (int64_t)r * a.C + c];
        const float xh = (x[c] - mean) * rstd;
        const float dxh = d * a.g[c];
        s1 += dxh;
        s2 += dxh * xh;
        wg[c] += d * xh;
        wb[c] += d;
      }
      s1 = warp_sum(s1) * invC;
      s2 = warp_sum(s2) * invC;
      for (int c = lane; c < a.C; c += 32) {
        float d = 0.f;
        for (int sp = 0; sp < a.dy_splits; ++sp) d += a.dy[sp * a.dy_split_stride + (int64_t)r * a.C + c];
        const float xh = (x[c] - mean) * rstd;
        float dx = rstd * (d * a.g[c] - s1 - xh * s2);
        if (din) dx += din[c];
        out[c] = dx;
        oa[c] = from_f<act_t>(dx);
      }
    }
  }
}

template <typename act_t>
__device__ inline void task_ln_bwd(const LnBwdArgs& a, int idx, float* smem) {
  const int r0 = idx * a.rows_per_task, r1 = min(r0 + a.rows_per_task, a.rows);
  float* sg = smem;                 // [kWarps][C]
  float* sb = smem + kWarps * a.C;  // [kWarps][C]
  for (int e = threadIdx.x; e < 2 * kWarps * a.C; e += kThreads) smem[e] = 0.f;
  __syncthreads();
  switch ((a.C & 127) ? 0 : a.C >> 7) {
    case 2: ln_bwd_rows<act_t, 2>(a, r0, r1, sg, sb); break;
    case 4: ln_bwd_rows<act_t, 4>(a, r0, r1, sg, sb); break;
    case 6: ln_bwd_rows<act_t, 6>(a, r0, r1, sg, sb); break;
    case 8: ln_bwd_rows<act_t, 8>(a, r0, r1, sg, sb); break;
    default: ln_bwd_rows<act_t, 0>(a, r0, r1, sg, sb); break;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < a.C; c += kThreads) {
    float g = 0.f, b = 0.f;
    for (int w = 0; w < kWarps; ++w) { g += sg[w * a.C + c]; b += sb[w * a.C + c]; }
    a.dg_part[(int64_t)idx * a.C + c] = g;
    if (a.db_part) a.db_part[(int64_t)idx * a.C + c] = b;
  }
}

// LayerNorm backward of a block of rows (same formulas as task_ln_bwd) with
// every input staged in shared memory first: thread 0 issues one bulk copy per
// array (dy and its split-K partials, x, the incoming residual gradient: the
// task's rows of each are contiguous), all in flight together, so the task
// waits about one memory latency instead of one per row a warp handles.  A
// warp then reduces its rows (C = 128 NV; lane holds float4 lane + 32 i) from
// shared memory and writes dres_out and its act copy with coalesced stores.
// The gain / bias partials of a warp's rows are summed in registers in row
// order, then across warps in warp order (a fixed order: steps stay bitwise
// repeatable).  Shared memory: (dy_splits + 1 + [dres_in]) x rows x C x 4 bytes.
template <typename act_t, int NV>
__device__ inline void task_ln_bwd_staged(const KParams& kp, const LnBwdArgs& a, int idx, uint8_t* smem,
                                          uint64_t* bars, uint32_t* iter) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = idx * a.rows_per_task, r1 = min(r0 + a.rows_per_task, a.rows);
  const int nr = r1 - r0;
  const int S = a.dy_splits;
  const uint32_t blk = (uint32_t)nr * (uint32_t)a.C * 4u;   // bytes of one array's rows (a multiple of 512)
  const uint32_t sbase = smem_u32(smem);
  const uint32_t it = *iter;
  const uint32_t bar = smem_u32(bars) + 8u * (it % kAdamStages);
  const uint32_t phase = (it / kAdamStages) & 1u;
  if (threadIdx.x == 0) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // earlier generic use of this memory
    const uint32_t total = blk * (uint32_t)(S + 1 + (a.dres_in ? 1 : 0));
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(total) : "memory");
    const int64_t off = (int64_t)r0 * a.C;
    for (int sp = 0; sp < S; ++sp) bulk_load(sbase + sp * blk, a.dy + sp * a.dy_split_stride + off, blk, bar);
    bulk_load(sbase + S * blk, a.x + off, blk, bar);
    if (a.dres_in) bulk_load(sbase + (S + 1) * blk, a.dres_in + off, blk, bar);
  }
  float4 g[NV], pg[NV], pb[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    g[i] = *reinterpret_cast<const float4*>(a.g + 4 * (lane + 32 * i));
    pg[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    pb[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const bool ok = __syncthreads_and(mbar_wait(kp, bar, phase));
  if (threadIdx.x == 0) *iter = it + 1u;  // this stage's phase is used (read by the next task after the block barrier)
  if (!ok) return;  // every thread leaves together
  const float invC = 1.0f / (float)a.C;
  act_t* dact = reinterpret_cast<act_t*>(a.dres_act);
  const float* sdy = reinterpret_cast<const float*>(smem);
  const float* sx = reinterpret_cast<const float*>(smem + S * blk);
  const float* sin = reinterpret_cast<const float*>(smem + (S + 1) * blk);
  for (int k = warp; k < nr; k += kWarps) {
    const int r = r0 + k;
    const float mean = a.mean[r], rstd = a.rstd[r];
    float4 dy[NV], xh[NV];
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int c = 4 * (lane + 32 * i);
      float4 d = *reinterpret_cast<const float4*>(sdy + (int64_t)k * a.C + c);
      for (int sp = 1; sp < S; ++sp) {
        const float4 e = *reinterpret_cast<const float4*>(sdy + (int64_t)sp * (blk / 4) + (int64_t)k * a.C + c);
        d.x += e.x; d.y += e.y; d.z += e.z; d.w += e.w;
      }
      dy[i] = d;
      const float4 xv = *reinterpret_cast<const float4*>(sx + (int64_t)k * a.C + c);
      xh[i] = make_float4((xv.x - mean) * rstd, (xv.y - mean) * rstd, (xv.z - mean) * rstd, (xv.w - mean) * rstd);
      const float a0 = d.x * g[i].x, a1 = d.y * g[i].y, a2 = d.z * g[i].z, a3 = d.w * g[i].w;
      s1 += (a0 + a1) + (a2 + a3);
      s2 += (a0 * xh[i].x + a1 * xh[i].y) + (a2 * xh[i].z + a3 * xh[i].w);
      pg[i].x += d.x * xh[i].x; pg[i].y += d.y * xh[i].y; pg[i].z += d.z * xh[i].z; pg[i].w += d.w * xh[i].w;
      pb[i].x += d.x; pb[i].y += d.y; pb[i].z += d.z; pb[i].w += d.w;
    }
    s1 = warp_sum(s1) * invC;
    s2 = warp_sum(s2) * invC;
    float* out = a.dres_out + (int64_t)r * a.C;
    act_t* oa = dact + (int64_t)r * a.C;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int c = 4 * (lane + 32 * i);
      float4 din = make_float4(0.f, 0.f, 0.f, 0.f);
      if (a.dres_in) din = *reinterpret_cast<const float4*>(sin + (int64_t)k * a.C + c);
      const float4 o = make_float4(rstd * (dy[i].x * g[i].x - s1 - xh[i].x * s2) + din.x,
                                   rstd * (dy[i].y * g[i].y - s1 - xh[i].y * s2) + din.y,
                                   rstd * (dy[i].z * g[i].z - s1 - xh[i].z * s2) + din.z,
                                   rstd * (dy[i].w * g[i].w - s1 - xh[i].w * s2) + din.w);
      *reinterpret_cast<float4*>(out + c) = o;
      store4<act_t>(oa + c, o.x, o.y, o.z, o.w);
    }
  }
  __syncthreads();  // every read of the staged rows is done: the area holds the warps' partials now
  float* wg = reinterpret_cast<float*>(smem);            // [kWarps][C]
  float* wb = wg + kWarps * a.C;                         // [kWarps][C]
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = 4 * (lane + 32 * i);
    *reinterpret_cast<float4*>(wg + warp * a.C + c) = pg[i];
    *reinterpret_cast<float4*>(wb + warp * a.C + c) = pb[i];
  }
  __syncthreads();
  for (int c = threadIdx.x; c < a.C; c += kThreads) {
    float sg = 0.f, sb = 0.f;
    for (int w = 0; w < kWarps; ++w) { sg += wg[w * a.C + c]; sb += wb[w * a.C + c]; }
    a.dg_part[(int64_t)idx * a.C + c] = sg;
    if (a.db_part) a.db_part[(int64_t)idx * a.C + c] = sb;
  }
}

template <typename act_t>
__device__ inline void task_ln_bwd_staged_any(const KParams& kp, const LnBwdArgs& a, int idx, uint8_t* smem,
                                              uint64_t* bars, uint32_t* iter) {
  switch (a.C >> 7) {  // the host stages only C = 128 NV, NV <= 8
    case 2: task_ln_bwd_staged<act_t, 2>(kp, a, idx, smem, bars, iter); break;
    case 4: task_ln_bwd_staged<act_t, 4>(kp, a, idx, smem, bars, iter); break;
    case 6: task_ln_bwd_staged<act_t, 6>(kp, a, idx, smem, bars, iter); break;
    case 8: task_ln_bwd_staged<act_t, 8>(kp, a, idx, smem, bars, iter); break;
    default: break;
  }
}

// Softmax cross-entropy of a block of rows, one warp per row:
// lse = log sum_j exp z_j (max subtracted), loss_n = lse - z[t_n],
// dz_j = (exp(z_j - lse) - [j = t_n]) / N written over the logits.
template <typename act_t>
__device__ inline void task_ce(const KParams& kp, const CeArgs& a, int idx) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = idx * a.rows_per_task, r1 = min(r0 + a.rows_per_task, a.N);
  act_t* L = reinterpret_cast<act_t*>(a.logits);
  const float invN = 1.0f / (float)a.N;
  for (int r = r0 + warp; r < r1; r += kWarps) {
    act_t* z = L + (int64_t)r * a.V;
    int t = step_targets(kp)[r];
    if (t < 0 || t >= a.V) {
      if (lane == 0) set_soft(kp, kSoftBadToken);
      t = t < 0 ? 0 : a.V - 1;
    }
    float m = -INFINITY, s = 0.f;
    for (int j = lane; j < a.V; j += 32) {
      const float x = to_f<act_t>(z[j]);
      if (x > m) { s = s * expf(m - x) + 1.0f; m = x; }
      else s += expf(x - m);
    }
    const float M = warp_max(m);
    s = (m == -INFINITY) ? 0.f : s * expf(m - M);
    const float S = warp_sum(s);
    const float lse = M + logf(S);
    const float zt = to_f<act_t>(z[t]);
    __syncwarp();
    if (lane == 0) {
      a.row_loss[r] = lse - zt;
      if (!isfinite(lse - zt)) set_soft(kp, kSoftNonFinite);
    }
    for (int j = lane; j < a.V; j += 32) {
      const float x = to_f<act_t>(z[j]);
      float p = expf(x - lse);
      if (j == t) p -= 1.0f;
      z[j] = from_f<act_t>(p * invN);
    }
  }
}

// Vectorised variant for bf16 logits with V % 8 == 0: 16-byte loads, 4 in flight.
// bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 word.
__device__ __forceinline__ void bf16x8_to_f(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ uint32_t f2_to_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ uint4 f_to_bf16x8(const float* f) {
  return make_uint4(f2_to_bf16x2(f[0], f[1]), f2_to_bf16x2(f[2], f[3]), f2_to_bf16x2(f[4], f[5]),
                    f2_to_bf16x2(f[6], f[7]));
}
// 2^x with the SFU's approximate base-2 exponential (relative error ~2^-22,
// subnormal results flushed to zero): one instruction.
__device__ __forceinline__ float ex2_sfu(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ inline void task_ce_bf16_vec(const KParams& kp, const CeArgs& a, int idx) {
  // One warp per row; every lane keeps eight 16-byte loads in flight in both
  // passes (a row of 50k logits is ~100 KB, mostly L2-resident right after the
  // LM-head tiles that wrote it).  exp is the fast hardware form (__expf):
  // its relative error (a few 1e-6 at these arguments) is far below the bf16
  // rounding of the gradient it feeds.
  constexpr int kU = 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = idx * a.rows_per_task, r1 = min(r0 + a.rows_per_task, a.N);
  const float invN = 1.0f / (float)a.N;
  const int nvec = a.V >> 3;
  for (int r = r0 + warp; r < r1; r += kWarps) {
    __nv_bfloat16* zr = reinterpret_cast<__nv_bfloat16*>(a.logits) + (int64_t)r * a.V;
    uint4* z = reinterpret_cast<uint4*>(zr);
    int t = step_targets(kp)[r];
    if (t < 0 || t >= a.V) {
      if (lane == 0) set_soft(kp, kSoftBadToken);
      t = t < 0 ? 0 : a.V - 1;
    }
    float m = -INFINITY, s = 0.f;
    for (int j = lane; j < nvec; j += 32 * kU) {
      uint4 u[kU];
#pragma unroll
      for (int q = 0; q < kU; ++q)
        if (j + 32 * q < nvec) u[q] = z[j + 32 * q];
#pragma unroll
      for (int q = 0; q < kU; ++q) {
        if (j + 32 * q >= nvec) break;
        float f[8];
        bf16x8_to_f(u[q], f);
        float lm = f[0];
#pragma unroll
        for (int e = 1; e < 8; ++e) lm = fmaxf(lm, f[e]);
        if (lm > m) { s *= __expf(m - lm); m = lm; }
#pragma unroll
        for (int e = 0; e < 8; ++e) s += __expf(f[e] - m);
      }
    }
    const float M = warp_max(m);
    s = (m == -INFINITY) ? 0.f : s * __expf(m - M);
    const float lse = M + logf(warp_sum(s));
    const float zt = __bfloat162float(zr[t]);
    __syncwarp();
    if (lane == 0) {
      a.row_loss[r] = lse - zt;
      if (!isfinite(lse - zt)) set_soft(kp, kSoftNonFinite);
    }
    for (int j = lane; j < nvec; j += 32 * kU) {
      uint4 u[kU];
#pragma unroll
      for (int q = 0; q < kU; ++q)
        if (j + 32 * q < nvec) u[q] = z[j + 32 * q];
#pragma unroll
      for (int q = 0; q < kU; ++q) {
        const int jq = j + 32 * q;
        if (jq >= nvec) break;
        float f[8];
        bf16x8_to_f(u[q], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float p = __expf(f[e] - lse);
          if (jq * 8 + e == t) p -= 1.0f;
          f[e] = p * invN;
        }
        z[jq] = f_to_bf16x8(f);
      }
    }
  }
}

// Staged variant (bf16, two rows of V logits fit in shared memory): one thread
// bulk-copies each row into one of two buffers, the next row while this one is
// processed; the whole block reduces the row (its maximum, then the sum of
// exp(z - max), each combined over the eight warps in a fixed order) and writes dz
// back with 16-byte coalesced stores.  A logit is read from memory once instead of twice.
// The row copies complete on the bars shared with AdamW (iter counts their
// phases); every copy issued here is also waited for here.
__device__ inline void task_ce_bf16_staged(const KParams& kp, const CeArgs& a, int idx, uint8_t* smem,
                                           uint64_t* bars, uint32_t* iter) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = idx * a.rows_per_task, r1 = min(r0 + a.rows_per_task, a.N);
  const int nrows = r1 - r0;
  const float invN = 1.0f / (float)a.N;
  const int nvec = a.V >> 3;
  const uint32_t row_bytes = (uint32_t)a.V * 2u;
  const uint32_t buf_stride = (row_bytes + 127u) & ~127u;
  float2* red = reinterpret_cast<float2*>(smem + 2 * buf_stride);  // [kWarps] (max, sum)
  const uint32_t it0 = *iter;
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem);
  const uint32_t bar0 = (uint32_t)__cvta_generic_to_shared(bars);
  const __nv_bfloat16* logits = reinterpret_cast<const __nv_bfloat16*>(a.logits);
  auto issue = [&](int k) {  // one thread: row r0 + k into buffer k & 1
    const uint32_t bar = bar0 + 8 * ((it0 + (uint32_t)k) % kAdamStages);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(row_bytes) : "memory");
    bulk_load(sbase + (uint32_t)(k & 1) * buf_stride, logits + (int64_t)(r0 + k) * a.V, row_bytes, bar);
  };
  if (threadIdx.x == 0) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // earlier generic use of the buffers
    for (int k = 0; k < min(nrows, 2); ++k) issue(k);
  }
  for (int k = 0; k < nrows; ++k) {
    const int r = r0 + k;
    const uint32_t st = (it0 + (uint32_t)k) % kAdamStages;
    const uint32_t phase = ((it0 + (uint32_t)k) / kAdamStages) & 1u;
    // every thread leaves together when a wait fails (no thread may be left
    // behind at a later barrier of this task)
    if (!__syncthreads_and(mbar_wait(kp, bar0 + 8 * st, phase))) return;
    const uint4* z = reinterpret_cast<const uint4*>(smem + (k & 1) * buf_stride);
    int t = step_targets(kp)[r];
    if (t < 0 || t >= a.V) {
      if (threadIdx.x == 0) set_soft(kp, kSoftBadToken);
      t = t < 0 ? 0 : a.V - 1;
    }
    // Three passes over the staged row, each with independent per-lane work (no
    // loop-carried chain through an exponential): the row maximum, the sum of
    // exp(z - max) in eight accumulators, then the gradient below.  Reductions run
    // in a fixed order (xor tree in the warp, warps in order).
    float m8[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 4
    for (int j = threadIdx.x; j < nvec; j += kThreads) {
      float f[8];
      bf16x8_to_f(z[j], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) m8[e & 3] = fmaxf(m8[e & 3], f[e]);
    }
    float m = fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp].x = m;
    __syncthreads();
    float M = red[0].x;
#pragma unroll
    for (int w = 1; w < kWarps; ++w) M = fmaxf(M, red[w].x);
    constexpr float kLog2e = 1.4426950408889634f;
    const float M2 = M * kLog2e;  // exp(z - M) = 2^(z log2 e - M log2 e)
    float s8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int j = threadIdx.x; j < nvec; j += kThreads) {
      float f[8];
      bf16x8_to_f(z[j], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) s8[e] += ex2_sfu(fmaf(f[e], kLog2e, -M2));
    }
    float s = ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) red[warp].y = s;
    __syncthreads();
    float S = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) S += red[w].y;
    const float lse = M + logf(S);
    const float lse2 = lse * kLog2e;
    if (threadIdx.x == 0) {
      const float zt = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(z)[t]);
      a.row_loss[r] = lse - zt;
      if (!isfinite(lse - zt)) set_soft(kp, kSoftNonFinite);
    }
    uint4* dz = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.logits) + (int64_t)r * a.V);
#pragma unroll 4
    for (int j = threadIdx.x; j < nvec; j += kThreads) {
      float f[8];
      bf16x8_to_f(z[j], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float p = ex2_sfu(fmaf(f[e], kLog2e, -lse2));
        if (j * 8 + e == t) p -= 1.0f;
        f[e] = p * invN;
      }
      dz[j] = f_to_bf16x8(f);
    }
    __syncthreads();  // buffer k & 1 and red[] are free again
    if (threadIdx.x == 0 && k + 2 < nrows) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(k + 2);
    }
  }
  if (threadIdx.x == 0) *iter = it0 + (uint32_t)nrows;
}

// loss = (1/N) sum_n row_loss[n], fixed order; flags a non-finite loss.
__device__ inline void task_loss(const KParams& kp, const LossArgs& a, float* smem) {
  float s = 0.f;
  for (int i = threadIdx.x; i < a.N; i += kThreads) s += a.row_loss[i];
  smem[threadIdx.x] = s;
  __syncthreads();
  for (int w = kThreads / 2; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) smem[threadIdx.x] += smem[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const float loss = smem[0] / (float)a.N;
    *a.loss = loss;
    if (!isfinite(loss)) set_soft(kp, kSoftNonFinite);
    // multi-step calls: the loss and the soft error bits of this step (every
    // cross-entropy row, which raises them, precedes this task) into the rings
    if (kp.loss_out) kp.loss_out[g_step] = loss;
    if (kp.status_out) kp.status_out[g_step] = ld_volatile_u32(&kp.err[1]);
  }
}

// dst[c] = sum_r src[r, c] for a chunk of columns; warp w sums rows w, w+8, ...,
// then the warps' partials are added in warp order.
template <typename act_t>
__device__ inline void task_colsum(const ColsumArgs& a, int idx, float* smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = idx * a.cols_per_task;
  const int ncol = min(a.cols_per_task, a.cols - c0);  // <= 64
  float acc0 = 0.f, acc1 = 0.f;
  const bool has0 = lane < ncol, has1 = lane + 32 < ncol;
  constexpr int U = 8;  // rows of one warp in flight
  if (a.src_f32) {
    const float* src = reinterpret_cast<const float*>(a.src) + c0;
    int r = warp;
    for (; r + (U - 1) * kWarps < a.rows; r += U * kWarps) {
      float x0[U], x1[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float* row = src + (int64_t)(r + u * kWarps) * a.ld;
        x0[u] = has0 ? row[lane] : 0.f;
        x1[u] = has1 ? row[lane + 32] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) { acc0 += x0[u]; acc1 += x1[u]; }
    }
    for (; r < a.rows; r += kWarps) {
      const float* row = src + (int64_t)r * a.ld;
      if (has0) acc0 += row[lane];
      if (has1) acc1 += row[lane + 32];
    }
  } else {
    const act_t* src = reinterpret_cast<const act_t*>(a.src) + c0;
    int r = warp;
    for (; r + (U - 1) * kWarps < a.rows; r += U * kWarps) {
      float x0[U], x1[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const act_t* row = src + (int64_t)(r + u * kWarps) * a.ld;
        x0[u] = has0 ? to_f<act_t>(row[lane]) : 0.f;
        x1[u] = has1 ? to_f<act_t>(row[lane + 32]) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) { acc0 += x0[u]; acc1 += x1[u]; }
    }
    for (; r < a.rows; r += kWarps) {
      const act_t* row = src + (int64_t)r * a.ld;
      if (has0) acc0 += to_f<act_t>(row[lane]);
      if (has1) acc1 += to_f<act_t>(row[lane + 32]);
    }
  }
  smem[warp * 64 + lane] = acc0;
  smem[warp * 64 + lane + 32] = acc1;
  __syncthreads();
  if ((int)threadIdx.x < ncol) {
    float s = 0.f;
    for (int w = 0; w < kWarps; ++w) s += smem[w * 64 + threadIdx.x];
    a.dst[c0 + threadIdx.x] = s;
  }
}

// Stable sort of the step's (token, position) pairs by token id, one block:
// least-significant-digit radix sort with 8-bit digits in shared memory.  The
// digit counts come from shared-memory atomics (order-free); the scatter walks
// the elements in order on one warp, ranking equal digits with __match_any_sync,
// so equal tokens keep increasing positions.
__device__ inline void task_token_sort(const KParams& kp, const EmbedArgs& a, int* smem) {
  const int N = a.N;
  int* ka = smem;
  int* va = ka + N;
  int* kb = va + N;
  int* vb = kb + N;
  int* hist = vb + N;  // [256]
  for (int n = threadIdx.x; n < N; n += kThreads) {
    int t = step_tokens(kp)[n];
    ka[n] = t < 0 ? 0 : (t >= a.V ? a.V - 1 : t);
    va[n] = n;
  }
  const int passes = a.V <= 256 ? 1 : (a.V <= 65536 ? 2 : 3);
  for (int pass = 0; pass < passes; ++pass) {
    const int shift = 8 * pass;
    for (int i = threadIdx.x; i < 256; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int n = threadIdx.x; n < N; n += kThreads) atomicAdd(&hist[(ka[n] >> shift) & 255], 1);
    __syncthreads();
    if (threadIdx.x == 0) {
      int run = 0;
      for (int i = 0; i < 256; ++i) { const int c = hist[i]; hist[i] = run; run += c; }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      const unsigned lt = (1u << lane) - 1u;
      for (int c0 = 0; c0 < N; c0 += 32) {
        const int n = c0 + lane;
        const bool live = n < N;
        const int key = live ? ka[n] : 0;
        const int d = live ? (key >> shift) & 255 : 256 + lane;  // dead lanes never match
        const unsigned peers = __match_any_sync(0xffffffffu, d);
        const int rank = __popc(peers & lt);
        const int base = live ? hist[d] : 0;
        __syncwarp();
        if (live) {
          kb[base + rank] = key;
          vb[base + rank] = va[n];
          if (rank == 0) hist[d] = base + __popc(peers);
        }
        __syncwarp();
      }
    }
    __syncthreads();
    int* t0 = ka; ka = kb; kb = t0;
    int* t1 = va; va = vb; vb = t1;
  }
  for (int n = threadIdx.x; n < N; n += kThreads) {
    a.sorted_tok[n] = ka[n];
    a.sorted_pos[n] = va[n];
  }
  // first sorted entry of every block of rows_per_task vocabulary rows
  const int nblk = (a.V + a.rows_per_task - 1) / a.rows_per_task;
  for (int n = threadIdx.x; n <= N; n += kThreads) {
    const int bprev = n == 0 ? -1 : ka[n - 1] / a.rows_per_task;
    const int bcur = n == N ? nblk : ka[n] / a.rows_per_task;
    for (int b = bprev + 1; b <= bcur; ++b) a.block_start[b] = n;
  }
}

// dwte[v] = sum over positions n with tok[n] = v of dx0[n] (in increasing n),
// for a block of vocabulary rows; rows no token hit are written as zeros.  The
// block's entries of the sorted token list are found by binary search.
__device__ __forceinline__ int lower_bound_i32(const int* a, int n, int key) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] < key) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// dwte[v] = sum of dx0 over the occurrences of token v, for a block of vocabulary
// rows [v0, v1), from the task's slice of the token-sorted positions (stok: the
// slice's token ids in shared memory).  Rows with fewer than kHotRow occurrences
// are summed by one warp each, four occurrences in flight; a hot row (Zipf-
// distributed tokens put hundreds of occurrences on the first few ids) is split
// over all warps in contiguous slices whose partial sums are then added in warp
// order — a fixed order, so the result is the same in every step.
constexpr int kHotRow = 32;

template <int NV>
__device__ __forceinline__ void wte_row_sum(const EmbedArgs& a, int i0, int j0, int j1, int lane, float4* acc) {
#pragma unroll
  for (int i = 0; i < NV; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  int j = j0;
  for (; j + 4 <= j1; j += 4) {  // four rows' loads in flight, added in order
    const float4* s0 = reinterpret_cast<const float4*>(a.dx0 + (int64_t)a.sorted_pos[i0 + j] * a.C);
    const float4* s1 = reinterpret_cast<const float4*>(a.dx0 + (int64_t)a.sorted_pos[i0 + j + 1] * a.C);
    const float4* s2 = reinterpret_cast<const float4*>(a.dx0 + (int64_t)a.sorted_pos[i0 + j + 2] * a.C);
    const float4* s3 = reinterpret_cast<const float4*>(a.dx0 + (int64_t)a.sorted_pos[i0 + j + 3] * a.C);
    float4 x0[NV], x1[NV], x2[NV], x3[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      x0[i] = s0[lane + 32 * i]; x1[i] = s1[lane + 32 * i]; x2[i] = s2[lane + 32 * i]; x3[i] = s3[lane + 32 * i];
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      acc[i].x += x0[i].x; acc[i].y += x0[i].y; acc[i].z += x0[i].z; acc[i].w += x0[i].w;
      acc[i].x += x1[i].x; acc[i].y += x1[i].y; acc[i].z += x1[i].z; acc[i].w += x1[i].w;
      acc[i].x += x2[i].x; acc[i].y += x2[i].y; acc[i].z += x2[i].z; acc[i].w += x2[i].w;
      acc[i].x += x3[i].x; acc[i].y += x3[i].y; acc[i].z += x3[i].z; acc[i].w += x3[i].w;
    }
  }
  for (; j < j1; ++j) {
    const float4* src = reinterpret_cast<const float4*>(a.dx0 + (int64_t)a.sorted_pos[i0 + j] * a.C);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const float4 x = src[lane + 32 * i];
      acc[i].x += x.x; acc[i].y += x.y; acc[i].z += x.z; acc[i].w += x.w;
    }
  }
}

template <int NV>
__device__ __forceinline__ void wte_rows(const EmbedArgs& a, int v0, int v1, int i0, const int* stok, int nseg,
                                         float* part) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if constexpr (NV > 0) {
    for (int v = v0 + warp; v < v1; v += kWarps) {
      const int j0 = lower_bound_i32(stok, nseg, v), j1 = lower_bound_i32(stok, nseg, v + 1);
      if (j1 - j0 >= kHotRow) continue;  // below, by the whole block
      if (a.accumulate && j1 == j0) continue;  // no occurrence: the LM-head part stays as it is
      float4 acc[NV];
      wte_row_sum<NV>(a, i0, j0, j1, lane, acc);
      float4* dst = reinterpret_cast<float4*>(a.dwte + (int64_t)v * a.C);
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        if (a.accumulate) {
          const float4 o = dst[lane + 32 * i];
          acc[i].x += o.x; acc[i].y += o.y; acc[i].z += o.z; acc[i].w += o.w;
        }
        dst[lane + 32 * i] = acc[i];
      }
    }
    for (int v = v0; v < v1; ++v) {  // every thread sees the same counts: uniform branches
      const int j0 = lower_bound_i32(stok, nseg, v), j1 = lower_bound_i32(stok, nseg, v + 1);
      if (j1 - j0 < kHotRow) continue;
      const int per = (j1 - j0 + kWarps - 1) / kWarps;
      const int w0 = min(j1, j0 + warp * per), w1 = min(j1, w0 + per);
      float4 acc[NV];
      wte_row_sum<NV>(a, i0, w0, w1, lane, acc);
#pragma unroll
      for (int i = 0; i < NV; ++i) reinterpret_cast<float4*>(part + warp * a.C)[lane + 32 * i] = acc[i];
      __syncthreads();
      for (int c = threadIdx.x; c < a.C; c += kThreads) {
        float s = part[c];
        for (int w = 1; w < kWarps; ++w) s += part[w * a.C + c];
        if (a.accumulate) s += a.dwte[(int64_t)v * a.C + c];
        a.dwte[(int64_t)v * a.C + c] = s;
      }
      __syncthreads();
    }
  } else {
    for (int v = v0 + warp; v < v1; v += kWarps) {
      const int jb = lower_bound_i32(stok, nseg, v);
      float* dst = a.dwte + (int64_t)v * a.C;
      if (a.accumulate && (jb >= nseg || stok[jb] != v)) continue;  // no occurrence
      for (int c = lane; c < a.C; c += 32) {
        float s = 0.f;
        for (int j = jb; j < nseg && stok[j] == v; ++j) s += a.dx0[(int64_t)a.sorted_pos[i0 + j] * a.C + c];
        dst[c] = a.accumulate ? dst[c] + s : s;
      }
    }
  }
}

__device__ inline void task_embed_bwd_wte(const KParams& kp, const EmbedArgs& a, int idx, int* smem) {
  (void)kp;
  const int v0 = idx * a.rows_per_task, v1 = min(v0 + a.rows_per_task, a.V);
  const int i0 = a.block_start[idx], nseg = a.block_start[idx + 1] - i0;
  int* stok = smem;
  float* part = reinterpret_cast<float*>(smem + ((a.N + 3) & ~3));  // [kWarps][C], after a slice of at most N ids
  for (int j = threadIdx.x; j < nseg; j += kThreads) stok[j] = a.sorted_tok[i0 + j];
  __syncthreads();
  switch ((a.C & 127) ? 0 : a.C >> 7) {
    case 2: wte_rows<2>(a, v0, v1, i0, stok, nseg, part); break;
    case 4: wte_rows<4>(a, v0, v1, i0, stok, nseg, part); break;
    case 6: wte_rows<6>(a, v0, v1, i0, stok, nseg, part); break;
    case 8: wte_rows<8>(a, v0, v1, i0, stok, nseg, part); break;
    default: wte_rows<0>(a, v0, v1, i0, stok, nseg, part); break;
  }
}

// dwpe[t] = sum_b dx0[b, t] for a block of positions.
__device__ inline void task_embed_bwd_wpe(const EmbedArgs& a, int idx) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = idx * a.rows_per_task, t1 = min(t0 + a.rows_per_task, a.T);
  for (int t = t0 + warp; t < t1; t += kWarps) {
    for (int c = lane; c < a.C; c += 32) {
      float s = 0.f;
      for (int b = 0; b < a.B; ++b) s += a.dx0[((int64_t)b * a.T + t) * a.C + c];
      a.dwpe[(int64_t)t * a.C + c] = s;
    }
  }
}

// AdamW on one chunk of a parameter tensor (decoupled weight decay first):
// p *= 1 - lr wd; m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2;
// p -= lr (m / bc1) / (sqrt(v / bc2) + eps); bf16 copy of p written if requested.
// The chunk streams through shared memory in sub-chunks of kAdamSub parameters:
// one thread issues 1-D bulk copies (cp.async.bulk, completion counted on an
// mbarrier) of p, g, m and v for kAdamStages - 1 sub-chunks ahead, all threads
// update a staged sub-chunk in place, and bulk stores write p, m, v and the bf16
// copy back — about 180 KB in flight per SM without spending registers on it.
// iter: this block's count of sub-chunks so far (stage = iter mod kAdamStages,
// phase = (iter / kAdamStages) mod 2), shared by the block's threads.
__device__ inline void task_adamw(const KParams& kp, const AdamArgs& a, int idx, uint8_t* smem, uint64_t* bars,
                                  uint32_t* iter) {
  // The loss task may raise the flag while this task runs: thread 0 reads it
  // once for the whole block, so all threads take the same branch.
  if (__syncthreads_or(threadIdx.x == 0 && (ld_volatile_u32(&kp.err[1]) & (kSoftBadToken | kSoftNonFinite)))) return;
  const int64_t lo = (int64_t)idx * a.chunk;
  const int64_t hi = min(lo + a.chunk, a.n);
  const int nsub = (int)((hi - lo + kAdamSub - 1) / kAdamSub);
  const uint32_t it0 = *iter;
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem);
  const uint32_t bar0 = (uint32_t)__cvta_generic_to_shared(bars);
  auto stage_of = [&](int s) { return (it0 + (uint32_t)s) % kAdamStages; };
  auto count_of = [&](int s) {
    const int64_t rest = hi - (lo + (int64_t)s * kAdamSub);
    return (int)(rest < kAdamSub ? rest : (int64_t)kAdamSub);
  };
  auto issue = [&](int s) {  // one thread
    const uint32_t st = stage_of(s);
    const int64_t base = lo + (int64_t)s * kAdamSub;
    const uint32_t bytes = (uint32_t)count_of(s) * 4u;
    const uint32_t buf = sbase + st * kAdamStageBytes;
    const uint32_t bar = bar0 + 8 * st;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(4 * bytes) : "memory");
    bulk_load(buf, a.p + base, bytes, bar);
    bulk_load(buf + kAdamSub * 4, a.g + base, bytes, bar);
    bulk_load(buf + kAdamSub * 8, a.m + base, bytes, bar);
    bulk_load(buf + kAdamSub * 12, a.v + base, bytes, bar);
  };
  // Sub-chunk s lives in stage (iter + s) mod kAdamStages.  Loads run
  // kAdamStages - 1 sub-chunks ahead: the load of s + kAdamStages - 1 goes into
  // the stage that sub-chunk s - 1 used, whose bulk stores (committed one
  // iteration earlier) have normally finished reading it already.
  constexpr int kAhead = kAdamStages - 1;
  if (threadIdx.x == 0) {
    bulk_wait_read_all();  // earlier bulk stores have finished reading these buffers
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    for (int s = 0; s < min(nsub, kAhead); ++s) issue(s);
  }
  const float decay = 1.0f - step_lr(kp) * kp.wd * a.decay;
  const AdamHyper hp = adam_hyper(kp);
  for (int s = 0; s < nsub; ++s) {
    const uint32_t st = stage_of(s);
    const uint32_t phase = ((it0 + (uint32_t)s) / kAdamStages) & 1u;
    if (!__syncthreads_and(mbar_wait(kp, bar0 + 8 * st, phase))) return;  // all threads leave together
    uint8_t* buf = smem + st * kAdamStageBytes;
    float4* P = reinterpret_cast<float4*>(buf);
    const float4* G = reinterpret_cast<const float4*>(buf + kAdamSub * 4);
    float4* Mo = reinterpret_cast<float4*>(buf + kAdamSub * 8);
    float4* Vo = reinterpret_cast<float4*>(buf + kAdamSub * 12);
    uint2* S = reinterpret_cast<uint2*>(buf + kAdamSub * 16);
    const int cnt4 = count_of(s) / 4;
    for (int i = threadIdx.x; i < cnt4; i += kThreads) {
      const float4 p = P[i], g = G[i], m = Mo[i], v = Vo[i];
      float pp[4] = {p.x, p.y, p.z, p.w}, gg[4] = {g.x, g.y, g.z, g.w};
      float mm[4] = {m.x, m.y, m.z, m.w}, vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) adamw_elem(hp, decay, gg[e], pp[e], mm[e], vv[e]);
      P[i] = make_float4(pp[0], pp[1], pp[2], pp[3]);
      Mo[i] = make_float4(mm[0], mm[1], mm[2], mm[3]);
      Vo[i] = make_float4(vv[0], vv[1], vv[2], vv[3]);
      if (a.shadow) {
        __nv_bfloat162 lo2 = __floats2bfloat162_rn(pp[0], pp[1]);
        __nv_bfloat162 hi2 = __floats2bfloat162_rn(pp[2], pp[3]);
        S[i] = make_uint2(*reinterpret_cast<uint32_t*>(&lo2), *reinterpret_cast<uint32_t*>(&hi2));
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic smem writes -> bulk stores
    __syncthreads();
    if (threadIdx.x == 0) {
      const int64_t base = lo + (int64_t)s * kAdamSub;
      const uint32_t bytes = (uint32_t)count_of(s) * 4u;
      const uint32_t sb = sbase + st * kAdamStageBytes;
      bulk_store(a.p + base, sb, bytes);
      bulk_store(a.m + base, sb + kAdamSub * 8, bytes);
      bulk_store(a.v + base, sb + kAdamSub * 12, bytes);
      if (a.shadow) bulk_store(a.shadow + base, sb + kAdamSub * 16, bytes / 2);
      bulk_commit();
      if (s + kAhead < nsub) {
        asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");  // sub-chunk s - 1's stores have read its stage
        issue(s + kAhead);
      }
    }
  }
  if (threadIdx.x == 0) {
    // Nothing later in the step reads an AdamW result, so only the staging
    // buffers need to be free before the next task; the stores to global memory
    // drain in the background (the kernel waits for them before it exits).
    bulk_wait_read_all();
    *iter = it0 + (uint32_t)nsub;
  }
}

}  // namespace pgs
