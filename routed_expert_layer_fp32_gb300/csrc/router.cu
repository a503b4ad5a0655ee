// Router: logits = x Wr^T + b in fp32, then top-k selection with the lowest index winning
// ties and the softmax renormalised over the selected experts.
// Layer definition: "We Ported Aleph Alpha's Kolibri to a MacBook. Our Own Gate Said No.",
// section "The gate" (384 experts scored per token in float32, top 6) and section 1
// (score plus a per-expert bias; forced ids replayed from a free run).
#include "common.cuh"

namespace moe {
namespace {

__device__ __forceinline__ void load4(const float* x, float (&v)[4]) {
  float4 f = *reinterpret_cast<const float4*>(x);
  v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* x, float (&v)[4]) {
  uint2 u = *reinterpret_cast<const uint2*>(x);
  v[0] = __uint_as_float(u.x << 16);
  v[1] = __uint_as_float(u.x & 0xffff0000u);
  v[2] = __uint_as_float(u.y << 16);
  v[3] = __uint_as_float(u.y & 0xffff0000u);
}

// Decode-sized router: one warp per expert, tokens in groups of 8.  Each lane owns the
// k-positions {4*lane + 128*j}; the warp sums its lanes at the end.
template <typename XT>
__global__ void __launch_bounds__(256) k_router_warp(const XT* __restrict__ x, int T, int d, int E,
                                                     const float* __restrict__ Wr, const float* __restrict__ bias,
                                                     float* __restrict__ logits) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp;
  if (e >= E) return;
  const float* wr = Wr + size_t(e) * d;
  const float b = bias ? bias[e] : 0.0f;
  for (int t0 = 0; t0 < T; t0 += 8) {
    const int nt = min(8, T - t0);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int k = lane * 4; k < d; k += 128) {
      float w[4];
      load4(wr + k, w);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (i < nt) {
          float xv[4];
          load4(x + size_t(t0 + i) * d + k, xv);
          acc[i] = fmaf(xv[0], w[0], acc[i]);
          acc[i] = fmaf(xv[1], w[1], acc[i]);
          acc[i] = fmaf(xv[2], w[2], acc[i]);
          acc[i] = fmaf(xv[3], w[3], acc[i]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float s = warp_sum(acc[i]);
      if (lane == 0 && i < nt) logits[size_t(t0 + i) * E + e] = s + b;
    }
  }
}

// Decode-sized router (T <= kRouterSplitMaxT): split over k so that every SM gets work.
// CTA (expert block of 32, k-slice of 128) stages Wr[32][128] and x[T][128] in shared
// memory and writes partial sums part[slice][t][e].  The last CTA of an expert block to
// finish (a counter in the status record, reset after use) adds the slices in slice order
// plus the bias, so the logits do not depend on which CTA finished last.
constexpr int kRsE = 32, kRsK = kRouterSplitK;
constexpr int kMaxRouterSlices = 2048 / kRouterSplitK;  // d <= 2048 on the split path
template <typename XT>
__global__ void __launch_bounds__(256) k_router_split(const XT* __restrict__ x, int T, int d, int E,
                                                      const float* __restrict__ Wr, const float* __restrict__ bias,
                                                      float* __restrict__ part, float* __restrict__ logits,
                                                      DevStatus* st) {
  __shared__ unsigned s_last;
  extern __shared__ __align__(16) float rs_smem[];
  float (*ws)[kRsK + 4] = reinterpret_cast<float (*)[kRsK + 4]>(rs_smem);
  float (*xs)[kRsK + 4] = reinterpret_cast<float (*)[kRsK + 4]>(rs_smem + kRsE * (kRsK + 4));
  const int e0 = blockIdx.x * kRsE, k0 = blockIdx.y * kRsK;
  const int tid = threadIdx.x;
  // Wr slice: 32 rows x 128 floats, float4 per thread per pass
  for (int i = tid; i < kRsE * kRsK / 4; i += blockDim.x) {
    const int r = i / (kRsK / 4), c = (i % (kRsK / 4)) * 4;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (e0 + r < E) load4(Wr + size_t(e0 + r) * d + k0 + c, v);
    *reinterpret_cast<float4*>(&ws[r][c]) = make_float4(v[0], v[1], v[2], v[3]);
  }
  for (int i = tid; i < T * kRsK / 4; i += blockDim.x) {
    const int t = i / (kRsK / 4), c = (i % (kRsK / 4)) * 4;
    float v[4];
    load4(x + size_t(t) * d + k0 + c, v);
    *reinterpret_cast<float4*>(&xs[t][c]) = make_float4(v[0], v[1], v[2], v[3]);
  }
  __syncthreads();
  const int e = tid & 31, tg = tid >> 5;  // lane = expert, warp = token group (t = tg + 8j)
  constexpr int kMaxJ = kRouterSplitMaxT / 8;
  float acc[kMaxJ];
#pragma unroll
  for (int j = 0; j < kMaxJ; ++j) acc[j] = 0.0f;
#pragma unroll 4
  for (int c = 0; c < kRsK; c += 4) {
    const float4 wv = *reinterpret_cast<const float4*>(&ws[e][c]);
#pragma unroll
    for (int j = 0; j < kMaxJ; ++j) {
      const int t = tg + 8 * j;
      if (t < T) {
        const float4 xv = *reinterpret_cast<const float4*>(&xs[t][c]);
        acc[j] = fmaf(xv.x, wv.x, acc[j]);
        acc[j] = fmaf(xv.y, wv.y, acc[j]);
        acc[j] = fmaf(xv.z, wv.z, acc[j]);
        acc[j] = fmaf(xv.w, wv.w, acc[j]);
      }
    }
  }
  if (e0 + e < E) {
#pragma unroll
    for (int j = 0; j < kMaxJ; ++j) {
      const int t = tg + 8 * j;
      if (t < T) part[(size_t(blockIdx.y) * T + t) * E + e0 + e] = acc[j];
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&st->router_done[blockIdx.x], 1u) == gridDim.y - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int n_part = gridDim.y;  // <= kMaxRouterSlices
  for (int i = tid; i < T * kRsE; i += blockDim.x) {
    const int t = i / kRsE, ee = e0 + i % kRsE;
    if (ee >= E) continue;
    float v[kMaxRouterSlices];
#pragma unroll
    for (int p = 0; p < kMaxRouterSlices; ++p) v[p] = p < n_part ? __ldcg(part + (size_t(p) * T + t) * E + ee) : 0.0f;
    float sum = v[0];
#pragma unroll
    for (int p = 1; p < kMaxRouterSlices; ++p)
      if (p < n_part) sum += v[p];
    logits[size_t(t) * E + ee] = sum + (bias ? bias[ee] : 0.0f);
  }
  if (tid == 0) st->router_done[blockIdx.x] = 0;
}

// Prefill-sized router: SIMT tiled GEMM, 64 tokens x 64 experts per CTA, 4x4 per thread.
template <typename XT>
__global__ void __launch_bounds__(256) k_router_gemm(const XT* __restrict__ x, int T, int d, int E,
                                                     const float* __restrict__ Wr, const float* __restrict__ bias,
                                                     float* __restrict__ logits) {
  constexpr int BM = 64, BN = 64, BK = 16;
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const int tid = threadIdx.x;
  const int t0 = blockIdx.y * BM, e0 = blockIdx.x * BN;
  const int tr = tid / 16, tc = tid % 16;  // 16 x 16 threads, 4 x 4 outputs each
  float acc[4][4] = {};
  // loader mapping: 64 rows x 16 k = 1024 elements = 256 threads x 4 (one float4 along k)
  const int lr = tid / 4, lk = (tid % 4) * 4;
  for (int k0 = 0; k0 < d; k0 += BK) {
    float xv[4] = {0.f, 0.f, 0.f, 0.f}, wv[4] = {0.f, 0.f, 0.f, 0.f};
    if (t0 + lr < T) load4(x + size_t(t0 + lr) * d + k0 + lk, xv);
    if (e0 + lr < E) load4(Wr + size_t(e0 + lr) * d + k0 + lk, wv);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      As[lk + j][lr] = xv[j];
      Bs[lk + j][lr] = wv[j];
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][tr * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tc * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + tr * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tc * 4 + j;
      if (e < E) logits[size_t(t) * E + e] = acc[i][j] + (bias ? bias[e] : 0.0f);
    }
  }
}

// "a is preferred over b": larger logit, or equal logit and lower index.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Selection: one warp per token.  Free routing picks k rounds of the preferred remaining
// expert (softmax is monotone in the logit, so selecting on logits selects on
// probabilities); forced routing validates the given ids.  Weights: softmax over the k
// selected logits, or forced_w as given.
__global__ void __launch_bounds__(256) k_select(const float* __restrict__ logits,
                                                const int32_t* __restrict__ forced_ids,
                                                const float* __restrict__ forced_w, int T, int E, int k,
                                                int32_t* __restrict__ ids, float* __restrict__ w, DevStatus* st) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  // lane-local logits of experts lane + 32 j
  constexpr int kPer = kMaxExperts / 32;
  float v[kPer];
  if (!(forced_ids && forced_w)) {
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int e = lane + 32 * j;
      v[j] = e < E ? logits[size_t(t) * E + e] : -INFINITY;
    }
  }
  int sel = -1;     // lane i < k holds slot i's expert
  float lsel = 0.f; // and its logit
  if (forced_ids) {
    int e = lane < k ? forced_ids[size_t(t) * k + lane] : -1;
    bool bad = lane < k && (e < 0 || e >= E);
    // a repeat of an earlier slot's id is rejected too
    for (int j = 0; j < k; ++j) {
      int ej = __shfl_sync(0xffffffffu, e, j);
      if (lane < k && j < lane && ej == e) bad = true;
    }
    unsigned badmask = __ballot_sync(0xffffffffu, bad);
    if (badmask && lane == 0) {
      set_status(st, kFlagBadForced);
      atomicAdd(&st->bad_forced, __popc(badmask));
    }
    sel = (lane < k && !bad) ? e : -1;
    if (forced_w) {
      if (lane < k) {
        ids[size_t(t) * k + lane] = sel;
        w[size_t(t) * k + lane] = sel >= 0 ? forced_w[size_t(t) * k + lane] : 0.0f;
      }
      return;
    }
    // each forced expert's logit, fetched from the lane that holds it
    for (int i = 0; i < k; ++i) {
      const int ei = __shfl_sync(0xffffffffu, sel, i);
      float li = 0.0f;
      if (ei >= 0) {
#pragma unroll
        for (int j = 0; j < kPer; ++j)
          if (ei == lane + 32 * j) li = v[j];
        li = __shfl_sync(0xffffffffu, li, ei & 31);
      }
      if (lane == i) lsel = li;
    }
  } else {
    unsigned taken = 0;
    for (int r = 0; r < k; ++r) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int e = lane + 32 * j;
        if (e < E && !(taken >> j & 1u) && better(v[j], e, bv, bi)) { bv = v[j]; bi = e; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == r) { sel = bi; lsel = bv; }
    }
  }
  // softmax over the valid selected logits, summed in slot order
  float m = -INFINITY;
  for (int j = 0; j < k; ++j) {
    int ej = __shfl_sync(0xffffffffu, sel, j);
    float lj = __shfl_sync(0xffffffffu, lsel, j);
    if (ej >= 0) m = fmaxf(m, lj);
  }
  float ex = (sel >= 0 && lane < k) ? expf(lsel - m) : 0.0f;
  float s = 0.0f;
  for (int j = 0; j < k; ++j) s += __shfl_sync(0xffffffffu, ex, j);
  if (lane < k) {
    ids[size_t(t) * k + lane] = sel;
    w[size_t(t) * k + lane] = sel >= 0 ? ex / s : 0.0f;
  }
}

}  // namespace

cudaError_t launch_router_logits(const void* x, bool x_bf16, int T, const LayerDev& L, float* logits, cudaStream_t s) {
  if (T <= 32) {
    dim3 grid((L.E + 7) / 8);
    if (x_bf16)
      k_router_warp<__nv_bfloat16><<<grid, 256, 0, s>>>((const __nv_bfloat16*)x, T, L.d, L.E, L.Wr, L.bias, logits);
    else
      k_router_warp<float><<<grid, 256, 0, s>>>((const float*)x, T, L.d, L.E, L.Wr, L.bias, logits);
  } else {
    dim3 grid((L.E + 63) / 64, (T + 63) / 64);
    if (x_bf16)
      k_router_gemm<__nv_bfloat16><<<grid, 256, 0, s>>>((const __nv_bfloat16*)x, T, L.d, L.E, L.Wr, L.bias, logits);
    else
      k_router_gemm<float><<<grid, 256, 0, s>>>((const float*)x, T, L.d, L.E, L.Wr, L.bias, logits);
  }
  return cudaGetLastError();
}

cudaError_t launch_router_split(const void* x, bool x_bf16, int T, const LayerDev& L, float* part, float* logits,
                                DevStatus* st, cudaStream_t s) {
  constexpr int most = (kRsE + kRouterSplitMaxT) * (kRsK + 4) * int(sizeof(float));
  static cudaError_t attr = [] {
    cudaError_t e1 = cudaFuncSetAttribute(k_router_split<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    cudaError_t e2 = cudaFuncSetAttribute(k_router_split<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    return e1 != cudaSuccess ? e1 : e2;
  }();
  if (attr != cudaSuccess) return attr;
  const size_t smem = size_t(kRsE + T) * (kRsK + 4) * sizeof(float);
  dim3 grid((L.E + kRsE - 1) / kRsE, L.d / kRsK);
  if (x_bf16)
    k_router_split<__nv_bfloat16><<<grid, 256, smem, s>>>((const __nv_bfloat16*)x, T, L.d, L.E, L.Wr, L.bias, part,
                                                          logits, st);
  else
    k_router_split<float><<<grid, 256, smem, s>>>((const float*)x, T, L.d, L.E, L.Wr, L.bias, part, logits, st);
  return cudaGetLastError();
}

cudaError_t launch_select(const float* logits, const int32_t* forced_ids, const float* forced_w, int T,
                          const LayerDev& L, int32_t* ids, float* w, DevStatus* st, cudaStream_t s) {
  k_select<<<(T + 7) / 8, 256, 0, s>>>(logits, forced_ids, forced_w, T, L.E, L.k, ids, w, st);
  return cudaGetLastError();
}

}  // namespace moe
