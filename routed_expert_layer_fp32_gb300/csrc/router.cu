// Router: logits = x Wr^T + b in fp32, then top-k selection with the lowest index winning
// ties and the softmax renormalised over the selected experts.
// Layer definition: "We Ported Aleph Alpha's Kolibri to a MacBook. Our Own Gate Said No.",
// section "The gate" (384 experts scored per token in float32, top 6) and section 1
// (score plus a per-expert bias; forced ids replayed from a free run).
#include <cooperative_groups.h>

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

// Decode router without a k split: CTA = kRsmE experts x all T tokens x all of k.  The CTA
// keeps its experts' rows of Wr in shared memory; warp w takes tokens 8w..8w+7, lanes split k
// (lane owns k = 4 lane + 128 j), and warp shuffles sum the lanes in a fixed order, so the
// logits are deterministic.
constexpr int kRsmE = 2;
template <typename XT>
__global__ void __launch_bounds__(512) k_router_small(const XT* __restrict__ x, int T, int d, int E,
                                                      const float* __restrict__ Wr, const float* __restrict__ bias,
                                                      float* __restrict__ logits) {
  pdl_begin();
  extern __shared__ __align__(16) float rsm_w[];  // [kRsmE][d]
  const int e0 = blockIdx.x * kRsmE;
  for (int i = threadIdx.x * 4; i < kRsmE * d; i += blockDim.x * 4) {
    const int r = i / d, c = i % d;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (e0 + r < E) v = *reinterpret_cast<const float4*>(Wr + size_t(e0 + r) * d + c);
    *reinterpret_cast<float4*>(rsm_w + i) = v;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = warp * 8;
  if (t0 >= T) return;
  const int nt = min(8, T - t0);
  float acc[8][kRsmE];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int e = 0; e < kRsmE; ++e) acc[i][e] = 0.0f;
#pragma unroll 4
  for (int k = lane * 4; k < d; k += 128) {
    float w[kRsmE][4];
#pragma unroll
    for (int e = 0; e < kRsmE; ++e) {
      const float4 wv = *reinterpret_cast<const float4*>(rsm_w + e * d + k);
      w[e][0] = wv.x; w[e][1] = wv.y; w[e][2] = wv.z; w[e][3] = wv.w;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < nt) {
        float xv[4];
        load4(x + size_t(t0 + i) * d + k, xv);
#pragma unroll
        for (int e = 0; e < kRsmE; ++e) {
          acc[i][e] = fmaf(xv[0], w[e][0], acc[i][e]);
          acc[i][e] = fmaf(xv[1], w[e][1], acc[i][e]);
          acc[i][e] = fmaf(xv[2], w[e][2], acc[i][e]);
          acc[i][e] = fmaf(xv[3], w[e][3], acc[i][e]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int e = 0; e < kRsmE; ++e) {
      const float sum = warp_sum(acc[i][e]);
      if (lane == 0 && i < nt && e0 + e < E) logits[size_t(t0 + i) * E + e0 + e] = sum + (bias ? bias[e0 + e] : 0.0f);
    }
}

// Decode router, split over k inside thread-block clusters.  CTA (32 experts, 256-wide
// k-slice) stages its slice of Wr (fp32) and of x in shared memory with all threads loading
// at once, computes partial logits [T][32] into its own shared memory, and the n_slice CTAs
// of the cluster (one per k-slice) then sum the partials through distributed shared memory,
// each CTA for a share of the tokens, adding the slices in rank order (deterministic).
constexpr int kRcE = 32, kRcK = 256, kRcThreads = 256;
template <typename XT>
__global__ void __launch_bounds__(kRcThreads) k_router_cluster(const XT* __restrict__ x, int T, int d, int E,
                                                               const float* __restrict__ Wr,
                                                               const float* __restrict__ bias,
                                                               float* __restrict__ logits) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(16) uint8_t rc_smem[];
  float* ws = reinterpret_cast<float*>(rc_smem);                      // [kRcE][kRcK + 4]
  XT* xs = reinterpret_cast<XT*>(ws + kRcE * (kRcK + 4));             // [T][kRcK + 8]
  float* part = reinterpret_cast<float*>(xs + size_t(T) * (kRcK + 8));  // [T][kRcE]
  pdl_begin();
  const int e0 = blockIdx.x * kRcE, k0 = blockIdx.y * kRcK;
  const int tid = threadIdx.x;
  for (int i = tid; i < kRcE * (kRcK / 4); i += kRcThreads) {
    const int r = i / (kRcK / 4), c = (i % (kRcK / 4)) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (e0 + r < E) v = *reinterpret_cast<const float4*>(Wr + size_t(e0 + r) * d + k0 + c);
    *reinterpret_cast<float4*>(ws + r * (kRcK + 4) + c) = v;
  }
  constexpr int kVec = 16 / sizeof(XT);  // elements per 16-byte load
  for (int i = tid; i < T * (kRcK / kVec); i += kRcThreads) {
    const int t = i / (kRcK / kVec), c = (i % (kRcK / kVec)) * kVec;
    *reinterpret_cast<uint4*>(xs + size_t(t) * (kRcK + 8) + c) =
        *reinterpret_cast<const uint4*>(x + size_t(t) * d + k0 + c);
  }
  __syncthreads();
  const int e = tid & 31, tg = tid >> 5;  // lane = expert, warp = tokens tg, tg + 8, ...
  for (int tb = tg; tb < T; tb += 8 * 8) {  // up to 8 tokens per pass
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    for (int c = 0; c < kRcK; c += 4) {
      const float4 wv = *reinterpret_cast<const float4*>(ws + e * (kRcK + 4) + c);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int t = tb + 8 * j;
        if (t < T) {
          float xv[4];
          load4(xs + size_t(t) * (kRcK + 8) + c, xv);
          acc[j] = fmaf(xv[0], wv.x, acc[j]);
          acc[j] = fmaf(xv[1], wv.y, acc[j]);
          acc[j] = fmaf(xv[2], wv.z, acc[j]);
          acc[j] = fmaf(xv[3], wv.w, acc[j]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int t = tb + 8 * j;
      if (t < T) part[t * kRcE + e] = acc[j];
    }
  }
  cluster.sync();
  const int n_slice = int(cluster.num_blocks());
  const int rank = int(cluster.block_rank());
  const int per = (T + n_slice - 1) / n_slice;
  const int t_lo = rank * per, t_hi = min(T, t_lo + per);
  for (int i = tid; i < (t_hi - t_lo) * kRcE; i += kRcThreads) {
    const int t = t_lo + i / kRcE, ee = i % kRcE;
    float sum = 0.0f;
    for (int r = 0; r < n_slice; ++r) sum += cluster.map_shared_rank(part, r)[t * kRcE + ee];
    if (e0 + ee < E) logits[size_t(t) * E + e0 + ee] = sum + (bias ? bias[e0 + ee] : 0.0f);
  }
  cluster.sync();  // no CTA leaves while another still reads its partials
}

// Prefill-sized router: SIMT tiled GEMM, 64 tokens x 64 experts per CTA, 4x4 per thread.
template <typename XT>
__global__ void __launch_bounds__(256) k_router_gemm(const XT* __restrict__ x, int T, int d, int E,
                                                     const float* __restrict__ Wr, const float* __restrict__ bias,
                                                     float* __restrict__ logits) {
  pdl_begin();
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
  pdl_begin();
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
      return launch_pdl(k_router_gemm<__nv_bfloat16>, grid, dim3(256), 0, s, (const __nv_bfloat16*)x, T, L.d, L.E, L.Wr,
                        L.bias, logits);
    return launch_pdl(k_router_gemm<float>, grid, dim3(256), 0, s, (const float*)x, T, L.d, L.E, L.Wr, L.bias, logits);
  }
  return cudaGetLastError();
}

cudaError_t launch_router_cluster(const void* x, bool x_bf16, int T, const LayerDev& L, float* logits, cudaStream_t s) {
  const int n_slice = L.d / kRcK;
  const size_t xel = x_bf16 ? 2 : 4;
  const size_t smem = size_t(kRcE) * (kRcK + 4) * 4 + size_t(T) * (kRcK + 8) * xel + size_t(T) * kRcE * 4;
  static cudaError_t attr = [] {
    const int most = 200 * 1024;
    cudaError_t e1 = cudaFuncSetAttribute(k_router_cluster<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    cudaError_t e2 = cudaFuncSetAttribute(k_router_cluster<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    return e1 != cudaSuccess ? e1 : e2;
  }();
  if (attr != cudaSuccess) return attr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((L.E + kRcE - 1) / kRcE, n_slice);
  cfg.blockDim = dim3(kRcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = 1;
  attrs[0].val.clusterDim.y = n_slice;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  if (x_bf16)
    return cudaLaunchKernelEx(&cfg, k_router_cluster<__nv_bfloat16>, (const __nv_bfloat16*)x, T, L.d, L.E, L.Wr, L.bias,
                              logits);
  return cudaLaunchKernelEx(&cfg, k_router_cluster<float>, (const float*)x, T, L.d, L.E, L.Wr, L.bias, logits);
}

cudaError_t launch_router_small(const void* x, bool x_bf16, int T, const LayerDev& L, float* logits, cudaStream_t s) {
  const size_t smem = size_t(kRsmE) * L.d * sizeof(float);
  static cudaError_t attr = [] {
    const int most = int(kRsmE * 8192 * sizeof(float));
    cudaError_t e1 = cudaFuncSetAttribute(k_router_small<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    cudaError_t e2 = cudaFuncSetAttribute(k_router_small<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    return e1 != cudaSuccess ? e1 : e2;
  }();
  if (attr != cudaSuccess) return attr;
  const int threads = ((T + 7) / 8) * 32;
  const dim3 grid((L.E + kRsmE - 1) / kRsmE);
  if (x_bf16)
    return launch_pdl(k_router_small<__nv_bfloat16>, grid, dim3(threads), smem, s, (const __nv_bfloat16*)x, T, L.d, L.E,
                      L.Wr, L.bias, logits);
  return launch_pdl(k_router_small<float>, grid, dim3(threads), smem, s, (const float*)x, T, L.d, L.E, L.Wr, L.bias,
                    logits);
}

cudaError_t launch_select(const float* logits, const int32_t* forced_ids, const float* forced_w, int T,
                          const LayerDev& L, int32_t* ids, float* w, DevStatus* st, cudaStream_t s) {
  return launch_pdl(k_select, dim3((T + 7) / 8), dim3(256), 0, s, logits, forced_ids, forced_w, T, L.E, L.k, ids, w, st);
}

}  // namespace moe
