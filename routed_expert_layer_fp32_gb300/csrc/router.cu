// Router: logits = x Wr^T + b in fp32, then top-k selection with the lowest index winning
// ties and the softmax renormalised over the selected experts.
// Layer definition: "We Ported Aleph Alpha's Kolibri to a MacBook. Our Own Gate Said No.",
// section "The gate" (384 experts scored per token in float32, top 6) and section 1
// (score plus a per-expert bias; forced ids replayed from a free run).
#include <cooperative_groups.h>

#include "common.cuh"
#include "dispatch_dev.cuh"
#include "select_dev.cuh"

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


// Weights of a forced selection: softmax over the valid selected logits (max subtracted, summed
// in slot order); an invalid slot (sel < 0) gets weight 0.
__device__ __forceinline__ void write_selection(int sel, float lsel, int k, int lane, int32_t* ids_row,
                                                float* w_row) {
  float m = -INFINITY;
  for (int j = 0; j < k; ++j) {
    const int ej = __shfl_sync(0xffffffffu, sel, j);
    const float lj = __shfl_sync(0xffffffffu, lsel, j);
    if (ej >= 0) m = fmaxf(m, lj);
  }
  const float ex = (sel >= 0 && lane < k) ? expf(lsel - m) : 0.0f;
  float s = 0.0f;
  for (int j = 0; j < k; ++j) s += __shfl_sync(0xffffffffu, ex, j);
  if (lane < k) {
    ids_row[lane] = sel;
    w_row[lane] = sel >= 0 ? ex / s : 0.0f;
  }
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

// Decode routers with the selection fused in.  Grid (expert groups of 16, k-slices of 256,
// token blocks of 64); the k-slices of one (expert group, token block) form a thread-block
// cluster.  Each CTA computes partial logits [64 tokens][16 experts] over its k-slice; then
// decode_router_tail sums the cluster's partials and selects.
constexpr int kRdE = 16, kRdK = 256, kRdT = 64, kRdThreads = 256;
static_assert(kRdThreads == kLeanWarps * 32, "the router's CTAs run the one-CTA dispatch");

// Activation quantisation fused into the bf16 decode router: cluster x (expert group x) of a
// token block quantises tokens [q_lo, q_hi) of it.  Each of its CTAs has the max |x| of those
// tokens over its k-slice in amax_part; after the cluster barrier every CTA takes the max over
// the cluster's slices (exact, in any order), forms the scale max/448 (1 for a zero row) and
// writes the E4M3 codes of its own slice, as the stand-alone quantisation kernel does.
struct XQuant {
  const __nv_bfloat16* xs;  // this CTA's staged x slice [kRdT][xs_ld]
  int xs_ld;
  const float* amax_part;   // [q_hi - q_lo] partial max |x| of this CTA's slice
  uint8_t* xq;              // [T, d] token order; nullptr: no fused quantisation
  float* sx;                // [T]
  int d, k0, q_lo, q_hi;
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    v[2 * j] = __uint_as_float(w[j] << 16);
    v[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
  }
}

// Cluster rank r sums the n_slice partials of token sub-block r through distributed shared
// memory in rank order (deterministic) and writes logits + bias.  With ids != NULL, the CTAs
// that wrote token sub-block r of token block z then count themselves on a ticket; the last of
// them (every expert group's logits for those tokens are written by then) picks top-k and
// weights for those tokens, a warp per token, as k_select does, and resets the ticket.  With
// one token block of at most kRdOneRank tokens, rank 0 takes them all: its selecting CTA then
// holds every token's ids, keeps them in shared memory and runs the dispatch at once, with no
// second ticket and no second read of the ids.
constexpr int kRdOneRank = kRdThreads / 32;  // a token per warp
__device__ __forceinline__ void decode_router_tail(const float* part, int T, int Tb, int E,
                                                   const float* __restrict__ bias, const float* sel_bias, float* logits,
                                                   int k, int32_t* __restrict__ ids, float* __restrict__ wts,
                                                   int* tickets, int* dispatch_ticket, const DispatchOut& dsp,
                                                   int rows_per_tile, int* scratch, int* last_flag,
                                                   const XQuant& xqz) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x;
  const int e0 = blockIdx.x * kRdE, t_base = blockIdx.z * kRdT;
  cluster.sync();
  const int n_slice = int(cluster.num_blocks()), rank = int(cluster.block_rank());
  const bool one = gridDim.z == 1 && Tb <= kRdOneRank;
  const int per = one ? Tb : (Tb + n_slice - 1) / n_slice;
  const int t_lo = min(Tb, rank * per), t_hi = min(Tb, t_lo + per);
  for (int i = tid; i < (t_hi - t_lo) * kRdE; i += kRdThreads) {  // one pass unless the cluster has < 4 slices
    const int t = t_lo + i / kRdE, e = i % kRdE;
    float v[8];  // all remote loads in flight at once, then summed in rank order
#pragma unroll
    for (int r = 0; r < 8; ++r) v[r] = cluster.map_shared_rank(part, min(r, n_slice - 1))[t * kRdE + e];
    float sum = 0.0f;
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (r < n_slice) sum += v[r];
    if (e0 + e < E) logits[size_t(t_base + t) * E + e0 + e] = sum + (bias ? bias[e0 + e] : 0.0f);
  }
  if (xqz.xq) {  // a warp per token, a lane per 8 columns of this CTA's 256
    const int warp = tid >> 5, lane = tid & 31;
    for (int i = warp; i < xqz.q_hi - xqz.q_lo; i += kRdThreads / 32) {
      float pm[8];  // all remote loads in flight at once
#pragma unroll
      for (int r = 0; r < 8; ++r) pm[r] = cluster.map_shared_rank(xqz.amax_part, min(r, n_slice - 1))[i];
      float m = 0.0f;
#pragma unroll
      for (int r = 0; r < 8; ++r) m = fmaxf(m, pm[r]);
      const float s = m > 0.0f ? __fdiv_rn(m, 448.0f) : 1.0f;
      const int t = xqz.q_lo + i;
      float v[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(xqz.xs + t * xqz.xs_ld + lane * 8), v);
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int j = 0; j < 4; j += 2) {
        lo |= uint32_t(e4m3_code2(__fdiv_rn(v[j], s), __fdiv_rn(v[j + 1], s))) << (8 * j);
        hi |= uint32_t(e4m3_code2(__fdiv_rn(v[4 + j], s), __fdiv_rn(v[5 + j], s))) << (8 * j);
      }
      *reinterpret_cast<uint2*>(xqz.xq + size_t(t_base + t) * xqz.d + xqz.k0 + lane * 8) = make_uint2(lo, hi);
      if (rank == 0 && lane == 0) xqz.sx[t_base + t] = s;
    }
  }
  // this CTA is done reading its peers' partials; it waits for them to be done with its own
  // only before it exits
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  if (ids && (!one || rank == 0)) {  // (one token block: ranks 1.. hold no tokens)
    __syncthreads();  // the CTA's logits are written ...
    if (tid == 0) {
      // ... released device-wide by the ticket, which also acquires what the earlier CTAs released
      int* ticket = tickets + blockIdx.z * 8 + rank;
      int old;
      asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(ticket) : "memory");
      const int last = old == int(gridDim.x) - 1;
      if (last) *ticket = 0;  // every contributor has counted: ready for the next launch
      *last_flag = last;
    }
    __syncthreads();
    if (*last_flag) {
      const int warp = tid >> 5, lane = tid & 31;
      int* stage = (one && dsp.counts) ? scratch + lean_dispatch_ids_offset(E) : nullptr;
      for (int t = t_lo + warp; t < t_hi; t += kRdThreads / 32) {
        const size_t row = size_t(t_base + t);
        select_write_free(logits + row * E, E, lane, ids + row * k, wts + row * k, sel_bias,
                          stage ? stage + row * k : nullptr);
      }
      if (stage) {  // every token's ids are in this CTA: dispatch now
        __syncthreads();
        dispatch_lean_body(ids, T, E, k, rows_per_tile, dsp, scratch, true);
      } else if (dsp.counts) {
        // the selecting CTAs count themselves; the last (every token's ids written by then)
        // runs the dispatch in this CTA, on its staging memory
        __syncthreads();
        if (tid == 0) {
          int old;
          asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(dispatch_ticket) : "memory");
          const int last = old == int(gridDim.z) * n_slice - 1;
          if (last) *dispatch_ticket = 0;  // ready for the next launch
          *last_flag = last ? 2 : 1;
        }
        __syncthreads();
        if (*last_flag == 2) dispatch_lean_body(ids, T, E, k, rows_per_tile, dsp, scratch);
      }
    }
  }
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// fp32 x: SIMT.  The CTA stages its slices of Wr and x in shared memory with every load
// issued up front; thread = 2 experts x 2 tokens, one sequential fp32 sum over the slice.
constexpr int kRdLd = kRdK + 4;
constexpr size_t kRdSmemF32 = size_t(kRdE + kRdT) * kRdLd * 4 + size_t(kRdT) * kRdE * 4 + 16;
static_assert(size_t(lean_dispatch_smem_ints(kRouterDecodeMaxT, 511, kTopK)) * 4 <= size_t(kRdE + kRdT) * kRdLd * 4,
              "dispatch scratch");
__global__ void __launch_bounds__(kRdThreads, 2) k_router_decode_f32(const float* __restrict__ x, int T, int d, int E,
                                                                  const float* __restrict__ Wr,
                                                                  const float* __restrict__ bias,
                                                                  const float* sel_bias, float* logits, int k,
                                                                  int32_t* __restrict__ ids, float* __restrict__ wts,
                                                                  int* tickets, int* dispatch_ticket, DispatchOut dsp,
                                                                  int rows_per_tile) {
  extern __shared__ __align__(16) uint8_t rd_smem[];
  float* ws = reinterpret_cast<float*>(rd_smem);  // [kRdE][kRdLd]
  float* xs = ws + kRdE * kRdLd;                   // [kRdT][kRdLd]
  float* part = xs + kRdT * kRdLd;                 // [kRdT][kRdE]
  int* last_flag = reinterpret_cast<int*>(part + kRdT * kRdE);
  const int tid = threadIdx.x;
  const int e0 = blockIdx.x * kRdE, k0 = blockIdx.y * kRdK, t_base = blockIdx.z * kRdT;
  const int Tb = min(kRdT, T - t_base);
  pdl_begin();
  {
    float4 wv[4], xv[16];  // Wr slice: 16 rows x 64 float4; x slice: 64 rows x 64 float4
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = tid + kRdThreads * j, r = i >> 6, c = (i & 63) * 4;
      wv[j] = e0 + r < E ? *reinterpret_cast<const float4*>(Wr + size_t(e0 + r) * d + k0 + c)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int i = tid + kRdThreads * j, t = i >> 6, c = (i & 63) * 4;
      xv[j] = t < Tb ? *reinterpret_cast<const float4*>(x + size_t(t_base + t) * d + k0 + c)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = tid + kRdThreads * j, r = i >> 6, c = (i & 63) * 4;
      *reinterpret_cast<float4*>(ws + r * kRdLd + c) = wv[j];
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int i = tid + kRdThreads * j, t = i >> 6, c = (i & 63) * 4;
      *reinterpret_cast<float4*>(xs + t * kRdLd + c) = xv[j];
    }
  }
  __syncthreads();
  // thread: experts eg and eg + 8 (rows 4 banks apart: conflict-free), tokens 2 tg and 2 tg + 1
  const int eg = tid & 7, tg = tid >> 3;
  if (2 * tg < Tb) {
    float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    const float* wa = ws + eg * kRdLd;
    const float* wb = ws + (eg + 8) * kRdLd;
    const float* xa = xs + (2 * tg) * kRdLd;
    const float* xb = xa + kRdLd;
#pragma unroll 4
    for (int c = 0; c < kRdK; c += 4) {
      const float4 w0 = *reinterpret_cast<const float4*>(wa + c), w1 = *reinterpret_cast<const float4*>(wb + c);
      const float4 x0 = *reinterpret_cast<const float4*>(xa + c), x1 = *reinterpret_cast<const float4*>(xb + c);
      acc[0][0] = fmaf(x0.x, w0.x, acc[0][0]); acc[0][0] = fmaf(x0.y, w0.y, acc[0][0]);
      acc[0][0] = fmaf(x0.z, w0.z, acc[0][0]); acc[0][0] = fmaf(x0.w, w0.w, acc[0][0]);
      acc[0][1] = fmaf(x0.x, w1.x, acc[0][1]); acc[0][1] = fmaf(x0.y, w1.y, acc[0][1]);
      acc[0][1] = fmaf(x0.z, w1.z, acc[0][1]); acc[0][1] = fmaf(x0.w, w1.w, acc[0][1]);
      acc[1][0] = fmaf(x1.x, w0.x, acc[1][0]); acc[1][0] = fmaf(x1.y, w0.y, acc[1][0]);
      acc[1][0] = fmaf(x1.z, w0.z, acc[1][0]); acc[1][0] = fmaf(x1.w, w0.w, acc[1][0]);
      acc[1][1] = fmaf(x1.x, w1.x, acc[1][1]); acc[1][1] = fmaf(x1.y, w1.y, acc[1][1]);
      acc[1][1] = fmaf(x1.z, w1.z, acc[1][1]); acc[1][1] = fmaf(x1.w, w1.w, acc[1][1]);
    }
    part[(2 * tg) * kRdE + eg] = acc[0][0];
    part[(2 * tg) * kRdE + eg + 8] = acc[0][1];
    part[(2 * tg + 1) * kRdE + eg] = acc[1][0];
    part[(2 * tg + 1) * kRdE + eg + 8] = acc[1][1];
  }
  decode_router_tail(part, T, Tb, E, bias, sel_bias, logits, k, ids, wts, tickets, dispatch_ticket, dsp,
                     rows_per_tile, reinterpret_cast<int*>(rd_smem), last_flag, XQuant{});
}

// bf16 x: tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate).  Wr rows are split on
// the fly into three bf16 terms hi + mid + lo that together carry its 24 significand bits;
// with x exact in bf16 every product is exact, so the logit keeps fp32 accuracy, as on the
// prefill router.  A = 16 experts x 16 k, B = 16 k x 8 tokens.  The CTA stages its slices of Wr
// (fp32) and x (bf16) in shared memory with 16-byte asynchronous copies, all in flight at
// once; warp w then takes k-steps 2w and 2w + 1 of the slice for all 8 token tiles (A
// fragments by 8-byte shared loads, B fragments by ldmatrix), and the 8 warps' accumulators
// are summed in warp order through shared memory.
constexpr int kRmLd = 20;          // token-row stride of a warp's partial tile: fragment stores are conflict-free
constexpr int kRmWLd = kRdK + 8;   // floats per staged Wr row: A-fragment loads are conflict-free
constexpr int kRmXLd = kRdK + 8;   // bf16 per staged x row: ldmatrix rows are conflict-free
constexpr size_t kRmOffX = size_t(kRdE) * kRmWLd * 4;
constexpr size_t kRmOffWpart = kRmOffX + size_t(kRdT) * kRmXLd * 2;
constexpr size_t kRmOffPart = kRmOffWpart + size_t(kRdThreads / 32) * kRdT * kRmLd * 4;
constexpr size_t kRmOffAmax = kRmOffPart + size_t(kRdT) * kRdE * 4;  // [kRdT] partial max |x| (fused quantisation)
// the dispatching CTA's scratch (T <= 128, E < 512) overlays the Wr and x staging only: the
// partials after them may still be read by the cluster's other CTAs
static_assert(size_t(lean_dispatch_smem_ints(kRouterDecodeMaxT, 511, kTopK)) * 4 <= kRmOffWpart, "dispatch scratch");
constexpr size_t kRdSmemBf16 = kRmOffAmax + size_t(kRdT) * 4 + 16;

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* smem_row) {
  const unsigned a = static_cast<unsigned>(__cvta_generic_to_shared(smem_row));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a)
               : "memory");
}

// (a, b) -> three packed bf16 pairs with a = hi.x + mid.x + lo.x (likewise b), low half = a.
__device__ __forceinline__ void split3(float2 v, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
  const float2 r1 = make_float2(v.x - __low2float(h), v.y - __high2float(h));
  const __nv_bfloat162 m = __floats2bfloat162_rn(r1.x, r1.y);
  const __nv_bfloat162 l = __floats2bfloat162_rn(r1.x - __low2float(m), r1.y - __high2float(m));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  mid = *reinterpret_cast<const uint32_t*>(&m);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__global__ void __launch_bounds__(kRdThreads, 2) k_router_decode_bf16(const __nv_bfloat16* __restrict__ x, int T, int d,
                                                                   int E, const float* __restrict__ Wr,
                                                                   const float* __restrict__ bias,
                                                                   const float* sel_bias, float* logits, int k,
                                                                   int32_t* __restrict__ ids, float* __restrict__ wts,
                                                                   int* tickets, int* dispatch_ticket, DispatchOut dsp,
                                                                   int rows_per_tile, uint8_t* xq, float* sx) {
  extern __shared__ __align__(16) uint8_t rd_smem[];
  float* ws = reinterpret_cast<float*>(rd_smem);                                  // [kRdE][kRmWLd]
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(rd_smem + kRmOffX);        // [kRdT][kRmXLd]
  float* wpart = reinterpret_cast<float*>(rd_smem + kRmOffWpart);                  // [8 warps][kRdT][kRmLd]
  float* part = reinterpret_cast<float*>(rd_smem + kRmOffPart);                    // [kRdT][kRdE]
  float* amax_part = reinterpret_cast<float*>(rd_smem + kRmOffAmax);               // [kRdT]
  int* last_flag = reinterpret_cast<int*>(amax_part + kRdT);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const int e0 = blockIdx.x * kRdE, k0 = blockIdx.y * kRdK, t_base = blockIdx.z * kRdT;
  const int Tb = min(kRdT, T - t_base);
  const int n_tiles = (Tb + 7) >> 3;
  // the router weights depend on no earlier kernel: their copies start before the wait for
  // the kernel that writes x
#pragma unroll
  for (int j = 0; j < 4; ++j) {  // Wr slice: 16 rows x 64 chunks of 16 bytes
    const int i = tid + kRdThreads * j, r = i >> 6, c = (i & 63) * 4;
    const bool ok = e0 + r < E;
    cp_async16(ws + r * kRmWLd + c, ok ? Wr + size_t(e0 + r) * d + k0 + c : Wr, ok ? 16 : 0);
  }
  pdl_begin();
#pragma unroll
  for (int j = 0; j < 8; ++j) {  // x slice: 64 rows x 32 chunks of 16 bytes (rows past the tokens zero-filled)
    const int i = tid + kRdThreads * j, t = i >> 5, c = (i & 31) * 8;
    const bool ok = t < Tb;
    cp_async16(xs + t * kRmXLd + c, ok ? x + size_t(t_base + t) * d + k0 + c : x, ok ? 16 : 0);
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  float acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
  uint32_t a_hi[2][4], a_mid[2][4], a_lo[2][4];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    // A registers: (row g, cols 2q..), (row g + 8, cols 2q..), (row g, cols 2q + 8..), (row g + 8, cols 2q + 8..)
    const int kk = warp * 32 + s * 16 + 2 * q;
    const float* w0 = ws + g * kRmWLd + kk;
    const float* w1 = w0 + 8 * kRmWLd;
    split3(*reinterpret_cast<const float2*>(w0), a_hi[s][0], a_mid[s][0], a_lo[s][0]);
    split3(*reinterpret_cast<const float2*>(w1), a_hi[s][1], a_mid[s][1], a_lo[s][1]);
    split3(*reinterpret_cast<const float2*>(w0 + 8), a_hi[s][2], a_mid[s][2], a_lo[s][2]);
    split3(*reinterpret_cast<const float2*>(w1 + 8), a_hi[s][3], a_mid[s][3], a_lo[s][3]);
  }
  // ldmatrix x4: matrix m = lane / 8 is (k-step m / 2, k half m % 2) of the token tile; lane
  // supplies row lane % 8 of it
  const int mrow = lane & 7, mk = warp * 32 + (lane >> 4) * 16 + ((lane >> 3) & 1) * 8;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < n_tiles) {
      uint32_t b[4];
      ldmatrix_x4(b, xs + (8 * j + mrow) * kRmXLd + mk);
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        mma_bf16_16816(acc[j], a_lo[s], b[2 * s], b[2 * s + 1]);
        mma_bf16_16816(acc[j], a_mid[s], b[2 * s], b[2 * s + 1]);
        mma_bf16_16816(acc[j], a_hi[s], b[2 * s], b[2 * s + 1]);
      }
    }
  }
  // C registers: (expert g, token 2q), (g, 2q + 1), (g + 8, 2q), (g + 8, 2q + 1) of tile j
  float* wp = wpart + warp * kRdT * kRmLd;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int t = 8 * j + 2 * q;
    wp[t * kRmLd + g] = acc[j][0];
    wp[(t + 1) * kRmLd + g] = acc[j][1];
    wp[t * kRmLd + g + 8] = acc[j][2];
    wp[(t + 1) * kRmLd + g + 8] = acc[j][3];
  }
  __syncthreads();
  {
    const int t = tid >> 2, c = (tid & 3) * 4;  // 64 tokens x 4 groups of 4 experts
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kRdThreads / 32; ++w) {
      const float4 v = *reinterpret_cast<const float4*>(wpart + (w * kRdT + t) * kRmLd + c);
      sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
    }
    *reinterpret_cast<float4*>(part + t * kRdE + c) = sum;
  }
  // fused activation quantisation: this cluster's tokens, max |x| over this CTA's slice
  XQuant xqz{xs, kRmXLd, amax_part, xq, sx, d, k0, 0, 0};
  if (xq) {
    const int tpc = (Tb + int(gridDim.x) - 1) / int(gridDim.x);
    xqz.q_lo = min(Tb, int(blockIdx.x) * tpc);
    xqz.q_hi = min(Tb, xqz.q_lo + tpc);
    for (int i = warp; i < xqz.q_hi - xqz.q_lo; i += kRdThreads / 32) {
      float v[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(xs + (xqz.q_lo + i) * kRmXLd + lane * 8), v);
      float m = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[j]));
      m = warp_max(m);
      if (lane == 0) amax_part[i] = m;
    }
  }
  decode_router_tail(part, T, Tb, E, bias, sel_bias, logits, k, ids, wts, tickets, dispatch_ticket, dsp,
                     rows_per_tile, reinterpret_cast<int*>(rd_smem), last_flag, xqz);
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

// Selection: one warp per token.  Free routing as select_write_free; forced routing validates
// the given ids (range and repeats) and takes the router's logits at them, or forced_w as
// given.
__global__ void __launch_bounds__(256, 2) k_select(const float* __restrict__ logits,
                                                const int32_t* __restrict__ forced_ids,
                                                const float* __restrict__ forced_w, int T, int E, int k,
                                                int32_t* __restrict__ ids, float* __restrict__ w, DevStatus* st,
                                                const float* sel_bias) {
  pdl_begin();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  if (!forced_ids) {
    select_write_free(logits + size_t(t) * E, E, lane, ids + size_t(t) * k, w + size_t(t) * k, sel_bias);
    return;
  }
  int sel = -1;      // lane i < k holds slot i's expert
  float lsel = 0.f;  // and its logit
  {
    int e = lane < k ? forced_ids[size_t(t) * k + lane] : -1;
    bool bad = lane < k && (e < 0 || e >= E);
    // a repeat of an earlier slot's id is rejected too
    for (int j = 0; j < k; ++j) {
      const int ej = __shfl_sync(0xffffffffu, e, j);
      if (lane < k && j < lane && ej == e) bad = true;
    }
    const unsigned badmask = __ballot_sync(0xffffffffu, bad);
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
    lsel = sel >= 0 ? logits[size_t(t) * E + sel] : 0.0f;
  }
  write_selection(sel, lsel, k, lane, ids + size_t(t) * k, w + size_t(t) * k);
}

}  // namespace

cudaError_t launch_router_logits(const void* x, bool x_bf16, int T, const LayerDev& L, float* logits, cudaStream_t s) {
  if (T <= 32) {
    dim3 grid((L.E + 7) / 8);
    if (x_bf16)
      k_router_warp<__nv_bfloat16><<<grid, 256, 0, s>>>((const __nv_bfloat16*)x, T, L.d, L.E, L.Wr, L.logit_bias(),
                                                        logits);
    else
      k_router_warp<float><<<grid, 256, 0, s>>>((const float*)x, T, L.d, L.E, L.Wr, L.logit_bias(), logits);
  } else {
    dim3 grid((L.E + 63) / 64, (T + 63) / 64);
    if (x_bf16)
      return launch_pdl(k_router_gemm<__nv_bfloat16>, grid, dim3(256), 0, s, (const __nv_bfloat16*)x, T, L.d, L.E, L.Wr,
                        L.logit_bias(), logits);
    return launch_pdl(k_router_gemm<float>, grid, dim3(256), 0, s, (const float*)x, T, L.d, L.E, L.Wr, L.logit_bias(),
                      logits);
  }
  return cudaGetLastError();
}

cudaError_t launch_router_decode(const void* x, bool x_bf16, int T, const LayerDev& L, float* logits, int32_t* ids,
                                 float* wts, DevStatus* st, const DispatchOut* dsp, int rows_per_tile, uint8_t* xq,
                                 float* sx, cudaStream_t s) {
  if (T > kRouterDecodeMaxT || L.d % kRdK || L.d / kRdK > 8) return cudaErrorInvalidValue;
  if (xq && (!x_bf16 || !sx)) return cudaErrorInvalidValue;
  const int n_slice = L.d / kRdK;
  static cudaError_t attr = [] {
    cudaError_t e1 = cudaFuncSetAttribute(k_router_decode_bf16, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          int(kRdSmemBf16));
    cudaError_t e2 = cudaFuncSetAttribute(k_router_decode_f32, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          int(kRdSmemF32));
    return e1 != cudaSuccess ? e1 : e2;
  }();
  if (attr != cudaSuccess) return attr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((L.E + kRdE - 1) / kRdE, n_slice, (T + kRdT - 1) / kRdT);
  cfg.blockDim = dim3(kRdThreads);
  cfg.dynamicSmemBytes = x_bf16 ? kRdSmemBf16 : kRdSmemF32;
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
  DispatchOut none{};
  const DispatchOut d = (dsp && ids) ? *dsp : none;  // dispatch only after a selection, and only if asked
  if (d.counts && !(L.E < 512 && T <= kDispatchChunk)) return cudaErrorInvalidValue;
  if (x_bf16)
    return cudaLaunchKernelEx(&cfg, k_router_decode_bf16, (const __nv_bfloat16*)x, T, L.d, L.E, L.Wr, L.logit_bias(),
                              L.sel_bias(), logits, L.k, ids, wts, st->tickets, &st->dispatch_ticket, d, rows_per_tile,
                              xq, sx);
  return cudaLaunchKernelEx(&cfg, k_router_decode_f32, (const float*)x, T, L.d, L.E, L.Wr, L.logit_bias(),
                            L.sel_bias(), logits, L.k, ids, wts, st->tickets, &st->dispatch_ticket, d, rows_per_tile);
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
                      L.Wr, L.logit_bias(), logits);
  return launch_pdl(k_router_small<float>, grid, dim3(threads), smem, s, (const float*)x, T, L.d, L.E, L.Wr, L.logit_bias(),
                    logits);
}

cudaError_t launch_select(const float* logits, const int32_t* forced_ids, const float* forced_w, int T,
                          const LayerDev& L, int32_t* ids, float* w, DevStatus* st, cudaStream_t s) {
  return launch_pdl(k_select, dim3((T + 7) / 8), dim3(256), 0, s, logits, forced_ids, forced_w, T, L.E, L.k, ids, w, st,
                    L.sel_bias());
}

}  // namespace moe
