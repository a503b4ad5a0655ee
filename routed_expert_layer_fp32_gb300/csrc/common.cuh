// Shared device helpers and the workspace layout of libmoe (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/libmoe.h"

namespace moe {

constexpr int kMaxExperts = 1024;
constexpr int kTopK = 6;
constexpr int kMaxTokens = 1 << 20;

// Device-side status record (first bytes of the workspace).
struct DevStatus {
  int flags;        // bit 0: bad forced id, bit 1: timeout
  int bad_forced;   // number of rejected forced slots
  int timeout_site; // where a bounded wait gave up (0 = none)
  int pad[61];
};
constexpr int kFlagBadForced = 1;
constexpr int kFlagTimeout = 2;

// One work tile of a grouped GEMM: rows [row0, row0 + nrows) of group `group`
// (group == n_experts is the shared expert).
struct Tile {
  int group, row0, nrows, pad;
};

// Where each buffer lives inside the caller's workspace, for T tokens.
struct WsLayout {
  size_t status, logits, ids, w, counts, offsets, chunk_counts, perm, pos, n_tiles, tiles, xq, sx, h, qh, sh, y_rows;
  size_t total;
  int T, R, n_chunks, max_tiles;
};

constexpr int kDispatchChunk = 1024;  // tokens per dispatch CTA
constexpr int kStreamRows = 32;        // rows per tile on the streaming path

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline WsLayout ws_layout(const moe_layer& L, int T) {
  WsLayout w{};
  const int E = L.n_experts, k = L.top_k, d = L.d_model, F = L.ffn;
  const size_t R = size_t(T) * (k + 1);
  const bool f32w = (L.w_dtype == MOE_F32);
  w.T = T;
  w.R = int(R);
  w.n_chunks = (T + kDispatchChunk - 1) / kDispatchChunk;
  w.max_tiles = int(R / 8 + 2 * (E + 1) + 8);  // tiles of >= 8 rows or a group's tail
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
  w.status = take(sizeof(DevStatus));
  w.logits = take(size_t(T) * E * 4);
  w.ids = take(size_t(T) * k * 4);
  w.w = take(size_t(T) * k * 4);
  w.counts = take(size_t(E + 1) * 4);
  w.offsets = take(size_t(E + 2) * 4);
  w.chunk_counts = take(size_t(w.n_chunks) * E * 4);
  w.perm = take(R * 4);
  w.pos = take(size_t(T) * k * 4);
  w.n_tiles = take(16);
  w.tiles = take(size_t(w.max_tiles) * sizeof(Tile));
  w.xq = take(R * d * (f32w ? 4 : 1));
  w.sx = take(R * 4);
  w.h = take(R * F * 4);
  w.qh = take(R * F);
  w.sh = take(R * 4);
  w.y_rows = take(R * d * 4);
  w.total = o;
  return w;
}

// ---------------------------------------------------------------- device helpers --------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// E4M3 code of v: round to nearest even, saturating to +-448 (hardware conversion).
__device__ __forceinline__ uint8_t e4m3_code(float v) {
  return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}
// Two codes packed little-endian: low byte = code(a), high byte = code(b).
__device__ __forceinline__ uint16_t e4m3_code2(float a, float b) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// 128-bit load of streamed weights: read once, do not keep in L1.
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// D += A(16x32 e4m3, row) * B(32x8 e4m3, col), fp32 accumulate (sm_89+ warp MMA).
__device__ __forceinline__ void mma_e4m3_16x8x32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                 uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ void set_status(DevStatus* st, int flag) { atomicOr(&st->flags, flag); }

}  // namespace moe

// Kernel launchers (defined in the .cu files, called by api.cu).
namespace moe {
struct LayerDev {
  int d, F, E, k;
  bool fp8;
  const float* Wr;
  const float* bias;
  const uint8_t* wgu;
  const float* sgu;
  const uint8_t* wd;
  const float* sd;
  const uint8_t* sh_wgu;
  const float* sh_sgu;
  const uint8_t* sh_wd;
  const float* sh_sd;
};

cudaError_t launch_router_logits(const void* x, bool x_bf16, int T, const LayerDev& L, float* logits, cudaStream_t s);
cudaError_t launch_select(const float* logits, const int32_t* forced_ids, const float* forced_w, int T,
                          const LayerDev& L, int32_t* ids, float* w, DevStatus* st, cudaStream_t s);
cudaError_t launch_dispatch(const int32_t* ids, int T, int E, int k, int rows_per_tile, const WsLayout& ws,
                            char* base, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* pos,
                            cudaStream_t s);
cudaError_t launch_act_quant(const void* x, bool x_bf16, int T, const LayerDev& L, const int32_t* pos, void* xq,
                             float* sx, cudaStream_t s);
cudaError_t launch_gateup_stream(const LayerDev& L, int T, const WsLayout& ws, char* base, cudaStream_t s);
cudaError_t launch_hquant(const LayerDev& L, int T, const WsLayout& ws, char* base, cudaStream_t s);
cudaError_t launch_down_stream(const LayerDev& L, int T, const WsLayout& ws, char* base, cudaStream_t s);
cudaError_t launch_combine(const float* y_rows, const int32_t* pos, const float* w, int T, const LayerDev& L,
                           void* y, moe_dtype y_dtype, bool residual_add, cudaStream_t s);
cudaError_t launch_e4m3_encode(const float* in, uint8_t* out, int64_t n, cudaStream_t s);
}  // namespace moe
