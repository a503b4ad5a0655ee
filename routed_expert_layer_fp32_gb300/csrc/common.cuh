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
  int dispatch_ticket;  // decode router: selecting CTAs done, the last one dispatches; 0 between launches
  int tickets[128];  // decode router: CTAs done per (64-token block, token sub-block); 0 between launches
  int pad[60];
};
static_assert(sizeof(DevStatus) == 768, "DevStatus is three 256-byte blocks");
constexpr int kFlagBadForced = 1;
constexpr int kFlagTimeout = 2;

// One work tile of a grouped GEMM: rows [row0, row0 + nrows) of group `group`
// (group == n_experts is the shared expert).
struct Tile {
  int group, row0, nrows, pad;
};

// Where each buffer lives inside the caller's workspace, for T tokens.
struct WsLayout {
  size_t status, logits, router_w3, ids, w, counts, offsets, chunk_counts, perm, pos, n_tiles, tiles, xq, sx, h,
      qh, sh, y_rows;
  size_t total;
  int T, R, R_alloc, n_chunks, max_tiles;
};

constexpr int kDispatchChunk = 1024;  // up to this many tokens the dispatch is one CTA
constexpr int kScatterChunk = 256;    // tokens per CTA of the multi-CTA dispatch
constexpr int kRouterSmallMaxT = 128;   // up to this many tokens the small fallback router runs
constexpr int kRouterDecodeMaxT = 512;   // up to this many tokens the cluster (decode) router runs (measured: 60 us at 512 tokens against ~100 us for the tensor-core router; 107 us at 1024)
static_assert(kRouterDecodeMaxT / 64 * 8 <= 128, "a ticket per (64-token block, k-slice rank)");
constexpr int kStreamRows = 16;        // rows per tile on the streaming path

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline WsLayout ws_layout(const moe_layer& L, int T) {
  WsLayout w{};
  const int E = L.n_experts, k = L.top_k, d = L.d_model, F = L.ffn;
  const size_t R = size_t(T) * (k + 1);
  const bool f32w = (L.w_dtype == MOE_F32);
  w.T = T;
  w.R = int(R);
  w.R_alloc = int(R) + 256;  // row padding: tensor-map boxes of up to 256 rows stay inside the buffers
  w.n_chunks = (T + kScatterChunk - 1) / kScatterChunk;
  w.max_tiles = int(R / 8 + 2 * (E + 1) + 8);  // tiles of >= 8 rows or a group's tail
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
  w.status = take(sizeof(DevStatus));
  w.logits = take(size_t(T) * E * 4);
  w.router_w3 = take(T > kRouterSmallMaxT ? size_t(3) * E * d * 2 : 0);  // bf16 split of Wr
  w.ids = take(size_t(T) * k * 4);
  w.w = take(size_t(T) * k * 4);
  w.counts = take(size_t(E + 1) * 4);
  w.offsets = take(size_t(E + 2) * 4);
  w.chunk_counts = take(size_t(w.n_chunks) * E * 4);
  w.perm = take(R * 4);
  w.pos = take(size_t(T) * k * 4);
  w.n_tiles = take(16);
  w.tiles = take(size_t(w.max_tiles) * sizeof(Tile));
  w.xq = take(size_t(T) * d * (f32w ? 4 : 1));  // activation rows in token order
  w.sx = take(size_t(T) * 4);
  w.h = take(R * F * 4);
  w.qh = take(size_t(w.R_alloc) * F);
  w.sh = take(R * 4);
  w.y_rows = take(R * d * (f32w ? 4 : 2));  // expert output rows: bf16 for E4M3 layers
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

// 16-byte asynchronous global->shared copy (L1 bypassed); src_bytes < 16 zero-fills the rest.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes = 16) {
  const unsigned dst = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(gmem), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
// Wait until at most n groups are pending (n folds to a constant in unrolled loops).
__device__ __forceinline__ void cp_async_wait_n(int n) {
  switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    case 6: cp_async_wait<6>(); break;
    case 7: cp_async_wait<7>(); break;
    case 8: cp_async_wait<8>(); break;
    case 9: cp_async_wait<9>(); break;
    default: cp_async_wait<0>(); break;
  }
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

// Programmatic dependent launch: every kernel of a layer is launched with programmatic
// stream serialisation, so it may start while its predecessor finishes.  pdl_begin() waits
// until the predecessor grid has completed (its writes visible) and then lets the next
// kernel launch; kernels call it before touching global memory.  Without the launch
// attribute both instructions are no-ops.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Lets the next kernel launch first, then waits.  Only for a kernel whose successor reads,
// before its own wait, nothing this kernel's predecessor may still be writing: the successor
// may then start while that predecessor runs (k_hquant: down's CTAs take the SMs as gate/up's
// retire and pull their first weights into L2; down's tile list was final before gate/up
// passed its wait).
__device__ __forceinline__ void pdl_trigger_then_wait() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void set_status(DevStatus* st, int flag) { atomicOr(&st->flags, flag); }

// ---- MOE_DEBUG builds: index checks -------------------------------------------------------
// Compiled with -DMOE_DEBUG, the kernels check every data-dependent index they read (tile
// descriptors, tokens in perm, rows in pos) against the buffers it addresses.  A failed check
// records kFlagIndex and the site in the status record (moe_get_status returns
// MOE_ERR_INDEX) and the access is redirected to an index inside the buffer, so the kernel
// finishes without touching memory outside its buffers; nothing traps.  Release builds
// compile the checks away.
constexpr int kFlagIndex = 4;
#ifdef MOE_DEBUG
constexpr bool kDebugIndexChecks = true;
#else
constexpr bool kDebugIndexChecks = false;
#endif

__device__ __forceinline__ void report_index(int* status_flags, int site) {
  atomicOr(status_flags, kFlagIndex);
  atomicCAS(status_flags + 2, 0, 1000 + site);
}

// Tile i of a tile list as an expert kernel reads it.  Debug builds check the group (<= E, the
// shared expert being group E), the rows (inside [0, R)) and the height (1 .. max_rows), and
// replace a bad tile by a clamped one; every role of a kernel reads its tiles through this, so
// the roles stay in step whatever they read.
__device__ __forceinline__ Tile checked_tile(const Tile* tiles, int i, int E, int R, int max_rows, int* status_flags,
                                             int site) {
  Tile t = tiles[i];
  if (kDebugIndexChecks) {
    const int hmax = min(max_rows, R);
    if (!(t.group >= 0 && t.group <= E && t.nrows >= 1 && t.nrows <= hmax && t.row0 >= 0 && t.row0 <= R - t.nrows)) {
      report_index(status_flags, site);
      t.group = min(max(t.group, 0), E);
      t.nrows = min(max(t.nrows, 1), hmax);
      t.row0 = min(max(t.row0, 0), R - t.nrows);
    }
  }
  return t;
}

// A token index read from perm: debug builds check 0 <= t < T (token 0 replaces a bad one).
__device__ __forceinline__ int checked_token(int t, int T, int* status_flags, int site) {
  if (kDebugIndexChecks && (t < 0 || t >= T)) {
    report_index(status_flags, site);
    return 0;
  }
  return t;
}

// Record a device-side timeout: flags |= kFlagTimeout, and the first site that gave up.
__device__ __forceinline__ void report_timeout_flag(int* status_flags, int site) {
  atomicOr(status_flags, kFlagTimeout);
  atomicCAS(status_flags + 2, 0, site);
}

template <typename... ExpTypes, typename... ActTypes>
inline cudaError_t launch_pdl(void (*kernel)(ExpTypes...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              ActTypes&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<ActTypes&&>(args)...);
}

}  // namespace moe

// Kernel launchers (defined in the .cu files, called by api.cu).
namespace moe {
struct LayerDev {
  int d, F, E, k;
  bool fp8;       // quantised weights (E4M3, or E2M1 with w4): E4M3 activations, bf16 expert rows
  bool w4;        // E2M1 weights (4-bit codes, two per byte)
  bool tiled;     // E4M3 weights in the tiled layout (MOE_LAYOUT_TILED)
  bool bias_sel;  // MOE_BIAS_SELECT: the bias ranks the experts but stays out of the logits
  // the bias added to the logits the routers write, and the one the selection adds on top
  const float* logit_bias() const { return bias_sel ? nullptr : bias; }
  const float* sel_bias() const { return bias_sel ? bias : nullptr; }
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
// The four E4M3 weight tensors of L (row layout) rewritten in the tiled layout.
cudaError_t launch_pack_weights(const LayerDev& L, void* gate_up, void* down, void* sh_gate_up, void* sh_down,
                                cudaStream_t s);
cudaError_t launch_select(const float* logits, const int32_t* forced_ids, const float* forced_w, int T,
                          const LayerDev& L, int32_t* ids, float* w, DevStatus* st, cudaStream_t s);
// Prefill router on tensor cores (bf16 x, Wr split into three bf16 terms in w3 [3, E, d]).
// logits (or NULL) receive the logits; with ids/wts not NULL the kernel also selects the
// top-k (free routing) and writes ids and renormalised weights.
bool router_tc_supported(const LayerDev& L, bool x_bf16);
cudaError_t launch_router_tc(const void* x, int T, const LayerDev& L, __nv_bfloat16* w3, float* logits, int32_t* ids,
                             float* wts, DevStatus* st, cudaStream_t s);
// Decode router (T <= kRouterDecodeMaxT, d % 256 == 0, d <= 2048): k split over the CTAs of a
// thread-block cluster, partials summed through distributed shared memory; deterministic.
// Writes logits; with ids/wts not NULL it also selects the top-k (free routing), using the
// ticket counters in st (zero between launches), and with dsp not NULL its last selecting CTA
// also runs the dispatch (E < 512).
struct DispatchOut;
// With xq (bf16 x only) the router also writes the per-token E4M3 activations and scales
// that launch_act_quant would.
cudaError_t launch_router_decode(const void* x, bool x_bf16, int T, const LayerDev& L, float* logits, int32_t* ids,
                                 float* wts, DevStatus* st, const DispatchOut* dsp, int rows_per_tile, uint8_t* xq,
                                 float* sx, cudaStream_t s);
// Decode router (T <= kRouterSmallMaxT, d <= 8192): all of k per CTA, deterministic.
cudaError_t launch_router_small(const void* x, bool x_bf16, int T, const LayerDev& L, float* logits, cudaStream_t s);


// The dispatch outputs run_layer hands to the decode router.
void dispatch_outputs(const WsLayout& ws, char* base, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* pos,
                      DispatchOut* o);
cudaError_t launch_dispatch(const int32_t* ids, int T, int E, int k, int rows_per_tile, const WsLayout& ws,
                            char* base, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* pos,
                            cudaStream_t s);
cudaError_t launch_act_quant(const void* x, bool x_bf16, int T, const LayerDev& L, void* xq, float* sx,
                             cudaStream_t s);
cudaError_t launch_gateup_stream(const LayerDev& L, int T, const WsLayout& ws, char* base, cudaStream_t s);
cudaError_t launch_hquant(const LayerDev& L, int T, const WsLayout& ws, char* base, int rows_per_tile, cudaStream_t s);
// tcgen05 grouped GEMMs (prefill and decode): E4M3 weights with d % 128 == 0, ffn % 128 == 0.
bool tc_supported(const LayerDev& L);
int tc_rows_per_tile(int T);
cudaError_t launch_gateup_tc(const LayerDev& L, int T, const WsLayout& ws, char* base, cudaStream_t s);
cudaError_t launch_down_tc(const LayerDev& L, int T, const WsLayout& ws, char* base, cudaStream_t s);
cudaError_t launch_down_stream(const LayerDev& L, int T, const WsLayout& ws, char* base, cudaStream_t s);
cudaError_t launch_combine(const void* y_rows, const int32_t* pos, const float* w, int T, const LayerDev& L,
                           void* y, moe_dtype y_dtype, bool residual_add, int* status_flags, cudaStream_t s);
cudaError_t launch_e4m3_encode(const float* in, uint8_t* out, int64_t n, cudaStream_t s);
}  // namespace moe
