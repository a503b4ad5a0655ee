// libmoe C ABI: validation, workspace carving and the launch sequence of one layer.
// The call names and the problem statement follow the pages' description of the layer
// ("We Ported Aleph Alpha's Kolibri to a MacBook. Our Own Gate Said No.", sections "The gate",
// 1 and 3): route (router + top-k), the forced variant, and a stack of layers on a residual.
#include <cstddef>
#include <cstring>

#include "common.cuh"
#include "tma.cuh"
#include "dispatch_dev.cuh"

using namespace moe;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shapes the weight-streaming kernels handle (their stages hold whole weight rows).
bool stream_ok(const moe_layer& L) {
  return L.w_dtype == MOE_F32 ||
         (L.d_model % 256 == 0 && L.d_model <= 2048 && L.ffn % 64 == 0 && L.ffn <= 640);
}

moe_status check_layer(const moe_layer* L) {
  if (!L) return MOE_ERR_INVALID_ARG;
  if (L->top_k != kTopK) return MOE_ERR_UNSUPPORTED;
  if (L->n_experts < kTopK || L->n_experts > kMaxExperts) return MOE_ERR_INVALID_ARG;
  if (L->d_model <= 0 || L->ffn <= 0) return MOE_ERR_INVALID_ARG;
  if (!L->w_router || !L->w_gate_up || !L->w_down || !L->sh_gate_up || !L->sh_down) return MOE_ERR_INVALID_ARG;
  if (!aligned16(L->w_router) || !aligned16(L->w_gate_up) || !aligned16(L->w_down) || !aligned16(L->sh_gate_up) ||
      !aligned16(L->sh_down))
    return MOE_ERR_INVALID_ARG;
  if (L->w_layout != MOE_LAYOUT_ROWS && L->w_layout != MOE_LAYOUT_TILED) return MOE_ERR_INVALID_ARG;
  if (L->bias_mode != MOE_BIAS_SCORE && L->bias_mode != MOE_BIAS_SELECT) return MOE_ERR_INVALID_ARG;
  if (L->w_dtype == MOE_E4M3) {
    if (!L->s_gate_up || !L->s_down || !L->sh_s_gate_up || !L->sh_s_down) return MOE_ERR_INVALID_ARG;
    if (L->w_layout == MOE_LAYOUT_TILED ? !(L->d_model % 128 == 0 && L->ffn % 128 == 0) : !stream_ok(*L))
      return MOE_ERR_UNSUPPORTED;
  } else if (L->w_dtype == MOE_E2M1) {
    // 4-bit weights run on the tensor-core kernels only
    if (!L->s_gate_up || !L->s_down || !L->sh_s_gate_up || !L->sh_s_down) return MOE_ERR_INVALID_ARG;
    if (L->w_layout != MOE_LAYOUT_TILED || L->d_model % 128 != 0 || L->ffn % 128 != 0) return MOE_ERR_UNSUPPORTED;
  } else if (L->w_dtype == MOE_F32) {
    if (L->w_layout != MOE_LAYOUT_ROWS) return MOE_ERR_INVALID_ARG;
    if (L->d_model % 128 != 0 || L->ffn % 32 != 0) return MOE_ERR_UNSUPPORTED;
  } else {
    return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

LayerDev to_dev(const moe_layer* L) {
  LayerDev d;
  d.d = L->d_model;
  d.F = L->ffn;
  d.E = L->n_experts;
  d.k = L->top_k;
  // quantised weights (E4M3 or E2M1) take the W8A8 / W4A8 path: E4M3 activations, bf16 rows
  d.fp8 = L->w_dtype == MOE_E4M3 || L->w_dtype == MOE_E2M1;
  d.w4 = L->w_dtype == MOE_E2M1;
  d.tiled = L->w_layout == MOE_LAYOUT_TILED;
  d.bias_sel = L->bias_mode == MOE_BIAS_SELECT && L->router_bias != nullptr;
  d.Wr = L->w_router;
  d.bias = L->router_bias;
  d.wgu = static_cast<const uint8_t*>(L->w_gate_up);
  d.sgu = L->s_gate_up;
  d.wd = static_cast<const uint8_t*>(L->w_down);
  d.sd = L->s_down;
  d.sh_wgu = static_cast<const uint8_t*>(L->sh_gate_up);
  d.sh_sgu = L->sh_s_gate_up;
  d.sh_wd = static_cast<const uint8_t*>(L->sh_down);
  d.sh_sd = L->sh_s_down;
  return d;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                          \
  do {                                         \
    cudaError_t err__ = (expr);                \
    if (err__ != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

// One layer on device buffers.  `residual_add`: y is the bf16 residual, updated in place.
moe_status run_layer(const void* x, moe_dtype x_dtype, int T, const moe_layer* Lh, const int32_t* forced_ids,
                     const float* forced_w, int32_t* ids_out, float* w_out, void* y, moe_dtype y_dtype,
                     bool residual_add, unsigned flags, void* ws, size_t ws_bytes, cudaStream_t s,
                     moe_event_t* ev) {
  const LayerDev L = to_dev(Lh);
  const WsLayout lay = ws_layout(*Lh, T);
  if (ws_bytes < lay.total) return MOE_ERR_WORKSPACE;
  char* base = static_cast<char*>(ws);
  DevStatus* st = reinterpret_cast<DevStatus*>(base + lay.status);
  float* logits = reinterpret_cast<float*>(base + lay.logits);
  int32_t* ids = ids_out ? ids_out : reinterpret_cast<int32_t*>(base + lay.ids);
  float* w = w_out ? w_out : reinterpret_cast<float*>(base + lay.w);
  int32_t* counts = reinterpret_cast<int32_t*>(base + lay.counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(base + lay.offsets);
  int32_t* perm = reinterpret_cast<int32_t*>(base + lay.perm);
  int32_t* pos = reinterpret_cast<int32_t*>(base + lay.pos);
  const bool x_bf16 = x_dtype == MOE_BF16;
  // expert path: the tcgen05 grouped GEMMs read tiled weights, the streaming kernels rows
  const bool use_tc = L.tiled && tc_supported(L);
  if ((flags & MOE_PATH_TC) && !use_tc) return MOE_ERR_UNSUPPORTED;
  if ((flags & MOE_PATH_STREAM) && use_tc) return MOE_ERR_UNSUPPORTED;
  if (!use_tc && (L.tiled || !stream_ok(*Lh))) return MOE_ERR_UNSUPPORTED;
  const int rows_per_tile = use_tc ? tc_rows_per_tile(T) : kStreamRows;
  // ev (optional): MOE_TRACE_POINTS events, recorded before the first stage and after each
  auto mark = [&](int i) -> cudaError_t {
    return ev ? cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev[i]), s) : cudaSuccess;
  };
  MOE_TRY(mark(0));
  bool selected = false;    // the decode and tensor-core routers select in-kernel under free routing
  bool dispatched = false;  // the decode router also dispatches then
  bool quantised = false;   // the bf16 decode router also quantises the activations (E4M3 layers)
  if (!(forced_ids && forced_w)) {
    if (T <= kRouterDecodeMaxT && L.d % 256 == 0 && L.d <= 2048) {
      selected = !forced_ids;
      // under free routing the router's last selecting CTA also dispatches
      dispatched = selected && L.E < 512;
      quantised = x_bf16 && L.fp8;
      DispatchOut dsp;
      dispatch_outputs(lay, base, counts, offsets, perm, pos, &dsp);
      MOE_TRY(launch_router_decode(x, x_bf16, T, L, logits, selected ? ids : nullptr, selected ? w : nullptr, st,
                                   dispatched ? &dsp : nullptr, rows_per_tile,
                                   quantised ? reinterpret_cast<uint8_t*>(base + lay.xq) : nullptr,
                                   quantised ? reinterpret_cast<float*>(base + lay.sx) : nullptr, s));
    } else if (T <= kRouterSmallMaxT && L.d <= 8192) {
      MOE_TRY(launch_router_small(x, x_bf16, T, L, logits, s));
    } else if (T > kRouterSmallMaxT && router_tc_supported(L, x_bf16)) {
      selected = !forced_ids;
      MOE_TRY(launch_router_tc(x, T, L, reinterpret_cast<__nv_bfloat16*>(base + lay.router_w3),
                               selected ? nullptr : logits, selected ? ids : nullptr, selected ? w : nullptr, st, s));
    } else {
      MOE_TRY(launch_router_logits(x, x_bf16, T, L, logits, s));
    }
  }
  MOE_TRY(mark(1));
  if (!selected) MOE_TRY(launch_select(logits, forced_ids, forced_w, T, L, ids, w, st, s));
  MOE_TRY(mark(2));
  if (!dispatched) MOE_TRY(launch_dispatch(ids, T, L.E, L.k, rows_per_tile, lay, base, counts, offsets, perm, pos, s));
  MOE_TRY(mark(3));
  if (!quantised) MOE_TRY(launch_act_quant(x, x_bf16, T, L, base + lay.xq, reinterpret_cast<float*>(base + lay.sx), s));
  MOE_TRY(mark(4));
  MOE_TRY(use_tc ? launch_gateup_tc(L, T, lay, base, s) : launch_gateup_stream(L, T, lay, base, s));
  MOE_TRY(mark(5));
  MOE_TRY(launch_hquant(L, T, lay, base, rows_per_tile, s));
  MOE_TRY(mark(6));
  MOE_TRY(use_tc ? launch_down_tc(L, T, lay, base, s) : launch_down_stream(L, T, lay, base, s));
  MOE_TRY(mark(7));
  MOE_TRY(launch_combine(base + lay.y_rows, pos, w, T, L, y, y_dtype, residual_add, &st->flags, s));
  MOE_TRY(mark(8));
  return MOE_OK;
}

// Self-test of the bounded-wait path: one CTA waits on an mbarrier that expects two arrivals
// but receives one, so the phase never completes; the wait gives up after limit_ns, records
// MOE_ERR_TIMEOUT in the status record and the kernel returns normally.
__global__ void k_selftest_wait_timeout(int* status_flags, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 2);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive(&bar);
    const unsigned long long t0 = global_timer_ns();
    bool done = false;
    while (!done) {
      done = mbar_try_wait(&bar, 0);
      if (!done && global_timer_ns() - t0 > limit_ns) break;
    }
    if (!done) report_timeout_flag(status_flags, 99);
  }
}

}  // namespace

extern "C" {

moe_status moe_selftest_wait_timeout(void* ws, size_t ws_bytes, unsigned timeout_us, moe_stream_t stream) {
  if (!ws || !aligned16(ws) || ws_bytes < sizeof(DevStatus) || timeout_us == 0 || timeout_us > 1000000)
    return MOE_ERR_INVALID_ARG;
  k_selftest_wait_timeout<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<int*>(ws), 1000ull * timeout_us);
  return cuda_status(cudaGetLastError());
}


size_t moe_workspace_bytes(const moe_layer* layer, int T) {
  if (!layer || T < 0 || check_layer(layer) != MOE_OK) return 0;
  return ws_layout(*layer, T).total;
}

moe_status moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!ws || !aligned16(ws) || ws_bytes < sizeof(DevStatus)) return MOE_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, sizeof(DevStatus), reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_pack_weights(const moe_layer* src, void* gate_up, void* down, void* sh_gate_up, void* sh_down,
                            moe_stream_t stream) {
  // only the four weight tensors are read: no check of the shapes the other kernels need
  if (!src || (src->w_dtype != MOE_E4M3 && src->w_dtype != MOE_E2M1) || src->w_layout != MOE_LAYOUT_ROWS)
    return MOE_ERR_INVALID_ARG;
  if (src->n_experts < 1 || src->n_experts > kMaxExperts || src->d_model <= 0 || src->ffn <= 0)
    return MOE_ERR_INVALID_ARG;
  if (!src->w_gate_up || !src->w_down || !src->sh_gate_up || !src->sh_down || !aligned16(src->w_gate_up) ||
      !aligned16(src->w_down) || !aligned16(src->sh_gate_up) || !aligned16(src->sh_down))
    return MOE_ERR_INVALID_ARG;
  if (src->d_model % 128 != 0 || src->ffn % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (!gate_up || !down || !sh_gate_up || !sh_down || !aligned16(gate_up) || !aligned16(down) ||
      !aligned16(sh_gate_up) || !aligned16(sh_down))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_pack_weights(to_dev(src), gate_up, down, sh_gate_up, sh_down,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_route(const void* x, moe_dtype x_dtype, int T, const moe_layer* layer, int k, int32_t* ids_out,
                     float* w_out, float* logits_out, void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status rc = check_layer(layer);
  if (rc != MOE_OK) return rc;
  if (k != layer->top_k) return MOE_ERR_UNSUPPORTED;
  if (T < 0 || T > kMaxTokens) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !ids_out || !w_out || !ws || !aligned16(x) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (x_dtype != MOE_F32 && x_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  const WsLayout lay = ws_layout(*layer, T);
  if (ws_bytes < lay.total) return MOE_ERR_WORKSPACE;
  char* base = static_cast<char*>(ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const LayerDev L = to_dev(layer);
  float* logits = logits_out ? logits_out : reinterpret_cast<float*>(base + lay.logits);
  DevStatus* st = reinterpret_cast<DevStatus*>(base + lay.status);
  if (T <= kRouterDecodeMaxT && L.d % 256 == 0 && L.d <= 2048) {
    MOE_TRY(launch_router_decode(x, x_dtype == MOE_BF16, T, L, logits, ids_out, w_out, st, nullptr, 0, nullptr, nullptr, s));
    return MOE_OK;
  } else if (T <= kRouterSmallMaxT && L.d <= 8192)
    MOE_TRY(launch_router_small(x, x_dtype == MOE_BF16, T, L, logits, s));
  else if (T > kRouterSmallMaxT && router_tc_supported(L, x_dtype == MOE_BF16)) {
    MOE_TRY(launch_router_tc(x, T, L, reinterpret_cast<__nv_bfloat16*>(base + lay.router_w3), logits_out, ids_out, w_out,
                             st, s));
    return MOE_OK;
  } else
    MOE_TRY(launch_router_logits(x, x_dtype == MOE_BF16, T, L, logits, s));
  MOE_TRY(launch_select(logits, nullptr, nullptr, T, L, ids_out, w_out, st, s));
  return MOE_OK;
}

moe_status moe_dispatch(const int32_t* ids, int T, int n_experts, int k, int32_t* counts, int32_t* offsets,
                        int32_t* perm, int32_t* pos, void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (k != kTopK) return MOE_ERR_UNSUPPORTED;
  if (n_experts < k || n_experts > kMaxExperts || T < 0 || T > kMaxTokens) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!ids || !counts || !offsets || !perm || !pos || !ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  moe_layer shape{};
  shape.d_model = 256;
  shape.ffn = 64;
  shape.n_experts = n_experts;
  shape.top_k = k;
  shape.w_dtype = MOE_E4M3;
  const WsLayout lay = ws_layout(shape, T);
  if (ws_bytes < lay.total) return MOE_ERR_WORKSPACE;
  return cuda_status(launch_dispatch(ids, T, n_experts, k, kStreamRows, lay, static_cast<char*>(ws), counts, offsets,
                                     perm, pos, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_forward_traced(const void* x, moe_dtype x_dtype, int T, const moe_layer* layer,
                              const int32_t* forced_ids, const float* forced_w, int32_t* ids_out, float* w_out,
                              void* y, moe_dtype y_dtype, unsigned flags, void* ws, size_t ws_bytes,
                              moe_stream_t stream, moe_event_t* events) {
  moe_status rc = check_layer(layer);
  if (rc != MOE_OK) return rc;
  if (T < 0 || T > kMaxTokens) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !y || !ws || !aligned16(x) || !aligned16(y) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (x_dtype != MOE_F32 && x_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (y_dtype != MOE_F32 && y_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (forced_w && !forced_ids) return MOE_ERR_INVALID_ARG;
  if (flags & ~(MOE_PATH_STREAM | MOE_PATH_TC) || flags == (MOE_PATH_STREAM | MOE_PATH_TC)) return MOE_ERR_INVALID_ARG;
  return run_layer(x, x_dtype, T, layer, forced_ids, forced_w, ids_out, w_out, y, y_dtype, false, flags, ws, ws_bytes,
                   reinterpret_cast<cudaStream_t>(stream), events);
}

moe_status moe_forward(const void* x, moe_dtype x_dtype, int T, const moe_layer* layer, const int32_t* forced_ids,
                       const float* forced_w, int32_t* ids_out, float* w_out, void* y, moe_dtype y_dtype,
                       unsigned flags, void* ws, size_t ws_bytes, moe_stream_t stream) {
  return moe_forward_traced(x, x_dtype, T, layer, forced_ids, forced_w, ids_out, w_out, y, y_dtype, flags, ws,
                            ws_bytes, stream, nullptr);
}

moe_status moe_forward_stack_traced(const moe_layer* layers, int L, void* residual, int T, int32_t* ids_out,
                                    unsigned flags, void* ws, size_t ws_bytes, moe_stream_t stream,
                                    moe_event_t* events) {
  if (!layers || L <= 0) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > kMaxTokens) return MOE_ERR_INVALID_ARG;
  for (int l = 0; l < L; ++l) {
    moe_status rc = check_layer(&layers[l]);
    if (rc != MOE_OK) return rc;
    if (layers[l].d_model != layers[0].d_model || layers[l].top_k != layers[0].top_k) return MOE_ERR_INVALID_ARG;
  }
  if (T == 0) return MOE_OK;
  if (!residual || !ws || !aligned16(residual) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (flags & ~(MOE_PATH_STREAM | MOE_PATH_TC) || flags == (MOE_PATH_STREAM | MOE_PATH_TC)) return MOE_ERR_INVALID_ARG;
  for (int l = 0; l < L; ++l)
    if (ws_bytes < ws_layout(layers[l], T).total) return MOE_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t per_layer_ids = size_t(T) * layers[0].top_k;
  for (int l = 0; l < L; ++l) {
    moe_status rc = run_layer(residual, MOE_BF16, T, &layers[l], nullptr, nullptr,
                              ids_out ? ids_out + size_t(l) * per_layer_ids : nullptr, nullptr, residual, MOE_BF16,
                              true, flags, ws, ws_bytes, s, events ? events + size_t(l) * MOE_TRACE_POINTS : nullptr);
    if (rc != MOE_OK) return rc;
  }
  return MOE_OK;
}

moe_status moe_forward_stack(const moe_layer* layers, int L, void* residual, int T, int32_t* ids_out, unsigned flags,
                             void* ws, size_t ws_bytes, moe_stream_t stream) {
  return moe_forward_stack_traced(layers, L, residual, T, ids_out, flags, ws, ws_bytes, stream, nullptr);
}

moe_status moe_get_status(void* ws, moe_stream_t stream) {
  if (!ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DevStatus h;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(ws, 0, sizeof(DevStatus)) != cudaSuccess) return MOE_ERR_CUDA;
  if (h.flags & kFlagIndex) return MOE_ERR_INDEX;
  if (h.flags & kFlagBadForced) return MOE_ERR_BAD_FORCED_ID;
  if (h.flags & kFlagTimeout) return MOE_ERR_TIMEOUT;
  return MOE_OK;
}

const char* moe_status_string(moe_status status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad dtype or shape)";
    case MOE_ERR_UNSUPPORTED: return "unsupported by this library (e.g. top_k != 6)";
    case MOE_ERR_WORKSPACE: return "workspace smaller than moe_workspace_bytes()";
    case MOE_ERR_BAD_FORCED_ID: return "a forced expert id was out of range or repeated within a token";
    case MOE_ERR_TIMEOUT: return "a device-side wait timed out";
    case MOE_ERR_CUDA: return "a CUDA runtime call failed";
    case MOE_ERR_INDEX: return "an index check of a MOE_DEBUG build failed (an internal error)";
  }
  return "unknown status";
}

moe_status moe_e4m3_encode(const float* in, uint8_t* out, int64_t n, moe_stream_t stream) {
  if (n < 0 || (n > 0 && (!in || !out))) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_e4m3_encode(in, out, n, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
