/* libmoe — the routed mixture-of-experts expert layer of a Kolibri-style model on one
 * NVIDIA GB300 (sm_103a), as a C ABI over hand-written CUDA kernels.
 *
 * The layer (page "We Ported Aleph Alpha's Kolibri to a MacBook. Our Own Gate Said No.",
 * section "The gate", and section 1 for the bias and the forced ids; section 3 for the
 * SwitchGLU expert layer): for every token a float32 router scores the routed experts
 * (384 in Kolibri-1), the top k = 6 are selected and weighted, one shared expert runs for
 * every token, and the weighted expert outputs are summed.  The expert choices can instead
 * be forced from a supplied id tensor (page "We Stopped the Kolibri Benchmark Before Scoring
 * One Answer", section "The gate, forced").  Numerical recipe of this library (the pages
 * leave it open):
 *   logits[t,e] = sum_k x[t,k] Wr[e,k] + b[e]                       (fp32)
 *   ids[t]      = the k largest softmax probabilities, lowest index on ties, in descending
 *                 order;  w[t,i] = p[ids_i] / sum_j p[ids_j]
 *   expert e    = W8A8 SwiGLU: x is quantised per token to E4M3 (scale max|x|/448),
 *                 g = (qx . Wg[e,n]) sx sg[e,n], u likewise, h = silu(g) u, h quantised per
 *                 row the same way, y_e[m] = (qh . Wd[e,m]) sh sd[e,m], stored as a bf16
 *                 activation (round to nearest even) before the combine
 *   y[t]        = y_shared[t] + sum_{i=0..k-1} w[t,i] y_{ids_i}[t]  (slot order, fp32)
 * With fp32 weights (MOE_F32) the experts run in fp32 without quantisation.
 *
 * Conventions for every call:
 *  - Every pointer argument is device memory owned by the caller, unless stated.  The
 *    library allocates nothing and keeps no state between calls.
 *  - Calls are asynchronous on `stream`; host-side validation errors return at once and
 *    launch nothing.  Device-side errors (bad forced ids, a wait that timed out) are
 *    recorded in the workspace and reported by moe_get_status().  Nothing traps.
 *  - T == 0 is a no-op returning MOE_OK.
 *  - Alignment: x, y, weights, scales and the workspace 16-byte aligned.
 *  - Shapes: top_k == 6 (else MOE_ERR_UNSUPPORTED), n_experts <= 1024, T <= 2^20;
 *    E4M3 or E2M1 weights in the tiled layout: d_model % 128 == 0 and ffn % 128 == 0 (E2M1
 *    weights only in the tiled layout); E4M3 weights
 *    in the row layout: d_model % 256 == 0, d_model <= 2048, ffn % 64 == 0, ffn <= 640;
 *    fp32 weights: d_model % 128 == 0 and ffn % 32 == 0.
 *  - Layout: row-major, last index contiguous.
 */
#ifndef LIBMOE_H
#define LIBMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (0 = the legacy default stream) and a cudaEvent_t. */
typedef struct CUstream_st* moe_stream_t;
typedef struct CUevent_st* moe_event_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,   /* null/misaligned pointer, bad dtype or shape */
  MOE_ERR_UNSUPPORTED = -2,   /* valid request this library does not implement (e.g. k != 6) */
  MOE_ERR_WORKSPACE = -3,     /* ws_bytes < moe_workspace_bytes() */
  MOE_ERR_BAD_FORCED_ID = -4, /* a forced id was out of range or repeated within a token */
  MOE_ERR_TIMEOUT = -5,       /* a device-side wait gave up */
  MOE_ERR_CUDA = -6,          /* a CUDA runtime call failed */
  MOE_ERR_INDEX = -7          /* MOE_DEBUG builds only: a kernel's index check failed (an internal
                                 error of the library; the access was kept inside its buffer) */
} moe_status;

/* MOE_E2M1: 4-bit weights (OCP E2M1 codes: sign bit 3, magnitudes 0, 0.5, 1, 1.5, 2, 3, 4,
 * 6), two per byte, element 2i in the low nibble of byte i, with one fp32 scale per output row
 * like MOE_E4M3 (this library's reading of the 4-bit "K4" builds of page "We Stopped the
 * Kolibri Benchmark Before Scoring One Answer", section "What this means if you want Kolibri
 * on a Mac"; the pages give no format).  Weight matrices keep their row count and halve their
 * bytes per row; activations enter the contractions as E4M3 as for MOE_E4M3 (W4A8). */
typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_E4M3 = 2, MOE_E2M1 = 3 } moe_dtype;

/* Byte order of the E4M3 expert weight tensors (w_gate_up, w_down, sh_gate_up, sh_down).
 *   MOE_LAYOUT_ROWS   the shapes below, row-major (a checkpoint's order).
 *   MOE_LAYOUT_TILED  the same bytes regrouped by moe_pack_weights into 16 KB tiles of 128
 *                     rows x 128 bytes of k, each tile stored in the 128-byte-swizzled order
 *                     the tensor cores read, and ordered so that the tiles one GEMM step
 *                     needs are contiguous:
 *                     gate/up tile (e, n, j, half) at byte ((((e * F/128) + n) * d/128 + j) * 2 + half) * 16384
 *                       = rows half*F + 128 n .. +127 of expert e's [2F, d] matrix, k = 128 j .. 128 j + 127
 *                     down tile (e, m, j) at byte (((e * d/128) + m) * F/128 + j) * 16384
 *                       = rows 128 m .. +127 of expert e's [d, F] matrix, k = 128 j .. +127
 *                     inside a tile, byte (r, c) sits at r*128 + 16*((c/16) ^ (r%8)) + c%16.
 *                     The shared expert's tensors are tiled the same way (as expert 0).
 *                     Requires E4M3 or E2M1, d_model % 128 == 0 and ffn % 128 == 0.
 *                     E2M1 weights use the same tile order with 8 KB tiles (tile index
 *                     x 8192 in place of x 16384): 128 rows of 64 bytes (128 codes of k)
 *                     each, rows in order and unswizzled (the tensor cores' swizzle is
 *                     applied when a tile is copied to shared memory).
 * The tensor-core expert kernels read the tiled layout (each pipeline stage is then one
 * contiguous copy of 32-80 KB); the weight-streaming kernels read the row layout.  E2M1
 * layers run only on the tensor-core kernels, so moe_forward takes them tiled. */
typedef enum { MOE_LAYOUT_ROWS = 0, MOE_LAYOUT_TILED = 1 } moe_layout;

/* How router_bias enters the routing (page "We Ported Aleph Alpha's Kolibri to a MacBook.
 * Our Own Gate Said No.", section 1: "router score plus a per-expert selection bias").
 *   MOE_BIAS_SCORE   logits = x Wr^T + b: the bias shifts both the selection and the weights.
 *   MOE_BIAS_SELECT  logits = x Wr^T: the experts are ranked on logits + b, and the weights are
 *                    the softmax of the unbiased logits renormalised over the selected six. */
typedef enum { MOE_BIAS_SCORE = 0, MOE_BIAS_SELECT = 1 } moe_bias_mode;

/* One layer: borrowed device pointers.  Shapes with d = d_model, F = ffn, E = n_experts.
 *   w_router     [E, d]  fp32            router_bias [E] fp32 or NULL
 *   w_gate_up    [E, 2, F, d]            gate rows (index 0) then up rows (index 1)
 *                (E2M1: the last dimension of each weight tensor holds two codes per byte)
 *   s_gate_up    [E, 2, F] fp32          per-output-row scales (E4M3 only, else NULL)
 *   w_down       [E, d, F]               s_down [E, d] fp32 (E4M3 only)
 *   sh_gate_up   [2, F, d]               sh_s_gate_up [2, F] (E4M3 only)
 *   sh_down      [d, F]                  sh_s_down [d] (E4M3 only)
 * Weights are E4M3 codes (w_dtype = MOE_E4M3, one byte each), E2M1 codes (MOE_E2M1, two
 * per byte) or fp32 (MOE_F32). */
typedef struct {
  int d_model, ffn, n_experts, top_k;
  moe_dtype w_dtype;
  const float* w_router;
  const float* router_bias;
  const void* w_gate_up;
  const float* s_gate_up;
  const void* w_down;
  const float* s_down;
  const void* sh_gate_up;
  const float* sh_s_gate_up;
  const void* sh_down;
  const float* sh_s_down;
  moe_layout w_layout; /* order of the four E4M3 weight tensors (MOE_LAYOUT_ROWS for fp32) */
  moe_bias_mode bias_mode; /* MOE_BIAS_SCORE (a zero-initialised struct) or MOE_BIAS_SELECT */
} moe_layer;

/* Flags for moe_forward / moe_forward_stack: which expert kernels run.  0 = automatic: the
 * tcgen05 grouped GEMMs for tiled E4M3 weights, the weight-streaming kernels otherwise. */
#define MOE_PATH_AUTO 0u
#define MOE_PATH_STREAM 1u /* weight-streaming kernels (row layout; any T) */
#define MOE_PATH_TC 2u     /* tcgen05 grouped GEMMs (tiled layout; any T) */

/* Writes the tiled layout (MOE_LAYOUT_TILED above) of src's four E4M3 (or E2M1) weight
 * tensors, which must be in the row layout, into gate_up [E*2*F*d], down [E*d*F], sh_gate_up
 * [2*F*d] and sh_down [d*F] bytes (half as many for E2M1) of caller-owned device memory
 * (16-byte aligned, not overlapping the sources).  The scales and the router are unchanged; a moe_layer with the four pointers
 * replaced and w_layout = MOE_LAYOUT_TILED then describes the same layer.  Asynchronous on
 * `stream`.  MOE_ERR_UNSUPPORTED unless E4M3 or E2M1 with d_model % 128 == 0 and
 * ffn % 128 == 0. */
moe_status moe_pack_weights(const moe_layer* src, void* gate_up, void* down, void* sh_gate_up, void* sh_down,
                            moe_stream_t stream);

/* Bytes of workspace the calls below need for T tokens of this layer (host only). */
size_t moe_workspace_bytes(const moe_layer* layer, int T);

/* Clears the workspace's status record.  Call once after allocating a workspace (or use
 * zero-filled memory).  Asynchronous on `stream`. */
moe_status moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream);

/* Router and selection (free routing) for T tokens: a float32 router scores every routed
 * expert and the top k = 6 are kept and weighted (page "We Ported Aleph Alpha's Kolibri to a
 * MacBook. Our Own Gate Said No.", section "The gate": 384 experts, top 6, a float32 router; the
 * per-expert bias: section 1).
 *   x           [T, d]  bf16 or fp32 (x_dtype)
 *   k           must equal layer->top_k (6)
 *   ids_out     [T, k] int32: selected experts, descending probability, lowest index on ties
 *   w_out       [T, k] fp32: renormalised softmax weights of the selected experts
 *   logits_out  [T, E] fp32 router logits (bias included under MOE_BIAS_SCORE, not under
 *               MOE_BIAS_SELECT), or NULL */
moe_status moe_route(const void* x, moe_dtype x_dtype, int T, const moe_layer* layer, int k,
                     int32_t* ids_out, float* w_out, float* logits_out, void* ws, size_t ws_bytes,
                     moe_stream_t stream);

/* Grouping of the T*k routed (token, slot) rows by expert, shared expert last: the sorted
 * grouping that turns the experts into one grouped GEMM (page "We Ported Aleph Alpha's Kolibri
 * to a MacBook. Our Own Gate Said No.", section 3, update of 5 October: the sorted path and its
 * row-count edge cases).
 *   counts  [E + 1]   rows per expert; counts[E] = T (the shared expert's rows)
 *   offsets [E + 2]   exclusive prefix sum of counts; offsets[E] = T*k, offsets[E+1] = T*k + T
 *   perm    [T*k + T] token of each row; tokens ascend within each expert (stable)
 *   pos     [T, k]    row holding (token t, slot i)
 * ids [T, k] must be valid (distinct within a token, in [0, E)). */
moe_status moe_dispatch(const int32_t* ids, int T, int n_experts, int k, int32_t* counts, int32_t* offsets,
                        int32_t* perm, int32_t* pos, void* ws, size_t ws_bytes, moe_stream_t stream);

/* The whole layer for T tokens.
 *   x            [T, d] bf16 or fp32 (x_dtype)
 *   forced_ids   [T, k] int32 or NULL: use these experts in this order instead of selecting.
 *                Ids out of range or repeated within a token contribute nothing and set
 *                MOE_ERR_BAD_FORCED_ID in the status record.
 *   forced_w     [T, k] fp32 or NULL (only with forced_ids): use these weights as given;
 *                without it the weights are the renormalised softmax over the forced ids.
 *   ids_out, w_out  [T, k] or NULL: the ids and weights used
 *   y            [T, d] bf16 or fp32 (y_dtype)
 *   flags        MOE_PATH_* */
moe_status moe_forward(const void* x, moe_dtype x_dtype, int T, const moe_layer* layer,
                       const int32_t* forced_ids, const float* forced_w, int32_t* ids_out, float* w_out,
                       void* y, moe_dtype y_dtype, unsigned flags, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/* L layers on a bf16 residual stream, free routing: for l = 0..L-1,
 * r <- bf16_round_nearest_even(r + layer_l(r)).  Kolibri-1 stacks 50 such MoE layers (page "We
 * Ported Aleph Alpha's Kolibri to a MacBook. Our Own Gate Said No.", section "The gate"); the
 * bf16 residual with one rounding per layer after an fp32 add is this library's reading of the
 * pages' bf16 activations.
 *   layers    host array of L layer descriptors (read during the call only)
 *   residual  [T, d] bf16, updated in place
 *   ids_out   [L, T, k] int32 or NULL: the experts each layer selected
 * ws must hold moe_workspace_bytes() of the largest layer; layers share it in turn. */
moe_status moe_forward_stack(const moe_layer* layers, int L, void* residual, int T, int32_t* ids_out,
                             unsigned flags, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Stage boundaries recorded by the *_traced calls: before the router, then after the router,
 * selection, dispatch, activation quantisation, gate/up, h quantisation, down, combine. */
#define MOE_TRACE_POINTS 9

/* moe_forward, recording `events` (MOE_TRACE_POINTS caller-created CUDA events, or NULL) on
 * `stream` at the stage boundaries, so the caller can time each kernel stage. */
moe_status moe_forward_traced(const void* x, moe_dtype x_dtype, int T, const moe_layer* layer,
                              const int32_t* forced_ids, const float* forced_w, int32_t* ids_out, float* w_out,
                              void* y, moe_dtype y_dtype, unsigned flags, void* ws, size_t ws_bytes,
                              moe_stream_t stream, moe_event_t* events);

/* moe_forward_stack with events [L][MOE_TRACE_POINTS] (or NULL) recorded per layer. */
moe_status moe_forward_stack_traced(const moe_layer* layers, int L, void* residual, int T, int32_t* ids_out,
                                    unsigned flags, void* ws, size_t ws_bytes, moe_stream_t stream,
                                    moe_event_t* events);

/* Synchronises `stream`, returns the first device-side error recorded in the workspace
 * since the last call (MOE_OK if none) and clears the record. */
moe_status moe_get_status(void* ws, moe_stream_t stream);

/* moe_route without a workspace, for callers that cannot allocate device memory (a host
 * runtime that owns all device memory through its own pool and forbids side allocations, or a
 * serving loop where an allocation, which may synchronise the device, is not allowed).  The
 * pages have no counterpart: this is a deployment variant of the router and selection.
 *   Same arguments and results as moe_route, minus logits_out and the workspace.
 *   Scratch: a fixed 4 MiB + 768 B array inside the library, resident on every GPU that loads
 *   it until the process exits; T * n_experts must be <= 1,048,576, else MOE_ERR_WORKSPACE.
 *   The first call on a device looks up the array's device address (once per device, with
 *   that device current); make that first call before any stream capture.  A device reset or
 *   another CUDA context on the device moves the array: the first call made under the new
 *   context looks the address up again.
 *   All calls on a device share the array: calls that overlap on the GPU race; serialise them.
 *   No device-side error can arise in this call (no forced ids, no device-side waits), so it
 *   has no status record to read: host-side errors are its return value, as for moe_route.
 *   Allocates nothing (no cudaMalloc, no cudaFree). */
moe_status moe_route_noalloc(const void* x, moe_dtype x_dtype, int T, const moe_layer* layer, int k,
                             int32_t* ids_out, float* w_out, moe_stream_t stream);

/* Exercises the device-side timeout path: launches one CTA whose wait on a barrier can never
 * complete; the wait gives up after timeout_us (<= 1 s) and records MOE_ERR_TIMEOUT in the
 * workspace's status record, which moe_get_status() then returns.  The GPU context stays
 * usable.  For failure-detection tests. */
moe_status moe_selftest_wait_timeout(void* ws, size_t ws_bytes, unsigned timeout_us, moe_stream_t stream);

/* Static description of a status code. */
const char* moe_status_string(moe_status status);

/* The device E4M3 encoder the kernels use (round to nearest even, saturating at +-448),
 * on n fp32 values: out[i] = code(in[i]).  For codec tests. */
moe_status moe_e4m3_encode(const float* in, uint8_t* out, int64_t n, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LIBMOE_H */
