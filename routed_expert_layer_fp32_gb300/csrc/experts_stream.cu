// Expert compute on the weight-streaming path, plus activation quantisation and combine.
//
// SwitchGLU experts ("We Ported Aleph Alpha's Kolibri to a MacBook. Our Own Gate Said No.",
// section 3) with FP8 E4M3 weights and one fp32 scale per output row; activations are
// quantised per row to E4M3 (scale max|v|/448) before each FP8 contraction (W8A8).
//
// At decode sizes the layer is a read of the selected experts' weights.  Each warp streams
// 16 weight rows with 128-bit loads straight into registers and multiplies them by up to 32
// activation rows with m16n8k32 E4M3 warp MMAs.  A thread's 16 contiguous bytes of a weight
// row feed two MMAs: since a dot product does not depend on the order of its k terms, the
// bytes are assigned to MMA k-slots in load order, and the activation fragment (16 bytes of
// the same k range, same assignment) follows it.  No shared-memory staging is needed.
#include <algorithm>

#include "common.cuh"
#include "tma.cuh"

namespace moe {
namespace {

// ------------------------------------------------------------ activation quantisation -----
// One CTA per token: sx = max|x| / 448 (1 if the row is zero), q = E4M3(x / sx), written to
// the token's row of xq (token order: the expert kernels gather rows through perm).  The
// fp32-weight path stores x itself, as fp32.
template <typename XT>
__device__ __forceinline__ void load8(const XT* p, float (&v)[8]);
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&v)[8]) {
  float4 a = *reinterpret_cast<const float4*>(p);
  float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename XT, bool kFp8>
__global__ void __launch_bounds__(256) k_act_quant(const XT* __restrict__ x, int T, int d, void* __restrict__ xq,
                                                   float* __restrict__ sx) {
  // A warp per token, eight tokens per CTA: a lane's loads of the row are all in flight at
  // once and the maximum is a warp reduction.  x was written before the kernel this launch
  // overlaps started: its scale is found before the dependency wait; the stores wait (the
  // previous layer's expert kernels read xq).
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const bool live = t < T;
  const XT* xr = x + size_t(live ? t : 0) * d;
  float amax = 0.0f;
#pragma unroll 8
  for (int c = lane * 8; c < d; c += 256) {
    float v[8];
    load8(xr + c, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
  amax = warp_max(amax);
  const float s = kFp8 ? (amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f) : 1.0f;
  pdl_begin();
  if (!live) return;
#pragma unroll 8
  for (int c = lane * 8; c < d; c += 256) {
    float v[8];
    load8(xr + c, v);
    if (kFp8) {
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int i = 0; i < 4; i += 2) {
        lo |= uint32_t(e4m3_code2(__fdiv_rn(v[i], s), __fdiv_rn(v[i + 1], s))) << (8 * i);
        hi |= uint32_t(e4m3_code2(__fdiv_rn(v[4 + i], s), __fdiv_rn(v[5 + i], s))) << (8 * i);
      }
      *reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(xq) + size_t(t) * d + c) = make_uint2(lo, hi);
    } else {
      float* dst = reinterpret_cast<float*>(xq) + size_t(t) * d + c;
      *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
      *reinterpret_cast<float4*>(dst + 4) = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
  if (lane == 0) sx[t] = s;
}

// ------------------------------------------------------------ gate/up, FP8 -----------------
struct ExpertArgs {
  int d, F, E, T, R;  // R = T (k + 1) rows
  const uint8_t* wgu;
  const float* sgu;
  const uint8_t* wd;
  const float* sd;
  const uint8_t* sh_wgu;
  const float* sh_sgu;
  const uint8_t* sh_wd;
  const float* sh_sd;
  const Tile* tiles;
  const int* n_tiles;
  const int32_t* perm;  // [R] token of each row
  const uint8_t* xq;    // [T, d] E4M3 in token order (or fp32 for the fp32 path)
  const float* sx;      // [T]
  float* h;           // [R, F]
  uint8_t* qh;        // [R, F]
  float* sh;          // [R]
  void* y_rows;       // [R, d]: bf16 rows (E4M3 layers) or fp32 rows (fp32 layers)
};

constexpr int kTG = kStreamRows / 8;     // token groups of 8 rows per tile

// Bulk-copy (TMA) pipeline shared by the two streaming kernels: one producer warp copies
// whole weight rows and activation rows of a work item into a shared-memory stage with
// cp.async.bulk (completion counted on the stage's "full" mbarrier); four MMA warps wait on
// it, compute, and release the stage on its "empty" mbarrier.  Rows are stored with a
// 16-byte pad so the fragment loads of 8 consecutive rows hit distinct banks.  Every wait is
// bounded (tma.cuh); on a timeout the CTA records MOE_ERR_TIMEOUT, the producer stops, the
// MMA warps leave at the same stage wait, and the producer waits for its copies in flight
// before the CTA exits.
constexpr int kConsumerWarps = 4;
constexpr int kStreamThreads = (kConsumerWarps + 1) * 32;
constexpr int kRowPad = 16;

struct PipeCtl {
  uint64_t full[8];
  uint64_t empty[8];
  int abort;
};

__device__ __forceinline__ void pipe_init(PipeCtl* ctl, int stages) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], kConsumerWarps);
    }
    ctl->abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
}

__device__ __forceinline__ void report_timeout(int* status_flags, int site) { report_timeout_flag(status_flags, site); }

// Producer epilogue: wait (bounded, ignoring the abort flag) until the last copies issued
// into every stage have landed, so no bulk copy targets this CTA's shared memory after exit.
__device__ __forceinline__ void pipe_drain(PipeCtl* ctl, int stages, int issued) {
  for (int s = 0; s < stages && s < issued; ++s) {
    const int last_use = (issued - 1 - s) / stages;  // uses of stage s: j = s, s + stages, ...
    int zero = 0;
    mbar_wait(&ctl->full[s], last_use & 1, &zero);
  }
}

// ------------------------------------------------------------ gate/up, FP8 -----------------
// Work item = (tile of <= kStreamRows rows, 16 output columns n of gate and of up).  The
// stage holds the 16 gate rows, the 16 up rows and the tile's activation rows (E4M3), all of
// length d.  MMA warp w covers k in [w*d/4, (w+1)*d/4); the four partial sums meet in shared
// memory; the epilogue forms h = silu(g) u.
constexpr int kGuStages = 2;

__global__ void __launch_bounds__(kStreamThreads) k_gateup_fp8(ExpertArgs a, int* status_flags) {
  extern __shared__ __align__(128) uint8_t gu_smem[];
  const int rs = a.d + kRowPad;
  const size_t stage_bytes = size_t(48) * rs;
  float (*red)[kTG][2][4][32] =
      reinterpret_cast<float (*)[kTG][2][4][32]>(gu_smem + kGuStages * stage_bytes);
  PipeCtl* ctl = reinterpret_cast<PipeCtl*>(gu_smem + kGuStages * stage_bytes + sizeof(float) * kConsumerWarps * kTG * 2 * 4 * 32);
  pipe_init(ctl, kGuStages);
  pdl_begin();
  const int n_tiles = *a.n_tiles;
  const int nblk = a.F / 16;
  const int total = n_tiles * nblk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == kConsumerWarps) {  // ---------------- producer
    const uint64_t pol = policy_evict_first();
    int j = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++j) {
      const int s = j % kGuStages, use = j / kGuStages;
      if (!mbar_wait(&ctl->empty[s], (use & 1) ^ 1, &ctl->abort)) {
        if (lane == 0) report_timeout(status_flags, 1);
        break;
      }
      const Tile tl = checked_tile(a.tiles, item / nblk, a.E, a.R, kStreamRows, status_flags, 11);
      const int n0 = (item % nblk) * 16;
      const uint8_t* Wg = tl.group == a.E ? a.sh_wgu : a.wgu + size_t(tl.group) * 2 * a.F * a.d;
      uint8_t* st = gu_smem + s * stage_bytes;
      if (lane == 0) mbar_arrive_expect_tx(&ctl->full[s], uint32_t((32 + tl.nrows) * a.d));
      __syncwarp();
      // lanes 0..15: gate rows n0 + lane; lanes 16..31: up rows n0 + lane - 16
      const uint8_t* src = Wg + (lane < 16 ? size_t(n0 + lane) : size_t(a.F + n0 + lane - 16)) * a.d;
      bulk_g2s_stream(st + lane * rs, src, a.d, &ctl->full[s], pol);
      if (lane < tl.nrows)
        bulk_g2s(st + (32 + lane) * rs, a.xq + size_t(checked_token(a.perm[tl.row0 + lane], a.T, status_flags, 12)) * a.d,
                 a.d, &ctl->full[s]);
    }
    pipe_drain(ctl, kGuStages, j);
    return;
  }

  // ---------------- MMA warps
  const int gq = lane >> 2, tig = lane & 3;
  const int kq = a.d / kConsumerWarps;
  int j = 0;
  for (int item = blockIdx.x; item < total; item += gridDim.x, ++j) {
    const int s = j % kGuStages, use = j / kGuStages;
    if (!mbar_wait(&ctl->full[s], use & 1, &ctl->abort)) {
      if (lane == 0) report_timeout(status_flags, 2);
      break;
    }
    const Tile tl = checked_tile(a.tiles, item / nblk, a.E, a.R, kStreamRows, status_flags, 13);
    const int n0 = (item % nblk) * 16;
    const int ntg = (tl.nrows + 7) >> 3;
    const uint8_t* st = gu_smem + s * stage_bytes;
    const int koff = warp * kq + tig * 16;
    float acc[kTG][2][4];
#pragma unroll
    for (int tg = 0; tg < kTG; ++tg)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[tg][jj][c] = 0.0f;
    for (int ks = 0; ks < kq; ks += 64) {
      const uint4 g0 = *reinterpret_cast<const uint4*>(st + gq * rs + koff + ks);
      const uint4 g1 = *reinterpret_cast<const uint4*>(st + (gq + 8) * rs + koff + ks);
      const uint4 u0 = *reinterpret_cast<const uint4*>(st + (16 + gq) * rs + koff + ks);
      const uint4 u1 = *reinterpret_cast<const uint4*>(st + (24 + gq) * rs + koff + ks);
#pragma unroll
      for (int tg = 0; tg < kTG; ++tg) {
        if (tg < ntg) {
          const int r = tg * 8 + gq;
          const uint4 xa = r < tl.nrows ? *reinterpret_cast<const uint4*>(st + (32 + r) * rs + koff + ks)
                                        : make_uint4(0, 0, 0, 0);
          mma_e4m3_16x8x32(acc[tg][0], g0.x, g1.x, g0.y, g1.y, xa.x, xa.y);
          mma_e4m3_16x8x32(acc[tg][0], g0.z, g1.z, g0.w, g1.w, xa.z, xa.w);
          mma_e4m3_16x8x32(acc[tg][1], u0.x, u1.x, u0.y, u1.y, xa.x, xa.y);
          mma_e4m3_16x8x32(acc[tg][1], u0.z, u1.z, u0.w, u1.w, xa.z, xa.w);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl->empty[s]);
#pragma unroll
    for (int tg = 0; tg < kTG; ++tg)
      if (tg < ntg)
#pragma unroll
        for (int jj = 0; jj < 2; ++jj)
#pragma unroll
          for (int c = 0; c < 4; ++c) red[warp][tg][jj][c][lane] = acc[tg][jj][c];
    named_bar_sync(1, kConsumerWarps * 32);
    const int tg = warp;
    if (tg < ntg) {
      const bool shared = tl.group == a.E;
      const float* sg = shared ? a.sh_sgu : a.sgu + size_t(tl.group) * 2 * a.F;
      const float* su = sg + a.F;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float gsum = 0.0f, usum = 0.0f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          gsum += red[w][tg][0][c][lane];
          usum += red[w][tg][1][c][lane];
        }
        const int r = tg * 8 + tig * 2 + (c & 1);
        const int n = n0 + gq + ((c & 2) ? 8 : 0);
        if (r < tl.nrows) {
          const int row = tl.row0 + r;
          const float sx = a.sx[checked_token(a.perm[row], a.T, status_flags, 14)];
          const float gv = gsum * sx * sg[n];
          const float uv = usum * sx * su[n];
          a.h[size_t(row) * a.F + n] = silu(gv) * uv;
        }
      }
    }
    named_bar_sync(1, kConsumerWarps * 32);
  }
}

// ------------------------------------------------------------ h quantisation ---------------
// One warp per row of a tile: sh = max|h| / 448 (1 if the row is zero), qh = E4M3(h / sh).
// Rows are taken in order 0..R-1; rows that no tile covers (slots of rejected forced ids)
// are quantised too, harmlessly: nothing reads them.
__global__ void __launch_bounds__(256) k_hquant(ExpertArgs a, int R) {
  pdl_trigger_then_wait();
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long row_l = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row_l < R; row_l += nwarps) {
    const int row = int(row_l);
    const float* hr = a.h + size_t(row) * a.F;
    float4 v[5];  // ffn <= 640 = 5 x 32 lanes x 4
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 5; ++j) {
      const int n = (j * 32 + lane) * 4;
      v[j] = n < a.F ? *reinterpret_cast<const float4*>(hr + n) : make_float4(0.f, 0.f, 0.f, 0.f);
      amax = fmaxf(fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))), amax);
    }
    for (int n = 640 + lane * 4; n < a.F; n += 128) {  // wider ffn: rare, second pass for the max
      const float4 u = *reinterpret_cast<const float4*>(hr + n);
      amax = fmaxf(fmaxf(fmaxf(fabsf(u.x), fabsf(u.y)), fmaxf(fabsf(u.z), fabsf(u.w))), amax);
    }
    amax = warp_max(amax);
    const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    uint8_t* qr = a.qh + size_t(row) * a.F;
#pragma unroll
    for (int j = 0; j < 5; ++j) {
      const int n = (j * 32 + lane) * 4;
      if (n < a.F)
        *reinterpret_cast<uint32_t*>(qr + n) = uint32_t(e4m3_code2(__fdiv_rn(v[j].x, s), __fdiv_rn(v[j].y, s))) |
                                               (uint32_t(e4m3_code2(__fdiv_rn(v[j].z, s), __fdiv_rn(v[j].w, s))) << 16);
    }
    for (int n = 640 + lane * 4; n < a.F; n += 128) {
      const float4 u = *reinterpret_cast<const float4*>(hr + n);
      *reinterpret_cast<uint32_t*>(qr + n) = uint32_t(e4m3_code2(__fdiv_rn(u.x, s), __fdiv_rn(u.y, s))) |
                                             (uint32_t(e4m3_code2(__fdiv_rn(u.z, s), __fdiv_rn(u.w, s))) << 16);
    }
    if (lane == 0) a.sh[row] = s;
  }
}

// ------------------------------------------------------------ down, FP8 --------------------
// Work item = (tile of <= kStreamRows rows, 64 output columns m).  The stage holds the 64
// weight rows (length ffn) and the tile's quantised h rows; MMA warp w owns 16 of the m
// columns and the whole k = ffn range, so no cross-warp reduction is needed.
constexpr int kDnStages = 4;

__global__ void __launch_bounds__(kStreamThreads) k_down_fp8(ExpertArgs a, int* status_flags) {
  extern __shared__ __align__(128) uint8_t dn_smem[];
  const int rs = a.F + kRowPad;
  const size_t stage_bytes = size_t(64 + kStreamRows) * rs;
  PipeCtl* ctl = reinterpret_cast<PipeCtl*>(dn_smem + kDnStages * stage_bytes);
  pipe_init(ctl, kDnStages);
  pdl_begin();
  const int n_tiles = *a.n_tiles;
  const int nblk = a.d / 64;
  const int total = n_tiles * nblk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == kConsumerWarps) {  // ---------------- producer
    const uint64_t pol = policy_evict_first();
    int j = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++j) {
      const int s = j % kDnStages, use = j / kDnStages;
      if (!mbar_wait(&ctl->empty[s], (use & 1) ^ 1, &ctl->abort)) {
        if (lane == 0) report_timeout(status_flags, 3);
        break;
      }
      const Tile tl = checked_tile(a.tiles, item / nblk, a.E, a.R, kStreamRows, status_flags, 15);
      const int m0 = (item % nblk) * 64;
      const uint8_t* W = tl.group == a.E ? a.sh_wd : a.wd + size_t(tl.group) * a.d * a.F;
      uint8_t* st = dn_smem + s * stage_bytes;
      if (lane == 0) mbar_arrive_expect_tx(&ctl->full[s], uint32_t((64 + tl.nrows) * a.F));
      __syncwarp();
      bulk_g2s_stream(st + lane * rs, W + size_t(m0 + lane) * a.F, a.F, &ctl->full[s], pol);
      bulk_g2s_stream(st + (32 + lane) * rs, W + size_t(m0 + 32 + lane) * a.F, a.F, &ctl->full[s], pol);
      if (lane < tl.nrows) bulk_g2s(st + (64 + lane) * rs, a.qh + size_t(tl.row0 + lane) * a.F, a.F, &ctl->full[s]);
    }
    pipe_drain(ctl, kDnStages, j);
    return;
  }

  const int gq = lane >> 2, tig = lane & 3;
  int j = 0;
  for (int item = blockIdx.x; item < total; item += gridDim.x, ++j) {
    const int s = j % kDnStages, use = j / kDnStages;
    if (!mbar_wait(&ctl->full[s], use & 1, &ctl->abort)) {
      if (lane == 0) report_timeout(status_flags, 4);
      break;
    }
    const Tile tl = checked_tile(a.tiles, item / nblk, a.E, a.R, kStreamRows, status_flags, 16);
    const int mw = warp * 16;  // this warp's columns within the item
    const int m0 = (item % nblk) * 64 + mw;
    const int ntg = (tl.nrows + 7) >> 3;
    const uint8_t* st = dn_smem + s * stage_bytes;
    float acc[kTG][4];
#pragma unroll
    for (int tg = 0; tg < kTG; ++tg)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[tg][c] = 0.0f;
    for (int ks = tig * 16; ks < a.F; ks += 64) {
      const uint4 w0 = *reinterpret_cast<const uint4*>(st + (mw + gq) * rs + ks);
      const uint4 w1 = *reinterpret_cast<const uint4*>(st + (mw + gq + 8) * rs + ks);
#pragma unroll
      for (int tg = 0; tg < kTG; ++tg) {
        if (tg < ntg) {
          const int r = tg * 8 + gq;
          const uint4 xa = r < tl.nrows ? *reinterpret_cast<const uint4*>(st + (64 + r) * rs + ks) : make_uint4(0, 0, 0, 0);
          mma_e4m3_16x8x32(acc[tg], w0.x, w1.x, w0.y, w1.y, xa.x, xa.y);
          mma_e4m3_16x8x32(acc[tg], w0.z, w1.z, w0.w, w1.w, xa.z, xa.w);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl->empty[s]);
    const float* sdn = tl.group == a.E ? a.sh_sd : a.sd + size_t(tl.group) * a.d;
#pragma unroll
    for (int tg = 0; tg < kTG; ++tg) {
      if (tg >= ntg) continue;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int r = tg * 8 + tig * 2 + (c & 1);
        const int m = m0 + gq + ((c & 2) ? 8 : 0);
        if (r < tl.nrows) {
          const int row = tl.row0 + r;
          static_cast<__nv_bfloat16*>(a.y_rows)[size_t(row) * a.d + m] = __float2bfloat16_rn(acc[tg][c] * a.sh[row] * sdn[m]);
        }
      }
    }
  }
}

// ------------------------------------------------------------ fp32 experts -----------------
// fp32 weights and activations (no quantisation): one warp per (tile, output column),
// lanes split k, for every row of the tile.
__global__ void __launch_bounds__(256) k_gateup_f32(ExpertArgs a) {
  pdl_begin();
  const int n_tiles = *a.n_tiles;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const float* xf = reinterpret_cast<const float*>(a.xq);
  for (int item = warp; item < n_tiles * a.F; item += nwarps) {
    const Tile tl = a.tiles[item / a.F];
    const int n = item % a.F;
    const float* Wg = tl.group == a.E ? reinterpret_cast<const float*>(a.sh_wgu)
                                      : reinterpret_cast<const float*>(a.wgu) + size_t(tl.group) * 2 * a.F * a.d;
    const float* wg = Wg + size_t(n) * a.d;
    const float* wu = Wg + size_t(a.F + n) * a.d;
    for (int r = 0; r < tl.nrows; ++r) {
      const float* xr = xf + size_t(a.perm[tl.row0 + r]) * a.d;
      float gs = 0.0f, us = 0.0f;
      for (int k = lane; k < a.d; k += 32) {
        gs = fmaf(xr[k], wg[k], gs);
        us = fmaf(xr[k], wu[k], us);
      }
      gs = warp_sum(gs);
      us = warp_sum(us);
      if (lane == 0) a.h[size_t(tl.row0 + r) * a.F + n] = silu(gs) * us;
    }
  }
}

__global__ void __launch_bounds__(256) k_down_f32(ExpertArgs a) {
  pdl_begin();
  const int n_tiles = *a.n_tiles;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  for (int item = warp; item < n_tiles * a.d; item += nwarps) {
    const Tile tl = a.tiles[item / a.d];
    const int m = item % a.d;
    const float* W = tl.group == a.E ? reinterpret_cast<const float*>(a.sh_wd)
                                     : reinterpret_cast<const float*>(a.wd) + size_t(tl.group) * a.d * a.F;
    const float* wr = W + size_t(m) * a.F;
    for (int r = 0; r < tl.nrows; ++r) {
      const float* hr = a.h + size_t(tl.row0 + r) * a.F;
      float s = 0.0f;
      for (int n = lane; n < a.F; n += 32) s = fmaf(hr[n], wr[n], s);
      s = warp_sum(s);
      if (lane == 0) static_cast<float*>(a.y_rows)[size_t(tl.row0 + r) * a.d + m] = s;
    }
  }
}

// ------------------------------------------------------------ combine ----------------------
// y[t] = Y[shared row of t] + sum_i w[t,i] Y[pos[t,i]] in slot order, in fp32; optionally
// r <- bf16(r + y) on a bf16 residual held in `out`.  Y holds bf16 rows (E4M3 layers) or fp32
// rows (fp32 layers).  One CTA per token, eight consecutive columns per thread and pass: the
// seven row loads of a pass are all issued before the first add, so a pass costs one memory
// latency, not seven.
__device__ __forceinline__ void load_row8(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    v[2 * j] = __uint_as_float(w[j] << 16);
    v[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
  }
}
__device__ __forceinline__ void load_row8(const __nv_bfloat16* p, float (&v)[8]) {
  bf16x8_to_f32(*reinterpret_cast<const uint4*>(p), v);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// kMinCtas: CTAs per SM the register budget allows (4 for many tokens per CTA, where the
// extra CTA hides more latency; 3 otherwise, without the spills the 64-register cap costs)
template <typename OT, bool kResidual, typename YT, int kMinCtas>
__global__ void __launch_bounds__(256, kMinCtas) k_combine(const YT* __restrict__ y_rows, const int32_t* __restrict__ pos,
                                                 const float* __restrict__ w, int T, int d, int k, OT* __restrict__ out,
                                                 int* status_flags) {
  // A few CTAs per SM walk the tokens; a token's slots (rows and weights) are loaded while the
  // previous token's rows are in flight.  The first token's slots come from the dispatch,
  // which completed before the kernel this launch overlaps started: read before the wait.
  int rows[kTopK];
  float wt[kTopK];
  auto load_slots = [&](int t, int (&r)[kTopK], float (&ww)[kTopK]) {
#pragma unroll
    for (int i = 0; i < kTopK; ++i) {
      const bool ok = t < T && i < k;
      r[i] = ok ? pos[size_t(t) * k + i] : -1;
      if (kDebugIndexChecks && r[i] >= k * T) {  // a routed row lies in [0, kT); -1 marks a dropped slot
        report_index(status_flags, 17);
        r[i] = -1;
      }
      ww[i] = ok ? w[size_t(t) * k + i] : 0.0f;
    }
  };
  int t = blockIdx.x;
  load_slots(t, rows, wt);
  pdl_begin();
  for (; t < T; t += gridDim.x) {
    int nrows[kTopK];
    float nwt[kTopK];
    load_slots(t + int(gridDim.x), nrows, nwt);
    const YT* ysh = y_rows + (size_t(k) * T + t) * d;
    for (int m = threadIdx.x * 8; m < d; m += blockDim.x * 8) {
      float acc[8], v[kTopK][8];
      load_row8(ysh + m, acc);
#pragma unroll
      for (int i = 0; i < kTopK; ++i)
        if (rows[i] >= 0) load_row8(y_rows + size_t(rows[i]) * d + m, v[i]);
#pragma unroll
      for (int i = 0; i < kTopK; ++i)
        if (rows[i] >= 0) {
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[j] = fmaf(wt[i], v[i][j], acc[j]);
        }
      OT* o = out + size_t(t) * d + m;
      if constexpr (sizeof(OT) == 4) {
        *reinterpret_cast<float4*>(o) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        *reinterpret_cast<float4*>(o + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
      } else {
        if (kResidual) {
          float r[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(o), r);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[j] += r[j];
        }
        *reinterpret_cast<uint4*>(o) = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                                  pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
      }
    }
#pragma unroll
    for (int i = 0; i < kTopK; ++i) {
      rows[i] = nrows[i];
      wt[i] = nwt[i];
    }
  }
}

__global__ void k_e4m3_encode(const float* __restrict__ in, uint8_t* __restrict__ out, int64_t n) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x)
    out[i] = e4m3_code(in[i]);
}

int num_sms() {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  return sms;
}

}  // namespace

cudaError_t launch_act_quant(const void* x, bool x_bf16, int T, const LayerDev& L, void* xq, float* sx,
                             cudaStream_t s) {
  const dim3 grid((T + 7) / 8);  // a warp per token
  if (x_bf16) {
    if (L.fp8)
      return launch_pdl(k_act_quant<__nv_bfloat16, true>, grid, dim3(256), 0, s, (const __nv_bfloat16*)x, T, L.d, xq, sx);
    return launch_pdl(k_act_quant<__nv_bfloat16, false>, grid, dim3(256), 0, s, (const __nv_bfloat16*)x, T, L.d, xq, sx);
  }
  if (L.fp8) return launch_pdl(k_act_quant<float, true>, grid, dim3(256), 0, s, (const float*)x, T, L.d, xq, sx);
  return launch_pdl(k_act_quant<float, false>, grid, dim3(256), 0, s, (const float*)x, T, L.d, xq, sx);
}

namespace {
ExpertArgs expert_args(const LayerDev& L, const WsLayout& ws, char* base) {
  ExpertArgs a;
  a.d = L.d;
  a.F = L.F;
  a.E = L.E;
  a.T = ws.T;
  a.R = ws.R;
  a.wgu = L.wgu;
  a.sgu = L.sgu;
  a.wd = L.wd;
  a.sd = L.sd;
  a.sh_wgu = L.sh_wgu;
  a.sh_sgu = L.sh_sgu;
  a.sh_wd = L.sh_wd;
  a.sh_sd = L.sh_sd;
  a.tiles = reinterpret_cast<const Tile*>(base + ws.tiles);
  a.n_tiles = reinterpret_cast<const int*>(base + ws.n_tiles);
  a.perm = reinterpret_cast<const int32_t*>(base + ws.perm);
  a.xq = reinterpret_cast<const uint8_t*>(base + ws.xq);
  a.sx = reinterpret_cast<const float*>(base + ws.sx);
  a.h = reinterpret_cast<float*>(base + ws.h);
  a.qh = reinterpret_cast<uint8_t*>(base + ws.qh);
  a.sh = reinterpret_cast<float*>(base + ws.sh);
  a.y_rows = base + ws.y_rows;
  return a;
}

// Upper bound of the tile count: one partial tile per non-empty group plus full tiles.
long long max_stream_tiles(const LayerDev& L, int T) {
  const long long R = (long long)T * (L.k + 1);
  return std::min<long long>(R, L.E + 1) + R / kStreamRows;
}
}  // namespace

size_t gateup_smem(int d) {
  return size_t(kGuStages) * 48 * (d + kRowPad) + sizeof(float) * kConsumerWarps * kTG * 2 * 4 * 32 + sizeof(PipeCtl);
}
size_t down_smem(int F) { return size_t(kDnStages) * (64 + kStreamRows) * (F + kRowPad) + sizeof(PipeCtl); }

cudaError_t launch_gateup_stream(const LayerDev& L, int T, const WsLayout& ws, char* base, cudaStream_t s) {
  const ExpertArgs a = expert_args(L, ws, base);
  const long long tiles = max_stream_tiles(L, T);
  const int sms = num_sms();
  if (L.fp8) {
    const size_t smem = gateup_smem(L.d);
    static cudaError_t attr = cudaFuncSetAttribute(k_gateup_fp8, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   int(gateup_smem(2048)));
    if (attr != cudaSuccess) return attr;
    const long long items = tiles * (L.F / 16);
    int* flags = reinterpret_cast<int*>(base + ws.status);
    return launch_pdl(k_gateup_fp8, dim3(int(std::min<long long>(items, sms))), dim3(kStreamThreads), smem, s, a, flags);
  }
  const long long items = tiles * L.F / 8;
  return launch_pdl(k_gateup_f32, dim3(int(std::min<long long>(items, (long long)sms * 16))), dim3(256), 0, s, a);
}

cudaError_t launch_hquant(const LayerDev& L, int T, const WsLayout& ws, char* base, int rows_per_tile, cudaStream_t s) {
  if (!L.fp8) return cudaSuccess;
  const ExpertArgs a = expert_args(L, ws, base);
  (void)rows_per_tile;
  const int R = T * (L.k + 1);
  return launch_pdl(k_hquant, dim3(int(std::min<long long>((R + 7) / 8, (long long)num_sms() * 16))), dim3(256), 0, s,
                    a, R);
}

cudaError_t launch_down_stream(const LayerDev& L, int T, const WsLayout& ws, char* base, cudaStream_t s) {
  const ExpertArgs a = expert_args(L, ws, base);
  const long long tiles = max_stream_tiles(L, T);
  const int sms = num_sms();
  if (L.fp8) {
    const size_t smem = down_smem(L.F);
    static cudaError_t attr = cudaFuncSetAttribute(k_down_fp8, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   int(down_smem(640)));
    if (attr != cudaSuccess) return attr;
    const long long items = tiles * (L.d / 64);
    int* flags = reinterpret_cast<int*>(base + ws.status);
    return launch_pdl(k_down_fp8, dim3(int(std::min<long long>(items, sms))), dim3(kStreamThreads), smem, s, a, flags);
  }
  const long long items = tiles * L.d / 8;
  return launch_pdl(k_down_f32, dim3(int(std::min<long long>(items, (long long)sms * 16))), dim3(256), 0, s, a);
}

template <typename YT, int kMinCtas>
cudaError_t launch_combine_k(const YT* y_rows, const int32_t* pos, const float* w, int T, const LayerDev& L, void* y,
                             moe_dtype y_dtype, bool residual_add, int* status_flags, cudaStream_t s) {
  const dim3 grid(std::max(1, std::min(T, num_sms() * kMinCtas)));
  if (y_dtype == MOE_F32)
    return launch_pdl(k_combine<float, false, YT, kMinCtas>, grid, dim3(256), 0, s, y_rows, pos, w, T, L.d, L.k,
                      (float*)y, status_flags);
  if (residual_add)
    return launch_pdl(k_combine<__nv_bfloat16, true, YT, kMinCtas>, grid, dim3(256), 0, s, y_rows, pos, w, T, L.d,
                      L.k, (__nv_bfloat16*)y, status_flags);
  return launch_pdl(k_combine<__nv_bfloat16, false, YT, kMinCtas>, grid, dim3(256), 0, s, y_rows, pos, w, T, L.d, L.k,
                    (__nv_bfloat16*)y, status_flags);
}

template <typename YT>
cudaError_t launch_combine_t(const YT* y_rows, const int32_t* pos, const float* w, int T, const LayerDev& L, void* y,
                             moe_dtype y_dtype, bool residual_add, int* status_flags, cudaStream_t s) {
  if (T > num_sms() * 8)  // CTAs walk several tokens each
    return launch_combine_k<YT, 4>(y_rows, pos, w, T, L, y, y_dtype, residual_add, status_flags, s);
  return launch_combine_k<YT, 3>(y_rows, pos, w, T, L, y, y_dtype, residual_add, status_flags, s);
}

cudaError_t launch_combine(const void* y_rows, const int32_t* pos, const float* w, int T, const LayerDev& L, void* y,
                           moe_dtype y_dtype, bool residual_add, int* status_flags, cudaStream_t s) {
  if (L.fp8)
    return launch_combine_t(static_cast<const __nv_bfloat16*>(y_rows), pos, w, T, L, y, y_dtype, residual_add,
                            status_flags, s);
  return launch_combine_t(static_cast<const float*>(y_rows), pos, w, T, L, y, y_dtype, residual_add, status_flags, s);
}

cudaError_t launch_e4m3_encode(const float* in, uint8_t* out, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int grid = int(std::min<int64_t>((n + 255) / 256, int64_t(num_sms()) * 32));
  k_e4m3_encode<<<grid, 256, 0, s>>>(in, out, n);
  return cudaGetLastError();
}

}  // namespace moe
