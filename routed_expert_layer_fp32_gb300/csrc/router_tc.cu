// Prefill router on the tensor cores with fp32 accuracy.
//
// The router is float32 ("We Ported Aleph Alpha's Kolibri to a MacBook. Our Own Gate Said
// No.", section "The gate": a bf16 router is one of the planted bugs).  Activations arrive in
// bf16, so x is exact in bf16; the fp32 router weights are split per call into three bf16
// terms, w = hi + mid + lo (+ a remainder below 2^-24 |w|): hi = bf16(w), mid = bf16(w - hi),
// lo = bf16(w - hi - mid), where both differences are exact in fp32.  Every product of bf16
// values is exact in fp32, so three accumulating bf16 MMAs with an fp32 accumulator give
// x . w to fp32 accuracy.
//
// Tile: 128 tokens (M) x all experts, the experts split into two MMAs of n_half columns
// (E = 384: 2 x 192) so one TMEM accumulator row holds a token's full logit row.  The two CTAs
// of a cluster work on two token tiles in lockstep and share the weight stream: each loads one
// n_half block of every (k-slice, term) weight stage and multicasts it to both, so each CTA
// reads half of the 4.7 MB of weight terms per tile pair from L2.  The x k-slice (16 KB) has
// its own ring and is loaded once for the three terms.  Warp roles as in the expert GEMMs
// (TMA producer, single-thread MMA issuer, four epilogue warps); bounded waits.  A CTA whose
// pair partner has a tile but it has none still loads and releases its weight halves.
#include "common.cuh"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace moe {
namespace {

constexpr int kRtThreads = 192;
constexpr int kRtM = 128;
constexpr int kRtATile = kRtM * 128;
constexpr size_t kRtSmemBudget = 200 * 1024;

__global__ void k_router_split_w(const float* __restrict__ Wr, long long n, __nv_bfloat16* __restrict__ out) {
  pdl_begin();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const float w = Wr[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    out[i] = hi;
    out[n + i] = mid;
    out[2 * n + i] = __float2bfloat16_rn(r2);
  }
}

constexpr int kRtC = 2;       // CTAs per cluster sharing the weight stream
constexpr int kRtMaxStages = 4;

struct RtCtl {
  uint64_t full_a[kRtMaxStages];
  uint64_t empty_a[kRtMaxStages];
  uint64_t full_b[kRtMaxStages];
  uint64_t empty_b[kRtMaxStages];  // one arrival per CTA of the cluster
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

__global__ void __launch_bounds__(kRtThreads, 1)
    k_router_tc(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                const float* __restrict__ bias, const float* __restrict__ sel_bias, int T, int d, int E, int n_half,
                int n_a, int n_b, int tmem_cols,
                float* __restrict__ logits, int32_t* __restrict__ ids, float* __restrict__ wts, int k,
                int* status_flags) {
  extern __shared__ uint8_t rt_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rt_smem_raw) + 1023) & ~uintptr_t(1023));
  const int b_half_bytes = n_half * 128;
  const int b_stage_bytes = 2 * b_half_bytes;
  uint8_t* ring_a = smem;
  uint8_t* ring_b = smem + size_t(n_a) * kRtATile;
  RtCtl* ctl = reinterpret_cast<RtCtl*>(ring_b + size_t(n_b) * b_stage_bytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = int(cluster_ctarank());
  const int pair = int(blockIdx.x) / kRtC, n_pairs = int(gridDim.x) / kRtC;
  if (threadIdx.x == 0) {
    for (int s = 0; s < n_a; ++s) {
      mbar_init(&ctl->full_a[s], 1);
      mbar_init(&ctl->empty_a[s], 1);
    }
    for (int s = 0; s < n_b; ++s) {
      mbar_init(&ctl->full_b[s], 1);
      mbar_init(&ctl->empty_b[s], kRtC);
    }
    mbar_init(&ctl->acc_full, 1);
    mbar_init(&ctl->acc_empty, 4);
    mbar_init(&ctl->mma_done, 1);
    ctl->abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the partner's barriers exist before any multicast or remote arrival
  tc_fence_after();
  pdl_begin();
  const uint32_t tmem = ctl->tmem_base;
  const int n_items = (T + kRtM - 1) / kRtM;
  const int KT = d / 64;  // 64 bf16 per 128-byte k-slice
  constexpr uint16_t kBoth = (1u << kRtC) - 1u;
  // round j: the pair's tiles are kRtC * (pair + j * n_pairs) + rank; the cluster runs while
  // rank 0's tile exists, rank 1 possibly without a tile of its own ("phantom")
  auto tile_of = [&](int j, int r) { return kRtC * (pair + j * n_pairs) + r; };
  auto sa = [&](int s) { return ring_a + size_t(s) * kRtATile; };
  auto sb = [&](int s, int h) { return ring_b + size_t(s) * b_stage_bytes + h * b_half_bytes; };

  if (warp == 0) {
    if (lane == 0) {  // TMA producer: x slice per k-slice (own tile), weight half per (k-slice, term)
      int ia = 0, ib = 0;
      bool stop = false;
      for (int j = 0; tile_of(j, 0) < n_items && !stop; ++j) {
        const int item = tile_of(j, rank);
        const bool real = item < n_items;
        for (int kt = 0; kt < KT && !stop; ++kt) {
          if (real) {
            const int s = ia % n_a, use = ia / n_a;
            if (!mbar_wait(&ctl->empty_a[s], (use & 1) ^ 1, &ctl->abort)) {
              report_timeout_flag(status_flags, 21);
              stop = true;
              break;
            }
            mbar_arrive_expect_tx(&ctl->full_a[s], kRtATile);
            tma_load_2d(sa(s), &map_x, kt * 64, item * kRtM, &ctl->full_a[s]);
            ++ia;
          }
          for (int term = 0; term < 3; ++term, ++ib) {
            const int s = ib % n_b, use = ib / n_b;
            if (!mbar_wait(&ctl->empty_b[s], (use & 1) ^ 1, &ctl->abort)) {
              report_timeout_flag(status_flags, 25);
              stop = true;
              break;
            }
            mbar_arrive_expect_tx(&ctl->full_b[s], b_stage_bytes);  // both halves land here
            tma_load_2d_mc(sb(s, rank), &map_w, kt * 64, term * E + rank * n_half, &ctl->full_b[s], kBoth);
          }
        }
      }
      for (int s = 0; s < n_a && s < ia; ++s) {
        int zero = 0;
        mbar_wait(&ctl->full_a[s], ((ia - 1 - s) / n_a) & 1, &zero);
      }
      for (int s = 0; s < n_b && s < ib; ++s) {
        int zero = 0;
        mbar_wait(&ctl->full_b[s], ((ib - 1 - s) / n_b) & 1, &zero);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      const uint32_t idesc = idesc_bf16(kRtM, n_half);
      int ia = 0, ib = 0, jt = 0;
      bool stop = false;
      for (int j = 0; tile_of(j, 0) < n_items && !stop; ++j) {
        const bool real = tile_of(j, rank) < n_items;
        if (real) {
          if (!mbar_wait(&ctl->acc_empty, (jt & 1) ^ 1, &ctl->abort)) {
            report_timeout_flag(status_flags, 22);
            break;
          }
          tc_fence_after();
        }
        for (int kt = 0; kt < KT && !stop; ++kt) {
          const int sa_i = ia % n_a;
          if (real && !mbar_wait(&ctl->full_a[sa_i], (ia / n_a) & 1, &ctl->abort)) {
            report_timeout_flag(status_flags, 23);
            stop = true;
            break;
          }
          for (int term = 0; term < 3; ++term, ++ib) {
            const int s = ib % n_b, use = ib / n_b;
            if (!mbar_wait(&ctl->full_b[s], use & 1, &ctl->abort)) {
              report_timeout_flag(status_flags, 26);
              stop = true;
              break;
            }
            tc_fence_after();
            if (real) {
              const uint64_t da = sw128_desc(sa(sa_i));
              const uint64_t db0 = sw128_desc(sb(s, 0)), db1 = sw128_desc(sb(s, 1));
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {  // 16 bf16 (32 bytes) per MMA
                const uint32_t acc = (kt > 0 || term > 0 || kk > 0) ? 1u : 0u;
                tc_mma_f16(tmem, da + 2 * kk, db0 + 2 * kk, idesc, acc);
                tc_mma_f16(tmem + uint32_t(n_half), da + 2 * kk, db1 + 2 * kk, idesc, acc);
              }
            }
            tc_commit_mc(&ctl->empty_b[s], kBoth);  // this CTA is done with both halves
          }
          if (stop) break;
          if (real) {
            tc_commit(&ctl->empty_a[sa_i]);
            ++ia;
          }
        }
        if (real && !stop) {
          tc_commit(&ctl->acc_full);
          ++jt;
        }
      }
      tc_commit(&ctl->mma_done);
      int zero = 0;
      mbar_wait(&ctl->mma_done, 0, &zero);
    }
  } else {  // epilogue: one token per TMEM lane, logits = acc + bias
    // With ids != nullptr the epilogue also selects: a sorted list of the kTopK best scores
    // (larger first, lower index first on equal scores; the scan visits experts in increasing
    // index, so an equal later score never displaces an earlier one), then the softmax over
    // the selected logits, summed in slot order.  The score is the logit, plus sel_bias in the
    // selection-only bias mode.
    const int q = warp & 3;
    int jt = 0;
    for (int j = 0; tile_of(j, rank) < n_items; ++j, ++jt) {
      const int item = tile_of(j, rank);
      if (!mbar_wait(&ctl->acc_full, jt & 1, &ctl->abort)) {
        if (lane == 0) report_timeout_flag(status_flags, 24);
        break;
      }
      tc_fence_after();
      const int t = item * kRtM + q * 32 + lane;
      const uint32_t taddr = tmem + (uint32_t(q * 32) << 16);
      float tv[kTopK], tl[kTopK];  // scores and their logits
      int ti[kTopK];
#pragma unroll
      for (int i = 0; i < kTopK; ++i) {
        tv[i] = -INFINITY;
        tl[i] = -INFINITY;
        ti[i] = 0x7fffffff;
      }
      for (int c0 = 0; c0 < 2 * n_half && c0 < E; c0 += 16) {
        float v[16];
        tmem_ld16(taddr + c0, v);
        if (t < T) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int e = c0 + i;
            if (e < E) {
              const float lg = v[i] + (bias ? bias[e] : 0.0f);
              const float sc = sel_bias ? lg + sel_bias[e] : lg;
              if (logits) logits[size_t(t) * E + e] = lg;
              if (ids && (sc > tv[kTopK - 1] || (sc == tv[kTopK - 1] && e < ti[kTopK - 1]))) {
                tv[kTopK - 1] = sc;
                tl[kTopK - 1] = lg;
                ti[kTopK - 1] = e;
#pragma unroll
                for (int j2 = kTopK - 1; j2 > 0; --j2) {
                  if (tv[j2] > tv[j2 - 1] || (tv[j2] == tv[j2 - 1] && ti[j2] < ti[j2 - 1])) {
                    const float fv = tv[j2];
                    tv[j2] = tv[j2 - 1];
                    tv[j2 - 1] = fv;
                    const float fl = tl[j2];
                    tl[j2] = tl[j2 - 1];
                    tl[j2 - 1] = fl;
                    const int fi = ti[j2];
                    ti[j2] = ti[j2 - 1];
                    ti[j2 - 1] = fi;
                  }
                }
              }
            }
          }
        }
      }
      if (ids && t < T) {
        float m = tl[0];  // the largest selected logit (slot 0 unless the bias reordered them)
#pragma unroll
        for (int i = 1; i < kTopK; ++i)
          if (i < k) m = fmaxf(m, tl[i]);
        float ex[kTopK], sum = 0.0f;
#pragma unroll
        for (int i = 0; i < kTopK; ++i) {
          ex[i] = i < k ? expf(tl[i] - m) : 0.0f;
          sum += ex[i];
        }
#pragma unroll
        for (int i = 0; i < kTopK; ++i) {
          if (i < k) {
            ids[size_t(t) * k + i] = ti[i];
            wts[size_t(t) * k + i] = ex[i] / sum;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->acc_empty);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while its partner may still multicast into it or arrive on it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

int rt_sm_count() {
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

bool router_tc_supported(const LayerDev& L, bool x_bf16) {
  return x_bf16 && L.d % 64 == 0 && L.E <= 512 && L.E % 32 == 0 && encode_fn() != nullptr;
}

cudaError_t launch_router_tc(const void* x, int T, const LayerDev& L, __nv_bfloat16* w3, float* logits, int32_t* ids,
                             float* wts, DevStatus* st, cudaStream_t s) {
  const long long n = (long long)L.E * L.d;
  cudaError_t e = launch_pdl(k_router_split_w, dim3(int(std::min<long long>((n + 255) / 256, 4096))), dim3(256), 0, s,
                             L.Wr, n, w3);
  if (e != cudaSuccess) return e;
  const int n_half = ((L.E / 2) + 15) / 16 * 16;
  const int b_stage_bytes = 2 * n_half * 128;
  // rings: x slices and weight stages, as many of each as fit (at most kRtMaxStages)
  int n_b = int(std::min<size_t>(kRtMaxStages, (kRtSmemBudget - 2 * size_t(kRtATile)) / b_stage_bytes));
  int n_a = int(std::min<size_t>(kRtMaxStages, (kRtSmemBudget - size_t(n_b) * b_stage_bytes) / kRtATile));
  if (n_b < 1 || n_a < 2) return cudaErrorInvalidValue;
  const int tmem_cols = 2 * n_half <= 256 ? 256 : 512;
  CUtensorMap mx, mw;
  if (!make_map_bytes(&mx, x, uint64_t(T), uint64_t(L.d), kRtM, 2) ||
      !make_map_bytes(&mw, w3, uint64_t(3) * L.E, uint64_t(L.d), uint32_t(n_half), 2))
    return cudaErrorInvalidValue;
  const size_t smem = size_t(n_a) * kRtATile + size_t(n_b) * b_stage_bytes + 1024 + sizeof(RtCtl);
  static cudaError_t attr = cudaFuncSetAttribute(k_router_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (attr != cudaSuccess) return attr;
  const int items = (T + kRtM - 1) / kRtM;
  const int pairs = std::max(1, std::min((items + kRtC - 1) / kRtC, rt_sm_count() / kRtC));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pairs * kRtC);
  cfg.blockDim = dim3(kRtThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = kRtC;
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_router_tc, mx, mw, L.logit_bias(), L.sel_bias(), T, L.d, L.E, n_half, n_a, n_b,
                            tmem_cols, logits, ids, wts, L.k, &st->flags);
}

}  // namespace moe
