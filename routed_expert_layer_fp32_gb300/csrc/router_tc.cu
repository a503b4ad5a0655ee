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
// Tile: 128 tokens (M) x all experts, the experts split into P parts of n_part columns (E =
// 384: P = 2 halves of 192, or 4 x 96) so one TMEM accumulator row holds a token's
// full logit row.  The split kernel writes the terms already in stage order and in the
// 128-byte-swizzled shared-memory layout: the three terms of one part for one 64-wide k-slice
// (n_part rows x 128 bytes each, 72 KB for a half at E = 384) are one contiguous block, so a
// weight stage is one bulk copy (on this GPU a row-strided tensor-map box of the same size
// streams several times slower per SM, and larger copies stream faster than smaller ones).
// The x k-slice (16 KB) has its own ring and is loaded once for all parts and all three terms.
//
// Two ways to spread the tiles.  With many tiles each CTA takes whole tiles (both halves, two
// weight stages per k-slice) and reads the 4.7 MB of weight terms from L2 for each of them.
// With few tiles each tile gets a thread-block cluster of P = 2 or 4 CTAs (the largest P for
// which every tile's cluster fits on the GPU at once), each CTA one part of the experts
// (one weight stage per k-slice), and ranks 1 .. P-1 hand their selected top-k lists to rank
// 0 through distributed shared memory for the final merge.  Every CTA loads only into its own
// shared memory.  Warp roles as in the expert GEMMs
// (TMA producer, single-thread MMA issuer, sixteen epilogue warps); bounded waits.
#include "common.cuh"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace moe {
namespace {

constexpr int kRtEpiParts = 4;                       // epilogue warps per TMEM lane quarter
constexpr int kRtEpiWarps = 4 * kRtEpiParts;
constexpr int kRtThreads = (2 + kRtEpiWarps) * 32;
// partial top-k lists of parts 1..3, merged by part 0: [part-1][token][slot] score, logit, id
constexpr size_t kRtMergeBytes = size_t(kRtEpiParts - 1) * 128 * kTopK * 12;
// split mode: each of ranks 1 .. P-1 hands rank 0 its merged lists, [128][kTopK] score, logit, id
constexpr size_t kRtRecvBytes = size_t(128) * kTopK * 12;
// the router bias row in shared memory (E <= 512 floats)
constexpr size_t kRtBiasBytes = 512 * 4;
// CTAs per cluster in split mode.  Measured (moe_route, 600-8192 tokens): 4 is 3 us faster
// than 2 up to 2048 tokens; 8 is no faster anywhere and at 2048 tokens its sixteen 8-CTA
// clusters of ~213 KB CTAs do not all fit at once (111 us against 56).
constexpr int kRtMaxParts = 4;
constexpr int kRtM = 128;
constexpr int kRtATile = kRtM * 128;
constexpr size_t kRtSmemBudget = 200 * 1024;  // at most this much for the two rings

// Split layout for P parts: block ((kt * P + h) * 3 + term) holds term `term` of experts
// [h n_part, (h + 1) n_part) over k = [64 kt, 64 kt + 64): n_part rows of 128 bytes, the
// 16-byte chunk c of row r stored at chunk c ^ (r % 8) (the MMA's 128-byte swizzle).  A thread
// converts one 8-element chunk of one expert row into its three terms.
__device__ __forceinline__ size_t split_block_offset(int kt, int term, int h, int n_part, int P) {
  return (size_t(kt * P + h) * 3 + term) * size_t(n_part) * 128;
}

__global__ void k_router_split_w(const float* __restrict__ Wr, int E, int d, int n_half, int P,
                                 uint8_t* __restrict__ out) {
  pdl_begin();
  const int chunks = d / 8;  // 16-byte chunks of bf16 per expert row
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < (long long)E * chunks;
       i += (long long)gridDim.x * blockDim.x) {
    const int e = int(i / chunks), q = int(i % chunks);
    const int kt = q >> 3, c = q & 7, h = e / n_half, r = e % n_half;  // n_half: the part height
    const float4 a = *reinterpret_cast<const float4*>(Wr + size_t(e) * d + q * 8);
    const float4 b = *reinterpret_cast<const float4*>(Wr + size_t(e) * d + q * 8 + 4);
    const float w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t t3[3][4];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      uint32_t p[3] = {0, 0, 0};
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float v = w[j + u];
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        const float r1 = v - __bfloat162float(hi);
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
        p[0] |= uint32_t(__bfloat16_as_ushort(hi)) << (16 * u);
        p[1] |= uint32_t(__bfloat16_as_ushort(mid)) << (16 * u);
        p[2] |= uint32_t(__bfloat16_as_ushort(lo)) << (16 * u);
      }
#pragma unroll
      for (int term = 0; term < 3; ++term) t3[term][j >> 1] = p[term];
    }
    const size_t in_block = size_t(r) * 128 + size_t((c ^ (r & 7)) * 16);
#pragma unroll
    for (int term = 0; term < 3; ++term)
      *reinterpret_cast<uint4*>(out + split_block_offset(kt, term, h, n_half, P) + in_block) =
          make_uint4(t3[term][0], t3[term][1], t3[term][2], t3[term][3]);
  }
}

constexpr int kRtMaxStages = 6;

struct RtCtl {
  uint64_t full_a[kRtMaxStages];
  uint64_t empty_a[kRtMaxStages];
  uint64_t full_b[kRtMaxStages];
  uint64_t empty_b[kRtMaxStages];
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t mma_done;
  uint64_t recv_full;  // split mode, rank 0: ranks 1 .. P-1's lists have arrived (one arrival per thread)
  uint32_t tmem_base;
  int abort;
  int epi_ok[2][4][kRtEpiParts];  // per tile parity: each epilogue warp's accumulator wait succeeded
};

// One token's running top-k list: scores tv (descending), logits tl, expert ids ti; an empty
// slot holds a NaN score.  Candidates are offered in increasing expert index (a scan visits its
// experts in order, and the lists it merges cover ever higher experts), so a candidate whose
// score equals a listed one goes in below it: the lower index ranks first.  The candidate
// takes the first slot whose score is below its own (or empty) and the slots from there down
// shift by one.  Every slot's new value is a select on the candidate's compares with the old
// list, so no slot waits on another.  A NaN candidate never enters.  Returns whether the
// candidate entered (it beat the last slot).
__device__ __forceinline__ bool rt_list_insert(float (&tv)[kTopK], float (&tl)[kTopK], int (&ti)[kTopK], float s,
                                               float l, int e) {
  bool gt[kTopK];
  const bool real = s == s;
#pragma unroll
  for (int j = 0; j < kTopK; ++j) gt[j] = real && !(s <= tv[j]);  // below s, or empty
#pragma unroll
  for (int j = kTopK - 1; j > 0; --j) {
    tv[j] = gt[j] ? (gt[j - 1] ? tv[j - 1] : s) : tv[j];
    tl[j] = gt[j] ? (gt[j - 1] ? tl[j - 1] : l) : tl[j];
    ti[j] = gt[j] ? (gt[j - 1] ? ti[j - 1] : e) : ti[j];
  }
  tv[0] = gt[0] ? s : tv[0];
  tl[0] = gt[0] ? l : tl[0];
  ti[0] = gt[0] ? e : ti[0];
  return gt[kTopK - 1];
}

template <bool split>
__global__ void __launch_bounds__(kRtThreads, 1)
    k_router_tc(const __grid_constant__ CUtensorMap map_x, const uint8_t* __restrict__ w_split,
                const float* __restrict__ bias, const float* __restrict__ sel_bias, int T, int d, int E, int n_half,
                int P, int n_a, int n_b, int tmem_cols,
                float* __restrict__ logits, int32_t* __restrict__ ids, float* __restrict__ wts, int k,
                int* status_flags) {
  extern __shared__ uint8_t rt_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rt_smem_raw) + 1023) & ~uintptr_t(1023));
  // split mode (few tiles): the P CTAs of a cluster take the same token tile, CTA r the experts
  // [r n_half, (r + 1) n_half) (n_half = E / P: the part height), and ranks 1 .. P-1 hand their
  // selected lists to rank 0.  Otherwise a CTA takes whole tiles, both halves (P = 2).
  const int b_half_bytes = n_half * 128;
  // a weight stage: the three terms of one half for one k-slice, one contiguous copy (72 KB at
  // E = 384); split mode loads its own half's stage per k-slice, otherwise both halves' in turn
  const int b_stage_bytes = 3 * b_half_bytes;
  const int b_per_kt = split ? 1 : P;  // weight stages per k-slice
  uint8_t* ring_a = smem;
  uint8_t* ring_b = smem + size_t(n_a) * kRtATile;
  RtCtl* ctl = reinterpret_cast<RtCtl*>(ring_b + size_t(n_b) * b_stage_bytes);
  uint8_t* merge = reinterpret_cast<uint8_t*>(ctl) + (sizeof(RtCtl) + 15) / 16 * 16;  // kRtMergeBytes
  uint8_t* recv = merge + kRtMergeBytes;                                               // (P-1) kRtRecvBytes (split)
  float* s_bias = reinterpret_cast<float*>(recv + (split ? size_t(P - 1) * kRtRecvBytes : 0));  // E floats
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = split ? int(cluster_ctarank()) : 0;
  // the CTA (split mode: the cluster) takes tiles unit, unit + n_units, ...
  const int per = split ? P : 1;
  const int unit = int(blockIdx.x) / per, n_units = int(gridDim.x) / per;
  if (threadIdx.x == 0) {
    for (int s = 0; s < n_a; ++s) {
      mbar_init(&ctl->full_a[s], 1);
      mbar_init(&ctl->empty_a[s], 1);
    }
    for (int s = 0; s < n_b; ++s) {
      mbar_init(&ctl->full_b[s], 1);
      mbar_init(&ctl->empty_b[s], 1);
    }
    mbar_init(&ctl->acc_full, 1);
    mbar_init(&ctl->acc_empty, kRtEpiWarps);
    mbar_init(&ctl->mma_done, 1);
    mbar_init(&ctl->recv_full, (split ? P - 1 : 1) * 4 * 32);  // every thread of the senders' part-0 warps
    ctl->abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if (split) cluster_sync_all();  // the partner's receive barrier exists before any remote arrival
  tc_fence_after();
  pdl_begin();
  const uint32_t tmem = ctl->tmem_base;
  const int n_items = (T + kRtM - 1) / kRtM;
  const int KT = d / 64;  // 64 bf16 per 128-byte k-slice
  auto tile_of = [&](int j) { return unit + j * n_units; };
  auto sa = [&](int s) { return ring_a + size_t(s) * kRtATile; };
  auto sb = [&](int s) { return ring_b + size_t(s) * b_stage_bytes; };
  // the expert half stage number hh of a k-slice covers
  auto half_of = [&](int hh) { return split ? rank : hh; };

  if (warp == 0) {
    if (lane == 0) {  // TMA producer: x slice per k-slice, the weight stages of every k-slice
      int ia = 0, ib = 0;
      bool stop = false;
      for (int j = 0; tile_of(j) < n_items && !stop; ++j) {
        const int item = tile_of(j);
        for (int kt = 0; kt < KT && !stop; ++kt) {
          {
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
          for (int hh = 0; hh < b_per_kt; ++hh, ++ib) {
            const int s = ib % n_b, use = ib / n_b;
            if (!mbar_wait(&ctl->empty_b[s], (use & 1) ^ 1, &ctl->abort)) {
              report_timeout_flag(status_flags, 25);
              stop = true;
              break;
            }
            mbar_arrive_expect_tx(&ctl->full_b[s], b_stage_bytes);
            bulk_g2s(sb(s), w_split + split_block_offset(kt, 0, half_of(hh), n_half, P), uint32_t(b_stage_bytes),
                     &ctl->full_b[s]);
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
      for (int j = 0; tile_of(j) < n_items && !stop; ++j) {
        if (!mbar_wait(&ctl->acc_empty, (jt & 1) ^ 1, &ctl->abort)) {
          report_timeout_flag(status_flags, 22);
          break;
        }
        tc_fence_after();
        for (int kt = 0; kt < KT && !stop; ++kt) {
          const int sa_i = ia % n_a;
          if (!mbar_wait(&ctl->full_a[sa_i], (ia / n_a) & 1, &ctl->abort)) {
            report_timeout_flag(status_flags, 23);
            stop = true;
            break;
          }
          for (int hh = 0; hh < b_per_kt; ++hh, ++ib) {
            const int s = ib % n_b, use = ib / n_b;
            if (!mbar_wait(&ctl->full_b[s], use & 1, &ctl->abort)) {
              report_timeout_flag(status_flags, 26);
              stop = true;
              break;
            }
            tc_fence_after();
            // the three terms of one half into that half's accumulator columns
            const uint64_t da = sw128_desc(sa(sa_i));
            const uint32_t d_cols = tmem + uint32_t(half_of(hh) * n_half);
            for (int tm = 0; tm < 3; ++tm) {
              const uint64_t db = sw128_desc(sb(s) + tm * b_half_bytes);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {  // 16 bf16 (32 bytes) per MMA
                const uint32_t acc = (kt > 0 || tm > 0 || kk > 0) ? 1u : 0u;
                tc_mma_f16(d_cols, da + 2 * kk, db + 2 * kk, idesc, acc);
              }
            }
            tc_commit(&ctl->empty_b[s]);
          }
          if (stop) break;
          tc_commit(&ctl->empty_a[sa_i]);
          ++ia;
        }
        if (!stop) {
          tc_commit(&ctl->acc_full);
          ++jt;
        }
      }
      tc_commit(&ctl->mma_done);
      int zero = 0;
      mbar_wait(&ctl->mma_done, 0, &zero);
    }
  } else {  // epilogue: one token per TMEM lane, logits = acc + bias
    // With ids != nullptr the epilogue also selects.  The four warps of a lane quarter each scan
    // a quarter of the experts (consecutive 16-column chunks) and keep a sorted list of the
    // kTopK best scores (larger first, lower index first on equal scores) with rt_list_insert.
    // A chunk whose best score is not above the list's last is skipped whole.  Part 0 merges
    // the four lists in expert order, then forms the softmax over the selected logits, summed
    // in slot order.  The score is the logit, plus sel_bias in the selection-only bias mode.
    // The bias row (whichever of the two is set) is read once into shared memory.
    const int q = warp & 3, part = (warp - 2) >> 2;
    const float* brow = bias ? bias : sel_bias;
    if (brow) {
      for (int i = int(threadIdx.x) - 64; i < E; i += kRtEpiWarps * 32) s_bias[i] = brow[i];
      named_bar_sync(5, kRtEpiWarps * 32);
    }
    float* m_sc = reinterpret_cast<float*>(merge);                       // [3][128][kTopK]
    float* m_lg = m_sc + (kRtEpiParts - 1) * 128 * kTopK;
    int* m_id = reinterpret_cast<int*>(m_lg + (kRtEpiParts - 1) * 128 * kTopK);
    // this CTA's experts in 16-column chunks (split mode: its half), a quarter per part
    const int n_chunks = split ? n_half / 16 : (E + 15) / 16;
    const int ch_base = split ? rank * (n_half / 16) : 0;
    const int ch_lo = ch_base + part * n_chunks / kRtEpiParts, ch_hi = ch_base + (part + 1) * n_chunks / kRtEpiParts;
    // split mode: rank r >= 1 writes its lists into block r - 1 of rank 0's receive buffer,
    // [block][score, logit, id][row][slot]
    int jt = 0;
    for (int j = 0; tile_of(j) < n_items; ++j, ++jt) {
      const int item = tile_of(j);
      // the four warps of a quarter meet at named barriers: they leave on a timeout together
      const bool ok = mbar_wait(&ctl->acc_full, jt & 1, &ctl->abort);
      if (lane == 0) ctl->epi_ok[jt & 1][q][part] = ok ? 1 : 0;
      named_bar_sync(1 + q, kRtEpiParts * 32);
      bool all_ok = true;
#pragma unroll
      for (int p2 = 0; p2 < kRtEpiParts; ++p2) all_ok = all_ok && ctl->epi_ok[jt & 1][q][p2] != 0;
      if (!all_ok) {
        if (lane == 0 && !ok) report_timeout_flag(status_flags, 24);
        break;
      }
      tc_fence_after();
      const int row = q * 32 + lane;
      const int t = item * kRtM + row;
      const uint32_t taddr = tmem + (uint32_t(q * 32) << 16);
      float tv[kTopK], tl[kTopK];  // scores and their logits
      int ti[kTopK];
#pragma unroll
      for (int i = 0; i < kTopK; ++i) {
        tv[i] = __int_as_float(0x7fc00000);  // empty
        tl[i] = -INFINITY;
        ti[i] = 0x7fffffff;
      }
      for (int ch = ch_lo; ch < ch_hi; ++ch) {
        const int c0 = ch * 16;
        float v[16];
        tmem_ld16(taddr + c0, v);
        if (t < T) {
          float sc[16];
          float cmax = -INFINITY;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int e = c0 + i;
            const float b = (brow && e < E) ? s_bias[e] : 0.0f;
            v[i] = e < E ? (bias ? v[i] + b : v[i]) : -INFINITY;
            sc[i] = e < E ? (sel_bias ? v[i] + b : v[i]) : __int_as_float(0x7fc00000);  // past E: never listed
            if (logits && e < E) logits[size_t(t) * E + e] = v[i];
            cmax = fmaxf(cmax, sc[i]);
          }
          if (ids && !(cmax <= tv[kTopK - 1])) {  // some score of the chunk may enter the list
#pragma unroll
            for (int i = 0; i < 16; ++i) rt_list_insert(tv, tl, ti, sc[i], v[i], c0 + i);
          }
        }
      }
      // the accumulator is free for the next tile once every warp has read its columns
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->acc_empty);
      if (ids) {  // (every warp of the quarter takes the same branches to both barriers)
        if (part > 0) {
#pragma unroll
          for (int i = 0; i < kTopK; ++i) {
            const int o = ((part - 1) * 128 + row) * kTopK + i;
            m_sc[o] = tv[i];
            m_lg[o] = tl[i];
            m_id[o] = ti[i];
          }
        }
        named_bar_sync(1 + q, kRtEpiParts * 32);  // the quarter's lists are written
        if (part == 0) {
          // merge parts 1..3 (ever higher experts) into this list; a list is sorted, so once one
          // of its candidates stays out the rest do
          for (int p2 = 1; p2 < kRtEpiParts; ++p2) {
#pragma unroll
            for (int i = 0; i < kTopK; ++i) {
              const int o = ((p2 - 1) * 128 + row) * kTopK + i;
              if (!rt_list_insert(tv, tl, ti, m_sc[o], m_lg[o], m_id[o])) break;
            }
          }
          if (split && rank >= 1) {  // hand the list to rank 0, which merges and writes
            const uint32_t base = mapa_shared(smem_u32(recv), 0) + uint32_t(rank - 1) * uint32_t(kRtRecvBytes);
#pragma unroll
            for (int i = 0; i < kTopK; ++i) {
              const uint32_t o = uint32_t(row * kTopK + i) * 4u;
              st_cluster_f32(base + o, tv[i]);
              st_cluster_f32(base + uint32_t(128 * kTopK * 4) + o, tl[i]);
              st_cluster_f32(base + uint32_t(2 * 128 * kTopK * 4) + o, __int_as_float(ti[i]));
            }
            mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->recv_full), 0));  // releases this thread's stores
          }
          bool merged = true;
          if (split && rank == 0) {  // ranks 1 .. P-1's lists for these tokens, in rank order
            merged = mbar_wait_cluster(&ctl->recv_full, jt & 1, &ctl->abort);
            if (!merged && lane == 0) report_timeout_flag(status_flags, 27);
            for (int src = 0; merged && src < P - 1; ++src) {
              const float* r_sc = reinterpret_cast<const float*>(recv + size_t(src) * kRtRecvBytes);
              const float* r_lg = r_sc + 128 * kTopK;
              const int* r_id = reinterpret_cast<const int*>(r_lg + 128 * kTopK);
#pragma unroll
              for (int i = 0; i < kTopK; ++i) {  // rank src + 1 covers higher experts than the list
                const int o = row * kTopK + i;
                if (!rt_list_insert(tv, tl, ti, r_sc[o], r_lg[o], r_id[o])) break;
              }
            }
          }
          if (t < T && merged && !(split && rank >= 1)) {
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
        }
        named_bar_sync(1 + q, kRtEpiParts * 32);  // the merge buffer may be written again
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (split) cluster_sync_all();  // no CTA leaves while its partner may still write its lists into it
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

// Stage counts of the two rings for one mode: weight stages first (three terms of one expert
// part, 3 n_part 128 bytes each), then x slices, as many as fit beside the control block and
// the merge buffers (at most kRtMaxStages each).  False unless both rings get two stages.
bool rt_rings(bool split, int n_part, int P, int* n_a, int* n_b, size_t* smem) {
  const size_t b_stage = size_t(3) * n_part * 128;
  const size_t fixed = 1024 + (sizeof(RtCtl) + 15) / 16 * 16 + kRtMergeBytes + (split ? size_t(P - 1) * kRtRecvBytes : 0) +
                       kRtBiasBytes;
  const size_t rings = std::min(kRtSmemBudget, 227 * 1024 - fixed);
  if (rings < 2 * b_stage + 2 * size_t(kRtATile)) return false;
  if (split && P >= 4) {  // one weight stage per x slice: rings of equal depth
    *n_a = *n_b = int(std::min<size_t>(kRtMaxStages, rings / (b_stage + size_t(kRtATile))));
  } else {
    *n_b = int(std::min<size_t>(kRtMaxStages, (rings - 2 * size_t(kRtATile)) / b_stage));
    *n_a = int(std::min<size_t>(kRtMaxStages, (rings - size_t(*n_b) * b_stage) / kRtATile));
  }
  *smem = size_t(*n_a) * kRtATile + size_t(*n_b) * b_stage + fixed;
  return *smem <= 227 * 1024;
}

}  // namespace

bool router_tc_supported(const LayerDev& L, bool x_bf16) {
  int n_a = 0, n_b = 0;
  size_t smem = 0;
  return x_bf16 && L.d % 64 == 0 && L.E <= 512 && L.E % 32 == 0 && rt_rings(false, L.E / 2, 2, &n_a, &n_b, &smem) &&
         rt_rings(true, L.E / 2, 2, &n_a, &n_b, &smem) && encode_fn() != nullptr;
}

cudaError_t launch_router_tc(const void* x, int T, const LayerDev& L, __nv_bfloat16* w3, float* logits, int32_t* ids,
                             float* wts, DevStatus* st, cudaStream_t s) {
  const int items = (T + kRtM - 1) / kRtM;
  // few tiles: split mode, a cluster of P CTAs per tile, each CTA E / P experts, with the
  // largest P (4 or 2) for which every tile's cluster fits on the GPU at once and the parts
  // are whole 16-column chunks; otherwise one CTA per tile at a time, both halves (P = 2)
  int split = 0, P = 2, n_a = 0, n_b = 0;
  size_t smem = 0;
  for (int p = kRtMaxParts; p >= 2 && !split; p /= 2)
    if (L.E % (16 * p) == 0 && items * p <= rt_sm_count() && rt_rings(true, L.E / p, p, &n_a, &n_b, &smem)) {
      split = 1;
      P = p;
    }
  if (!split && !rt_rings(false, L.E / 2, 2, &n_a, &n_b, &smem)) return cudaErrorInvalidValue;
  const int n_half = L.E / P;  // the part height (E % 32 == 0: P = 2 gives whole 16-column chunks)
  const long long n = (long long)L.E * (L.d / 8);
  cudaError_t e = launch_pdl(k_router_split_w, dim3(int(std::min<long long>((n + 255) / 256, 4096))), dim3(256), 0, s,
                             L.Wr, L.E, L.d, n_half, P, reinterpret_cast<uint8_t*>(w3));
  if (e != cudaSuccess) return e;
  const int tmem_cols = L.E <= 256 ? 256 : 512;
  CUtensorMap mx;
  if (!make_map_bytes(&mx, x, uint64_t(T), uint64_t(L.d), kRtM, 2)) return cudaErrorInvalidValue;
  static cudaError_t attr = [] {
    const cudaError_t e0 = cudaFuncSetAttribute(k_router_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    const cudaError_t e1 = cudaFuncSetAttribute(k_router_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    return e0 != cudaSuccess ? e0 : e1;
  }();
  if (attr != cudaSuccess) return attr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(split ? items * P : std::min(items, rt_sm_count()));
  cfg.blockDim = dim3(kRtThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = P;
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = split ? 2 : 1;
  const uint8_t* w_split = static_cast<const uint8_t*>(static_cast<const void*>(w3));
  if (split)
    return cudaLaunchKernelEx(&cfg, k_router_tc<true>, mx, w_split, L.logit_bias(), L.sel_bias(), T, L.d, L.E, n_half,
                              P, n_a, n_b, tmem_cols, logits, ids, wts, L.k, &st->flags);
  return cudaLaunchKernelEx(&cfg, k_router_tc<false>, mx, w_split, L.logit_bias(), L.sel_bias(), T, L.d, L.E, n_half,
                            P, n_a, n_b, tmem_cols, logits, ids, wts, L.k, &st->flags);
}

}  // namespace moe
