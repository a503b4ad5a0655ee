// Grouped FP8 expert GEMMs on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// The experts are SwitchGLU FFNs with E4M3 weights and one fp32 scale per output row
// ("We Ported Aleph Alpha's Kolibri to a MacBook. Our Own Gate Said No.", section 3, and the
// E4M3 checkpoint of the vllm.cpp Kolibri-1 CPU FP8 pull request); activations enter each
// contraction as per-row E4M3 codes (W8A8).
//
// One kernel shape serves decode and prefill ("swap-AB"): the A operand (M = 128) is a block
// of 128 weight rows, the B operand (N = kN) is a tile of up to kN token rows of one expert
// group, D[weight row][token] accumulates in TMEM in fp32.  Gate/up issues two MMAs per
// k-step (gate and up rows of the same 128 outputs) into two accumulators, so the epilogue
// sees g and u side by side and writes h = silu(g) u directly (the per-row maximum of |h|
// that scales its quantisation is taken afterwards, by the h-quantisation pass).  Down produces
// y_e[token][m] for 128 output columns m.
//
// Warp roles (320 threads): warp 0 fills a ring of shared-memory stages (128-byte swizzle, the
// layout the MMA descriptors name): lane 0 copies the weight tiles, and for gate/up the lanes
// gather the tile's activation rows by token (TMA tile::gather4 on the token-order E4M3 rows,
// so the activations are quantised once per token, not once per routed copy); warp 1 owns the TMEM
// allocation and its lane 0 issues tcgen05.mma and tcgen05.commit (the commit frees a stage
// when its MMAs have read it, and marks an accumulator ready after the last k-step); warps
// 2-9 (two per TMEM lane quarter, each half of the token columns) read the accumulators
// with tcgen05.ld and write the outputs (h = silu(g) u for gate/up, scaled rows for down).
// Accumulators are double-buffered when TMEM has room, so an item's epilogue overlaps the
// next item's MMAs.
//
// For a handful of tokens (fewer gate/up items than SMs) the two CTAs of a cluster share each
// item: rank 0 runs the first half of the k-steps, rank 1 the second; rank 1's epilogue
// writes its fp32 partial accumulators into rank 0's shared memory (distributed shared
// memory, an mbarrier counting the writers), and rank 0 adds them to its own (always in that
// order, so results do not depend on timing) before the nonlinearity.
//
// Every wait is bounded (tma.cuh): on a timeout the CTA records MOE_ERR_TIMEOUT, all roles
// leave their loops, the producer waits for its loads in flight, the MMA issuer waits for its
// MMAs, and TMEM is freed before the CTA exits.
#include <algorithm>

#include "common.cuh"
#include "tma.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace {

constexpr int kEpiWarps = 8;                      // two per TMEM lane quarter, splitting the columns
constexpr int kTcThreads = (2 + kEpiWarps) * 32;
constexpr int kTileM = 128;       // weight rows per accumulator (MMA M)
constexpr int kKTile = 128;       // bytes (= E4M3 elements) of k per chunk: one 128-byte swizzle atom
constexpr int kATileBytes = kTileM * kKTile;  // one weight tile of the tiled layout (16 KB)
constexpr size_t kTcSmemCap = 226 * 1024;     // dynamic shared memory per CTA
constexpr int kPrefetchBytes = 256 * 1024;  // weights a CTA pulls into L2 before its dependency wait
constexpr int kMaxStages = 8;
constexpr int kDownPairMinN = 64;
constexpr int kSplitMaxT = 16;  // gate/up k-steps split over a CTA pair up to this many tokens
constexpr int kGateUpPairChunkMaxN = 32;  // gate/up stages of two k-chunks up to this tile width

struct TcArgs {
  int d, F, E, T, R;  // R = T (k + 1) rows
  const uint8_t* w;    // tiled weights of the routed experts (gate/up or down)
  const uint8_t* wsh;  // the shared expert's, same layout
  const Tile* tiles;
  const int* n_tiles;
  const int32_t* perm;  // [R] token of each row (gate/up gathers activation rows through it)
  const uint8_t* xq;    // [T, d] E4M3 activations in token order (gate/up)
  const float* sx;      // [T] activation scales, token order (gate/up)
  const float* sgu;     // [E, 2, F]
  const float* sh_sgu;  // [2, F]
  const float* sd;      // [E, d]
  const float* sh_sd;   // [d]
  float* h;             // [R, F]
  const float* sh;      // [R] h scales (down)
  __nv_bfloat16* y_rows;  // [R, d] expert output rows (bf16 activations)
  int* status_flags;
};

// MMA width for a tile of `nrows` token rows: the rows rounded up to the 16 columns an M = 128
// MMA steps in, at most the tile width.  Columns past it are neither loaded nor computed (the
// padding of an expert's last tile would otherwise cost up to a whole tile of MMA work).
template <int kN>
__device__ __forceinline__ int mma_cols(int nrows) {
  return kN <= 16 ? kN : min(kN, max(16, (nrows + 15) & ~15));
}

// An instruction descriptor with its N field (bits 17-22, N / 8) replaced.
__device__ __forceinline__ uint32_t with_n(uint32_t idesc, int n) {
  return (idesc & ~(0x3Fu << 17)) | (uint32_t(n >> 3) << 17);
}

struct TcCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t mma_done;
  uint64_t recv_full;  // split-K, rank 0: the partner's partial accumulators have arrived
  uint64_t recv_free;  // split-K, rank 1: rank 0 has consumed the receive buffer
  int stage_n[kMaxStages];  // MMA width (token columns) of the item a stage belongs to
  uint32_t tmem_base;
  int abort;
};

// kA accumulators of kN columns (gate/up: gate and up rows of the same 128 outputs; down:
// 1 or 2 blocks of 128 output rows); a stage holds kC consecutive 128-byte k-chunks: the kA
// weight tiles of each chunk (one contiguous copy for gate/up, one per block for down) and the
// kN activation rows of those chunks (gate/up: gathered by token, four rows per TMA gather;
// down: one 3-D tensor-map box of h rows).
template <int kN, bool kGateUp, int kA_, int kSplit_, int kC_>
struct TcCfg {
  // gate/up activation rows: wide tiles gather with per-lane cp.async (16 bytes each; TMA's
  // cost per request makes 512-byte gathers slow at 128 rows per stage), narrow ones with
  // TMA gather4
  static constexpr bool kLdgsts = kGateUp && kN >= 64;
  static constexpr int kA = kA_;
  static constexpr int kSplit = kSplit_;  // CTAs (one cluster) sharing an item's k-steps
  static constexpr int kC = kC_;
  static constexpr int kABytes = kA * kC * kATileBytes;
  static constexpr int kBBytes = kC * kN * kKTile;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kRecvBytes = kSplit == 2 ? kA * kTileM * kN * 4 : 0;  // [kA][kN cols][128 rows] fp32
  static constexpr int kStages =
      int(std::min<size_t>(kMaxStages, (kTcSmemCap - kRecvBytes - 1024 - sizeof(TcCtl)) / kStageBytes));
  static_assert(kStages >= 2, "at least a double-buffered stage ring");
  static_assert(kStageBytes % 1024 == 0 && (kN * kKTile) % 1024 == 0, "stages and chunks keep the swizzle atoms aligned");
  static constexpr int kColsPerAcc = kA * kN;
  static constexpr int kBufs = (2 * kColsPerAcc <= 512) ? 2 : 1;
  static constexpr int kTmemCols = (kBufs * kColsPerAcc <= 32)    ? 32
                                   : (kBufs * kColsPerAcc <= 64)  ? 64
                                   : (kBufs * kColsPerAcc <= 128) ? 128
                                   : (kBufs * kColsPerAcc <= 256) ? 256
                                                                  : 512;
  static constexpr size_t kSmemBytes =
      size_t(kStages) * kStageBytes + kRecvBytes + 1024 /* alignment slack */ + sizeof(TcCtl);
};

template <int kN, bool kGateUp, int kA, int kSplit, int kC, bool kW4>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_expert_tc(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                const __grid_constant__ CUtensorMap map_wsh, TcArgs a) {
  using C = TcCfg<kN, kGateUp, kA, kSplit, kC>;
  static_assert(!kGateUp || kA == 2, "gate/up stages hold the gate and the up rows");
  static_assert(kSplit == 1 || kSplit == 2, "items are split over one or two CTAs");
  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  float* recv = reinterpret_cast<float*>(smem + size_t(C::kStages) * C::kStageBytes);
  TcCtl* ctl = reinterpret_cast<TcCtl*>(smem + size_t(C::kStages) * C::kStageBytes + C::kRecvBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // split-K: the two CTAs of a cluster take the first and the second half of every item's
  // k-steps; rank 1 hands its partial accumulators to rank 0, which finishes the item
  const int rank = kSplit == 2 ? int(cluster_ctarank()) : 0;
  const int unit = int(blockIdx.x) / kSplit, n_units = int(gridDim.x) / kSplit;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&ctl->full[s], C::kLdgsts ? 33 : 1);  // + one cp.async arrival per producer lane
      mbar_init(&ctl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl->acc_full[b], 1);
      mbar_init(&ctl->acc_empty[b], kEpiWarps);
    }
    mbar_init(&ctl->mma_done, 1);
    mbar_init(&ctl->recv_full, kEpiWarps * 32);
    mbar_init(&ctl->recv_free, kEpiWarps * 32);
    ctl->abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if (kSplit == 2) cluster_sync_all();  // the partner's barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  // The tile list is read after the dependency wait: gate/up may directly follow the kernel
  // that writes it (the decode router dispatches in its last CTA).  Down launches only once
  // gate/up has passed its own wait (the h-quantisation kernel between them lets down launch
  // early, while gate/up still runs), so the list is final and down's prefetch may read it
  // before its wait.
  const int nblk = kGateUp ? a.F / kTileM : a.d / (kTileM * kA);  // items per tile
  const int KT = (kGateUp ? a.d : a.F) / kKTile;                  // 128-byte k-chunks per item
  const int KS = KT / kC;                                          // stages per item
  const int ks_lo = rank * KS / kSplit, ks_hi = (rank + 1) * KS / kSplit;  // this CTA's share
  int total = 0;                                                   // items, set after the wait
  const int nb_rows = (kGateUp ? a.F : a.d) / kTileM;              // 128-row blocks per expert
  auto stage_a = [&](int s) { return smem + size_t(s) * C::kStageBytes; };
  auto stage_b = [&](int s) { return smem + size_t(s) * C::kStageBytes + C::kABytes; };
  // weight tile (accumulator ai, chunk c) of a stage
  auto a_tile = [&](int s, int ai, int c) {
    return stage_a(s) + (kGateUp ? (c * 2 + ai) : (ai * kC + c)) * kATileBytes;
  };
  // tiled-layout index of the first tile of an item's block ai (down) or of its gate/up pairs,
  // chunk j; the copy's tiles follow it
  auto w_tile = [&](const Tile& tl, int nb, int ai, int j) -> size_t {
    const size_t e = tl.group == a.E ? 0 : size_t(tl.group);
    if (kGateUp) return ((e * nb_rows + nb) * KT + j) * 2;
    return (e * nb_rows + size_t(nb) * kA + ai) * KT + j;
  };
  // E4M3 tiles are 16 KB in memory and in shared memory; E2M1 tiles 8 KB in memory, unpacked
  // to the 16 KB operand layout by the copy (tensor map type 16U4_ALIGN16B)
  constexpr uint32_t kTileMem = kW4 ? kATileBytes / 2 : kATileBytes;
  auto w_src = [&](const Tile& tl, int nb, int ai, int j) {
    return (tl.group == a.E ? a.wsh : a.w) + w_tile(tl, nb, ai, j) * kTileMem;
  };
  constexpr uint32_t kCopyTiles = kGateUp ? 2 * kC : kC;  // tiles per weight copy
  constexpr uint32_t kCopyBytes = kCopyTiles * kATileBytes;  // shared-memory bytes per weight copy
  constexpr int kCopies = kGateUp ? 1 : kA;

  if (warp == 0) {  // -------------------------------------------------- TMA producer warp
    // Weights need nothing from the kernel this launch overlaps: pull this CTA's first items
    // into L2 while that kernel runs (up to kPrefetchBytes), then wait for it.  Gate/up knows
    // only the shared expert's items before the wait (the list starts with its ceil(T / kN)
    // tiles); down knows its whole list.
    if (lane == 0) {
      int budget = kPrefetchBytes;
      const int known = kGateUp ? ((a.T + kN - 1) / kN) * nblk : *a.n_tiles * nblk;
      for (int item = unit; item < known && budget > 0; item += n_units) {
        const Tile tl = kGateUp ? Tile{a.E, 0, 0, 0} : checked_tile(a.tiles, item / nblk, a.E, a.R, kN, a.status_flags, 1);
        for (int ks = ks_lo; ks < ks_hi && budget > 0; ++ks, budget -= kCopies * int(kCopyBytes))
          for (int ai = 0; ai < kCopies; ++ai)
            prefetch_l2_bulk(w_src(tl, item % nblk, ai, ks * kC), kCopyTiles * kTileMem);
      }
    }
    pdl_begin();
    total = *a.n_tiles * nblk;
    // Lane 0 waits for a free stage and copies the weights; gate/up activation rows are
    // gathered by token (perm) with tile::gather4, lane l bringing rows 4l..4l+3 of the tile
    // (rows past the tile's end repeat its first token; their columns are never read).
    // Down reads h rows, already in row order, as one 3-D box.
    const uint64_t pol = policy_evict_first();
    int it = 0;
    bool stop = false;
    for (int item = unit; item < total && !stop; item += n_units) {
      const Tile tl = checked_tile(a.tiles, item / nblk, a.E, a.R, kN, a.status_flags, 2);
      const int nb = item % nblk;
      const int n_mma = mma_cols<kN>(tl.nrows);
      // the tokens of this lane's rows: gather4 lanes own rows 4l..4l+3; cp.async lanes own
      // 16-byte column l % 8 of rows l / 8 + 4j
      constexpr int kG = C::kLdgsts ? kN / 4 : 4;
      int g[kG];
#pragma unroll
      for (int i = 0; i < kG; ++i) g[i] = 0;
      if (kGateUp) {
        const int first = checked_token(a.perm[tl.row0], a.T, a.status_flags, 3);
#pragma unroll
        for (int i = 0; i < kG; ++i) {
          const int r = C::kLdgsts ? (lane >> 3) + 4 * i : 4 * lane + i;
          g[i] = (r < tl.nrows && (C::kLdgsts || 4 * lane < kN)) ? checked_token(a.perm[tl.row0 + r], a.T, a.status_flags, 3)
                                                                 : first;
        }
      }
      for (int ks = ks_lo; ks < ks_hi; ++ks, ++it) {
        const int s = it % C::kStages, use = it / C::kStages;
        int ok = 1;
        if (lane == 0) ok = mbar_wait(&ctl->empty[s], (use & 1) ^ 1, &ctl->abort) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          if (lane == 0) report_timeout_flag(a.status_flags, 11);
          stop = true;
          break;
        }
        if (lane == 0) {
          ctl->stage_n[s] = n_mma;  // published to the MMA issuer by the arrive below
          // the weights' bytes in memory (E2M1: half their shared-memory bytes), then the
          // activations' unless cp.async brings them
          mbar_arrive_expect_tx(&ctl->full[s], (kW4 ? C::kABytes / 2 : C::kABytes) + (C::kLdgsts ? 0 : C::kBBytes));
#pragma unroll
          for (int ai = 0; ai < kCopies; ++ai) {
            if (kW4) {  // one tensor-map box per tile, rows of the [tiles x 128, 128] code matrix
              const CUtensorMap* mw = tl.group == a.E ? &map_wsh : &map_w;
              const int y0 = int(w_tile(tl, nb, ai, ks * kC) * kTileM);
              for (int t = 0; t < int(kCopyTiles); ++t)
                tma_load_2d(stage_a(s) + ai * kCopyBytes + t * kATileBytes, mw, 0, y0 + t * kTileM, &ctl->full[s]);
            } else {
              bulk_g2s_stream(stage_a(s) + ai * kCopyBytes, w_src(tl, nb, ai, ks * kC), kCopyBytes, &ctl->full[s], pol);
            }
          }
          if (!kGateUp) tma_load_3d(stage_b(s), &map_x, 0, tl.row0, ks * kC, &ctl->full[s]);
        }
        if (C::kLdgsts) {
          // row r, 16-byte column cc of chunk c lands at (c kN + r) 128 + (cc ^ r % 8) 16: the
          // 128-byte swizzle the MMA descriptor names
          const int cc = lane & 7;
#pragma unroll
          for (int c = 0; c < kC; ++c) {
            uint8_t* dst = stage_b(s) + c * kN * kKTile;
            const size_t col = size_t(ks * kC + c) * kKTile + cc * 16;
#pragma unroll
            for (int i = 0; i < kG; ++i) {
              const int r = (lane >> 3) + 4 * i;
              if (r < n_mma)  // rows past the MMA's width are never read
                cp_async16(dst + r * kKTile + ((cc ^ (r & 7)) << 4), a.xq + size_t(g[i]) * a.d + col);
            }
          }
          cp_async_arrive_noinc(&ctl->full[s]);
        } else if (kGateUp) {
          __syncwarp();
          if (4 * lane < kN) {
#pragma unroll
            for (int c = 0; c < kC; ++c)
              tma_gather4(stage_b(s) + (c * kN + 4 * lane) * kKTile, &map_x, (ks * kC + c) * kKTile, g[0], g[1], g[2],
                          g[3], &ctl->full[s]);
          }
        }
      }
    }
    // wait for the loads still in flight (bounded, regardless of abort)
    if (lane == 0) {
      for (int s = 0; s < C::kStages && s < it; ++s) {
        const int last_use = (it - 1 - s) / C::kStages;
        int zero = 0;
        mbar_wait(&ctl->full[s], last_use & 1, &zero);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    pdl_begin();
    total = *a.n_tiles * nblk;
    if (lane == 0) {  // ------------------------------------------------ MMA issuer
      constexpr uint32_t idesc0 = kW4 ? idesc_f8f6f4(kTileM, kN, kFmtE2M1, kFmtE4M3) : idesc_e4m3(kTileM, kN);
      int it = 0, jt = 0;
      bool stop = false;
      for (int item = unit; item < total && !stop; item += n_units, ++jt) {
        const int b = jt % C::kBufs, ub = jt / C::kBufs;
        if (!mbar_wait(&ctl->acc_empty[b], (ub & 1) ^ 1, &ctl->abort)) {
          report_timeout_flag(a.status_flags, 12);
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem + uint32_t(b * C::kColsPerAcc);
        for (int ks = ks_lo; ks < ks_hi; ++ks, ++it) {
          const int s = it % C::kStages, use = it / C::kStages;
          if (!mbar_wait(&ctl->full[s], use & 1, &ctl->abort)) {
            report_timeout_flag(a.status_flags, 13);
            stop = true;
            break;
          }
          tc_fence_after();
          if (C::kLdgsts) fence_proxy_async_smem();  // the activation rows were written by cp.async
          const uint32_t idesc = kN > 16 ? with_n(idesc0, ctl->stage_n[s]) : idesc0;
#pragma unroll
          for (int c = 0; c < kC; ++c) {
            const uint64_t db = sw128_desc(stage_b(s) + c * kN * kKTile);
            uint64_t da[kA];
#pragma unroll
            for (int ai = 0; ai < kA; ++ai) da[ai] = sw128_desc(a_tile(s, ai, c));
#pragma unroll
            for (int kk = 0; kk < kKTile / 32; ++kk) {
              const uint32_t acc = (ks > ks_lo || c > 0 || kk > 0) ? 1u : 0u;
#pragma unroll
              for (int ai = 0; ai < kA; ++ai)  // accumulators interleaved
                tc_mma_f8(d0 + uint32_t(ai * kN), da[ai] + 2 * kk, db + 2 * kk, idesc, acc);
            }
          }
          tc_commit(&ctl->empty[s]);
        }
        if (!stop) tc_commit(&ctl->acc_full[b]);
      }
      // every MMA issued has completed before TMEM is released
      tc_commit(&ctl->mma_done);
      int zero = 0;
      mbar_wait(&ctl->mma_done, 0, &zero);
    }
  } else {  // ------------------------------------------------------------ epilogue
    pdl_begin();
    total = *a.n_tiles * nblk;
    // warps 2..9: lane quarter q = warp % 4 (the TMEM lanes this warp may read), column half
    // ch = (warp - 2) / 4 of the kN token columns
    const int q = warp & 3, ch = (warp - 2) >> 2;
    const int rloc = q * 32 + lane;
    constexpr int kHalf = kN / 2 >= 16 ? kN / 2 : 16;
    const int cbeg = kN / 2 >= 16 ? ch * kHalf : (ch == 0 ? 0 : kN);  // kN = 16: one warp set
    const int cend = kN / 2 >= 16 ? cbeg + kHalf : (ch == 0 ? kN : kN);
    // split-K exchange: rank 1 writes its partials into rank 0's receive buffer
    // [kA][kN columns][128 rows] (a warp's 32 rows contiguous) and both sides count every
    // epilogue thread on the partner's barrier
    const uint32_t peer_recv = kSplit == 2 ? mapa_shared(smem_u32(recv), 0) : 0;
    const uint32_t peer_recv_full = kSplit == 2 ? mapa_shared(smem_u32(&ctl->recv_full), 0) : 0;
    const uint32_t peer_recv_free = kSplit == 2 ? mapa_shared(smem_u32(&ctl->recv_free), 1) : 0;
    int jt = 0;
    constexpr int kGroups = kHalf / 16;  // 16-column groups of this warp's columns
    for (int item = unit; item < total; item += n_units, ++jt) {
      const int b = jt % C::kBufs, ub = jt / C::kBufs;
      // The item's tile, its row scales and its token columns' scales do not depend on the
      // accumulators: load them before the wait, so their latency (a tile -> perm -> scale
      // chain through L2) overlaps the item's MMAs instead of following them.
      const Tile tl = checked_tile(a.tiles, item / nblk, a.E, a.R, kN, a.status_flags, 4);
      const int nb = item % nblk;
      const bool shared = tl.group == a.E;
      const int cols = min(cend, tl.nrows);  // this warp's columns of the item end here
      float colscale[kGroups];               // lane i < 16: the scale of column cbeg + 16 g + i
#pragma unroll
      for (int g = 0; g < kGroups; ++g) {
        const int c = cbeg + 16 * g + lane;
        colscale[g] = 0.0f;
        if (lane < 16 && c < cols)
          colscale[g] = kGateUp ? a.sx[checked_token(a.perm[tl.row0 + c], a.T, a.status_flags, 5)] : a.sh[tl.row0 + c];
      }
      float rowscale[kA];  // gate/up: the gate and up scales of this lane's output; down: per block
#pragma unroll
      for (int ai = 0; ai < kA; ++ai) {
        if (kGateUp) {
          const float* sgp = shared ? a.sh_sgu : a.sgu + size_t(tl.group) * 2 * a.F;
          rowscale[ai] = sgp[ai * a.F + nb * kTileM + rloc];
        } else {
          const int m = (nb * kA + ai) * kTileM + rloc;
          rowscale[ai] = shared ? a.sh_sd[m] : a.sd[size_t(tl.group) * a.d + m];
        }
      }
      if (!mbar_wait(&ctl->acc_full[b], ub & 1, &ctl->abort)) {
        if (lane == 0) report_timeout_flag(a.status_flags, 14);
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem + (uint32_t(q * 32) << 16) + uint32_t(b * C::kColsPerAcc);
      if (kSplit == 2 && rank == 1) {  // hand the partial accumulators to rank 0
        if (!mbar_wait_cluster(&ctl->recv_free, (jt & 1) ^ 1, &ctl->abort)) {
          if (lane == 0) report_timeout_flag(a.status_flags, 15);
          break;
        }
#pragma unroll
        for (int ai = 0; ai < kA; ++ai) {
          for (int c0 = cbeg; c0 < cend && c0 < tl.nrows; c0 += 16) {
            float v[16];
            tmem_ld16(taddr + ai * kN + c0, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) st_cluster_f32(peer_recv + uint32_t(((ai * kN + c0 + i) * kTileM + rloc) * 4), v[i]);
          }
        }
        mbar_arrive_cluster(peer_recv_full);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->acc_empty[b]);
        continue;
      }
      if (kSplit == 2 && !mbar_wait_cluster(&ctl->recv_full, jt & 1, &ctl->abort)) {
        if (lane == 0) report_timeout_flag(a.status_flags, 16);
        break;
      }
      // accumulator ai, columns c0..c0+15 of this lane's row: own k-steps, then the partner's
      auto load_acc = [&](int ai, int c0, float (&v)[16]) {
        tmem_ld16(taddr + ai * kN + c0, v);
        if (kSplit == 2) {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] += recv[(ai * kN + c0 + i) * kTileM + rloc];
        }
      };
      if (kGateUp) {
        const int n = nb * kTileM + rloc;
        const float sg = rowscale[0], su = rowscale[1];
#pragma unroll
        for (int gi = 0; gi < kGroups; ++gi) {
          const int c0 = cbeg + 16 * gi;
          if (c0 >= cols) break;
          float gv[16], uv[16];
          load_acc(0, c0, gv);
          load_acc(1, c0, uv);
          const float sx_l = colscale[gi];  // shuffles hand lane i's token scale to every lane
          float* hp = a.h + size_t(tl.row0 + c0) * a.F + n;
          if (c0 + 16 <= tl.nrows) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float sx = __shfl_sync(0xffffffffu, sx_l, i);
              const float gq = gv[i] * sx * sg;
              const float uq = uv[i] * sx * su;
              hp[size_t(i) * a.F] = __fdividef(gq, 1.0f + expf(-gq)) * uq;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float sx = __shfl_sync(0xffffffffu, sx_l, i);
              if (c0 + i < tl.nrows) {
                const float gq = gv[i] * sx * sg;
                const float uq = uv[i] * sx * su;
                hp[size_t(i) * a.F] = __fdividef(gq, 1.0f + expf(-gq)) * uq;
              }
            }
          }
        }
      } else {
#pragma unroll
       for (int ai = 0; ai < kA; ++ai) {  // row block ai of the item: accumulator columns ai * kN
        const int m = (nb * kA + ai) * kTileM + rloc;
        const float sdm = rowscale[ai];
#pragma unroll
        for (int gi = 0; gi < kGroups; ++gi) {
          const int c0 = cbeg + 16 * gi;
          if (c0 >= cols) break;
          float yv[16];
          load_acc(ai, c0, yv);
          const float sh_l = colscale[gi];
          __nv_bfloat16* yp = a.y_rows + size_t(tl.row0 + c0) * a.d + m;
          if (c0 + 16 <= tl.nrows) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              yp[size_t(i) * a.d] = __float2bfloat16_rn(yv[i] * __shfl_sync(0xffffffffu, sh_l, i) * sdm);
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float shv = __shfl_sync(0xffffffffu, sh_l, i);
              if (c0 + i < tl.nrows) yp[size_t(i) * a.d] = __float2bfloat16_rn(yv[i] * shv * sdm);
            }
          }
        }
       }
      }
      if (kSplit == 2) mbar_arrive_cluster(peer_recv_free);  // this thread is done with the receive buffer
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->acc_empty[b]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (kSplit == 2) cluster_sync_all();  // no CTA leaves while its partner may still reach its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side --------------
int sm_count() {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  return sms;
}

template <int kN, bool kGateUp, int kA, int kSplit, int kC, bool kW4 = false>
cudaError_t launch_tc(const CUtensorMap& mx, const CUtensorMap& mw, const CUtensorMap& mwsh, const TcArgs& a,
                      long long max_items, cudaStream_t s) {
  using C = TcCfg<kN, kGateUp, kA, kSplit, kC>;
  static cudaError_t attr = cudaFuncSetAttribute(k_expert_tc<kN, kGateUp, kA, kSplit, kC, kW4>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::kSmemBytes));
  if (attr != cudaSuccess) return attr;
  // one CTA (or one CTA pair) per SM
  const int units = int(std::max<long long>(1, std::min<long long>(max_items, sm_count() / kSplit)));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(units * kSplit);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = kSplit;
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = kSplit == 2 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k_expert_tc<kN, kGateUp, kA, kSplit, kC, kW4>, mx, mw, mwsh, a);
}

template <int kN, int kC, bool kSplit2>
cudaError_t launch_gateup_w(bool w4, const CUtensorMap& mx, const CUtensorMap& mw, const CUtensorMap& mwsh,
                            const TcArgs& a, long long items, cudaStream_t s) {
  constexpr int kS = kSplit2 ? 2 : 1;
  return w4 ? launch_tc<kN, true, 2, kS, kC, true>(mx, mw, mwsh, a, items, s)
            : launch_tc<kN, true, 2, kS, kC, false>(mx, mw, mwsh, a, items, s);
}

// Gate/up: decode tiles (16 or 32 token rows) take two k-chunks per stage (64 KB of weights in
// one copy); wider tiles one chunk (their activation boxes are larger).  E2M1 weights (w4)
// load through the tensor maps mw / mwsh.
cudaError_t launch_gateup_n(int kN, int kC, bool split, bool w4, const CUtensorMap& mx, const CUtensorMap& mw,
                            const CUtensorMap& mwsh, const TcArgs& a, long long items, cudaStream_t s) {
  if (kN == 16 && kC == 2) return split ? launch_gateup_w<16, 2, true>(w4, mx, mw, mwsh, a, items, s)
                                        : launch_gateup_w<16, 2, false>(w4, mx, mw, mwsh, a, items, s);
  if (kN == 16) return split ? launch_gateup_w<16, 1, true>(w4, mx, mw, mwsh, a, items, s)
                             : launch_gateup_w<16, 1, false>(w4, mx, mw, mwsh, a, items, s);
  if (kN == 32) return kC == 2 ? launch_gateup_w<32, 2, false>(w4, mx, mw, mwsh, a, items, s)
                               : launch_gateup_w<32, 1, false>(w4, mx, mw, mwsh, a, items, s);
  if (kN == 64) return kC == 2 ? launch_gateup_w<64, 2, false>(w4, mx, mw, mwsh, a, items, s)
                               : launch_gateup_w<64, 1, false>(w4, mx, mw, mwsh, a, items, s);
  if (kN == 128) return kC == 2 ? launch_gateup_w<128, 2, false>(w4, mx, mw, mwsh, a, items, s)
                                : launch_gateup_w<128, 1, false>(w4, mx, mw, mwsh, a, items, s);
  return cudaErrorInvalidValue;
}

// Down: decode tiles take an item's whole k range (ffn = 640: five chunks, 80 KB in one
// copy) per stage; wider tiles pair two 128-row blocks per stage, one chunk at a time.
template <int kN, int kA, int kC>
cudaError_t launch_down_w(bool w4, const CUtensorMap& mx, const CUtensorMap& mw, const CUtensorMap& mwsh,
                          const TcArgs& a, long long items, cudaStream_t s) {
  return w4 ? launch_tc<kN, false, kA, 1, kC, true>(mx, mw, mwsh, a, items, s)
            : launch_tc<kN, false, kA, 1, kC, false>(mx, mw, mwsh, a, items, s);
}

cudaError_t launch_down_n(int kN, int kA, int kC, bool w4, const CUtensorMap& mx, const CUtensorMap& mw,
                          const CUtensorMap& mwsh, const TcArgs& a, long long items, cudaStream_t s) {
  if (kA == 2) {
    if (kN == 64) return launch_down_w<64, 2, 1>(w4, mx, mw, mwsh, a, items, s);
    if (kN == 128) return launch_down_w<128, 2, 1>(w4, mx, mw, mwsh, a, items, s);
    return cudaErrorInvalidValue;
  }
  if (kN == 16) return kC == 5 ? launch_down_w<16, 1, 5>(w4, mx, mw, mwsh, a, items, s)
                               : launch_down_w<16, 1, 1>(w4, mx, mw, mwsh, a, items, s);
  if (kN == 32) return kC == 5 ? launch_down_w<32, 1, 5>(w4, mx, mw, mwsh, a, items, s)
                               : launch_down_w<32, 1, 1>(w4, mx, mw, mwsh, a, items, s);
  if (kN == 64) return launch_down_w<64, 1, 1>(w4, mx, mw, mwsh, a, items, s);
  if (kN == 128) return launch_down_w<128, 1, 1>(w4, mx, mw, mwsh, a, items, s);
  return cudaErrorInvalidValue;
}

TcArgs tc_args(const LayerDev& L, int T, const WsLayout& ws, char* base) {
  TcArgs a;
  a.T = T;
  a.R = T * (L.k + 1);
  a.d = L.d;
  a.F = L.F;
  a.E = L.E;
  a.tiles = reinterpret_cast<const Tile*>(base + ws.tiles);
  a.n_tiles = reinterpret_cast<const int*>(base + ws.n_tiles);
  a.perm = reinterpret_cast<const int32_t*>(base + ws.perm);
  a.xq = reinterpret_cast<const uint8_t*>(base + ws.xq);
  a.sx = reinterpret_cast<const float*>(base + ws.sx);
  a.sgu = L.sgu;
  a.sh_sgu = L.sh_sgu;
  a.sd = L.sd;
  a.sh_sd = L.sh_sd;
  a.h = reinterpret_cast<float*>(base + ws.h);
  a.sh = reinterpret_cast<const float*>(base + ws.sh);
  a.y_rows = reinterpret_cast<__nv_bfloat16*>(base + ws.y_rows);
  a.status_flags = reinterpret_cast<int*>(base + ws.status);
  a.w = nullptr;
  a.wsh = nullptr;
  return a;
}

long long max_tc_tiles(const LayerDev& L, int T, int kN) {
  const long long R = (long long)T * (L.k + 1);
  return std::min<long long>(R, L.E + 1) + R / kN;
}

}  // namespace

bool tc_supported(const LayerDev& L) { return L.fp8 && L.d % 128 == 0 && L.F % 128 == 0 && encode_fn() != nullptr; }

int tc_rows_per_tile(int T) {
  if (T <= 64) return 16;
  if (T <= 256) return 32;
  if (T <= 1024) return 64;
  return 128;
}

cudaError_t launch_gateup_tc(const LayerDev& L, int T, const WsLayout& ws, char* base, cudaStream_t s) {
  if (!L.tiled) return cudaErrorInvalidValue;
  const int kN = tc_rows_per_tile(T);
  const int KT = L.d / kKTile;
  const int kC = (kN <= kGateUpPairChunkMaxN && KT % 2 == 0) ? 2 : 1;
  CUtensorMap mx;  // activation rows in token order, gathered four rows at a time
  if (!make_map_bytes(&mx, base + ws.xq, uint64_t(T), L.d, 1, 1)) return cudaErrorInvalidValue;
  TcArgs a = tc_args(L, T, ws, base);
  a.w = L.wgu;
  a.wsh = L.sh_wgu;
  CUtensorMap mw = mx, mwsh = mx;  // E2M1 weights: [tiles x 128, 128] code matrices, one tile per box
  if (L.w4) {
    const uint64_t tiles_e = uint64_t(L.F / kTileM) * (L.d / kKTile) * 2;
    if (!make_map_e2m1(&mw, L.wgu, uint64_t(L.E) * tiles_e * kTileM, kTileM) ||
        !make_map_e2m1(&mwsh, L.sh_wgu, tiles_e * kTileM, kTileM))
      return cudaErrorInvalidValue;
  }
  const long long items = max_tc_tiles(L, T, kN) * (L.F / kTileM);
  // a handful of tokens touch few experts: fewer items than SMs, so the k-steps of each item
  // are split over a CTA pair
  const bool split = T <= kSplitMaxT;
  return launch_gateup_n(kN, kC, split, L.w4, mx, mw, mwsh, a, items, s);
}

cudaError_t launch_down_tc(const LayerDev& L, int T, const WsLayout& ws, char* base, cudaStream_t s) {
  if (!L.tiled) return cudaErrorInvalidValue;
  const int kN = tc_rows_per_tile(T);
  const int KT = L.F / kKTile;
  // two 128-row blocks per item (two accumulators fed from one activation stage) where d allows
  // and the tiles are wide enough for the activation traffic to matter
  const int kA = (L.d % (2 * kTileM) == 0 && kN >= kDownPairMinN) ? 2 : 1;
  const int kC = (kA == 1 && kN <= 32 && KT == 5) ? 5 : 1;
  CUtensorMap mx;
  if (!make_map_chunks(&mx, base + ws.qh, uint64_t(ws.R_alloc), L.F, kN, kC)) return cudaErrorInvalidValue;
  TcArgs a = tc_args(L, T, ws, base);
  a.w = L.wd;
  a.wsh = L.sh_wd;
  CUtensorMap mw = mx, mwsh = mx;  // E2M1 weights: [tiles x 128, 128] code matrices, one tile per box
  if (L.w4) {
    const uint64_t tiles_e = uint64_t(L.d / kTileM) * KT;
    if (!make_map_e2m1(&mw, L.wd, uint64_t(L.E) * tiles_e * kTileM, kTileM) ||
        !make_map_e2m1(&mwsh, L.sh_wd, tiles_e * kTileM, kTileM))
      return cudaErrorInvalidValue;
  }
  const long long items = max_tc_tiles(L, T, kN) * (L.d / (kA * kTileM));
  return launch_down_n(kN, kA, kC, L.w4, mx, mw, mwsh, a, items, s);
}

}  // namespace moe
