// Dispatch building blocks shared by the dispatch kernels and the decode router, which runs
// the one-CTA dispatch itself once the last token's experts are selected.
#pragma once

#include "common.cuh"

namespace moe {

template <class F>
__device__ __forceinline__ void warp_walk(const int32_t* __restrict__ ids, int t0, int t1, int k, int E, int* cnt,
                                          F f) {
  const int lane = threadIdx.x & 31;
  const int tpi = 32 / k;
  const int tl = lane / k, s = lane - (lane / k) * k;
  for (int base = t0; base < t1; base += tpi) {
    const int t = base + tl;
    int e = (tl < tpi && t < t1) ? ids[size_t(t) * k + s] : -1;
    if (e >= E) e = -1;  // out-of-range ids get no row
    const unsigned m = __match_any_sync(0xffffffffu, e);
    if (e >= 0) f(t, s, cnt[e] + __popc(m & ((1u << lane) - 1u)));
    __syncwarp();
    if (e >= 0 && (31 - __clz(m)) == lane) cnt[e] += __popc(m);
    __syncwarp();
  }
}

// Exclusive scan of n <= 2 * blockDim ints in shared memory (blockDim = 1024).  Returns the
// total to every thread.
__device__ __forceinline__ int block_exclusive_scan(int* a, int n, int* warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i0 = 2 * tid, i1 = 2 * tid + 1;
  const int v0 = i0 < n ? a[i0] : 0, v1 = i1 < n ? a[i1] : 0;
  int s = v0 + v1, incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int wt = lane < (blockDim.x >> 5) ? warp_tot[lane] : 0, wi = wt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_tot[lane] = wi - wt;  // exclusive warp offsets
    if (lane == 31) warp_tot[32] = wi;
  }
  __syncthreads();
  const int ex = warp_tot[warp] + incl - s;
  const int total = warp_tot[32];
  __syncthreads();
  if (i0 < n) a[i0] = ex;
  if (i1 < n) a[i1] = ex + v0;
  __syncthreads();
  return total;
}

struct DispatchOut {
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* pos;
  int32_t* chunk_base;  // [n_chunks, E]: counts per chunk, then their exclusive prefix
  Tile* tiles;
  int32_t* n_tiles;
};

// T <= kDispatchChunk and E < 512: the whole dispatch in one CTA of kLeanWarps warps,
// everything in shared memory (lean_dispatch_smem_ints(T, E, k) ints at smem).  The ids are
// staged first, read through L2 (they may have been written by other CTAs of the caller's
// grid); warp w owns the run of tokens [w*tpw, (w+1)*tpw); per-warp counts become per-warp
// row bases by a prefix over the warps, then over the experts.
constexpr int kLeanWarps = 8;
__host__ __device__ constexpr int lean_dispatch_smem_ints(int T, int E, int k) {
  return kLeanWarps * E + 3 * (E + 1) + T * k + 33;
}

__device__ __forceinline__ void dispatch_lean_body(const int32_t* ids_g, int T, int E, int k, int rows_per_tile,
                                                   const DispatchOut& o, int* smem) {
  int* wcnt = smem;                  // [kLeanWarps][E]
  int* tot = smem + kLeanWarps * E;  // [E + 1] counts, then offsets
  int* cnt = tot + E + 1;            // [E + 1] counts (the tile list reads them here, not back from global)
  int* ntile = cnt + E + 1;          // [E + 1] tiles per group (shared expert first), then their prefix
  int* ids = ntile + E + 1;          // [T * k], the staged ids
  int* warp_tot = ids + T * k;       // [33]
  const int warp = threadIdx.x >> 5;
  const int tpw = (T + kLeanWarps - 1) / kLeanWarps;
  const int t0 = min(T, warp * tpw), t1 = min(T, t0 + tpw);
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) ids[i] = __ldcg(ids_g + i);
  for (int i = threadIdx.x; i < kLeanWarps * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  warp_walk(ids, t0, t1, k, E, wcnt + warp * E, [](int, int, int) {});
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < kLeanWarps; ++w) {
      const int v = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += v;
    }
    tot[e] = run;
    cnt[e] = run;
    o.counts[e] = run;
  }
  __syncthreads();
  block_exclusive_scan(tot, E, warp_tot);  // tot[e] = offset of expert e
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    o.offsets[e] = tot[e];
    for (int w = 0; w < kLeanWarps; ++w) wcnt[w * E + e] += tot[e];
  }
  if (threadIdx.x == 0) {
    o.counts[E] = T;
    o.offsets[E] = k * T;
    o.offsets[E + 1] = (k + 1) * T;
  }
  __syncthreads();
  // tile list, shared expert first: tile counts per group, scanned
  for (int q = threadIdx.x; q <= E; q += blockDim.x) {
    const int g = q == 0 ? E : q - 1;
    const int c = g == E ? T : cnt[g];
    ntile[q] = (c + rows_per_tile - 1) / rows_per_tile;
  }
  __syncthreads();
  const int total_tiles = block_exclusive_scan(ntile, E + 1, warp_tot);
  for (int q = threadIdx.x; q <= E; q += blockDim.x) {
    const int g = q == 0 ? E : q - 1;
    const int c = g == E ? T : cnt[g];
    const int base_row = g == E ? k * T : tot[g];
    int ti = ntile[q];
    for (int r = 0; r < c; r += rows_per_tile, ++ti) {
      Tile tl;
      tl.group = g;
      tl.row0 = base_row + r;
      tl.nrows = min(rows_per_tile, c - r);
      tl.pad = 0;
      o.tiles[ti] = tl;
    }
  }
  if (threadIdx.x == 0) *o.n_tiles = total_tiles;
  // rows: invalid slots get pos = -1; valid ones are placed in token order
  for (int i = (threadIdx.x & 31); i < (t1 - t0) * k; i += 32) {
    const int t = t0 + i / k;
    const int e = ids[size_t(t) * k + (i % k)];
    if (e < 0 || e >= E) o.pos[size_t(t) * k + (i % k)] = -1;
  }
  int32_t* perm = o.perm;
  int32_t* pos = o.pos;
  warp_walk(ids, t0, t1, k, E, wcnt + warp * E, [&](int t, int s, int row) {
    perm[row] = t;
    pos[size_t(t) * k + s] = row;
  });
  for (int t = threadIdx.x; t < T; t += blockDim.x) perm[size_t(k) * T + t] = t;
}


}  // namespace moe
