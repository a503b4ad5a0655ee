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
// grid), unless the caller staged them already (ids_staged: T * k ints at
// smem + lean_dispatch_ids_offset(E)); warp w owns the run of tokens [w*tpw, (w+1)*tpw).
// Per-warp counts become per-warp row bases within each expert by a prefix over the warps;
// one scan over the experts then gives both the row offsets and the tile indices: each
// expert's (rows << 16 | tiles) is scanned as one int (rows <= 6144 and tiles <= 6656 here, so
// neither half carries into the other).  The shared expert's tiles come first.
constexpr int kLeanWarps = 8;
__host__ __device__ constexpr int lean_dispatch_ids_offset(int E) { return kLeanWarps * E + 3 * (E + 1); }
__host__ __device__ constexpr int lean_dispatch_smem_ints(int T, int E, int k) {
  return lean_dispatch_ids_offset(E) + T * k + 33;
}

__device__ __forceinline__ void dispatch_lean_body(const int32_t* ids_g, int T, int E, int k, int rows_per_tile,
                                                   const DispatchOut& o, int* smem, bool ids_staged = false) {
  int* wcnt = smem;                  // [kLeanWarps][E]
  int* pk = smem + kLeanWarps * E;   // [E + 1] packed rows and tiles per expert, then their exclusive prefix
  int* cnt = pk + E + 1;             // [E + 1] rows per expert
  int* ids = smem + lean_dispatch_ids_offset(E);  // [T * k], the staged ids
  int* warp_tot = ids + T * k;       // [33]
  const int warp = threadIdx.x >> 5;
  const int tpw = (T + kLeanWarps - 1) / kLeanWarps;
  const int t0 = min(T, warp * tpw), t1 = min(T, t0 + tpw);
  if (!ids_staged)
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
    cnt[e] = run;
    o.counts[e] = run;
    pk[e] = (run << 16) | ((run + rows_per_tile - 1) / rows_per_tile);
  }
  __syncthreads();
  const int total = block_exclusive_scan(pk, E, warp_tot);
  const int sh_tiles = (T + rows_per_tile - 1) / rows_per_tile;  // the shared expert's, first
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int off = pk[e] >> 16, c = cnt[e];
    o.offsets[e] = off;
    for (int w = 0; w < kLeanWarps; ++w) wcnt[w * E + e] += off;
    int ti = sh_tiles + (pk[e] & 0xffff);
    for (int r = 0; r < c; r += rows_per_tile, ++ti) {
      Tile tl;
      tl.group = e;
      tl.row0 = off + r;
      tl.nrows = min(rows_per_tile, c - r);
      tl.pad = 0;
      o.tiles[ti] = tl;
    }
  }
  if (threadIdx.x == 0) {
    o.counts[E] = T;
    o.offsets[E] = k * T;
    o.offsets[E + 1] = (k + 1) * T;
    int ti = 0;
    for (int r = 0; r < T; r += rows_per_tile, ++ti) {
      Tile tl;
      tl.group = E;
      tl.row0 = k * T + r;
      tl.nrows = min(rows_per_tile, T - r);
      tl.pad = 0;
      o.tiles[ti] = tl;
    }
    *o.n_tiles = sh_tiles + (total & 0xffff);
  }
  __syncthreads();
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
