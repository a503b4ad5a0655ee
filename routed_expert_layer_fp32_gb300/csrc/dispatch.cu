// Dispatch: group the T*k routed (token, slot) rows by expert, stably (tokens ascend within
// an expert), append the shared expert's T rows, and cut every group into row tiles for the
// expert kernels.  This is the "sorted" grouping that the batched expert layer relies on
// ("We Ported Aleph Alpha's Kolibri to a MacBook. Our Own Gate Said No.", section 3: the
// sorted gather path, used once a call has 64 or more (token, expert) rows).
//
// Each warp owns a run of consecutive tokens and walks it in steps of 32/k tokens, one lane
// per (token, slot).  __match_any_sync groups the lanes that name the same expert; a lane's
// rank is its warp-private counter plus the number of lower lanes in its group (lower lane =
// earlier token, so the order is stable), and the group's highest lane advances the counter.
// The per-warp counts are combined by prefix sums across warps, CTAs and experts.
#include "common.cuh"
#include "dispatch_dev.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;  // warps per chunk CTA (256 threads)
constexpr int kTokensPerWarp = kScatterChunk / kWarps;


// Phase 1 (per CTA): per-warp counts of the chunk -> chunk totals [chunk][e].
// Warps of this CTA that own tokens (the rest skip every per-warp loop).
__device__ __forceinline__ int active_warps(int T) {
  const int n = min(T - int(blockIdx.x) * kScatterChunk, kScatterChunk);
  return min(kWarps, (n + kTokensPerWarp - 1) / kTokensPerWarp);
}

// The chunk's ids, staged in shared memory with every load issued at once (the walks then
// read shared memory, not one L2 round trip per step).  Returns the chunk's token count.
__device__ __forceinline__ int stage_chunk_ids(const int32_t* ids, int T, int k, int* ids_s) {
  const int c0 = blockIdx.x * kScatterChunk;
  const int n = min(T - c0, kScatterChunk);
  for (int i = threadIdx.x; i < n * k; i += blockDim.x) ids_s[i] = __ldcg(ids + size_t(c0) * k + i);
  return n;
}

// smem: [kWarps][E] per-warp counters, then the chunk's ids [kScatterChunk][k]
__device__ void count_chunk(const int32_t* ids, int T, int E, int k, int* wcnt, int32_t* chunk_row) {
  const int warp = threadIdx.x >> 5;
  const int nw = active_warps(T);
  int* ids_s = wcnt + kWarps * E;
  const int n = stage_chunk_ids(ids, T, k, ids_s);
  for (int i = threadIdx.x; i < nw * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  const int t0 = min(n, warp * kTokensPerWarp), t1 = min(n, t0 + kTokensPerWarp);  // chunk-relative
  warp_walk(ids_s, t0, t1, k, E, wcnt + warp * E, [](int, int, int) {});
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int s = 0;
    for (int w = 0; w < nw; ++w) s += wcnt[w * E + e];
    chunk_row[e] = s;
  }
}

// Scan across chunks and experts, and the tile list (shared expert's tiles first).
__device__ void scan_and_tiles(int T, int E, int k, int n_chunks, int rows_per_tile, const DispatchOut& o,
                               int* sm_a, int* warp_tot) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int c0 = 0; c0 < n_chunks; c0 += 16) {  // sixteen chunks' loads in flight at once
      int v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = c0 + j < n_chunks ? o.chunk_base[size_t(c0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (c0 + j < n_chunks) {
          o.chunk_base[size_t(c0 + j) * E + e] = run;
          run += v[j];
        }
    }
    sm_a[e] = run;
    o.counts[e] = run;
  }
  __syncthreads();
  block_exclusive_scan(sm_a, E, warp_tot);
  for (int e = threadIdx.x; e < E; e += blockDim.x) o.offsets[e] = sm_a[e];
  if (threadIdx.x == 0) {
    o.counts[E] = T;
    o.offsets[E] = k * T;
    o.offsets[E + 1] = (k + 1) * T;
  }
  __syncthreads();
  // tiles: group order shared (E), 0, 1, ..., E-1
  for (int q = threadIdx.x; q <= E; q += blockDim.x) {
    const int g = q == 0 ? E : q - 1;
    const int c = g == E ? T : o.counts[g];
    sm_a[q] = (c + rows_per_tile - 1) / rows_per_tile;
  }
  __syncthreads();
  const int total = block_exclusive_scan(sm_a, E + 1, warp_tot);
  for (int q = threadIdx.x; q <= E; q += blockDim.x) {
    const int g = q == 0 ? E : q - 1;
    const int c = g == E ? T : o.counts[g];
    const int base_row = g == E ? k * T : o.offsets[g];
    int ti = sm_a[q];
    for (int r = 0; r < c; r += rows_per_tile, ++ti) {
      Tile t;
      t.group = g;
      t.row0 = base_row + r;
      t.nrows = min(rows_per_tile, c - r);
      t.pad = 0;
      o.tiles[ti] = t;
    }
  }
  if (threadIdx.x == 0) *o.n_tiles = total;
}

// Phase 3 (per CTA): ranks again, now offset by the rows of earlier warps, chunks and
// experts; writes perm and pos, plus the shared expert's rows.
__device__ void scatter_chunk(const int32_t* ids, int T, int E, int k, int* wcnt, const DispatchOut& o) {
  const int warp = threadIdx.x >> 5;
  const int nw = active_warps(T);
  int* ids_s = wcnt + kWarps * E;
  const int n = stage_chunk_ids(ids, T, k, ids_s);
  const int cbase = blockIdx.x * kScatterChunk;  // token index of the chunk's first token
  for (int i = threadIdx.x; i < nw * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  const int t0 = min(n, warp * kTokensPerWarp), t1 = min(n, t0 + kTokensPerWarp);  // chunk-relative
  warp_walk(ids_s, t0, t1, k, E, wcnt + warp * E, [](int, int, int) {});
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = o.offsets[e] + o.chunk_base[size_t(blockIdx.x) * E + e];
    for (int w = 0; w < nw; ++w) {
      int v = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += v;
    }
  }
  __syncthreads();
  int32_t* perm = o.perm;
  int32_t* pos = o.pos;
  // invalid slots (id < 0) get no row
  for (int i = (threadIdx.x & 31); i < (t1 - t0) * k; i += 32) {
    const int t = t0 + i / k;
    const int e = ids_s[t * k + (i % k)];
    if (e < 0 || e >= E) pos[size_t(cbase + t) * k + (i % k)] = -1;
  }
  warp_walk(ids_s, t0, t1, k, E, wcnt + warp * E, [&](int t, int s, int row) {
    perm[row] = cbase + t;
    pos[size_t(cbase + t) * k + s] = row;
  });
  for (int t = blockIdx.x * kScatterChunk + threadIdx.x; t < min(T, (blockIdx.x + 1) * kScatterChunk); t += blockDim.x)
    perm[size_t(k) * T + t] = t;
}

__global__ void __launch_bounds__(kWarps * 32) k_dispatch_count(const int32_t* __restrict__ ids, int T, int E, int k,
                                                         DispatchOut o) {
  pdl_begin();
  extern __shared__ int smem[];
  count_chunk(ids, T, E, k, smem, o.chunk_base + size_t(blockIdx.x) * E);
}

__global__ void __launch_bounds__(1024) k_dispatch_scan(int T, int E, int k, int n_chunks, int rows_per_tile,
                                                        DispatchOut o) {
  pdl_begin();
  __shared__ int sm_a[kMaxExperts + 1];
  __shared__ int warp_tot[33];
  scan_and_tiles(T, E, k, n_chunks, rows_per_tile, o, sm_a, warp_tot);
}

__global__ void __launch_bounds__(kWarps * 32) k_dispatch_scatter(const int32_t* __restrict__ ids, int T, int E, int k,
                                                           DispatchOut o) {
  pdl_begin();
  extern __shared__ int smem[];
  scatter_chunk(ids, T, E, k, smem, o);
}

__global__ void __launch_bounds__(kLeanWarps * 32) k_dispatch_lean(const int32_t* __restrict__ ids_g, int T, int E,
                                                                  int k, int rows_per_tile, DispatchOut o) {
  pdl_begin();
  extern __shared__ int lean_smem[];
  dispatch_lean_body(ids_g, T, E, k, rows_per_tile, o, lean_smem);
}

}  // namespace

void dispatch_outputs(const WsLayout& ws, char* base, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* pos,
                      DispatchOut* o) {
  o->counts = counts;
  o->offsets = offsets;
  o->perm = perm;
  o->pos = pos;
  o->chunk_base = reinterpret_cast<int32_t*>(base + ws.chunk_counts);
  o->tiles = reinterpret_cast<Tile*>(base + ws.tiles);
  o->n_tiles = reinterpret_cast<int32_t*>(base + ws.n_tiles);
}

cudaError_t launch_dispatch(const int32_t* ids, int T, int E, int k, int rows_per_tile, const WsLayout& ws, char* base,
                            int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* pos, cudaStream_t s) {
  DispatchOut o;
  dispatch_outputs(ws, base, counts, offsets, perm, pos, &o);
  const size_t smem = (size_t(kWarps) * E + size_t(kScatterChunk) * k) * sizeof(int);
  const int n_chunks = (T + kScatterChunk - 1) / kScatterChunk;
  // opt in once per process to the largest per-warp counter table (E <= kMaxExperts); later
  // calls (also inside a stream capture) only launch
  static cudaError_t attr = [] {
    const int most = int((size_t(kWarps) * kMaxExperts + size_t(kScatterChunk) * kTopK) * sizeof(int));
    cudaError_t e2 = cudaFuncSetAttribute(k_dispatch_count, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    cudaError_t e3 = cudaFuncSetAttribute(k_dispatch_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    return e2 != cudaSuccess ? e2 : e3;
  }();
  if (attr != cudaSuccess) return attr;
  if (T <= kDispatchChunk && E < 512) {
    const size_t lean = size_t(lean_dispatch_smem_ints(T, E, k)) * sizeof(int);
    return launch_pdl(k_dispatch_lean, dim3(1), dim3(kLeanWarps * 32), lean, s, ids, T, E, k, rows_per_tile, o);
  }
  cudaError_t e = launch_pdl(k_dispatch_count, dim3(n_chunks), dim3(kWarps * 32), smem, s, ids, T, E, k, o);
  if (e == cudaSuccess) e = launch_pdl(k_dispatch_scan, dim3(1), dim3(1024), 0, s, T, E, k, n_chunks, rows_per_tile, o);
  if (e == cudaSuccess) e = launch_pdl(k_dispatch_scatter, dim3(n_chunks), dim3(kWarps * 32), smem, s, ids, T, E, k, o);
  return e;
}

}  // namespace moe
