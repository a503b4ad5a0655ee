// Repacking of the E4M3 (or E2M1) expert weights into the tiled layout the tensor-core kernels stream
// (include/libmoe.h, MOE_LAYOUT_TILED): 16 KB tiles of 128 rows x 128 bytes of k in the
// 128-byte-swizzled order of the MMA operand descriptors, the tiles of one GEMM step
// contiguous.  One thread moves one 16-byte chunk.
#include "common.cuh"

namespace moe {
namespace {

// Tile t of a matrix group: rows row_of(t) .. +127, k bytes 128 kt .. +127.  Gate/up: t =
// ((e * NB + n) * KT + j) * 2 + half, rows half*F + 128 n of expert e (rows 2F, cols d);
// down: t = (e * NB + m) * KT + j, rows 128 m of expert e (rows d, cols F).
__global__ void k_pack_tiles(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, long long n_tiles, int K,
                             int NB, int F, bool gate_up) {
  const int KT = K / 128;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n_tiles * 1024;
       i += (long long)gridDim.x * blockDim.x) {
    const long long t = i >> 10;
    const int within = int(i & 1023);        // 16-byte chunk of the tile, in destination order
    const int r = within >> 3, cd = within & 7;
    const int cs = cd ^ (r & 7);             // the source chunk stored at this position
    long long row;
    int j;
    if (gate_up) {
      const int half = int(t & 1);
      const long long q = t >> 1;
      j = int(q % KT);
      const long long en = q / KT;
      const int n = int(en % NB);
      const long long e = en / NB;
      row = e * 2 * F + half * F + n * 128 + r;
    } else {
      j = int(t % KT);
      const long long em = t / KT;  // = e * NB + m, rows of down are consecutive over (e, m)
      row = em * 128 + r;
    }
    const uint4 v = *reinterpret_cast<const uint4*>(src + row * K + j * 128 + cs * 16);
    *reinterpret_cast<uint4*>(dst + t * 16384 + r * 128 + cd * 16) = v;
  }
}

// The 4-bit tiles: the same tile order, 128 rows of 64 bytes (128 codes of k) per 8 KB tile,
// rows in order and unswizzled.  One thread moves one 16-byte chunk (four per row).
__global__ void k_pack_tiles4(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, long long n_tiles, int K,
                              int NB, int F, bool gate_up) {
  const int KT = K / 128;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n_tiles * 512;
       i += (long long)gridDim.x * blockDim.x) {
    const long long t = i >> 9;
    const int within = int(i & 511);
    const int r = within >> 2, c = within & 3;
    long long row;
    int j;
    if (gate_up) {
      const int half = int(t & 1);
      const long long q = t >> 1;
      j = int(q % KT);
      const long long en = q / KT;
      const int n = int(en % NB);
      const long long e = en / NB;
      row = e * 2 * F + half * F + n * 128 + r;
    } else {
      j = int(t % KT);
      row = (t / KT) * 128 + r;
    }
    const uint4 v = *reinterpret_cast<const uint4*>(src + row * (K / 2) + j * 64 + c * 16);
    *reinterpret_cast<uint4*>(dst + t * 8192 + r * 64 + c * 16) = v;
  }
}

cudaError_t pack4(const void* src, void* dst, long long n_tiles, int K, int NB, int F, bool gate_up, cudaStream_t s) {
  const long long chunks = n_tiles * 512;
  const int grid = int(std::min<long long>((chunks + 255) / 256, 152LL * 32));
  k_pack_tiles4<<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), n_tiles, K, NB, F,
                                      gate_up);
  return cudaGetLastError();
}

cudaError_t pack(const void* src, void* dst, long long n_tiles, int K, int NB, int F, bool gate_up, cudaStream_t s) {
  const long long chunks = n_tiles * 1024;
  const int grid = int(std::min<long long>((chunks + 255) / 256, 152LL * 32));
  k_pack_tiles<<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), n_tiles, K, NB, F,
                                     gate_up);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pack_weights(const LayerDev& L, void* gate_up, void* down, void* sh_gate_up, void* sh_down,
                                cudaStream_t s) {
  const int d = L.d, F = L.F;
  const long long E = L.E;
  if (L.w4) {
    cudaError_t e = pack4(L.wgu, gate_up, E * (F / 128) * (d / 128) * 2, d, F / 128, F, true, s);
    if (e == cudaSuccess) e = pack4(L.wd, down, E * (d / 128) * (F / 128), F, d / 128, F, false, s);
    if (e == cudaSuccess) e = pack4(L.sh_wgu, sh_gate_up, (F / 128) * (d / 128) * 2, d, F / 128, F, true, s);
    if (e == cudaSuccess) e = pack4(L.sh_wd, sh_down, (d / 128) * (F / 128), F, d / 128, F, false, s);
    return e;
  }
  // gate/up: per expert (F/128) x (d/128) x 2 tiles; down: per expert (d/128) x (F/128) tiles
  cudaError_t e = pack(L.wgu, gate_up, E * (F / 128) * (d / 128) * 2, d, F / 128, F, true, s);
  if (e == cudaSuccess) e = pack(L.wd, down, E * (d / 128) * (F / 128), F, d / 128, F, false, s);
  if (e == cudaSuccess) e = pack(L.sh_wgu, sh_gate_up, (F / 128) * (d / 128) * 2, d, F / 128, F, true, s);
  if (e == cudaSuccess) e = pack(L.sh_wd, sh_down, (d / 128) * (F / 128), F, d / 128, F, false, s);
  return e;
}

}  // namespace moe
