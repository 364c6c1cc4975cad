// nvfp4_pack.cu -- NVFP4 expert weights rearranged into the tile layout the W4A16 GEMMs stream
// (flashinfer PR #4048 serves its NVFP4 weights in a kernel-specific scale layout too; this one
// is this library's own).
//
// Input, per matrix m (one expert's gate/up or down projection): codes [rows, K/2] bytes (two
// E2M1 codes per byte, element 2i in the low nibble) and scales [rows, K/16] bytes (E4M3, one
// per 16 consecutive k).  Output: for every (m, 128-row slab s, 128-k block b), in that order, a
// 9216-byte tile:
//   bytes [0, 8192)     the slab's 128 rows of 64 code bytes; row r at r * 64, and its 16-byte
//                       chunk j (codes of k = 32j .. 32j+31 of the block) at chunk position
//                       j ^ ((r >> 1) & 3), so that a warp reading one row per thread touches
//                       every shared-memory bank once per 128 bytes;
//   bytes [8192, 9216)  the 128 rows' 8 scale bytes, row r at 8192 + r * 8.
// The GEMM reads one tile per slab and stage with a single contiguous bulk copy, instead of 128
// strided 64-byte rows and 128 separate 8-byte scale rows.
#include "common.cuh"

namespace gb300moe {

namespace {

constexpr int kPackRows = 128;
constexpr int kPackK = 128;
constexpr int kPackTileBytes = kPackRows * kPackK / 2 + kPackRows * kPackK / 16;  // 9216

// One thread per (tile, row): four 16-byte code chunks and one 8-byte scale row.
__global__ void __launch_bounds__(256) nvfp4_pack_kernel(int64_t n_tiles, int slabs, int blocks,
                                                         int K, const uint8_t* __restrict__ codes,
                                                         const uint8_t* __restrict__ scales,
                                                         uint8_t* __restrict__ tiles) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_tiles * kPackRows) return;
  const int r = (int)(i % kPackRows);
  const int64_t t = i / kPackRows;
  const int b = (int)(t % blocks);
  const int64_t ms = t / blocks;  // m * slabs + s
  const int64_t grow = ms * kPackRows + r;  // row over all matrices
  const uint8_t* src = codes + grow * (K / 2) + (int64_t)b * (kPackK / 2);
  uint8_t* dst = tiles + t * kPackTileBytes;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * j);
    *reinterpret_cast<uint4*>(dst + r * 64 + 16 * (j ^ ((r >> 1) & 3))) = v;
  }
  *reinterpret_cast<uint2*>(dst + kPackRows * kPackK / 2 + r * 8) =
      *reinterpret_cast<const uint2*>(scales + grow * (K / 16) + (int64_t)b * (kPackK / 16));
  (void)slabs;
}

}  // namespace

cudaError_t launch_nvfp4_pack(int64_t n_mats, int rows, int K, const uint8_t* codes,
                              const uint8_t* scales, uint8_t* tiles, cudaStream_t s) {
  const int slabs = rows / kPackRows, blocks = K / kPackK;
  const int64_t n_tiles = n_mats * slabs * blocks;
  if (n_tiles == 0) return cudaSuccess;
  const int64_t threads = n_tiles * kPackRows;
  const int64_t grid = (threads + 255) / 256;
  return launch_k(nvfp4_pack_kernel, dim3((unsigned)grid), dim3(256), 0, s, false, n_tiles,
                  slabs, blocks, K, codes, scales, tiles);
}

}  // namespace gb300moe
