// sort.cu -- expert sort (TileOPs "MoE" page, op MoEPermuteAlignFwd), row gather (op
// MoEPrePermuteFwd), GEMM tile schedule, and the deterministic top-k combine (op
// MoEPostPermuteFwd; aiter PR #5973 "Changes": sorted_sum writes the output in full).
//
// The sort is a stable counting sort of the flat route index r = t*top_k + j by expert id,
// done in three launches over 256-route chunks:
//   count:   per-chunk expert histogram (shared-memory integer atomics: order-independent)
//   scan:    per expert, exclusive prefix over chunks; block-wide scan of the block_m-padded
//            counts gives the segment offsets; padding slots are filled with -1
//   scatter: rank of a route among the equal ids before it in its chunk, plus the chunk base,
//            plus the segment offset = its sorted position
// so every route lands at a position that depends only on topk_ids (bit-exact and
// deterministic).
#include "common.cuh"

namespace gb300moe {

namespace {

constexpr int kChunk = 256;

__global__ void __launch_bounds__(kChunk)
    sort_count_kernel(const int32_t* __restrict__ ids, int P, int E,
                      int32_t* __restrict__ chunk_counts, int* status) {
  extern __shared__ int hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int r = blockIdx.x * kChunk + threadIdx.x;
  if (r < P) {
    const int e = ids[r];
    if (e >= 0 && e < E)
      atomicAdd(&hist[e], 1);
    else if (e != -1)
      set_status(status, MOE_ERR_BAD_EXPERT_ID);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_counts[(size_t)blockIdx.x * E + e] = hist[e];
}

// Block-wide inclusive scan of one int per thread (blockDim.x <= 1024).
__device__ int block_inclusive_scan(int v, int* warp_tot) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  if (lane == 31) warp_tot[w] = v;
  __syncthreads();
  if (w == 0) {
    const int nw = (blockDim.x + 31) >> 5;
    int s = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += o;
    }
    if (lane < nw) warp_tot[lane] = s;  // inclusive totals per warp
  }
  __syncthreads();
  const int before = w > 0 ? warp_tot[w - 1] : 0;
  return v + before;
}

__global__ void __launch_bounds__(1024)
    sort_scan_kernel(int n_chunks, int E, int block_m, int64_t cap,
                     int32_t* __restrict__ chunk_counts, int32_t* __restrict__ counts,
                     int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_ids,
                     int32_t* __restrict__ tile_expert, int64_t tile_len) {
  __shared__ int warp_tot[32];
  __shared__ int s_total;
  const int e = threadIdx.x;
  int total = 0;
  if (e < E) {
    for (int c = 0; c < n_chunks; ++c) {
      const size_t i = (size_t)c * E + e;
      const int v = chunk_counts[i];
      chunk_counts[i] = total;  // becomes the chunk's base within expert e
      total += v;
    }
  }
  const int padded = e < E ? (total + block_m - 1) / block_m * block_m : 0;
  const int incl = block_inclusive_scan(padded, warp_tot);
  const int excl = incl - padded;
  if (e < E) {
    counts[e] = total;
    offsets[e] = excl;
  }
  if (e == E - 1) {
    offsets[E] = incl;
    s_total = incl;
  }
  __syncthreads();
  const int tot = s_total;
  if (e < E)
    for (int q = excl + total; q < excl + padded; ++q) sorted_ids[q] = -1;
  for (int64_t q = tot + threadIdx.x; q < cap; q += blockDim.x) sorted_ids[q] = -1;
  if (tile_expert) {
    if (e < E)
      for (int i = excl / block_m; i < (excl + padded) / block_m; ++i) tile_expert[i] = e;
    for (int64_t i = tot / block_m + threadIdx.x; i < tile_len; i += blockDim.x)
      tile_expert[i] = -1;
  }
}

__global__ void __launch_bounds__(kChunk)
    sort_scatter_kernel(const int32_t* __restrict__ ids, int P, int E,
                        const int32_t* __restrict__ chunk_base,
                        const int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_ids,
                        int32_t* __restrict__ inv_route) {
  __shared__ int s_ids[kChunk];
  const int r = blockIdx.x * kChunk + threadIdx.x;
  int e = r < P ? ids[r] : -1;
  if (e < -1 || e >= E) e = -1;  // reported by the count kernel; treated as padding
  s_ids[threadIdx.x] = e;
  __syncthreads();
  if (r >= P) return;
  if (e < 0) {
    inv_route[r] = -1;
    return;
  }
  int rank = 0;
  for (int i = 0; i < (int)threadIdx.x; ++i) rank += (s_ids[i] == e);
  const int pos = offsets[e] + chunk_base[(size_t)blockIdx.x * E + e] + rank;
  sorted_ids[pos] = r;
  inv_route[r] = pos;
}

// Tiles of at most kTileRows rows over each expert segment [offsets[e], offsets[e+1]).
__global__ void __launch_bounds__(1024)
    build_tiles_kernel(int E, const int32_t* __restrict__ offsets, Tile* __restrict__ tiles,
                       int* __restrict__ n_tiles) {
  __shared__ int warp_tot[32];
  const int e = threadIdx.x;
  const int seg = e < E ? offsets[e + 1] - offsets[e] : 0;
  const int nt = (seg + kTileRows - 1) / kTileRows;
  const int incl = block_inclusive_scan(nt, warp_tot);
  const int base = incl - nt;
  if (e < E) {
    const int r0 = offsets[e];
    for (int i = 0; i < nt; ++i) {
      Tile t;
      t.e = e;
      t.row0 = r0 + i * kTileRows;
      t.nrows = min(kTileRows, seg - i * kTileRows);
      t.pad = 0;
      tiles[base + i] = t;
    }
  }
  if (e == E - 1) *n_tiles = incl;
}

// a_sorted[p, :] = hidden[sorted_ids[p] / top_k, :] for p < offsets[E]; padding rows are zero.
__global__ void __launch_bounds__(128)
    permute_kernel(int top_k, int H, const uint16_t* __restrict__ hidden,
                   const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ offsets,
                   int E, uint16_t* __restrict__ a_sorted) {
  const int64_t rows = offsets[E];
  const int nvec = H / 8;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const int sid = sorted_ids[row];
    uint4* dst = reinterpret_cast<uint4*>(a_sorted + row * H);
    if (sid < 0) {
      for (int v = threadIdx.x; v < nvec; v += blockDim.x) dst[v] = make_uint4(0, 0, 0, 0);
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(hidden + (int64_t)(sid / top_k) * H);
      for (int v = threadIdx.x; v < nvec; v += blockDim.x) dst[v] = src[v];
    }
  }
}

// out[t, :] = round(sum_j y[inv[t*K+j], :] + shared[t, :]): f32 rows in, one rounding out.
template <typename T>
__global__ void __launch_bounds__(128)
    combine_kernel(int K, int H, const float* __restrict__ y, const int32_t* __restrict__ inv,
                   const int32_t* __restrict__ ids, const float* __restrict__ shared,
                   T* __restrict__ out) {
  const int t = blockIdx.y;
  const int v = blockIdx.x * blockDim.x + threadIdx.x;  // 8 columns per thread
  if (v >= H / 8) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  for (int j = 0; j < K; ++j) {
    const int r = t * K + j;
    if (ids && ids[r] < 0) continue;
    const int p = inv ? inv[r] : r;
    if (p < 0) continue;
    const float4* src = reinterpret_cast<const float4*>(y + (int64_t)p * H) + 2 * v;
    const float4 a = src[0], b = src[1];
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
  }
  if (shared) {
    const float4* src = reinterpret_cast<const float4*>(shared + (int64_t)t * H) + 2 * v;
    const float4 a = src[0], b = src[1];
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
  }
  uint4 o;
  T* oe = reinterpret_cast<T*>(&o);
#pragma unroll
  for (int i = 0; i < 8; ++i) oe[i] = DT<T>::from_f(acc[i]);
  reinterpret_cast<uint4*>(out + (int64_t)t * H)[v] = o;
}

}  // namespace

cudaError_t launch_align_sort(const moe_problem_t& p, int block_m, const int32_t* ids,
                              int32_t* counts, int32_t* offsets, int32_t* sorted_ids,
                              int64_t cap, int32_t* tile_expert, int32_t* inv_route,
                              int32_t* chunk_scratch, int* status, cudaStream_t s) {
  const int P = p.T * p.top_k;
  const int n_chunks = (P + kChunk - 1) / kChunk;
  const int64_t tile_len = (cap + block_m - 1) / block_m;
  if (n_chunks > 0) {
    sort_count_kernel<<<n_chunks, kChunk, sizeof(int) * p.E, s>>>(ids, P, p.E, chunk_scratch,
                                                                   status);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  sort_scan_kernel<<<1, 1024, 0, s>>>(n_chunks, p.E, block_m, cap, chunk_scratch, counts,
                                      offsets, sorted_ids, tile_expert, tile_len);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess || n_chunks == 0) return err;
  sort_scatter_kernel<<<n_chunks, kChunk, 0, s>>>(ids, P, p.E, chunk_scratch, offsets,
                                                  sorted_ids, inv_route);
  return cudaGetLastError();
}

cudaError_t launch_build_tiles(int E, const int32_t* offsets, Tile* tiles, int* n_tiles,
                               cudaStream_t s) {
  build_tiles_kernel<<<1, 1024, 0, s>>>(E, offsets, tiles, n_tiles);
  return cudaGetLastError();
}

cudaError_t launch_permute(int dtype, int top_k, int H, const void* hidden,
                           const int32_t* sorted_ids, const int32_t* offsets, int E, int64_t cap,
                           void* a_sorted, cudaStream_t s) {
  (void)dtype;  // a row copy: the element type does not matter
  if (cap <= 0) return cudaSuccess;
  const int64_t grid = cap < 4096 ? cap : 4096;
  permute_kernel<<<(int)grid, 128, 0, s>>>(top_k, H, static_cast<const uint16_t*>(hidden),
                                           sorted_ids, offsets, E,
                                           static_cast<uint16_t*>(a_sorted));
  return cudaGetLastError();
}

cudaError_t launch_combine(const moe_problem_t& p, const void* y_route,
                           const int32_t* inv_route, const int32_t* ids, const void* shared_out,
                           void* out, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  dim3 grid((p.H / 8 + 127) / 128, p.T);
  if (p.dtype == MOE_BF16) {
    combine_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(
        p.top_k, p.H, static_cast<const float*>(y_route), inv_route, ids,
        static_cast<const float*>(shared_out), static_cast<__nv_bfloat16*>(out));
  } else {
    combine_kernel<__half><<<grid, 128, 0, s>>>(
        p.top_k, p.H, static_cast<const float*>(y_route), inv_route, ids,
        static_cast<const float*>(shared_out), static_cast<__half*>(out));
  }
  return cudaGetLastError();
}

}  // namespace gb300moe
