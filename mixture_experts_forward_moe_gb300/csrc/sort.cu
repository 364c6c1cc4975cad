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
#include "ptx.cuh"

namespace gb300moe {

namespace {

constexpr int kChunk = 256;

__global__ void __launch_bounds__(kChunk)
    sort_count_kernel(const int32_t* __restrict__ ids, int P, int E,
                      int32_t* __restrict__ chunk_counts, int* status) {
  extern __shared__ int hist[];
  pdl_wait();
  pdl_trigger();
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

// Tile lists of `rows` rows over the padded expert segments (thread e owns expert e); the
// caller has synchronised the block, and warp_tot is reused by the block scan.
__device__ void write_tile_list(int E, int excl, int padded, int rows, Tile* tiles, int* n_tiles,
                                int* warp_tot) {
  const int e = threadIdx.x;
  const int nt = e < E ? (padded + rows - 1) / rows : 0;
  const int incl = block_inclusive_scan(nt, warp_tot);
  const int base = incl - nt;
  for (int i = 0; i < nt; ++i) {
    Tile t;
    t.e = e;
    t.row0 = excl + i * rows;
    t.nrows = min(rows, padded - i * rows);
    t.first = base;
    t.count = nt;
    t.pad0 = t.pad1 = t.pad2 = 0;
    tiles[base + i] = t;
  }
  if (e == E - 1) *n_tiles = incl;
}

// Per expert, the exclusive prefix of the chunk histograms over chunks (a thread per expert),
// then the block scan of the padded totals into the segment offsets, the padding slots,
// tile_expert and (optionally) the two GEMM tile lists.
__global__ void __launch_bounds__(1024)
    sort_scan_kernel(int n_chunks, int E, int block_m, int64_t cap,
                     int32_t* __restrict__ chunk_counts, int32_t* __restrict__ counts,
                     int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_ids,
                     int32_t* __restrict__ tile_expert, int64_t tile_len, Tile* __restrict__ tiles,
                     int* __restrict__ n_tiles, int tile_rows, Tile* __restrict__ tiles2,
                     int* __restrict__ n_tiles2, int tile_rows2) {
  __shared__ int warp_tot[32];
  __shared__ int s_total;
  __shared__ int s_expert_total[1024];
  pdl_wait();
  pdl_trigger();
  {
    // Thread e walks expert e's column of the chunk histograms: at each step the warp reads
    // one contiguous row segment, 16 chunks ahead (independent loads), and leaves the
    // exclusive prefix (the chunk's base within the expert) in their place.
    constexpr int kAhead = 16;
    const int ex = threadIdx.x;
    int carry = 0;
    if (ex < E) {
      for (int c0 = 0; c0 < n_chunks; c0 += kAhead) {
        int v[kAhead];
#pragma unroll
        for (int i = 0; i < kAhead; ++i)
          v[i] = c0 + i < n_chunks ? chunk_counts[(size_t)(c0 + i) * E + ex] : 0;
#pragma unroll
        for (int i = 0; i < kAhead; ++i) {
          if (c0 + i < n_chunks) chunk_counts[(size_t)(c0 + i) * E + ex] = carry;
          carry += v[i];
        }
      }
      s_expert_total[ex] = carry;
    }
  }
  __syncthreads();
  const int e = threadIdx.x;
  const int total = e < E ? s_expert_total[e] : 0;
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
  if (tiles) {
    __syncthreads();
    write_tile_list(E, excl, padded, tile_rows, tiles, n_tiles, warp_tot);
  }
  if (tiles2) {
    __syncthreads();
    write_tile_list(E, excl, padded, tile_rows2, tiles2, n_tiles2, warp_tot);
  }
}

__global__ void __launch_bounds__(kChunk)
    sort_scatter_kernel(const int32_t* __restrict__ ids, int P, int E,
                        const int32_t* __restrict__ chunk_base,
                        const int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_ids,
                        int32_t* __restrict__ inv_route) {
  __shared__ int s_ids[kChunk];
  pdl_wait();
  pdl_trigger();
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

// Tiles of at most tile_rows rows over each expert segment [offsets[e], offsets[e+1]).
__global__ void __launch_bounds__(1024)
    build_tiles_kernel(int E, const int32_t* __restrict__ offsets, Tile* __restrict__ tiles,
                       int* __restrict__ n_tiles, int tile_rows) {
  __shared__ int warp_tot[32];
  pdl_wait();
  pdl_trigger();
  const int e = threadIdx.x;
  const int seg = e < E ? offsets[e + 1] - offsets[e] : 0;
  const int nt = (seg + tile_rows - 1) / tile_rows;
  const int incl = block_inclusive_scan(nt, warp_tot);
  const int base = incl - nt;
  if (e < E) {
    const int r0 = offsets[e];
    for (int i = 0; i < nt; ++i) {
      Tile t;
      t.e = e;
      t.row0 = r0 + i * tile_rows;
      t.nrows = min(tile_rows, seg - i * tile_rows);
      t.first = base;
      t.count = nt;
      t.pad0 = t.pad1 = t.pad2 = 0;
      tiles[base + i] = t;
    }
  }
  if (e == E - 1) *n_tiles = incl;
}

// Tiles of at most tile_rows rows over the groups of a grouped-GEMM layout (TileOPs "MoE" page,
// op MoEGroupedGemmFwd): masked (max_m > 0) group e owns rows e*max_m .. + clamp(meta[e], 0,
// max_m); contiguous (max_m == 0) meta holds the inclusive prefix sums of the groups' rows.  A
// decreasing prefix sum or one past `rows` sets MOE_ERR_INVALID_ARG and drops the group.
__global__ void __launch_bounds__(1024)
    build_tiles_meta_kernel(int E, int max_m, int64_t rows, const int32_t* __restrict__ meta,
                            Tile* __restrict__ tiles, int* __restrict__ n_tiles, int tile_rows,
                            int* __restrict__ status) {
  __shared__ int warp_tot[32];
  pdl_wait();
  pdl_trigger();
  const int e = threadIdx.x;
  int r0 = 0, seg = 0;
  if (e < E) {
    if (max_m > 0) {
      r0 = e * max_m;
      seg = min(max(meta[e], 0), max_m);
    } else {
      r0 = e == 0 ? 0 : meta[e - 1];
      seg = meta[e] - r0;
      if (r0 < 0 || seg < 0 || (int64_t)meta[e] > rows) {
        set_status(status, MOE_ERR_INVALID_ARG);
        seg = 0;
      }
    }
  }
  const int nt = (seg + tile_rows - 1) / tile_rows;
  const int incl = block_inclusive_scan(nt, warp_tot);
  const int base = incl - nt;
  for (int i = 0; i < nt; ++i) {
    Tile t;
    t.e = e;
    t.row0 = r0 + i * tile_rows;
    t.nrows = min(tile_rows, seg - i * tile_rows);
    t.first = base;
    t.count = nt;
    t.pad0 = t.pad1 = t.pad2 = 0;
    tiles[base + i] = t;
  }
  if (e == E - 1) *n_tiles = incl;
}

// Mask of the lanes whose v equals this lane's (0 <= v < 2^nbits), from one ballot per bit: the
// mask __match_any_sync returns, at a fraction of its cost when most values differ.
__device__ __forceinline__ unsigned match_by_ballots(int v, int nbits) {
  unsigned m = 0xffffffffu;
  for (int b = 0; b < nbits; ++b) {
    const int bit = (v >> b) & 1;
    const unsigned bb = __ballot_sync(0xffffffffu, bit);
    m &= bit ? bb : ~bb;
  }
  return m;
}

// The whole sort in one CTA of 1024 threads (32 warps), for up to kFusedSortMaxRoutes routes
// (beyond that the chunked kernels, which spread the ranking over many CTAs, are faster):
// warp w owns the contiguous routes [w*per, (w+1)*per), per <= 256, which it reads once into
// registers.  Pass A counts each warp's routes per expert (shared-memory atomics into the
// warp's own counters); a per-expert prefix over the warps, after the block scan of the padded
// totals, turns the counts into each warp's first position in every expert segment; pass B
// walks the same routes in the same order and places each one at that base plus its rank among
// the equal ids before it (lanes with the same id found by ballots on the id's bits).  The
// result is the same stable order as the chunked kernels, from a single launch.  With `tiles`
// it also writes the GEMM tile list over the segments.
constexpr int kFusedSortMaxRoutes = 8192;

__global__ void __launch_bounds__(1024)
    sort_fused_kernel(const int32_t* __restrict__ ids, int P, int E, int block_m, int64_t cap,
                      int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                      int32_t* __restrict__ sorted_ids, int32_t* __restrict__ tile_expert,
                      int64_t tile_len, int32_t* __restrict__ inv_route, Tile* __restrict__ tiles,
                      int* __restrict__ n_tiles, int tile_rows, Tile* __restrict__ tiles2,
                      int* __restrict__ n_tiles2, int tile_rows2, int* status,
                      int* __restrict__ zero, int n_zero) {
  extern __shared__ int warp_cnt[];  // [32][E]
  __shared__ int warp_tot[32];
  __shared__ int s_total;
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  for (int i = tid; i < n_zero; i += blockDim.x) zero[i] = 0;
  for (int i = tid; i < 32 * E; i += blockDim.x) warp_cnt[i] = 0;
  __syncthreads();
  int* wc = warp_cnt + w * E;
  const int per = (P + 31) / 32;
  const int r0 = w * per, r1 = min(P, r0 + per);
  const unsigned lt_mask = (1u << lane) - 1u;
  // A warp's routes are read once, 8 groups of 32 (independent loads, one latency), and kept in
  // registers for both passes: per <= 32 * kBatch because P <= kFusedSortMaxRoutes.
  constexpr int kBatch = 8;
  static_assert(32 * 32 * kBatch >= kFusedSortMaxRoutes, "one batch per warp");
  int eb[kBatch];
#pragma unroll
  for (int g = 0; g < kBatch; ++g) {
    const int r = r0 + 32 * g + lane;
    int e = r < r1 ? ids[r] : -1;
    if (e < -1 || e >= E) {
      set_status(status, MOE_ERR_BAD_EXPERT_ID);
      e = -1;
    }
    eb[g] = e;
  }
#pragma unroll
  for (int g = 0; g < kBatch; ++g)  // pass A: per-warp histogram
    if (eb[g] >= 0) atomicAdd(&wc[eb[g]], 1);
  __syncthreads();
  int total = 0;
  if (tid < E)
    for (int ww = 0; ww < 32; ++ww) total += warp_cnt[ww * E + tid];
  const int padded = tid < E ? (total + block_m - 1) / block_m * block_m : 0;
  const int incl = block_inclusive_scan(padded, warp_tot);
  const int excl = incl - padded;
  if (tid < E) {
    counts[tid] = total;
    offsets[tid] = excl;
    int base = excl;
    for (int ww = 0; ww < 32; ++ww) {
      const int c = warp_cnt[ww * E + tid];
      warp_cnt[ww * E + tid] = base;
      base += c;
    }
  }
  if (tid == E - 1) {
    offsets[E] = incl;
    s_total = incl;
  }
  __syncthreads();
  {  // pass B: stable scatter
    const int nbits = 32 - __clz(E);  // e + 1 lies in [0, E]
#pragma unroll
    for (int g = 0; g < kBatch; ++g) {
      if (r0 + 32 * g >= r1) break;  // warp-uniform
      const int r = r0 + 32 * g + lane;
      const int e = eb[g];
      const unsigned m = match_by_ballots(e + 1, nbits);
      const int base = e >= 0 ? wc[e] : 0;
      __syncwarp();
      if (r < r1) {
        if (e >= 0) {
          const int pos = base + __popc(m & lt_mask);
          sorted_ids[pos] = r;
          inv_route[r] = pos;
        } else {
          inv_route[r] = -1;
        }
      }
      if (e >= 0 && lane == __ffs(m) - 1) wc[e] = base + __popc(m);
      __syncwarp();
    }
  }
  const int tot = s_total;
  if (tid < E)
    for (int q = excl + total; q < excl + padded; ++q) sorted_ids[q] = -1;
  for (int64_t q = tot + tid; q < cap; q += blockDim.x) sorted_ids[q] = -1;
  if (tile_expert) {
    if (tid < E)
      for (int i = excl / block_m; i < (excl + padded) / block_m; ++i) tile_expert[i] = tid;
    for (int64_t i = tot / block_m + tid; i < tile_len; i += blockDim.x) tile_expert[i] = -1;
  }
  if (tiles) {
    __syncthreads();  // warp_tot is reused by every scan
    write_tile_list(E, excl, padded, tile_rows, tiles, n_tiles, warp_tot);
  }
  if (tiles2) {
    __syncthreads();
    write_tile_list(E, excl, padded, tile_rows2, tiles2, n_tiles2, warp_tot);
  }
}

// a_sorted[p, :] = hidden[sorted_ids[p] / top_k, :] for p < offsets[E]; padding rows are zero.
// A CTA copies whole rows (grid-stride): each thread loads up to 8 of its 16-byte pieces of the
// row before it stores any, and the next row's source index is fetched during the copy.
// kToF16: bf16 rows in, f16 rows out (the NVFP4 path), a value past the f16 range flagged.
constexpr int kPermuteThreads = 128;
constexpr int kPermuteAhead = 8;

template <bool kToF16>
__global__ void __launch_bounds__(kPermuteThreads)
    permute_kernel(int top_k, int H, const uint16_t* __restrict__ hidden,
                   const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ offsets,
                   int E, uint16_t* __restrict__ a_sorted, int* __restrict__ status) {
  pdl_wait();
  pdl_trigger();
  bool over = false;
  const int64_t rows = offsets[E];
  const int nvec = H / 8;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  int64_t row = blockIdx.x;
  int sid = row < rows ? sorted_ids[row] : -1;
  for (; row < rows; row += gridDim.x) {
    const int64_t next = row + gridDim.x;
    const int next_sid = next < rows ? sorted_ids[next] : -1;
    uint4* dst = reinterpret_cast<uint4*>(a_sorted + row * H);
    const uint4* src =
        reinterpret_cast<const uint4*>(hidden + (int64_t)(sid < 0 ? 0 : sid / top_k) * H);
    for (int v0 = 0; v0 < nvec; v0 += kPermuteThreads * kPermuteAhead) {
      uint4 buf[kPermuteAhead];
#pragma unroll
      for (int i = 0; i < kPermuteAhead; ++i) {
        const int v = v0 + i * kPermuteThreads + threadIdx.x;
        buf[i] = (sid >= 0 && v < nvec) ? __ldg(src + v) : zero;
      }
#pragma unroll
      for (int i = 0; i < kPermuteAhead; ++i) {
        const int v = v0 + i * kPermuteThreads + threadIdx.x;
        if (v < nvec) dst[v] = kToF16 ? bf16x8_to_f16x8(buf[i], over) : buf[i];
      }
    }
    sid = next_sid;
  }
  if (kToF16 && over) set_status(status, MOE_ERR_F16_RANGE);
}

// out[t, :] = round(sum_j y[inv[t*K+j], :] + shared[t, :]): f32 rows in, one rounding out.
// A CTA owns one token and `cpc` chunks of 512 columns (4 per thread); the token's route rows
// are looked up once into shared memory, and each thread then streams its columns of those rows
// with up to 16 loads of 16 bytes in flight (two chunks of 8 routes).  The routes are summed in
// j order, so the sum is the same on every run and for every cpc.
constexpr int kCombineThreads = 128;

// 16-byte read-only load when `pred`, else zeros: a predicated load, so that a group of them
// can all be in flight before the first add.
__device__ __forceinline__ float4 ld_f4_if(const float* ptr, bool pred) {
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  asm("{\n\t.reg .pred q;\n\t"
      "setp.ne.b32 q, %5, 0;\n\t"
      "@q ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];\n\t}\n"
      : "+f"(v.x), "+f"(v.y), "+f"(v.z), "+f"(v.w)
      : "l"(ptr), "r"((int)pred));
  return v;
}

template <typename T>
__device__ __forceinline__ void combine_store(T* out, float4 a) {
  T o[4] = {DT<T>::from_f(a.x), DT<T>::from_f(a.y), DT<T>::from_f(a.z), DT<T>::from_f(a.w)};
  *reinterpret_cast<uint2*>(out) = *reinterpret_cast<const uint2*>(o);
}

__device__ __forceinline__ void add4(float4& a, const float4 b) {
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
}

template <typename T>
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(int K, int H, int cpc, const float* __restrict__ y,
                   const int32_t* __restrict__ inv, const int32_t* __restrict__ ids,
                   const float* __restrict__ shared, T* __restrict__ out) {
  __shared__ int s_row[32];  // y row of each route of the token, -1 to skip
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.y;
  if (threadIdx.x < K) {
    const int r = t * K + threadIdx.x;
    s_row[threadIdx.x] = (ids && ids[r] < 0) ? -1 : (inv ? inv[r] : r);
  }
  __syncthreads();
  const int nv = H / 4;  // float4 columns of a row
  const int v_end = min(nv, (blockIdx.x + 1) * cpc * kCombineThreads);
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  int v = blockIdx.x * cpc * kCombineThreads + threadIdx.x;
  // two chunks at a time: 16 independent loads before the first add
  for (; v + kCombineThreads < v_end; v += 2 * kCombineThreads) {
    float4 acc0 = zero, acc1 = zero;
    for (int j0 = 0; j0 < K; j0 += 8) {
      float4 r0[8], r1[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int p = j0 + jj < K ? s_row[j0 + jj] : -1;
        const float* src = y + (int64_t)(p < 0 ? 0 : p) * H + 4 * v;
        r0[jj] = ld_f4_if(src, p >= 0);
        r1[jj] = ld_f4_if(src + 4 * kCombineThreads, p >= 0);
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        add4(acc0, r0[jj]);
        add4(acc1, r1[jj]);
      }
    }
    if (shared) {
      add4(acc0, reinterpret_cast<const float4*>(shared + (int64_t)t * H)[v]);
      add4(acc1, reinterpret_cast<const float4*>(shared + (int64_t)t * H)[v + kCombineThreads]);
    }
    combine_store(out + (int64_t)t * H + 4 * v, acc0);
    combine_store(out + (int64_t)t * H + 4 * (v + kCombineThreads), acc1);
  }
  if (v < v_end) {  // the last, odd chunk (or its ragged end)
    float4 acc = zero;
    for (int j0 = 0; j0 < K; j0 += 8) {
      float4 r0[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int p = j0 + jj < K ? s_row[j0 + jj] : -1;
        r0[jj] = ld_f4_if(y + (int64_t)(p < 0 ? 0 : p) * H + 4 * v, p >= 0);
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) add4(acc, r0[jj]);
    }
    if (shared) add4(acc, reinterpret_cast<const float4*>(shared + (int64_t)t * H)[v]);
    combine_store(out + (int64_t)t * H + 4 * v, acc);
  }
}

// The same sum on an expert-parallel shard, where a token has about one route to this GPU's
// experts (the others are -1 in ids).  With the loop above, one route keeps only two loads in
// flight per thread.  Here warp 0 first lists the routes that have a row (in j order), and a
// thread then loads 8 column chunks of one route at a time (of two to eight routes, two chunks
// of eight routes), so the sum is still taken in j order.
template <int G, int J, typename T>
__device__ __forceinline__ void combine_cols(int na, const int* rows, const float* y, int H,
                                             int v0, int v_end, const float* shared_row,
                                             T* out_row) {
  for (int v = v0; v < v_end; v += G * kCombineThreads) {
    float4 acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) acc[g] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 < na; j0 += J) {
      float4 r[J][G];
#pragma unroll
      for (int jj = 0; jj < J; ++jj) {
        const int p = j0 + jj < na ? rows[j0 + jj] : -1;
        const float* src = y + (int64_t)(p < 0 ? 0 : p) * H;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const int c = v + g * kCombineThreads;
          r[jj][g] = ld_f4_if(src + 4 * c, p >= 0 && c < v_end);
        }
      }
#pragma unroll
      for (int jj = 0; jj < J; ++jj) {
#pragma unroll
        for (int g = 0; g < G; ++g) add4(acc[g], r[jj][g]);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int c = v + g * kCombineThreads;
      if (c < v_end) {
        if (shared_row) add4(acc[g], reinterpret_cast<const float4*>(shared_row)[c]);
        combine_store(out_row + 4 * c, acc[g]);
      }
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kCombineThreads, 6)
    combine_sparse_kernel(int K, int H, int cpc, const float* __restrict__ y,
                          const int32_t* __restrict__ inv, const int32_t* __restrict__ ids,
                          const float* __restrict__ shared, T* __restrict__ out) {
  __shared__ int s_row[32];  // y rows of the token's routes that have one, in j order
  __shared__ int s_na;
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.y;
  if (threadIdx.x < 32) {
    const int j = threadIdx.x;
    int row = -1;
    if (j < K) {
      const int r = t * K + j;
      row = (ids && ids[r] < 0) ? -1 : (inv ? inv[r] : r);
    }
    const unsigned has = __ballot_sync(0xffffffffu, row >= 0);
    if (row >= 0) s_row[__popc(has & ((1u << j) - 1u))] = row;
    if (j == 0) s_na = __popc(has);
  }
  __syncthreads();
  const int na = s_na;
  const int v_end = min(H / 4, (blockIdx.x + 1) * cpc * kCombineThreads);
  const int v0 = blockIdx.x * cpc * kCombineThreads + threadIdx.x;
  const float* sh = shared ? shared + (int64_t)t * H : nullptr;
  T* o = out + (int64_t)t * H;
  if (na <= 1)
    combine_cols<8, 1>(na, s_row, y, H, v0, v_end, sh, o);
  else
    combine_cols<2, 8>(na, s_row, y, H, v0, v_end, sh, o);
}

// out[t, :] = round( sum_j w[t, j] * rows[inv[t*K + j], :] ), f32 in fixed j order (TileOPs
// "MoE" page, op MoEPostPermuteFwd), 8 columns per thread; routes with inv = -1 are skipped.
template <typename T>
__global__ void __launch_bounds__(128)
    post_permute_kernel(int K, int H, const T* __restrict__ rows, const float* __restrict__ w,
                        const int32_t* __restrict__ inv, T* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.y;
  const int v = blockIdx.x * blockDim.x + threadIdx.x;  // 8 columns per thread
  if (v >= H / 8) return;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < K; ++j) {
    const int r = t * K + j;
    const int p = inv[r];
    if (p < 0) continue;
    const float wj = w[r];
    const uint4 raw = reinterpret_cast<const uint4*>(rows + (int64_t)p * H)[v];
    const T* x = reinterpret_cast<const T*>(&raw);
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = fmaf(wj, DT<T>::to_f(x[c]), acc[c]);
  }
  T o[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) o[c] = DT<T>::from_f(acc[c]);
  reinterpret_cast<uint4*>(out + (int64_t)t * H)[v] = *reinterpret_cast<const uint4*>(o);
}

}  // namespace

cudaError_t launch_build_tiles_meta(int E, int max_m, int64_t rows, const int32_t* meta,
                                    Tile* tiles, int* n_tiles, int tile_rows, int* status,
                                    cudaStream_t s, bool pdl) {
  return launch_k(build_tiles_meta_kernel, dim3(1), dim3(1024), 0, s, pdl, E, max_m, rows, meta,
                  tiles, n_tiles, tile_rows, status);
}

cudaError_t launch_post_permute(int dtype, int T, int K, int H, const void* rows,
                                const float* w, const int32_t* inv, void* out, cudaStream_t s,
                                bool pdl) {
  if (T == 0) return cudaSuccess;
  const dim3 grid((H / 8 + 127) / 128, T);
  if (dtype == MOE_BF16)
    return launch_k(post_permute_kernel<__nv_bfloat16>, grid, dim3(128), 0, s, pdl, K, H,
                    static_cast<const __nv_bfloat16*>(rows), w, inv,
                    static_cast<__nv_bfloat16*>(out));
  return launch_k(post_permute_kernel<__half>, grid, dim3(128), 0, s, pdl, K, H,
                  static_cast<const __half*>(rows), w, inv, static_cast<__half*>(out));
}

bool fused_sort_fits(const moe_problem_t& p) {
  return (int64_t)p.T * p.top_k <= kFusedSortMaxRoutes && p.E <= 1024;
}

cudaError_t launch_sort_fused(const moe_problem_t& p, int block_m, const int32_t* ids,
                              int32_t* counts, int32_t* offsets, int32_t* sorted_ids,
                              int64_t cap, int32_t* tile_expert, int32_t* inv_route, Tile* tiles,
                              int* n_tiles, int tile_rows, Tile* tiles2, int* n_tiles2,
                              int tile_rows2, int* status, cudaStream_t s, bool pdl, int* zero,
                              int n_zero) {
  const int P = p.T * p.top_k;
  const size_t smem = sizeof(int) * 32 * (size_t)p.E;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(sort_fused_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(sizeof(int) * 32 * 1024));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t tile_len = (cap + block_m - 1) / block_m;
  return launch_k(sort_fused_kernel, dim3(1), dim3(1024), smem, s, pdl, ids, P, p.E, block_m,
                  cap, counts, offsets, sorted_ids, tile_expert, tile_len, inv_route, tiles,
                  n_tiles, tile_rows, tiles2, n_tiles2, tile_rows2, status, zero,
                  zero ? n_zero : 0);
}

cudaError_t launch_align_sort_chunked(const moe_problem_t& p, int block_m, const int32_t* ids,
                                      int32_t* counts, int32_t* offsets, int32_t* sorted_ids,
                                      int64_t cap, int32_t* tile_expert, int32_t* inv_route,
                                      int32_t* chunk_scratch, int* status, cudaStream_t s,
                                      bool pdl, Tile* tiles, int* n_tiles, int tile_rows,
                                      Tile* tiles2, int* n_tiles2, int tile_rows2) {
  const int P = p.T * p.top_k;
  const int n_chunks = (P + kChunk - 1) / kChunk;
  const int64_t tile_len = (cap + block_m - 1) / block_m;
  if (n_chunks > 0) {
    cudaError_t err = launch_k(sort_count_kernel, dim3(n_chunks), dim3(kChunk),
                               sizeof(int) * p.E, s, pdl, ids, P, p.E, chunk_scratch, status);
    if (err != cudaSuccess) return err;
    pdl = true;
  }
  cudaError_t err = launch_k(sort_scan_kernel, dim3(1), dim3(1024), 0, s, pdl, n_chunks, p.E,
                             block_m, cap, chunk_scratch, counts, offsets, sorted_ids,
                             tile_expert, tile_len, tiles, n_tiles, tile_rows, tiles2, n_tiles2,
                             tile_rows2);
  if (err != cudaSuccess || n_chunks == 0) return err;
  return launch_k(sort_scatter_kernel, dim3(n_chunks), dim3(kChunk), 0, s, true, ids, P, p.E,
                  static_cast<const int32_t*>(chunk_scratch),
                  static_cast<const int32_t*>(offsets), sorted_ids, inv_route);
}

cudaError_t launch_align_sort(const moe_problem_t& p, int block_m, const int32_t* ids,
                              int32_t* counts, int32_t* offsets, int32_t* sorted_ids,
                              int64_t cap, int32_t* tile_expert, int32_t* inv_route,
                              int32_t* chunk_scratch, int* status, cudaStream_t s, bool pdl) {
  if (fused_sort_fits(p))
    return launch_sort_fused(p, block_m, ids, counts, offsets, sorted_ids, cap, tile_expert,
                             inv_route, nullptr, nullptr, kTileRows, nullptr, nullptr, kTileRows,
                             status, s, pdl);
  return launch_align_sort_chunked(p, block_m, ids, counts, offsets, sorted_ids, cap,
                                   tile_expert, inv_route, chunk_scratch, status, s, pdl,
                                   nullptr, nullptr, kTileRows, nullptr, nullptr, kTileRows);
}

cudaError_t launch_build_tiles(int E, const int32_t* offsets, Tile* tiles, int* n_tiles,
                               int tile_rows, cudaStream_t s, bool pdl) {
  return launch_k(build_tiles_kernel, dim3(1), dim3(1024), 0, s, pdl, E, offsets, tiles,
                  n_tiles, tile_rows);
}

cudaError_t launch_permute(int dtype, int top_k, int H, const void* hidden,
                           const int32_t* sorted_ids, const int32_t* offsets, int E, int64_t cap,
                           void* a_sorted, cudaStream_t s, bool pdl, bool to_f16, int* status) {
  if (cap <= 0) return cudaSuccess;
  if (to_f16 && dtype != MOE_BF16) return cudaErrorInvalidValue;
  // without to_f16 a row copy: the element type does not matter
  const int64_t grid = cap < 4096 ? cap : 4096;
  auto kern = to_f16 ? permute_kernel<true> : permute_kernel<false>;
  return launch_k(kern, dim3((int)grid), dim3(kPermuteThreads), 0, s, pdl, top_k, H,
                  static_cast<const uint16_t*>(hidden), sorted_ids, offsets, E,
                  static_cast<uint16_t*>(a_sorted), status);
}

cudaError_t launch_combine(const moe_problem_t& p, const void* y_route,
                           const int32_t* inv_route, const int32_t* ids, const void* shared_out,
                           void* out, cudaStream_t s, bool pdl) {
  // An expert-parallel shard whose tokens average at most two routes to its experts.
  const bool sparse = p.ep_num_local > 0 && (int64_t)p.top_k * p.ep_num_local <= 2ll * p.E;
  if (p.T == 0) return cudaSuccess;
  // Chunks of 512 columns per CTA: as many as keep about 16 CTAs of 128 threads per SM busy in
  // one round (a whole row per CTA at prefill sizes, one chunk per CTA at decode sizes).
  const int nch = (p.H / 4 + kCombineThreads - 1) / kCombineThreads;
  const int64_t want = 16ll * num_sms();
  int cpc = (int)((int64_t)nch * p.T / want);
  cpc = cpc < 1 ? 1 : (cpc > nch ? nch : cpc);
  dim3 grid((nch + cpc - 1) / cpc, p.T);
  const float* y = static_cast<const float*>(y_route);
  const float* sh = static_cast<const float*>(shared_out);
  // The sparse kernel's 8-chunk steps add loads in flight only where a CTA has 8 chunks (large
  // T); below, it only lowers the occupancy (measured 0.2-0.4 % slower at 512 tokens).
  if (sparse && ids && cpc >= 8) {
    if (p.dtype == MOE_BF16)
      return launch_k(combine_sparse_kernel<__nv_bfloat16>, grid, dim3(kCombineThreads), 0, s,
                      pdl, p.top_k, p.H, cpc, y, inv_route, ids, sh,
                      static_cast<__nv_bfloat16*>(out));
    return launch_k(combine_sparse_kernel<__half>, grid, dim3(kCombineThreads), 0, s, pdl,
                    p.top_k, p.H, cpc, y, inv_route, ids, sh, static_cast<__half*>(out));
  }
  if (p.dtype == MOE_BF16)
    return launch_k(combine_kernel<__nv_bfloat16>, grid, dim3(kCombineThreads), 0, s, pdl,
                    p.top_k, p.H, cpc, y, inv_route, ids, sh, static_cast<__nv_bfloat16*>(out));
  return launch_k(combine_kernel<__half>, grid, dim3(kCombineThreads), 0, s, pdl, p.top_k, p.H,
                  cpc, y, inv_route, ids, sh, static_cast<__half*>(out));
}

}  // namespace gb300moe
