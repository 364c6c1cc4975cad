// gemm_pair.cu -- the grouped down projection at prefill sizes on pairs of SMs (tcgen05
// cta_group::2).
//
// TileOPs "MoE" page, op MoEGroupedGemmFwd (contiguous layout) -- the arithmetic of gemm.cu's
// down projection (y_route[p,:] = topk_w[route(p)] * act[p,:] . W_down[e]^T, f32 rows), organised
// for experts with hundreds of routed rows (DeepSeek-V3-shaped prefill: 32768 routes over 256
// experts, up to ~1250 rows per expert).  There the single-SM kernel, with 256-row token tiles,
// stages 48 KB per 64-k block per SM (16 KB of weights, 32 KB of token rows) and keeps a single
// accumulator when both buffers would not fit.  A pair of SMs (a cluster of two CTAs) issues one
// M = 256 MMA over a 256-row token tile instead: each CTA stages only its own 128 rows of w_down
// and its own half (128 rows) of the token tile, 32 KB per 64-k block, and keeps two 256-column
// accumulator buffers so that a unit's epilogue overlaps the next unit's MMAs.  The epilogue
// multiplies by the route weight and stores f32 rows (rounded once, later, by the combine).
// A pipeline stage holds two 64-k blocks of both (64 KB per CTA, three stages).
// Roles per CTA (192 threads, one CTA per SM, persistent over the pair's units):
//   warp 0  TMA producer of this CTA's weight rows and token half (its own barriers);
//   warp 1  even CTA: MMA issuer (tcgen05.mma.cta_group::2, M = 256, N = 32..256);
//           odd CTA: forwarder, which tells the even CTA's full barrier that a stage of the
//           odd CTA's shared memory has landed (one remote arrive per stage);
//   warps 2-5  epilogue (tcgen05.ld of this CTA's 128 accumulator rows).
// The MMA's completion is committed to the barriers of both CTAs (stage free, accumulator
// ready); the epilogue warps of both CTAs arrive on the even CTA's accumulator-free barrier.
// No copy is multicast: every CTA loads its own tiles.  Every wait is bounded; on expiry the CTA
// records MOE_ERR_TIMEOUT, raises its own and the peer's abort flag, waits (bounded) for its
// own copies and MMAs in flight, and both CTAs meet at a final cluster barrier before TMEM is
// freed.
//
// The same pairing for the gate/up projection (64 gate and 64 up rows per CTA, the two
// accumulator halves swapped between epilogue warps) measured slower than the single-SM kernel
// at DeepSeek-V3 prefill (2.48 against 2.23 ms): at that routing most experts have fewer than
// 128 rows, so most units only stream weights, and the single-SM kernel keeps more weight bytes
// in flight per SM (128 KB against 96 KB).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace gb300moe {

namespace {

constexpr int kPN = kTileRowsWide;              // token rows of a pair tile (the MMA's N)
constexpr int kPHalf = kPN / 2;                 // token rows each CTA stages
// A stage carries two 64-k blocks: the MMA issuer's per-stage wait and commits and the
// producer's and forwarder's per-stage barrier operations are paid once per 8 MMAs.  With one
// block per stage (4 MMAs) the issuer spent 0.31 us of each 0.40 us stage issuing at
// DeepSeek-V3 prefill, with the tensor pipe half idle.
constexpr int kPKps = 2;
constexpr int kPStages = 3;
constexpr int kPABytes = kSlab * kBlockK * 2;   // 16 KB: the CTA's 128 weight rows of 64 k
constexpr int kPBBytes = kPHalf * kBlockK * 2;  // 16 KB: the CTA's token rows of 64 k
constexpr int kPStageBytes = kPKps * (kPABytes + kPBBytes);
constexpr int kPAccCols = kPN;                  // f32 accumulator columns per buffer
constexpr int kPAccBufs = 2;
constexpr int kPTmemCols = kPAccBufs * kPAccCols;
constexpr int kPThreads = 192;
constexpr int kPSmemBytes = kPStages * kPStageBytes + 1024;
static_assert(kPSmemBytes <= 227 * 1024, "shared memory");
static_assert(kPTmemCols == 512, "two accumulator buffers of 256 columns");

struct PParams {
  int n_out, n_slabs, num_kb;
  int w_rows_per_expert;
  const Tile* tiles;
  const int* n_tiles;
  const int32_t* sorted_ids;  // the route of each sorted row (null: weight 1)
  const float* topk_w;
  float* out;
  int* status;
  uint64_t limit_ns;
  int prefetch_steps;  // K steps of first-unit weights pulled into L2 before the dependency wait
};

struct PUnit {
  int e, row0, nrows, n, slab;
};

// Unit u of the pair schedule: the units of expert e are [n_slabs*first, n_slabs*(first+count))
// of its tiles, slab-major (the tiles of one weight slab are adjacent, so the pairs that run them
// at the same time share the slab through L2).
__device__ __forceinline__ bool pair_unit(const PParams& p, int u, PUnit& U) {
  const Tile owner = p.tiles[u / p.n_slabs];
  const int local = u - p.n_slabs * owner.first;
  U.slab = local / owner.count;
  const Tile t = p.tiles[owner.first + local % owner.count];
  U.e = t.e;
  U.row0 = t.row0;
  U.nrows = t.nrows;
  U.n = (t.nrows + 31) & ~31;  // MMA N: each CTA's half a multiple of 16 rows
  return t.nrows > 0;
}

// First row of w_down this CTA loads for unit U (the pair's slab is 256 rows).
__device__ __forceinline__ int pair_wrow(const PParams& p, const PUnit& U, uint32_t rank) {
  return U.e * p.w_rows_per_expert + U.slab * 2 * kSlab + kSlab * (int)rank;
}

constexpr uint64_t kPDrainNs = 1000000000ull;  // total budget of a CTA's drain waits

template <typename T>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPThreads, 1)
    moe_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmW,
                         const __grid_constant__ CUtensorMap tmB16,
                         const __grid_constant__ CUtensorMap tmB64,
                         const __grid_constant__ CUtensorMap tmB128, const PParams p) {
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[kPStages];
  __shared__ __align__(8) uint64_t empty_bar[kPStages];
  __shared__ __align__(8) uint64_t tfull_bar[kPAccBufs];
  __shared__ __align__(8) uint64_t tempty_bar[kPAccBufs];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  __shared__ int s_n_units;
  __shared__ int ent_dst[kPN];
  __shared__ float col_scale[kPN];

  // Both CTAs run the same kernel with the same static shared memory, so the 1024-byte aligned
  // ring sits at the same offset in both: the MMA reads the peer's tiles at these addresses.
  const uint32_t raw = smem_u32(dsmem);
  uint8_t* smem = dsmem + ((1024u - (raw & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  volatile int* abort_flag = &s_abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      // the even CTA's stage is full when its own copies have landed and the odd CTA has
      // forwarded that its copies have landed
      mbar_init(&full_bar[s], leader ? 2 : 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < kPAccBufs; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 8);  // one arrival per epilogue warp of both CTAs
    }
    mbar_init(&drain_bar, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmW);
    prefetch_tensormap(&tmB16);
    prefetch_tensormap(&tmB64);
    prefetch_tensormap(&tmB128);
  }
  if (warp == 1) {
    tmem_alloc_pair(&s_tmem_base, kPTmemCols);
    tmem_relinquish_pair();
  }
  const uint32_t cid = cluster_id_x();
  const uint32_t ncl = num_clusters_x();
  // The tile list was written at least two launches earlier (it is complete): pull this CTA's
  // first units' weights into L2 while the previous kernel finishes on other SMs.
  if (p.prefetch_steps > 0 && threadIdx.x == 0) {
    const int n = (*p.n_tiles) * p.n_slabs;
    int left = p.prefetch_steps;
    for (int u = (int)cid; u < n && left > 0; u += (int)ncl) {
      PUnit U;
      if (!pair_unit(p, u, U)) continue;
      const int wrow = pair_wrow(p, U, rank);
      for (int kb = 0; kb < p.num_kb && left > 0; ++kb, --left)
        tma_prefetch_l2_2d(&tmW, kb * kBlockK, wrow);
    }
  }
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) s_n_units = (*p.n_tiles) * p.n_slabs;
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, TMEM of both allocated
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  const int n_units = s_n_units;
  const uint32_t peer_abort = cluster_map(smem_u32(&s_abort), rank ^ 1u);

  // Bounded wait on one of this CTA's barriers; on expiry the peer CTA is told to stop too.
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_wait(bar, parity, abort_flag, p.limit_ns, p.status)) return true;
    st_cluster_u32(peer_abort, 1u);
    return false;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int u = (int)cid; u < n_units && ok; u += (int)ncl) {
        PUnit U;
        if (!pair_unit(p, u, U)) continue;
        const int half = U.n >> 1;
        const int b0 = U.row0 + (int)rank * half;
        // This CTA's token rows of the tile (the rest of its half is never read into a kept
        // output column, so it is not loaded).
        int rows = U.nrows - (int)rank * half;
        rows = rows < 0 ? 0 : (rows > half ? half : rows);
        rows = (rows + 15) & ~15;
        const int wrow = pair_wrow(p, U, rank);
        const uint32_t bytes = (uint32_t)(kPABytes + rows * kBlockK * 2);  // per 64-k block
        for (int kb = 0; kb < p.num_kb; kb += kPKps) {
          const int nsub = p.num_kb - kb < kPKps ? p.num_kb - kb : kPKps;
          if (!wait(&empty_bar[stage], phase ^ 1u)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + stage * kPStageBytes;
          mbar_arrive_expect_tx(&full_bar[stage], bytes * nsub);
          for (int j = 0; j < nsub; ++j) {
            uint8_t* sa = st + j * kPABytes;
            uint8_t* sb = st + kPKps * kPABytes + j * kPBBytes;
            const int kx = (kb + j) * kBlockK;
            tma_load_2d(sa, &tmW, &full_bar[stage], kx, wrow);
            int r = 0;
            for (; r + 128 <= rows; r += 128)
              tma_load_2d(sb + r * kBlockK * 2, &tmB128, &full_bar[stage], kx, b0 + r);
            for (; r + 64 <= rows; r += 64)
              tma_load_2d(sb + r * kBlockK * 2, &tmB64, &full_bar[stage], kx, b0 + r);
            for (; r < rows; r += 16)
              tma_load_2d(sb + r * kBlockK * 2, &tmB16, &full_bar[stage], kx, b0 + r);
          }
          ++issued;
          if (++stage == kPStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort_flag) {
        // Let this CTA's copies in flight land before it goes away (the even CTA's full phase
        // also waits for the odd CTA's forward, hence one total budget).
        const uint64_t t0 = global_timer_ns();
        const int n = issued < kPStages ? issued : kPStages;
        for (int i = issued - n; i < issued; ++i)
          while (!mbar_try_wait(&full_bar[i % kPStages], (uint32_t)((i / kPStages) & 1)))
            if (global_timer_ns() - t0 > kPDrainNs) break;
      }
    }
  } else if (warp == 1 && !leader) {
    // ---------------------------------------------------------------- forwarder (odd CTA)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = (int)cid; u < n_units && ok; u += (int)ncl) {
        PUnit U;
        if (!pair_unit(p, u, U)) continue;
        for (int kb = 0; kb < p.num_kb; kb += kPKps) {
          if (!wait(&full_bar[stage], phase)) {
            ok = false;
            break;
          }
          mbar_arrive_cluster(cluster_map(smem_u32(&full_bar[stage]), 0));
          if (++stage == kPStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (even CTA)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool issued_any = false;
      const uint32_t smem_base = smem_u32(smem);
      for (int u = (int)cid; u < n_units && ok; u += (int)ncl) {
        PUnit U;
        if (!pair_unit(p, u, U)) continue;
        if (!wait(&tempty_bar[acc], acc_phase ^ 1u)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * kPAccCols);
        const uint32_t idesc = idesc_f16(256, U.n, DT<T>::kIsBF16);
        for (int kb = 0; kb < p.num_kb; kb += kPKps) {
          const int nsub = p.num_kb - kb < kPKps ? p.num_kb - kb : kPKps;
          if (!wait(&full_bar[stage], phase)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_base + (uint32_t)(stage * kPStageBytes);
#pragma unroll
          for (int j = 0; j < kPKps; ++j) {
            if (j >= nsub) break;
            const uint32_t sa = st + (uint32_t)(j * kPABytes);
            const uint32_t sb = st + (uint32_t)(kPKps * kPABytes + j * kPBBytes);
#pragma unroll
            for (int k = 0; k < kBlockK / 16; ++k)
              umma_f16_pair(d, sw128_kmajor_desc(sa + k * 32), sw128_kmajor_desc(sb + k * 32),
                            idesc, (kb | j | k) != 0 ? 1u : 0u);
          }
          umma_commit_pair(smem_u32(&empty_bar[stage]));
          umma_commit_pair(cluster_map(smem_u32(&empty_bar[stage]), 1));
          issued_any = true;
          if (++stage == kPStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(smem_u32(&tfull_bar[acc]));
        umma_commit_pair(cluster_map(smem_u32(&tfull_bar[acc]), 1));
        if (++acc == kPAccBufs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (issued_any) {  // every MMA issued has completed once drain_bar flips
        umma_commit_pair(smem_u32(&drain_bar));
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&drain_bar, 0))
          if (global_timer_ns() - t0 > kPDrainNs) break;
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (128 threads)
    const int q = warp & 3;  // the TMEM lane quarter this warp reads
    const int row = q * 32 + lane;
    const int et = threadIdx.x - 64;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = (int)cid; u < n_units; u += (int)ncl) {
      PUnit U;
      if (!pair_unit(p, u, U)) continue;
      {
        // Each accumulator column (a sorted row) goes to one f32 output row, scaled by its
        // route's weight (padding rows by 0).
        for (int i = et; i < U.n; i += 128) {
          int dst = -1;
          float sc = 0.0f;
          if (i < U.nrows) {
            dst = U.row0 + i;
            if (p.sorted_ids) {
              const int sid = p.sorted_ids[dst];
              sc = sid >= 0 ? p.topk_w[sid] : 0.0f;
            } else {
              sc = 1.0f;
            }
          }
          ent_dst[i] = dst;
          col_scale[i] = sc;
        }
      }
      const bool got = wait(&tfull_bar[acc], acc_phase);
      if (!named_bar_and(1, 128, got)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kPAccCols);
      {
        float* out = p.out;
        const int h = U.slab * 2 * kSlab + kSlab * (int)rank + row;
        for (int c0 = 0; c0 < U.n; c0 += 16) {
          float g[16];
          tmem_ld_x16(tb + (uint32_t)c0, g);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int dst = ent_dst[c0 + j];
            if (dst >= 0) out[(int64_t)dst * p.n_out + h] = g[j] * col_scale[c0 + j];
          }
        }
      }
      // This warp has read its TMEM lanes of the buffer: tell the even CTA's MMA issuer.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(cluster_map(smem_u32(&tempty_bar[acc]), 0));
      named_bar_sync(1, 128);  // the per-column tables are rewritten for the next unit
      if (++acc == kPAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  cluster_sync();  // neither CTA leaves while the other may still touch its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kPTmemCols);
  }
}

// ---- host side -----------------------------------------------------------------------------

// Clusters of two that can be resident at once for moe_gemm_pair_kernel<T> on the current
// device (0 when none can); also sets the kernel's shared-memory limit.
template <typename T>
int max_pairs() {
  static int cached[64];
  static std::once_flag once[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::call_once(once[dev], [] {
    auto kern = moe_gemm_pair_kernel<T>;
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmemBytes) ==
        cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * 256);
      cfg.blockDim = dim3(kPThreads);
      cfg.dynamicSmemBytes = kPSmemBytes;
      if (cudaOccupancyMaxActiveClusters(&n, (void*)kern, &cfg) != cudaSuccess) n = 0;
    }
    (void)cudaGetLastError();
    int d = 0;
    cudaGetDevice(&d);
    cached[d] = n;
  });
  return cached[dev];
}

template <typename T>
cudaError_t launch_pair_typed(const GemmCall& c, const PParams& pp, int64_t upper,
                              cudaStream_t s, bool pdl) {
  auto kern = moe_gemm_pair_kernel<T>;
  const int pairs = max_pairs<T>();
  if (pairs <= 0) return cudaErrorNotSupported;
  const int n_pairs = (int)(upper < pairs ? upper : pairs);
  CUtensorMap tmW, tmB16, tmB64, tmB128;
  const uint64_t w_rows = (uint64_t)c.E * (uint64_t)pp.w_rows_per_expert;
  if (!make_map16(&tmW, c.dtype, c.w, (uint64_t)c.K, w_rows, kSlab) ||
      !make_map16(&tmB16, c.dtype, c.b, (uint64_t)c.K, (uint64_t)c.b_rows, 16) ||
      !make_map16(&tmB64, c.dtype, c.b, (uint64_t)c.K, (uint64_t)c.b_rows, 64) ||
      !make_map16(&tmB128, c.dtype, c.b, (uint64_t)c.K, (uint64_t)c.b_rows, 128))
    return cudaErrorInvalidValue;
  return launch_k(kern, dim3(2 * n_pairs), dim3(kPThreads), kPSmemBytes, s, pdl, tmW, tmB16,
                  tmB64, tmB128, pp);
}

}  // namespace

bool pair_gemm_available(int dtype) {
  return dtype == MOE_BF16 ? max_pairs<__nv_bfloat16>() > 0 : max_pairs<__half>() > 0;
}

cudaError_t launch_gemm_pair(const GemmCall& c, cudaStream_t s, bool pdl) {
  // The down projection in sorted mode over 256-row tiles, 16-bit weights, H a multiple of 256
  // (a pair unit never crosses an expert).
  if (c.gemm1 || c.mode != kSorted || c.w4 || c.tile_rows != kPN) return cudaErrorInvalidValue;
  if (c.n_out % (2 * kSlab) != 0 || c.K % 8 != 0) return cudaErrorInvalidValue;
  PParams pp;
  pp.n_out = c.n_out;
  pp.n_slabs = c.n_out / (2 * kSlab);
  pp.num_kb = (c.K + kBlockK - 1) / kBlockK;
  pp.w_rows_per_expert = c.n_out;
  pp.tiles = c.tiles;
  pp.n_tiles = c.n_tiles;
  pp.sorted_ids = c.sorted_ids;
  pp.topk_w = c.topk_w;
  pp.out = static_cast<float*>(c.out);
  pp.status = c.status;
  pp.limit_ns = wait_limit_ns();
  pp.prefetch_steps = 0;
  const int64_t upper = (int64_t)c.max_tiles * pp.n_slabs;
  if (upper <= 0 || c.b_rows <= 0) return cudaSuccess;
  if (c.early_tiles) {
    // Up to ~48 MB (well under the L2) of first-unit weights over the whole grid.
    const int64_t ctas = num_sms();
    const int64_t step_bytes = (int64_t)kSlab * kBlockK * 2;  // one CTA's weights of a K step
    const int64_t budget = (48ll << 20) / ctas / step_bytes;
    pp.prefetch_steps = (int)(budget < pp.num_kb * 4 ? budget : pp.num_kb * 4);
  }
  return c.dtype == MOE_BF16 ? launch_pair_typed<__nv_bfloat16>(c, pp, upper, s, pdl)
                             : launch_pair_typed<__half>(c, pp, upper, s, pdl);
}

}  // namespace gb300moe
