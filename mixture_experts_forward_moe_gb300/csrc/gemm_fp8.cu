// gemm_fp8.cu -- FP8 (E4M3) block-scaled grouped GEMM on the sm_103a tensor cores.
//
// TileOPs "MoE" page, op MoEGroupedGemmFP8Fwd: a [rows, K] and b [E, N, K] in E4M3 with f32
// scales per 128-k block of a row of a and per 128 x 128 block of b,
//   out[r, n] = sum_kb a_scale[r, kb] * b_scale[e, n/128, kb] * sum_{k in kb} a[r, k] b[e, n, k],
// in the masked or contiguous grouped layout (the tile list comes from the layout metadata).
//
// Design: weight-stationary like the 16-bit GEMMs.  A unit is (group, 128-row weight slab, token
// tile of up to 128 rows); the 128 weight rows of a slab share one scale per k block, so the
// k-block partial D_kb = W_slab(kb) . A_tile(kb)^T (four tcgen05.mma kind::f8f6f4 of k = 32, A =
// weights, B = tokens, both from 128-byte-swizzled shared memory) only needs one scalar b_scale
// times a per-column (token) a_scale before it is added to the running sum.  Each k block is
// therefore accumulated in a fresh TMEM buffer (4 in flight), and eight epilogue warps fold
// scale * D_kb into f32 registers (warp w reads TMEM lanes 32*(w%4)..; warpgroups split the 128
// token columns in halves), then store the bf16 rows.
//
// Warp roles (320 threads, one CTA per SM, persistent): warp 0 TMA producer, warp 1 MMA issuer,
// warps 2-9 scale-and-accumulate epilogue.  Every wait is bounded as in gemm.cu.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace gb300moe {

namespace {

constexpr int kF8Stages = 6;
constexpr int kF8BlockK = 128;                                // k per stage = one scale block
constexpr int kF8WBytes = kSlab * kF8BlockK;                  // 16 KB of weights
constexpr int kF8TBytes = kTileRows * kF8BlockK;              // up to 16 KB of tokens
constexpr int kF8StageBytes = kF8WBytes + kF8TBytes;
constexpr int kF8PBufs = 4;                                   // TMEM partial buffers
constexpr int kF8Threads = 320;
constexpr int kF8SmemBytes = kF8Stages * kF8StageBytes + 1024;
constexpr uint64_t kF8DrainNs = 1000000000ull;

struct F8Params {
  int N, num_kb, n_slabs;
  const Tile* tiles;
  const int* n_tiles;
  const float* a_scale;  // [rows, num_kb]
  const float* b_scale;  // [E, n_slabs, num_kb]
  __nv_bfloat16* out;    // [rows, N]
  int* status;
  uint64_t limit_ns;
};

struct F8Unit {
  int e, slab, row0, nrows, n_mma;
};

// Units of group e occupy [n_slabs*first, n_slabs*(first+count)), slab-major (as in gemm.cu).
__device__ __forceinline__ bool f8_unit(const F8Params& p, int u, F8Unit& U) {
  const Tile owner = p.tiles[u / p.n_slabs];
  const int local = u - p.n_slabs * owner.first;
  U.slab = local / owner.count;
  const Tile t = p.tiles[owner.first + local % owner.count];
  U.e = t.e;
  U.row0 = t.row0;
  U.nrows = t.nrows;
  U.n_mma = (t.nrows + 15) & ~15;
  return U.nrows > 0;
}

__device__ __forceinline__ void f8_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kF8DrainNs) return;
}

__global__ void __launch_bounds__(kF8Threads, 1)
    moe_gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmB16,
                        const __grid_constant__ CUtensorMap tmB64,
                        const __grid_constant__ CUtensorMap tmB128, const F8Params p) {
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[kF8Stages];
  __shared__ __align__(8) uint64_t empty_bar[kF8Stages];
  __shared__ __align__(8) uint64_t pfull_bar[kF8PBufs];
  __shared__ __align__(8) uint64_t pempty_bar[kF8PBufs];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  __shared__ int s_n_units;
  __shared__ __align__(16) float s_sa[2][kTileRows];  // column scales of one k block

  const uint32_t raw = smem_u32(dsmem);
  uint8_t* smem = dsmem + ((1024u - (raw & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &s_abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kF8Stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < kF8PBufs; ++b) {
      mbar_init(&pfull_bar[b], 1);
      mbar_init(&pempty_bar[b], 8);  // one arrival per epilogue warp
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
    tmem_alloc(&s_tmem_base, kF8PBufs * kTileRows);
    tmem_relinquish();
  }
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) s_n_units = (*p.n_tiles) * p.n_slabs;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  const int n_units = s_n_units;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        F8Unit U;
        if (!f8_unit(p, u, U)) continue;
        const uint32_t bytes = kF8WBytes + U.n_mma * kF8BlockK;
        const int wrow = U.e * p.N + U.slab * kSlab;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, p.limit_ns, p.status)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * kF8StageBytes;
          uint8_t* sb = sa + kF8WBytes;
          mbar_arrive_expect_tx(&full_bar[stage], bytes);
          const int kx = kb * kF8BlockK;
          tma_load_2d(sa, &tmW, &full_bar[stage], kx, wrow);
          int r = 0;
          for (; r + 128 <= U.n_mma; r += 128)
            tma_load_2d(sb + r * kF8BlockK, &tmB128, &full_bar[stage], kx, U.row0 + r);
          for (; r + 64 <= U.n_mma; r += 64)
            tma_load_2d(sb + r * kF8BlockK, &tmB64, &full_bar[stage], kx, U.row0 + r);
          for (; r < U.n_mma; r += 16)
            tma_load_2d(sb + r * kF8BlockK, &tmB16, &full_bar[stage], kx, U.row0 + r);
          ++issued;
          if (++stage == kF8Stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort_flag) {
        const int n = issued < kF8Stages ? issued : kF8Stages;
        for (int i = issued - n; i < issued; ++i)
          f8_wait_drain(&full_bar[i % kF8Stages], (uint32_t)((i / kF8Stages) & 1));
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, pb = 0;
      uint32_t phase = 0, pphase = 0;
      bool ok = true, issued_any = false;
      const uint32_t smem_base = smem_u32(smem);
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        F8Unit U;
        if (!f8_unit(p, u, U)) continue;
        const uint32_t idesc = idesc_e4m3_m128(U.n_mma);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, abort_flag, p.limit_ns, p.status) ||
              !mbar_wait(&pempty_bar[pb], pphase ^ 1u, abort_flag, p.limit_ns, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_base + (uint32_t)(stage * kF8StageBytes);
          const uint32_t sb = sa + kF8WBytes;
          const uint32_t d = tmem_base + (uint32_t)(pb * kTileRows);
#pragma unroll
          for (int k = 0; k < kF8BlockK / 32; ++k)
            umma_f8(d, sw128_kmajor_desc(sa + k * 32), sw128_kmajor_desc(sb + k * 32), idesc,
                    k != 0 ? 1u : 0u);
          umma_commit(&empty_bar[stage]);
          umma_commit(&pfull_bar[pb]);
          issued_any = true;
          if (++stage == kF8Stages) {
            stage = 0;
            phase ^= 1u;
          }
          if (++pb == kF8PBufs) {
            pb = 0;
            pphase ^= 1u;
          }
        }
      }
      if (issued_any) {
        umma_commit(&drain_bar);
        f8_wait_drain(&drain_bar, 0);
      }
    }
  } else {
    // ------------------------------------------------- scale-and-accumulate epilogue (8 warps)
    const int q = warp & 3;          // TMEM lane quarter this warp may read
    const int g = (warp - 2) >> 2;   // token-column half: [64g, 64g + 64)
    const int row = q * 32 + lane;   // weight row within the slab
    const int et = threadIdx.x - 64;  // 0..255
    int pb = 0, kbc = 0;
    uint32_t pphase = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      F8Unit U;
      if (!f8_unit(p, u, U)) continue;
      float acc[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
      // The scales of k blocks kb .. kb+3 are loaded ahead into registers, so their global
      // latency overlaps the MMAs instead of every k block waiting for it.
      const float* bs = p.b_scale + ((int64_t)U.e * p.n_slabs + U.slab) * p.num_kb;
      const bool has_row = et < U.nrows;
      const float* as = p.a_scale + (int64_t)(U.row0 + (has_row ? et : 0)) * p.num_kb;
      float nsa[4], nsw[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        nsa[i] = (has_row && i < p.num_kb) ? as[i] : 0.0f;
        nsw[i] = i < p.num_kb ? bs[i] : 0.0f;
      }
      for (int kb = 0; kb < p.num_kb; ++kb, ++kbc) {
        const int buf = kbc & 1;
        // column scale of this k block: b_scale (one per slab) times the token's a_scale
        if (et < kTileRows) s_sa[buf][et] = nsw[0] * nsa[0];
#pragma unroll
        for (int i = 0; i < 3; ++i) {
          nsa[i] = nsa[i + 1];
          nsw[i] = nsw[i + 1];
        }
        nsa[3] = (has_row && kb + 4 < p.num_kb) ? as[kb + 4] : 0.0f;
        nsw[3] = kb + 4 < p.num_kb ? bs[kb + 4] : 0.0f;
        const bool got = mbar_wait(&pfull_bar[pb], pphase, abort_flag, p.limit_ns, p.status);
        if (!named_bar_and(1, 256, got)) {  // also publishes s_sa[buf]
          ok = false;
          break;
        }
        tc_fence_after();
        const int ncols = U.n_mma - g * 64;  // warp-uniform
        const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) +
                            (uint32_t)(pb * kTileRows + g * 64);
        const float4* sc4 = reinterpret_cast<const float4*>(&s_sa[buf][g * 64]);
        if (ncols >= 64) {  // the whole half in one TMEM load
          float v[64];
          tmem_ld_x64(tb, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float4 sc = sc4[j];
            acc[4 * j] = fmaf(sc.x, v[4 * j], acc[4 * j]);
            acc[4 * j + 1] = fmaf(sc.y, v[4 * j + 1], acc[4 * j + 1]);
            acc[4 * j + 2] = fmaf(sc.z, v[4 * j + 2], acc[4 * j + 2]);
            acc[4 * j + 3] = fmaf(sc.w, v[4 * j + 3], acc[4 * j + 3]);
          }
        } else {  // decode-sized tiles: only the 16-column chunks that hold tokens
#pragma unroll
          for (int ch = 0; ch < 3; ++ch) {
            if (ch * 16 < ncols) {
              float v[16];
              tmem_ld_x16(tb + (uint32_t)(ch * 16), v);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float4 sc = sc4[ch * 4 + j];
                acc[ch * 16 + 4 * j] = fmaf(sc.x, v[4 * j], acc[ch * 16 + 4 * j]);
                acc[ch * 16 + 4 * j + 1] = fmaf(sc.y, v[4 * j + 1], acc[ch * 16 + 4 * j + 1]);
                acc[ch * 16 + 4 * j + 2] = fmaf(sc.z, v[4 * j + 2], acc[ch * 16 + 4 * j + 2]);
                acc[ch * 16 + 4 * j + 3] = fmaf(sc.w, v[4 * j + 3], acc[ch * 16 + 4 * j + 3]);
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pempty_bar[pb]);
        if (++pb == kF8PBufs) {
          pb = 0;
          pphase ^= 1u;
        }
      }
      if (!ok) break;
      // bf16 rows: column n = slab*128 + row of token row row0 + c (a warp writes 64 bytes).
      __nv_bfloat16* o = p.out + (int64_t)U.row0 * p.N + U.slab * kSlab + row;
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const int c = g * 64 + i;
        if (c < U.nrows) o[(int64_t)c * p.N] = __float2bfloat16_rn(acc[i]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kF8PBufs * kTileRows);
  }
}

}  // namespace

cudaError_t launch_gemm_fp8(int E, int N, int K, int64_t rows, const uint8_t* a,
                            const float* a_scale, const uint8_t* b, const float* b_scale,
                            const Tile* tiles, const int* n_tiles, int max_tiles,
                            __nv_bfloat16* out, int* status, cudaStream_t s, bool pdl) {
  if (N % kSlab != 0 || K % kF8BlockK != 0 || rows <= 0) return cudaErrorInvalidValue;
  CUtensorMap tmW, tmB16, tmB64, tmB128;
  if (!make_map_bytes(&tmW, b, (uint64_t)K, (uint64_t)E * N, kF8BlockK, kSlab) ||
      !make_map_bytes(&tmB16, a, (uint64_t)K, (uint64_t)rows, kF8BlockK, 16) ||
      !make_map_bytes(&tmB64, a, (uint64_t)K, (uint64_t)rows, kF8BlockK, 64) ||
      !make_map_bytes(&tmB128, a, (uint64_t)K, (uint64_t)rows, kF8BlockK, 128))
    return cudaErrorInvalidValue;
  F8Params p;
  p.N = N;
  p.num_kb = K / kF8BlockK;
  p.n_slabs = N / kSlab;
  p.tiles = tiles;
  p.n_tiles = n_tiles;
  p.a_scale = a_scale;
  p.b_scale = b_scale;
  p.out = out;
  p.status = status;
  p.limit_ns = wait_limit_ns();
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(moe_gemm_fp8_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kF8SmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const long long upper = (long long)max_tiles * p.n_slabs;
  const int sms = num_sms();
  const int grid = (int)(upper < sms ? upper : sms);
  if (grid <= 0) return cudaSuccess;
  return launch_k(moe_gemm_fp8_kernel, dim3(grid), dim3(kF8Threads), kF8SmemBytes, s, pdl, tmW,
                  tmB16, tmB64, tmB128, p);
}

}  // namespace gb300moe
