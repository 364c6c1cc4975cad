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
// therefore accumulated in a fresh TMEM buffer, and eight epilogue warps fold scale * D_kb into
// f32 registers (warp w reads TMEM lanes 32*(w%4)..; warpgroups split the token columns in
// halves), then store the bf16 rows.
//
// At decode sizes the MMA issuer, not HBM, sets the pace: every barrier wait, tcgen05.mma and
// commit costs the single issuing thread tens to a hundred cycles, while the MMAs themselves
// (N = 16..64 tokens) are short.  So for token tiles of up to 64 rows a pipeline stage carries
// two k blocks (256 k: two weight boxes and two token boxes) and the MMA thread pays one
// full-barrier wait, one TMEM-buffer wait and one commit per two k blocks; taller tiles keep one
// k block per stage, where the longer MMAs hide the issue cost and four TMEM buffers keep the
// epilogue's scale-and-accumulate work off the critical path.  In both, the epilogue learns that
// a stage's MMAs are done from the stage's empty barrier (the commit that frees its shared
// memory) instead of a second commit.  The stage count follows the stage size: six stages of
// 36 KB for 16-row tiles, six of 32 KB for 128.
//
// Units are taken round-robin (CTA c: units c, c + G, ...).  Splitting the last partial wave's
// units along k over all SMs (stream-K, with f32 partials handed between CTAs) was measured on
// the page's workloads and lost: the pieces are short, and their fixups cost more than the
// imbalance they remove.
//
// Warp roles (384 threads, one CTA per SM, persistent): warp 0 TMA producer, warp 1 MMA issuer
// (warps 2-3 idle; their warpgroup hands registers to the epilogue), warps 4-11
// scale-and-accumulate epilogue.  Every wait is bounded as in gemm.cu.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace gb300moe {

namespace {

constexpr int kF8BlockK = 128;                  // k per scale block
constexpr int kF8WBytes = kSlab * kF8BlockK;    // 16 KB of weights per k block
constexpr int kF8MaxStages = 6;
// One CTA per SM: 12 warps in three warpgroups.  Warpgroup 0 holds the TMA producer (warp 0)
// and the MMA issuer (warp 1; warps 2-3 idle) and gives up registers (setmaxnreg) to
// warpgroups 1-2, the epilogue (token columns 0-63 and 64-127), whose 64 f32 accumulators and
// 64-column TMEM loads per thread need them: 128 * 56 + 256 * 224 = 64512 = 384 threads * 168
// registers at launch.
// Two CTAs per SM (k2Cta; token tiles of at most 64 rows, which leave warpgroup 2 idle): 8
// warps, warpgroup 1 alone is the epilogue; 256 TMEM columns and half the shared memory each.
// Each SM then runs two MMA issuers: one issuing thread is latency bound and slows further
// next to the epilogue warps on its SMSP.  128 * 56 + 128 * 200 = 32768 = 256 threads * 128.
template <bool k2Cta>
struct F8Cfg {
  static constexpr int kThreads = k2Cta ? 256 : 384;
  static constexpr int kEpiThreads = kThreads - 128;
  static constexpr int kProducerRegs = 56;
  static constexpr int kEpilogueRegs = k2Cta ? 200 : 224;
  static constexpr int kLaunchRegs = k2Cta ? 128 : 168;
  static constexpr int kMinBlocks = k2Cta ? 2 : 1;
  static constexpr int kTmemCols = k2Cta ? 256 : 512;
  // Dynamic shared memory the kernel may use: the block's share of the SM's 228 KB, less the
  // per-block reserve and the static part.
  static constexpr int kSmemLimit = k2Cta ? 233472 / 2 - 1024 - 4096 : 232448 - 4096;
  static_assert(128 * kProducerRegs + kEpiThreads * kEpilogueRegs <= kThreads * kLaunchRegs,
                "register split exceeds the launch allocation");
  static_assert(kThreads * kLaunchRegs * kMinBlocks <= 65536, "registers of the SM");
};
constexpr uint64_t kF8DrainNs = 1000000000ull;

struct F8Params {
  int N, num_kb, n_slabs;
  int tcap;          // token rows a stage holds per k block (16..128, a multiple of 16)
  int tile_h;        // rows per tile of a group (128, or 64 at two CTAs per SM)
  int stage_bytes;   // KPS * (16 KB + tcap * 128), KPS = k blocks per stage
  int stages;        // pipeline stages (<= kF8MaxStages)
  int nbuf;          // TMEM buffers (KPS * tcap columns each), <= stages
  const Tile* tiles;
  const int* n_tiles;
  // With `meta`, the tile list is not read from `tiles` but derived in the prologue from the
  // layout metadata (at most kF8FusedGroups groups): masked (max_m > 0) counts, or contiguous
  // (max_m == 0) inclusive prefix sums over `rows` rows.
  const int32_t* meta;
  int E, max_m;
  long long rows;
  const float* a_scale;  // [rows, num_kb]
  const float* b_scale;  // [E, n_slabs, num_kb]
  __nv_bfloat16* out;    // [rows, N]
  int* status;
  uint64_t limit_ns;
};

struct F8Unit {
  int e, slab, row0, nrows, n_mma;
};

// Groups a launch can take its tile list from directly (shared-memory tables below).
constexpr int kF8FusedGroups = 128;

// The groups as the prologue tabulates them: tile g of the list belongs to the group e with
// tfirst[e] <= g < tfirst[e + 1]; its rows start at row0[e] + 128 * (g - tfirst[e]).
struct F8Groups {
  const int* tfirst;  // [E + 1]
  const int* row0;    // [E]
  const int* cnt;     // [E]
  int E;
};

// Units of group e occupy [n_slabs*first, n_slabs*(first+count)), slab-major (as in gemm.cu).
// `cur` is the caller's group cursor: a CTA visits its units in increasing order, so the owning
// group (the last whose first tile is <= the unit's tile) is found by stepping it forward.
__device__ __forceinline__ void f8_unit(const F8Params& p, const F8Groups& gr, int u, int& cur,
                                        F8Unit& U) {
  if (p.meta != nullptr) {
    const int ti = u / p.n_slabs;
    while (cur + 1 < gr.E && gr.tfirst[cur + 1] <= ti) ++cur;
    const int lo = cur;
    const int first = gr.tfirst[lo], count = gr.tfirst[lo + 1] - first;
    const int local = u - p.n_slabs * first;
    const int j = local % count;
    U.slab = local / count;
    U.e = lo;
    U.row0 = gr.row0[lo] + j * p.tile_h;
    U.nrows = min(p.tile_h, gr.cnt[lo] - j * p.tile_h);
  } else {
    const Tile owner = p.tiles[u / p.n_slabs];
    const int local = u - p.n_slabs * owner.first;
    U.slab = local / owner.count;
    const Tile t = p.tiles[owner.first + local % owner.count];
    U.e = t.e;
    U.row0 = t.row0;
    U.nrows = t.nrows;
  }
  U.n_mma = (U.nrows + 15) & ~15;
}

__device__ __forceinline__ void f8_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kF8DrainNs) return;
}

template <int KPS, bool k2Cta>
__global__ void __launch_bounds__(F8Cfg<k2Cta>::kThreads, F8Cfg<k2Cta>::kMinBlocks)
    moe_gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmB16,
                        const __grid_constant__ CUtensorMap tmB64,
                        const __grid_constant__ CUtensorMap tmB128, const F8Params p) {
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[kF8MaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kF8MaxStages];  // MMAs of the stage done
  __shared__ __align__(8) uint64_t pempty_bar[kF8MaxStages];  // TMEM buffer read by the epilogue
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  __shared__ int s_n_units;
  __shared__ int s_tfirst[kF8FusedGroups + 1], s_row0[kF8FusedGroups], s_cnt[kF8FusedGroups];
  __shared__ __align__(16) float s_sa[2][2][kTileRows];  // column scales of a stage's k blocks

  const uint32_t raw = smem_u32(dsmem);
  uint8_t* smem = dsmem + ((1024u - (raw & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &s_abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kF8MaxStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
      mbar_init(&pempty_bar[s], F8Cfg<k2Cta>::kEpiThreads / 32);  // one per epilogue warp
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
    tmem_alloc(&s_tmem_base, F8Cfg<k2Cta>::kTmemCols);
    tmem_relinquish();
  }
  pdl_wait();
  pdl_trigger();
  if (p.meta == nullptr) {
    if (threadIdx.x == 0) s_n_units = (*p.n_tiles) * p.n_slabs;
  } else if (warp == 0) {
    // The tile list from the layout metadata: lane l tabulates groups 4l .. 4l+3 (rows and
    // 128-row tiles), a warp scan gives each group's first tile.  As in the tile-list kernel,
    // a contiguous prefix sum that decreases or passes `rows` sets MOE_ERR_INVALID_ARG and
    // drops its group.
    int nt[4], tot = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = lane * 4 + i;
      int r0 = 0, c = 0;
      if (e < p.E) {
        if (p.max_m > 0) {
          r0 = e * p.max_m;
          c = min(max(p.meta[e], 0), p.max_m);
        } else {
          r0 = e == 0 ? 0 : p.meta[e - 1];
          c = p.meta[e] - r0;
          if (r0 < 0 || c < 0 || (long long)p.meta[e] > p.rows) {
            if (p.status) atomicCAS(p.status, 0, (int)MOE_ERR_INVALID_ARG);
            c = 0;
          }
        }
        s_row0[e] = r0;
        s_cnt[e] = c;
      }
      nt[i] = (c + p.tile_h - 1) / p.tile_h;
      tot += nt[i];
    }
    int incl = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    int run = incl - tot;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = lane * 4 + i;
      if (e < p.E) s_tfirst[e] = run;
      run += nt[i];
    }
    if (lane == 31) {
      s_tfirst[p.E] = incl;
      s_n_units = incl * p.n_slabs;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  const int n_units = s_n_units;
  const F8Groups gr{s_tfirst, s_row0, s_cnt, p.E};
  const int tblk = p.tcap * kF8BlockK;  // bytes of one k block of token rows

  if (warp < 4) {  // warpgroup 0: producer and MMA issuer
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(F8Cfg<k2Cta>::kProducerRegs));
    if (warp == 0) {
      // ------------------------------------------------------------------ TMA producer
      if (lane == 0) {
        int stage = 0, issued = 0;
        uint32_t phase = 0;
        bool ok = true;
        int gcur = 0;  // group cursor (tile list from the metadata)
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
          F8Unit U;
          f8_unit(p, gr, u, gcur, U);
          const int wrow = U.e * p.N + U.slab * kSlab;
          for (int kb = 0; kb < p.num_kb; kb += KPS) {
            const int nk = p.num_kb - kb >= KPS ? KPS : 1;
            if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, p.limit_ns, p.status)) {
              ok = false;
              break;
            }
            uint8_t* sw = smem + stage * p.stage_bytes;
            uint8_t* st = sw + KPS * kF8WBytes;
            mbar_arrive_expect_tx(&full_bar[stage],
                                  (uint32_t)(nk * (kF8WBytes + U.n_mma * kF8BlockK)));
  #pragma unroll
            for (int j = 0; j < KPS; ++j) {
              if (j >= nk) break;
              const int kx = (kb + j) * kF8BlockK;
              tma_load_2d(sw + j * kF8WBytes, &tmW, &full_bar[stage], kx, wrow);
              uint8_t* tb = st + j * tblk;
              int r = 0;
              for (; r + 128 <= U.n_mma; r += 128)
                tma_load_2d(tb + r * kF8BlockK, &tmB128, &full_bar[stage], kx, U.row0 + r);
              for (; r + 64 <= U.n_mma; r += 64)
                tma_load_2d(tb + r * kF8BlockK, &tmB64, &full_bar[stage], kx, U.row0 + r);
              for (; r < U.n_mma; r += 16)
                tma_load_2d(tb + r * kF8BlockK, &tmB16, &full_bar[stage], kx, U.row0 + r);
            }
            ++issued;
            if (++stage == p.stages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (*abort_flag) {
          const int n = issued < p.stages ? issued : p.stages;
          for (int i = issued - n; i < issued; ++i)
            f8_wait_drain(&full_bar[i % p.stages], (uint32_t)((i / p.stages) & 1));
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        int stage = 0, pb = 0;
        uint32_t phase = 0, pphase = 0;
        bool ok = true, issued_any = false;
        const uint32_t smem_base = smem_u32(smem);
        int gcur = 0;  // group cursor (tile list from the metadata)
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
          F8Unit U;
          f8_unit(p, gr, u, gcur, U);
          const uint32_t idesc = idesc_e4m3_m128(U.n_mma);
          for (int kb = 0; kb < p.num_kb; kb += KPS) {
            const int nk = p.num_kb - kb >= KPS ? KPS : 1;
            if (!mbar_wait(&full_bar[stage], phase, abort_flag, p.limit_ns, p.status) ||
                !mbar_wait(&pempty_bar[pb], pphase ^ 1u, abort_flag, p.limit_ns, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sw = smem_base + (uint32_t)(stage * p.stage_bytes);
            // descriptors of k = 0; a step of 32 bytes along k adds 2 to the address field
            const uint64_t da = sw128_kmajor_desc(sw);
            const uint64_t db = sw128_kmajor_desc(sw + (uint32_t)(KPS * kF8WBytes));
            const uint32_t d = tmem_base + (uint32_t)(pb * KPS * p.tcap);
  #pragma unroll
            for (int j = 0; j < KPS; ++j) {
              if (j >= nk) break;
              const uint64_t daj = da + (uint64_t)((j * kF8WBytes) >> 4);
              const uint64_t dbj = db + (uint64_t)((j * tblk) >> 4);
              const uint32_t dj = d + (uint32_t)(j * p.tcap);
  #pragma unroll
              for (int k = 0; k < kF8BlockK / 32; ++k)
                umma_f8(dj, daj + 2 * k, dbj + 2 * k, idesc, k != 0 ? 1u : 0u);
            }
            umma_commit(&empty_bar[stage]);  // frees the smem stage; tells the epilogue
            issued_any = true;
            if (++stage == p.stages) {
              stage = 0;
              phase ^= 1u;
            }
            if (++pb == p.nbuf) {
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
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(F8Cfg<k2Cta>::kEpilogueRegs));
    // ------------------------------------------------- scale-and-accumulate epilogue (8 warps)
    const int q = warp & 3;          // TMEM lane quarter this warp may read
    const int g = (warp - 4) >> 2;   // token-column half: [64g, 64g + 64)
    const int row = q * 32 + lane;   // weight row within the slab
    const int et = threadIdx.x - 128;  // 0 .. kEpiThreads - 1
    int stage = 0, pb = 0, sc = 0;
    uint32_t phase = 0, pphase = 0;
    bool ok = true;
    int gcur = 0;  // group cursor (tile list from the metadata)
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      F8Unit U;
      f8_unit(p, gr, u, gcur, U);
      float acc[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
      // The scales of k blocks kb .. kb+3 are loaded ahead into registers, so their global
      // latency overlaps the MMAs instead of every stage waiting for it.
      const float* bs = p.b_scale + ((int64_t)U.e * p.n_slabs + U.slab) * p.num_kb;
      const bool has_row = et < U.nrows;
      const float* as = p.a_scale + (int64_t)(U.row0 + (has_row ? et : 0)) * p.num_kb;
      float nsa[4], nsw[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        nsa[i] = (has_row && i < p.num_kb) ? as[i] : 0.0f;
        nsw[i] = i < p.num_kb ? bs[i] : 0.0f;
      }
      const int ncols = U.n_mma - g * 64;  // warp-uniform; may be <= 0
      for (int kb = 0; kb < p.num_kb; kb += KPS) {
        const int nk = p.num_kb - kb >= KPS ? KPS : 1;
        const int buf = sc & 1;
        // column scales of the stage's k blocks: b_scale (one per slab) times the token's
        // a_scale; the k blocks 4 ahead are fetched in their place
#pragma unroll
        for (int j = 0; j < KPS; ++j) {
          if (j < nk) {
            if (et < kTileRows) s_sa[buf][j][et] = nsw[0] * nsa[0];
#pragma unroll
            for (int i = 0; i < 3; ++i) {
              nsa[i] = nsa[i + 1];
              nsw[i] = nsw[i + 1];
            }
            nsa[3] = (has_row && kb + j + 4 < p.num_kb) ? as[kb + j + 4] : 0.0f;
            nsw[3] = kb + j + 4 < p.num_kb ? bs[kb + j + 4] : 0.0f;
          }
        }
        const bool got = mbar_wait(&empty_bar[stage], phase, abort_flag, p.limit_ns, p.status);
        if (!named_bar_and(1, F8Cfg<k2Cta>::kEpiThreads, got)) {  // also publishes s_sa[buf]
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < KPS; ++j) {
          if (j < nk) {
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) +
                                (uint32_t)((KPS * pb + j) * p.tcap + g * 64);
            const float4* sc4 = reinterpret_cast<const float4*>(&s_sa[buf][j][g * 64]);
            if (ncols >= 64) {  // the whole half in one TMEM load
              float v[64];
              tmem_ld_x64(tb, v);
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float4 s4 = sc4[i];
                acc[4 * i] = fmaf(s4.x, v[4 * i], acc[4 * i]);
                acc[4 * i + 1] = fmaf(s4.y, v[4 * i + 1], acc[4 * i + 1]);
                acc[4 * i + 2] = fmaf(s4.z, v[4 * i + 2], acc[4 * i + 2]);
                acc[4 * i + 3] = fmaf(s4.w, v[4 * i + 3], acc[4 * i + 3]);
              }
            } else {  // decode-sized tiles: only the 16-column chunks that hold tokens
#pragma unroll
              for (int ch = 0; ch < 3; ++ch) {
                if (ch * 16 < ncols) {
                  float v[16];
                  tmem_ld_x16(tb + (uint32_t)(ch * 16), v);
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    const float4 s4 = sc4[ch * 4 + i];
                    acc[ch * 16 + 4 * i] = fmaf(s4.x, v[4 * i], acc[ch * 16 + 4 * i]);
                    acc[ch * 16 + 4 * i + 1] = fmaf(s4.y, v[4 * i + 1], acc[ch * 16 + 4 * i + 1]);
                    acc[ch * 16 + 4 * i + 2] = fmaf(s4.z, v[4 * i + 2], acc[ch * 16 + 4 * i + 2]);
                    acc[ch * 16 + 4 * i + 3] = fmaf(s4.w, v[4 * i + 3], acc[ch * 16 + 4 * i + 3]);
                  }
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pempty_bar[pb]);
        ++sc;
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1u;
        }
        if (++pb == p.nbuf) {
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
    tmem_dealloc(tmem_base, F8Cfg<k2Cta>::kTmemCols);
  }
}

}  // namespace

cudaError_t launch_gemm_fp8(int E, int N, int K, int64_t rows, int max_tile_rows,
                            const uint8_t* a, const float* a_scale, const uint8_t* b,
                            const float* b_scale, const Tile* tiles, const int* n_tiles,
                            int max_tiles, const int32_t* meta, int max_m,
                            __nv_bfloat16* out, int* status, cudaStream_t s, bool pdl) {
  if (meta != nullptr && E > kF8FusedGroups) return cudaErrorInvalidValue;
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
  // Token rows per stage and k block: the tallest tile this layout can produce.
  int tcap = max_tile_rows < 1 ? 1 : (max_tile_rows > kTileRows ? kTileRows : max_tile_rows);
  tcap = (tcap + 15) & ~15;
  // 64-row tiles with two k blocks per stage ("narrow"): always when no group can exceed 64
  // rows; for a masked layout of at least 256 rows per group too.  The layout's capacity does
  // not say how many rows its groups hold (the counts live on the device), so this is a rule:
  // the page's 256-row layouts hold 5-16 rows a group and gained 8-21 % with narrow tiles
  // (a group's weight slab is read from HBM once by adjacent units, the rest from L2), while
  // its 128-row layout holds about 96 a group, and its up projection lost 33 % to twice the
  // units.  Narrow tiles of at most 16 k blocks run two CTAs per SM (one epilogue warpgroup
  // covers a 64-row tile): the b64 down projections gained 6-8 %, the up projections (32-56 k
  // blocks) lost up to 4 % to the halved pipeline depth of each CTA.
  const bool narrow = tcap <= 64 || (meta != nullptr && max_m >= 256);
  const bool two = narrow && p.num_kb <= 16;
  if (narrow && tcap > 64) tcap = 64;
  p.tcap = tcap;
  p.tile_h = narrow ? 64 : kTileRows;
  const int kps = tcap <= 64 ? 2 : 1;
  const int smem_limit = two ? F8Cfg<true>::kSmemLimit : F8Cfg<false>::kSmemLimit;
  p.stage_bytes = kps * (kF8WBytes + tcap * kF8BlockK);
  p.stages = (smem_limit - 1024) / p.stage_bytes;
  if (p.stages > kF8MaxStages) p.stages = kF8MaxStages;
  p.nbuf = (two ? F8Cfg<true>::kTmemCols : F8Cfg<false>::kTmemCols) / (kps * tcap);
  if (p.nbuf > p.stages) p.nbuf = p.stages;  // the epilogue never falls a full ring behind
  p.tiles = tiles;
  p.n_tiles = n_tiles;
  p.meta = meta;
  p.E = E;
  p.max_m = max_m;
  p.rows = rows;
  p.a_scale = a_scale;
  p.b_scale = b_scale;
  p.out = out;
  p.status = status;
  p.limit_ns = wait_limit_ns();
  static bool attr_set = false;
  if (!attr_set) {
    for (auto k : {moe_gemm_fp8_kernel<1, false>, moe_gemm_fp8_kernel<2, false>}) {
      cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           F8Cfg<false>::kSmemLimit);
      if (e != cudaSuccess) return e;
    }
    cudaError_t e = cudaFuncSetAttribute(moe_gemm_fp8_kernel<2, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         F8Cfg<true>::kSmemLimit);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const long long upper = (long long)max_tiles * p.n_slabs;
  const int sms = num_sms();
  const long long slots = two ? 2ll * sms : sms;
  const int grid = (int)(upper < slots ? upper : slots);
  if (grid <= 0) return cudaSuccess;
  const size_t smem = (size_t)p.stages * p.stage_bytes + 1024;
  if (two)
    return launch_k(moe_gemm_fp8_kernel<2, true>, dim3(grid), dim3(F8Cfg<true>::kThreads), smem,
                    s, pdl, tmW, tmB16, tmB64, tmB128, p);
  return launch_k(kps == 2 ? moe_gemm_fp8_kernel<2, false> : moe_gemm_fp8_kernel<1, false>,
                  dim3(grid), dim3(F8Cfg<false>::kThreads), smem, s, pdl, tmW, tmB16, tmB64,
                  tmB128, p);
}

}  // namespace gb300moe
