// common.cuh -- shared definitions of the GB300 MoE kernels (status word, dtype traits, launch
// prototypes).  Everything here is device-side product code; nothing is shared with the oracle.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace gb300moe {

// Number of SMs on a GB300 (2 dies x 76); the launchers read the real count at run time and
// use this only as an upper bound for static tables.
constexpr int kMaxSMs = 256;

// Token rows per GEMM tile (the N side of the tcgen05 MMA: 128, or 256 when experts have many
// rows) and weight rows per slab (the M side); K is staged 64 elements (128 bytes) at a time
// with the 128-byte swizzle.
constexpr int kTileRows = 128;
constexpr int kTileRowsWide = 256;
constexpr int kTileRowsNarrow = 64;  // 16-bit down projection at decode sizes; NVFP4 gate/up
constexpr int kTileRowsNvfp4Min = 32;  // NVFP4 gate/up tiles at the smallest decode sizes
constexpr int kSlab = 128;
constexpr int kBlockK = 64;

// Workspace header: status word at offset 0, tile counter at offset 64.
constexpr size_t kHeaderBytes = 256;

// Experts whose weights this GPU holds (an expert-parallel shard, or all E), and the problem
// as the post-routing stages see it: ids are local indices in [0, local_experts) or -1.
// CTAs a persistent GEMM uses for `units` equal units when it has `ctas` of them: the fewest
// that keep each CTA's share at ceil(units / ctas), so every working CTA gets that share or one
// less and none sits out the last wave's tail.  CTAs from this count on take no unit.  (The
// 16-bit-weight GEMMs use it: their units stream weights at HBM speed, so a last wave on fewer
// SMs leaves HBM idle.  The FP8 and NVFP4 GEMMs do not: their units run at the SM's own pace,
// and the FP8 one measured slower on fewer CTAs.)
__host__ __device__ __forceinline__ int balanced_ctas(int units, int ctas) {
  if (units <= 0 || ctas <= 0) return ctas;
  const int waves = (units + ctas - 1) / ctas;
  return (units + waves - 1) / waves;
}

inline int local_experts(const moe_problem_t& p) {
  return p.ep_num_local > 0 ? p.ep_num_local : p.E;
}
inline moe_problem_t local_view(const moe_problem_t& p) {
  moe_problem_t q = p;
  q.E = local_experts(p);
  q.ep_num_local = 0;
  q.ep_local_offset = 0;
  return q;
}

// First error wins; later errors are dropped until the host reads and clears the word.
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

template <typename T> struct DT;
template <> struct DT<__nv_bfloat16> {
  static constexpr int kIsBF16 = 1;
  __device__ __forceinline__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  __device__ __forceinline__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};
template <> struct DT<__half> {
  static constexpr int kIsBF16 = 0;
  __device__ __forceinline__ static float to_f(__half v) { return __half2float(v); }
  __device__ __forceinline__ static __half from_f(float v) { return __float2half_rn(v); }
};

// A tile of the grouped GEMM schedule: expert, first row, number of rows (<= kTileRows), and
// the index of the expert's first tile and its tile count (the tiles of an expert are
// contiguous), so that a unit index maps to (expert, weight slab, tile) in O(1).
struct __align__(16) Tile {
  int e, row0, nrows, first;
  int count, pad0, pad1, pad2;
};

// Launch `kern` on `s`; with pdl the launch may overlap the tail of the previous kernel on the
// stream (programmatic stream serialization): the kernel itself waits for it with pdl_wait().
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---- launchers (defined in the .cu files, called by api.cu) ------------------------------
// `pdl`: true when the launch follows another kernel of the same entry point.
// With `rows_f16`, extra CTAs of the same launch also write hidden_states ([T, H] bf16) to
// rows_f16 as f16 (the NVFP4 path's token rows), setting MOE_ERR_F16_RANGE in `status` for a
// value past the f16 range.
cudaError_t launch_route(const moe_problem_t& p, const float* gating, const float* bias,
                         int32_t* ids, float* w, cudaStream_t s, bool pdl,
                         const void* hidden = nullptr, void* rows_f16 = nullptr,
                         int* status = nullptr);

// The sort: one launch when it fits, else the chunked form.
cudaError_t launch_align_sort(const moe_problem_t& p, int block_m, const int32_t* ids,
                              int32_t* counts, int32_t* offsets, int32_t* sorted_ids,
                              int64_t cap, int32_t* tile_expert, int32_t* inv_route,
                              int32_t* chunk_scratch, int* status, cudaStream_t s, bool pdl);

// The sort in one launch (one CTA) when it fits (T*top_k <= 8192); with `tiles` (`tiles2`)
// it also writes the GEMM tile list of tile_rows (tile_rows2) rows per tile, and it zeroes
// zero[0, n_zero) (the split-K counters of the GEMM that follows).
bool fused_sort_fits(const moe_problem_t& p);
cudaError_t launch_sort_fused(const moe_problem_t& p, int block_m, const int32_t* ids,
                              int32_t* counts, int32_t* offsets, int32_t* sorted_ids,
                              int64_t cap, int32_t* tile_expert, int32_t* inv_route, Tile* tiles,
                              int* n_tiles, int tile_rows, Tile* tiles2, int* n_tiles2,
                              int tile_rows2, int* status, cudaStream_t s, bool pdl,
                              int* zero = nullptr, int n_zero = 0);
// The sort as three launches over 256-route chunks (any size), using chunk_scratch
// (ceil(T*top_k/256) * E int32); with `tiles` (`tiles2`) the scan also writes the GEMM tile
// lists.
cudaError_t launch_align_sort_chunked(const moe_problem_t& p, int block_m, const int32_t* ids,
                                      int32_t* counts, int32_t* offsets, int32_t* sorted_ids,
                                      int64_t cap, int32_t* tile_expert, int32_t* inv_route,
                                      int32_t* chunk_scratch, int* status, cudaStream_t s,
                                      bool pdl, Tile* tiles, int* n_tiles, int tile_rows,
                                      Tile* tiles2, int* n_tiles2, int tile_rows2);

cudaError_t launch_build_tiles(int E, const int32_t* offsets, Tile* tiles, int* n_tiles,
                               int tile_rows, cudaStream_t s, bool pdl);

// to_f16: bf16 rows in, f16 rows out (the NVFP4 path), MOE_ERR_F16_RANGE in `status` for a
// value past the f16 range.
cudaError_t launch_permute(int dtype, int top_k, int H, const void* hidden,
                           const int32_t* sorted_ids, const int32_t* offsets, int E, int64_t cap,
                           void* a_sorted, cudaStream_t s, bool pdl, bool to_f16 = false,
                           int* status = nullptr);

// Tile list over a grouped-GEMM layout (masked or prefix sums) and the weighted post-permute.
cudaError_t launch_build_tiles_meta(int E, int max_m, int64_t rows, const int32_t* meta,
                                    Tile* tiles, int* n_tiles, int tile_rows, int* status,
                                    cudaStream_t s, bool pdl);
cudaError_t launch_post_permute(int dtype, int T, int K, int H, const void* rows,
                                const float* w, const int32_t* inv, void* out, cudaStream_t s,
                                bool pdl);

// FP8 (E4M3) block-scaled grouped GEMM (gemm_fp8.cu); out is bf16 [rows, N].
// max_tile_rows bounds the rows of any tile of the layout (it sizes the token stages).
// With `meta` (E <= 128 groups) the kernel derives the tile list itself from the layout
// metadata (max_m > 0: masked counts; 0: inclusive prefix sums) and `tiles` is not read.
cudaError_t launch_gemm_fp8(int E, int N, int K, int64_t rows, int max_tile_rows,
                            const uint8_t* a, const float* a_scale, const uint8_t* b,
                            const float* b_scale, const Tile* tiles, const int* n_tiles,
                            int max_tiles, const int32_t* meta, int max_m,
                            __nv_bfloat16* out, int* status, cudaStream_t s, bool pdl);

// Activation code of the single-projection GEMM that writes the product itself (the plain
// grouped GEMM); not a moe_activation_t a caller can pass.
constexpr int kActIdentity = 3;
// Magnitude from which a value rounds to an infinite f16 (the NVFP4 path's token rows and act
// are f16).
constexpr float kF16Overflow = 65520.0f;

// Eight bf16 values (one 16-byte vector) to f16: exact from 2^-14 to 65504 in magnitude,
// rounded to the nearest f16 below 2^-14 (an error of at most 2^-25); returns true when one
// of them is at or past kF16Overflow (it becomes infinite).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v, bool& over) {
  const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
  over |= fabsf(f.x) >= kF16Overflow || fabsf(f.y) >= kF16Overflow;
  const __half2 h = __floats2half2_rn(f.x, f.y);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint4 bf16x8_to_f16x8(const uint4 v, bool& over) {
  return make_uint4(bf16x2_to_f16x2(v.x, over), bf16x2_to_f16x2(v.y, over),
                    bf16x2_to_f16x2(v.z, over), bf16x2_to_f16x2(v.w, over));
}

// NVFP4 weights -> the packed tile layout the W4A16 GEMMs read (nvfp4_pack.cu).
cudaError_t launch_nvfp4_pack(int64_t n_mats, int rows, int K, const uint8_t* codes,
                              const uint8_t* scales, uint8_t* tiles, cudaStream_t s);

// p is the caller's whole problem (its expert-parallel fields decide the kernel: a shard whose
// tokens average at most two routes to its experts lists each token's routes first).
cudaError_t launch_combine(const moe_problem_t& p, const void* y_route,
                           const int32_t* inv_route, const int32_t* ids, const void* shared_out,
                           void* out, cudaStream_t s, bool pdl);

// Grouped GEMM on tcgen05.  mode: 0 = sorted segments (tile list), 1 = direct from topk_ids
// (T <= 8), 2 = dense rows (one expert, all rows: the shared expert).
enum GemmMode { kSorted = 0, kDirect = 1, kDense = 2 };

struct GemmCall {
  int gemm1;      // 1: gate/up + activation; 0: down projection with route weight
  int act;        // gemm1: moe_activation_t (ReLU2: w has n_out rows per expert, not 2*n_out)
  int mode;       // GemmMode
  int dtype;      // moe_dtype_t
  int K;          // reduction length (H for gemm1, F for gemm2)
  int n_out;      // output columns (F for gemm1, H for gemm2)
  int E;          // experts (1 for dense)
  const void* w;  // weights: gemm1 [E, 2*n_out, K] ([E, n_out, K] for ReLU2); gemm2 [E, n_out, K]
                  // (NVFP4: the packed tiles of moe_nvfp4_pack)
  int w4;         // 1: NVFP4 weights (E2M1 codes, E4M3 scales per 16 k, FP32 scale per expert)
  const float* alpha;   // NVFP4 per-expert scale [E]
  const void* b;  // token rows [b_rows, K]
  int64_t b_rows; // rows of b (tensor extent)
  void* out;      // [*, n_out]
  // sorted mode
  const Tile* tiles;
  const int* n_tiles;
  int max_tiles;  // upper bound of *n_tiles (grid sizing)
  int tile_rows;  // token rows per tile: 128 or 256 (sorted tiles must be built with it)
  int token_rows; // sorted gemm1 with T <= 128 and no padding slots: b is hidden_states [T, K]
                  // and each sorted row takes the column of its route's token (no gather)
  const int32_t* sorted_ids;  // gemm2 scale lookup
  // direct mode
  const int32_t* topk_ids;
  int P, top_k, T;
  // dense mode
  int dense_rows;
  // gemm2 route weights
  const float* topk_w;
  // sorted mode: the tile list was written at least two launches before this GEMM, so the
  // kernel may read it (and prefetch its first units' weights) before its dependency wait
  int early_tiles;
  // NVFP4 gate/up GEMM over token rows: when it shortens the last wave, each unit's K range is
  // split in two halves run by different CTAs.  Both store their f32 accumulators in
  // split_part (split_cols columns per accumulator); the half that finishes second, told by
  // split_cnt[unit] (zeroed before the launch), adds the other's and writes the output.  Only
  // when the units number at most split_cap (0: never).
  int split_cap;
  int split_cols;
  float* split_part;
  int* split_cnt;
  // 16-bit gate/up GEMM over token rows: the router's ids [P].  The unit list (one tile per
  // routed expert, in expert order) follows from them, so the weight producer and the MMA
  // issuer start before the sort has finished; only the epilogue waits for it.
  const int32_t* route_ids;
  int* status;
};

cudaError_t launch_gemm(const GemmCall& c, cudaStream_t s, bool pdl);

// The grouped down projection on pairs of SMs (gemm_pair.cu): sorted mode with 256-row tiles,
// 16-bit weights, n_out a multiple of 256.  pair_gemm_available: whether clusters of two fit on
// this device.
cudaError_t launch_gemm_pair(const GemmCall& c, cudaStream_t s, bool pdl);
bool pair_gemm_available(int dtype);

uint64_t wait_limit_ns();
int num_sms();

// Checks a problem description (sizes, routing options, the expert-parallel shard, the limits
// of the kernels: E <= 1024, top_k <= 32, T*top_k <= 2^30); returns MOE_OK,
// MOE_ERR_INVALID_ARG or MOE_ERR_UNSUPPORTED.
moe_status_t check_problem(const moe_problem_t* p);

}  // namespace gb300moe
