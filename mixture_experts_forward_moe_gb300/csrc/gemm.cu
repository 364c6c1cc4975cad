// gemm.cu -- grouped expert GEMMs on the sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// TileOPs "MoE" page, op MoEGroupedGemmFwd (contiguous layout; activation=silu_and_mul for the
// gate/up projection) and op SharedExpertMLPFwd.  The design is GB300-first:
//
//  * Weight-stationary orientation ("swap AB").  Every config on the pages streams far more
//    weight bytes than activation bytes, so the 128-row MMA side (M) is a slab of 128 weight
//    rows and the N side is the expert's token rows (16..128, a multiple of 16).  Each unit of
//    work reads its weight slab from HBM exactly once along K, whatever the number of tokens.
//  * gemm1: the slab is 128 gate rows [f0, f0+128) and the matching 128 up rows [F+f0, ...),
//    two MMAs per K step into two TMEM accumulators, so epilogue thread i holds gate row i and
//    up row i and computes SiLU(g)*u (or GELU_tanh(g)*u) in f32 with no data exchange.  The
//    single-projection ReLU2 MLP has no up rows: its unit takes 256 consecutive rows as two
//    128-row halves in the same two accumulators (the second skipped past the last row) and
//    the epilogue writes max(h,0)^2 of each half to its own 128 output columns.
//  * gemm2: the slab is 128 rows of w_down; the epilogue multiplies by the route weight.
//  * Warp roles (192 threads, one CTA per SM, persistent over units):
//      warp 0  TMA producer: weight boxes {64 x 128} and token boxes of 128, 64 and 16 rows
//              (as few copies as the tile's rows allow), 128-byte swizzle, into a multi-stage
//              shared-memory ring (mbarrier complete_tx);
//      warp 1  MMA issuer: tcgen05.mma kind::f16, f32 accumulators in TMEM, double-buffered
//              so the epilogue of one unit overlaps the K loop of the next;
//      warps 2-5  epilogue: tcgen05.ld -> f32 math.  gemm1 rounds SiLU(g)*u once to bf16/f16,
//              transposes the tile through shared memory and stores whole output rows with
//              16-byte stores; gemm2 keeps the weighted rows in f32 (rounded once, later, by the
//              combine) and stores them straight from registers.
//  * Cluster size 1 and no multicast: each CTA fetches its own tiles.
//  * Every wait is bounded (global timer); on expiry the kernel records MOE_ERR_TIMEOUT, the
//    roles stop, in-flight copies and MMAs are drained, TMEM is freed and the kernel returns.
//
// Modes (how a unit index maps to an expert, token rows and output rows):
//   sorted  units = tiles x slabs; tile = (expert, first row, rows) over the expert-contiguous
//           rows produced by the sort; output row = input row.
//   direct  units = routes x slabs for T <= 8 (aiter PR #5973 "Changes": direct decoding runs
//           straight from topk_ids without sorting); a unit is owned by the first route of its
//           expert; the token side is every token (gemm1) or every route row (gemm2), and the
//           epilogue writes the rows of the routes that chose the expert.
//   dense   one expert over all rows in order (the shared expert).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "nvfp4.cuh"
#include "ptx.cuh"

namespace gb300moe {

namespace {

// Tile configurations: kN token rows per tile (the MMA's N).  kN = 128 keeps two accumulator
// buffers in TMEM for every GEMM (the epilogue of one unit overlaps the K loop of the next);
// kN = 256 halves how often an expert with many rows streams its weights, at the cost of a
// single gemm1 accumulator buffer (2 x 256 columns fill TMEM) and fewer pipeline stages.
//
// NVFP4 weights (kW4, the W4A16 GEMMs).  A stage covers 128 k, and the weights and the tokens
// travel in separate rings so that a weight slot is refilled as soon as it has been decoded:
//  * weight ring (kNW slots): per slab one 9216-byte tile of the packed weight layout
//    (moe_nvfp4_pack: the 128 rows' E2M1 codes for 128 k, then their E4M3 block scales), one
//    contiguous bulk copy; freed by the decoders;
//  * token ring (kNT slots): two 128-byte-swizzled 64-k boxes of token rows; freed by the MMA;
//  * TMEM ring (kAStages slots of 64 k): the decoder warps (eight, or four per CTA with two
//    CTAs per SM) turn the codes into exact f16 values and store them there (one column holds
//    two consecutive k of one weight row); the MMA reads its A operand from it.  The
//    accumulators take the first columns and the ring the rest.
//  * MMA issue: one thread per chain.  The gate/up GEMMs issue the gate and the up chain from
//    two warps, and the 64-row down projection the first and the second 64-k half of every
//    stage into two accumulators that the epilogue adds.
// Every tcgen05.mma of M = 128 and k = 16 takes about the same time whatever N and wherever A
// comes from, so at decode sizes the MMA issue rate bounds these GEMMs; the rings are sized so
// that the decoders and the loads keep it fed.
//
// 64-row token tiles of the 16-bit GEMMs (the down projection at decode sizes): a stage carries
// two 64-k blocks (kKps = 2), so the MMA issuer pays one barrier wait and one commit per 32 KB of
// weights instead of per 16 KB; at a few tokens per expert those per-stage costs, not HBM,
// would otherwise set the pace.
//
// Two CTAs per SM (k2Cta): the NVFP4 down projection (128- or 64-row tiles) and the NVFP4
// gate/up GEMM with 64- or 32-row tiles (at most 64 tokens, or gathered rows at decode sizes)
// run two CTAs on each SM, each with half the TMEM (256 columns: one accumulator buffer and the
// decoded-weight ring),
// about half the shared memory and four decoder warps.  One MMA-issuing thread is latency
// bound (about 44 cycles per tcgen05.mma at these N when nothing else runs on its SMSP, and
// twice that next to busy decoder warps), so a second issuer per SM measured 19-21 % faster on
// the down projection and 12 % on the gate/up GEMM.  32-row gate/up accumulators (64 columns)
// leave three 64-k slots for the decoded weights instead of two (another 9 %).  The 128-row
// gate/up GEMM keeps one CTA: its accumulators alone fill 256 columns.
template <bool kGemm1, int kN, bool kW4 = false, bool k2Cta = false>
struct Cfg {
  static_assert(kN == 32 || kN == 64 || kN == 128 || kN == 256, "tile rows");
  static_assert(kN != 64 || kW4 || !kGemm1, "64-row tiles: 16-bit down proj. or NVFP4");
  static_assert(kN != 32 || (kGemm1 && kW4 && k2Cta), "32-row tiles: NVFP4 gate/up, two CTAs");
  static_assert(!kW4 || kN == 128 || kN == 64 || (kN == 32 && kGemm1),
                "NVFP4 tiles are 128 or 64 rows (32 for gate/up)");
  static_assert(!k2Cta || (kW4 && (kGemm1 ? kN <= 64 : kN >= 64)),
                "two CTAs per SM: the NVFP4 down proj. and 32/64-row gate/up");
  static constexpr int kSlabs = kGemm1 ? 2 : 1;
  static constexpr int kKps = (kN == 64 && !kW4) ? 2 : 1;  // 64-k blocks per stage (16-bit)
  static constexpr int kStageK = kW4 ? 128 : kBlockK * kKps;  // k per pipeline stage
  static constexpr int kStages = kGemm1 ? (kN == 128 ? 4 : 3) : (kN == 64 ? 4 : (kN == 128 ? 7 : 4));
  static constexpr int kASubBytes = kSlabs * kSlab * kBlockK * 2;  // weights of one 64-k block
  static constexpr int kBSubBytes = kN * kBlockK * 2;              // tokens of one 64-k block
  static constexpr int kABytes = kASubBytes * (kW4 ? 1 : kKps);
  static constexpr int kBBytes = kN * kStageK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  // NVFP4 rings
  static constexpr int kQBytes = kSlab * 64;  // packed codes of one slab (128 k)
  static constexpr int kSfBytes = kSlab * 8;  // block scales of one slab (128 k)
  static constexpr int kTileBytes = kQBytes + kSfBytes;  // one tile of the packed layout
  static constexpr int kWBytes = kSlabs * kTileBytes;
  static constexpr int kNW = k2Cta ? (kGemm1 ? 3 : 4) : (kGemm1 ? 6 : 8);
  static constexpr int kNT = k2Cta ? ((kN == 32 || (!kGemm1 && kN == 64)) ? 4 : 2) : (kGemm1 ? 3 : 4);
  static constexpr int kRingBytes = kW4 ? kNW * kWBytes + kNT * kBBytes : kStages * kStageBytes;
  static constexpr int kFullBars = kW4 ? kNT : kStages;  // token (or combined) ring barriers
  // gemm1 transposes 64 token columns at a time through shared memory; gemm2 writes f32 rows
  // straight from registers.
  static constexpr int kPassCols = 64;
  static constexpr int kStagingBytes = kGemm1 ? kPassCols * kSlab * 2 : 0;
  // The NVFP4 down projection over 64-row tiles accumulates each stage's two 64-k halves in two
  // accumulators (one per MMA issuer, below), which the epilogue adds.
  static constexpr bool kKHalves = kW4 && !kGemm1 && kN == 64;
  static constexpr int kAccCols = (kGemm1 || kKHalves) ? 2 * kN : kN;  // per accumulator buffer
  static constexpr int kAccBufs =
      kW4 ? ((k2Cta || (kGemm1 && kN == 128)) ? 1 : 2) : ((kGemm1 && kN == 256) ? 1 : 2);
  static constexpr int kABase = kAccBufs * kAccCols;  // first TMEM ring column
  static constexpr int kASlotCols = kSlabs * 32;      // 64 k of every slab
  static constexpr int kTmemTotal = k2Cta ? 256 : 512;  // two CTAs per SM share the 512 columns
  static constexpr int kAStages = kW4 ? (kTmemTotal - kABase) / kASlotCols : 1;
  static constexpr int kTmemCols = kW4 ? kTmemTotal : kAccBufs * kAccCols;
  // NVFP4 warps: 0 weight producer, 1 MMA, 2-5 epilogue, then the decoders (eight; four, each
  // doing both groups' rows, with two CTAs per SM), then the token producer.
  static constexpr int kDecWarps = k2Cta ? 4 : 8;
  static constexpr int kTokWarp = 6 + kDecWarps;
  // The NVFP4 gate/up GEMMs issue the up projection's MMAs from a second thread, in a warp of
  // its own after the others (on another SMSP than warp 1), and the 64-row down projection the
  // second 64-k half of every stage: the token stage and the accumulator then count two
  // commits, and a decoded-weight slot the commits of the issuers that read it.  (The 16-bit
  // GEMMs, paced by HBM, measured slower with two issuers.)
  static constexpr bool kDual = kW4 && (kGemm1 || kKHalves);
  static constexpr int kIssuers = kDual ? 2 : 1;
  static constexpr int kSlotReaders = kKHalves ? 1 : kIssuers;
  static constexpr int kMma2Warp = kTokWarp + 1;
  static constexpr int kThreads = kW4 ? 32 * (kTokWarp + 1 + (kDual ? 1 : 0)) : 192;
  static constexpr int kMinBlocks = k2Cta ? 2 : 1;
  // Warps that write each decoded-weight slot: gemm1 slots hold both slabs (two groups).
  static constexpr int kSlotWriters = (kGemm1 && !k2Cta) ? 8 : 4;
  static constexpr int kSmemBytes = kRingBytes + kStagingBytes + 1024;
  static_assert(!kW4 || kABase + kAStages * kASlotCols <= kTmemTotal, "TMEM columns");
  static_assert(!k2Cta || kSmemBytes <= 110 * 1024, "shared memory of two CTAs per SM");
  static_assert(kStageBytes % 1024 == 0 && kABytes % 1024 == 0 && kWBytes % 1024 == 0 &&
                    kBBytes % 1024 == 0,
                "swizzle-atom alignment");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

struct KParams {
  int mode;
  int token_rows;  // sorted gemm1 with T <= 128: the token side is every row of hidden_states
  int act;         // gemm1: moe_activation_t
  int gated;       // gemm1: second weight tile is the up projection (else the next 128 rows)
  int slab_rows;   // weight rows (output columns) a unit covers: 128, or 256 for ReLU2 gemm1
  int second_off;  // gemm1: row offset of the second weight tile (F gated, 128 ReLU2)
  int K, n_out, E, n_slabs, num_kb, w_rows_per_expert;
  // NVFP4 weights: packed tiles (moe_nvfp4_pack) and the per-expert FP32 scale
  const uint8_t* w4;
  const float* alpha;
  const Tile* tiles;
  const int* n_tiles;
  const int32_t* sorted_ids;
  const int32_t* topk_ids;
  const float* topk_w;
  int P, top_k, T, dense_rows;
  // Sorted mode, bf16/f16 weights: before waiting for the previous kernel, the CTA pulls the
  // first `prefetch_steps` K steps of weights of its first units into L2.  Only set when the
  // tile list was written at least two launches earlier (it is then complete when this kernel
  // starts).
  int prefetch_steps;
  // 16-bit gate/up GEMM over token rows: the router's ids (GemmCall::route_ids).
  const int32_t* route_ids;
  // NVFP4 gate/up GEMM: split-K in two halves when it shortens the last wave (GemmCall).
  int split_cap, split_cols;
  float* split_part;
  int* split_cnt;
  void* out;
  int* status;
  uint64_t limit_ns;
};

struct Unit {
  int e, row0, nrows, n_mma, slab;
  int b_row0;    // first token-side row the unit loads
  bool two;      // gemm1: the second weight tile is used (always when gated)
  int kb0, kb1;  // K steps [kb0, kb1) of this piece of work
  int part;      // split-K: index of this half's partial accumulators (-1: no split)
};

__device__ __forceinline__ int round16(int n) { return (n + 15) & ~15; }

template <bool kGemm1, int kN>
__device__ __forceinline__ bool decode_unit(const KParams& p, int u, Unit& U) {
  if (p.mode == kSorted) {
    // Units of expert e occupy [n_slabs*first, n_slabs*(first+count)), ordered slab-major:
    // the `count` tiles of one (expert, weight slab) are adjacent, so they run at the same time
    // on neighbouring CTAs and can share the slab's weights through L2.  Tile u / n_slabs
    // always lies in the range of the unit's expert.
    const Tile owner = p.tiles[u / p.n_slabs];
    const int local = u - p.n_slabs * owner.first;
    U.slab = local / owner.count;
    const Tile t = p.tiles[owner.first + local % owner.count];
    U.e = t.e;
    U.row0 = t.row0;
    U.nrows = t.nrows;
  } else if (p.mode == kDense) {
    // One expert over all rows, slab-major: the row tiles of a weight slab are adjacent.
    const int n_tiles = (p.dense_rows + kN - 1) / kN;
    U.slab = u / n_tiles;
    U.e = 0;
    U.row0 = (u % n_tiles) * kN;
    U.nrows = min(kN, p.dense_rows - U.row0);
  } else {
    U.slab = u % p.n_slabs;
    const int q = u / p.n_slabs;
    const int e = p.topk_ids[q];
    if (e < 0 || e >= p.E) {
      if (e != -1) set_status(p.status, MOE_ERR_BAD_EXPERT_ID);
      return false;
    }
    for (int r = 0; r < q; ++r)
      if (p.topk_ids[r] == e) return false;  // owned by an earlier route
    U.e = e;
    U.row0 = 0;
    U.nrows = kGemm1 ? p.T : p.P;
  }
  U.b_row0 = U.row0;
  U.n_mma = round16(U.nrows);
  U.two = kGemm1 && (p.gated || U.slab * p.slab_rows + kSlab < p.n_out);
  if (kGemm1 && p.token_rows) {  // load all T token rows; the epilogue picks each row's token
    U.b_row0 = 0;
    U.n_mma = round16(p.T);
  }
  return U.nrows > 0;
}

// Work item u of ks per unit (ks = 2: split-K; item 2v runs K steps [0, num_kb/2) of unit v and
// item 2v+1 the rest).
template <bool kGemm1, int kN>
__device__ __forceinline__ bool decode_item(const KParams& p, int u, int ks, Unit& U) {
  const bool split = ks == 2;
  if (!decode_unit<kGemm1, kN>(p, split ? (u >> 1) : u, U)) return false;
  U.kb0 = 0;
  U.kb1 = p.num_kb;
  U.part = -1;
  if (split) {
    const int mid = p.num_kb >> 1;
    if (u & 1)
      U.kb0 = mid;
    else
      U.kb1 = mid;
    U.part = u;
  }
  return true;
}

// decode_item for the roles that run before the sort has finished (gate/up over token rows):
// unit v is slab v % n_slabs of the (v / n_slabs)-th routed expert in `emask`, the bitmask of
// the experts the router chose, because the sort's tile list holds one tile per routed expert
// in expert order.  These roles need neither the unit's rows nor its position in the sorted
// order; the epilogue reads those from the tile list after its dependency wait.
template <bool kGemm1, int kN>
__device__ __forceinline__ bool decode_item_routed(const KParams& p, const uint32_t* emask, int u,
                                                   int ks, Unit& U) {
  const bool split = ks == 2;
  const int v = split ? (u >> 1) : u;
  const int rank = v / p.n_slabs;
  int word = 0, seen = 0;
  while (word < 32 && seen + __popc(emask[word]) <= rank) seen += __popc(emask[word++]);
  if (word == 32) return false;
  uint32_t m = emask[word];
  for (int i = seen; i < rank; ++i) m &= m - 1;  // drop the lower routed experts of the word
  U.e = word * 32 + __ffs(m) - 1;
  U.slab = v % p.n_slabs;
  U.row0 = 0;
  U.nrows = p.T;
  U.b_row0 = 0;
  U.n_mma = round16(p.T);
  U.two = kGemm1 && (p.gated || U.slab * p.slab_rows + kSlab < p.n_out);
  U.kb0 = 0;
  U.kb1 = p.num_kb;
  U.part = -1;
  if (split) {
    const int mid = p.num_kb >> 1;
    if (u & 1)
      U.kb0 = mid;
    else
      U.kb1 = mid;
    U.part = u;
  }
  return true;
}

// Split-K cost model of the NVFP4 gate/up GEMM over at most 64 token rows, in K steps per CTA:
// a whole unit costs its num_kb steps plus kSplitWholeOver, a half its num_kb/2 plus
// kSplitHalfOver (the extra epilogue and the exchange of partials), fitted to timings of both
// forms on GB300 at one CTA per SM (DeepSeek-V3 EP8 shard, T = 32: 56 K steps a unit, 224 units
// on 152 SMs, 135 us whole, 108 us split; Qwen3-30B-A3B, T = 32: 16 K steps, 660 units, where
// the model keeps whole units).  With two CTAs per SM it counts CTAs: the EP8 shard's 224 units
// then fit one round of 304 CTAs and stay whole (72 us, against 77 us split).
constexpr int kSplitWholeOver = 3;
constexpr int kSplitHalfOver = 4;

__host__ __device__ inline bool split_pays(int n, int ctas, int num_kb) {
  if (n <= 0 || ctas <= 0 || num_kb < 2) return false;
  const int whole = (n + ctas - 1) / ctas, halves = (2 * n + ctas - 1) / ctas;
  return halves * (num_kb + 2 * kSplitHalfOver) < whole * (2 * num_kb + 2 * kSplitWholeOver);
}

// GELU, tanh form: g/2 * (1 + tanh(sqrt(2/pi) * (g + 0.044715 g^3))), in f32.
__device__ __forceinline__ float gelu_tanh_f32(float g) {
  const float u = 0.7978845608028654f * (g + 0.044715f * g * g * g);
  return 0.5f * g * (1.0f + tanhf(u));
}

// Plain bounded wait (ignores the abort flag and the wait-limit knob) used while draining the
// copies and MMAs a CTA has in flight before it frees TMEM and exits; they finish in
// microseconds, so one second is only a backstop.
constexpr uint64_t kDrainLimitNs = 1000000000ull;
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kDrainLimitNs) return;
  }
}

// kBal: the units are spread evenly over balanced_ctas(units, gridDim.x) CTAs (decode-sized
// launches); otherwise every CTA takes units c, c + gridDim.x, ...  kRouted: the NVFP4 gate/up
// kernel for token rows, whose roles may take their units from the router's ids (the 16-bit
// kernels decide at run time; the NVFP4 loops measured 1 % slower with that branch in them).
template <bool kGemm1, int kN, typename T, bool kW4, bool kBal, bool kRouted = false,
          bool k2Cta = false>
__global__ void __launch_bounds__(Cfg<kGemm1, kN, kW4, k2Cta>::kThreads,
                                  Cfg<kGemm1, kN, kW4, k2Cta>::kMinBlocks)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmW,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmB64,
                    const __grid_constant__ CUtensorMap tmB128, const KParams p) {
  using C = Cfg<kGemm1, kN, kW4, k2Cta>;
  // Split-K is built into the NVFP4 gate/up kernel for at most 64 token rows only: the other
  // kernels keep K loops with compile-time bounds.
  constexpr bool kSplit = kW4 && kGemm1 && kN <= 64;
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[C::kFullBars];   // NVFP4: the token ring
  __shared__ __align__(8) uint64_t empty_bar[C::kFullBars];
  __shared__ __align__(8) uint64_t tfull_bar[C::kAccBufs];
  __shared__ __align__(8) uint64_t tempty_bar[C::kAccBufs];
  __shared__ __align__(8) uint64_t drain_bar[2];  // one per MMA issuer
  __shared__ __align__(8) uint64_t afull_bar[C::kAStages];   // NVFP4: decoded slot ready
  __shared__ __align__(8) uint64_t aempty_bar[C::kAStages];  // NVFP4: slot consumed by the MMA
  __shared__ __align__(8) uint64_t wfull_bar[kW4 ? C::kNW : 1];   // NVFP4: weights landed
  __shared__ __align__(8) uint64_t wempty_bar[kW4 ? C::kNW : 1];  // NVFP4: weights decoded
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  __shared__ int s_n_units;
  __shared__ int s_ks;          // work items per unit (2: split-K)
  __shared__ int s_split_last;  // epilogue: this half finished the unit second
  __shared__ uint32_t s_emask[(kGemm1 && (!kW4 || kRouted)) ? 32 : 1];  // routed experts
  __shared__ int ent_col[kGemm1 ? kN : 1];
  __shared__ int ent_dst[kN];
  __shared__ float col_scale[kGemm1 ? 1 : kN];

  // 1024-byte alignment for the 128-byte swizzle atoms.
  const uint32_t raw = smem_u32(dsmem);
  uint8_t* smem = dsmem + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* staging = smem + C::kRingBytes;
  uint8_t* tring = smem + (kW4 ? C::kNW * C::kWBytes : 0);  // NVFP4 token ring
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &s_abort;

  // Prologue that touches no global memory: it overlaps the previous kernel's tail.
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kFullBars; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], C::kIssuers);  // freed by every MMA issuer's commit
    }
    if (kW4) {
      for (int s = 0; s < C::kNW; ++s) {
        mbar_init(&wfull_bar[s], 1);
        mbar_init(&wempty_bar[s], C::kDecWarps);  // one arrival per decoder warp
      }
      for (int a = 0; a < C::kAStages; ++a) {
        mbar_init(&afull_bar[a], C::kSlotWriters);  // the warps that write the slot
        mbar_init(&aempty_bar[a], C::kSlotReaders);
      }
    }
    for (int a = 0; a < C::kAccBufs; ++a) {
      mbar_init(&tfull_bar[a], C::kIssuers);
      mbar_init(&tempty_bar[a], 128);
    }
    mbar_init(&drain_bar[0], 1);
    mbar_init(&drain_bar[1], 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmW);
    prefetch_tensormap(&tmB);
    prefetch_tensormap(&tmB64);
    prefetch_tensormap(&tmB128);
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  if constexpr (!kW4) {
    // The previous kernel may still be running on other SMs (this grid starts as its CTAs
    // finish): stream the first units' weights into L2 meanwhile.  They depend on nothing that
    // kernel writes.
    if (p.prefetch_steps > 0 && p.mode == kSorted && threadIdx.x == 0) {
      const int n = (*p.n_tiles) * p.n_slabs;
      const int G = kBal ? balanced_ctas(n, gridDim.x) : (int)gridDim.x;  // as below
      int left = p.prefetch_steps;
      for (int u = blockIdx.x < G ? blockIdx.x : n; u < n && left > 0; u += G) {
        Unit U;
        if (!decode_unit<kGemm1, kN>(p, u, U)) continue;
        const int wrow = U.e * p.w_rows_per_expert + U.slab * p.slab_rows;
        for (int kb = 0; kb < p.num_kb && left > 0; ++kb, --left) {
          tma_prefetch_l2_2d(&tmW, kb * kBlockK, wrow);
          if (kGemm1 && U.two) tma_prefetch_l2_2d(&tmW, kb * kBlockK, wrow + p.second_off);
        }
      }
    }
  }
  // 16-bit gate/up over token rows: the units follow from the router's ids, so only the
  // epilogue waits for the sort (below); the router finished before the sort released this
  // grid, and the ids are read from L2.
  const bool routed =
      (!kW4 || kRouted) && kGemm1 && p.route_ids != nullptr && p.mode == kSorted;
  const uint32_t* emask = routed ? s_emask : nullptr;
  if (routed) {
    if (warp == 0) {
      s_emask[lane] = 0u;
      __syncwarp();
      for (int r = lane; r < p.P; r += 32) {
        const int e = __ldcg(p.route_ids + r);
        if (e >= 0 && e < p.E) atomicOr(&s_emask[e >> 5], 1u << (e & 31));
      }
      __syncwarp();
    }
  } else {
    pdl_wait();
    pdl_trigger();
  }
  if (threadIdx.x == 0) {
    int n = 0;
    if (routed) {
      int active = 0;
      for (int i = 0; i < 32; ++i) active += __popc(s_emask[i]);
      n = active * p.n_slabs;
    } else if (p.mode == kSorted)
      n = (*p.n_tiles) * p.n_slabs;
    else if (p.mode == kDirect)
      n = p.P * p.n_slabs;
    else
      n = ((p.dense_rows + kN - 1) / kN) * p.n_slabs;
    // NVFP4 gate/up: split every unit's K range in two when, by the cost model, the halves end
    // the last wave sooner than whole units would (the MMA issue rate, not HBM, paces these
    // kernels, so an SM left idle is time lost).
    int ks = 1;
    if (kSplit && p.split_cap > 0 && n <= p.split_cap && split_pays(n, gridDim.x, p.num_kb))
      ks = 2;
    s_ks = ks;
    s_n_units = n * ks;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  const int n_units = s_n_units;       // work items
  const int ks = kSplit ? s_ks : 1;
  // CTAs that take units (the stride) and this CTA's first unit.  At decode sizes (kBal) the
  // 16-bit weights stream at HBM speed, so the units are spread evenly over as few CTAs as keep
  // the per-CTA share.  Otherwise the loops read the stride from gridDim directly: held in a
  // register instead, it measured 3 % slower at prefill sizes and 14 % slower in the NVFP4
  // kernels (same register counts).
  const int G = balanced_ctas(n_units, gridDim.x);
  const int u0 = blockIdx.x < G ? (int)blockIdx.x : n_units;
#define UNIT_FIRST (kBal ? u0 : (int)blockIdx.x)
#define UNIT_STRIDE (kBal ? G : (int)gridDim.x)

  if (kW4 && warp == 0) {
    // ---------------------------------------------- NVFP4 weight producer (one lane)
    // One bulk copy per slab and stage: the tile of (expert, 128 rows, 128 k) is contiguous.
    if (lane == 0) {
      int ws = 0;
      uint32_t wph = 0;
      int issued = 0;
      bool ok = true;
      const int64_t slabs_per_expert = p.w_rows_per_expert / kSlab;
      for (int u = UNIT_FIRST; u < n_units && ok; u += UNIT_STRIDE) {
        Unit U;
        if (!(routed ? decode_item_routed<kGemm1, kN>(p, emask, u, ks, U)
                     : decode_item<kGemm1, kN>(p, u, ks, U)))
          continue;
        const int n_w = U.two ? 2 : 1;
        const int64_t t0 = ((int64_t)U.e * slabs_per_expert + U.slab * p.slab_rows / kSlab) *
                           p.num_kb;
        const int64_t t1 = t0 + (int64_t)(p.second_off / kSlab) * p.num_kb;
        for (int kb = U.kb0; kb < U.kb1; ++kb) {
          if (!mbar_wait(&wempty_bar[ws], wph ^ 1u, abort_flag, p.limit_ns, p.status)) {
            ok = false;
            break;
          }
          uint8_t* sw = smem + ws * C::kWBytes;
          mbar_arrive_expect_tx(&wfull_bar[ws], n_w * C::kTileBytes);
          bulk_load(sw, p.w4 + (t0 + kb) * C::kTileBytes, C::kTileBytes, &wfull_bar[ws]);
          if (kGemm1 && U.two)
            bulk_load(sw + C::kTileBytes, p.w4 + (t1 + kb) * C::kTileBytes, C::kTileBytes,
                      &wfull_bar[ws]);
          ++issued;
          if (++ws == C::kNW) {
            ws = 0;
            wph ^= 1u;
          }
        }
      }
      if (*abort_flag) {
        const int n = issued < C::kNW ? issued : C::kNW;
        for (int i = issued - n; i < issued; ++i)
          mbar_wait_drain(&wfull_bar[i % C::kNW], (uint32_t)((i / C::kNW) & 1));
      }
    }
  } else if (kW4 && warp == C::kTokWarp) {
    // ---------------------------------------------- NVFP4 token producer (one lane)
    if (lane == 0) {
      int ts = 0;
      uint32_t tph = 0;
      int issued = 0;
      bool ok = true;
      for (int u = UNIT_FIRST; u < n_units && ok; u += UNIT_STRIDE) {
        Unit U;
        if (!(routed ? decode_item_routed<kGemm1, kN>(p, emask, u, ks, U)
                     : decode_item<kGemm1, kN>(p, u, ks, U)))
          continue;
        for (int kb = U.kb0; kb < U.kb1; ++kb) {
          if (!mbar_wait(&empty_bar[ts], tph ^ 1u, abort_flag, p.limit_ns, p.status)) {
            ok = false;
            break;
          }
          uint8_t* sb = tring + ts * C::kBBytes;
          mbar_arrive_expect_tx(&full_bar[ts], U.n_mma * C::kStageK * 2);
#pragma unroll
          for (int a = 0; a < C::kStageK / kBlockK; ++a) {
            uint8_t* sba = sb + a * kN * kBlockK * 2;
            const int kx = kb * C::kStageK + a * kBlockK;
            int r = 0;
            for (; r + 128 <= U.n_mma; r += 128)
              tma_load_2d(sba + r * kBlockK * 2, &tmB128, &full_bar[ts], kx, U.b_row0 + r);
            for (; r + 64 <= U.n_mma; r += 64)
              tma_load_2d(sba + r * kBlockK * 2, &tmB64, &full_bar[ts], kx, U.b_row0 + r);
            for (; r < U.n_mma; r += 16)
              tma_load_2d(sba + r * kBlockK * 2, &tmB, &full_bar[ts], kx, U.b_row0 + r);
          }
          ++issued;
          if (++ts == C::kNT) {
            ts = 0;
            tph ^= 1u;
          }
        }
      }
      if (*abort_flag) {
        const int n = issued < C::kNT ? issued : C::kNT;
        for (int i = issued - n; i < issued; ++i)
          mbar_wait_drain(&full_bar[i % C::kNT], (uint32_t)((i / C::kNT) & 1));
      }
    }
  } else if (kW4 && warp >= 6 && warp < 6 + C::kDecWarps) {
    // ------------------------------------------------------- NVFP4 decoders (8 or 4 warps)
    // Warp w owns TMEM lanes 32*(w%4)..+31, i.e. weight rows of the slab.  Two groups of work:
    // gemm1: group g decodes slab g (gate, up) into columns 32g..32g+31 of each 64-k ring slot;
    // gemm2: group g decodes k 64g..64g+63 of the stage into its own slot.  With eight decoder
    // warps, warps 6-9 are group 0 and 10-13 group 1; with four (two CTAs per SM) every warp
    // does both.  A thread decodes one weight row: 16-byte chunks of 32 codes, two scales
    // each.  Stores are pipelined: a slot's tcgen05.st is waited for and the slot handed to the
    // MMA only after the next slot's first decode, so the store latency hides behind ALU work.
    constexpr int kG = C::kDecWarps == 4 ? 2 : 1;  // groups per warp
    const int g0 = kG == 2 ? 0 : (warp - 6) >> 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
    int ws = 0;
    uint32_t wph = 0;
    int a_cnt = 0;
    int pending = -1;  // ring slot whose store is in flight
    bool ok = true;
    auto hand_over = [&](int slot) {  // make this warp's part of `slot` visible to the MMA
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&afull_bar[slot]);
    };
    for (int u = UNIT_FIRST; u < n_units && ok; u += UNIT_STRIDE) {
      Unit U;
      if (!(routed ? decode_item_routed<kGemm1, kN>(p, emask, u, ks, U)
                   : decode_item<kGemm1, kN>(p, u, ks, U)))
        continue;
      for (int kb = U.kb0; kb < U.kb1; ++kb) {
        if (!mbar_wait(&wfull_bar[ws], wph, abort_flag, p.limit_ns, p.status)) {
          ok = false;
          break;
        }
        const uint8_t* wslot = smem + ws * C::kWBytes;
        // the row's block scales in each slab this warp decodes (gemm2: one slab)
        constexpr int kSc = kGemm1 ? kG : 1;
        uint32_t s2[kSc][8];
#pragma unroll
        for (int i = 0; i < kSc; ++i) {
          const uint8_t* tile = wslot + (kGemm1 ? g0 + i : 0) * C::kTileBytes;
          const uint2 sfw = *reinterpret_cast<const uint2*>(tile + C::kQBytes + row * 8);
          nvfp4_scales(sfw.x, *reinterpret_cast<uint32_t(*)[4]>(&s2[i][0]));
          nvfp4_scales(sfw.y, *reinterpret_cast<uint32_t(*)[4]>(&s2[i][4]));
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          // gemm1: every group writes half hh of the stage; gemm2: only group hh does.
          if (!kGemm1 && kG == 1 && hh != g0) continue;
          const int idx = a_cnt + hh;
          const int slot = idx % C::kAStages;
          if (!mbar_wait(&aempty_bar[slot], (uint32_t)(((idx / C::kAStages) & 1) ^ 1),
                         abort_flag, p.limit_ns, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          bool stored = false;
#pragma unroll
          for (int gi = 0; gi < kG; ++gi) {
            const int g = g0 + gi;
            if (!kGemm1 && g != hh) continue;
            if (kGemm1 && g == 1 && !U.two) continue;  // no second slab: nothing to decode
            const int slab = kGemm1 ? g : 0;
            const uint32_t* sc = s2[kGemm1 ? gi : 0];
            const uint8_t* qrow = wslot + slab * C::kTileBytes + row * 64;
            uint32_t v[32];
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              const int j = 2 * hh + jj;  // 32-k chunk of the stage
              // packed layout: chunk j of row r sits at chunk j ^ ((r >> 1) & 3)
              const uint4 qw =
                  *reinterpret_cast<const uint4*>(qrow + ((j ^ ((row >> 1) & 3)) << 4));
              nvfp4_decode8(qw.x, sc[2 * j], *reinterpret_cast<uint32_t(*)[4]>(&v[16 * jj]));
              nvfp4_decode8(qw.y, sc[2 * j], *reinterpret_cast<uint32_t(*)[4]>(&v[16 * jj + 4]));
              nvfp4_decode8(qw.z, sc[2 * j + 1],
                            *reinterpret_cast<uint32_t(*)[4]>(&v[16 * jj + 8]));
              nvfp4_decode8(qw.w, sc[2 * j + 1],
                            *reinterpret_cast<uint32_t(*)[4]>(&v[16 * jj + 12]));
            }
            if (pending >= 0) {  // the previous store has had a whole decode to land
              tmem_wait_st();
              hand_over(pending);
              pending = -1;
            }
            const uint32_t col =
                (uint32_t)(C::kABase + slot * C::kASlotCols + (kGemm1 ? slab * 32 : 0));
            tmem_st_x32(tmem_base + lane_addr + col, v);
            stored = true;
          }
          if (stored)
            pending = slot;
          else
            hand_over(slot);
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&wempty_bar[ws]);  // this warp has read the weight slot
        a_cnt += 2;
        if (++ws == C::kNW) {
          ws = 0;
          wph ^= 1u;
        }
      }
    }
    if (pending >= 0) {  // the last store (also on the way out after a timeout)
      tmem_wait_st();
      if (ok) hand_over(pending);
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int u = UNIT_FIRST; u < n_units && ok; u += UNIT_STRIDE) {
        Unit U;
        if (!(routed ? decode_item_routed<kGemm1, kN>(p, emask, u, ks, U)
                     : decode_item<kGemm1, kN>(p, u, ks, U)))
          continue;
        const uint32_t wbytes = U.two ? 2 * kSlab * kBlockK * 2 : kSlab * kBlockK * 2;
        const uint32_t bytes = wbytes + U.n_mma * kBlockK * 2;  // per 64-k block
        const int wrow = U.e * p.w_rows_per_expert + U.slab * p.slab_rows;
        for (int kb = 0; kb < p.num_kb; kb += C::kKps) {
          const int nsub = p.num_kb - kb < C::kKps ? p.num_kb - kb : C::kKps;
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, p.limit_ns, p.status)) {
            ok = false;
            break;
          }
          uint8_t* sa0 = smem + stage * C::kStageBytes;
          mbar_arrive_expect_tx(&full_bar[stage], bytes * nsub);
#pragma unroll
          for (int j = 0; j < C::kKps; ++j) {
            if (j >= nsub) break;
            uint8_t* sa = sa0 + j * C::kASubBytes;
            uint8_t* sb = sa0 + C::kABytes + j * C::kBSubBytes;
            const int kx = (kb + j) * kBlockK;
            tma_load_2d(sa, &tmW, &full_bar[stage], kx, wrow);
            if (kGemm1 && U.two)
              tma_load_2d(sa + kSlab * kBlockK * 2, &tmW, &full_bar[stage], kx,
                          wrow + p.second_off);
            // Token rows in as few copies as possible: 128-, then 64-, then 16-row boxes.
            int r = 0;
            for (; r + 128 <= U.n_mma; r += 128)
              tma_load_2d(sb + r * kBlockK * 2, &tmB128, &full_bar[stage], kx, U.b_row0 + r);
            for (; r + 64 <= U.n_mma; r += 64)
              tma_load_2d(sb + r * kBlockK * 2, &tmB64, &full_bar[stage], kx, U.b_row0 + r);
            for (; r < U.n_mma; r += 16)
              tma_load_2d(sb + r * kBlockK * 2, &tmB, &full_bar[stage], kx, U.b_row0 + r);
          }
          ++issued;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort_flag) {
        // Let every copy still in flight land before the CTA goes away.
        const int n = issued < C::kStages ? issued : C::kStages;
        for (int i = issued - n; i < issued; ++i)
          mbar_wait_drain(&full_bar[i % C::kStages], (uint32_t)((i / C::kStages) & 1));
      }
    }
  } else if (warp == 1 || (C::kDual && warp == C::kMma2Warp)) {
    // ------------------------------------------------------------------ MMA issuer(s)
    // kDual: warp 1 issues the gate (first slab) MMAs and warp kMma2Warp the up (second slab)
    // ones, or (kKHalves) the first and the second 64-k half of every stage, each into its own
    // accumulator; both wait for the same token stages and commit to the barriers they free.
    const bool upper = C::kDual && warp != 1;
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int a_cnt = 0;  // NVFP4: TMEM ring slots consumed so far
      bool ok = true;
      bool issued_any = false;
      const uint32_t smem_base = smem_u32(smem);
      for (int u = UNIT_FIRST; u < n_units && ok; u += UNIT_STRIDE) {
        Unit U;
        if (!(routed ? decode_item_routed<kGemm1, kN>(p, emask, u, ks, U)
                     : decode_item<kGemm1, kN>(p, u, ks, U)))
          continue;
        if (!mbar_wait(&tempty_bar[acc], acc_phase ^ 1u, abort_flag, p.limit_ns, p.status)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * C::kAccCols);
        const uint32_t idesc = idesc_f16_m128(U.n_mma, DT<T>::kIsBF16);
        for (int kb = U.kb0; kb < U.kb1; kb += C::kKps) {  // NVFP4: kKps = 1, 128-k stages
          if (!mbar_wait(&full_bar[stage], phase, abort_flag, p.limit_ns, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_base + (uint32_t)(stage * C::kStageBytes);
          const uint32_t sb = sa + C::kABytes;
          if constexpr (kW4) {
            // A (decoded weights) from two TMEM ring slots of 64 k each; B: the token slot.  The
            // descriptor of a 64-k half of the token slot is the slot's plus (half offset) / 16.
            const uint64_t tdesc = sw128_kmajor_desc(
                smem_base + (uint32_t)(C::kNW * C::kWBytes + stage * C::kBBytes));
            const bool two = kGemm1 && U.two;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              if (C::kKHalves && (hh != 0) != upper) continue;  // the other issuer's half
              const int idx = a_cnt + hh;
              const int slot = idx % C::kAStages;
              if (!mbar_wait(&afull_bar[slot], (uint32_t)((idx / C::kAStages) & 1), abort_flag,
                             p.limit_ns, p.status)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t a = tmem_base + (uint32_t)(C::kABase + slot * C::kASlotCols);
              const uint64_t bdesc = tdesc + (uint64_t)(hh * (kN * kBlockK * 2 / 16));
              const uint32_t accum = (kb != U.kb0 || (hh != 0 && !C::kKHalves)) ? 1u : 0u;
              if (C::kKHalves) {
                umma_tmem_a_kblock(d + (uint32_t)(hh * kN), a, bdesc, idesc, accum);
                issued_any = true;
              } else if (!C::kDual) {
                if (two)
                  umma_tmem_a_kblock2(d, a, d + kN, a + 32, bdesc, idesc, accum);
                else
                  umma_tmem_a_kblock(d, a, bdesc, idesc, accum);
                issued_any = true;
              } else if (!upper) {
                umma_tmem_a_kblock(d, a, bdesc, idesc, accum);
                issued_any = true;
              } else if (two) {
                umma_tmem_a_kblock(d + kN, a + 32, bdesc, idesc, accum);
                issued_any = true;
              }
              umma_commit(&aempty_bar[slot]);
            }
            if (!ok) break;
            a_cnt += 2;
            umma_commit(&empty_bar[stage]);
            if (++stage == C::kFullBars) {
              stage = 0;
              phase ^= 1u;
            }
          } else {
            const int nsub = U.kb1 - kb < C::kKps ? U.kb1 - kb : C::kKps;
#pragma unroll
            for (int j = 0; j < C::kKps; ++j) {
              if (j >= nsub) break;
              const uint32_t aj = sa + (uint32_t)(j * C::kASubBytes);
              const uint32_t bj = sb + (uint32_t)(j * C::kBSubBytes);
#pragma unroll
              for (int k = 0; k < kBlockK / 16; ++k) {
                const uint64_t bdesc = sw128_kmajor_desc(bj + k * 32);
                const uint32_t accum = (kb | j | k) != 0 ? 1u : 0u;
                if (!upper) umma_f16(d, sw128_kmajor_desc(aj + k * 32), bdesc, idesc, accum);
                if (kGemm1 && U.two && (upper || !C::kDual))
                  umma_f16(d + kN, sw128_kmajor_desc(aj + kSlab * kBlockK * 2 + k * 32), bdesc,
                           idesc, accum);
              }
            }
            umma_commit(&empty_bar[stage]);
            issued_any |= !upper || (kGemm1 && U.two);
            if (++stage == C::kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!ok) break;
        umma_commit(&tfull_bar[acc]);
        if (++acc == C::kAccBufs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // Every MMA issued by this thread has completed once its drain barrier flips.
      if (issued_any) {
        umma_commit(&drain_bar[upper ? 1 : 0]);
        mbar_wait_drain(&drain_bar[upper ? 1 : 0], 0);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue (128 thr)
    const int q = warp & 3;  // the TMEM lane quarter this warp may read
    const int row = q * 32 + lane;
    const int et = threadIdx.x - 64;
    int acc = 0;
    uint32_t acc_phase = 0;
    if (routed) {
      // The tile list and the sorted ids come from the sort.  Dependents are released only
      // after this wait: the next kernel may read what the sort wrote before its own wait.
      pdl_wait();
      pdl_trigger();
    }
    for (int u = UNIT_FIRST; u < n_units; u += UNIT_STRIDE) {
      Unit U;
      if (!decode_item<kGemm1, kN>(p, u, ks, U)) continue;
      // NVFP4: the expert's FP32 scale multiplies the FP32 accumulator (before the activation)
      const float al = kW4 ? p.alpha[U.e] : 1.0f;
      if constexpr (kGemm1) {
        // Output rows of this unit as (accumulator column, destination row) entries.  In direct
        // mode a column is a token and each route of that token to this expert is an entry; with
        // token_rows a column is a token and sorted row p reads the column of its route's token.
        const bool direct = p.mode == kDirect;
        const bool by_token = direct || p.token_rows;
        const int n_ent = direct ? p.P : U.nrows;
        for (int i = et; i < n_ent; i += 128) {
          if (direct) {
            ent_col[i] = p.topk_ids[i] == U.e ? i / p.top_k : -1;
            ent_dst[i] = i;
          } else if (p.token_rows) {
            const int sid = p.sorted_ids[U.row0 + i];
            ent_col[i] = sid >= 0 ? sid / p.top_k : -1;
            ent_dst[i] = U.row0 + i;
          } else {
            ent_col[i] = i;
            ent_dst[i] = U.row0 + i;
          }
        }
        const bool got = mbar_wait(&tfull_bar[acc], acc_phase, abort_flag, p.limit_ns, p.status);
        if (!named_bar_and(1, 128, got)) break;
        tc_fence_after();
        const uint32_t tb =
            tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * C::kAccCols);
        const float* other = nullptr;  // split-K: the other half's accumulators
        if constexpr (kW4) {
          if (U.part >= 0) {
            // Store both accumulators (f32, column-major: a warp writes 128 bytes per column),
            // then count this half in.  The half that comes second adds the first one's
            // partials to its own: a + b is the same either way round, so the result does not
            // depend on which half finished first.
            const int64_t stride = (int64_t)2 * p.split_cols * kSlab;  // floats per half
            float* mine = p.split_part + (int64_t)U.part * stride;
            for (int c = 0; c < U.n_mma; c += 16) {
              float g[16], v[16];
              tmem_ld2_x16(tb + c, tb + kN + c, g, v);
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                __stcg(mine + (int64_t)(c + j) * kSlab + row, g[j]);
                __stcg(mine + (int64_t)(p.split_cols + c + j) * kSlab + row, v[j]);
              }
            }
            __threadfence();
            named_bar_sync(1, 128);
            if (et == 0) s_split_last = atomicAdd(&p.split_cnt[U.part >> 1], 1);
            named_bar_sync(1, 128);
            if (s_split_last == 0) {  // the other half writes the unit's output
              tc_fence_before();
              mbar_arrive(&tempty_bar[acc]);
              if (++acc == C::kAccBufs) {
                acc = 0;
                acc_phase ^= 1u;
              }
              continue;
            }
            __threadfence();
            other = p.split_part + (int64_t)(U.part ^ 1) * stride;
          }
        }
        T* stg = reinterpret_cast<T*>(staging);
        T* out = static_cast<T*>(p.out);
        const int n_halves = p.gated ? 1 : (U.two ? 2 : 1);
        for (int half = 0; half < n_halves; ++half) {
          const int col0 = U.slab * p.slab_rows + half * kSlab;  // first output column
          const int width = min(kSlab, p.n_out - col0);
          const int nch = width / 8;
          for (int c0 = 0; c0 < U.n_mma; c0 += C::kPassCols) {
            const int c1 = min(U.n_mma, c0 + C::kPassCols);
            for (int c = c0; c < c1; c += 16) {
              float h[16];
              if (p.gated) {
                float g[16], v[16];
                tmem_ld2_x16(tb + c, tb + kN + c, g, v);
                if constexpr (kW4) {
                  if (other) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                      g[j] += __ldcg(other + (int64_t)(c + j) * kSlab + row);
                      v[j] += __ldcg(other + (int64_t)(p.split_cols + c + j) * kSlab + row);
                    }
                  }
#pragma unroll
                  for (int j = 0; j < 16; ++j) {
                    g[j] *= al;
                    v[j] *= al;
                  }
                }
                if (p.act == MOE_ACT_GELU_TANH) {
#pragma unroll
                  for (int j = 0; j < 16; ++j) h[j] = gelu_tanh_f32(g[j]) * v[j];
                } else {
#pragma unroll
                  for (int j = 0; j < 16; ++j)
                    h[j] = __fdividef(g[j], 1.0f + __expf(-g[j])) * v[j];
                }
              } else {
                tmem_ld_x16(tb + (uint32_t)(half * kN) + c, h);
                if constexpr (kW4) {
                  if (other) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                      h[j] += __ldcg(other + (int64_t)(half * p.split_cols + c + j) * kSlab + row);
                  }
                }
                if (p.act == kActIdentity) {
#pragma unroll
                  for (int j = 0; j < 16; ++j) h[j] *= al;
                } else {
#pragma unroll
                  for (int j = 0; j < 16; ++j) {
                    const float r = fmaxf(h[j] * al, 0.0f);
                    h[j] = r * r;
                  }
                }
              }
              if constexpr (kW4) {  // the f16 act: a value past the f16 range is an error
                bool over = false;
#pragma unroll
                for (int j = 0; j < 16; ++j) over |= fabsf(h[j]) >= kF16Overflow;
                if (over) set_status(p.status, MOE_ERR_F16_RANGE);
              }
#pragma unroll
              for (int j = 0; j < 16; ++j) stg[(c - c0 + j) * kSlab + row] = DT<T>::from_f(h[j]);
            }
            if (half == n_halves - 1 && c1 == U.n_mma) {  // every TMEM column has been read
              tc_fence_before();
              mbar_arrive(&tempty_bar[acc]);
            }
            named_bar_sync(1, 128);
            // 16-byte stores of whole output rows: entry en, chunk ch of 8 columns.
            const int en_lo = by_token ? 0 : c0, en_hi = by_token ? n_ent : min(n_ent, c1);
            for (int idx = et; idx < (en_hi - en_lo) * 16; idx += 128) {
              const int en = en_lo + (idx >> 4), ch = idx & 15;
              if (ch >= nch) continue;
              const int col = ent_col[en];
              if (col < c0 || col >= c1) continue;
              const uint4 val =
                  *reinterpret_cast<const uint4*>(stg + (col - c0) * kSlab + ch * 8);
              *reinterpret_cast<uint4*>(out + (int64_t)ent_dst[en] * p.n_out + col0 + ch * 8) =
                  val;
            }
            named_bar_sync(1, 128);
          }
        }
      } else {
        // Each accumulator column (token row) goes to at most one f32 output row, scaled by its
        // route weight; thread `row` owns output column slab*128 + row, so a warp stores one
        // 128-byte line per column.
        for (int i = et; i < U.n_mma; i += 128) {
          int dst = -1;
          float sc = 0.0f;
          if (p.mode == kSorted) {
            if (i < U.nrows) {
              dst = U.row0 + i;
              if (p.sorted_ids) {  // a route's row, scaled by its weight; padding rows give 0
                const int sid = p.sorted_ids[dst];
                sc = sid >= 0 ? p.topk_w[sid] : 0.0f;
              } else {  // the plain grouped GEMM
                sc = 1.0f;
              }
            }
          } else if (p.mode == kDirect) {
            if (i < p.P && p.topk_ids[i] == U.e) {
              dst = i;
              sc = p.topk_w[i];
            }
          } else if (i < U.nrows) {
            dst = U.row0 + i;
            sc = 1.0f;
          }
          ent_dst[i] = dst;
          col_scale[i] = sc;
        }
        const bool got = mbar_wait(&tfull_bar[acc], acc_phase, abort_flag, p.limit_ns, p.status);
        if (!named_bar_and(1, 128, got)) break;
        tc_fence_after();
        const uint32_t tb =
            tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * C::kAccCols);
        float* out = static_cast<float*>(p.out);
        const int h = U.slab * kSlab + row;
        const bool in_range = h < p.n_out;
        for (int c0 = 0; c0 < U.n_mma; c0 += 16) {
          float g[16];
          if constexpr (C::kKHalves) {  // the two 64-k halves' accumulators
            float v[16];
            tmem_ld2_x16(tb + c0, tb + kN + c0, g, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) g[j] += v[j];
          } else {
            tmem_ld_x16(tb + c0, g);
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int dst = ent_dst[c0 + j];
            if (dst >= 0 && in_range)
              out[(int64_t)dst * p.n_out + h] = (kW4 ? g[j] * al : g[j]) * col_scale[c0 + j];
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty_bar[acc]);
        named_bar_sync(1, 128);
      }
      if (++acc == C::kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}
#undef UNIT_FIRST
#undef UNIT_STRIDE

// ---- host side -----------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 2-D map over a row-major [rows, inner] 16-bit tensor, box {64, box_rows}, 128-byte swizzle,
// zero fill outside the tensor.
bool make_map(CUtensorMap* m, int dtype, const void* base, uint64_t inner, uint64_t rows,
              uint32_t box_rows) {
  if (!get_encode()) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBlockK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m,
                        dtype == MOE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <bool kGemm1, int kN, typename T, bool kW4, bool kBal = false, bool kRouted = false,
          bool k2Cta = false>
cudaError_t launch_typed(const GemmCall& c, const KParams& kp, int grid, cudaStream_t s,
                         bool pdl) {
  using C = Cfg<kGemm1, kN, kW4, k2Cta>;
  CUtensorMap tmW, tmB, tmB64, tmB128;
  const uint64_t w_rows = (uint64_t)c.E * (uint64_t)kp.w_rows_per_expert;
  // The token rows are of the kernel's 16-bit type (f16 for the NVFP4 kernels, whatever the
  // problem's type); so are 16-bit weights.  NVFP4 weights are read with plain bulk copies: tmW
  // is then a copy of the token map, unused.
  const int tdt = DT<T>::kIsBF16 ? MOE_BF16 : MOE_F16;
  if (!kW4 && !make_map(&tmW, tdt, c.w, (uint64_t)c.K, w_rows, kSlab))
    return cudaErrorInvalidValue;
  if (!make_map(&tmB, tdt, c.b, (uint64_t)c.K, (uint64_t)c.b_rows, 16) ||
      !make_map(&tmB64, tdt, c.b, (uint64_t)c.K, (uint64_t)c.b_rows, 64) ||
      !make_map(&tmB128, tdt, c.b, (uint64_t)c.K, (uint64_t)c.b_rows, 128))
    return cudaErrorInvalidValue;
  if (kW4) tmW = tmB;
  auto kern = moe_gemm_kernel<kGemm1, kN, T, kW4, kBal, kRouted, k2Cta>;
  static bool attr_set = false;  // one per instantiation: set once per process
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_k(kern, dim3(grid), dim3(C::kThreads), C::kSmemBytes, s, pdl, tmW, tmB, tmB64,
                  tmB128, kp);
}

// Decode-sized launch: sorted or direct units of experts that average at most 64 routed rows.
bool decode_sized(const GemmCall& c) {
  if (c.P <= 0 || (c.mode != kSorted && c.mode != kDirect)) return false;
  const int64_t active = c.P < c.E ? c.P : c.E;
  return (int64_t)c.P / active <= 64;
}

template <bool kGemm1, typename T>
cudaError_t launch_rows(const GemmCall& c, const KParams& kp, long long units, cudaStream_t s,
                        bool pdl) {
  const int sms = num_sms();
  const int grid = (int)(units < sms ? units : sms);
  if (c.w4) {
    if constexpr (kGemm1) {
      // At most 64 tokens over token rows, the direct path with at most 64 routes (its epilogue
      // keeps one entry per route, in arrays of the tile's rows), or 32/64-row tiles of gathered
      // rows: two CTAs per SM, split-K (token rows only) when the cost model says it pays.  Up
      // to 32 tokens (routes, tile rows) the tiles have 32 rows: their accumulators take 64 TMEM
      // columns, which leaves three 64-k slots for the decoded weights instead of two.
      const bool gathered = c.mode == kSorted && !kp.token_rows;
      const bool narrow = (kp.token_rows && c.T <= 32) || (c.mode == kDirect && c.P <= 32) ||
                          (gathered && c.tile_rows == kTileRowsNvfp4Min);
      if ((kp.token_rows && c.T <= 64) || (c.mode == kDirect && c.P <= 64) ||
          (gathered && c.tile_rows <= kTileRowsNarrow)) {
        const int grid2 = (int)(units < 2 * sms ? units : 2 * sms);
        if (narrow)
          return launch_typed<true, 32, __half, true, false, true, true>(c, kp, grid2, s, pdl);
        return launch_typed<true, 64, __half, true, false, true, true>(c, kp, grid2, s, pdl);
      }
      if (kp.route_ids)  // token rows: units from the router's ids
        return launch_typed<true, 128, __half, true, false, true>(c, kp, grid, s, pdl);
      return launch_typed<true, 128, __half, true>(c, kp, grid, s, pdl);
    } else {
      // Two CTAs per SM, each with its own MMA issuer: one issuing thread is latency bound
      // and, next to the decoders, reaches well under half the tensor pipe's MMA rate.  With
      // 64-row tiles (and on the direct path with at most 64 routes) the two accumulators of
      // the k halves fit TMEM, and each CTA has two issuers.
      const int grid2 = (int)(units < 2 * sms ? units : 2 * sms);
      if ((c.mode == kSorted && c.tile_rows == kTileRowsNarrow) ||
          (c.mode == kDirect && c.P <= 64))
        return launch_typed<false, 64, __half, true, false, false, true>(c, kp, grid2, s, pdl);
      return launch_typed<false, 128, __half, true, false, false, true>(c, kp, grid2, s, pdl);
    }
  }
  if constexpr (!kGemm1) {  // 64-row tiles are decode tiles: balanced
    if (c.tile_rows == 64) return launch_typed<false, 64, T, false, true>(c, kp, grid, s, pdl);
  }
  if (c.tile_rows == 256) return launch_typed<kGemm1, 256, T, false>(c, kp, grid, s, pdl);
  return decode_sized(c) ? launch_typed<kGemm1, 128, T, false, true>(c, kp, grid, s, pdl)
                         : launch_typed<kGemm1, 128, T, false>(c, kp, grid, s, pdl);
}

}  // namespace

cudaError_t launch_gemm(const GemmCall& c, cudaStream_t s, bool pdl) {
  KParams kp;
  kp.mode = c.mode;
  kp.token_rows = c.gemm1 && c.mode == kSorted && c.token_rows;
  if (c.token_rows && (!kp.token_rows || c.T > kTileRows || c.tile_rows != kTileRows))
    return cudaErrorInvalidValue;
  if (c.gemm1 && (c.act < MOE_ACT_SILU || c.act > kActIdentity)) return cudaErrorInvalidValue;
  kp.act = c.act;
  kp.gated = c.gemm1 && c.act != MOE_ACT_RELU2 && c.act != kActIdentity;
  kp.slab_rows = (c.gemm1 && !kp.gated) ? 2 * kSlab : kSlab;
  kp.second_off = kp.gated ? c.n_out : kSlab;
  kp.K = c.K;
  kp.n_out = c.n_out;
  kp.E = c.E;
  kp.n_slabs = (c.n_out + kp.slab_rows - 1) / kp.slab_rows;
  kp.num_kb = (c.K + kBlockK - 1) / kBlockK;
  kp.w_rows_per_expert = kp.gated ? 2 * c.n_out : c.n_out;
  kp.w4 = nullptr;
  kp.alpha = nullptr;
  if (c.w4) {
    // NVFP4 weights: a bf16 problem (its token rows and act reach the GEMMs as f16), 128-row
    // token tiles (64 for the down projection, 64 or 32 for the gate/up GEMM over gathered
    // rows), K and the output width whole multiples of 128 (one stage is 128 k; a weight slab
    // never crosses an expert).
    const bool tiles_ok =
        c.tile_rows == kTileRows ||
        (c.tile_rows == kTileRowsNarrow && !c.gemm1 && c.mode == kSorted) ||
        ((c.tile_rows == kTileRowsNarrow || c.tile_rows == kTileRowsNvfp4Min) && c.gemm1 &&
         c.mode == kSorted && !c.token_rows);
    if (c.dtype != MOE_BF16 || !tiles_ok || c.K % 128 != 0 || c.n_out % 128 != 0 || !c.alpha ||
        (reinterpret_cast<uintptr_t>(c.w) & 15) != 0)
      return cudaErrorInvalidValue;
    kp.num_kb = c.K / 128;
    kp.w4 = static_cast<const uint8_t*>(c.w);
    kp.alpha = c.alpha;
  }
  kp.tiles = c.tiles;
  kp.n_tiles = c.n_tiles;
  kp.sorted_ids = c.sorted_ids;
  kp.topk_ids = c.topk_ids;
  kp.topk_w = c.topk_w;
  kp.P = c.P;
  kp.top_k = c.top_k;
  kp.T = c.T;
  kp.dense_rows = c.dense_rows;
  kp.out = c.out;
  kp.status = c.status;
  kp.limit_ns = wait_limit_ns();
  kp.prefetch_steps = 0;
  kp.route_ids = (c.gemm1 && kp.token_rows && c.E <= 1024) ? c.route_ids : nullptr;
  kp.split_cap = 0;
  kp.split_cols = 0;
  kp.split_part = nullptr;
  kp.split_cnt = nullptr;
  if (c.w4 && c.gemm1 && kp.token_rows && c.T <= 64 && c.split_cap > 0 && c.split_part &&
      c.split_cnt) {
    if (c.split_cols < ((c.T + 15) & ~15)) return cudaErrorInvalidValue;
    // Split scratch only when splitting pays for the most units the call can have (one tile
    // per routed expert); the kernel (two CTAs per SM, the model counts CTAs) then decides on
    // the actual count.
    const int64_t active = (int64_t)c.P < c.E ? (int64_t)c.P : (int64_t)c.E;
    const int64_t n_max = active * kp.n_slabs;
    const int64_t ctas = 2 * n_max < 2 * num_sms() ? 2 * n_max : 2 * num_sms();
    if (n_max <= c.split_cap && split_pays((int)n_max, (int)ctas, kp.num_kb)) {
      kp.split_cap = c.split_cap;
      kp.split_cols = c.split_cols;
      kp.split_part = c.split_part;
      kp.split_cnt = c.split_cnt;
    }
  }

  if (c.tile_rows != 128 && c.tile_rows != 256 &&
      !(c.tile_rows == 64 && c.mode == kSorted && (c.w4 || !c.gemm1)) &&
      !(c.tile_rows == 32 && c.mode == kSorted && c.w4 && c.gemm1))
    return cudaErrorInvalidValue;
  long long upper = 0;
  if (c.mode == kSorted)
    upper = (long long)c.max_tiles * kp.n_slabs;
  else if (c.mode == kDirect)
    upper = (long long)c.P * kp.n_slabs;
  else
    upper = (long long)((c.dense_rows + c.tile_rows - 1) / c.tile_rows) * kp.n_slabs;
  if (upper <= 0 || c.b_rows <= 0) return cudaSuccess;
  const int sms = num_sms();
  if (kp.split_cap > 0) upper *= 2;  // room for the split halves
  const int grid = (int)(upper < sms ? upper : sms);  // the prefetch budget's CTA count
  if (c.early_tiles && c.mode == kSorted && !c.w4) {
    // Up to ~48 MB (well under the L2) of first-unit weights over the whole grid.
    const int64_t step_bytes = (int64_t)kSlab * kBlockK * 2 * (c.gemm1 && kp.gated ? 2 : 1);
    const int64_t budget = (48ll << 20) / grid / step_bytes;
    kp.prefetch_steps = (int)(budget < kp.num_kb * 4 ? budget : kp.num_kb * 4);
  }

  if (c.gemm1) {
    return c.dtype == MOE_BF16 ? launch_rows<true, __nv_bfloat16>(c, kp, upper, s, pdl)
                               : launch_rows<true, __half>(c, kp, upper, s, pdl);
  }
  return c.dtype == MOE_BF16 ? launch_rows<false, __nv_bfloat16>(c, kp, upper, s, pdl)
                             : launch_rows<false, __half>(c, kp, upper, s, pdl);
}

}  // namespace gb300moe
