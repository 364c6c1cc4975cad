// api.cu -- the C ABI declared in include/moe.h: argument validation, workspace carving and
// the launch sequence of the fused MoE forward (router -> sort -> gather -> gemm1+SwiGLU ->
// gemm2 x route weight -> combine, plus the shared expert).
#include <stdio.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace gb300moe {

namespace {

std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};

// ---- stage profiler: event pairs around each stage of fused_moe_fwd (opt-in) ----------------
enum Stage { kRoute, kSort, kTiles, kPermute, kGemm1, kGemm2, kSharedGemm1, kSharedGemm2,
             kCombine, kNumStages };
static_assert(kNumStages == MOE_NUM_STAGES, "stage count");
const char* const kStageNames[kNumStages] = {"route", "sort", "tiles", "permute", "gemm1",
                                             "gemm2", "shared_gemm1", "shared_gemm2",
                                             "combine"};

struct Profiler {
  std::mutex mu;
  uint32_t mask = 0;
  std::vector<cudaEvent_t> ev[kNumStages];  // pairs: start at 2i, end at 2i+1
  size_t used[kNumStages] = {};
  int64_t launches[kNumStages] = {};
};
Profiler g_prof;

// Records the start of `stage` on `s`; returns the pair index or -1 when profiling is off.
int prof_begin(int stage, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (!((g_prof.mask >> stage) & 1u)) return -1;
  auto& v = g_prof.ev[stage];
  const size_t i = g_prof.used[stage];
  if (2 * i + 2 > v.size()) {
    cudaEvent_t a, b;
    if (cudaEventCreate(&a) != cudaSuccess) return -1;
    if (cudaEventCreate(&b) != cudaSuccess) {
      cudaEventDestroy(a);
      return -1;
    }
    v.push_back(a);
    v.push_back(b);
  }
  if (cudaEventRecord(v[2 * i], s) != cudaSuccess) return -1;
  g_prof.used[stage] = i + 1;
  return (int)i;
}

void prof_end(int stage, int idx, cudaStream_t s, int n_launches) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  g_prof.launches[stage] += n_launches;
  if (idx >= 0 && ((g_prof.mask >> stage) & 1u)) cudaEventRecord(g_prof.ev[stage][2 * idx + 1], s);
}

struct StageTimer {
  int stage, idx;
  cudaStream_t s;
  StageTimer(int st, cudaStream_t st_s) : stage(st), idx(prof_begin(st, st_s)), s(st_s) {}
  void done(int n_launches) { prof_end(stage, idx, s, n_launches); }
};

constexpr int kMaxE = 1024;
constexpr int kMaxTopK = 32;
constexpr int kDirectMaxT = 8;
constexpr int kDirectMaxRoutes = kTileRows;
constexpr int kSortChunk = 256;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int elt_bytes(const moe_problem_t&) { return 2; }

}  // namespace

// Declared in common.cuh.
moe_status_t check_problem(const moe_problem_t* p) {
  if (!p) return MOE_ERR_INVALID_ARG;
  if (p->T < 0 || p->H <= 0 || p->E <= 0 || p->F <= 0 || p->top_k <= 0 || p->S < 0)
    return MOE_ERR_INVALID_ARG;
  if (p->top_k > p->E) return MOE_ERR_INVALID_ARG;
  if (p->dtype != MOE_BF16 && p->dtype != MOE_F16) return MOE_ERR_INVALID_ARG;
  if (p->scoring != MOE_SOFTMAX && p->scoring != MOE_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (p->activation < MOE_ACT_SILU || p->activation > MOE_ACT_RELU2) return MOE_ERR_INVALID_ARG;
  if (p->ep_num_local < 0 || p->ep_local_offset < 0) return MOE_ERR_INVALID_ARG;
  if (p->ep_num_local > 0 && (int64_t)p->ep_local_offset + p->ep_num_local > p->E)
    return MOE_ERR_INVALID_ARG;
  if (p->ep_num_local == 0 && p->ep_local_offset != 0) return MOE_ERR_INVALID_ARG;
  if (!(p->routed_scaling_factor == p->routed_scaling_factor)) return MOE_ERR_INVALID_ARG;
  if (p->num_expert_group < 0 || p->topk_group < 0) return MOE_ERR_INVALID_ARG;
  if (p->num_expert_group > 1) {
    const int G = p->num_expert_group;
    if (p->E % G != 0 || p->E / G < 2) return MOE_ERR_INVALID_ARG;
    if (p->topk_group < 1 || p->topk_group > G) return MOE_ERR_INVALID_ARG;
    if ((int64_t)p->topk_group * (p->E / G) < p->top_k) return MOE_ERR_INVALID_ARG;
    if (G > 32) return MOE_ERR_UNSUPPORTED;
    if (p->scoring != MOE_SIGMOID && p->topk_group < G) return MOE_ERR_UNSUPPORTED;
  }
  if (p->E > kMaxE || p->top_k > kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (p->H % 8 != 0 || p->F % 8 != 0 || p->S % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)p->T * p->top_k > (int64_t)1 << 30) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

namespace {

bool use_direct(const moe_problem_t& p) {
  return p.T <= kDirectMaxT && (int64_t)p.T * p.top_k <= kDirectMaxRoutes;
}

// Token rows per tile of the sorted down-projection GEMM: 256 when the experts average at
// least 96 routed rows (prefill), so an expert's weights reach the SMs at most once per 256
// rows; 64 when they average at most 32 (decode), whose tiles stage two 64-k blocks at a time
// and so pay the MMA issuer's per-stage costs once per 32 KB of weights; 128 in between.  The
// gate/up GEMM always uses 128-row tiles: at 256 rows its two accumulators fill TMEM and the
// epilogue could no longer overlap the next unit's K loop, which measured slower on the
// prefill shapes.  The averages are over all E experts of the problem, not the shard's: an
// expert-parallel shard's experts receive their share of the T * top_k routes, and the routes
// to other shards are padding.
int64_t rows_per_expert(const moe_problem_t& p) {
  const int64_t P = (int64_t)p.T * p.top_k;
  const int64_t active = P < p.E ? P : p.E;
  return active > 0 ? P / active : 0;
}

int sorted_tile_rows(const moe_problem_t& p) {
  const int64_t r = rows_per_expert(p);
  if (r <= 0) return kTileRows;
  if (r >= 96) return kTileRowsWide;
  return r <= 32 ? kTileRowsNarrow : kTileRows;
}

// Token rows per tile of the NVFP4 gate/up GEMM over gathered rows: 32 while the experts average
// at most 16 routed rows and 64 while they average at most 64 (two CTAs per SM, each with its
// own MMA issuer; 32-row accumulators leave three decoded-weight slots in TMEM instead of two);
// 128 above, where the narrow tiles' extra MMAs cost more than the second issuer gains.
int w4_gate_up_tile_rows(const moe_problem_t& p) {
  const int64_t r = rows_per_expert(p);
  return r <= 16 ? kTileRowsNvfp4Min : (r <= 64 ? kTileRowsNarrow : kTileRows);
}

// Token rows per tile of the NVFP4 down projection: 64 while the experts average at most 64
// routed rows (the accumulators of a stage's two 64-k halves then fit TMEM, one per MMA issuer),
// 128 above.
int w4_down_tile_rows(const moe_problem_t& p) {
  return rows_per_expert(p) <= 64 ? kTileRowsNarrow : kTileRows;
}

// The down projection of fused_moe_fwd runs on pairs of SMs (gemm_pair.cu) when its tiles have
// 256 rows (experts average at least 96 routed rows) and H splits into whole 256-row pair units.
bool use_pair_gemm2(const moe_problem_t& p) {
  if (p.T <= kTileRows || sorted_tile_rows(p) != kTileRowsWide) return false;
  if (p.H % (2 * kSlab) != 0) return false;
  return pair_gemm_available(p.dtype);
}

// Token rows per tile of the dense shared-expert GEMMs.
int dense_tile_rows(const moe_problem_t& p) { return p.T > kTileRows ? kTileRowsWide : kTileRows; }

// Workspace layout of a call (all offsets 256-byte aligned).
struct Layout {
  int64_t P, cap, n_chunks, max_tiles;
  size_t ids, w, counts, offsets, sorted, inv, chunk, tiles, tiles2, a_sorted, act, y, sh_act,
      sh_out;
  size_t total;
};

Layout make_layout(const moe_problem_t& p, int block_m) {
  Layout L;
  const int eb = elt_bytes(p);
  L.P = (int64_t)p.T * p.top_k;
  L.cap = L.P + (int64_t)p.E * (block_m - 1);
  L.n_chunks = (L.P + kSortChunk - 1) / kSortChunk;
  L.max_tiles = L.cap / kTileRowsNvfp4Min + p.E + 1;  // the most tiles any tile height gives
  size_t off = kHeaderBytes;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.ids = take(sizeof(int32_t) * L.P);
  L.w = take(sizeof(float) * L.P);
  L.counts = take(sizeof(int32_t) * p.E);
  L.offsets = take(sizeof(int32_t) * (p.E + 1));
  L.sorted = take(sizeof(int32_t) * L.cap);
  L.inv = take(sizeof(int32_t) * L.P);
  L.chunk = take(sizeof(int32_t) * L.n_chunks * p.E);
  L.tiles = take(sizeof(Tile) * L.max_tiles);
  L.tiles2 = take(sizeof(Tile) * L.max_tiles);
  // The gathered rows: the staged gate/up GEMM always gathers; fused_moe_fwd needs them only
  // for T > 128 (it reads hidden_states directly on the direct path and when T <= 128, except
  // that the NVFP4 path then keeps its f16 copy of hidden_states here).
  L.a_sorted = take((size_t)L.cap * p.H * eb);
  L.act = take((size_t)L.cap * p.F * eb);
  L.y = take((size_t)L.cap * p.H * sizeof(float));  // weighted down-projection rows, f32
  L.sh_act = take((size_t)p.T * p.S * eb);
  L.sh_out = take(p.S > 0 ? (size_t)p.T * p.H * sizeof(float) : 0);
  L.total = off;
  return L;
}

// Split-K scratch of the NVFP4 gate/up GEMM in fused_moe_fwd_w4a16 (token rows, T <= 64),
// placed after the common layout: a counter per unit, then per unit two halves of f32 partial
// accumulators (gate and up, round16(T) columns of 128 rows each), for up to kSplitMaxUnits
// units.  Its bytes are what moe_workspace_size_w4a16 adds; with a smaller workspace the GEMM
// runs unsplit.
constexpr int64_t kSplitMaxUnits = 1024;
constexpr int kSplitMaxT = 64;

struct SplitLayout {
  int64_t units, cols;
  size_t cnt, part, total;  // offsets from the start of the scratch, and its bytes
};

SplitLayout split_layout(const moe_problem_t& lp) {  // lp: the local view of the problem
  SplitLayout S{0, 0, 0, 0, 0};
  if (lp.T <= 0 || lp.T > kSplitMaxT || !fused_sort_fits(lp) || lp.F % kSlab != 0) return S;
  const int64_t P = (int64_t)lp.T * lp.top_k;
  const int64_t active = P < lp.E ? P : lp.E;  // one tile per active expert over token rows
  const int64_t units = active * (lp.F / kSlab);
  S.units = units < kSplitMaxUnits ? units : kSplitMaxUnits;
  S.cols = (lp.T + 15) & ~15;
  S.cnt = 0;
  S.part = align_up(sizeof(int) * (size_t)S.units, 256);
  S.total = S.part + (size_t)S.units * 2 * 2 * (size_t)S.cols * kSlab * sizeof(float);
  return S;
}

template <typename P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<char*>(ws) + off);
}

int* status_word(void* ws) { return static_cast<int*>(ws); }
int* tile_counter(void* ws) { return reinterpret_cast<int*>(static_cast<char*>(ws) + 64); }
int* tile_counter2(void* ws) { return reinterpret_cast<int*>(static_cast<char*>(ws) + 128); }

moe_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                                 \
  do {                                                \
    cudaError_t _e = (expr);                          \
    if (_e != cudaSuccess) return MOE_ERR_CUDA;       \
  } while (0)

GemmCall base_call(const moe_problem_t& p, int* status) {
  GemmCall c{};
  c.dtype = p.dtype;
  c.status = status;
  c.top_k = p.top_k;
  c.T = p.T;
  c.P = p.T * p.top_k;
  c.E = p.E;
  c.act = p.activation;
  c.tile_rows = kTileRows;
  return c;
}

// Shared expert: dense gemm1 (hidden -> sh_act) and dense gemm2 (sh_act -> sh_out).
cudaError_t run_shared(const moe_problem_t& p, const void* hidden, const void* sgu,
                       const void* sd, void* sh_act, void* sh_out, int* status, cudaStream_t s,
                       bool pdl) {
  GemmCall g1 = base_call(p, status);
  g1.gemm1 = 1;
  g1.mode = kDense;
  g1.K = p.H;
  g1.n_out = p.S;
  g1.E = 1;
  g1.w = sgu;
  g1.b = hidden;
  g1.b_rows = p.T;
  g1.out = sh_act;
  g1.dense_rows = p.T;
  g1.tile_rows = dense_tile_rows(p);
  cudaError_t e;
  {
    StageTimer t(kSharedGemm1, s);
    e = launch_gemm(g1, s, pdl);
    t.done(1);
  }
  if (e != cudaSuccess) return e;
  GemmCall g2 = base_call(p, status);
  g2.gemm1 = 0;
  g2.mode = kDense;
  g2.K = p.S;
  g2.n_out = p.H;
  g2.E = 1;
  g2.w = sd;
  g2.b = sh_act;
  g2.b_rows = p.T;
  g2.out = sh_out;
  g2.dense_rows = p.T;
  g2.tile_rows = dense_tile_rows(p);
  StageTimer t(kSharedGemm2, s);
  e = launch_gemm(g2, s, true);
  t.done(1);
  return e;
}

}  // namespace

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(); }

int num_sms() {
  static int cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace gb300moe

using namespace gb300moe;

extern "C" {

size_t moe_workspace_size(const moe_problem_t* p) {
  if (check_problem(p) != MOE_OK) return 0;
  return make_layout(*p, 1).total;
}

size_t moe_workspace_size_w4a16(const moe_problem_t* p) {
  if (check_problem(p) != MOE_OK) return 0;
  return make_layout(*p, 1).total + split_layout(local_view(*p)).total;
}

size_t moe_stage_workspace_size(const moe_problem_t* p, int32_t block_m) {
  if (check_problem(p) != MOE_OK || block_m <= 0 || block_m > 1024) return 0;
  return make_layout(*p, block_m).total;
}

int64_t moe_sorted_capacity(const moe_problem_t* p, int32_t block_m) {
  if (check_problem(p) != MOE_OK || block_m <= 0) return -1;
  return (int64_t)p->T * p->top_k + (int64_t)p->E * (block_m - 1);
}

moe_status_t moe_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes < kHeaderBytes) return MOE_ERR_INVALID_ARG;
  return from_cuda(cudaMemsetAsync(workspace, 0, kHeaderBytes, (cudaStream_t)stream));
}

// The routed experts' weights: 16-bit (w1, w2), or NVFP4 packed tiles (w1, w2) with their
// per-expert scales (a1, a2).
struct Experts {
  const void* w1;
  const void* w2;
  const float* a1;
  const float* a2;
  int w4;
};

void set_weights(GemmCall& g, const Experts& X, bool first) {
  g.w = first ? X.w1 : X.w2;
  g.w4 = X.w4;
  g.alpha = first ? X.a1 : X.a2;
}

// Limits of the NVFP4 GEMMs (bf16 activations, 128-k stages, 128-row weight slabs).
moe_status_t check_w4(const moe_problem_t& p) {
  if (p.dtype != MOE_BF16 || p.H % 128 != 0 || p.F % 128 != 0 || p.S != 0)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status_t run_fused(const moe_problem_t* p, const Experts& X, const void* hidden_states,
                       const float* gating_output, const float* correction_bias,
                       const void* shared_w_gate_up, const void* shared_w_down, void* out,
                       void* workspace, size_t workspace_bytes, void* stream) {
  moe_status_t st = check_problem(p);
  if (st != MOE_OK) return st;
  if (X.w4 && (st = check_w4(*p)) != MOE_OK) return st;
  if (!workspace) return MOE_ERR_INVALID_ARG;
  if (p->T > 0 && (!hidden_states || !gating_output || !X.w1 || !X.w2 || !out))
    return MOE_ERR_INVALID_ARG;
  if (X.w4 && p->T > 0 && (!X.a1 || !X.a2)) return MOE_ERR_INVALID_ARG;
  if ((p->S > 0) != (shared_w_gate_up != nullptr) || (p->S > 0) != (shared_w_down != nullptr))
    return MOE_ERR_INVALID_ARG;
  if (correction_bias && p->scoring != MOE_SIGMOID) return MOE_ERR_UNSUPPORTED;
  const Layout L = make_layout(*p, 1);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (p->T == 0) return MOE_OK;
  cudaStream_t s = (cudaStream_t)stream;
  void* ws = workspace;
  int* status = status_word(ws);
  int32_t* ids = at<int32_t>(ws, L.ids);
  float* w = at<float>(ws, L.w);
  // The NVFP4 GEMMs take f16 token rows.  Up to 128 tokens the router's launch writes them (in
  // the gathered-rows buffer, unused then); beyond, the permute converts while it gathers.
  void* rows16 = (X.w4 && p->T <= kTileRows) ? at<void>(ws, L.a_sorted) : nullptr;
  {
    StageTimer t(kRoute, s);
    MOE_TRY(launch_route(*p, gating_output, correction_bias, ids, w, s, false, hidden_states,
                         rows16, status));
    t.done(1);
  }
  const void* tokens = rows16 ? rows16 : hidden_states;  // the gate/up GEMM's token rows
  // Past the router every id is a local expert index (or -1): the stages see E_local experts.
  const moe_problem_t P = local_view(*p);

  const void* y_rows = at<void>(ws, L.y);
  const int32_t* inv = nullptr;
  if (use_direct(P)) {
    GemmCall g1 = base_call(P, status);
    g1.gemm1 = 1;
    g1.mode = kDirect;
    g1.K = P.H;
    g1.n_out = P.F;
    set_weights(g1, X, true);
    g1.b = tokens;
    g1.b_rows = P.T;
    g1.out = at<void>(ws, L.act);
    g1.topk_ids = ids;
    {
      StageTimer t(kGemm1, s);
      MOE_TRY(launch_gemm(g1, s, true));
      t.done(1);
    }
    GemmCall g2 = base_call(P, status);
    g2.gemm1 = 0;
    g2.mode = kDirect;
    g2.K = P.F;
    g2.n_out = P.H;
    set_weights(g2, X, false);
    g2.b = at<void>(ws, L.act);
    g2.b_rows = L.P;
    g2.out = at<void>(ws, L.y);
    g2.topk_ids = ids;
    g2.topk_w = w;
    {
      StageTimer t(kGemm2, s);
      MOE_TRY(launch_gemm(g2, s, true));
      t.done(1);
    }
  } else {
    int32_t* counts = at<int32_t>(ws, L.counts);
    int32_t* offsets = at<int32_t>(ws, L.offsets);
    int32_t* sorted = at<int32_t>(ws, L.sorted);
    int32_t* inv_route = at<int32_t>(ws, L.inv);
    Tile* tiles = at<Tile>(ws, L.tiles);    // gemm1: tile_rows1-row tiles
    Tile* tiles2 = at<Tile>(ws, L.tiles2);  // gemm2: tile_rows2-row tiles
    const int tile_rows2 = X.w4 ? w4_down_tile_rows(*p) : sorted_tile_rows(*p);
    // With T <= 128 every expert's rows fit one tile of all T tokens: gemm1 reads hidden_states
    // directly and no gathered copy is made.
    const bool token_rows = P.T <= kTileRows;
    const int tile_rows1 = (X.w4 && !token_rows) ? w4_gate_up_tile_rows(*p) : kTileRows;
    const bool pair2 = !X.w4 && use_pair_gemm2(*p);
    SplitLayout S{0, 0, 0, 0, 0};
    if (X.w4 && token_rows) {
      S = split_layout(P);
      if (S.total == 0 || workspace_bytes < L.total + S.total) S.units = 0;
    }
    int* split_cnt = S.units ? at<int>(ws, L.total + S.cnt) : nullptr;
    if (fused_sort_fits(P)) {  // sort and both tile lists in one launch (and split counters)
      StageTimer t(kSort, s);
      MOE_TRY(launch_sort_fused(P, 1, ids, counts, offsets, sorted, L.cap, nullptr, inv_route,
                                tiles, tile_counter(ws), tile_rows1, tiles2, tile_counter2(ws),
                                tile_rows2, status, s, true, split_cnt, (int)S.units));
      t.done(1);
    } else {
      StageTimer t(kSort, s);
      MOE_TRY(launch_align_sort_chunked(P, 1, ids, counts, offsets, sorted, L.cap, nullptr,
                                        inv_route, at<int32_t>(ws, L.chunk), status, s, true,
                                        tiles, tile_counter(ws), tile_rows1, tiles2,
                                        tile_counter2(ws), tile_rows2));
      t.done(3);
    }
    if (!token_rows) {
      StageTimer t(kPermute, s);
      MOE_TRY(launch_permute(P.dtype, P.top_k, P.H, hidden_states, sorted, offsets, P.E, L.cap,
                             at<void>(ws, L.a_sorted), s, true, X.w4 != 0, status));
      t.done(1);
    }
    GemmCall g1 = base_call(P, status);
    g1.gemm1 = 1;
    g1.mode = kSorted;
    g1.K = P.H;
    g1.n_out = P.F;
    set_weights(g1, X, true);
    g1.b = token_rows ? tokens : at<void>(ws, L.a_sorted);
    g1.b_rows = token_rows ? P.T : L.cap;
    g1.token_rows = token_rows ? 1 : 0;
    g1.sorted_ids = sorted;
    g1.out = at<void>(ws, L.act);
    g1.tiles = tiles;
    g1.n_tiles = tile_counter(ws);
    g1.max_tiles = (int)L.max_tiles;
    g1.tile_rows = tile_rows1;
    g1.early_tiles = token_rows ? 0 : 1;  // sort, then permute, then gemm1
    g1.route_ids = token_rows ? ids : nullptr;  // route, sort, then gemm1
    if (split_cnt) {
      g1.split_cap = (int)S.units;
      g1.split_cols = (int)S.cols;
      g1.split_part = at<float>(ws, L.total + S.part);
      g1.split_cnt = split_cnt;
    }
    {
      StageTimer t(kGemm1, s);
      MOE_TRY(launch_gemm(g1, s, true));
      t.done(1);
    }
    GemmCall g2 = g1;
    g2.route_ids = nullptr;
    g2.split_cap = 0;
    g2.split_part = nullptr;
    g2.split_cnt = nullptr;
    g2.gemm1 = 0;
    g2.token_rows = 0;
    g2.b_rows = L.cap;
    g2.K = P.F;
    g2.n_out = P.H;
    set_weights(g2, X, false);
    g2.b = at<void>(ws, L.act);
    g2.out = at<void>(ws, L.y);
    g2.sorted_ids = sorted;
    g2.topk_w = w;
    g2.tiles = tiles2;
    g2.n_tiles = tile_counter2(ws);
    g2.tile_rows = tile_rows2;
    g2.early_tiles = 1;  // sort, [permute,] gemm1, then gemm2
    {
      StageTimer t(kGemm2, s);
      MOE_TRY(pair2 ? launch_gemm_pair(g2, s, true) : launch_gemm(g2, s, true));
      t.done(1);
    }
    inv = inv_route;
  }
  const void* sh_out = nullptr;
  if (P.S > 0) {
    MOE_TRY(run_shared(P, hidden_states, shared_w_gate_up, shared_w_down, at<void>(ws, L.sh_act),
                       at<void>(ws, L.sh_out), status, s, true));
    sh_out = at<void>(ws, L.sh_out);
  }
  {
    StageTimer t(kCombine, s);
    // the whole problem: its expert-parallel fields choose the combine kernel
    MOE_TRY(launch_combine(*p, y_rows, inv, ids, sh_out, out, s, true));
    t.done(1);
  }
  return MOE_OK;
}

moe_status_t fused_moe_fwd(const moe_problem_t* p, const void* hidden_states,
                           const float* gating_output, const void* w_gate_up, const void* w_down,
                           const float* correction_bias, const void* shared_w_gate_up,
                           const void* shared_w_down, void* out, void* workspace,
                           size_t workspace_bytes, void* stream) {
  const Experts X{w_gate_up, w_down, nullptr, nullptr, 0};
  return run_fused(p, X, hidden_states, gating_output, correction_bias, shared_w_gate_up,
                   shared_w_down, out, workspace, workspace_bytes, stream);
}

moe_status_t fused_moe_fwd_w4a16(const moe_problem_t* p, const void* hidden_states,
                                 const float* gating_output, const uint8_t* w_gate_up_tiles,
                                 const float* w_gate_up_alpha, const uint8_t* w_down_tiles,
                                 const float* w_down_alpha, const float* correction_bias,
                                 void* out, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  const Experts X{w_gate_up_tiles, w_down_tiles, w_gate_up_alpha, w_down_alpha, 1};
  return run_fused(p, X, hidden_states, gating_output, correction_bias, nullptr, nullptr, out,
                   workspace, workspace_bytes, stream);
}

// ---- from host buffers -------------------------------------------------------------------
namespace {

// Staging for the host entry points, carved from the END of the caller's workspace: hidden
// states [T,H] dtype, router logits [T,E] f32 and the output [T,H] dtype, each 256-byte aligned.
struct HostStaging {
  size_t hidden, gating, out, total;
};

HostStaging host_staging(const moe_problem_t& p) {
  HostStaging h;
  h.hidden = align_up((size_t)p.T * p.H * elt_bytes(p), 256);
  h.gating = align_up((size_t)p.T * p.E * sizeof(float), 256);
  h.out = h.hidden;
  h.total = h.hidden + h.gating + h.out;
  return h;
}

}  // namespace

size_t moe_host_staging_bytes(const moe_problem_t* p) {
  if (check_problem(p) != MOE_OK) return 0;
  return host_staging(*p).total;
}

namespace {

moe_status_t run_fused_host(const moe_problem_t* p, const Experts& X, const void* hidden_host,
                            const float* gating_host, const float* correction_bias,
                            const void* shared_w_gate_up, const void* shared_w_down,
                            void* out_host, void* workspace, size_t workspace_bytes,
                            void* stream) {
  moe_status_t st = check_problem(p);
  if (st != MOE_OK) return st;
  if (!workspace) return MOE_ERR_INVALID_ARG;
  if (p->T > 0 && (!hidden_host || !gating_host || !out_host)) return MOE_ERR_INVALID_ARG;
  const HostStaging h = host_staging(*p);
  if (workspace_bytes < h.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  // The staging sits at the 256-byte-aligned end; the fused path gets the bytes before it.
  const uintptr_t end = (reinterpret_cast<uintptr_t>(workspace) + workspace_bytes) & ~(uintptr_t)255;
  if (end < reinterpret_cast<uintptr_t>(workspace) + h.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  char* stage = reinterpret_cast<char*>(end - h.total);
  const size_t fused_bytes = (size_t)(stage - static_cast<char*>(workspace));
  void* d_hidden = stage;
  float* d_gating = reinterpret_cast<float*>(stage + h.hidden);
  void* d_out = stage + h.hidden + h.gating;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t hid_bytes = (size_t)p->T * p->H * elt_bytes(*p);
  if (p->T > 0) {
    // Argument errors of the fused call come back before anything is enqueued: check them on
    // the device staging addresses first (T = 0 would skip the checks of the weights).
    if (!X.w1 || !X.w2 || (X.w4 && (!X.a1 || !X.a2))) return MOE_ERR_INVALID_ARG;
    if (X.w4 && (st = check_w4(*p)) != MOE_OK) return st;
    if ((p->S > 0) != (shared_w_gate_up != nullptr) || (p->S > 0) != (shared_w_down != nullptr))
      return MOE_ERR_INVALID_ARG;
    if (correction_bias && p->scoring != MOE_SIGMOID) return MOE_ERR_UNSUPPORTED;
    if (fused_bytes < make_layout(*p, 1).total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    MOE_TRY(cudaMemcpyAsync(d_hidden, hidden_host, hid_bytes, cudaMemcpyHostToDevice, s));
    MOE_TRY(cudaMemcpyAsync(d_gating, gating_host, (size_t)p->T * p->E * sizeof(float),
                            cudaMemcpyHostToDevice, s));
  }
  st = run_fused(p, X, d_hidden, d_gating, correction_bias, shared_w_gate_up, shared_w_down,
                 d_out, workspace, fused_bytes, stream);
  if (st != MOE_OK || p->T == 0) return st;
  MOE_TRY(cudaMemcpyAsync(out_host, d_out, hid_bytes, cudaMemcpyDeviceToHost, s));
  return MOE_OK;
}

}  // namespace

moe_status_t fused_moe_fwd_host(const moe_problem_t* p, const void* hidden_states_host,
                                const float* gating_output_host, const void* w_gate_up,
                                const void* w_down, const float* correction_bias,
                                const void* shared_w_gate_up, const void* shared_w_down,
                                void* out_host, void* workspace, size_t workspace_bytes,
                                void* stream) {
  const Experts X{w_gate_up, w_down, nullptr, nullptr, 0};
  return run_fused_host(p, X, hidden_states_host, gating_output_host, correction_bias,
                        shared_w_gate_up, shared_w_down, out_host, workspace, workspace_bytes,
                        stream);
}

moe_status_t fused_moe_fwd_w4a16_host(const moe_problem_t* p, const void* hidden_states_host,
                                      const float* gating_output_host,
                                      const uint8_t* w_gate_up_tiles,
                                      const float* w_gate_up_alpha, const uint8_t* w_down_tiles,
                                      const float* w_down_alpha, const float* correction_bias,
                                      void* out_host, void* workspace, size_t workspace_bytes,
                                      void* stream) {
  const Experts X{w_gate_up_tiles, w_down_tiles, w_gate_up_alpha, w_down_alpha, 1};
  return run_fused_host(p, X, hidden_states_host, gating_output_host, correction_bias, nullptr,
                        nullptr, out_host, workspace, workspace_bytes, stream);
}

moe_status_t moe_route(const moe_problem_t* p, const float* gating_output,
                       const float* correction_bias, int32_t* topk_ids, float* topk_weights,
                       void* stream) {
  moe_status_t st = check_problem(p);
  if (st != MOE_OK) return st;
  if (p->T > 0 && (!gating_output || !topk_ids || !topk_weights)) return MOE_ERR_INVALID_ARG;
  if (correction_bias && p->scoring != MOE_SIGMOID) return MOE_ERR_UNSUPPORTED;
  return from_cuda(launch_route(*p, gating_output, correction_bias, topk_ids, topk_weights,
                                (cudaStream_t)stream, false));
}

moe_status_t moe_align_sort(const moe_problem_t* p, int32_t block_m, const int32_t* topk_ids,
                            int32_t* counts, int32_t* offsets, int32_t* sorted_ids,
                            int32_t* tile_expert, int32_t* inv_route, void* workspace,
                            size_t workspace_bytes, void* stream) {
  moe_status_t st = check_problem(p);
  if (st != MOE_OK) return st;
  if (block_m <= 0 || block_m > 1024) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets || !sorted_ids || !inv_route || !workspace) return MOE_ERR_INVALID_ARG;
  if (p->T > 0 && !topk_ids) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(*p, 1);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const int64_t cap = moe_sorted_capacity(p, block_m);
  return from_cuda(launch_align_sort(local_view(*p), block_m, topk_ids, counts, offsets,
                                     sorted_ids, cap,
                                     tile_expert, inv_route, at<int32_t>(workspace, L.chunk),
                                     status_word(workspace), (cudaStream_t)stream, false));
}

moe_status_t gemm1_staged(const moe_problem_t* p, int32_t block_m, const void* hidden_states,
                          const int32_t* sorted_ids, const int32_t* offsets, const Experts& X,
                          void* act, void* workspace, size_t workspace_bytes, void* stream) {
  moe_status_t st = check_problem(p);
  if (st != MOE_OK) return st;
  if (X.w4 && (st = check_w4(*p)) != MOE_OK) return st;
  if (block_m <= 0 || block_m > 1024) return MOE_ERR_INVALID_ARG;
  if (!workspace || !sorted_ids || !offsets || !act) return MOE_ERR_INVALID_ARG;
  if (p->T > 0 && (!hidden_states || !X.w1)) return MOE_ERR_INVALID_ARG;
  if (X.w4 && p->T > 0 && !X.a1) return MOE_ERR_INVALID_ARG;
  const moe_problem_t P = local_view(*p);
  const Layout L = make_layout(*p, block_m);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = (cudaStream_t)stream;
  void* ws = workspace;
  Tile* tiles = at<Tile>(ws, L.tiles);
  const int tile_rows = X.w4 ? w4_gate_up_tile_rows(*p) : kTileRows;
  MOE_TRY(launch_build_tiles(P.E, offsets, tiles, tile_counter(ws), tile_rows, s, false));
  MOE_TRY(launch_permute(P.dtype, P.top_k, P.H, hidden_states, sorted_ids, offsets, P.E, L.cap,
                         at<void>(ws, L.a_sorted), s, true, X.w4 != 0, status_word(ws)));
  GemmCall g1 = base_call(P, status_word(ws));
  g1.gemm1 = 1;
  g1.mode = kSorted;
  g1.K = P.H;
  g1.n_out = P.F;
  set_weights(g1, X, true);
  g1.b = at<void>(ws, L.a_sorted);
  g1.b_rows = L.cap;
  g1.out = act;
  g1.tiles = tiles;
  g1.n_tiles = tile_counter(ws);
  g1.max_tiles = (int)L.max_tiles;
  g1.tile_rows = tile_rows;
  return from_cuda(launch_gemm(g1, s, true));
}

moe_status_t gemm2_staged(const moe_problem_t* p, int32_t block_m, const void* act,
                          const int32_t* sorted_ids, const int32_t* offsets,
                          const float* topk_weights, const Experts& X, void* y_route,
                          void* workspace, size_t workspace_bytes, void* stream) {
  moe_status_t st = check_problem(p);
  if (st != MOE_OK) return st;
  if (X.w4 && (st = check_w4(*p)) != MOE_OK) return st;
  if (block_m <= 0 || block_m > 1024) return MOE_ERR_INVALID_ARG;
  if (!workspace || !sorted_ids || !offsets || !y_route) return MOE_ERR_INVALID_ARG;
  if (p->T > 0 && (!act || !topk_weights || !X.w2)) return MOE_ERR_INVALID_ARG;
  if (X.w4 && p->T > 0 && !X.a2) return MOE_ERR_INVALID_ARG;
  const moe_problem_t P = local_view(*p);
  const Layout L = make_layout(*p, block_m);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = (cudaStream_t)stream;
  void* ws = workspace;
  Tile* tiles = at<Tile>(ws, L.tiles);
  const int tile_rows = X.w4 ? w4_down_tile_rows(*p) : sorted_tile_rows(*p);
  MOE_TRY(launch_build_tiles(P.E, offsets, tiles, tile_counter(ws), tile_rows, s, false));
  GemmCall g2 = base_call(P, status_word(ws));
  g2.gemm1 = 0;
  g2.mode = kSorted;
  g2.K = P.F;
  g2.n_out = P.H;
  set_weights(g2, X, false);
  g2.b = act;
  g2.b_rows = L.cap;
  g2.out = y_route;
  g2.tiles = tiles;
  g2.n_tiles = tile_counter(ws);
  g2.max_tiles = (int)L.max_tiles;
  g2.tile_rows = tile_rows;
  g2.sorted_ids = sorted_ids;
  g2.topk_w = topk_weights;
  return from_cuda(launch_gemm(g2, s, true));
}

moe_status_t moe_gemm1_swiglu(const moe_problem_t* p, int32_t block_m, const void* hidden_states,
                              const int32_t* sorted_ids, const int32_t* offsets,
                              const void* w_gate_up, void* act, void* workspace,
                              size_t workspace_bytes, void* stream) {
  const Experts X{w_gate_up, nullptr, nullptr, nullptr, 0};
  return gemm1_staged(p, block_m, hidden_states, sorted_ids, offsets, X, act, workspace,
                      workspace_bytes, stream);
}

moe_status_t moe_gemm1_w4a16(const moe_problem_t* p, int32_t block_m, const void* hidden_states,
                             const int32_t* sorted_ids, const int32_t* offsets,
                             const uint8_t* w_gate_up_tiles, const float* w_gate_up_alpha,
                             void* act, void* workspace, size_t workspace_bytes, void* stream) {
  const Experts X{w_gate_up_tiles, nullptr, w_gate_up_alpha, nullptr, 1};
  return gemm1_staged(p, block_m, hidden_states, sorted_ids, offsets, X, act, workspace,
                      workspace_bytes, stream);
}

moe_status_t moe_gemm2(const moe_problem_t* p, int32_t block_m, const void* act,
                       const int32_t* sorted_ids, const int32_t* offsets,
                       const float* topk_weights, const void* w_down, void* y_route,
                       void* workspace, size_t workspace_bytes, void* stream) {
  const Experts X{nullptr, w_down, nullptr, nullptr, 0};
  return gemm2_staged(p, block_m, act, sorted_ids, offsets, topk_weights, X, y_route, workspace,
                      workspace_bytes, stream);
}

moe_status_t moe_gemm2_w4a16(const moe_problem_t* p, int32_t block_m, const void* act,
                             const int32_t* sorted_ids, const int32_t* offsets,
                             const float* topk_weights, const uint8_t* w_down_tiles,
                             const float* w_down_alpha, void* y_route, void* workspace,
                             size_t workspace_bytes, void* stream) {
  const Experts X{nullptr, w_down_tiles, nullptr, w_down_alpha, 1};
  return gemm2_staged(p, block_m, act, sorted_ids, offsets, topk_weights, X, y_route, workspace,
                      workspace_bytes, stream);
}

moe_status_t moe_combine(const moe_problem_t* p, const void* y_route, const int32_t* inv_route,
                         const int32_t* topk_ids, const void* shared_out, void* out,
                         void* stream) {
  moe_status_t st = check_problem(p);
  if (st != MOE_OK) return st;
  if (p->T > 0 && (!y_route || !out)) return MOE_ERR_INVALID_ARG;
  return from_cuda(launch_combine(*p, y_route, inv_route, topk_ids, shared_out, out,
                                  (cudaStream_t)stream, false));
}

moe_status_t moe_shared_expert_fwd(const moe_problem_t* p, const void* hidden_states,
                                   const void* shared_w_gate_up, const void* shared_w_down,
                                   void* shared_out, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  moe_status_t st = check_problem(p);
  if (st != MOE_OK) return st;
  if (p->S <= 0) return MOE_ERR_INVALID_ARG;
  if (!workspace || (p->T > 0 && (!hidden_states || !shared_w_gate_up || !shared_w_down ||
                                  !shared_out)))
    return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(*p, 1);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (p->T == 0) return MOE_OK;
  return from_cuda(run_shared(*p, hidden_states, shared_w_gate_up, shared_w_down,
                              at<void>(workspace, L.sh_act), shared_out,
                              status_word(workspace), (cudaStream_t)stream, false));
}

// ---- expert-parallel building blocks ------------------------------------------------------

moe_status_t moe_pre_permute(const moe_problem_t* p, const void* hidden_states,
                             const int32_t* local_ids, void* permuted, int32_t* offsets,
                             int32_t* sorted_ids, int32_t* inv_route, void* workspace,
                             size_t workspace_bytes, void* stream) {
  moe_status_t st = check_problem(p);
  if (st != MOE_OK) return st;
  if (!workspace || !offsets || !sorted_ids || !inv_route) return MOE_ERR_INVALID_ARG;
  if (p->T > 0 && (!hidden_states || !local_ids || !permuted)) return MOE_ERR_INVALID_ARG;
  const moe_problem_t P = local_view(*p);
  const Layout L = make_layout(*p, 1);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = (cudaStream_t)stream;
  void* ws = workspace;
  MOE_TRY(launch_align_sort(P, 1, local_ids, at<int32_t>(ws, L.counts), offsets, sorted_ids,
                            L.cap, nullptr, inv_route, at<int32_t>(ws, L.chunk), status_word(ws),
                            s, false));
  if (p->T == 0) return MOE_OK;
  return from_cuda(launch_permute(P.dtype, P.top_k, P.H, hidden_states, sorted_ids, offsets, P.E,
                                  L.cap, permuted, s, true));
}

namespace {

bool grouped_gemm_valid(const moe_grouped_gemm_t* g) {
  if (!g || g->E < 1 || g->E > 1024 || g->N <= 0 || g->K <= 0 || g->max_m < 0) return false;
  if (g->N % 8 != 0 || g->K % 8 != 0) return false;
  if (g->dtype != MOE_BF16 && g->dtype != MOE_F16) return false;
  if (g->activation != 0 && g->activation != 1) return false;
  if (g->out_f32 && g->activation != 0) return false;
  if (g->max_m == 0 && g->rows < 0) return false;
  const int64_t rows = g->max_m > 0 ? (int64_t)g->E * g->max_m : g->rows;
  return rows < ((int64_t)1 << 31);
}

int64_t grouped_gemm_rows(const moe_grouped_gemm_t* g) {
  return g->max_m > 0 ? (int64_t)g->E * g->max_m : g->rows;
}

int64_t grouped_gemm_max_tiles(const moe_grouped_gemm_t* g) {
  return grouped_gemm_rows(g) / kTileRows + g->E + 1;
}

}  // namespace

size_t moe_grouped_gemm_workspace_size(const moe_grouped_gemm_t* g) {
  if (!grouped_gemm_valid(g)) return 0;
  return kHeaderBytes + align_up(sizeof(Tile) * (size_t)grouped_gemm_max_tiles(g), 256);
}

moe_status_t moe_grouped_gemm(const moe_grouped_gemm_t* g, const void* a, const void* b,
                              const int32_t* layout_metadata, void* out, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (!grouped_gemm_valid(g)) return MOE_ERR_INVALID_ARG;
  if (!workspace || !layout_metadata) return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < moe_grouped_gemm_workspace_size(g)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const int64_t rows = grouped_gemm_rows(g);
  if (rows == 0) return MOE_OK;
  if (!a || !b || !out) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  void* ws = workspace;
  Tile* tiles = at<Tile>(ws, kHeaderBytes);
  MOE_TRY(launch_build_tiles_meta(g->E, g->max_m, rows, layout_metadata, tiles, tile_counter(ws),
                                  kTileRows, status_word(ws), s, false));
  GemmCall c{};
  c.dtype = g->dtype;
  c.status = status_word(ws);
  c.E = g->E;
  c.mode = kSorted;
  c.K = g->K;
  c.n_out = g->N;
  c.w = b;
  c.b = a;
  c.b_rows = rows;
  c.out = out;
  c.tiles = tiles;
  c.n_tiles = tile_counter(ws);
  c.max_tiles = (int)grouped_gemm_max_tiles(g);
  c.tile_rows = kTileRows;
  if (g->out_f32) {
    c.gemm1 = 0;  // f32 rows, scale 1 (no sorted_ids)
  } else {
    c.gemm1 = 1;
    c.act = g->activation ? MOE_ACT_SILU : kActIdentity;
  }
  return from_cuda(launch_gemm(c, s, true));
}

moe_status_t moe_grouped_gemm_fp8(const moe_grouped_gemm_t* g, const uint8_t* a,
                                  const float* a_scale, const uint8_t* b, const float* b_scale,
                                  const int32_t* layout_metadata, void* out, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  if (!grouped_gemm_valid(g)) return MOE_ERR_INVALID_ARG;
  if (g->dtype != MOE_BF16 || g->activation != 0 || g->out_f32) return MOE_ERR_UNSUPPORTED;
  if (g->N % 128 != 0 || g->K % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (!workspace || !layout_metadata) return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < moe_grouped_gemm_workspace_size(g)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const int64_t rows = grouped_gemm_rows(g);
  if (rows == 0) return MOE_OK;
  if (!a || !a_scale || !b || !b_scale || !out) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  void* ws = workspace;
  Tile* tiles = at<Tile>(ws, kHeaderBytes);
  // Up to 128 groups the GEMM derives its tile list from the metadata itself (one launch);
  // beyond, the tile-list kernel writes it first.
  const bool own_tiles = g->E <= 128;
  if (!own_tiles)
    MOE_TRY(launch_build_tiles_meta(g->E, g->max_m, rows, layout_metadata, tiles,
                                    tile_counter(ws), kTileRows, status_word(ws), s, false));
  // the tallest tile: a group's rows, at most max_m (masked) or all rows (contiguous), and 128
  const int64_t tall = g->max_m > 0 ? g->max_m : rows;
  return from_cuda(launch_gemm_fp8(g->E, g->N, g->K, rows,
                                   (int)(tall < kTileRows ? tall : kTileRows), a, a_scale, b,
                                   b_scale, tiles, tile_counter(ws),
                                   (int)grouped_gemm_max_tiles(g),
                                   own_tiles ? layout_metadata : nullptr, g->max_m,
                                   static_cast<__nv_bfloat16*>(out), status_word(ws), s, true));
}

moe_status_t moe_post_permute(const moe_problem_t* p, const void* rows,
                              const float* topk_weights, const int32_t* inv_route, void* out,
                              void* stream) {
  moe_status_t st = check_problem(p);
  if (st != MOE_OK) return st;
  if (p->T > 0 && (!rows || !topk_weights || !inv_route || !out)) return MOE_ERR_INVALID_ARG;
  return from_cuda(launch_post_permute(p->dtype, p->T, p->top_k, p->H, rows, topk_weights,
                                       inv_route, out, (cudaStream_t)stream, false));
}

int64_t moe_nvfp4_packed_bytes(int64_t n_mats, int32_t rows, int32_t K) {
  if (n_mats < 0 || rows <= 0 || K <= 0 || rows % 128 != 0 || K % 128 != 0) return -1;
  return n_mats * (int64_t)rows * K / 2 + n_mats * (int64_t)rows * K / 16;
}

moe_status_t moe_nvfp4_pack(int64_t n_mats, int32_t rows, int32_t K, const uint8_t* codes,
                            const uint8_t* scales, uint8_t* tiles, void* stream) {
  if (moe_nvfp4_packed_bytes(n_mats, rows, K) < 0) return MOE_ERR_UNSUPPORTED;
  if (n_mats > 0 && (!codes || !scales || !tiles)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(codes) & 15) || (reinterpret_cast<uintptr_t>(scales) & 7) ||
      (reinterpret_cast<uintptr_t>(tiles) & 15))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(launch_nvfp4_pack(n_mats, rows, K, codes, scales, tiles, (cudaStream_t)stream));
}

moe_status_t moe_get_device_status(void* workspace, void* stream) {
  if (!workspace) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaMemset(workspace, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  return (moe_status_t)v;
}

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported problem size or option";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA launch or API error";
    case MOE_ERR_TIMEOUT: return "a bounded wait inside a kernel timed out";
    case MOE_ERR_BAD_EXPERT_ID: return "expert id outside [-1, E)";
    case MOE_ERR_F16_RANGE: return "an NVFP4-path value past the f16 range";
  }
  return "unknown status";
}

uint64_t moe_set_wait_limit_ns(uint64_t limit_ns) { return g_wait_limit_ns.exchange(limit_ns); }

const char* moe_stage_name(int32_t stage) {
  return stage >= 0 && stage < kNumStages ? kStageNames[stage] : nullptr;
}

moe_status_t moe_profile_enable(int32_t stage_mask) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  g_prof.mask = (uint32_t)stage_mask;
  for (int i = 0; i < kNumStages; ++i) {
    g_prof.used[i] = 0;
    g_prof.launches[i] = 0;
  }
  return MOE_OK;
}

int32_t moe_profile_collect(double* total_ms, int64_t* calls, int64_t* launches,
                            int32_t max_stages) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  const int n = max_stages < kNumStages ? max_stages : kNumStages;
  for (int i = 0; i < n; ++i) {
    double tot = 0.0;
    for (size_t j = 0; j < g_prof.used[i]; ++j) {
      float ms = 0.0f;
      cudaEventSynchronize(g_prof.ev[i][2 * j + 1]);
      if (cudaEventElapsedTime(&ms, g_prof.ev[i][2 * j], g_prof.ev[i][2 * j + 1]) == cudaSuccess)
        tot += ms;
    }
    if (total_ms) total_ms[i] = tot;
    if (calls) calls[i] = (int64_t)g_prof.used[i];
    if (launches) launches[i] = g_prof.launches[i];
  }
  for (int i = 0; i < kNumStages; ++i) {
    g_prof.used[i] = 0;
    g_prof.launches[i] = 0;
  }
  return n;
}

}  // extern "C"
