/*
 * moe.h -- C ABI of the GB300 fused Mixture-of-Experts forward library (libgb300moe.so).
 *
 * The problem statement follows the TileOPs benchmark page, "MoE" section:
 *   op FusedMoEFwd:  hidden_states[T,H], gating_output[T,E] f32, w_gate_up[E,2F,H],
 *                    w_down[E,H,F], top_k, renormalize; the sigmoid form adds
 *                    correction_bias[E] f32, num_expert_group, topk_group and
 *                    routed_scaling_factor;
 *   op FusedMoESharedExpertFwd: adds shared_w_gate_up[2S,H] and shared_w_down[H,S].
 * The path has five steps: router top-k, expert sort, grouped gate/up GEMM with SiLU(gate)*up,
 * grouped down GEMM with the route weight, and the top-k combine (plus the shared expert).
 *
 * Conventions (all entry points):
 *  - Pointers are DEVICE pointers unless stated; tensors are row-major and contiguous, with the
 *    shapes given.  16-bit tensors (hidden_states, weights, out, intermediate rows) all have the
 *    problem's dtype (bf16 or f16).  gating_output, correction_bias and route weights are f32.
 *  - `stream` is a cudaStream_t passed as void*; all device work is enqueued on it and the call
 *    returns without synchronising (except moe_get_device_status).
 *  - Ownership: the caller owns every buffer.  The library never allocates device memory and
 *    keeps no cached arenas; scratch space comes from the caller's `workspace`, sized by
 *    moe_workspace_size.  Buffer addresses are fixed for the life of a call, so a call can be
 *    captured into a CUDA graph and replayed with the same buffers.
 *  - Errors: argument errors return synchronously, before any launch, and enqueue nothing.
 *    A failed launch returns MOE_ERR_CUDA.  Errors found on the device (an expert id outside
 *    [-1, E), a bounded wait that gave up, an NVFP4-path value past the f16 range) are written
 *    to a status word inside the workspace and read with moe_get_device_status.
 *  - Expert id -1 in a caller-supplied topk_ids marks a padding route: it is skipped and
 *    contributes nothing (ROCm/aiter PR #5973 "[FlyDSL] Optimize MI308 MoE decoding (3/3)",
 *    "Changes": routes with expert ID -1 are skipped).
 *  - Supported sizes: H, F, S multiples of 8 (16-byte row pitch); 1 <= top_k <= 32;
 *    top_k <= E <= 1024; T >= 0.  Unsupported combinations return MOE_ERR_UNSUPPORTED.
 *  - Functions are reentrant given distinct workspaces.
 */
#ifndef GB300_MOE_H
#define GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,         /* null pointer, negative or inconsistent size */
  MOE_ERR_UNSUPPORTED = 2,         /* a valid problem outside the supported sizes */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < the size the call needs */
  MOE_ERR_CUDA = 4,                /* a CUDA launch or API call failed */
  MOE_ERR_TIMEOUT = 5,             /* device: a bounded wait inside a kernel gave up */
  MOE_ERR_BAD_EXPERT_ID = 6,       /* device: an expert id outside [-1, E) was seen */
  MOE_ERR_F16_RANGE = 7            /* device: an NVFP4-path token or act value at or past
                                      65520 in magnitude (the f16 range it computes in) */
} moe_status_t;

typedef enum { MOE_BF16 = 0, MOE_F16 = 1 } moe_dtype_t;
typedef enum { MOE_SOFTMAX = 0, MOE_SIGMOID = 1 } moe_scoring_t;

/* Expert activation (the routed experts and the shared expert use the same one).
 *   MOE_ACT_SILU       act = SiLU(gate) * up, SiLU(g) = g / (1 + e^-g)  (TileOPs "MoE" page,
 *                      op MoEGroupedGemmFwd, activation=silu_and_mul)
 *   MOE_ACT_GELU_TANH  act = GELU_tanh(gate) * up, GELU_tanh(g) = g/2 (1 + tanh(sqrt(2/pi)
 *                      (g + 0.044715 g^3)))  (flashinfer W4A16 follow-up PR, "GeGLU-tanh")
 *   MOE_ACT_RELU2      act = max(h, 0)^2 of a single projection h  (the W4A8 validation list's
 *                      "ReLU2"; read as squared ReLU with no up half)
 * The gated forms keep 2F rows per expert in w_gate_up (gate rows [0,F), up rows [F,2F)); ReLU2
 * keeps F rows.  The same holds for shared_w_gate_up with S. */
typedef enum { MOE_ACT_SILU = 0, MOE_ACT_GELU_TANH = 1, MOE_ACT_RELU2 = 2 } moe_activation_t;

/* Problem description.  Enumerations are stored as int32 so the layout is fixed. */
typedef struct {
  int32_t T;           /* tokens */
  int32_t H;           /* hidden size */
  int32_t E;           /* routed experts */
  int32_t F;           /* expert intermediate size (w_gate_up rows per expert: 2F, or F for
                          MOE_ACT_RELU2) */
  int32_t top_k;       /* experts per token */
  int32_t dtype;       /* moe_dtype_t of hidden_states, weights and outputs */
  int32_t scoring;     /* moe_scoring_t */
  int32_t renormalize; /* nonzero: route weights are normalised over the selected experts */
  int32_t num_expert_group; /* 0 or 1: no grouping; else E % G == 0 and E/G >= 2 (sigmoid) */
  int32_t topk_group;       /* groups kept when grouping, 1 <= topk_group <= G */
  float routed_scaling_factor; /* multiplies every route weight; 1.0f when unused */
  int32_t S;           /* shared-expert intermediate size; 0 = no shared expert */
  int32_t activation;  /* moe_activation_t; 0 (MOE_ACT_SILU) when zero-initialised */
  /* Expert-parallel shard (flashinfer PR #4048 benchmark: a DeepSeek-V3 EP8 rank holds 32 of
   * the 256 experts).  0 = every expert is local.  Otherwise this GPU holds the experts
   * [ep_local_offset, ep_local_offset + ep_num_local) of the E the router scores: the weight
   * tensors hold only those (index e - ep_local_offset), the router's ids are local indices
   * with routes to other experts set to -1 (padding), and out[t] is the sum over the local
   * experts only (plus the shared expert), which the caller's collective adds across shards. */
  int32_t ep_num_local;
  int32_t ep_local_offset;
} moe_problem_t;

/* ---------------------------------------------------------------------------------------- */
/* Sizes (host only, no device work).                                                         */
/* ---------------------------------------------------------------------------------------- */

/* Bytes of workspace fused_moe_fwd needs for problem p (0 if p is invalid).  The first 256
 * bytes hold the device status word; they must be zero before the workspace is first used
 * (moe_workspace_init does this).  It also serves the staged entry points when the sort ran
 * with block_m = 1 (see moe_stage_workspace_size for other alignments). */
size_t moe_workspace_size(const moe_problem_t* p);

/* Bytes of workspace fused_moe_fwd_w4a16 can use for problem p (0 if p is invalid): those of
 * moe_workspace_size(p), plus, for T <= 64, scratch that lets the NVFP4 gate/up GEMM split
 * each unit's K range over two CTAs when that shortens its last wave (a per-unit counter and
 * two halves of f32 partial accumulators: 2048 * round16(T) bytes per unit, at most 1024
 * units of 128 gate/up rows).  Given only moe_workspace_size(p) bytes, fused_moe_fwd_w4a16
 * runs unsplit; the results agree to f32 rounding either way, and each setting is
 * deterministic. */
size_t moe_workspace_size_w4a16(const moe_problem_t* p);

/* Slots of sorted_ids (and rows of the sorted intermediate buffers) moe_align_sort may use for
 * alignment block_m: T*top_k + E*(block_m-1).  -1 if the arguments are invalid. */
int64_t moe_sorted_capacity(const moe_problem_t* p, int32_t block_m);

/* Bytes of workspace the staged entry points need when moe_align_sort ran with block_m
 * (block_m = 1 gives moe_workspace_size(p)).  0 if the arguments are invalid. */
size_t moe_stage_workspace_size(const moe_problem_t* p, int32_t block_m);

/* Zero the workspace's status header on `stream` (one 256-byte memset). */
moe_status_t moe_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------------------- */
/* Whole path.                                                                                */
/* ---------------------------------------------------------------------------------------- */

/*
 * fused_moe_fwd -- TileOPs "MoE" page, ops FusedMoEFwd and FusedMoESharedExpertFwd.
 *   out[t,:] = sum_j w[t,j] * W_down[e_tj] . (SiLU(W_gate[e_tj] x_t) * (W_up[e_tj] x_t))
 *              + shared(x_t)
 * where W_gate[e] = w_gate_up[e, 0:F, :], W_up[e] = w_gate_up[e, F:2F, :], (e_tj, w[t,j]) come
 * from the router (moe_route), and shared(x) = shared_w_down . (SiLU(Wsg x) * (Wsu x)) with
 * Wsg = shared_w_gate_up[0:S, :], Wsu = shared_w_gate_up[S:2S, :] (added unweighted).
 * (shown for p->activation = MOE_ACT_SILU; the other activations replace SiLU(.)*(.) as
 * moe_activation_t states, for the routed and the shared experts alike).
 *   hidden_states   [T,H] dtype
 *   gating_output   [T,E] f32 router logits
 *   w_gate_up       [E,2F,H] dtype ([E,F,H] for MOE_ACT_RELU2);  w_down [E,H,F] dtype
 *   correction_bias [E] f32 or NULL (sigmoid scoring only)
 *   shared_w_gate_up [2S,H] ([S,H] for MOE_ACT_RELU2), shared_w_down [H,S] dtype; both NULL
 *                   iff p->S == 0
 *   out             [T,H] dtype (written in full)
 * For T <= 8 the experts run straight from the router's ids (no sort); otherwise the routes are
 * sorted into expert-contiguous rows first.
 */
moe_status_t fused_moe_fwd(const moe_problem_t* p, const void* hidden_states,
                           const float* gating_output, const void* w_gate_up, const void* w_down,
                           const float* correction_bias, const void* shared_w_gate_up,
                           const void* shared_w_down, void* out, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * fused_moe_fwd_host -- fused_moe_fwd (TileOPs "MoE" page, ops FusedMoEFwd and
 * FusedMoESharedExpertFwd) for a caller whose batch lives in HOST memory:
 *   hidden_states_host  [T,H] dtype, host memory
 *   gating_output_host  [T,E] f32, host memory
 *   out_host            [T,H] dtype, host memory (written in full)
 * The weights, correction_bias and workspace are device memory, as in fused_moe_fwd.  On
 * `stream` the call enqueues one cudaMemcpyAsync host->device per input into staging buffers
 * at the end of the workspace, the fused forward, and one cudaMemcpyAsync device->host of the
 * output; it returns without synchronising, and out_host holds the result once the stream has
 * passed that point.  Page-locked host buffers keep the copies asynchronous (with pageable
 * memory CUDA stages them and the call may block the host).  The host buffers must stay valid
 * and unmodified until then.
 *   workspace_bytes >= moe_workspace_size(p) + moe_host_staging_bytes(p); the staging takes the
 * last moe_host_staging_bytes(p) bytes below the 256-byte-aligned end of the workspace.
 * Argument errors (the checks of fused_moe_fwd included) return before anything is enqueued.
 */
size_t moe_host_staging_bytes(const moe_problem_t* p);
moe_status_t fused_moe_fwd_host(const moe_problem_t* p, const void* hidden_states_host,
                                const float* gating_output_host, const void* w_gate_up,
                                const void* w_down, const float* correction_bias,
                                const void* shared_w_gate_up, const void* shared_w_down,
                                void* out_host, void* workspace, size_t workspace_bytes,
                                void* stream);

/*
 * fused_moe_fwd_w4a16 -- fused_moe_fwd with NVFP4 routed experts and bf16 activations
 * (flashinfer PR #4048, quant_mode "w4a16": NVFP4 weights decoded for a 16-bit MMA, the FP32
 * per-expert scale applied to the FP32 accumulator, as its weight-scale placement ablation
 * keeps).  Each routed weight is
 *   W[e,n,k] = e2m1(code[e,n,k]) * e4m3(sf[e,n,k/16]) * alpha[e]
 * with E2M1 = 1 sign, 2 exponent (bias 1), 1 mantissa bit, and E4M3 = 1 sign, 4 exponent
 * (bias 7), 3 mantissa bits (OCP 8-bit floating point; S.1111.111 is NaN).  The codes and
 * scales are passed in the packed tile layout moe_nvfp4_pack produces:
 *   w_gate_up_tiles moe_nvfp4_pack of codes [E_l, R1, H/2] and scales [E_l, R1, H/16]
 *                   (R1 = 2F, gate rows then up rows, or F for MOE_ACT_RELU2)
 *   w_gate_up_alpha [E_l] f32
 *   w_down_tiles    moe_nvfp4_pack of codes [E_l, H, F/2] and scales [E_l, H, F/16]
 *   w_down_alpha    [E_l] f32
 * (E_l = p->ep_num_local, or E).  Other arguments as fused_moe_fwd.  Requires p->dtype
 * MOE_BF16, H and F multiples of 128 and p->S == 0 (MOE_ERR_UNSUPPORTED otherwise).
 * The GEMMs compute in f16: e2m1 * e4m3 is an exact f16, the bf16 hidden states are converted
 * to f16 (exact from 2^-14 to 65504 in magnitude; smaller ones round to the f16 grid, an error
 * of at most 2^-25) and the act intermediate is kept in f16 (three more bits than bf16).  A
 * hidden or act value of 65520 or more in magnitude would overflow: the call then sets
 * MOE_ERR_F16_RANGE in the device status word and its output is not valid.
 */
moe_status_t fused_moe_fwd_w4a16(const moe_problem_t* p, const void* hidden_states,
                                 const float* gating_output, const uint8_t* w_gate_up_tiles,
                                 const float* w_gate_up_alpha, const uint8_t* w_down_tiles,
                                 const float* w_down_alpha, const float* correction_bias,
                                 void* out, void* workspace, size_t workspace_bytes,
                                 void* stream);

/* fused_moe_fwd_w4a16 from host buffers, as fused_moe_fwd_host: workspace_bytes >=
 * moe_workspace_size(p) (or moe_workspace_size_w4a16(p), for the split-K scratch) +
 * moe_host_staging_bytes(p). */
moe_status_t fused_moe_fwd_w4a16_host(const moe_problem_t* p, const void* hidden_states_host,
                                      const float* gating_output_host,
                                      const uint8_t* w_gate_up_tiles,
                                      const float* w_gate_up_alpha, const uint8_t* w_down_tiles,
                                      const float* w_down_alpha, const float* correction_bias,
                                      void* out_host, void* workspace, size_t workspace_bytes,
                                      void* stream);

/*
 * moe_nvfp4_pack -- rearrange NVFP4 weights into the tile layout the W4A16 GEMMs stream (a
 * one-time step when weights are loaded; no counterpart on the pages beyond their use of a
 * kernel-specific scale layout).  For n_mats matrices of `rows` x K:
 *   codes  [n_mats, rows, K/2] u8 (two E2M1 codes per byte, element 2i in the low nibble),
 *   scales [n_mats, rows, K/16] u8 (E4M3, one per 16 consecutive k)
 *   tiles  moe_nvfp4_packed_bytes(n_mats, rows, K) bytes (out): for each (matrix, 128-row slab,
 *          128-k block) in that order a 9216-byte tile holding the slab's 128 rows of 64 code
 *          bytes (row r at r*64, its 16-byte chunk j at chunk position j ^ ((r>>1)&3)) followed
 *          by their 8 scale bytes (row r at 8192 + r*8).
 * rows and K must be multiples of 128 (MOE_ERR_UNSUPPORTED); codes and tiles 16-byte aligned,
 * scales 8-byte aligned (MOE_ERR_INVALID_ARG).  Runs on `stream`; the caller owns all buffers.
 */
moe_status_t moe_nvfp4_pack(int64_t n_mats, int32_t rows, int32_t K, const uint8_t* codes,
                            const uint8_t* scales, uint8_t* tiles, void* stream);

/* Bytes of moe_nvfp4_pack's output (codes plus scales), or -1 for unsupported sizes. */
int64_t moe_nvfp4_packed_bytes(int64_t n_mats, int32_t rows, int32_t K);

/* ---------------------------------------------------------------------------------------- */
/* Staged entry points (the same kernels, callable one at a time).                          */
/* ---------------------------------------------------------------------------------------- */

/*
 * moe_route -- TileOPs "MoE" page, op FusedTopKFwd (and the routing of FusedMoEFwd).
 * Per token, ids in selection order (descending key, equal keys -> lower expert id):
 *   softmax: key = the raw logit (softmax is monotone); weight_j = exp(x_j - max) / D with D
 *            summed over the selected experts if renormalize, else over all E.
 *   sigmoid: s_e = sigmoid(x_e); key = s_e + correction_bias_e.  With num_expert_group G > 1
 *            the experts form G contiguous groups; a group's score is the sum of its two
 *            largest keys; the topk_group best groups are kept (ties -> lower group) and only
 *            their experts are candidates.  weight_j = s_j / sum_selected(s) if renormalize,
 *            else s_j.
 *   Every weight is then multiplied by routed_scaling_factor.
 * The f32 sigmoid used for the selection key is a fixed sequence of correctly rounded f32
 * operations (Cody-Waite reduction of exp with a degree-7 Taylor polynomial), so the same
 * logits give the same ids on every run.  With an expert-parallel shard (p->ep_num_local > 0)
 * the ids are local indices, -1 for experts outside the shard.
 *   gating_output [T,E] f32; correction_bias [E] f32 or NULL
 *   topk_ids [T,top_k] int32 (out); topk_weights [T,top_k] f32 (out)
 */
moe_status_t moe_route(const moe_problem_t* p, const float* gating_output,
                       const float* correction_bias, int32_t* topk_ids, float* topk_weights,
                       void* stream);

/*
 * moe_align_sort -- TileOPs "MoE" page, op MoEPermuteAlignFwd; the inverse map follows aiter
 * PR #5973 "Changes" (the sort returns each route's sorted row).  A stable counting sort of the
 * flat route index r = t*top_k + j by expert.
 *   topk_ids     [T,top_k] int32 in; -1 = padding route (skipped)
 *   counts       [E] out: live routes per expert
 *   offsets      [E+1] out: start of each expert's segment; each segment is padded to a
 *                multiple of block_m; offsets[E] = padded total
 *   sorted_ids   [cap] out, cap = moe_sorted_capacity(p, block_m): the routes of each segment
 *                in ascending r, then -1 in padding slots; -1 from offsets[E] to cap
 *   tile_expert  [ceil(cap/block_m)] out or NULL: expert owning rows [i*block_m,(i+1)*block_m),
 *                -1 past the end
 *   inv_route    [T*top_k] out: sorted position of each route, -1 for padding routes
 *   workspace    scratch (moe_workspace_size bytes) also holding the status word; an id outside
 *                [-1,E) is treated as padding and sets MOE_ERR_BAD_EXPERT_ID there.
 */
moe_status_t moe_align_sort(const moe_problem_t* p, int32_t block_m, const int32_t* topk_ids,
                            int32_t* counts, int32_t* offsets, int32_t* sorted_ids,
                            int32_t* tile_expert, int32_t* inv_route, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * moe_gemm1_swiglu -- TileOPs "MoE" page, op MoEGroupedGemmFwd with activation=silu_and_mul
 * (contiguous layout): gathers hidden_states rows in sorted order and, per expert segment e,
 *   act[p, f] = SiLU(sum_h Wg[e,f,h] x[h]) * (sum_h Wu[e,f,h] x[h]),  x = hidden[sorted_ids[p]/k]
 * on the tensor cores (bf16/f16 operands, f32 accumulation, f32 epilogue, one rounding to dtype).
 * p->activation selects GELU_tanh(.)*(.) or the single-projection max(.,0)^2 instead
 * (moe_activation_t); the name keeps the default form.
 *   hidden_states [T,H]; block_m, sorted_ids, offsets: as given to / produced by
 *   moe_align_sort; w_gate_up [E,2F,H] ([E,F,H] for MOE_ACT_RELU2); act [cap,F] out,
 *   cap = moe_sorted_capacity(p,block_m)
 *   (rows of padding slots are written as zero).  workspace: moe_stage_workspace_size bytes.
 */
moe_status_t moe_gemm1_swiglu(const moe_problem_t* p, int32_t block_m, const void* hidden_states,
                              const int32_t* sorted_ids, const int32_t* offsets,
                              const void* w_gate_up, void* act, void* workspace,
                              size_t workspace_bytes, void* stream);

/* moe_gemm1_w4a16 -- moe_gemm1_swiglu with NVFP4 gate/up weights (packed tiles and scale as
 * in fused_moe_fwd_w4a16): hidden_states bf16 as there, act written as f16 [cap, F] (the type
 * these GEMMs compute in; MOE_ERR_F16_RANGE as in fused_moe_fwd_w4a16).  Requires MOE_BF16, H
 * and F multiples of 128. */
moe_status_t moe_gemm1_w4a16(const moe_problem_t* p, int32_t block_m, const void* hidden_states,
                             const int32_t* sorted_ids, const int32_t* offsets,
                             const uint8_t* w_gate_up_tiles, const float* w_gate_up_alpha,
                             void* act, void* workspace, size_t workspace_bytes, void* stream);

/*
 * moe_gemm2 -- TileOPs "MoE" page, op MoEGroupedGemmFwd (down projection, contiguous layout),
 * with the route weight applied in the epilogue:
 *   y_route[p, h] = topk_weights[sorted_ids[p]] * sum_f Wd[e,h,f] act[p,f]   (0 for padding)
 *   block_m, sorted_ids, offsets: as for moe_gemm1_swiglu; act [cap,F] dtype;
 *   topk_weights [T*top_k] f32; w_down [E,H,F] dtype; y_route [cap,H] f32 out (kept in f32
 *   so that the only rounding after the down projection is the combine's final one).
 */
moe_status_t moe_gemm2(const moe_problem_t* p, int32_t block_m, const void* act,
                       const int32_t* sorted_ids,
                       const int32_t* offsets, const float* topk_weights, const void* w_down,
                       void* y_route, void* workspace, size_t workspace_bytes, void* stream);

/* moe_gemm2_w4a16 -- moe_gemm2 with NVFP4 down weights (packed tiles and scale as in
 * fused_moe_fwd_w4a16), act read as f16 [cap, F] (what moe_gemm1_w4a16 writes).  Requires
 * MOE_BF16 (the problem's type), H and F multiples of 128. */
moe_status_t moe_gemm2_w4a16(const moe_problem_t* p, int32_t block_m, const void* act,
                             const int32_t* sorted_ids, const int32_t* offsets,
                             const float* topk_weights, const uint8_t* w_down_tiles,
                             const float* w_down_alpha, void* y_route, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * moe_combine -- TileOPs "MoE" page, op MoEPostPermuteFwd; aiter PR #5973 "Changes"
 * (sorted_sum writes the output in full, so no pre-clear is needed):
 *   out[t,:] = round( sum_{j=0..k-1} y_route[inv_route[t*k+j], :] (+ shared_out[t,:]) )
 * summed in f32 in fixed j order, shared term last (deterministic: no atomics), rounded once
 * to dtype.  Routes with inv_route -1, or with topk_ids -1 when topk_ids is given, are
 * skipped.  inv_route NULL means the identity (route r at row r).  On an expert-parallel shard
 * (p->ep_num_local > 0; topk_ids are then the shard's local ids, -1 for a route to another
 * shard) the result is the same; when its tokens average at most two local routes, large calls
 * use a kernel that lists each token's local routes before it loads their rows.
 *   y_route [rows,H] f32; inv_route [T*k] or NULL; topk_ids [T*k] or NULL;
 *   shared_out [T,H] f32 or NULL; out [T,H] dtype
 */
moe_status_t moe_combine(const moe_problem_t* p, const void* y_route, const int32_t* inv_route,
                         const int32_t* topk_ids, const void* shared_out, void* out,
                         void* stream);

/*
 * moe_shared_expert_fwd -- TileOPs "MoE" page, op SharedExpertMLPFwd: the dense SwiGLU MLP
 *   shared_out = shared_w_down . (SiLU(Wsg x) * (Wsu x)) for every token, no routing weight
 *   (or the activation p->activation selects).
 *   hidden_states [T,H]; shared_w_gate_up [2S,H] ([S,H] for MOE_ACT_RELU2); shared_w_down
 *   [H,S];
 *   shared_out [T,H] f32 out (the form moe_combine adds).
 */
moe_status_t moe_shared_expert_fwd(const moe_problem_t* p, const void* hidden_states,
                                   const void* shared_w_gate_up, const void* shared_w_down,
                                   void* shared_out, void* workspace, size_t workspace_bytes,
                                   void* stream);

/*
 * moe_align_sort_noalloc -- the sort of moe_align_sort for callers that cannot allocate device
 * memory when they need it: a serving engine that has handed all device memory to its own pool
 * and forbids later cudaMalloc (which would synchronise the device and fragment the pool), or a
 * plugin entry point whose framework passes only input and output buffers and no workspace.
 * The source pages have no counterpart of this entry point.
 * Same arguments and results as moe_align_sort, minus the workspace: the scratch (per-chunk
 * expert histograms and a status word) lives in a static device array of 256 KiB + 256 bytes
 * inside the library, which every GPU that loads the library holds until the process exits.
 *   status_out  device int32 or NULL: receives MOE_OK or MOE_ERR_BAD_EXPERT_ID for this call
 * The problem is checked as in moe_align_sort (argument errors MOE_ERR_INVALID_ARG, E > 1024 or
 * top_k > 32 MOE_ERR_UNSUPPORTED); with an expert-parallel shard the ids index its ep_num_local
 * experts.  Limit of the static array: ceil(T*top_k/256) * (local experts) <= 65536, else
 * MOE_ERR_WORKSPACE_TOO_SMALL (nothing enqueued).  The first call on a device looks up the array's address (cudaGetSymbolAddress,
 * with that device current); make it before any stream capture.  No call allocates.  Every call
 * shares the array and the array keeps the last call's contents: each call clears the status
 * word itself, and calls that overlap on the GPU (concurrent streams or threads) race.
 */
moe_status_t moe_align_sort_noalloc(const moe_problem_t* p, int32_t block_m,
                                    const int32_t* topk_ids, int32_t* counts, int32_t* offsets,
                                    int32_t* sorted_ids, int32_t* tile_expert,
                                    int32_t* inv_route, int32_t* status_out, void* stream);

/* ---------------------------------------------------------------------------------------- */
/* Expert-parallel building blocks (TileOPs "MoE" page: ops MoEPrePermuteFwd, MoEGroupedGemmFwd */
/* in its masked and contiguous layouts, MoEPostPermuteFwd), for callers that move tokens      */
/* between GPUs themselves and run the experts on local expert ids.                            */
/* ---------------------------------------------------------------------------------------- */

/*
 * moe_pre_permute -- op MoEPrePermuteFwd: the rows of hidden_states in local-expert order
 * (contiguous layout, tight packing, alignment 1).  p->E is the number of local experts;
 * local_ids [T, top_k] int32 holds local expert ids in [0, E), or -1 for a route to another GPU.
 *   permuted   [T*top_k, H] dtype out: rows [offsets[e], offsets[e+1]) are the tokens routed to
 *              local expert e, in ascending route order; rows from offsets[E] on are untouched
 *   offsets    [E+1] out (prefix sums; offsets[E] = local routes), sorted_ids [T*top_k] out
 *              (route index r = t*top_k + j of each row, then -1), inv_route [T*top_k] out
 *              (row of each route, -1 for other GPUs' routes)
 *   workspace  moe_workspace_size(p) bytes (scratch and status word).
 * An id outside [-1, E) is treated as -1 and sets MOE_ERR_BAD_EXPERT_ID in the status word.
 */
moe_status_t moe_pre_permute(const moe_problem_t* p, const void* hidden_states,
                             const int32_t* local_ids, void* permuted, int32_t* offsets,
                             int32_t* sorted_ids, int32_t* inv_route, void* workspace,
                             size_t workspace_bytes, void* stream);

/* Grouped GEMM description (op MoEGroupedGemmFwd). */
typedef struct {
  int32_t E;          /* groups (experts), 1 <= E <= 1024 */
  int32_t N;          /* output columns; a multiple of 8 */
  int32_t K;          /* reduction length; a multiple of 8 */
  int32_t max_m;      /* > 0: masked layout; 0: contiguous layout */
  int64_t rows;       /* contiguous layout: rows P of a and out (ignored when masked) */
  int32_t dtype;      /* moe_dtype_t of a, b and a 16-bit out */
  int32_t activation; /* 0: plain product; 1: silu_and_mul (b holds gate rows then up rows) */
  int32_t out_f32;    /* plain product only: out is f32 (the "bf16/f32" form) */
} moe_grouped_gemm_t;

/*
 * moe_grouped_gemm -- op MoEGroupedGemmFwd: out[r, :] = a[r, :] . b[e(r)]^T for the rows r of
 * each group e, on the tcgen05 tensor cores (f32 accumulation, one rounding to dtype unless
 * out_f32), with silu_and_mul when activation = 1:
 *   masked layout (max_m > 0): a [E, max_m, K], out [E, max_m, N]; layout_metadata [E] int32 is
 *     the number of valid rows of each group (clamped to [0, max_m]); group e owns rows
 *     e*max_m .. e*max_m + layout_metadata[e] - 1, and the other rows of out are untouched;
 *   contiguous layout (max_m == 0): a [rows, K], out [rows, N]; layout_metadata [E] int32 holds
 *     the inclusive prefix sums of the groups' row counts (group e owns rows
 *     layout_metadata[e-1] .. layout_metadata[e] - 1, with layout_metadata[-1] = 0).
 *   b [E, N, K] (activation 0) or [E, 2N, K] (activation 1) dtype, K contiguous.
 *   workspace  moe_grouped_gemm_workspace_size(g) bytes; a prefix sum that decreases or passes
 *              `rows` sets MOE_ERR_INVALID_ARG in its status word (moe_get_device_status).
 */
size_t moe_grouped_gemm_workspace_size(const moe_grouped_gemm_t* g);
moe_status_t moe_grouped_gemm(const moe_grouped_gemm_t* g, const void* a, const void* b,
                              const int32_t* layout_metadata, void* out, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * moe_grouped_gemm_fp8 -- op MoEGroupedGemmFP8Fwd: the grouped GEMM of E4M3 operands with f32
 * block scales, on the tcgen05 tensor cores (kind::f8f6f4):
 *   out[r, n] = sum_kb a_scale[r, kb] * b_scale[e, n/128, kb]
 *                      * sum_{k in block kb} e4m3(a[r, k]) * e4m3(b[e, n, k])
 * with 128-k blocks, f32 accumulation and one rounding to bf16.  Layouts and layout_metadata as
 * for moe_grouped_gemm (masked or contiguous); a is [E, max_m, K] or [rows, K] E4M3 bytes,
 * a_scale [.., K/128] f32 (one per row and 128-k block), b [E, N, K] E4M3 bytes, b_scale
 * [E, N/128, K/128] f32 (one per 128 x 128 block), out bf16 [.., N].  g->dtype must be MOE_BF16
 * (the output type), activation 0, out_f32 0; N and K multiples of 128 (MOE_ERR_UNSUPPORTED).
 * workspace: moe_grouped_gemm_workspace_size(g) bytes.
 */
moe_status_t moe_grouped_gemm_fp8(const moe_grouped_gemm_t* g, const uint8_t* a,
                                  const float* a_scale, const uint8_t* b, const float* b_scale,
                                  const int32_t* layout_metadata, void* out, void* workspace,
                                  size_t workspace_bytes, void* stream);

/*
 * moe_post_permute -- op MoEPostPermuteFwd: the weighted top-k combine
 *   out[t, :] = round( sum_{j=0..k-1} topk_weights[t*k+j] * rows[inv_route[t*k+j], :] )
 * summed in f32 in fixed j order (deterministic), rounded once to dtype; routes with
 * inv_route -1 are skipped (a token with none gets a zero row).
 *   rows [*, H] dtype; topk_weights [T*k] f32; inv_route [T*k] int32; out [T, H] dtype.
 */
moe_status_t moe_post_permute(const moe_problem_t* p, const void* rows,
                              const float* topk_weights, const int32_t* inv_route, void* out,
                              void* stream);

/* ---------------------------------------------------------------------------------------- */
/* Status.                                                                                    */
/* ---------------------------------------------------------------------------------------- */

/* Synchronises `stream`, returns the first device-side error recorded in the workspace's
 * status word since it was last read (MOE_OK if none) and clears it. */
moe_status_t moe_get_device_status(void* workspace, void* stream);

/* Static English description of a status code. */
const char* moe_status_string(moe_status_t s);

/* Test-only knob: the limit, in nanoseconds, of every bounded wait inside the kernels
 * (default 2e9).  A limit of 0 makes the first wait that is not already satisfied give up, so
 * the timeout path can be exercised without a hang.  Returns the previous value. */
uint64_t moe_set_wait_limit_ns(uint64_t limit_ns);

/* ---------------------------------------------------------------------------------------- */
/* Stage profiling (benchmarks).                                                              */
/* ---------------------------------------------------------------------------------------- */

/* Stages of fused_moe_fwd, in launch order: 0 route, 1 sort, 2 tiles, 3 permute, 4 gemm1,
 * 5 gemm2, 6 shared_gemm1, 7 shared_gemm2, 8 combine.  The sort also writes the GEMM tile
 * lists, so stage 2 launches nothing; stage 3 launches only for T > 128 (below that gemm1 reads
 * hidden_states directly); stages 1-3 are skipped on the direct path (T <= 8). */
#define MOE_NUM_STAGES 9

/* Name of stage i (NULL when out of range). */
const char* moe_stage_name(int32_t stage);

/* stage_mask != 0: from now on fused_moe_fwd records a CUDA event pair around every stage i
 * whose bit (1 << i) is set, on the call's stream (host-side event objects, no device memory);
 * kernel launches are counted for every stage.  Totals are reset.  stage_mask == 0 stops the
 * event recording.  Must not be enabled while a call is being captured into a CUDA graph. */
moe_status_t moe_profile_enable(int32_t stage_mask);

/* Synchronises on the recorded events and writes, per stage, the summed device milliseconds,
 * the number of recorded calls and the number of kernel launches since moe_profile_enable;
 * returns the number of stages written (<= max_stages) and resets the totals. */
int32_t moe_profile_collect(double* total_ms, int64_t* calls, int64_t* launches,
                            int32_t max_stages);

#ifdef __cplusplus
}
#endif

#endif /* GB300_MOE_H */
