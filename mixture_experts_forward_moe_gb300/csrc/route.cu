// route.cu -- router top-k (TileOPs "MoE" page, op FusedTopKFwd and the routing of FusedMoEFwd):
// one warp per token, expert e held by lane e % 32, selection by warp-wide argmax with shuffles.
#include <limits.h>
#include <math.h>

#include "common.cuh"
#include "ptx.cuh"

namespace gb300moe {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarpsPerBlock = 8;

// f32 sigmoid used as the selection key for scoring_func=sigmoid.  It is a fixed sequence of
// correctly rounded f32 operations, so the same logit always gives the same key:
//   exp(z): n = rint(z*log2 e); r = z - n*ln2 (ln2 as a 16-bit head, exact when multiplied by
//   n, plus an f32 tail) by two fused multiply-adds; e^r by the degree-7 Taylor polynomial
//   (coefficients 1/k!) in Horner form with fused multiply-adds; times 2^n built from bits.
//   sigmoid(x) = 1 / (1 + exp(-x)), with -x clamped to [-80, 80] so 2^n stays normal.
// The polynomial remainder is below 1e-8 relative on |r| <= ln2/2.
__device__ __forceinline__ float key_exp_f32(float z) {
  const float n = rintf(__fmul_rn(z, 0x1.715476p+0f));
  float r = __fmaf_rn(-n, 0x1.62e4p-1f, z);
  r = __fmaf_rn(-n, 0x1.7f7d1cp-20f, r);
  float q = 0x1.a01a02p-13f;        // 1/7!
  q = __fmaf_rn(q, r, 0x1.6c16c2p-10f);  // 1/6!
  q = __fmaf_rn(q, r, 0x1.111112p-7f);   // 1/5!
  q = __fmaf_rn(q, r, 0x1.555556p-5f);   // 1/4!
  q = __fmaf_rn(q, r, 0x1.555556p-3f);   // 1/3!
  q = __fmaf_rn(q, r, 0x1p-1f);          // 1/2!
  q = __fmaf_rn(q, r, 1.0f);
  q = __fmaf_rn(q, r, 1.0f);
  const int ni = static_cast<int>(n);
  return __fmul_rn(q, __int_as_float((ni + 127) << 23));
}

__device__ __forceinline__ float key_sigmoid_f32(float x) {
  const float z = fminf(fmaxf(-x, -80.0f), 80.0f);
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, key_exp_f32(z)));
}

// (ka, ea) ranks before (kb, eb): larger key, then lower expert id.
__device__ __forceinline__ bool before(float ka, int ea, float kb, int eb) {
  return ka > kb || (ka == kb && ea < eb);
}

template <int VPL>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    route_kernel(int T, int E, int K, int scoring, int renorm, int G, int keepG, float rsf,
                 int loc0, int nloc, const float* __restrict__ gating,
                 const float* __restrict__ bias, int32_t* __restrict__ ids,
                 float* __restrict__ wout, int conv_ctas, int64_t conv_vec,
                 const uint4* __restrict__ conv_src, uint4* __restrict__ conv_dst,
                 int* __restrict__ status) {
  __shared__ float s_gscore[kWarpsPerBlock][32];
  pdl_wait();
  pdl_trigger();
  const int route_ctas = (int)gridDim.x - conv_ctas;
  if ((int)blockIdx.x >= route_ctas) {
    // The NVFP4 path's token rows: hidden_states to f16, 16 bytes at a time.
    bool over = false;
    for (int64_t v = (int64_t)(blockIdx.x - route_ctas) * blockDim.x + threadIdx.x; v < conv_vec;
         v += (int64_t)conv_ctas * blockDim.x)
      conv_dst[v] = bf16x8_to_f16x8(__ldg(conv_src + v), over);
    if (over) set_status(status, MOE_ERR_F16_RANGE);
    return;
  }
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int t = blockIdx.x * kWarpsPerBlock + wib;
  if (t >= T) return;
  const float* x = gating + (size_t)t * E;

  float key[VPL], sc[VPL];
  bool live[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    live[i] = e < E;
    const float v = live[i] ? x[e] : 0.0f;
    if (scoring == MOE_SOFTMAX) {
      sc[i] = v;
      key[i] = v;
    } else {
      const float s = key_sigmoid_f32(v);
      sc[i] = s;
      key[i] = (bias != nullptr && live[i]) ? __fadd_rn(s, bias[e]) : s;
    }
    if (key[i] != key[i]) key[i] = -INFINITY;  // NaN ranks lowest
  }

  // Grouped selection: group g = experts [g*E/G, (g+1)*E/G); score = sum of its two largest
  // keys; keep the keepG best groups (ties -> lower group id); exclude the rest.
  if (G > 1 && keepG < G && E == 32 * VPL && G == VPL) {
    // Groups of exactly 32 experts (DeepSeek-V3: 256 in 8): lane value i belongs to group i.
    // All G top-2 reductions run interleaved, every lane ends with every group's score, and
    // each lane ranks the groups itself (no shared memory, no serial selection).
    float m1[VPL], m2[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      m1[i] = key[i];
      m2[i] = -INFINITY;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const float o1 = __shfl_xor_sync(kFull, m1[i], off);
        const float o2 = __shfl_xor_sync(kFull, m2[i], off);
        const float hi = fmaxf(m1[i], o1);
        const float lo = fmaxf(fminf(m1[i], o1), fmaxf(m2[i], o2));
        m1[i] = hi;
        m2[i] = lo;
      }
    }
    float gs[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) gs[i] = __fadd_rn(m1[i], m2[i]);
#pragma unroll
    for (int g = 0; g < VPL; ++g) {
      int rank = 0;  // groups that rank before g (larger score, ties -> lower group id)
#pragma unroll
      for (int h = 0; h < VPL; ++h) rank += (h != g && before(gs[h], h, gs[g], g)) ? 1 : 0;
      if (rank >= keepG) live[g] = false;
    }
  } else if (G > 1 && keepG < G) {
    const int gsz = E / G;
    int gi[VPL];  // group of each of this lane's experts (-1 past E)
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      gi[i] = e < E ? e / gsz : -1;
    }
    for (int g = 0; g < G; ++g) {
      float m1 = -INFINITY, m2 = -INFINITY;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        if (gi[i] == g) {
          const float v = key[i];
          if (v > m1) {
            m2 = m1;
            m1 = v;
          } else if (v > m2) {
            m2 = v;
          }
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float o1 = __shfl_xor_sync(kFull, m1, off);
        const float o2 = __shfl_xor_sync(kFull, m2, off);
        const float hi = fmaxf(m1, o1);
        const float lo = fmaxf(fminf(m1, o1), fmaxf(m2, o2));
        m1 = hi;
        m2 = lo;
      }
      if (lane == 0) s_gscore[wib][g] = __fadd_rn(m1, m2);
    }
    __syncwarp();
    uint32_t kept = 0;
    for (int j = 0; j < keepG; ++j) {
      int bg = -1;
      float bs = 0.0f;
      for (int g = 0; g < G; ++g) {
        if ((kept >> g) & 1u) continue;
        const float v = s_gscore[wib][g];
        if (bg < 0 || before(v, g, bs, bg)) {
          bs = v;
          bg = g;
        }
      }
      kept |= 1u << bg;
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (gi[i] >= 0 && !((kept >> gi[i]) & 1u)) live[i] = false;
  }

  // top_k rounds of warp argmax; lane j keeps the j-th selection.
  int my_e = -1;
  float my_v = 0.0f;
  if constexpr (VPL <= 4) {
    // Each lane first sorts its candidates (best first; dead ones last), so a round compares
    // only the lanes' heads and the winning lane shifts its list down by one.  (Measured: at 8
    // values a lane its registers left the 4096-token grid a second wave, and at 12 the
    // unrolled insertion sort cost more than rescanning.)
    float hk[VPL], hs[VPL];
    int he[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      hk[i] = live[i] ? key[i] : -INFINITY;
      he[i] = live[i] ? lane + 32 * i : INT_MAX;
      hs[i] = sc[i];
    }
#pragma unroll
    for (int i = 1; i < VPL; ++i) {  // insertion sort, fully unrolled (registers only)
#pragma unroll
      for (int j = i; j > 0; --j) {
        if (before(hk[j], he[j], hk[j - 1], he[j - 1])) {
          const float tk = hk[j], ts = hs[j];
          const int te = he[j];
          hk[j] = hk[j - 1];
          he[j] = he[j - 1];
          hs[j] = hs[j - 1];
          hk[j - 1] = tk;
          he[j - 1] = te;
          hs[j - 1] = ts;
        }
      }
    }
    for (int j = 0; j < K; ++j) {
      float bk = hk[0];
      int be = he[0];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ok = __shfl_xor_sync(kFull, bk, off);
        const int oe = __shfl_xor_sync(kFull, be, off);
        if (before(ok, oe, bk, be)) {
          bk = ok;
          be = oe;
        }
      }
      const int wl = be & 31;  // the winning lane holds expert be at its head
      const float v = __shfl_sync(kFull, hs[0], wl);
      if (lane == wl) {
#pragma unroll
        for (int i = 0; i + 1 < VPL; ++i) {
          hk[i] = hk[i + 1];
          he[i] = he[i + 1];
          hs[i] = hs[i + 1];
        }
        hk[VPL - 1] = -INFINITY;
        he[VPL - 1] = INT_MAX;
      }
      if (lane == j) {
        my_e = be;
        my_v = v;
      }
    }
  } else {
    for (int j = 0; j < K; ++j) {
      float bk = -INFINITY;
      int be = INT_MAX;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        if (live[i] && (be == INT_MAX || before(key[i], e, bk, be))) {
          bk = key[i];
          be = e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ok = __shfl_xor_sync(kFull, bk, off);
        const int oe = __shfl_xor_sync(kFull, be, off);
        if (before(ok, oe, bk, be)) {
          bk = ok;
          be = oe;
        }
      }
      float cand = 0.0f;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        if (lane + 32 * i == be) {
          live[i] = false;
          cand = sc[i];
        }
      }
      const float v = __shfl_sync(kFull, cand, be & 31);
      if (lane == j) {
        my_e = be;
        my_v = v;
      }
    }
  }

  // Weights.
  float w = 0.0f;
  if (scoring == MOE_SOFTMAX) {
    const float m = __shfl_sync(kFull, my_v, 0);  // the first selection is the largest logit
    float part = 0.0f;
    if (renorm) {
      if (lane < K) part = expf(my_v - m);
    } else {
#pragma unroll
      for (int i = 0; i < VPL; ++i)
        if (lane + 32 * i < E) part += expf(sc[i] - m);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(kFull, part, off);
    w = expf(my_v - m) / part;
  } else {
    float part = lane < K ? my_v : 0.0f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(kFull, part, off);
    w = renorm ? my_v / part : my_v;
  }
  if (lane < K) {
    // Expert-parallel shard: local index, or -1 (padding) for an expert held elsewhere.
    const int le = my_e - loc0;
    ids[(size_t)t * K + lane] = (le >= 0 && le < nloc) ? le : -1;
    wout[(size_t)t * K + lane] = w * rsf;
  }
}

template <int VPL>
cudaError_t launch_vpl(const moe_problem_t& p, const float* gating, const float* bias,
                       int32_t* ids, float* w, cudaStream_t s, bool pdl, const void* hidden,
                       void* rows_f16, int* status) {
  const int G = p.num_expert_group > 1 ? p.num_expert_group : 1;
  const int keepG = G > 1 ? p.topk_group : 1;
  const int blocks = (p.T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const int loc0 = p.ep_num_local > 0 ? p.ep_local_offset : 0;
  const int nloc = local_experts(p);
  // Conversion CTAs: about two 16-byte vectors per thread, at most one wave of the SMs.
  const int64_t conv_vec = rows_f16 ? (int64_t)p.T * p.H / 8 : 0;
  const int64_t per_cta = 2ll * kWarpsPerBlock * 32;
  int64_t conv = (conv_vec + per_cta - 1) / per_cta;
  if (conv > num_sms()) conv = num_sms();
  return launch_k(route_kernel<VPL>, dim3(blocks + (int)conv), dim3(kWarpsPerBlock * 32), 0, s,
                  pdl, p.T, p.E, p.top_k, p.scoring, p.renormalize, G, keepG,
                  p.routed_scaling_factor, loc0, nloc, gating, bias, ids, w, (int)conv, conv_vec,
                  static_cast<const uint4*>(hidden), static_cast<uint4*>(rows_f16), status);
}

}  // namespace

cudaError_t launch_route(const moe_problem_t& p, const float* gating, const float* bias,
                         int32_t* ids, float* w, cudaStream_t s, bool pdl, const void* hidden,
                         void* rows_f16, int* status) {
  if (p.T == 0) return cudaSuccess;
  if (rows_f16 && (!hidden || p.H % 8 != 0)) return cudaErrorInvalidValue;
  const int need = (p.E + 31) / 32;
#define ROUTE_VPL(V) launch_vpl<V>(p, gating, bias, ids, w, s, pdl, hidden, rows_f16, status)
  if (need <= 1) return ROUTE_VPL(1);
  if (need <= 2) return ROUTE_VPL(2);
  if (need <= 4) return ROUTE_VPL(4);
  if (need <= 8) return ROUTE_VPL(8);
  if (need <= 12) return ROUTE_VPL(12);
  if (need <= 16) return ROUTE_VPL(16);
  return ROUTE_VPL(32);
#undef ROUTE_VPL
}

}  // namespace gb300moe
