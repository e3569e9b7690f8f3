// rlk_grpo_loss kernels: GRPO/DAPO clipped-ratio loss with truncated
// importance sampling (TIS) and the k3 KL estimate.
//
// Method: GRPO with standard-deviation-normalised group advantages and KL
// coefficient 0.01 (RL-Kernel "ROCm sparse performance" notes); TIS clips large
// importance ratios (LumenRL README, section "Rollout Correction"); the loss
// backward seed is normalised before model derivatives (RL-Kernel "Qwen3-8B
// VIME train-rollout consistency", section "Canonical topology strategy"), so
// the gradient written here already carries the aggregation weight.
//
// Launches (all on the caller's stream, each a programmatic dependent of the
// one before, which it waits for before reading; no atomics on floats, no
// waits between CTAs of one launch, every sum in a fixed order):
//  1. seq kernel, one CTA per sequence: the sequence's advantage from its
//     group's rewards, then per-token terms; per-sequence partial sums (and
//     the advantage) go to the workspace.
//  2. finalize kernel, one CTA: fixed-order sums over sequences, then over
//     the aggregation units -> loss, statistics, the gradient weights.
//  3. grad kernel, one CTA per sequence (only when a gradient is requested):
//     each token's gradient, recomputed from the inputs, times its weight.
//
// The variants (policy term, importance weight, baseline, aggregation) follow
// the prime-rl v0.10.0 release notes, section "2. RL Algorithms" (IPO mask
// |pi_train(y) - pi_infer(y)| > eps; IcePop's ratio band; length-weighted
// baseline; prompt-mean aggregation) and the LumenRL README, section "Rollout
// Correction" (TIS caps the ratio, MIS normalises it).

#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "rlk.h"

namespace rlk {
namespace {

constexpr int LT = 256;
constexpr int LWARP = LT / 32;
constexpr int NP = kLossPartials;  // partial sums per sequence, see below
// Partial slots: 0 sum m l (MIS: sum m kl_coef k3 only), 1 sum m, 2 clip-low
// count, 3 clip-high count, 4 sum m w (MIS: sum m raw), 5 capped count,
// 6 sum m k3, 7 sum m pg, 8 count dropped by the IPO / IcePop mask,
// 9 sum m raw pg (MIS), 10 the sequence's advantage, 11 1 when the
// sequence's offsets are out of order or outside the n_tok packed tokens.
// Scalars after the partials: 0 1 / sum m, 1 live aggregation units,
// 2 the importance-weight scale (1 / mean raw for MIS, else 1).

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xFFFFFFFFu, v, o);
  return v;
}

// The per-token policy term: pg, its derivative in logp_new (g), the mask
// value (keep) and the raw importance ratio exp(old - rollout).
struct TokTerms {
  float pg, g, keep, r, raw;
};
__device__ __forceinline__ TokTerms token_terms(const LossArgs& a, float A, float nw, float od,
                                                float ro) {
  TokTerms t;
  t.r = expf(nw - od);
  t.raw = expf(od - ro);
  t.keep = 1.f;
  if (a.loss_type == RLK_LOSS_IPO) {
    const float rho = expf(nw - ro);
    t.keep = fabsf(expf(nw) - expf(ro)) <= a.ipo_eps ? 1.f : 0.f;
    t.pg = -(t.keep * rho * A);
    t.g = t.pg;
  } else {
    const float rc = fminf(fmaxf(t.r, 1.0f - a.eps_low), 1.0f + a.eps_high);
    const float un = t.r * A, cl = rc * A;
    t.pg = -fminf(un, cl);
    t.g = (un <= cl) ? -un : 0.f;
    if (a.loss_type == RLK_LOSS_ICEPOP) {
      const float rho = expf(nw - ro);
      t.keep = (rho >= a.band_low && rho <= a.band_high) ? 1.f : 0.f;
      t.pg *= t.keep;
      t.g *= t.keep;
    }
  }
  return t;
}

// The importance weight for everything but MIS (whose scale is known only
// after the batch reduction).
__device__ __forceinline__ float is_weight(const LossArgs& a, float raw) {
  return a.is_method == RLK_IS_TIS ? fminf(raw, a.tis_cap) : 1.f;
}

// Sequence s's packed tokens [t0, t1), clamped to the n_tok tokens that start
// at seq_offsets[0]; returns whether the offsets were valid (non-decreasing
// and inside that range).  Invalid offsets make the loss NaN, and no token
// outside the range is read or written.
__device__ __forceinline__ bool seq_range(const LossArgs& a, int s, int64_t& t0, int64_t& t1) {
  const int64_t base = a.seq_offsets[0], lim = base + a.n_tok;
  t0 = a.seq_offsets[s];
  t1 = a.seq_offsets[s + 1];
  const bool ok = t0 >= base && t1 >= t0 && t1 <= lim;
  t0 = t0 < base ? base : (t0 > lim ? lim : t0);
  t1 = t1 < t0 ? t0 : (t1 > lim ? lim : t1);
  return ok;
}

__global__ void __launch_bounds__(LT) loss_seq_kernel(LossArgs a) {
  pdl_trigger();
  pdl_wait();   // the log-probabilities may come from the kernel before
  __shared__ float s_adv;
  __shared__ float s_red[LWARP][NP];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.group_size;
  const bool mis = a.is_method == RLK_IS_MIS;
  for (int s = blockIdx.x; s < a.n_seq; s += gridDim.x) {
    if (tid == 0) {
      // Group statistics in a fixed order: the mean as a double-float sum,
      // then the squared deviations from it (two passes over G rewards); the
      // length-weighted baseline weights each reward by its packed length.
      const int s0 = (s / G) * G;
      DF sum{0.f, 0.f};
      for (int j = 0; j < G; ++j) sum = df_add_f(sum, a.rewards[s0 + j]);
      const float mu = __fdiv_rn(__fadd_rn(sum.hi, sum.lo), (float)G);
      float ss = 0.f;
      for (int j = 0; j < G; ++j) {
        const float d = __fsub_rn(a.rewards[s0 + j], mu);
        ss = __fmaf_rn(d, d, ss);
      }
      const float sigma = G > 1 ? sqrtf(__fdiv_rn(ss, (float)(G - 1))) : 0.f;
      float b = mu;
      if (a.baseline == RLK_BASELINE_LENGTH_WEIGHTED) {
        DF lw{0.f, 0.f};
        float ln = 0.f;   // lengths are integers: exact in fp32 up to 2^24 tokens a group
        for (int j = 0; j < G; ++j) {
          const float len = (float)(a.seq_offsets[s0 + j + 1] - a.seq_offsets[s0 + j]);
          lw = df_add_f(lw, __fmul_rn(len, a.rewards[s0 + j]));
          ln = __fadd_rn(ln, len);
        }
        if (ln > 0.f) b = __fdiv_rn(__fadd_rn(lw.hi, lw.lo), ln);
      }
      s_adv = __fdiv_rn(__fsub_rn(a.rewards[s], b), __fadd_rn(sigma, 1e-6f));
    }
    __syncthreads();
    const float A = s_adv;
    int64_t t0, t1;
    const bool range_ok = seq_range(a, s, t0, t1);
    float acc[NP];
#pragma unroll
    for (int k = 0; k < NP; ++k) acc[k] = 0.f;
    const float lo_b = 1.0f - a.eps_low, hi_b = 1.0f + a.eps_high;
    const bool clipped_type = a.loss_type != RLK_LOSS_IPO;
    for (int64_t t = t0 + tid; t < t1; t += LT) {
      const float nw = a.logp_new[t], od = a.logp_old[t];
      const float ro = a.logp_rollout[t], rf = a.logp_ref[t];
      const float m = a.mask ? (a.mask[t] ? 1.f : 0.f) : 1.f;
      const TokTerms tt = token_terms(a, A, nw, od, ro);
      const float dl = rf - nw;
      const float k3 = expm1f(dl) - dl;
      if (mis) {
        acc[0] += m * (a.kl_coef * k3);
        acc[4] += m * tt.raw;
        acc[9] += m * (tt.raw * tt.pg);
      } else {
        const float w = is_weight(a, tt.raw);
        acc[0] += m * (w * tt.pg + a.kl_coef * k3);
        acc[4] += m * w;
      }
      acc[1] += m;
      if (clipped_type) {
        acc[2] += (A < 0.f && tt.r < lo_b) ? m : 0.f;
        acc[3] += (A > 0.f && tt.r > hi_b) ? m : 0.f;
      }
      acc[5] += (a.is_method == RLK_IS_TIS && tt.raw > a.tis_cap) ? m : 0.f;
      acc[6] += m * k3;
      acc[7] += m * tt.pg;
      acc[8] += m * (1.f - tt.keep);
    }
#pragma unroll
    for (int k = 0; k < NP; ++k) acc[k] = warp_sum(acc[k]);
    if (lane == 0)
      for (int k = 0; k < NP; ++k) s_red[warp][k] = acc[k];
    __syncthreads();
    if (tid < NP) {
      float v = 0.f;
      for (int w2 = 0; w2 < LWARP; ++w2) v += s_red[w2][tid];
      a.workspace[(int64_t)s * NP + tid] = tid == 10 ? A : (tid == 11 ? (range_ok ? 0.f : 1.f) : v);
    }
    __syncthreads();
  }
}

// A sequence's sum of m l, given the MIS scale (1 when not MIS).
__device__ __forceinline__ float seq_lsum(const float* p, bool mis, float scale) {
  return mis ? __fmaf_rn(p[9], scale, p[0]) : p[0];
}

// Fixed-order double-float reduction of NV values over the CTA; valid on
// thread 0.
template <int NV>
__device__ void cta_sum_df(DF (&acc)[NV], DF (*s_red)[NV], float (&out)[NV]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      acc[k] = df_add(acc[k], DF{shfl_down(acc[k].hi, o), shfl_down(acc[k].lo, o)});
  }
  if (lane == 0)
    for (int k = 0; k < NV; ++k) s_red[warp][k] = acc[k];
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      DF v = lane < LWARP ? s_red[lane][k] : DF{0.f, 0.f};
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v = df_add(v, DF{shfl_down(v.hi, o), shfl_down(v.lo, o)});
      out[k] = __fadd_rn(v.hi, v.lo);
    }
  }
  __syncthreads();
}

// One CTA: fixed-order sums over the sequences' partials, then (the MIS scale
// being known) over the aggregation units: the batch, sequences or groups.
__global__ void __launch_bounds__(LT) loss_finalize_kernel(LossArgs a) {
  pdl_trigger();
  pdl_wait();   // the sequences' partials
  __shared__ DF s_red1[LWARP][NP];
  __shared__ DF s_red2[LWARP][2];
  __shared__ float s_t[NP];
  const int tid = threadIdx.x;
  DF acc[NP];
#pragma unroll
  for (int k = 0; k < NP; ++k) acc[k] = DF{0.f, 0.f};
  for (int s = tid; s < a.n_seq; s += LT) {
    const float* p = a.workspace + (int64_t)s * NP;
#pragma unroll
    for (int k = 0; k < NP; ++k) acc[k] = df_add_f(acc[k], p[k]);
  }
  float t[NP];
  cta_sum_df<NP>(acc, s_red1, t);
  if (tid == 0)
    for (int k = 0; k < NP; ++k) s_t[k] = t[k];
  __syncthreads();
  const bool mis = a.is_method == RLK_IS_MIS;
  const float M = s_t[1];
  // MIS: w = raw / (sum m raw / sum m)
  const float scale = mis && s_t[4] > 0.f ? __fdiv_rn(M, s_t[4]) : 1.f;
  // Aggregation units: the batch (token mean) sums every sequence's m l;
  // sequences or groups add their own token means.
  const int per = a.agg == RLK_AGG_PROMPT_MEAN ? a.group_size : 1;
  const int n_unit = a.agg == RLK_AGG_TOKEN_MEAN ? a.n_seq : a.n_seq / per;
  DF u2[2] = {DF{0.f, 0.f}, DF{0.f, 0.f}};   // sum of unit values, live units
  for (int u = tid; u < n_unit; u += LT) {
    float ls = 0.f, ms = 0.f;
    for (int j = 0; j < per; ++j) {
      const float* p = a.workspace + (int64_t)(u * per + j) * NP;
      ls = __fadd_rn(ls, seq_lsum(p, mis, scale));
      ms = __fadd_rn(ms, p[1]);
    }
    if (a.agg == RLK_AGG_TOKEN_MEAN) {
      u2[0] = df_add_f(u2[0], ls);
    } else if (ms > 0.f) {
      u2[0] = df_add_f(u2[0], __fdiv_rn(ls, ms));
      u2[1] = df_add_f(u2[1], 1.f);
    }
  }
  float v[2];
  cta_sum_df<2>(u2, s_red2, v);
  if (tid == 0) {
    float L;
    if (a.agg == RLK_AGG_TOKEN_MEAN) L = M > 0.f ? __fdiv_rn(v[0], M) : 0.f;
    else L = v[1] > 0.f ? __fdiv_rn(v[0], v[1]) : 0.f;
    const bool bad_offsets = s_t[11] != 0.f;   // some sequence's offsets were invalid
    if (bad_offsets) L = NAN;
    *a.out_loss = L;
    if (a.out_stats) {
      const float d = bad_offsets ? NAN : (M > 0.f ? M : 1.f);
      a.out_stats[RLK_STAT_LOSS] = L;
      a.out_stats[RLK_STAT_TOKENS] = bad_offsets ? NAN : M;
      a.out_stats[RLK_STAT_CLIP_LOW] = __fdiv_rn(s_t[2], d);
      a.out_stats[RLK_STAT_CLIP_HIGH] = __fdiv_rn(s_t[3], d);
      a.out_stats[RLK_STAT_TIS_MEAN] = __fdiv_rn(__fmul_rn(s_t[4], scale), d);
      a.out_stats[RLK_STAT_TIS_CAPPED] = __fdiv_rn(s_t[5], d);
      a.out_stats[RLK_STAT_K3_MEAN] = __fdiv_rn(s_t[6], d);
      a.out_stats[RLK_STAT_PG_MEAN] = __fdiv_rn(s_t[7], d);
      if (a.nstats > RLK_STAT_MASK_DROPPED)
        a.out_stats[RLK_STAT_MASK_DROPPED] = __fdiv_rn(s_t[8], d);
    }
    float* sc = a.workspace + (int64_t)a.n_seq * NP;
    sc[0] = bad_offsets ? NAN : (M > 0.f ? __fdiv_rn(1.f, M) : 0.f);   // token-mean weight
    sc[1] = bad_offsets ? NAN : v[1];                                    // live sequences or groups
    sc[2] = scale;
  }
}

// Each token's gradient with its weight in the loss, recomputed from the
// inputs (the weight and the MIS scale are known only after the reduction).
__global__ void __launch_bounds__(LT) loss_grad_kernel(LossArgs a) {
  pdl_trigger();
  pdl_wait();   // the batch sums
  const float* sc = a.workspace + (int64_t)a.n_seq * NP;
  const bool mis = a.is_method == RLK_IS_MIS;
  for (int s = blockIdx.x; s < a.n_seq; s += gridDim.x) {
    const float* p = a.workspace + (int64_t)s * NP;
    float wgt;
    if (a.agg == RLK_AGG_TOKEN_MEAN) {
      wgt = sc[0];
    } else {
      float mu = p[1];   // the unit's token count: the sequence's, or its group's
      if (a.agg == RLK_AGG_PROMPT_MEAN) {
        const int s0 = (s / a.group_size) * a.group_size;
        mu = 0.f;
        for (int j = 0; j < a.group_size; ++j) mu = __fadd_rn(mu, a.workspace[(int64_t)(s0 + j) * NP + 1]);
      }
      wgt = mu > 0.f ? __fdiv_rn(1.f, __fmul_rn(mu, sc[1])) : 0.f;
    }
    const float A = p[10];
    int64_t t0, t1;
    seq_range(a, s, t0, t1);
    for (int64_t t = t0 + threadIdx.x; t < t1; t += LT) {
      const float nw = a.logp_new[t], od = a.logp_old[t];
      const float ro = a.logp_rollout[t], rf = a.logp_ref[t];
      const float m = a.mask ? (a.mask[t] ? 1.f : 0.f) : 1.f;
      const TokTerms tt = token_terms(a, A, nw, od, ro);
      const float w = mis ? __fmul_rn(tt.raw, sc[2]) : is_weight(a, tt.raw);
      const float em1 = expm1f(rf - nw);
      a.out_grad[t] = wgt * (m * (w * tt.g - a.kl_coef * em1));
    }
  }
}

}  // namespace

size_t loss_workspace_bytes(int64_t n_seq) {
  const size_t floats = (size_t)n_seq * NP + 4;
  return (floats * sizeof(float) + 255) & ~(size_t)255;
}

cudaError_t launch_grpo_loss(const LossArgs& a, cudaStream_t stream) {
  const int cap = 8 * sm_count();
  const int grid = a.n_seq < cap ? (a.n_seq > 0 ? a.n_seq : 1) : cap;
  // each launch overlaps the end of the kernel before it (programmatic
  // dependent launch; every kernel waits for its predecessor's writes)
  cudaError_t e = cudaSuccess;
  if (a.n_seq > 0) e = launch_after(loss_seq_kernel, dim3(grid), dim3(LT), 0, stream, a);
  if (e == cudaSuccess) e = launch_after(loss_finalize_kernel, dim3(1), dim3(LT), 0, stream, a);
  if (e == cudaSuccess && a.out_grad && a.n_seq > 0)
    e = launch_after(loss_grad_kernel, dim3(grid), dim3(LT), 0, stream, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace rlk

// ---------------------------------------------------------------------------
// rlk_grpo_loss_noalloc: the same loss for callers that cannot allocate device
// memory -- a framework that has reserved the whole device for its own pool
// (cudaMalloc would fail or take memory the pool counts on), code that runs
// inside an allocator callback (allocating there would re-enter the
// allocator), or a latency-critical loop that bans cudaMalloc because it may
// synchronise the device.  The caller passes inputs and outputs only; the
// per-sequence partial sums live in the static array below, which every GPU
// that loads the library holds until the process exits.
//
// The kernels write every partial sum and every scalar before reading it, so
// nothing in the array has to start at zero; the array keeps the last call's
// contents.  All calls share it: calls whose work overlaps on the GPU (on
// different streams or from different host threads) race and give wrong
// results, so callers must serialise them.

#include <atomic>

namespace rlk {
namespace {

constexpr int kNoallocFloats = RLK_NOALLOC_MAX_SEQ * NP + 4;
static __device__ __align__(256) float g_noalloc_scratch[kNoallocFloats];

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
float* noalloc_scratch(cudaError_t& err) {
  static std::atomic<float*> cache[64];
  int dev = -1;
  err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    err = cudaErrorInvalidDevice;
    return nullptr;
  }
  float* p = cache[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* addr = nullptr;
  err = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
  if (err != cudaSuccess) return nullptr;
  p = static_cast<float*>(addr);
  cache[dev].store(p, std::memory_order_release);
  return p;
}

}  // namespace
}  // namespace rlk

extern "C" rlk_status rlk_grpo_loss_noalloc(
    const float* logp_new, const float* logp_old, const float* logp_rollout,
    const float* logp_ref, const uint8_t* loss_mask, const float* rewards,
    const int32_t* seq_offsets, int32_t n_seq, int32_t group_size, int64_t n_tok,
    float eps_low, float eps_high, float tis_cap, float kl_coef, rlk_agg agg, float* out_loss,
    float* out_dloss_dlogp_new, float* out_stats, rlk_stream stream) {
  if (n_seq > RLK_NOALLOC_MAX_SEQ) return RLK_ERR_INVALID_ARG;
  rlk::LossArgs a;
  const int st = rlk::grpo_loss_args(logp_new, logp_old, logp_rollout, logp_ref, loss_mask,
                                     rewards, seq_offsets, n_seq, group_size, n_tok, eps_low,
                                     eps_high, tis_cap, kl_coef, (int)agg, out_loss,
                                     out_dloss_dlogp_new, out_stats, a);
  if (st != RLK_OK) return (rlk_status)st;
  cudaError_t err;
  float* scratch = rlk::noalloc_scratch(err);
  if (!scratch) return RLK_ERR_CUDA;
  a.workspace = scratch;
  if (rlk::take_injected_failure()) return RLK_ERR_CUDA;
  return rlk::launch_grpo_loss(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RLK_OK
             : RLK_ERR_CUDA;
}
