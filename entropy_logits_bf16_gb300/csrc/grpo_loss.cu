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
// Launches (all on the caller's stream, no atomics on floats, no inter-CTA
// waits, every sum in a fixed order):
//  1. seq kernel, one CTA per sequence: the sequence's advantage from its
//     group's rewards, then per-token terms; per-sequence partial sums go to
//     the workspace and the unscaled per-token gradient to the output.
//  2. finalize kernel, one CTA: fixed-order sums over sequences -> loss,
//     statistics and the gradient weights.
//  3. scale kernel, one CTA per sequence (only when a gradient is requested).

#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "rlk.h"

namespace rlk {
namespace {

constexpr int LT = 256;
constexpr int LWARP = LT / 32;
constexpr int NP = kLossPartials;  // partial sums per sequence, see below
// Partial slots: 0 sum m*l, 1 sum m, 2 clip-low count, 3 clip-high count,
// 4 sum m*w, 5 TIS-capped count, 6 sum m*k3, 7 sum m*pg.

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xFFFFFFFFu, v, o);
  return v;
}

__global__ void __launch_bounds__(LT) loss_seq_kernel(LossArgs a) {
  __shared__ float s_adv;
  __shared__ float s_red[LWARP][NP];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.group_size;
  const float lo_b = 1.0f - a.eps_low, hi_b = 1.0f + a.eps_high;
  for (int s = blockIdx.x; s < a.n_seq; s += gridDim.x) {
    if (tid == 0) {
      // Group statistics in a fixed order: the mean as a double-float sum,
      // then the squared deviations from it (two passes over G rewards).
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
      s_adv = __fdiv_rn(__fsub_rn(a.rewards[s], mu), __fadd_rn(sigma, 1e-6f));
    }
    __syncthreads();
    const float A = s_adv;
    const int64_t t0 = a.seq_offsets[s], t1 = a.seq_offsets[s + 1];
    float acc[NP];
#pragma unroll
    for (int k = 0; k < NP; ++k) acc[k] = 0.f;
    for (int64_t t = t0 + tid; t < t1; t += LT) {
      const float nw = a.logp_new[t], od = a.logp_old[t];
      const float ro = a.logp_rollout[t], rf = a.logp_ref[t];
      const float m = a.mask ? (a.mask[t] ? 1.f : 0.f) : 1.f;
      const float r = expf(nw - od);
      const float rc = fminf(fmaxf(r, lo_b), hi_b);
      const float un = r * A, cl = rc * A;
      const float pg = -fminf(un, cl);
      const float gpg = (un <= cl) ? -un : 0.f;
      const float raw = expf(od - ro);
      const float w = fminf(raw, a.tis_cap);
      const float dl = rf - nw;
      const float em1 = expm1f(dl);
      const float k3 = em1 - dl;
      const float ell = w * pg + a.kl_coef * k3;
      acc[0] += m * ell;
      acc[1] += m;
      acc[2] += (A < 0.f && r < lo_b) ? m : 0.f;
      acc[3] += (A > 0.f && r > hi_b) ? m : 0.f;
      acc[4] += m * w;
      acc[5] += (raw > a.tis_cap) ? m : 0.f;
      acc[6] += m * k3;
      acc[7] += m * pg;
      if (a.out_grad) a.out_grad[t] = m * (w * gpg - a.kl_coef * em1);
    }
#pragma unroll
    for (int k = 0; k < NP; ++k) acc[k] = warp_sum(acc[k]);
    if (lane == 0)
      for (int k = 0; k < NP; ++k) s_red[warp][k] = acc[k];
    __syncthreads();
    if (tid < NP) {
      float v = 0.f;
      for (int w2 = 0; w2 < LWARP; ++w2) v += s_red[w2][tid];
      a.workspace[(int64_t)s * NP + tid] = v;
    }
    __syncthreads();
  }
}

// One CTA: fixed-order sums over the sequences' partials.
__global__ void __launch_bounds__(LT) loss_finalize_kernel(LossArgs a) {
  // Double-float (fp32 pair) sums in a fixed order: thread t takes sequences
  // t, t + LT, ...; then a shuffle tree per warp and one over the warps.
  constexpr int NV = NP + 2;   // NP partial sums, sum of per-sequence means, live sequences
  __shared__ DF s_red[LWARP][NV];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  DF acc[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) acc[k] = DF{0.f, 0.f};
  for (int s = tid; s < a.n_seq; s += LT) {
    const float* p = a.workspace + (int64_t)s * NP;
#pragma unroll
    for (int k = 0; k < NP; ++k) acc[k] = df_add_f(acc[k], p[k]);
    if (p[1] > 0.f) {
      acc[NP] = df_add_f(acc[NP], __fdiv_rn(p[0], p[1]));
      acc[NP + 1] = df_add_f(acc[NP + 1], 1.f);
    }
  }
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
    float t[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      DF v = lane < LWARP ? s_red[lane][k] : DF{0.f, 0.f};
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v = df_add(v, DF{shfl_down(v.hi, o), shfl_down(v.lo, o)});
      t[k] = __fadd_rn(v.hi, v.lo);
    }
    if (lane == 0) {
      const float M = t[1];
      float L;
      if (a.agg == RLK_AGG_TOKEN_MEAN) L = M > 0.f ? __fdiv_rn(t[0], M) : 0.f;
      else L = t[NP + 1] > 0.f ? __fdiv_rn(t[NP], t[NP + 1]) : 0.f;
      *a.out_loss = L;
      if (a.out_stats) {
        const float d = M > 0.f ? M : 1.f;
        a.out_stats[RLK_STAT_LOSS] = L;
        a.out_stats[RLK_STAT_TOKENS] = M;
        a.out_stats[RLK_STAT_CLIP_LOW] = __fdiv_rn(t[2], d);
        a.out_stats[RLK_STAT_CLIP_HIGH] = __fdiv_rn(t[3], d);
        a.out_stats[RLK_STAT_TIS_MEAN] = __fdiv_rn(t[4], d);
        a.out_stats[RLK_STAT_TIS_CAPPED] = __fdiv_rn(t[5], d);
        a.out_stats[RLK_STAT_K3_MEAN] = __fdiv_rn(t[6], d);
        a.out_stats[RLK_STAT_PG_MEAN] = __fdiv_rn(t[7], d);
      }
      float* sc = a.workspace + (int64_t)a.n_seq * NP;
      sc[0] = M > 0.f ? __fdiv_rn(1.f, M) : 0.f;   // token-mean weight
      sc[1] = t[NP + 1];                             // sequences with tokens
    }
  }
}

// Multiply each token's unscaled gradient by its weight in the loss.
__global__ void __launch_bounds__(LT) loss_scale_kernel(LossArgs a) {
  const float* sc = a.workspace + (int64_t)a.n_seq * NP;
  for (int s = blockIdx.x; s < a.n_seq; s += gridDim.x) {
    float wgt;
    if (a.agg == RLK_AGG_TOKEN_MEAN) {
      wgt = sc[0];
    } else {
      const float ms = a.workspace[(int64_t)s * NP + 1];
      wgt = ms > 0.f ? __fdiv_rn(1.f, __fmul_rn(ms, sc[1])) : 0.f;
    }
    const int64_t t0 = a.seq_offsets[s], t1 = a.seq_offsets[s + 1];
    for (int64_t t = t0 + threadIdx.x; t < t1; t += LT) a.out_grad[t] *= wgt;
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
  if (a.n_seq > 0) loss_seq_kernel<<<grid, LT, 0, stream>>>(a);
  loss_finalize_kernel<<<1, LT, 0, stream>>>(a);
  if (a.out_grad && a.n_seq > 0) loss_scale_kernel<<<grid, LT, 0, stream>>>(a);
  return cudaGetLastError();
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
  if (n_seq < 0 || n_seq > RLK_NOALLOC_MAX_SEQ || group_size < 1 || n_seq % group_size != 0 ||
      n_tok < 0)
    return RLK_ERR_INVALID_ARG;
  if (!(isfinite(eps_low) && eps_low >= 0.0f && isfinite(eps_high) && eps_high >= 0.0f))
    return RLK_ERR_INVALID_ARG;
  if (!(isfinite(tis_cap) && tis_cap > 0.0f) || !(isfinite(kl_coef) && kl_coef >= 0.0f))
    return RLK_ERR_INVALID_ARG;
  if (agg != RLK_AGG_TOKEN_MEAN && agg != RLK_AGG_SEQ_MEAN_TOKEN_MEAN) return RLK_ERR_INVALID_ARG;
  if (!seq_offsets || !out_loss) return RLK_ERR_INVALID_ARG;
  if (n_seq > 0 && (!logp_new || !logp_old || !logp_rollout || !logp_ref || !rewards))
    return RLK_ERR_INVALID_ARG;
  cudaError_t err;
  float* scratch = rlk::noalloc_scratch(err);
  if (!scratch) return RLK_ERR_CUDA;
  rlk::LossArgs a;
  a.logp_new = logp_new;
  a.logp_old = logp_old;
  a.logp_rollout = logp_rollout;
  a.logp_ref = logp_ref;
  a.mask = loss_mask;
  a.rewards = rewards;
  a.seq_offsets = seq_offsets;
  a.n_seq = n_seq;
  a.group_size = group_size;
  a.n_tok = n_tok;
  a.eps_low = eps_low;
  a.eps_high = eps_high;
  a.tis_cap = tis_cap;
  a.kl_coef = kl_coef;
  a.agg = agg;
  a.out_loss = out_loss;
  a.out_grad = out_dloss_dlogp_new;
  a.out_stats = out_stats;
  a.workspace = scratch;
  return rlk::launch_grpo_loss(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RLK_OK
             : RLK_ERR_CUDA;
}
