// The canonical vocabulary partition for the top_p = 1 path.
//
// RL-Kernel "Qwen3-8B VIME train-rollout consistency", section "Canonical
// topology strategy": the launcher fixes a virtual tensor-parallel degree of 8
// and a padded vocabulary of 152576 for every physical topology; a physical
// rank executes its adjacent virtual shards separately and combines them in
// the same fixed order, and the selected-token log-probability uses the same
// virtual partition.  So a shard's partial depends only on that shard's
// logits, and the row's result only on the partials taken in shard order: the
// same bits whatever the physical degree.
//
// shard_partial_kernel: one warp per (row, shard) pair.  The shard's columns
// are folded into an online state (max m, sum of 2^d as a double-float, sum of
// 2^d d; d = (z - m) log2(e) / T) per lane, merged along a fixed tree, plus the
// selected logit when the selected id lies in the shard.  shard_combine_kernel: one thread per row merges the row's partials
// in shard order and writes the log-probability and entropy.

#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "rlk.h"

namespace rlk {
namespace {

constexpr int NTP = 256;
constexpr int NWP = NTP / 32;

struct Part {
  float m, hi, lo, u;
};

__device__ __forceinline__ bool part_empty(const Part& a) {
  return a.m == -INFINITY && a.hi == 0.f && a.lo == 0.f && a.u == 0.f;
}

// Merge b into a (a is the left operand; the caller fixes the order).
__device__ __forceinline__ Part part_merge(const Part& a, const Part& b, float c) {
  if (part_empty(b)) return a;
  if (part_empty(a)) return b;
  const float M = fmaxf(a.m, b.m);
  const float da = __fmul_rn(__fsub_rn(M, a.m), c);
  const float db = __fmul_rn(__fsub_rn(M, b.m), c);
  const float fa = (a.m == M) ? 1.f : ex2(-da);
  const float fb = (b.m == M) ? 1.f : ex2(-db);
  const float sa = __fadd_rn(a.hi, a.lo), sb = __fadd_rn(b.hi, b.lo);
  Part r;
  r.m = M;
  r.u = __fadd_rn(__fmul_rn(fa, __fmaf_rn(-da, sa, a.u)), __fmul_rn(fb, __fmaf_rn(-db, sb, b.u)));
  float s, e;
  two_sum(__fmul_rn(a.hi, fa), __fmul_rn(b.hi, fb), s, e);
  e = __fadd_rn(e, __fadd_rn(__fmul_rn(a.lo, fa), __fmul_rn(b.lo, fb)));
  r.hi = __fadd_rn(s, e);
  r.lo = __fsub_rn(e, __fsub_rn(r.hi, s));
  return r;
}

// Fold n (<= 8) values into the state: one rescale per group of eight.
__device__ __forceinline__ void part_absorb8(Part& st, const float (&v)[8], int n, float c) {
  float gm = -INFINITY;
  bool fin = true;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (k < n) {
      gm = fmaxf(gm, v[k]);
      fin = fin && isfinite(v[k]);
    }
  }
  if (!fin) {   // a non-finite logit: the row has no distribution
    st.u = NAN;
    return;
  }
  if (gm == -INFINITY) return;
  if (gm > st.m) {
    if (st.m != -INFINITY) {
      const float delta = __fmul_rn(__fsub_rn(gm, st.m), c);
      const float f = ex2(-delta);
      st.u = __fmul_rn(f, __fmaf_rn(-delta, __fadd_rn(st.hi, st.lo), st.u));
      st.hi = __fmul_rn(st.hi, f);
      st.lo = __fmul_rn(st.lo, f);
    }
    st.m = gm;
  }
  float w[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float d = k < n ? __fmul_rn(__fsub_rn(v[k], st.m), c) : 0.f;
    w[k] = k < n ? ex2(d) : 0.f;
    st.u = __fmaf_rn(w[k], d, st.u);
  }
  const float s4 = __fadd_rn(__fadd_rn(__fadd_rn(w[0], w[1]), __fadd_rn(w[2], w[3])),
                             __fadd_rn(__fadd_rn(w[4], w[5]), __fadd_rn(w[6], w[7])));
  float s, e;
  two_sum(st.hi, s4, s, e);
  st.hi = s;
  st.lo = __fadd_rn(st.lo, e);
}

// Fold one packed group of eight bf16 into the state with packed arithmetic:
// bf16x2 max / min (the NaN-propagating max flags NaN, the extremes flag
// +-inf), then d = z c - E with E = fp32(m c) as fp32x2 fmas.
__device__ __forceinline__ void part_absorb_packed(Part& st, const uint4 q, float c) {
  const __nv_bfloat162 mx = __hmax2_nan(__hmax2_nan(bf2(q.x), bf2(q.y)),
                                        __hmax2_nan(bf2(q.z), bf2(q.w)));
  const __nv_bfloat162 mn = __hmin2(__hmin2(bf2(q.x), bf2(q.y)), __hmin2(bf2(q.z), bf2(q.w)));
  const float gm = fmaxf(__low2float(mx), __high2float(mx));
  const float gn = fminf(__low2float(mn), __high2float(mn));
  if (!(isfinite(__low2float(mx)) && isfinite(__high2float(mx)) && isfinite(gn))) {
    st.u = NAN;   // a non-finite logit: the row has no distribution
    return;
  }
  if (gm > st.m) {
    if (st.m != -INFINITY) {
      const float delta = __fmul_rn(__fsub_rn(gm, st.m), c);
      const float f = ex2(-delta);
      st.u = __fmul_rn(f, __fmaf_rn(-delta, __fadd_rn(st.hi, st.lo), st.u));
      st.hi = __fmul_rn(st.hi, f);
      st.lo = __fmul_rn(st.lo, f);
    }
    st.m = gm;
  }
  // d relative to m itself: E = fp32(m c), and fma(z, c, -E) differs from
  // (z - m) c by the rounding of E, which every term and the rescales share
  const float E = __fmul_rn(st.m, c);
  const float2 c2 = make_float2(c, c), nE2 = make_float2(-E, -E);
  const float2 d0 = __ffma2_rn(bf16x2_to_f2(q.x), c2, nE2);
  const float2 d1 = __ffma2_rn(bf16x2_to_f2(q.y), c2, nE2);
  const float2 d2 = __ffma2_rn(bf16x2_to_f2(q.z), c2, nE2);
  const float2 d3 = __ffma2_rn(bf16x2_to_f2(q.w), c2, nE2);
  const float2 w0 = make_float2(ex2(d0.x), ex2(d0.y)), w1 = make_float2(ex2(d1.x), ex2(d1.y));
  const float2 w2 = make_float2(ex2(d2.x), ex2(d2.y)), w3 = make_float2(ex2(d3.x), ex2(d3.y));
  float2 u2 = __fmul2_rn(w0, d0);
  u2 = __ffma2_rn(w1, d1, u2);
  u2 = __ffma2_rn(w2, d2, u2);
  u2 = __ffma2_rn(w3, d3, u2);
  const float2 s2 = __fadd2_rn(__fadd2_rn(w0, w1), __fadd2_rn(w2, w3));
  st.u = __fadd_rn(st.u, __fadd_rn(u2.x, u2.y));
  float s, e;
  two_sum(st.hi, __fadd_rn(s2.x, s2.y), s, e);
  st.hi = s;
  st.lo = __fadd_rn(st.lo, e);
}

// One warp per (row, shard) pair; lane l takes the 8-column groups l, l + 32,
// ... of the shard (four 16-byte loads in flight), and the lanes' states
// merge along a fixed shuffle tree.
__global__ void __launch_bounds__(NTP) shard_partial_kernel(ShardArgs a, float c) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t n_pairs = a.T * (int64_t)a.n_shards;
  const int64_t nwarps = (int64_t)gridDim.x * NWP;
  for (int64_t pr = (int64_t)blockIdx.x * NWP + warp; pr < n_pairs; pr += nwarps) {
    const int64_t r = pr / a.n_shards;
    const int s = (int)(pr % a.n_shards);
    // the shard's columns, local to the logits given: [l0, l1)
    const int64_t g0 = a.first_col + (int64_t)s * a.shard_width;   // global index
    const int64_t l0 = (int64_t)s * a.shard_width;
    int64_t l1 = l0 + a.shard_width;
    if (g0 + a.shard_width > a.V) l1 = a.V - a.first_col;          // padding is not a column
    if (l1 < l0) l1 = l0;
    Part st{-INFINITY, 0.f, 0.f, 0.f};
    if (a.dtype == 0) {
      const uint16_t* p = reinterpret_cast<const uint16_t*>(a.logits) + r * a.ld;
      const bool vec = ((reinterpret_cast<uintptr_t>(p + l0)) & 15u) == 0;
      int64_t j = l0 + (int64_t)lane * 8;
      if (vec) {
        constexpr int B = 4;
        for (; j + (int64_t)(B - 1) * 256 + 8 <= l1; j += (int64_t)B * 256) {
          uint4 q[B];
#pragma unroll
          for (int b = 0; b < B; ++b)
            q[b] = __ldg(reinterpret_cast<const uint4*>(p + j + (int64_t)b * 256));
#pragma unroll
          for (int b = 0; b < B; ++b) part_absorb_packed(st, q[b], c);
        }
        for (; j + 8 <= l1; j += 256) part_absorb_packed(st, __ldg(reinterpret_cast<const uint4*>(p + j)), c);
      }
      for (; j < l1; j += 256) {
        float v[8];
        const int n = (int)(l1 - j < 8 ? l1 - j : 8);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = k < n ? bf16_val(__ldg(p + j + k)) : -INFINITY;
        part_absorb8(st, v, n, c);
      }
    } else {
      const float* p = reinterpret_cast<const float*>(a.logits) + r * a.ld;
      for (int64_t j = l0 + (int64_t)lane * 8; j < l1; j += 256) {
        float v[8];
        const int n = (int)(l1 - j < 8 ? l1 - j : 8);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = k < n ? __ldg(p + j + k) : -INFINITY;
        part_absorb8(st, v, n, c);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const Part x{shfl_down(st.m, o), shfl_down(st.hi, o), shfl_down(st.lo, o), shfl_down(st.u, o)};
      st = part_merge(st, x, c);
    }
    if (lane == 0) {
      // the selected logit, when the selected id is one of this shard's columns
      const int64_t y = a.ids[r];
      float zy = NAN;
      if (y >= a.first_col + l0 && y < a.first_col + l1) {
        const int64_t jy = y - a.first_col;
        zy = a.dtype == 0
                 ? bf16_val(reinterpret_cast<const uint16_t*>(a.logits)[r * a.ld + jy])
                 : reinterpret_cast<const float*>(a.logits)[r * a.ld + jy];
      }
      float4* o = reinterpret_cast<float4*>(a.partials) + 2 * ((int64_t)s * a.T + r);
      o[0] = make_float4(st.m, st.hi, st.lo, st.u);
      o[1] = make_float4(zy, isnan(zy) ? 0.f : 1.f, 0.f, 0.f);   // every column is in S
    }
  }
}

// Fold one value into a lane's state.
__device__ __forceinline__ void part_absorb1(Part& st, float z, float c) {
  if (!isfinite(z)) {
    st.u = NAN;
    return;
  }
  if (z > st.m) {
    if (st.m != -INFINITY) {
      const float delta = __fmul_rn(__fsub_rn(z, st.m), c);
      const float f = ex2(-delta);
      st.u = __fmul_rn(f, __fmaf_rn(-delta, __fadd_rn(st.hi, st.lo), st.u));
      st.hi = __fmul_rn(st.hi, f);
      st.lo = __fmul_rn(st.lo, f);
    }
    st.m = z;
  }
  const float d = __fmul_rn(__fsub_rn(z, st.m), c);
  const float w = ex2(d);
  float s, e;
  two_sum(st.hi, w, s, e);
  st.hi = s;
  st.lo = __fadd_rn(st.lo, e);
  st.u = __fmaf_rn(w, d, st.u);
}

// The retained set supplied by the sampler (CSR), under the same partition:
// one warp per (row, shard); lane l takes list positions l, l + 32, ... and
// keeps those in the shard's columns.  The list's checks (empty, decreasing
// offsets, an id outside [0, V)) are the row's, made by every shard alike.
__global__ void __launch_bounds__(NTP) shard_support_partial_kernel(ShardArgs a, float c) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t n_pairs = a.T * (int64_t)a.n_shards;
  const int64_t nwarps = (int64_t)gridDim.x * NWP;
  for (int64_t pr = (int64_t)blockIdx.x * NWP + warp; pr < n_pairs; pr += nwarps) {
    const int64_t r = pr / a.n_shards;
    const int s = (int)(pr % a.n_shards);
    const int64_t g0 = a.first_col + (int64_t)s * a.shard_width;   // global columns [g0, g1)
    int64_t g1 = g0 + a.shard_width;
    if (g1 > a.V) g1 = a.V;
    const int64_t j0 = a.offsets[r], j1 = a.offsets[r + 1];
    const int64_t y = a.ids[r];
    Part st{-INFINITY, 0.f, 0.f, 0.f};
    uint32_t bad = j1 <= j0 ? RLK_STATUS_BAD_SUPPORT : 0u;
    bool y_here = false;
    for (int64_t j = j0 + lane; j < j1; j += 32) {
      const int64_t id = a.support[j];
      if (id < 0 || id >= a.V) {
        bad |= RLK_STATUS_BAD_SUPPORT;
        continue;
      }
      if (id < g0 || id >= g1) continue;
      const int64_t col = (id - a.first_col);
      const float z = a.dtype == 0
                          ? bf16_val(__ldg(reinterpret_cast<const uint16_t*>(a.logits) + r * a.ld + col))
                          : __ldg(reinterpret_cast<const float*>(a.logits) + r * a.ld + col);
      part_absorb1(st, z, c);
      if (id == y) y_here = true;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const Part x{shfl_down(st.m, o), shfl_down(st.hi, o), shfl_down(st.lo, o), shfl_down(st.u, o)};
      st = part_merge(st, x, c);
    }
    bad = __reduce_or_sync(0xFFFFFFFFu, bad);
    y_here = __any_sync(0xFFFFFFFFu, y_here);
    if (lane == 0) {
      float zy = NAN;
      if (y_here) {
        const int64_t col = y - a.first_col;
        zy = a.dtype == 0
                 ? bf16_val(reinterpret_cast<const uint16_t*>(a.logits)[r * a.ld + col])
                 : reinterpret_cast<const float*>(a.logits)[r * a.ld + col];
      }
      float4* o = reinterpret_cast<float4*>(a.partials) + 2 * ((int64_t)s * a.T + r);
      o[0] = make_float4(st.m, st.hi, st.lo, st.u);
      o[1] = make_float4(zy, y_here ? 1.f : 0.f, __uint_as_float(bad), 0.f);
    }
  }
}

// One thread per row: the row's partials merged in shard order.
__global__ void __launch_bounds__(256) shard_combine_kernel(ShardCombineArgs a, float c) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= a.T) return;
  const int64_t y = a.ids[r];
  if (y < 0 || y >= a.V) {
    a.out_logprob[r] = NAN;
    a.out_entropy[r] = NAN;
    if (a.status) atomicOr(a.status, RLK_STATUS_BAD_TOKEN_ID);
    return;
  }
  const float4* p = reinterpret_cast<const float4*>(a.partials);
  Part st{-INFINITY, 0.f, 0.f, 0.f};
  for (int s = 0; s < a.n_shards; ++s) {
    const float4 q = p[2 * ((int64_t)s * a.T + r)];
    st = part_merge(st, Part{q.x, q.y, q.z, q.w}, c);
  }
  uint32_t bad = 0u;   // status bits the shards raised (a supplied list's checks)
  for (int s = 0; s < a.n_shards; ++s) bad |= __float_as_uint(p[2 * ((int64_t)s * a.T + r) + 1].z);
  const int ys = (int)(y / a.shard_width);
  const float4 py = ys < a.n_shards ? p[2 * ((int64_t)ys * a.T + r) + 1] : make_float4(NAN, 0.f, 0.f, 0.f);
  const bool y_in = py.y > 0.5f;   // the selected id is in the scored set
  const float zf = __fadd_rn(st.hi, st.lo);
  if (!bad && !(isfinite(zf) && isfinite(st.u) && isfinite(st.m) && (!y_in || isfinite(py.x))))
    bad = RLK_STATUS_NONFINITE;
  if (bad) {
    a.out_logprob[r] = NAN;
    a.out_entropy[r] = NAN;
    if (a.status) atomicOr(a.status, bad);
    return;
  }
  const float lz = logf(zf);
  a.out_logprob[r] = y_in ? __fsub_rn(__fdiv_rn(__fsub_rn(py.x, st.m), a.temperature), lz)
                          : -INFINITY;
  a.out_entropy[r] = __fsub_rn(lz, __fdiv_rn(__fmul_rn(kLn2, st.u), zf));
}

}  // namespace

cudaError_t launch_shard_partials(const ShardArgs& a, cudaStream_t stream) {
  const float c = (float)(1.4426950408889634 / (double)a.temperature);
  const int64_t n_pairs = a.T * (int64_t)a.n_shards;
  const int64_t blocks = (n_pairs + NWP - 1) / NWP;
  const int64_t cap = (int64_t)8 * sm_count();
  shard_partial_kernel<<<(unsigned)(blocks < cap ? blocks : cap), NTP, 0, stream>>>(a, c);
  return cudaGetLastError();
}

cudaError_t launch_shard_support_partials(const ShardArgs& a, cudaStream_t stream) {
  const float c = (float)(1.4426950408889634 / (double)a.temperature);
  const int64_t n_pairs = a.T * (int64_t)a.n_shards;
  const int64_t blocks = (n_pairs + NWP - 1) / NWP;
  const int64_t cap = (int64_t)8 * sm_count();
  shard_support_partial_kernel<<<(unsigned)(blocks < cap ? blocks : cap), NTP, 0, stream>>>(a, c);
  return cudaGetLastError();
}

cudaError_t launch_shard_combine(const ShardCombineArgs& a, cudaStream_t stream) {
  const float c = (float)(1.4426950408889634 / (double)a.temperature);
  shard_combine_kernel<<<(unsigned)((a.T + 255) / 256), 256, 0, stream>>>(a, c);
  return cudaGetLastError();
}

}  // namespace rlk
