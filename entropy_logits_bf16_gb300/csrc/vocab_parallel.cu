// The canonical vocabulary partition: top_p = 1, a supplied retained set, and
// top_p < 1 (window counts per shard after one exchange of the partials).
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

// A state's sums are relative to 2^E with E = ceil(fp32(m c)), an integer
// fixed by its max m alone: every weight is 2^d with d = fma(z, c, -E) (one
// rounding), states merge and rescale by exact powers of two, and the
// window's bins, formed the same way against the row's E, carry the very
// weights the sums hold for the row max's tokens.  (A reference of fp32(m c)
// itself rescaled by ex2 of rounded differences, and left the bins and Z
// apart by up to 2^-19 relative: enough to move a boundary whose gap is
// 1e-6.)
struct Part {
  float m, hi, lo, u;
  float e = -INFINITY;   // part_ref(m): kept by the absorbs and merges (not stored)
};

__device__ __forceinline__ float part_ref(float m, float c) { return ceilf(__fmul_rn(m, c)); }

// 2^n for an integer-valued n <= 0, exactly (0 below 2^-126).
__device__ __forceinline__ float pow2_int(float n) {
  return n >= -126.f ? __int_as_float(((int)n + 127) << 23) : 0.f;
}

// Moves a state's sums from the reference of max m to that of max gm > m.
__device__ __forceinline__ void part_raise(Part& st, float gm, float c) {
  const float En = part_ref(gm, c);
  if (st.m != -INFINITY) {
    const float k = __fsub_rn(En, st.e);   // an integer >= 0
    if (k > 0.f) {
      const float f = pow2_int(-k);
      st.u = __fmul_rn(f, __fmaf_rn(-k, __fadd_rn(st.hi, st.lo), st.u));
      st.hi = __fmul_rn(st.hi, f);
      st.lo = __fmul_rn(st.lo, f);
    }
  }
  st.m = gm;
  st.e = En;
}

__device__ __forceinline__ bool part_empty(const Part& a) {
  return a.m == -INFINITY && a.hi == 0.f && a.lo == 0.f && a.u == 0.f;
}

// Merge b into a (a is the left operand; the caller fixes the order).
__device__ __forceinline__ Part part_merge(const Part& a, const Part& b, float c) {
  if (part_empty(b)) return a;
  if (part_empty(a)) return b;
  const float M = fmaxf(a.m, b.m);
  const float E = part_ref(M, c);
  const float da = __fsub_rn(E, part_ref(a.m, c));   // integers >= 0
  const float db = __fsub_rn(E, part_ref(b.m, c));
  const float fa = pow2_int(-da);
  const float fb = pow2_int(-db);
  const float sa = __fadd_rn(a.hi, a.lo), sb = __fadd_rn(b.hi, b.lo);
  Part r;
  r.m = M;
  r.e = E;
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
  if (gm > st.m) part_raise(st, gm, c);
  const float E = st.e;
  float w[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float d = k < n ? __fmaf_rn(v[k], c, -E) : 0.f;
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
// +-inf), then d = z c - E as fp32x2 fmas.
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
  if (gm > st.m) part_raise(st, gm, c);
  const float E = st.e;
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
__global__ void __launch_bounds__(NTP, 5) shard_partial_kernel(ShardArgs a, float c) {
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
  if (z > st.m) part_raise(st, z, c);
  const float d = __fmaf_rn(z, c, -st.e);
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
  a.out_logprob[r] = y_in ? __fsub_rn(__fmul_rn(kLn2, __fmaf_rn(py.x, c, -part_ref(st.m, c))), lz)
                          : -INFINITY;
  a.out_entropy[r] = __fsub_rn(lz, __fdiv_rn(__fmul_rn(kLn2, st.u), zf));
}


// ------------------------------------------------------------- top_p < 1
// The retained set at top_p < 1 under the same partition, with no supplied
// set: every rank first gathers all shards' partials, so each one knows the
// row's max m and Z.  From them every shard derives the same window
// z >= m - L T with L = ln(V / ((1 - top_p) Z)) + 0.5 (Z relative to the
// max's weight): below it lies less than V e^-L < (1 - top_p) Z of the mass,
// so the nucleus boundary lies inside.  Each shard counts its logits in the
// window per bf16 value -- every token of one value carries the same mass --
// and the integer counts of all shards add up exactly, in any order.  Values
// with |z| < 2^-12 share one bin whose mass each shard sums in a fixed order
// (combined in shard order).  The combine scans the bins largest value first
// with a fixed-order double-float prefix, as the single-device scorer does.

constexpr int HBW = 4096;   // window bins (compressed keys below the row max)
// Ordered 16-bit keys of the bf16 values with |z| < 2^-12 (exponent field
// < 115) form the contiguous interval [MERGE_LO, MERGE_HI], compressed into
// the single key MERGE_LO.
constexpr uint32_t MERGE_LO = 0x4680u;
constexpr uint32_t MERGE_HI = 0xB97Fu;
constexpr uint32_t MERGE_SPAN = MERGE_HI - MERGE_LO;

__device__ __forceinline__ uint32_t ckey(uint32_t k) {
  return k < MERGE_LO ? k : (k <= MERGE_HI ? MERGE_LO : k - MERGE_SPAN);
}
__device__ __forceinline__ uint32_t ckey_expand(uint32_t ck) {   // ck != MERGE_LO
  return ck < MERGE_LO ? ck : ck + MERGE_SPAN;
}
__device__ __forceinline__ uint32_t key_of_f(float v) { return okey16(__float_as_uint(v) >> 16); }

struct ShardCounts {      // one row's window counts of one shard (8224 bytes)
  uint32_t ties;          // tokens whose value is y's and whose id is below y
  uint32_t merged_n;      // tokens in the near-zero bin
  float merged_hi, merged_lo;   // their sum of 2^d, d = fma(z, c, -E), a double-float
  float merged_u;         // their sum of 2^d d
  uint32_t over;          // a bin of this shard passed 65535 tokens
  uint32_t pad[2];
  uint16_t cnt[HBW];      // bins 0..dmax
};
static_assert(sizeof(ShardCounts) == 8224, "the counts' layout is part of the ABI");

struct Window {
  float m, E, zf;         // the row max, E = ceil(fp32(m c)), Z relative to 2^E
  DF Z;
  uint32_t key_m, key_lo, ck_m, dmax;
  bool fits;              // the window has at most HBW bins and the row is finite
};

// Every shard and the combine derive the row's window from the gathered
// partials (merged in shard order), so they all agree on it.  Called by a
// whole warp: lane k loads shard k's partial (32 at a time) and every lane
// merges them all in shard order, so each lane returns the same window.
__device__ Window row_window(const float4* p, int n_all, int64_t T, int64_t r, int64_t V, float c,
                             float temp, float top_p, int lane) {
  Part st{-INFINITY, 0.f, 0.f, 0.f};
  for (int s0 = 0; s0 < n_all; s0 += 32) {
    float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
    if (s0 + lane < n_all) q = p[2 * ((int64_t)(s0 + lane) * T + r)];
    const int n = n_all - s0 < 32 ? n_all - s0 : 32;
    for (int k = 0; k < n; ++k) {
      const Part b{__shfl_sync(0xFFFFFFFFu, q.x, k), __shfl_sync(0xFFFFFFFFu, q.y, k),
                   __shfl_sync(0xFFFFFFFFu, q.z, k), __shfl_sync(0xFFFFFFFFu, q.w, k)};
      st = part_merge(st, b, c);
    }
  }
  Window w{};
  w.m = st.m;
  w.E = part_ref(st.m, c);
  w.Z = DF{st.hi, st.lo};
  w.zf = __fadd_rn(st.hi, st.lo);
  const float one_m_p = __fsub_rn(1.f, top_p);
  // Z relative to the max's own weight 2^(m c - E), in (1/2, 1]
  const float zmax = __fdiv_rn(w.zf, ex2(__fmaf_rn(st.m, c, -w.E)));
  const float L = fmaxf(logf(__fdiv_rn((float)V, __fmul_rn(one_m_p, zmax))), 0.f) + 0.5f;
  const float zlo = __fsub_rn(w.m, __fmul_rn(L, temp));
  w.key_m = key_of_f(w.m);
  const uint32_t kl = key_of_f(zlo);
  w.key_lo = kl > 0u ? kl - 1u : 0u;
  w.ck_m = ckey(w.key_m);
  const uint32_t ck_lo = ckey(w.key_lo);
  w.dmax = w.ck_m - ck_lo;
  w.fits = isfinite(w.m) && isfinite(w.zf) && isfinite(st.u) && w.zf > 0.f &&
           w.key_lo <= w.key_m && w.dmax < (uint32_t)HBW;
  return w;
}

// One CTA per (row, shard): the shard's window counts.
__global__ void __launch_bounds__(NTP, 8) shard_window_kernel(ShardWindowArgs a, float c) {
  __shared__ uint32_t hist[HBW];
  __shared__ Window win;
  __shared__ float red_hi[NWP], red_lo[NWP], red_u[NWP];
  __shared__ uint32_t red_n[NWP], red_t[NWP];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n_pairs = a.T * (int64_t)a.n_shards;
  for (int64_t pr = blockIdx.x; pr < n_pairs; pr += gridDim.x) {
    const int64_t r = pr / a.n_shards;
    const int s = (int)(pr % a.n_shards);
    if (warp == 0) {
      const Window w0 = row_window(reinterpret_cast<const float4*>(a.all_partials), a.n_all, a.T, r,
                                   a.V, c, a.temperature, a.top_p, lane);
      if (lane == 0) win = w0;
    }
    __syncthreads();
    const Window w = win;
    ShardCounts* out = reinterpret_cast<ShardCounts*>(a.counts) + ((int64_t)s * a.T + r);
    const int64_t y = a.ids[r];
    if (!w.fits || y < 0 || y >= a.V) {   // nothing to count (the combine reports the row)
      if (tid == 0) {
        out->ties = 0u;
        out->merged_n = 0u;
        out->merged_hi = out->merged_lo = out->merged_u = 0.f;
        out->over = 0u;
      }
      __syncthreads();
      continue;
    }
    for (uint32_t d = tid; d <= w.dmax; d += NTP) hist[d] = 0u;
    __syncthreads();
    const uint32_t fb = okey16_inverse(w.key_lo);
    const __nv_bfloat162 f2 = bf2(fb | (fb << 16));
    // y's logit, from the shard that holds it (every shard's partial is here)
    const int ys = (int)(y / a.shard_width);
    const float zy = ys < a.n_all ? reinterpret_cast<const float4*>(a.all_partials)[2 * ((int64_t)ys * a.T + r) + 1].x
                                  : NAN;
    const uint32_t key_y = isfinite(zy) ? key_of_f(zy) : 0xFFFFFFFFu;
    const int64_t g0 = a.first_col + (int64_t)s * a.shard_width;   // global columns [g0, g1)
    const int64_t l0 = (int64_t)s * a.shard_width;
    int64_t l1 = l0 + a.shard_width;
    if (g0 + a.shard_width > a.V) l1 = a.V - a.first_col;
    if (l1 < l0) l1 = l0;
    const uint16_t* p = reinterpret_cast<const uint16_t*>(a.logits) + r * a.ld;
    DF mz{0.f, 0.f};
    float mu = 0.f;
    uint32_t mn = 0u, tie = 0u;
    const int64_t ylim = y - a.first_col;   // columns below this one precede y
    auto take = [&](uint32_t bits, int64_t col) {   // one logit in the window
      const uint32_t k = okey16(bits);
      const uint32_t ck = ckey(k);
      if (ck == MERGE_LO) {
        const float d = __fmaf_rn(bf16_lo(bits), c, -w.E);
        const float e = ex2(d);
        mz = df_add_f(mz, e);
        mu = __fmaf_rn(e, d, mu);
        ++mn;
      } else {
        atomicAdd(&hist[w.ck_m - ck], 1u);
      }
      tie += (k == key_y && col < ylim) ? 1u : 0u;
    };
    const bool vec = ((reinterpret_cast<uintptr_t>(p + l0)) & 15u) == 0;
    int64_t j = l0 + (int64_t)tid * 8;
    if (vec) {
      for (; j + 8 <= l1; j += (int64_t)NTP * 8) {
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(p + j));
        // bit k: logit k of the eight reaches the floor (two packed compares a word)
        uint32_t cand = 0u;
        cand |= (__hge2_mask(bf2(q.x), f2) & 0x00010001u) * 1u;
        cand |= (__hge2_mask(bf2(q.y), f2) & 0x00010001u) * 4u;
        cand |= (__hge2_mask(bf2(q.z), f2) & 0x00010001u) * 16u;
        cand |= (__hge2_mask(bf2(q.w), f2) & 0x00010001u) * 64u;
        cand = (cand & 0xFFu) | ((cand >> 15) & 0x1FEu);
        // the window's logits only, in column order (a loop of each lane's own
        // length, not a branch per logit that the warp takes for all eight)
        while (cand) {
          const int k = __ffs(cand) - 1;
          cand &= cand - 1u;
          const int h = k >> 1;
          const uint32_t wsel = h == 0 ? q.x : (h == 1 ? q.y : (h == 2 ? q.z : q.w));
          take((wsel >> (16 * (k & 1))) & 0xFFFFu, j + k);
        }
      }
    }
    for (; j < l1; j += (int64_t)NTP * 8) {
      for (int i = 0; i < 8 && j + i < l1; ++i) {
        const uint32_t bits = __ldg(p + j + i);
        if (bf16_lo(bits) >= bf16_lo(fb)) take(bits, j + i);
      }
    }
    // fixed-order reductions: lanes along a shuffle tree, then the warps in order
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const DF x{shfl_down(mz.hi, o), shfl_down(mz.lo, o)};
      mz = df_add(mz, x);
      mu = __fadd_rn(mu, shfl_down(mu, o));
      mn += __shfl_down_sync(0xFFFFFFFFu, mn, o);
      tie += __shfl_down_sync(0xFFFFFFFFu, tie, o);
    }
    if (lane == 0) {
      red_hi[warp] = mz.hi;
      red_lo[warp] = mz.lo;
      red_u[warp] = mu;
      red_n[warp] = mn;
      red_t[warp] = tie;
    }
    __syncthreads();
    uint32_t over = 0u;
    for (uint32_t d = tid; d <= w.dmax; d += NTP) {
      const uint32_t n = hist[d];
      over |= n > 0xFFFFu ? 1u : 0u;
      out->cnt[d] = (uint16_t)(n > 0xFFFFu ? 0xFFFFu : n);
    }
    over = __syncthreads_or(over);
    if (tid == 0) {
      DF z{0.f, 0.f};
      float u = 0.f;
      uint32_t n = 0u, t = 0u;
      for (int k = 0; k < NWP; ++k) {
        z = df_add(z, DF{red_hi[k], red_lo[k]});
        u = __fadd_rn(u, red_u[k]);
        n += red_n[k];
        t += red_t[k];
      }
      out->ties = t;
      out->merged_n = n;
      out->merged_hi = z.hi;
      out->merged_lo = z.lo;
      out->merged_u = u;
      out->over = over;
    }
    __syncthreads();
  }
}

// One warp per row: the shards' counts added up, then the fixed-order scan.
__global__ void __launch_bounds__(NTP) shard_combine_topp_kernel(ShardCombineArgs a, float c) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t r = (int64_t)blockIdx.x * NWP + warp;
  if (r >= a.T) return;
  const float4* P = reinterpret_cast<const float4*>(a.partials);
  const ShardCounts* C = reinterpret_cast<const ShardCounts*>(a.counts);
  const int64_t y = a.ids[r];
  auto finish_bad = [&](uint32_t bit) {
    if (lane == 0) {
      a.out_logprob[r] = NAN;
      a.out_entropy[r] = NAN;
      if (a.out_k) a.out_k[r] = 0;
      if (a.status) atomicOr(a.status, bit);
    }
  };
  if (y < 0 || y >= a.V) return finish_bad(RLK_STATUS_BAD_TOKEN_ID);
  const Window w = row_window(P, a.n_shards, a.T, r, a.V, c, a.temperature, a.top_p, lane);
  const int ys = (int)(y / a.shard_width);
  const float4 py = ys < a.n_shards ? P[2 * ((int64_t)ys * a.T + r) + 1] : make_float4(NAN, 0.f, 0.f, 0.f);
  const float zy = py.x;
  if (!(isfinite(w.m) && isfinite(w.zf) && isfinite(zy))) return finish_bad(RLK_STATUS_NONFINITE);
  {
    bool fin = true;   // a non-finite logit in any shard leaves NaN in its partial
    for (int s = 0; s < a.n_shards; ++s) fin = fin && !isnan(P[2 * ((int64_t)s * a.T + r)].w);
    if (!fin) return finish_bad(RLK_STATUS_NONFINITE);
  }
  if (!w.fits) return finish_bad(RLK_STATUS_UNRESOLVED);
  uint32_t ties = 0u, over = 0u, mn = 0u;
  DF mz{0.f, 0.f};
  float mu = 0.f;
  for (int s = 0; s < a.n_shards; ++s) {
    const ShardCounts& q = C[(int64_t)s * a.T + r];
    ties += q.ties;
    over |= q.over;
    mn += q.merged_n;
    mz = df_add(mz, DF{q.merged_hi, q.merged_lo});
    mu = __fadd_rn(mu, q.merged_u);
  }
  if (over) return finish_bad(RLK_STATUS_UNRESOLVED);
  const uint32_t key_y = key_of_f(zy);
  const uint32_t d_merged = w.ck_m >= MERGE_LO ? w.ck_m - MERGE_LO : 0xFFFFFFFFu;
  const uint32_t dmax = w.dmax;
  const DF target = df_mul_f(w.Z, a.top_p);
  // Bin d: the tokens of compressed key ck_m - d (d_merged: the near-zero bin).
  auto bin = [&](uint32_t d, uint32_t& nb, DF& mass, float& um, float& wv, float& dv) {
    nb = 0u; mass = DF{0.f, 0.f}; um = 0.f; wv = 0.f; dv = 0.f;
    if (d > dmax) return;
    if (d == d_merged) {
      nb = mn; mass = mz; um = mu;
      return;
    }
    for (int s = 0; s < a.n_shards; ++s) nb += C[(int64_t)s * a.T + r].cnt[d];
    if (nb == 0u) return;
    dv = __fmaf_rn(bf16_val(okey16_inverse(ckey_expand(w.ck_m - d))), c, -w.E);
    wv = ex2(dv);
    const float ms = __fmul_rn((float)nb, wv);
    mass = DF{ms, 0.f};
    um = __fmul_rn(ms, dv);
  };
  const uint32_t bpl = (dmax + 32u) / 32u;
  const uint32_t d0 = (uint32_t)lane * bpl;
  DF tot{0.f, 0.f};
  uint32_t tcnt = 0u;
  float tum = 0.f;
  for (uint32_t j = 0; j < bpl; ++j) {
    uint32_t nb; DF ms; float um, wv, dv;
    bin(d0 + j, nb, ms, um, wv, dv);
    tot = df_add(tot, ms);
    tcnt += nb;
    tum = __fadd_rn(tum, um);
  }
  DF inc = tot;
  uint32_t icnt = tcnt;
  float ium = tum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF lft{shfl_up(inc.hi, o), shfl_up(inc.lo, o)};
    const uint32_t lc = __shfl_up_sync(0xFFFFFFFFu, icnt, o);
    const float lu = shfl_up(ium, o);
    if (lane >= o) {
      inc = df_add(lft, inc);
      icnt += lc;
      ium = __fadd_rn(lu, ium);
    }
  }
  DF P0{shfl_up(inc.hi, 1), shfl_up(inc.lo, 1)};
  uint32_t pc = __shfl_up_sync(0xFFFFFFFFu, icnt, 1);
  float pu = shfl_up(ium, 1);
  if (lane == 0) { P0 = DF{0.f, 0.f}; pc = 0u; pu = 0.f; }
  int my_d = -1;
  DF pb{0.f, 0.f};
  uint32_t cb = 0u, nt = 0u;
  float ub = 0.f, wt = 0.f, dt = 0.f;
  for (uint32_t j = 0; j < bpl; ++j) {
    uint32_t nb; DF ms; float um, wv, dv;
    bin(d0 + j, nb, ms, um, wv, dv);
    const DF Pn = df_add(P0, ms);
    if (nb > 0u && df_ge(Pn, target)) {
      my_d = (int)(d0 + j);
      pb = P0; cb = pc; ub = pu; wt = wv; dt = dv; nt = nb;
      break;
    }
    P0 = Pn;
    pc += nb;
    pu = __fadd_rn(pu, um);
  }
  const uint32_t bal = __ballot_sync(0xFFFFFFFFu, my_d >= 0);
  if (bal == 0u) return finish_bad(RLK_STATUS_UNRESOLVED);   // (the window holds the crossing)
  const int win_lane = __ffs(bal) - 1;
  const int cross = __shfl_sync(0xFFFFFFFFu, my_d, win_lane);
  // A crossing inside the near-zero bin would need its values' order.
  if ((uint32_t)cross == d_merged) return finish_bad(RLK_STATUS_UNRESOLVED);
  if (lane == win_lane) {
    const float need = df_sub_to_f(target, pb);
    const float cf = ceilf(__fdiv_rn(need, wt));
    const uint32_t cneed = cf < 1.f ? 1u : (cf > (float)nt ? nt : (uint32_t)cf);
    const float wn = __fmul_rn((float)cneed, wt);
    const DF zs = df_add_f(pb, wn);
    const float us = __fmaf_rn(wn, dt, ub);
    const uint32_t ck_y = ckey(key_y);
    const uint32_t d_y = w.ck_m - ck_y;
    const bool y_in = (d_y < (uint32_t)my_d) || (d_y == (uint32_t)my_d && ties < cneed);
    const float zsf = __fadd_rn(zs.hi, zs.lo);
    const float lz = logf(zsf);
    a.out_logprob[r] = y_in ? __fsub_rn(__fmul_rn(kLn2, __fmaf_rn(zy, c, -w.E)), lz) : -INFINITY;
    a.out_entropy[r] = __fsub_rn(lz, __fdiv_rn(__fmul_rn(kLn2, us), zsf));
    if (a.out_k) a.out_k[r] = (int32_t)(cb + cneed);
  }
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

cudaError_t launch_shard_window(const ShardWindowArgs& a, cudaStream_t stream) {
  const float c = (float)(1.4426950408889634 / (double)a.temperature);
  const int64_t n_pairs = a.T * (int64_t)a.n_shards;
  const int64_t cap = (int64_t)16 * sm_count();
  shard_window_kernel<<<(unsigned)(n_pairs < cap ? n_pairs : cap), NTP, 0, stream>>>(a, c);
  return cudaGetLastError();
}

cudaError_t launch_shard_combine_topp(const ShardCombineArgs& a, cudaStream_t stream) {
  const float c = (float)(1.4426950408889634 / (double)a.temperature);
  shard_combine_topp_kernel<<<(unsigned)((a.T + NWP - 1) / NWP), NTP, 0, stream>>>(a, c);
  return cudaGetLastError();
}

cudaError_t launch_shard_combine(const ShardCombineArgs& a, cudaStream_t stream) {
  const float c = (float)(1.4426950408889634 / (double)a.temperature);
  shard_combine_kernel<<<(unsigned)((a.T + 255) / 256), 256, 0, stream>>>(a, c);
  return cudaGetLastError();
}

}  // namespace rlk
