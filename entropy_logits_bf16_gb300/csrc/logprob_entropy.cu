// rlk_logprob_entropy kernels: per-token top-p log-probability and entropy.
//
// What is computed follows RL-Kernel "Qwen3-8B VIME train-rollout
// consistency", section "ROCm MI300X and gfx942" (sparse logp /
// monitoring-entropy fusion over the complete retained top-p support; the
// full-vocabulary scorer at top_p = 1; temperature > 0, top_p in (0,1]) and the
// RL-Kernel "ROCm sparse performance" notes (temperature, softmax, sort and
// top-p thresholding with the sampler's semantics; a fixed reduction order so
// that recomputed log-probabilities are bitwise reproducible).
//
// Design: one CTA of 512 threads per row; rows are strided over a persistent
// grid of 2 CTAs per SM.
//  Pass 1 streams the row once from HBM with 16-byte loads.  Thread t owns the
//   8-element groups t, t+512, t+1024, ... and keeps an online state: the max
//   m, the sum of 2^d as a double-float and the sum of 2^d * d, where
//   d = (z - m) log2(e) / T.  The 512 states merge along a fixed tree.  At
//   top_p = 1 this is the answer: logprob = (z_y - m)/T - ln Z and
//   H = ln Z - ln2 * (sum 2^d d) / Z.
//  top_p < 1, bf16: the retained set lies in a window z >= m - L T.  All
//   tokens of one bf16 value carry the same mass, so the window is summarised
//   exactly by integer counts per distinct value (a histogram over the
//   order-preserving 16-bit key; the values with |z| < 2^-12 share one bin
//   whose mass is summed per token in fixed point).  Counts and fixed-point
//   sums do not depend on the order of the atomics that build them.
//   - Fast path: during pass 1 the CTA shares a running max; a group holding a
//     token within the speculative depth L_spec T (L_spec = ln(1/(1-top_p)) + 7)
//     of it is pushed on a per-warp shared-memory queue (one packed bf16x2
//     compare per word, a ballot per group) and expanded with all lanes busy
//     into an absolute-key histogram of 16-bit counts.  The running max never
//     exceeds the final one, so every token of the final window is counted.
//   - A fixed-order double-float scan over the window's bins (largest value
//     first) finds the bin where the prefix mass reaches top_p * Z and how
//     many of its tied tokens are needed (ties are kept lower id first).  If
//     the window's own mass falls short, the worst-case window
//     L = ln(V / ((1 - top_p) Z)) + 0.5 -- below which lies less than
//     V e^-L < (1 - top_p) Z of the mass -- is counted by a second pass over
//     the row (an L2 hit) and scanned the same way.  The same pass serves rows
//     the fast path cannot take (a window touching the near-zero bin, or more
//     than 65535 counted tokens); on rows where a quarter of the groups or
//     more hold window tokens it counts each thread's groups in place.
//     Every path feeds identical bins to the same scan, so the result does
//     not depend on which path ran.
//   - Rows whose window spans more than the histogram, rows whose threshold
//     falls in the near-zero bin, and fp32 rows bisect on the value key with
//     fixed-order passes over the row (exact, slower).  This choice depends
//     only on the row's values.
//  No sum depends on thread timing, so a row's output bits never depend on
//  the batch around it.

#include <cuda_bf16.h>
#include <math.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "rlk.h"

namespace rlk {
namespace {

constexpr int NT = 256;
constexpr int NWARP = NT / 32;
constexpr int HB = 4096;         // largest window (bins) the histogram path takes
constexpr int QCAP = 64;         // per-warp queue of candidate groups (flushed at >= 32)
constexpr int SK_ROUNDS = 76;    // rows of up to SK_ROUNDS * NT groups keep a group-max sketch
constexpr int WL = 256;          // per-warp list of candidate groups (sketch pass)

// Ordered 16-bit keys of the bf16 values with |z| < 2^-12 (exponent field
// < 115) form the contiguous interval [MERGE_LO, MERGE_HI]; it is compressed
// into the single key MERGE_LO.
constexpr uint32_t MERGE_LO = 0x4680u;
constexpr uint32_t MERGE_HI = 0xB97Fu;
constexpr uint32_t MERGE_SPAN = MERGE_HI - MERGE_LO;

__device__ __forceinline__ uint32_t compress_key(uint32_t k) {
  return k < MERGE_LO ? k : (k <= MERGE_HI ? MERGE_LO : k - MERGE_SPAN);
}
__device__ __forceinline__ uint32_t expand_key(uint32_t ck) {  // ck != MERGE_LO
  return ck < MERGE_LO ? ck : ck + MERGE_SPAN;
}

// ---------------------------------------------------------------- row access
struct RowBf16 {
  static constexpr int E = 8;          // elements per 16-byte group
  static constexpr int KEYBITS = 16;
  const uint16_t* p;
  int64_t V;
  bool aligned;
  __device__ __forceinline__ void vec(int64_t g, float (&v)[E]) const {
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(p) + g);
    v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x); v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
    v[4] = bf16_lo(q.z); v[5] = bf16_hi(q.z); v[6] = bf16_lo(q.w); v[7] = bf16_hi(q.w);
  }
  __device__ __forceinline__ int scal(int64_t g, float (&v)[E]) const {
    const int64_t base = g * E;
    const int n = (int)(V - base < E ? V - base : E);
#pragma unroll
    for (int k = 0; k < E; ++k) v[k] = k < n ? bf16_val(__ldg(p + base + k)) : -INFINITY;
    return n;
  }
  __device__ __forceinline__ float elem(int64_t i) const { return bf16_val(__ldg(p + i)); }
  // The group as four packed words; missing tail elements read as -inf.
  __device__ __forceinline__ uint4 packed(int64_t g, int64_t nfull) const {
    if (g < nfull && aligned) return __ldg(reinterpret_cast<const uint4*>(p) + g);
    float v[E];
    scal(g, v);
    uint32_t b[E];
#pragma unroll
    for (int k = 0; k < E; ++k) b[k] = __float_as_uint(v[k]) >> 16;
    return make_uint4(b[0] | (b[1] << 16), b[2] | (b[3] << 16), b[4] | (b[5] << 16),
                      b[6] | (b[7] << 16));
  }
  __device__ static __forceinline__ uint32_t key(float v) {
    return okey16(__float_as_uint(v) >> 16);
  }
  __device__ static __forceinline__ float value_of_key(uint32_t k) {
    return bf16_val(okey16_inverse(k));
  }
};

struct RowF32 {
  static constexpr int E = 4;
  static constexpr int KEYBITS = 32;
  const float* p;
  int64_t V;
  bool aligned;
  __device__ __forceinline__ void vec(int64_t g, float (&v)[E]) const {
    const float4 q = __ldg(reinterpret_cast<const float4*>(p) + g);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
  __device__ __forceinline__ int scal(int64_t g, float (&v)[E]) const {
    const int64_t base = g * E;
    const int n = (int)(V - base < E ? V - base : E);
#pragma unroll
    for (int k = 0; k < E; ++k) v[k] = k < n ? __ldg(p + base + k) : -INFINITY;
    return n;
  }
  __device__ __forceinline__ float elem(int64_t i) const { return __ldg(p + i); }
  __device__ static __forceinline__ uint32_t key(float v) { return okey32(__float_as_uint(v)); }
  __device__ static __forceinline__ float value_of_key(uint32_t k) {
    return __uint_as_float(okey32_inverse(k));
  }
};

__device__ __forceinline__ void unpack8(const uint4 q, float (&v)[8]) {
  v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x); v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
  v[4] = bf16_lo(q.z); v[5] = bf16_hi(q.z); v[6] = bf16_lo(q.w); v[7] = bf16_hi(q.w);
}

// Calls f(values, n_valid, group) for this thread's groups in a fixed order
// (g = tid, tid + NT, ...), whatever the row's alignment.  Aligned rows issue
// BATCH 16-byte loads before using them (memory-level parallelism).
template <int BATCH = 4, class Row, class F>
__device__ __forceinline__ void for_groups(const Row& row, int tid, F&& f) {
  constexpr int E = Row::E;
  const int64_t nfull = row.V / E;
  int64_t g = tid;
  if (row.aligned) {
    for (; g + (BATCH - 1) * NT < nfull; g += BATCH * NT) {
      float a[BATCH][E];
#pragma unroll
      for (int b = 0; b < BATCH; ++b) row.vec(g + b * NT, a[b]);
#pragma unroll
      for (int b = 0; b < BATCH; ++b) f(a[b], E, g + b * NT);
    }
    for (; g < nfull; g += NT) {
      float a[E];
      row.vec(g, a);
      f(a, E, g);
    }
  } else {
    for (; g < nfull; g += NT) {
      float a[E];
      row.scal(g, a);
      f(a, E, g);
    }
  }
  if (g == nfull && row.V % E != 0) {
    float a[E];
    const int n = row.scal(g, a);
    f(a, n, g);
  }
}

// ------------------------------------------------------- online LSE state
struct Online {
  float m;        // running max of z
  float hi, lo;   // sum of 2^d, d = (z - m) * c, as a double-float
  float u;        // sum of 2^d * d
};

__device__ __forceinline__ bool online_empty(const Online& a) {
  return a.m == -INFINITY && a.hi == 0.f && a.lo == 0.f && a.u == 0.f;
}

// Merge two states (a is the left operand; the tree fixes which is which).
__device__ __forceinline__ Online online_merge(const Online& a, const Online& b, float c) {
  if (online_empty(b)) return a;
  if (online_empty(a)) return b;
  const float M = fmaxf(a.m, b.m);
  const float da = __fmul_rn(__fsub_rn(M, a.m), c);
  const float db = __fmul_rn(__fsub_rn(M, b.m), c);
  const float fa = (a.m == M) ? 1.f : ex2(-da);
  const float fb = (b.m == M) ? 1.f : ex2(-db);
  const float sa = __fadd_rn(a.hi, a.lo), sb = __fadd_rn(b.hi, b.lo);
  Online r;
  r.m = M;
  r.u = __fadd_rn(__fmul_rn(fa, __fmaf_rn(-da, sa, a.u)), __fmul_rn(fb, __fmaf_rn(-db, sb, b.u)));
  float s, e;
  two_sum(__fmul_rn(a.hi, fa), __fmul_rn(b.hi, fb), s, e);
  e = __fadd_rn(e, __fadd_rn(__fmul_rn(a.lo, fa), __fmul_rn(b.lo, fb)));
  r.hi = __fadd_rn(s, e);
  r.lo = __fsub_rn(e, __fsub_rn(r.hi, s));
  return r;
}

// Fold one group of N values (the first n valid) into the state; returns the
// group's max.
template <int N>
__device__ __forceinline__ float absorb(Online& st, const float (&v)[N], int n, float c) {
  float gm = -INFINITY;
#pragma unroll
  for (int k = 0; k < N; ++k)
    if (k < n) gm = fmaxf(gm, v[k]);
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
  float w[N], d[N];
#pragma unroll
  for (int k = 0; k < N; ++k) {
    if (k < n) {
      d[k] = __fmul_rn(__fsub_rn(v[k], st.m), c);
      w[k] = ex2(d[k]);
    } else {
      d[k] = 0.f;
      w[k] = 0.f;
    }
  }
  float gsum;
  if constexpr (N == 8) {
    gsum = __fadd_rn(__fadd_rn(__fadd_rn(w[0], w[1]), __fadd_rn(w[2], w[3])),
                     __fadd_rn(__fadd_rn(w[4], w[5]), __fadd_rn(w[6], w[7])));
  } else {
    gsum = __fadd_rn(__fadd_rn(w[0], w[1]), __fadd_rn(w[2], w[3]));
  }
  float s, e;
  two_sum(st.hi, gsum, s, e);
  st.hi = s;
  st.lo = __fadd_rn(st.lo, e);
#pragma unroll
  for (int k = 0; k < N; ++k) st.u = __fmaf_rn(w[k], d[k], st.u);
  return gm;
}

// Fold one full group of 8 bf16 values (packed words) into the state: the
// group max by packed bf16x2 compares, then the same arithmetic as absorb().
// With WITH_U the entropy numerator is accumulated too; *gmin gets the group
// min (to detect -inf inputs when WITH_U is off).  Returns the group max.
__device__ __forceinline__ __nv_bfloat162 as_bf162w(uint32_t w) {
  return *reinterpret_cast<const __nv_bfloat162*>(&w);
}
template <bool WITH_U>
__device__ __forceinline__ float absorb_packed(Online& st, const uint4 q, float c, float& gmin) {
  const __nv_bfloat162 mx = __hmax2(__hmax2(as_bf162w(q.x), as_bf162w(q.y)),
                                    __hmax2(as_bf162w(q.z), as_bf162w(q.w)));
  const float gm = fmaxf(__low2float(mx), __high2float(mx));
  if (!WITH_U) {
    const __nv_bfloat162 mn = __hmin2(__hmin2(as_bf162w(q.x), as_bf162w(q.y)),
                                      __hmin2(as_bf162w(q.z), as_bf162w(q.w)));
    gmin = fminf(__low2float(mn), __high2float(mn));
  }
  if (gm > st.m) {
    if (st.m != -INFINITY) {
      const float delta = __fmul_rn(__fsub_rn(gm, st.m), c);
      const float f = ex2(-delta);
      if (WITH_U) st.u = __fmul_rn(f, __fmaf_rn(-delta, __fadd_rn(st.hi, st.lo), st.u));
      st.hi = __fmul_rn(st.hi, f);
      st.lo = __fmul_rn(st.lo, f);
    }
    st.m = gm;
  }
  float v[8], w[8], d[8];
  unpack8(q, v);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    d[k] = __fmul_rn(__fsub_rn(v[k], st.m), c);
    w[k] = ex2(d[k]);
  }
  const float gsum = __fadd_rn(__fadd_rn(__fadd_rn(w[0], w[1]), __fadd_rn(w[2], w[3])),
                               __fadd_rn(__fadd_rn(w[4], w[5]), __fadd_rn(w[6], w[7])));
  float s, e;
  two_sum(st.hi, gsum, s, e);
  st.hi = s;
  st.lo = __fadd_rn(st.lo, e);
  if (WITH_U) {
#pragma unroll
    for (int k = 0; k < 8; ++k) st.u = __fmaf_rn(w[k], d[k], st.u);
  }
  return gm;
}

// ------------------------------------------------------------ shared memory
struct __align__(16) Smem {
  // Histogram of 32-bit counts indexed by distance from the max (in keys).
  struct {
    uint32_t rel[HB];
  } hist;
  uint16_t gmax[SK_ROUNDS][NT];            // bf16 max of each group (the sketch)
  union {
    struct {
      uint4 qdata[NWARP][QCAP];
      uint32_t qidx[NWARP][QCAP];
    } q;
    uint32_t wlist[NWARP][WL];
  } lists;
  float red[NWARP][4];
  float bc[8];
  uint32_t ured[NWARP][4];
  uint32_t ubc[4];
  DF scan_wtot[NWARP];
  uint32_t scan_wcnt[NWARP];
  float scan_wum[NWARP];
  DF scan_woff[NWARP];
  uint32_t scan_woffc[NWARP];
  float scan_woffu[NWARP];
  unsigned long long merged_w, merged_u;  // fixed-point sums of the near-zero bin
  uint32_t merged_n;
  uint32_t gmin_key;                      // ordered key of the row's smallest value
  uint32_t marked[NWARP];                 // recompute pass: which of the next NT rows are marked,
  uint32_t wide[NWARP];                   // and which of them take the guaranteed window at once
  int dstar;
  // result of the scan, written by the thread owning the threshold bin
  float r_pb_hi, r_pb_lo, r_um_before, r_w, r_x;
  uint32_t r_cnt_before, r_n;
};

__device__ Online block_reduce_online(Online st, float c, Smem& sm, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Online x{shfl_down(st.m, o), shfl_down(st.hi, o), shfl_down(st.lo, o), shfl_down(st.u, o)};
    st = online_merge(st, x, c);
  }
  if (lane == 0) {
    sm.red[warp][0] = st.m; sm.red[warp][1] = st.hi;
    sm.red[warp][2] = st.lo; sm.red[warp][3] = st.u;
  }
  __syncthreads();
  if (warp == 0) {
    Online x = (lane < NWARP) ? Online{sm.red[lane][0], sm.red[lane][1], sm.red[lane][2], sm.red[lane][3]}
                              : Online{-INFINITY, 0.f, 0.f, 0.f};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Online y{shfl_down(x.m, o), shfl_down(x.hi, o), shfl_down(x.lo, o), shfl_down(x.u, o)};
      x = online_merge(x, y, c);
    }
    if (lane == 0) {
      sm.bc[0] = x.m; sm.bc[1] = x.hi; sm.bc[2] = x.lo; sm.bc[3] = x.u;
    }
  }
  __syncthreads();
  Online r{sm.bc[0], sm.bc[1], sm.bc[2], sm.bc[3]};
  __syncthreads();
  return r;
}

// Fixed-order block sum of a double-float and a float.
__device__ void block_sum_df(DF& x, float& f, Smem& sm, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    DF y{shfl_down(x.hi, o), shfl_down(x.lo, o)};
    const float g = shfl_down(f, o);
    x = df_add(x, y);
    f = __fadd_rn(f, g);
  }
  if (lane == 0) {
    sm.red[warp][0] = x.hi; sm.red[warp][1] = x.lo; sm.red[warp][2] = f;
  }
  __syncthreads();
  if (tid == 0) {
    DF a{sm.red[0][0], sm.red[0][1]};
    float b = sm.red[0][2];
    for (int w = 1; w < NWARP; ++w) {
      a = df_add(a, DF{sm.red[w][0], sm.red[w][1]});
      b = __fadd_rn(b, sm.red[w][2]);
    }
    sm.bc[0] = a.hi; sm.bc[1] = a.lo; sm.bc[2] = b;
  }
  __syncthreads();
  x = DF{sm.bc[0], sm.bc[1]};
  f = sm.bc[2];
  __syncthreads();
}

// Block sums of up to four unsigned counters (order-free).
__device__ void block_sum_u32(uint32_t (&v)[4], Smem& sm, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __reduce_add_sync(0xFFFFFFFFu, v[i]);
  if (lane == 0)
    for (int i = 0; i < 4; ++i) sm.ured[warp][i] = v[i];
  __syncthreads();
  if (tid < 4) {
    uint32_t a = 0;
    for (int w = 0; w < NWARP; ++w) a += sm.ured[w][tid];
    sm.ubc[tid] = a;
  }
  __syncthreads();
  for (int i = 0; i < 4; ++i) v[i] = sm.ubc[i];
  __syncthreads();
}

// ------------------------------------------------------ candidate queues
// Largest of the 8 bf16 values of a packed group (packed bf16x2 max).
__device__ __forceinline__ float group_max(const uint4 q) {
  const __nv_bfloat162 mx = __hmax2(__hmax2(as_bf162w(q.x), as_bf162w(q.y)),
                                    __hmax2(as_bf162w(q.z), as_bf162w(q.w)));
  return fmaxf(__low2float(mx), __high2float(mx));
}

// Per-warp queue of groups that hold a candidate.  offer() is called by every
// lane of the warp in lockstep; process(q, g) expands one queued group.
struct WarpQueue {
  uint4* data;
  uint32_t* idx;
  uint32_t n;          // warp-uniform fill
  uint32_t lt_mask;
  int lane;
  template <class P>
  __device__ __forceinline__ void flush(P&& process) {
    __syncwarp();
    for (uint32_t i = (uint32_t)lane; i < n; i += 32) process(data[i], idx[i]);
    __syncwarp();
    n = 0;
  }
  template <class P>
  __device__ __forceinline__ void offer(const uint4& q, int64_t g, bool cand, P&& process) {
    const uint32_t b = __ballot_sync(0xFFFFFFFFu, cand);
    if (b) {
      if (cand) {
        const uint32_t pos = n + __popc(b & lt_mask);
        data[pos] = q;
        idx[pos] = (uint32_t)g;
      }
      n += __popc(b);
      if (n >= 32u) flush(process);
    }
  }
};

// Expands a queued group: calls f(bits16, element index) for every element
// with value >= thr.
template <class F>
__device__ __forceinline__ void for_candidates(const uint4 q, uint32_t g, int64_t V, float thr,
                                               F&& f) {
  const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
  uint32_t mask = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t bits = (w4[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
    if (bf16_val(bits) >= thr && (int64_t)g * 8 + k < V) mask |= 1u << k;
  }
  while (mask) {
    const int k = __ffs(mask) - 1;
    mask &= mask - 1u;
    const int h = k >> 1;
    const uint32_t wsel = h == 0 ? w4[0] : h == 1 ? w4[1] : h == 2 ? w4[2] : w4[3];
    f((wsel >> (16 * (k & 1))) & 0xFFFFu, (int64_t)g * 8 + k);
  }
}

// ---------------------------------------------------------- packed pass 1
// Pass 1 over a bf16 row with the groups kept packed (four registers each) so
// that BATCH 16-byte loads per thread are in flight before they are used.
// Same group order as for_groups (g = tid, tid + NT, ...).  *gmin gets the
// thread's smallest value when WITH_U is off (-inf detection).
template <int BATCH, bool WITH_U>
__device__ __forceinline__ void pass1_packed(const RowBf16& row, int tid, float c, Online& st,
                                             float& gmin, uint16_t (*sketch)[NT]) {
  const int V = (int)row.V;   // V <= 2^24
  const int nfull = V / 8;
  int g = tid;
  auto record = [&](int gg, float gm) {
    if (sketch) sketch[gg / NT][tid] = (uint16_t)(__float_as_uint(gm) >> 16);
  };
  if (row.aligned) {
    const uint4* base = reinterpret_cast<const uint4*>(row.p);
    for (; g + (BATCH - 1) * NT < nfull; g += BATCH * NT) {
      uint4 q[BATCH];
#pragma unroll
      for (int b = 0; b < BATCH; ++b) q[b] = __ldg(base + g + b * NT);
#pragma unroll
      for (int b = 0; b < BATCH; ++b) {
        float gn = INFINITY;
        record(g + b * NT, absorb_packed<WITH_U>(st, q[b], c, gn));
        gmin = fminf(gmin, gn);
      }
    }
  }
  for (; g < nfull; g += NT) {
    float gn = INFINITY;
    record(g, absorb_packed<WITH_U>(st, row.packed(g, nfull), c, gn));
    gmin = fminf(gmin, gn);
  }
  if (g == nfull && V % 8 != 0) {
    float v[8];
    const int n = row.scal(g, v);
    for (int k = 0; k < n; ++k) gmin = fminf(gmin, v[k]);
    record(g, absorb<8>(st, v, n, c));
  }
}

// ------------------------------------------------------------ second pass
// Counts one window token (bf16 bits): into the distance histogram (bin =
// ck_m - ck), or, in the near-zero bin, into its fixed-point sums.  Every
// window pass counts through here, so they all build the same integers.
__device__ __forceinline__ void count_window_token(uint32_t ck, uint32_t bits, float m, float c,
                                                   float inv_t, uint32_t ck_m, Smem& sm) {
  if (ck == MERGE_LO) {
    const float dd = __fsub_rn(bf16_val(bits), m);
    const float w = ex2(__fmul_rn(dd, c));
    atomicAdd(&sm.merged_w, __float2ull_rn(__fmul_rn(w, 1099511627776.0f)));      // 2^40
    atomicAdd(&sm.merged_u, __float2ull_rn(__fmul_rn(-__fmul_rn(w, __fmul_rn(dd, inv_t)),
                                                     4294967296.0f)));                  // 2^32
    atomicAdd(&sm.merged_n, 1u);
  } else {
    atomicAdd(&sm.hist.rel[ck_m - ck], 1u);
  }
}

// The window pass for rows where a quarter of the groups or more hold window
// tokens (flat rows, wide nuclei): each thread counts the tokens of its own
// groups in place, unrolled, without the queue.  Same counts and sums as
// window_pass (absent tail logits read as -inf, below any window floor).
__device__ __forceinline__ uint32_t window_pass_dense(const RowBf16& row, int tid, float zlo, float m,
                                                   float c, float inv_t, uint32_t ck_m,
                                                   uint32_t key_y, int64_t y, Smem& sm) {
  const int64_t nfull = row.V / 8;
  const int64_t ngroups = (row.V + 7) / 8;
  uint32_t tie = 0;
  auto group = [&](const uint4 q, int64_t g) {
    if (group_max(q) < zlo) return;
    const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
    // ids of this group ahead of y: 0..8
    const int64_t ahead64 = y - g * 8;
    const int ahead = ahead64 < 0 ? 0 : (ahead64 > 8 ? 8 : (int)ahead64);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t bits = (w4[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
      if (bf16_val(bits) >= zlo) {
        const uint32_t key = okey16(bits);
        count_window_token(compress_key(key), bits, m, c, inv_t, ck_m, sm);
        tie += (key == key_y && k < ahead) ? 1u : 0u;
      }
    }
  };
  constexpr int B = 4;
  int64_t g = tid;
  if (row.aligned) {   // whole batches of full groups: plain vector loads
    const uint4* base = reinterpret_cast<const uint4*>(row.p);
    for (; g + (B - 1) * NT < nfull; g += B * NT) {
      uint4 q[B];
#pragma unroll
      for (int b = 0; b < B; ++b) q[b] = __ldg(base + g + b * NT);
#pragma unroll
      for (int b = 0; b < B; ++b) group(q[b], g + b * NT);
    }
  }
  for (; g < ngroups; g += NT) group(row.packed(g, nfull), g);
  return tie;
}

// Counts the tokens with z >= zlo into the distance histogram (bin = ck_m - ck),
// the near-zero bin into fixed-point sums, and the ties of y ahead of it
// (dense: by window_pass_dense).
__device__ __noinline__ uint32_t window_pass(const RowBf16& row, int tid, float zlo, float m, float c,
                                float inv_t, uint32_t ck_m, uint32_t key_y, int64_t y,
                                Smem& sm, bool dense) {
  if (dense) return window_pass_dense(row, tid, zlo, m, c, inv_t, ck_m, key_y, y, sm);
  const int lane = tid & 31, warp = tid >> 5;
  const int64_t nfull = row.V / 8;
  const int64_t ngroups = (row.V + 7) / 8;
  const int64_t rounds = (ngroups + NT - 1) / NT;
  WarpQueue wq{sm.lists.q.qdata[warp], sm.lists.q.qidx[warp], 0u, (1u << lane) - 1u, lane};
  uint32_t tie = 0;
  auto process = [&](const uint4 q, uint32_t g) {
    for_candidates(q, g, row.V, zlo, [&](uint32_t bits, int64_t i) {
      const uint32_t key = okey16(bits);
      count_window_token(compress_key(key), bits, m, c, inv_t, ck_m, sm);
      if (key == key_y && i < y) ++tie;
    });
  };
  constexpr int B = 4;
  int64_t r0 = 0;
  if (row.aligned) {   // whole batches of full groups: plain vector loads
    const uint4* base = reinterpret_cast<const uint4*>(row.p);
    for (; (r0 + B - 1) * NT + (NT - 1) < nfull; r0 += B) {
      uint4 q[B];
#pragma unroll
      for (int b = 0; b < B; ++b) q[b] = __ldg(base + tid + (r0 + b) * NT);
#pragma unroll
      for (int b = 0; b < B; ++b)
        wq.offer(q[b], tid + (r0 + b) * NT, group_max(q[b]) >= zlo, process);
    }
  }
  for (; r0 < rounds; ++r0) {
    const int64_t g = tid + r0 * NT;
    const bool val = g < ngroups;
    const uint4 q = val ? row.packed(g, nfull) : make_uint4(0u, 0u, 0u, 0u);
    wq.offer(q, g, val && group_max(q) >= zlo, process);
  }
  wq.flush(process);
  return tie;
}

// ------------------------------------------------------------ sketch pass
// The second pass when pass 1 kept the group-max sketch: a group can hold a
// token with z >= zlo only if its max is >= zlo, so each warp ballots over its
// sketch entries into a list of candidate group indices and then reloads just
// those groups (four per lane in flight) and counts their window tokens
// exactly as window_pass does.
__device__ __forceinline__ uint32_t sketch_pass(const RowBf16& row, int tid, float zlo, float m, float c,
                                float inv_t, uint32_t ck_m, uint32_t key_y, int64_t y,
                                Smem& sm) {
  const int lane = tid & 31, warp = tid >> 5;
  const int V = (int)row.V;
  const int nfull = V / 8;
  const int ngroups = (V + 7) / 8;
  const int rounds = (ngroups + NT - 1) / NT;
  const uint32_t lt_mask = (1u << lane) - 1u;
  uint32_t* wl = sm.lists.wlist[warp];
  uint32_t tie = 0;
  auto expand = [&](const uint4 q, uint32_t g) {
    for_candidates(q, g, row.V, zlo, [&](uint32_t bits, int64_t i) {
      const uint32_t key = okey16(bits);
      count_window_token(compress_key(key), bits, m, c, inv_t, ck_m, sm);
      if (key == key_y && i < y) ++tie;
    });
  };
  auto drain = [&](uint32_t n) {
    __syncwarp();
    for (uint32_t i0 = 0; i0 < n; i0 += 128) {
      uint4 q[4];
      uint32_t gi[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t i = i0 + b * 32 + lane;
        gi[b] = i < n ? wl[i] : 0xFFFFFFFFu;
        if (gi[b] != 0xFFFFFFFFu) q[b] = row.packed(gi[b], nfull);
      }
#pragma unroll
      for (int b = 0; b < 4; ++b)
        if (gi[b] != 0xFFFFFFFFu) expand(q[b], gi[b]);
    }
    __syncwarp();
  };
  uint32_t wn = 0;    // warp-uniform list fill
  for (int r = 0; r < rounds; ++r) {
    const int g = tid + r * NT;
    const bool cand = g < ngroups && bf16_val(sm.gmax[r][tid]) >= zlo;
    const uint32_t b = __ballot_sync(0xFFFFFFFFu, cand);
    if (cand) wl[wn + __popc(b & lt_mask)] = (uint32_t)g;
    wn += __popc(b);
    if (wn > (uint32_t)(WL - 32)) {
      drain(wn);
      wn = 0;
    }
  }
  drain(wn);
  return tie;
}

// ------------------------------------------------------------ bin scan
// Bins 0..dmax (bin d = compressed key ck_m - d, largest value first): a
// fixed-order double-float scan for the first bin whose inclusive prefix
// mass reaches the target.  Bins are split into equal contiguous chunks per
// thread (one bin per thread while the window has <= 512 bins).  The winner's
// data lands in sm.r_*; returns false when the window's mass is short.
__device__ __forceinline__ bool scan_bins(int tid, uint32_t dmax, uint32_t d_merged, uint32_t ck_m, float m,
                          float c, float inv_t, DF target, Smem& sm, int& dstar_out) {
  DF mmerged{0.f, 0.f};
  float umerged = 0.f;
  uint32_t nmerged = 0u;
  if (d_merged != 0xFFFFFFFFu) {
    const double mw = (double)sm.merged_w * (1.0 / 1099511627776.0);
    mmerged.hi = (float)mw;
    mmerged.lo = (float)(mw - (double)mmerged.hi);
    umerged = (float)(-(double)sm.merged_u * (1.0 / 4294967296.0));
    nmerged = sm.merged_n;
  }
  const uint32_t bpt = (dmax + NT) / NT;   // ceil((dmax + 1) / NT)
  const uint32_t d0 = (uint32_t)tid * bpt;
  auto bin = [&](uint32_t d, uint32_t& nb, DF& mass, float& um, float& wv, float& xv) {
    nb = 0u; mass = DF{0.f, 0.f}; um = 0.f; wv = 0.f; xv = 0.f;
    if (d > dmax) return;
    if (d == d_merged) {
      nb = nmerged; mass = mmerged; um = umerged;
      return;
    }
    nb = sm.hist.rel[d];
    if (nb == 0u) return;
    const float vv = RowBf16::value_of_key(expand_key(ck_m - d));
    const float dd = __fsub_rn(vv, m);
    wv = ex2(__fmul_rn(dd, c));
    xv = __fmul_rn(dd, inv_t);
    mass.hi = __fmul_rn((float)nb, wv);
    um = __fmul_rn(mass.hi, xv);
  };
  DF tot{0.f, 0.f};
  uint32_t tcnt = 0u;
  float tum = 0.f;
  if (d0 <= dmax) {
    for (uint32_t j = 0; j < bpt; ++j) {
      uint32_t nb; DF ms; float um, wv, xv;
      bin(d0 + j, nb, ms, um, wv, xv);
      tot = df_add(tot, ms);
      tcnt += nb;
      tum = __fadd_rn(tum, um);
    }
  }
  // exclusive scan of the per-thread totals in thread order
  const int lane = tid & 31, warp = tid >> 5;
  DF inc = tot;
  uint32_t icnt = tcnt;
  float ium = tum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    DF lft{shfl_up(inc.hi, o), shfl_up(inc.lo, o)};
    const uint32_t lc = __shfl_up_sync(0xFFFFFFFFu, icnt, o);
    const float lu = shfl_up(ium, o);
    if (lane >= o) {
      inc = df_add(lft, inc);
      icnt += lc;
      ium = __fadd_rn(lu, ium);
    }
  }
  DF exc{shfl_up(inc.hi, 1), shfl_up(inc.lo, 1)};
  uint32_t ecnt = __shfl_up_sync(0xFFFFFFFFu, icnt, 1);
  float eum = shfl_up(ium, 1);
  if (lane == 0) { exc = DF{0.f, 0.f}; ecnt = 0u; eum = 0.f; }
  if (lane == 31) {
    sm.scan_wtot[warp] = inc;
    sm.scan_wcnt[warp] = icnt;
    sm.scan_wum[warp] = ium;
  }
  __syncthreads();
  if (warp == 0) {   // exclusive scan of the warp totals, in warp order
    DF t = lane < NWARP ? sm.scan_wtot[lane] : DF{0.f, 0.f};
    uint32_t tc = lane < NWARP ? sm.scan_wcnt[lane] : 0u;
    float tu = lane < NWARP ? sm.scan_wum[lane] : 0.f;
#pragma unroll
    for (int o = 1; o < NWARP; o <<= 1) {
      DF lft{shfl_up(t.hi, o), shfl_up(t.lo, o)};
      const uint32_t lc = __shfl_up_sync(0xFFFFFFFFu, tc, o);
      const float lu = shfl_up(tu, o);
      if (lane >= o) {
        t = df_add(lft, t);
        tc += lc;
        tu = __fadd_rn(lu, tu);
      }
    }
    DF e{shfl_up(t.hi, 1), shfl_up(t.lo, 1)};
    uint32_t ec = __shfl_up_sync(0xFFFFFFFFu, tc, 1);
    float eu = shfl_up(tu, 1);
    if (lane == 0) { e = DF{0.f, 0.f}; ec = 0u; eu = 0.f; }
    if (lane < NWARP) {
      sm.scan_woff[lane] = e;
      sm.scan_woffc[lane] = ec;
      sm.scan_woffu[lane] = eu;
    }
  }
  __syncthreads();
  exc = df_add(sm.scan_woff[warp], exc);
  ecnt += sm.scan_woffc[warp];
  eum = __fadd_rn(sm.scan_woffu[warp], eum);
  // first bin whose inclusive prefix reaches the target; smallest index wins
  int my_d = -1;
  DF my_pb{0.f, 0.f};
  uint32_t my_cb = 0u, my_n = 0u;
  float my_ub = 0.f, my_w = 0.f, my_x = 0.f;
  if (d0 <= dmax) {
    DF P = exc;
    uint32_t pc = ecnt;
    float pu = eum;
    for (uint32_t j = 0; j < bpt; ++j) {
      uint32_t nb; DF ms; float um, wv, xv;
      bin(d0 + j, nb, ms, um, wv, xv);
      const DF Pn = df_add(P, ms);
      if (nb > 0u && df_ge(Pn, target)) {
        my_d = (int)(d0 + j);
        my_pb = P; my_cb = pc; my_ub = pu; my_w = wv; my_x = xv; my_n = nb;
        break;
      }
      P = Pn;
      pc += nb;
      pu = __fadd_rn(pu, um);
    }
    if (my_d >= 0) atomicMin(&sm.dstar, my_d);
  }
  __syncthreads();
  const int dstar = sm.dstar;
  if (my_d >= 0 && my_d == dstar) {
    sm.r_pb_hi = my_pb.hi; sm.r_pb_lo = my_pb.lo;
    sm.r_cnt_before = my_cb; sm.r_um_before = my_ub;
    sm.r_w = my_w; sm.r_x = my_x; sm.r_n = my_n;
  }
  __syncthreads();
  dstar_out = dstar;
  return dstar != 0x7FFFFFFF;
}

// Bin span of the window z >= zlo: the smallest key it can hold (truncating
// zlo's fp32 bits to bf16 moves it by less than one bf16 step) to ck_m.
__device__ __forceinline__ uint32_t window_dmax(float zlo, uint32_t ck_m, bool& merged_in) {
  const uint32_t k_lo_raw = okey16(__float_as_uint(zlo) >> 16);
  const uint32_t ck_lo = compress_key(k_lo_raw > 0u ? k_lo_raw - 1u : 0u);
  merged_in = (ck_lo <= MERGE_LO) && (MERGE_LO <= ck_m);
  return ck_m - ck_lo;   // ck_lo <= ck_m since zlo < m
}

// ------------------------------------------------ exact bisection fallback
// Largest key tau with mass(key >= tau) >= target, then the tie count at tau;
// every mass is a fixed-order pass over the row.  Results go to the output
// references (valid on all threads).
template <class Row>
__device__ __noinline__ void select_by_bisection(const Row& row, int tid, float m, float c, float inv_t,
                                    DF target, uint32_t key_y, int64_t y, Smem& sm,
                                    bool& all_tokens, DF& zs, float& us, uint32_t& kstar,
                                    bool& y_in, uint32_t& key_thr, uint32_t& ties) {
  auto mass_ge = [&](uint32_t t) -> DF {
    DF acc{0.f, 0.f};
    float dummy = 0.f;
    for_groups(row, tid, [&](const float (&v)[Row::E], int n, int64_t) {
#pragma unroll
      for (int k = 0; k < Row::E; ++k) {
        if (k < n && Row::key(v[k]) >= t)
          acc = df_add_f(acc, ex2(__fmul_rn(__fsub_rn(v[k], m), c)));
      }
    });
    block_sum_df(acc, dummy, sm, tid);
    return acc;
  };
  const DF full = mass_ge(0u);
  all_tokens = !df_ge(full, target);
  if (all_tokens) return;
  uint32_t tau = 0u;
  for (int b = Row::KEYBITS - 1; b >= 0; --b) {
    const uint32_t cand = tau | (1u << b);
    if (df_ge(mass_ge(cand), target)) tau = cand;
  }
  // One more pass: mass / count / entropy numerator above tau, ties at tau,
  // and the selected token's rank among the ties.
  DF mgt{0.f, 0.f};
  float ugt = 0.f;
  uint32_t cnt[4] = {0u, 0u, 0u, 0u};  // [0] key > tau, [1] key == tau, [2] ties before y
  for_groups(row, tid, [&](const float (&v)[Row::E], int n, int64_t g) {
#pragma unroll
    for (int k = 0; k < Row::E; ++k) {
      if (k >= n) continue;
      const uint32_t kk = Row::key(v[k]);
      if (kk > tau) {
        const float dd = __fsub_rn(v[k], m);
        const float w = ex2(__fmul_rn(dd, c));
        mgt = df_add_f(mgt, w);
        ugt = __fmaf_rn(w, __fmul_rn(dd, inv_t), ugt);
        cnt[0] += 1u;
      } else if (kk == tau) {
        cnt[1] += 1u;
        if (g * Row::E + k < y) cnt[2] += 1u;
      }
    }
  });
  block_sum_df(mgt, ugt, sm, tid);
  block_sum_u32(cnt, sm, tid);
  const float vt = Row::value_of_key(tau);
  const float dt = __fsub_rn(vt, m);
  const float wt = ex2(__fmul_rn(dt, c));
  const float xt = __fmul_rn(dt, inv_t);
  const float need = df_sub_to_f(target, mgt);
  float cf = ceilf(__fdiv_rn(need, wt));
  uint32_t cneed = cf < 1.f ? 1u : (cf > (float)cnt[1] ? cnt[1] : (uint32_t)cf);
  zs = df_add_f(mgt, __fmul_rn((float)cneed, wt));
  us = __fmaf_rn(__fmul_rn((float)cneed, wt), xt, ugt);
  kstar = cnt[0] + cneed;
  y_in = (key_y > tau) || (key_y == tau && cnt[2] < cneed);
  key_thr = tau;
  ties = cneed == cnt[1] ? kTiesAll : cneed;
}

// Threshold-bin bookkeeping shared by the histogram paths: the number of tied
// tokens needed, retained mass and entropy numerator, k*, membership of y.
__device__ __forceinline__ void finish_from_scan(const Smem& sm, DF target, int dstar,
                                                 uint32_t ck_m, uint32_t key_y, uint32_t tie_y,
                                                 DF& zs, float& us, uint32_t& kstar,
                                                 bool& y_in, uint32_t& key_thr, uint32_t& ties) {
  const DF pb{sm.r_pb_hi, sm.r_pb_lo};
  const float wt = sm.r_w, xt = sm.r_x;
  const uint32_t nt = sm.r_n;
  const float need = df_sub_to_f(target, pb);
  const float cf = ceilf(__fdiv_rn(need, wt));
  const uint32_t cneed = cf < 1.f ? 1u : (cf > (float)nt ? nt : (uint32_t)cf);
  zs = df_add_f(pb, __fmul_rn((float)cneed, wt));
  us = __fmaf_rn(__fmul_rn((float)cneed, wt), xt, sm.r_um_before);
  kstar = sm.r_cnt_before + cneed;
  key_thr = expand_key(ck_m - (uint32_t)dstar);
  ties = cneed == nt ? kTiesAll : cneed;
  const uint32_t d_y = ck_m - compress_key(key_y);
  y_in = (d_y < (uint32_t)dstar) || (d_y == (uint32_t)dstar && tie_y < cneed);
}

// Sum of w x over the whole row (fixed order), for rows whose nucleus turns out
// to be the whole vocabulary on the path that skipped it in pass 1.
__device__ __noinline__ float full_entropy_numerator(const RowBf16& row, int tid, float m, float c,
                                        float inv_t, Smem& sm) {
  DF dummy{0.f, 0.f};
  float u = 0.f;
  for_groups(row, tid, [&](const float (&v)[8], int n, int64_t) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (k < n) {
        const float dd = __fsub_rn(v[k], m);
        u = __fmaf_rn(ex2(__fmul_rn(dd, c)), __fmul_rn(dd, inv_t), u);
      }
    }
  });
  block_sum_df(dummy, u, sm, tid);
  return u;
}

// The saved state of a finished row.  The sums here are taken relative to m
// (w = 2^((z - m) c)); the state's reference is E = fp32(m c), so ln Z_S moves
// by ln2 (m c - E), computed exactly by one fma.
__device__ __forceinline__ void write_state(const LpeArgs& a, int64_t r, float m, float c, float lz,
                                            float h, uint32_t key_thr, uint32_t ties, bool y_in,
                                            uint32_t kstar, float row_t) {
  const float E = __fmul_rn(m, c);
  const float lzE = __fmaf_rn(kLn2, __fmaf_rn(m, c, -E), lz);
  a.state[r] = RowState{E, lzE, h, key_thr, ties, kStateValid | (y_in ? kStateYIn : 0u),
                        (int32_t)kstar, row_t};
}

__device__ __forceinline__ void write_bad_state(const LpeArgs& a, int64_t r, uint32_t bit) {
  if (a.state) a.state[r] = RowState{0.f, 0.f, 0.f, 0u, 0u, bit << 8, 0, 0u};
}

// --------------------------------------------------------------- kernel
template <class Row, bool TOPP>
__global__ void __launch_bounds__(NT, 3) lpe_kernel(LpeArgs a, float c0, float inv_t0) {
  pdl_trigger();
  pdl_wait();   // as the recompute pass, the streaming kernel's marks and outputs
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int tid = threadIdx.x;
  constexpr bool BF = Row::KEYBITS == 16;
  constexpr bool HIST = TOPP && BF;   // histogram select (else bisection at top_p < 1)
  int64_t i_row = 0;   // this CTA's row count (the recompute pass reads its marks NT at a time)
  for (int64_t r = blockIdx.x; r < a.T; r += gridDim.x, ++i_row) {
    bool wide_first = false;   // the streaming kernel found its window's mass short
    if (a.only_marked) {
      const int slot = (int)(i_row % NT);
      if (slot == 0) {
        __syncthreads();
        const int64_t rr = r + (int64_t)tid * gridDim.x;
        const uint32_t mb = rr < a.T ? __float_as_uint(a.out_logprob[rr]) : 0u;
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, mb == kRecomputeMark || mb == kRecomputeMarkWide);
        const uint32_t wbal = __ballot_sync(0xFFFFFFFFu, mb == kRecomputeMarkWide);
        if ((tid & 31) == 0) {
          sm.marked[tid >> 5] = bal;
          sm.wide[tid >> 5] = wbal;
        }
        __syncthreads();
      }
      if (((sm.marked[slot >> 5] >> (slot & 31)) & 1u) == 0u) continue;
      wide_first = ((sm.wide[slot >> 5] >> (slot & 31)) & 1u) != 0u;
    }
    Row row;
    row.p = reinterpret_cast<decltype(row.p)>(a.logits) + r * a.ld;
    row.V = a.V;
    row.aligned = (reinterpret_cast<uintptr_t>(row.p) & 15u) == 0;
    const int64_t y = a.ids[r];
    if (y < 0 || y >= a.V) {
      if (tid == 0) {
        a.out_logprob[r] = NAN;
        a.out_entropy[r] = NAN;
        if (a.out_k) a.out_k[r] = 0;
        if (a.status) atomicOr(a.status, RLK_STATUS_BAD_TOKEN_ID);
        write_bad_state(a, r, RLK_STATUS_BAD_TOKEN_ID);
      }
      continue;
    }
    // The row's sampling parameters: the call's, or its own (per-row mode,
    // with c and 1 / T formed exactly as the host forms the call's).
    float c = c0, inv_t = inv_t0, temp = a.temperature, top_p = a.top_p, row_t = 0.f;
    if (a.temps || a.top_ps) {
      if (a.temps) temp = a.temps[r];
      if (a.top_ps) top_p = a.top_ps[r];
      if (!(isfinite(temp) && temp > 0.f && top_p > 0.f && top_p <= 1.f)) {
        if (tid == 0) {
          a.out_logprob[r] = NAN;
          a.out_entropy[r] = NAN;
          if (a.out_k) a.out_k[r] = 0;
          if (a.status) atomicOr(a.status, RLK_STATUS_BAD_PARAM);
          write_bad_state(a, r, RLK_STATUS_BAD_PARAM);
        }
        continue;
      }
      c = (float)(1.4426950408889634 / (double)temp);
      inv_t = (float)(1.0 / (double)temp);
      if (a.temps) row_t = temp;
    }
    const bool row_topp = TOPP && top_p < 1.0f;
    const float zy = row.elem(y);    // the selected logit
    const uint32_t key_y = Row::key(zy);

    // ---- pass 1: online max / sum (/ entropy numerator)
    Online st{-INFINITY, 0.f, 0.f, 0.f};
    if constexpr (BF) {
      float gmin = INFINITY;
      if constexpr (HIST) {
        if (tid == 0) sm.gmin_key = 0xFFFFFFFFu;
        const bool sketch = (a.V + 8 * NT - 1) / (8 * NT) <= SK_ROUNDS;
        pass1_packed<4, false>(row, tid, c, st, gmin, sketch ? sm.gmax : nullptr);
        const uint32_t gk = __reduce_min_sync(0xFFFFFFFFu, okey32(__float_as_uint(gmin)));
        if ((tid & 31) == 0) atomicMin(&sm.gmin_key, gk);
      } else {
        pass1_packed<8, true>(row, tid, c, st, gmin, nullptr);
      }
    } else {
      for_groups<TOPP ? 4 : 8>(row, tid, [&](const float (&v)[Row::E], int n, int64_t) {
        absorb<Row::E>(st, v, n, c);
      });
    }
    st = block_reduce_online(st, c, sm, tid);   // its barriers also publish gmin_key
    const float m = st.m;
    const DF Z{st.hi, st.lo};
    const float zf = __fadd_rn(st.hi, st.lo);
    bool bad = !(isfinite(zf) && isfinite(st.u) && isfinite(m));
    if constexpr (HIST) bad = bad || isinf(__uint_as_float(okey32_inverse(sm.gmin_key)));
    if (bad) {
      if (tid == 0) {
        a.out_logprob[r] = NAN;
        a.out_entropy[r] = NAN;
        if (a.out_k) a.out_k[r] = 0;
        if (a.status) atomicOr(a.status, RLK_STATUS_NONFINITE);
        write_bad_state(a, r, RLK_STATUS_NONFINITE);
      }
      __syncthreads();
      continue;
    }
    const float x_y = __fdiv_rn(__fsub_rn(zy, m), temp);
    if (!row_topp) {
      // top_p = 1 (a per-row top_p of 1 in a top-p launch has no entropy
      // numerator from the packed pass 1: one more pass gives it)
      float u_ln2 = __fmul_rn(kLn2, st.u);
      if constexpr (HIST) u_ln2 = full_entropy_numerator(row, tid, m, c, inv_t, sm);
      if (tid == 0) {
        const float lz = logf(zf);
        const float h = __fsub_rn(lz, __fdiv_rn(u_ln2, zf));
        a.out_logprob[r] = __fsub_rn(x_y, lz);
        a.out_entropy[r] = h;
        if (a.out_k) a.out_k[r] = (int32_t)a.V;
        if (a.state) write_state(a, r, m, c, lz, h, 0u, kTiesAll, true, (uint32_t)a.V, row_t);
      }
      __syncthreads();
      continue;
    }

    // ---- top_p < 1: nucleus select
    const DF target = df_mul_f(Z, top_p);
    const float one_m_p = __fsub_rn(1.f, top_p);
    // Speculative window depth (units of T), kept only if its own mass reaches
    // the target; worst-case depth, below which lies less than
    // V e^-L < (1 - top_p) Z of the mass.
    const float L_spec = logf(__fdiv_rn(1.f, one_m_p)) + 7.0f;
    const float L_worst =
        fmaxf(logf(__fdiv_rn((float)a.V, __fmul_rn(one_m_p, zf))), 0.f) + 0.5f;

    bool all_tokens = false, y_in = false, use_bisect = !HIST;
    DF zs{0.f, 0.f};
    float us = 0.f;
    uint32_t kstar = 0u, key_thr = 0u, ties = kTiesAll;

    if constexpr (HIST) {
      const uint32_t ck_m = compress_key(Row::key(m));
      bool done = false;
      // Second pass over the row (served from L2): the speculative window,
      // then, if its mass falls short, the worst-case window (at once for a
      // row whose speculative window the streaming kernel found short).
      for (int att = 0; att < 2 && !done && !use_bisect; ++att) {
        if (att == 0 && (!(L_spec < L_worst) || wide_first)) continue;
        const float L = att == 0 ? L_spec : L_worst;
        const float zlo = __fsub_rn(m, __fmul_rn(L, temp));
        bool merged_in;
        const uint32_t dmax = window_dmax(zlo, ck_m, merged_in);
        if (dmax >= (uint32_t)HB) { use_bisect = true; break; }
        const uint32_t d_merged = merged_in ? ck_m - MERGE_LO : 0xFFFFFFFFu;
        for (uint32_t i = tid; i <= dmax; i += NT) sm.hist.rel[i] = 0u;
        if (tid == 0) {
          sm.dstar = 0x7FFFFFFF;
          sm.merged_w = 0ull;
          sm.merged_u = 0ull;
          sm.merged_n = 0u;
        }
        __syncthreads();
        // The sketch pass lists the candidate groups and reloads only those:
        // worth it while they are sparse.  When a quarter of the groups or
        // more are candidates (flat rows, wide nuclei) the window pass reads
        // the row whole and counts each thread's groups in place (dense);
        // rows too long for the sketch take the window pass with its queue.
        // All three build the same integer counts.
        const bool has_sketch = (a.V + 8 * NT - 1) / (8 * NT) <= SK_ROUNDS;
        bool use_sketch = has_sketch;
        if (use_sketch) {
          const int64_t ngroups = (a.V + 7) / 8;
          uint32_t cc[4] = {0u, 0u, 0u, 0u};
          for (int r2 = 0; (int64_t)r2 * NT + tid < ngroups; ++r2)
            cc[0] += bf16_val(sm.gmax[r2][tid]) >= zlo ? 1u : 0u;
          block_sum_u32(cc, sm, tid);
          use_sketch = (int64_t)cc[0] * 4 < ngroups;
        }
        uint32_t cnt2[4] = {0u, 0u, 0u, 0u};
        cnt2[0] = use_sketch ? sketch_pass(row, tid, zlo, m, c, inv_t, ck_m, key_y, y, sm)
                             : window_pass(row, tid, zlo, m, c, inv_t, ck_m, key_y, y, sm, has_sketch);
        block_sum_u32(cnt2, sm, tid);  // also the barrier after the histogram
        int dstar;
        const bool found = scan_bins(tid, dmax, d_merged, ck_m, m, c, inv_t, target, sm, dstar);
        if (!found) {
          if (att == 1) all_tokens = true;   // rounding left the total below top_p
          continue;
        }
        if ((uint32_t)dstar == d_merged) { use_bisect = true; break; }
        finish_from_scan(sm, target, dstar, ck_m, key_y, cnt2[0], zs, us, kstar, y_in, key_thr,
                         ties);
        done = true;
      }
      __syncthreads();
      if (all_tokens) us = full_entropy_numerator(row, tid, m, c, inv_t, sm);
    }
    if (use_bisect) {
      all_tokens = false;
      select_by_bisection(row, tid, m, c, inv_t, target, key_y, y, sm, all_tokens, zs, us,
                          kstar, y_in, key_thr, ties);
      if (all_tokens) {
        if constexpr (HIST) us = full_entropy_numerator(row, tid, m, c, inv_t, sm);
        else us = __fmul_rn(kLn2, st.u);
      }
    }
    if (tid == 0) {
      float lz, hval;
      if (all_tokens) {
        lz = logf(zf);
        hval = __fsub_rn(lz, __fdiv_rn(us, zf));
        kstar = (uint32_t)a.V;
        y_in = true;
        key_thr = 0u;
        ties = kTiesAll;
      } else {
        const float zsf = __fadd_rn(zs.hi, zs.lo);
        lz = logf(zsf);
        hval = __fsub_rn(lz, __fdiv_rn(us, zsf));
      }
      a.out_logprob[r] = y_in ? __fsub_rn(x_y, lz) : -INFINITY;
      a.out_entropy[r] = hval;
      if (a.out_k) a.out_k[r] = (int32_t)kstar;
      if (a.state) write_state(a, r, m, c, lz, hval, key_thr, ties, y_in, kstar, row_t);
    }
    __syncthreads();
  }
}

}  // namespace

constexpr int64_t kMarkedRowsPerCta = 8;   // rows per CTA of the recompute pass

cudaError_t launch_logprob_entropy(const LpeArgs& a, cudaStream_t stream) {
  // c = log2(e) / T rounded once; inv_t = 1 / T.
  const float c = (float)(1.4426950408889634 / (double)a.temperature);
  const float inv_t = (float)(1.0 / (double)a.temperature);
  const int64_t grid64 = a.T < (int64_t)3 * sm_count() ? a.T : (int64_t)3 * sm_count();
  const dim3 grid((unsigned)grid64), block(NT);
  // per-row parameters: the kernels' top-p form (rows with top_p = 1 take
  // its all-tokens branch)
  const bool per_row = a.temps != nullptr || a.top_ps != nullptr;
  const bool topp = per_row || a.top_p < 1.0f;
  const size_t smem = sizeof(Smem);

  static std::atomic<int> attr_done[64];   // once per device
  const int ds = device_slot();
  if (ds < 0 || !attr_done[ds].load()) {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(lpe_kernel<RowBf16, true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(lpe_kernel<RowBf16, false>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(lpe_kernel<RowF32, true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(lpe_kernel<RowF32, false>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
      return e;
    if (ds >= 0) attr_done[ds].store(1);
  }
  if (!a.only_marked && lpe_stream_eligible(a)) {
    cudaError_t e = launch_lpe_stream(a, stream, debug_wait_limit(), debug_take_withheld());
    if (e != cudaSuccess || !topp) return e;
    LpeArgs b = a;   // rows the streaming kernel marked for recomputation
    b.only_marked = 1;
    // About a CTA for every 8 rows, in whole multiples of the usual grid: a
    // CTA without marked rows ends at once, so the block scheduler hands the
    // marked rows to the SMs as they free up, and when every row is marked
    // the waves stay full.  (With only the usual grid, each CTA taking every
    // 456th row, a few CTAs got several marked rows and set the launch's
    // time.)
    const int64_t waves = (a.T + grid64 * kMarkedRowsPerCta - 1) / (grid64 * kMarkedRowsPerCta);
    const int64_t rg = grid64 * waves;
    const dim3 rgrid((unsigned)(rg < 0x7FFFFFFF ? rg : 0x7FFFFFFF));
    cudaError_t le = launch_after(lpe_kernel<RowBf16, true>, rgrid, block, smem, stream, b, c, inv_t);
    return le != cudaSuccess ? le : cudaGetLastError();
  }
  if (a.dtype == 0) {
    if (topp) lpe_kernel<RowBf16, true><<<grid, block, smem, stream>>>(a, c, inv_t);
    else lpe_kernel<RowBf16, false><<<grid, block, smem, stream>>>(a, c, inv_t);
  } else {
    if (topp) lpe_kernel<RowF32, true><<<grid, block, smem, stream>>>(a, c, inv_t);
    else lpe_kernel<RowF32, false><<<grid, block, smem, stream>>>(a, c, inv_t);
  }
  return cudaGetLastError();
}

}  // namespace rlk
