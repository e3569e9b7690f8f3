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
//  top_p < 1: every retained token lies in the window z >= m - L T with
//   L = ln(V / ((1 - top_p) Z)) + 0.5, because the tokens below it carry less
//   than V e^-L < (1 - top_p) Z of the mass.  Pass 2 re-reads the row (an L2
//   hit) and counts the window's tokens per distinct bf16 value into a
//   shared-memory histogram indexed by key distance from the max; values with
//   |z| < 2^-12 share one bin whose mass is summed token by token.  All tokens
//   of one value carry the same mass, so a bin's mass is count x w(value):
//   integer counts make the histogram independent of thread timing.  A
//   fixed-order double-float scan over the bins (largest value first) finds
//   the bin where the prefix mass reaches top_p * Z and how many of its tied
//   tokens are needed (ties are kept lower id first).  The retained mass Z_S,
//   the entropy and the selected token's membership (its rank among equal
//   values is counted in pass 2) follow.
//  Rows whose window is wider than the histogram, rows whose threshold falls
//   in the shared near-zero bin, and fp32 rows at top_p < 1 instead bisect
//   on the value key with fixed-order passes over the row (exact, slower).
//  Each of these choices depends only on the row's own values, and every sum
//   has a fixed order, so a row's output bits never depend on the batch.

#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "rlk.h"

namespace rlk {
namespace {

constexpr int NT = 512;
constexpr int NWARP = NT / 32;
constexpr int HB = 8192;         // histogram bins (32 KB of shared memory)
constexpr int BPT = HB / NT;     // bins per thread in the scan

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
  __device__ static __forceinline__ uint32_t key(float v) { return okey32(__float_as_uint(v)); }
  __device__ static __forceinline__ float value_of_key(uint32_t k) {
    return __uint_as_float(okey32_inverse(k));
  }
};

// Calls f(values, n_valid, group) for this thread's groups in a fixed order
// (g = tid, tid + NT, ...), whatever the row's alignment.  Aligned rows issue
// four 16-byte loads before using them.
template <class Row, class F>
__device__ __forceinline__ void for_groups(const Row& row, int tid, F&& f) {
  constexpr int E = Row::E;
  const int64_t nfull = row.V / E;
  int64_t g = tid;
  if (row.aligned) {
    for (; g + 3 * NT < nfull; g += 4 * NT) {
      float a[E], b[E], c[E], d[E];
      row.vec(g, a);
      row.vec(g + NT, b);
      row.vec(g + 2 * NT, c);
      row.vec(g + 3 * NT, d);
      f(a, E, g);
      f(b, E, g + NT);
      f(c, E, g + 2 * NT);
      f(d, E, g + 3 * NT);
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

// Fold one group of N values (the first n valid) into the state.
template <int N>
__device__ __forceinline__ void absorb(Online& st, const float (&v)[N], int n, float c) {
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
}

// ------------------------------------------------------ block reductions
struct Smem {
  uint32_t hist[HB];
  float red[NWARP][4];
  float bc[8];          // broadcast slots
  uint32_t ured[NWARP][4];
  uint32_t ubc[4];
  DF scan_wtot[NWARP];
  uint32_t scan_wcnt[NWARP];
  float scan_wum[NWARP];
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

// ------------------------------------------------ exact bisection fallback
// Largest key tau with mass(key >= tau) >= target, then the tie count at tau;
// every mass is a fixed-order pass over the row.  Results go to the output
// references (valid on all threads).
template <class Row>
__device__ void select_by_bisection(const Row& row, int tid, float m, float c, float inv_t,
                                    DF target, uint32_t key_y, int64_t y, Smem& sm,
                                    bool& all_tokens, DF& zs, float& us, uint32_t& kstar,
                                    bool& y_in) {
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
}

// --------------------------------------------------------------- kernel
template <class Row, bool TOPP>
__global__ void __launch_bounds__(NT, 2) lpe_kernel(LpeArgs a, float c, float inv_t) {
  __shared__ Smem sm;
  const int tid = threadIdx.x;
  for (int64_t r = blockIdx.x; r < a.T; r += gridDim.x) {
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
      }
      continue;
    }
    const float zy = [&] {
      float v[Row::E];
      // the selected logit, read through the same element decoding
      const int64_t gy = y / Row::E;
      row.scal(gy, v);
      return v[y - gy * Row::E];
    }();

    // ---- pass 1: online max / sum / entropy numerator
    Online st{-INFINITY, 0.f, 0.f, 0.f};
    for_groups(row, tid, [&](const float (&v)[Row::E], int n, int64_t) {
      absorb<Row::E>(st, v, n, c);
    });
    st = block_reduce_online(st, c, sm, tid);
    const float m = st.m;
    const DF Z{st.hi, st.lo};
    const float zf = __fadd_rn(st.hi, st.lo);
    if (!(isfinite(zf) && isfinite(st.u) && isfinite(m))) {
      if (tid == 0) {
        a.out_logprob[r] = NAN;
        a.out_entropy[r] = NAN;
        if (a.out_k) a.out_k[r] = 0;
        if (a.status) atomicOr(a.status, RLK_STATUS_NONFINITE);
      }
      continue;
    }
    const float x_y = __fdiv_rn(__fsub_rn(zy, m), a.temperature);
    if (!TOPP) {
      if (tid == 0) {
        const float lz = logf(zf);
        a.out_logprob[r] = __fsub_rn(x_y, lz);
        a.out_entropy[r] = __fsub_rn(lz, __fdiv_rn(__fmul_rn(kLn2, st.u), zf));
        if (a.out_k) a.out_k[r] = (int32_t)a.V;
      }
      continue;
    }

    // ---- top_p < 1: nucleus select
    const DF target = df_mul_f(Z, a.top_p);
    const float L = fmaxf(logf(__fdiv_rn((float)a.V, __fmul_rn(__fsub_rn(1.f, a.top_p), zf))), 0.f) + 0.5f;
    const float zlo = __fsub_rn(m, __fmul_rn(L, a.temperature));
    const uint32_t key_y = Row::key(zy);

    bool all_tokens = false, y_in = false, use_bisect = (Row::KEYBITS != 16);
    DF zs{0.f, 0.f};
    float us = 0.f;
    uint32_t kstar = 0u;

    if constexpr (Row::KEYBITS == 16) {
     if (!use_bisect) {
      const uint32_t ck_m = compress_key(Row::key(m));
      // smallest key the window can hold: truncating zlo's fp32 bits to bf16
      // moves it by less than one bf16 step.
      const uint32_t k_lo_raw = okey16(__float_as_uint(zlo) >> 16);
      const uint32_t ck_lo = compress_key(k_lo_raw > 0u ? k_lo_raw - 1u : 0u);
      const uint32_t dmax = ck_m - ck_lo;  // ck_lo <= ck_m since zlo < m
      if (dmax >= (uint32_t)HB) {
        use_bisect = true;
      } else {
        const bool merged_in = (ck_lo <= MERGE_LO) && (MERGE_LO <= ck_m);
        const uint32_t d_merged = merged_in ? ck_m - MERGE_LO : 0xFFFFFFFFu;
        for (uint32_t i = tid; i <= dmax; i += NT) sm.hist[i] = 0u;
        if (tid == 0) sm.dstar = 0x7FFFFFFF;
        __syncthreads();
        // ---- pass 2: window histogram (re-read, served from L2)
        DF mm{0.f, 0.f};      // merged-bin mass
        float mu = 0.f;       // merged-bin mass * x
        uint32_t cnt[4] = {0u, 0u, 0u, 0u};  // [0] merged count, [1] ties before y
        for_groups(row, tid, [&](const float (&v)[Row::E], int n, int64_t g) {
#pragma unroll
          for (int k = 0; k < Row::E; ++k) {
            if (k < n && v[k] >= zlo) {
              const uint32_t kk = Row::key(v[k]);
              const uint32_t ck = compress_key(kk);
              if (ck == MERGE_LO) {
                const float dd = __fsub_rn(v[k], m);
                const float w = ex2(__fmul_rn(dd, c));
                mm = df_add_f(mm, w);
                mu = __fmaf_rn(w, __fmul_rn(dd, inv_t), mu);
                cnt[0] += 1u;
              } else {
                atomicAdd(&sm.hist[ck_m - ck], 1u);
              }
              if (kk == key_y && g * Row::E + k < y) cnt[1] += 1u;
            }
          }
        });
        if (merged_in) block_sum_df(mm, mu, sm, tid);
        block_sum_u32(cnt, sm, tid);  // includes a barrier after the histogram

        // ---- scan: chunk totals per thread
        const uint32_t d0 = (uint32_t)tid * BPT;
        auto bin = [&](uint32_t d, uint32_t& nb, float& mass_hi, float& mass_lo, float& um,
                       float& wv, float& xv) {
          nb = 0u; mass_hi = 0.f; mass_lo = 0.f; um = 0.f; wv = 0.f; xv = 0.f;
          if (d > dmax) return;
          if (d == d_merged) {
            nb = cnt[0]; mass_hi = mm.hi; mass_lo = mm.lo; um = mu;
            return;
          }
          nb = sm.hist[d];
          if (nb == 0u) return;
          const float vv = Row::value_of_key(expand_key(ck_m - d));
          const float dd = __fsub_rn(vv, m);
          wv = ex2(__fmul_rn(dd, c));
          xv = __fmul_rn(dd, inv_t);
          mass_hi = __fmul_rn((float)nb, wv);
          um = __fmul_rn(mass_hi, xv);
        };
        DF tot{0.f, 0.f};
        uint32_t tcnt = 0u;
        float tum = 0.f;
        if (d0 <= dmax) {
          for (int j = 0; j < BPT; ++j) {
            uint32_t nb; float mh, ml, um, wv, xv;
            bin(d0 + j, nb, mh, ml, um, wv, xv);
            tot = df_add(tot, DF{mh, ml});
            tcnt += nb;
            tum = __fadd_rn(tum, um);
          }
        }
        // ---- exclusive scan of chunk totals in thread order
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
        DF woff{0.f, 0.f};
        uint32_t wcnt = 0u;
        float wum = 0.f;
        for (int w = 0; w < warp; ++w) {
          woff = df_add(woff, sm.scan_wtot[w]);
          wcnt += sm.scan_wcnt[w];
          wum = __fadd_rn(wum, sm.scan_wum[w]);
        }
        exc = df_add(woff, exc);
        ecnt += wcnt;
        eum = __fadd_rn(wum, eum);
        // ---- first bin (in scan order) whose inclusive prefix reaches the
        // target.  Every thread checks its own bins; the smallest index wins.
        int my_d = -1;
        DF my_pb{0.f, 0.f};
        uint32_t my_cb = 0u, my_n = 0u;
        float my_ub = 0.f, my_w = 0.f, my_x = 0.f;
        if (d0 <= dmax) {
          DF P = exc;
          uint32_t pc = ecnt;
          float pu = eum;
          for (int j = 0; j < BPT; ++j) {
            uint32_t nb; float mh, ml, um, wv, xv;
            bin(d0 + j, nb, mh, ml, um, wv, xv);
            const DF Pn = df_add(P, DF{mh, ml});
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
        if (dstar == 0x7FFFFFFF) {
          all_tokens = true;
        } else if ((uint32_t)dstar == d_merged) {
          use_bisect = true;
        } else {
          const DF pb{sm.r_pb_hi, sm.r_pb_lo};
          const float wt = sm.r_w, xt = sm.r_x;
          const uint32_t nt = sm.r_n;
          const float need = df_sub_to_f(target, pb);
          const float cf = ceilf(__fdiv_rn(need, wt));
          const uint32_t cneed = cf < 1.f ? 1u : (cf > (float)nt ? nt : (uint32_t)cf);
          zs = df_add_f(pb, __fmul_rn((float)cneed, wt));
          us = __fmaf_rn(__fmul_rn((float)cneed, wt), xt, sm.r_um_before);
          kstar = sm.r_cnt_before + cneed;
          const uint32_t d_y = ck_m - compress_key(key_y);
          y_in = (d_y < (uint32_t)dstar) || (d_y == (uint32_t)dstar && cnt[1] < cneed);
        }
        __syncthreads();
      }
     }
    }
    if (use_bisect) {
      select_by_bisection(row, tid, m, c, inv_t, target, key_y, y, sm, all_tokens, zs, us,
                          kstar, y_in);
    }
    if (tid == 0) {
      float lz, hval;
      if (all_tokens) {
        lz = logf(zf);
        hval = __fsub_rn(lz, __fdiv_rn(__fmul_rn(kLn2, st.u), zf));
        kstar = (uint32_t)a.V;
        y_in = true;
      } else {
        const float zsf = __fadd_rn(zs.hi, zs.lo);
        lz = logf(zsf);
        hval = __fsub_rn(lz, __fdiv_rn(us, zsf));
      }
      a.out_logprob[r] = y_in ? __fsub_rn(x_y, lz) : -INFINITY;
      a.out_entropy[r] = hval;
      if (a.out_k) a.out_k[r] = (int32_t)kstar;
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_logprob_entropy(const LpeArgs& a, cudaStream_t stream) {
  // c = log2(e) / T rounded once; inv_t = 1 / T.
  const float c = (float)(1.4426950408889634 / (double)a.temperature);
  const float inv_t = (float)(1.0 / (double)a.temperature);
  const int64_t grid64 = a.T < (int64_t)2 * sm_count() ? a.T : (int64_t)2 * sm_count();
  const dim3 grid((unsigned)grid64), block(NT);
  const bool topp = a.top_p < 1.0f;
  if (a.dtype == 0) {
    if (topp) lpe_kernel<RowBf16, true><<<grid, block, 0, stream>>>(a, c, inv_t);
    else lpe_kernel<RowBf16, false><<<grid, block, 0, stream>>>(a, c, inv_t);
  } else {
    if (topp) lpe_kernel<RowF32, true><<<grid, block, 0, stream>>>(a, c, inv_t);
    else lpe_kernel<RowF32, false><<<grid, block, 0, stream>>>(a, c, inv_t);
  }
  return cudaGetLastError();
}

}  // namespace rlk
