// rlk_logprob_entropy_support kernel: log-probability of the selected token
// and entropy over a retained set supplied by the sampler.
//
// RL-Kernel "Qwen3-8B VIME train-rollout consistency", section "ROCm MI300X
// and gfx942": the sparse path scores the complete retained support the
// sampler produced (its CSR retained set) rather than recomputing it.  Row t
// keeps exactly the ids support_ids[support_offsets[t] .. support_offsets[t+1]).
//
// One CTA of NTS threads per row, rows strided over the grid.  List position
// j goes to thread (j - start) mod NTS, so the order of every sum depends only
// on the list.  Each thread gathers its listed logits (four loads in flight),
// keeps an online state (max m, sum of 2^d as a double-float, sum of 2^d d,
// d = (z - m) log2(e) / T), and the states merge along a fixed tree.  Only the
// listed logits are read: the traffic is one 32-byte sector per listed token
// at worst, instead of the whole row.

#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "rlk.h"

namespace rlk {
namespace {

constexpr int NTS = 128;
constexpr int NWS = NTS / 32;
constexpr int NCACHE = 2048;   // listed logits a backward CTA keeps in shared memory

struct St {
  float m, hi, lo, u;
};

__device__ __forceinline__ bool st_empty(const St& a) {
  return a.m == -INFINITY && a.hi == 0.f && a.lo == 0.f && a.u == 0.f;
}

// Merge two states (a is the left operand; the tree fixes which is which).
__device__ __forceinline__ St st_merge(const St& a, const St& b, float c) {
  if (st_empty(b)) return a;
  if (st_empty(a)) return b;
  const float M = fmaxf(a.m, b.m);
  const float da = __fmul_rn(__fsub_rn(M, a.m), c);
  const float db = __fmul_rn(__fsub_rn(M, b.m), c);
  const float fa = (a.m == M) ? 1.f : ex2(-da);
  const float fb = (b.m == M) ? 1.f : ex2(-db);
  const float sa = __fadd_rn(a.hi, a.lo), sb = __fadd_rn(b.hi, b.lo);
  St r;
  r.m = M;
  r.u = __fadd_rn(__fmul_rn(fa, __fmaf_rn(-da, sa, a.u)), __fmul_rn(fb, __fmaf_rn(-db, sb, b.u)));
  float s, e;
  two_sum(__fmul_rn(a.hi, fa), __fmul_rn(b.hi, fb), s, e);
  e = __fadd_rn(e, __fadd_rn(__fmul_rn(a.lo, fa), __fmul_rn(b.lo, fb)));
  r.hi = __fadd_rn(s, e);
  r.lo = __fsub_rn(e, __fsub_rn(r.hi, s));
  return r;
}

// Fold one value into the state.
__device__ __forceinline__ void st_absorb(St& st, float z, float c) {
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

template <bool BF>
__device__ __forceinline__ float load_z(const void* logits, int64_t off) {
  if (BF) return bf16_val(__ldg(reinterpret_cast<const uint16_t*>(logits) + off));
  return __ldg(reinterpret_cast<const float*>(logits) + off);
}

// The row's sums over its list, merged along a fixed tree; valid in t / f on
// thread 0 (f: 1 y listed, 2 a non-finite listed logit, 4 a listed id out of
// range).
// With s_cache, list position j0 + i (i < NCACHE) also keeps its logit in
// s_cache[i]; position j always belongs to thread (j - j0) mod NTS, so the
// same thread reads it back later without a barrier.
template <bool BF>
__device__ void row_sums(const SupportArgs& a, int64_t j0, int64_t j1, int64_t y, int64_t base,
                         float c, St (&s_red)[NWS], uint32_t (&s_flags)[NWS], St& t, uint32_t& f,
                         float* s_cache = nullptr) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  {
    St st{-INFINITY, 0.f, 0.f, 0.f};
    uint32_t flags = 0u;   // 1: y listed, 2: non-finite listed logit, 4: listed id out of range
    for (int64_t j = j0 + tid; j < j1; j += 4 * NTS) {
      int32_t id[4];
      float z[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) id[k] = (j + k * NTS < j1) ? __ldg(a.support + j + k * NTS) : -1;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        z[k] = (id[k] >= 0 && id[k] < a.V) ? load_z<BF>(a.logits, base + id[k]) : 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (j + k * NTS >= j1) continue;
        if (id[k] < 0 || id[k] >= a.V) {
          flags |= 4u;
          continue;
        }
        if (s_cache && j + k * NTS - j0 < NCACHE) s_cache[j + k * NTS - j0] = z[k];
        if (!isfinite(z[k])) flags |= 2u;
        if (id[k] == y) flags |= 1u;
        st_absorb(st, z[k], c);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const St x{shfl_down(st.m, o), shfl_down(st.hi, o), shfl_down(st.lo, o), shfl_down(st.u, o)};
      st = st_merge(st, x, c);
    }
    flags = __reduce_or_sync(0xFFFFFFFFu, flags);
    if (lane == 0) {
      s_red[warp] = st;
      s_flags[warp] = flags;
    }
    __syncthreads();
    if (tid == 0) {
      t = s_red[0];
      f = s_flags[0];
      for (int w = 1; w < NWS; ++w) {
        t = st_merge(t, s_red[w], c);
        f |= s_flags[w];
      }
    }
  }
}

// Status of a row from its sums (0 when the row is good).
__device__ __forceinline__ uint32_t row_status(const SupportArgs& a, int64_t j0, int64_t j1,
                                               int64_t y, const St& t, uint32_t f) {
  uint32_t bad = 0u;
  if (y < 0 || y >= a.V) bad = RLK_STATUS_BAD_TOKEN_ID;
  else if (j1 <= j0 || (f & 4u)) bad = RLK_STATUS_BAD_SUPPORT;
  else if (f & 2u) bad = RLK_STATUS_NONFINITE;
  const float zf = __fadd_rn(t.hi, t.lo);
  if (!bad && !(isfinite(zf) && isfinite(t.u))) bad = RLK_STATUS_NONFINITE;
  return bad;
}

template <bool BF>
__global__ void __launch_bounds__(NTS) support_kernel(SupportArgs a, float c) {
  __shared__ St s_red[NWS];
  __shared__ uint32_t s_flags[NWS];
  const int tid = threadIdx.x;
  for (int64_t r = blockIdx.x; r < a.T; r += gridDim.x) {
    const int64_t j0 = a.offsets[r], j1 = a.offsets[r + 1];
    const int64_t y = a.ids[r];
    const int64_t base = r * a.ld;
    St t;
    uint32_t f;
    row_sums<BF>(a, j0, j1, y, base, c, s_red, s_flags, t, f);
    if (tid == 0) {
      const uint32_t bad = row_status(a, j0, j1, y, t, f);
      const float zf = __fadd_rn(t.hi, t.lo);
      if (bad) {
        a.out_logprob[r] = NAN;
        a.out_entropy[r] = NAN;
        if (a.status) atomicOr(a.status, bad);
      } else {
        const float lz = logf(zf);
        const float zy = load_z<BF>(a.logits, base + y);
        a.out_logprob[r] = (f & 1u) ? __fsub_rn(__fdiv_rn(__fsub_rn(zy, t.m), a.temperature), lz)
                                    : -INFINITY;
        a.out_entropy[r] = __fsub_rn(lz, __fdiv_rn(__fmul_rn(kLn2, t.u), zf));
      }
    }
    __syncthreads();
  }
}

// Backward: for every list position j, dL/dz of the listed id with the set
// held fixed, L = g_lp logprob + g_H H:
//   g_lp ([i = y] - q_i) / T (when y is listed) - g_H q_i (ln q_i + H) / T,
// q_i = exp((z_i - m) / T) / Z_S.  The first pass keeps the first NCACHE
// listed logits of the row in shared memory; the second pass takes them from
// there and gathers only the rest again (from L2, where the first pass left
// them).
template <bool BF>
__global__ void __launch_bounds__(NTS) support_backward_kernel(SupportArgs a, float c) {
  __shared__ St s_red[NWS];
  __shared__ uint32_t s_flags[NWS];
  __shared__ float s_b[6];   // m, 1 / Z_S, ln Z_S, H, g_lp (0 when y is not listed), g_H; NaN: bad row
  __shared__ float s_z[NCACHE];
  const int tid = threadIdx.x;
  for (int64_t r = blockIdx.x; r < a.T; r += gridDim.x) {
    const int64_t j0 = a.offsets[r], j1 = a.offsets[r + 1];
    const int64_t y = a.ids[r];
    const int64_t base = r * a.ld;
    St t;
    uint32_t f;
    row_sums<BF>(a, j0, j1, y, base, c, s_red, s_flags, t, f, s_z);
    if (tid == 0) {
      const uint32_t bad = row_status(a, j0, j1, y, t, f);
      const float zf = __fadd_rn(t.hi, t.lo);
      if (bad) {
        if (a.status) atomicOr(a.status, bad);
        s_b[0] = NAN;
      } else {
        const float lz = logf(zf);
        s_b[0] = t.m;
        s_b[1] = __fdiv_rn(1.f, zf);
        s_b[2] = lz;
        s_b[3] = __fsub_rn(lz, __fdiv_rn(__fmul_rn(kLn2, t.u), zf));
        s_b[4] = (f & 1u) && a.grad_logprob ? a.grad_logprob[r] : 0.f;
        s_b[5] = a.grad_entropy ? a.grad_entropy[r] : 0.f;
      }
    }
    __syncthreads();
    const float m = s_b[0];
    if (isnan(m)) {
      for (int64_t j = j0 + tid; j < j1; j += NTS) a.grad_support[j] = NAN;
    } else {
      const float rz = s_b[1], lz = s_b[2], H = s_b[3], glp = s_b[4], gh = s_b[5];
      const float inv_t = __fdiv_rn(1.f, a.temperature);
      for (int64_t j = j0 + tid; j < j1; j += NTS) {
        const int32_t id = __ldg(a.support + j);
        const float z = j - j0 < NCACHE ? s_z[j - j0] : load_z<BF>(a.logits, base + id);
        const float d = __fmul_rn(__fsub_rn(z, m), c);
        const float q = __fmul_rn(ex2(d), rz);
        const float lq = __fsub_rn(__fmul_rn(d, kLn2), lz);      // ln q
        const float dlp = __fsub_rn(id == y ? 1.f : 0.f, q);
        const float dh = -__fmul_rn(q, __fadd_rn(lq, H));
        a.grad_support[j] = __fmul_rn(__fmaf_rn(glp, dlp, __fmul_rn(gh, dh)), inv_t);
      }
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_support_backward(const SupportArgs& a, cudaStream_t stream) {
  const float c = (float)(1.4426950408889634 / (double)a.temperature);
  const int64_t cap = (int64_t)16 * sm_count();
  const dim3 grid((unsigned)(a.T < cap ? a.T : cap)), block(NTS);
  if (a.dtype == 0) support_backward_kernel<true><<<grid, block, 0, stream>>>(a, c);
  else support_backward_kernel<false><<<grid, block, 0, stream>>>(a, c);
  return cudaGetLastError();
}

cudaError_t launch_support(const SupportArgs& a, cudaStream_t stream) {
  const float c = (float)(1.4426950408889634 / (double)a.temperature);
  const int64_t cap = (int64_t)16 * sm_count();
  const dim3 grid((unsigned)(a.T < cap ? a.T : cap)), block(NTS);
  if (a.dtype == 0) support_kernel<true><<<grid, block, 0, stream>>>(a, c);
  else support_kernel<false><<<grid, block, 0, stream>>>(a, c);
  return cudaGetLastError();
}

}  // namespace rlk
