// rlk_logprob_entropy_bwd kernel: dL/dz over the whole vocabulary for
// L = sum_t g_lp[t] logprob_t + g_H[t] H_t, the retained set of each row held
// fixed (it only moves where a logit crosses the boundary, so almost
// everywhere it is locally constant).
//
// RL-Kernel "Qwen3-8B VIME train-rollout consistency", section "ROCm MI300X
// and gfx942": top-p < 1 rows are scored over the complete retained set,
// renormalised; its gradient is the softmax gradient restricted to S at
// temperature T:
//   grad_i = 0                                                     (i not in S)
//   grad_i = (g_lp [y in S] ([i = y] - q_i) - g_H q_i (ln q_i + H)) / T   (i in S)
// with q_i = 2^(z_i c - E) / e^lz from the state the forward saved.
//
// One CTA of NTB threads per row, rows strided over the grid.  Each step a
// thread owns 16 consecutive ids (32 bytes of bf16), so the row streams in id
// order with 16-byte loads and stores.  S is "key > key_thr, plus the first
// `ties` ids with key == key_thr": when the boundary's ties are split, the
// rank of each tied id is a running count over the row, taken per step with a
// warp scan and one block barrier (double-buffered warp totals).  Rows whose
// ties are all kept need no barrier.  Ids outside S cost one integer compare
// and a zero store; only members evaluate ex2.

#include <cuda_bf16.h>
#include <math.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "rlk.h"

namespace rlk {
namespace {

constexpr int NTB = 256;
constexpr int NWB = NTB / 32;
constexpr int EPT = 16;   // consecutive ids per thread per step
constexpr float kLog2e = 1.4426950408889634f;

template <bool BF>
__device__ __forceinline__ uint32_t key_of(float v) {
  if (BF) return okey16(__float_as_uint(v) >> 16);
  return okey32(__float_as_uint(v));
}

// 16 logits from id i0 (vector loads when the whole run is inside the row and
// the row is 16-byte aligned; ids past V read as -inf and are never members).
template <bool BF>
__device__ __forceinline__ void load16(const void* row, bool vec, int64_t i0, int64_t V,
                                       float (&v)[EPT]) {
  if (BF) {
    const uint16_t* p = reinterpret_cast<const uint16_t*>(row);
    if (vec && i0 + EPT <= V) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(p + i0));
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(p + i0) + 1);
      const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        v[2 * k] = bf16_lo(w[k]);
        v[2 * k + 1] = bf16_hi(w[k]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < EPT; ++e) v[e] = i0 + e < V ? bf16_val(__ldg(p + i0 + e)) : -INFINITY;
    }
  } else {
    const float* p = reinterpret_cast<const float*>(row);
    if (vec && i0 + EPT <= V) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 q = __ldg(reinterpret_cast<const float4*>(p + i0) + k);
        v[4 * k] = q.x; v[4 * k + 1] = q.y; v[4 * k + 2] = q.z; v[4 * k + 3] = q.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < EPT; ++e) v[e] = i0 + e < V ? __ldg(p + i0 + e) : -INFINITY;
    }
  }
}

template <bool BO>
__device__ __forceinline__ void store16(void* row, bool vec, int64_t i0, int64_t V,
                                        const float (&g)[EPT]) {
  if (BO) {
    uint16_t* p = reinterpret_cast<uint16_t*>(row);
    if (vec && i0 + EPT <= V) {
      uint32_t w[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(g[2 * k], g[2 * k + 1]);
        w[k] = *reinterpret_cast<const uint32_t*>(&h);
      }
      uint4* q = reinterpret_cast<uint4*>(p + i0);
      q[0] = make_uint4(w[0], w[1], w[2], w[3]);
      q[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        if (i0 + e < V) {
          const __nv_bfloat16 h = __float2bfloat16_rn(g[e]);
          p[i0 + e] = *reinterpret_cast<const uint16_t*>(&h);
        }
      }
    }
  } else {
    float* p = reinterpret_cast<float*>(row);
    if (vec && i0 + EPT <= V) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        reinterpret_cast<float4*>(p + i0)[k] =
            make_float4(g[4 * k], g[4 * k + 1], g[4 * k + 2], g[4 * k + 3]);
    } else {
#pragma unroll
      for (int e = 0; e < EPT; ++e)
        if (i0 + e < V) p[i0 + e] = g[e];
    }
  }
}

// The lowest n set bits of m (0 <= n).
__device__ __forceinline__ uint32_t lowest_bits(uint32_t m, int n) {
  uint32_t r = 0u;
  for (int j = 0; j < n && m; ++j) {
    const uint32_t b = m & (0u - m);
    r |= b;
    m ^= b;
  }
  return r;
}

template <bool BF, bool BO>
__global__ void __launch_bounds__(NTB, 4) lpe_backward_kernel(LpeBwdArgs a, float c, float inv_t) {
  __shared__ uint32_t s_wt[2][NWB];   // per-warp tie counts of a step (double-buffered)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t per_step = (int64_t)NTB * EPT;
  const int64_t nstep = (a.V + per_step - 1) / per_step;
  uint32_t phase = 0u;   // barrier steps taken by this CTA (selects the buffer)
  for (int64_t r = blockIdx.x; r < a.T; r += gridDim.x) {
    const RowState st = a.state[r];
    const int64_t y = a.ids[r];
    const char* lrow = reinterpret_cast<const char*>(a.logits) + r * a.ld * (BF ? 2 : 4);
    char* grow = reinterpret_cast<char*>(a.grad_logits) + r * a.ldg * (BO ? 2 : 4);
    const bool vin = (reinterpret_cast<uintptr_t>(lrow) & 15u) == 0;
    const bool vout = (reinterpret_cast<uintptr_t>(grow) & 15u) == 0;
    const bool good = (st.flags & kStateValid) != 0u && y >= 0 && y < a.V;
    if (!good) {
      if (tid == 0 && a.status) {
        uint32_t bits = st.flags >> 8;
        if (y < 0 || y >= a.V) bits |= RLK_STATUS_BAD_TOKEN_ID;
        if (bits == 0u) bits = RLK_STATUS_NO_STATE;
        atomicOr(a.status, bits);
      }
      float g[EPT];
#pragma unroll
      for (int e = 0; e < EPT; ++e) g[e] = NAN;
      for (int64_t s = 0; s < nstep; ++s) store16<BO>(grow, vout, (s * NTB + tid) * EPT, a.V, g);
      continue;
    }
    const float glp = (st.flags & kStateYIn) && a.grad_logprob ? a.grad_logprob[r] : 0.f;
    const float gh = a.grad_entropy ? a.grad_entropy[r] : 0.f;
    const float lz2 = __fmul_rn(st.lz, kLog2e);
    const bool split = st.ties != kTiesAll;   // uniform over the CTA
    uint32_t carry = 0u;                      // tied ids before this step
    for (int64_t s = 0; s < nstep; ++s) {
      const int64_t i0 = (s * NTB + tid) * EPT;
      float v[EPT];
      load16<BF>(lrow, vin, i0, a.V, v);
      uint32_t gt = 0u, tie = 0u;
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        const uint32_t k = key_of<BF>(v[e]);
        if (i0 + e < a.V) {
          if (k > st.key_thr) gt |= 1u << e;
          else if (k == st.key_thr) tie |= 1u << e;
        }
      }
      uint32_t in = gt | tie;
      if (split) {
        const uint32_t n = (uint32_t)__popc(tie);
        uint32_t inc = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t l = __shfl_up_sync(0xFFFFFFFFu, inc, o);
          if (lane >= o) inc += l;
        }
        const int b = (int)(phase & 1u);
        if (lane == 31) s_wt[b][warp] = inc;
        __syncthreads();
        uint32_t before = carry, total = 0u;
#pragma unroll
        for (int w = 0; w < NWB; ++w) {
          const uint32_t t = s_wt[b][w];
          if (w < warp) before += t;
          total += t;
        }
        carry += total;
        ++phase;
        const uint32_t first = before + inc - n;   // rank of this thread's first tied id
        const int keep = st.ties > first ? (int)min(st.ties - first, n) : 0;
        in = gt | lowest_bits(tie, keep);
      }
      float g[EPT];
      if (in == 0u) {
#pragma unroll
        for (int e = 0; e < EPT; ++e) g[e] = 0.f;
      } else {
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
          g[e] = 0.f;
          if ((in >> e) & 1u) {
            const float t = __fsub_rn(__fmaf_rn(v[e], c, -st.E), lz2);   // log2 q
            const float q = ex2(t);
            const float lnq = __fmul_rn(t, kLn2);
            const float dlp = __fsub_rn(i0 + e == y ? 1.f : 0.f, q);
            const float dh = -__fmul_rn(q, __fadd_rn(lnq, st.H));
            g[e] = __fmul_rn(__fmaf_rn(glp, dlp, __fmul_rn(gh, dh)), inv_t);
          }
        }
      }
      store16<BO>(grow, vout, i0, a.V, g);
    }
  }
}

template <bool BF, bool BO>
cudaError_t launch_typed(const LpeBwdArgs& a, float c, float inv_t, cudaStream_t stream) {
  static std::atomic<int> per_sm{0};   // resident CTAs per SM (one GPU type per process)
  int occ = per_sm.load();
  if (occ == 0) {
    const cudaError_t e =
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, lpe_backward_kernel<BF, BO>, NTB, 0);
    if (e != cudaSuccess) return e;
    occ = occ < 1 ? 1 : occ;
    per_sm.store(occ);
  }
  const int64_t cap = (int64_t)occ * sm_count();
  const dim3 grid((unsigned)(a.T < cap ? a.T : cap)), block(NTB);
  lpe_backward_kernel<BF, BO><<<grid, block, 0, stream>>>(a, c, inv_t);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_logprob_entropy_backward(const LpeBwdArgs& a, cudaStream_t stream) {
  // The same c = log2(e) / T, rounded once, as the forward.
  const float c = (float)(1.4426950408889634 / (double)a.temperature);
  const float inv_t = (float)(1.0 / (double)a.temperature);
  if (a.dtype == 0) {
    return a.grad_dtype == 0 ? launch_typed<true, true>(a, c, inv_t, stream)
                             : launch_typed<true, false>(a, c, inv_t, stream);
  }
  return a.grad_dtype == 0 ? launch_typed<false, true>(a, c, inv_t, stream)
                           : launch_typed<false, false>(a, c, inv_t, stream);
}

}  // namespace rlk
