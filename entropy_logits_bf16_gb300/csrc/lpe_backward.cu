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

// The row's c = log2(e) / T and 1 / T: from the temperature its state
// recorded (a forward with per-row temperatures), else the call's.
__device__ __forceinline__ void row_consts(const RowState& st, float c0, float inv_t0, float& c,
                                           float& inv_t) {
  c = c0;
  inv_t = inv_t0;
  if (st.temperature > 0.f) {
    c = (float)(1.4426950408889634 / (double)st.temperature);
    inv_t = (float)(1.0 / (double)st.temperature);
  }
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
__global__ void __launch_bounds__(NTB, 4) lpe_backward_kernel(LpeBwdArgs a, float c0, float inv_t0) {
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
    float c, inv_t;
    row_consts(st, c0, inv_t0, c, inv_t);
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

// ------------------------------------------------------------ pipelined
// Rows of 16-byte-aligned bf16 logits with V % 8 == 0 (and aligned gradient
// rows) stream through a ring of NSTG shared-memory stages filled by
// cp.async.bulk, so ~NSTG x 16 KB per CTA are in flight whatever the register
// budget (the register-staged kernel above keeps 32 bytes a thread in flight
// and reaches about a third of HBM bandwidth).  A stage holds PT x GPT
// 16-byte groups; thread t takes groups t, t + PT, ... (conflict-free shared
// reads, coalesced stores).  The one block barrier per stage releases the
// stage to its refill and publishes the warps' tie counts, four 8-group
// counts packed two to a word.
constexpr int PT = 256;
constexpr int PW = PT / 32;
constexpr int GPT = 4;                        // 16-byte groups per thread per stage
constexpr int64_t STG = (int64_t)PT * GPT * 16;   // stage bytes (16 KB)
constexpr int NSTG = 4;

struct PSmem {
  unsigned long long full[NSTG];   // mbarriers, one per stage
  uint4 wt[2][PW / 2];             // inclusive warp tie counts (2 words a warp), double-buffered
  int abort;
};
constexpr int RING_OFF = 256;   // the ring starts here (16-byte aligned for the bulk copies)
static_assert(sizeof(PSmem) <= RING_OFF, "PSmem fits below the ring");

// Waits for a phase with no abort short-cut, for at most ~2^31 cycles (the
// copies still in flight when a CTA that timed out leaves).
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > (1ll << 31)) return;
}

template <bool BO>
__global__ void __launch_bounds__(PT, 3) lpe_backward_pipe_kernel(LpeBwdArgs a, float c0, float inv_t0) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  PSmem& sm = *reinterpret_cast<PSmem*>(smem_raw);
  uint8_t* ring = smem_raw + RING_OFF;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t RB = a.V * 2;   // row bytes, a multiple of 16
  const int64_t nch = (RB + STG - 1) / STG;
  const int64_t nrow = (a.T - (int64_t)blockIdx.x + gridDim.x - 1) / gridDim.x;
  const int64_t G = nrow * nch;   // stages this CTA consumes
  const char* logits = reinterpret_cast<const char*>(a.logits);

  auto issue = [&](int64_t g) {   // one thread: stage g's bytes into slot g % NSTG
    const int64_t r = blockIdx.x + (g / nch) * (int64_t)gridDim.x;
    const int64_t off = (g % nch) * STG;
    const uint32_t bytes = (uint32_t)(RB - off < STG ? RB - off : STG);
    const int sl = (int)(g % NSTG);
    const uint32_t bar = smem_u32(&sm.full[sl]);
    mbar_expect_tx(bar, bytes);
    bulk_copy_g2s(smem_u32(ring + sl * STG), logits + r * a.ld * 2 + off, bytes, bar);
  };
  if (tid == 0) {
    for (int sl = 0; sl < NSTG; ++sl) mbar_init(smem_u32(&sm.full[sl]), 1u);
    sm.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int64_t g = 0; g < G && g < NSTG; ++g) issue(g);

  RowState st{};
  int64_t r = 0, y = 0;
  bool good = false, split = false;
  // Per member: t = log2 q = z c - (E + log2 Z_S), q = 2^t and
  //   grad = q (-C t - B) + A [i = y],
  // A = g_lp / T, B = (g_lp + g_H H) / T, C = g_H ln2 / T.
  float thr_v = 0.f, thr_up = 0.f, A = 0.f;   // the boundary value and the next bf16 above it
  float2 c2 = make_float2(c0, c0), nE2 = c2, nB2 = c2, nC2 = c2;
  uint32_t carry = 0u, phase = 0u;
  for (int64_t g = 0; g < G; ++g) {
    const int64_t ch = g % nch;
    if (ch == 0) {   // the first stage of a row
      r = blockIdx.x + (g / nch) * (int64_t)gridDim.x;
      st = a.state[r];
      y = a.ids[r];
      good = (st.flags & kStateValid) != 0u && y >= 0 && y < a.V;
      if (!good && tid == 0 && a.status) {
        uint32_t bits = st.flags >> 8;
        if (y < 0 || y >= a.V) bits |= RLK_STATUS_BAD_TOKEN_ID;
        if (bits == 0u) bits = RLK_STATUS_NO_STATE;
        atomicOr(a.status, bits);
      }
      float c, inv_t;
      row_consts(st, c0, inv_t0, c, inv_t);
      c2 = make_float2(c, c);
      const float glp = good && (st.flags & kStateYIn) && a.grad_logprob ? a.grad_logprob[r] : 0.f;
      const float gh = good && a.grad_entropy ? a.grad_entropy[r] : 0.f;
      const float eref = __fadd_rn(st.E, __fmul_rn(st.lz, kLog2e));
      A = __fmul_rn(glp, inv_t);
      const float B = __fmul_rn(__fmaf_rn(gh, st.H, glp), inv_t);
      const float C = __fmul_rn(__fmul_rn(gh, kLn2), inv_t);
      nE2 = make_float2(-eref, -eref);
      nB2 = make_float2(-B, -B);
      nC2 = make_float2(-C, -C);
      // key 0 is below every finite value: the whole row is kept
      thr_v = st.key_thr == 0u ? -INFINITY : bf16_val(okey16_inverse(st.key_thr));
      thr_up = bf16_val(okey16_inverse(st.key_thr + 1u));
      split = good && st.ties != kTiesAll;
      carry = 0u;
    }
    const int sl = (int)(g % NSTG);
    if (!mbar_wait_sleep(smem_u32(&sm.full[sl]), (uint32_t)((g / NSTG) & 1), &sm.abort) &&
        tid == 0 && a.status)
      atomicOr(a.status, RLK_STATUS_TIMEOUT);
    const int64_t off = ch * STG;
    const int ngroups = (int)((RB - off < STG ? RB - off : STG) >> 4);
    const uint4* sv = reinterpret_cast<const uint4*>(ring + sl * STG);
    uint4 qv[GPT];
#pragma unroll
    for (int j = 0; j < GPT; ++j)
      qv[j] = j * PT + tid < ngroups ? sv[j * PT + tid] : make_uint4(0u, 0u, 0u, 0u);
    // Members: z > thr, or z == thr and the tie is kept.  Every group is
    // evaluated (candidates are too dense for skipping them to pay: most warps
    // hold one); ties are counted with packed compares.
    uint32_t cnt01 = 0u, cnt23 = 0u, inc01 = 0u, inc23 = 0u;
    uint32_t ntie[GPT] = {0u, 0u, 0u, 0u};
    if (split) {
      const __nv_bfloat162 thr2 = __float2bfloat162_rn(thr_v);   // exact: thr_v is a bf16 value
#pragma unroll
      for (int j = 0; j < GPT; ++j) {
        if (j * PT + tid >= ngroups) continue;
        const uint32_t m0 = __heq2_mask(bf2(qv[j].x), thr2), m1 = __heq2_mask(bf2(qv[j].y), thr2);
        const uint32_t m2 = __heq2_mask(bf2(qv[j].z), thr2), m3 = __heq2_mask(bf2(qv[j].w), thr2);
        if ((m0 | m1 | m2 | m3) != 0u) {   // rare: a tied id in this group
          const uint32_t s4 = (m0 & 0x00010001u) + (m1 & 0x00010001u) + (m2 & 0x00010001u) +
                              (m3 & 0x00010001u);
          ntie[j] = (s4 & 0xFFFFu) + (s4 >> 16);
        }
      }
      cnt01 = ntie[0] | (ntie[1] << 16);
      cnt23 = ntie[2] | (ntie[3] << 16);
      inc01 = cnt01;
      inc23 = cnt23;
      if (__any_sync(0xFFFFFFFFu, (cnt01 | cnt23) != 0u)) {   // most warps hold no tie
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {   // 16-bit fields: at most 256 per warp
          const uint32_t l01 = __shfl_up_sync(0xFFFFFFFFu, inc01, o);
          const uint32_t l23 = __shfl_up_sync(0xFFFFFFFFu, inc23, o);
          if (lane >= o) {
            inc01 += l01;
            inc23 += l23;
          }
        }
      }
      if (lane == 31) {
        uint32_t* wt = reinterpret_cast<uint32_t*>(&sm.wt[phase & 1u][0]);
        wt[2 * warp] = inc01;
        wt[2 * warp + 1] = inc23;
      }
    }
    __syncthreads();   // the stage is free; the warps' tie counts are visible
    if (tid == 0 && g + NSTG < G) {
      fence_proxy_async_smem();
      issue(g + NSTG);
    }
    // Per group: members are z >= thr_eff, where thr_eff is the boundary
    // value while the group's ties are kept and the next value up once they are
    // not; the one group where the kept ties end also carries a mask (kt, bit e)
    // of the tied ids it keeps.
    float thr_eff[GPT] = {thr_v, thr_v, thr_v, thr_v};
    uint32_t kt[GPT] = {0xFFu, 0xFFu, 0xFFu, 0xFFu};
    if (split) {
      uint4 wv[PW / 2];
#pragma unroll
      for (int k = 0; k < PW / 2; ++k) wv[k] = sm.wt[phase & 1u][k];
      ++phase;
      uint32_t tot01 = 0u, tot23 = 0u;
#pragma unroll
      for (int k = 0; k < PW / 2; ++k) {
        tot01 += wv[k].x + wv[k].z;
        tot23 += wv[k].y + wv[k].w;
      }
      const uint32_t T0 = tot01 & 0xFFFFu, T1 = tot01 >> 16, T2 = tot23 & 0xFFFFu;
      const uint32_t c0 = carry;
      carry += T0 + T1 + T2 + (tot23 >> 16);
      if ((cnt01 | cnt23) != 0u) {   // only threads holding a tied id need its rank
        uint32_t pre01 = 0u, pre23 = 0u;
#pragma unroll
        for (int k = 0; k < PW / 2; ++k) {
          if (2 * k < warp) {
            pre01 += wv[k].x;
            pre23 += wv[k].y;
          }
          if (2 * k + 1 < warp) {
            pre01 += wv[k].z;
            pre23 += wv[k].w;
          }
        }
        const uint32_t ex01 = pre01 + inc01 - cnt01, ex23 = pre23 + inc23 - cnt23;
        const uint32_t base[GPT] = {c0 + (ex01 & 0xFFFFu), c0 + T0 + (ex01 >> 16),
                                    c0 + T0 + T1 + (ex23 & 0xFFFFu),
                                    c0 + T0 + T1 + T2 + (ex23 >> 16)};
#pragma unroll
        for (int j = 0; j < GPT; ++j) {
        const uint32_t keep = st.ties > base[j] ? min(st.ties - base[j], ntie[j]) : 0u;
        if (keep == ntie[j]) continue;          // all of this group's ties kept (or none tied)
        if (keep == 0u) {
          thr_eff[j] = thr_up;
          continue;
        }
        const uint32_t w[4] = {qv[j].x, qv[j].y, qv[j].z, qv[j].w};   // the split group
        uint32_t tm = 0u;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float z = (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]);
          if (z == thr_v) tm |= 1u << e;
        }
        kt[j] = lowest_bits(tm, (int)keep);
        }
      }
    }
    char* grow = reinterpret_cast<char*>(a.grad_logits) + r * a.ldg * (BO ? 2 : 4);
#pragma unroll
    for (int j = 0; j < GPT; ++j) {
      if (j * PT + tid >= ngroups) continue;
      const int64_t i0 = (off >> 1) + (int64_t)(j * PT + tid) * 8;
      float gv[8];
      if (!good) {
#pragma unroll
        for (int e = 0; e < 8; ++e) gv[e] = NAN;
      } else {
        const uint32_t w[4] = {qv[j].x, qv[j].y, qv[j].z, qv[j].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 z2 = bf16x2_to_f2(w[k]);
          const float2 t2 = __ffma2_rn(z2, c2, nE2);
          const float2 q2 = make_float2(ex2(t2.x), ex2(t2.y));
          const float2 g2 = __fmul2_rn(q2, __ffma2_rn(nC2, t2, nB2));
          gv[2 * k] = z2.x >= thr_eff[j] ? g2.x : 0.f;
          gv[2 * k + 1] = z2.y >= thr_eff[j] ? g2.y : 0.f;
        }
        if (kt[j] != 0xFFu) {   // the group where the kept ties end: drop the others
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float z = (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]);
            if (z == thr_v && !((kt[j] >> e) & 1u)) gv[e] = 0.f;
          }
        }
        const uint64_t ey = (uint64_t)(y - i0);   // the selected id's slot, if in this group
        if (ey < 8u && (st.flags & kStateYIn)) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if ((uint64_t)e == ey) gv[e] = __fadd_rn(gv[e], A);
        }
      }
      if (BO) {
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(gv[2 * k], gv[2 * k + 1]);
          o[k] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(grow + i0 * 2) = make_uint4(o[0], o[1], o[2], o[3]);
      } else {
        float4* p = reinterpret_cast<float4*>(grow + i0 * 4);
        p[0] = make_float4(gv[0], gv[1], gv[2], gv[3]);
        p[1] = make_float4(gv[4], gv[5], gv[6], gv[7]);
      }
    }
  }
  // After a timeout, wait (boundedly) for this CTA's copies still in flight:
  // the last phase issued on each slot.
  if (sm.abort && tid == 0) {
    for (int sl = 0; sl < NSTG; ++sl) {
      if (sl >= G) break;
      const int64_t g_last = sl + ((G - 1 - sl) / NSTG) * NSTG;
      mbar_drain(smem_u32(&sm.full[sl]), (uint32_t)((g_last / NSTG) & 1));
    }
  }
}

template <bool BO>
cudaError_t launch_pipe(const LpeBwdArgs& a, float c, float inv_t, cudaStream_t stream) {
  static std::atomic<int> per_sm[64];   // resident CTAs per SM, per device
  const int smem = RING_OFF + NSTG * (int)STG;
  const int ds = device_slot();
  int occ = ds >= 0 ? per_sm[ds].load() : 0;
  if (occ == 0) {
    cudaError_t e = cudaFuncSetAttribute(lpe_backward_pipe_kernel<BO>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, lpe_backward_pipe_kernel<BO>, PT, smem);
    if (e != cudaSuccess) return e;
    occ = occ < 1 ? 1 : occ;
    if (ds >= 0) per_sm[ds].store(occ);
  }
  const int64_t cap = (int64_t)occ * sm_count();
  const dim3 grid((unsigned)(a.T < cap ? a.T : cap)), block(PT);
  lpe_backward_pipe_kernel<BO><<<grid, block, smem, stream>>>(a, c, inv_t);
  return cudaGetLastError();
}

bool pipe_eligible(const LpeBwdArgs& a) {
  const uintptr_t lb = reinterpret_cast<uintptr_t>(a.logits);
  const uintptr_t gb = reinterpret_cast<uintptr_t>(a.grad_logits);
  return a.dtype == 0 && a.V % 8 == 0 && a.ld % 8 == 0 && lb % 16 == 0 && gb % 16 == 0 &&
         a.ldg % (a.grad_dtype == 0 ? 8 : 4) == 0;
}

template <bool BF, bool BO>
cudaError_t launch_typed(const LpeBwdArgs& a, float c, float inv_t, cudaStream_t stream) {
  static std::atomic<int> per_sm[64];   // resident CTAs per SM, per device
  const int ds = device_slot();
  int occ = ds >= 0 ? per_sm[ds].load() : 0;
  if (occ == 0) {
    const cudaError_t e =
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, lpe_backward_kernel<BF, BO>, NTB, 0);
    if (e != cudaSuccess) return e;
    occ = occ < 1 ? 1 : occ;
    if (ds >= 0) per_sm[ds].store(occ);
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
  if (pipe_eligible(a))
    return a.grad_dtype == 0 ? launch_pipe<true>(a, c, inv_t, stream)
                             : launch_pipe<false>(a, c, inv_t, stream);
  if (a.dtype == 0) {
    return a.grad_dtype == 0 ? launch_typed<true, true>(a, c, inv_t, stream)
                             : launch_typed<true, false>(a, c, inv_t, stream);
  }
  return a.grad_dtype == 0 ? launch_typed<false, true>(a, c, inv_t, stream)
                           : launch_typed<false, false>(a, c, inv_t, stream);
}

}  // namespace rlk
