// rlk_lmhead_logprob: the top_p = 1 logits path fused with the LM-head GEMM.
//
// What is computed: logits[t, v] = sum_k hidden[t, k] W[v, k] (bf16 inputs,
// fp32 accumulation, never rounded or stored), then for each row the
// full-vocabulary log-probability of the selected token and the entropy at
// temperature T (RL-Kernel "Qwen3-8B VIME train-rollout consistency", section
// "ROCm MI300X and gfx942": the full-vocabulary strict scorer at top_p = 1;
// prime-rl v0.10.0 notes, "1. Trainer Performance": the loss is chunked so the
// full logits need not exist at once; RL-Kernel "ROCm sparse performance"
// notes: a deterministic GEMM with a fixed reduction order).
//
// Design (sm_103a, one CTA per SM, persistent):
//  * Work unit = (128-row tile of hidden, one of NSLICE fixed vocabulary
//    slices).  Units are strided over the grid; the slice boundaries depend
//    only on V, so a row's result never depends on the batch size.
//  * warp 0: TMA producer.  Each stage holds a 128 x 64 tile of hidden and a
//    256 x 64 tile of W (bf16, 128-byte swizzle), 4 stages in shared memory,
//    completion tracked by mbarriers.
//  * warp 1: allocates 512 TMEM columns (two 128 x 256 fp32 accumulators) and
//    one elected thread issues tcgen05.mma (M=128, N=256, K=16) over K, then
//    commits to the stage's "empty" barrier and, after the last K step, to
//    the accumulator's "full" barrier.
//  * warps 2-5: epilogue, one TMEM lane (= one row) per thread.  tcgen05.ld
//    brings 32 columns at a time into registers; the columns fold into an
//    online (max, sum of 2^d as double-float, sum of 2^d d) state in column
//    order, and the selected token's logit is captured.  The accumulator is
//    handed back while the next tile's MMAs run into the other one.
//  * After a unit, each row's state goes to the workspace; a combine kernel
//    merges the NSLICE states of a row in slice order (fixed) and writes the
//    log-probability and entropy.
//  * Every wait on an mbarrier is bounded; on expiry the CTA raises
//    RLK_STATUS_TIMEOUT in the status word and winds down.

#include <cuda.h>
#include <math.h>

#include <atomic>
#include <mutex>


#include "common.cuh"
#include "internal.h"
#include "rlk.h"

namespace rlk {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int NSLICE = 19;
constexpr int THREADS = 192;
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t B_BYTES = BN * BK * 2;
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SPIN_LIMIT = 1u << 22;
constexpr size_t SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;

// ------------------------------------------------------------ PTX wrappers
// Bounded wait: false when `limit` clock cycles ran out (the abort flag is
// then raised) or another role gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u) {
      if (*abort) return false;
      if (clock64() - t0 > limit) {
        *abort = 1;
        return false;
      }
    }
  }
}

// The row-state marker of a slice that a timed-out CTA never finished: a
// negative sum, which no data produces; the combine turns it into NaN rows.
constexpr float kTimedOutSum = -1.0f;
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Shared-memory matrix descriptor: K-major tile written by TMA with the
// 128-byte swizzle; 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);   // start address
  d |= (uint64_t)1u << 16;                   // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024u >> 4) << 32;         // stride byte offset: next 8-row group
  d |= (uint64_t)1u << 46;                   // descriptor version
  d |= (uint64_t)2u << 61;                   // 128-byte swizzle
  return d;
}
// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, M x N.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(kIdesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// ------------------------------------------------------------ row state
struct RowState {
  float m, hi, lo, u;
};

__device__ __forceinline__ bool state_empty(const RowState& a) {
  return a.m == -INFINITY && a.hi == 0.f && a.lo == 0.f && a.u == 0.f;
}

__device__ __forceinline__ RowState state_merge(const RowState& a, const RowState& b, float c) {
  if (state_empty(b)) return a;
  if (state_empty(a)) return b;
  const float M = fmaxf(a.m, b.m);
  const float da = __fmul_rn(__fsub_rn(M, a.m), c);
  const float db = __fmul_rn(__fsub_rn(M, b.m), c);
  const float fa = (a.m == M) ? 1.f : ex2(-da);
  const float fb = (b.m == M) ? 1.f : ex2(-db);
  const float sa = __fadd_rn(a.hi, a.lo), sb = __fadd_rn(b.hi, b.lo);
  RowState r;
  r.m = M;
  r.u = __fadd_rn(__fmul_rn(fa, __fmaf_rn(-da, sa, a.u)), __fmul_rn(fb, __fmaf_rn(-db, sb, b.u)));
  float s, e;
  two_sum(__fmul_rn(a.hi, fa), __fmul_rn(b.hi, fb), s, e);
  e = __fadd_rn(e, __fadd_rn(__fmul_rn(a.lo, fa), __fmul_rn(b.lo, fb)));
  r.hi = __fadd_rn(s, e);
  r.lo = __fsub_rn(e, __fsub_rn(r.hi, s));
  return r;
}

// Fold 32 consecutive logits (the first n valid) into the state.
__device__ __forceinline__ void absorb32(RowState& st, const float (&v)[32], int n, float c) {
  float gm = -INFINITY;
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (j < n) gm = fmaxf(gm, v[j]);
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
  float w[32], d[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (j < n) {
      d[j] = __fmul_rn(__fsub_rn(v[j], st.m), c);
      w[j] = ex2(d[j]);
    } else {
      d[j] = 0.f;
      w[j] = 0.f;
    }
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) st.u = __fmaf_rn(w[j], d[j], st.u);
#pragma unroll
  for (int h = 16; h > 0; h >>= 1) {
#pragma unroll
    for (int j = 0; j < h; ++j) w[j] = __fadd_rn(w[j], w[j + h]);
  }
  float s, e;
  two_sum(st.hi, w[0], s, e);
  st.hi = s;
  st.lo = __fadd_rn(st.lo, e);
}

struct LmParams {
  int64_t T, V;
  int n_mt, n_nt, n_units, k_steps;
  const int32_t* ids;
  float c;               // log2(e) / temperature
  float4* part;          // [NSLICE][T] row states
  float* zy;             // [T] the selected token's logit
  float* debug_logits;   // [T][V] when non-null (validation aid)
  uint32_t* status;
  // gradient mode (grad == 1): the epilogue writes dL/dz (bf16) instead of
  // folding row states; emit mode (grad == 2): it writes the logits (bf16)
  int grad;
  const float* lse;      // [T] ln sum exp(z / T) from the forward
  const float* ent;      // [T] entropy from the forward
  const float* glp;      // [T] or NULL
  const float* gh;       // [T] or NULL
  uint16_t* dz;          // [T][ldz] bf16
  int64_t ldz;
  float inv_t;
  long long wait_limit;  // clock cycles a wait may take
  long long withhold;    // debug: the k-step copy the first CTA never issues (-1: none)
};

// Work unit u -> (row tile mt, vocabulary slice sl).  The slices go in blocks of
// SLICE_BLOCK and, inside a block, the row tiles: the CTAs at work at any time
// cover many row tiles of a few slices, so each W tile they read serves many
// row tiles from L2 while their hidden tiles stay resident too.  The order only
// changes which CTA runs a unit, never what it computes.
constexpr int SLICE_BLOCK = 4;
__device__ __forceinline__ void unit_coords(int u, int n_mt, int& mt, int& sl) {
  const int full = n_mt * SLICE_BLOCK;                 // units of a whole block of slices
  const int nfb = NSLICE / SLICE_BLOCK;                // whole blocks
  const int b = u / full;
  if (b < nfb) {
    const int r = u - b * full;
    mt = r / SLICE_BLOCK;
    sl = b * SLICE_BLOCK + r % SLICE_BLOCK;
  } else {                                             // the last, partial block
    const int last = NSLICE - nfb * SLICE_BLOCK;
    const int r = u - nfb * full;
    mt = r / last;
    sl = nfb * SLICE_BLOCK + r % last;
  }
}

__device__ __forceinline__ void slice_bounds(int n_nt, int sl, int& nt0, int& nt1) {
  nt0 = (int)((int64_t)sl * n_nt / NSLICE);
  nt1 = (int)((int64_t)(sl + 1) * n_nt / NSLICE);
}

__global__ void __launch_bounds__(THREADS, 1)
    lmhead_kernel(const __grid_constant__ CUtensorMap tmap_a,
                  const __grid_constant__ CUtensorMap tmap_b, LmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;            // 1024-aligned stage area
  uint8_t* base_ptr = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + STAGES * STAGE_BYTES);
  // bars: full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], then the
  // abort flag, the TMEM address and the drain barrier of an aborted MMA issuer
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * STAGES;
  const uint32_t accf0 = empty0 + 8 * STAGES, acce0 = accf0 + 16;
  const uint32_t drain_bar = smem_u32(bars + 2 * STAGES + 6);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf0 + 8 * a, 1);
      mbar_init(acce0 + 8 * a, 4);   // one arrive per epilogue warp
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0u, issued_parity = 0u;  // per stage: used, parity of last issue
      long long n_issue = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
        int mt, sl;
        unit_coords(u, p.n_mt, mt, sl);
        int nt0, nt1;
        slice_bounds(p.n_nt, sl, nt0, nt1);
        for (int nt = nt0; nt < nt1 && ok; ++nt) {
          for (int k = 0; k < p.k_steps; ++k, ++n_issue) {
            if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag, p.wait_limit)) { ok = false; break; }
            if (*abort_flag) { ok = false; break; }
            if (blockIdx.x == 0 && n_issue == p.withhold) {   // debug: a copy never issued
              if (++stage == STAGES) { stage = 0; phase ^= 1u; }
              continue;
            }
            const uint32_t fb = full0 + 8 * stage;
            mbar_expect_tx(fb, STAGE_BYTES);
            const uint32_t sa = base + stage * STAGE_BYTES;
            tma_load_2d(sa, &tmap_a, fb, k * BK, mt * BM);
            tma_load_2d(sa + A_BYTES, &tmap_b, fb, k * BK, nt * BN);
            issued_mask |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
        }
      }
      // If any role gave up, let every issued copy land before the CTA exits
      // (each wait bounded).
      if (!ok || *abort_flag) {
        for (int s2 = 0; s2 < STAGES; ++s2) {
          if (!(issued_mask & (1u << s2))) continue;
          const uint32_t par = (issued_parity >> s2) & 1u;
          for (uint32_t i = 0; i < SPIN_LIMIT; ++i)
            if (mbar_try_wait(full0 + 8 * s2, par)) break;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t tile = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
        int mt_unused, sl;
        unit_coords(u, p.n_mt, mt_unused, sl);
        int nt0, nt1;
        slice_bounds(p.n_nt, sl, nt0, nt1);
        for (int nt = nt0; nt < nt1 && ok; ++nt, ++tile) {
          const uint32_t acc = tile & 1u, accph = (tile >> 1) & 1u;
          if (!mbar_wait(acce0 + 8 * acc, accph ^ 1u, abort_flag, p.wait_limit)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_tmem = tmem + acc * BN;
          for (int k = 0; k < p.k_steps; ++k) {
            if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, p.wait_limit)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sa = base + stage * STAGE_BYTES;
            const uint64_t da = smem_desc_sw128(sa), db = smem_desc_sw128(sa + A_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              // advance 16 bf16 (32 bytes) along K inside the swizzle atom
              mma_bf16(d_tmem, da + (uint64_t)(kk * 2), db + (uint64_t)(kk * 2),
                       (k > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(empty0 + 8 * stage);
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
          if (ok) mma_commit(accf0 + 8 * acc);
        }
      }
      if (!ok) {
        // Let every MMA already issued finish before TMEM is freed (bounded).
        mma_commit(drain_bar);
        for (uint32_t i = 0; i < SPIN_LIMIT; ++i)
          if (mbar_try_wait(drain_bar, 0u)) break;
      }
    }
  } else {
    // ------------------------------------------------------ epilogue
    const int q = warp & 3;                     // TMEM lane quadrant of this warp
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t tile = 0;
    bool ok = true;
    int u_fail = p.n_units;
    for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
      u_fail = u;
      int mt, sl;
      unit_coords(u, p.n_mt, mt, sl);
      int nt0, nt1;
      slice_bounds(p.n_nt, sl, nt0, nt1);
      const int64_t row = (int64_t)mt * BM + q * 32 + lane;
      const int64_t y = row < p.T ? (int64_t)p.ids[row] : -1;
      // gradient mode: dz = q (-C t - B) + A [v = y] with t = log2 q
      // = z c - lse log2(e), A = g_lp / T, B = (g_lp + g_H H) / T,
      // C = g_H ln2 / T
      float gnE = 0.f, gA = 0.f, gB = 0.f, gC = 0.f;
      if (p.grad == 1 && row < p.T) {
        const float glp = p.glp ? p.glp[row] : 0.f, gh = p.gh ? p.gh[row] : 0.f;
        gnE = -__fmul_rn(p.lse[row], kLog2e);
        gA = __fmul_rn(glp, p.inv_t);
        gB = __fmul_rn(__fmaf_rn(gh, p.ent[row], glp), p.inv_t);
        gC = __fmul_rn(__fmul_rn(gh, kLn2), p.inv_t);
      }
      RowState st{-INFINITY, 0.f, 0.f, 0.f};
      float zy = 0.f;
      bool have_zy = false;
      for (int nt = nt0; nt < nt1; ++nt, ++tile) {
        const uint32_t acc = tile & 1u, accph = (tile >> 1) & 1u;
        if (!mbar_wait(accf0 + 8 * acc, accph, abort_flag, p.wait_limit)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int ch = 0; ch < BN / 32; ++ch) {
          float v[32];
          tmem_ld32(tmem + lane_base + acc * BN + ch * 32, v);
          const int64_t col0 = (int64_t)nt * BN + ch * 32;
          const int n = (int)(p.V - col0 < 32 ? (p.V - col0 > 0 ? p.V - col0 : 0) : 32);
          if (p.grad) {
            if (row < p.T && n > 0) {
              uint32_t o[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                float g2[2] = {v[2 * j], v[2 * j + 1]};
                if (p.grad == 1) {
#pragma unroll
                  for (int e = 0; e < 2; ++e) {
                    const float t = __fmaf_rn(v[2 * j + e], p.c, gnE);
                    const float qv = ex2(t);
                    g2[e] = __fmul_rn(qv, __fmaf_rn(-gC, t, -gB));
                    if (col0 + 2 * j + e == y) g2[e] = __fadd_rn(g2[e], gA);
                  }
                }
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(g2[0], g2[1]);
                o[j] = *reinterpret_cast<const uint32_t*>(&h2);
              }
              uint16_t* dst = p.dz + row * p.ldz + col0;
              if (n == 32) {
                uint4* d4 = reinterpret_cast<uint4*>(dst);   // ldz % 8 == 0, col0 % 32 == 0
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  d4[k] = make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (j < n) dst[j] = (uint16_t)((o[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
              }
            }
            continue;
          }
          if (n > 0) absorb32(st, v, n, p.c);
          if (y >= col0 && y < col0 + n) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (col0 + j == y) zy = v[j];
            have_zy = true;
          }
          if (p.debug_logits && row < p.T) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < n) p.debug_logits[row * p.V + col0 + j] = v[j];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce0 + 8 * acc);
      }
      if (ok && row < p.T && !p.grad) {
        p.part[(int64_t)sl * p.T + row] = make_float4(st.m, st.hi, st.lo, st.u);
        if (have_zy) p.zy[row] = zy;
      }
      if (ok) u_fail = p.n_units;
    }
    if (!ok) {
      // A wait ran out: every unit this CTA has not finished is marked, so
      // its rows come out NaN instead of normal-looking values.
      for (int u = u_fail; u < p.n_units; u += gridDim.x) {
        int umt, usl;
        unit_coords(u, p.n_mt, umt, usl);
        const int64_t row = (int64_t)umt * BM + q * 32 + lane;
        if (row >= p.T) continue;
        if (!p.grad) {
          p.part[(int64_t)usl * p.T + row] = make_float4(0.f, kTimedOutSum, 0.f, 0.f);
        } else {   // NaN logits or gradients: every result built on them is NaN
          int nt0, nt1;
          slice_bounds(p.n_nt, usl, nt0, nt1);
          const int64_t c1 = (int64_t)nt1 * BN < p.V ? (int64_t)nt1 * BN : p.V;
          for (int64_t col = (int64_t)nt0 * BN; col < c1; ++col) p.dz[row * p.ldz + col] = 0x7FC0u;
        }
      }
      if (lane == 0 && p.status) atomicOr(p.status, RLK_STATUS_TIMEOUT);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// Merge each row's slice states in slice order and write the outputs.
__global__ void __launch_bounds__(256) lmhead_combine_kernel(LmParams p, float* out_lp,
                                                             float* out_ent, float* out_lse,
                                                             float temperature) {
  const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= p.T) return;
  const int64_t y = p.ids[row];
  if (y < 0 || y >= p.V) {
    out_lp[row] = NAN;
    out_ent[row] = NAN;
    if (out_lse) out_lse[row] = NAN;
    if (p.status) atomicOr(p.status, RLK_STATUS_BAD_TOKEN_ID);
    return;
  }
  RowState st{-INFINITY, 0.f, 0.f, 0.f};
  bool timed_out = false;
  for (int sl = 0; sl < NSLICE; ++sl) {
    const float4 s = p.part[(int64_t)sl * p.T + row];
    timed_out = timed_out || s.y == kTimedOutSum;
    st = state_merge(st, RowState{s.x, s.y, s.z, s.w}, p.c);
  }
  if (timed_out) {   // the kernel has set RLK_STATUS_TIMEOUT
    out_lp[row] = NAN;
    out_ent[row] = NAN;
    if (out_lse) out_lse[row] = NAN;
    return;
  }
  const float z = __fadd_rn(st.hi, st.lo);
  if (!(isfinite(z) && isfinite(st.u) && isfinite(st.m))) {
    out_lp[row] = NAN;
    out_ent[row] = NAN;
    if (out_lse) out_lse[row] = NAN;
    if (p.status) atomicOr(p.status, RLK_STATUS_NONFINITE);
    return;
  }
  const float lz = logf(z);
  if (out_lse) out_lse[row] = __fadd_rn(__fdiv_rn(st.m, temperature), lz);
  out_lp[row] = __fsub_rn(__fdiv_rn(__fsub_rn(p.zy[row], st.m), temperature), lz);
  out_ent[row] = __fsub_rn(lz, __fdiv_rn(__fmul_rn(kLn2, st.u), z));
}

// ------------------------------------------------------------ plain GEMM
// D[M, N] (fp32, row-major, row stride ldd) = A[M, K] B[K, N] + beta D, with
// bf16 operands brought in by TMA and the products on the tensor cores
// (tcgen05, fp32 accumulators in TMEM), each tile's K in order (so the result
// is deterministic).  A_MN: A is stored with M contiguous (a [K][M] array),
// else with K contiguous ([M][K]); B_MN: B is stored with N contiguous
// ([K][N]), else with K contiguous ([N][K]).  An MN-contiguous operand comes in
// 64-element-wide TMA boxes of 64 K rows: 8-row groups of 128-byte swizzled
// rows, 1024 bytes apart, and the 64-element blocks 8192 bytes apart.
// Persistent: CTA b takes tiles b, b + grid, ...; warp 0 loads, one thread of
// warp 1 issues the MMAs into one of two TMEM accumulators, warps 2-5 store.
constexpr int GBM = 128, GBN = 256, GBK = 64, GSTAGES = 4;
constexpr uint32_t GA_BYTES = GBM * GBK * 2;
constexpr uint32_t GB_BYTES = GBN * GBK * 2;
constexpr uint32_t GSTAGE_BYTES = GA_BYTES + GB_BYTES;
constexpr uint32_t GMN_BLOCK = 64 * GBK * 2;   // one 64-element-wide MN block of a stage
constexpr size_t GSMEM_BYTES = GSTAGES * GSTAGE_BYTES + 1024 + 256;

struct GemmParams {
  int64_t M, N, K;
  int n_mt, n_nt, n_tiles, k_steps;
  int m_fast;          // consecutive tiles walk M (else N): CTAs at work share the other operand in L2
  float* D;
  int64_t ldd;
  float beta;
  long long wait_limit;
};

// MN-contiguous operand: lbo = byte distance between 64-element blocks.
__device__ __forceinline__ uint64_t smem_desc_mn_sw128(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);   // start address
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;   // leading byte offset: next 64-element block
  d |= (uint64_t)(1024u >> 4) << 32;         // stride byte offset: next 8-row group along K
  d |= (uint64_t)1u << 46;                   // descriptor version
  d |= (uint64_t)2u << 61;                   // 128-byte swizzle
  return d;
}

template <bool A_MN, bool B_MN>
constexpr uint32_t gemm_idesc() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((A_MN ? 1u : 0u) << 15) | ((B_MN ? 1u : 0u) << 16) |
         ((uint32_t)(GBN >> 3) << 17) | ((uint32_t)(GBM >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16_i(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                           uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void gemm_tile(const GemmParams& p, int t, int& mt, int& nt) {
  if (p.m_fast) {
    mt = t % p.n_mt;
    nt = t / p.n_mt;
  } else {
    nt = t % p.n_nt;
    mt = t / p.n_nt;
  }
}

template <bool A_MN, bool B_MN>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + GSTAGES * GSTAGE_BYTES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * GSTAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * GSTAGES + 5);
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * GSTAGES;
  const uint32_t accf0 = empty0 + 8 * GSTAGES, acce0 = accf0 + 16;
  const uint32_t drain_bar = smem_u32(bars + 2 * GSTAGES + 6);
  constexpr uint32_t idesc = gemm_idesc<A_MN, B_MN>();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < GSTAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf0 + 8 * a, 1);
      mbar_init(acce0 + 8 * a, 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0u, issued_parity = 0u;
      bool ok = true;
      for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x) {
        int mt, nt;
        gemm_tile(p, t, mt, nt);
        for (int k = 0; k < p.k_steps; ++k) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag, p.wait_limit)) { ok = false; break; }
          if (*abort_flag) { ok = false; break; }
          const uint32_t fb = full0 + 8 * stage;
          mbar_expect_tx(fb, GSTAGE_BYTES);
          const uint32_t sa = base + stage * GSTAGE_BYTES, sb = sa + GA_BYTES;
          if (A_MN) {
#pragma unroll
            for (int j = 0; j < GBM / 64; ++j) tma_load_2d(sa + j * GMN_BLOCK, &tmap_a, fb, mt * GBM + j * 64, k * GBK);
          } else {
            tma_load_2d(sa, &tmap_a, fb, k * GBK, mt * GBM);
          }
          if (B_MN) {
#pragma unroll
            for (int j = 0; j < GBN / 64; ++j) tma_load_2d(sb + j * GMN_BLOCK, &tmap_b, fb, nt * GBN + j * 64, k * GBK);
          } else {
            tma_load_2d(sb, &tmap_b, fb, k * GBK, nt * GBN);
          }
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == GSTAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok || *abort_flag) {   // let every issued copy land before the CTA exits
        for (int s2 = 0; s2 < GSTAGES; ++s2) {
          if (!(issued_mask & (1u << s2))) continue;
          const uint32_t par = (issued_parity >> s2) & 1u;
          for (uint32_t i = 0; i < SPIN_LIMIT; ++i)
            if (mbar_try_wait(full0 + 8 * s2, par)) break;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, tile = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x, ++tile) {
        const uint32_t acc = tile & 1u, accph = (tile >> 1) & 1u;
        if (!mbar_wait(acce0 + 8 * acc, accph ^ 1u, abort_flag, p.wait_limit)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * GBN;
        for (int k = 0; k < p.k_steps; ++k) {
          if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, p.wait_limit)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = base + stage * GSTAGE_BYTES, sb = sa + GA_BYTES;
#pragma unroll
          for (int kk = 0; kk < GBK / 16; ++kk) {
            // 16 K-elements: 32 bytes inside a K-contiguous row, 16 rows of an MN-contiguous block
            const uint64_t da = A_MN ? smem_desc_mn_sw128(sa + kk * 2048, GMN_BLOCK)
                                     : smem_desc_sw128(sa) + (uint64_t)(kk * 2);
            const uint64_t db = B_MN ? smem_desc_mn_sw128(sb + kk * 2048, GMN_BLOCK)
                                     : smem_desc_sw128(sb) + (uint64_t)(kk * 2);
            mma_bf16_i(d_tmem, da, db, idesc, (k > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(empty0 + 8 * stage);
          if (++stage == GSTAGES) { stage = 0; phase ^= 1u; }
        }
        if (ok) mma_commit(accf0 + 8 * acc);
      }
      if (!ok) {
        mma_commit(drain_bar);
        for (uint32_t i = 0; i < SPIN_LIMIT; ++i)
          if (mbar_try_wait(drain_bar, 0u)) break;
      }
    }
  } else {
    // ------------------------------------------------------ epilogue
    const int q = warp & 3;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t tile = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x, ++tile) {
      int mt, nt;
      gemm_tile(p, t, mt, nt);
      const uint32_t acc = tile & 1u, accph = (tile >> 1) & 1u;
      if (!mbar_wait(accf0 + 8 * acc, accph, abort_flag, p.wait_limit)) { ok = false; break; }
      tc_fence_after();
      const int64_t row = (int64_t)mt * GBM + q * 32 + lane;
      float* drow = p.D + row * p.ldd;
#pragma unroll 1
      for (int ch = 0; ch < GBN / 32; ++ch) {
        float v[32];
        tmem_ld32(tmem + lane_base + acc * GBN + ch * 32, v);
        const int64_t col0 = (int64_t)nt * GBN + ch * 32;
        if (row >= p.M || col0 >= p.N) continue;
        const int n = (int)(p.N - col0 < 32 ? p.N - col0 : 32);
        if (n == 32 && ((reinterpret_cast<uintptr_t>(drow + col0) & 15u) == 0)) {
          float4* d4 = reinterpret_cast<float4*>(drow + col0);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float4 o = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
            if (p.beta != 0.f) {
              const float4 old = d4[k];
              o.x = __fmaf_rn(p.beta, old.x, o.x);
              o.y = __fmaf_rn(p.beta, old.y, o.y);
              o.z = __fmaf_rn(p.beta, old.z, o.z);
              o.w = __fmaf_rn(p.beta, old.w, o.w);
            }
            d4[k] = o;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < n) drow[col0 + j] = p.beta != 0.f ? __fmaf_rn(p.beta, drow[col0 + j], v[j]) : v[j];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce0 + 8 * acc);
    }
    if (!ok && lane == 0) *abort_flag = 1;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load();
  if (f) return f;
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  f = reinterpret_cast<EncodeTiledFn>(ptr);
  fn.store(f);
  return f;
}

bool make_map(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {BK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return f(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 2-D bf16 map over rows x cols (row stride ld elements) with a box of
// box_inner columns by box_outer rows.
bool make_map_box(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint64_t ld,
                  uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return f(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// D = A B + beta D with the GEMM above.  A_MN / B_MN as there; a and b are
// the stored arrays (a: [K][M] when A_MN else [M][K]; b: [K][N] when B_MN else
// [N][K]), with row strides lda, ldb (elements, multiples of 8).
template <bool A_MN, bool B_MN>
cudaError_t gemm(const void* a, int64_t lda, const void* b, int64_t ldb, int64_t M, int64_t N,
                 int64_t K, float* D, int64_t ldd, float beta, bool m_fast, cudaStream_t stream) {
  static std::atomic<int> done[64];
  const int ds = device_slot();
  if (ds < 0 || !done[ds].load()) {
    const cudaError_t e = cudaFuncSetAttribute(gemm_kernel<A_MN, B_MN>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)GSMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (ds >= 0) done[ds].store(1);
  }
  CUtensorMap ma, mb;
  const bool oka = A_MN ? make_map_box(&ma, a, (uint64_t)K, (uint64_t)M, (uint64_t)lda, 64, GBK)
                        : make_map_box(&ma, a, (uint64_t)M, (uint64_t)K, (uint64_t)lda, GBK, GBM);
  const bool okb = B_MN ? make_map_box(&mb, b, (uint64_t)K, (uint64_t)N, (uint64_t)ldb, 64, GBK)
                        : make_map_box(&mb, b, (uint64_t)N, (uint64_t)K, (uint64_t)ldb, GBK, GBN);
  if (!oka || !okb) return cudaErrorInvalidValue;
  GemmParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.n_mt = (int)((M + GBM - 1) / GBM);
  p.n_nt = (int)((N + GBN - 1) / GBN);
  p.n_tiles = p.n_mt * p.n_nt;
  p.k_steps = (int)((K + GBK - 1) / GBK);
  p.m_fast = m_fast ? 1 : 0;
  p.D = D;
  p.ldd = ldd;
  p.beta = beta;
  p.wait_limit = debug_wait_limit();
  const int grid = p.n_tiles < sm_count() ? p.n_tiles : sm_count();
  gemm_kernel<A_MN, B_MN><<<grid, THREADS, GSMEM_BYTES, stream>>>(ma, mb, p);
  return cudaGetLastError();
}

}  // namespace

size_t lmhead_workspace_bytes(int64_t T, int64_t V, int64_t H) {
  (void)V;
  (void)H;
  const size_t b = (size_t)NSLICE * (size_t)T * sizeof(float4) + (size_t)T * sizeof(float);
  return (b + 255) & ~(size_t)255;
}

// The kernel's shared-memory attribute, once per device.
cudaError_t set_lmhead_smem() {
  static std::atomic<int> done[64];
  const int ds = device_slot();
  if (ds >= 0 && done[ds].load()) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(lmhead_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)SMEM_BYTES);
  if (e == cudaSuccess && ds >= 0) done[ds].store(1);
  return e;
}

cudaError_t launch_lmhead_impl(const LmheadArgs& a, float* debug_logits, cudaStream_t stream) {
  CUtensorMap ma, mb;
  if (!make_map(&ma, a.hidden, (uint64_t)a.T, (uint64_t)a.H, BM)) return cudaErrorInvalidValue;
  if (!make_map(&mb, a.w_vocab, (uint64_t)a.V, (uint64_t)a.H, BN)) return cudaErrorInvalidValue;
  if (cudaError_t e = set_lmhead_smem(); e != cudaSuccess) return e;
  LmParams p{};
  p.T = a.T;
  p.V = a.V;
  p.n_mt = (int)((a.T + BM - 1) / BM);
  p.n_nt = (int)((a.V + BN - 1) / BN);
  p.n_units = p.n_mt * NSLICE;
  p.k_steps = (int)(a.H / BK);
  p.ids = a.ids;
  p.c = (float)(1.4426950408889634 / (double)a.temperature);
  p.part = static_cast<float4*>(a.workspace);
  p.zy = reinterpret_cast<float*>(static_cast<char*>(a.workspace) +
                                  (size_t)NSLICE * (size_t)a.T * sizeof(float4));
  p.debug_logits = debug_logits;
  p.status = a.status;
  p.grad = 0;
  p.wait_limit = debug_wait_limit();
  p.withhold = debug_take_withheld();
  const int grid = p.n_units < sm_count() ? p.n_units : sm_count();
  lmhead_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(ma, mb, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  lmhead_combine_kernel<<<(unsigned)((a.T + 255) / 256), 256, 0, stream>>>(
      p, a.out_logprob, a.out_entropy, a.out_lse, a.temperature);
  return cudaGetLastError();
}

// ------------------------------------------------------------ backward
// dL/dhidden = dZ W and dL/dW = dZ^T hidden, with dZ = dL/dz recomputed by
// the GEMM above (gradient epilogue) one chunk of rows at a time, so the
// gradient logits exist for at most kBwdRows rows (the chunked-loss layout of
// prime-rl v0.10.0 notes, "1. Trainer Performance").  The two weight-side
// products are the tcgen05 GEMM above with MN-contiguous operands: bf16
// inputs, fp32 accumulation and output, each tile's K and the chunks in a
// fixed order.
namespace {

constexpr int64_t kBwdRows = 4096;

int64_t dz_ld(int64_t V) { return (V + 7) / 8 * 8; }   // 16-byte rows

size_t dz_bytes(int64_t T, int64_t V) {
  const int64_t rows = T < kBwdRows ? T : kBwdRows;
  return ((size_t)rows * (size_t)dz_ld(V) * 2 + 255) & ~(size_t)255;
}

}  // namespace

size_t lmhead_bwd_workspace_bytes(int64_t T, int64_t V, int64_t H) {
  (void)H;
  return dz_bytes(T, V);
}

cudaError_t launch_lmhead_backward(const LmheadBwdArgs& a, cudaStream_t stream) {
  if (cudaError_t e = set_lmhead_smem(); e != cudaSuccess) return e;
  CUtensorMap mb;
  if (!make_map(&mb, a.w_vocab, (uint64_t)a.V, (uint64_t)a.H, BN)) return cudaErrorInvalidValue;
  uint16_t* dz = static_cast<uint16_t*>(a.workspace);
  const int64_t ldz = dz_ld(a.V);
  const uint16_t* hid = static_cast<const uint16_t*>(a.hidden);
  for (int64_t r0 = 0; r0 < a.T; r0 += kBwdRows) {
    const int64_t rows = a.T - r0 < kBwdRows ? a.T - r0 : kBwdRows;
    CUtensorMap ma;
    if (!make_map(&ma, hid + r0 * a.H, (uint64_t)rows, (uint64_t)a.H, BM))
      return cudaErrorInvalidValue;
    LmParams p{};
    p.T = rows;
    p.V = a.V;
    p.n_mt = (int)((rows + BM - 1) / BM);
    p.n_nt = (int)((a.V + BN - 1) / BN);
    p.n_units = p.n_mt * NSLICE;
    p.k_steps = (int)(a.H / BK);
    p.ids = a.ids + r0;
    p.c = (float)(1.4426950408889634 / (double)a.temperature);
    p.inv_t = (float)(1.0 / (double)a.temperature);
    p.grad = 1;   // no status word: a timed-out tile leaves NaN gradients
    p.wait_limit = debug_wait_limit();
    p.withhold = -1;
    p.lse = a.lse + r0;
    p.ent = a.entropy + r0;
    p.glp = a.grad_logprob ? a.grad_logprob + r0 : nullptr;
    p.gh = a.grad_entropy ? a.grad_entropy + r0 : nullptr;
    p.dz = dz;
    p.ldz = ldz;
    const int grid = p.n_units < sm_count() ? p.n_units : sm_count();
    lmhead_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(ma, mb, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // dH[r0 : r0 + rows] = dZ W: A = dZ [rows][V] (K contiguous), B = W [V][H]
    // (N contiguous); consecutive tiles walk the rows, so the CTAs at work read
    // the same columns of W
    e = gemm<false, true>(dz, ldz, a.w_vocab, a.H, rows, a.H, a.V, a.grad_hidden + r0 * a.H, a.H,
                          0.0f, true, stream);
    if (e != cudaSuccess) return e;
    // dW (+)= dZ^T hidden: A = dZ^T (M = V contiguous in dZ), B = hidden [rows][H]
    // (N contiguous); consecutive tiles walk H, so the chunk's hidden stays in L2
    const float beta = (r0 > 0 || a.accumulate_w) ? 1.0f : 0.0f;
    e = gemm<true, true>(dz, ldz, hid + r0 * a.H, a.H, a.V, a.H, rows, a.grad_w, a.H, beta, false,
                         stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

size_t lmhead_topp_workspace_bytes(int64_t T, int64_t V, int64_t H) {
  (void)H;
  return dz_bytes(T, V);
}

// top_p < 1: the nucleus needs every logit of a row, so each chunk of at most
// kBwdRows rows is emitted once as bf16 logits (the same GEMM, emit epilogue)
// into the workspace and scored there by the top-p logits path.
cudaError_t launch_lmhead_topp(const LmheadArgs& a, cudaStream_t stream) {
  if (cudaError_t e = set_lmhead_smem(); e != cudaSuccess) return e;
  CUtensorMap mb;
  if (!make_map(&mb, a.w_vocab, (uint64_t)a.V, (uint64_t)a.H, BN)) return cudaErrorInvalidValue;
  uint16_t* zbuf = static_cast<uint16_t*>(a.workspace);
  const int64_t ldz = dz_ld(a.V);
  const uint16_t* hid = static_cast<const uint16_t*>(a.hidden);
  for (int64_t r0 = 0; r0 < a.T; r0 += kBwdRows) {
    const int64_t rows = a.T - r0 < kBwdRows ? a.T - r0 : kBwdRows;
    CUtensorMap ma;
    if (!make_map(&ma, hid + r0 * a.H, (uint64_t)rows, (uint64_t)a.H, BM))
      return cudaErrorInvalidValue;
    LmParams p{};
    p.T = rows;
    p.V = a.V;
    p.n_mt = (int)((rows + BM - 1) / BM);
    p.n_nt = (int)((a.V + BN - 1) / BN);
    p.n_units = p.n_mt * NSLICE;
    p.k_steps = (int)(a.H / BK);
    p.ids = a.ids + r0;
    p.c = (float)(1.4426950408889634 / (double)a.temperature);
    p.grad = 2;
    p.status = a.status;
    p.wait_limit = debug_wait_limit();
    p.withhold = -1;
    p.dz = zbuf;
    p.ldz = ldz;
    const int grid = p.n_units < sm_count() ? p.n_units : sm_count();
    lmhead_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(ma, mb, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    LpeArgs l{};
    l.logits = zbuf;
    l.dtype = 0;
    l.T = rows;
    l.V = a.V;
    l.ld = ldz;
    l.ids = a.ids + r0;
    l.temperature = a.temperature;
    l.top_p = a.top_p;
    l.out_logprob = a.out_logprob + r0;
    l.out_entropy = a.out_entropy + r0;
    l.status = a.status;
    e = launch_logprob_entropy(l, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_lmhead(const LmheadArgs& a, cudaStream_t stream) {
  return launch_lmhead_impl(a, nullptr, stream);
}

}  // namespace rlk
