// Cluster-resident rlk_logprob_entropy kernel for bf16 rows of a large
// vocabulary (the Qwen3-8B shape: V = 151,936).
//
// What is computed is the same as the per-row kernel: the temperature-scaled,
// top-p-truncated, renormalised log-probability of the selected token and the
// Shannon entropy of the retained distribution, following RL-Kernel
// "Qwen3-8B VIME train-rollout consistency", section "ROCm MI300X and gfx942"
// (sparse logp / monitoring-entropy fusion over the complete retained top-p
// support, the full-vocabulary scorer at top_p = 1) and the RL-Kernel "ROCm
// sparse performance" notes (the sampler's temperature / top-p semantics,
// fixed reduction order).
//
// Layout: a cluster of CL = 4 CTAs owns one row at a time; CTA q holds the
// columns [q CW, (q+1) CW) of the row in its own shared memory (CW = ceil(V/4)
// rounded up to 8 columns: 75,968 bytes at V = 151,936), filled by
// one-dimensional TMA bulk copies in four sub-chunks that complete on
// mbarriers.  Each sub-chunk is refilled with the next row as soon as the last
// warp is done with it, so the next row streams in while this one is being
// finished.  Two clusters' CTAs share each SM.  The row is read from HBM once.
//
// Arithmetic, in base-2 units with c = log2(e) / T: against a reference
// exponent E (an fp32 number near m c, m a max), each token contributes
// w = 2^d, d = fma(z, c, -E) (one rounding; the rounding of E itself shifts
// every d alike and cancels in the log-probability ln2 fma(z_y, c, -E) - ln S
// and in the entropy ln S - ln2 (sum w d) / S).  S is summed per thread in
// packed fp32 pairs and folded into a double-float every sub-chunk.
//
//  * top_p = 1: each warp takes its own max as reference, sums S and sum w d
//    over its groups and pushes (E, S, sum w d) into the shared memory of the
//    CTA that finishes the row (a rotating one); that CTA's warp 0 merges the
//    48 warp partials along a fixed tree (rescaling to the larger reference).
//  * top_p < 1: every warp first pushes its (max, min) to every CTA, one
//    cluster barrier later all warps know the row max m (E = m c, common to
//    all sums).  The retained set lies in the window z >= m - L T,
//    L = ln(1/(1-top_p)) + 7: a group whose max (kept in registers from the
//    first pass) reaches it is queued per warp, and its tokens are counted per
//    distinct bf16 value with remote atomic adds into the finishing CTA's
//    histogram (all tokens of one value carry the same mass, so integer counts
//    summarise the window exactly and in any order).  The finishing warp
//    scans the bins largest value first in a fixed-order double-float prefix
//    sum: the bin where the retained mass reaches top_p S, how many of its tied
//    tokens are needed (lower ids first), Z_S and the entropy numerator.
//  * Rows this path does not finish -- a window wider than the histogram
//    (e.g. one that crosses zero), or a window whose mass falls short of the
//    target -- get a marker in out_logprob and are recomputed by the per-row
//    kernel launched right after.  The choice depends only on the row's own
//    values; every sum runs in a fixed order; so a row's output bits never
//    depend on the batch around it.
//
// The finishing warp does its merge / scan one step late, inside the slack of
// the next cluster barrier, so it does not hold up the other warps.

#include <cuda_bf16.h>
#include <math.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "rlk.h"

namespace rlk {
namespace {

constexpr int CL = 4;             // CTAs per cluster (one row)
constexpr int NTC = 384;          // compute threads per CTA
constexpr int NWC = NTC / 32;     // compute warps; warp NWC finishes rows
constexpr int NTB = NTC + 32;     // threads per CTA
constexpr int JMAX = 14;          // 8-column groups per thread: CW <= JMAX * NTC * 8
constexpr int JS = 4;             // group rounds per bulk-copy sub-chunk
constexpr int NSUB = (JMAX + JS - 1) / JS;
constexpr int HBC = 2048;         // largest window (bins) this path takes
constexpr int NSLOT = 3;          // warp-partial slots (the top_p = 1 finish lags by a row)

struct __align__(16) CSmem {
  unsigned long long full[NSUB];   // sub-chunk landed (TMA complete_tx)
  unsigned long long cmax_bar;     // every warp has posted its max (top_p < 1)
  uint32_t released[NSUB];         // warps done with a sub-chunk (the last one refills it)
  float4 wpart[NSLOT][CL][NWC];    // every warp's sums, pushed to the row's finishing CTA
  uint4 wcta[NSLOT][CL];           // every CTA's (max key, min key), pushed likewise
  uint2 wmax[2][NWC];              // this CTA's warps' (max key, min key)
  unsigned long long wpeer[2][CL][NWC];   // every warp's (row, max key), pushed to all CTAs
  uint32_t hist[NSLOT][HBC / 2];   // this CTA's window counts, two 16-bit bins a word
  uint32_t merged[HBC];            // the finishing warp's counts for the whole row
  uint16_t queue[NWC][JS * 32];    // per-warp candidate groups of one sub-chunk
  int abort;
};

struct Geom {
  int64_t CW;   // columns per CTA (multiple of 8)
};

// ------------------------------------------------------------ cluster PTX
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_cluster_u64(uint32_t addr, unsigned long long v) {
  asm volatile("st.relaxed.cluster.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(uint32_t addr) {
  unsigned long long v;
  asm volatile("ld.relaxed.cluster.shared::cta.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ float value_of_key(uint32_t k) { return bf16_val(okey16_inverse(k)); }

// ----------------------------------------------------------------- helpers
// Fixed-order warp sum of (double-float, float); lane 0 gets the total.
__device__ __forceinline__ void warp_sum_df(DF& x, float& v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const DF y{shfl_down(x.hi, o), shfl_down(x.lo, o)};
    const float w = shfl_down(v, o);
    x = df_add(x, y);
    v = __fadd_rn(v, w);
  }
}

// A partial sum against the reference exponent e: S = sum 2^d as a
// double-float (hi, lo) and U = sum 2^d d, d = z c - e.
struct P2 {
  float e, hi, lo, u;
};
__device__ __forceinline__ bool p2_empty(const P2& a) {
  return a.e == -INFINITY && a.hi == 0.f && a.lo == 0.f && a.u == 0.f;
}
// Merge two partials (a is the left operand; the tree fixes which is which),
// rescaling to the larger reference.
__device__ __forceinline__ P2 p2_merge(const P2& a, const P2& b) {
  if (p2_empty(b)) return a;
  if (p2_empty(a)) return b;
  const float E = fmaxf(a.e, b.e);
  const float da = __fsub_rn(E, a.e), db = __fsub_rn(E, b.e);
  const float fa = (a.e == E) ? 1.f : ex2(-da);
  const float fb = (b.e == E) ? 1.f : ex2(-db);
  const float sa = __fadd_rn(a.hi, a.lo), sb = __fadd_rn(b.hi, b.lo);
  P2 r;
  r.e = E;
  r.u = __fadd_rn(__fmul_rn(fa, __fmaf_rn(-da, sa, a.u)), __fmul_rn(fb, __fmaf_rn(-db, sb, b.u)));
  float s, e;
  two_sum(__fmul_rn(a.hi, fa), __fmul_rn(b.hi, fb), s, e);
  e = __fadd_rn(e, __fadd_rn(__fmul_rn(a.lo, fa), __fmul_rn(b.lo, fb)));
  r.hi = __fadd_rn(s, e);
  r.lo = __fsub_rn(e, __fsub_rn(r.hi, s));
  return r;
}

struct ScanOut {
  uint32_t kstar;
  float lz, h;
  bool y_in;
  uint32_t key_thr, ties;   // the boundary key and its tied tokens kept (kTiesAll: all)
};

// One warp scans the window's bins 0..dmax (distance below the max key) in a
// fixed order, largest value first: the first bin whose inclusive prefix mass
// reaches the target, how many of its tied tokens are needed (lower ids
// first), Z_S and the entropy numerator.  Lane l owns the contiguous bins
// [l b, (l+1) b).  Returns false (on every lane) when the window's mass falls
// short; else the results are valid on every lane.
__device__ bool warp_scan_window(int lane, uint32_t dmax, uint32_t key_m, float c, float E,
                                 DF target, const uint32_t* hist, uint32_t key_y, uint32_t tie_y,
                                 ScanOut& out) {
  const uint32_t bpl = (dmax + 32u) / 32u;   // ceil((dmax + 1) / 32)
  const uint32_t d0 = (uint32_t)lane * bpl;
  auto bin = [&](uint32_t d, uint32_t& nb, float& mass, float& um, float& wv, float& dv) {
    nb = 0u; mass = 0.f; um = 0.f; wv = 0.f; dv = 0.f;
    if (d > dmax) return;
    nb = hist[d];
    if (nb == 0u) return;
    dv = __fmaf_rn(value_of_key(key_m - d), c, -E);
    wv = ex2(dv);
    mass = __fmul_rn((float)nb, wv);
    um = __fmul_rn(mass, dv);
  };
  DF tot{0.f, 0.f};
  uint32_t tcnt = 0u;
  float tum = 0.f;
  for (uint32_t j = 0; j < bpl; ++j) {
    uint32_t nb; float ms, um, wv, dv;
    bin(d0 + j, nb, ms, um, wv, dv);
    tot = df_add_f(tot, ms);
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
  DF P{shfl_up(inc.hi, 1), shfl_up(inc.lo, 1)};
  uint32_t pc = __shfl_up_sync(0xFFFFFFFFu, icnt, 1);
  float pu = shfl_up(ium, 1);
  if (lane == 0) { P = DF{0.f, 0.f}; pc = 0u; pu = 0.f; }
  int my_d = -1;
  DF pb{0.f, 0.f};
  uint32_t cb = 0u, nt = 0u;
  float ub = 0.f, wt = 0.f, dt = 0.f;
  for (uint32_t j = 0; j < bpl; ++j) {
    uint32_t nb; float ms, um, wv, dv;
    bin(d0 + j, nb, ms, um, wv, dv);
    const DF Pn = df_add_f(P, ms);
    if (nb > 0u && df_ge(Pn, target)) {
      my_d = (int)(d0 + j);
      pb = P; cb = pc; ub = pu; wt = wv; dt = dv; nt = nb;
      break;
    }
    P = Pn;
    pc += nb;
    pu = __fadd_rn(pu, um);
  }
  const uint32_t bal = __ballot_sync(0xFFFFFFFFu, my_d >= 0);
  if (bal == 0u) return false;
  const int win = __ffs(bal) - 1;   // the lowest lane holds the lowest crossing bin
  uint32_t kstar = 0u, ties = 0u;
  int y_in = 0;
  float lz = 0.f, h = 0.f;
  if (lane == win) {
    const float need = df_sub_to_f(target, pb);
    const float cf = ceilf(__fdiv_rn(need, wt));
    const uint32_t cneed = cf < 1.f ? 1u : (cf > (float)nt ? nt : (uint32_t)cf);
    const float wn = __fmul_rn((float)cneed, wt);
    const DF zs = df_add_f(pb, wn);
    const float us = __fmaf_rn(wn, dt, ub);
    const uint32_t d_y = key_m - key_y;
    kstar = cb + cneed;
    ties = cneed == nt ? kTiesAll : cneed;
    y_in = (d_y < (uint32_t)my_d) || (d_y == (uint32_t)my_d && tie_y < cneed);
    const float zsf = __fadd_rn(zs.hi, zs.lo);
    lz = logf(zsf);
    h = __fsub_rn(lz, __fdiv_rn(__fmul_rn(kLn2, us), zsf));
  }
  out.kstar = __shfl_sync(0xFFFFFFFFu, kstar, win);
  out.ties = __shfl_sync(0xFFFFFFFFu, ties, win);
  out.key_thr = key_m - (uint32_t)__shfl_sync(0xFFFFFFFFu, my_d, win);
  out.y_in = __shfl_sync(0xFFFFFFFFu, y_in, win) != 0;
  out.lz = __shfl_sync(0xFFFFFFFFu, lz, win);
  out.h = __shfl_sync(0xFFFFFFFFu, h, win);
  return true;
}

__device__ __forceinline__ void write_bad(const LpeArgs& a, int64_t r, uint32_t bit) {
  a.out_logprob[r] = NAN;
  a.out_entropy[r] = NAN;
  if (a.out_k) a.out_k[r] = 0;
  if (a.status) atomicOr(a.status, bit);
  if (a.state) a.state[r] = RowState{0.f, 0.f, 0.f, 0u, 0u, bit << 8, 0, 0u};
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// --------------------------------------------------------------- kernel
template <bool TOPP>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(NTB, 2)
    lpe_cluster_kernel(LpeArgs a, Geom geo, float c) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  CSmem& sm = *reinterpret_cast<CSmem*>(smem_raw);
  uint8_t* buf = smem_raw + ((sizeof(CSmem) + 127) & ~size_t(127));
  const uint4* bufv = reinterpret_cast<const uint4*>(buf);
  const uint32_t buf_s = smem_u32(buf);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t q = cluster_rank();
  const int64_t ncl = cluster_count();
  const int64_t r0 = cluster_id();

  const int64_t col0 = (int64_t)q * geo.CW;
  const int64_t nq = a.V - col0 < geo.CW ? a.V - col0 : geo.CW;  // >= 8 NTC (checked on the host)
  const int gfull = (int)(nq >> 3);                // full 8-column groups, resident in smem
  const int tail = (int)(nq & 7);                  // columns of the last, partial group
  const int nsub = (gfull + JS * NTC - 1) / (JS * NTC);
  const bool tail_owner = tail != 0 && tid == (gfull % NTC);
  const uint16_t* logits = reinterpret_cast<const uint16_t*>(a.logits);

  auto issue_sub = [&](int64_t r, int s) {   // one thread: sub-chunk s of row r
    const int g0 = s * JS * NTC;
    const int g1 = min(gfull, g0 + JS * NTC);
    const uint32_t bytes = (uint32_t)(g1 - g0) * 16u;
    const uint32_t bar = smem_u32(&sm.full[s]);
    mbar_expect_tx(bar, bytes);
    bulk_copy_g2s(buf_s + (uint32_t)g0 * 16u, logits + r * a.ld + col0 + (int64_t)g0 * 8, bytes, bar);
  };

  if (tid == 0) {
    for (int s = 0; s < NSUB; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1u);
      sm.released[s] = 0u;
    }
    mbar_init(smem_u32(&sm.cmax_bar), (uint32_t)NWC);
    sm.abort = 0;
    fence_mbar_init();
  }
  // Shared memory keeps whatever an earlier launch left: the row-tagged warp
  // maxima start with a tag no row has (the first cluster barrier orders this
  // before any peer's push).
  for (int i = tid; i < 2 * CL * NWC; i += blockDim.x) (&sm.wpeer[0][0][0])[i] = ~0ull;
  __syncthreads();
  if (tid == 0 && r0 < a.T)
    for (int s = 0; s < nsub; ++s) issue_sub(r0, s);
  cluster_arrive();   // barrier initialisation visible before any peer pushes here
  cluster_wait();

  // ---- the finishing warp's work for a row, one row late
  struct Fin {
    int64_t r;
    bool bad_id;
    float zy;
    uint32_t key_y, slot;
  };
  auto finish_p1 = [&](const Fin& f) {
    const float4* wp = &sm.wpart[f.slot][0][0];
    const float4 p0 = wp[lane];
    P2 M{p0.x, p0.y, p0.z, p0.w};
    if (lane + 32 < CL * NWC) {
      const float4 p1 = wp[lane + 32];
      M = p2_merge(M, P2{p1.x, p1.y, p1.z, p1.w});
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const P2 x{shfl_down(M.e, o), shfl_down(M.hi, o), shfl_down(M.lo, o), shfl_down(M.u, o)};
      M = p2_merge(M, x);
    }
    if (lane == 0) {
      const float zf = __fadd_rn(M.hi, M.lo);
      if (f.bad_id) {
        write_bad(a, f.r, RLK_STATUS_BAD_TOKEN_ID);
      } else if (!(isfinite(zf) && isfinite(M.u) && isfinite(M.e))) {
        write_bad(a, f.r, RLK_STATUS_NONFINITE);
      } else {
        const float lz = logf(zf);
        const float h = __fsub_rn(lz, __fdiv_rn(__fmul_rn(kLn2, M.u), zf));
        a.out_logprob[f.r] = __fsub_rn(__fmul_rn(kLn2, __fmaf_rn(f.zy, c, -M.e)), lz);
        a.out_entropy[f.r] = h;
        if (a.out_k) a.out_k[f.r] = (int32_t)a.V;
        if (a.state)
          a.state[f.r] = RowState{M.e, lz, h, 0u, kTiesAll, kStateValid | kStateYIn,
                                  (int32_t)a.V, 0u};
      }
    }
  };
  const float L_spec = TOPP ? logf(__fdiv_rn(1.f, __fsub_rn(1.f, a.top_p))) + 7.0f : 0.f;
  auto finish_topp = [&](const Fin& f) {
    // The row's max and min from the four CTAs.
    const uint4 ci = sm.wcta[f.slot][lane & (CL - 1)];
    const uint32_t key_m = __reduce_max_sync(0xFFFFFFFFu, ci.x);
    const uint32_t gmin = __reduce_min_sync(0xFFFFFFFFu, ci.y);
    const float m = value_of_key(key_m);
    const float E = __fmul_rn(m, c);
    // Total mass at the reference E = m c (the largest of the CTAs' references).
    const float4* wp = &sm.wpart[f.slot][0][0];
    const float4 p0 = wp[lane];
    P2 M{p0.x, p0.y, p0.z, 0.f};
    float ties = p0.w;
    if (lane + 32 < CL * NWC) {
      const float4 p1 = wp[lane + 32];
      M = p2_merge(M, P2{p1.x, p1.y, p1.z, 0.f});
      ties = __fadd_rn(ties, p1.w);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const P2 x{shfl_down(M.e, o), shfl_down(M.hi, o), shfl_down(M.lo, o), shfl_down(M.u, o)};
      M = p2_merge(M, x);
      ties = __fadd_rn(ties, shfl_down(ties, o));
    }
    const DF Z{__shfl_sync(0xFFFFFFFFu, M.hi, 0), __shfl_sync(0xFFFFFFFFu, M.lo, 0)};
    const float ME = __shfl_sync(0xFFFFFFFFu, M.e, 0);
    const uint32_t tie_y = (uint32_t)__shfl_sync(0xFFFFFFFFu, ties, 0);
    const float zf = __fadd_rn(Z.hi, Z.lo);
    const bool nonfinite = !isfinite(m) || isinf(__uint_as_float(okey32_inverse(gmin))) ||
                           !isfinite(zf) || ME != E;
    // The window z >= m - L T as keys [key_lo, key_m] (key_lo one key below zlo
    // truncated to bf16); every CTA counted at least these keys.
    const float zlo = __fsub_rn(m, __fmul_rn(L_spec, a.temperature));
    const uint32_t kl = okey16(__float_as_uint(zlo) >> 16);
    const uint32_t key_lo = kl > 0u ? kl - 1u : 0u;
    const uint32_t dmax = key_m - key_lo;
    const bool hist_ok = !f.bad_id && !nonfinite && key_lo <= key_m && dmax < (uint32_t)HBC;
    ScanOut so{0u, 0.f, 0.f, false};
    bool found = false;
    if (hist_ok) {
      // Gather the four CTAs' counts for the row's bins into this CTA's memory.
      uint32_t kmq[CL], base[CL];
#pragma unroll
      for (int k = 0; k < CL; ++k) {
        kmq[k] = __shfl_sync(0xFFFFFFFFu, ci.x, k);
        base[k] = map_rank(smem_u32(&sm.hist[f.slot][0]), (uint32_t)k);
      }
      for (uint32_t d = (uint32_t)lane; d <= dmax; d += 32u) {
        const uint32_t key = key_m - d;
        uint32_t n = 0u;
#pragma unroll
        for (int k = 0; k < CL; ++k) {
          if (key <= kmq[k]) {
            const uint32_t idx = kmq[k] - key;
            n += (ld_cluster_u32(base[k] + 4u * (idx >> 1)) >> (16u * (idx & 1u))) & 0xFFFFu;
          }
        }
        sm.merged[d] = n;
      }
      __syncwarp();
      found = warp_scan_window(lane, dmax, key_m, c, E, df_mul_f(Z, a.top_p), sm.merged, f.key_y,
                               tie_y, so);
    }
    if (lane == 0) {
      if (f.bad_id) {
        write_bad(a, f.r, RLK_STATUS_BAD_TOKEN_ID);
      } else if (nonfinite) {
        write_bad(a, f.r, RLK_STATUS_NONFINITE);
      } else if (!found) {
        a.out_logprob[f.r] = __uint_as_float(kRecomputeMark);   // the per-row kernel redoes it
      } else {
        a.out_logprob[f.r] = so.y_in ? __fsub_rn(__fmul_rn(kLn2, __fmaf_rn(f.zy, c, -E)), so.lz)
                                     : -INFINITY;
        a.out_entropy[f.r] = so.h;
        if (a.out_k) a.out_k[f.r] = (int32_t)so.kstar;
        if (a.state)
          a.state[f.r] = RowState{E, so.lz, so.h, so.key_thr, so.ties,
                                  kStateValid | (so.y_in ? kStateYIn : 0u), (int32_t)so.kstar, 0u};
      }
    }
  };

  if (warp == NWC) {
    // ---- the finishing warp: one cluster-barrier phase per row, always ahead
    // of the compute warps (which publish a row at the next row's arrive).
    int itf = 0;
    for (int64_t r = r0; r < a.T; r += ncl, ++itf) {
      cluster_arrive();
      cluster_wait();
      if ((uint32_t)(itf % CL) == q) {
        Fin f;
        f.r = r;
        const int64_t y = a.ids[r];
        f.bad_id = y < 0 || y >= a.V;
        f.zy = f.bad_id ? 0.f : bf16_val(__ldg(logits + r * a.ld + y));
        f.key_y = okey16(__float_as_uint(f.zy) >> 16);
        f.slot = (uint32_t)(itf % NSLOT);
        if (TOPP) finish_topp(f);
        else finish_p1(f);
      }
    }
    cluster_arrive();   // no CTA leaves while another may still touch its memory
    cluster_wait();
    return;
  }

  bool pending = false;   // a cluster-barrier phase arrived on but not yet waited for
  const float2 c2 = make_float2(c, c);
  const uint32_t lt_mask = (1u << lane) - 1u;
  int it = 0;
  for (int64_t r = r0; r < a.T; r += ncl, ++it) {
    const uint32_t ph = (uint32_t)it & 1u;
    const uint32_t slot = (uint32_t)(it % NSLOT);
    const bool has_next = r + ncl < a.T;
    const int64_t y = a.ids[r];
    const bool bad_id = y < 0 || y >= a.V;
    const float zy = bad_id ? 0.f : bf16_val(__ldg(logits + r * a.ld + y));
    const uint32_t frank = (uint32_t)(it % CL);   // the CTA that finishes this row
    float tv[8];                                   // the partial last group, from global
#pragma unroll
    for (int k = 0; k < 8; ++k)
      tv[k] = (tail_owner && k < tail) ? bf16_val(__ldg(logits + r * a.ld + col0 + (int64_t)gfull * 8 + k))
                                       : -INFINITY;

    // ---- A0: the warp's max (and min), each group's max (top_p < 1)
    __nv_bfloat162 mx2 = bf2(0xFF80FF80u), mn2 = bf2(0x7F807F80u);   // (-inf, -inf), (+inf, +inf)
    uint32_t sk[(JMAX + 1) / 2];
#pragma unroll
    for (int j = 0; j < (JMAX + 1) / 2; ++j) sk[j] = 0u;
    auto a0_group = [&](const uint4 v, const int j) {
      if (TOPP) {
        const __nv_bfloat162 gm = __hmax2(__hmax2(bf2(v.x), bf2(v.y)), __hmax2(bf2(v.z), bf2(v.w)));
        mx2 = __hmax2(mx2, gm);
        mn2 = __hmin2(mn2, __hmin2(__hmin2(bf2(v.x), bf2(v.y)), __hmin2(bf2(v.z), bf2(v.w))));
        const uint32_t gw = *reinterpret_cast<const uint32_t*>(&gm);
        sk[j >> 1] |= (__float_as_uint(fmaxf(bf16_lo(gw), bf16_hi(gw))) >> 16) << (16 * (j & 1));
      } else {
        mx2 = __hmax2(__hmax2(mx2, bf2(v.x)), __hmax2(bf2(v.y), __hmax2(bf2(v.z), bf2(v.w))));
      }
    };
#pragma unroll
    for (int s = 0; s < NSUB; ++s) {
      if (s < nsub) {
        if (!mbar_wait_sleep(smem_u32(&sm.full[s]), ph, &sm.abort) && a.status)
          atomicOr(a.status, RLK_STATUS_TIMEOUT);
        const int J1 = (s * JS + JS < JMAX) ? s * JS + JS : JMAX;
        if (J1 * NTC <= gfull) {   // every thread's groups of this sub-chunk are whole
          uint4 v[JS];
#pragma unroll
          for (int jj = 0; jj < JS; ++jj)
            if (s * JS + jj < JMAX) v[jj] = bufv[tid + (s * JS + jj) * NTC];
#pragma unroll
          for (int jj = 0; jj < JS; ++jj)
            if (s * JS + jj < JMAX) a0_group(v[jj], s * JS + jj);
        } else {
#pragma unroll
          for (int jj = 0; jj < JS; ++jj)
            if (s * JS + jj < JMAX && tid + (s * JS + jj) * NTC < gfull)
              a0_group(bufv[tid + (s * JS + jj) * NTC], s * JS + jj);
        }
      }
    }
    float mt = fmaxf(__low2float(mx2), __high2float(mx2));
    float nt = fminf(__low2float(mn2), __high2float(mn2));
    if (tail_owner) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k < tail) {
          mt = fmaxf(mt, tv[k]);
          nt = fminf(nt, tv[k]);
        }
    }
    const uint32_t kx = __reduce_max_sync(0xFFFFFFFFu, okey32(__float_as_uint(mt)));

    // Publish the previous row's pushes (they have landed by now, so the
    // release is cheap); the finishing warp then finishes that row.
    if (it > 0) {
      if (pending) cluster_wait();
      cluster_arrive();
      pending = true;
    }

    // ---- the reference exponent; top_p < 1: this CTA's max and its window
    float E;
    uint32_t key_mq = 0u, key_lo = 0u;
    bool win_empty = false;
    float zlo_k = 0.f;
    if (TOPP) {
      const uint32_t kn = __reduce_min_sync(0xFFFFFFFFu, okey32(__float_as_uint(nt)));
      // Offer this warp's max to every CTA: a larger max than this CTA's own
      // raises its window floor (any value between the CTA max and the row
      // max gives a window that holds the row's; the finishing warp reads only
      // the row window's bins, so what arrives in time does not change them).
      if (lane < CL)
        st_cluster_u64(map_rank(smem_u32(&sm.wpeer[ph][q][warp]), (uint32_t)lane),
                       ((unsigned long long)(uint32_t)r << 32) | kx);
      // This row's counts go to buffer `slot`, last read two rows ago (every
      // CTA has passed the barrier that follows that read): clear it.
      for (int i = tid; i < HBC / 2; i += NTC) sm.hist[slot][i] = 0u;
      __syncwarp();   // the lanes' clearing is ordered before lane 0's release
      if (lane == 0) {
        sm.wmax[ph][warp] = make_uint2(kx, kn);
        mbar_arrive(smem_u32(&sm.cmax_bar));
      }
      if (!mbar_wait_sleep(smem_u32(&sm.cmax_bar), ph, &sm.abort) && a.status)
        atomicOr(a.status, RLK_STATUS_TIMEOUT);
      uint32_t km = lane < NWC ? sm.wmax[ph][lane].x : 0u;
      uint32_t kmn = lane < NWC ? sm.wmax[ph][lane].y : 0xFFFFFFFFu;
      km = __reduce_max_sync(0xFFFFFFFFu, km);
      kmn = __reduce_min_sync(0xFFFFFFFFu, kmn);
      const float mq = __uint_as_float(okey32_inverse(km));
      E = __fmul_rn(mq, c);
      // The largest warp max of this row that has reached this CTA so far.
      uint32_t kpeer = km;
      {
        const uint32_t wp = smem_u32(&sm.wpeer[ph][0][0]);
        const unsigned long long a0 = ld_relaxed_u64(wp + 8u * lane);
        if ((uint32_t)(a0 >> 32) == (uint32_t)r) kpeer = max(kpeer, (uint32_t)a0);
        if (lane + 32 < CL * NWC) {
          const unsigned long long a1 = ld_relaxed_u64(wp + 8u * (lane + 32));
          if ((uint32_t)(a1 >> 32) == (uint32_t)r) kpeer = max(kpeer, (uint32_t)a1);
        }
        kpeer = __reduce_max_sync(0xFFFFFFFFu, kpeer);
      }
      const float mfloor = __uint_as_float(okey32_inverse(kpeer));
      if (warp == 0 && lane == 0)
        st_cluster_v4(map_rank(smem_u32(&sm.wcta[slot][q]), frank),
                      make_float4(__uint_as_float(okey16(__float_as_uint(mq) >> 16)),
                                  __uint_as_float(kmn), 0.f, 0.f));
      // Window of this CTA: z >= mq - L T, at most HBC keys below its max (the
      // row's window, which is what the finishing warp reads, lies inside).
      const float zlo = __fsub_rn(mfloor, __fmul_rn(L_spec, a.temperature));
      key_mq = okey16(__float_as_uint(mq) >> 16);
      const uint32_t kl = okey16(__float_as_uint(zlo) >> 16);
      key_lo = kl > 0u ? kl - 1u : 0u;
      if (key_lo > key_mq) {
        win_empty = true;   // every token of this CTA lies below the row's window
        zlo_k = INFINITY;
      } else {
        if (key_mq - key_lo >= (uint32_t)HBC)
          key_lo = key_mq > (uint32_t)(HBC - 1) ? key_mq - (uint32_t)(HBC - 1) : 0u;
        zlo_k = value_of_key(key_lo);
      }
    } else {
      E = __fmul_rn(__uint_as_float(okey32_inverse(kx)), c);
    }
    const uint32_t key_y = okey16(__float_as_uint(zy) >> 16);
    const uint32_t dmq = win_empty ? 0u : key_mq - key_lo;   // window: idx = key_mq - key <= dmq
    const int32_t ycol = (int32_t)(y - col0);         // y's column within this CTA's chunk

    // ---- A1: S = sum 2^d (and U = sum 2^d d), d = fma(z, c, -E); window counts
    const float2 nE2 = make_float2(-E, -E);
    DF acc{0.f, 0.f};
    float2 u2 = make_float2(0.f, 0.f);
    uint32_t tie = 0u;
    uint32_t* hist = sm.hist[slot];
#pragma unroll
    for (int s = 0; s < NSUB; ++s) {
      if (s < nsub) {
        float2 sacc = make_float2(0.f, 0.f);
        uint32_t qn = 0u;   // warp-uniform queue fill
        auto a1_group = [&](const uint4 v) {
          const float2 d0 = __ffma2_rn(bf16x2_to_f2(v.x), c2, nE2);
          const float2 d1 = __ffma2_rn(bf16x2_to_f2(v.y), c2, nE2);
          const float2 d2 = __ffma2_rn(bf16x2_to_f2(v.z), c2, nE2);
          const float2 d3 = __ffma2_rn(bf16x2_to_f2(v.w), c2, nE2);
          const float2 w0 = make_float2(ex2(d0.x), ex2(d0.y));
          const float2 w1 = make_float2(ex2(d1.x), ex2(d1.y));
          const float2 w2 = make_float2(ex2(d2.x), ex2(d2.y));
          const float2 w3 = make_float2(ex2(d3.x), ex2(d3.y));
          sacc = __fadd2_rn(sacc, __fadd2_rn(__fadd2_rn(w0, w1), __fadd2_rn(w2, w3)));
          if (!TOPP) {
            u2 = __ffma2_rn(w0, d0, u2);
            u2 = __ffma2_rn(w1, d1, u2);
            u2 = __ffma2_rn(w2, d2, u2);
            u2 = __ffma2_rn(w3, d3, u2);
          }
        };
        auto enqueue = [&](const int j, const bool valid) {   // top_p < 1: candidate groups
          const int g = tid + j * NTC;
          const bool cand = valid && bf16_val((sk[j >> 1] >> (16 * (j & 1))) & 0xFFFFu) >= zlo_k;
          const uint32_t bal = __ballot_sync(0xFFFFFFFFu, cand);
          if (cand) sm.queue[warp][qn + __popc(bal & lt_mask)] = (uint16_t)g;
          qn += __popc(bal);
        };
        const int J1 = (s * JS + JS < JMAX) ? s * JS + JS : JMAX;
        if (J1 * NTC <= gfull) {   // every thread's groups of this sub-chunk are whole
          uint4 v[JS];
#pragma unroll
          for (int jj = 0; jj < JS; ++jj)
            if (s * JS + jj < JMAX) v[jj] = bufv[tid + (s * JS + jj) * NTC];
#pragma unroll
          for (int jj = 0; jj < JS; ++jj)
            if (s * JS + jj < JMAX) a1_group(v[jj]);
          if (TOPP) {
#pragma unroll
            for (int jj = 0; jj < JS; ++jj)
              if (s * JS + jj < JMAX) enqueue(s * JS + jj, true);
          }
        } else {
#pragma unroll
          for (int jj = 0; jj < JS; ++jj) {
            if (s * JS + jj < JMAX) {
              const bool valid = tid + (s * JS + jj) * NTC < gfull;
              if (valid) a1_group(bufv[tid + (s * JS + jj) * NTC]);
              if (TOPP) enqueue(s * JS + jj, valid);
            }
          }
        }
        float t, e;
        two_sum(acc.hi, __fadd_rn(sacc.x, sacc.y), t, e);
        acc.hi = t;
        acc.lo = __fadd_rn(acc.lo, e);
        if (TOPP && qn != 0u) {
          // Count the queued groups' window tokens: one lane per group, an
          // 8-bit mask of its tokens >= zlo_k from packed bf16 compares, one
          // atomic per set bit.
          __syncwarp();
          const __nv_bfloat162 z2 = __float2bfloat162_rn(zlo_k);   // zlo_k is a bf16 value
          for (uint32_t e0 = 0; e0 < qn; e0 += 32) {
            const uint32_t e = e0 + (uint32_t)lane;
            const bool act = e < qn;
            const int g = act ? (int)sm.queue[warp][e] : 0;
            const uint4 v = act ? bufv[g] : make_uint4(0u, 0u, 0u, 0u);
            uint32_t msk = 0u;
            if (act)
              msk = (__hge2_mask(bf2(v.x), z2) & 0x00010001u) |
                    ((__hge2_mask(bf2(v.y), z2) & 0x00010001u) << 1) |
                    ((__hge2_mask(bf2(v.z), z2) & 0x00010001u) << 2) |
                    ((__hge2_mask(bf2(v.w), z2) & 0x00010001u) << 3);
            while (msk != 0u) {
              const int b = __ffs(msk) - 1;   // bit b: word b & 3, high half if b >= 16
              msk &= msk - 1u;
              const int wi = b & 3, hi = b >> 4;
              const uint32_t wd = wi == 0 ? v.x : (wi == 1 ? v.y : (wi == 2 ? v.z : v.w));
              const uint32_t kk = okey16(hi ? (wd >> 16) : wd);
              const uint32_t idx = key_mq - kk;
              if (idx <= dmq) {
                atomicAdd(&hist[idx >> 1], 1u << ((idx & 1u) << 4));
                if (kk == key_y && g * 8 + 2 * wi + hi < ycol) ++tie;
              }
            }
          }
        }
        // The last warp done with the sub-chunk refills it with the next row.
        // Every value this warp read from it has been consumed by now.
        __syncwarp();
        if (lane == 0 && has_next && (atomicAdd(&sm.released[s], 1u) + 1u) % NWC == 0u) {
          fence_proxy_async_smem();
          issue_sub(r + ncl, s);
        }
      }
    }
    if (tail_owner) {
      float gs = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (k < tail) {
          const float d = __fmaf_rn(tv[k], c, -E);
          const float w = ex2(d);
          gs = __fadd_rn(gs, w);
          if (!TOPP) u2.x = __fmaf_rn(w, d, u2.x);
          if (TOPP) {
            const uint32_t kk = okey16(__float_as_uint(tv[k]) >> 16);
            const uint32_t idx = key_mq - kk;
            if (!win_empty && idx <= dmq) {
              atomicAdd(&hist[idx >> 1], 1u << ((idx & 1u) << 4));
              if (kk == key_y && gfull * 8 + k < ycol) ++tie;
            }
          }
        }
      }
      float t, e;
      two_sum(acc.hi, gs, t, e);
      acc.hi = t;
      acc.lo = __fadd_rn(acc.lo, e);
    }
    // Warp sums (the tie count rides along as an exact float), pushed to the
    // finishing CTA; published by the next row's cluster arrive.
    float wv = TOPP ? (float)tie : __fadd_rn(u2.x, u2.y);
    warp_sum_df(acc, wv);
    if (lane == 0)
      st_cluster_v4(map_rank(smem_u32(&sm.wpart[slot][q][warp]), frank),
                    make_float4(E, acc.hi, acc.lo, wv));
  }
  // Publish the last row; no CTA leaves while another may still read or
  // write its shared memory.
  if (it > 0) {
    if (pending) cluster_wait();
    cluster_arrive();
    cluster_wait();
  }
  cluster_arrive();
  cluster_wait();
}

}  // namespace

bool lpe_cluster_eligible(const LpeArgs& a) {
  if (a.dtype != 0 || a.T >= 0xFFFFFFFFll) return false;   // rows are tagged with 32 bits
  if ((reinterpret_cast<uintptr_t>(a.logits) & 15u) != 0 || (a.ld & 7) != 0) return false;
  const int64_t cw = (((a.V + CL - 1) / CL) + 7) & ~int64_t(7);
  if (a.V - (CL - 1) * cw < 8 * NTC) return false;    // every CTA gets a sizeable chunk
  return cw / 8 + 1 <= (int64_t)JMAX * NTC;          // chunk (and partial group) fit
}

cudaError_t launch_lpe_cluster(const LpeArgs& a, cudaStream_t stream) {
  // c = log2(e) / T rounded once.
  const float c = (float)(1.4426950408889634 / (double)a.temperature);
  Geom geo;
  geo.CW = (((a.V + CL - 1) / CL) + 7) & ~int64_t(7);
  const size_t smem = ((sizeof(CSmem) + 127) & ~size_t(127)) + (size_t)geo.CW * 2;
  const bool topp = a.top_p < 1.0f;

  // Max active clusters for this shared-memory size, per device and variant
  // (packed as size << 32 | clusters).
  static std::atomic<unsigned long long> cached[64][2];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int di = dev & 63, vi = topp ? 1 : 0;
  const unsigned long long cv = cached[di][vi].load();
  int ncl = (int)(cv & 0xFFFFFFFFull);
  if ((cv >> 32) != smem || ncl < 1) {
    const void* fn = topp ? (const void*)lpe_cluster_kernel<true> : (const void*)lpe_cluster_kernel<false>;
    const int smax = (int)(((sizeof(CSmem) + 127) & ~size_t(127)) + (size_t)JMAX * NTC * 16);
    if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smax)) != cudaSuccess)
      return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL);
    cfg.blockDim = dim3(NTB);
    cfg.dynamicSmemBytes = smem;
    if ((e = cudaOccupancyMaxActiveClusters(&ncl, fn, &cfg)) != cudaSuccess) return e;
    if (ncl < 1) return cudaErrorLaunchOutOfResources;
    cached[di][vi].store(((unsigned long long)smem << 32) | (unsigned)ncl);
  }
  const int64_t nclusters = a.T < (int64_t)ncl ? a.T : (int64_t)ncl;
  const dim3 grid((unsigned)(nclusters * CL)), block(NTB);
  if (topp) lpe_cluster_kernel<true><<<grid, block, smem, stream>>>(a, geo, c);
  else lpe_cluster_kernel<false><<<grid, block, smem, stream>>>(a, geo, c);
  return cudaGetLastError();
}

}  // namespace rlk
