// Streaming rlk_logprob_entropy kernel for bf16 rows of a large vocabulary
// (every bf16 batch with 14,336 <= V <= 174,080, whatever its row stride or
// alignment, and whichever entry point -- scalar or per-row parameters -- so a
// row gets one set of bits from every call that scores it).
//
// What is computed: the temperature-scaled, top-p-truncated, renormalised
// log-probability of the selected token and the Shannon entropy of the
// retained distribution, following RL-Kernel "Qwen3-8B VIME train-rollout
// consistency", section "ROCm MI300X and gfx942" (sparse logp /
// monitoring-entropy fusion over the complete retained top-p support, the
// full-vocabulary scorer at top_p = 1) and the RL-Kernel "ROCm sparse
// performance" notes (the sampler's temperature / top-p semantics, a fixed
// reduction order so recomputed log-probabilities are bitwise reproducible).
//
// One CTA of 1024 threads per SM; CTA b scores rows b, b + grid, ...  Warp
// roles, pipelined over rows:
//  * the producer (warp 28): one thread streams each row through a ring of
//    four shared-memory stages with cp.async.bulk (one unit of 16 logits = 32
//    bytes per compute thread per stage), and forms each row's parameters
//    (c = log2(e) / T exactly as the host forms it);
//  * the compute warps (0-27): thread t owns the units t, t + 896, ... of a
//    row and keeps one running state: an integer reference E_t,
//    S = sum 2^d as a double-float and U = sum 2^d d with d = fma(z, c, -E_t)
//    (one rounding).  A unit's max comes first (packed bf16x2 max); the
//    reference moves up (by an exact power of two) only when a unit's max
//    exceeds it by more than LAZY, so the exponentials run against a fixed
//    reference almost always.  At top_p < 1 each unit's largest and second
//    largest logits also go to a sketch.  At the end of a row each warp
//    merges its 32 thread states in a fixed order, writes the warp state to
//    shared memory and starts the next row at once;
//  * the merge warp (29), one row behind: merges the 28 warp states in a
//    fixed order (rescaling to E = ceil(m c), m the row max: exact powers of
//    two) and decides the row: at top_p = 1 its answer; at top_p < 1 the
//    window z >= m - L T (L = ln(1/(1-top_p)) + 7) in which the retained set
//    must lie.  All tokens of one bf16 value carry the same mass, so the
//    window is summarised exactly by integer counts per distinct value;
//  * side work of the compute warps, at the end of the next row: the threads
//    test the sketch of the finished row against the window.  A unit whose
//    largest logit reaches the window and whose second largest does not holds
//    one window token, its max, counted from the sketch alone.  A unit with
//    more has its two largest counted from the sketch and is listed.  Tokens
//    are counted per key with shared-memory atomics (integer counts do not
//    depend on the atomics' order);
//  * the scan warps (30 and 31, alternate rows): the counts are now exact for
//    every token but the third and later largest of listed units.  A first
//    scan over them, largest value first, bounds the crossing from below; the
//    listed units whose second largest logit reaches that bound, and the
//    selected token's unit, are read once more and their remaining tokens
//    above it counted, which makes every count above the bound exact.  The
//    final scan (a fixed-order double-float prefix) finds the bin where the
//    retained mass reaches top_p Z, how many of its tied tokens are needed
//    (lower ids first), Z_S and the entropy numerator; the warp writes the
//    row's outputs.
//  * Rows this path does not finish -- a window wider than the histogram (one
//    that crosses zero) or a window whose mass falls short of the target --
//    get a marker in out_logprob and are recomputed by the per-row kernel
//    launched right after.  The choice depends only on the row's own values;
//    every sum runs in a fixed order; so a row's output bits never depend on
//    the batch around it, nor on the layout of the batch (aligned rows stream
//    through the ring, other rows are read with scalar loads into the same
//    units, with the same arithmetic).
//
// Every wait is bounded: a wait that runs out raises RLK_STATUS_TIMEOUT and an
// abort flag; every role then stops waiting, the rows not yet finished get
// NaN outputs, the producer lets the copies it issued land, and the kernel
// returns.

#include <cuda_bf16.h>
#include <math.h>

#include <atomic>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "rlk.h"

namespace rlk {
namespace {

constexpr int NWC = 28;                  // compute warps
constexpr int NTC = NWC * 32;            // compute threads
constexpr int WPROD = NWC;               // producer warp
constexpr int WMRG = NWC + 1;            // merge warp
constexpr int WSCN = NWC + 2;            // scan warps (two: even and odd rows of the CTA)
constexpr int NTB = (NWC + 4) * 32;
static_assert(NTB == 1024, "one 1024-thread CTA per SM");
constexpr int UNIT = 16;                 // logits per unit (32 bytes)
constexpr int NSTAGE = 4;                // ring stages
constexpr int STAGE_BYTES = NTC * 32;    // one unit per compute thread
constexpr int HBC = 2048;                // window bins (keys below the row max)
constexpr int NRP = 16;                  // row-parameter slots
constexpr float LAZY = 4.0f;             // re-base when a unit's max exceeds E_t by this (base 2)
constexpr int64_t V_MIN = (int64_t)UNIT * NTC;
constexpr int64_t V_MAX = 174080;        // the sketch's share of shared memory (10,880 units)
static_assert((V_MAX / UNIT + NTC - 1) / NTC <= 32, "a thread's units of a row fit a 32-bit mask");
constexpr uint32_t PART_BYTES = 2u * 4u * 32u * 4u;   // [2][4][32] warp states
constexpr int NSTM = (int)((V_MAX / UNIT + NTC - 1) / NTC);   // a thread's units of a row, at most
constexpr uint32_t LCAP = 1500;          // units with two or more window tokens listed per row

struct RowParam {
  float c, temp, top_p, row_t;   // row_t: the row's own temperature (per-row calls), else 0
  uint32_t bad;                  // the row's parameters are invalid (RLK_STATUS_BAD_PARAM)
  uint32_t pad[3];
};

// What the merge warp decides for a row.
enum : uint32_t { REC_DONE = 0, REC_COUNT = 1, REC_MARK = 2, REC_BAD = 3 };
constexpr uint32_t MGCAP = 24;    // entries of a row's shared near-zero bin kept (see ck_of)
struct RowRec {
  uint32_t mode, bad_bit;
  uint32_t zf2;          // window floor, a bf16 value in both halves
  uint32_t key_m, dmax, key_y;
  uint32_t cz;           // the window crosses zero: bins by compressed key (ck_of)
  uint32_t ckm, key_lo;  // the max's compressed key (bins are ckm - ck); the floor's key
  int32_t y;
  float E, c, U, zy, top_p, row_t;
  float zhi, zlo;        // Z as a double-float
  float lp, ent, lz;     // REC_DONE: the outputs and ln Z
  int32_t kstar;
};

struct __align__(16) Ctrl {
  unsigned long long full[NSTAGE];
  unsigned long long empty[NSTAGE];
  unsigned long long rowpub[2];     // compute warps -> merge warp: a row's states written
  unsigned long long floorpub[2];   // merge warp -> compute warps, scan warp: the row's record
  unsigned long long counted[2];    // compute warps -> scan warp: the row's window counted
  unsigned long long hclear[2];     // scan warp -> merge warp: the row's counts consumed
  uint32_t mgn[2];                  // the shared near-zero bin's entries (may exceed MGCAP)
  uint32_t mgv[2][MGCAP];           // bf16 value | 1 << 16 for a token taken out again
  RowParam rp[NRP];
  RowRec rec[2];
  uint32_t wkey[2][NWC];
  uint32_t tie[2];
  uint32_t lcnt[2];                 // units listed for the scan warp (may exceed LCAP)
  int abort;
};

struct Geom {
  int nunits;     // ceil(V / 16)
  int nfull;      // V / 16: units whose 16 logits all exist
  int nst;        // stages per row: ceil(nunits / NTC)
  int tma;        // rows stream through the ring (16-byte aligned rows)
  uint32_t tma_bytes;   // bytes of a row the ring copies: floor(V / 8) * 16
  uint32_t off_part, off_hist, off_list, off_sk, skb, off_ring;
  long long wait_limit;   // clock cycles a wait may take before it gives up
  long long withhold;     // debug: the stage CTA 0 never issues (-1: none)
};

__host__ __device__ constexpr uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------------ helpers

// 2^n for an integer-valued n <= 0 (-inf gives 0), exactly.
__device__ __forceinline__ float exp2_int(float n) {
  return n >= -126.f ? __int_as_float(((int)n + 127) << 23) : 0.f;
}

// Waits for the mbarrier phase of the given parity, suspending in hardware.
// Gives up after `limit` clock cycles (raising the abort flag and the status
// bit) or at once when the abort flag is up.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort,
                                           long long limit, uint32_t* status) {
  const long long t0 = clock64();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(100000u)
        : "memory");
    if (ok) return true;
    if (*abort) return false;
    if (clock64() - t0 > limit) {
      *abort = 1;
      if (status) atomicOr(status, RLK_STATUS_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ float value_of_key(uint32_t k) { return bf16_val(okey16_inverse(k)); }
__device__ __forceinline__ uint32_t key_of(float v) { return okey16(__float_as_uint(v) >> 16); }

// Windows that cross zero.  The bf16 keys between -2^-4 and 2^-4 (bits
// 0xBD7F .. 0x3D7F, the zeros included) are ~31,000 keys of which a window
// would need a bin each; such a row's bins are indexed by compressed keys
// instead: those keys share one bin, MG_LO, and the keys above them move down
// by MG_W.  The shared bin's tokens differ in value, so its mass and its
// entropy term are sums over the tokens, kept in fixed point (w 2^40 and
// -w d 2^36, truncated: exact and independent of the order of the atomics);
// a crossing inside it cannot be placed by counts and hands the row on.
constexpr uint32_t MG_LO = 0x4280u, MG_HI = 0xBD7Fu, MG_W = MG_HI - MG_LO;
constexpr float kFixW = 1099511627776.0f;   // 2^40
constexpr float kFixU = 68719476736.0f;     // 2^36
// The code that counts and scans a row comes in two instantiations: CZ for
// rows whose window crosses zero, and the plain one (keys as they are) for
// every other row, which thus runs no extra instruction.
template <bool CZ>
__device__ __forceinline__ uint32_t ck_of(uint32_t k) {
  if (!CZ) return k;
  return k > MG_HI ? k - MG_W : (k >= MG_LO ? MG_LO : k);
}
template <bool CZ>
__device__ __forceinline__ uint32_t raw_of(uint32_t ck) {
  return (CZ && ck > MG_LO) ? ck + MG_W : ck;
}
// An entry of the shared near-zero bin's list: a token (bf16 bits) counted,
// or (remove) taken out again.
__device__ __forceinline__ void mg_list(Ctrl& ctl, int sb, uint32_t bits, bool remove) {
  const uint32_t i = atomicAdd(&ctl.mgn[sb], 1u);
  if (i < MGCAP) ctl.mgv[sb][i] = bits | (remove ? 0x10000u : 0u);
}

// Counts one window token (bf16 bits) into the bins of buffer sb; a token of
// the shared near-zero bin also goes to that bin's list.
template <bool CZ>
__device__ __forceinline__ void count_token(uint32_t* hist, uint32_t ckm, uint32_t bits, Ctrl& ctl,
                                            int sb) {
  const uint32_t ck = ck_of<CZ>(okey16(bits));
  atomicAdd(&hist[ckm - ck], 1u);
  if (CZ && ck == MG_LO) mg_list(ctl, sb, bits, false);
}

// The shared bin's mass and entropy term, sum w and sum w d over its listed
// tokens (less those taken out again), summed by one warp in fixed point
// (w 2^40, -w d 2^36, truncated: exact in any order, modulo 2^64).
__device__ __forceinline__ void mg_sums(const Ctrl& ctl, int sb, int lane, float c, float E,
                                        float& mass, float& um) {
  const uint32_t n = ctl.mgn[sb] < MGCAP ? ctl.mgn[sb] : MGCAP;
  unsigned long long sw = 0ull, su = 0ull;
  for (uint32_t k = (uint32_t)lane; k < n; k += 32u) {
    const uint32_t e = ctl.mgv[sb][k];
    const float d = __fmaf_rn(bf16_val(e & 0xFFFFu), c, -E);   // <= 0: E >= m c >= v c
    const float w = ex2(d);
    const unsigned long long fw = __float2ull_rz(__fmul_rn(w, kFixW));
    const unsigned long long fu = __float2ull_rz(__fmul_rn(__fmul_rn(w, -d), kFixU));
    sw += (e >> 16) ? 0ull - fw : fw;
    su += (e >> 16) ? 0ull - fu : fu;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sw += __shfl_xor_sync(0xFFFFFFFFu, sw, o);
    su += __shfl_xor_sync(0xFFFFFFFFu, su, o);
  }
  mass = (float)((double)sw * (1.0 / 1099511627776.0));
  um = -(float)((double)su * (1.0 / 68719476736.0));
}

// The running state of one compute thread for one row.
struct Acc {
  float E;      // reference (integer-valued, or -inf before the first unit)
  DF S;         // sum 2^d
  float2 U;     // sum 2^d d (two packed lanes)
  float mx;     // largest logit seen
  uint32_t mn;  // without U: smallest logit seen per bf16x2 lane (a -inf logit makes the row
                // non-finite, which U would otherwise show as NaN)
};

// Moves the reference up to En (> E): every sum scales by 2^(E - En), exactly.
// NOU: U is not kept (it stays 0).
template <bool NOU = false>
__device__ __forceinline__ void rebase(Acc& st, float En) {
  if (st.E == -INFINITY) {
    st.E = En;
    return;
  }
  const float n = __fsub_rn(st.E, En);   // integer, < 0
  const float f = exp2_int(n);
  if (!NOU) {
    st.U.x = __fmul_rn(f, __fmaf_rn(n, st.S.hi, st.U.x));
    st.U.y = __fmul_rn(f, st.U.y);
  }
  st.S.hi = __fmul_rn(st.S.hi, f);
  st.S.lo = __fmul_rn(st.S.lo, f);
  st.E = En;
}

__device__ __forceinline__ uint32_t u32(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t*>(&v); }

// Merges two (largest, second largest) pairs of bf16x2 lanes.
__device__ __forceinline__ void top2_merge(__nv_bfloat162& a1, __nv_bfloat162& b1, __nv_bfloat162 a2,
                                           __nv_bfloat162 b2) {
  b1 = __hmax2(__hmin2(a1, a2), __hmax2(b1, b2));
  a1 = __hmax2(a1, a2);
}

// Folds a unit's 16 logits into the state and returns the unit's max.  The
// words w[0..7] hold the logits in the order the thread reads them (two bf16
// a word, low half first).  MASKED: only the logits whose bit is set in vmask
// (bit j: half j & 1 of word j >> 1) exist -- the row's last, partial unit.
// TOP2: *ent receives the unit's sketch entry, its largest logit (low half)
// and its second largest (high half; -inf for a unit of one logit), as bf16.
// NOU: U is not kept -- a row at top_p < 1 takes its entropy from the
// retained set's counts, not from the whole row.
template <bool MASKED, bool UNIFORM = false, bool TOP2 = false, bool NOU = false>
__device__ __forceinline__ float absorb_unit(Acc& st, const uint32_t (&w)[8], float c,
                                             uint32_t vmask = 0xFFFFu, uint32_t* ent = nullptr) {
  uint32_t wm[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    wm[k] = w[k];
    if (MASKED) {   // absent logits read as -inf for the max
      if (!((vmask >> (2 * k)) & 1u)) wm[k] = (wm[k] & 0xFFFF0000u) | 0xFF80u;
      if (!((vmask >> (2 * k + 1)) & 1u)) wm[k] = (wm[k] & 0xFFFFu) | 0xFF800000u;
    }
  }
  float gm;
  if (TOP2) {
    // tournament: (max, second) per bf16x2 lane over the 8 words, then across the lanes
    __nv_bfloat162 A[4], B[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      A[k] = __hmax2(bf2(wm[2 * k]), bf2(wm[2 * k + 1]));
      B[k] = __hmin2(bf2(wm[2 * k]), bf2(wm[2 * k + 1]));
    }
    if (NOU) {
      if (MASKED) {   // absent logits read as +inf for the min
        uint32_t mn = 0x7F807F80u;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          uint32_t v = w[k];
          if (!((vmask >> (2 * k)) & 1u)) v = (v & 0xFFFF0000u) | 0x7F80u;
          if (!((vmask >> (2 * k + 1)) & 1u)) v = (v & 0xFFFFu) | 0x7F800000u;
          mn = u32(__hmin2(bf2(mn), bf2(v)));
        }
        st.mn = u32(__hmin2(bf2(st.mn), bf2(mn)));
      } else {
        st.mn = u32(__hmin2(bf2(st.mn), __hmin2(__hmin2(B[0], B[1]), __hmin2(B[2], B[3]))));
      }
    }
    top2_merge(A[0], B[0], A[1], B[1]);
    top2_merge(A[2], B[2], A[3], B[3]);
    top2_merge(A[0], B[0], A[2], B[2]);
    const __nv_bfloat162 As = bf2(__byte_perm(u32(A[0]), 0u, 0x1032));
    const __nv_bfloat162 Bs = bf2(__byte_perm(u32(B[0]), 0u, 0x1032));
    top2_merge(A[0], B[0], As, Bs);   // both lanes now hold the unit's pair
    *ent = __byte_perm(u32(A[0]), u32(B[0]), 0x5410);
    gm = bf16_lo(u32(A[0]));
  } else {
    const __nv_bfloat162 m01 = __hmax2(bf2(wm[0]), bf2(wm[1])), m23 = __hmax2(bf2(wm[2]), bf2(wm[3]));
    const __nv_bfloat162 m45 = __hmax2(bf2(wm[4]), bf2(wm[5])), m67 = __hmax2(bf2(wm[6]), bf2(wm[7]));
    const __nv_bfloat162 mm = __hmax2(__hmax2(m01, m23), __hmax2(m45, m67));
    const uint32_t mw = u32(mm);
    gm = fmaxf(bf16_lo(mw), bf16_hi(mw));
  }
  st.mx = fmaxf(st.mx, gm);
  // rare after a row's first units (E = -inf before the first: always taken)
  const bool up = __fmaf_rn(gm, c, -st.E) > LAZY;
  if (UNIFORM) {   // every lane is here: one warp-uniform test guards the rare re-base
    if (__any_sync(0xFFFFFFFFu, up)) {
      if (up) rebase<NOU>(st, ceilf(__fmul_rn(gm, c)));
    }
  } else if (up) {
    rebase<NOU>(st, ceilf(__fmul_rn(gm, c)));
  }
  const float2 c2 = make_float2(c, c);
  const float2 nE2 = make_float2(-st.E, -st.E);
  // Two halves of four words: sum ((e0+e1)+(e2+e3)) + ((e4+e5)+(e6+e7)) and
  // U += e_k d_k for k = 0..7 in order.
  float2 sh[2];
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    float2 d[4], e[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int k = 4 * hf + i;
      d[i] = __ffma2_rn(bf16x2_to_f2(w[k]), c2, nE2);
      e[i] = make_float2(ex2(d[i].x), ex2(d[i].y));
      if (MASKED) {
        if (!((vmask >> (2 * k)) & 1u)) { d[i].x = 0.f; e[i].x = 0.f; }
        if (!((vmask >> (2 * k + 1)) & 1u)) { d[i].y = 0.f; e[i].y = 0.f; }
      }
    }
    sh[hf] = __fadd2_rn(__fadd2_rn(e[0], e[1]), __fadd2_rn(e[2], e[3]));
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (!NOU) st.U = __ffma2_rn(e[i], d[i], st.U);
  }
  const float2 s = __fadd2_rn(sh[0], sh[1]);
  float t, r;
  two_sum(st.S.hi, __fadd_rn(s.x, s.y), t, r);
  st.S.hi = t;
  st.S.lo = __fadd_rn(st.S.lo, r);
  return gm;
}

// The 8 words of unit u of a row read with scalar loads (any alignment);
// absent logits (beyond V) read as -inf (the stream masks them besides).
__device__ __forceinline__ void load_unit_scalar(const uint16_t* row, int64_t V, int u, int h,
                                                 uint32_t (&w)[8]) {
  const int64_t c0 = (int64_t)u * UNIT;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int hh = half == 0 ? h : 1 - h;   // the half read first goes to words 0..3
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t i0 = c0 + hh * 8 + 2 * k;
      const uint32_t lo = i0 < V ? (uint32_t)__ldg(row + i0) : 0xFF80u;
      const uint32_t hi = i0 + 1 < V ? (uint32_t)__ldg(row + i0 + 1) : 0xFF80u;
      w[half * 4 + k] = lo | (hi << 16);
    }
  }
}

// ---------------------------------------------------------------- the scan
struct ScanOut {
  uint32_t kstar;
  float lz, h;
  bool y_in;
  uint32_t key_thr, ties;
};

// One warp scans the window's bins 0..dmax (distance below the max key) in a
// fixed order, largest value first: the first bin whose inclusive prefix mass
// reaches the target, how many of its tied tokens are needed (lower ids
// first), Z_S and the entropy numerator.  Lane l owns the contiguous bins
// [l b, (l+1) b).  Returns false (on every lane) when the window's mass falls
// short; else the results are valid on every lane.
template <bool CZ>
__device__ bool warp_scan_window(int lane, uint32_t dmax, uint32_t key_m, float c, float E,
                                 DF target, const uint32_t* hist, uint32_t key_y, uint32_t tie_y,
                                 ScanOut& out, bool& short_mass, float mg_mass = 0.f,
                                 float mg_um = 0.f) {
  // key_m: the max's key, compressed when cz (bin d holds compressed key key_m - d)
  const uint32_t bpl = (dmax + 32u) / 32u;
  const uint32_t d0 = (uint32_t)lane * bpl;
  // the shared near-zero bin (its mass and entropy term given, as fp32)
  const uint32_t d_mg = CZ ? key_m - MG_LO : 0xFFFFFFFFu;
  auto bin = [&](uint32_t d, uint32_t& nb, float& mass, float& um, float& wv, float& dv) {
    nb = 0u; mass = 0.f; um = 0.f; wv = 0.f; dv = 0.f;
    if (d > dmax) return;
    nb = hist[d];
    if (nb == 0u) return;
    if (CZ && d == d_mg) {
      mass = mg_mass;
      um = mg_um;
      return;
    }
    dv = __fmaf_rn(value_of_key(raw_of<CZ>(key_m - d)), c, -E);
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
  short_mass = bal == 0u;   // no bin reaches the target: the window holds too little
  if (bal == 0u) return false;
  const int win = __ffs(bal) - 1;   // the lowest lane holds the lowest crossing bin
  // a crossing inside the shared near-zero bin needs its tokens' order
  if (CZ && (uint32_t)__shfl_sync(0xFFFFFFFFu, my_d, win) == d_mg) return false;
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
    const uint32_t d_y = key_m - ck_of<CZ>(key_y);
    kstar = cb + cneed;
    ties = cneed == nt ? kTiesAll : cneed;
    y_in = (d_y < (uint32_t)my_d) || (d_y == (uint32_t)my_d && tie_y < cneed);
    const float zsf = __fadd_rn(zs.hi, zs.lo);
    lz = logf(zsf);
    h = __fsub_rn(lz, __fdiv_rn(__fmul_rn(kLn2, us), zsf));
  }
  out.kstar = __shfl_sync(0xFFFFFFFFu, kstar, win);
  out.ties = __shfl_sync(0xFFFFFFFFu, ties, win);
  out.key_thr = raw_of<CZ>(key_m - (uint32_t)__shfl_sync(0xFFFFFFFFu, my_d, win));
  out.y_in = __shfl_sync(0xFFFFFFFFu, y_in, win) != 0;
  out.lz = __shfl_sync(0xFFFFFFFFu, lz, win);
  out.h = __shfl_sync(0xFFFFFFFFu, h, win);
  return true;
}

__device__ __forceinline__ void write_bad(const LpeArgs& a, int64_t r, uint32_t bit) {
  a.out_logprob[r] = NAN;
  a.out_entropy[r] = NAN;
  if (a.out_k) a.out_k[r] = 0;
  if (a.status && bit) atomicOr(a.status, bit);
  if (a.state) a.state[r] = RowState{0.f, 0.f, 0.f, 0u, 0u, bit << 8, 0, 0u};
}

// wait_phase with a fast path: one suspending try first (the phase has
// usually completed or completes within the hardware's suspend window).
__device__ __forceinline__ bool wait_full(uint32_t bar, uint32_t parity, volatile int* abort,
                                          long long limit, uint32_t* status) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(100000u)
      : "memory");
  if (ok) return true;
  return wait_phase(bar, parity, abort, limit, status);
}

// wait_full for a whole warp, its lanes agreeing on the result.
__device__ __forceinline__ bool wait_full_warp(uint32_t bar, uint32_t parity, volatile int* abort,
                                               long long limit, uint32_t* status) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(100000u)
      : "memory");
  if (__all_sync(0xFFFFFFFFu, ok != 0u)) return true;
  return __all_sync(0xFFFFFFFFu, wait_phase(bar, parity, abort, limit, status));
}

// Counts the tokens of unit u of a row that reach the window floor (zf2w, a
// bf16 value in both halves) into hist (bins below key_m); ny receives how
// many carry key_y.  The unit is read again (whole with two 16-byte loads from
// a 16-byte aligned row, else with scalar loads; absent logits read as -inf).
template <bool CZ>
__device__ __forceinline__ void count_unit(const uint16_t* row, int64_t V, int u, bool aligned_full,
                                           uint32_t zf2w, uint32_t key_m, uint32_t key_y,
                                           uint32_t* hist, uint32_t& ny, Ctrl& ctl, int sb) {
  uint32_t w[8];
  if (aligned_full) {
    const uint4* q = reinterpret_cast<const uint4*>(row) + 2 * u;
    const uint4 v0 = __ldg(q), v1 = __ldg(q + 1);
    w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
    w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
  } else {
    load_unit_scalar(row, V, u, 0, w);
  }
  const __nv_bfloat162 zf2 = bf2(zf2w);
  ny = 0u;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t hm = __hge2_mask(bf2(w[k]), zf2);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      if ((hm >> (16 * hf)) & 1u) {
        const uint32_t bits = (w[k] >> (16 * hf)) & 0xFFFFu;
        count_token<CZ>(hist, key_m, bits, ctl, sb);
        ny += okey16(bits) == key_y ? 1u : 0u;
      }
    }
  }
}

// The scan warp's second look at a listed unit (two or more window tokens,
// whose two largest logits the sketch already counted): reads the unit again
// (whole with two 16-byte loads from a 16-byte aligned row, else with scalar
// loads; absent logits beyond V read as -inf) and adds its other tokens whose
// key reaches the one of kv (a bf16 value in both halves).  Returns how many
// were added; ny receives how many of them carry key_y.
template <bool CZ>
__device__ __forceinline__ uint32_t recount_unit(const uint16_t* row, int64_t V, int u, bool aligned_full,
                                                 uint32_t kv2w, uint32_t key_m, uint32_t key_y,
                                                 uint32_t* hist, uint32_t& ny, Ctrl& ctl, int sb) {
  uint32_t w[8];
  if (aligned_full) {
    const uint4* q = reinterpret_cast<const uint4*>(row) + 2 * u;
    const uint4 v0 = __ldg(q), v1 = __ldg(q + 1);
    w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
    w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
  } else {
    load_unit_scalar(row, V, u, 0, w);
  }
  const __nv_bfloat162 kv2 = bf2(kv2w);
  uint32_t n = 0u;
  ny = 0u;
  float m1 = -INFINITY, m2 = -INFINITY;   // the unit's two largest logits
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t hm = __hge2_mask(bf2(w[k]), kv2);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const uint32_t bits = (w[k] >> (16 * hf)) & 0xFFFFu;
      const float f = bf16_lo(bits);
      if (f > m1) {
        m2 = m1;
        m1 = f;
      } else {
        m2 = fmaxf(m2, f);
      }
      if ((hm >> (16 * hf)) & 1u) {
        count_token<CZ>(hist, key_m, bits, ctl, sb);
        ++n;
        ny += okey16(bits) == key_y ? 1u : 0u;
      }
    }
  }
  // the two largest were counted from the sketch
  const uint32_t k1 = key_of(m1), k2 = key_of(m2);
  const uint32_t c1 = ck_of<CZ>(k1), c2 = ck_of<CZ>(k2);
  atomicAdd(&hist[key_m - c1], 0xFFFFFFFFu);
  atomicAdd(&hist[key_m - c2], 0xFFFFFFFFu);
  if (CZ && c1 == MG_LO) mg_list(ctl, sb, __float_as_uint(m1) >> 16, true);
  if (CZ && c2 == MG_LO) mg_list(ctl, sb, __float_as_uint(m2) >> 16, true);
  ny -= (k1 == key_y ? 1u : 0u) + (k2 == key_y ? 1u : 0u);
  return n - 2u;
}

// --------------------------------------------------------------- kernel
template <bool TOPP, bool TMA>
__global__ void __launch_bounds__(NTB, 1) lpe_stream_kernel(LpeArgs a, Geom g, float c0) {
  pdl_trigger();   // the recompute pass may be scheduled (it waits for this grid)
  pdl_wait();      // the logits may come from the kernel before
  extern __shared__ __align__(128) uint8_t smem[];
  Ctrl& ctl = *reinterpret_cast<Ctrl*>(smem);
  float* part = reinterpret_cast<float*>(smem + g.off_part);         // [2][4][32]: E, S hi, S lo, U
  uint32_t* hist0 = reinterpret_cast<uint32_t*>(smem + g.off_hist);  // [2][HBC]
  uint8_t* skb = smem + g.off_sk;                                     // [2][skb]: u32 per unit
  uint8_t* ring = smem + g.off_ring;                                  // [NSTAGE][STAGE_BYTES]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint16_t* logits = reinterpret_cast<const uint16_t*>(a.logits);
  volatile int* abort = &ctl.abort;

  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(smem_u32(&ctl.full[s]), 1u);
      mbar_init(smem_u32(&ctl.empty[s]), (uint32_t)NTC);   // every compute lane releases
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctl.rowpub[b]), (uint32_t)NWC);
      mbar_init(smem_u32(&ctl.floorpub[b]), 1u);
      mbar_init(smem_u32(&ctl.counted[b]), (uint32_t)NWC);
      mbar_init(smem_u32(&ctl.hclear[b]), 1u);
      ctl.tie[b] = 0u;
      ctl.lcnt[b] = 0u;
      ctl.mgn[b] = 0u;
    }
    ctl.abort = 0;
    fence_mbar_init();
  }
  for (int i = tid; i < 2 * HBC; i += NTB) hist0[i] = 0u;
  __syncthreads();

  if (warp < NWC) {
    // ------------------------------------------------------ compute warps
    const int t = tid;
    const int h = (lane >> 2) & 1;   // the half of its unit a thread reads first (bank spread)
    uint32_t gs = 0;   // stages consumed (ring slot gs % NSTAGE, phase gs / NSTAGE)
    int it = 0;
    // Side work: the window count of the previous row, done by each warp at
    // the end of a row.  Each lane tests the sketch entries of its own units
    // of that row (only the thread that wrote an entry reads it: a warp may
    // already be a few stages into the next row, writing the other buffer's
    // entries of its own units).  A unit whose largest logit reaches the
    // window floor but whose second largest does not holds exactly one window
    // token, its max, counted from the sketch.  A unit with two or more window
    // tokens has its two largest counted the same way and is listed for the
    // scan warp, which reads again only the listed units whose second largest
    // logit reaches the crossing (units the list has no room for are read
    // again here and counted whole).  The selected token's unit is left to the
    // scan warp (its ties need positions).
    auto side_row = [&](int rs) {   // rs: the side row's place in this CTA's sequence
      const int sb = rs & 1;
      const uint32_t par = (uint32_t)((rs >> 1) & 1);
      bool ready = wait_phase(smem_u32(&ctl.floorpub[sb]), par, abort, g.wait_limit, a.status);
      ready = __shfl_sync(0xFFFFFFFFu, ready ? 1 : 0, 0) != 0;
      uint32_t tie = 0u;
      if (ready && ctl.rec[sb].mode == REC_COUNT && !*abort) {
        auto count_row = [&](auto czc) {
          constexpr bool CZ = decltype(czc)::value;
            const uint32_t zf2w = ctl.rec[sb].zf2;
            const __nv_bfloat162 zf2 = bf2(zf2w);
            const uint32_t key_m = ctl.rec[sb].ckm, key_y = ctl.rec[sb].key_y;   // key_m compressed
            const int uy = ctl.rec[sb].y >> 4;
            uint32_t* hist = hist0 + sb * HBC;
            const uint32_t* sk = reinterpret_cast<const uint32_t*>(skb + (size_t)sb * g.skb);
            uint32_t sm = 0u, cm = 0u;   // bit j: unit t + j NTC holds one / several window tokens
#pragma unroll
            for (int j = 0; j < NSTM; ++j) {
              const int u = t + j * NTC;
              if (u < g.nunits) {
                const uint32_t mk = __hge2_mask(bf2(sk[u]), zf2);
                if ((mk & 1u) && u != uy) {
                  if (mk >> 16) cm |= 1u << j;
                  else sm |= 1u << j;
                }
              }
            }
            // Candidates are handed out warp-densely, one per lane and round:
            // candidate k of the warp belongs to the lane whose inclusive count
            // first exceeds k, as that lane's (k - exclusive count)-th set bit.
            const int ns = __popc(sm), nc = __popc(cm);
            int is = ns, ic = nc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const int vs = __shfl_up_sync(0xFFFFFFFFu, is, o), vc = __shfl_up_sync(0xFFFFFFFFu, ic, o);
              if (lane >= o) { is += vs; ic += vc; }
            }
            const int tot_s = __shfl_sync(0xFFFFFFFFu, is, 31), tot_c = __shfl_sync(0xFFFFFFFFu, ic, 31);
            auto pick = [&](int k, int incl, int n, uint32_t mask) -> int {   // the unit, or -1
              int L = 0;
#pragma unroll
              for (int st = 16; st > 0; st >>= 1) {
                const int v = __shfl_sync(0xFFFFFFFFu, incl, L + st - 1);
                if (v <= k) L += st;
              }
              const int x = __shfl_sync(0xFFFFFFFFu, incl - n, L);
              const uint32_t mL = __shfl_sync(0xFFFFFFFFu, mask, L);
              if (L > 31) return -1;
              const int j = (int)__fns(mL, 0u, k - x + 1);
              return warp * 32 + L + j * NTC;
            };
            for (int k0 = 0; k0 < tot_s; k0 += 32) {
              const int k = k0 + lane;
              const int u = pick(k, is, ns, sm);
              if (k < tot_s) {
                const uint32_t kk = okey16(sk[u] & 0xFFFFu);
                count_token<CZ>(hist, key_m, sk[u] & 0xFFFFu, ctl, sb);
                tie += (kk == key_y && u < uy) ? 1u : 0u;
              }
            }
            if (tot_c) {
              uint32_t base = 0u;
              if (lane == 0) base = atomicAdd(&ctl.lcnt[sb], (uint32_t)tot_c);
              base = __shfl_sync(0xFFFFFFFFu, base, 0);
              uint32_t* lst = reinterpret_cast<uint32_t*>(smem + g.off_list) + sb * LCAP;
              const uint16_t* srow = logits + (int64_t)(blockIdx.x + (int64_t)rs * gridDim.x) * a.ld;
              for (int k0 = 0; k0 < tot_c; k0 += 32) {
                const int k = k0 + lane;
                const int u = pick(k, ic, nc, cm);
                if (k < tot_c) {
                  const uint32_t idx = base + (uint32_t)k;
                  if (idx < LCAP) {
                    const uint32_t e = sk[u];
                    const uint32_t kg = okey16(e & 0xFFFFu), k2 = okey16(e >> 16);
                    count_token<CZ>(hist, key_m, e & 0xFFFFu, ctl, sb);
                    count_token<CZ>(hist, key_m, e >> 16, ctl, sb);
                    if (u < uy) tie += (kg == key_y ? 1u : 0u) + (k2 == key_y ? 1u : 0u);
                    lst[idx] = (uint32_t)u | (e & 0xFFFF0000u);
                  } else if (!CZ || *reinterpret_cast<volatile const uint32_t*>(&ctl.mgn[sb]) <= MGCAP) {
                    // no room in the list: counted whole here (unless the
                    // shared near-zero bin's list has run out of room: such a
                    // row is handed on, so its count can stop)
                    uint32_t ny;
                    count_unit<CZ>(srow, a.V, u, TMA && u < g.nfull, zf2w, key_m, key_y, hist, ny, ctl, sb);
                    if (u < uy) tie += ny;
                  }
                }
              }
            }
        };
        if (ctl.rec[sb].cz) count_row(std::true_type{});
        else count_row(std::false_type{});
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tie += __shfl_down_sync(0xFFFFFFFFu, tie, o);
      if (lane == 0 && tie) atomicAdd(&ctl.tie[sb], tie);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl.counted[sb]));
    };

    for (int64_t r = blockIdx.x; r < a.T; r += gridDim.x, ++it) {
      const int b = it & 1;
      Acc st{-INFINITY, DF{0.f, 0.f}, make_float2(0.f, 0.f), -INFINITY, 0x7F807F80u};
      float c = 0.f;
      bool nou = false;   // a row at top_p < 1: U is not needed
      const uint16_t* row = logits + r * a.ld;
      uint32_t* sk = reinterpret_cast<uint32_t*>(skb + (size_t)b * g.skb);
      // One stage: wait for the slot, fold this thread's unit (whole units
      // on every stage but the last), release the slot, then side work.
      auto stage = [&](int s, bool last) {
        const uint32_t slot = gs & (NSTAGE - 1);
        const bool ok = wait_full_warp(smem_u32(&ctl.full[slot]), (gs / NSTAGE) & 1u, abort, g.wait_limit,
                                  a.status);
        const int u = t + s * NTC;
        if (ok && (!last || u < g.nunits)) {
          uint32_t w[8];
          uint32_t ent = 0u;
          if (!last || u < g.nfull) {
            if (TMA) {
              const uint4* q = reinterpret_cast<const uint4*>(ring + slot * STAGE_BYTES) + 2 * t;
              const uint4 v0 = q[h], v1 = q[1 - h];
              w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
              w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
            } else {
              load_unit_scalar(row, a.V, u, h, w);
            }
            if (nou) {
              if (last) absorb_unit<false, false, TOPP, true>(st, w, c, 0xFFFFu, &ent);
              else absorb_unit<false, true, TOPP, true>(st, w, c, 0xFFFFu, &ent);
            } else {
              if (last) absorb_unit<false, false, TOPP>(st, w, c, 0xFFFFu, &ent);
              else absorb_unit<false, true, TOPP>(st, w, c, 0xFFFFu, &ent);
            }
          } else {
            // the row's last, partial unit: slot j of the words holds logit
            // 8 * (j < 8 ? h : 1 - h) + (j & 7) of the unit
            load_unit_scalar(row, a.V, u, h, w);
            const int nv = (int)(a.V - (int64_t)u * UNIT);   // 1..15 logits exist
            uint32_t vm = 0u;
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (8 * (j < 8 ? h : 1 - h) + (j & 7) < nv) vm |= 1u << j;
            if (nou) absorb_unit<true, false, TOPP, true>(st, w, c, vm, &ent);
            else absorb_unit<true, false, TOPP>(st, w, c, vm, &ent);
          }
          if (TOPP) sk[u] = ent;
        }
        mbar_arrive(smem_u32(&ctl.empty[slot]));   // this lane is done with the slot
        ++gs;
      };
      // The row's parameters are published with its first stage.
      {
        const uint32_t slot = gs & (NSTAGE - 1);
        wait_full(smem_u32(&ctl.full[slot]), (gs / NSTAGE) & 1u, abort, g.wait_limit, a.status);
        c = ctl.rp[it % NRP].c;
        nou = TOPP && ctl.rp[it % NRP].top_p < 1.0f;
      }
      for (int s = 0; s + 1 < g.nst; ++s) stage(s, false);
      stage(g.nst - 1, true);
      // The previous row's side work, by every warp at once: the producer
      // meanwhile fills the ring's stages for the next row.
      if (TOPP && it > 0) side_row(it - 1);
      // Merge the warp's 32 thread states in a fixed order: rescale to the
      // warp's largest reference (exact powers of two), then a shuffle tree.
      // (At top_p < 1 the side work above has waited for the previous row's
      // record, so the merge warp is done with this row's state buffer.)
      float Ew = st.E;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) Ew = fmaxf(Ew, __shfl_xor_sync(0xFFFFFFFFu, Ew, o));
      DF ws_s{0.f, 0.f};
      float ws_u = 0.f;
      {
        const float n = __fsub_rn(st.E, Ew);
        const float f = exp2_int(n);
        if (f != 0.f) {
          ws_s = DF{__fmul_rn(st.S.hi, f), __fmul_rn(st.S.lo, f)};
          ws_u = __fmul_rn(f, __fmaf_rn(n, __fadd_rn(st.S.hi, st.S.lo), __fadd_rn(st.U.x, st.U.y)));
        }
        if (nou && (bf16_lo(st.mn) == -INFINITY || bf16_hi(st.mn) == -INFINITY)) ws_u = NAN;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const DF x{shfl_down(ws_s.hi, o), shfl_down(ws_s.lo, o)};
        const float ux = shfl_down(ws_u, o);
        ws_s = df_add(ws_s, x);
        ws_u = __fadd_rn(ws_u, ux);
      }
      // The state buffer was last read by the merge warp two rows ago (at
      // top_p < 1 the side work above has already waited for that).
      if (!TOPP && it >= 2)
        wait_phase(smem_u32(&ctl.floorpub[b]), (uint32_t)(((it - 2) >> 1) & 1), abort, g.wait_limit,
                   a.status);
      const uint32_t kx = __reduce_max_sync(0xFFFFFFFFu, okey32(__float_as_uint(st.mx)));
      if (lane == 0) {
        float* pb = part + b * 4 * 32;
        pb[warp] = Ew;
        pb[32 + warp] = ws_s.hi;
        pb[64 + warp] = ws_s.lo;
        pb[96 + warp] = ws_u;
        ctl.wkey[b][warp] = kx;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl.rowpub[b]));
    }
    if (TOPP && it > 0) side_row(it - 1);
  } else if (warp == WPROD) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    uint32_t gs = 0;
    int it = 0;
    int issued[NSTAGE];   // parity of the last copy issued on a slot (-1: none pending)
    for (int s = 0; s < NSTAGE; ++s) issued[s] = -1;
    const bool per_row = a.temps || a.top_ps;
    for (int64_t r = blockIdx.x; r < a.T && !*abort; r += gridDim.x, ++it) {
      RowParam p{c0, a.temperature, a.top_p, 0.f, 0u, {0u, 0u, 0u}};
      if (per_row) {
        if (a.temps) p.temp = a.temps[r];
        if (a.top_ps) p.top_p = a.top_ps[r];
        p.bad = !(isfinite(p.temp) && p.temp > 0.f && p.top_p > 0.f && p.top_p <= 1.f);
        p.c = p.bad ? 1.f : (float)(1.4426950408889634 / (double)p.temp);
        if (a.temps) p.row_t = p.temp;
      }
      ctl.rp[it % NRP] = p;
      const char* src = reinterpret_cast<const char*>(logits + r * a.ld);
      for (int s = 0; s < g.nst; ++s, ++gs) {
        const uint32_t slot = gs & (NSTAGE - 1);
        // Once a wait of this CTA has run out no further copy is issued: the
        // consumers may have left a slot unread.
        if (gs >= NSTAGE &&
            !wait_phase(smem_u32(&ctl.empty[slot]), ((gs / NSTAGE) - 1) & 1u, abort,
                        g.wait_limit, a.status))
          break;
        if (*abort) break;
        if (blockIdx.x == 0 && (long long)gs == g.withhold) continue;   // debug: a copy never issued
        const uint32_t bar = smem_u32(&ctl.full[slot]);
        const uint32_t b0 = (uint32_t)s * STAGE_BYTES;
        uint32_t bytes = 0u;
        if (TMA && b0 < g.tma_bytes) bytes = min((uint32_t)STAGE_BYTES, g.tma_bytes - b0);
        if (bytes) {
          mbar_expect_tx(bar, bytes);
          bulk_copy_g2s(smem_u32(ring + slot * STAGE_BYTES), src + b0, bytes, bar);
          issued[slot] = (int)((gs / NSTAGE) & 1);
        } else {
          mbar_arrive(bar);
          issued[slot] = -1;
        }
      }
    }
    // Let every copy this thread issued land before the CTA may exit.
    volatile int never = 0;
    for (int s = 0; s < NSTAGE; ++s)
      if (issued[s] >= 0)
        wait_phase(smem_u32(&ctl.full[s]), (uint32_t)issued[s], &never, g.wait_limit, a.status);
  } else if (warp == WMRG) {
    // ---------------------------------------------------------- merge warp
    int it = 0;
    for (int64_t r = blockIdx.x; r < a.T; r += gridDim.x, ++it) {
      const int b = it & 1;
      const uint32_t par = (uint32_t)((it >> 1) & 1);
      // A row is trusted only if no wait of this CTA has run out (the compute
      // warps still publish rows after an abort, without having read them).
      const bool waited = wait_phase(smem_u32(&ctl.rowpub[b]), par, abort, g.wait_limit, a.status);
      const bool ok = __shfl_sync(0xFFFFFFFFu, (waited && !*abort) ? 1 : 0, 0) != 0;
      const RowParam p = ctl.rp[it % NRP];
      const int64_t y = a.ids[r];
      const bool bad_id = y < 0 || y >= a.V;
      const uint16_t* row = logits + r * a.ld;
      const float zy = bad_id ? 0.f : bf16_val(__ldg(row + y));
      uint32_t km = lane < NWC ? ctl.wkey[b][lane] : 0u;
      km = __reduce_max_sync(0xFFFFFFFFu, km);
      const float m = __uint_as_float(okey32_inverse(km));
      const float c = p.c;
      const float E = ceilf(__fmul_rn(m, c));
      // Merge the warp states in a fixed order: lane l takes warp l's state,
      // rescaled to E (exact powers of two), then a shuffle tree.
      DF Z{0.f, 0.f};
      float U = 0.f;
      if (ok && lane < NWC) {
        const float* pb = part + b * 4 * 32;
        const float n = __fsub_rn(pb[lane], E);
        const float f = exp2_int(n);
        if (f != 0.f) {
          const float shi = pb[32 + lane], slo = pb[64 + lane];
          Z = DF{__fmul_rn(shi, f), __fmul_rn(slo, f)};
          U = __fmul_rn(f, __fmaf_rn(n, __fadd_rn(shi, slo), pb[96 + lane]));
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const DF x{shfl_down(Z.hi, o), shfl_down(Z.lo, o)};
        const float ux = shfl_down(U, o);
        Z = df_add(Z, x);
        U = __fadd_rn(U, ux);
      }
      RowRec rc{};
      if (lane == 0) {
        const float zf = __fadd_rn(Z.hi, Z.lo);
        const bool nonfinite = !(isfinite(zf) && isfinite(U) && isfinite(m) && isfinite(E));
        const bool topp = TOPP && p.top_p < 1.0f;
        rc.E = E; rc.c = c; rc.U = U; rc.zy = zy; rc.top_p = p.top_p; rc.row_t = p.row_t;
        rc.zhi = Z.hi; rc.zlo = Z.lo;
        rc.y = (int32_t)y;
        if (!ok) { rc.mode = REC_BAD; rc.bad_bit = 0u; }
        else if (p.bad) { rc.mode = REC_BAD; rc.bad_bit = RLK_STATUS_BAD_PARAM; }
        else if (bad_id) { rc.mode = REC_BAD; rc.bad_bit = RLK_STATUS_BAD_TOKEN_ID; }
        else if (nonfinite) { rc.mode = REC_BAD; rc.bad_bit = RLK_STATUS_NONFINITE; }
        else if (!topp) {
          rc.mode = REC_DONE;
          const float lz = logf(zf);
          rc.lp = __fsub_rn(__fmul_rn(kLn2, __fmaf_rn(zy, c, -E)), lz);
          rc.ent = __fsub_rn(lz, __fdiv_rn(__fmul_rn(kLn2, U), zf));
          rc.lz = lz;
          rc.kstar = (int32_t)a.V;
        } else {
          // The window z >= m - L T as keys [key_lo, key_m].
          const float L_spec = logf(__fdiv_rn(1.f, __fsub_rn(1.f, p.top_p))) + 7.0f;
          const float zlo = __fsub_rn(m, __fmul_rn(L_spec, p.temp));
          const uint32_t key_m = key_of(m);
          const uint32_t kl = key_of(zlo);
          const uint32_t key_lo = kl > 0u ? kl - 1u : 0u;
          uint32_t dmax = key_m - key_lo;
          uint32_t cz = 0u, ckm = key_m;
          if (key_lo <= key_m && dmax >= (uint32_t)HBC && key_m >= MG_LO && key_lo <= MG_HI) {
            // the window reaches into the near-zero keys (from above them, or
            // from a max among them): bins by compressed key
            cz = 1u;
            ckm = ck_of<true>(key_m);
            dmax = ckm - ck_of<true>(key_lo);
          }
          if (key_lo <= key_m && dmax < (uint32_t)HBC) {
            rc.mode = REC_COUNT;
            const uint32_t fb = okey16_inverse(key_lo);
            rc.zf2 = fb | (fb << 16);
            rc.key_m = key_m;
            rc.dmax = dmax;
            rc.key_y = key_of(zy);
            rc.cz = cz;
            rc.ckm = ckm;
            rc.key_lo = key_lo;
          } else {
            rc.mode = REC_MARK;
          }
        }
      }
      // The record buffer and the counts of this buffer were last used two
      // rows ago: wait until the scan warp is done with them.
      if (it >= 2)
        wait_phase(smem_u32(&ctl.hclear[b]), (uint32_t)(((it - 2) >> 1) & 1), abort, g.wait_limit,
                   a.status);
      if (lane == 0) {
        if (*abort && rc.mode != REC_BAD) { rc.mode = REC_BAD; rc.bad_bit = 0u; }
        ctl.rec[b] = rc;
        mbar_arrive(smem_u32(&ctl.floorpub[b]));
      }
      __syncwarp();
    }
  } else {
    // ---------------------------------------------------------- scan warps
    // Warp WSCN + s finishes the CTA's rows it = s, s + 2, ... (buffer s), so
    // each has two rows' time for one.
    const int s0 = warp - WSCN;
    int it = s0;
    for (int64_t r = blockIdx.x + (int64_t)s0 * gridDim.x; r < a.T; r += 2 * (int64_t)gridDim.x, it += 2) {
      const int b = it & 1;
      const uint32_t par = (uint32_t)((it >> 1) & 1);
      bool ok = wait_phase(smem_u32(&ctl.floorpub[b]), par, abort, g.wait_limit, a.status);
      const RowRec rc = ctl.rec[b];
      const uint16_t* row = logits + r * a.ld;
      // The selected token's unit, read while the compute warps count.
      const bool counting = TOPP && rc.mode == REC_COUNT;
      uint32_t ybits = 0xFF80u;
      const int64_t ypos = (int64_t)(rc.y & ~15) + lane;
      if (ok && counting && lane < UNIT && ypos >= 0 && ypos < a.V) ybits = __ldg(row + ypos);
      // every row's count phase completes (the compute warps report each one)
      if (TOPP) ok = wait_phase(smem_u32(&ctl.counted[b]), par, abort, g.wait_limit, a.status) && ok;
      ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
      uint32_t* hist = hist0 + b * HBC;
      if (!ok || *abort) {
        if (lane == 0) write_bad(a, r, 0u);
      } else if (rc.mode == REC_BAD) {
        if (lane == 0) write_bad(a, r, rc.bad_bit);
      } else if (rc.mode == REC_DONE) {
        if (lane == 0) {
          a.out_logprob[r] = rc.lp;
          a.out_entropy[r] = rc.ent;
          if (a.out_k) a.out_k[r] = rc.kstar;
          if (a.state)
            a.state[r] = RowState{rc.E, rc.lz, rc.ent, 0u, kTiesAll, kStateValid | kStateYIn,
                                  rc.kstar, rc.row_t};
        }
      } else if (rc.mode == REC_MARK) {
        if (lane == 0) a.out_logprob[r] = __uint_as_float(kRecomputeMark);
      } else {
        auto scan_row = [&](auto czc) {
          constexpr bool CZ = decltype(czc)::value;
            // The counts so far are exact for every token but the third and
            // later largest of the listed units.  A first scan on them bounds the
            // crossing from below; the listed units whose second largest logit
            // reaches that bound are read again and their other tokens above it
            // added; a second scan then sees exact counts above the bound.
            const DF Z{rc.zhi, rc.zlo};
            const DF target = df_mul_f(Z, rc.top_p);
            uint32_t ty = 0u;
            if (lane < UNIT && bf16_lo(ybits) >= bf16_lo(rc.zf2)) {
              const uint32_t kk = okey16(ybits);
              count_token<CZ>(hist, rc.ckm, ybits, ctl, b);
              ty = (kk == rc.key_y && ypos < rc.y) ? 1u : 0u;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ty += __shfl_xor_sync(0xFFFFFFFFu, ty, o);
            uint32_t tie_all = ctl.tie[b] + ty;
            __syncwarp();
            ScanOut so{};
            float mg_mass = 0.f, mg_um = 0.f;
            // A shared near-zero bin whose list ran out of room has no exact
            // mass: the row is handed on without a scan (the compute warps
            // stopped counting it too).
            const bool lost = CZ && ctl.mgn[b] > MGCAP;
            bool found = false, short_mass = false;
            if (!lost) {
              if (CZ) mg_sums(ctl, b, lane, rc.c, rc.E, mg_mass, mg_um);
              found = warp_scan_window<CZ>(lane, rc.dmax, rc.ckm, rc.c, rc.E, target, hist, rc.key_y,
                                           tie_all, so, short_mass, mg_mass, mg_um);
              // (units beyond the list's room were counted whole by the compute warps)
              const uint32_t ncx = ctl.lcnt[b] < LCAP ? ctl.lcnt[b] : LCAP;
              if (ncx > 0u) {
                const uint32_t kap = found ? so.key_thr : rc.key_lo;
                const uint32_t kvb = okey16_inverse(kap);
                const uint32_t* lst = reinterpret_cast<const uint32_t*>(smem + g.off_list) + b * LCAP;
                const int uy = rc.y >> 4;
                uint32_t* lstw = reinterpret_cast<uint32_t*>(smem + g.off_list) + b * LCAP;
                // keep the listed units whose second largest reaches kap (in place, in order)
                uint32_t nneed = 0u;
                for (uint32_t k0 = 0u; k0 < ncx; k0 += 32u) {
                  const uint32_t k = k0 + (uint32_t)lane;
                  const uint32_t item = k < ncx ? lst[k] : 0u;
                  const bool need = k < ncx && okey16(item >> 16) >= kap;
                  const uint32_t bal = __ballot_sync(0xFFFFFFFFu, need);
                  __syncwarp();
                  if (need) lstw[nneed + __popc(bal & ((1u << lane) - 1u))] = item;
                  nneed += __popc(bal);
                }
                __syncwarp();
                uint32_t added = 0u, tx = 0u;
                for (uint32_t k = (uint32_t)lane; k < nneed; k += 32u) {
                  const uint32_t item = lstw[k];
                  const int u = (int)(item & 0xFFFFu);
                  uint32_t ny;
                  added += recount_unit<CZ>(row, a.V, u, TMA && u < g.nfull, kvb | (kvb << 16), rc.ckm,
                                        rc.key_y, hist, ny, ctl, b);
                  if (u < uy) tx += ny;
                }
                if (__any_sync(0xFFFFFFFFu, added != 0u)) {
#pragma unroll
                  for (int o = 16; o > 0; o >>= 1) tx += __shfl_xor_sync(0xFFFFFFFFu, tx, o);
                  tie_all += tx;
                  __syncwarp();
                  __syncwarp();
                  if (CZ) mg_sums(ctl, b, lane, rc.c, rc.E, mg_mass, mg_um);
                  found = warp_scan_window<CZ>(lane, rc.dmax, rc.ckm, rc.c, rc.E, target, hist, rc.key_y,
                                           tie_all, so, short_mass, mg_mass, mg_um);
                }
              }
            }
            // the second look can fill the shared bin's list too
            if (CZ && ctl.mgn[b] > MGCAP) found = short_mass = false;
            if (lane == 0) {
              if (!found) {
                a.out_logprob[r] = __uint_as_float(short_mass ? kRecomputeMarkWide : kRecomputeMark);
              } else {
                a.out_logprob[r] = so.y_in
                                       ? __fsub_rn(__fmul_rn(kLn2, __fmaf_rn(rc.zy, rc.c, -rc.E)), so.lz)
                                       : -INFINITY;
                a.out_entropy[r] = so.h;
                if (a.out_k) a.out_k[r] = (int32_t)so.kstar;
                if (a.state)
                  a.state[r] = RowState{rc.E, so.lz, so.h, so.key_thr, so.ties,
                                        kStateValid | (so.y_in ? kStateYIn : 0u), (int32_t)so.kstar,
                                        rc.row_t};
              }
            }
        };
        if (rc.cz) scan_row(std::true_type{});
        else scan_row(std::false_type{});
      }
      if (TOPP && rc.mode == REC_COUNT) {
        __syncwarp();
        for (uint32_t d = (uint32_t)lane; d <= rc.dmax; d += 32u) hist[d] = 0u;
        if (lane == 0) {
          ctl.tie[b] = 0u;
          ctl.lcnt[b] = 0u;
          ctl.mgn[b] = 0u;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl.hclear[b]));
    }
  }
}

}  // namespace

constexpr uint32_t kSmemMax =
    align_up(align_up((uint32_t)sizeof(Ctrl), 128) + PART_BYTES + 2u * HBC * 4u + 2u * LCAP * 4u +
                 2u * align_up((uint32_t)(V_MAX / UNIT) * 4u, 16),
             128) +
    NSTAGE * STAGE_BYTES;
static_assert(kSmemMax <= 232448u, "shared memory of one CTA");

bool lpe_stream_eligible(const LpeArgs& a) {
  return a.dtype == 0 && a.V >= V_MIN && a.V <= V_MAX;
}

cudaError_t launch_lpe_stream(const LpeArgs& a, cudaStream_t stream, long long wait_limit,
                              long long withhold) {
  Geom g{};
  g.nunits = (int)((a.V + UNIT - 1) / UNIT);
  g.nfull = (int)(a.V / UNIT);
  g.nst = (g.nunits + NTC - 1) / NTC;
  g.tma = ((reinterpret_cast<uintptr_t>(a.logits) & 15u) == 0 && (a.ld & 7) == 0) ? 1 : 0;
  g.tma_bytes = (uint32_t)((a.V / 8) * 16);
  uint32_t off = align_up((uint32_t)sizeof(Ctrl), 128);
  g.off_part = off;
  off += PART_BYTES;
  g.off_hist = off;
  off += 2u * HBC * 4u;
  g.off_list = off;
  off += 2u * LCAP * 4u;
  g.skb = align_up((uint32_t)g.nunits * 4u, 16);
  g.off_sk = off;
  off += 2u * g.skb;
  off = align_up(off, 128);
  g.off_ring = off;
  off += NSTAGE * STAGE_BYTES;
  const size_t smem = off;
  g.wait_limit = wait_limit;
  g.withhold = withhold;
  const float c = (float)(1.4426950408889634 / (double)a.temperature);
  const bool topp = a.temps || a.top_ps || a.top_p < 1.0f;

  // The shared-memory attribute is set once per device and variant.
  static std::atomic<int> attr[64][4];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int vi = (topp ? 2 : 0) + (g.tma ? 1 : 0);
  const void* fns[4] = {(const void*)lpe_stream_kernel<false, false>, (const void*)lpe_stream_kernel<false, true>,
                        (const void*)lpe_stream_kernel<true, false>, (const void*)lpe_stream_kernel<true, true>};
  const int smax = (int)kSmemMax;
  if (dev < 0 || dev >= 64 || attr[dev][vi].load() < smax) {
    if ((e = cudaFuncSetAttribute(fns[vi], cudaFuncAttributeMaxDynamicSharedMemorySize, smax)) !=
        cudaSuccess)
      return e;
    if (dev >= 0 && dev < 64) attr[dev][vi].store(smax);
  }
  const int nsm = sm_count();
  const int64_t grid = a.T < (int64_t)nsm ? a.T : (int64_t)nsm;
  // a programmatic dependent of the kernel before it on the stream (it waits
  // for that kernel's writes before reading anything)
  void (*const ks[4])(LpeArgs, Geom, float) = {lpe_stream_kernel<false, false>, lpe_stream_kernel<false, true>,
                                               lpe_stream_kernel<true, false>, lpe_stream_kernel<true, true>};
  e = launch_after(ks[vi], dim3((unsigned)grid), dim3(NTB), smem, stream, a, g, c);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace rlk
