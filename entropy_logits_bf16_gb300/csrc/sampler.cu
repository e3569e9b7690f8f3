// rlk_sample_top_p kernel: a deterministic top-p sampler.
//
// The sampler draws the id at which the cumulative renormalised probability,
// taken over the retained set S in ranking order (logit descending, id
// ascending), first reaches u (RL-Kernel "Qwen3-8B VIME train-rollout
// consistency", section "ROCm MI300X and gfx942": sampling keeps the
// sampler's native temperature / softmax / sort / top-p semantics; "ROCm
// sparse performance" notes: a deterministic top-p sampler).  u is supplied
// per row; S is the one rlk_logprob_entropy_fwd selected (its row state).
//
// Instead of a sort and a prefix scan over the vocabulary, one CTA per row,
// four rows in flight per SM, each thread keeping NLD 16-byte loads in flight
// (groups whose maximum reaches the retained range are queued per warp and
// tested 32 at a time, one per lane).  Direct mode, when the members' keys lie within NBD of the boundary
// key (the top key is known to within a bf16 step from the saved E =
// fp32(m c)): one read of the row counts members into bins by key - boundary
// with exact fixed-point masses and lists each member's position; a block
// scan from the top finds the draw's key, and the member list gives the
// need-th lowest position holding it (a scan of the row in id order only when
// the list ran out of room or the key's tie group is too large to rank).
// Otherwise (or when a member lands above the estimate) a radix descent on the
// 16-bit order-preserving key of the bf16 logits:
//  1. members (key > boundary, or == boundary among the kept ties) counted
//     into 256 bins by key >> 8, with masses w = 2^(z c - E) as fixed-point
//     integers (w 2^40, truncated), so every sum is exact and order-free;
//     the bins are scanned from the top for the first whose cumulative mass
//     reaches u Z_S;
//  2. the same inside that bin by key & 255: the exact key, and how many of
//     its tokens (lowest ids first) the draw needs;
//  3. the need-th id holding that key, by a block scan of matches in id order.
// Tokens whose weight is below 2^-40 of the row maximum count with mass 0.

#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "rlk.h"

namespace rlk {
namespace {

constexpr int NTM = 256;
constexpr int NWM = NTM / 32;
constexpr float kFix = 1099511627776.0f;   // 2^40

constexpr int NBD = 2048;   // direct mode: members' keys within NBD of the boundary key
// the direct-mode scan gives each thread exactly 8 consecutive bins
static_assert(NBD == 8 * NTM, "direct-mode bins: 8 per thread");
constexpr uint32_t LCAP = 4096;   // direct mode: members listed per row
constexpr uint32_t GCAP = 1024;   // largest tie group ranked from the list
constexpr int64_t kListMaxV = int64_t(1) << 21;   // a position and a bin in 32 bits
constexpr int NLD = 5;            // 16-byte loads in flight per thread (5 measured fastest of 2..8)
constexpr uint32_t QCAP = 64;     // a warp's queue of passing groups (at most 63 held)

struct MSmem {
  union {
    struct {                        // radix descent: 256 bins per level
      unsigned long long mass[256];
      uint32_t cnt[256];
    };
    struct {                        // direct mode: bin = key - boundary key
      unsigned long long dmass[NBD];
      uint32_t dcnt[NBD];
    };
    uint32_t grp[GCAP];             // direct mode, after the scan: the draw's tie group
  };
  uint32_t lst[LCAP];             // direct mode: members, position << 11 | bin
  uint32_t q[NWM][QCAP];          // each warp's queue of groups that reach the range
  uint32_t lcnt;                  // members listed (may exceed LCAP)
  uint32_t gn;                    // tie group gathered
  unsigned long long wsum[NWM];   // per-warp sums (direct-mode scan)
  uint32_t n_thr;                 // tokens holding the boundary key
  int ovf;                        // direct mode: a member above the estimated top key
  int dsel;                       // direct mode: the winning distance
  uint32_t wt[2][NWM];            // per-warp match counts (pass 3), double-buffered
  int sel;                        // scan result: the bin (or -1)
  unsigned long long before;      // mass ahead of the selected bin
  int found;
};

__device__ __forceinline__ uint64_t fixed_w(float z, float c, float E) {
  return (uint64_t)__float2ull_rz(__fmul_rn(ex2(__fmaf_rn(z, c, -E)), kFix));
}

// Bins of the current level scanned from bin 255 down by warp 0 in a fixed
// order; the first non-empty bin whose inclusive cumulative mass (from
// `base`) reaches target.  Results in sm.sel / sm.before (sel = -1: none).
__device__ void scan256(MSmem& sm, unsigned long long base, unsigned long long target) {
  const int lane = threadIdx.x & 31;
  if (threadIdx.x >= 32) return;
  // lane l owns bins 255 - 8 l ... 248 - 8 l (descending)
  unsigned long long own = 0ull;
#pragma unroll
  for (int k = 0; k < 8; ++k) own += sm.mass[255 - 8 * lane - k];
  unsigned long long inc = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long l = __shfl_up_sync(0xFFFFFFFFu, inc, o);
    if (lane >= o) inc += l;
  }
  unsigned long long cum = base + inc - own;
  int my = -1;
  unsigned long long my_before = 0ull;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int b = 255 - 8 * lane - k;
    const unsigned long long nx = cum + sm.mass[b];
    if (my < 0 && sm.cnt[b] > 0u && nx >= target) {
      my = b;
      my_before = cum;
    }
    cum = nx;
  }
  const uint32_t bal = __ballot_sync(0xFFFFFFFFu, my >= 0);
  if (bal == 0u) {
    // the draw is past the total (truncation): the lowest non-empty bin
    int last = -1;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int b = 255 - 8 * lane - k;
      if (sm.cnt[b] > 0u) last = b;
    }
    const uint32_t b2 = __ballot_sync(0xFFFFFFFFu, last >= 0);
    const int src = b2 ? 31 - __clz(b2) : 0;
    const int lb = __shfl_sync(0xFFFFFFFFu, last, src);
    unsigned long long bef = 0ull;   // mass ahead of bin lb
    if (lane == 0) {
      bef = base;
      for (int b = 255; b > lb; --b) bef += sm.mass[b];
      sm.sel = lb;
      sm.before = bef;
    }
    return;
  }
  const int src = __ffs(bal) - 1;   // the lowest lane holds the highest bins
  const int sel = __shfl_sync(0xFFFFFFFFu, my, src);
  const unsigned long long bef = __shfl_sync(0xFFFFFFFFu, my_before, src);
  if (lane == 0) {
    sm.sel = sel;
    sm.before = bef;
  }
}

__global__ void __launch_bounds__(NTM, 4) sample_kernel(SampleArgs a, float c0, int mode) {
  __shared__ MSmem sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t ngroups = (a.V + 7) / 8;
  uint32_t phase = 0u;
  for (int64_t r = blockIdx.x; r < a.T; r += gridDim.x) {
    const RowState st = a.state[r];
    if (!(st.flags & kStateValid)) {
      if (tid == 0) {
        a.out_ids[r] = -1;
        if (a.status) atomicOr(a.status, (st.flags >> 8) ? (st.flags >> 8) : RLK_STATUS_NO_STATE);
      }
      continue;
    }
    // the row's c: from the temperature its state recorded, else the call's
    const float c = st.temperature > 0.f ? (float)(1.4426950408889634 / (double)st.temperature)
                                         : c0;
    const uint16_t* p = reinterpret_cast<const uint16_t*>(a.logits) + r * a.ld;
    const bool vec = (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
    const uint32_t thr = st.key_thr;
    const float E = st.E;
    float u = a.uniforms[r];
    u = u < 0.f ? 0.f : (u < 1.f ? u : 0.99999994f);
    // The elements of the row whose keys lie in [klo, khi], each through
    // f(has, k, z, index), called by every lane of the warp together (has:
    // this lane holds an element this round).  A thread takes groups g,
    // g + NTM, ..., NLD of them per step, all loads issued before any is used;
    // a group whose largest value is below the range is dropped after one
    // packed max.  The others go into the warp's queue (their indices), and
    // every 32 queued groups are taken one per lane: the group read again
    // (from L2), tested two elements at a time by packed bf16 compares
    // against the range's end values (-0 == +0, as the keys have it), and its
    // elements in the range handed to f in rounds, one per lane and round.
    // The range test and the rounds thus run once per 32 passing groups, not
    // once per lane slot that holds one.
    auto for_row = [&](uint32_t klo, uint32_t khi, auto&& f) {
      // the range as values (keys below 0x7F are NaN, above 0xFF80 too; 0x7FFF
      // is the key -0 would have without its mapping to +0)
      const float lo_val = klo > 0x7Fu ? bf16_val(okey16_inverse(klo)) : -INFINITY;
      const float hi_val = khi >= 0xFF80u ? INFINITY : bf16_val(okey16_inverse(khi == 0x7FFFu ? 0x7FFEu : khi));
      const bool bounded = hi_val != INFINITY;
      const __nv_bfloat162 lo2 = __float2bfloat162_rn(lo_val), hi2 = __float2bfloat162_rn(hi_val);
      uint32_t* q = sm.q[warp];
      uint32_t head = 0u, tail = 0u;   // the warp's queue (warp-uniform counters, ring of QCAP)
      // lanes below n take queue entries head + lane
      auto drain = [&](uint32_t n) {
        __syncwarp();   // the entries written by other lanes are visible
        uint32_t m8 = 0u, w[4] = {0u, 0u, 0u, 0u};
        int64_t g = 0;
        if ((uint32_t)lane < n) {
          g = q[(head + (uint32_t)lane) & (QCAP - 1)];
          if (vec && g * 8 + 8 <= a.V) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(p) + g);
            w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
          } else {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const int64_t i0 = g * 8 + 2 * h;
              const uint32_t lo = i0 < a.V ? __ldg(p + i0) : 0xFF80u;
              const uint32_t hi = i0 + 1 < a.V ? __ldg(p + i0 + 1) : 0xFF80u;
              w[h] = lo | (hi << 16);
            }
          }
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            uint32_t mk = __hge2_mask(bf2(w[h]), lo2);
            if (bounded) mk &= __hle2_mask(bf2(w[h]), hi2);
            m8 |= ((mk & 1u) | ((mk >> 15) & 2u)) << (2 * h);
          }
          const int64_t left = a.V - g * 8;   // elements of the group inside the row
          if (left < 8) m8 &= (1u << left) - 1u;
        }
        head += n;
        while (__any_sync(0xFFFFFFFFu, m8 != 0u)) {
          const bool has = m8 != 0u;
          uint32_t bits = 0u;
          int64_t i = 0;
          if (has) {
            const int e = __ffs(m8) - 1;
            m8 &= m8 - 1u;
            const uint32_t wa = (e & 2) ? w[1] : w[0], wb = (e & 2) ? w[3] : w[2];
            bits = (((e & 4) ? wb : wa) >> (16 * (e & 1))) & 0xFFFFu;
            i = g * 8 + e;
          }
          f(has, okey16(bits), bf16_val(bits), i);
        }
        __syncwarp();   // the entries are read before later pushes reuse them
      };
      // the bound is the warp's (its first lane's): every lane of a warp runs
      // the same steps, as the ballots and the drains need; groups past the
      // row load nothing and never pass
      for (int64_t g0 = tid; g0 - lane < ngroups; g0 += (int64_t)NLD * NTM) {
        uint32_t w4[NLD][4];
#pragma unroll
        for (int j = 0; j < NLD; ++j) {
          const int64_t g = g0 + (int64_t)j * NTM;
          if (vec && g * 8 + 8 <= a.V) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(p) + g);
            w4[j][0] = v.x; w4[j][1] = v.y; w4[j][2] = v.z; w4[j][3] = v.w;
          } else {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const int64_t i0 = g * 8 + 2 * h;
              const uint32_t lo = i0 < a.V ? __ldg(p + i0) : 0xFF80u;
              const uint32_t hi = i0 + 1 < a.V ? __ldg(p + i0 + 1) : 0xFF80u;
              w4[j][h] = lo | (hi << 16);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < NLD; ++j) {
          const int64_t g = g0 + (int64_t)j * NTM;
          const __nv_bfloat162 m2 = __hmax2(__hmax2(bf2(w4[j][0]), bf2(w4[j][1])),
                                            __hmax2(bf2(w4[j][2]), bf2(w4[j][3])));
          const bool pass = g < ngroups && fmaxf(__low2float(m2), __high2float(m2)) >= lo_val;
          const uint32_t bal = __ballot_sync(0xFFFFFFFFu, pass);
          if (pass) q[(tail + (uint32_t)__popc(bal & ((1u << lane) - 1u))) & (QCAP - 1)] = (uint32_t)g;
          tail += (uint32_t)__popc(bal);
          if (tail - head >= 32u) drain(32u);
        }
      }
      if (tail != head) drain(tail - head);
    };
    const float zt = bf16_val(okey16_inverse(thr));
    const uint64_t w_thr = thr == 0u ? 0ull : fixed_w(zt, c, E);
    uint32_t key_sel = 0u, n_sel = 0u, need = 1u;
    bool have = false;          // key_sel / need found (block-uniform)
    bool direct_done = false;   // direct mode: the answer is written (block-uniform)
    {
      const float m_est = __fdiv_rn(E, c);   // the row max to within rounding
      uint32_t kmax = okey16(__float_as_uint(m_est) >> 16) + 4u;
      kmax = kmax > 0xFFFFu ? 0xFFFFu : kmax;
      if (mode >= 1 && thr != 0u && kmax >= thr && kmax - thr < (uint32_t)NBD) {
        const bool listing = mode == 1 && a.V <= kListMaxV;
        for (int i = tid; i < NBD; i += NTM) {
          sm.dmass[i] = 0ull;
          sm.dcnt[i] = 0u;
        }
        if (tid == 0) {
          sm.ovf = 0;
          sm.dsel = 0x7FFFFFFF;
          sm.lcnt = 0u;
          sm.gn = 0u;
        }
        __syncthreads();
        for_row(thr, 0xFFFFu, [&](bool has, uint32_t k, float z, int64_t i) {
          const uint32_t d = k - thr;
          const bool in = has && d < (uint32_t)NBD;
          if (has && !in) sm.ovf = 1;
          if (in) {
            atomicAdd(&sm.dcnt[d], 1u);
            atomicAdd(&sm.dmass[d], fixed_w(z, c, E));
          }
          if (listing) {   // one list slot reservation per warp and round
            const uint32_t bal = __ballot_sync(0xFFFFFFFFu, in);
            if (bal) {
              const int lead = __ffs(bal) - 1;
              uint32_t base = 0u;
              if (lane == lead) base = atomicAdd(&sm.lcnt, (uint32_t)__popc(bal));
              base = __shfl_sync(0xFFFFFFFFu, base, lead);
              const uint32_t idx = base + (uint32_t)__popc(bal & ((1u << lane) - 1u));
              if (in && idx < LCAP) sm.lst[idx] = ((uint32_t)i << 11) | d;
            }
          }
        });
        __syncthreads();
        if (!sm.ovf) {
          const uint32_t n_thr = sm.dcnt[0];   // tokens holding the boundary key
          uint32_t drop = 0u;
          if (st.ties != kTiesAll && n_thr > st.ties) drop = n_thr - st.ties;
          // thread t owns distances 8t .. 8t + 7 from the top (bin NBD - 1 - distance)
          unsigned long long own = 0ull;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int b = NBD - 1 - (8 * tid + k);
            own += sm.dmass[b] - (b == 0 ? (unsigned long long)drop * w_thr : 0ull);
          }
          unsigned long long inc = own;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long l = __shfl_up_sync(0xFFFFFFFFu, inc, o);
            if (lane >= o) inc += l;
          }
          if (lane == 31) sm.wsum[warp] = inc;
          __syncthreads();
          unsigned long long pre = 0ull, Z = 0ull;
#pragma unroll
          for (int w = 0; w < NWM; ++w) {
            if (w < warp) pre += sm.wsum[w];
            Z += sm.wsum[w];
          }
          const unsigned long long target = (unsigned long long)ceil((double)u * (double)Z);
          unsigned long long cum = pre + inc - own;
          int my = -1;
          unsigned long long my_before = 0ull;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int b = NBD - 1 - (8 * tid + k);
            const uint32_t n = sm.dcnt[b] - (b == 0 ? drop : 0u);
            const unsigned long long mb = sm.dmass[b] - (b == 0 ? (unsigned long long)drop * w_thr : 0ull);
            if (my < 0 && n > 0u && cum + mb >= target) {
              my = 8 * tid + k;
              my_before = cum;
            }
            cum += mb;
          }
          if (my >= 0) atomicMin(&sm.dsel, my);
          __syncthreads();
          const int dsel = sm.dsel;   // always found: the last member bin reaches Z
          if (my >= 0 && my == dsel) sm.before = my_before;
          __syncthreads();
          if (dsel != 0x7FFFFFFF) {
            const int b = NBD - 1 - dsel;
            const uint32_t n_all = sm.dcnt[b];   // tokens holding the key, kept or not
            n_sel = n_all - (b == 0 ? drop : 0u);
            const unsigned long long w_sel =
                (sm.dmass[b] - (b == 0 ? (unsigned long long)drop * w_thr : 0ull)) / n_sel;
            need = 1u;
            if (w_sel > 0ull && target > sm.before) {
              const unsigned long long q = (target - sm.before + w_sel - 1ull) / w_sel;
              need = q < 1ull ? 1u : (q > n_sel ? n_sel : (uint32_t)q);
            }
            key_sel = thr + (uint32_t)b;
            have = true;
            const uint32_t nl = sm.lcnt;
            if (listing && nl <= LCAP && n_all <= GCAP) {
              // every member is listed: gather the key's tie group (its
              // positions; the kept ties of the boundary key are its lowest)
              // and take the need-th lowest
              if (tid == 0) a.out_ids[r] = -1;   // overwritten below (the group holds need tokens)
              __syncthreads();   // the bins are read: grp overlays them
              for (uint32_t k = tid; k < nl; k += NTM) {
                const uint32_t e = sm.lst[k];
                if ((e & 2047u) == (uint32_t)b) {
                  const uint32_t gi = atomicAdd(&sm.gn, 1u);
                  if (gi < GCAP) sm.grp[gi] = e >> 11;
                }
              }
              __syncthreads();
              const uint32_t gn = min(sm.gn, GCAP);   // == n_all
              for (uint32_t t = tid; t < gn; t += NTM) {
                const uint32_t pos = sm.grp[t];
                uint32_t rank = 0u;
                for (uint32_t j = 0; j < gn; ++j) rank += sm.grp[j] < pos ? 1u : 0u;
                if (rank == need - 1u) a.out_ids[r] = (int32_t)pos;
              }
              direct_done = true;
            }
          }
        }
        __syncthreads();
      }
    }
    if (direct_done) continue;
    if (!have) {
    // ---- pass 1: bins by key >> 8
    for (int i = tid; i < 256; i += NTM) {
      sm.mass[i] = 0ull;
      sm.cnt[i] = 0u;
    }
    if (tid == 0) sm.n_thr = 0u;
    __syncthreads();
    for_row(thr, 0xFFFFu, [&](bool has, uint32_t k, float z, int64_t) {
      if (!has) return;
      atomicAdd(&sm.cnt[k >> 8], 1u);
      atomicAdd(&sm.mass[k >> 8], fixed_w(z, c, E));
      if (k == thr) atomicAdd(&sm.n_thr, 1u);
    });
    __syncthreads();
    uint32_t drop = 0u;   // tied tokens at the boundary that S does not keep
    if (st.ties != kTiesAll && sm.n_thr > st.ties) drop = sm.n_thr - st.ties;
    if (tid == 0 && drop) {
      sm.cnt[thr >> 8] -= drop;
      sm.mass[thr >> 8] -= (unsigned long long)drop * w_thr;
    }
    __syncthreads();
    // Z_S and the draw's target: the first token whose cumulative mass is >= u Z_S
    if (warp == 0) {   // integer sums: the order does not matter
      unsigned long long z = 0ull;
#pragma unroll
      for (int k = 0; k < 8; ++k) z += sm.mass[8 * lane + k];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) z += __shfl_down_sync(0xFFFFFFFFu, z, o);
      if (lane == 0) sm.before = z;
    }
    __syncthreads();
    const unsigned long long Z = sm.before;
    const unsigned long long target =
        (unsigned long long)ceil((double)u * (double)Z);
    __syncthreads();
    scan256(sm, 0ull, target);
    __syncthreads();
    const int hi_bin = sm.sel;
    const unsigned long long before1 = sm.before;
    __syncthreads();
    if (hi_bin < 0) {   // no member at all: a state that does not belong to these logits
      if (tid == 0) {
        a.out_ids[r] = -1;
        if (a.status) atomicOr(a.status, RLK_STATUS_NO_STATE);
      }
      continue;
    }
    // ---- pass 2: inside bin hi_bin, by key & 255
    for (int i = tid; i < 256; i += NTM) {
      sm.mass[i] = 0ull;
      sm.cnt[i] = 0u;
    }
    __syncthreads();
    for_row(max(thr, (uint32_t)hi_bin << 8), ((uint32_t)hi_bin << 8) | 255u,
            [&](bool has, uint32_t k, float z, int64_t) {
      if (!has) return;
      atomicAdd(&sm.cnt[k & 255u], 1u);
      atomicAdd(&sm.mass[k & 255u], fixed_w(z, c, E));
    });
    __syncthreads();
    if (tid == 0 && drop && (int)(thr >> 8) == hi_bin) {
      sm.cnt[thr & 255u] -= drop;
      sm.mass[thr & 255u] -= (unsigned long long)drop * w_thr;
    }
    __syncthreads();
    scan256(sm, before1, target);
    __syncthreads();
    if (sm.sel < 0) {   // unreachable for a state of these logits (pass 1 found members here)
      if (tid == 0) {
        a.out_ids[r] = -1;
        if (a.status) atomicOr(a.status, RLK_STATUS_NO_STATE);
      }
      __syncthreads();
      continue;
    }
    key_sel = ((uint32_t)hi_bin << 8) | (uint32_t)sm.sel;
    n_sel = sm.cnt[sm.sel];
    const unsigned long long w_sel = sm.mass[sm.sel] / (n_sel ? n_sel : 1u);   // equal values
    need = 1u;
    if (w_sel > 0ull && target > sm.before) {
      const unsigned long long q = (target - sm.before + w_sel - 1ull) / w_sel;
      need = q < 1ull ? 1u : (q > n_sel ? n_sel : (uint32_t)q);
    }
    }   // radix descent
    if (tid == 0) {
      sm.found = 0;
      a.out_ids[r] = -1;   // overwritten below (a member always holds key_sel)
    }
    __syncthreads();
    // ---- pass 3: the need-th id (ascending) holding key_sel
    const __nv_bfloat162 sel2 = bf2(okey16_inverse(key_sel) * 0x10001u);
    // Each step covers 4 NTM groups: thread t takes the four consecutive
    // groups 4 t .. 4 t + 3 of the step (ids stay in thread order).
    constexpr int GPS = 4;
    uint32_t carry = 0u;
    for (int64_t g0 = 0; g0 < ngroups; g0 += (int64_t)GPS * NTM) {
      const int64_t gb = g0 + (int64_t)GPS * tid;
      uint32_t mm = 0u;   // bit 8 j + e: element e of group gb + j holds key_sel
#pragma unroll
      for (int j = 0; j < GPS; ++j) {
        const int64_t g = gb + j;
        if (g >= ngroups) break;
        if (vec && g * 8 + 8 <= a.V) {
          // equal values <=> equal keys (-0 == +0; a valid row holds no NaN)
          const uint4 q = __ldg(reinterpret_cast<const uint4*>(p) + g);
          const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const uint32_t eq = __heq2_mask(bf2(w4[h]), sel2);
            mm |= ((eq & 1u) | ((eq >> 15) & 2u)) << (8 * j + 2 * h);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int64_t i = g * 8 + e;
            if (i < a.V && okey16(__ldg(p + i)) == key_sel) mm |= 1u << (8 * j + e);
          }
        }
      }
      const int64_t g = gb;   // ids: gb * 8 + bit
      const uint32_t n = (uint32_t)__popc(mm);
      uint32_t inc = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t l = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += l;
      }
      const int b = (int)(phase & 1u);
      if (lane == 31) sm.wt[b][warp] = inc;
      __syncthreads();
      uint32_t before = carry, total = 0u;
#pragma unroll
      for (int w = 0; w < NWM; ++w) {
        const uint32_t t = sm.wt[b][w];
        if (w < warp) before += t;
        total += t;
      }
      ++phase;
      const uint32_t first = before + inc - n;   // matches ahead of this thread's group
      if (n > 0u && first < need && need <= first + n) {
        uint32_t m2 = mm;
        for (uint32_t j = first + 1u; j < need; ++j) m2 &= m2 - 1u;
        a.out_ids[r] = (int32_t)(g * 8 + (__ffs(m2) - 1));
        sm.found = 1;
      }
      carry += total;
      __syncthreads();
      if (sm.found) break;
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_sample(const SampleArgs& a, cudaStream_t stream) {
  const float c = (float)(1.4426950408889634 / (double)a.temperature);
  // a row's serial phases (the scans, the barriers) are hidden by the other
  // rows in flight: four CTAs per SM (64 registers a thread; five would fit
  // in shared memory but spill at 48 registers, and measured slower)
  const int64_t cap = (int64_t)4 * sm_count();
  sample_kernel<<<(unsigned)(a.T < cap ? a.T : cap), NTM, 0, stream>>>(a, c, debug_sampler_mode());
  return cudaGetLastError();
}

}  // namespace rlk
