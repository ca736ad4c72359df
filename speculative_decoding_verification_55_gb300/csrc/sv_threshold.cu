// Thresholds of top-k / top-p filtering on sm_103a ([R] "Speculative decoding", rayaq.ca ml-models
// -- Why the output is exactly the target's: temperature, top-p and any penalties are applied to p
// and q before the test, and the rule then preserves exactly the distribution it is given).
//
// For every row the filters touch (the target rows 0..gamma_b and the draft rows 0..gamma_b - 1 of a
// sampled batch row whose top_k or top_p is on), the kernel finds the smallest logit the filters
// keep, tau, and writes it; every other row gets -inf. The filters keep exactly the logits z >= tau:
//   top-k   the logits at or above the k-th largest (ties at the boundary all kept);
//   top-p   on the renormalised top-k set, a logit is kept when the mass of the logits strictly
//           larger than it is below top_p times the set's mass (equal logits go together, the
//           largest is always kept).
// Both sets are upper sets of the logits' order, so one threshold describes them. The streaming
// kernel then verifies the batch with every logit below its row's threshold read as -inf: the
// softmax of the kept logits is the renormalised filtered distribution.
//
// One CTA of 512 threads per row at a time (persistent, two CTAs per SM so that one streams while
// the other selects; rows claimed from a counter when one is given); nothing is shared between
// CTAs. Masses are w = 2^-d with d = (M - z) log2(e) / T, the logit's log2 probability below the
// row max M. Per row:
//   1  top-k rows: a strided sample of 1/64 of the row's 16-byte vectors. Top-p rows (top-k off):
//      one pass over the row for M, a 1/16 sample and the row's mass (summed against each thread's
//      running max).
//   2  the sample's histogram over fine bins of d (8 per unit over [0, 64), then a tail bin; top-k
//      rows measure d from the sample's max) gives value cut points that hold the boundary with a
//      wide margin: top-k, the logits above the bin where the sample holds k's share plus three
//      deviations; top-p, the top bins (T), the bins counted as a whole (A) and the bins around
//      where the mass below, estimated from the sample's tail with a five-sigma margin, reaches
//      (1 - top_p) of the row's mass (C).
//   3  one pass (top-k: from DRAM, also the row max; top-p: the second pass, mostly from L2):
//      packed compares against the cut points, the logits of T and C appended to a shared-memory
//      list (one warp-aggregated atomic per four-vector step), A's mass summed per thread.
//   4  the exact selection on the list by radix levels of 8 bits over the logits' order keys from
//      the list's known key range (counts for top-k, 42-bit fixed-point masses for top-p; integer
//      sums, the same result for any order of the atomics), after checking that the boundary does
//      lie in the window.
//   5  with list outputs given: a top-k row's kept set, when it holds at most kList logits, as an
//      (index, logit) list for the list kernel.
// A row whose window misses the boundary or whose candidates do not fit (a large k, an unusual
// sample) takes the exact path instead: level-0 histograms of counts and masses over the whole
// row in coarse bins of d, then the same radix levels over the row (several passes, each exact).
// Within a bin, decisions are on exact keys and integer masses; bins and cut points only choose
// what is listed (membership is recomputed with the same compares in every pass).

#include <type_traits>

#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kTT = 512;                  // threads per CTA
constexpr int kCtasT = 2;                 // CTAs per SM: one streams while the other selects
constexpr int kTW = kTT / 32;
constexpr int kFB = 512;                  // fine bins (bin kFB is the tail)
constexpr float kFBPerLog2 = 8.0f;        // fine bins per unit of log2 probability
constexpr int kL0 = 256;                  // exact path: level-0 bins (bin kL0 is the tail)
constexpr float kL0PerLog2 = 4.0f;
constexpr float kFix = 4398046511104.0f;  // 2^42: the fixed-point scale of a mass 2^-d in [0, 1]
constexpr int kSampleVecs = 2048;         // sampled 16-byte vectors at most
constexpr int kCandMax = 16384;           // candidate logits (fp32)
constexpr int kIdxMax = kSampleVecs * 4;  // candidate indices kept (in the sample's place)
#ifndef SV_THRESHOLD_UNROLL
#define SV_THRESHOLD_UNROLL 4
#endif
constexpr int kU = SV_THRESHOLD_UNROLL;   // vectors in flight per thread in the two passes

// Dynamic shared memory holds either the fast path's sample and candidates or the exact path's
// per-warp level-0 histograms (never both at once).
constexpr int kSampleBytes = kSampleVecs * 16;
constexpr int kFastBytes = kSampleBytes + kCandMax * 4;
constexpr int kSlowBytes = kTW * kL0 * (8 + 4);
constexpr int kDynBytesT = kFastBytes > kSlowBytes ? kFastBytes : kSlowBytes;

struct TShared {
  unsigned fc[kFB + 1];                   // sample: fine-bin counts
  unsigned fd[kFB + 1];                   // sample: fine-bin sums of 2^16 (w / 2^-(b+1)/8 - 1)
  unsigned c0[kL0 + 1];                   // exact path: level-0 counts (index kL0: the tail)
  unsigned long long m0[kL0 + 1];
  unsigned rc[256];                       // a radix level
  unsigned long long rm[256];
  float redf[kTW];
  unsigned redu[kTW];
  unsigned long long redm[kTW];
  unsigned long long redm2[kTW];
  int bi[8];                              // broadcasts
  unsigned long long bm[8];
  float bx[4];                            // broadcast cut points
  unsigned ncand;
  int claim[2];                           // claimed rows (alternating slots)
};

// Order key: unsigned order of keys is the order of the values; -0 reads as +0. bf16 logits keep
// their 16 bits (keys < 2^16), fp32 their 32.
template <bool BF16>
__device__ __forceinline__ uint32_t order_key(float z) {
  uint32_t b = __float_as_uint(z);
  if (b == 0x80000000u) b = 0u;
  if (BF16) b >>= 16;
  const uint32_t sign = BF16 ? 0x8000u : 0x80000000u;
  const uint32_t mask = BF16 ? 0xffffu : 0xffffffffu;
  return (b & sign) ? (~b & mask) : (b | sign);
}

template <bool BF16>
__device__ __forceinline__ float key_value(uint32_t key) {
  const uint32_t sign = BF16 ? 0x8000u : 0x80000000u;
  const uint32_t mask = BF16 ? 0xffffu : 0xffffffffu;
  uint32_t b = (key & sign) ? (key & ~sign & mask) : (~key & mask);
  if (BF16) b <<= 16;
  return __uint_as_float(b);
}

// Bin of a logit at `per` bins per unit of d = (M - z) k over [0, nb / per), else the tail nb
// (-inf included). The rounding of M k can leave d slightly below 0 at the max: bin 0.
__device__ __forceinline__ int d_bin(float z, float Mk, float k, float per, int nb) {
  const float dd = fmaf(-z, k * per, Mk * per);
  if (!(dd < static_cast<float>(nb))) return nb;
  return dd > 0.0f ? static_cast<int>(dd) : 0;
}

// Mass of a logit relative to the max, 2^-d, in fixed point; at most 1 (the max's own mass, which
// the rounding of M k can push a little above 1), so V masses sum below 2^64 for V < 2^22.
// An approximate square root (the hardware's, not correctly rounded).
__device__ __forceinline__ float sqrt_approx(float x) {
  float y;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ unsigned long long fix_mass(float z, float Mk, float k) {
  const float w = fminf(ex2(fmaf(z, k, -Mk)), 1.0f);
  return __float2ull_rn(w * kFix);
}

// A 16-byte vector of the row with an L2 eviction policy.
__device__ __forceinline__ uint4 ld_pol_v4(const void* p, uint64_t pol) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
}

// The largest value of the storage type at or below x (fp32: x itself); -inf stays -inf.
template <bool BF16>
__device__ __forceinline__ float store_floor(float x) {
  if (!BF16) return x;
  uint32_t t = __float_as_uint(x) & 0xffff0000u;
  if (__uint_as_float(t) > x) t += 0x10000u;     // a negative x: one step down in value
  return __uint_as_float(t);
}

// Class words of a 16-byte vector against the cut points xt >= xa >= xl (values of the storage
// type): per logit, all ones in cw where it is a candidate (z >= xt, or xl <= z < xa) and in aw
// where it falls between (xa <= z < xt). bf16: one word per pair of logits, 16 bits per logit;
// fp32: one word per logit. kP: top-p over the whole row (three cut points), else top-k (z >= xt
// only, aw empty).
template <bool BF16, bool kP>
__device__ __forceinline__ void class_words(const uint4& v, float xt, float xa, float xl,
                                            uint32_t cw[4], uint32_t aw[4]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if (BF16) {
    const uint32_t t = __float_as_uint(xt) >> 16, a = __float_as_uint(xa) >> 16,
                   l = __float_as_uint(xl) >> 16;
    const uint32_t t2 = t | (t << 16), a2 = a | (a << 16), l2 = l | (l << 16);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t mt;
      asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(mt) : "r"(w[q]), "r"(t2));   // 0xffff where z >= x
      if (kP) {
        uint32_t ma, ml;
        asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(ma) : "r"(w[q]), "r"(a2));
        asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(ml) : "r"(w[q]), "r"(l2));
        cw[q] = mt | (ml & ~ma);
        aw[q] = ma & ~mt;
      } else {
        cw[q] = mt;
        aw[q] = 0u;
      }
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float z = __uint_as_float(w[q]);
      const bool gt = z >= xt;
      if (kP) {
        const bool ga = z >= xa, gl = z >= xl;
        cw[q] = (gt || (gl && !ga)) ? 0xffffffffu : 0u;
        aw[q] = (ga && !gt) ? 0xffffffffu : 0u;
      } else {
        cw[q] = gt ? 0xffffffffu : 0u;
        aw[q] = 0u;
      }
    }
  }
}

// Bit e of the result: logit e's entry of the class words. bf16: a byte of each half per logit
// (in logit order, by byte permutes), then one bit of each byte gathered by a multiply (the four
// partial products land on distinct bits, so nothing carries).
template <bool BF16>
__device__ __forceinline__ unsigned word_bits(const uint32_t m[4]) {
  if (BF16) {
    const uint32_t lo = __byte_perm(m[0], m[1], 0x6420) & 0x01010101u;   // logits 0..3
    const uint32_t hi = __byte_perm(m[2], m[3], 0x6420) & 0x01010101u;   // logits 4..7
    constexpr uint32_t kGather = (1u << 28) | (1u << 21) | (1u << 14) | (1u << 7);
    return ((lo * kGather) >> 28) | (((hi * kGather) >> 24) & 0xf0u);
  }
  unsigned bits = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) bits |= (m[q] & 1u) << q;
  return bits;
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// One warp over kPer * 32 bins h[idx(j)] in scan order j = 0, 1, ... (idx(j) = j ascending, or
// base - j descending): the first position whose inclusive cumulative sum reaches `target`.
// Returns the bin index (or -1 if the total stays below target) and the sum before it; every lane
// gets the answer.
template <int kPer, bool kDesc, typename T>
__device__ __forceinline__ int warp_first_reach(const T* h, int base, T target, int lane, T& before,
                                                T& total) {
  T loc[kPer];
  T s = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int j = lane * kPer + i;
    loc[i] = h[kDesc ? base - j : j];
    s += loc[i];
  }
  T incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  total = __shfl_sync(kFull, incl, 31);
  const unsigned hit = __ballot_sync(kFull, incl >= target);
  if (hit == 0u) {
    before = total;
    return -1;
  }
  const int L = __ffs(hit) - 1;
  int jr = 0;
  T b = 0;
  if (lane == L) {
    T a = incl - s;
    bool found = false;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      if (!found && a + loc[i] >= target) {
        found = true;
        jr = lane * kPer + i;
        b = a;
      }
      a += loc[i];
    }
  }
  jr = __shfl_sync(kFull, jr, L);
  before = __shfl_sync(kFull, b, L);
  return kDesc ? base - jr : jr;
}

// One warp over the 256 sub-bins of a radix level in descending order (255 first), with `above`
// the mass of every logit above the level's range: the last non-empty sub-bin entered with less
// than `target` above it (the smallest candidate key range still kept by top-p), and the mass
// above that sub-bin. -1 if none.
__device__ __forceinline__ int warp_last_below(const unsigned* cnt, const unsigned long long* mass,
                                               unsigned long long above, double target, int lane,
                                               unsigned long long& above_sel) {
  constexpr int kPer = 8;
  unsigned long long loc[kPer];
  unsigned long long s = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    loc[i] = mass[255 - (lane * kPer + i)];
    s += loc[i];
  }
  unsigned long long incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  unsigned long long a = above + (incl - s);
  int jsel = -1;
  unsigned long long asel = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int j = 255 - (lane * kPer + i);
    if (cnt[j] > 0u && static_cast<double>(a) < target) {
      jsel = j;
      asel = a;
    }
    a += loc[i];
  }
  const unsigned has = __ballot_sync(kFull, jsel >= 0);
  if (has == 0u) {
    above_sel = above;
    return -1;
  }
  const int L = 31 - __clz(has);
  above_sel = __shfl_sync(kFull, asel, L);
  return __shfl_sync(kFull, jsel, L);
}

// Group-wide sums over kN threads (kN = 32: one warp, no shared memory; kN = kTT: the CTA, in warp
// order so the sums are the same every run). Every thread of the group calls; every one gets them.
template <int kN>
__device__ __forceinline__ void group_sum2(TShared& sm, unsigned long long& a, unsigned long long& b,
                                           int lane, int warp) {
  a = warp_sum(a);
  b = warp_sum(b);
  if (kN == 32) return;
  if (lane == 0) {
    sm.redm[warp] = a;
    sm.redm2[warp] = b;
  }
  __syncthreads();
  a = 0;
  b = 0;
#pragma unroll 8
  for (int w = 0; w < kTW; ++w) {
    a += sm.redm[w];
    b += sm.redm2[w];
  }
  __syncthreads();
}

__device__ __forceinline__ void block_sum2(TShared& sm, unsigned long long& a, unsigned long long& b,
                                           int lane, int warp) {
  group_sum2<kTT>(sm, a, b, lane, warp);
}

template <int kN>
__device__ __forceinline__ void group_sync() {
  if (kN == 32) {
    __syncwarp();
  } else {
    __syncthreads();
  }
}

template <bool BF16>
struct RowCtx {
  const uint4* rv;
  int nvec;
  float Mk, k;
  int topk;
  float topp;
  bool kon, pon;
};

// ---- radix levels over the candidate list (fast path), by a group of kN threads ----
// Candidates that take part: class test `in_set` and key >= kmin. Counts (and masses) per
// sub-range of 2^shift keys inside [kl, kl + 2^(shift + 8)).
template <int kN, bool BF16, typename InSet>
__device__ __forceinline__ void cand_level(TShared& sm, const float* cand, int nc, uint32_t kl,
                                           int shift, uint32_t kmin, bool masses, float Mk, float k,
                                           InSet in_set, int tid) {
  for (int j = tid; j < 256; j += kN) {
    sm.rc[j] = 0u;
    sm.rm[j] = 0ull;
  }
  group_sync<kN>();
  // At the last level a sub-range is one key, and every logit of a key has the same mass: the
  // sub-range's mass is its count times that mass (the same integer as the sum), no atomics.
  const bool by_key = masses && shift == 0;
  const unsigned long long span = 256ull << shift;
  for (int i = tid; i < nc; i += kN) {
    const float z = cand[i];
    const uint32_t key = order_key<BF16>(z);
    const unsigned long long off = static_cast<unsigned long long>(key) - kl;
    if (key >= kl && off < span && key >= kmin && in_set(z)) {
      const int s = static_cast<int>(off >> shift);
      atomicAdd(&sm.rc[s], 1u);
      if (masses && !by_key) atomicAdd(&sm.rm[s], fix_mass(z, Mk, k));
    }
  }
  group_sync<kN>();
  if (by_key) {
    for (int j = tid; j < 256; j += kN) {
      const unsigned c = sm.rc[j];
      if (c != 0u) sm.rm[j] = static_cast<unsigned long long>(c) * fix_mass(key_value<BF16>(kl + j), Mk, k);
    }
    group_sync<kN>();
  }
}

// The first radix shift for keys in [lo, hi]: levels of 8 bits from lo cover the span (one level
// when it spans fewer than 256 keys).
__device__ __forceinline__ int radix_shift0(uint32_t lo, uint32_t hi) {
  const uint32_t span = hi > lo ? hi - lo : 0u;
  const int bits = span ? 32 - __clz(span) : 0;
  return bits <= 8 ? 0 : 8 * ((bits + 7) / 8) - 8;
}

// The k-th largest key among the candidates in the set (rank k counted from the top).
// Every candidate key lies in [lo, hi].
template <int kN, bool BF16, typename InSet>
__device__ uint32_t cand_kth(TShared& sm, const float* cand, int nc, int rank, uint32_t lo,
                             uint32_t hi, float Mk, float k, InSet in_set, int tid, int lane,
                             int warp) {
  uint32_t kl = lo;
  for (int shift = radix_shift0(lo, hi); shift >= 0; shift -= 8) {
    cand_level<kN, BF16>(sm, cand, nc, kl, shift, 0u, false, Mk, k, in_set, tid);
    int s = 0, r2 = rank;
    if (warp == 0) {
      unsigned before = 0, total = 0;
      s = warp_first_reach<8, true, unsigned>(sm.rc, 255, static_cast<unsigned>(rank), lane, before,
                                              total);
      s = s < 0 ? 0 : s;
      r2 = rank - static_cast<int>(before);
      if (kN != 32 && lane == 0) {
        sm.bi[4] = s;
        sm.bi[5] = r2;
      }
    }
    if (kN != 32) {
      __syncthreads();
      s = sm.bi[4];
      r2 = sm.bi[5];
      __syncthreads();
    }
    kl += static_cast<uint32_t>(s) << shift;
    rank = r2;
  }
  return kl;
}

// The smallest key (>= kmin, in the set) whose strictly-larger mass, plus `base`, stays below
// `target`. The set's keys lie in [kmin, hi].
template <int kN, bool BF16, typename InSet>
__device__ uint32_t cand_topp(TShared& sm, const float* cand, int nc, uint32_t kmin, uint32_t hi,
                              unsigned long long base, double target, float Mk, float k,
                              InSet in_set, int tid, int lane, int warp) {
  uint32_t kl = kmin;
  unsigned long long above = base;
  for (int shift = radix_shift0(kmin, hi); shift >= 0; shift -= 8) {
    cand_level<kN, BF16>(sm, cand, nc, kl, shift, kmin, true, Mk, k, in_set, tid);
    int s = 0;
    unsigned long long asel = above;
    if (warp == 0) {
      s = warp_last_below(sm.rc, sm.rm, above, target, lane, asel);
      s = s < 0 ? 0 : s;
      if (kN != 32 && lane == 0) {
        sm.bi[6] = s;
        sm.bm[2] = asel;
      }
    }
    if (kN != 32) {
      __syncthreads();
      s = sm.bi[6];
      asel = sm.bm[2];
      __syncthreads();
    }
    kl += static_cast<uint32_t>(s) << shift;
    above = asel;
  }
  return kl > kmin ? kl : kmin;
}

// The exact selection on the candidate list by a group of kN threads (one warp for a short list,
// the CTA otherwise). top-k rows: the k-th largest among all candidates, then (top-p) the nucleus of
// the candidates at or above it. top-p rows: the boundary among T (z >= x_t) or among C (z < x_a)
// with base mass mT + mA, as the caller decided. Returns the threshold key.
template <int kN, bool BF16>
__device__ uint32_t cand_solve(TShared& sm, const float* cand, int nc, bool kon, bool pon, int topk,
                               float topp, int where, unsigned long long base, double target_p,
                               float x_t, float x_a, float x_l, float M, float Mk, float k, int tid,
                               int lane, int warp) {
  const uint32_t kM = order_key<BF16>(M);                // the largest key of the row
  if (kon) {
    auto all = [](float) { return true; };
    const uint32_t kth = cand_kth<kN, BF16>(sm, cand, nc, topk, order_key<BF16>(x_t), kM, Mk, k,
                                            all, tid, lane, warp);
    if (!pon) return kth;
    unsigned long long km = 0, unused = 0;
    for (int j = tid; j < nc; j += kN) {
      const float z = cand[j];
      if (order_key<BF16>(z) >= kth) km += fix_mass(z, Mk, k);
    }
    group_sum2<kN>(sm, km, unused, lane, warp);
    const double target = static_cast<double>(topp) * static_cast<double>(km);
    return cand_topp<kN, BF16>(sm, cand, nc, kth, kM, 0ull, target, Mk, k, all, tid, lane, warp);
  }
  if (where == 0) {
    auto in_t = [=](float z) { return z >= x_t; };
    return cand_topp<kN, BF16>(sm, cand, nc, order_key<BF16>(x_t), kM, 0ull, target_p, Mk, k, in_t,
                               tid, lane, warp);
  }
  auto in_c = [=](float z) { return z < x_a; };
  const uint32_t ka = order_key<BF16>(x_a);
  return cand_topp<kN, BF16>(sm, cand, nc, order_key<BF16>(x_l), ka > 0u ? ka - 1u : 0u, base,
                             target_p, Mk, k, in_c, tid, lane, warp);
}

// ---- the exact path over the whole row ----
template <bool BF16>
__device__ __noinline__ uint32_t exact_row(TShared& sm, unsigned char* dyn, const RowCtx<BF16> R,
                                           int tid, int lane, int warp) {
  constexpr int E = BF16 ? 8 : 4;
  constexpr int kKeyBits = BF16 ? 16 : 32;
  unsigned long long* wm = reinterpret_cast<unsigned long long*>(dyn);                 // [kTW][kL0]
  unsigned* wc = reinterpret_cast<unsigned*>(dyn + kTW * kL0 * 8);                    // [kTW][kL0]
  const float Mk = R.Mk, k = R.k;
  const bool kon = R.kon, pon = R.pon;

  for (int j = lane; j < kL0; j += 32) {
    wc[warp * kL0 + j] = 0u;
    wm[warp * kL0 + j] = 0ull;
  }
  __syncwarp();
  unsigned tail_c = 0;
  unsigned long long tail_m = 0;
  for (int u = tid; u < R.nvec; u += kTT) {
    const uint4 v = ld_stream_v4(R.rv + u);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float z = vec_get<BF16>(v, e);
      const int bin = d_bin(z, Mk, k, kL0PerLog2, kL0);
      if (bin < kL0) {
        atomicAdd(&wc[warp * kL0 + bin], 1u);
        if (pon) atomicAdd(&wm[warp * kL0 + bin], fix_mass(z, Mk, k));
      } else {
        ++tail_c;
        if (pon) tail_m += fix_mass(z, Mk, k);
      }
    }
  }
  tail_c = __reduce_add_sync(kFull, tail_c);
  tail_m = warp_sum(tail_m);
  if (lane == 0) {
    sm.redu[warp] = tail_c;
    sm.redm[warp] = tail_m;
  }
  __syncthreads();
  for (int j = tid; j < kL0; j += kTT) {     // warp order: the same sums every run
    unsigned c = 0;
    unsigned long long m = 0;
    for (int w = 0; w < kTW; ++w) {
      c += wc[w * kL0 + j];
      m += wm[w * kL0 + j];
    }
    sm.c0[j] = c;
    sm.m0[j] = m;
  }
  if (tid == 0) {
    unsigned c = 0;
    unsigned long long m = 0;
    for (int w = 0; w < kTW; ++w) {
      c += sm.redu[w];
      m += sm.redm[w];
    }
    sm.c0[kL0] = c;
    sm.m0[kL0] = m;
  }
  __syncthreads();

  // One radix level over the row's logits in level-0 bin `bin` with key in [kl, kl + 2^(shift+8))
  // and key >= kmin.
  auto radix_level = [&](int bin, uint32_t kl, int shift, uint32_t kmin, bool masses) {
    for (int j = tid; j < 256; j += kTT) {
      sm.rc[j] = 0u;
      sm.rm[j] = 0ull;
    }
    __syncthreads();
    const unsigned long long span = 256ull << shift;
    for (int u = tid; u < R.nvec; u += kTT) {
      const uint4 v = ld_stream_v4(R.rv + u);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float z = vec_get<BF16>(v, e);
        const uint32_t key = order_key<BF16>(z);
        const unsigned long long off = static_cast<unsigned long long>(key) - kl;
        if (key >= kl && off < span && key >= kmin && d_bin(z, Mk, k, kL0PerLog2, kL0) == bin) {
          const int s = static_cast<int>(off >> shift);
          atomicAdd(&sm.rc[s], 1u);
          if (masses) atomicAdd(&sm.rm[s], fix_mass(z, Mk, k));
        }
      }
    }
    __syncthreads();
  };
  const int shift0 = kKeyBits - 8;

  // K: the k-th largest logit (its key) and the mass at or above it.
  uint32_t kth_key = 0;
  unsigned long long kept_mass = 0;
  int kbin = kL0;
  unsigned long long kbin_mass = 0;
  if (kon) {
    if (tid == 0) {
      unsigned cum = 0;
      int bsel = kL0;
      for (int j = 0; j <= kL0; ++j) {
        if (cum + sm.c0[j] >= static_cast<unsigned>(R.topk)) {
          bsel = j;
          break;
        }
        cum += sm.c0[j];
      }
      sm.bi[0] = bsel;
      sm.bi[1] = R.topk - static_cast<int>(cum);
    }
    __syncthreads();
    kbin = sm.bi[0];
    int rank = sm.bi[1];
    __syncthreads();
    uint32_t kl = 0;
    unsigned long long above = 0;
    for (int shift = shift0; shift >= 0; shift -= 8) {
      radix_level(kbin, kl, shift, 0u, pon);
      if (tid == 0) {
        unsigned cum = 0;
        int s = 0;
        for (int j = 255; j >= 0; --j) {
          if (cum + sm.rc[j] >= static_cast<unsigned>(rank)) {
            s = j;
            break;
          }
          cum += sm.rc[j];
          above += sm.rm[j];
        }
        sm.bi[2] = s;
        sm.bi[3] = rank - static_cast<int>(cum);
        sm.bm[0] = above;
        sm.bm[1] = sm.rm[s];
      }
      __syncthreads();
      const int s = sm.bi[2];
      rank = sm.bi[3];
      above = sm.bm[0];
      kl += static_cast<uint32_t>(s) << shift;
      if (shift == 0) kbin_mass = above + sm.bm[1];
      __syncthreads();
    }
    kth_key = kl;
    if (pon) {
      unsigned long long m = kbin_mass;
      for (int j = 0; j < kbin; ++j) m += sm.m0[j];
      kept_mass = m;
    }
  } else if (pon) {
    unsigned long long m = 0;
    for (int j = 0; j <= kL0; ++j) m += sm.m0[j];
    kept_mass = m;
  }

  // P: the smallest key whose strictly-larger mass stays below top_p times the kept mass.
  uint32_t tau_key = kth_key;
  if (pon) {
    const double target = static_cast<double>(R.topp) * static_cast<double>(kept_mass);
    if (tid == 0) {
      unsigned long long A = 0, A_sel = 0;
      int psel = -1;
      const int last = kon ? kbin : kL0;
      for (int j = 0; j <= last; ++j) {
        const unsigned long long mj = (kon && j == kbin) ? kbin_mass : sm.m0[j];
        if (sm.c0[j] == 0u) continue;
        if (static_cast<double>(A) < target) {
          psel = j;
          A_sel = A;
          A += mj;
        } else {
          break;
        }
      }
      sm.bi[2] = psel;
      sm.bm[0] = A_sel;
    }
    __syncthreads();
    const int pbin = sm.bi[2];
    unsigned long long above = sm.bm[0];
    __syncthreads();
    const uint32_t kmin = (kon && pbin == kbin) ? kth_key : 0u;
    uint32_t kl = 0;
    for (int shift = shift0; shift >= 0; shift -= 8) {
      radix_level(pbin, kl, shift, kmin, true);
      if (warp == 0) {
        unsigned long long asel = 0;
        const int s = warp_last_below(sm.rc, sm.rm, above, target, lane, asel);
        if (lane == 0) {
          sm.bi[3] = s < 0 ? 0 : s;
          sm.bm[1] = asel;
        }
      }
      __syncthreads();
      kl += static_cast<uint32_t>(sm.bi[3]) << shift;
      above = sm.bm[1];
      __syncthreads();
    }
    tau_key = kl > kth_key ? kl : kth_key;
  }
  return tau_key;
}

// Pass 2 over the row: candidates (cut points of class_words) appended to `cand` in shared memory
// (warp-aggregated: one atomic per warp and vector step with a candidate), and (kP) the thread's
// fp32 sum of the masses between the cut points; kMax: also the thread's max (NaN-propagating) in
// mx; cidx (or null): each candidate's logit index, for the first kIdxMax candidates. Every thread
// calls it with the same trip count.
template <bool BF16, bool kP, bool kMax>
__device__ __forceinline__ float pass2(TShared& sm, float* cand, int* cidx, const uint4* rv,
                                       int nvec, float xt, float xa, float xl, float Mk, float k,
                                       uint64_t pol, int tid, int lane, float& mx) {
  constexpr int E = BF16 ? 8 : 4;
  float s_a = 0.0f;
  static_assert(kU * E <= 32, "one bit per logit of a step in a word");
  const f32x2 k2 = pk(k, k), c2 = pk(-Mk, -Mk);
  uint32_t pmx = 0xFF80FF80u;                       // bf16: the running max of both halves (-inf)
  // One step of kU vectors per thread; a full step (every vector inside the row, all but the
  // row's last step) skips the bounds checks.
  auto step = [&](int u0, auto full_tag) {
    constexpr bool kAll = decltype(full_tag)::value;
    uint4 vv[kU];
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const int u = u0 + j * kTT + tid;
      if (kAll) {
        vv[j] = ld_pol_v4(rv + u, pol);
      } else {
        vv[j] = make_uint4(0u, 0u, 0u, 0u);
        if (u < nvec) vv[j] = ld_pol_v4(rv + u, pol);
      }
    }
    unsigned bits = 0;                              // bit j*E + e: logit e of vector j is a candidate
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const bool in = kAll || u0 + j * kTT + tid < nvec;
      const uint4 v = vv[j];
      uint32_t cw[4], aw[4];
      if (kMax && in) {
        if (BF16) pmx = bmax2_nan(pmx, bmax2_nan(bmax2_nan(v.x, v.y), bmax2_nan(v.z, v.w)));
        else mx = max_nan(mx, vec_max<BF16>(v));
      }
      class_words<BF16, kP>(v, xt, xa, xl, cw, aw);
      if (in && (cw[0] | cw[1] | cw[2] | cw[3]) != 0u) bits |= word_bits<BF16>(cw) << (j * E);
      if (kP && in && (aw[0] | aw[1] | aw[2] | aw[3]) != 0u) {
        // Two logits per packed step; a logit outside A adds zero.
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        f32x2 sa = pk(0.0f, 0.0f);
#pragma unroll
        for (int q = 0; q < 4; q += BF16 ? 1 : 2) {
          float a0, a1;
          bool in0, in1;
          if (BF16) {
            upk(fma2(pk(bf_lo(w[q]), bf_hi(w[q])), k2, c2), a0, a1);
            in0 = (aw[q] & 0xffffu) != 0u;
            in1 = (aw[q] >> 16) != 0u;
          } else {
            upk(fma2(pk(__uint_as_float(w[q]), __uint_as_float(w[q + 1])), k2, c2), a0, a1);
            in0 = aw[q] != 0u;
            in1 = aw[q + 1] != 0u;
          }
          sa = add2(sa, pk(in0 ? ex2(a0) : 0.0f, in1 ? ex2(a1) : 0.0f));
        }
        float s0, s1;
        upk(sa, s0, s1);
        s_a += s0 + s1;
      }
    }
    if (__any_sync(kFull, bits != 0u)) {            // append the step's candidates, once a warp
      const int c = __popc(bits);
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
      }
      unsigned pos0 = 0;
      if (lane == 31) pos0 = atomicAdd(&sm.ncand, static_cast<unsigned>(incl));
      pos0 = __shfl_sync(kFull, pos0, 31);
      unsigned pos = pos0 + static_cast<unsigned>(incl - c);
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        unsigned bj = (bits >> (j * E)) & ((1u << E) - 1u);
        const int ubase = (u0 + j * kTT + tid) * E;
        while (bj != 0u) {
          const int e = __ffs(bj) - 1;
          bj &= bj - 1u;
          if (pos < static_cast<unsigned>(kCandMax)) cand[pos] = vec_get<BF16>(vv[j], e);
          if (cidx != nullptr && pos < static_cast<unsigned>(kIdxMax)) cidx[pos] = ubase + e;
          ++pos;
        }
      }
    }
  };
  int u0 = 0;
  for (; u0 + kTT * kU <= nvec; u0 += kTT * kU) step(u0, std::true_type{});
  if (u0 < nvec) step(u0, std::false_type{});
  if (kMax && BF16) mx = max_nan(mx, max_nan(bf_lo(pmx), bf_hi(pmx)));
  return s_a;
}

// rows: null, or a zeroed counter from which CTAs claim rows one at a time (rows differ in cost by
// a few times); without it, CTA c takes rows c, c + gridDim.x, ...
// lists / list_n: see launch_threshold.
template <bool BF16>
__global__ void __launch_bounds__(kTT, kCtasT) sv_threshold_kernel(const Params P, float* tau,
                                                              unsigned* rows, int2* lists,
                                                              int* list_n) {
  __shared__ TShared sm;
  extern __shared__ __align__(16) unsigned char dyn_t[];
  uint4* samp = reinterpret_cast<uint4*>(dyn_t);
  float* cand = reinterpret_cast<float*>(dyn_t + kSampleBytes);
  constexpr size_t ES = BF16 ? 2 : 4;
  constexpr int E = BF16 ? 8 : 4;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = P.B, G = P.G, V = P.V;
  const int ntarget = B * (G + 1);
  const int nrows = ntarget + B * G;
  const int nvec = static_cast<int>(static_cast<size_t>(V) * ES / 16);
  const size_t Vs = static_cast<size_t>(V);
  const uint64_t keep = l2_policy_evict_last();
  const uint64_t first = l2_policy_evict_first();
  // Sampled vectors: every sstride-th (a power of two >= 16), at most kSampleVecs of them.
  int sstride = 16;
  while ((nvec + sstride - 1) / sstride > kSampleVecs) sstride *= 2;
  const int nsv = (nvec + sstride - 1) / sstride;

  int nclaim = 0;
  // The next row: claimed by thread 0 into one of two slots (a slot is rewritten only after every
  // thread has passed the barrier that follows its next claim).
  auto next_row = [&](int r) -> int {
    if (rows == nullptr) return r + static_cast<int>(gridDim.x);
    const int slot = nclaim++ & 1;
    if (tid == 0) sm.claim[slot] = static_cast<int>(atomicAdd(rows, 1u));
    __syncthreads();
    return sm.claim[slot];
  };
  for (int r = rows ? next_row(0) : static_cast<int>(blockIdx.x); r < nrows; r = next_row(r)) {
    // ---- which row, and does a filter touch it ----
    const bool draft = r >= ntarget;
    const int b = draft ? (r - ntarget) / G : r / (G + 1);
    const int i = draft ? (r - ntarget) % G : r % (G + 1);
    const int gb = P.draft_len ? __ldg(P.draft_len + b) : G;
    const float T = __ldg(P.temperature + b);
    const int topk = P.top_k ? __ldg(P.top_k + b) : 0;
    const float topp = P.top_p ? __ldg(P.top_p + b) : 1.0f;
    const bool kon = topk > 0 && topk < V;
    const bool pon = topp < 1.0f;
    const bool read = gb >= 0 && gb <= G && (draft ? i < gb : i <= gb);
    const bool sampled = T >= FLT_MIN && T <= FLT_MAX;
    if (!(read && sampled && (kon || pon) && topp > 0.0f)) {
      if (tid == 0) tau[r] = -INFINITY;
      continue;
    }
    const char* row = draft ? static_cast<const char*>(P.zd) + ((size_t)b * G + i) * Vs * ES
                            : static_cast<const char*>(P.zt) + ((size_t)b * (G + 1) + i) * Vs * ES;
    RowCtx<BF16> R;
    R.rv = reinterpret_cast<const uint4*>(row);
    R.nvec = nvec;
    R.k = kLog2e / T;
    R.topk = topk;
    R.topp = topp;
    R.kon = kon;
    R.pon = pon;
    const float k = R.k;

    // ---- 1: the sample, and for top-p over the whole row also the row max and mass ----
    // Top-k rows read only every fourth sampled vector here (k's share needs few; the row max comes
    // with the candidates in pass 2). Top-p rows read the whole row: the max, the sample and the
    // mass, summed kU vectors at a time against the thread's running max m_run (the sum rescaled
    // when m_run grows; packed pairs, as in the streaming kernel's pass 1).
    const bool pmass = pon && !kon;
    const int nsamp = pmass ? nsv : (nvec + 4 * sstride - 1) / (4 * sstride);
    float mx = -INFINITY, m_run = -INFINITY;
    f32x2 s_run = pk(0.0f, 0.0f);
    if (!pmass) {
      for (int s2 = tid; s2 < nsamp; s2 += kTT) {
        const uint4 v = ld_pol_v4(R.rv + s2 * 4 * sstride, keep);
        samp[s2] = v;
        mx = max_nan(mx, vec_max<BF16>(v));
      }
    }
    // Full steps (every vector inside the row) skip the bounds checks.
    auto mass_step = [&](int u0, auto full_tag) {
      constexpr bool kAll = decltype(full_tag)::value;
      constexpr uint32_t ninf = BF16 ? 0xFF80FF80u : 0xFF800000u;
      uint4 v[kU];
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int u = u0 + j * kTT;
        v[j] = (kAll || u < nvec) ? ld_pol_v4(R.rv + u, keep) : make_uint4(ninf, ninf, ninf, ninf);
      }
      online_update_batch<BF16, kU>(v, k, m_run, s_run, mx);
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int u = u0 + j * kTT;
        if ((kAll || u < nvec) && (u & (sstride - 1)) == 0) samp[u / sstride] = v[j];
      }
    };
    if (pmass) {
      int u0 = tid;
      for (; u0 - tid + kTT * kU <= nvec; u0 += kTT * kU) mass_step(u0, std::true_type{});
      if (u0 - tid < nvec) mass_step(u0, std::false_type{});
    }
    mx = warp_max_nan(mx);
    if (lane == 0) sm.redf[warp] = mx;
    for (int j = tid; j <= kFB; j += kTT) {
      sm.fc[j] = 0u;
      sm.fd[j] = 0u;
    }
    __syncthreads();
    float M = -INFINITY;                     // top-k rows: the sample's max
#pragma unroll 8
    for (int w = 0; w < kTW; ++w) M = max_nan(M, sm.redf[w]);
    const bool m_ok = M > -INFINITY && M < INFINITY;
    if (pmass && !m_ok) {        // NaN, +inf or only -inf: the streaming kernel's row error
      if (tid == 0) tau[r] = -INFINITY;
      __syncthreads();
      continue;
    }
    float Mk = M * k;
    R.Mk = Mk;
    // The row's mass relative to M, in fixed point (every thread gets it).
    unsigned long long S = 0, unused0 = 0;
    if (pmass) {
      float s0, s1;
      upk(s_run, s0, s1);
      const float sc = m_run > -INFINITY ? (s0 + s1) * ex2((m_run - M) * k) : 0.0f;
      S = __float2ull_rn(sc * kFix);
      block_sum2(sm, S, unused0, lane, warp);
    }

    // ---- 2: the sample's fine-bin histogram and the window ----
    for (int s = tid; m_ok && s < nsamp; s += kTT) {
      const uint4 v = samp[s];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float z = vec_get<BF16>(v, e);
        const int bin = d_bin(z, Mk, k, kFBPerLog2, kFB);
        atomicAdd(&sm.fc[bin], 1u);
        if (pmass && bin < kFB) {
          // A logit of bin b has w in (2^-(b+1)/8, 2^-b/8]: its mass is 2^-(b+1)/8 (1 + delta),
          // delta in [0, 2^(1/8) - 1], summed in 16-bit fixed point (a bin of 16,384 sampled logits
          // stays below 2^27). Native 32-bit atomics; the bin's mass is rebuilt from the two sums.
          const float e = fmaf(z, k, -Mk) + static_cast<float>(bin + 1) / kFBPerLog2;
          const float dlt = fminf(fmaxf(ex2(e) - 1.0f, 0.0f), 0.125f);
          atomicAdd(&sm.fd[bin], __float2uint_rn(dlt * 65536.0f));
        }
      }
    }
    __syncthreads();
    if (warp == 0) {
      // Logits a sampled logit stands for.
      const float f = static_cast<float>(nvec) / static_cast<float>(nsamp);
      int b_t, b_c, b_lo;
      unsigned est = 0;
      unsigned before = 0, total = 0;
      if (kon) {
        // Down to where the sample holds k's share plus three deviations and three more (more
        // than that many sampled logits among the top k has a chance near 1e-4; the check after
        // pass 2 sends such a row to the exact path).
        const float ks = static_cast<float>(topk) / f;
        const unsigned want = static_cast<unsigned>(ceilf(ks + 3.0f * sqrtf(ks) + 3.0f));
        const int j = warp_first_reach<16, false, unsigned>(sm.fc, 0, want, lane, before, total);
        b_lo = j < 0 ? kFB : j;
        est = j < 0 ? total + sm.fc[kFB] : before + sm.fc[j];
        b_t = b_lo;
        b_c = b_lo + 1;
      } else {
        // T: the bins holding the sample's top eight logits.
        const int j = warp_first_reach<16, false, unsigned>(sm.fc, 0, 8u, lane, before, total);
        b_t = j < 0 ? kFB : j;
        const unsigned cnt_t = j < 0 ? total + sm.fc[kFB] : before + sm.fc[j];
        // The mass of the bins below b estimated from the sample, m_lo(b) = f * (sample mass of
        // the bins >= b), with its standard deviation sqrt(f (f - 1) * sample squared mass), gives
        // est_above(b) = S - m_lo(b). A: bins < b_c, the largest b_c with est_above + 5 sd below
        // top_p * S; C ends at b_lo, the smallest with est_above(b_lo + 1) - 5 sd at or above it.
        // Masses in units of the max's: the row's S, the sample's per bin.
        const float Sf = static_cast<float>(S) * (1.0f / kFix);
        const float target = topp * Sf;
        auto bin_mass = [&](int bb) {
          return ex2(-static_cast<float>(bb + 1) / kFBPerLog2) *
                 (static_cast<float>(sm.fc[bb]) + static_cast<float>(sm.fd[bb]) * (1.0f / 65536.0f));
        };
        // Squared masses bounded by mass times the bin's largest weight 2^(-b/8). The tail bin's
        // logits (w < 2^-64) add nothing.
        float tm = 0.0f, tm2 = 0.0f;
        for (int i2 = 0; i2 < 16; ++i2) {
          const int bb = lane * 16 + i2;
          const float mb = bin_mass(bb);
          tm += mb;
          tm2 += mb * ex2(-static_cast<float>(bb) / kFBPerLog2);
        }
        // Sample mass of the bins >= this lane's first bin: the lanes above.
        float sfx = tm, sfx2 = tm2;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_down_sync(kFull, sfx, o);
          const float y2 = __shfl_down_sync(kFull, sfx2, o);
          if (lane + o < 32) {
            sfx += y;
            sfx2 += y2;
          }
        }
        // Variances: f (f - 1) times the sample's squared masses.
        const float ffk = f * (f - 1.0f);
        // est_above(b) and 5 sd(b) from the sample masses of the bins >= b, once per bin (the
        // margin needs no correctly rounded square root). Bin b decides b_c with its own pair and
        // b_lo for bin b - 1.
        int bc_l = -1, blo_l = kFB;
        float sb = sfx, sb2 = sfx2;                  // sample mass of bins >= lane * 16 + i2
        for (int i2 = 0; i2 <= 16; ++i2) {
          const int bb = lane * 16 + i2;
          const float ea = Sf - f * fmaxf(sb, 0.0f);
          const float sd = 5.0f * sqrt_approx(ffk * fmaxf(sb2, 0.0f));
          if (i2 > 0 && blo_l == kFB && ea - sd >= target) blo_l = bb - 1;   // bins <= bb - 1 reach it
          if (i2 == 16) break;
          if (ea + sd <= target) bc_l = bb;          // A = bins < bb stays below the target
          const float mb = bin_mass(bb);
          sb -= mb;
          sb2 -= mb * ex2(-static_cast<float>(bb) / kFBPerLog2);
        }
        const unsigned hc = __ballot_sync(kFull, bc_l >= 0);
        b_c = hc ? __shfl_sync(kFull, bc_l, 31 - __clz(hc)) : 0;
        const unsigned hl = __ballot_sync(kFull, blo_l < kFB);
        b_lo = hl ? __shfl_sync(kFull, blo_l, __ffs(hl) - 1) : kFB;
        if (b_c <= b_t) b_c = b_t + 1;
        if (b_lo < b_c) b_lo = b_c - 1;          // C empty: the boundary is estimated inside T
        // The sample's logits in C.
        unsigned cc = 0;
        for (int jj = b_c + lane; jj <= b_lo; jj += 32) cc += sm.fc[jj];
        cc = __reduce_add_sync(kFull, cc);
        est = cnt_t + cc;
      }
      if (lane == 0) {
        // Cut points: the lower value edge of a bin, M - (b + 1) / (8 k), in the storage type
        // (-inf for the tail bin); the classes of pass 2 and of the selection are these compares.
        auto edge = [&](int bb) {
          return bb >= kFB ? -INFINITY
                           : store_floor<BF16>(M - static_cast<float>(bb + 1) / (kFBPerLog2 * k));
        };
        sm.bx[0] = edge(b_t);
        sm.bx[1] = edge(b_c - 1);
        sm.bx[2] = edge(b_lo);
        sm.bi[0] = b_t;
        sm.bi[1] = b_c;
        sm.bi[2] = b_lo;
        // The fast path; a top-k row whose sample max is not finite takes the exact path (the
        // main pass then collects nothing).
        const bool fast_row = m_ok && static_cast<float>(est) * f <= 0.6f * kCandMax;
        sm.bi[3] = fast_row;
        if (!fast_row) sm.bx[0] = sm.bx[1] = sm.bx[2] = INFINITY;
        sm.ncand = 0u;
      }
    }
    __syncthreads();
    const float x_t = sm.bx[0], x_a = sm.bx[1], x_l = sm.bx[2];
    bool fast = sm.bi[3] != 0;
    __syncthreads();

    uint32_t tau_key = 0;
    if (!pmass) {
      // ---- 3 (top-k rows): the row max and the candidates in one pass ----
      float m2 = -INFINITY;
      pass2<BF16, false, true>(sm, cand, lists ? reinterpret_cast<int*>(samp) : nullptr, R.rv,
                               nvec, x_t, x_t, x_t, Mk, k, first, tid, lane, m2);
      m2 = warp_max_nan(m2);
      if (lane == 0) sm.redf[warp] = m2;
      __syncthreads();
      M = -INFINITY;
#pragma unroll 8
      for (int w = 0; w < kTW; ++w) M = max_nan(M, sm.redf[w]);
      if (!(M > -INFINITY && M < INFINITY)) {   // NaN, +inf or only -inf: a row error
        if (tid == 0) tau[r] = -INFINITY;
        __syncthreads();
        continue;
      }
      Mk = M * k;
      R.Mk = Mk;
    }
    if (fast) {
      // ---- 3 (top-p rows): the mass of A, the candidates of T and C ----
      unsigned long long mA = 0, unused1 = 0;
      if (pmass) {
        float unused_mx = 0.0f;
        const float s_a = pass2<BF16, true, false>(sm, cand, nullptr, R.rv, nvec, x_t, x_a, x_l,
                                                   Mk, k, first, tid, lane, unused_mx);
        mA = __float2ull_rn(s_a * kFix);       // per-thread sums in fixed point, then block sums
      }
      block_sum2(sm, mA, unused1, lane, warp);
      const unsigned ncand = sm.ncand;
      const int nc = static_cast<int>(ncand < static_cast<unsigned>(kCandMax) ? ncand : kCandMax);
      fast = ncand <= static_cast<unsigned>(kCandMax);

      // ---- 4: the exact selection on the candidates ----
      int where = 0;                             // top-p rows: the boundary in T (0) or C (1)
      unsigned long long base = 0;
      double target_p = 0.0;
      if (fast && kon) {
        fast = nc >= topk;                       // the k-th largest lies in the window
      } else if (fast) {                         // top-p over the whole row
        unsigned long long mT = 0, mC = 0;
        for (int j = tid; j < nc; j += kTT) {
          const float z = cand[j];
          const unsigned long long w = fix_mass(z, Mk, k);
          if (z >= x_t) {
            mT += w;
          } else {
            mC += w;
          }
        }
        block_sum2(sm, mT, mC, lane, warp);
        target_p = static_cast<double>(topp) * static_cast<double>(S);
        if (static_cast<double>(mT) >= target_p) {                  // the boundary lies in T
          where = 0;
        } else if (static_cast<double>(mT + mA) < target_p &&
                   static_cast<double>(mT + mA + mC) >= target_p) { // ... in C
          where = 1;
          base = mT + mA;
        } else {                                                     // in A, or below the window
          fast = false;
        }
      }
      if (fast) {
        tau_key = cand_solve<kTT, BF16>(sm, cand, nc, kon, pon, topk, topp, where, base, target_p,
                                        x_t, x_a, x_l, M, Mk, k, tid, lane, warp);
      }
      // ---- 5 (top-k rows): the kept set, when it is short, as an (index, logit) list ----
      if (fast && kon && lists != nullptr && nc <= kIdxMax) {
        const int* cidx = reinterpret_cast<const int*>(samp);
        unsigned nk = 0;
        for (int j = tid; j < nc; j += kTT) nk += order_key<BF16>(cand[j]) >= tau_key ? 1u : 0u;
        nk = __reduce_add_sync(kFull, nk);
        if (lane == 0) sm.redu[warp] = nk;
        if (tid == 0) sm.ncand = 0u;             // reused as the list's fill counter
        __syncthreads();
        nk = 0;
#pragma unroll 8
        for (int w = 0; w < kTW; ++w) nk += sm.redu[w];
        if (nk <= static_cast<unsigned>(kList)) {
          int2* out = lists + static_cast<size_t>(r) * kList;
          for (int j = tid; j < nc; j += kTT) {
            const float z = cand[j];
            if (order_key<BF16>(z) >= tau_key) {
              const unsigned pos = atomicAdd(&sm.ncand, 1u);
              out[pos] = make_int2(cidx[j], __float_as_int(z));
            }
          }
          if (tid == 0) list_n[r] = static_cast<int>(nk);
        }
      }
    }
    __syncthreads();
    if (!fast) tau_key = exact_row<BF16>(sm, dyn_t, R, tid, lane, warp);
    if (tid == 0) tau[r] = key_value<BF16>(tau_key);
    __syncthreads();
  }
}

}  // namespace

int threshold_rows(const Params& P) { return P.B * (2 * P.G + 1); }

cudaError_t launch_threshold(const Params& P, bool bf16, float* tau, unsigned* rows, int2* lists,
                             int* list_n, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int nrows = threshold_rows(P);
  const int grid = nrows < kCtasT * sms ? nrows : kCtasT * sms;
  const void* fn = bf16 ? reinterpret_cast<const void*>(sv_threshold_kernel<true>)
                        : reinterpret_cast<const void*>(sv_threshold_kernel<false>);
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynBytesT);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  if (bf16) {
    sv_threshold_kernel<true><<<grid, kTT, kDynBytesT, stream>>>(P, tau, rows, lists, list_n);
  } else {
    sv_threshold_kernel<false><<<grid, kTT, kDynBytesT, stream>>>(P, tau, rows, lists, list_n);
  }
  return cudaGetLastError();
}

}  // namespace sv
