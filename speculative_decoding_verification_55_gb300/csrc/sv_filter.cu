// Filtered verification on sm_103a: top-k and top-p applied to p and q before the test ([R]
// "Speculative decoding", rayaq.ca ml-models -- Why the output is exactly the target's: temperature,
// top-p and any penalties are applied to p and q before the test; the rule then preserves exactly
// the distribution it is given). Rows of 16-byte multiples, 16-byte aligned.
//
// One cluster of C CTAs verifies one position at a time (persistent over positions); CTA r holds the
// r-th chunk of the position's target row (and draft row) in shared memory, loaded once with
// cp.async.bulk, and every pass below runs on that copy:
//   A   the chunk max (and, for a row without filtering, the sum of exp2((z - M) k)); one cluster
//       exchange gives the row max M (greedy rows: the argmax, then the finish).
//   K   top-k: the threshold of the k largest logits, ties at the boundary all kept.
//   P   top-p, on the top-k set: the largest logit whose kept mass at or above it reaches top_p
//       times the mass of the set (tokens with equal logits go together).
//       Both are selections over a total order of the logits, by histogram levels: level 0 bins
//       by f = (M - z) k (8 bins per unit of log2 probability, 32 units, the rest in one bin), a
//       function monotone in z, so the bins are intervals of the order and the mode of a logit
//       distribution spreads over many bins (few shared-memory atomic conflicts); the next levels
//       refine the chosen bin on 8-bit digits of the logit's order key (2 levels for bf16, 4 for
//       fp32), and a selection stops early once the boundary bin is decided whole. Every level is
//       a count and mass histogram per CTA, read across the cluster in rank order, so every CTA
//       sums the same numbers in the same order and takes the same decision. A level's candidates
//       are one interval of floats (kept_threshold finds its ends), so a logit outside it costs
//       two compares.
//   V   the filtered p~ (and q~), a logit kept when z >= the row's smallest kept float: the
//       accept test u < min(1, p~(x)/q~(x)), then the chunk totals of
//       max(0, p~ - q~) and of p~ in one exchange: alpha = 1 - sum max(0, p~ - q~), and the chunk
//       holding the draw's threshold (the residual draw, its fallback to p~, or the bonus draw).
//   D   that CTA scans its chunk in index order (block-wide prefix sum over per-thread runs) and
//       finishes the position; the row's last finished position emits the row (finish_position).
//   L   a position with top-k takes a shorter road first: one count pass over the value bins near
//       the max gives the bin of the k-th largest logit, one pass writes every logit of that bin
//       or above (a superset of the top-k set, typically k plus a few) into a per-CTA list, and
//       when the lists fit, rank 0 gathers them in index order and runs K, P, V and D on them
//       alone while the other CTAs move on (and every CTA starts the next position's copies).
//       Same levels and decisions as the chunk-wide passes.
// With Params::split the kernel takes only the rows that row_unfiltered leaves out; the streaming
// kernel verifies the others in the same call.
// Control flow depends on cluster-wide data only, so every CTA passes the same cluster barriers.
// The bulk-copy wait is bounded; a CTA whose wait gives up reports it in the next exchange, the
// position is marked bad, the status word is set and the cluster stops.

#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kFT = 512;                        // threads per CTA
constexpr int kFW = kFT / 32;
constexpr int kFRowBytes = 65536;               // a row chunk held in shared memory
constexpr int kFRowUnits = kFRowBytes / 16;
constexpr int kBins = 256;
// Per-warp histograms (count and mass per row and bin) beside the two row chunks: a warp's atomics
// only meet its own lanes'.
constexpr int kHistBytes = kFW * 2 * kBins * 8;
constexpr int kFDynBytes = 2 * kFRowBytes + kHistBytes;
constexpr int kCopyPiece = 16384;               // bytes per bulk copy
constexpr float kBinsPerLog2 = 8.0f;            // level-0 resolution
// Top-k rows: the count pass counts the value bins from kHighBin up, and from kLowBin up (logits
// within 24 units of log2 probability of the max) when fewer than k logits lie that high. A
// candidate list holds at most kLCap logits of a row, per CTA and for the whole cluster. A CTA's
// lists (the target list's four arrays, the draft list's one) sit in the upper half of the
// histogram area, which the count-only passes do not use; rank 0's gathered lists in the lower.
constexpr int kLowBin = 64;
constexpr int kHighBin = 192;                   // within 8 units of log2 probability of the max
constexpr int kLCap = 1024;
static_assert(kFW * 2 * kBins * 4 <= kHistBytes / 2, "count histograms exceed half the area");
static_assert(5 * kLCap * 4 <= kHistBytes / 2 && 4 * kLCap * 4 <= kHistBytes / 2,
              "candidate lists exceed half the histogram area");

enum : unsigned { kStatusTimeout = 1u };

// The state of one row's selection (top-k or top-p), kept in shared memory.
struct FSel {
  int act;            // still refining
  int lvl;            // level of the next histogram: 0 value bins, 1.. key digits
  int D0;             // level-0 bin of the boundary
  uint32_t pre;       // key digits chosen so far
  unsigned need;      // top-k: rank of the boundary among the current candidates
  float above;        // mass of the kept logits above the current candidates
  float tau;          // top-p: mass to reach (set at level 0 from the candidates' total)
  int lbD0;           // candidates at or above (lbD0, lbkey) only
  uint32_t lbkey;
  int thD0;           // result: logits at or above (thD0, thkey) are kept
  uint32_t thkey;
  float mass;         // result: their mass, relative to exp2(M k)
};

struct FShared {
  uint64_t bar;                                 // the chunk copies of the current position
  float xrec[2][8];                             // exchange record, by exchange parity
  unsigned hc[2][2][kBins];                     // this CTA's histograms [parity][row][bin]
  float hm[2][2][kBins];
  unsigned gc[2][kBins];                        // the cluster's histograms [row][bin]
  float gm[2][kBins];
  FSel sel[2];
  float redf[kFW][4];
  int redi[kFW][2];
  float bc[16];                                 // broadcast of cluster-wide values
  int bi[16];
  int stop;
  // candidate lists: boundary bins, this CTA's counts, the cluster's offsets and totals, and the
  // thresholds and masses found on the gathered lists
  int lD[2];
  int lnum[2];
  int loff[2][kMaxCluster];
  int ltot[2];
  int lth[2];
  uint32_t lkey[2];
  float lmass[2];
};

struct FPos {
  int b, i, gb;
  float T;
  bool len_ok, t_ok, greedy, load, two;
};

__device__ __forceinline__ FPos fclassify(const Params& P, int s) {
  FPos p;
  p.i = s / P.B;
  p.b = s - p.i * P.B;
  p.gb = P.draft_len ? __ldg(P.draft_len + p.b) : P.G;
  p.T = __ldg(P.temperature + p.b);
  p.len_ok = p.gb >= 0 && p.gb <= P.G;
  p.greedy = (p.T == 0.0f);
  p.t_ok = p.greedy || (p.T >= FLT_MIN && p.T <= FLT_MAX);   // NaN fails both
  p.load = p.len_ok && p.t_ok && p.i <= p.gb;
  p.two = p.load && !p.greedy && p.i < p.gb;
  if (P.split && row_unfiltered(P, p.b)) {    // the streaming kernel's row: no work, no error here
    p.len_ok = p.t_ok = true;
    p.load = p.two = false;
  }
  return p;
}

// Order key of a logit: unsigned order of keys is the order of the values (-0 reads as +0); bf16
// logits keep their 16 significant bits.
template <bool BF16>
__device__ __forceinline__ uint32_t okey(float z) {
  uint32_t b = __float_as_uint(z);
  if ((b << 1) == 0u) b = 0u;
  const uint32_t k = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return BF16 ? (k >> 16) : k;
}

// Level-0 bin: 255 at the max, one bin per 1/8 unit of log2 probability below it, 0 for the rest.
// Non-decreasing in z (each step rounds monotonically).
__device__ __forceinline__ int vbin(float z, float M, float k) {
  const float f = (M - z) * k * kBinsPerLog2;
  return 255 - static_cast<int>(fminf(f, 255.0f));
}

// (bin, key) at or above the threshold (D0, key0) in the lexicographic order.
__device__ __forceinline__ bool at_or_above(int vb, uint32_t key, int D0, uint32_t key0) {
  return vb > D0 || (vb == D0 && key >= key0);
}

// The smallest float whose (value bin, order key) lies at or above (D0, key0). Both are
// non-decreasing in z, so for every z <= M: (vbin(z), okey(z)) >= (D0, key0) exactly when
// z >= the result. One warp: a 32-way search over the order of the floats (about 7 steps). +inf
// when not even M lies that high.
template <bool BF16>
__device__ float kept_threshold(float M, float k, int D0, uint32_t key0, int lane) {
  auto f2k = [](float z) -> uint32_t {
    const uint32_t b = __float_as_uint(z);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  };
  auto k2f = [](uint32_t q) -> float {
    return __uint_as_float((q & 0x80000000u) ? (q & 0x7fffffffu) : ~q);
  };
  auto keep = [&](float z) { return at_or_above(vbin(z, M, k), okey<BF16>(z), D0, key0); };
  if (keep(-INFINITY)) return -INFINITY;
  if (!keep(M)) return INFINITY;
  uint32_t lo = f2k(-INFINITY), hi = f2k(M);    // keep(lo) false, keep(hi) true
  while (hi - lo > 1u) {
    const uint64_t span = hi - lo;
    const uint32_t q = lo + static_cast<uint32_t>(span * static_cast<uint64_t>(lane + 1) / 33u);
    const bool t = q <= lo ? false : (q >= hi ? true : keep(k2f(q)));
    const unsigned m = __ballot_sync(kFull, t);
    const int f = m ? __ffs(m) - 1 : 32;         // the first lane whose point is kept
    const uint32_t qh = __shfl_sync(kFull, q, f < 32 ? f : 31);
    const uint32_t ql = __shfl_sync(kFull, q, f > 0 ? f - 1 : 0);
    if (f < 32) hi = qh;
    if (f > 0) lo = ql;
  }
  return k2f(hi);
}

// The logits a selection level looks at, as an interval [zlo, zhi) of floats (one warp): level 0
// takes every logit at or above the lower bound (lbD0, lbkey); a deeper level takes the level-0 bin
// D0 at or above the bound, with the key digits chosen so far. Each end is a threshold on
// (value bin, order key), both non-decreasing in z.
template <bool BF16, int KB>
__device__ void level_interval(const FSel& S, float M, float k, int lane, float& zlo, float& zhi) {
  if (S.lvl == 0) {
    zlo = kept_threshold<BF16>(M, k, S.lbD0, S.lbkey, lane);
    zhi = INFINITY;
    return;
  }
  const int sp = KB - 8 * (S.lvl - 1);          // the digits chosen so far sit at bits >= sp
  uint32_t klo = 0u;
  uint64_t khi = 1ull << KB;                     // one past the largest key of the bin
  if (S.lvl > 1) {
    klo = S.pre << sp;
    khi = static_cast<uint64_t>(S.pre + 1u) << sp;
  }
  if (S.D0 == S.lbD0 && S.lbkey > klo) klo = S.lbkey;
  zlo = kept_threshold<BF16>(M, k, S.D0, klo, lane);
  if (khi < (1ull << KB)) zhi = kept_threshold<BF16>(M, k, S.D0, static_cast<uint32_t>(khi), lane);
  else zhi = S.D0 == 255 ? INFINITY : kept_threshold<BF16>(M, k, S.D0 + 1, 0u, lane);
}

// Block-wide max (NaN-propagating) and sum of the two rows of a position at once, in warp order
// (one pair of barriers each).
__device__ __forceinline__ void block_max2_nan(float& a, float& b, FShared& sm) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  a = warp_max_nan(a);
  b = warp_max_nan(b);
  if (lane == 0) {
    sm.redf[w][0] = a;
    sm.redf[w][1] = b;
  }
  __syncthreads();
  float ta = -INFINITY, tb = -INFINITY;
#pragma unroll
  for (int j = 0; j < kFW; ++j) {
    ta = max_nan(ta, sm.redf[j][0]);
    tb = max_nan(tb, sm.redf[j][1]);
  }
  __syncthreads();
  a = ta;
  b = tb;
}

__device__ __forceinline__ void block_sum2(float& a, float& b, FShared& sm) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  a = warp_sum_lane0(a);
  b = warp_sum_lane0(b);
  if (lane == 0) {
    sm.redf[w][2] = a;
    sm.redf[w][3] = b;
  }
  __syncthreads();
  float ta = 0.0f, tb = 0.0f;
#pragma unroll
  for (int j = 0; j < kFW; ++j) {
    ta += sm.redf[j][2];
    tb += sm.redf[j][3];
  }
  __syncthreads();
  a = ta;
  b = tb;
}

__device__ __forceinline__ unsigned warp_incl_scan_u(unsigned v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// One decision of a selection (one warp, on the cluster histogram of its row). Lane l owns the
// eight bins 255 - 8l .. 248 - 8l, so lanes run from the largest logits down. count_mode: the bin
// holding the need-th largest candidate; else the first bin with mass whose running mass (from the
// top, plus S.above) reaches S.tau. The owning lane updates S.
template <int KB>
__device__ void decide(FSel& S, const unsigned* gc, const float* gm, bool count_mode, float topp,
                       int lane) {
  constexpr int kLast = KB / 8;
  const int base = 255 - 8 * lane;
  unsigned c[8];
  float m[8];
  unsigned cl = 0u;
  float ml = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    c[j] = gc[base - j];
    m[j] = gm[base - j];
    cl += c[j];
    ml += m[j];
  }
  const unsigned ci = warp_incl_scan_u(cl, lane);
  const float mi = warp_incl_scan(ml, lane);
  const unsigned ce = ci - cl;
  float me = __shfl_up_sync(kFull, mi, 1);
  if (lane == 0) me = 0.0f;
  const int lvl = S.lvl;
  const float above0 = S.above;
  float tau = S.tau;
  if (!count_mode && lvl == 0) tau = topp * __shfl_sync(kFull, mi, 31);

  int D = -1;
  unsigned cum = 0u, cD = 0u;
  float am = 0.0f, mD = 0.0f;
  int owner = 0;
  if (count_mode) {
    const unsigned need = S.need;
    const unsigned hit = __ballot_sync(kFull, ci >= need);
    owner = hit ? __ffs(hit) - 1 : 31;
    if (lane == owner) {
      cum = ce;
      am = me;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (D < 0) {
          if (cum + c[j] >= need || j == 7) {
            D = base - j;
            cD = c[j];
            mD = m[j];
          } else {
            cum += c[j];
            am += m[j];
          }
        }
      }
      am += above0;
    }
  } else {
    const unsigned hit = __ballot_sync(kFull, ml > 0.0f && above0 + mi >= tau);
    if (hit) {
      owner = __ffs(hit) - 1;
      if (lane == owner) {
        float a = above0 + me;
        int jl = 0;
        bool done = false;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (!done && m[j] > 0.0f) {
            jl = j;
            am = a;
            cD = c[j];
            mD = m[j];
            if (a + m[j] >= tau) done = true;      // the crossing bin
            else a += m[j];
          }
        }
        // Without a crossing (the lane's scan rounded past tau) the lane's last bin with mass.
        D = base - jl;
      }
    } else {
      // Rounding left the total below tau: every candidate is kept (the lowest non-empty bin).
      const unsigned ne = __ballot_sync(kFull, cl > 0u);
      owner = ne ? 31 - __clz(ne) : 0;
      if (lane == owner) {
        int jl = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (c[j] > 0u) {
            jl = j;
            cD = c[j];
            mD = m[j];
          }
        float a = above0 + me;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < jl) a += m[j];
        D = base - jl;
        am = a;
      }
    }
  }
  if (lane == owner) {
    const unsigned need2 = count_mode ? S.need - cum : 0u;
    const bool whole = count_mode ? (cD == need2) : (cD <= 1u);
    const uint32_t pre = lvl == 0 ? 0u : ((S.pre << 8) | static_cast<uint32_t>(D));
    if (lvl == kLast || whole) {
      S.act = 0;
      if (lvl == 0) {
        S.thD0 = D;
        S.thkey = 0u;
      } else {
        S.thD0 = S.D0;
        S.thkey = pre << (KB - 8 * lvl);
      }
      S.mass = am + mD;
    } else {
      if (lvl == 0) S.D0 = D;
      S.pre = pre;
      S.lvl = lvl + 1;
      S.need = need2;
      S.above = am;
    }
    S.tau = tau;
  }
}

// A value below which every logit has a value bin below L: vbin is non-decreasing in z and the
// value is checked with vbin itself, so skipping the logits below it skips no logit of bin L or
// above. -inf when no such value is found (nothing is skipped).
__device__ __forceinline__ float cut_below(float M, float k, int L) {
  const float zc = M - static_cast<float>(257 - L) / (k * kBinsPerLog2);
  return (zc == zc && vbin(zc, M, k) < L) ? zc : -INFINITY;
}

// The value bin holding the need-th largest logit, from the cluster's counts (one warp; lane l owns
// the bins 255 - 8l .. 248 - 8l); -1 when the counted bins hold fewer than need logits.
__device__ int boundary_bin(const unsigned* gc, unsigned need, int lane) {
  const int base = 255 - 8 * lane;
  unsigned c[8];
  unsigned cl = 0u;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    c[j] = gc[base - j];
    cl += c[j];
  }
  const unsigned ci = warp_incl_scan_u(cl, lane);
  const unsigned hit = __ballot_sync(kFull, ci >= need);
  if (!hit) return -1;
  const int owner = __ffs(hit) - 1;
  int D = 0;
  if (lane == owner) {
    unsigned cum = ci - cl;
    bool found = false;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (!found) {
        cum += c[j];
        if (cum >= need) {
          D = base - j;
          found = true;
        }
      }
    }
  }
  return __shfl_sync(kFull, D, owner);
}

// The remaining levels of a selection (count mode: top-k; else top-p), from the state in S, by one
// warp over a row's gathered candidates: the levels and decisions of the chunk-wide selection, on
// histograms of the list's entries. Every candidate the remaining levels look at (every logit at
// or above the lower bound (lbD0, lbkey), in the level-0 bin D0 once level 0 is decided) must be on
// the list; other entries are harmless.
template <bool BF16, int KB>
__device__ void list_refine(FSel& S, const float* zl, int n, float M, float k, unsigned* hc,
                            float* hm, bool count_mode, float topp, int lane) {
  while (S.act) {
    for (int j = lane; j < kBins; j += 32) {
      hc[j] = 0u;
      hm[j] = 0.0f;
    }
    __syncwarp();
    const int lvl = S.lvl, D0 = S.D0, lbD0 = S.lbD0;
    const uint32_t pre = S.pre, lbkey = S.lbkey;
    const int sh = KB - 8 * lvl;
    for (int e = lane; e < n; e += 32) {
      const float z = zl[e];
      const int vb = vbin(z, M, k);
      if (lvl == 0 ? vb < lbD0 : vb != D0) continue;
      const uint32_t key = okey<BF16>(z);
      bool cand = vb != lbD0 || key >= lbkey;
      int digit = vb;
      if (lvl > 0) {
        cand = cand && (lvl == 1 || (key >> (sh + 8)) == pre);
        digit = static_cast<int>((key >> sh) & 255u);
      }
      if (cand) {
        atomicAdd(hc + digit, 1u);
        atomicAdd(hm + digit, ex2((z - M) * k));
      }
    }
    __syncwarp();
    decide<KB>(S, hc, hm, count_mode, topp, lane);
    __syncwarp();
  }
}

// A whole selection on a gathered list: the state of level 0 with the lower bound (lbD0, lbkey)
// (a top-p selection on the top-k set takes the top-k threshold), then list_refine.
template <bool BF16, int KB>
__device__ void list_select(FSel& S, const float* zl, int n, float M, float k, unsigned* hc,
                            float* hm, bool count_mode, unsigned need, float topp, int lbD0,
                            uint32_t lbkey, int lane) {
  if (lane == 0) {
    S.act = 1;
    S.lvl = 0;
    S.D0 = 0;
    S.pre = 0u;
    S.need = need;
    S.above = 0.0f;
    S.tau = 0.0f;
    S.lbD0 = lbD0;
    S.lbkey = lbkey;
  }
  __syncwarp();
  list_refine<BF16, KB>(S, zl, n, M, k, hc, hm, count_mode, topp, lane);
}

template <bool BF16>
__global__ void __launch_bounds__(kFT, 1) sv_filter_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ FShared sm;
  constexpr int E = BF16 ? 8 : 4;
  constexpr size_t ES = BF16 ? 2 : 4;
  constexpr int KB = BF16 ? 16 : 32;            // significant bits of the order key

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = static_cast<int>(cluster_rank());
  const int C = P.C, G = P.G, G1 = G + 1;
  const int cid = static_cast<int>(blockIdx.x) / C;
  const int total = P.B * G1;
  const int u0 = min(rank * P.per, P.units);
  const int cu = min(u0 + P.per, P.units) - u0;
  const size_t Vs = static_cast<size_t>(P.V);
  const uint4* dt = reinterpret_cast<const uint4*>(dyn);
  const uint4* dd = reinterpret_cast<const uint4*>(dyn + kFRowBytes);

  if (tid == 0) {
    mbar_init(smem_addr(&sm.bar), 1);
    fence_mbarrier_init_cluster();
    sm.stop = 0;
  }
  __syncthreads();
  cluster_sync_all();

  uint32_t npos = 0;        // positions loaded (the copy barrier's phase)
  uint32_t ex = 0;          // exchanges (record parity)
  bool my_tmo = false;      // this CTA gave up on a copy

  // Exchange: after this returns, peers' records of parity `par` can be read.
  auto publish = [&]() -> uint32_t {
    const uint32_t par = ex & 1;
    ++ex;
    __syncthreads();
    cluster_sync_all();
    return par;
  };
  auto peer = [&](uint32_t par, int field, int r) -> float {
    return ld_cluster_f32(map_to_rank(smem_addr(&sm.xrec[par][field]), static_cast<uint32_t>(r)));
  };

  // Bulk copies of this CTA's chunk of position q's row(s) (thread 0), completing on sm.bar.
  auto issue_copy = [&](const FPos& q) {
    const int nr = q.two ? 2 : 1;
    const uint32_t bytes = static_cast<uint32_t>(cu) * 16;
    mbar_arrive_expect_tx(smem_addr(&sm.bar), bytes * nr);
    const uint64_t once = l2_policy_evict_first();
    for (int r = 0; r < nr; ++r) {
      const char* g = r == 0
          ? static_cast<const char*>(P.zt) + ((size_t)q.b * G1 + q.i) * Vs * ES
          : static_cast<const char*>(P.zd) + ((size_t)q.b * G + q.i) * Vs * ES;
      g += static_cast<size_t>(u0) * 16;
      const uint32_t dst = smem_addr(dyn) + r * kFRowBytes;
      for (uint32_t off = 0; off < bytes; off += kCopyPiece)
        bulk_g2s(dst + off, g + off, min(static_cast<uint32_t>(kCopyPiece), bytes - off),
                 smem_addr(&sm.bar), once);
    }
  };
  int pf = -1;              // thread 0: the position slot whose copies were issued ahead

  for (int s = cid; s < total; s += P.nclusters) {
    if (sm.stop) break;                         // set from exchanged data: the same on every CTA
    const FPos p = fclassify(P, s);
    if (!p.load) {
      if (!(p.len_ok && p.t_ok) && p.i == 0 && rank == 0 && warp == 0) write_row_error(P, p.b, lane);
      continue;
    }
    const int nrows = p.two ? 2 : 1;
    const char* rowt = static_cast<const char*>(P.zt) + ((size_t)p.b * G1 + p.i) * Vs * ES;
    const char* rowd = p.two ? static_cast<const char*>(P.zd) + ((size_t)p.b * G + p.i) * Vs * ES
                             : nullptr;
    // ---- the chunk(s) into shared memory (unless issued ahead) ----
    if (tid == 0) {
      if (pf != s) issue_copy(p);
      pf = -1;
    }
    const bool landed = __syncthreads_and(mbar_wait(smem_addr(&sm.bar), npos & 1)) != 0;
    ++npos;
    if (!landed) {
      my_tmo = true;
      if (tid == 0) atomicOr(P.status, kStatusTimeout);
    }

    const bool ok = row_scalars_ok(P, p.b, p.gb, p.greedy, lane) &&
                    (p.greedy || !P.top_p || __ldg(P.top_p + p.b) > 0.0f);   // NaN fails too
    const int x = p.i < p.gb ? __ldg(P.tokens + (size_t)p.b * G + p.i) : -1;

    if (p.greedy) {
      // ---- greedy: the argmax (lowest index on ties); filtering keeps the argmax ----
      float m = -INFINITY, mx = -INFINITY;
      int idx = INT_MAX;
      if (landed)
        for (int u = tid; u < cu; u += kFT) {
          const uint4 v = dt[u];
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const float z = vec_get<BF16>(v, e);
            mx = max_nan(mx, z);
            if (z > m) {
              m = z;
              idx = (u0 + u) * E + e;
            }
          }
        }
      warp_argmax(m, idx);
      const int wbad = __any_sync(kFull, (mx != mx) || mx == INFINITY);
      if (lane == 0) {
        sm.redf[warp][0] = m;
        sm.redi[warp][0] = idx;
        sm.redi[warp][1] = wbad;
      }
      __syncthreads();
      if (tid == 0) {
        float bm = -INFINITY;
        int bidx = INT_MAX, bb = 0;
        for (int w = 0; w < kFW; ++w) {
          const float wm = sm.redf[w][0];
          const int wi = sm.redi[w][0];
          if (wm > bm || (wm == bm && wi < bidx)) {
            bm = wm;
            bidx = wi;
          }
          bb |= sm.redi[w][1];
        }
        const uint32_t par = ex & 1;
        sm.xrec[par][0] = bm;
        sm.xrec[par][1] = __int_as_float(bidx);
        sm.xrec[par][2] = __int_as_float(bb | (my_tmo ? 2 : 0));
      }
      const uint32_t par = publish();
      if (warp == 0) {
        float v = lane < C ? peer(par, 0, lane) : -INFINITY;
        int ii = lane < C ? __float_as_int(peer(par, 1, lane)) : INT_MAX;
        const int fl = lane < C ? __float_as_int(peer(par, 2, lane)) : 0;
        const bool gbad = __any_sync(kFull, fl & 1);
        const bool gtmo = __any_sync(kFull, fl & 2);
        lanes_argmax(v, ii, 32);
        v = __shfl_sync(kFull, v, 0);
        ii = __shfl_sync(kFull, ii, 0);
        if (lane == 0) sm.stop = gtmo ? 1 : 0;
        if (rank == 0) {
          if (!ok) {
            if (p.i == 0) write_row_error(P, p.b, lane);
          } else {
            const bool bad = gbad || gtmo || !(v > -INFINITY);
            const bool acc = (p.i < p.gb) && (x == ii);
            const float a = acc ? 1.0f : 0.0f;
            finish_position(P, p.b, p.i, p.gb, ii, (bad ? kFlagBad : 0) | (acc ? kFlagAccept : 0),
                            a, a, 1.0f, lane);
          }
        }
      }
      __syncthreads();
      continue;
    }

    // ---- A: chunk max (and the sum when the row is not filtered) ----
    const float k = kLog2e / p.T;
    const int topk = P.top_k ? __ldg(P.top_k + p.b) : 0;
    const float topp = P.top_p ? __ldg(P.top_p + p.b) : 1.0f;
    const bool kon = ok && topk > 0 && topk < P.V;
    const bool pon = ok && topp < 1.0f;
    const bool filt = kon || pon;
    float lm[2] = {-INFINITY, -INFINITY}, ls[2] = {0.0f, 0.0f};
    if (landed) {
      for (int u = tid; u < cu; u += kFT) lm[0] = max_nan(lm[0], vec_max<BF16>(dt[u]));
      if (nrows > 1)
        for (int u = tid; u < cu; u += kFT) lm[1] = max_nan(lm[1], vec_max<BF16>(dd[u]));
    }
    block_max2_nan(lm[0], lm[1], sm);
    int lbad = 0;
#pragma unroll
    for (int r = 0; r < 2; ++r)
      if (r < nrows) lbad |= (lm[r] != lm[r]) || lm[r] == INFINITY;
    if (!filt) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const uint4* src = r == 0 ? dt : dd;
        const float m = lm[r];
        if (r < nrows && landed && m > -INFINITY && m < INFINITY)
          for (int u = tid; u < cu; u += kFT) {
            const uint4 v = src[u];
#pragma unroll
            for (int e = 0; e < E; ++e) ls[r] += ex2((vec_get<BF16>(v, e) - m) * k);
          }
      }
      block_sum2(ls[0], ls[1], sm);
    }
    if (tid == 0) {
      const uint32_t par = ex & 1;
      sm.xrec[par][0] = lm[0];
      sm.xrec[par][1] = ls[0];
      sm.xrec[par][2] = lm[1];
      sm.xrec[par][3] = ls[1];
      sm.xrec[par][4] = __int_as_float(lbad | (my_tmo ? 2 : 0));
    }
    {
      const uint32_t par = publish();
      if (warp == 0) {
        const int fl = lane < C ? __float_as_int(peer(par, 4, lane)) : 0;
        const bool gbad = __any_sync(kFull, fl & 1);
        const bool gtmo = __any_sync(kFull, fl & 2);
        float Mg[2], Sg[2];
        for (int r = 0; r < 2; ++r) {
          const float m = lane < C ? peer(par, 2 * r, lane) : -INFINITY;
          const float sv = lane < C ? peer(par, 2 * r + 1, lane) : 0.0f;
          Mg[r] = __shfl_sync(kFull, lanes_max(m, 32), 0);
          Sg[r] = __shfl_sync(kFull, lanes_sum((sv > 0.0f) ? sv * ex2((m - Mg[r]) * k) : 0.0f, 32), 0);
        }
        if (lane == 0) {
          const bool b2 = gbad || gtmo || !(Mg[0] > -INFINITY && Mg[0] < INFINITY) ||
                          (p.two && !(Mg[1] > -INFINITY && Mg[1] < INFINITY));
          sm.bc[0] = Mg[0];
          sm.bc[1] = Sg[0];
          sm.bc[2] = Mg[1];
          sm.bc[3] = Sg[1];
          sm.bi[0] = b2 || !ok;
          sm.stop = gtmo ? 1 : 0;
        }
      }
      __syncthreads();
    }
    const float M[2] = {sm.bc[0], sm.bc[2]};
    float Sk[2] = {sm.bc[1], sm.bc[3]};          // mass of the kept set, relative to exp2(M k)
    const bool bad = sm.bi[0] != 0;
    if (tid == 0) {
      sm.lnum[0] = 0;
      sm.lnum[1] = 0;
    }
    __syncthreads();

    // this CTA's lists: target [index, z_t, z_d at that index, rank by index], draft [z_d]; in
    // the half of the histogram area that the count passes leave alone (they are written while
    // the per-warp counts are live)
    uint32_t* li0 = reinterpret_cast<uint32_t*>(dyn + 2 * kFRowBytes + kHistBytes / 2);
    float* lz0 = reinterpret_cast<float*>(li0 + kLCap);
    float* lw0 = lz0 + kLCap;
    int* lr0 = reinterpret_cast<int*>(lw0 + kLCap);
    float* lz1 = reinterpret_cast<float*>(lr0 + kLCap);
    // the gathered lists (rank 0, written after the counts were summed)
    uint32_t* mi0 = reinterpret_cast<uint32_t*>(dyn + 2 * kFRowBytes);
    float* mz0 = reinterpret_cast<float*>(mi0 + kLCap);
    float* mw0 = mz0 + kLCap;
    float* mz1 = mw0 + kLCap;

    // Warp 0: the peers' list lengths (exchange record `par`), their offsets and totals.
    auto list_offsets = [&](uint32_t par) {
      if (warp != 0) return;
      const int c0 = lane < C ? __float_as_int(peer(par, 0, lane)) : 0;
      const int c1 = lane < C ? __float_as_int(peer(par, 1, lane)) : 0;
      int i0 = c0, i1 = c1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y0 = __shfl_up_sync(kFull, i0, o), y1 = __shfl_up_sync(kFull, i1, o);
        if (lane >= o) {
          i0 += y0;
          i1 += y1;
        }
      }
      if (lane < C) {
        sm.loff[0][lane] = i0 - c0;
        sm.loff[1][lane] = i1 - c1;
      }
      if (lane == 31) {
        sm.ltot[0] = i0;
        sm.ltot[1] = i1;
      }
    };
    // ---- L: a top-k position on short lists of candidates ----
    // The cluster's counts of the value bins near the max give each row's boundary bin D (the bin
    // of the k-th largest logit): first from kHighBin up (few logits pass the prefilter), again from
    // kLowBin up when fewer than k logits lie that high. A second pass writes every logit of bin D
    // or above into this CTA's list of the row (the top-k set, and so the top-p set on it, lies
    // inside). When every list fits, rank 0 gathers them in index order and finishes the position
    // from them alone; the other CTAs go on to their next position. Otherwise the chunk-wide passes
    // below run. (Listing every logit from kHighBin up during the first count saves the second pass
    // and its exchange, but the longer lists cost rank 0 more than that on the benchmark rows.)
    if (kon && !bad) {
      // Appends logit e of vector u of row r (value z) to this CTA's list of the row.
      auto append = [&](int r, int u, int e, float z) {
        const int slot = atomicAdd(&sm.lnum[r], 1);
        if (slot < kLCap) {
          if (r == 0) {
            li0[slot] = static_cast<uint32_t>((u0 + u) * E + e);
            lz0[slot] = z;
            lw0[slot] = p.two ? vec_get<BF16>(dd[u], e) : 0.0f;
          } else {
            lz1[slot] = z;
          }
        }
      };
      // Ranks of the target list's entries by vocabulary index.
      auto rank_entries = [&]() {
        const int n0 = min(sm.lnum[0], kLCap);
        for (int e = tid; e < n0; e += kFT) {
          const uint32_t ie = li0[e];
          int rk = 0;
          for (int j = 0; j < n0; ++j) rk += li0[j] < ie ? 1 : 0;
          lr0[e] = rk;
        }
      };
      // Counts the value bins from `lo` up, exchanges the counts and finds each row's boundary bin
      // (sm.lD; -1 when the counted bins hold fewer than k logits).
      auto count_pass = [&](int lo) {
        const uint32_t hpar = ex & 1;
        unsigned* whc = reinterpret_cast<unsigned*>(dyn + 2 * kFRowBytes) + warp * 2 * kBins;
        for (int j = lane; j < 2 * kBins; j += 32) whc[j] = 0u;
        __syncwarp();
        for (int r = 0; r < nrows; ++r) {
          const uint4* src = r == 0 ? dt : dd;
          const float Mr = M[r];
          const float zc = cut_below(Mr, k, lo);
          unsigned* hc = whc + r * kBins;
          for (int u = tid; u < cu; u += kFT) {
            const uint4 v = src[u];
            if (!(vec_max<BF16>(v) >= zc)) continue;  // one packed test for the vector's logits
#pragma unroll
            for (int e = 0; e < E; ++e) {
              const float z = vec_get<BF16>(v, e);
              if (z >= zc) {
                const int vb = vbin(z, Mr, k);
                if (vb >= lo) atomicAdd(hc + vb, 1u);
              }
            }
          }
        }
        __syncthreads();
        {
          const unsigned* ahc = reinterpret_cast<const unsigned*>(dyn + 2 * kFRowBytes);
          for (int j = tid; j < 2 * kBins; j += kFT) {
            unsigned c = 0u;
            if (j / kBins < nrows) {
#pragma unroll 4
              for (int w = 0; w < kFW; ++w) c += ahc[w * 2 * kBins + j];
            }
            (&sm.hc[hpar][0][0])[j] = c;
          }
        }
        publish();
        for (int j = tid; j < 2 * kBins; j += kFT) {
          unsigned c = 0u;
          if (j / kBins < nrows && j % kBins >= lo) {
            const uint32_t ac = smem_addr(&sm.hc[hpar][0][0] + j);
            int cq[kMaxCluster];
#pragma unroll
            for (int q = 0; q < kMaxCluster; ++q)
              if (q < C) cq[q] = ld_cluster_s32(map_to_rank(ac, static_cast<uint32_t>(q)));
#pragma unroll
            for (int q = 0; q < kMaxCluster; ++q)
              if (q < C) c += static_cast<unsigned>(cq[q]);
          }
          (&sm.gc[0][0])[j] = c;
        }
        __syncthreads();
        if (warp < nrows) {
          const int D = boundary_bin(sm.gc[warp], static_cast<unsigned>(topk), lane);
          if (lane == 0) sm.lD[warp] = D;
        }
        if (tid == 0) {
          sm.lnum[0] = 0;
          sm.lnum[1] = 0;
        }
        __syncthreads();
      };

      bool listed = false;
      count_pass(kHighBin);
      int Dr[2] = {sm.lD[0], nrows > 1 ? sm.lD[1] : kHighBin};
      if (!(Dr[0] >= kHighBin && Dr[1] >= kHighBin)) {   // cluster-wide counts: same on every CTA
        count_pass(kLowBin);
        Dr[0] = sm.lD[0];
        Dr[1] = nrows > 1 ? sm.lD[1] : kLowBin;
      }
      if (Dr[0] >= kLowBin && Dr[1] >= kLowBin) {
        for (int r = 0; r < nrows; ++r) {
          const uint4* src = r == 0 ? dt : dd;
          const float Mr = M[r];
          const int D = Dr[r];
          const float zc = cut_below(Mr, k, D);
          for (int u = tid; u < cu; u += kFT) {
            const uint4 v = src[u];
            if (!(vec_max<BF16>(v) >= zc)) continue;
#pragma unroll
            for (int e = 0; e < E; ++e) {
              const float z = vec_get<BF16>(v, e);
              if (z >= zc && vbin(z, Mr, k) >= D) append(r, u, e, z);
            }
          }
        }
        __syncthreads();
        rank_entries();
        if (tid == 0) {
          const uint32_t par = ex & 1;
          sm.xrec[par][0] = __int_as_float(sm.lnum[0]);
          sm.xrec[par][1] = __int_as_float(nrows > 1 ? sm.lnum[1] : 0);
        }
        list_offsets(publish());
        __syncthreads();
        listed = sm.ltot[0] <= kLCap && sm.ltot[1] <= kLCap;
      }
      if (listed) {
        const int N0 = sm.ltot[0], N1 = sm.ltot[1];
        {
          // Every list fits: this position reads no row chunk any more, so the next position's
          // copies start now, under the gathering and rank 0's work on the lists.
          if (tid == 0) {
            int s2 = s + P.nclusters;
            while (s2 < total && !fclassify(P, s2).load) s2 += P.nclusters;
            if (s2 < total) {
              issue_copy(fclassify(P, s2));
              pf = s2;
            }
          }
          if (rank != 0) continue;
          // warp 0's global reads for the accept test and the draw, issued first so that their
          // latency passes under the gathering and the selections
          float e_zt = 0.0f, e_zd = 0.0f, e_uacc = 0.0f, e_udraw = 0.0f;
          if (warp == 0) {
            const float* ur = P.uniforms + (size_t)p.b * (G + 2);
            if (p.two) {
              e_zt = load_logit<BF16>(rowt, x);
              e_zd = load_logit<BF16>(rowd, x);
              e_uacc = __ldg(ur + p.i);
            }
            e_udraw = p.two ? __ldg(ur + G) : __ldg(ur + G + 1);
          }
          // gather: CTA q's target entries go to loff[q] + their rank by index (chunks are in index
          // order by rank, so the list is in index order); draft entries in any order
          for (int j = tid; j < N0; j += kFT) {
            int q = 0;
            while (q + 1 < C && j >= sm.loff[0][q + 1]) ++q;
            const int e = j - sm.loff[0][q];
            const uint32_t qq = static_cast<uint32_t>(q);
            const int dst = sm.loff[0][q] + ld_cluster_s32(map_to_rank(smem_addr(lr0 + e), qq));
            mi0[dst] = static_cast<uint32_t>(ld_cluster_s32(map_to_rank(smem_addr(li0 + e), qq)));
            mz0[dst] = ld_cluster_f32(map_to_rank(smem_addr(lz0 + e), qq));
            mw0[dst] = ld_cluster_f32(map_to_rank(smem_addr(lw0 + e), qq));
          }
          for (int j = tid; j < N1; j += kFT) {
            int q = 0;
            while (q + 1 < C && j >= sm.loff[1][q + 1]) ++q;
            mz1[j] = ld_cluster_f32(map_to_rank(smem_addr(lz1 + (j - sm.loff[1][q])),
                                                static_cast<uint32_t>(q)));
          }
          __syncthreads();
          // K, P on the gathered lists: warp r selects row r
          if (warp < nrows) {
            FSel& S = sm.sel[warp];
            const float* zl = warp == 0 ? mz0 : mz1;
            const int nl = warp == 0 ? N0 : N1;
            const float Mr = M[warp];
            list_select<BF16, KB>(S, zl, nl, Mr, k, sm.gc[warp], sm.gm[warp], true,
                                  static_cast<unsigned>(topk), topp, 0, 0u, lane);
            int tD = S.thD0;
            uint32_t tK = S.thkey;
            if (pon) {
              list_select<BF16, KB>(S, zl, nl, Mr, k, sm.gc[warp], sm.gm[warp], false,
                                    static_cast<unsigned>(topk), topp, tD, tK, lane);
              if (S.thD0 > tD || (S.thD0 == tD && S.thkey > tK)) {
                tD = S.thD0;
                tK = S.thkey;
              }
            }
            if (lane == 0) {
              sm.lth[warp] = tD;
              sm.lkey[warp] = tK;
              sm.lmass[warp] = S.mass;
            }
          }
          __syncthreads();
          // V, D on the gathered target list (one warp; lane l takes a contiguous run of entries)
          if (warp == 0) {
            const int t0 = sm.lth[0], t1 = sm.lth[1];
            const uint32_t k0 = sm.lkey[0], k1 = sm.lkey[1];
            const float lt = -log2f(sm.lmass[0]);
            const float ld = p.two ? -log2f(sm.lmass[1]) : 0.0f;
            auto wt_l = [&](float z) -> float {
              return at_or_above(vbin(z, M[0], k), okey<BF16>(z), t0, k0)
                         ? ex2(fmaf(z - M[0], k, lt)) : 0.0f;
            };
            auto wd_l = [&](float z) -> float {
              return at_or_above(vbin(z, M[1], k), okey<BF16>(z), t1, k1)
                         ? ex2(fmaf(z - M[1], k, ld)) : 0.0f;
            };
            float px = 0.0f, qx = 0.0f, acc = 1.0f;
            if (p.two) {
              px = wt_l(e_zt);
              qx = wd_l(e_zd);
              const float ratio = accept_ratio(px, qx);
              acc = e_uacc < ratio ? 1.0f : 0.0f;
            }
            const int run = (N0 + 31) / 32;
            const int e0 = min(lane * run, N0), e1 = min(e0 + run, N0);
            float sp = 0.0f, sw = 0.0f;
            int lastp = -1, lastw = -1;
            for (int e = e0; e < e1; ++e) {
              const float wt = wt_l(mz0[e]);
              sp += wt;
              if (wt > 0.0f) lastp = e;
              if (p.two) {
                const float w = fmaxf(wt - wd_l(mw0[e]), 0.0f);
                sw += w;
                if (w > 0.0f) lastw = e;
              }
            }
            const float ip = warp_incl_scan(sp, lane), iw = warp_incl_scan(sw, lane);
            const float Pt = __shfl_sync(kFull, ip, 31), Wt = __shfl_sync(kFull, iw, 31);
            const float alpha = p.two ? fminf(1.0f, fmaxf(0.0f, 1.0f - Wt)) : 0.0f;
            if (p.two && acc != 0.0f) {
              finish_position(P, p.b, p.i, p.gb, -1, kFlagAccept, alpha, px, qx, lane);
            } else {
              // the residual (rejection), p~ when the residual has no mass, or the bonus draw
              const bool resid = p.two && Wt > 0.0f;
              const float uu = e_udraw;
              const float t = uu * (resid ? Wt : Pt);
              const float ts = resid ? sw : sp, incl = resid ? iw : ip;
              float excl = __shfl_up_sync(kFull, incl, 1);
              if (lane == 0) excl = 0.0f;
              const unsigned cm = __ballot_sync(kFull, ts > 0.0f && incl > t);
              int pick;
              if (cm) {
                const int wl = __ffs(cm) - 1;
                int pk = -1;
                if (lane == wl) {
                  float c = excl;
                  int lp = -1;
                  for (int e = e0; e < e1 && pk < 0; ++e) {
                    const float wt = wt_l(mz0[e]);
                    const float w = resid ? fmaxf(wt - wd_l(mw0[e]), 0.0f) : wt;
                    if (w > 0.0f) {
                      lp = e;
                      c += w;
                      if (c > t) pk = e;
                    }
                  }
                  if (pk < 0) pk = lp;
                }
                pick = __shfl_sync(kFull, pk, wl);
              } else {
                // rounding left the running sum at or below t: the last entry with weight
                int lj = resid ? lastw : lastp;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) lj = max(lj, __shfl_xor_sync(kFull, lj, o));
                pick = lj;
              }
              const int tok = pick >= 0 ? static_cast<int>(mi0[pick]) : -1;
              finish_position(P, p.b, p.i, p.gb, tok,
                              (tok < 0 ? kFlagBad : 0) | (p.two ? 0 : kFlagAccept), alpha, px, qx,
                              lane);
            }
          }
          continue;
        }
      }
    }

    // ---- K, P: the thresholds ----
    int thD0[2] = {0, 0};
    uint32_t thkey[2] = {0u, 0u};
    if (filt && !bad) {
      // One selection (count mode: top-k; else top-p) for the position's rows.
      auto select = [&](bool count_mode) {
        if (tid < nrows) {
          FSel& S = sm.sel[tid];
          S.act = 1;
          S.lvl = 0;
          S.D0 = 0;
          S.pre = 0u;
          S.need = static_cast<unsigned>(topk);
          S.above = 0.0f;
          S.tau = 0.0f;
          S.lbD0 = thD0[tid];
          S.lbkey = thkey[tid];
        }
        __syncthreads();
        while (sm.sel[0].act || (nrows > 1 && sm.sel[1].act)) {
          if (warp < nrows && sm.sel[warp].act) {
            float zlo, zhi;
            level_interval<BF16, KB>(sm.sel[warp], warp == 0 ? M[0] : M[1], k, lane, zlo, zhi);
            if (lane == 0) {
              sm.bc[10 + 2 * warp] = zlo;
              sm.bc[11 + 2 * warp] = zhi;
            }
          }
          __syncthreads();
          // histograms of the active rows' candidates: per warp, then summed over the warps in order
          const uint32_t par = ex & 1;
          unsigned* whc = reinterpret_cast<unsigned*>(dyn + 2 * kFRowBytes) + warp * 2 * kBins;
          float* whm = reinterpret_cast<float*>(dyn + 2 * kFRowBytes + kFW * 2 * kBins * 4) + warp * 2 * kBins;
          for (int j = lane; j < 2 * kBins; j += 32) {
            whc[j] = 0u;
            whm[j] = 0.0f;
          }
          __syncwarp();
          for (int r = 0; r < nrows; ++r) {
            const FSel S = sm.sel[r];
            if (!S.act) continue;
            const uint4* src = r == 0 ? dt : dd;
            const float Mr = M[r];
            const int sh = KB - 8 * S.lvl;
            unsigned* hc = whc + r * kBins;
            float* hm = whm + r * kBins;
            // the level's candidates are the logits in [zlo, zhi); only they get a bin or a key
            const float zlo = sm.bc[10 + 2 * r], zhi = sm.bc[11 + 2 * r];
            for (int u = tid; u < cu; u += kFT) {
              const uint4 v = src[u];
              if (!(vec_max<BF16>(v) >= zlo)) continue;
#pragma unroll
              for (int e = 0; e < E; ++e) {
                const float z = vec_get<BF16>(v, e);
                if (z >= zlo && z < zhi) {
                  const int digit = S.lvl == 0 ? vbin(z, Mr, k)
                                               : static_cast<int>((okey<BF16>(z) >> sh) & 255u);
                  atomicAdd(hc + digit, 1u);
                  atomicAdd(hm + digit, ex2((z - Mr) * k));
                }
              }
            }
          }
          __syncthreads();
          {
            const unsigned* ahc = reinterpret_cast<const unsigned*>(dyn + 2 * kFRowBytes);
            const float* ahm = reinterpret_cast<const float*>(dyn + 2 * kFRowBytes + kFW * 2 * kBins * 4);
            for (int j = tid; j < 2 * kBins; j += kFT) {
              unsigned c = 0u;
              float mm = 0.0f;
              if (j / kBins < nrows) {
#pragma unroll 4
                for (int w = 0; w < kFW; ++w) {
                  c += ahc[w * 2 * kBins + j];
                  mm += ahm[w * 2 * kBins + j];
                }
              }
              (&sm.hc[par][0][0])[j] = c;
              (&sm.hm[par][0][0])[j] = mm;
            }
          }
          publish();
          // the cluster's histograms, summed in rank order
          for (int j = tid; j < 2 * kBins; j += kFT) {
            const int r = j / kBins;
            unsigned c = 0u;
            float mm = 0.0f;
            if (r < nrows && sm.sel[r].act) {
              // Every peer's entry is requested before any is added, so the remote latencies overlap;
              // the sums then run in rank order.
              const uint32_t ac = smem_addr(&sm.hc[par][0][0] + j);
              const uint32_t am = smem_addr(&sm.hm[par][0][0] + j);
              int cq[kMaxCluster];
              float mq[kMaxCluster];
#pragma unroll
              for (int q = 0; q < kMaxCluster; ++q) {
                if (q < C) {
                  cq[q] = ld_cluster_s32(map_to_rank(ac, static_cast<uint32_t>(q)));
                  mq[q] = ld_cluster_f32(map_to_rank(am, static_cast<uint32_t>(q)));
                }
              }
#pragma unroll
              for (int q = 0; q < kMaxCluster; ++q) {
                if (q < C) {
                  c += static_cast<unsigned>(cq[q]);
                  mm += mq[q];
                }
              }
            }
            (&sm.gc[0][0])[j] = c;
            (&sm.gm[0][0])[j] = mm;
          }
          __syncthreads();
          if (warp < nrows && sm.sel[warp].act)
            decide<KB>(sm.sel[warp], sm.gc[warp], sm.gm[warp], count_mode, topp, lane);
          __syncthreads();
        }
        for (int r = 0; r < nrows; ++r) {
          const int D = sm.sel[r].thD0;
          const uint32_t kk = sm.sel[r].thkey;
          if (D > thD0[r] || (D == thD0[r] && kk > thkey[r])) {
            thD0[r] = D;
            thkey[r] = kk;
          }
          Sk[r] = sm.sel[r].mass;
        }
        __syncthreads();
      };
      if (kon) select(true);
      if (pon) select(false);
    }

    // ---- V: the filtered p~ (and q~), the accept test, the chunk totals ----
    // kept: (vbin, okey) at or above the row's threshold, i.e. z at or above its smallest float
    float zth[2] = {-INFINITY, -INFINITY};
    if (filt && !bad) {
      if (warp < nrows) {
        const float t = kept_threshold<BF16>(M[warp], k, warp == 0 ? thD0[0] : thD0[1],
                                             warp == 0 ? thkey[0] : thkey[1], lane);
        if (lane == 0) sm.bc[4 + warp] = t;
      }
      __syncthreads();
      zth[0] = sm.bc[4];
      zth[1] = sm.bc[5];
    }
    auto kept = [&](float z, int r) -> bool { return !filt || z >= zth[r]; };
    const float lt = -log2f(Sk[0]);              // p~(v) = exp2((z - M) k - log2 Sk) on kept logits
    const float ld = p.two ? -log2f(Sk[1]) : 0.0f;
    auto wt_of = [&](float z) -> float { return kept(z, 0) ? ex2(fmaf(z - M[0], k, lt)) : 0.0f; };
    auto wd_of = [&](float z) -> float { return kept(z, 1) ? ex2(fmaf(z - M[1], k, ld)) : 0.0f; };
    float px = 0.0f, qx = 0.0f, acc = 1.0f;
    if (p.two && !bad) {
      px = wt_of(load_logit<BF16>(rowt, x));
      qx = wd_of(load_logit<BF16>(rowd, x));
      const float ratio = accept_ratio(px, qx);
      acc = __ldg(P.uniforms + (size_t)p.b * (G + 2) + p.i) < ratio ? 1.0f : 0.0f;
    }
    float wsum = 0.0f, psum = 0.0f;
    if (!bad) {
      for (int u = tid; u < cu; u += kFT) {
        const uint4 vt = dt[u];
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float wt = wt_of(vec_get<BF16>(vt, e));
          psum += wt;
          if (p.two) wsum += fmaxf(wt - wd_of(vec_get<BF16>(dd[u], e)), 0.0f);
        }
      }
    }
    block_sum2(wsum, psum, sm);
    if (tid == 0) {
      const uint32_t par = ex & 1;
      sm.xrec[par][0] = wsum;
      sm.xrec[par][1] = psum;
    }
    {
      const uint32_t par = publish();
      if (warp == 0) {
        const float w_r = lane < C ? peer(par, 0, lane) : 0.0f;
        const float p_r = lane < C ? peer(par, 1, lane) : 0.0f;
        const float iw = warp_incl_scan(w_r, lane);
        const float ip = warp_incl_scan(p_r, lane);
        const float Wt = __shfl_sync(kFull, iw, 31), Pt = __shfl_sync(kFull, ip, 31);
        float ew = __shfl_up_sync(kFull, iw, 1), ep = __shfl_up_sync(kFull, ip, 1);
        if (lane == 0) ew = ep = 0.0f;
        const float* ur = P.uniforms + (size_t)p.b * (G + 2);
        // The draw: the residual (rejection), p~ when the residual has no mass, or the bonus.
        const bool draw_resid = p.two && acc == 0.0f && Wt > 0.0f;
        const float uu = p.two ? __ldg(ur + G) : __ldg(ur + G + 1);
        const float t = uu * (draw_resid ? Wt : Pt);
        const float wv = draw_resid ? w_r : p_r, iv = draw_resid ? iw : ip;
        const float evv = draw_resid ? ew : ep;
        const unsigned hit = __ballot_sync(kFull, lane < C && wv > 0.0f && iv > t);
        const unsigned pos = __ballot_sync(kFull, lane < C && wv > 0.0f);
        const int c = hit ? (__ffs(hit) - 1) : (pos ? (31 - __clz(pos)) : 0);
        const float tl = t - __shfl_sync(kFull, evv, c);
        if (lane == 0) {
          sm.bi[8] = (bad || (p.two && acc != 0.0f)) ? -1 : c;
          sm.bi[9] = draw_resid;
          sm.bc[8] = tl;
          sm.bc[9] = fminf(1.0f, fmaxf(0.0f, 1.0f - Wt));
        }
      }
      __syncthreads();
    }
    const int dch = sm.bi[8];
    const bool resid = sm.bi[9] != 0;
    const float tl = sm.bc[8];
    const float alpha = p.two ? sm.bc[9] : 0.0f;
    __syncthreads();
    if (!ok) {
      if (p.i == 0 && rank == 0 && warp == 0) write_row_error(P, p.b, lane);
      continue;
    }
    if (dch < 0) {
      if (rank == 0 && warp == 0) {
        if (bad) finish_position(P, p.b, p.i, p.gb, -1, kFlagBad, 0.0f, 0.0f, 0.0f, lane);
        else finish_position(P, p.b, p.i, p.gb, -1, kFlagAccept, alpha, px, qx, lane);
      }
      continue;
    }
    if (rank != dch) continue;

    // ---- D: the draw inside this CTA's chunk (a contiguous run per thread, block-wide scan) ----
    auto weight = [&](int j) -> float {
      const float wt = wt_of(vec_get<BF16>(dt[j / E], j % E));
      if (!resid) return wt;
      return fmaxf(wt - wd_of(vec_get<BF16>(dd[j / E], j % E)), 0.0f);
    };
    const int nel = cu * E;
    const int run = (nel + kFT - 1) / kFT;
    const int e0 = min(tid * run, nel), e1 = min(e0 + run, nel);
    float tsum = 0.0f;
    int lastp = -1;
    for (int j = e0; j < e1; ++j) {
      const float w = weight(j);
      tsum += w;
      if (w > 0.0f) lastp = j;
    }
    const float incl = warp_incl_scan(tsum, lane);
    if (lane == 31) sm.redf[warp][0] = incl;
    int lj = lastp;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lj = max(lj, __shfl_xor_sync(kFull, lj, o));
    if (lane == 0) sm.redi[warp][0] = lj;
    __syncthreads();
    float wex = 0.0f;
    for (int w = 0; w < warp; ++w) wex += sm.redf[w][0];
    float excl = __shfl_up_sync(kFull, incl, 1);
    if (lane == 0) excl = 0.0f;
    const bool cross = tsum > 0.0f && wex + incl > tl;
    const unsigned cm = __ballot_sync(kFull, cross);
    if (lane == 0) sm.redi[warp][1] = cm ? warp * 32 + __ffs(cm) - 1 : INT_MAX;
    __syncthreads();
    int win = INT_MAX, best = -1;
    for (int w = 0; w < kFW; ++w) {
      win = min(win, sm.redi[w][1]);
      best = max(best, sm.redi[w][0]);
    }
    if (win != INT_MAX && tid == win) {
      float c = wex + excl;
      int pick = -1, lp = -1;
      for (int j = e0; j < e1 && pick < 0; ++j) {
        const float w = weight(j);
        if (w > 0.0f) {
          lp = j;
          c += w;
          if (c > tl) pick = j;
        }
      }
      sm.bi[10] = pick >= 0 ? pick : lp;
    } else if (win == INT_MAX && tid == 0) {
      sm.bi[10] = best;
    }
    __syncthreads();
    const int pick = sm.bi[10];
    __syncthreads();
    if (warp == 0) {
      const int tok = pick >= 0 ? u0 * E + pick : -1;
      finish_position(P, p.b, p.i, p.gb, tok, (tok < 0 ? kFlagBad : 0) | (p.two ? 0 : kFlagAccept),
                      alpha, px, qx, lane);
    }
  }
  // A copy that timed out, or one issued ahead for a position the cluster did not reach, may still
  // land: wait for it (bounded) before this CTA can exit.
  if (tid == 0) {
    if (my_tmo) mbar_wait_drain(smem_addr(&sm.bar), (npos - 1) & 1);
    if (pf >= 0) mbar_wait_drain(smem_addr(&sm.bar), npos & 1);
  }
  cluster_sync_all();        // no CTA leaves while a peer may still read its shared memory
}

const void* filter_fn(bool bf16) {
  return bf16 ? reinterpret_cast<const void*>(sv_filter_kernel<true>)
              : reinterpret_cast<const void*>(sv_filter_kernel<false>);
}

cudaError_t filter_attrs(const void* fn, int C) {
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kFDynBytes);
  if (e != cudaSuccess) return e;
  if (C > 8) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

cudaLaunchConfig_t filter_config(int C, int nclusters, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nclusters * C), 1, 1);
  cfg.blockDim = dim3(kFT, 1, 1);
  cfg.dynamicSmemBytes = kFDynBytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

int filter_max_row_units() { return kFRowUnits; }

cudaError_t filter_max_clusters(bool bf16, int C, int* n) {
  const void* fn = filter_fn(bf16);
  const cudaError_t e = filter_attrs(fn, C);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = filter_config(C, 16, nullptr, attr);
  return cudaOccupancyMaxActiveClusters(n, fn, &cfg);
}

cudaError_t launch_filter(Params P, bool bf16, cudaStream_t stream) {
  const void* fn = filter_fn(bf16);
  const cudaError_t e = filter_attrs(fn, P.C);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = filter_config(P.C, P.nclusters, stream, attr);
  void* args[] = {&P};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace sv
