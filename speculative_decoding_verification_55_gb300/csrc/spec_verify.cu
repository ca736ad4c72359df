// Batched speculative-decoding verification (accept-or-resample) for GB300 / sm_103a.
//
// The operation is defined on these pages (page title, section):
//   [R] "Speculative decoding", rayaq.ca ml-models -- Mechanics, One round, steps 3-5; Why the
//       output is exactly the target's; The greedy case; Implementation.
//   [B] "Inference: distillation and speculative decoding", brunomaga.github.io -- Draft-model
//       speculative decoding (greedy rule, speculative-sampling rule, ragged batched rows).
//   [C] "Speculative decoding", cgnarendiran.github.io blog -- The correction that makes it exact.
// p is the target distribution, q the draft distribution.
//
// Design. One thread-block cluster of C CTAs (C <= 16) verifies one position (b, i) of the batch.
// The V-wide logit row(s) of the position are split into C contiguous chunks; each CTA reads its
// chunk ONCE from HBM with 16-byte streaming loads straight into registers (the row never goes
// through shared memory and is never re-read), and all later passes run on those registers:
//   phase A  chunk max (NaN-propagating; greedy: argmax with the lowest index)
//   phase B  chunk sum of exp2((z - m_chunk) * log2(e) / T)
//   xchg 1   the C chunk records meet over distributed shared memory: global max M, normaliser
//            S = sum_r s_r * 2^((m_r - M) k) (an inclusive scan over ranks, so chunk-level CDF
//            prefixes come for free), then the accept test on p(x), q(x)
//   phase C  (draft positions) alpha partial = sum min(p, q), residual partial = sum max(0, p - q)
//   xchg 2   alpha and the residual chunk totals (inclusive scan over ranks)
//   phase D  only the CTA whose chunk holds the inverse-CDF threshold scans its chunk in index order
//            (block-wide prefix sum) to pick the residual or bonus token
//   emit     the last position of a row to finish (an atomic arrival counter per row in the
//            caller's workspace, no spinning) finds the first rejection and writes the row's outputs.
// There is no dense contraction anywhere in this operation, so no tensor-core path is used: the
// kernel is bound by HBM bandwidth (and, for bf16, by the exp2 rate of the special-function units).

#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <cstdint>
#include <mutex>

#include "../../include/spec_verify.h"

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 16;
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;

enum : int { kVerify = 0, kBonus = 1, kArgmax = 2 };
enum : int { kFlagAccept = 1, kFlagBad = 2 };

struct Params {
  const void* zt;            // [B, G+1, V]
  const void* zd;            // [B, G, V]
  const int32_t* tokens;     // [B, G]
  const int32_t* draft_len;  // [B] or null
  const float* temperature;  // [B]
  const float* uniforms;     // [B, G+2]
  int32_t* out_tokens;       // [B, G+1]
  int32_t* out_num;          // [B]
  float* out_alpha;          // [B, G] or null
  float* out_p;              // [B, G] or null
  float* out_q;              // [B, G] or null
  int2* rec;                 // [B, G+1] per-position records {candidate token, flags}
  unsigned* cnt;             // [B] arrival counters (zero between calls)
  int B, G, V;
  int C;                     // CTAs per position (cluster size)
  int units;                 // load units per row (16-byte vectors, or elements on the scalar path)
  int per;                   // units per CTA chunk
};

// ------------------------------------------------------------------------------------------------
// Small device helpers (inline PTX for the cluster, exp2 and NaN-propagating max)
// ------------------------------------------------------------------------------------------------

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

__device__ __forceinline__ uint32_t map_to_rank(const void* smem_ptr, uint32_t rank) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(smem_ptr));
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ int ld_cluster_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void st_cluster_s32(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// One stored logit widened to fp32 (exact for both storage types).
template <bool BF16>
__device__ __forceinline__ float load_logit(const void* row, int v) {
  if (BF16) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(row) + v);
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  }
  return __ldg(reinterpret_cast<const float*>(row) + v);
}

// A load unit: a 16-byte vector (8 bf16 or 4 fp32 logits) on the vector path, one logit on the
// scalar path (rows whose byte length is not a multiple of 16). Units past the chunk read as -inf.
template <bool BF16, bool VEC>
struct Unit;

template <bool BF16>
struct Unit<BF16, true> {
  static constexpr int E = BF16 ? 8 : 4;
  uint4 v;
  __device__ __forceinline__ void load(const void* row, int u, bool ok) {
    if (ok) {
      v = ld_stream_v4(reinterpret_cast<const uint4*>(row) + u);
    } else {
      const uint32_t ninf = BF16 ? 0xFF80FF80u : 0xFF800000u;
      v = make_uint4(ninf, ninf, ninf, ninf);
    }
  }
  __device__ __forceinline__ uint32_t word(int w) const {
    return w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
  }
  __device__ __forceinline__ float get(int e) const {
    if (BF16) {
      const uint32_t w = word(e >> 1);
      return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
    }
    return __uint_as_float(word(e));
  }
  __device__ __forceinline__ float vmax() const {
    if (BF16) {
      const uint32_t m = bmax2_nan(bmax2_nan(v.x, v.y), bmax2_nan(v.z, v.w));
      return max_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    }
    return max_nan(max_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                   max_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
};

template <bool BF16>
struct Unit<BF16, false> {
  static constexpr int E = 1;
  float v;
  __device__ __forceinline__ void load(const void* row, int u, bool ok) {
    v = ok ? load_logit<BF16>(row, u) : -INFINITY;
  }
  __device__ __forceinline__ float get(int) const { return v; }
  __device__ __forceinline__ float vmax() const { return v; }
};

// exp2((z - M) * k) * inv_s with every rounding explicit, so that phase C and phase D recompute
// bit-identical probabilities.
__device__ __forceinline__ float scaled_exp(float z, float M, float k) {
  return ex2(__fmul_rn(__fsub_rn(z, M), k));
}
__device__ __forceinline__ float prob(float z, float M, float k, float inv_s) {
  return __fmul_rn(scaled_exp(z, M, k), inv_s);
}
__device__ __forceinline__ float resid_weight(float zt, float zd, float Mt, float Md, float k,
                                              float it, float id) {
  return fmaxf(__fsub_rn(prob(zt, Mt, k, it), prob(zd, Md, k, id)), 0.0f);
}

struct __align__(16) Smem {
  float red[3][kWarps][2];     // block-reduction scratch, one buffer per stage
  int ired[kWarps][2];
  float xch1[4];               // this CTA's chunk record for exchange 1
  int xch1i[2];
  float xch2[2];               // this CTA's chunk record for exchange 2
  float scan_wt[2][kWarps];    // phase D warp totals (double-buffered by segment)
  int scan_slot[2][kWarps];    // phase D first crossing thread per warp
  int result;                  // the drawn token (written into rank 0's copy)
};

__device__ __forceinline__ float warp_sum_lane0(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return __shfl_sync(kFull, v, 0);
}

__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ float warp_incl_scan(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// Writes the all-error outputs of row b (warp-wide).
__device__ void write_row_error(const Params& P, int b, int lane) {
  const int G = P.G;
  for (int j = lane; j <= G; j += 32) P.out_tokens[(size_t)b * (G + 1) + j] = -1;
  for (int j = lane; j < G; j += 32) {
    if (P.out_alpha) P.out_alpha[(size_t)b * G + j] = 0.0f;
    if (P.out_p) P.out_p[(size_t)b * G + j] = 0.0f;
    if (P.out_q) P.out_q[(size_t)b * G + j] = 0.0f;
  }
  if (lane == 0) P.out_num[b] = -1;
}

// Phase D: block-wide inverse-CDF scan of this CTA's chunk in index order. Picks the first element
// whose running weight exceeds t_local (the threshold minus the weight of the chunks before this
// one); if rounding leaves none, the last element with positive weight. resid selects the weight:
// max(0, p - q) (residual draw) or exp2((z - Mt) k) (draw from p). Returns the token on every
// thread of the CTA.
template <bool BF16, bool VEC, int VPT>
__device__ int chunk_draw(const Unit<BF16, VEC> (&rt)[VPT], const Unit<BF16, VEC> (&rd)[VPT],
                          bool resid, float Mt, float Md, float k, float it, float id,
                          float t_local, int u0, int u1, Smem& sm) {
  constexpr int E = Unit<BF16, VEC>::E;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float running = 0.0f;
  int last_pos = -1;
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int u = u0 + tid + j * kThreads;
    float wv[E];
    float tsum = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      float w = 0.0f;
      if (u < u1) {
        w = resid ? resid_weight(rt[j].get(e), rd[j].get(e), Mt, Md, k, it, id)
                  : scaled_exp(rt[j].get(e), Mt, k);
      }
      wv[e] = w;
      tsum = __fadd_rn(tsum, w);
      if (w > 0.0f) last_pos = u * E + e;
    }
    const float incl = warp_incl_scan(tsum, lane);
    float excl = __shfl_up_sync(kFull, incl, 1);
    if (lane == 0) excl = 0.0f;
    const int pb = j & 1;
    if (lane == 31) sm.scan_wt[pb][warp] = incl;
    __syncthreads();
    float wexcl = 0.0f, seg = 0.0f;
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) {
      const float v = sm.scan_wt[pb][w2];
      if (w2 < warp) wexcl += v;
      seg += v;
    }
    const bool cross = (tsum > 0.0f) && (running + (wexcl + incl) > t_local);
    const unsigned m = __ballot_sync(kFull, cross);
    if (lane == 0) sm.scan_slot[pb][warp] = m ? (warp * 32 + __ffs(m) - 1) : INT_MAX;
    __syncthreads();
    int win = INT_MAX;
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) win = min(win, sm.scan_slot[pb][w2]);
    if (win != INT_MAX) {
      if (tid == win) {
        float c = running + (wexcl + excl);
        int pick = -1, lastp = -1;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if (wv[e] > 0.0f) {
            lastp = e;
            c += wv[e];
            if (pick < 0 && c > t_local) pick = e;
          }
        }
        if (pick < 0) pick = lastp;
        sm.ired[0][0] = u * E + pick;
      }
      __syncthreads();
      return sm.ired[0][0];
    }
    running = running + seg;
  }
  // Overrun by rounding: the last element with positive weight in this chunk.
  int lp = last_pos;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(kFull, lp, o));
  if (lane == 0) sm.ired[warp][1] = lp;
  __syncthreads();
  int best = -1;
#pragma unroll
  for (int w2 = 0; w2 < kWarps; ++w2) best = max(best, sm.ired[w2][1]);
  return best;
}

// ------------------------------------------------------------------------------------------------
// The kernel: one cluster of P.C CTAs per (row, position) slot.
// ------------------------------------------------------------------------------------------------

template <bool BF16, bool VEC, int VPT>
__global__ void __launch_bounds__(kThreads, (VPT <= 4 ? 2 : 1)) sv_verify_kernel(const Params P) {
  using U = Unit<BF16, VEC>;
  constexpr int E = U::E;
  constexpr size_t ES = BF16 ? 2 : 4;
  __shared__ Smem sm;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = static_cast<int>(cluster_rank());
  const int C = P.C;
  const int G = P.G, G1 = G + 1;
  const int slot = static_cast<int>(blockIdx.x) / C;
  const int b = slot / G1, i = slot % G1;

  // ---- Row scalars and the row-error rules (every warp computes the same answer) ----
  const int gb = P.draft_len ? __ldg(P.draft_len + b) : G;
  const float T = __ldg(P.temperature + b);
  const bool len_ok = gb >= 0 && gb <= G;
  if (len_ok && i > gb) return;                       // padding slot: never read
  const bool greedy = (T == 0.0f);
  bool ok = len_ok && (greedy || (T >= FLT_MIN && T <= FLT_MAX));   // NaN fails both
  if (ok) {
    bool good = true;
    const int32_t* xr = P.tokens + (size_t)b * G;
    for (int j = lane; j < gb; j += 32) {
      const int x = __ldg(xr + j);
      good &= (x >= 0 && x < P.V);
    }
    if (!greedy) {
      const float* ur = P.uniforms + (size_t)b * (G + 2);
      for (int j = lane; j < gb + 2; j += 32) {
        const float u = __ldg(ur + (j < gb ? j : G + (j - gb)));
        good &= (u >= 0.0f && u < 1.0f);
      }
    }
    ok = __all_sync(kFull, good);
  }
  if (!ok) {
    if (i == 0 && rank == 0 && warp == 0) write_row_error(P, b, lane);
    return;
  }

  const int kind = greedy ? kArgmax : (i < gb ? kVerify : kBonus);
  const bool two = (kind == kVerify);
  const size_t Vs = static_cast<size_t>(P.V);
  const char* rowt = static_cast<const char*>(P.zt) + ((size_t)b * G1 + i) * Vs * ES;
  const char* rowd = two ? static_cast<const char*>(P.zd) + ((size_t)b * G + i) * Vs * ES : nullptr;
  const int u0 = rank * P.per;
  const int u1 = min(u0 + P.per, P.units);
  const int x = (i < gb) ? __ldg(P.tokens + (size_t)b * G + i) : -1;
  if (rank == 0 && tid == 0) sm.result = -1;

  // ---- Load the chunk once: 16-byte streaming loads into registers ----
  U rt[VPT], rd[VPT];
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int u = u0 + tid + j * kThreads;
    rt[j].load(rowt, u, u < u1);
  }
  if (two) {
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int u = u0 + tid + j * kThreads;
      rd[j].load(rowd, u, u < u1);
    }
  }

  // ---- Phase A: chunk max (NaN and +inf propagate, so a bad row shows in the max) ----
  float mt = -INFINITY, md = -INFINITY;
#pragma unroll
  for (int j = 0; j < VPT; ++j) mt = max_nan(mt, rt[j].vmax());
  if (two) {
#pragma unroll
    for (int j = 0; j < VPT; ++j) md = max_nan(md, rd[j].vmax());
  }

  int cand = -1;
  int flags = 0;
  float alpha = 0.0f, px = 0.0f, qx = 0.0f;

  if (kind == kArgmax) {
    // Greedy: target argmax, lowest index on ties ([B] greedy rule; [R] The greedy case).
    bool bad = (mt != mt) || (mt == INFINITY);
    int idx = INT_MAX;
    if (!bad && mt > -INFINITY) {
#pragma unroll
      for (int j = 0; j < VPT; ++j) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if (idx == INT_MAX && rt[j].get(e) == mt) idx = (u0 + tid + j * kThreads) * E + e;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(kFull, mt, o);
      const int oi = __shfl_xor_sync(kFull, idx, o);
      if (ov > mt || (ov == mt && oi < idx)) { mt = ov; idx = oi; }
    }
    bad = __any_sync(kFull, bad);
    if (lane == 0) {
      sm.red[0][warp][0] = mt;
      sm.ired[warp][0] = idx;
      sm.ired[warp][1] = bad;
    }
    __syncthreads();
    float cv = -INFINITY;
    int ci = INT_MAX, cb = 0;
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) {
      const float v = sm.red[0][w2][0];
      const int ii = sm.ired[w2][0];
      if (v > cv || (v == cv && ii < ci)) { cv = v; ci = ii; }
      cb |= sm.ired[w2][1];
    }
    if (tid == 0) {
      sm.xch1[0] = cv;
      sm.xch1i[0] = ci;
      sm.xch1i[1] = cb;
    }
    cluster_sync_all();                                   // exchange 1
    float gv = -INFINITY;
    int gi = INT_MAX, gbad = 0;
    if (lane < C) {
      gv = ld_cluster_f32(map_to_rank(&sm.xch1[0], lane));
      gi = ld_cluster_s32(map_to_rank(&sm.xch1i[0], lane));
      gbad = ld_cluster_s32(map_to_rank(&sm.xch1i[1], lane));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(kFull, gv, o);
      const int oi = __shfl_xor_sync(kFull, gi, o);
      if (ov > gv || (ov == gv && oi < gi)) { gv = ov; gi = oi; }
    }
    gbad = __any_sync(kFull, gbad != 0) || !(gv > -INFINITY);
    cand = gi;
    const bool acc = (i < gb) && (x == gi);
    flags = (gbad ? kFlagBad : 0) | (acc ? kFlagAccept : 0);
    alpha = px = acc ? 1.0f : 0.0f;
    qx = 1.0f;
  } else {
    // ---- Sampled rows: temperature softmax of p (and q) ([R] Implementation) ----
    const float k = kLog2e / T;
    mt = warp_max_nan(mt);
    md = warp_max_nan(md);
    if (lane == 0) { sm.red[0][warp][0] = mt; sm.red[0][warp][1] = md; }
    __syncthreads();
    float mct = -INFINITY, mcd = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) {
      mct = max_nan(mct, sm.red[0][w2][0]);
      mcd = max_nan(mcd, sm.red[0][w2][1]);
    }
    // ---- Phase B: chunk sums against the chunk max ----
    const float reft = (mct == -INFINITY) ? 0.0f : mct;
    const float refd = (mcd == -INFINITY) ? 0.0f : mcd;
    float st = 0.0f, sd = 0.0f;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
#pragma unroll
      for (int e = 0; e < E; ++e) st += scaled_exp(rt[j].get(e), reft, k);
    }
    if (two) {
#pragma unroll
      for (int j = 0; j < VPT; ++j) {
#pragma unroll
        for (int e = 0; e < E; ++e) sd += scaled_exp(rd[j].get(e), refd, k);
      }
    }
    st = warp_sum_lane0(st);
    sd = warp_sum_lane0(sd);
    if (lane == 0) { sm.red[1][warp][0] = st; sm.red[1][warp][1] = sd; }
    __syncthreads();
    float sct = 0.0f, scd = 0.0f;
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) {
      sct += sm.red[1][w2][0];
      scd += sm.red[1][w2][1];
    }
    if (tid == 0) {
      sm.xch1[0] = mct; sm.xch1[1] = sct; sm.xch1[2] = mcd; sm.xch1[3] = scd;
    }
    cluster_sync_all();                                   // exchange 1
    // Every warp combines the C chunk records in the same fixed order (bit-identical results).
    float m_r = -INFINITY, s_r = 0.0f, md_r = -INFINITY, sd_r = 0.0f;
    if (lane < C) {
      m_r = ld_cluster_f32(map_to_rank(&sm.xch1[0], lane));
      s_r = ld_cluster_f32(map_to_rank(&sm.xch1[1], lane));
      md_r = ld_cluster_f32(map_to_rank(&sm.xch1[2], lane));
      sd_r = ld_cluster_f32(map_to_rank(&sm.xch1[3], lane));
    }
    const float Mt = warp_max_nan(m_r);
    const float Md = warp_max_nan(md_r);
    const float term_t = (s_r > 0.0f) ? s_r * scaled_exp(m_r, Mt, k) : 0.0f;
    const float incl_t = warp_incl_scan(term_t, lane);
    const float St = __shfl_sync(kFull, incl_t, 31);
    float Sd = 1.0f;
    bool bad = !(Mt > -INFINITY && Mt < INFINITY);        // NaN, +inf, or every logit -inf
    if (two) {
      const float term_d = (sd_r > 0.0f) ? sd_r * scaled_exp(md_r, Md, k) : 0.0f;
      Sd = __shfl_sync(kFull, warp_incl_scan(term_d, lane), 31);
      bad = bad || !(Md > -INFINITY && Md < INFINITY);
    }
    const float* ur = P.uniforms + (size_t)b * (G + 2);

    // Which chunk holds the threshold t of a draw whose chunk CDF is incl: the first chunk with
    // positive weight whose inclusive prefix exceeds t, else (rounding) the last positive chunk.
    auto pick_chunk = [&](float incl, float term, float t, float& t_local) -> int {
      const unsigned hit = __ballot_sync(kFull, lane < C && term > 0.0f && incl > t);
      const unsigned pos = __ballot_sync(kFull, lane < C && term > 0.0f);
      const int c = hit ? (__ffs(hit) - 1) : (pos ? (31 - __clz(pos)) : 0);
      float excl = __shfl_up_sync(kFull, incl, 1);
      if (lane == 0) excl = 0.0f;
      t_local = t - __shfl_sync(kFull, excl, c);
      return c;
    };

    int draw_chunk = -1;          // chunk of the residual / bonus draw, -1: no draw
    bool draw_resid = false;
    float t_local = 0.0f;
    float it = 0.0f, id = 0.0f;
    bool acc = true;
    if (kind == kBonus) {
      // Bonus token from p at position gamma_b ([R] One round, step 5).
      const float t = __ldg(ur + G + 1) * St;
      draw_chunk = pick_chunk(incl_t, term_t, t, t_local);
    } else {
      // Accept test u < min(1, p(x)/q(x)) ([R] One round, step 3).
      const float zx_t = load_logit<BF16>(rowt, x);
      const float zx_d = load_logit<BF16>(rowd, x);
      px = __fdiv_rn(scaled_exp(zx_t, Mt, k), St);
      qx = __fdiv_rn(scaled_exp(zx_d, Md, k), Sd);
      const float ratio = (qx > 0.0f) ? fminf(1.0f, __fdiv_rn(px, qx)) : 1.0f;
      acc = __ldg(ur + i) < ratio;

      // ---- Phase C: alpha = sum min(p, q) and residual mass sum max(0, p - q) ----
      it = __frcp_rn(St);
      id = __frcp_rn(Sd);
      float a = 0.0f, w = 0.0f;
#pragma unroll
      for (int j = 0; j < VPT; ++j) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float pt = prob(rt[j].get(e), Mt, k, it);
          const float pd = prob(rd[j].get(e), Md, k, id);
          a += fminf(pt, pd);
          w += fmaxf(__fsub_rn(pt, pd), 0.0f);
        }
      }
      a = warp_sum_lane0(a);
      w = warp_sum_lane0(w);
      if (lane == 0) { sm.red[2][warp][0] = a; sm.red[2][warp][1] = w; }
      __syncthreads();
      float ac = 0.0f, wc = 0.0f;
#pragma unroll
      for (int w2 = 0; w2 < kWarps; ++w2) {
        ac += sm.red[2][w2][0];
        wc += sm.red[2][w2][1];
      }
      if (tid == 0) { sm.xch2[0] = ac; sm.xch2[1] = wc; }
      cluster_sync_all();                                 // exchange 2
      float a_r = 0.0f, w_r = 0.0f;
      if (lane < C) {
        a_r = ld_cluster_f32(map_to_rank(&sm.xch2[0], lane));
        w_r = ld_cluster_f32(map_to_rank(&sm.xch2[1], lane));
      }
      alpha = warp_sum_lane0(a_r);                         // [R] alpha = sum min(p, q)
      const float incl_w = warp_incl_scan(w_r, lane);
      const float W = __shfl_sync(kFull, incl_w, 31);
      if (!acc) {
        // Replacement from max(0, p - q) / sum max(0, p - q) ([R] One round, step 4).
        const float u_res = __ldg(ur + G);
        if (W > 0.0f) {
          draw_resid = true;
          draw_chunk = pick_chunk(incl_w, w_r, u_res * W, t_local);
        } else {
          draw_chunk = pick_chunk(incl_t, term_t, u_res * St, t_local);   // zero residual mass
        }
      }
    }
    if (draw_chunk >= 0 && !bad && rank == draw_chunk) {
      const int tok = chunk_draw<BF16, VEC, VPT>(rt, rd, draw_resid, Mt, Md, k, it, id, t_local,
                                                 u0, u1, sm);
      if (tid == 0) st_cluster_s32(map_to_rank(&sm.result, 0), tok);
    }
    flags = (bad ? kFlagBad : 0) | (acc ? kFlagAccept : 0);
  }

  cluster_sync_all();                                     // no CTA leaves while peers read it
  if (rank != 0 || warp != 0) return;

  // ---- Position record, arrival, and (last arriver) the row's outputs ----
  if (kind != kArgmax) cand = sm.result;
  if ((kind == kBonus || (kind == kVerify && !(flags & kFlagAccept))) && cand < 0) flags |= kFlagBad;
  if (lane == 0 && i < gb) {
    if (P.out_alpha) P.out_alpha[(size_t)b * G + i] = alpha;
    if (P.out_p) P.out_p[(size_t)b * G + i] = px;
    if (P.out_q) P.out_q[(size_t)b * G + i] = qx;
  }
  if (i == gb) {
    for (int j = gb + lane; j < G; j += 32) {              // padding positions
      if (P.out_alpha) P.out_alpha[(size_t)b * G + j] = 0.0f;
      if (P.out_p) P.out_p[(size_t)b * G + j] = 0.0f;
      if (P.out_q) P.out_q[(size_t)b * G + j] = 0.0f;
    }
  }
  unsigned old = 0;
  if (lane == 0) {
    P.rec[(size_t)b * G1 + i] = make_int2(cand, flags);
    __threadfence();
    old = atomicAdd(P.cnt + b, 1u);
  }
  old = __shfl_sync(kFull, old, 0);
  if (old != static_cast<unsigned>(gb)) return;
  __threadfence();

  // Last arriver: k = first rejected position, else gamma_b ([R] One round, steps 3-5).
  int kk = gb;
  bool err = false;
  for (int j0 = 0; j0 <= gb; j0 += 32) {
    const int j = j0 + lane;
    int2 r = make_int2(-1, kFlagAccept);
    if (j <= gb) r = __ldcg(P.rec + (size_t)b * G1 + j);
    err |= (j <= gb) && (r.y & kFlagBad);
    const unsigned rej = __ballot_sync(kFull, j < gb && !(r.y & kFlagAccept));
    if (rej && kk == gb) kk = j0 + __ffs(rej) - 1;
  }
  err = __any_sync(kFull, err);
  const int tok_k = __ldcg(P.rec + (size_t)b * G1 + kk).x;
  for (int j = lane; j <= G; j += 32) {
    int v = -1;
    if (!err) v = (j < kk) ? __ldg(P.tokens + (size_t)b * G + j) : (j == kk ? tok_k : -1);
    P.out_tokens[(size_t)b * G1 + j] = v;
  }
  if (err) {
    for (int j = lane; j < G; j += 32) {
      if (P.out_alpha) P.out_alpha[(size_t)b * G + j] = 0.0f;
      if (P.out_p) P.out_p[(size_t)b * G + j] = 0.0f;
      if (P.out_q) P.out_q[(size_t)b * G + j] = 0.0f;
    }
  }
  if (lane == 0) {
    P.out_num[b] = err ? -1 : kk + 1;
    P.cnt[b] = 0u;                                         // leave the workspace zeroed
  }
}

// ------------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------------

using KernelFn = void (*)(const Params);

constexpr int kVptOptions[4] = {1, 2, 4, 8};

template <bool BF16, bool VEC>
KernelFn kernel_for(int vpt_index) {
  switch (vpt_index) {
    case 0: return sv_verify_kernel<BF16, VEC, 1>;
    case 1: return sv_verify_kernel<BF16, VEC, 2>;
    case 2: return sv_verify_kernel<BF16, VEC, 4>;
    default: return sv_verify_kernel<BF16, VEC, 8>;
  }
}

KernelFn select_kernel(bool bf16, bool vec, int vpt_index) {
  if (bf16) return vec ? kernel_for<true, true>(vpt_index) : kernel_for<true, false>(vpt_index);
  return vec ? kernel_for<false, true>(vpt_index) : kernel_for<false, false>(vpt_index);
}

struct Plan {
  bool vec;
  int vpt_index;
  int C;
  int units;
  int per;
};

// Splits a row of V logits into C <= 16 chunks of at most 512 * VPT load units, preferring the
// smallest VPT (fewest registers per thread, most CTAs per SM).
bool make_plan(int V, bool bf16, bool vec, Plan* plan) {
  const int es = bf16 ? 2 : 4;
  const int E = vec ? 16 / es : 1;
  const int units = vec ? V / E : V;
  for (int vi = 0; vi < 4; ++vi) {
    const long long cap = static_cast<long long>(kThreads) * kVptOptions[vi];
    const long long C = (units + cap - 1) / cap;
    if (C <= kMaxCluster) {
      plan->vec = vec;
      plan->vpt_index = vi;
      plan->C = static_cast<int>(C < 1 ? 1 : C);
      plan->units = units;
      plan->per = static_cast<int>((units + plan->C - 1) / plan->C);
      return true;
    }
  }
  return false;
}

std::mutex g_mu;
int g_device_ok[64];          // 0 unknown, 1 sm_103, 2 other
bool g_attr_set[2][2][4];

int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  if (dev < 0 || dev >= 64) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_device_ok[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return SV_ERR_CUDA;
    g_device_ok[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  return g_device_ok[dev] == 1 ? SV_OK : SV_ERR_UNSUPPORTED_DEVICE;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t records_bytes(int32_t B, int32_t G) {
  return align_up(static_cast<size_t>(B) * (G + 1) * sizeof(int2), 256);
}

bool sizes_ok(int32_t B, int32_t G, int32_t V, int32_t dtype) {
  if (B < 1 || G < 0 || G > SV_MAX_GAMMA || V < 1) return false;
  if (dtype != SV_DTYPE_F32 && dtype != SV_DTYPE_BF16) return false;
  return true;
}

}  // namespace

extern "C" {

size_t spec_verify_workspace_size(int32_t B, int32_t gamma_max, int32_t V, int32_t dtype) {
  if (!sizes_ok(B, gamma_max, V, dtype)) return 0;
  return align_up(records_bytes(B, gamma_max) + static_cast<size_t>(B) * sizeof(unsigned), 256);
}

const char* spec_verify_status_string(int status) {
  switch (status) {
    case SV_OK: return "SV_OK: success";
    case SV_ERR_NULL_POINTER: return "SV_ERR_NULL_POINTER: a required pointer is NULL";
    case SV_ERR_BAD_SHAPE: return "SV_ERR_BAD_SHAPE: B, gamma_max or V out of range";
    case SV_ERR_BAD_DTYPE: return "SV_ERR_BAD_DTYPE: dtype is not SV_DTYPE_F32 or SV_DTYPE_BF16";
    case SV_ERR_WORKSPACE_TOO_SMALL: return "SV_ERR_WORKSPACE_TOO_SMALL: workspace missing or too small";
    case SV_ERR_MISALIGNED: return "SV_ERR_MISALIGNED: a pointer is not aligned to its element type";
    case SV_ERR_CUDA: return "SV_ERR_CUDA: a CUDA runtime call failed";
    case SV_ERR_UNSUPPORTED_DEVICE: return "SV_ERR_UNSUPPORTED_DEVICE: the device is not sm_103";
    default: return "unknown sv_status";
  }
}

int spec_verify_version(void) { return SV_VERSION; }

int spec_verify_ex(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                   const int32_t* draft_len, const float* temperature, const float* uniforms,
                   int32_t* out_tokens, int32_t* out_num_emitted, float* out_alpha,
                   float* out_p_draft, float* out_q_draft,
                   int32_t B, int32_t gamma_max, int32_t V, int32_t dtype,
                   void* workspace, size_t workspace_bytes, void* cuda_stream) {
  if (dtype != SV_DTYPE_F32 && dtype != SV_DTYPE_BF16) return SV_ERR_BAD_DTYPE;
  if (!sizes_ok(B, gamma_max, V, dtype)) return SV_ERR_BAD_SHAPE;
  const int G = gamma_max;
  if (!target_logits || !temperature || !uniforms || !out_tokens || !out_num_emitted)
    return SV_ERR_NULL_POINTER;
  if (G > 0 && (!draft_logits || !draft_tokens)) return SV_ERR_NULL_POINTER;
  const bool bf16 = dtype == SV_DTYPE_BF16;
  const uintptr_t es = bf16 ? 2 : 4;
  auto mis = [](const void* p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) != 0; };
  if (mis(target_logits, es) || mis(draft_logits, es) || mis(draft_tokens, 4) || mis(draft_len, 4) ||
      mis(temperature, 4) || mis(uniforms, 4) || mis(out_tokens, 4) || mis(out_num_emitted, 4) ||
      mis(out_alpha, 4) || mis(out_p_draft, 4) || mis(out_q_draft, 4) || mis(workspace, 16))
    return SV_ERR_MISALIGNED;
  const size_t need = spec_verify_workspace_size(B, G, V, dtype);
  if (!workspace || workspace_bytes < need) return SV_ERR_WORKSPACE_TOO_SMALL;

  const bool vec = (static_cast<size_t>(V) * es) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(target_logits) % 16 == 0 &&
                   (!draft_logits || reinterpret_cast<uintptr_t>(draft_logits) % 16 == 0);
  Plan plan;
  if (!make_plan(V, bf16, vec, &plan)) return SV_ERR_BAD_SHAPE;
  const long long grid = static_cast<long long>(B) * (G + 1) * plan.C;
  if (grid > INT_MAX) return SV_ERR_BAD_SHAPE;

  const int dev_status = check_device();
  if (dev_status != SV_OK) return dev_status;

  Params P;
  P.zt = target_logits;
  P.zd = draft_logits;
  P.tokens = draft_tokens;
  P.draft_len = draft_len;
  P.temperature = temperature;
  P.uniforms = uniforms;
  P.out_tokens = out_tokens;
  P.out_num = out_num_emitted;
  P.out_alpha = out_alpha;
  P.out_p = out_p_draft;
  P.out_q = out_q_draft;
  P.rec = static_cast<int2*>(workspace);
  P.cnt = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + records_bytes(B, G));
  P.B = B;
  P.G = G;
  P.V = V;
  P.C = plan.C;
  P.units = plan.units;
  P.per = plan.per;

  KernelFn fn = select_kernel(bf16, plan.vec, plan.vpt_index);
  if (plan.C > 8) {
    std::lock_guard<std::mutex> lock(g_mu);
    bool& done = g_attr_set[bf16][plan.vec][plan.vpt_index];
    if (!done) {
      if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                               cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return SV_ERR_CUDA;
      done = true;
    }
  }

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(cuda_stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(plan.C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, fn, P) != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
}

int spec_verify(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                const int32_t* draft_len, const float* temperature, const float* uniforms,
                int32_t* out_tokens, int32_t* out_num_emitted, float* out_alpha,
                int32_t B, int32_t gamma_max, int32_t V, int32_t dtype,
                void* workspace, size_t workspace_bytes, void* cuda_stream) {
  return spec_verify_ex(target_logits, draft_logits, draft_tokens, draft_len, temperature, uniforms,
                        out_tokens, out_num_emitted, out_alpha, nullptr, nullptr, B, gamma_max, V,
                        dtype, workspace, workspace_bytes, cuda_stream);
}

}  // extern "C"
