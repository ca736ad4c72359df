// Element path of the sm_103a verifier: rows whose byte length is not a multiple of 16 or whose
// base is not 16-byte aligned (small or odd vocabularies). One thread-block cluster of C CTAs
// verifies one (row, position) slot; each CTA loads its chunk of the logit row(s) once, logit by
// logit, into registers and every later pass runs on those registers:
//   phase A  chunk max (NaN-propagating; greedy rows: argmax with the lowest index)
//   phase B  chunk sum of exp2((z - m_chunk) * log2(e) / T)
//   xchg 1   chunk records meet over distributed shared memory: global max M, normaliser S (an
//            inclusive scan over ranks gives the chunk-level CDF), then the accept test
//   phase C  (draft positions) alpha = sum min(p, q), residual mass sum max(0, p - q)
//   xchg 2   alpha and the residual chunk totals
//   phase D  the CTA whose chunk holds the inverse-CDF threshold scans its chunk in index order
// Rows of 16-byte multiples take the streaming path (sv_stream.cu) instead.
//
// The operation: [R] "Speculative decoding", rayaq.ca ml-models -- Mechanics, One round, steps 3-5;
// The greedy case. [B] brunomaga.github.io "Inference: distillation and speculative decoding" --
// Draft-model speculative decoding. [C] cgnarendiran.github.io "Speculative decoding" -- The
// correction that makes it exact.

#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

// One logit per load unit; units past the chunk read as -inf.
template <bool BF16>
struct ElemUnit {
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

// Phase D: block-wide inverse-CDF scan of this CTA's chunk in index order. Picks the first element
// whose running weight exceeds t_local (the threshold minus the weight of the chunks before this
// one); if rounding leaves none, the last element with positive weight. resid selects the weight:
// max(0, p - q) (residual draw) or exp2((z - Mt) k) (draw from p). Returns the token on every
// thread of the CTA.
template <bool BF16, int VPT>
__device__ int chunk_draw(const ElemUnit<BF16> (&rt)[VPT], const ElemUnit<BF16> (&rd)[VPT],
                          bool resid, float Mt, float Md, float k, float it, float id,
                          float t_local, int u0, int u1, Smem& sm) {
  constexpr int E = ElemUnit<BF16>::E;
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

template <bool BF16, int VPT>
__global__ void __launch_bounds__(kThreads, (VPT <= 4 ? 2 : 1)) sv_element_kernel(const Params P) {
  using U = ElemUnit<BF16>;
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
      gv = ld_cluster_f32(map_to_rank(smem_addr(&sm.xch1[0]), lane));
      gi = ld_cluster_s32(map_to_rank(smem_addr(&sm.xch1i[0]), lane));
      gbad = ld_cluster_s32(map_to_rank(smem_addr(&sm.xch1i[1]), lane));
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
      m_r = ld_cluster_f32(map_to_rank(smem_addr(&sm.xch1[0]), lane));
      s_r = ld_cluster_f32(map_to_rank(smem_addr(&sm.xch1[1]), lane));
      md_r = ld_cluster_f32(map_to_rank(smem_addr(&sm.xch1[2]), lane));
      sd_r = ld_cluster_f32(map_to_rank(smem_addr(&sm.xch1[3]), lane));
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
      const float ratio = accept_ratio(px, qx);
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
        a_r = ld_cluster_f32(map_to_rank(smem_addr(&sm.xch2[0]), lane));
        w_r = ld_cluster_f32(map_to_rank(smem_addr(&sm.xch2[1]), lane));
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
      const int tok = chunk_draw<BF16, VPT>(rt, rd, draw_resid, Mt, Md, k, it, id, t_local,
                                                 u0, u1, sm);
      if (tid == 0) st_cluster_s32(map_to_rank(smem_addr(&sm.result), 0), tok);
    }
    flags = (bad ? kFlagBad : 0) | (acc ? kFlagAccept : 0);
  }

  cluster_sync_all();                                     // no CTA leaves while peers read it
  if (rank != 0 || warp != 0) return;

  // ---- The position's result, its arrival and (last arriver) the row's outputs ----
  if (kind != kArgmax) cand = sm.result;
  if ((kind == kBonus || (kind == kVerify && !(flags & kFlagAccept))) && cand < 0) flags |= kFlagBad;
  finish_position(P, b, i, gb, cand, flags, alpha, px, qx, lane);
}


using KernelFn = void (*)(const Params);

template <bool BF16>
KernelFn element_kernel(int vpt_index) {
  switch (vpt_index) {
    case 0: return sv_element_kernel<BF16, 1>;
    case 1: return sv_element_kernel<BF16, 2>;
    case 2: return sv_element_kernel<BF16, 4>;
    case 3: return sv_element_kernel<BF16, 8>;
    case 4: return sv_element_kernel<BF16, 16>;
    default: return sv_element_kernel<BF16, 32>;
  }
}

}  // namespace

cudaError_t launch_element(const Params& P, bool bf16, int vpt_index, cudaStream_t stream) {
  KernelFn fn = bf16 ? element_kernel<true>(vpt_index) : element_kernel<false>(vpt_index);
  if (P.C > 8) {
    const cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                               cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  const long long grid = static_cast<long long>(P.B) * (P.G + 1) * P.C;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(P.C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, P);
}

}  // namespace sv
