// Verification of filtered batch rows from their kept lists on sm_103a ([R] "Speculative decoding",
// rayaq.ca ml-models -- One round, steps 3-5; Why the output is exactly the target's: the filters
// are applied to p and q before the test).
//
// With top-k on, a logit row's filtered distribution lives on its kept set: at most k logits plus
// ties (then cut by top-p). The threshold kernel writes each such set, when it holds at most kList
// logits, as an (index, logit) list. A batch row all of whose read logit rows have lists is verified
// here from the lists alone, without reading its rows again:
//   p~(v) = 2^((z_v - M) k) / Z over the target list (M its max, Z its sum), q~ likewise;
//   accept x_i while u[b,i] < min(1, p~(x)/q~(x)) (where q~(x) = 0 the ratio is 1 if p~(x) > 0,
//   else 0); alpha_i = sum over v of min(p~(v), q~(v)); at the first rejection the token is drawn
//   from max(0, p~ - q~) (from p~ when that has no mass) with u[b,G], after gamma_b accepts from p~
//   of position gamma_b with u[b,G+1]; both draws by inverse CDF in index order (the first index
//   whose running weight exceeds u times the total, else the last index with weight).
// Logits outside a list have p~ = 0 (or q~ = 0), so the lists carry every term of these sums.
// Rows this kernel does not take (greedy rows, rows without lists, rows with a bad scalar) are left
// untouched for the streaming kernel, which skips the rows marked in `listed`.
//
// One CTA of kList threads per batch row; a list entry per thread after the lists are sorted by
// index (rank sort), so every sum runs in index order and the results do not depend on the order the
// threshold kernel wrote the entries in.

#include <climits>

#include "../../include/spec_verify.h"
#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kLT = kList;                 // threads per CTA
constexpr int kLW = kLT / 32;

struct LShared {
  int2 stage[kList];                       // a list as written
  int idx_t[kList];                        // target list sorted by index
  float w_t[kList];                        // its weights 2^((z - M) k)
  int idx_d[kList];                        // draft list sorted by index
  float w_d[kList];
  float redf[kLW];
  int n_t, n_d;
  float px, qx;
  int acc[SV_MAX_GAMMA];
  float alpha[SV_MAX_GAMMA], pxs[SV_MAX_GAMMA], qxs[SV_MAX_GAMMA];
  int tok, ok;
};

// Block sums over the kLT threads (a fixed tree: the same result every run).
__device__ __forceinline__ float block_sum(LShared& sm, float v, int lane, int warp) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  if (lane == 0) sm.redf[warp] = v;
  __syncthreads();
  float s = 0.0f;
#pragma unroll
  for (int w = 0; w < kLW; ++w) s += sm.redf[w];
  __syncthreads();
  return s;
}

__device__ __forceinline__ float block_max(LShared& sm, float v, int lane, int warp) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  if (lane == 0) sm.redf[warp] = v;
  __syncthreads();
  float s = -INFINITY;
#pragma unroll
  for (int w = 0; w < kLW; ++w) s = fmaxf(s, sm.redf[w]);
  __syncthreads();
  return s;
}

// Loads the list of n entries into idx / w sorted by index, weights 2^((z - M) k) with M the list's
// max. Returns the sum of the weights (every thread).
__device__ float load_list(LShared& sm, const int2* src, int n, int* idx, float* w, float k, int tid,
                           int lane, int warp) {
  if (tid < n) sm.stage[tid] = src[tid];
  __syncthreads();
  float z = -INFINITY;
  if (tid < n) {
    const int2 e = sm.stage[tid];
    int rank = 0;
    for (int m = 0; m < n; ++m) rank += sm.stage[m].x < e.x ? 1 : 0;
    z = __int_as_float(e.y);
    idx[rank] = e.x;
    w[rank] = z;                           // the logit for now
  }
  const float M = block_max(sm, z, lane, warp);    // also orders the writes above
  float wv = 0.0f;
  if (tid < n) {
    wv = ex2(fmaf(w[tid], k, -M * k));
    w[tid] = wv;
  }
  return block_sum(sm, wv, lane, warp);
}

// Position of index v in the sorted list idx[0..n), or -1.
__device__ __forceinline__ int find_index(const int* idx, int n, int v) {
  int lo = 0, hi = n - 1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    const int x = idx[mid];
    if (x == v) return mid;
    if (x < v) lo = mid + 1; else hi = mid - 1;
  }
  return -1;
}

// Inverse CDF over the weights r (thread j holds the weight of the j-th smallest index, 0 past the
// list) with uniform u: the first j whose running weight exceeds u times the total (strict), else
// the last j with a positive weight. -1 when every weight is 0. Every thread gets the answer.
__device__ int draw_index(LShared& sm, int* redi, float r, float u, int lane, int warp) {
  float incl = r;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm.redf[warp] = incl;
  __syncthreads();
  float off = 0.0f, total = 0.0f;
#pragma unroll
  for (int w = 0; w < kLW; ++w) {
    if (w < warp) off += sm.redf[w];
    total += sm.redf[w];
  }
  incl += off;
  const float t = u * total;
  const unsigned hit = __ballot_sync(kFull, incl > t);
  const unsigned pos = __ballot_sync(kFull, r > 0.0f);
  if (lane == 0) {
    redi[warp] = hit ? warp * 32 + __ffs(hit) - 1 : INT_MAX;
    redi[kLW + warp] = pos ? warp * 32 + 31 - __clz(pos) : -1;
  }
  __syncthreads();
  int first = INT_MAX, last = -1;
#pragma unroll
  for (int w = 0; w < kLW; ++w) {
    first = min(first, redi[w]);
    last = max(last, redi[kLW + w]);
  }
  __syncthreads();
  if (!(total > 0.0f)) return -1;
  return first != INT_MAX ? first : last;
}

__global__ void __launch_bounds__(kLT) sv_listed_kernel(const Params P, const int2* lists,
                                                        const int* list_n, int* listed) {
  __shared__ LShared sm;
  __shared__ int redi[2 * kLW];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  const int B = P.B, G = P.G, G1 = G + 1, V = P.V;

  // ---- does this kernel take the row: sampled, top-k on, good scalars, every read row listed ----
  if (tid == 0) {
    bool ok = true;
    const int gb = P.draft_len ? __ldg(P.draft_len + b) : G;
    const float T = __ldg(P.temperature + b);
    ok = gb >= 0 && gb <= G && T >= FLT_MIN && T <= FLT_MAX;
    if (ok) {
      const int topk = P.top_k ? __ldg(P.top_k + b) : 0;
      ok = topk > 0 && topk < V;
      if (P.top_p) ok = ok && __ldg(P.top_p + b) > 0.0f;   // NaN fails
    }
    for (int i = 0; ok && i <= gb; ++i) {
      ok = __ldg(list_n + (size_t)b * G1 + i) > 0;
      if (ok && i < gb) {
        ok = __ldg(list_n + (size_t)B * G1 + (size_t)b * G + i) > 0;
        const int x = __ldg(P.tokens + (size_t)b * G + i);
        ok = ok && x >= 0 && x < V;
      }
    }
    const float* ur = P.uniforms + (size_t)b * (G + 2);
    for (int j = 0; ok && j < gb + 2; ++j) {
      const float u = __ldg(ur + (j < gb ? j : G + (j - gb)));
      ok = u >= 0.0f && u < 1.0f;
    }
    sm.ok = ok ? 1 : 0;
    sm.tok = -1;
  }
  __syncthreads();
  if (!sm.ok) return;
  const int gb = P.draft_len ? __ldg(P.draft_len + b) : G;
  const float k = kLog2e / __ldg(P.temperature + b);
  const float* ur = P.uniforms + (size_t)b * (G + 2);

  // ---- positions 0 .. gamma_b ----
  bool rejected = false;
  for (int i = 0; i <= gb; ++i) {
    const size_t rt = (size_t)b * G1 + i;
    const int n_t = __ldg(list_n + rt);
    const float Zt = load_list(sm, lists + rt * kList, n_t, sm.idx_t, sm.w_t, k, tid, lane, warp);
    const float p_t = tid < n_t ? sm.w_t[tid] / Zt : 0.0f;
    if (i == gb) {
      if (!rejected) {                     // the bonus token from p~ of position gamma_b
        const int j = draw_index(sm, redi, p_t, __ldg(ur + G + 1), lane, warp);
        if (tid == 0) sm.tok = j >= 0 ? sm.idx_t[j] : -1;
      }
      break;
    }
    const size_t rd = (size_t)B * G1 + (size_t)b * G + i;
    const int n_d = __ldg(list_n + rd);
    const float Zd = load_list(sm, lists + rd * kList, n_d, sm.idx_d, sm.w_d, k, tid, lane, warp);
    const int x = __ldg(P.tokens + (size_t)b * G + i);
    if (tid == 0) {
      sm.px = 0.0f;
      sm.qx = 0.0f;
    }
    __syncthreads();
    if (tid < n_t && sm.idx_t[tid] == x) sm.px = p_t;
    if (tid < n_d && sm.idx_d[tid] == x) sm.qx = sm.w_d[tid] / Zd;
    // min(p~, q~) and the residual max(0, p~ - q~) at this thread's target entry
    float q_at = 0.0f;
    if (tid < n_t) {
      const int m = find_index(sm.idx_d, n_d, sm.idx_t[tid]);
      if (m >= 0) q_at = sm.w_d[m] / Zd;
    }
    const float alpha = block_sum(sm, fminf(p_t, q_at), lane, warp);   // also orders px / qx
    const float px = sm.px, qx = sm.qx;
    const bool acc = __ldg(ur + i) < accept_ratio(px, qx);
    if (tid == 0) {
      sm.acc[i] = acc ? 1 : 0;
      sm.alpha[i] = alpha;
      sm.pxs[i] = px;
      sm.qxs[i] = qx;
    }
    if (!acc && !rejected) {               // the first rejection: the residual draw
      int j = draw_index(sm, redi, fmaxf(p_t - q_at, 0.0f), __ldg(ur + G), lane, warp);
      if (j < 0) j = draw_index(sm, redi, p_t, __ldg(ur + G), lane, warp);   // no residual mass
      if (tid == 0) sm.tok = j >= 0 ? sm.idx_t[j] : -1;
      rejected = true;
    }
    __syncthreads();                       // the lists are reloaded for the next position
  }
  __syncthreads();

  // ---- the row's outputs ----
  int kk = gb;
  for (int i = 0; i < gb; ++i) {
    if (!sm.acc[i]) {
      kk = i;
      break;
    }
  }
  const int tok = sm.tok;
  const bool err = tok < 0;                // no token with weight (only on degenerate lists)
  for (int j = tid; j <= G; j += kLT) {
    int v = -1;
    if (!err) v = j < kk ? __ldg(P.tokens + (size_t)b * G + j) : (j == kk ? tok : -1);
    P.out_tokens[(size_t)b * G1 + j] = v;
  }
  for (int j = tid; j < G; j += kLT) {
    const bool in = !err && j < gb;
    if (P.out_alpha) P.out_alpha[(size_t)b * G + j] = in ? sm.alpha[j] : 0.0f;
    if (P.out_p) P.out_p[(size_t)b * G + j] = in ? sm.pxs[j] : 0.0f;
    if (P.out_q) P.out_q[(size_t)b * G + j] = in ? sm.qxs[j] : 0.0f;
  }
  if (tid == 0) {
    P.out_num[b] = err ? -1 : kk + 1;
    listed[b] = 1;
  }
}

}  // namespace

cudaError_t launch_listed(const Params& P, const int2* lists, const int* list_n, int* listed,
                          cudaStream_t stream) {
  sv_listed_kernel<<<P.B, kLT, 0, stream>>>(P, lists, list_n, listed);
  return cudaGetLastError();
}

}  // namespace sv
