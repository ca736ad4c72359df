// Shared device code of the sm_103a verification kernels: kernel parameters, inline-PTX helpers
// (exp2, NaN-propagating max, clusters, mbarriers, bulk copies), warp reductions, and the
// per-position finish (record, arrival counter, row emit) both kernels end with.
//
// The operation is defined on these pages (page title, section):
//   [R] "Speculative decoding", rayaq.ca ml-models -- Mechanics, One round, steps 3-5; Why the
//       output is exactly the target's; The greedy case; Implementation.
//   [B] "Inference: distillation and speculative decoding", brunomaga.github.io -- Draft-model
//       speculative decoding (greedy rule, speculative-sampling rule, ragged batched rows).
//   [C] "Speculative decoding", cgnarendiran.github.io blog -- The correction that makes it exact.
// p is the target distribution, q the draft distribution.
#pragma once

#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <cstdint>

namespace sv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxCluster = 16;
// Largest chunk (in 16-byte vectors) one CTA of the streaming kernel owns per row: its group
// sums of the residual weights must fit in shared memory beside the copy ring (bf16: a two-slot
// ring, 128 KB chunks; fp32: a three-slot ring).
#ifndef SV_STREAM_MAX_UNITS_BF16
#define SV_STREAM_MAX_UNITS_BF16 8192
#endif
#ifndef SV_STREAM_MAX_UNITS_F32
#define SV_STREAM_MAX_UNITS_F32 4864
#endif
// wide: the draw groups of bf16 one-hot launches, twice as long (twice the chunk, same table).
constexpr int stream_max_units(bool bf16, bool wide = false) {
  return bf16 ? (wide ? 2 * SV_STREAM_MAX_UNITS_BF16 : SV_STREAM_MAX_UNITS_BF16)
              : SV_STREAM_MAX_UNITS_F32;
}

enum : int { kVerify = 0, kBonus = 1, kArgmax = 2, kOneHot = 3 };
enum : int { kFlagAccept = 1, kFlagBad = 2, kFlagDone = 4 };

struct Params {
  const void* zt;            // [B, G+1, V] target logits
  const void* zd;            // [B, G, V] draft logits
  const int32_t* tokens;     // [B, G] drafted tokens
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
  unsigned* status;          // [1] sticky kernel status (0 = fine)
  int B, G, V;
  int C;                     // CTAs per position (cluster size)
  int units;                 // load units per row (16-byte vectors, or logits on the element path)
  int per;                   // units per CTA chunk
  int nclusters;             // clusters in the grid (persistent kernel)
  int onehot;                // drafted positions have one-hot drafts q = [v == x] (no draft logits)
  // Greedy tree verification (tree != 0): positions are the N = G + 1 tree nodes of each row.
  int tree;
  const int32_t* tparent;    // [B, N] parent of each node, -1 at the root
  const int32_t* ttok;       // [B, N] token of each node
  const int32_t* tsize;      // [B] nodes per row, or null (N)
  int32_t* out_path;         // [B, N] longest accepted path, root first
  int32_t* out_plen;         // [B] nodes on the path
  int32_t* out_pred;         // [B, N] target argmax per node, or null
  // Filtered verification: per-row top-k and top-p, applied to p and q alike.
  const int32_t* top_k;      // [B] or null (0 or >= V: off)
  const float* top_p;        // [B] or null (>= 1: off)
  // Filtered verification by thresholds: per row the smallest logit the filters keep (target rows
  // [B, G+1], then draft rows [B, G]); the streaming kernel reads every logit below it as -inf.
  const float* tau;
  // Filtered batch rows already verified from their kept lists (nonzero: the streaming kernel
  // leaves the row alone), or null.
  const int* listed;
};

constexpr int kMaxTreeNodes = 65;    // N <= SV_MAX_GAMMA + 1
// Kept lists of filtered logit rows: at most kList (index, logit) entries per row.
constexpr int kList = 128;

// ------------------------------------------------------------------------------------------------
// Arithmetic
// ------------------------------------------------------------------------------------------------

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The accept probability min(1, p(x)/q(x)) ([R] One round, step 3). q(x) = 0 gives 1 when p(x) > 0
// (p >= q is always kept) and 0 when p(x) = 0 as well: a token the target gives no mass is never
// emitted ([R] The output distribution is exactly the target's). Round-to-nearest division.
__device__ __forceinline__ float accept_ratio(float px, float qx) {
  if (qx > 0.0f) return fminf(1.0f, __fdiv_rn(px, qx));
  return px > 0.0f ? 1.0f : 0.0f;
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

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Packed fp32 pairs (sm_100+ f32x2 arithmetic).
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pk(float a, float b) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk(f32x2 v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ------------------------------------------------------------------------------------------------
// Memory
// ------------------------------------------------------------------------------------------------

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// L2 eviction-priority policies: evict_last for data read again soon (a drafted position's chunk,
// re-read by the residual pass), evict_first for data read for the last time.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
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

// Logit e (0 <= e < 8 for bf16, < 4 for fp32) of a 16-byte vector.
template <bool BF16>
__device__ __forceinline__ float vec_get(const uint4& v, int e) {
  const int w = BF16 ? (e >> 1) : e;
  const uint32_t x = w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
  if (BF16) return __uint_as_float((e & 1) ? (x & 0xffff0000u) : (x << 16));
  return __uint_as_float(x);
}

// The vector with every logit below tau read as -inf (NaN stays: it still marks a bad row). tau is a
// stored logit value (exact in the storage type) or -inf.
template <bool BF16>
__device__ __forceinline__ uint4 mask_below(const uint4& v, float tau) {
  if (BF16) {
    const uint32_t t = __float_as_uint(tau) >> 16;
    const uint32_t t2 = t | (t << 16);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t m;
      asm("set.lt.u32.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(w[q]), "r"(t2));   // 0xffff where z < tau
      w[q] = (w[q] & ~m) | (0xff80ff80u & m);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  const uint32_t ninf = 0xff800000u;
  return make_uint4(__uint_as_float(v.x) < tau ? ninf : v.x, __uint_as_float(v.y) < tau ? ninf : v.y,
                    __uint_as_float(v.z) < tau ? ninf : v.z, __uint_as_float(v.w) < tau ? ninf : v.w);
}

// NaN-propagating max of the logits of a 16-byte vector.
template <bool BF16>
__device__ __forceinline__ float vec_max(const uint4& v) {
  if (BF16) {
    const uint32_t m = bmax2_nan(bmax2_nan(v.x, v.y), bmax2_nan(v.z, v.w));
    return max_nan(bf_lo(m), bf_hi(m));
  }
  return max_nan(max_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                 max_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
}

// ------------------------------------------------------------------------------------------------
// Clusters and mbarriers
// ------------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
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

// Asynchronous stores into another CTA's shared memory that complete their bytes on that CTA's
// mbarrier (no fence, no round trip for the storing thread).
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                            uint32_t d, uint32_t mbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
      ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d), "r"(mbar) : "memory");
}

__device__ __forceinline__ void st_async_v2(uint32_t addr, uint32_t a, uint32_t b, uint32_t mbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];"
               ::"r"(addr), "r"(a), "r"(b), "r"(mbar) : "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init_cluster() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded waits: every spin gives up after kSpinLimit polls (each poll may suspend the thread for a
// hardware-chosen time), so a broken protocol ends the kernel with an error status instead of a hang.
// A CTA that waits for its own bulk copies to land before it exits (they always land: they read
// valid memory) allows kDrainLimit polls.
#ifndef SV_SPIN_LIMIT
#define SV_SPIN_LIMIT (1 << 22)
#endif
constexpr int kSpinLimit = SV_SPIN_LIMIT;
constexpr int kDrainLimit = 1 << 26;

__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  for (int n = 0; n < kDrainLimit; ++n)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (int n = 0; n < kSpinLimit; ++n)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity) {
  for (int n = 0; n < kSpinLimit; ++n)
    if (mbar_try_wait_cluster(bar, parity)) return true;
  return false;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Arrive on an mbarrier of any CTA of the cluster, releasing this thread's earlier writes.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// Bulk copy global -> this CTA's shared memory, completing `bytes` transactions on `bar`, with an
// L2 eviction-priority policy for the source lines.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}


// ------------------------------------------------------------------------------------------------
// Warp reductions
// ------------------------------------------------------------------------------------------------

__device__ __forceinline__ float warp_sum_lane0(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return __shfl_sync(kFull, v, 0);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
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

// The same over the first n lanes only (n a power of two, 1 <= n <= 32): log2(n) shuffle stages
// instead of five. Lanes below n get the result; the others hold partial values.
__device__ __forceinline__ float lanes_max(float v, int n) {
  for (int o = 1; o < n; o <<= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ float lanes_sum(float v, int n) {
  for (int o = 1; o < n; o <<= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ float lanes_incl_scan(float v, int lane, int n) {
  for (int o = 1; o < n; o <<= 1) {
    const float y = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

__device__ __forceinline__ void lanes_argmax(float& v, int& i, int n) {
  for (int o = 1; o < n; o <<= 1) {
    const float ov = __shfl_xor_sync(kFull, v, o);
    const int oi = __shfl_xor_sync(kFull, i, o);
    if (ov > v || (ov == v && oi < i)) {
      v = ov;
      i = oi;
    }
  }
}

// (value, index) argmax over the warp: larger value wins, equal values keep the lower index.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(kFull, v, o);
    const int oi = __shfl_xor_sync(kFull, i, o);
    if (ov > v || (ov == v && oi < i)) {
      v = ov;
      i = oi;
    }
  }
}

// ------------------------------------------------------------------------------------------------
// Inner loops over 16-byte vectors of logits (8 bf16 or 4 fp32)
// ------------------------------------------------------------------------------------------------

// Online softmax update with N vectors of one thread (a ring slot's share in the streaming
// kernel's pass 1, a step of a top-p row's first pass in the threshold kernel): one max and one
// rescale check for the batch, then every exp2 with two independent accumulators.
template <bool BF16, int N>
__device__ __forceinline__ void online_update_batch(const uint4 (&v)[N], float k, float& m, f32x2& s,
                                                    float& mx) {
  float vm = -INFINITY;
  if (BF16) {
    uint32_t a = bmax2_nan(bmax2_nan(v[0].x, v[0].y), bmax2_nan(v[0].z, v[0].w));
#pragma unroll
    for (int j = 1; j < N; ++j)
      a = bmax2_nan(a, bmax2_nan(bmax2_nan(v[j].x, v[j].y), bmax2_nan(v[j].z, v[j].w)));
    vm = max_nan(bf_lo(a), bf_hi(a));
  } else {
#pragma unroll
    for (int j = 0; j < N; ++j) vm = max_nan(vm, vec_max<false>(v[j]));
  }
  mx = max_nan(mx, vm);
  if (vm > m) {                                   // rescale the running sum to the new max
    if (m > -INFINITY) {
      float s0, s1;
      upk(s, s0, s1);
      const float f = ex2((m - vm) * k);
      s = pk(s0 * f, s1 * f);
    }
    m = vm;
  }
  // Every logit so far is -inf (NaN is caught by mx): nothing to add, and -m k would be +inf.
  if (!(m > -INFINITY)) return;
  const float c = -m * k;
  const f32x2 k2 = pk(k, k), c2 = pk(c, c);
  f32x2 acc[4] = {pk(0.0f, 0.0f), pk(0.0f, 0.0f), pk(0.0f, 0.0f), pk(0.0f, 0.0f)};
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float a0, a1;
      if (BF16) {
        upk(fma2(pk(bf_lo(w[q]), bf_hi(w[q])), k2, c2), a0, a1);
      } else {
        if (q >= 2) break;
        upk(fma2(pk(__uint_as_float(w[2 * q]), __uint_as_float(w[2 * q + 1])), k2, c2), a0, a1);
      }
      acc[(j * 4 + q) & 3] = add2(acc[(j * 4 + q) & 3], pk(ex2(a0), ex2(a1)));
    }
  }
  s = add2(s, add2(add2(acc[0], acc[1]), add2(acc[2], acc[3])));
}

// Pass-1 greedy update: running max and the lowest index holding it.
template <bool BF16>
__device__ __forceinline__ void argmax_update(const uint4& v, int base, float& m, int& idx, float& mx) {
  constexpr int E = BF16 ? 8 : 4;
  const float vm = vec_max<BF16>(v);
  mx = max_nan(mx, vm);
  if (vm > m) {
#pragma unroll
    for (int e = E - 1; e >= 0; --e)
      if (vec_get<BF16>(v, e) == vm) idx = base + e;
    m = vm;
  }
}

// Residual weights max(0, p - q) of element pair e, e+1 of a target vector and its draft vector,
// p and q normalised inside the exponent (ct, cd), two logits per packed instruction.
template <bool BF16>
__device__ __forceinline__ void resid_pair(const uint4& t, const uint4& d, int e, f32x2 k2, f32x2 c2,
                                           float& w0, float& w1) {
  float a0, b0, a1, b1;
  upk(fma2(pk(vec_get<BF16>(t, e), vec_get<BF16>(d, e)), k2, c2), a0, b0);
  upk(fma2(pk(vec_get<BF16>(t, e + 1), vec_get<BF16>(d, e + 1)), k2, c2), a1, b1);
  upk(sub2(pk(ex2(a0), ex2(a1)), pk(ex2(b0), ex2(b1))), w0, w1);
  w0 = fmaxf(w0, 0.0f);
  w1 = fmaxf(w1, 0.0f);
}

// Sum of the residual weights of one vector pair (the order the draw's rescan reproduces).
template <bool BF16>
__device__ __forceinline__ float resid_vec_sum(const uint4& t, const uint4& d, f32x2 k2, f32x2 c2) {
  constexpr int E = BF16 ? 8 : 4;
  float w[E];
#pragma unroll
  for (int e = 0; e < E; e += 2) resid_pair<BF16>(t, d, e, k2, c2, w[e], w[e + 1]);
#pragma unroll
  for (int h = 1; h < E; h *= 2) {
#pragma unroll
    for (int e = 0; e < E; e += 2 * h) w[e] += w[e + h];
  }
  return w[0];
}

// Sum of the unnormalised p weights exp2(z k + cb) of one vector.
template <bool BF16>
__device__ __forceinline__ float p_vec_sum(const uint4& t, float k, float cb) {
  constexpr int E = BF16 ? 8 : 4;
  float s = 0.0f;
#pragma unroll
  for (int e = 0; e < E; ++e) s += ex2(fmaf(vec_get<BF16>(t, e), k, cb));
  return s;
}

// ------------------------------------------------------------------------------------------------
// Row scalars and row errors
// ------------------------------------------------------------------------------------------------

// Writes the all-error outputs of row b (one full warp).
__device__ __forceinline__ void write_row_error(const Params& P, int b, int lane) {
  const int G = P.G;
  for (int j = lane; j <= G; j += 32) P.out_tokens[(size_t)b * (G + 1) + j] = -1;
  for (int j = lane; j < G; j += 32) {
    if (P.out_alpha) P.out_alpha[(size_t)b * G + j] = 0.0f;
    if (P.out_p) P.out_p[(size_t)b * G + j] = 0.0f;
    if (P.out_q) P.out_q[(size_t)b * G + j] = 0.0f;
  }
  if (lane == 0) P.out_num[b] = -1;
}

// Drafted tokens in [0, V) for i < gamma_b, and (sampled rows) the used uniforms in [0, 1). Every
// lane of the warp returns the same answer.
__device__ __forceinline__ bool row_scalars_ok(const Params& P, int b, int gb, bool greedy, int lane) {
  const int G = P.G;
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
  return __all_sync(kFull, good);
}

// ------------------------------------------------------------------------------------------------
// Positions of the batch
// ------------------------------------------------------------------------------------------------

struct Pos {
  int b, i, gb;
  float T;
  bool len_ok, t_ok, greedy, load, two, oh;   // two: a draft row is read; oh: one-hot draft
};

// Slot s in position-major order (s = i * B + b): the slots a cluster strides over mix every
// position index, so ragged rows (fewer positions at large i) and the cheaper bonus positions
// spread evenly over the clusters.
// kMask: a filtered launch, where a sampled row also needs top_p > 0.
template <bool kMask = false>
__device__ __forceinline__ Pos classify(const Params& P, int s) {
  Pos p;
  p.i = s / P.B;
  p.b = s - p.i * P.B;
  if (P.tree) {                       // tree nodes: greedy positions 0 .. size-1 of the row
    p.gb = (P.tsize ? __ldg(P.tsize + p.b) : P.G + 1) - 1;
    p.T = 0.0f;
    p.len_ok = p.gb >= 0 && p.gb <= P.G;
    p.greedy = p.t_ok = true;
    p.load = p.len_ok && p.i <= p.gb;
    p.two = p.oh = false;
    return p;
  }
  p.gb = P.draft_len ? __ldg(P.draft_len + p.b) : P.G;
  p.T = __ldg(P.temperature + p.b);
  p.len_ok = p.gb >= 0 && p.gb <= P.G;
  p.greedy = (p.T == 0.0f);
  p.t_ok = p.greedy || (p.T >= FLT_MIN && p.T <= FLT_MAX);   // NaN fails both
  p.load = p.len_ok && p.t_ok && p.i <= p.gb;
  p.two = p.load && !p.greedy && p.i < p.gb && !P.onehot;
  p.oh = p.load && !p.greedy && p.i < p.gb && P.onehot;
  if (kMask && P.listed && __ldg(P.listed + p.b) != 0) {   // verified from its kept lists
    p.len_ok = p.t_ok = true;
    p.load = p.two = p.oh = false;
    return p;
  }
  if (kMask && !p.greedy && P.top_p) {
    const float pp = __ldg(P.top_p + p.b);
    if (!(pp > 0.0f)) {                        // NaN fails too
      p.t_ok = false;
      p.load = p.two = p.oh = false;
    }
  }
  return p;
}

// ------------------------------------------------------------------------------------------------
// Finish a position (one full warp of the CTA that holds the position's final result): outputs of
// the position, its record, its arrival on the row counter and, for the row's last arrival, the
// row's emit: k = first rejected position (else gamma_b), tokens x_0..x_{k-1} then the correction
// or bonus token ([R] One round, steps 3-5). The counter scheme needs no waiting: the arrivals are
// ordered by release fences and the last one acquires.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void finish_position(const Params& P, int b, int i, int gb, int cand,
                                                int flags, float alpha, float px, float qx,
                                                int lane) {
  const int G = P.G, G1 = G + 1;
  if (lane == 0 && i < gb) {
    if (P.out_alpha) P.out_alpha[(size_t)b * G + i] = alpha;
    if (P.out_p) P.out_p[(size_t)b * G + i] = px;
    if (P.out_q) P.out_q[(size_t)b * G + i] = qx;
  }
  if (i == gb) {
    for (int j = gb + lane; j < G; j += 32) {   // padding positions of the row
      if (P.out_alpha) P.out_alpha[(size_t)b * G + j] = 0.0f;
      if (P.out_p) P.out_p[(size_t)b * G + j] = 0.0f;
      if (P.out_q) P.out_q[(size_t)b * G + j] = 0.0f;
    }
  }
  unsigned old = 0;
  __syncwarp();
  if (lane == 0) {
    P.rec[(size_t)b * G1 + i] = make_int2(cand, flags | kFlagDone);
    __threadfence();
    old = atomicAdd(P.cnt + b, 1u);
  }
  old = __shfl_sync(kFull, old, 0);
  if (old != static_cast<unsigned>(gb)) return;
  __threadfence();

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
  err = err || tok_k < 0;
  __syncwarp();
  for (int j = lane; j <= gb; j += 32) P.rec[(size_t)b * G1 + j] = make_int2(0, 0);  // leave zeros
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
    P.cnt[b] = 0u;                                     // leave the workspace zeroed
  }
}

// ------------------------------------------------------------------------------------------------
// Greedy tree verification: the row's outputs when the tree itself is invalid, and the finish of
// one node (its argmax recorded, then, for the row's last node, the walk of the tree).
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void write_tree_row_error(const Params& P, int b, int lane) {
  const int N = P.G + 1;
  for (int j = lane; j < N; j += 32) {
    P.out_path[(size_t)b * N + j] = -1;
    if (P.out_pred) P.out_pred[(size_t)b * N + j] = -1;
  }
  for (int j = lane; j <= N; j += 32) P.out_tokens[(size_t)b * (N + 1) + j] = -1;
  if (lane == 0) P.out_plen[b] = -1;
}

// [B] "Inference: distillation and speculative decoding" -- Medusa: the root (node 0) is the
// target's own next token; a node is accepted when its parent is accepted and its token equals the
// target's argmax at the parent; the longest accepted path is kept (the lowest node index among
// the deepest), and the target's argmax at its last node is the next token. `scr` is 2 *
// kMaxTreeNodes ints of the calling warp's shared memory. One full warp.
__device__ __forceinline__ void finish_tree_node(const Params& P, int b, int i, int nb, int cand,
                                                 int bad, int* scr, int lane) {
  const int N = P.G + 1;
  unsigned old = 0;
  __syncwarp();
  if (lane == 0) {
    P.rec[(size_t)b * N + i] = make_int2(cand, (bad ? kFlagBad : 0) | kFlagDone);
    __threadfence();
    old = atomicAdd(P.cnt + b, 1u);
  }
  old = __shfl_sync(kFull, old, 0);
  if (old != static_cast<unsigned>(nb - 1)) return;
  __threadfence();
  int* pred = scr;                    // target argmax per node
  int* len = scr + kMaxTreeNodes;     // nodes on the accepted path ending at a node, 0 if rejected
  bool err = false;
  for (int j = lane; j < nb; j += 32) {
    const int2 r = __ldcg(P.rec + (size_t)b * N + j);
    pred[j] = r.x;
    const int t = __ldg(P.ttok + (size_t)b * N + j);
    const int pa = __ldg(P.tparent + (size_t)b * N + j);
    err |= (r.y & kFlagBad) || t < 0 || t >= P.V || (j == 0 ? pa != -1 : (pa < 0 || pa >= j));
  }
  err = __any_sync(kFull, err);
  for (int j = lane; j < nb; j += 32) P.rec[(size_t)b * N + j] = make_int2(0, 0);   // leave zeros
  __syncwarp();
  int best = 0, blen = 1;
  if (lane == 0 && !err) {
    len[0] = 1;
    for (int j = 1; j < nb; ++j) {
      const int pa = __ldg(P.tparent + (size_t)b * N + j);
      const int t = __ldg(P.ttok + (size_t)b * N + j);
      len[j] = (len[pa] > 0 && t == pred[pa]) ? len[pa] + 1 : 0;
      if (len[j] > blen) {
        best = j;
        blen = len[j];
      }
    }
  }
  __syncwarp();
  best = __shfl_sync(kFull, best, 0);
  blen = __shfl_sync(kFull, blen, 0);
  if (err) {
    write_tree_row_error(P, b, lane);
  } else {
    if (lane == 0) {
      int node = best;
      for (int d = blen - 1; d >= 0; --d) {     // root first: fill from the end of the path
        P.out_path[(size_t)b * N + d] = node;
        P.out_tokens[(size_t)b * (N + 1) + d] = __ldg(P.ttok + (size_t)b * N + node);
        node = d > 0 ? __ldg(P.tparent + (size_t)b * N + node) : node;
      }
      P.out_tokens[(size_t)b * (N + 1) + blen] = pred[best];
      P.out_plen[b] = blen;
    }
    for (int j = blen + lane; j < N; j += 32) P.out_path[(size_t)b * N + j] = -1;
    for (int j = blen + 1 + lane; j <= N; j += 32) P.out_tokens[(size_t)b * (N + 1) + j] = -1;
    if (P.out_pred)
      for (int j = lane; j < N; j += 32) P.out_pred[(size_t)b * N + j] = j < nb ? pred[j] : -1;
  }
  if (lane == 0) P.cnt[b] = 0u;                  // leave the workspace zeroed
}

// Whether a position of row b before position i has already recorded a rejection (visible to this
// thread now; one full warp, every lane gets the answer). A rejected or bonus position after such
// a rejection is never emitted, so its draw can be skipped. Records not yet visible read as
// "no rejection", which only means the draw is done.
__device__ __forceinline__ bool earlier_rejection(const Params& P, int b, int i, int lane) {
  bool rej = false;
  for (int j = lane; j < i; j += 32) {
    const int f = __ldcg(&P.rec[(size_t)b * (P.G + 1) + j].y);
    rej |= (f & kFlagDone) && !(f & kFlagAccept);
  }
  return __any_sync(kFull, rej);
}

// ------------------------------------------------------------------------------------------------
// Draws inside one CTA's chunk
// ------------------------------------------------------------------------------------------------

// The vector with element e set to -inf (a one-hot draft's token, left out of a sum).
template <bool BF16>
__device__ __forceinline__ uint4 mask_elem(uint4 v, int e) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (BF16) {
      if (e == 2 * q) w[q] = (w[q] & 0xffff0000u) | 0xff80u;
      if (e == 2 * q + 1) w[q] = (w[q] & 0x0000ffffu) | 0xff800000u;
    } else if (e == q) {
      w[q] = 0xff800000u;
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Sum over the G consecutive lanes of a group (vectors u, u+1, ... of a chunk sit in consecutive
// lanes); every lane of the group gets the total.
template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = 1; o < G; o <<= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// The draw inside this CTA's chunk (kNT consumer threads meeting at named barrier kBarId; `sm`
// provides scan_wt, scan_slot, widx (one entry per warp), dj, dbefore, dover). usum[g] holds the weight of vectors u0 + g*kGrp ... +kGrp-1
// (residual or p weights, per `resid`); the token is the first logit whose running weight exceeds
// t_local, else (rounding) the last logit with positive weight. Block-wide prefix sum over the
// group sums, then one reload of the crossing group. Returns the token in warp `finisher` (all its
// lanes); other warps return -1. All consumer threads call it. Token `skip_tok` (if >= 0) has weight 0
// (the usum entries already leave it out).
template <bool BF16, int kGrp, int kNT, int kBarId, bool kMask = false, typename SM>
__device__ int chunk_draw(const float* usum, int cu, int u0, float t_local, const char* rowt,
                          const char* rowd, bool resid, float k, float ct, float cd, float cb,
                          SM& sm, int ctid, int& finisher, int skip_tok = -1,
                          float tau_t = -INFINITY, float tau_d = -INFINITY) {
  constexpr int kCT = kNT, kCW = kNT / 32;
  constexpr int E = BF16 ? 8 : 4;
  const int lane = ctid & 31, cw = ctid >> 5;
  const int cg = (cu + kGrp - 1) / kGrp;
  const int run = (cg + kCT - 1) / kCT;
  const int r0 = min(ctid * run, cg), r1 = min(r0 + run, cg);
  float tsum = 0.0f;
  int last_j = -1;
  for (int j = r0; j < r1; ++j) {
    const float v = usum[j];
    tsum += v;
    if (v > 0.0f) last_j = j;
  }
  const float incl = warp_incl_scan(tsum, lane);
  float excl = __shfl_up_sync(kFull, incl, 1);
  if (lane == 0) excl = 0.0f;
  if (lane == 31) sm.scan_wt[cw] = incl;
  int lj = last_j;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lj = max(lj, __shfl_xor_sync(kFull, lj, o));
  if (lane == 0) sm.widx[cw] = lj;
  named_bar_sync(kBarId, kCT);
  float wexcl = 0.0f;
#pragma unroll
  for (int w2 = 0; w2 < kCW; ++w2)
    if (w2 < cw) wexcl += sm.scan_wt[w2];
  const bool cross = (tsum > 0.0f) && (wexcl + incl > t_local);
  const unsigned m = __ballot_sync(kFull, cross);
  if (lane == 0) sm.scan_slot[cw] = m ? (cw * 32 + __ffs(m) - 1) : INT_MAX;
  named_bar_sync(kBarId, kCT);
  int win = INT_MAX, best_j = -1;
#pragma unroll
  for (int w2 = 0; w2 < kCW; ++w2) {
    win = min(win, sm.scan_slot[w2]);
    best_j = max(best_j, sm.widx[w2]);
  }
  // The crossing vector and the weight before it (winner thread), else the last positive vector.
  if (win != INT_MAX && ctid == win) {
    float c = wexcl + excl;
    int lastpos = -1, vj = -1;
    float c_last = c, before = 0.0f;
    for (int j = r0; j < r1; ++j) {
      const float v = usum[j];
      if (v > 0.0f) {
        if (c + v > t_local) {
          vj = j;
          before = c;
          break;
        }
        lastpos = j;
        c_last = c;
        c += v;
      }
    }
    const bool over = vj < 0;        // rounding: the run's sums crossed, its vectors did not
    sm.dj = over ? lastpos : vj;
    sm.dbefore = over ? c_last : before;
    sm.dover = over;
  } else if (win == INT_MAX && ctid == 0) {
    sm.dj = best_j;
    sm.dbefore = 0.0f;
    sm.dover = 1;
  }
  named_bar_sync(kBarId, kCT);   // after this no thread reads usum: the caller may reuse it
  finisher = (win == INT_MAX) ? 0 : (win >> 5);
  if (cw != finisher) return -1;
  const int vj = sm.dj;
  const float before = sm.dbefore;
  const bool overrun = sm.dover != 0;
  int tok = -1;
  if (lane == 0 && vj >= 0) {
    // Scan the group's vectors in index order: the first logit whose running weight exceeds the
    // threshold, else the last positive one.
    const f32x2 k2 = pk(k, k), c2 = pk(ct, cd);
    const int ga = u0 + vj * kGrp, gz = min(ga + kGrp, u0 + cu);
    float c = before;
    int pick = -1, lastp = -1;
    for (int u = ga; u < gz && (pick < 0 || overrun); ++u) {
      uint4 t = ld_stream_v4(reinterpret_cast<const uint4*>(rowt) + u);
      if (skip_tok >= 0 && u == skip_tok / E) t = mask_elem<BF16>(t, skip_tok - u * E);   // weight 0
      if (kMask) t = mask_below<BF16>(t, tau_t);                  // filtered rows
      uint4 d = resid ? ld_stream_v4(reinterpret_cast<const uint4*>(rowd) + u) : t;
      if (kMask && resid) d = mask_below<BF16>(d, tau_d);
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        float w0, w1;
        if (resid) {
          resid_pair<BF16>(t, d, e, k2, c2, w0, w1);
        } else {
          w0 = ex2(fmaf(vec_get<BF16>(t, e), k, cb));
          w1 = ex2(fmaf(vec_get<BF16>(t, e + 1), k, cb));
        }
        if (w0 > 0.0f) {
          lastp = u * E + e;
          c += w0;
          if (pick < 0 && c > t_local) pick = u * E + e;
        }
        if (w1 > 0.0f) {
          lastp = u * E + e + 1;
          c += w1;
          if (pick < 0 && c > t_local) pick = u * E + e + 1;
        }
      }
    }
    if (pick < 0 || overrun) pick = lastp;
    tok = pick;
  }
  return __shfl_sync(kFull, tok, 0);
}

// ------------------------------------------------------------------------------------------------
// Host-side launchers (defined in the kernel translation units)
// ------------------------------------------------------------------------------------------------

// Every check spec_verify_ex makes before it enqueues anything (sizes, dtype, pointers, alignment,
// the row layout, the device), without the workspace: the status it would return, or SV_OK.
int verify_args_status(const void* target_logits, const void* draft_logits,
                       const int32_t* draft_tokens, const int32_t* draft_len,
                       const float* temperature, const float* uniforms, int32_t* out_tokens,
                       int32_t* out_num_emitted, float* out_alpha, float* out_p_draft,
                       float* out_q_draft, int32_t B, int32_t gamma_max, int32_t V, int32_t dtype);

// spec_verify_ex with the streaming path's chunks planned as for a batch of plan_slots position
// slots (0: this batch's own).
int verify_ex_planned(const void* target_logits, const void* draft_logits,
                      const int32_t* draft_tokens, const int32_t* draft_len,
                      const float* temperature, const float* uniforms, int32_t* out_tokens,
                      int32_t* out_num_emitted, float* out_alpha, float* out_p_draft,
                      float* out_q_draft, int32_t B, int32_t gamma_max, int32_t V, int32_t dtype,
                      void* workspace, size_t workspace_bytes, void* cuda_stream,
                      long long plan_slots);

// Element path (any alignment, V <= 16 * 512 * 32): one cluster per position slot.
cudaError_t launch_element(const Params& P, bool bf16, int vpt_index, cudaStream_t stream);
// Streaming path (16-byte aligned rows): persistent clusters fed by bulk copies.
cudaError_t launch_stream(Params P, bool bf16, cudaStream_t stream);
// Clusters of `C` CTAs of the streaming kernel that fit on the current device at once (masked: the
// instantiation of filtered verification).
cudaError_t stream_max_clusters(bool bf16, bool wide, int C, int* n, bool masked = false);
// Per-row thresholds of top-k / top-p filtering (16-byte aligned rows): tau [B * (2G + 1)], target
// rows [B, G+1] then draft rows [B, G]. rows: a zeroed device counter the CTAs claim rows from (it
// ends at rows + grid size), or null for a static split.
int threshold_rows(const Params& P);
// lists / list_n (or null): per threshold row, kList (index, logit bits) entries and their count;
// a top-k row solved on its candidate list writes its kept set there when it fits, the other rows
// leave list_n at 0.
cudaError_t launch_threshold(const Params& P, bool bf16, float* tau, unsigned* rows, int2* lists,
                             int* list_n, cudaStream_t stream);
// Verifies the filtered batch rows whose logit rows all have kept lists, and marks them in listed.
cudaError_t launch_listed(const Params& P, const int2* lists, const int* list_n, int* listed,
                          cudaStream_t stream);

}  // namespace sv
