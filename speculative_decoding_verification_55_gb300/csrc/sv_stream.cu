// Streaming path of the sm_103a verifier (rows of 16-byte multiples): persistent thread-block
// clusters fed by bulk copies.
//
// Work split. A position (b, i) of the batch is one target row (plus the draft row for a drafted
// position) of V logits. Each cluster of C CTAs owns every nclusters-th position slot; CTA r of the
// cluster owns the r-th contiguous chunk of every row it touches. Four or five CTAs share an SM, so
// one CTA's exchanges and barriers overlap the others' arithmetic. A CTA is 4 consumer warps and
// one producer warp.
//
// Producer warp (one thread). Walks the cluster's positions and streams this CTA's chunks through a
// ring of kNumSlots x kSlotBytes shared-memory slots with cp.async.bulk (the TMA engine), one full/empty
// mbarrier pair per slot. It runs ahead of the consumers by the ring's capacity, so HBM keeps
// streaming while the consumers exchange partial results.
//
// One cluster exchange per position: after pass 1 of position n, every CTA pushes its softmax
// partials of n together with its residual total of the previous drafted position (st.async into
// every peer's shared memory, completing bytes on the peer's mbarrier). The previous position's
// alpha, draw and finish follow that exchange; position n's own residual pass follows it too, and
// n's totals ride on the next exchange.
//
// Consumer warps, per position:
//   pass 1   online softmax of the chunk straight out of the ring: running max (with a
//            NaN-propagating tracker beside it) and sum of exp2((z - m) log2(e) / T); greedy rows:
//            running argmax with the lowest index.
//   xchg     each CTA combines the C records in the same fixed order: global max M, normaliser S
//            (an inclusive scan over ranks = the chunk-level CDF of p), the accept test
//            u < min(1, p(x)/q(x)), the chunk that holds a bonus-draw threshold.
//   pass 2   (drafted positions) the chunk again, copied from L2 where pass 1 left it through
//            the same ring, last block first (each slot half target vectors, half the matching
//            draft vectors):
//            residual weights max(0, p - q), p and q normalised inside the exponent; one sum per
//            group of kGrp 16-byte vectors (4, or 8 for bf16 one-hot launches) is kept in shared
//            memory for the draw. alpha = 1 - W
//            with W the residual mass: sum min(p, q) + sum max(0, p - q) = sum p = 1 ([R] Why the
//            output is exactly the target's).
//   next     the residual chunk totals (inclusive scan over ranks) arrive with the next exchange.
//   draw     the CTA whose chunk holds the inverse-CDF threshold scans its group sums in index
//            order (block-wide prefix sum), reloads the group that crosses the threshold and
//            picks the token inside it. A bonus draw first fills the group sums of p from L2.
//   finish   the CTA holding the position's final result writes it; the row's last position to
//            finish writes the row's outputs (an arrival counter per row, no waiting).
// Every wait is bounded; a wait that gives up sets the status word, marks the rows the CTA was
// working on as errors and ends the CTA's work. The CTAs of a cluster leave together, at a hardware
// cluster barrier that every thread reaches (all waits before it are bounded), so none leaves while
// a peer may still push into its shared memory, and a producer that stopped first lets its own
// in-flight copies land.
//
// The operation: [R] "Speculative decoding", rayaq.ca ml-models -- Mechanics, One round, steps 3-5;
// Why the output is exactly the target's; The greedy case; Implementation. [B]
// brunomaga.github.io "Inference: distillation and speculative decoding" -- Draft-model speculative
// decoding. [C] cgnarendiran.github.io "Speculative decoding" -- The correction that makes it exact.

#include "sv_common.cuh"

namespace sv {
namespace {

// Several CTAs per SM, each 4 consumer warps + 1 producer warp with a ring of 16 KB slots:
// independent position streams per SM, so one CTA's exchange waits overlap another's arithmetic.
// bf16 logits: five CTAs per SM with two slots each (V=256000: 1470 vs 1497 us with four CTAs and
// three slots; V=128256: 72.8 vs 78.2 us). fp32 logits: four CTAs with three slots (five: 524 vs
// 511 us at V=152064).
#ifndef SV_STREAM_CONSUMER_WARPS
#define SV_STREAM_CONSUMER_WARPS 4
#endif
#ifndef SV_STREAM_RING_SLOTS_BF16
#define SV_STREAM_RING_SLOTS_BF16 2
#endif
#ifndef SV_STREAM_CTAS_PER_SM_BF16
#define SV_STREAM_CTAS_PER_SM_BF16 5
#endif
#ifndef SV_STREAM_RING_SLOTS_F32
#define SV_STREAM_RING_SLOTS_F32 3
#endif
#ifndef SV_STREAM_CTAS_PER_SM_F32
#define SV_STREAM_CTAS_PER_SM_F32 4
#endif
constexpr int kCW = SV_STREAM_CONSUMER_WARPS;   // consumer warps
constexpr int kCT = kCW * 32;                 // consumer threads
constexpr int kThreadsS = kCT + 32;           // plus the producer warp
#ifndef SV_STREAM_SLOT_BYTES
#define SV_STREAM_SLOT_BYTES 16384
#endif
// Consecutive 16-byte vectors summed into one entry of the draw's weight table.
#ifndef SV_STREAM_GROUP
#define SV_STREAM_GROUP 4
#endif
constexpr int kSlotBytes = SV_STREAM_SLOT_BYTES;
constexpr int kSlotUnits = kSlotBytes / 16;
template <bool BF16>
constexpr int kSlotsOf = BF16 ? SV_STREAM_RING_SLOTS_BF16 : SV_STREAM_RING_SLOTS_F32;
template <bool BF16>
constexpr int kCtasPerSm = BF16 ? SV_STREAM_CTAS_PER_SM_BF16 : SV_STREAM_CTAS_PER_SM_F32;
constexpr int kMaxSlots = SV_STREAM_RING_SLOTS_BF16 > SV_STREAM_RING_SLOTS_F32
                              ? SV_STREAM_RING_SLOTS_BF16
                              : SV_STREAM_RING_SLOTS_F32;
static_assert(kSlotUnits % kCT == 0, "a ring slot splits evenly over the consumer threads");
// A residual-pass slot holds kHalfUnits target vectors and the matching kHalfUnits draft vectors.
constexpr int kHalfUnits = kSlotUnits / 2;
static_assert(kHalfUnits % kCT == 0, "a residual slot splits evenly over the consumer threads");
// Draw groups: kGrpNarrow vectors per group, or kGrpWide for bf16 one-hot launches, which take
// chunks twice as long (the group table keeps its size).
constexpr int kGrpNarrow = SV_STREAM_GROUP;
constexpr int kGrpWide = 8;
static_assert(kGrpNarrow == 1 || kGrpNarrow == 2 || kGrpNarrow == 4 || kGrpNarrow == 8,
              "groups of lanes for a shuffle sum");
static_assert(kHalfUnits % kGrpWide == 0 && kHalfUnits % kGrpNarrow == 0,
              "a vector group never straddles two ring slots");
template <bool BF16, int G>
constexpr int kMaxGroupsOf = (stream_max_units(BF16, G == kGrpWide) + G - 1) / G;
// ring, then the draw's group weights
template <bool BF16, int G>
constexpr int kDynBytesOf = kSlotBytes * kSlotsOf<BF16> + kMaxGroupsOf<BF16, G> * 4;
constexpr int kConsumerBar = 1;               // named barrier of the consumer warps
#ifndef SV_STREAM_STOP_POLL
#define SV_STREAM_STOP_POLL 64
#endif
constexpr int kStopPoll = SV_STREAM_STOP_POLL;   // producer polls between looks at the stop flag
static_assert((kStopPoll & (kStopPoll - 1)) == 0, "a power of two");

enum : unsigned { kStatusTimeout = 1u };

struct Shared {
  uint64_t full[kMaxSlots];
  uint64_t empty[kMaxSlots];
  uint64_t xbar[2];                  // exchange: bytes pushed by every CTA complete it, by parity
  float4 xrec[2][kMaxCluster];       // per rank: (m_p, s_p, m_q, s_q), or (argmax value, index)
  uint2 xaux[2][kMaxCluster];        // per rank: (bad flag, residual total of the pending position)
  float4 wpart[kCW];                 // warp partials
  int wbad[kCW];
  int widx[kCW];
  float wsum2[kCW];
  float scan_wt[kCW];
  int scan_slot[kCW];
  int stop;                          // set by any thread that gave up a wait
  int stop_snap;                     // its value as published by consumer warp 0 under a barrier
  // broadcast from consumer warp 0 after an exchange: the current position ...
  float k, ct, cd, cb;               // log2(e)/T; exponent offsets of p, q and of unnormalised p
  float px, qx, t_local, p_tlocal;
  int acc, bad, cand, draw_chunk, p_chunk;
  int resid_mass;                    // one-hot drafts: p without x has positive mass
  int tree_scr[2 * kMaxTreeNodes];   // the tree walk at a row's end (consumer warp 0)
  // ... and the pending drafted position whose residual totals this exchange carried
  float pend_alpha, pend_tlocal;
  int pend_chunk, pend_resid;
  // the draw's crossing vector, handed from the thread that found it to the finishing warp
  int dj, dover;
  float dbefore;
  int skip;                          // the drawing CTA saw an earlier rejection in the row
  // the pending drafted position (kept here, not in registers, to leave room for the hot loops)
  struct {
    const char* rt;
    const char* rd;
    int b, i, gb, acc, bad, p_chunk, fin;
    float k, ct, cd, cb, px, qx, p_tlocal, u_res, tau_t, tau_d;
  } pend;
};

__device__ __forceinline__ void set_status(const Params& P, Shared& sm, unsigned code) {
  atomicOr(P.status, code);
  sm.stop = 1;
}

// Bytes every CTA pushes into every CTA of its cluster per exchange: one float4 record and one uint2.
constexpr uint32_t kXchBytes = 24;

// kMask: filtered verification. Every logit below its row's threshold P.tau reads as -inf (the
// thresholds come from the threshold kernel): the softmax of the kept logits is the filtered
// distribution, and the rest of the path is unchanged.
template <bool BF16, int kGrp, bool kMask>
__global__ void __launch_bounds__(kThreadsS, kCtasPerSm<BF16>) sv_stream_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ Shared sm;
  constexpr int kNumSlots = kSlotsOf<BF16>;
  constexpr int kRingBytes = kSlotBytes * kNumSlots;
  constexpr size_t ES = BF16 ? 2 : 4;
  constexpr int E = BF16 ? 8 : 4;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = static_cast<int>(cluster_rank());
  const int C = P.C, G = P.G, G1 = G + 1;
  const int cid = static_cast<int>(blockIdx.x) / C;
  const int total = P.B * G1;
  const int u0 = min(rank * P.per, P.units);
  const int u1 = min(u0 + P.per, P.units);
  const int cu = u1 - u0;
  const int nsl = (cu + kSlotUnits - 1) / kSlotUnits;      // pass-1 slots per row
  const int nsl2 = (cu + kHalfUnits - 1) / kHalfUnits;     // residual-pass slots per position
  const size_t Vs = static_cast<size_t>(P.V);
  float* usum = reinterpret_cast<float*>(dyn + kRingBytes);   // the draw's group weights

  if (tid == 0) {
    for (int s = 0; s < kNumSlots; ++s) {
      mbar_init(smem_addr(&sm.full[s]), 1);
      mbar_init(smem_addr(&sm.empty[s]), kCW);
    }
    for (int s = 0; s < 2; ++s) mbar_init(smem_addr(&sm.xbar[s]), 1);
    sm.stop = 0;
    sm.stop_snap = 0;
    fence_mbarrier_init_cluster();
  }
  cluster_sync_all();                      // every CTA's barriers exist before any remote arrival

  const uint32_t ring_addr = smem_addr(dyn);

  // ------------------------------------------------------------------ producer
  // The whole warp walks the loop in step (so it never diverges and reaches the final cluster
  // barrier together); lane 0 alone arms the barriers and issues the copies.
  if (warp == kCW) {
    uint32_t tc = 0;
    bool ok = true;
    const uint64_t keep = l2_policy_evict_last(), once = l2_policy_evict_first();
    // A free ring slot; gives up when the consumers stopped (looked at every kStopPoll polls) or
    // after the spin limit. Warp-uniform.
    auto acquire = [&](uint32_t slot, uint32_t par) -> bool {
      for (int n = 0; n < kSpinLimit; ++n) {
        if (__all_sync(kFull, mbar_try_wait(smem_addr(&sm.empty[slot]), par))) return true;
        if ((n & (kStopPoll - 1)) == kStopPoll - 1 &&
            __any_sync(kFull, *reinterpret_cast<volatile int*>(&sm.stop) != 0))
          return false;
      }
      return false;
    };
    for (int s = cid; s < total && ok; s += P.nclusters) {
      const Pos p = classify<kMask>(P, s);
      if (!p.load) continue;
      for (int row = 0; row < (p.two ? 2 : 1) && ok; ++row) {
        const char* g = row == 0
            ? static_cast<const char*>(P.zt) + ((size_t)p.b * G1 + p.i) * Vs * ES
            : static_cast<const char*>(P.zd) + ((size_t)p.b * G + p.i) * Vs * ES;
        g += static_cast<size_t>(u0) * 16;
        for (int ks = 0; ks < nsl; ++ks, ++tc) {
          const uint32_t slot = tc % kNumSlots, par = (tc / kNumSlots) & 1;
          if (!acquire(slot, par ^ 1)) {
            ok = false;
            break;
          }
          const uint32_t bytes = static_cast<uint32_t>(min(kSlotUnits, cu - ks * kSlotUnits)) * 16;
          if (lane == 0) {
            mbar_arrive_expect_tx(smem_addr(&sm.full[slot]), bytes);
            // A drafted position's chunks are read again by the residual pass: keep them in L2.
            bulk_g2s(ring_addr + slot * kSlotBytes, g + static_cast<size_t>(ks) * kSlotBytes, bytes,
                     smem_addr(&sm.full[slot]), p.two ? keep : once);
          }
        }
      }
      if (!p.two || !ok) continue;
      // Residual pass of a drafted position: the same chunk again, now from L2, each slot holding
      // kHalfUnits target vectors and the matching draft vectors, last block first (the most
      // recently streamed lines are the likeliest still in L2). These copies depend on nothing the
      // exchange produces, so they land while the consumers wait for it.
      const char* gt = static_cast<const char*>(P.zt) + ((size_t)p.b * G1 + p.i) * Vs * ES + (size_t)u0 * 16;
      const char* gd = static_cast<const char*>(P.zd) + ((size_t)p.b * G + p.i) * Vs * ES + (size_t)u0 * 16;
      for (int ks = 0; ks < nsl2; ++ks, ++tc) {
        const uint32_t slot = tc % kNumSlots, par = (tc / kNumSlots) & 1;
        if (!acquire(slot, par ^ 1)) {
          ok = false;
          break;
        }
        const int blk = nsl2 - 1 - ks;
        const uint32_t bytes = static_cast<uint32_t>(min(kHalfUnits, cu - blk * kHalfUnits)) * 16;
        const size_t off = static_cast<size_t>(blk) * kHalfUnits * 16;
        if (lane == 0) {
          mbar_arrive_expect_tx(smem_addr(&sm.full[slot]), 2 * bytes);
          bulk_g2s(ring_addr + slot * kSlotBytes, gt + off, bytes, smem_addr(&sm.full[slot]), once);
          bulk_g2s(ring_addr + slot * kSlotBytes + kSlotBytes / 2, gd + off, bytes,
                   smem_addr(&sm.full[slot]), once);
        }
      }
    }
    if (!ok && lane == 0) set_status(P, sm, kStatusTimeout);
    // Let the copies already issued land before this CTA can exit (the consumers may have stopped
    // before reading them; when they read every slot, these phases are complete already).
    for (uint32_t t = tc > kNumSlots ? tc - kNumSlots : 0; t < tc; ++t)
      mbar_wait_drain(smem_addr(&sm.full[t % kNumSlots]), (t / kNumSlots) & 1);
    __syncwarp();
  } else {

  // ------------------------------------------------------------------ consumers
  const int ctid = tid;          // 0 .. kCT-1
  const int cw = warp;
  uint32_t tc = 0;               // ring slots consumed
  uint32_t ex = 0;               // exchanges done
  const uint4* ringv = reinterpret_cast<const uint4*>(dyn);

  // The pending drafted position: pass 2 done, its residual chunk totals ride on the next exchange,
  // after which its draw (if rejected) and finish happen. Uniform across the cluster.
  bool pv = false;                 // a pending position exists (its fields are in sm.pend)

  // Group sums of p's unnormalised weights exp2(z k + cb) over this CTA's chunk, from L2; token
  // `excl` (if >= 0) left out.
  auto fill_p_sums = [&](const char* rt, float kk, float cbv, int excl, float tau_r = -INFINITY) {
    const uint4* vt = reinterpret_cast<const uint4*>(rt) + u0;
    const int xu = excl >= 0 ? excl / E - u0 : -1;     // the chunk-local vector holding excl
    int base = 0;
    for (; base + 8 * kCT <= cu; base += 8 * kCT) {
      uint4 t[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        t[j] = ld_stream_v4(vt + base + ctid + j * kCT);
        if (base + ctid + j * kCT == xu) t[j] = mask_elem<BF16>(t[j], excl - (u0 + xu) * E);
        if (kMask) t[j] = mask_below<BF16>(t[j], tau_r);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float g = group_sum<kGrp>(p_vec_sum<BF16>(t[j], kk, cbv));
        if ((ctid & (kGrp - 1)) == 0) usum[(base + ctid + j * kCT) / kGrp] = g;
      }
    }
    for (; base < cu; base += kCT) {             // uniform trip count: every lane shuffles
      const int uu = base + ctid;
      float sv = 0.0f;
      if (uu < cu) {
        uint4 t = ld_stream_v4(vt + uu);
        if (uu == xu) t = mask_elem<BF16>(t, excl - (u0 + xu) * E);
        if (kMask) t = mask_below<BF16>(t, tau_r);
        sv = p_vec_sum<BF16>(t, kk, cbv);
      }
      const float g = group_sum<kGrp>(sv);
      if ((ctid & (kGrp - 1)) == 0 && uu < cu) usum[uu / kGrp] = g;
    }
  };

  // One cluster exchange (consumer warp 0 pushes and combines; every consumer thread calls it).
  // It carries the current position's pass-1 partials (has_cur) and the pending position's
  // residual total (pv), and broadcasts the combined results through shared memory.
  auto exchange = [&](bool has_cur, int kind, const Pos& p, int x, float k, float zx_t, float zx_d,
                      float u_acc, float u_res, float u_bon) {
    const uint32_t par = ex & 1, ph = (ex >> 1) & 1;
    ++ex;
    if (cw == 0) {
      // The pending position's CTA residual total (its warp partials are ordered by the barrier
      // every consumer passed before this exchange).
      // Reductions over the kCW warp partials (lanes below kCW), then broadcast from lane 0 to the
      // lanes that push.
      const float pw = pv ? __shfl_sync(kFull, lanes_sum(lane < kCW ? sm.wsum2[lane] : 0.0f, kCW), 0) : 0.0f;
      float4 rec = make_float4(-INFINITY, 0.0f, -INFINITY, 0.0f);
      int rbad = 0;
      if (has_cur) {
        if (kind == kArgmax) {
          float v = lane < kCW ? sm.wpart[lane].x : -INFINITY;
          int ii = lane < kCW ? sm.widx[lane] : INT_MAX;
          lanes_argmax(v, ii, kCW);
          rec = make_float4(__shfl_sync(kFull, v, 0), __int_as_float(__shfl_sync(kFull, ii, 0)), 0.0f, 0.0f);
        } else {
          const float4 w = lane < kCW ? sm.wpart[lane] : make_float4(-INFINITY, 0.0f, -INFINITY, 0.0f);
          const float Mct = lanes_max(w.x, kCW), Mcd = lanes_max(w.z, kCW);
          const float a = (w.y > 0.0f) ? w.y * ex2((w.x - Mct) * k) : 0.0f;
          const float c = (w.w > 0.0f) ? w.w * ex2((w.z - Mcd) * k) : 0.0f;
          const float sa = lanes_sum(a, kCW), sc = lanes_sum(c, kCW);
          rec = make_float4(__shfl_sync(kFull, Mct, 0), __shfl_sync(kFull, sa, 0),
                            __shfl_sync(kFull, Mcd, 0), __shfl_sync(kFull, sc, 0));
        }
        rbad = __any_sync(kFull, lane < kCW && sm.wbad[lane]);
      }
#ifdef SV_TEST_DROP_RANK0_PUSHES
      // Test builds only: rank 0 pushes nothing, so every exchange wait of the cluster runs out.
      if (lane < C && rank != 0) {
#else
      if (lane < C) {
#endif
        const uint32_t bar_r = map_to_rank(smem_addr(&sm.xbar[par]), lane);
        st_async_v4(map_to_rank(smem_addr(&sm.xrec[par][rank]), lane), __float_as_uint(rec.x),
                    __float_as_uint(rec.y), __float_as_uint(rec.z), __float_as_uint(rec.w), bar_r);
        st_async_v2(map_to_rank(smem_addr(&sm.xaux[par][rank]), lane), rbad ? 1u : 0u,
                    __float_as_uint(pw), bar_r);
      }
      if (lane == 0) mbar_arrive_expect_tx(smem_addr(&sm.xbar[par]), kXchBytes * C);
      const bool arrived = mbar_wait_cluster(smem_addr(&sm.xbar[par]), ph);
      if (!arrived) set_status(P, sm, kStatusTimeout);
      const float4 r = lane < C ? sm.xrec[par][lane] : make_float4(-INFINITY, 0.0f, -INFINITY, 0.0f);
      const uint2 au = lane < C ? sm.xaux[par][lane] : make_uint2(0u, 0u);
      const int gbad = __any_sync(kFull, au.x != 0u) || !arrived;
      if (has_cur && kind == kArgmax) {
        float v = lane < C ? r.x : -INFINITY;
        int ii = lane < C ? __float_as_int(r.y) : INT_MAX;
        lanes_argmax(v, ii, C);
        if (lane == 0) {
          sm.bad = gbad || !(v > -INFINITY);
          sm.cand = ii;
          sm.acc = (p.i < p.gb) && (x == ii);
        }
      } else if (has_cur) {
        // Global max and normaliser of p (and q); the chunk-level CDF of p by an inclusive scan.
        // One-hot drafts: the chunks' sums leave x out (the residual p without x, chunk by chunk);
        // x's own term joins the normaliser, against a reference no lower than z(x).
        float Mt = lanes_max(r.x, C);
        const float Md = lanes_max(r.z, C);
        const bool oh = kind == kOneHot;
        if (oh && zx_t > Mt && zx_t < INFINITY) Mt = zx_t;
        const float term_t = (lane < C && r.y > 0.0f) ? r.y * ex2((r.x - Mt) * k) : 0.0f;
        const float incl_t = lanes_incl_scan(term_t, lane, C);
        const float ex_x = oh ? ex2((zx_t - Mt) * k) : 0.0f;   // x's unnormalised weight
        const float St = __shfl_sync(kFull, incl_t, C - 1) + ex_x;
        float excl_t = __shfl_up_sync(kFull, incl_t, 1);
        if (lane == 0) excl_t = 0.0f;
        bool b2 = gbad || !(Mt > -INFINITY && Mt < INFINITY);
        if (oh) b2 = b2 || (zx_t != zx_t) || zx_t == INFINITY;   // x's logit was left out of the scan
        float Sd = 1.0f;
        if (kind == kVerify) {
          const float term_d = (lane < C && r.w > 0.0f) ? r.w * ex2((r.z - Md) * k) : 0.0f;
          Sd = __shfl_sync(kFull, lanes_incl_scan(term_d, lane, C), C - 1);
          b2 = b2 || !(Md > -INFINITY && Md < INFINITY);
        }
        // Chunk of a draw from p with threshold t (the bonus draw, or the residual fallback).
        auto chunk_of = [&](float t, float& t_loc) -> int {
          const unsigned hit = __ballot_sync(kFull, lane < C && term_t > 0.0f && incl_t > t);
          const unsigned pos = __ballot_sync(kFull, lane < C && term_t > 0.0f);
          const int c = hit ? (__ffs(hit) - 1) : (pos ? (31 - __clz(pos)) : 0);
          t_loc = t - __shfl_sync(kFull, excl_t, c);
          return c;
        };
        float tl_b = 0.0f, tl_p = 0.0f;
        // Bonus ([R] One round, step 5); one-hot drafts: the residual p without x, whose chunk CDF
        // is the scan itself ([R] One round, step 4 with q = [v == x]).
        const float Wr = __shfl_sync(kFull, incl_t, C - 1);
        const int cb_chunk = chunk_of(oh ? u_res * Wr : u_bon * St, tl_b);
        // Zero-residual fallback: the draw from p with u[G]; for one-hot drafts p without x has no
        // mass, so that draw is x itself.
        const int cp_chunk = chunk_of(u_res * St, tl_p);
        if (lane == 0) {
          const float ct = -fmaf(Mt, k, log2f(St));
          const float cd = -fmaf(Md, k, log2f(Sd));
          sm.k = k;
          sm.cb = -Mt * k;
          sm.ct = ct;
          sm.cd = cd;
          sm.bad = b2;
          sm.acc = 1;
          sm.px = sm.qx = 0.0f;
          if (kind == kVerify) {
            // [R] One round, step 3: keep x while u < min(1, p(x)/q(x)); q(x) = 0 keeps x when
            // p(x) > 0 and rejects it when p(x) = 0 too (zero target mass is never emitted).
            const float px = ex2(fmaf(zx_t, k, ct));
            const float qx = ex2(fmaf(zx_d, k, cd));
            const float ratio = accept_ratio(px, qx);
            sm.px = px;
            sm.qx = qx;
            sm.acc = u_acc < ratio;
          } else if (oh) {
            // q(x) = 1: keep x while u < p(x); alpha = sum min(p, q) = p(x).
            const float px = __fdividef(ex_x, St);
            sm.px = px;
            sm.qx = 1.0f;
            sm.acc = u_acc < px;
            sm.resid_mass = Wr > 0.0f;
          }
          sm.draw_chunk = (kind == kBonus || oh) ? cb_chunk : -1;
          sm.t_local = tl_b;
          sm.p_chunk = cp_chunk;
          sm.p_tlocal = tl_p;
        }
      }
      if (pv) {
        // The pending position's residual mass W and alpha = 1 - W; on a rejection, the chunk whose
        // inclusive prefix first exceeds u * W ([R] One round, step 4), else (rounding) the last
        // positive chunk; with no residual mass at all, the draw from p picked at its exchange.
        const float w_r = lane < C ? __uint_as_float(au.y) : 0.0f;
        const float incl_w = lanes_incl_scan(w_r, lane, C);
        const float Wt = __shfl_sync(kFull, incl_w, C - 1);
        float excl_w = __shfl_up_sync(kFull, incl_w, 1);
        if (lane == 0) excl_w = 0.0f;
        const float t = sm.pend.u_res * Wt;
        const unsigned hit = __ballot_sync(kFull, lane < C && w_r > 0.0f && incl_w > t);
        const unsigned pos = __ballot_sync(kFull, lane < C && w_r > 0.0f);
        const int c = hit ? (__ffs(hit) - 1) : (pos ? (31 - __clz(pos)) : 0);
        const float tl = t - __shfl_sync(kFull, excl_w, c);
        if (lane == 0) {
          sm.pend_alpha = fminf(1.0f, fmaxf(0.0f, 1.0f - Wt));
          sm.pend_chunk = (sm.pend.acc || sm.pend.bad) ? -1 : (Wt > 0.0f ? c : -2);
          sm.pend_tlocal = tl;
          sm.pend_resid = Wt > 0.0f;
        }
      }
      if (lane == 0) sm.stop_snap = sm.stop;
    }
    named_bar_sync(kConsumerBar, kCT);
  };

  // Draw (if rejected) and finish of the pending position; every consumer thread calls it.
  auto finish_pending = [&]() {
    if (!pv) return;
    pv = false;
    int dch = sm.pend_chunk;
    const float alpha = sm.pend_alpha;
    bool resid = sm.pend_resid != 0;
    float tl = sm.pend_tlocal;
    const int pb = sm.pend.b, pi = sm.pend.i, pgb = sm.pend.gb;
    const float ppx = sm.pend.px, pqx = sm.pend.qx;
    if (dch == -2) {                 // zero residual mass: draw from p with the residual uniform
      dch = sm.pend.p_chunk;
      tl = sm.pend.p_tlocal;
      resid = false;
    }
    if (dch < 0) {
      if (rank == sm.pend.fin && cw == 0)
        finish_position(P, pb, pi, pgb, -1, sm.pend.bad ? kFlagBad : kFlagAccept, alpha, ppx, pqx,
                        lane);
      return;
    }
    if (rank != dch) return;
    if (cw == 0) {
      const bool early = earlier_rejection(P, pb, pi, lane);
      if (lane == 0) sm.skip = early;
    }
    named_bar_sync(kConsumerBar, kCT);
    if (sm.skip) {                   // a rejection earlier in the row: this draw is never emitted
      if (cw == 0) finish_position(P, pb, pi, pgb, -1, 0, alpha, ppx, pqx, lane);
      return;
    }
    const char* prt = sm.pend.rt;
    const char* prd = sm.pend.rd;
    const float pkk = sm.pend.k, pct = sm.pend.ct, pcd = sm.pend.cd, pcb = sm.pend.cb;
    const float ptt = sm.pend.tau_t, ptd = sm.pend.tau_d;
    if (!resid) {
      fill_p_sums(prt, pkk, pcb, -1, ptt);
      named_bar_sync(kConsumerBar, kCT);
    }
    int finisher = 0;
    const int tok = chunk_draw<BF16, kGrp, kCT, kConsumerBar, kMask>(usum, cu, u0, tl, prt, prd, resid, pkk, pct, pcd, pcb, sm,
                                           ctid, finisher, -1, ptt, ptd);
    if (cw == finisher) finish_position(P, pb, pi, pgb, tok, tok < 0 ? kFlagBad : 0, alpha, ppx, pqx,
                                        lane);
  };

  for (int s = cid; s < total; s += P.nclusters) {
    const Pos p = classify<kMask>(P, s);
    if (!p.load) {
      if (!(p.len_ok && p.t_ok) && p.i == 0 && rank == 0 && cw == 0) {
        if (P.tree) write_tree_row_error(P, p.b, lane);
        else write_row_error(P, p.b, lane);
      }
      continue;
    }
    // (tree rows: the tree's parents and tokens are checked by the walk at the row's end)
    const bool ok = P.tree || row_scalars_ok(P, p.b, p.gb, p.greedy, lane);
    const int kind = p.greedy ? kArgmax : (p.two ? kVerify : (p.oh ? kOneHot : kBonus));
    const char* rowt = static_cast<const char*>(P.zt) + ((size_t)p.b * G1 + p.i) * Vs * ES;
    const char* rowd = p.two ? static_cast<const char*>(P.zd) + ((size_t)p.b * G + p.i) * Vs * ES
                             : nullptr;
    const int x = (!P.tree && p.i < p.gb) ? __ldg(P.tokens + (size_t)p.b * G + p.i) : -1;

    // Filtered rows: the thresholds of this position's rows (-inf: nothing dropped).
    float tau_t = -INFINITY, tau_d = -INFINITY;
    if (kMask) {
      tau_t = __ldg(P.tau + (size_t)p.b * G1 + p.i);
      if (p.two) tau_d = __ldg(P.tau + (size_t)P.B * G1 + (size_t)p.b * G + p.i);
    }
    // Early scalar loads for the accept test (their latency hides behind pass 1).
    float zx_t = 0.0f, zx_d = 0.0f, u_acc = 0.0f, u_res = 0.0f, u_bon = 0.0f;
    if (ok && cw == 0 && !p.greedy) {
      const float* ur = P.uniforms + (size_t)p.b * (G + 2);
      u_res = __ldg(ur + G);
      u_bon = __ldg(ur + G + 1);
      if (kind == kVerify || kind == kOneHot) {
        u_acc = __ldg(ur + p.i);
        zx_t = load_logit<BF16>(rowt, x);
      }
      if (kind == kVerify) zx_d = load_logit<BF16>(rowd, x);
      if (kMask) {                 // a drafted token outside a filtered set has probability 0
        if (zx_t < tau_t) zx_t = -INFINITY;
        if (zx_d < tau_d) zx_d = -INFINITY;
      }
    }

    // ---- pass 1 out of the ring ----
    const float k = p.greedy ? 0.0f : kLog2e / p.T;
    float mt = -INFINITY, md = -INFINITY, mxt = -INFINITY, mxd = -INFINITY;
    f32x2 st = pk(0.0f, 0.0f), sd = pk(0.0f, 0.0f);
    int idx = INT_MAX;
    bool timed_out = false;
    for (int row = 0; row < (p.two ? 2 : 1); ++row) {
      for (int ks = 0; ks < nsl; ++ks, ++tc) {
        const uint32_t slot = tc % kNumSlots, par = (tc / kNumSlots) & 1;
        if (!mbar_wait(smem_addr(&sm.full[slot]), par)) timed_out = true;
        const int nu = min(kSlotUnits, cu - ks * kSlotUnits);
        const uint4* src = ringv + slot * kSlotUnits;
        if (ok && !timed_out) {
          constexpr int N = kSlotUnits / kCT;
          const uint32_t ninf = BF16 ? 0xFF80FF80u : 0xFF800000u;
          uint4 v[N];
          if (nu == kSlotUnits) {      // a full slot: no tail to mask
#pragma unroll
            for (int j = 0; j < N; ++j) v[j] = src[ctid + j * kCT];
          } else {
#pragma unroll
            for (int j = 0; j < N; ++j) {
              const int uu = ctid + j * kCT;
              v[j] = uu < nu ? src[uu] : make_uint4(ninf, ninf, ninf, ninf);
            }
          }
          if (kMask && kind != kArgmax) {
            const float tr = row == 0 ? tau_t : tau_d;
#pragma unroll
            for (int j = 0; j < N; ++j) v[j] = mask_below<BF16>(v[j], tr);
          }
          if (kind == kOneHot) {
            // The drafted token's own term is added at the exchange: the chunk sums leave it out,
            // so the residual mass of every chunk (p without x) has no cancellation.
#pragma unroll
            for (int j = 0; j < N; ++j)
              if (u0 + ks * kSlotUnits + ctid + j * kCT == x / E) v[j] = mask_elem<BF16>(v[j], x % E);
          }
          if (kind == kArgmax) {
#pragma unroll
            for (int j = 0; j < N; ++j)
              argmax_update<BF16>(v[j], (u0 + ks * kSlotUnits + ctid + j * kCT) * E, mt, idx, mxt);
          } else if (row == 0) {
            online_update_batch<BF16, N>(v, k, mt, st, mxt);
          } else {
            online_update_batch<BF16, N>(v, k, md, sd, mxd);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.empty[slot]));
      }
    }
    if (timed_out) set_status(P, sm, kStatusTimeout);
    if (!ok) {                       // drafted token or uniform out of range: the row is an error
      if (p.two) {                   // the producer also streamed the residual-pass slots: drain
        for (int ks = 0; ks < nsl2; ++ks, ++tc) {
          const uint32_t slot = tc % kNumSlots, par = (tc / kNumSlots) & 1;
          if (!mbar_wait(smem_addr(&sm.full[slot]), par)) set_status(P, sm, kStatusTimeout);
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&sm.empty[slot]));
        }
      }
      if (p.i == 0 && rank == 0 && cw == 0) write_row_error(P, p.b, lane);
      continue;
    }

    // ---- warp partials ----
    if (kind == kArgmax) {
      warp_argmax(mt, idx);
      const int bad = __any_sync(kFull, (mxt != mxt) || mxt == INFINITY);
      if (lane == 0) {
        sm.wpart[cw] = make_float4(mt, 0.0f, 0.0f, 0.0f);
        sm.widx[cw] = idx;
        sm.wbad[cw] = bad;
      }
    } else {
      float s0, s1;
      upk(st, s0, s1);
      float sT = s0 + s1;
      upk(sd, s0, s1);
      float sD = s0 + s1;
      const float Mwt = warp_max(mt), Mwd = warp_max(md);
      sT = (sT > 0.0f) ? sT * ex2((mt - Mwt) * k) : 0.0f;
      sD = (sD > 0.0f) ? sD * ex2((md - Mwd) * k) : 0.0f;
      sT = warp_sum_lane0(sT);
      sD = warp_sum_lane0(sD);
      const float mxa = max_nan(mxt, mxd);
      const int bad = __any_sync(kFull, (mxa != mxa) || mxa == INFINITY);
      if (lane == 0) {
        sm.wpart[cw] = make_float4(Mwt, sT, Mwd, sD);
        sm.wbad[cw] = bad;
      }
    }
    named_bar_sync(kConsumerBar, kCT);

    // ---- the cluster exchange: this position's softmax partials + the pending residual totals ----
    exchange(true, kind, p, x, k, zx_t, zx_d, u_acc, u_res, u_bon);
    if (sm.stop_snap) {
      // A wait gave up: this position (and the pending one) will never finish, so their rows
      // would never be written. Mark them as errors; the status word tells the caller why.
      if (cw == 0) {
        if (P.tree) write_tree_row_error(P, p.b, lane);
        else write_row_error(P, p.b, lane);
        if (pv && !P.tree) write_row_error(P, sm.pend.b, lane);
      }
      break;
    }
    finish_pending();
    // The CTA that finishes this position when no draw picks one: rotates over the ranks so that
    // the finishing work (records, counters, row emits) does not slow one rank down.
    const int fin = static_cast<int>((ex - 1) % static_cast<uint32_t>(C));

    if (kind == kArgmax && P.tree) {
      if (rank == fin && cw == 0) finish_tree_node(P, p.b, p.i, p.gb + 1, sm.cand, sm.bad, sm.tree_scr, lane);
      continue;
    }
    if (kind == kArgmax) {
      if (rank == fin && cw == 0) {
        const int acc = sm.acc;
        const int flags = (sm.bad ? kFlagBad : 0) | (acc ? kFlagAccept : 0);
        const float a = acc ? 1.0f : 0.0f;
        finish_position(P, p.b, p.i, p.gb, sm.cand, flags, a, a, 1.0f, lane);
      }
      continue;
    }

    const float kk = sm.k, ct = sm.ct, cd = sm.cd, cb = sm.cb;
    const int cbad = sm.bad;

    if (kind == kOneHot) {
      // One-hot draft: finished at its exchange (alpha = p(x) needs no residual pass). On a
      // rejection the residual p without x is drawn by the CTA holding its threshold. With no
      // residual mass the fallback draw from p can only give x (all of p is on x).
      const float apx = sm.px;
      const bool rej = !(cbad || sm.acc);
      if (!rej || !sm.resid_mass) {
        if (rank == fin && cw == 0) {
          if (cbad) finish_position(P, p.b, p.i, p.gb, -1, kFlagBad, 0.0f, 0.0f, 0.0f, lane);
          else if (!rej) finish_position(P, p.b, p.i, p.gb, -1, kFlagAccept, apx, apx, 1.0f, lane);
          else finish_position(P, p.b, p.i, p.gb, x, 0, apx, apx, 1.0f, lane);
        }
      } else if (rank == sm.draw_chunk) {
        const float tl = sm.t_local;
        if (cw == 0) {
          const bool early = earlier_rejection(P, p.b, p.i, lane);
          if (lane == 0) sm.skip = early;
        }
        named_bar_sync(kConsumerBar, kCT);
        if (sm.skip) {               // a rejection earlier in the row: this draw is never emitted
          if (cw == 0) finish_position(P, p.b, p.i, p.gb, -1, 0, apx, apx, 1.0f, lane);
          named_bar_sync(kConsumerBar, kCT);   // sm.skip is read before it is reused
          continue;
        }
        fill_p_sums(rowt, kk, cb, x);
        named_bar_sync(kConsumerBar, kCT);
        int finisher = 0;
        const int tok = chunk_draw<BF16, kGrp, kCT, kConsumerBar, kMask>(usum, cu, u0, tl, rowt, rowd, false, kk, ct, cd, cb, sm,
                                               ctid, finisher, x);
        if (cw == finisher)
          finish_position(P, p.b, p.i, p.gb, tok, tok < 0 ? kFlagBad : 0, apx, apx, 1.0f, lane);
      }
      continue;
    }

    if (kind == kBonus) {
      // Bonus token from p at position gamma_b ([R] One round, step 5).
      const int dch = cbad ? -1 : sm.draw_chunk;
      const float tl = sm.t_local;
      if (dch < 0) {
        if (rank == fin && cw == 0) finish_position(P, p.b, p.i, p.gb, -1, kFlagBad, 0.0f, 0.0f, 0.0f, lane);
      } else if (rank == dch) {
        if (cw == 0) {
          const bool early = earlier_rejection(P, p.b, p.i, lane);
          if (lane == 0) sm.skip = early;
        }
        named_bar_sync(kConsumerBar, kCT);
        if (sm.skip) {               // a rejection earlier in the row: the bonus is never emitted
          if (cw == 0) finish_position(P, p.b, p.i, p.gb, -1, kFlagAccept, 0.0f, 0.0f, 0.0f, lane);
          continue;
        }
        fill_p_sums(rowt, kk, cb, -1, tau_t);
        named_bar_sync(kConsumerBar, kCT);
        int finisher = 0;
        const int tok = chunk_draw<BF16, kGrp, kCT, kConsumerBar, kMask>(usum, cu, u0, tl, rowt, rowd, false, kk, ct, cd, cb, sm,
                                               ctid, finisher, -1, tau_t);
        if (cw == finisher)
          finish_position(P, p.b, p.i, p.gb, tok, (tok < 0 ? kFlagBad : 0) | kFlagAccept, 0.0f, 0.0f,
                          0.0f, lane);
      }
      continue;
    }

    // ---- drafted position: pass 2, the residual weights of the chunk, out of the ring ----
    float W = 0.0f;
    {
      const f32x2 k2 = pk(kk, kk), c2 = pk(ct, cd);
      bool tmo = false;
      for (int ks = 0; ks < nsl2; ++ks, ++tc) {
        const uint32_t slot = tc % kNumSlots, par = (tc / kNumSlots) & 1;
        // Warp-uniform, so that a wait given up by one lane cannot split a group's shuffle.
        if (!__all_sync(kFull, mbar_wait(smem_addr(&sm.full[slot]), par))) tmo = true;
        const int blk = nsl2 - 1 - ks;               // the producer's order: last block first
        const int nu = min(kHalfUnits, cu - blk * kHalfUnits);
        const uint4* st4 = ringv + slot * kSlotUnits;
        const uint4* sd4 = st4 + kHalfUnits;
        if (!cbad && !tmo) {
          // Uniform trip count over the slot (kHalfUnits is a multiple of kCT): every lane of a
          // group takes part in the shuffle; lanes past the chunk's end add zero.
#pragma unroll
          for (int j = 0; j < kHalfUnits / kCT; ++j) {
            const int uu = ctid + j * kCT;
            float sv = 0.0f;
            if (uu < nu) {
              if (kMask) {
                sv = resid_vec_sum<BF16>(mask_below<BF16>(st4[uu], tau_t),
                                         mask_below<BF16>(sd4[uu], tau_d), k2, c2);
              } else {
                sv = resid_vec_sum<BF16>(st4[uu], sd4[uu], k2, c2);
              }
            }
            W += sv;
            const float g = group_sum<kGrp>(sv);
            if ((ctid & (kGrp - 1)) == 0 && uu < nu) usum[(blk * kHalfUnits + uu) / kGrp] = g;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.empty[slot]));
      }
      if (tmo) set_status(P, sm, kStatusTimeout);
    }
    const float ws = warp_sum_lane0(W);
    if (lane == 0) sm.wsum2[cw] = ws;
    // The position becomes pending: its residual totals ride on the next exchange. Consumer
    // thread 0 records it (every consumer reads it only after the next exchange's barrier).
    pv = true;
    if (ctid == 0) {
      sm.pend.b = p.b;
      sm.pend.i = p.i;
      sm.pend.gb = p.gb;
      sm.pend.acc = sm.acc;
      sm.pend.bad = cbad;
      sm.pend.rt = rowt;
      sm.pend.rd = rowd;
      sm.pend.k = kk;
      sm.pend.ct = ct;
      sm.pend.cd = cd;
      sm.pend.cb = cb;
      sm.pend.px = sm.px;
      sm.pend.qx = sm.qx;
      sm.pend.p_chunk = sm.p_chunk;
      sm.pend.p_tlocal = sm.p_tlocal;
      sm.pend.u_res = u_res;
      sm.pend.fin = fin;
      if (kMask) {
        sm.pend.tau_t = tau_t;
        sm.pend.tau_d = tau_d;
      }
    }
  }
  if (pv && !sm.stop_snap) {
    named_bar_sync(kConsumerBar, kCT);   // the last residual partials are in place
    exchange(false, kVerify, Pos{}, -1, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f);
    if (!sm.stop_snap) {
      finish_pending();
    } else if (cw == 0 && !P.tree) {     // the pending position will never finish
      write_row_error(P, sm.pend.b, lane);
    }
  }

  }

  // ---- no CTA leaves while a peer may still write into its shared memory ----
  cluster_sync_all();
}

// bf16 one-hot launches take the wide draw groups; the rest the narrow ones. Filtered launches
// (thresholds given) take the masked instantiation.
const void* stream_fn(bool bf16, bool wide, bool masked = false) {
  if (masked) {
    return bf16 ? reinterpret_cast<const void*>(sv_stream_kernel<true, kGrpNarrow, true>)
                : reinterpret_cast<const void*>(sv_stream_kernel<false, kGrpNarrow, true>);
  }
  if (bf16) {
    return wide ? reinterpret_cast<const void*>(sv_stream_kernel<true, kGrpWide, false>)
                : reinterpret_cast<const void*>(sv_stream_kernel<true, kGrpNarrow, false>);
  }
  return reinterpret_cast<const void*>(sv_stream_kernel<false, kGrpNarrow, false>);
}

int stream_dyn_bytes(bool bf16, bool wide) {
  if (bf16) return wide ? kDynBytesOf<true, kGrpWide> : kDynBytesOf<true, kGrpNarrow>;
  return kDynBytesOf<false, kGrpNarrow>;
}

cudaError_t stream_attrs(const void* fn, int C, bool bf16, bool wide) {
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       stream_dyn_bytes(bf16, wide));
  if (e != cudaSuccess) return e;
  // Several CTAs per SM need the largest shared-memory carveout.
  e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  if (C > 8) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

cudaLaunchConfig_t stream_config(int C, int nclusters, bool bf16, bool wide, cudaStream_t stream,
                                 cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nclusters * C), 1, 1);
  cfg.blockDim = dim3(kThreadsS, 1, 1);
  cfg.dynamicSmemBytes = stream_dyn_bytes(bf16, wide);
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

cudaError_t stream_max_clusters(bool bf16, bool wide, int C, int* n, bool masked) {
  wide = wide && bf16 && !masked;
  const void* fn = stream_fn(bf16, wide, masked);
  const cudaError_t e = stream_attrs(fn, C, bf16, wide);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = stream_config(C, 64, bf16, wide, nullptr, attr);
  return cudaOccupancyMaxActiveClusters(n, fn, &cfg);
}

cudaError_t launch_stream(Params P, bool bf16, cudaStream_t stream) {
  const bool masked = P.tau != nullptr;
  const bool wide = bf16 && P.onehot && !masked;
  const void* fn = stream_fn(bf16, wide, masked);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = stream_config(P.C, P.nclusters, bf16, wide, stream, attr);
  void* args[] = {&P};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace sv
