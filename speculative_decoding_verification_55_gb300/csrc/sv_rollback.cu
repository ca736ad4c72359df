// Batched KV-cache rollback after a verification round ([R] "Speculative decoding", rayaq.ca
// ml-models -- Verification attention and the cache: after verification the cache holds entries for
// all gamma + 1 new positions; with k drafts accepted the first n + k + 1 are kept (the prefix, the
// last token, the accepted drafts) and the rest is truncated; the drafter's cache is rolled back the
// same way. [B] brunomaga.github.io "Inference: distillation and speculative decoding" --
// Draft-model speculative decoding: the drafter keeps the prefix of its cache that is still valid).
//
// One CTA per row: thread 0 writes the row's new lengths; when a cache is given, every thread zeroes
// its share of the dropped entries [n + k + 1, n + gamma_b + 1) with 16-byte stores, in order, so a
// row's bytes are written by consecutive threads (coalesced).

#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/spec_verify.h"

namespace {

constexpr int kRollbackThreads = 256;

struct RollbackParams {
  const int32_t* prefix_len;
  const int32_t* draft_len;
  const int32_t* num_emitted;
  const int32_t* drafter_in;
  int32_t* target_out;
  int32_t* drafter_out;
  unsigned char* cache;
  long long row_stride;      // bytes between rows of the cache
  int entry_bytes;
  int cache_entries;         // entries one cache row holds
  int B, G;
};

__global__ void __launch_bounds__(kRollbackThreads) sv_rollback_kernel(const RollbackParams P) {
  const int b = blockIdx.x;
  const int n = __ldg(P.prefix_len + b);
  int g = P.draft_len ? __ldg(P.draft_len + b) : P.G;
  g = min(max(g, 0), P.G);
  const int e = __ldg(P.num_emitted + b);          // k + 1, or -1 for a row error
  const int keep = e >= 1 ? n + e : n;             // n + k + 1; a failed round commits nothing
  if (threadIdx.x == 0) {
    P.target_out[b] = keep;
    if (P.drafter_out) {
      const int d = P.drafter_in ? __ldg(P.drafter_in + b) : keep;
      P.drafter_out[b] = min(d, keep);
    }
  }
  if (!P.cache) return;
  // Dropped entries of this row, clamped to the row's capacity.
  const long long lo = static_cast<long long>(max(keep, 0));
  const long long hi = static_cast<long long>(min(n + g + 1, P.cache_entries));
  if (hi <= lo) return;
  uint4* p = reinterpret_cast<uint4*>(P.cache + P.row_stride * b + lo * P.entry_bytes);
  const long long nv = (hi - lo) * (P.entry_bytes / 16);
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (long long v = threadIdx.x; v < nv; v += kRollbackThreads) p[v] = z;
}

}  // namespace

extern "C" int spec_verify_kv_rollback(const int32_t* prefix_len, const int32_t* draft_len,
                                       const int32_t* out_num_emitted, const int32_t* drafter_len_in,
                                       int32_t* target_len_out, int32_t* drafter_len_out, void* cache,
                                       int64_t cache_row_stride, int32_t entry_bytes,
                                       int32_t cache_entries, int32_t B, int32_t gamma_max,
                                       void* cuda_stream) {
  if (B < 1 || gamma_max < 0 || gamma_max > SV_MAX_GAMMA) return SV_ERR_BAD_SHAPE;
  if (!prefix_len || !out_num_emitted || !target_len_out) return SV_ERR_NULL_POINTER;
  auto mis = [](const void* p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) != 0; };
  if (mis(prefix_len, 4) || mis(draft_len, 4) || mis(out_num_emitted, 4) || mis(drafter_len_in, 4) ||
      mis(target_len_out, 4) || mis(drafter_len_out, 4))
    return SV_ERR_MISALIGNED;
  if (cache) {
    if (entry_bytes <= 0 || cache_entries < 0 || cache_row_stride < static_cast<int64_t>(entry_bytes) * cache_entries)
      return SV_ERR_BAD_SHAPE;
    if (entry_bytes % 16 != 0 || cache_row_stride % 16 != 0 || mis(cache, 16)) return SV_ERR_MISALIGNED;
  }
  RollbackParams P;
  P.prefix_len = prefix_len;
  P.draft_len = draft_len;
  P.num_emitted = out_num_emitted;
  P.drafter_in = drafter_len_in;
  P.target_out = target_len_out;
  P.drafter_out = drafter_len_out;
  P.cache = static_cast<unsigned char*>(cache);
  P.row_stride = cache_row_stride;
  P.entry_bytes = entry_bytes;
  P.cache_entries = cache_entries;
  P.B = B;
  P.G = gamma_max;
  sv_rollback_kernel<<<B, kRollbackThreads, 0, static_cast<cudaStream_t>(cuda_stream)>>>(P);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
