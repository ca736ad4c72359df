// Host-buffer entry point (include/spec_verify.h: spec_verify_staged): stages into device memory
// only the logit rows the accept-or-resample rule reads, runs spec_verify_ex on them and copies the
// outputs back. The rows go in groups: group g + 1 crosses the host link on an internal stream while
// group g verifies on the caller's stream. Page-locked host logits are gathered by a kernel reading
// host memory directly (no per-row copy calls); other host memory goes through one cudaMemcpyAsync
// per run of contiguous rows.
//
// Rows read ([R] "Speculative decoding", rayaq.ca ml-models -- Mechanics, One round, steps 3-5; The
// greedy case): target rows 0..gamma_b of row b (the drafted positions and the bonus position) and,
// for a sampled row, draft rows 0..gamma_b - 1. A greedy row (temperature exactly 0) reads no draft
// logits. Everything past gamma_b is padding.

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/spec_verify.h"
#include "sv_common.cuh"

namespace {

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

bool shape_ok(int32_t B, int32_t G, int32_t V, int32_t dtype) {
  if (B < 1 || G < 0 || G > SV_MAX_GAMMA || V < 1) return false;
  if (dtype != SV_DTYPE_F32 && dtype != SV_DTYPE_BF16) return false;
  // B * (G + 1) * V * s must not overflow int64 (and the staged target tensor must be addressable).
  const unsigned long long s = dtype == SV_DTYPE_BF16 ? 2ull : 4ull;
  const unsigned long long rows = static_cast<unsigned long long>(B) * static_cast<unsigned>(G + 1);
  return rows <= (static_cast<unsigned long long>(INT64_MAX) / s) / static_cast<unsigned>(V);
}

// Byte offsets of the staged tensors inside the staging buffer (each 256-byte aligned).
struct Layout {
  size_t zt, zd, tok, len, temp, u, otok, onum, oalpha, total;
};

Layout layout(int32_t B, int32_t G, int32_t V, int32_t dtype) {
  const size_t s = dtype == SV_DTYPE_BF16 ? 2 : 4;
  const size_t b = static_cast<size_t>(B), g = static_cast<size_t>(G), v = static_cast<size_t>(V);
  Layout L{};
  size_t o = 0;
  L.zt = o;
  o += align256(b * (g + 1) * v * s);
  L.zd = o;
  o += align256(b * g * v * s);
  L.tok = o;
  o += align256(b * g * 4);
  L.len = o;
  o += align256(b * 4);
  L.temp = o;
  o += align256(b * 4);
  L.u = o;
  o += align256(b * (g + 2) * 4);
  L.otok = o;
  o += align256(b * (g + 1) * 4);
  L.onum = o;
  o += align256(b * 4);
  L.oalpha = o;
  o += align256(b * g * 4);
  L.total = o;
  return L;
}

// Visits the contiguous byte runs [off, off + len) of the target and draft tensors that the rule
// reads, merging consecutive rows b whose runs touch (row b with gamma_b = gamma_max ends where row
// b + 1 starts).
template <typename F>
void for_each_run(const int32_t* h_len, const float* h_temp, int32_t b0, int32_t b1, int32_t G,
                  int32_t V, size_t s, F&& visit) {
  const size_t row = static_cast<size_t>(V) * s;
  size_t t_off = 0, t_len = 0, d_off = 0, d_len = 0;
  for (int32_t b = b0; b < b1; ++b) {
    const int32_t g = h_len ? h_len[b] : G;
    if (g < 0 || g > G) continue;
    const size_t to = static_cast<size_t>(b) * (G + 1) * row, tl = static_cast<size_t>(g + 1) * row;
    if (t_len && t_off + t_len == to) {
      t_len += tl;
    } else {
      if (t_len) visit(false, t_off, t_len);
      t_off = to;
      t_len = tl;
    }
    if (g > 0 && h_temp[b] != 0.0f) {
      const size_t dof = static_cast<size_t>(b) * G * row, dl = static_cast<size_t>(g) * row;
      if (d_len && d_off + d_len == dof) {
        d_len += dl;
      } else {
        if (d_len) visit(true, d_off, d_len);
        d_off = dof;
        d_len = dl;
      }
    }
  }
  if (t_len) visit(false, t_off, t_len);
  if (d_len) visit(true, d_off, d_len);
}

// Zero-copy gather: the device reads the logit rows the rule reads straight from page-locked host
// memory (mapped into the device's address space) into the staging buffer, one CTA per position
// slot at a time. The same row selection as for_each_run, taken from the staged copies of draft_len
// and temperature, so the bytes moved are the ones counted on the host. Rows of 16-byte multiples.
constexpr int kGatherThreads = 128;
// One CTA per SM at most: the host link, not the SMs, bounds the gather, and the CTAs stay small
// (128 threads of at most 40 registers, no shared memory: 5,120 registers, which fit beside five
// streaming-kernel CTAs of 160 threads x 72 registers) so that the verification of the previous
// row group runs beside them.
constexpr int kGatherCtasPerSm = 1;

// One row of 16-byte vectors by the CTA, kGatherDepth loads in flight per thread before the stores
// (the host link's latency is long; the bytes in flight set its throughput).
constexpr int kGatherDepth = 6;
__device__ __forceinline__ void copy_row(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                         unsigned row16) {
  constexpr unsigned kStep = kGatherThreads * kGatherDepth;
  const uint4* s = src + threadIdx.x;
  uint4* d = dst + threadIdx.x;
  unsigned u0 = 0;
  for (; u0 + kStep <= row16; u0 += kStep) {
    uint4 v[kGatherDepth];
#pragma unroll
    for (int j = 0; j < kGatherDepth; ++j) v[j] = s[u0 + j * kGatherThreads];
#pragma unroll
    for (int j = 0; j < kGatherDepth; ++j) d[u0 + j * kGatherThreads] = v[j];
  }
  for (unsigned u = u0 + threadIdx.x; u < row16; u += kGatherThreads) dst[u] = src[u];
}

__global__ void __launch_bounds__(kGatherThreads, 12) sv_gather_rows(
    const uint4* __restrict__ zt_h, const uint4* __restrict__ zd_h, uint4* __restrict__ zt_d,
    uint4* __restrict__ zd_d, const int32_t* __restrict__ len, const float* __restrict__ temp,
    int32_t b0, int32_t nb, int32_t G, size_t row16) {
  const long long slots = static_cast<long long>(nb) * (G + 1);
  for (long long s = blockIdx.x; s < slots; s += gridDim.x) {
    const int32_t b = b0 + static_cast<int32_t>(s / (G + 1));
    const int32_t i = static_cast<int32_t>(s - static_cast<long long>(b - b0) * (G + 1));
    const int32_t g = len ? len[b] : G;
    if (g < 0 || g > G || i > g) continue;
    const size_t t0 = (static_cast<size_t>(b) * (G + 1) + i) * row16;
    copy_row(zt_h + t0, zt_d + t0, static_cast<unsigned>(row16));
    if (i < g && temp[b] != 0.0f) {
      const size_t d0 = (static_cast<size_t>(b) * G + i) * row16;
      copy_row(zd_h + d0, zd_d + d0, static_cast<unsigned>(row16));
    }
  }
}

// Device addresses of the host logit buffers when both are page-locked, mapped and 16-byte aligned
// with rows of 16-byte multiples; false otherwise (the copy engines then move the rows).
bool mapped_rows(const void* h_zt, const void* h_zd, int32_t G, size_t row_bytes, const void** d_zt,
                 const void** d_zd) {
  auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (row_bytes % 16 != 0 || !al(h_zt) || (G > 0 && !al(h_zd))) return false;
  void* a = nullptr;
  void* b = nullptr;
  if (cudaHostGetDevicePointer(&a, const_cast<void*>(h_zt), 0) != cudaSuccess ||
      (G > 0 && cudaHostGetDevicePointer(&b, const_cast<void*>(h_zd), 0) != cudaSuccess)) {
    (void)cudaGetLastError();            // not page-locked: clear the error this lookup left
    return false;
  }
  if (!al(a) || (G > 0 && !al(b))) return false;
  *d_zt = a;
  *d_zd = b;
  return true;
}

// The internal stream that copies row group g + 1 while group g verifies on the caller's stream:
// one per device, created on first use and kept for the process.
std::mutex g_copy_mu;
cudaStream_t g_copy_stream[64];

cudaError_t copy_stream(cudaStream_t* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_copy_mu);
  if (g_copy_stream[dev] == nullptr) {
    e = cudaStreamCreateWithFlags(&g_copy_stream[dev], cudaStreamNonBlocking);
    if (e != cudaSuccess) return e;
  }
  *out = g_copy_stream[dev];
  return cudaSuccess;
}

// Row groups of the pipelined call: a few, each of at least 64 rows.
int32_t row_groups(int32_t B) {
  int32_t g = B / 64;
  return g < 1 ? 1 : (g > 4 ? 4 : g);
}

size_t small_h2d_bytes(const int32_t* h_len, int32_t B, int32_t G) {
  const size_t b = static_cast<size_t>(B), g = static_cast<size_t>(G);
  return b * g * 4 + (h_len ? b * 4 : 0) + b * 4 + b * (g + 2) * 4;
}

}  // namespace

extern "C" {

size_t spec_verify_staging_size(int32_t B, int32_t gamma_max, int32_t V, int32_t dtype) {
  if (!shape_ok(B, gamma_max, V, dtype)) return 0;
  return layout(B, gamma_max, V, dtype).total;
}

size_t spec_verify_staged_h2d_bytes(const int32_t* h_draft_len, const float* h_temperature,
                                    int32_t B, int32_t gamma_max, int32_t V, int32_t dtype) {
  if (!shape_ok(B, gamma_max, V, dtype) || !h_temperature) return 0;
  size_t n = small_h2d_bytes(h_draft_len, B, gamma_max);
  for_each_run(h_draft_len, h_temperature, 0, B, gamma_max, V, dtype == SV_DTYPE_BF16 ? 2 : 4,
               [&](bool, size_t, size_t len) { n += len; });
  return n;
}

int spec_verify_staged(const void* h_target_logits, const void* h_draft_logits,
                       const int32_t* h_draft_tokens, const int32_t* h_draft_len,
                       const float* h_temperature, const float* h_uniforms,
                       int32_t* h_out_tokens, int32_t* h_out_num_emitted, float* h_out_alpha,
                       int32_t B, int32_t gamma_max, int32_t V, int32_t dtype, void* staging,
                       size_t staging_bytes, void* workspace, size_t workspace_bytes,
                       size_t* h2d_bytes, void* cuda_stream) {
  if (dtype != SV_DTYPE_F32 && dtype != SV_DTYPE_BF16) return SV_ERR_BAD_DTYPE;
  if (!shape_ok(B, gamma_max, V, dtype)) return SV_ERR_BAD_SHAPE;
  const int32_t G = gamma_max;
  if (!h_target_logits || !h_temperature || !h_uniforms || !h_out_tokens || !h_out_num_emitted ||
      !staging || !workspace)
    return SV_ERR_NULL_POINTER;
  if (G > 0 && (!h_draft_logits || !h_draft_tokens)) return SV_ERR_NULL_POINTER;
  if (reinterpret_cast<uintptr_t>(staging) % 256 != 0) return SV_ERR_MISALIGNED;
  const Layout L = layout(B, G, V, dtype);
  if (staging_bytes < L.total) return SV_ERR_WORKSPACE_TOO_SMALL;
  if (workspace_bytes < spec_verify_workspace_size(B, G, V, dtype))
    return SV_ERR_WORKSPACE_TOO_SMALL;

  const cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  char* d = static_cast<char*>(staging);
  const size_t b = static_cast<size_t>(B), g = static_cast<size_t>(G);
  size_t n = 0;
  bool failed = false;
  auto h2d = [&](size_t dst, const void* src, size_t len) {
    if (failed || len == 0) return;
    if (cudaMemcpyAsync(d + dst, src, len, cudaMemcpyHostToDevice, st) == cudaSuccess) n += len;
    else failed = true;
  };
  if (G > 0) h2d(L.tok, h_draft_tokens, b * g * 4);
  if (h_draft_len) h2d(L.len, h_draft_len, b * 4);
  h2d(L.temp, h_temperature, b * 4);
  h2d(L.u, h_uniforms, b * (g + 2) * 4);
  const size_t es = dtype == SV_DTYPE_BF16 ? 2 : 4;
  const size_t row_bytes = static_cast<size_t>(V) * es;
  if (failed) return SV_ERR_CUDA;
  const void* m_zt = nullptr;
  const void* m_zd = nullptr;
  const bool mapped = mapped_rows(h_target_logits, h_draft_logits, G, row_bytes, &m_zt, &m_zd);
  int dev = 0, sms = 0;
  cudaStream_t cs = nullptr;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      copy_stream(&cs) != cudaSuccess)
    return SV_ERR_CUDA;

  // The rows in NG groups: the logit rows of group g + 1 cross the host link on the internal stream
  // while group g verifies on `cuda_stream`; events order each verification after its rows.
  const int32_t NG = row_groups(B), per = (B + NG - 1) / NG;
  cudaEvent_t ev[5] = {};
  auto cleanup = [&]() {
    for (cudaEvent_t& e : ev)
      if (e) cudaEventDestroy(e);                  // released once the event has completed
  };
  for (int e = 0; e <= NG; ++e)
    if (cudaEventCreateWithFlags(&ev[e], cudaEventDisableTiming) != cudaSuccess) {
      cleanup();
      return SV_ERR_CUDA;
    }
  // The internal stream starts after the small copies (the gather reads draft_len, temperature).
  if (cudaEventRecord(ev[NG], st) != cudaSuccess || cudaStreamWaitEvent(cs, ev[NG], 0) != cudaSuccess) {
    cleanup();
    return SV_ERR_CUDA;
  }
  int status = SV_OK;
  for (int32_t gi = 0; gi < NG && status == SV_OK; ++gi) {
    const int32_t b0 = gi * per, b1 = (b0 + per < B) ? b0 + per : B;
    if (b0 >= b1) break;
    if (mapped) {
      for_each_run(h_draft_len, h_temperature, b0, b1, G, V, es,
                   [&](bool, size_t, size_t len) { n += len; });
      const long long slots = static_cast<long long>(b1 - b0) * (G + 1);
      const long long cap = static_cast<long long>(sms) * kGatherCtasPerSm;
      const unsigned grid = static_cast<unsigned>(slots < cap ? slots : cap);
      sv_gather_rows<<<grid, kGatherThreads, 0, cs>>>(
          static_cast<const uint4*>(m_zt), static_cast<const uint4*>(m_zd),
          reinterpret_cast<uint4*>(d + L.zt), reinterpret_cast<uint4*>(d + L.zd),
          h_draft_len ? reinterpret_cast<const int32_t*>(d + L.len) : nullptr,
          reinterpret_cast<const float*>(d + L.temp), b0, b1 - b0, G, row_bytes / 16);
      if (cudaGetLastError() != cudaSuccess) failed = true;
    } else {
      for_each_run(h_draft_len, h_temperature, b0, b1, G, V, es,
                   [&](bool draft, size_t off, size_t len) {
        if (failed || len == 0) return;
        if (cudaMemcpyAsync(d + (draft ? L.zd : L.zt) + off,
                            static_cast<const char*>(draft ? h_draft_logits : h_target_logits) + off,
                            len, cudaMemcpyHostToDevice, cs) == cudaSuccess)
          n += len;
        else
          failed = true;
      });
    }
    if (failed || cudaEventRecord(ev[gi], cs) != cudaSuccess ||
        cudaStreamWaitEvent(st, ev[gi], 0) != cudaSuccess) {
      failed = true;
      break;
    }
    const size_t bg = static_cast<size_t>(b0);
    status = sv::verify_ex_planned(
        d + L.zt + bg * (G + 1) * row_bytes,
        G > 0 ? d + L.zd + bg * G * row_bytes : nullptr,
        G > 0 ? reinterpret_cast<const int32_t*>(d + L.tok) + bg * G : nullptr,
        h_draft_len ? reinterpret_cast<const int32_t*>(d + L.len) + bg : nullptr,
        reinterpret_cast<const float*>(d + L.temp) + bg, reinterpret_cast<const float*>(d + L.u) + bg * (G + 2),
        reinterpret_cast<int32_t*>(d + L.otok) + bg * (G + 1), reinterpret_cast<int32_t*>(d + L.onum) + bg,
        reinterpret_cast<float*>(d + L.oalpha) + bg * G, nullptr, nullptr, b1 - b0, G, V, dtype,
        workspace, workspace_bytes, cuda_stream, static_cast<long long>(B) * (G + 1));
  }
  cleanup();
  if (h2d_bytes) *h2d_bytes = n;
  if (failed) return SV_ERR_CUDA;
  if (status != SV_OK) return status;

  auto d2h = [&](void* dst, size_t src, size_t len) {
    return cudaMemcpyAsync(dst, d + src, len, cudaMemcpyDeviceToHost, st) == cudaSuccess;
  };
  if (!d2h(h_out_tokens, L.otok, b * (g + 1) * 4) || !d2h(h_out_num_emitted, L.onum, b * 4) ||
      (G > 0 && h_out_alpha && !d2h(h_out_alpha, L.oalpha, b * g * 4)))
    return SV_ERR_CUDA;
  return SV_OK;
}

}  // extern "C"
