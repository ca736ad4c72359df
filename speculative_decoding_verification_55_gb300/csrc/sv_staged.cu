// Host-buffer entry point (include/spec_verify.h: spec_verify_staged): stages into device memory
// only the logit rows the accept-or-resample rule reads, runs spec_verify_ex on them and copies the
// outputs back, all enqueued on the caller's stream. Page-locked host logits are gathered by one
// kernel reading host memory directly (no per-row copy calls); other host memory goes through one
// cudaMemcpyAsync per run of contiguous rows.
//
// Rows read ([R] "Speculative decoding", rayaq.ca ml-models -- Mechanics, One round, steps 3-5; The
// greedy case): target rows 0..gamma_b of row b (the drafted positions and the bonus position) and,
// for a sampled row, draft rows 0..gamma_b - 1. A greedy row (temperature exactly 0) reads no draft
// logits. Everything past gamma_b is padding.

#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/spec_verify.h"

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
void for_each_run(const int32_t* h_len, const float* h_temp, int32_t B, int32_t G, int32_t V,
                  size_t s, F&& visit) {
  const size_t row = static_cast<size_t>(V) * s;
  size_t t_off = 0, t_len = 0, d_off = 0, d_len = 0;
  for (int32_t b = 0; b < B; ++b) {
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
constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads) sv_gather_rows(
    const uint4* __restrict__ zt_h, const uint4* __restrict__ zd_h, uint4* __restrict__ zt_d,
    uint4* __restrict__ zd_d, const int32_t* __restrict__ len, const float* __restrict__ temp,
    int32_t B, int32_t G, size_t row16) {
  const long long slots = static_cast<long long>(B) * (G + 1);
  for (long long s = blockIdx.x; s < slots; s += gridDim.x) {
    const int32_t b = static_cast<int32_t>(s / (G + 1));
    const int32_t i = static_cast<int32_t>(s - static_cast<long long>(b) * (G + 1));
    const int32_t g = len ? len[b] : G;
    if (g < 0 || g > G || i > g) continue;
    const size_t t0 = static_cast<size_t>(s) * row16;
    for (size_t u = threadIdx.x; u < row16; u += kGatherThreads) zt_d[t0 + u] = zt_h[t0 + u];
    if (i < g && temp[b] != 0.0f) {
      const size_t d0 = (static_cast<size_t>(b) * G + i) * row16;
      for (size_t u = threadIdx.x; u < row16; u += kGatherThreads) zd_d[d0 + u] = zd_h[d0 + u];
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
  for_each_run(h_draft_len, h_temperature, B, gamma_max, V, dtype == SV_DTYPE_BF16 ? 2 : 4,
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
  const void* m_zt = nullptr;
  const void* m_zd = nullptr;
  if (!failed && mapped_rows(h_target_logits, h_draft_logits, G, row_bytes, &m_zt, &m_zd)) {
    for_each_run(h_draft_len, h_temperature, B, G, V, es,
                 [&](bool, size_t, size_t len) { n += len; });
    const long long slots = static_cast<long long>(B) * (G + 1);
    const unsigned grid = static_cast<unsigned>(slots < 2048 ? slots : 2048);
    sv_gather_rows<<<grid, kGatherThreads, 0, st>>>(
        static_cast<const uint4*>(m_zt), static_cast<const uint4*>(m_zd),
        reinterpret_cast<uint4*>(d + L.zt), reinterpret_cast<uint4*>(d + L.zd),
        h_draft_len ? reinterpret_cast<const int32_t*>(d + L.len) : nullptr,
        reinterpret_cast<const float*>(d + L.temp), B, G, row_bytes / 16);
    if (cudaGetLastError() != cudaSuccess) failed = true;
  } else {
    for_each_run(h_draft_len, h_temperature, B, G, V, es, [&](bool draft, size_t off, size_t len) {
      h2d((draft ? L.zd : L.zt) + off,
          static_cast<const char*>(draft ? h_draft_logits : h_target_logits) + off, len);
    });
  }
  if (h2d_bytes) *h2d_bytes = n;
  if (failed) return SV_ERR_CUDA;

  const int status = spec_verify_ex(
      d + L.zt, G > 0 ? d + L.zd : nullptr,
      G > 0 ? reinterpret_cast<const int32_t*>(d + L.tok) : nullptr,
      h_draft_len ? reinterpret_cast<const int32_t*>(d + L.len) : nullptr,
      reinterpret_cast<const float*>(d + L.temp), reinterpret_cast<const float*>(d + L.u),
      reinterpret_cast<int32_t*>(d + L.otok), reinterpret_cast<int32_t*>(d + L.onum),
      reinterpret_cast<float*>(d + L.oalpha), nullptr, nullptr, B, G, V, dtype, workspace,
      workspace_bytes, cuda_stream);
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
