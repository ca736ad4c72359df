// C ABI of the verifier (include/spec_verify.h): host-side validation, launch planning and
// dispatch to the streaming kernel (16-byte aligned rows) or the element kernel (any alignment).

#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "../../include/spec_verify.h"
#include "sv_common.cuh"

namespace {

#ifndef SV_STREAM_CHUNK_BYTES
#define SV_STREAM_CHUNK_BYTES 65536   // target bytes of one row chunk per CTA on the streaming path
#endif
// bf16 rows of a batch with many position slots per cluster: 128 KB chunks, half the CTAs per
// position and so half the exchange participants (V=256000, B=1024: 1.28 vs 1.47 ms; one-hot
// drafts 0.66 vs 0.89 ms). A small batch keeps SV_STREAM_CHUNK_BYTES to fill the GPU (B=64,
// V=128256: 73 vs 76 us); fp32 rows too (B=256, V=152064: 513 vs 662 us).
#ifndef SV_STREAM_CHUNK_BYTES_LARGE
#define SV_STREAM_CHUNK_BYTES_LARGE 131072
#endif
// bf16 one-hot drafts of such a batch (no residual pass): 256 KB chunks with the wide draw groups
// (V=256000, B=1024: 0.57 vs 0.66 ms).
#ifndef SV_STREAM_CHUNK_BYTES_ONEHOT
#define SV_STREAM_CHUNK_BYTES_ONEHOT 262144
#endif
#ifndef SV_STREAM_LARGE_MIN_SLOTS
#define SV_STREAM_LARGE_MIN_SLOTS 16   // position slots per cluster that make a batch large
#endif
#ifndef SV_STREAM_MAX_CLUSTER
#define SV_STREAM_MAX_CLUSTER 8
#endif

constexpr int kElemThreads = 512;
// Logits per thread of the element kernel: up to 16 CTAs x 512 threads x 32 = 262144 logits a row.
constexpr int kVptOptions[6] = {1, 2, 4, 8, 16, 32};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t records_bytes(int32_t B, int32_t G) {
  return align_up(static_cast<size_t>(B) * (G + 1) * sizeof(int2), 256);
}

// Workspace: records [B, G+1] int2, row counters [B], the status word, then (filtered
// verification) the row thresholds [B * (2G + 1)] fp32 and the threshold kernel's row counter,
// which the call clears again after use.
size_t thresholds_offset(int32_t B, int32_t G) {
  return align_up(records_bytes(B, G) + static_cast<size_t>(B) * sizeof(unsigned) + 4, 256);
}
size_t threshold_rows_of(int32_t B, int32_t G) { return static_cast<size_t>(B) * (2 * G + 1); }

// Past spec_verify_workspace_size, the larger workspace of spec_verify_filtered_workspace_size
// holds the kept lists: per threshold row a count, per batch row a "verified from its lists" flag,
// then per threshold row kList (index, logit) entries. All of it is cleared after each call.
constexpr size_t kListBytes = sv::kList * sizeof(int2);   // one row's kept list
size_t list_counts_offset(int32_t B, int32_t G, int32_t V, int32_t dtype) {
  return spec_verify_workspace_size(B, G, V, dtype);
}
size_t lists_offset(int32_t B, int32_t G, int32_t V, int32_t dtype) {
  return list_counts_offset(B, G, V, dtype) +
         align_up((threshold_rows_of(B, G) + static_cast<size_t>(B)) * sizeof(int), 256);
}

bool sizes_ok(int32_t B, int32_t G, int32_t V, int32_t dtype) {
  if (B < 1 || G < 0 || G > SV_MAX_GAMMA || V < 1) return false;
  if (dtype != SV_DTYPE_F32 && dtype != SV_DTYPE_BF16) return false;
  return true;
}

// Element path: a row of V logits split into C <= 16 chunks of at most 512 * VPT logits.
bool element_plan(int V, int* vpt_index, int* C, int* per) {
  for (int vi = 0; vi < 6; ++vi) {
    const long long cap = static_cast<long long>(kElemThreads) * kVptOptions[vi];
    const long long c = (V + cap - 1) / cap;
    if (c <= sv::kMaxCluster) {
      *vpt_index = vi;
      *C = static_cast<int>(c < 1 ? 1 : c);
      *per = (V + *C - 1) / *C;
      return true;
    }
  }
  return false;
}

// Streaming path: CTAs per position, the power of two that brings a row chunk near chunk_bytes
// (at most SV_STREAM_MAX_CLUSTER), raised until a chunk fits the group sums buffer. 0 when even 16
// CTAs leave chunks too large.
int stream_cluster_size(long long row_bytes, bool bf16,
                        long long chunk_bytes = SV_STREAM_CHUNK_BYTES, bool wide = false) {
  int C = 1;
  while (C < SV_STREAM_MAX_CLUSTER && row_bytes > static_cast<long long>(C) * chunk_bytes) C *= 2;
  const long long units = row_bytes / 16;
  while ((units + C - 1) / C > sv::stream_max_units(bf16, wide)) {
    if (C >= sv::kMaxCluster) return 0;
    C *= 2;
  }
  return C;
}

std::mutex g_mu;
int g_device_ok[64];                 // 0 unknown, 1 sm_103, 2 other
int g_max_clusters[64][2][3][5];     // by device, bf16, variant (narrow, wide, masked), log2(C);
                                     // 0 = not queried

int check_device(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  if (dev < 0 || dev >= 64) return SV_ERR_CUDA;
  *dev_out = dev;
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

// masked: the instantiation of filtered verification (narrow draw groups).
int max_clusters(int dev, bool bf16, int C, int* n, bool masked = false, bool wide = false) {
  int lg = 0;
  while ((1 << lg) < C) ++lg;
  std::lock_guard<std::mutex> lock(g_mu);
  wide = wide && bf16 && !masked;
  int& slot = g_max_clusters[dev][bf16 ? 1 : 0][masked ? 2 : (wide ? 1 : 0)][lg];
  if (slot == 0) {
    int m = 0;
    const cudaError_t e = sv::stream_max_clusters(bf16, wide, C, &m, masked);
    if (e != cudaSuccess || m < 1) return SV_ERR_CUDA;
    slot = m;
  }
  *n = slot;
  return SV_OK;
}

// CTAs per position on the streaming path: C (from SV_STREAM_CHUNK_BYTES), or for bf16 rows the
// smaller C of SV_STREAM_CHUNK_BYTES_LARGE chunks when the batch holds at least
// SV_STREAM_LARGE_MIN_SLOTS position slots per cluster of that size.
// One-hot launches (bf16) take SV_STREAM_CHUNK_BYTES_ONEHOT chunks on the same condition.
int stream_plan_C(int dev, bool bf16, long long row_bytes, long long slots, int C,
                  bool onehot = false) {
  if (!bf16) return C;
  const int Cl = stream_cluster_size(
      row_bytes, bf16, onehot ? SV_STREAM_CHUNK_BYTES_ONEHOT : SV_STREAM_CHUNK_BYTES_LARGE, onehot);
  if (Cl == 0 || Cl >= C) return C;
  int mc = 0;
  if (max_clusters(dev, bf16, Cl, &mc, false, onehot) != SV_OK) return C;
  return slots >= static_cast<long long>(SV_STREAM_LARGE_MIN_SLOTS) * mc ? Cl : C;
}

// Greedy tree nodes draw nothing, so the draw-group table does not bound their chunks: a batch
// with at least 8 node slots per cluster takes chunks of up to SV_STREAM_CHUNK_BYTES_ONEHOT
// (one CTA per node row at V=128256 bf16); otherwise the plan of stream_plan_C.
int tree_plan_C(int dev, bool bf16, long long row_bytes, long long slots, int C) {
  const int Ct = stream_cluster_size(row_bytes, bf16, SV_STREAM_CHUNK_BYTES_ONEHOT, true);
  if (bf16 && Ct > 0 && Ct < C) {
    int mc = 0;
    if (max_clusters(dev, bf16, Ct, &mc) == SV_OK && slots >= 8LL * mc) return Ct;
  }
  return stream_plan_C(dev, bf16, row_bytes, slots, C);
}

}  // namespace

extern "C" {

size_t spec_verify_workspace_size(int32_t B, int32_t gamma_max, int32_t V, int32_t dtype) {
  if (!sizes_ok(B, gamma_max, V, dtype)) return 0;
  return thresholds_offset(B, gamma_max) +
         align_up((threshold_rows_of(B, gamma_max) + 1) * sizeof(float), 256);
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
    case SV_ERR_SCRATCH_TOO_SMALL:
      return "SV_ERR_SCRATCH_TOO_SMALL: the sizes need more than the library's static scratch "
             "(SV_NOALLOC_SCRATCH_BYTES)";
    default: return "unknown sv_status";
  }
}

int spec_verify_version(void) { return SV_VERSION; }

int spec_verify_workspace_status(const void* workspace, int32_t B, int32_t gamma_max,
                                 int32_t* status_out, void* cuda_stream) {
  if (!workspace || !status_out) return SV_ERR_NULL_POINTER;
  if (B < 1 || gamma_max < 0 || gamma_max > SV_MAX_GAMMA) return SV_ERR_BAD_SHAPE;
  const char* w = static_cast<const char*>(workspace) + records_bytes(B, gamma_max) +
                  static_cast<size_t>(B) * sizeof(unsigned);
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  unsigned v = 0;
  if (cudaMemcpyAsync(&v, w, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess) return SV_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SV_ERR_CUDA;
  *status_out = static_cast<int32_t>(v);
  return SV_OK;
}

}  // extern "C"

namespace {

// Validation, planning and launch shared by spec_verify_ex (draft logits) and spec_verify_onehot
// (one-hot drafts: no draft logits, 16-byte rows only).
int verify_impl(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                const int32_t* draft_len, const float* temperature, const float* uniforms,
                int32_t* out_tokens, int32_t* out_num_emitted, float* out_alpha,
                float* out_p_draft, float* out_q_draft,
                int32_t B, int32_t gamma_max, int32_t V, int32_t dtype,
                void* workspace, size_t workspace_bytes, void* cuda_stream, bool onehot,
                bool check_only = false, long long plan_slots = 0) {
  if (dtype != SV_DTYPE_F32 && dtype != SV_DTYPE_BF16) return SV_ERR_BAD_DTYPE;
  if (!sizes_ok(B, gamma_max, V, dtype)) return SV_ERR_BAD_SHAPE;
  const int G = gamma_max;
  if (!target_logits || !temperature || !uniforms || !out_tokens || !out_num_emitted)
    return SV_ERR_NULL_POINTER;
  if (G > 0 && ((!onehot && !draft_logits) || !draft_tokens)) return SV_ERR_NULL_POINTER;
  const bool bf16 = dtype == SV_DTYPE_BF16;
  const uintptr_t es = bf16 ? 2 : 4;
  auto mis = [](const void* p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) != 0; };
  if (mis(target_logits, es) || mis(draft_logits, es) || mis(draft_tokens, 4) || mis(draft_len, 4) ||
      mis(temperature, 4) || mis(uniforms, 4) || mis(out_tokens, 4) || mis(out_num_emitted, 4) ||
      mis(out_alpha, 4) || mis(out_p_draft, 4) || mis(out_q_draft, 4) || mis(workspace, 16))
    return SV_ERR_MISALIGNED;
  const size_t need = spec_verify_workspace_size(B, G, V, dtype);
  if (!check_only && (!workspace || workspace_bytes < need)) return SV_ERR_WORKSPACE_TOO_SMALL;
  if (static_cast<long long>(B) * (G + 1) > INT_MAX / sv::kMaxCluster) return SV_ERR_BAD_SHAPE;

  const bool vec = (static_cast<size_t>(V) * es) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(target_logits) % 16 == 0 &&
                   (!draft_logits || reinterpret_cast<uintptr_t>(draft_logits) % 16 == 0);
  if (onehot && !vec)   // one-hot drafts run on the streaming kernel only
    return (static_cast<size_t>(V) * es) % 16 != 0 ? SV_ERR_BAD_SHAPE : SV_ERR_MISALIGNED;
  int vpt_index = 0, eC = 1, eper = 1;
  if (!vec && !element_plan(V, &vpt_index, &eC, &eper)) return SV_ERR_BAD_SHAPE;
  const int sC =
      vec ? stream_cluster_size(static_cast<long long>(V) * static_cast<long long>(es), bf16) : 0;
  if (vec && sC == 0) return SV_ERR_BAD_SHAPE;

  int dev = 0;
  const int dev_status = check_device(&dev);
  if (dev_status != SV_OK || check_only) return dev_status;

  sv::Params P{};
  P.onehot = onehot ? 1 : 0;
  P.zt = target_logits;
  P.zd = onehot ? nullptr : draft_logits;
  P.tokens = draft_tokens;
  P.draft_len = draft_len;
  P.temperature = temperature;
  P.uniforms = uniforms;
  P.out_tokens = out_tokens;
  P.out_num = out_num_emitted;
  P.out_alpha = out_alpha;
  P.out_p = out_p_draft;
  P.out_q = out_q_draft;
  char* ws = static_cast<char*>(workspace);
  P.rec = reinterpret_cast<int2*>(ws);
  P.cnt = reinterpret_cast<unsigned*>(ws + records_bytes(B, G));
  P.status = P.cnt + B;
  P.B = B;
  P.G = G;
  P.V = V;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);

  if (vec) {
    const int E = static_cast<int>(16 / es);
    const long long slots = static_cast<long long>(B) * (G + 1);
    P.units = V / E;
    // plan_slots: plan the chunks as for a batch of that many slots (the staged call verifies row
    // groups with the whole batch's plan, so every row gets the same arithmetic as in one call).
    P.C = stream_plan_C(dev, bf16, static_cast<long long>(V) * static_cast<long long>(es),
                        plan_slots > 0 ? plan_slots : slots, sC, onehot);
    P.per = (P.units + P.C - 1) / P.C;
    int maxc = 0;
    if (max_clusters(dev, bf16, P.C, &maxc, false, onehot) != SV_OK) return SV_ERR_CUDA;
    P.nclusters = static_cast<int>(slots < maxc ? slots : maxc);
    if (sv::launch_stream(P, bf16, stream) != cudaSuccess) return SV_ERR_CUDA;
    return SV_OK;
  }
  P.units = V;
  P.C = eC;
  P.per = eper;
  P.nclusters = B * (G + 1);
  if (sv::launch_element(P, bf16, vpt_index, stream) != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
}

}  // namespace

namespace sv {

int verify_args_status(const void* target_logits, const void* draft_logits,
                       const int32_t* draft_tokens, const int32_t* draft_len,
                       const float* temperature, const float* uniforms, int32_t* out_tokens,
                       int32_t* out_num_emitted, float* out_alpha, float* out_p_draft,
                       float* out_q_draft, int32_t B, int32_t gamma_max, int32_t V, int32_t dtype) {
  return verify_impl(target_logits, draft_logits, draft_tokens, draft_len, temperature, uniforms,
                     out_tokens, out_num_emitted, out_alpha, out_p_draft, out_q_draft, B, gamma_max,
                     V, dtype, nullptr, 0, nullptr, false, true);
}

int verify_ex_planned(const void* target_logits, const void* draft_logits,
                      const int32_t* draft_tokens, const int32_t* draft_len,
                      const float* temperature, const float* uniforms, int32_t* out_tokens,
                      int32_t* out_num_emitted, float* out_alpha, float* out_p_draft,
                      float* out_q_draft, int32_t B, int32_t gamma_max, int32_t V, int32_t dtype,
                      void* workspace, size_t workspace_bytes, void* cuda_stream,
                      long long plan_slots) {
  return verify_impl(target_logits, draft_logits, draft_tokens, draft_len, temperature, uniforms,
                     out_tokens, out_num_emitted, out_alpha, out_p_draft, out_q_draft, B, gamma_max,
                     V, dtype, workspace, workspace_bytes, cuda_stream, false, false, plan_slots);
}

}  // namespace sv

extern "C" {

int spec_verify_ex(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                   const int32_t* draft_len, const float* temperature, const float* uniforms,
                   int32_t* out_tokens, int32_t* out_num_emitted, float* out_alpha,
                   float* out_p_draft, float* out_q_draft,
                   int32_t B, int32_t gamma_max, int32_t V, int32_t dtype,
                   void* workspace, size_t workspace_bytes, void* cuda_stream) {
  return verify_impl(target_logits, draft_logits, draft_tokens, draft_len, temperature, uniforms,
                     out_tokens, out_num_emitted, out_alpha, out_p_draft, out_q_draft, B, gamma_max,
                     V, dtype, workspace, workspace_bytes, cuda_stream, false);
}

int spec_verify_tree_greedy(const void* target_logits, const int32_t* tree_tokens,
                            const int32_t* tree_parents, const int32_t* tree_size,
                            int32_t* out_path, int32_t* out_path_len, int32_t* out_tokens,
                            int32_t* out_pred, int32_t B, int32_t N, int32_t V, int32_t dtype,
                            void* workspace, size_t workspace_bytes, void* cuda_stream) {
  if (dtype != SV_DTYPE_F32 && dtype != SV_DTYPE_BF16) return SV_ERR_BAD_DTYPE;
  if (N < 1 || !sizes_ok(B, N - 1, V, dtype)) return SV_ERR_BAD_SHAPE;
  if (!target_logits || !tree_tokens || !tree_parents || !out_path || !out_path_len || !out_tokens)
    return SV_ERR_NULL_POINTER;
  const bool bf16 = dtype == SV_DTYPE_BF16;
  const uintptr_t es = bf16 ? 2 : 4;
  auto mis = [](const void* p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) != 0; };
  if (mis(target_logits, es) || mis(tree_tokens, 4) || mis(tree_parents, 4) || mis(tree_size, 4) ||
      mis(out_path, 4) || mis(out_path_len, 4) || mis(out_tokens, 4) || mis(out_pred, 4) ||
      mis(workspace, 16))
    return SV_ERR_MISALIGNED;
  const int G = N - 1;
  const size_t need = spec_verify_workspace_size(B, G, V, dtype);
  if (!workspace || workspace_bytes < need) return SV_ERR_WORKSPACE_TOO_SMALL;
  if (static_cast<long long>(B) * N > INT_MAX / sv::kMaxCluster) return SV_ERR_BAD_SHAPE;
  // Tree rows run on the streaming kernel only (rows of 16-byte multiples, 16-byte aligned base).
  if ((static_cast<size_t>(V) * es) % 16 != 0) return SV_ERR_BAD_SHAPE;
  if (reinterpret_cast<uintptr_t>(target_logits) % 16 != 0) return SV_ERR_MISALIGNED;
  const int sC = stream_cluster_size(static_cast<long long>(V) * static_cast<long long>(es), bf16);
  if (sC == 0) return SV_ERR_BAD_SHAPE;
  int dev = 0;
  const int dev_status = check_device(&dev);
  if (dev_status != SV_OK) return dev_status;

  sv::Params P{};
  P.tree = 1;
  P.zt = target_logits;
  P.ttok = tree_tokens;
  P.tparent = tree_parents;
  P.tsize = tree_size;
  P.out_path = out_path;
  P.out_plen = out_path_len;
  P.out_tokens = out_tokens;
  P.out_pred = out_pred;
  char* ws = static_cast<char*>(workspace);
  P.rec = reinterpret_cast<int2*>(ws);
  P.cnt = reinterpret_cast<unsigned*>(ws + records_bytes(B, G));
  P.status = P.cnt + B;
  P.B = B;
  P.G = G;
  P.V = V;
  const int E = static_cast<int>(16 / es);
  const long long slots = static_cast<long long>(B) * N;
  P.units = V / E;
  P.C = tree_plan_C(dev, bf16, static_cast<long long>(V) * static_cast<long long>(es), slots, sC);
  P.per = (P.units + P.C - 1) / P.C;
  int maxc = 0;
  if (max_clusters(dev, bf16, P.C, &maxc) != SV_OK) return SV_ERR_CUDA;
  P.nclusters = static_cast<int>(slots < maxc ? slots : maxc);
  if (sv::launch_stream(P, bf16, static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}

int spec_verify_onehot(const void* target_logits, const int32_t* draft_tokens,
                       const int32_t* draft_len, const float* temperature, const float* uniforms,
                       int32_t* out_tokens, int32_t* out_num_emitted, float* out_alpha,
                       float* out_p_draft, float* out_q_draft,
                       int32_t B, int32_t gamma_max, int32_t V, int32_t dtype,
                       void* workspace, size_t workspace_bytes, void* cuda_stream) {
  return verify_impl(target_logits, nullptr, draft_tokens, draft_len, temperature, uniforms,
                     out_tokens, out_num_emitted, out_alpha, out_p_draft, out_q_draft, B, gamma_max,
                     V, dtype, workspace, workspace_bytes, cuda_stream, true);
}

}  // extern "C"

namespace {

// The checks both filtered entry points make before anything is enqueued (the logits' rows: 16-byte
// multiples on 16-byte aligned bases, within the streaming kernel's row limits).
int filter_args_status(const void* target_logits, const void* draft_logits, const void* const* ptrs4,
                       int nptrs, int32_t B, int32_t G, int32_t V, int32_t dtype, int* sC) {
  if (dtype != SV_DTYPE_F32 && dtype != SV_DTYPE_BF16) return SV_ERR_BAD_DTYPE;
  if (!sizes_ok(B, G, V, dtype)) return SV_ERR_BAD_SHAPE;
  const bool bf16 = dtype == SV_DTYPE_BF16;
  const uintptr_t es = bf16 ? 2 : 4;
  auto mis = [](const void* p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) != 0; };
  for (int k = 0; k < nptrs; ++k)
    if (mis(ptrs4[k], 4)) return SV_ERR_MISALIGNED;
  if ((static_cast<size_t>(V) * es) % 16 != 0) return SV_ERR_BAD_SHAPE;
  if (mis(target_logits, 16) || mis(draft_logits, 16)) return SV_ERR_MISALIGNED;
  if (static_cast<long long>(B) * (2 * G + 1) > INT_MAX / sv::kMaxCluster) return SV_ERR_BAD_SHAPE;
  *sC = stream_cluster_size(static_cast<long long>(V) * static_cast<long long>(es), bf16);
  return *sC == 0 ? SV_ERR_BAD_SHAPE : SV_OK;
}

}  // namespace

extern "C" {

size_t spec_verify_filtered_workspace_size(int32_t B, int32_t gamma_max, int32_t V, int32_t dtype) {
  if (!sizes_ok(B, gamma_max, V, dtype)) return 0;
  return lists_offset(B, gamma_max, V, dtype) +
         align_up(threshold_rows_of(B, gamma_max) * kListBytes, 256);
}

int spec_verify_filter_thresholds(const void* target_logits, const void* draft_logits,
                                  const int32_t* draft_len, const float* temperature,
                                  const int32_t* top_k, const float* top_p, float* out_thresholds,
                                  int32_t B, int32_t gamma_max, int32_t V, int32_t dtype,
                                  void* cuda_stream) {
  const int G = gamma_max;
  if (!target_logits || !temperature || !out_thresholds) return SV_ERR_NULL_POINTER;
  if (G > 0 && !draft_logits) return SV_ERR_NULL_POINTER;
  const void* p4[] = {draft_len, temperature, top_k, top_p, out_thresholds};
  int sC = 0;
  const int st = filter_args_status(target_logits, draft_logits, p4, 5, B, G, V, dtype, &sC);
  if (st != SV_OK) return st;
  int dev = 0;
  const int dev_status = check_device(&dev);
  if (dev_status != SV_OK) return dev_status;
  sv::Params P{};
  P.zt = target_logits;
  P.zd = draft_logits;
  P.draft_len = draft_len;
  P.temperature = temperature;
  P.top_k = top_k;
  P.top_p = top_p;
  P.B = B;
  P.G = G;
  P.V = V;
  if (sv::launch_threshold(P, dtype == SV_DTYPE_BF16, out_thresholds, nullptr, nullptr, nullptr,
                           static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}

int spec_verify_filtered(const void* target_logits, const void* draft_logits,
                         const int32_t* draft_tokens, const int32_t* draft_len,
                         const float* temperature, const int32_t* top_k, const float* top_p,
                         const float* uniforms, int32_t* out_tokens, int32_t* out_num_emitted,
                         float* out_alpha, float* out_p_draft, float* out_q_draft,
                         int32_t B, int32_t gamma_max, int32_t V, int32_t dtype,
                         void* workspace, size_t workspace_bytes, void* cuda_stream) {
  const int G = gamma_max;
  if (dtype != SV_DTYPE_F32 && dtype != SV_DTYPE_BF16) return SV_ERR_BAD_DTYPE;
  if (!sizes_ok(B, G, V, dtype)) return SV_ERR_BAD_SHAPE;
  if (!target_logits || !temperature || !uniforms || !out_tokens || !out_num_emitted)
    return SV_ERR_NULL_POINTER;
  if (G > 0 && (!draft_logits || !draft_tokens)) return SV_ERR_NULL_POINTER;
  if (workspace && reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return SV_ERR_MISALIGNED;
  const void* p4[] = {draft_tokens, draft_len, temperature, top_k, top_p, uniforms, out_tokens,
                      out_num_emitted, out_alpha, out_p_draft, out_q_draft};
  int sC = 0;
  const int st = filter_args_status(target_logits, draft_logits, p4, 11, B, G, V, dtype, &sC);
  if (st != SV_OK) return st;
  const size_t need = spec_verify_workspace_size(B, G, V, dtype);
  if (!workspace || workspace_bytes < need) return SV_ERR_WORKSPACE_TOO_SMALL;
  int dev = 0;
  const int dev_status = check_device(&dev);
  if (dev_status != SV_OK) return dev_status;

  const bool bf16 = dtype == SV_DTYPE_BF16;
  const long long row_bytes = static_cast<long long>(V) * (bf16 ? 2 : 4);
  sv::Params P{};
  P.zt = target_logits;
  P.zd = draft_logits;
  P.tokens = draft_tokens;
  P.draft_len = draft_len;
  P.temperature = temperature;
  P.top_k = top_k;
  P.top_p = top_p;
  P.uniforms = uniforms;
  P.out_tokens = out_tokens;
  P.out_num = out_num_emitted;
  P.out_alpha = out_alpha;
  P.out_p = out_p_draft;
  P.out_q = out_q_draft;
  char* ws = static_cast<char*>(workspace);
  P.rec = reinterpret_cast<int2*>(ws);
  P.cnt = reinterpret_cast<unsigned*>(ws + records_bytes(B, G));
  P.status = P.cnt + B;
  float* tau = reinterpret_cast<float*>(ws + thresholds_offset(B, G));
  P.B = B;
  P.G = G;
  P.V = V;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  // 1. The threshold of every row a filter touches (-inf for the others).
  unsigned* row_counter = reinterpret_cast<unsigned*>(tau + threshold_rows_of(B, G));
  // A workspace of spec_verify_filtered_workspace_size bytes also takes the kept lists.
  const size_t need_lists = spec_verify_filtered_workspace_size(B, G, V, dtype);
  const bool with_lists = workspace_bytes >= need_lists;
  int* list_n = with_lists ? reinterpret_cast<int*>(ws + list_counts_offset(B, G, V, dtype)) : nullptr;
  int* listed = with_lists ? list_n + threshold_rows_of(B, G) : nullptr;
  int2* lists = with_lists ? reinterpret_cast<int2*>(ws + lists_offset(B, G, V, dtype)) : nullptr;
  if (sv::launch_threshold(P, bf16, tau, row_counter, lists, list_n, stream) != cudaSuccess)
    return SV_ERR_CUDA;
  // 2. Batch rows whose logit rows all have kept lists: verified from the lists.
  if (with_lists) {
    if (sv::launch_listed(P, lists, list_n, listed, stream) != cudaSuccess) return SV_ERR_CUDA;
    P.listed = listed;
  }
  // 3. The streaming kernel (the other rows) with every logit below its row's threshold read as
  //    -inf.
  P.tau = tau;
  const long long slots = static_cast<long long>(B) * (G + 1);
  P.units = static_cast<int>(row_bytes / 16);
  P.C = stream_plan_C(dev, bf16, row_bytes, slots, sC);
  P.per = (P.units + P.C - 1) / P.C;
  int maxc = 0;
  if (max_clusters(dev, bf16, P.C, &maxc, true) != SV_OK) return SV_ERR_CUDA;
  P.nclusters = static_cast<int>(slots < maxc ? slots : maxc);
  if (sv::launch_stream(P, bf16, stream) != cudaSuccess) return SV_ERR_CUDA;
  // 4. Leave the workspace zeroed: a later call of other sizes keeps its counters where these
  //    thresholds, the row counter and the lists were.
  const size_t used = (with_lists ? need_lists : need) - thresholds_offset(B, G);
  if (cudaMemsetAsync(tau, 0, used, stream) != cudaSuccess) return SV_ERR_CUDA;
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
