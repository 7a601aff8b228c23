// csa_recall.cu — Level-1 recall (FlashMemory-DeepSeek-V4, "Two-level recall
// algorithm", Level 1, and "Joint checkpoint + ensemble"): the Memory Indexer
// scores the full history at several target layers with 128-head queries, the
// per-layer sigmoid scores are combined per chunk (max or mean), and a chunk is
// resident when the combined score reaches the threshold or it lies in the
// row's attention sink or recency tail. The output is the resident set per
// chunk and, per query row, the ascending list of logical pages that hold a
// resident chunk (the Level-2 resident list).
//
// The scoring kernel runs once per layer with the layer's 128-head query in its
// logit mode (csa_index_logits), reading each layer's cache once; a small kernel
// applies the sigmoid and folds the layer into the combined score.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "csa_index.h"

namespace {

constexpr int kHeads = 128, kD = 128, kPage = 64;
constexpr int kMaxLayers = 8;
constexpr int kFinalThreads = 256;  // one page of the window per thread

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace: one layer's logits and the running combined score.
struct Layout {
  size_t la, acc, total;
};

Layout layout_of(int64_t num_q, int64_t stride) {
  Layout L;
  size_t off = 0;
  L.la = off;
  off += round256(static_cast<size_t>(num_q) * stride * 4);
  L.acc = off;
  off += round256(static_cast<size_t>(num_q) * stride * 4);
  L.total = off;
  return L;
}

struct Rows {
  const int32_t* q_len;
  const int32_t* q_req;
  int32_t num_req;
  int32_t pt_stride;
};

// Request of row b (q_req, or b itself when q_req is NULL).
__device__ __forceinline__ int32_t row_req(const Rows& R, int32_t b) { return R.q_req ? R.q_req[b] : b; }

// Visible length of row b, as the scorer sees it: q_len clamped to
// [0, 64 * pt_stride]; 0 for a request id out of range.
__device__ __forceinline__ int64_t row_len(const Rows& R, int32_t b) {
  const int32_t req = row_req(R, b);
  if (req < 0 || req >= R.num_req) return 0;
  int64_t L = R.q_len[b];
  const int64_t cap = static_cast<int64_t>(kPage) * R.pt_stride;
  return L < 0 ? 0 : (L > cap ? cap : L);
}

// acc = layer 0 ? s : combine(acc, s), s = sigmoid(la), for the visible
// positions of row blockIdx.x (blockIdx.y strides over the positions). A
// position on a page this layer's page table maps out of range was not scored
// (the scorer flags it); it counts 0 in this layer.
__global__ void combine_kernel(const float* la, float* acc, int64_t stride, Rows R,
                               const int32_t* page_table, int64_t num_pages, int layer, int ensemble) {
  const int32_t b = blockIdx.x;
  const int64_t L = row_len(R, b);
  if (L == 0) return;
  const int32_t* pt = page_table + static_cast<int64_t>(row_req(R, b)) * R.pt_stride;
  for (int64_t n = static_cast<int64_t>(blockIdx.y) * blockDim.x + threadIdx.x; n < L;
       n += static_cast<int64_t>(gridDim.y) * blockDim.x) {
    const int64_t o = static_cast<int64_t>(b) * stride + n;
    const int32_t phys = pt[n / kPage];
    const float s = phys < 0 || phys >= num_pages ? 0.0f : 1.0f / (1.0f + expf(-la[o]));
    acc[o] = layer == 0 ? s : (ensemble == CSA_ENSEMBLE_MAX ? fmaxf(acc[o], s) : acc[o] + s);
  }
}

// One CTA per row: the combined score, the keep decision and the ascending list
// of pages with a kept chunk, a window of 256 pages at a time.
__global__ void __launch_bounds__(kFinalThreads) select_kernel(const float* acc, int64_t stride, Rows R, int n_layers,
                                                               int ensemble, float threshold, int32_t sink,
                                                               int32_t recent, uint8_t* keep, float* scores,
                                                               int32_t* pages, int32_t pages_stride,
                                                               int32_t* n_pages) {
  __shared__ uint8_t any[kFinalThreads];
  __shared__ int32_t warp_count[kFinalThreads / 32];
  const int32_t b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t L = row_len(R, b);
  const int64_t npages = (L + kPage - 1) / kPage;
  const float inv_layers = 1.0f / static_cast<float>(n_layers);
  int32_t listed = 0;  // uniform
  for (int64_t p0 = 0; p0 < npages; p0 += kFinalThreads) {
    any[tid] = 0;
    __syncthreads();
    const int64_t n1 = (p0 + kFinalThreads) * kPage < L ? (p0 + kFinalThreads) * kPage : L;
    for (int64_t n = p0 * kPage + tid; n < n1; n += kFinalThreads) {
      const int64_t o = static_cast<int64_t>(b) * stride + n;
      const float e = ensemble == CSA_ENSEMBLE_MEAN ? acc[o] * inv_layers : acc[o];
      const bool k = e >= threshold || n < sink || n >= L - recent;
      keep[o] = k ? 1 : 0;
      if (scores) scores[o] = e;
      if (k) any[(n / kPage) - p0] = 1;  // several threads may write the same 1
    }
    __syncthreads();
    const bool f = p0 + tid < npages && any[tid] != 0;
    const uint32_t ballot = __ballot_sync(0xFFFFFFFFu, f);
    if (lane == 0) warp_count[warp] = __popc(ballot);
    __syncthreads();
    int32_t before = listed, total = 0;
    for (int w = 0; w < kFinalThreads / 32; ++w) {
      if (w < warp) before += warp_count[w];
      total += warp_count[w];
    }
    if (f) pages[static_cast<int64_t>(b) * pages_stride + before + __popc(ballot & ((1u << lane) - 1u))] =
        static_cast<int32_t>(p0 + tid);
    listed += total;
    __syncthreads();
  }
  if (tid == 0) n_pages[b] = listed;
}

// Every layer scores the same rows (layer 0's q_len and q_req) over a cache of
// the same geometry.
bool same_rows(const csa_index_args& a, const csa_index_args& b) {
  return a.num_q == b.num_q && a.num_req == b.num_req && a.pt_stride == b.pt_stride;
}

}  // namespace

extern "C" size_t csa_recall_workspace_bytes(const csa_recall_args* a) {
  if (!a || !a->layers || a->keep_stride < 0 || a->layers[0].num_q < 0) return 0;
  return layout_of(a->layers[0].num_q, a->keep_stride).total;
}

extern "C" csa_status csa_recall_level1(const csa_recall_args* a, void* ws, size_t ws_bytes, void* stream) {
  if (!a || !a->layers || a->n_layers < 1 || a->n_layers > kMaxLayers) return CSA_ERR_INVALID_ARG;
  if (a->ensemble != CSA_ENSEMBLE_MAX && a->ensemble != CSA_ENSEMBLE_MEAN) return CSA_ERR_INVALID_ARG;
  if (std::isnan(a->threshold) || a->sink < 0 || a->recent < 0) return CSA_ERR_INVALID_ARG;
  const csa_index_args& L0 = a->layers[0];
  for (int l = 0; l < a->n_layers; ++l) {
    const csa_index_args& L = a->layers[l];
    if (!same_rows(L0, L) || L.num_heads != kHeads || L.head_dim != kD || L.resident || L.n_resident)
      return CSA_ERR_INVALID_ARG;
  }
  const int64_t num_q = L0.num_q;
  if (num_q < 0 || L0.pt_stride < 1) return CSA_ERR_INVALID_ARG;
  if (num_q == 0) return CSA_OK;
  if (!a->keep || !a->pages || !a->n_pages) return CSA_ERR_INVALID_ARG;
  if (a->keep_stride < static_cast<int64_t>(kPage) * L0.pt_stride || a->pages_stride < L0.pt_stride)
    return CSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(a->pages) & 3) || (reinterpret_cast<uintptr_t>(a->n_pages) & 3) ||
      (a->scores && (reinterpret_cast<uintptr_t>(a->scores) & 3)))
    return CSA_ERR_ALIGNMENT;
  const Layout W = layout_of(num_q, a->keep_stride);
  if (!ws || ws_bytes < W.total) return CSA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 255) return CSA_ERR_ALIGNMENT;
  uint8_t* base = static_cast<uint8_t*>(ws);
  float* la = reinterpret_cast<float*>(base + W.la);
  float* acc = reinterpret_cast<float*>(base + W.acc);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Rows R{L0.q_len, L0.q_req, L0.num_req, L0.pt_stride};
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return CSA_ERR_CUDA;
  for (int l = 0; l < a->n_layers; ++l) {
    const csa_index_args& L = a->layers[l];
    csa_index_args layer = L;
    layer.q_len = L0.q_len;  // every layer scores layer 0's rows
    layer.q_req = L0.q_req;
    layer.dev_status = L0.dev_status;
    const csa_status st = csa_index_logits(&layer, la, a->keep_stride, stream);
    if (st != CSA_OK) return st;
    int64_t gy = (static_cast<int64_t>(sms) * 8 + num_q - 1) / num_q;  // about 8 CTAs per SM in all
    gy = gy < 1 ? 1 : (gy > 65535 ? 65535 : gy);
    combine_kernel<<<dim3(static_cast<unsigned>(num_q), static_cast<unsigned>(gy)), 256, 0, s>>>(
        la, acc, a->keep_stride, R, L.page_table, L.num_pages, l, a->ensemble);
    if (cudaGetLastError() != cudaSuccess) return CSA_ERR_CUDA;
  }
  select_kernel<<<static_cast<unsigned>(num_q), kFinalThreads, 0, s>>>(
      acc, a->keep_stride, R, a->n_layers, a->ensemble, a->threshold, a->sink, a->recent, a->keep, a->scores,
      a->pages, a->pages_stride, a->n_pages);
  return cudaGetLastError() == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}
