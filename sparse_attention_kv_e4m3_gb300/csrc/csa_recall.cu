// csa_recall.cu — Level-1 recall (FlashMemory-DeepSeek-V4, "Two-level recall
// algorithm", Level 1, and "Joint checkpoint + ensemble"): the Memory Indexer
// scores the full history at several target layers with 128-head queries, the
// per-layer sigmoid scores are combined per chunk (max or mean), and a chunk is
// resident when the combined score reaches the threshold or it lies in the
// row's attention sink or recency tail. The output is the resident set per
// chunk and, per query row, the ascending list of logical pages that hold a
// resident chunk (the Level-2 resident list).
//
// The combined score lives in a workspace plane, zeroed first; the scoring
// kernel runs once per layer with the layer's 128-head query and folds each
// visible record's score into the plane (max, or sum for the mean) in its
// epilogue, so each layer's cache is read once and no per-layer plane is
// written. A record the layer cannot read (a page out of range) leaves the
// plane as it is: it counts 0 for that layer. A kernel over (row, window of
// pages) then writes keep, the scores and a flag per page, and a small kernel
// per row compacts the flags into the page list.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "csa_index.h"
#include "csa_internal.h"

namespace {

constexpr int kHeads = 128, kD = 128, kPage = 64;
constexpr int kMaxLayers = 8;
constexpr int kWinPages = 64;          // pages per CTA of the keep kernel
constexpr int kWinThreads = 256;
constexpr int kListThreads = 256;      // pages per pass of the list kernel

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace: the combined score plane and one flag per (row, logical page).
struct Layout {
  size_t acc, flags, total;
};

Layout layout_of(int64_t num_q, int64_t stride, int32_t pt_stride) {
  Layout L;
  size_t off = 0;
  L.acc = off;
  off += round256(static_cast<size_t>(num_q) * stride * 4);
  L.flags = off;
  off += round256(static_cast<size_t>(num_q) * pt_stride);
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

// Row blockIdx.x, pages [64 w, 64 w + 64) with w = blockIdx.y: the ensemble
// score e, keep = e >= threshold or n < sink or n >= L - recent, and a flag per
// page that holds a kept chunk.
__global__ void __launch_bounds__(kWinThreads) keep_kernel(const float* acc, int64_t stride, Rows R, int n_layers,
                                                           int ensemble, float threshold, int32_t sink,
                                                           int32_t recent, uint8_t* keep, float* scores,
                                                           uint8_t* flags) {
  __shared__ uint32_t pflag[kWinPages];
  const int32_t b = blockIdx.x;
  const int64_t L = row_len(R, b);
  const int64_t n0 = static_cast<int64_t>(blockIdx.y) * kWinPages * kPage;
  if (n0 >= L) return;  // uniform
  const int64_t n1 = n0 + kWinPages * kPage < L ? n0 + kWinPages * kPage : L;
  if (threadIdx.x < kWinPages) pflag[threadIdx.x] = 0;
  __syncthreads();
  const float inv_layers = 1.0f / static_cast<float>(n_layers);
  for (int64_t n = n0 + threadIdx.x; n < n1; n += kWinThreads) {
    const int64_t o = static_cast<int64_t>(b) * stride + n;
    const float e = ensemble == CSA_ENSEMBLE_MEAN ? acc[o] * inv_layers : acc[o];
    const bool k = e >= threshold || n < sink || n >= L - recent;
    keep[o] = k ? 1 : 0;
    if (scores) scores[o] = e;
    if (k) pflag[(n - n0) / kPage] = 1;  // several threads may write the same 1
  }
  __syncthreads();
  const int64_t p = n0 / kPage + threadIdx.x;
  if (threadIdx.x < kWinPages && p * kPage < L)
    flags[static_cast<int64_t>(b) * R.pt_stride + p] = static_cast<uint8_t>(pflag[threadIdx.x]);
}

// One CTA per row: the ascending list of flagged pages, kListThreads pages at a
// time (a ballot scan per pass).
__global__ void __launch_bounds__(kListThreads) list_kernel(const uint8_t* flags, Rows R, int32_t* pages,
                                                            int32_t pages_stride, int32_t* n_pages) {
  __shared__ int32_t warp_count[kListThreads / 32];
  const int32_t b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t L = row_len(R, b);
  const int64_t npages = (L + kPage - 1) / kPage;
  int32_t listed = 0;  // uniform
  for (int64_t p0 = 0; p0 < npages; p0 += kListThreads) {
    const bool f = p0 + tid < npages && flags[static_cast<int64_t>(b) * R.pt_stride + p0 + tid] != 0;
    const uint32_t ballot = __ballot_sync(0xFFFFFFFFu, f);
    if (lane == 0) warp_count[warp] = __popc(ballot);
    __syncthreads();
    int32_t before = listed, total = 0;
    for (int w = 0; w < kListThreads / 32; ++w) {
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
  if (!a || !a->layers || a->keep_stride < 0 || a->layers[0].num_q < 0 || a->layers[0].pt_stride < 0) return 0;
  return layout_of(a->layers[0].num_q, a->keep_stride, a->layers[0].pt_stride).total;
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
  if ((L0.pt_stride + kWinPages - 1) / kWinPages > 65535) return CSA_ERR_UNSUPPORTED;  // grid y of keep_kernel
  if (num_q == 0) return CSA_OK;
  if (!a->keep || !a->pages || !a->n_pages) return CSA_ERR_INVALID_ARG;
  if (a->keep_stride < static_cast<int64_t>(kPage) * L0.pt_stride || a->pages_stride < L0.pt_stride)
    return CSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(a->pages) & 3) || (reinterpret_cast<uintptr_t>(a->n_pages) & 3) ||
      (a->scores && (reinterpret_cast<uintptr_t>(a->scores) & 3)))
    return CSA_ERR_ALIGNMENT;
  const Layout W = layout_of(num_q, a->keep_stride, L0.pt_stride);
  if (!ws || ws_bytes < W.total) return CSA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 255) return CSA_ERR_ALIGNMENT;
  uint8_t* base = static_cast<uint8_t*>(ws);
  float* acc = reinterpret_cast<float*>(base + W.acc);
  uint8_t* flags = base + W.flags;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Rows R{L0.q_len, L0.q_req, L0.num_req, L0.pt_stride};
  if (cudaMemsetAsync(acc, 0, static_cast<size_t>(num_q) * a->keep_stride * 4, s) != cudaSuccess) return CSA_ERR_CUDA;
  const int fold = a->ensemble == CSA_ENSEMBLE_MAX ? CSA_FOLD_MAX : CSA_FOLD_ADD;
  for (int l = 0; l < a->n_layers; ++l) {
    csa_index_args layer = a->layers[l];
    layer.q_len = L0.q_len;  // every layer scores layer 0's rows
    layer.q_req = L0.q_req;
    layer.dev_status = L0.dev_status;
    const csa_status st = csa_score_fold(&layer, acc, a->keep_stride, fold, stream);
    if (st != CSA_OK) return st;
  }
  const unsigned windows = static_cast<unsigned>((L0.pt_stride + kWinPages - 1) / kWinPages);
  keep_kernel<<<dim3(static_cast<unsigned>(num_q), windows), kWinThreads, 0, s>>>(
      acc, a->keep_stride, R, a->n_layers, a->ensemble, a->threshold, a->sink, a->recent, a->keep, a->scores, flags);
  if (cudaGetLastError() != cudaSuccess) return CSA_ERR_CUDA;
  list_kernel<<<static_cast<unsigned>(num_q), kListThreads, 0, s>>>(flags, R, a->pages, a->pages_stride, a->n_pages);
  return cudaGetLastError() == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}
