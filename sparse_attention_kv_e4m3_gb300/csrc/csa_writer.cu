// csa_writer.cu — the compressed-K writer: quantises key rows into the cache's
// 132-byte records (FlashMemory-DeepSeek-V4, "compressed_k format": 128 e4m3
// bytes, then the fp32 scale; the BatchGen #153 commit log's store kernel for
// that "[128B fp8 | 4B fp32 scale]" layout). Per row: scale = amax / 448 in
// binary32 and codes = e4m3(x / scale), x / scale in binary32, rounded to the
// nearest e4m3 value with ties to even and saturating at 448; a row whose
// scale is 0 (all zero, or amax / 448 underflows) is zero codes and scale 0.
//
// A warp quantises a row at a time (32 rows per pass, their loads in flight
// together): each lane holds 4 of the 128 values, a shuffle tree finds amax,
// and each lane stores its 4 codes as one 32-bit word (records are 4-byte
// aligned); lane 0 stores the scale. Memory-bound: the row is read once,
// coalesced, and the record written once.
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "csa_index.h"

namespace {

constexpr int kWriterThreads = 256;
constexpr int kRec = 132, kPage = 64, kD = 128;

struct WriteParams {
  const void* keys;
  int32_t bf16;
  int64_t n;
  const int32_t* row_req;
  const int32_t* row_pos;
  uint8_t* kv;
  int64_t num_pages;
  int64_t page_stride;
  const int32_t* page_table;
  int32_t num_req;
  int32_t pt_stride;
  int32_t* dev_status;
};

// Row i's record address, or the CSA_DEV_* bit that stops it (checked in the
// documented order: request, position, page).
__device__ __forceinline__ int32_t record_of(const WriteParams& W, int64_t i, uint8_t** rec) {
  const int64_t req = W.row_req ? W.row_req[i] : i;
  if (req < 0 || req >= W.num_req) return CSA_DEV_BAD_REQUEST;
  const int32_t pos = W.row_pos[i];
  if (pos < 0 || pos >= static_cast<int64_t>(kPage) * W.pt_stride) return CSA_DEV_LEN_OOB;
  const int64_t phys = W.page_table[req * W.pt_stride + pos / kPage];
  if (phys < 0 || phys >= W.num_pages) return CSA_DEV_PAGE_OOB;
  *rec = W.kv + phys * W.page_stride + static_cast<int64_t>(pos % kPage) * kRec;
  return 0;
}

// A warp takes 32 rows per pass: each lane resolves one row's record (request,
// position, page table) so that those loads are in flight together; then the
// rows' values are loaded kChunk rows at a time, every lane holding 4 values of
// each, and each row is quantised and stored.
constexpr int kRowsPerPass = 32, kChunk = 8;
constexpr int32_t kNoRow = 1 << 30;

__device__ __forceinline__ void load_row(const WriteParams& W, int64_t i, int lane, float (&x)[4]) {
  if (W.bf16) {
    const uint2 raw = reinterpret_cast<const uint2*>(W.keys)[i * (kD / 4) + lane];
    x[0] = __uint_as_float(raw.x << 16);
    x[1] = __uint_as_float(raw.x & 0xFFFF0000u);
    x[2] = __uint_as_float(raw.y << 16);
    x[3] = __uint_as_float(raw.y & 0xFFFF0000u);
  } else {
    const float4 v = reinterpret_cast<const float4*>(W.keys)[i * (kD / 4) + lane];
    x[0] = v.x;
    x[1] = v.y;
    x[2] = v.z;
    x[3] = v.w;
  }
}

__global__ void __launch_bounds__(kWriterThreads) write_keys_kernel(const WriteParams W) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kWriterThreads / 32);
  int32_t flags = 0;
  for (int64_t i0 = ((static_cast<int64_t>(blockIdx.x) * kWriterThreads + threadIdx.x) >> 5) * kRowsPerPass;
       i0 < W.n; i0 += warps * kRowsPerPass) {
    uint8_t* my_rec = nullptr;
    const int32_t my_f = i0 + lane < W.n ? record_of(W, i0 + lane, &my_rec) : kNoRow;
    const int rows = W.n - i0 < kRowsPerPass ? static_cast<int>(W.n - i0) : kRowsPerPass;  // uniform
    for (int c = 0; c < rows; c += kChunk) {
      float x[kChunk][4];
#pragma unroll
      for (int r = 0; r < kChunk; ++r) load_row(W, c + r < rows ? i0 + c + r : i0, lane, x[r]);
#pragma unroll
      for (int r = 0; r < kChunk; ++r) {
        if (c + r >= rows) break;  // uniform
        const int32_t f0 = __shfl_sync(0xFFFFFFFFu, my_f, c + r);
        uint8_t* rec =
            reinterpret_cast<uint8_t*>(__shfl_sync(0xFFFFFFFFu, reinterpret_cast<uintptr_t>(my_rec), c + r));
        int32_t f = f0;
        const bool finite = isfinite(x[r][0]) && isfinite(x[r][1]) && isfinite(x[r][2]) && isfinite(x[r][3]);
        if (f == 0 && !__all_sync(0xFFFFFFFFu, finite)) f = CSA_DEV_RANGE;
        if (f != 0) {  // uniform
          flags |= f;
          continue;
        }
        float amax = fmaxf(fmaxf(fabsf(x[r][0]), fabsf(x[r][1])), fmaxf(fabsf(x[r][2]), fabsf(x[r][3])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        const float scale = amax / 448.0f;  // IEEE division, round to nearest even
        uint32_t word = 0;
        if (scale > 0.0f) {  // a scale of 0 (amax == 0, or amax / 448 underflows): zero codes
          const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
              make_float2(x[r][0] / scale, x[r][1] / scale), __NV_SATFINITE, __NV_E4M3);
          const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
              make_float2(x[r][2] / scale, x[r][3] / scale), __NV_SATFINITE, __NV_E4M3);
          word = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
        }
        uint32_t* rw = reinterpret_cast<uint32_t*>(rec);
        rw[lane] = word;  // bytes 4 lane .. 4 lane + 3: codes of d = 4 lane .. 4 lane + 3
        if (lane == 0) rw[kD / 4] = __float_as_uint(scale);  // little-endian fp32 at byte 128
      }
    }
  }
  if (flags && W.dev_status && lane == 0) atomicOr(W.dev_status, flags);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" csa_status csa_index_write_keys(const csa_write_args* a, void* stream) {
  if (!a) return CSA_ERR_INVALID_ARG;
  if (a->n < 0 || a->reserved0 != 0 || (a->key_dtype != CSA_KEYS_F32 && a->key_dtype != CSA_KEYS_BF16))
    return CSA_ERR_INVALID_ARG;
  if (a->n == 0) return CSA_OK;
  if (!a->keys || !a->row_pos || !a->kv || !a->page_table) return CSA_ERR_INVALID_ARG;
  if (a->num_req < 1 || a->pt_stride < 1 || a->num_pages < 1) return CSA_ERR_INVALID_ARG;
  if (a->page_stride_bytes < static_cast<int64_t>(kPage) * kRec || a->page_stride_bytes % 16 != 0)
    return CSA_ERR_INVALID_ARG;
  if (!aligned(a->keys, 16) || !aligned(a->kv, 16) || !aligned(a->row_pos, 4) || !aligned(a->page_table, 4) ||
      (a->row_req && !aligned(a->row_req, 4)) || (a->dev_status && !aligned(a->dev_status, 4)))
    return CSA_ERR_ALIGNMENT;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return CSA_ERR_CUDA;
  WriteParams W;
  W.keys = a->keys;
  W.bf16 = a->key_dtype == CSA_KEYS_BF16;
  W.n = a->n;
  W.row_req = a->row_req;
  W.row_pos = a->row_pos;
  W.kv = a->kv;
  W.num_pages = a->num_pages;
  W.page_stride = a->page_stride_bytes;
  W.page_table = a->page_table;
  W.num_req = a->num_req;
  W.pt_stride = a->pt_stride;
  W.dev_status = a->dev_status;
  int per_sm = 0;  // resident CTAs per SM: one full wave, grid-stride beyond
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, write_keys_kernel, kWriterThreads, 0) != cudaSuccess ||
      per_sm < 1)
    return CSA_ERR_CUDA;
  const int64_t rows_per_block = kRowsPerPass * (kWriterThreads / 32);
  const int64_t want = (a->n + rows_per_block - 1) / rows_per_block;
  const int64_t cap = static_cast<int64_t>(sms) * per_sm;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  write_keys_kernel<<<grid, kWriterThreads, 0, static_cast<cudaStream_t>(stream)>>>(W);
  return cudaGetLastError() == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}
