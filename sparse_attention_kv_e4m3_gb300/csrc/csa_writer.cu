// csa_writer.cu — the compressed-K writer: quantises key rows into the cache's
// 132-byte records (FlashMemory-DeepSeek-V4, "compressed_k format": 128 e4m3
// bytes, then the fp32 scale; the BatchGen #153 commit log's store kernel for
// that "[128B fp8 | 4B fp32 scale]" layout). Per row: scale = amax / 448 in
// binary32 and codes = e4m3(x / scale), x / scale in binary32, rounded to the
// nearest e4m3 value with ties to even and saturating at 448; a row whose
// scale is 0 (all zero, or amax / 448 underflows) is zero codes and scale 0.
//
// Eight lanes quantise a row (a warp four rows at a time): each lane holds 16 of
// the 128 values, a reduction over the group's magnitude bits gives amax and
// tells whether all are finite, and each lane stores its 16 codes as four
// 32-bit words (records are 4-byte aligned); the group's first lane stores the
// scale. The per-row work (amax, the scale, its reciprocal) is thus shared by
// eight lanes instead of a whole warp. The row is read once, coalesced, and the
// record written once.
//
// The quotients x / scale are the correctly rounded binary32 ones, computed
// without a division per value: with y = RN(1/scale) (one correctly rounded
// reciprocal per row), q0 = RN(x y) is within a few ulps of x / scale; one
// correction q1 = RN(q0 + RN(x - q0 scale) y) brings it within one ulp, and a
// second one (the same step from q1) gives RN(x / scale) by Markstein's theorem
// on FMA-based division (P. Markstein, "Computation of elementary functions on
// the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990; restated
// in Muller et al., "Handbook of Floating-Point Arithmetic", the section on
// Newton-Raphson-based division with an FMA): the residuals x - q scale are
// exact under an FMA when nothing underflows. That holds for every quotient
// that can reach a nonzero code (|x / scale| >= 2^-10, so |x| >= 2^-100) once
// scale >= 2^-90; smaller scales take the division itself. Quotients below
// 2^-10 become a signed zero code either way.
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

// Row i's request and position words (an index past the rows reads row 0's,
// which the caller drops), loaded without a branch on any loaded value so that
// they stay in flight while the warp works on earlier rows.
struct RowRef {
  int32_t req, pos;
};

__device__ __forceinline__ RowRef row_ref(const WriteParams& W, int64_t i) {
  const int64_t k = i < W.n ? i : 0;
  return {W.row_req ? W.row_req[k] : static_cast<int32_t>(k), W.row_pos[k]};
}

__device__ __forceinline__ bool ref_in_range(const WriteParams& W, RowRef r) {
  return r.req >= 0 && r.req < W.num_req && r.pos >= 0 && r.pos < static_cast<int64_t>(kPage) * W.pt_stride;
}

// The row's page-table word (the table's first word when the request or the
// position is out of range: record_at then flags the row).
__device__ __forceinline__ int32_t page_word(const WriteParams& W, RowRef r) {
  return W.page_table[ref_in_range(W, r) ? static_cast<int64_t>(r.req) * W.pt_stride + r.pos / kPage : 0];
}

// The row's record address, or the CSA_DEV_* bit that stops it (checked in the
// documented order: request, position, page).
__device__ __forceinline__ int32_t record_at(const WriteParams& W, RowRef r, int32_t phys, uint8_t** rec) {
  if (r.req < 0 || r.req >= W.num_req) return CSA_DEV_BAD_REQUEST;
  if (r.pos < 0 || r.pos >= static_cast<int64_t>(kPage) * W.pt_stride) return CSA_DEV_LEN_OOB;
  if (phys < 0 || phys >= W.num_pages) return CSA_DEV_PAGE_OOB;
  *rec = W.kv + static_cast<int64_t>(phys) * W.page_stride + static_cast<int64_t>(r.pos % kPage) * kRec;
  return 0;
}

// A warp takes 32 rows per pass, each lane resolving one row's record; the
// resolution runs ahead of the quantisation: while a pass is quantised, the
// page-table words of the next pass and the request and position words of the
// one after are in flight. The pass is quantised four rows (one per eight-lane
// group) per step, the loads of several steps in flight together.
constexpr int kRowsPerPass = 32;  // one row's record resolved per lane
constexpr int kRowLanes = 8, kVals = kD / kRowLanes;  // lanes per row, values per lane
constexpr int32_t kNoRow = 1 << 30;

// The 16 values of row i that lane s of the row's group holds (d = 16 s .. 16 s + 15).
template <bool kBf16>
struct RowSlice {
  static constexpr int kWords = kBf16 ? 2 : 4;  // 16-byte loads per lane
  uint4 raw[kWords];
  __device__ __forceinline__ void load(const WriteParams& W, int64_t i, int sl) {
    const uint4* base = reinterpret_cast<const uint4*>(W.keys) + i * (kWords * kRowLanes) + kWords * sl;
#pragma unroll
    for (int k = 0; k < kWords; ++k) raw[k] = base[k];
  }
  __device__ __forceinline__ void values(float (&v)[kVals]) const {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(raw);
#pragma unroll
    for (int k = 0; k < kVals; ++k) {
      if constexpr (kBf16)
        v[k] = __uint_as_float((k & 1) ? (w[k >> 1] & 0xFFFF0000u) : (w[k >> 1] << 16));
      else
        v[k] = __uint_as_float(w[k]);
    }
  }
};

// RN(x / b) from y = RN(1 / b) by two FMA corrections (see the file header);
// b >= 2^-90, finite. The quotient takes x's sign (b > 0): a zero x gives a zero
// residual, whose sum with -0 would otherwise round to +0.
__device__ __forceinline__ float quotient_rn(float x, float b, float y) {
  const float q0 = x * y;
  const float q1 = fmaf(fmaf(-q0, b, x), y, q0);
  return copysignf(fmaf(fmaf(-q1, b, x), y, q1), x);
}

template <bool kBf16>
__global__ void __launch_bounds__(kWriterThreads) write_keys_kernel(const WriteParams W) {
  constexpr int kStepRows = 32 / kRowLanes;          // rows a warp quantises at once
  constexpr int kChunkSteps = kBf16 ? 4 : 2;         // steps whose loads are in flight together
  constexpr int kSteps = kRowsPerPass / kStepRows;   // steps per pass
  const int lane = threadIdx.x & 31, g = lane / kRowLanes, sl = lane % kRowLanes;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kWriterThreads / 32);
  int32_t flags = 0;
  const int64_t step = warps * kRowsPerPass;
  int64_t i0 = ((static_cast<int64_t>(blockIdx.x) * kWriterThreads + threadIdx.x) >> 5) * kRowsPerPass;
  RowRef r0 = row_ref(W, i0 + lane), r1 = row_ref(W, i0 + step + lane);
  int32_t pg0 = page_word(W, r0);
  for (; i0 < W.n; i0 += step) {
    const RowRef r2 = row_ref(W, i0 + 2 * step + lane);
    const int32_t pg1 = page_word(W, r1);
    uint8_t* my_rec = nullptr;
    const int32_t my_f = i0 + lane < W.n ? record_at(W, r0, pg0, &my_rec) : kNoRow;
    r0 = r1;
    r1 = r2;
    pg0 = pg1;
    const int rows = W.n - i0 < kRowsPerPass ? static_cast<int>(W.n - i0) : kRowsPerPass;  // uniform
    for (int c = 0; c < kSteps; c += kChunkSteps) {
      RowSlice<kBf16> x[kChunkSteps];
#pragma unroll
      for (int j = 0; j < kChunkSteps; ++j) {
        const int r = kStepRows * (c + j) + g;  // this group's row of the step, within the pass
        x[j].load(W, r < rows ? i0 + r : i0, sl);
      }
#pragma unroll
      for (int j = 0; j < kChunkSteps; ++j) {
        const int r = kStepRows * (c + j) + g;
        const int32_t f0 = __shfl_sync(0xFFFFFFFFu, my_f, r);
        uint8_t* rec = reinterpret_cast<uint8_t*>(__shfl_sync(0xFFFFFFFFu, reinterpret_cast<uintptr_t>(my_rec), r));
        float v[kVals];
        x[j].values(v);
        // magnitude bits order like the magnitudes; at or above 0x7F800000: inf or NaN
        uint32_t mbits = 0;
#pragma unroll
        for (int k = 0; k < kVals; ++k) mbits = max(mbits, __float_as_uint(v[k]) & 0x7FFFFFFFu);
#pragma unroll
        for (int o = 1; o < kRowLanes; o <<= 1) mbits = max(mbits, __shfl_xor_sync(0xFFFFFFFFu, mbits, o));
        if (r >= rows) continue;  // the group's row is past the last one
        int32_t f = f0;
        if (f == 0 && mbits >= 0x7F800000u) f = CSA_DEV_RANGE;
        if (f != 0) {  // uniform over the group
          flags |= f;
          continue;
        }
        const float amax = __uint_as_float(mbits);
        const float scale = amax / 448.0f;  // IEEE division, round to nearest even
        uint32_t word[kVals / 4] = {};
        if (scale > 0.0f) {  // a scale of 0 (amax == 0, or amax / 448 underflows): zero codes
          if (scale >= 0x1p-90f) {  // uniform over the group
            const float y = __frcp_rn(scale);
#pragma unroll
            for (int k = 0; k < kVals; ++k) v[k] = quotient_rn(v[k], scale, y);
          } else {
#pragma unroll
            for (int k = 0; k < kVals; ++k) v[k] = v[k] / scale;
          }
#pragma unroll
          for (int k = 0; k < kVals / 4; ++k) {
            const __nv_fp8x2_storage_t lo =
                __nv_cvt_float2_to_fp8x2(make_float2(v[4 * k], v[4 * k + 1]), __NV_SATFINITE, __NV_E4M3);
            const __nv_fp8x2_storage_t hi =
                __nv_cvt_float2_to_fp8x2(make_float2(v[4 * k + 2], v[4 * k + 3]), __NV_SATFINITE, __NV_E4M3);
            word[k] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
          }
        }
        uint32_t* rw = reinterpret_cast<uint32_t*>(rec);
#pragma unroll
        for (int k = 0; k < kVals / 4; ++k) rw[(kVals / 4) * sl + k] = word[k];  // codes of d = 16 sl ..
        if (sl == 0) rw[kD / 4] = __float_as_uint(scale);  // little-endian fp32 at byte 128
      }
    }
  }
  flags = static_cast<int32_t>(__reduce_or_sync(0xFFFFFFFFu, static_cast<uint32_t>(flags)));
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
  const auto kernel = W.bf16 ? write_keys_kernel<true> : write_keys_kernel<false>;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kWriterThreads, 0) != cudaSuccess || per_sm < 1)
    return CSA_ERR_CUDA;
  const int64_t rows_per_block = kRowsPerPass * (kWriterThreads / 32);
  const int64_t want = (a->n + rows_per_block - 1) / rows_per_block;
  const int64_t cap = static_cast<int64_t>(sms) * per_sm;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  kernel<<<grid, kWriterThreads, 0, static_cast<cudaStream_t>(stream)>>>(W);
  return cudaGetLastError() == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}
