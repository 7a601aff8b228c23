// csa_index.cu — the CSA indexer hot path on GB300 (sm_103a) and its C ABI.
//
// What is computed (FlashMemory-DeepSeek-V4, "Retriever architecture",
// "compressed_k format", "Two-level recall algorithm"):
//   k_n      = e4m3(record_n[0:128]) * fp32(record_n[128:132])
//   logit_bn = sum_h relu(k_n . q_b[h]) * fused_w_b[h]
//   score_bn = sigmoid(logit_bn)
// and the top-k records of each query row by (logit desc, position asc).
//
// Design (one persistent CTA per SM, warp-specialised):
//   warp 0      issuer: 1-D bulk copies of whole 8448-byte pages into a ring of
//               shared-memory stages (a record's 132-byte pitch is not 16-byte
//               aligned, so tiled tensor maps cannot address rows; whole pages can).
//   warp 1      MMA: allocates TMEM, issues tcgen05.mma kind::f8f6f4 with the
//               128-record key tile as the A operand in TMEM and the query as the
//               B operand in shared memory, accumulating fp32 in TMEM.
//   warp 2      page walker: turns (query, tile) into physical pages through the
//               page table / resident list, 32 pages at a time.
//   warp 3      query prep: splits each bf16 query row into two e4m3 terms
//               (q * 2^e_h = hi + lo, exact for every element of magnitude
//               >= 2^-2 after the per-head power-of-two scale) written in the
//               128-byte-swizzled K-major layout the MMA reads, and folds 2^-e_h
//               into the head weight.
//   warps 4-7   loader: copies each record's 128 e4m3 bytes from the staged page
//               into TMEM as the A operand (raw bytes, no conversion), and its
//               scale (NaN for an invisible record) and position beside the
//               accumulator.
//   warps 8-11  epilogue: reads the fp32 head dots from TMEM and computes
//               s * sum_h relu(x_h) w'_h; then either writes sigmoid scores or
//               keeps a thresholded candidate buffer in shared memory and writes
//               each segment's best k to a workspace slot.
// A second kernel merges the slots of each query into the exact, sorted top-k.
//
// Work split: a query row covers ceil(visible pages / 2) tiles of 128 records;
// the tiles of all rows are laid end to end and cut into one contiguous,
// equal-sized range per CTA. A CTA's range falls into "segments" (maximal runs
// of one row); segment (row b, CTA c) owns workspace slot b + c, which is unique
// because b + c grows by at least one from one segment to the next.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "csa_index.h"
#include "csa_internal.h"
#include "csa_ptx.cuh"
#include "csa_select.cuh"

namespace csa {

constexpr int kH = 64;
constexpr int kD = 128;
constexpr int kPage = 64;
constexpr int kRec = 132;
constexpr int kPageBytes = kPage * kRec;  // 8448
constexpr int kFp4Rec = 68;                // MXFP4 record: 64 code bytes + 4 UE8M0 block scales
constexpr int kFp4PageBytes = kPage * kFp4Rec;  // 4352
constexpr int kMmaRows = 128;             // records per MMA (M)
constexpr int kSub = 2;                   // MMA sub-tiles per tile
constexpr int kTile = kSub * kMmaRows;    // records per tile: the unit of every hand-off
constexpr int kTilePages = kTile / kPage; // 4

constexpr int kAStages = 2;    // TMEM A (key tile) stages: one per worker group

// Per head count H: page stages in shared memory and TMEM accumulator stages.
// The indexer runs with 64 heads: an accumulator stage holds a whole tile
// (2 sub-tiles x 64 columns). The scorer also runs with 128 heads (score and
// logit modes, for the Level-1 recall): its query buffers double, which leaves
// shared memory for 12 page stages, and a whole tile's accumulator would leave
// TMEM room for one stage, which serialises the MMA and the epilogue; so its
// stages hold one sub-tile (128 columns) each, taken and freed per sub-tile.
template <int H> struct Geo;
template <> struct Geo<64> {
  static constexpr int kStages = 16, kDStages = 3, kDCols = 2 * 64;
  static constexpr bool kSubStaged = false;
};
template <> struct Geo<128> {
  static constexpr int kStages = 12, kDStages = 3, kDCols = 128;
  static constexpr bool kSubStaged = true;
};
constexpr int kRing = 4;       // page-walker ring slots of 32 pages
constexpr int kSlotKeysMax = 2048;  // most keys a workspace slot has room for (see slot_bytes_fused)
constexpr int32_t kShortRowsMin = 512;  // rows from which the fused path takes the short-row scorer
constexpr int kCap = 2048;     // candidate buffer of one segment (keys)
constexpr int kKeyRing = 8;    // tiles of ranking keys between the workers and the selector

constexpr int kThreads = 512;
// warp roles
constexpr int kWarpIssuer = 0, kWarpMma = 1, kWarpWalker = 2, kWarpQprep = 3;
constexpr int kWarpWorker = 4;   // warps 4-7: worker group 0 (even tiles), 8-11: group 1 (odd tiles)
constexpr int kWorkerGroups = 2;
constexpr int kWarpSelect = 12;  // warps 12-15: top-k selector
constexpr int kBarSelect = 1;
constexpr int kQEmptyCount = 1 + 4 * kWorkerGroups;  // MMA commit + every worker warp

constexpr uint32_t kTmemCols = 512;
// A stage: kSub x 32 columns (128 lanes x 128 e4m3 bytes per sub-tile);
// D stage: Geo<H>::kDCols fp32 columns (128 records x H heads per sub-tile it holds).
__host__ __device__ constexpr uint32_t a_col(int s) { return static_cast<uint32_t>(s) * 32u * kSub; }
template <int H>
__host__ __device__ constexpr uint32_t d_col(int s) {
  return 32u * kSub * kAStages + static_cast<uint32_t>(s) * Geo<H>::kDCols;
}
static_assert(d_col<64>(Geo<64>::kDStages) <= kTmemCols && d_col<128>(Geo<128>::kDStages) <= kTmemCols,
              "TMEM column map");
static_assert(kAStages == kWorkerGroups, "each worker group owns one key stage");
static_assert(Geo<64>::kStages % 4 == 0 && Geo<128>::kStages % 4 == 0 && kCap >= CSA_MAX_K + kTile,
              "stage and buffer sizes");

// One MMA: 128 records x H heads x 32 bytes of K. A sub-tile takes 8 of them:
// the query's hi term over K = 0..127, then its lo term over the same K, all
// into one accumulator, so each head's column holds k . (q * 2^e_h) directly.
template <int H>
constexpr uint32_t kIdesc = idesc_e4m3_f32(128, H);
constexpr uint32_t kNaNBits = 0x7FC00000u;

// Keys kept by a cut of a candidate buffer: at least k, at most half as many
// again (or the scratch size). The window is wide enough for a sampled
// threshold to land in it almost always; a segment's slot holds this many keys
// at most, unsorted, and only the merge finds the exact k best.
__host__ __device__ __forceinline__ int loose_keep(int k) {
  const int m = k + (k >> 1);
  return m < CSA_MAX_K ? m : CSA_MAX_K;
}

// Keys the merge sorts: the power of two at or above 2k (at least 64, at most
// CSA_MAX_K); a row with more candidates is first cut to between k and this.
__host__ __device__ __forceinline__ int merge_window(int k) {
  int w = 64;
  while (w < 2 * k) w <<= 1;
  return w < CSA_MAX_K ? w : CSA_MAX_K;
}

struct Params {
  const uint16_t* q;
  const float* w;
  const uint8_t* kv;
  int64_t num_pages;
  int64_t page_stride;
  const int32_t* page_table;
  const int32_t* q_req;
  const int32_t* q_len;
  const int32_t* resident;
  const int32_t* n_resident;
  int32_t* dev_status;
  float* scores;        // score mode
  const float* in_scores;  // unfused top-k
  int64_t score_stride;
  uint8_t* ws;          // top-k modes
  int64_t slot_bytes;
  int64_t slots_offset;
  int32_t num_q;
  int32_t num_req;
  int32_t pt_stride;
  int32_t res_stride;
  int32_t k;
  int32_t grid;         // CTAs of the phase-1 kernel (slot numbering)
  int32_t fmt;          // record format: CSA_RECORD_E4M3 or CSA_RECORD_MXFP4
  int32_t raw_logits;   // score mode: write the logit instead of its sigmoid
  int32_t fold;         // score mode: 0 store, CSA_FOLD_MAX / CSA_FOLD_ADD fold the score into the output
};

struct PageInfo {
  int32_t lp;     // logical page (positions lp*64 + r)
  int32_t nrows;  // visible rows of the page (0: nothing to score)
  int32_t phys;   // physical page
  int32_t pad;
};

// ------------------------------------------------------------------ geometry

// Request of row b, or -1 when out of range.
__device__ __forceinline__ int32_t row_request(const Params& P, int32_t b) {
  const int32_t req = P.q_req ? P.q_req[b] : b;
  return (req < 0 || req >= P.num_req) ? -1 : req;
}

// Visible length of row b: q_len clamped to [0, 64 * pt_stride].
__device__ __forceinline__ int64_t row_length(const Params& P, int32_t b, int32_t* flags) {
  int64_t L = P.q_len[b];
  const int64_t cap = static_cast<int64_t>(kPage) * P.pt_stride;
  if (L < 0) {
    *flags |= CSA_DEV_LEN_OOB;
    L = 0;
  }
  if (L > cap) {
    *flags |= CSA_DEV_LEN_OOB;
    L = cap;
  }
  return L;
}

__device__ __forceinline__ int32_t resident_count(const Params& P, int32_t req, int32_t* flags) {
  int32_t n = P.n_resident[req];
  if (n < 0) {
    *flags |= CSA_DEV_LEN_OOB;
    n = 0;
  }
  if (n > P.res_stride) {
    *flags |= CSA_DEV_LEN_OOB;
    n = P.res_stride;
  }
  return n;
}

// Tiles (TP page slots each) that row b covers.
template <int TP = kTilePages>
__device__ __forceinline__ int64_t query_tiles(const Params& P, int32_t b, int32_t* flags) {
  const int32_t req = row_request(P, b);
  if (req < 0) {
    *flags |= CSA_DEV_BAD_REQUEST;
    return 0;
  }
  if (P.resident) return (resident_count(P, req, flags) + TP - 1) / TP;
  return (row_length(P, b, flags) + kPage * TP - 1) / (kPage * TP);
}

template <int TP = kTilePages>
__device__ __forceinline__ int64_t query_tiles(const Params& P, int32_t b) {
  int32_t f = 0;
  return query_tiles<TP>(P, b, &f);
}

template <int TP = kTilePages>
__device__ __forceinline__ int32_t next_nonempty(const Params& P, int32_t b) {
  while (b < P.num_q && query_tiles<TP>(P, b) == 0) ++b;
  return b;
}

__host__ __device__ __forceinline__ int64_t cta_begin(int64_t c, int64_t total, int64_t grid) {
  return c * total / grid;
}

// CTA whose (non-empty) range holds tile t, 0 <= t < total.
__host__ __device__ __forceinline__ int64_t cta_of(int64_t t, int64_t total, int64_t grid) {
  const int64_t c = ((t + 1) * grid - 1) / total;
  return c < grid - 1 ? c : grid - 1;
}

// Visible rows, logical page and physical page of page slot `j` (0..TP-1) of
// tile `lt` of row b. nrows = 0 marks a slot with nothing to score.
template <int TP = kTilePages>
__device__ PageInfo page_of(const Params& P, int32_t b, int64_t lt, int j, int32_t* flags) {
  PageInfo e{0, 0, 0, 0};
  const int32_t req = row_request(P, b);
  if (req < 0) return e;
  const int64_t L = row_length(P, b, flags);
  const int64_t npages = (L + kPage - 1) / kPage;
  const int64_t slot = static_cast<int64_t>(TP) * lt + j;
  int64_t p;
  if (P.resident) {
    if (slot >= resident_count(P, req, flags)) return e;
    p = P.resident[static_cast<int64_t>(req) * P.res_stride + slot];
    if (p < 0 || p >= npages) {
      *flags |= CSA_DEV_RESIDENT_OOB;
      return e;
    }
  } else {
    p = slot;
    if (p >= npages) return e;
  }
  e.lp = static_cast<int32_t>(p);
  if (P.page_table) {  // the unfused top-k may run without a page table
    const int32_t phys = P.page_table[static_cast<int64_t>(req) * P.pt_stride + p];
    if (phys < 0 || phys >= P.num_pages) {
      *flags |= CSA_DEV_PAGE_OOB;
      return e;
    }
    e.phys = phys;
  }
  const int64_t rows = L - p * kPage;
  e.nrows = static_cast<int32_t>(rows < kPage ? rows : kPage);
  return e;
}

// ------------------------------------------------------------------ planning

// The CTAs split the rows' tiles in row order into contiguous ranges of equal
// cost. When rows are long (at least kLongRowTiles tiles on average), each row
// that has tiles also costs kSegTiles "virtual" tiles placed before its first
// tile, so that a CTA pays for every row it starts (the selection of a new
// segment starts from nothing: every key passes until the segment has seen k
// of them): measured on this GPU, a second segment cost a CTA three to five
// tiles of time, and without the charge the CTAs that cross a row boundary
// finished last. Batches of short rows (chunked prefill) keep the plain split:
// there the charge made a few CTAs several times slower, for reasons not yet
// understood. Both figures are in records, so that they mean the same for
// every tile size: a row start costs 1024 records, and rows count as long from
// 4096 records on average.
constexpr int64_t kSegRecords = 1024, kLongRowRecords = 4096;

struct Plan {
  int64_t total;   // virtual tiles of all rows
  int64_t t0;      // first virtual tile of this CTA
  int64_t ntiles;  // tiles of this CTA (real ones)
  int64_t lt0;     // local tile of row b0 where the CTA starts
  int32_t b0;      // row of the CTA's first tile
  int32_t flags;
  int64_t r0, r1;  // real tiles before virtual tiles t0 and t0 + share (planning scratch)
};

// Block-wide: virtual tiles of every row, their running sum, and this CTA's
// share of the real tiles. CTA 0 also writes, when given, the exclusive prefix
// sums of the virtual tiles (tile_off[0 .. num_q]) and the charge per row W
// (tile_off[num_q + 1]): row b's tiles are virtual tiles tile_off[b] + W ..
// tile_off[b + 1] - 1.
template <int NT, int TP = kTilePages>
__device__ void make_plan(const Params& P, Plan* plan, int64_t* warp_sums, int32_t* tile_off) {
  constexpr int64_t kSegTiles = kSegRecords / (kPage * TP), kLongRowTiles = kLongRowRecords / (kPage * TP);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = NT / 32;
  int32_t flags = 0;
  // sums of (non-empty rows << 32) | tiles: one scan gives both (tile sums, like
  // tile_off, stay below 2^31; row counts below 2^31)
  constexpr int kShift = 32;
  constexpr int64_t kLow = (int64_t{1} << kShift) - 1;
  // pass 1: real tiles and non-empty rows, hence the charge per row and the virtual total
  int64_t part = 0;
  for (int32_t b = tid; b < P.num_q; b += NT) {
    const int64_t t = query_tiles<TP>(P, b, &flags);
    part += t | (t > 0 ? int64_t{1} << kShift : 0);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o);
  if (lane == 0) warp_sums[warp] = part;
  __syncthreads();
  int64_t packed_total = 0;
  for (int i = 0; i < NW; ++i) packed_total += warp_sums[i];
  __syncthreads();
  const int64_t real_total = packed_total & kLow, rows = packed_total >> kShift;
  const int64_t W = real_total >= kLongRowTiles * rows ? kSegTiles : 0;
  const int64_t total = real_total + W * rows;
  const int64_t t0 = cta_begin(blockIdx.x, total, gridDim.x);
  const int64_t t1 = cta_begin(blockIdx.x + 1, total, gridDim.x);
  if (tid == 0) {
    plan->total = total;
    plan->t0 = t0;
    plan->ntiles = 0;
    plan->b0 = P.num_q;
    plan->lt0 = 0;
    plan->r0 = -1;
    plan->r1 = t1 >= total ? -2 : -1;  // -2: the range runs to the last tile
  }
  __syncthreads();
  // pass 2: ordered prefix sums of the packed virtual tiles, chunk by chunk; real
  // tiles before virtual position x inside row b: real_before(b) + max(0, x - vstart(b) - W)
  const bool write_off = tile_off != nullptr && blockIdx.x == 0;
  int64_t running = 0;
  for (int32_t base = 0; base < P.num_q; base += NT) {
    const int32_t b = base + tid;
    const int64_t tr = b < P.num_q ? query_tiles<TP>(P, b) : 0;
    const int64_t t = tr > 0 ? (tr + W) | (int64_t{1} << kShift) : 0;
    int64_t incl = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    __syncthreads();
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    int64_t before = running;
    for (int i = 0; i < warp; ++i) before += warp_sums[i];
    int64_t chunk = 0;
    for (int i = 0; i < NW; ++i) chunk += warp_sums[i];
    const int64_t excl_packed = before + incl - t;
    const int64_t excl = excl_packed & kLow, v = t & kLow;
    const int64_t real_before = excl - W * (excl_packed >> kShift);
    if (b < P.num_q) {
      if (write_off) tile_off[b] = static_cast<int32_t>(excl);
      if (v > 0 && excl <= t0 && t0 < excl + v) {  // the row holding t0 (one thread)
        const int64_t lt = t0 - excl - W;
        plan->b0 = b;
        plan->lt0 = lt > 0 ? lt : 0;
        plan->r0 = real_before + (lt > 0 ? lt : 0);
      }
      if (v > 0 && excl <= t1 && t1 < excl + v) {  // the row holding t1 (one thread)
        const int64_t lt = t1 - excl - W;
        plan->r1 = real_before + (lt > 0 ? lt : 0);
      }
    }
    running += chunk;
    if (!write_off && (running & kLow) > t1) break;  // uniform: every thread sees the same running sum
  }
  __syncthreads();
  if (tid == 0) {
    // a range that runs to the last tile ends after every real tile; the loop did not
    // stop early then, so `running` holds the whole packed sum
    const int64_t r1 = plan->r1 == -2 ? (running & kLow) - W * (running >> kShift) : plan->r1;
    plan->ntiles = (plan->r0 >= 0 && r1 > plan->r0) ? r1 - plan->r0 : 0;
  }
  if (write_off && tid == 0) {
    tile_off[P.num_q] = static_cast<int32_t>(total);
    tile_off[P.num_q + 1] = static_cast<int32_t>(W);
  }
  if (flags) atomicOr(&plan->flags, flags);
  __syncthreads();
}

// ------------------------------------------------------------------ shared memory

template <int H>
struct __align__(1024) Smem {
  static constexpr int kStages = Geo<H>::kStages, kDStages = Geo<H>::kDStages;
  // Accumulator-ready signals, MMA -> worker group. The two groups take turns,
  // so a group waits on every other signal; with fewer than three slots its
  // next wait (same slot, same parity two phases later) could be satisfied by
  // the completion it has just consumed.
  static constexpr int kDSignals = kDStages >= 3 ? kDStages : 4;
  uint8_t qbuf[2][2][H * kD];      // [slot][hi/lo] e4m3, K-major, 128-byte swizzle
  uint8_t pages[kStages][kPageBytes];
  uint64_t cand[kCap];
  uint64_t scratch[CSA_MAX_K];
  uint64_t keys[kKeyRing][kTile];  // a tile's admissible keys, worker -> selector: 64 per worker warp
  uint32_t kcnt[kKeyRing][4];      // keys in each worker warp's region of the slot
  uint64_t filt;                   // (segment << 32) | value word of the selector's current threshold
  alignas(16) float wbuf[2][H];    // read as float4
  PageInfo ring[kRing * 32];
  PageInfo info[kStages];
  uint64_t full[kStages], empty[kStages];
  uint64_t afull[kAStages], aempty[kAStages];
  uint64_t dfull[kDSignals], dempty[kDStages];
  uint64_t qfull[2], qempty[2];
  uint64_t rfull[kRing], rempty[kRing];
  uint64_t kfull[kKeyRing], kempty[kKeyRing];
  uint64_t drain;
  SelectShared sel;
  Plan plan;
  int64_t warp_sums[32];
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t status;
  int32_t go[2];                   // selector leader's wait result, by tile parity
};
// alignment each field's accesses need: swizzle atoms, bulk-copy destinations, float4 loads
template <int H>
constexpr bool smem_layout_ok() {
  return offsetof(Smem<H>, qbuf) % 1024 == 0 && offsetof(Smem<H>, pages) % 16 == 0 && kPageBytes % 16 == 0 &&
         offsetof(Smem<H>, wbuf) % 16 == 0 && offsetof(Smem<H>, full) % 8 == 0 && offsetof(Smem<H>, filt) % 8 == 0;
}
static_assert(smem_layout_ok<64>() && smem_layout_ok<128>(),
              "swizzle atoms 1024-byte, bulk copies and float4 loads 16-byte, mbarriers 8-byte aligned");

// The worker-side filter of segment `seg`: a key whose value word is below the
// returned word cannot reach the segment's best k (the selector has already
// seen k keys at or above it); 0 admits every key. A word tagged with another
// segment is stale and admits everything.
template <int H>
__device__ __forceinline__ uint32_t filter_word(const Smem<H>& S, int seg) {
  const uint64_t f = *reinterpret_cast<const volatile uint64_t*>(&S.filt);
  return static_cast<uint32_t>(f >> 32) == static_cast<uint32_t>(seg) ? static_cast<uint32_t>(f) : 0u;
}

template <int H>
constexpr size_t kSmemBytes = sizeof(Smem<H>) + 1024;  // + alignment slack
static_assert(kSmemBytes<64> <= 232448 && kSmemBytes<128> <= 232448, "shared memory budget");

template <int H>
__device__ __forceinline__ Smem<H>& smem_of(uint8_t* raw) {
  return *reinterpret_cast<Smem<H>*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
}

// ------------------------------------------------------------------ roles

template <int TP = kTilePages>
struct CursorT {
  int32_t b;
  int64_t lt;
  int64_t tiles;
  __device__ void init(const Params& P, const Plan& pl) {
    b = pl.b0;
    lt = pl.lt0;
    tiles = b < P.num_q ? query_tiles<TP>(P, b) : 0;
  }
  // the row after b that has tiles, and its tile count
  static __device__ __forceinline__ void next_row(const Params& P, int32_t& b, int64_t& tiles) {
    b = next_nonempty<TP>(P, b + 1);
    tiles = b < P.num_q ? query_tiles<TP>(P, b) : 0;
  }
  __device__ void advance(const Params& P) {
    if (++lt >= tiles) {
      next_row(P, b, tiles);
      lt = 0;
    }
  }
};
using Cursor = CursorT<>;

// Broadcast of lane 0's value to the warp.
__device__ __forceinline__ bool warp_ok(bool ok) { return __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0; }


// Page walker: fills the ring with the PageInfo of the CTA's pages, 32 at a
// time (TP page slots per tile; 32 / TP tiles per ring slot). SM is the
// kernel's shared-memory struct (ring, rfull, rempty, plan, abort_flag, status).
template <int TP, class SM, class Cur = CursorT<TP>>
__device__ void walk_pages(const Params& P, SM& S) {
  static_assert(32 % TP == 0, "a ring slot holds whole tiles");
  const int lane = threadIdx.x & 31;
  const int64_t npg = static_cast<int64_t>(TP) * S.plan.ntiles;
  Cur cur;
  cur.init(P, S.plan);
  int32_t flags = 0;
#ifdef CSA_TEST_WALKER_DELAY_NS
  // Test build only: the walker publishes nothing for this long, so that the
  // roles waiting on it run out of their (shortened) wait limit.
  if (lane == 0) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < CSA_TEST_WALKER_DELAY_NS) __nanosleep(1000);
  }
  __syncwarp();
#endif
  for (int64_t pg = 0; pg < npg; pg += 32) {
    const int64_t batch = pg >> 5;
    const int slot = static_cast<int>(batch % kRing);
    int ok = 1;
    if (lane == 0) ok = mbar_wait(smem_u32(&S.rempty[slot]), static_cast<uint32_t>(((batch / kRing) & 1) ^ 1),
                                  &S.abort_flag);
    if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
    // lane j handles page pg + j: tile offset j / TP, slot j % TP
    int32_t bb = cur.b;
    int64_t ll = cur.lt + lane / TP, tb = cur.tiles;
    while (bb < P.num_q && ll >= tb) {
      ll -= tb;
      Cur::next_row(P, bb, tb);
    }
    PageInfo e{0, -1, 0, 0};
    if (pg + lane < npg && bb < P.num_q) e = page_of<TP>(P, bb, ll, lane % TP, &flags);
    S.ring[slot * 32 + lane] = e;
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&S.rfull[slot]));
    // the cursor moves on by 32 pages
    for (int t = 0; t < 32 / TP; ++t) cur.advance(P);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) flags |= __shfl_xor_sync(0xFFFFFFFFu, flags, o);
  if (lane == 0 && flags) atomicOr(&S.status, flags);
}

template <int H>
__device__ void role_walker(const Params& P, Smem<H>& S) {
  walk_pages<kTilePages>(P, S);
}

// Page copies are issued by kIssueLanes lanes in lockstep, one page each: the
// per-copy instruction latencies (ring read, barrier wait, expect_tx, copy) are
// paid once per group instead of once per page.
constexpr int kIssueLanes = 4;
static_assert(Geo<64>::kStages % kIssueLanes == 0 && Geo<128>::kStages % kIssueLanes == 0 && 32 % kIssueLanes == 0,
              "issue groups");

template <int H>
__device__ void role_issuer(const Params& P, Smem<H>& S) {
  constexpr int kStages = Smem<H>::kStages, kDStages = Smem<H>::kDStages;
  (void)kStages;
  (void)kDStages;
  const int lane = threadIdx.x & 31;
  const int64_t npg = kTilePages * S.plan.ntiles;
  const uint64_t policy = policy_evict_first();
  int64_t last = -1;  // last page this lane issued
  for (int64_t pg0 = 0; pg0 < npg; pg0 += kIssueLanes) {
    const int64_t batch = pg0 >> 5;
    const int slot = static_cast<int>(batch % kRing);
    const uint32_t rph = static_cast<uint32_t>((batch / kRing) & 1);
    if ((pg0 & 31) == 0) {
      bool ok = true;
      if (lane == 0) ok = mbar_wait(smem_u32(&S.rfull[slot]), rph, &S.abort_flag);
      if (!warp_ok(ok)) break;
    }
    const int64_t pg = pg0 + lane;
    bool ok = true;
    if (lane < kIssueLanes && pg < npg) {
      mbar_wait_drain(smem_u32(&S.rfull[slot]), rph);  // complete: acquire the walker's entries
      const PageInfo e = S.ring[slot * 32 + static_cast<int>(pg & 31)];
      const int s = static_cast<int>(pg % kStages);
      ok = mbar_wait(smem_u32(&S.empty[s]), static_cast<uint32_t>(((pg / kStages) & 1) ^ 1), &S.abort_flag);
      if (ok) {
        S.info[s] = e;
        const uint32_t fb = smem_u32(&S.full[s]);
        if (e.nrows > 0) {
          mbar_arrive_expect_tx(fb, kPageBytes);
          bulk_g2s_hint(smem_u32(S.pages[s]), P.kv + static_cast<int64_t>(e.phys) * P.page_stride, kPageBytes,
                        fb, policy);
        } else {
          mbar_arrive(fb);
        }
        last = pg;
      }
    }
    if (!__all_sync(0xFFFFFFFFu, ok)) break;
    if (lane == 0 && (((pg0 + kIssueLanes) & 31) == 0 || pg0 + kIssueLanes >= npg))
      mbar_arrive(smem_u32(&S.rempty[slot]));
  }
  // Wait for every copy this lane still has in flight before the CTA may exit.
  for (int64_t p = last; p >= 0 && p > last - kStages; p -= kIssueLanes)
    mbar_wait_drain(smem_u32(&S.full[p % kStages]), static_cast<uint32_t>((p / kStages) & 1));
}

template <int H>
__device__ void role_mma(const Params& P, Smem<H>& S) {
  constexpr int kStages = Smem<H>::kStages, kDStages = Smem<H>::kDStages;
  (void)kStages;
  (void)kDStages;
  Cursor cur;
  cur.init(P, S.plan);
  const uint32_t tmem = S.tmem_base;
  int seg = 0;
  for (int64_t i = 0; i < S.plan.ntiles; ++i) {
    const bool seg_start = (i == 0) || (cur.lt == 0);
    if (seg_start && i > 0) ++seg;
    const int qs = seg & 1;
    const int ta = static_cast<int>(i % kAStages);
    if (seg_start &&
        !mbar_wait(smem_u32(&S.qfull[qs]), static_cast<uint32_t>((seg >> 1) & 1), &S.abort_flag))
      break;
    if (!mbar_wait(smem_u32(&S.afull[ta]), static_cast<uint32_t>((i / kAStages) & 1), &S.abort_flag)) break;
    if constexpr (Geo<H>::kSubStaged) {
      bool ok = true;
#pragma unroll
      for (int sub = 0; sub < kSub && ok; ++sub) {
        // sub-tile u of the accumulator ring: its stage is free once the epilogue
        // of the sub-tile kDStages earlier has read it
        const int64_t u = kSub * i + sub;
        const int td = static_cast<int>(u % kDStages);
        ok = mbar_wait(smem_u32(&S.dempty[td]), static_cast<uint32_t>(((u / kDStages) & 1) ^ 1), &S.abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t dt = tmem + d_col<H>(td);
        const uint32_t at = tmem + a_col(ta) + 32 * sub;
#pragma unroll
        for (int term = 0; term < 2; ++term) {
          const uint32_t bq = smem_u32(S.qbuf[qs][term]);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_e4m3_ts(dt, at + kk * 8, sdesc_kmajor_sw128(bq + kk * 32), kIdesc<H>, (term | kk) != 0);
        }
      }
      if (!ok) break;
    } else {
      const int td = static_cast<int>(i % kDStages);
      if (!mbar_wait(smem_u32(&S.dempty[td]), static_cast<uint32_t>(((i / kDStages) & 1) ^ 1), &S.abort_flag))
        break;
      tc_fence_after();
#pragma unroll
      for (int sub = 0; sub < kSub; ++sub) {
        const uint32_t dt = tmem + d_col<H>(td) + H * sub;
        const uint32_t at = tmem + a_col(ta) + 32 * sub;
#pragma unroll
        for (int term = 0; term < 2; ++term) {
          const uint32_t bq = smem_u32(S.qbuf[qs][term]);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_e4m3_ts(dt, at + kk * 8, sdesc_kmajor_sw128(bq + kk * 32), kIdesc<H>, (term | kk) != 0);
        }
      }
    }
    mma_commit(smem_u32(&S.aempty[ta]));
    mma_commit(smem_u32(&S.dfull[i % Smem<H>::kDSignals]));
    const bool seg_end = (i == S.plan.ntiles - 1) || (cur.lt == cur.tiles - 1);
    if (seg_end) mma_commit(smem_u32(&S.qempty[qs]));
    cur.advance(P);
  }
  mma_commit(smem_u32(&S.drain));
  mbar_wait_drain(smem_u32(&S.drain), 0);
}

// Per-head power-of-two scale 2^e (and 1 / 2^e) mapping the head's largest |q|,
// m, into (224, 448] for every finite bf16 m, subnormals included (2^-133 up to
// 2^128): e runs from -120 to 141. 2^e above 2^126 is not an fp32 value, so the
// scale is returned as two factors, sc * sc2 (sc2 = 1 unless e > 126), which a
// value is multiplied by in turn (each product exact); 1 / 2^e is then an fp32
// subnormal, still exact. A non-finite m is flagged and treated as 1.
__device__ __forceinline__ void head_scale(float m, int32_t* flags, float* sc, float* sc2, float* isc) {
  if (!isfinite(m)) {
    *flags |= CSA_DEV_RANGE;
    m = 1.0f;
  }
  int E2;
  const float f = frexpf(m, &E2);
  int e = (f <= 0.875f) ? 9 - E2 : 8 - E2;
  e = e < -126 ? -126 : (e > 141 ? 141 : e);
  const int e1 = e > 126 ? 126 : e;
  *sc = __uint_as_float(static_cast<uint32_t>(e1 + 127) << 23);
  *sc2 = __uint_as_float(static_cast<uint32_t>(e - e1 + 127) << 23);
  *isc = e <= 126 ? __uint_as_float(static_cast<uint32_t>(127 - e) << 23) : __uint_as_float(1u << (149 - e));
}

// e4m3 hi and lo terms of two scaled query values (a in the low byte of each):
// hi = e4m3(x), lo = e4m3(x - hi).
__device__ __forceinline__ void split_pair(float a, float c, uint32_t* hi2, uint32_t* lo2) {
  uint16_t h2, l2;
  uint32_t hf;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h2) : "f"(c), "f"(a));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hf) : "h"(h2));
  const float ah = __half2float(__ushort_as_half(static_cast<uint16_t>(hf & 0xFFFFu)));
  const float ch = __half2float(__ushort_as_half(static_cast<uint16_t>(hf >> 16)));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(l2) : "f"(c - ch), "f"(a - ah));
  *hi2 = h2;
  *lo2 = l2;
}

// Byte offset of K-chunk `chunk` (16 bytes) of head h in a 128-byte-swizzled,
// K-major query buffer (8-row atoms of 1024 bytes).
__device__ __forceinline__ uint32_t qbuf_offset(int h, int chunk) {
  return (h >> 3) * 1024 + (h & 7) * 128 + (((chunk ^ (h & 7)) & 7) << 4);
}

// Splits one bf16 query row into e4m3 hi + lo terms (per-head power-of-two
// scale so that the largest |q| maps into (224, 448]) in the swizzled layout.
//
// The whole row is requested before the loop (the head weights, one per lane
// and half, the first batch of q, and the rest of q into L2), and each batch's
// loads are issued before the previous batch is processed: the first query of
// a CTA is prepared while every CTA's first page copies load HBM, and a loop
// that waits for memory once per head or per batch took about 11 us there.
template <int H, class SM>
__device__ void prep_query(const Params& P, SM& S, int32_t b, int qs, int32_t* flags) {
  const int lane = threadIdx.x & 31;
  const uint16_t* qrow = P.q + static_cast<int64_t>(b) * H * kD;
  const float* wrow = P.w + static_cast<int64_t>(b) * H;
  uint8_t* hi = S.qbuf[qs][0];
  uint8_t* lo = S.qbuf[qs][1];
  // 64 heads: each lane holds the weights of heads lane and lane + 32. 128 heads: the raw
  // weights go to the slot first and each is scaled in place once its head's scale is known
  // (four per lane would be indexed by a run-time head).
  float w_first = 0.0f, w_second = 0.0f;
  if constexpr (H == 64) {
    w_first = __ldg(wrow + lane);
    w_second = __ldg(wrow + 32 + lane);
  } else {
#pragma unroll
    for (int j = 0; j < H / 32; ++j) S.wbuf[qs][32 * j + lane] = __ldg(wrow + 32 * j + lane);
    __syncwarp();
  }
  {
    const char* base = reinterpret_cast<const char*>(qrow);  // H rows of 256 bytes: H / 16 lines per lane
#pragma unroll
    for (int j = 0; j < H / 16; ++j) asm volatile("prefetch.global.L2 [%0];" ::"l"(base + (lane + 32 * j) * 128));
  }
  uint2 raw[8], nxt[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) raw[j] = __ldg(reinterpret_cast<const uint2*>(qrow + j * kD + lane * 4));
#pragma unroll 1
  for (int h0 = 0; h0 < H; h0 += 8) {
    if (h0 + 8 < H) {
#pragma unroll
      for (int j = 0; j < 8; ++j) nxt[j] = __ldg(reinterpret_cast<const uint2*>(qrow + (h0 + 8 + j) * kD + lane * 4));
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int h = h0 + j;
      float x[4];
      x[0] = __uint_as_float(raw[j].x << 16);
      x[1] = __uint_as_float(raw[j].x & 0xFFFF0000u);
      x[2] = __uint_as_float(raw[j].y << 16);
      x[3] = __uint_as_float(raw[j].y & 0xFFFF0000u);
      float m = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      float sc, sc2, isc;
      head_scale(m, flags, &sc, &sc2, &isc);
      uint32_t whi = 0, wlo = 0;
#pragma unroll
      for (int pr = 0; pr < 2; ++pr) {
        uint32_t h2, l2;
        split_pair(x[2 * pr] * sc * sc2, x[2 * pr + 1] * sc * sc2, &h2, &l2);
        whi |= h2 << (16 * pr);
        wlo |= l2 << (16 * pr);
      }
      const uint32_t off = qbuf_offset(h, lane >> 2) + (lane & 3) * 4;
      *reinterpret_cast<uint32_t*>(hi + off) = whi;
      *reinterpret_cast<uint32_t*>(lo + off) = wlo;
      if constexpr (H == 64) {
        if (lane == (h & 31)) S.wbuf[qs][h] = (h < 32 ? w_first : w_second) * isc;
      } else {
        if (lane == (h & 31)) S.wbuf[qs][h] *= isc;
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) raw[j] = nxt[j];
  }
}

// The first segment's query, prepared by the whole CTA in the kernel's prologue,
// before any page copy is in flight, into query slot 0: thread t takes the 16
// elements 16p .. 16p+15 of head h = t / 8 (p = t % 8), so that the row's loads
// are all issued at once. Same arithmetic and layout as prep_query.
static_assert(kThreads == 64 * (kD / 16), "64 heads per pass, one thread per 16 elements");
template <int H, class SM>
__device__ void prep_first_query(const Params& P, SM& S, int32_t b, int32_t* flags) {
  const int tid = threadIdx.x, p = tid & 7;
#pragma unroll
  for (int pass = 0; pass < H / 64; ++pass) {
  const int h = (tid >> 3) + 64 * pass;
  const uint16_t* src = P.q + (static_cast<int64_t>(b) * H + h) * kD + p * 16;
  const uint4 r0 = __ldg(reinterpret_cast<const uint4*>(src));
  const uint4 r1 = __ldg(reinterpret_cast<const uint4*>(src + 8));
  const float wv = p == 0 ? __ldg(P.w + static_cast<int64_t>(b) * H + h) : 0.0f;
  const uint32_t u[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
  float x[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(u[i] << 16);
    x[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(x[i]));
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));  // the head's 8 threads
  float sc, sc2, isc;
  head_scale(m, flags, &sc, &sc2, &isc);
  uint32_t whi[4], wlo[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t h0, l0, h1, l1;
    split_pair(x[4 * i] * sc * sc2, x[4 * i + 1] * sc * sc2, &h0, &l0);
    split_pair(x[4 * i + 2] * sc * sc2, x[4 * i + 3] * sc * sc2, &h1, &l1);
    whi[i] = h0 | (h1 << 16);
    wlo[i] = l0 | (l1 << 16);
  }
  const uint32_t off = qbuf_offset(h, p);
  *reinterpret_cast<uint4*>(S.qbuf[0][0] + off) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
  *reinterpret_cast<uint4*>(S.qbuf[0][1] + off) = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
  if (p == 0) S.wbuf[0][h] = wv * isc;
  }
}

// Prepares the queries of the CTA's later segments (the first one is prepared
// in the prologue), each as soon as its slot is free. TP: pages per tile of the
// calling kernel; SM: its shared-memory struct (qbuf, wbuf, qfull, qempty, plan,
// abort_flag, status).
template <int H, int TP, class SM>
__device__ void prep_segments(const Params& P, SM& S) {
  const int lane = threadIdx.x & 31;
  int32_t flags = 0;
  int64_t done = query_tiles<TP>(P, S.plan.b0) - S.plan.lt0;
  int32_t b = next_nonempty<TP>(P, S.plan.b0 + 1);
  for (int seg = 1; done < S.plan.ntiles; ++seg) {
    const int qs = seg & 1;
    int ok = 1;
    if (lane == 0)
      ok = mbar_wait(smem_u32(&S.qempty[qs]), static_cast<uint32_t>(((seg >> 1) & 1) ^ 1), &S.abort_flag);
    if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
    prep_query<H>(P, S, b, qs, &flags);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&S.qfull[qs]));
    done += query_tiles<TP>(P, b);
    b = next_nonempty<TP>(P, b + 1);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) flags |= __shfl_xor_sync(0xFFFFFFFFu, flags, o);
  if (lane == 0 && flags) atomicOr(&S.status, flags);
}

template <int H>
__device__ void role_qprep(const Params& P, Smem<H>& S) {
  prep_segments<H, kTilePages>(P, S);
}

// Packed fp32 pairs (two IEEE binary32 operations per instruction, round to nearest).
__device__ __forceinline__ uint64_t f2pack_(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2unpack_(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2fma_(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// The head sum of one record (TMEM address tc: its accumulator row) when a
// record of the warp has a negative scale: relu(s x) = |s| relu(sign(s) x), with
// g = sign(s); the caller multiplies by |s|. Out of line: it is rare.
template <int H>
__device__ __noinline__ float head_sum_signed(uint32_t tc, const float4* wv, float g) {
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll 1
  for (int c = 0; c < H; c += 32) {
    uint32_t x[32];
    tmem_ld16(tc + c, *reinterpret_cast<uint32_t(*)[16]>(&x[0]));
    tmem_ld16(tc + c + 16, *reinterpret_cast<uint32_t(*)[16]>(&x[16]));
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 wq = wv[(c >> 2) + j];
      float a[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = g * __uint_as_float(x[4 * j + i]);
      acc[(2 * j) & 3] = f2fma_(f2pack_(fmaxf(a[0], 0.f), fmaxf(a[1], 0.f)), f2pack_(wq.x, wq.y), acc[(2 * j) & 3]);
      acc[(2 * j + 1) & 3] =
          f2fma_(f2pack_(fmaxf(a[2], 0.f), fmaxf(a[3], 0.f)), f2pack_(wq.z, wq.w), acc[(2 * j + 1) & 3]);
    }
  }
  float p[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) f2unpack_(acc[i], p[2 * i], p[2 * i + 1]);
  return ((p[0] + p[4]) + (p[1] + p[5])) + ((p[2] + p[6]) + (p[3] + p[7]));
}

// One warp of a worker group: TMEM lane quarter q of every tile the group owns
// (tiles i with i % kWorkerGroups == group). It moves its records' key bytes
// (32 rows of each of the kSub sub-tiles) from the staged pages into the TMEM
// A operand ("load") and turns the MMA's head dots into logits ("epilogue").
// Once the MMA of own tile t is done, the group's key stage is free: the warp
// loads own tile t + kWorkerGroups first, so that its MMA overlaps the
// epilogue of t. The warps never wait on each other.
template <bool kTopk, int H>
__device__ void role_worker(const Params& P, Smem<H>& S) {
  constexpr int kStages = Smem<H>::kStages, kDStages = Smem<H>::kDStages;
  const int wi = (threadIdx.x >> 5) - kWarpWorker;
  const int group = wi >> 2;
  const int q = wi & 3;
  const int lane = threadIdx.x & 31;
  const int half = q >> 1;                 // page of each sub-tile this quarter reads
  const int r = 32 * (q & 1) + lane;       // record row inside that page
  const int row = 32 * q + lane;           // record row inside a sub-tile
  const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
  const uint32_t tmem = S.tmem_base;
  const int64_t nt = S.plan.ntiles;

  // Loads own tile i. Returns false on abort; per sub-tile, the scale bits (NaN
  // when the record is not visible) and the record's logical position.
  auto load = [&](int64_t i, uint32_t (&sc)[kSub], uint32_t (&pos)[kSub]) -> bool {
    const int ta = static_cast<int>(i % kAStages);
    // every lane waits, and so acquires the pages itself: no divergent branch, no broadcast
    bool ok = mbar_wait(smem_u32(&S.aempty[ta]), static_cast<uint32_t>(((i / kAStages) & 1) ^ 1), &S.abort_flag);
#pragma unroll
    for (int sub = 0; sub < kSub; ++sub) {
      const int64_t pg = kTilePages * i + 2 * sub + half;
      ok = ok && mbar_wait(smem_u32(&S.full[pg % kStages]), static_cast<uint32_t>((pg / kStages) & 1),
                           &S.abort_flag);
    }
    if (!__all_sync(0xFFFFFFFFu, ok)) return false;
#pragma unroll
    for (int sub = 0; sub < kSub; ++sub) {
      const int64_t pg = kTilePages * i + 2 * sub + half;
      const int s = static_cast<int>(pg % kStages);
      const PageInfo e = S.info[s];
      const uint8_t* src = S.pages[s] + r * kRec;
      uint32_t v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = *reinterpret_cast<const uint32_t*>(src + 4 * j);
      const uint32_t scale = *reinterpret_cast<const uint32_t*>(src + kD);
      sc[sub] = r < e.nrows ? scale : kNaNBits;
      pos[sub] = static_cast<uint32_t>(e.lp * kPage + r);
      tmem_st32(tmem + a_col(ta) + 32 * sub + lane_off, v);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
#pragma unroll
      for (int sub = 0; sub < kSub; ++sub)
        mbar_arrive(smem_u32(&S.empty[(kTilePages * i + 2 * sub + half) % kStages]));
      mbar_arrive(smem_u32(&S.afull[ta]));
    }
    return true;
  };

  // Logits of this lane's two records (one per sub-tile) in D stage td. Both
  // sub-tiles are read per TMEM wait, and their sums are independent chains.
  // relu(s * x) = |s| * relu(sign(s) * x); in practice every record of the warp
  // has s >= 0 (one vote), and then the sign multiply drops out.
  static_assert(kSub == 2, "the epilogue reads two sub-tiles at a time");
  auto logits_of = [&](int td, const uint32_t (&sc)[kSub], int seg, float (&logit)[kSub]) {
    const float4* wv = reinterpret_cast<const float4*>(S.wbuf[seg & 1]);
    const float s0 = __uint_as_float(sc[0]), s1 = __uint_as_float(sc[1]);
    const float g0 = s0 < 0.0f ? -1.0f : 1.0f, g1 = s1 < 0.0f ? -1.0f : 1.0f;
    const bool all_pos = __all_sync(0xFFFFFFFFu, g0 > 0.0f && g1 > 0.0f);
    float a0[8], a1[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) a0[j] = a1[j] = 0.f;
#pragma unroll 1
    for (int c = 0; c < H; c += 16) {  // heads c .. c+15 of both records
      uint32_t x0[16], x1[16];
      tmem_ld16(tmem + d_col<H>(td) + c + lane_off, x0);
      tmem_ld16(tmem + d_col<H>(td) + H + c + lane_off, x1);
      tmem_wait_ld();
      float4 w4[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) w4[j] = wv[(c >> 2) + j];
      const float* w = reinterpret_cast<const float*>(w4);
      if (all_pos) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          a0[j & 7] = fmaf(fmaxf(__uint_as_float(x0[j]), 0.f), w[j], a0[j & 7]);
          a1[j & 7] = fmaf(fmaxf(__uint_as_float(x1[j]), 0.f), w[j], a1[j & 7]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          a0[j & 7] = fmaf(fmaxf(g0 * __uint_as_float(x0[j]), 0.f), w[j], a0[j & 7]);
          a1[j & 7] = fmaf(fmaxf(g1 * __uint_as_float(x1[j]), 0.f), w[j], a1[j & 7]);
        }
      }
    }
    logit[0] = fabsf(s0) * (((a0[0] + a0[4]) + (a0[1] + a0[5])) + ((a0[2] + a0[6]) + (a0[3] + a0[7])));
    logit[1] = fabsf(s1) * (((a1[0] + a1[4]) + (a1[1] + a1[5])) + ((a1[2] + a1[6]) + (a1[3] + a1[7])));
  };

  // Logit of this lane's record in the sub-tile whose accumulator is stage td
  // (sub-staged accumulators): two 16-head chunks per TMEM wait, four packed
  // pairs of sums (two fp32 multiply-adds per instruction).
  auto logit_one = [&](int td, uint32_t scb, int seg) -> float {
    const float4* wv = reinterpret_cast<const float4*>(S.wbuf[seg & 1]);
    const float s = __uint_as_float(scb);
    const float g = s < 0.0f ? -1.0f : 1.0f;
    if (!__all_sync(0xFFFFFFFFu, g > 0.0f))  // rare: out of line, away from this loop
      return fabsf(s) * head_sum_signed<H>(tmem + d_col<H>(td) + lane_off, wv, g);
    uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll 1
    for (int c = 0; c < H; c += 32) {  // heads c .. c+31
      uint32_t x[32];
      tmem_ld16(tmem + d_col<H>(td) + c + lane_off, *reinterpret_cast<uint32_t(*)[16]>(&x[0]));
      tmem_ld16(tmem + d_col<H>(td) + c + 16 + lane_off, *reinterpret_cast<uint32_t(*)[16]>(&x[16]));
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 wq = wv[(c >> 2) + j];
        float a[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = __uint_as_float(x[4 * j + i]);
        acc[(2 * j) & 3] = f2fma_(f2pack_(fmaxf(a[0], 0.f), fmaxf(a[1], 0.f)), f2pack_(wq.x, wq.y), acc[(2 * j) & 3]);
        acc[(2 * j + 1) & 3] =
            f2fma_(f2pack_(fmaxf(a[2], 0.f), fmaxf(a[3], 0.f)), f2pack_(wq.z, wq.w), acc[(2 * j + 1) & 3]);
      }
    }
    float p[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) f2unpack_(acc[i], p[2 * i], p[2 * i + 1]);
    return fabsf(s) * (((p[0] + p[4]) + (p[1] + p[5])) + ((p[2] + p[6]) + (p[3] + p[7])));
  };

  // Sub-staged accumulators: the first sub-tile's logit, read and its stage freed
  // before the next own tile is loaded (the next tile's MMA waits for this stage).
  auto first_half = [&](int64_t i, uint32_t sc0, int seg) -> float {
    tc_fence_after();
    const int td = static_cast<int>((kSub * i) % kDStages);
    const float l = logit_one(td, sc0, seg);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&S.dempty[td]));
    return l;
  };

  // Epilogue of own tile i of row b, local tile lt, segment `seg`; the caller
  // has seen the tile's accumulator complete.
  auto epilogue = [&](int64_t i, int32_t b, int64_t lt, int seg, const uint32_t (&sc)[kSub],
                      const uint32_t (&pos)[kSub], float logit0, const float (&prev)[kSub]) -> bool {
    tc_fence_after();
    float logit[kSub];
    if constexpr (Geo<H>::kSubStaged) {
      static_assert(kSub == 2, "first_half reads sub-tile 0, this sub-tile 1");
      logit[0] = logit0;
      const int td = static_cast<int>((kSub * i + 1) % kDStages);
      logit[1] = logit_one(td, sc[1], seg);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&S.dempty[td]));
    } else {
      (void)logit0;
      const int td = static_cast<int>(i % kDStages);
      logits_of(td, sc, seg, logit);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&S.dempty[td]));
    }

    if constexpr (!kTopk) {
      float* out = P.scores + static_cast<int64_t>(b) * P.score_stride + lt * kTile + row;
#pragma unroll
      for (int sub = 0; sub < kSub; ++sub)
        if (!isnan(__uint_as_float(sc[sub]))) {
          const float v = P.raw_logits ? logit[sub] : __frcp_rn(1.0f + __expf(-logit[sub]));
          float* o = out + kMmaRows * sub;
          *o = P.fold == 0 ? v : (P.fold == CSA_FOLD_MAX ? fmaxf(prev[sub], v) : prev[sub] + v);
        }
    } else {
      const int slot = static_cast<int>(i % kKeyRing);
      const bool ok2 = mbar_wait(smem_u32(&S.kempty[slot]), static_cast<uint32_t>(((i / kKeyRing) & 1) ^ 1),
                                 &S.abort_flag);
      if (!__all_sync(0xFFFFFFFFu, ok2)) return false;
      // keys that can still make the segment's best k, packed into this warp's region
      const uint32_t thr = filter_word(S, seg);
      const uint32_t lt = lanemask_lt();
      uint64_t* region = S.keys[slot] + 64 * q;
      uint32_t cnt = 0;
#pragma unroll
      for (int sub = 0; sub < kSub; ++sub) {
        const bool valid = !isnan(__uint_as_float(sc[sub])) && !isnan(logit[sub]);
        const uint64_t key = valid ? make_key(logit[sub], static_cast<int32_t>(pos[sub])) : 0ull;
        const bool take = valid && static_cast<uint32_t>(key >> 32) >= thr;
        const uint32_t ballot = __ballot_sync(0xFFFFFFFFu, take);
        if (take) region[cnt + __popc(ballot & lt)] = key;
        cnt += __popc(ballot);
      }
      if (lane == 0) S.kcnt[slot][q] = cnt;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&S.kfull[slot]));
    }
    return true;
  };

  // scale bits and positions of the current own tile and of the next one
  uint32_t cur_sc[kSub], cur_pos[kSub], nxt_sc[kSub], nxt_pos[kSub];
#pragma unroll
  for (int u = 0; u < kSub; ++u) cur_sc[u] = cur_pos[u] = nxt_sc[u] = nxt_pos[u] = 0;
  bool ok = true;
  if (group < nt) ok = load(group, cur_sc, cur_pos);

  Cursor cur;
  cur.init(P, S.plan);
  int seg = 0, wseg = -1;
  for (int64_t t = 0; ok && t < nt; ++t) {
    const bool seg_start = (t == 0) || (cur.lt == 0);
    if (seg_start && t > 0) ++seg;
    const bool seg_end = (t == nt - 1) || (cur.lt == cur.tiles - 1);
    if (t % kWorkerGroups == group) {
      if (seg != wseg) {  // first own tile of this segment: its head weights must be ready
        const bool okq = mbar_wait(smem_u32(&S.qfull[seg & 1]), static_cast<uint32_t>((seg >> 1) & 1), &S.abort_flag);
        if (!__all_sync(0xFFFFFFFFu, okq)) break;
        wseg = seg;
      }
      // MMA of tile t done: its accumulator is ready and the group's key stage is free
      constexpr int kDSignals = Smem<H>::kDSignals;
      const bool okd = mbar_wait(smem_u32(&S.dfull[t % kDSignals]), static_cast<uint32_t>((t / kDSignals) & 1),
                                 &S.abort_flag);
      if (!__all_sync(0xFFFFFFFFu, okd)) break;
      // a fold reads the plane's current values: issue those loads now, so that they
      // arrive while the accumulators are read and the next tile is staged
      float prev[kSub] = {0.0f, 0.0f};
      if constexpr (!kTopk) {
        if (P.fold != 0) {
          const float* out = P.scores + static_cast<int64_t>(cur.b) * P.score_stride + cur.lt * kTile + row;
#pragma unroll
          for (int sub = 0; sub < kSub; ++sub)
            if (!isnan(__uint_as_float(cur_sc[sub]))) prev[sub] = out[kMmaRows * sub];
        }
      }
      float logit0 = 0.0f;
      if constexpr (Geo<H>::kSubStaged) logit0 = first_half(t, cur_sc[0], seg);
      if (t + kWorkerGroups < nt) {
        ok = load(t + kWorkerGroups, nxt_sc, nxt_pos);
        if (!ok) break;
      }
      ok = epilogue(t, cur.b, cur.lt, seg, cur_sc, cur_pos, logit0, prev);
#pragma unroll
      for (int u = 0; u < kSub; ++u) {
        cur_sc[u] = nxt_sc[u];
        cur_pos[u] = nxt_pos[u];
      }
    }
    if (seg_end) {  // done with this segment's head weights
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&S.qempty[seg & 1]));
    }
    cur.advance(P);
  }
}

// Top-k selector (warps 12-15): takes each tile's admissible keys in tile
// order (the workers have dropped keys below the segment's published
// threshold), keeps those above the running threshold in a shared-memory
// buffer, cuts the buffer back to between k and loose_keep(k) keys when it
// fills, publishes the new threshold to the workers, and writes each segment's
// survivors (at most loose_keep(k), unsorted) to workspace slot (row + CTA).
template <int H>
__device__ void role_select(const Params& P, Smem<H>& S) {
  constexpr int kStages = Smem<H>::kStages, kDStages = Smem<H>::kDStages;
  (void)kStages;
  (void)kDStages;
  const int g = threadIdx.x - kWarpSelect * 32;
  const int sw = g >> 5, lane = g & 31;
  Cursor cur;
  cur.init(P, S.plan);
  int seg = 0;
  for (int64_t t = 0; t < S.plan.ntiles; ++t) {
    const int slot = static_cast<int>(t % kKeyRing);
    const uint32_t ph = static_cast<uint32_t>((t / kKeyRing) & 1);
    if (g == 0) S.go[t & 1] = mbar_wait(smem_u32(&S.kfull[slot]), ph, &S.abort_flag) ? 1 : 0;
    named_bar_sync(kBarSelect, 128);  // passes the leader's acquire of the slot on to the group
    if (!S.go[t & 1]) break;
    const uint64_t tau = S.sel.tau;
    const int c = static_cast<int>(S.kcnt[slot][sw]);
    const uint64_t* region = S.keys[slot] + 64 * sw;
    const uint64_t k0 = lane < c ? region[lane] : 0ull;
    const uint64_t k1 = lane + 32 < c ? region[lane + 32] : 0ull;
    append_keys2(S.cand, k0, k0 > tau, k1, k1 > tau, &S.sel);
    named_bar_sync(kBarSelect, 128);
    if (g == 0) mbar_arrive(smem_u32(&S.kempty[slot]));
    shrink_if_above<128, 128>(S.cand, S.scratch, kCap - kTile, P.k, loose_keep(P.k), &S.sel, kBarSelect, g);
    const bool seg_end = (t == S.plan.ntiles - 1) || (cur.lt == cur.tiles - 1);
    if (seg_end) {
      shrink_if_above<128, 128>(S.cand, S.scratch, loose_keep(P.k), P.k, loose_keep(P.k), &S.sel, kBarSelect, g);
      const int n = static_cast<int>(S.sel.n);
      uint8_t* out = P.ws + P.slots_offset + (static_cast<int64_t>(cur.b) + blockIdx.x) * P.slot_bytes;
      uint64_t* ent = reinterpret_cast<uint64_t*>(out + 16);
      for (int j = g; j < n; j += 128) ent[j] = S.cand[j];
      named_bar_sync(kBarSelect, 128);
      if (g == 0) {
        *reinterpret_cast<int32_t*>(out) = n;
        S.sel.n = 0;
        S.sel.tau = 0;
      }
      named_bar_sync(kBarSelect, 128);
      ++seg;
    }
    if (g == 0) {
      const uint64_t T = S.sel.tau + 1;  // keys >= T are admitted
      *reinterpret_cast<volatile uint64_t*>(&S.filt) =
          (static_cast<uint64_t>(static_cast<uint32_t>(seg)) << 32) | static_cast<uint32_t>(S.sel.tau ? T >> 32 : 0);
    }
    cur.advance(P);
  }
}

template <bool kTopk, int H>
__global__ void __launch_bounds__(kThreads, 1) score_kernel(const Params P) {
  constexpr int kStages = Smem<H>::kStages, kDStages = Smem<H>::kDStages;
  extern __shared__ uint8_t smem_raw[];
  Smem<H>& S = smem_of<H>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    S.plan.flags = 0;
    S.abort_flag = 0;
    S.status = 0;
    S.sel.n = 0;
    S.sel.tau = 0;
    S.filt = ~0ull;  // tagged with no segment: admits everything
  }
  __syncthreads();
  make_plan<kThreads>(P, &S.plan, S.warp_sums,
                      kTopk ? reinterpret_cast<int32_t*>(P.ws) : nullptr);
  if (tid == 0 && blockIdx.x == 0 && S.plan.flags && P.dev_status) atomicOr(P.dev_status, S.plan.flags);
  if (S.plan.ntiles == 0) return;  // uniform

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&S.full[s]), 1);
      mbar_init(smem_u32(&S.empty[s]), 2);
    }
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(smem_u32(&S.afull[s]), 4);  // the four warps of the loading worker group
      mbar_init(smem_u32(&S.aempty[s]), 1);
    }
    for (int s = 0; s < Smem<H>::kDSignals; ++s) mbar_init(smem_u32(&S.dfull[s]), 1);
    for (int s = 0; s < kDStages; ++s) mbar_init(smem_u32(&S.dempty[s]), 4);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&S.qfull[s]), 1);
      mbar_init(smem_u32(&S.qempty[s]), kQEmptyCount);
    }
    for (int s = 0; s < kKeyRing; ++s) {
      mbar_init(smem_u32(&S.kfull[s]), 4);
      mbar_init(smem_u32(&S.kempty[s]), 1);
    }
    for (int s = 0; s < kRing; ++s) {
      mbar_init(smem_u32(&S.rfull[s]), 1);
      mbar_init(smem_u32(&S.rempty[s]), 1);
    }
    mbar_init(smem_u32(&S.drain), 1);
    mbar_init_fence();
    fence_proxy_async_smem();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(&S.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  {
    int32_t qflags = 0;
    prep_first_query<H>(P, S, S.plan.b0, &qflags);
    fence_proxy_async_smem();  // the MMA reads the query through the async proxy
    if (qflags) atomicOr(&S.status, qflags);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) mbar_arrive(smem_u32(&S.qfull[0]));

  if (warp == kWarpIssuer) {
    role_issuer(P, S);
  } else if (warp == kWarpMma) {
    if ((tid & 31) == 0) role_mma(P, S);
  } else if (warp == kWarpWalker) {
    role_walker(P, S);
  } else if (warp == kWarpQprep) {
    role_qprep(P, S);
  } else if (warp < kWarpSelect) {
    role_worker<kTopk, H>(P, S);
  } else if (kTopk) {
    role_select(P, S);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(S.tmem_base, kTmemCols);
  }
  if (tid == 0 && P.dev_status) {
    const int32_t st = S.status | (S.abort_flag ? CSA_DEV_TIMEOUT : 0);
    if (st) atomicOr(P.dev_status, st);
  }
}

}  // namespace csa

#include "csa_score64.cuh"

namespace csa {

// ------------------------------------------------------------------ merge

// A merge CTA is small so that several rows run on each SM: the merge is
// latency-bound (a few dependent global reads, then shared-memory passes).
constexpr int kMergeThreads = 256;
constexpr int kMergeCap = 4096;   // candidate buffer; a row with more is cut back between chunks of slots
constexpr int kMergeSlots = CSA_MAX_CTAS + 1;
static_assert(CSA_MAX_K + kSlotKeysMax <= kMergeCap, "after a cut to merge_window(k), any slot must fit");

constexpr int kRankBins = 1024;  // bins of the final rank sort
static_assert(kMergeThreads / 32 <= 8, "the rank sort's per-warp partials fit sel.part");

struct MergeSmem {
  uint64_t cand[kMergeCap];
  uint64_t scratch[CSA_MAX_K];  // also the rank sort's scatter buffer (merge_window(k) <= CSA_MAX_K keys)
  uint32_t rank_hist[kRankBins], rank_cur[kRankBins];
  int32_t offs[kMergeSlots];  // exclusive prefix of the row's slot counts
  SelectShared sel;
};

// Sorts the n <= merge_window(k) candidates descending: by rank over value bins,
// or by the sorting network when the values crowd into a few bins.
__device__ __forceinline__ void merge_sort_desc(MergeSmem& S, int n, int tid) {
  if (!rank_sort_desc<kMergeThreads, kRankBins>(S.cand, n, S.scratch, S.rank_hist, S.rank_cur, &S.sel.part[0][0], 0,
                                                tid))
    sort_prefix_desc<kMergeThreads>(S.cand, n, 0, tid);
}

// One CTA per query row: the row's segment slots each hold at most
// loose_keep(k) keys, unsorted. They are gathered into shared memory (a row
// with more candidates than fit is cut back between chunks of slots), cut to
// between k and merge_window(k) keys, sorted, and the first k written out by
// (value desc, position asc), padded with -1 / 0.
template <bool kFromLogit>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const Params P, int32_t* idx, float* vals) {
  extern __shared__ uint8_t smem_raw[];
  MergeSmem& S = *reinterpret_cast<MergeSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~uintptr_t(15));
  const int tid = threadIdx.x;
  const int32_t b = blockIdx.x;
  const int32_t* tile_off = reinterpret_cast<const int32_t*>(P.ws);
  const int cap = static_cast<int>((P.slot_bytes - 16) / 8), window = merge_window(P.k);
  if (tid == 0) {
    S.sel.n = 0;
    S.sel.tau = 0;
  }
  // Launched as a programmatic dependent of the scoring kernel, this CTA may
  // start while that grid still runs: wait here until it has completed and its
  // slot writes are visible (returns at once after an ordinary launch).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // row b's tiles are virtual tiles t0 + W .. t1 - 1 (none when t0 == t1)
  const int64_t t0 = tile_off[b], t1 = tile_off[b + 1], total = tile_off[P.num_q], W = tile_off[P.num_q + 1];
  int64_t c0 = 0, c1 = -1;
  if (t0 < t1) {
    c0 = cta_of(t0 + W, total, P.grid);
    c1 = cta_of(t1 - 1, total, P.grid);
  }
  const int nslots = static_cast<int>(c1 - c0 + 1);  // 0 for an empty row
  auto slot_ptr = [&](int j) {
    return P.ws + P.slots_offset + (static_cast<int64_t>(b) + c0 + j) * P.slot_bytes;
  };
  // slot counts (0 for CTAs with an empty range) and their prefix, by warp 0
  if (tid < 32) {
    int run = 0;
    for (int base = 0; base < nslots; base += 32) {
      const int j = base + tid;
      int cnt = 0;
      if (j < nslots) {
        const int64_t c = c0 + j;
        if (cta_begin(c, total, P.grid) != cta_begin(c + 1, total, P.grid)) {
          cnt = *reinterpret_cast<const int32_t*>(slot_ptr(j));
          cnt = cnt < 0 ? 0 : (cnt > cap ? cap : cnt);  // a slot never holds more than it has room for
        }
      }
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (tid >= o) incl += v;
      }
      if (j < nslots) S.offs[j] = run + incl - cnt;
      run += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (tid == 0) S.offs[nslots] = run;
  }
  __syncthreads();
  // Gather whole slots while they fit, one warp per slot with four loads in
  // flight per lane; when the next slot would not fit, cut the buffer to at
  // most `window` keys (never below k) and go on. After a cut any slot fits:
  // window + a slot's room <= CSA_MAX_K + kSlotKeysMax <= kMergeCap.
  const int warp = tid >> 5, lane = tid & 31;
  int n = 0;
  for (int j0 = 0; j0 < nslots;) {
    int j1 = j0;
    while (j1 < nslots && n + (S.offs[j1 + 1] - S.offs[j0]) <= kMergeCap) ++j1;
    const int base = n - S.offs[j0];
    for (int j = j0 + warp; j < j1; j += kMergeThreads / 32) {
      const int o = S.offs[j], cnt = S.offs[j + 1] - o;
      const uint64_t* ent = reinterpret_cast<const uint64_t*>(slot_ptr(j) + 16);
      uint64_t* dst = S.cand + base + o;
      for (int i = lane; i < cnt; i += 128) {
        uint64_t v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = (i + 32 * u < cnt) ? ent[i + 32 * u] : 0ull;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (i + 32 * u < cnt) dst[i + 32 * u] = v[u];
      }
    }
    n += S.offs[j1] - S.offs[j0];
    j0 = j1;
    if (tid == 0) S.sel.n = static_cast<uint32_t>(n);
    __syncthreads();
    if (j0 < nslots) {
      shrink_if_above_reg<kMergeThreads, kMergeCap / kMergeThreads>(S.cand, S.scratch, window, P.k, window, &S.sel,
                                                                    0, tid);
      n = static_cast<int>(S.sel.n);
    }
  }
  shrink_if_above_reg<kMergeThreads, kMergeCap / kMergeThreads>(S.cand, S.scratch, window, P.k, window, &S.sel, 0,
                                                                tid);
  n = static_cast<int>(S.sel.n);
  merge_sort_desc(S, n, tid);
  for (int j = tid; j < P.k; j += kMergeThreads) {
    const int64_t o = static_cast<int64_t>(b) * P.k + j;
    if (j < n) {
      const uint64_t key = S.cand[j];
      const float v = key_value(key);
      idx[o] = key_position(key);
      vals[o] = kFromLogit ? 1.0f / (1.0f + expf(-v)) : v;
    } else {
      idx[o] = -1;
      vals[o] = 0.0f;
    }
  }
}

// ------------------------------------------------------------------ merge of top-k lists

// Context-parallel scoring splits one request's pages across G GPUs; each
// returns its rows' local top-k (position, value). The global top-k of a row is
// contained in the union of the local ones (every record of the global top-k
// ranks at least as high in its own shard), so merging the G lists is exact.
struct MergeListArgs {
  const int32_t* idx;  // [G, num_q, k_in]
  const float* vals;   // [G, num_q, k_in]
  int32_t* out_idx;    // [num_q, k]
  float* out_vals;     // [num_q, k]
  int32_t num_lists, num_q, k_in, k;
};

// One CTA per row: the lists' valid entries (position >= 0, value not NaN)
// become keys (value desc, position asc) appended to the candidate buffer; the
// buffer is cut back to between k and merge_window(k) keys whenever the next
// list might not fit, then sorted, and the first k written with their values
// unchanged, padded with -1 / 0.
__global__ void __launch_bounds__(kMergeThreads) merge_lists_kernel(const MergeListArgs A) {
  extern __shared__ uint8_t smem_raw[];
  MergeSmem& S = *reinterpret_cast<MergeSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~uintptr_t(15));
  const int tid = threadIdx.x;
  const int32_t b = blockIdx.x;
  const int window = merge_window(A.k);
  if (tid == 0) {
    S.sel.n = 0;
    S.sel.tau = 0;
  }
  __syncthreads();
  for (int g = 0; g < A.num_lists; ++g) {
    if (static_cast<int>(S.sel.n) + A.k_in > kMergeCap)  // uniform: read after a barrier
      shrink_if_above_reg<kMergeThreads, kMergeCap / kMergeThreads>(S.cand, S.scratch, kMergeCap - A.k_in, A.k,
                                                                    window, &S.sel, 0, tid);
    const int64_t base = (static_cast<int64_t>(g) * A.num_q + b) * A.k_in;
    for (int j0 = 0; j0 < A.k_in; j0 += kMergeThreads) {  // whole warps in every round
      const int j = j0 + tid;
      int32_t pos = -1;
      float v = 0.0f;
      if (j < A.k_in) {
        pos = A.idx[base + j];
        v = A.vals[base + j];
      }
      const bool take = pos >= 0 && !isnan(v);
      append_key(S.cand, take ? make_key(v, pos) : 0ull, take, &S.sel);
    }
    __syncthreads();
  }
  shrink_if_above_reg<kMergeThreads, kMergeCap / kMergeThreads>(S.cand, S.scratch, window, A.k, window, &S.sel, 0,
                                                                tid);
  const int n = static_cast<int>(S.sel.n);
  merge_sort_desc(S, n, tid);
  for (int j = tid; j < A.k; j += kMergeThreads) {
    const int64_t o = static_cast<int64_t>(b) * A.k + j;
    if (j < n) {
      const uint64_t key = S.cand[j];
      A.out_idx[o] = key_position(key);
      A.out_vals[o] = key_value(key);
    } else {
      A.out_idx[o] = -1;
      A.out_vals[o] = 0.0f;
    }
  }
}

// ------------------------------------------------------------------ unfused top-k

constexpr int kTopkThreads = 128;
constexpr int kTopkBatch = 4;
constexpr int kTopkCtasPerSm = 4;

struct TopkSmem {
  uint64_t cand[kCap];
  uint64_t scratch[CSA_MAX_K];
  SelectShared sel;
  Plan plan;
  int64_t warp_sums[32];
};

// Phase 1 of top-k over a score matrix: same tiles, CTA ranges and slots as the
// fused kernel; each thread owns one column of a 128-column tile.
__global__ void __launch_bounds__(kTopkThreads) topk_scores_kernel(const Params P) {
  extern __shared__ uint8_t smem_raw[];
  TopkSmem& S = *reinterpret_cast<TopkSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~uintptr_t(15));
  const int tid = threadIdx.x;
  if (tid == 0) {
    S.plan.flags = 0;
    S.sel.n = 0;
    S.sel.tau = 0;
  }
  __syncthreads();
  make_plan<kTopkThreads>(P, &S.plan, S.warp_sums, reinterpret_cast<int32_t*>(P.ws));
  if (tid == 0 && blockIdx.x == 0 && S.plan.flags && P.dev_status) atomicOr(P.dev_status, S.plan.flags);
  if (S.plan.ntiles == 0) return;
  int32_t flags = 0;
  Cursor cur;
  cur.init(P, S.plan);
  for (int64_t i0 = 0; i0 < S.plan.ntiles; i0 += kTopkBatch) {
    const int nb = static_cast<int>(S.plan.ntiles - i0 < kTopkBatch ? S.plan.ntiles - i0 : kTopkBatch);
    // this thread's columns of the next nb tiles: tid and tid + 128 of each
    float val[kTopkBatch][2];
    int32_t pos[kTopkBatch][2];
    bool ok[kTopkBatch][2];
    Cursor c = cur;
#pragma unroll
    for (int u = 0; u < kTopkBatch; ++u) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        ok[u][h] = false;
        pos[u][h] = 0;
        val[u][h] = 0.f;
      }
      if (u < nb) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int colt = 128 * h + tid;  // column inside the tile
          const PageInfo e = page_of(P, c.b, c.lt, colt >> 6, &flags);
          const int r = colt & 63;
          if (r < e.nrows) {
            ok[u][h] = true;
            pos[u][h] = e.lp * kPage + r;
            val[u][h] = P.in_scores[static_cast<int64_t>(c.b) * P.score_stride + c.lt * kTile + colt];
          }
        }
        c.advance(P);
      }
    }
    for (int u = 0; u < nb; ++u) {
      const uint64_t tau = S.sel.tau;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint64_t key = (ok[u][h] && !isnan(val[u][h])) ? make_key(val[u][h], pos[u][h]) : 0ull;
        append_key(S.cand, key, key != 0ull && key > tau, &S.sel);
      }
      __syncthreads();
      shrink_if_above<kTopkThreads, kTopkThreads>(S.cand, S.scratch, kCap - kTile, P.k, loose_keep(P.k), &S.sel, 0,
                                                  tid);
      const bool seg_end = (i0 + u == S.plan.ntiles - 1) || (cur.lt == cur.tiles - 1);
      if (seg_end) {
        shrink_if_above<kTopkThreads, kTopkThreads>(S.cand, S.scratch, loose_keep(P.k), P.k, loose_keep(P.k), &S.sel,
                                                    0, tid);
        const int n = static_cast<int>(S.sel.n);
        uint8_t* slot = P.ws + P.slots_offset + (static_cast<int64_t>(cur.b) + blockIdx.x) * P.slot_bytes;
        uint64_t* ent = reinterpret_cast<uint64_t*>(slot + 16);
        for (int j = tid; j < n; j += kTopkThreads) ent[j] = S.cand[j];
        __syncthreads();
        if (tid == 0) {
          *reinterpret_cast<int32_t*>(slot) = n;
          S.sel.n = 0;
          S.sel.tau = 0;
        }
        __syncthreads();
      }
      cur.advance(P);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) flags |= __shfl_xor_sync(0xFFFFFFFFu, flags, o);
  if ((tid & 31) == 0 && flags && P.dev_status) atomicOr(P.dev_status, flags);
}

}  // namespace csa

// ====================================================================== C ABI

namespace {

using namespace csa;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices];
bool g_ready[kMaxDevices];

// A slot: a 16-byte header (the key count) and room for the keys. Segments are
// cut to at most loose_keep(k) keys before they are written, except in the
// short-row scorer (kShortRowsMin rows and more, on a caller's workspace),
// whose slots take a whole uncut row of up to kSlotKeysMax keys.
size_t slot_bytes_for(int32_t k) { return (16 + 8 * static_cast<size_t>(loose_keep(k)) + 15) & ~size_t(15); }
size_t slot_bytes_fused(int32_t num_q, int32_t k) {
  return num_q >= kShortRowsMin ? (16 + 8 * static_cast<size_t>(kSlotKeysMax) + 15) & ~size_t(15) : slot_bytes_for(k);
}
// tile_off[num_q + 2] (virtual prefix sums and the charge per row), then the slots
size_t slots_offset_for(int32_t num_q) { return (4 * (static_cast<size_t>(num_q) + 2) + 255) & ~size_t(255); }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

enum { kNeedQ = 1, kNeedKv = 2, kAllowWide = 4 };  // kAllowWide: 128 heads accepted as well as 64

csa_status check_args(const csa_index_args* a, int need) {
  if (!a) return CSA_ERR_INVALID_ARG;
  if (a->reserved0 != 0) return CSA_ERR_INVALID_ARG;
  if (a->record_format != CSA_RECORD_E4M3 && a->record_format != CSA_RECORD_MXFP4) return CSA_ERR_INVALID_ARG;
  if (a->num_q < 0 || a->num_req < 0 || a->pt_stride < 0 || a->res_stride < 0) return CSA_ERR_INVALID_ARG;
  if (a->num_q == 0) return CSA_OK;
  if (!a->q_len) return CSA_ERR_INVALID_ARG;
  if (!aligned(a->q_len, 4) || (a->q_req && !aligned(a->q_req, 4))) return CSA_ERR_ALIGNMENT;
  if (!a->q_req && a->num_req < a->num_q) return CSA_ERR_INVALID_ARG;
  if (a->resident) {
    if (!a->n_resident || a->res_stride < 1) return CSA_ERR_INVALID_ARG;
    if (!aligned(a->resident, 4) || !aligned(a->n_resident, 4)) return CSA_ERR_ALIGNMENT;
  }
  if (a->dev_status && !aligned(a->dev_status, 4)) return CSA_ERR_ALIGNMENT;
  if (need & kNeedQ) {
    if (a->head_dim != kD || !(a->num_heads == kH || ((need & kAllowWide) && a->num_heads == 2 * kH)))
      return CSA_ERR_UNSUPPORTED;
    if (a->record_format == CSA_RECORD_MXFP4 && a->num_heads != kH) return CSA_ERR_UNSUPPORTED;
    if (!a->q || !a->fused_w) return CSA_ERR_INVALID_ARG;
    if (!aligned(a->q, 16) || !aligned(a->fused_w, 4)) return CSA_ERR_ALIGNMENT;
  }
  if (need & kNeedKv) {
    if (!a->kv || !a->page_table || a->num_pages < 1 || a->pt_stride < 1 || a->num_req < 1)
      return CSA_ERR_INVALID_ARG;
    if (a->num_pages > INT32_MAX) return CSA_ERR_INVALID_ARG;
    if (a->page_stride_bytes < (a->record_format == CSA_RECORD_MXFP4 ? kFp4PageBytes : kPageBytes))
      return CSA_ERR_INVALID_ARG;
    if (a->page_stride_bytes % 16 != 0 || !aligned(a->kv, 16)) return CSA_ERR_ALIGNMENT;
    if (!aligned(a->page_table, 4)) return CSA_ERR_ALIGNMENT;
  } else if (a->page_table && !aligned(a->page_table, 4)) {
    return CSA_ERR_ALIGNMENT;
  }
  if (static_cast<int64_t>(kPage) * a->pt_stride > INT32_MAX) return CSA_ERR_INVALID_ARG;
  return CSA_OK;
}

csa_status device_setup(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ready[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return CSA_ERR_CUDA;
    if (n * kTopkCtasPerSm > CSA_MAX_CTAS) return CSA_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(w64::score_kernel_w64<false, CSA_RECORD_E4M3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(w64::kSmemBytes)) != cudaSuccess ||
        cudaFuncSetAttribute(w64::score_kernel_w64<true, CSA_RECORD_E4M3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(w64::kSmemBytes)) != cudaSuccess ||
        cudaFuncSetAttribute(w64::score_kernel_w64<true, CSA_RECORD_E4M3, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(w64::kSmemBytes)) != cudaSuccess ||
        cudaFuncSetAttribute(w64::score_kernel_w64<false, CSA_RECORD_MXFP4>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(w64::kSmemBytes)) != cudaSuccess ||
        cudaFuncSetAttribute(w64::score_kernel_w64<true, CSA_RECORD_MXFP4>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(w64::kSmemBytes)) != cudaSuccess ||
        cudaFuncSetAttribute(score_kernel<false, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes<128>)) != cudaSuccess ||
        cudaFuncSetAttribute(merge_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(MergeSmem) + 16)) != cudaSuccess ||
        cudaFuncSetAttribute(merge_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(MergeSmem) + 16)) != cudaSuccess ||
        cudaFuncSetAttribute(merge_lists_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(MergeSmem) + 16)) != cudaSuccess ||
        cudaFuncSetAttribute(topk_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(TopkSmem) + 16)) != cudaSuccess)
      return CSA_ERR_CUDA;
    g_sms[dev] = n;
    g_ready[dev] = true;
  }
  *sms = g_sms[dev];
  return CSA_OK;
}

Params params_of(const csa_index_args* a) {
  Params P;
  std::memset(&P, 0, sizeof(P));
  P.q = static_cast<const uint16_t*>(a->q);
  P.w = a->fused_w;
  P.kv = a->kv;
  P.num_pages = a->num_pages;
  P.page_stride = a->page_stride_bytes;
  P.page_table = a->page_table;
  P.q_req = a->q_req;
  P.q_len = a->q_len;
  P.resident = a->resident;
  P.n_resident = a->n_resident;
  P.dev_status = a->dev_status;
  P.num_q = a->num_q;
  P.num_req = a->num_req;
  P.pt_stride = a->pt_stride;
  P.res_stride = a->res_stride;
  P.fmt = a->record_format;
  return P;
}

int64_t min_score_stride(const csa_index_args* a) {
  return static_cast<int64_t>(kPage) * (a->resident ? a->res_stride : a->pt_stride);
}

csa_status launch_status() { return cudaGetLastError() == cudaSuccess ? CSA_OK : CSA_ERR_CUDA; }

}  // namespace

// The 64-head scorer in score / logit mode or top-k mode.
csa_status launch_w64(const Params& P, bool topk, int sms, cudaStream_t s) {
  const bool fp4 = P.fmt == CSA_RECORD_MXFP4;
  if (topk && fp4)
    w64::score_kernel_w64<true, CSA_RECORD_MXFP4><<<sms, w64::kThreads, w64::kSmemBytes, s>>>(P);
  else if (topk && P.num_q >= kShortRowsMin)  // many rows: the short-row scorer
    w64::score_kernel_w64<true, CSA_RECORD_E4M3, true><<<sms, w64::kThreads, w64::kSmemBytes, s>>>(P);
  else if (topk)
    w64::score_kernel_w64<true, CSA_RECORD_E4M3><<<sms, w64::kThreads, w64::kSmemBytes, s>>>(P);
  else if (fp4)
    w64::score_kernel_w64<false, CSA_RECORD_MXFP4><<<sms, w64::kThreads, w64::kSmemBytes, s>>>(P);
  else
    w64::score_kernel_w64<false, CSA_RECORD_E4M3><<<sms, w64::kThreads, w64::kSmemBytes, s>>>(P);
  return launch_status();
}

// Score or logit mode (P.raw_logits) of the scoring kernel for 64 or 128 heads.
csa_status launch_score(const csa_index_args* a, const Params& P, int sms, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a->num_heads == 2 * kH) {
    score_kernel<false, 128><<<sms, kThreads, kSmemBytes<128>, s>>>(P);
    return launch_status();
  }
  return launch_w64(P, false, sms, s);
}

extern "C" {

int32_t csa_index_abi_version(void) { return CSA_ABI_VERSION; }

const char* csa_status_str(csa_status s) {
  switch (s) {
    case CSA_OK: return "ok";
    case CSA_ERR_INVALID_ARG: return "invalid argument";
    case CSA_ERR_UNSUPPORTED: return "unsupported shape or device";
    case CSA_ERR_ALIGNMENT: return "misaligned pointer or stride";
    case CSA_ERR_WORKSPACE: return "workspace missing or too small";
    case CSA_ERR_CUDA: return "CUDA runtime error";
  }
  return "unknown status";
}

size_t csa_index_workspace_bytes(const csa_index_args* args, int32_t k) {
  if (!args || args->num_q < 0 || k < 1 || k > CSA_MAX_K) return 0;
  return slots_offset_for(args->num_q) +
         (static_cast<size_t>(args->num_q) + CSA_MAX_CTAS) * slot_bytes_fused(args->num_q, k);
}

csa_status csa_index_score(const csa_index_args* args, float* scores, int64_t score_stride, void* stream) {
  csa_status st = check_args(args, kNeedQ | kNeedKv | kAllowWide);
  if (st != CSA_OK) return st;
  if (args->num_q == 0) return CSA_OK;
  if (!scores) return CSA_ERR_INVALID_ARG;
  if (!aligned(scores, 4)) return CSA_ERR_ALIGNMENT;
  if (score_stride < min_score_stride(args)) return CSA_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = device_setup(&sms)) != CSA_OK) return st;
  Params P = params_of(args);
  P.scores = scores;
  P.score_stride = score_stride;
  P.grid = sms;
  return launch_score(args, P, sms, stream);
}

csa_status csa_index_logits(const csa_index_args* args, float* logits, int64_t stride, void* stream) {
  csa_status st = check_args(args, kNeedQ | kNeedKv | kAllowWide);
  if (st != CSA_OK) return st;
  if (args->num_q == 0) return CSA_OK;
  if (!logits) return CSA_ERR_INVALID_ARG;
  if (!aligned(logits, 4)) return CSA_ERR_ALIGNMENT;
  if (stride < min_score_stride(args)) return CSA_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = device_setup(&sms)) != CSA_OK) return st;
  Params P = params_of(args);
  P.scores = logits;
  P.score_stride = stride;
  P.grid = sms;
  P.raw_logits = 1;
  return launch_score(args, P, sms, stream);
}

}  // extern "C"

csa_status csa_score_fold(const csa_index_args* args, float* acc, int64_t stride, int fold, void* stream) {
  csa_status st = check_args(args, kNeedQ | kNeedKv | kAllowWide);
  if (st != CSA_OK) return st;
  if (args->num_q == 0) return CSA_OK;
  if (!acc || args->resident || (fold != CSA_FOLD_MAX && fold != CSA_FOLD_ADD)) return CSA_ERR_INVALID_ARG;
  if (args->num_heads != 2 * kH) return CSA_ERR_UNSUPPORTED;  // the fold mode is the 128-head scorer's
  if (!aligned(acc, 4)) return CSA_ERR_ALIGNMENT;
  if (stride < min_score_stride(args)) return CSA_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = device_setup(&sms)) != CSA_OK) return st;
  Params P = params_of(args);
  P.scores = acc;
  P.score_stride = stride;
  P.grid = sms;
  P.fold = fold;
  return launch_score(args, P, sms, stream);
}

// Launches the merge right behind the kernel that filled the slots on stream s.
// When nothing else sits between the two on the stream (pdl), it is a
// programmatic dependent launch: its CTAs are placed on SMs as the scoring CTAs
// leave them and wait inside the kernel for the scoring grid to complete, so
// the launch latency is off the critical path.
template <bool kFromLogit>
csa_status launch_merge(const Params& P, int32_t num_q, int32_t* idx, float* vals, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_q));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = sizeof(MergeSmem) + 16;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, merge_kernel<kFromLogit>, P, idx, vals) != cudaSuccess) return CSA_ERR_CUDA;
  return launch_status();
}

extern "C" {

csa_status csa_index_score_topk_fused(const csa_index_args* args, int32_t k, int32_t* idx, float* vals, void* ws,
                                      size_t ws_bytes, void* stream) {
  return csa_index_score_topk_fused_marked(args, k, idx, vals, ws, ws_bytes, stream, nullptr);
}

csa_status csa_index_score_topk_fused_marked(const csa_index_args* args, int32_t k, int32_t* idx, float* vals,
                                             void* ws, size_t ws_bytes, void* stream, void* event) {
  csa_status st = check_args(args, kNeedQ | kNeedKv);
  if (st != CSA_OK) return st;
  if (k < 1 || k > CSA_MAX_K) return CSA_ERR_INVALID_ARG;
  if (args->num_q == 0) return CSA_OK;
  if (!idx || !vals) return CSA_ERR_INVALID_ARG;
  if (!aligned(idx, 4) || !aligned(vals, 4)) return CSA_ERR_ALIGNMENT;
  if (!ws || ws_bytes < csa_index_workspace_bytes(args, k)) return CSA_ERR_WORKSPACE;
  if (!aligned(ws, 16)) return CSA_ERR_ALIGNMENT;
  int sms = 0;
  if ((st = device_setup(&sms)) != CSA_OK) return st;
  Params P = params_of(args);
  P.ws = static_cast<uint8_t*>(ws);
  P.k = k;
  P.slot_bytes = static_cast<int64_t>(slot_bytes_fused(args->num_q, k));
  P.slots_offset = static_cast<int64_t>(slots_offset_for(args->num_q));
  P.grid = sms;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = launch_w64(P, true, sms, s)) != CSA_OK) return st;
  if (event && cudaEventRecord(static_cast<cudaEvent_t>(event), s) != cudaSuccess) return CSA_ERR_CUDA;
  return launch_merge<true>(P, args->num_q, idx, vals, s, event == nullptr);
}

csa_status csa_index_merge_topk(const int32_t* idx, const float* vals, int32_t num_lists, int32_t num_q,
                                int32_t k_in, int32_t k, int32_t* out_idx, float* out_vals, void* stream) {
  if (num_lists < 1 || num_q < 0 || k_in < 1 || k_in > CSA_MAX_K || k < 1 || k > CSA_MAX_K)
    return CSA_ERR_INVALID_ARG;
  if (num_q == 0) return CSA_OK;
  if (!idx || !vals || !out_idx || !out_vals) return CSA_ERR_INVALID_ARG;
  if (!aligned(idx, 4) || !aligned(vals, 4) || !aligned(out_idx, 4) || !aligned(out_vals, 4))
    return CSA_ERR_ALIGNMENT;
  int sms = 0;
  csa_status st = device_setup(&sms);
  if (st != CSA_OK) return st;
  MergeListArgs A{idx, vals, out_idx, out_vals, num_lists, num_q, k_in, k};
  merge_lists_kernel<<<num_q, kMergeThreads, sizeof(MergeSmem) + 16, static_cast<cudaStream_t>(stream)>>>(A);
  return launch_status();
}

csa_status csa_index_topk(const float* scores, int64_t score_stride, const csa_index_args* args, int32_t k,
                          int32_t* idx, float* vals, void* ws, size_t ws_bytes, void* stream) {
  csa_status st = check_args(args, 0);
  if (st != CSA_OK) return st;
  if (k < 1 || k > CSA_MAX_K) return CSA_ERR_INVALID_ARG;
  if (args->num_q == 0) return CSA_OK;
  if (args->pt_stride < 1 || args->num_req < 1) return CSA_ERR_INVALID_ARG;
  if (!scores || !idx || !vals) return CSA_ERR_INVALID_ARG;
  if (!aligned(scores, 4) || !aligned(idx, 4) || !aligned(vals, 4)) return CSA_ERR_ALIGNMENT;
  if (score_stride < min_score_stride(args)) return CSA_ERR_INVALID_ARG;
  if (!ws || ws_bytes < csa_index_workspace_bytes(args, k)) return CSA_ERR_WORKSPACE;
  if (!aligned(ws, 16)) return CSA_ERR_ALIGNMENT;
  int sms = 0;
  if ((st = device_setup(&sms)) != CSA_OK) return st;
  Params P = params_of(args);
  P.num_pages = args->page_table ? args->num_pages : 0;
  P.in_scores = scores;
  P.score_stride = score_stride;
  P.ws = static_cast<uint8_t*>(ws);
  P.k = k;
  P.slot_bytes = static_cast<int64_t>(slot_bytes_for(k));
  P.slots_offset = static_cast<int64_t>(slots_offset_for(args->num_q));
  P.grid = sms * kTopkCtasPerSm;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  topk_scores_kernel<<<P.grid, kTopkThreads, sizeof(TopkSmem) + 16, s>>>(P);
  if ((st = launch_status()) != CSA_OK) return st;
  return launch_merge<false>(P, args->num_q, idx, vals, s, true);
}

}  // extern "C"

// ====================================================================== built-in scratch

// Scratch of csa_index_score_topk_fused_static: the row tile offsets and the
// per-segment candidate slots that csa_index_score_topk_fused otherwise keeps in
// the caller's workspace. Every GPU that loads the library holds this array
// until the process exits; all calls on a device share it.
static __device__ __align__(256) uint8_t csa_static_scratch[CSA_STATIC_SCRATCH_BYTES];

namespace {

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];

// Device address of csa_static_scratch on the current device, looked up once per
// device (host code may not use the symbol itself: it names a host-side shadow).
csa_status static_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, csa_static_scratch) != cudaSuccess || !p) return CSA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return CSA_OK;
}

}  // namespace

extern "C" csa_status csa_index_score_topk_fused_static(const csa_index_args* args, int32_t k, int32_t* idx,
                                                        float* vals, void* stream) {
  csa_status st = check_args(args, kNeedQ | kNeedKv);
  if (st != CSA_OK) return st;
  if (k < 1 || k > CSA_MAX_K) return CSA_ERR_INVALID_ARG;
  if (args->num_q == 0) return CSA_OK;
  if (!idx || !vals) return CSA_ERR_INVALID_ARG;
  if (!aligned(idx, 4) || !aligned(vals, 4)) return CSA_ERR_ALIGNMENT;
  int sms = 0;
  if ((st = device_setup(&sms)) != CSA_OK) return st;
  // The scoring kernel writes slot (row + CTA) for CTA < grid = SM count.
  const size_t need =
      slots_offset_for(args->num_q) + (static_cast<size_t>(args->num_q) + sms) * slot_bytes_for(k);
  if (need > CSA_STATIC_SCRATCH_BYTES) return CSA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((st = static_scratch_address(&scratch)) != CSA_OK) return st;
  Params P = params_of(args);
  P.ws = static_cast<uint8_t*>(scratch);
  P.k = k;
  P.slot_bytes = static_cast<int64_t>(slot_bytes_for(k));
  P.slots_offset = static_cast<int64_t>(slots_offset_for(args->num_q));
  P.grid = sms;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = launch_w64(P, true, sms, s)) != CSA_OK) return st;
  return launch_merge<true>(P, args->num_q, idx, vals, s, true);
}
