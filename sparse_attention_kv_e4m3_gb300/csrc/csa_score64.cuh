// csa_score64.cuh — the 64-head scoring kernel (the indexer's hot path).
//
// Included by csa_index.cu after the shared definitions (Params, PageInfo, the
// plan, the page walker, the query preparation, the selection helpers).
//
// Data path. Whole 8448-byte pages are streamed into a ring of shared-memory
// slots with 1-D bulk copies (one copy-engine instruction per page: measured on
// this GPU, tiled tensor copies of the page's rows cost about 140 cycles per
// box and 7.6 per 128-byte row, which caps them below the HBM rate). A record
// is 132 bytes, so record rows are not 16-byte aligned; four records are
// (528 = 33 x 16). The records of a page are therefore taken in "classes":
// class r (r = 0..3) is record r of each of the page's 16 four-record groups,
// and record r of group g starts 4r bytes past the 16-byte-aligned offset
// 528g + 128r. A worker thread loads the nine aligned 16-byte chunks from there
// (conflict-free across a warp) and passes words r .. r + 31 — exactly the
// record's 128 key bytes — to its TMEM lane; word r + 32 is the record's
// fp32 scale. Every lane of a warp works on the same class, so the word
// selection is a warp-uniform choice between four register assignments.
//
// A class sub-tile is record r of the 128 groups of one tile (8 pages = 512
// records): TMEM lane m holds group m % 16 of page m / 16. It is scored by
// M=128, N=64, K=32 e4m3 MMAs with the key bytes in TMEM (A) and the query in
// shared memory (B, K-major, one buffer per term): the query's e4m3 hi term
// over K = 0..127 (four MMAs), then its lo term into the same accumulator (four
// more), so each head's column holds k . (q * 2^e_h) itself. A half-tile is two
// class sub-tiles (classes 2g and 2g + 1 of a tile) and belongs to worker group
// g; a worker lane then carries two records per iteration, which amortises the
// iteration's fixed barrier and hand-off latencies. Two threads in two warps
// issue the MMAs, one class sub-tile of each half-tile each (8 MMAs back to
// back from precomputed operands), and both commit to the half-tile's
// accumulator-ready barrier: measured here, one thread issues at most one
// tcgen05.mma every ~50 cycles in a tight loop (~80 beside the busy warps of
// its scheduler), two issuing warps reach the tensor pipe's ~32 cycles per N=64
// MMA, and a loop that rebuilds descriptors and branches per MMA takes ~95-106.
//
// Warp roles (512 threads):
//   0      issuer: 8 lanes in lockstep, one 1-D bulk copy per page into a ring of
//          kPages slots
//   1      MMA issue for class sub-tiles 0 and 2 (one thread); allocates the
//          512 TMEM columns
//   2      page walker (shared with the other scorer)
//   3      MMA issue for class sub-tiles 1 and 3 (one thread)
//   4-11   workers, two groups of four (one warp per TMEM lane quarter): group
//          g owns classes 2g and 2g + 1 of every tile. For each tile: wait for
//          the MMAs of its half-tile, stage the next tile's half-tile into the
//          group's TMEM A stage (its MMAs then overlap), then the epilogue of
//          both records.
//   12-15  selector (top-k mode): one tile of keys (all four classes) per step;
//          also splits the queries of the CTA's later segments (the first is
//          split by the whole CTA in the prologue; two query slots), 16 heads
//          per warp: segment s + 2's into the slot of segment s once it has
//          taken s's last keys, by which time the MMAs and the epilogues of s
//          are done. In score mode warp 12 prepares them instead, each as soon
//          as the MMAs and the workers release its slot.
//
// TMEM: one 64-column A stage per worker group (columns 0 and 64: two class
// sub-tiles of 32 columns) and three 128-column accumulator stages (columns
// 128, 256, 384: two class sub-tiles of 64 columns).
#pragma once

namespace csa {
namespace w64 {

constexpr int kH = 64;
constexpr int kTP = 8;                               // pages per tile
constexpr int kTileRecs = kTP * kPage;               // 512
constexpr int kGroupBytes = 4 * kRec;                // 528
constexpr int kGroupsPerPage = kPage / 4;            // 16
constexpr int kRows = kTP * kGroupsPerPage;          // 128 rows per class sub-tile (MMA M)
constexpr int kPages = 17;                           // page ring slots
constexpr int kDStages = 3;                          // accumulator stages
constexpr int kKeyRing = 4;                          // tiles of keys, workers -> selector
constexpr int kCapW = 2048;                          // candidate buffer of one segment
constexpr int kThreads = 512;
constexpr int kWarpIssuer = 0, kWarpMma = 1, kWarpWalker = 2, kWarpMma2 = 3, kWarpWorker = 4, kWarpSelect = 12;
constexpr int kWorkerWarps = 8;
constexpr int kBarSelect = 1;
constexpr int kQEmptyCount = 2 + kWorkerWarps;       // both MMA threads' commits + every worker warp
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdesc = idesc_e4m3_f32(128, kH);

__host__ __device__ constexpr uint32_t a_col(int g) { return 64u * static_cast<uint32_t>(g); }
__host__ __device__ constexpr uint32_t d_col(int s) { return 128u + 128u * static_cast<uint32_t>(s); }

static_assert(kGroupBytes % 16 == 0 && kPageBytes % 16 == 0, "group offsets and pages are 16-byte aligned");
static_assert(kH == 64, "one N = 64 B operand per query term");
static_assert(kCapW >= CSA_MAX_K + kTileRecs, "a cut leaves room for one more tile of keys");
static_assert(kCapW <= kSlotKeysMax, "a workspace slot for short rows has room for the whole buffer");
static_assert(a_col(2) <= d_col(0) && d_col(kDStages) <= kTmemCols, "TMEM column map");
static_assert(32 % kTP == 0 && kTP == 8, "a walker ring slot holds four tiles; the issuer uses 8 lanes");
static_assert(kThreads == 64 * (kD / 16), "the prologue splits the first query with one thread per 16 elements");

struct __align__(1024) Smem {
  uint8_t qbuf[2][2][kH * kD];                // [slot][hi/lo] e4m3, K-major, 128-byte swizzle: N=64 operands
  uint8_t pages[kPages][kPageBytes];
  uint64_t cand[kCapW];
  uint64_t scratch[CSA_MAX_K];
  uint64_t keys[kKeyRing][kTileRecs];         // a tile's admissible keys: 32 per (class, worker warp)
  alignas(16) uint32_t kcnt[kKeyRing][16];    // keys in region 4 * class + lane quarter
  PageInfo ring[kRing * 32];
  PageInfo info[kPages];
  int64_t last_pg[kPages];                    // most recent page copied into each ring slot (-1: none)
  alignas(16) float wbuf[2][kH];              // head weights x 2^-e_h, by query slot
  uint64_t full[kPages], empty[kPages];
  uint64_t afull[2];
  uint64_t dfull[kDStages], dempty[kDStages];
  uint64_t kfull[kKeyRing], kempty[kKeyRing];
  uint64_t rfull[kRing], rempty[kRing];
  uint64_t qfull[2], qempty[2];
  uint64_t drain;
  uint64_t filt;                              // (segment << 32) | value word of the selector's threshold
  SelectShared sel;
  Plan plan;
  int64_t warp_sums[32];
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t status;
  int32_t go[2];
};

constexpr bool smem_layout_ok() {
  return offsetof(Smem, qbuf) % 1024 == 0 && offsetof(Smem, pages) % 16 == 0 && offsetof(Smem, wbuf) % 16 == 0 &&
         offsetof(Smem, full) % 8 == 0 && offsetof(Smem, filt) % 8 == 0;
}
static_assert(smem_layout_ok(), "swizzle atoms 1024-byte aligned, copies 16-byte, mbarriers 8-byte aligned");
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ Smem& smem_of(uint8_t* raw) {
  return *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ uint32_t filter_word(const Smem& S, int seg) {
  const uint64_t f = *reinterpret_cast<const volatile uint64_t*>(&S.filt);
  return static_cast<uint32_t>(f >> 32) == static_cast<uint32_t>(seg) ? static_cast<uint32_t>(f) : 0u;
}

// The row after b that has tiles, and its tile count: the cursors' step at a
// segment end, kept out of line so that the roles' loops stay small (the
// parameters live in the kernel's parameter space: no copy is made).
struct RowTiles {
  int32_t b;
  int64_t tiles;
};
__device__ __noinline__ RowTiles next_row_tiles(const Params& P, int32_t b) {
  b = next_nonempty<kTP>(P, b + 1);
  return {b, b < P.num_q ? query_tiles<kTP>(P, b) : 0};
}

// A role's position: row b, tile lt of its `tiles` (the segment plan's order).
struct Cursor64 {
  int32_t b;
  int64_t lt;
  int64_t tiles;
  __device__ __forceinline__ void init(const Params& P, const Plan& pl) {
    b = pl.b0;
    lt = pl.lt0;
    tiles = b < P.num_q ? query_tiles<kTP>(P, b) : 0;
  }
  static __device__ __forceinline__ void next_row(const Params& P, int32_t& b, int64_t& tiles) {
    const RowTiles r = next_row_tiles(P, b);
    b = r.b;
    tiles = r.tiles;
  }
  __device__ __forceinline__ void advance(const Params& P) {
    if (++lt >= tiles) {
      next_row(P, b, tiles);
      lt = 0;
    }
  }
};

// ------------------------------------------------------------------ issuer

// Lanes 0..7 copy the 8 pages of each tile in lockstep, page j of tile t into
// ring slot (8t + j) % kPages.
template <int kFmt>
__device__ void role_issuer(const Params& P, Smem& S) {
  constexpr uint32_t kBytes = kFmt == CSA_RECORD_MXFP4 ? kFp4PageBytes : kPageBytes;  // a page's records
  const int lane = threadIdx.x & 31;
  const int64_t nt = S.plan.ntiles;
  const uint64_t policy = policy_evict_first();
  for (int s = lane; s < kPages; s += 32) S.last_pg[s] = -1;
  __syncwarp();
  for (int64_t t = 0; t < nt; ++t) {
    const int64_t batch = t >> 2;  // a walker ring slot holds 32 pages = 4 tiles
    const int rs = static_cast<int>(batch % kRing);
    const uint32_t rph = static_cast<uint32_t>((batch / kRing) & 1);
    if ((t & 3) == 0) {
      bool ok = true;
      if (lane == 0) ok = mbar_wait(smem_u32(&S.rfull[rs]), rph, &S.abort_flag);
      if (!warp_ok(ok)) break;
    }
    bool ok = true;
    if (lane < kTP) {
      mbar_wait_drain(smem_u32(&S.rfull[rs]), rph);  // complete: acquire the walker's entries
      const PageInfo e = S.ring[rs * 32 + static_cast<int>(t & 3) * kTP + lane];
      const int64_t pg = kTP * t + lane;
      const int s = static_cast<int>(pg % kPages);
      ok = mbar_wait(smem_u32(&S.empty[s]), static_cast<uint32_t>(((pg / kPages) & 1) ^ 1), &S.abort_flag);
      if (ok) {
        S.info[s] = e;
        const uint32_t fb = smem_u32(&S.full[s]);
        if (e.nrows > 0) {
          mbar_arrive_expect_tx(fb, kBytes);
          bulk_g2s_hint(smem_u32(S.pages[s]), P.kv + static_cast<int64_t>(e.phys) * P.page_stride, kBytes, fb,
                        policy);
        } else {
          mbar_arrive(fb);
        }
        S.last_pg[s] = pg;
      }
    }
    if (!__all_sync(0xFFFFFFFFu, ok)) break;
    if (lane == 0 && ((t & 3) == 3 || t == nt - 1)) mbar_arrive(smem_u32(&S.rempty[rs]));
  }
  // Every copy issued must land before the CTA may exit: the most recent one of
  // each ring slot (a slot's earlier pages were consumed before it was reused).
  __syncwarp();
  for (int s = lane; s < kPages; s += 32) {
    const int64_t p = S.last_pg[s];
    if (p >= 0) mbar_wait_drain(smem_u32(&S.full[s]), static_cast<uint32_t>((p / kPages) & 1));
  }
}

// ------------------------------------------------------------------ MMA

// One of the two issuing threads: class sub-tile c of every half-tile (classes
// c and 2 + c of each tile). Both commit to the half-tile's accumulator-ready
// barrier, to the query slot's release at a segment end and to the final drain.
template <int kFmt>
__device__ void role_mma(const Params& P, Smem& S, const int c) {
  constexpr int kTerms = kFmt == CSA_RECORD_MXFP4 ? 1 : 2;  // an MXFP4 query is one e4m3 term
  Cursor64 cur;
  cur.init(P, S.plan);
  const uint32_t tmem = S.tmem_base;
  int seg = 0;
  bool ok = true;
  uint64_t bdesc[2][4];  // B descriptors of the current query slot: [hi/lo][K step]
  for (int64_t t = 0; ok && t < S.plan.ntiles; ++t) {
    const bool seg_start = (t == 0) || (cur.lt == 0);
    if (seg_start && t > 0) ++seg;
    const int qs = seg & 1;
    if (seg_start) {
      if (!mbar_wait(smem_u32(&S.qfull[qs]), static_cast<uint32_t>((seg >> 1) & 1), &S.abort_flag)) break;
#pragma unroll
      for (int term = 0; term < 2; ++term)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) bdesc[term][kk] = sdesc_kmajor_sw128(smem_u32(S.qbuf[qs][term]) + 32 * kk);
    }
#pragma unroll 1
    for (int g = 0; g < 2; ++g) {  // the two half-tiles of tile t
      const uint32_t h = static_cast<uint32_t>(2 * t + g);  // half-tiles of a CTA stay far below 2^32
      const int ds = static_cast<int>(h % kDStages);
      ok = mbar_wait(smem_u32(&S.afull[g]), static_cast<uint32_t>(t & 1), &S.abort_flag) &&
           mbar_wait(smem_u32(&S.dempty[ds]), ((h / kDStages) & 1) ^ 1, &S.abort_flag);
      if (!ok) break;
      tc_fence_after();
      const uint32_t d = tmem + d_col(ds) + kH * c, a = tmem + a_col(g) + 32 * c;
#pragma unroll
      for (int term = 0; term < kTerms; ++term)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_e4m3_ts(d, a + 8 * kk, bdesc[term][kk], kIdesc, (term | kk) != 0);
      mma_commit(smem_u32(&S.dfull[ds]));
    }
    if (!ok) break;
    const bool seg_end = (t == S.plan.ntiles - 1) || (cur.lt == cur.tiles - 1);
    if (seg_end) mma_commit(smem_u32(&S.qempty[qs]));
    cur.advance(P);
  }
  mma_commit(smem_u32(&S.drain));
  mbar_wait_drain(smem_u32(&S.drain), 0);
}

// ------------------------------------------------------------------ workers

// Words R .. R + 31 of the 36 loaded (the record's key bytes) into v; word
// R + 32 (its scale) into sc.
template <int R>
__device__ __forceinline__ void pick_record(const uint32_t (&w)[36], uint32_t (&v)[32], uint32_t& sc) {
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = w[R + j];
  sc = w[R + 32];
}

// Loads the 36 words at src (9 aligned 16-byte chunks): a record of class R
// and its scale are words R .. R + 32.
__device__ __forceinline__ void load36(const uint8_t* src, uint32_t (&w)[36]) {
#pragma unroll
  for (int j = 0; j < 9; ++j) {
    const uint4 c = *reinterpret_cast<const uint4*>(src + 16 * j);
    w[4 * j] = c.x;
    w[4 * j + 1] = c.y;
    w[4 * j + 2] = c.z;
    w[4 * j + 3] = c.w;
  }
}

// Stages this lane's record of class r (run-time, warp-uniform) from the
// 16-byte-aligned group row `row` into TMEM column address ta; returns the
// record's scale bits. The class is a run-time value selected by a switch whose
// four cases each issue their own TMEM store of the picked words (one store
// site per case saves the register copies into a shared array: measured 186.5
// -> 181.9 us per fused step on the long ragged batch). Two earlier variants
// that instead specialised a whole worker function on a compile-time class
// raised "illegal instruction" on the GPU (cause not identified); this form has
// run cleanly in every test.
__device__ __forceinline__ uint32_t stage_record(const uint8_t* row, int r, uint32_t ta) {
  uint32_t w[36];
  load36(row + 128 * r, w);
  uint32_t scale;
  switch (r) {  // warp-uniform: every lane stages the same class
    case 0: { uint32_t v[32]; pick_record<0>(w, v, scale); tmem_st32(ta, v); break; }
    case 1: { uint32_t v[32]; pick_record<1>(w, v, scale); tmem_st32(ta, v); break; }
    case 2: { uint32_t v[32]; pick_record<2>(w, v, scale); tmem_st32(ta, v); break; }
    default: { uint32_t v[32]; pick_record<3>(w, v, scale); tmem_st32(ta, v); break; }
  }
  return scale;
}

// ------------------------------------------------------------------ MXFP4 records and queries
//
// An MXFP4 record (68 bytes: 64 bytes of e2m1 codes, element 2j in the low nibble
// of byte j, then the UE8M0 scale bytes of its four 32-element blocks) is turned
// into the 128 e4m3 bytes the MMA reads, exactly: with e_b the exponent of block
// b and E the record's largest, element x = v * 2^e_b (v an e2m1 value) is
// stored as the e4m3 value v * 2^(e_b - E + 6), and 2^(E - 6) becomes the
// record's scale for the epilogue. v * 2^k is an e4m3 value for every e2m1 v
// when -8 <= k <= 6 (the largest, 6 * 2^6 = 384, stays below 448; the smallest,
// 0.5 * 2^-8 = 2^-9, is e4m3's smallest subnormal), i.e. whenever the record's
// block exponents span at most 14. The query is MXFP4-rounded per head the same
// way and converted relative to its head's largest block exponent, so a single
// e4m3 term carries it exactly (no lo term: half the MMAs).

// e4m3 codes of the 8 e2m1 magnitudes (0, 0.5, 1, 1.5, 2, 3, 4, 6), four per word.
constexpr uint32_t kE2m1ToE4m3Lo = 0x3C383000u, kE2m1ToE4m3Hi = 0x4C484440u;

// e2m1 magnitude code (0..7) of a >= 0 (a value already divided by its block
// scale): round to nearest, ties to the even code, saturating at 6. Each
// comparison is one of the midpoints 0.25, 0.75, ..., 5; a tie stays on the even
// side (e.g. 0.75 goes up to 1.0 = code 2, 1.25 stays at 1.0).
__device__ __forceinline__ uint32_t e2m1_mag(float a) {
  return static_cast<uint32_t>(a > 0.25f) + static_cast<uint32_t>(a >= 0.75f) + static_cast<uint32_t>(a > 1.25f) +
         static_cast<uint32_t>(a >= 1.75f) + static_cast<uint32_t>(a > 2.5f) + static_cast<uint32_t>(a >= 3.5f) +
         static_cast<uint32_t>(a > 5.0f);
}

// Value of e2m1 magnitude code m: exponent m >> 1 (bias 1, 0 subnormal), mantissa m & 1.
__device__ __forceinline__ float e2m1_value(uint32_t m) {
  const int E = static_cast<int>(m >> 1);
  const float mant = (m & 1u) ? 1.5f : 1.0f;
  return E == 0 ? 0.5f * static_cast<float>(m & 1u) : mant * __int_as_float((E - 1 + 127) << 23);
}

// 2^k as an fp32 value for -149 <= k <= 127 (subnormal below -126).
__device__ __forceinline__ float pow2f(int k) {
  return k >= -126 ? __int_as_float((k + 127) << 23) : __int_as_float(1 << (k + 149));
}

// Two fp32 values as e4m3 codes (a in the low byte), round to nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// Block exponent of MXFP4: floor(log2 amax) - 2, clamped to [-127, 127]; -127
// for a block of zeros.
__device__ __forceinline__ int mx_block_exp(float amax) {
  if (!(amax > 0.0f)) return -127;
  int E2;
  (void)frexpf(amax, &E2);  // amax = f * 2^E2, f in [0.5, 1)
  const int e = E2 - 3;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// The 8 e4m3 codes of the e2m1 magnitudes times 2^k (k <= 6), as (lo, hi) words
// for a byte-permute lookup. For k >= -5 all eight are normal and the exponent
// fields just move by k; below, each is converted (exact down to k = -8).
// The table for k < -5 (blocks far below the record's largest: rare), out of
// line so that the workers' loop stays small.
__device__ __noinline__ uint2 e4m3_table_low(int k) {
  const float f = pow2f(k < -40 ? -40 : k);
  return make_uint2(e4m3x2(0.0f, 0.5f * f) | (e4m3x2(1.0f * f, 1.5f * f) << 16),
                    e4m3x2(2.0f * f, 3.0f * f) | (e4m3x2(4.0f * f, 6.0f * f) << 16));
}
__device__ __forceinline__ void e4m3_table(int k, uint32_t& lo, uint32_t& hi) {
  if (k >= -5) {
    const uint32_t add = static_cast<uint32_t>(k * 8);
    lo = kE2m1ToE4m3Lo + add * 0x01010100u;  // code 0 stays 0
    hi = kE2m1ToE4m3Hi + add * 0x01010101u;
  } else {
    const uint2 t = e4m3_table_low(k);
    lo = t.x;
    hi = t.y;
  }
}

// PTX byte permute in its default mode: byte n of the result is byte (sel nibble n
// & 7) of {b, a} (a bytes 0-3); bit 3 of the nibble replicates that byte's sign bit
// over the whole result byte instead.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Four e2m1 codes (the low four nibbles of c, element i in nibble i; the
// selector of a default-mode byte permute reads only bits 0-15) as four e4m3
// bytes (element i in byte i) through the table (lo, hi): the magnitude by a
// byte-permute lookup on the low three bits of each nibble, the sign from bit 3
// (a permute of 0x80 bytes in sign-replicate mode gives 0xFF for a set bit and
// 0x80 otherwise, so bit 6 of each byte is the sign: one shift moves it to bit 7;
// the carry-out of each byte lands in bit 0 of the next, which the mask drops).
__device__ __forceinline__ uint32_t e2m1x4_to_e4m3(uint32_t c, uint32_t lo, uint32_t hi) {
  const uint32_t mag = prmt(lo, hi, c & 0x7777u);
  const uint32_t rep = prmt(0x80808080u, 0x80808080u, c);
  return mag | ((rep << 1) & 0x80808080u);
}

// Words r .. r + 15 of the 20 loaded (the record's code bytes) into c; word
// r + 16 (its four scale bytes) into sb.
template <int R>
__device__ __forceinline__ void pick_record_fp4(const uint32_t (&w)[20], uint32_t (&c)[16], uint32_t& sb) {
#pragma unroll
  for (int j = 0; j < 16; ++j) c[j] = w[R + j];
  sb = w[R + 16];
}

// Stages this lane's MXFP4 record of class r (run-time, warp-uniform: the same
// reason as stage_record) from the 16-byte-aligned group row `row` (272 bytes =
// 4 records) into TMEM column address ta as 128 e4m3 bytes; returns the record's
// scale bits 2^(E - 6), NaN bits for a record holding a NaN scale byte. A block
// span above 14 is flagged (CSA_DEV_RANGE) and scored with its smallest blocks
// rounded.
__device__ __forceinline__ uint32_t stage_record_fp4(const uint8_t* row, int r, uint32_t ta, int32_t* flags) {
  uint32_t w[20];
#pragma unroll
  for (int j = 0; j < 5; ++j) {
    const uint4 q4 = *reinterpret_cast<const uint4*>(row + 64 * r + 16 * j);
    w[4 * j] = q4.x;
    w[4 * j + 1] = q4.y;
    w[4 * j + 2] = q4.z;
    w[4 * j + 3] = q4.w;
  }
  uint32_t c[16], sb;
  switch (r) {
    case 0: pick_record_fp4<0>(w, c, sb); break;
    case 1: pick_record_fp4<1>(w, c, sb); break;
    case 2: pick_record_fp4<2>(w, c, sb); break;
    default: pick_record_fp4<3>(w, c, sb); break;
  }
  int e[4], emax = -127;
  bool nan_scale = false;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const int byte = static_cast<int>((sb >> (8 * b)) & 0xFFu);
    nan_scale |= byte == 255;
    e[b] = byte - 127;
    emax = max(emax, e[b]);
  }
  uint32_t v[32];
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const int k = e[b] - emax + 6;
    if (k < -8) *flags |= CSA_DEV_RANGE;
    uint32_t lo, hi;
    e4m3_table(k, lo, hi);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t cw = c[4 * b + j];
      v[8 * b + 2 * j] = e2m1x4_to_e4m3(cw, lo, hi);
      v[8 * b + 2 * j + 1] = e2m1x4_to_e4m3(cw >> 16, lo, hi);
    }
  }
  tmem_st32(ta, v);
  if (nan_scale) {
    *flags |= CSA_DEV_RANGE;
    return kNaNBits;
  }
  return __float_as_uint(pow2f(emax - 6));
}

// MXFP4 rounding of 4 elements of one head (x[0..3], its block's exponent e_b,
// its head's largest E) as one word of e4m3 codes of v * 2^(e_b - E + 6).
__device__ __forceinline__ uint32_t fp4_query_word(const float (&x)[4], int eb, int E, int32_t* flags) {
  const float inv = pow2f(-eb);                   // 1 / block scale (e_b in [-127, 127])
  const int k = eb - E + 6;
  if (k < -8) *flags |= CSA_DEV_RANGE;
  const float f = pow2f(k < -40 ? -40 : k);
  float y[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float m = e2m1_value(e2m1_mag(fabsf(x[i]) * inv)) * f;
    y[i] = signbit(x[i]) ? -m : m;
  }
  return e4m3x2(y[0], y[1]) | (e4m3x2(y[2], y[3]) << 16);
}

// Splits heads h0 .. h0 + 15 of query row b into query slot qs (one warp), MXFP4:
// lane l holds elements 4l .. 4l + 3 of each head, so the 8 lanes of a block
// reduce its amax and all 32 lanes the head's largest block exponent.
__device__ void prep_query_part_fp4(const Params& P, Smem& S, int32_t b, int qs, int h0, int32_t* flags) {
  const int lane = threadIdx.x & 31;
  const uint16_t* qrow = P.q + (static_cast<int64_t>(b) * kH + h0) * kD;
  const float w_mine = lane < 16 ? __ldg(P.w + static_cast<int64_t>(b) * kH + h0 + lane) : 0.0f;
  uint8_t* hi = S.qbuf[qs][0];
  uint2 raw[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) raw[j] = __ldg(reinterpret_cast<const uint2*>(qrow + j * kD + lane * 4));
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int h = h0 + j;
    float x[4];
    x[0] = __uint_as_float(raw[j].x << 16);
    x[1] = __uint_as_float(raw[j].x & 0xFFFF0000u);
    x[2] = __uint_as_float(raw[j].y << 16);
    x[3] = __uint_as_float(raw[j].y & 0xFFFF0000u);
    float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));  // the block's 8 lanes
    if (!isfinite(a)) *flags |= CSA_DEV_RANGE;
    const int eb = mx_block_exp(isfinite(a) ? a : 0.0f);
    int E = eb;
#pragma unroll
    for (int o = 16; o >= 8; o >>= 1) E = max(E, __shfl_xor_sync(0xFFFFFFFFu, E, o));
    *reinterpret_cast<uint32_t*>(hi + qbuf_offset(h, lane >> 2) + (lane & 3) * 4) = fp4_query_word(x, eb, E, flags);
    if (lane == j) S.wbuf[qs][h] = w_mine * pow2f(E - 6);
  }
}

// The first segment's MXFP4 query by the whole CTA in the prologue (thread t:
// the 16 elements 16p .. 16p + 15 of head t / 8, p = t % 8; a block is two
// threads).
__device__ void prep_first_query_fp4(const Params& P, Smem& S, int32_t b, int32_t* flags) {
  const int tid = threadIdx.x, p = tid & 7, h = tid >> 3;
  const uint16_t* src = P.q + (static_cast<int64_t>(b) * kH + h) * kD + p * 16;
  const uint4 r0 = __ldg(reinterpret_cast<const uint4*>(src));
  const uint4 r1 = __ldg(reinterpret_cast<const uint4*>(src + 8));
  const float wv = p == 0 ? __ldg(P.w + static_cast<int64_t>(b) * kH + h) : 0.0f;
  const uint32_t u[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
  float x[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(u[i] << 16);
    x[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(x[i]));
  a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));  // the block's two threads
  if (!isfinite(a)) *flags |= CSA_DEV_RANGE;
  const int eb = mx_block_exp(isfinite(a) ? a : 0.0f);
  int E = eb;
#pragma unroll
  for (int o = 4; o >= 2; o >>= 1) E = max(E, __shfl_xor_sync(0xFFFFFFFFu, E, o));  // the head's 8 threads
  uint32_t wd[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float xi[4] = {x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]};
    wd[i] = fp4_query_word(xi, eb, E, flags);
  }
  *reinterpret_cast<uint4*>(S.qbuf[0][0] + qbuf_offset(h, p)) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
  if (p == 0) S.wbuf[0][h] = wv * pow2f(E - 6);
}

// The head sums of both records of a lane when a record of the warp has a
// negative scale (rare): relu(s x) = |s| relu(sign(s) x), the sign applied to
// each accumulator; kept out of line, away from the common path's code.
__device__ __noinline__ float2 head_sums_signed(uint32_t tc, const float4* wv, float g0, float g1) {
  float sa[4] = {0.0f, 0.0f, 0.0f, 0.0f}, sb[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 1
  for (int c = 0; c < kH; c += 16) {
    uint32_t x0[16], x1[16];
    tmem_ld16(tc + c, x0);
    tmem_ld16(tc + kH + c, x1);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 wq = wv[(c >> 2) + j];
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = __uint_as_float(x0[4 * j + i]) * g0;
        b[i] = __uint_as_float(x1[4 * j + i]) * g1;
      }
      sa[0] = fmaf(fmaxf(a[0], 0.0f), wq.x, sa[0]);
      sa[1] = fmaf(fmaxf(a[1], 0.0f), wq.y, sa[1]);
      sa[2] = fmaf(fmaxf(a[2], 0.0f), wq.z, sa[2]);
      sa[3] = fmaf(fmaxf(a[3], 0.0f), wq.w, sa[3]);
      sb[0] = fmaf(fmaxf(b[0], 0.0f), wq.x, sb[0]);
      sb[1] = fmaf(fmaxf(b[1], 0.0f), wq.y, sb[1]);
      sb[2] = fmaf(fmaxf(b[2], 0.0f), wq.z, sb[2]);
      sb[3] = fmaf(fmaxf(b[3], 0.0f), wq.w, sb[3]);
    }
  }
  return make_float2((sa[0] + sa[2]) + (sa[1] + sa[3]), (sb[0] + sb[2]) + (sb[1] + sb[3]));
}

// One warp of a worker group: group gi owns classes 2gi and 2gi + 1 of every tile.
template <bool kTopk, int kFmt>
__device__ void role_worker(const Params& P, Smem& S) {
  int32_t wflags = 0;  // CSA_DEV_RANGE from MXFP4 records
  const int e = (threadIdx.x >> 5) - kWarpWorker;  // 0..7
  const int gi = e >> 2;                            // worker group
  const int c0 = 2 * gi;                            // the group's first class
  const int q = e & 3;                              // TMEM lane quarter (warp index % 4)
  const int lane = threadIdx.x & 31;
  const int m = 32 * q + lane;                      // row of a class sub-tile: page m / 16, group m % 16
  const int pg_in_tile = m >> 4, grp = m & 15;
  const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
  const uint32_t tmem = S.tmem_base;
  const int64_t nt = S.plan.ntiles;

  // Stages the group's half-tile of tile t into its A stage: this lane's two
  // records (group grp of page pg_in_tile, records c0 and c0 + 1 of the group).
  // Returns false on abort; sets each record's scale bits (NaN when the record
  // is not visible) and position.
  auto stage = [&](int64_t t, uint32_t (&sc)[2], uint32_t (&pos)[2]) -> bool {
    const int64_t pg = kTP * t + pg_in_tile;
    const int s = static_cast<int>(pg % kPages);
    const bool ok = mbar_wait(smem_u32(&S.full[s]), static_cast<uint32_t>((pg / kPages) & 1), &S.abort_flag);
    if (!__all_sync(0xFFFFFFFFu, ok)) return false;
    const PageInfo pi = S.info[s];
    const uint32_t ta = tmem + a_col(gi) + lane_off;
    if constexpr (kFmt == CSA_RECORD_MXFP4) {
      // a slot's records past the page's visible rows (or a slot never filled) hold
      // whatever bytes were there: only visible records raise flags
      const uint8_t* row = S.pages[s] + grp * (4 * kFp4Rec);
      int32_t f0 = 0, f1 = 0;
      sc[0] = stage_record_fp4(row, c0, ta, &f0);
      sc[1] = stage_record_fp4(row, c0 + 1, ta + 32, &f1);
      wflags |= (4 * grp + c0 < pi.nrows ? f0 : 0) | (4 * grp + c0 + 1 < pi.nrows ? f1 : 0);
    } else {
      const uint8_t* row = S.pages[s] + grp * kGroupBytes;
      sc[0] = stage_record(row, c0, ta);
      sc[1] = stage_record(row, c0 + 1, ta + 32);
    }
    // the TMEM stores (warp-collective) have read every lane's loaded words: the
    // group is done with the warp's two pages
    __syncwarp();
    if ((lane & 15) == 0) mbar_arrive(smem_u32(&S.empty[s]));
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&S.afull[gi]));
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int rec = 4 * grp + c0 + c;
      sc[c] = rec < pi.nrows ? sc[c] : kNaNBits;
      pos[c] = static_cast<uint32_t>(pi.lp * kPage + rec);
    }
    return true;
  };

  uint32_t cur_sc[2] = {0, 0}, cur_pos[2] = {0, 0}, nxt_sc[2] = {0, 0}, nxt_pos[2] = {0, 0};
  bool ok = stage(0, cur_sc, cur_pos);

  Cursor64 cur;
  cur.init(P, S.plan);
  int seg = 0;
  for (int64_t t = 0; ok && t < nt; ++t) {
    const bool seg_start = (t == 0) || (cur.lt == 0);
    if (seg_start && t > 0) ++seg;
    const bool seg_end = (t == nt - 1) || (cur.lt == cur.tiles - 1);
    const int qs = seg & 1;
    if (seg_start) {  // this segment's head weights are in place
      ok = mbar_wait(smem_u32(&S.qfull[qs]), static_cast<uint32_t>((seg >> 1) & 1), &S.abort_flag);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
    }
    const float4* wv = reinterpret_cast<const float4*>(S.wbuf[qs]);
    const uint32_t h = static_cast<uint32_t>(2 * t + gi);  // half-tiles of a CTA stay far below 2^32
    const int ds = static_cast<int>(h % kDStages);
    // MMAs of h done: the accumulators are ready and the group's A stage is free
    ok = mbar_wait(smem_u32(&S.dfull[ds]), (h / kDStages) & 1, &S.abort_flag);
    if (!__all_sync(0xFFFFFFFFu, ok)) break;
    if (t + 1 < nt) {
      ok = stage(t + 1, nxt_sc, nxt_pos);
      if (!ok) break;
    }
    tc_fence_after();
    // logit = s * sum_h relu(x_h) w_h for both records; relu(s x) = |s| relu(sign(s) x).
    // Scalar multiply-adds into four partial sums per record: measured faster here
    // than packed fp32 pairs (179 against 182 us per fused step), which have half
    // as many independent chains. When no record of the warp has a negative scale
    // the sign products are left out; the other case runs out of line
    // (head_sums_signed), which keeps this loop's code small: 174 against 177 us
    // with both cases inlined here.
    const float s0 = __uint_as_float(cur_sc[0]), s1 = __uint_as_float(cur_sc[1]);
    const float g0 = s0 < 0.0f ? -1.0f : 1.0f, g1 = s1 < 0.0f ? -1.0f : 1.0f;
    const bool all_pos = __all_sync(0xFFFFFFFFu, g0 > 0.0f && g1 > 0.0f);
    const uint32_t tc = tmem + lane_off + d_col(ds);
    float logit[2];
    if (all_pos) {  // the common case: no sign products
      float sa[4] = {0.0f, 0.0f, 0.0f, 0.0f}, sb[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 1
      for (int c = 0; c < kH; c += 16) {  // heads c .. c+15 of both records per TMEM wait
        uint32_t x0[16], x1[16];
        tmem_ld16(tc + c, x0);
        tmem_ld16(tc + kH + c, x1);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 wq = wv[(c >> 2) + j];
          float a[4], b[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            a[i] = __uint_as_float(x0[4 * j + i]);
            b[i] = __uint_as_float(x1[4 * j + i]);
          }
          sa[0] = fmaf(fmaxf(a[0], 0.0f), wq.x, sa[0]);
          sa[1] = fmaf(fmaxf(a[1], 0.0f), wq.y, sa[1]);
          sa[2] = fmaf(fmaxf(a[2], 0.0f), wq.z, sa[2]);
          sa[3] = fmaf(fmaxf(a[3], 0.0f), wq.w, sa[3]);
          sb[0] = fmaf(fmaxf(b[0], 0.0f), wq.x, sb[0]);
          sb[1] = fmaf(fmaxf(b[1], 0.0f), wq.y, sb[1]);
          sb[2] = fmaf(fmaxf(b[2], 0.0f), wq.z, sb[2]);
          sb[3] = fmaf(fmaxf(b[3], 0.0f), wq.w, sb[3]);
        }
      }
      logit[0] = fabsf(s0) * ((sa[0] + sa[2]) + (sa[1] + sa[3]));
      logit[1] = fabsf(s1) * ((sb[0] + sb[2]) + (sb[1] + sb[3]));
    } else {
      const float2 r = head_sums_signed(tc, wv, g0, g1);
      logit[0] = fabsf(s0) * r.x;
      logit[1] = fabsf(s1) * r.y;
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&S.dempty[ds]));
    if constexpr (!kTopk) {
#pragma unroll
      for (int c = 0; c < 2; ++c)
        if (!isnan(__uint_as_float(cur_sc[c]))) {
          const float val = P.raw_logits ? logit[c] : __frcp_rn(1.0f + __expf(-logit[c]));
          P.scores[static_cast<int64_t>(cur.b) * P.score_stride + cur.lt * kTileRecs + pg_in_tile * kPage + 4 * grp +
                   c0 + c] = val;
        }
    } else {
      const int slot = static_cast<int>(t % kKeyRing);
      ok = mbar_wait(smem_u32(&S.kempty[slot]), static_cast<uint32_t>(((t / kKeyRing) & 1) ^ 1), &S.abort_flag);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      const uint32_t thr = filter_word(S, seg);
      const uint32_t ltm = lanemask_lt();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const bool valid = !isnan(__uint_as_float(cur_sc[c])) && !isnan(logit[c]);
        const uint64_t key = valid ? make_key(logit[c], static_cast<int32_t>(cur_pos[c])) : 0ull;
        const bool take = valid && static_cast<uint32_t>(key >> 32) >= thr;
        const uint32_t ballot = __ballot_sync(0xFFFFFFFFu, take);
        const int region = 4 * (c0 + c) + q;
        if (take) S.keys[slot][32 * region + __popc(ballot & ltm)] = key;
        if (lane == 0) S.kcnt[slot][region] = static_cast<uint32_t>(__popc(ballot));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&S.kfull[slot]));
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      cur_sc[c] = nxt_sc[c];
      cur_pos[c] = nxt_pos[c];
    }
    if (seg_end) {  // done with this segment's head weights
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&S.qempty[qs]));
    }
    cur.advance(P);
  }
  if constexpr (kFmt == CSA_RECORD_MXFP4) {
    wflags = __reduce_or_sync(0xFFFFFFFFu, static_cast<uint32_t>(wflags));
    if (lane == 0 && wflags) atomicOr(&S.status, wflags);
  }
}

// ------------------------------------------------------------------ selector

// Splits heads h0 .. h0 + 15 of query row b into query slot qs (one warp): the
// arithmetic and layout of prep_query over a quarter of the heads, with all 16
// heads' loads in flight at once.
__device__ void prep_query_part(const Params& P, Smem& S, int32_t b, int qs, int h0, int32_t* flags) {
  const int lane = threadIdx.x & 31;
  const uint16_t* qrow = P.q + (static_cast<int64_t>(b) * kH + h0) * kD;
  const float w_mine = lane < 16 ? __ldg(P.w + static_cast<int64_t>(b) * kH + h0 + lane) : 0.0f;
  uint8_t* hi = S.qbuf[qs][0];
  uint8_t* lo = S.qbuf[qs][1];
  uint2 raw[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) raw[j] = __ldg(reinterpret_cast<const uint2*>(qrow + j * kD + lane * 4));
#pragma unroll
  for (int j = 0; j < 16; ++j) {
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
    if (lane == j) S.wbuf[qs][h] = w_mine * isc;
  }
}

// Same selection as the other scorer, per tile: the tile's admissible keys
// (16 regions, one per class and worker warp) enter a shared buffer, which is
// cut back to between k and loose_keep(k) keys when it could overflow; each
// segment's survivors go to workspace slot (row + CTA).
// kShort: the instantiation for batches of many short rows (chunked prefill),
// where a whole row inside the CTA that fits the buffer is written uncut when
// its slot has room and the merge, which then reads that one slot, cuts it (the
// selector, not the workers, bounds those batches).
template <int kFmt, bool kShort>
__device__ void role_select(const Params& P, Smem& S) {
  const int g = threadIdx.x - kWarpSelect * 32;
  const int sw = g >> 5, lane = g & 31;
  Cursor64 cur;
  cur.init(P, S.plan);
  int seg = 0;
  // query preparation: the next segment to prepare (1, then 2, ...), its row,
  // and the tiles that the segments prepared so far cover
  int32_t qflags = 0;
  int prep_seg = 1;
  int64_t prep_done = query_tiles<kTP>(P, S.plan.b0) - S.plan.lt0;
  int32_t prep_b = next_nonempty<kTP>(P, S.plan.b0 + 1);
  auto prep_next = [&]() {
    if (prep_done >= S.plan.ntiles) return;  // uniform
    const int qs = prep_seg & 1;
    if constexpr (kFmt == CSA_RECORD_MXFP4)
      prep_query_part_fp4(P, S, prep_b, qs, 16 * sw, &qflags);
    else
      prep_query_part(P, S, prep_b, qs, 16 * sw, &qflags);
    fence_proxy_async_smem();  // the MMA reads the query through the async proxy
    named_bar_sync(kBarSelect, 128);
    if (g == 0) mbar_arrive(smem_u32(&S.qfull[qs]));
    prep_done += query_tiles<kTP>(P, prep_b);
    prep_b = next_nonempty<kTP>(P, prep_b + 1);
    ++prep_seg;
  };
  prep_next();  // segment 1 into the free slot 1
  for (int64_t t = 0; t < S.plan.ntiles; ++t) {
    const int slot = static_cast<int>(t % kKeyRing);
    const uint32_t ph = static_cast<uint32_t>((t / kKeyRing) & 1);
    if (g == 0) S.go[t & 1] = mbar_wait(smem_u32(&S.kfull[slot]), ph, &S.abort_flag) ? 1 : 0;
    named_bar_sync(kBarSelect, 128);  // passes the leader's acquire of the slot on to the group
    if (!S.go[t & 1]) break;
    // The workers kept the keys at or above the threshold word they last read;
    // the selector's own threshold may have risen since (a cut that finished
    // after they read it: they run up to kKeyRing tiles ahead), so every key is
    // checked again on the way in. Warp sw takes lane quarter sw of each class
    // (regions 4c + sw) and places its survivors after those of warps 0 .. sw-1.
    {
      const uint64_t tau = S.sel.tau;  // keys must exceed it; 0 at a segment start
      const uint32_t n0 = S.sel.n;
      uint64_t key[4];
      uint32_t bal[4], mine = 0;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int i = 4 * c + sw;
        const bool have = static_cast<uint32_t>(lane) < S.kcnt[slot][i];
        key[c] = have ? S.keys[slot][32 * i + lane] : 0ull;
        bal[c] = __ballot_sync(0xFFFFFFFFu, have && key[c] > tau);
        mine += static_cast<uint32_t>(__popc(bal[c]));
      }
      if (lane == 0) S.sel.part[0][sw] = mine;
      named_bar_sync(kBarSelect, 128);
      uint32_t off = n0, total = n0;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t c = S.sel.part[0][w];
        off += w < sw ? c : 0u;
        total += c;
      }
      const uint32_t ltm = lanemask_lt();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if ((bal[c] >> lane) & 1u) S.cand[off + __popc(bal[c] & ltm)] = key[c];
        off += static_cast<uint32_t>(__popc(bal[c]));
      }
      if (g == 0) S.sel.n = total;
    }
    named_bar_sync(kBarSelect, 128);
    if (g == 0) mbar_arrive(smem_u32(&S.kempty[slot]));
    bool whole_short = false;
    if constexpr (kShort)
      whole_short = cur.tiles * kTileRecs <= kCapW && cur.lt == cur.tiles - 1 && (seg > 0 || S.plan.lt0 == 0);
    shrink_if_above_reg<128, kCapW / 128, 512>(S.cand, S.scratch, whole_short ? kCapW : kCapW - kTileRecs, P.k,
                                               loose_keep(P.k), &S.sel, kBarSelect, g);
    const bool seg_end = (t == S.plan.ntiles - 1) || (cur.lt == cur.tiles - 1);
    if (seg_end) {
      const int limit = whole_short ? static_cast<int>((P.slot_bytes - 16) / 8) : loose_keep(P.k);  // slot room
      shrink_if_above_reg<128, kCapW / 128, 512>(S.cand, S.scratch, limit, P.k, loose_keep(P.k), &S.sel, kBarSelect, g);
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
      // the keys of segment seg - 1's last tile are in: its MMAs and epilogues
      // are done with query slot (seg - 1) & 1, which segment seg + 1 takes
      if (prep_seg == seg + 1) prep_next();
    }
    if (g == 0) {
      const uint64_t T = S.sel.tau + 1;  // keys >= T are admitted
      *reinterpret_cast<volatile uint64_t*>(&S.filt) =
          (static_cast<uint64_t>(static_cast<uint32_t>(seg)) << 32) | static_cast<uint32_t>(S.sel.tau ? T >> 32 : 0);
    }
    cur.advance(P);
  }
  if (qflags) atomicOr(&S.status, qflags);
}

// Score mode, MXFP4: warp 12 splits the CTA's later queries (as prep_segments
// does for e4m3 records), 16 heads at a time.
__device__ void prep_segments_fp4(const Params& P, Smem& S) {
  const int lane = threadIdx.x & 31;
  int32_t flags = 0;
  int64_t done = query_tiles<kTP>(P, S.plan.b0) - S.plan.lt0;
  int32_t b = next_nonempty<kTP>(P, S.plan.b0 + 1);
  for (int seg = 1; done < S.plan.ntiles; ++seg) {
    const int qs = seg & 1;
    int ok = 1;
    if (lane == 0)
      ok = mbar_wait(smem_u32(&S.qempty[qs]), static_cast<uint32_t>(((seg >> 1) & 1) ^ 1), &S.abort_flag);
    if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
    for (int h0 = 0; h0 < kH; h0 += 16) prep_query_part_fp4(P, S, b, qs, h0, &flags);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&S.qfull[qs]));
    done += query_tiles<kTP>(P, b);
    b = next_nonempty<kTP>(P, b + 1);
  }
  flags = static_cast<int32_t>(__reduce_or_sync(0xFFFFFFFFu, static_cast<uint32_t>(flags)));
  if (lane == 0 && flags) atomicOr(&S.status, flags);
}

// ------------------------------------------------------------------ kernel

template <bool kTopk, int kFmt, bool kShort = false>
__global__ void __launch_bounds__(kThreads, 1) score_kernel_w64(const __grid_constant__ Params P) {
  extern __shared__ uint8_t smem_raw[];
  Smem& S = smem_of(smem_raw);
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
  make_plan<kThreads, kTP>(P, &S.plan, S.warp_sums, kTopk ? reinterpret_cast<int32_t*>(P.ws) : nullptr);
  if (tid == 0 && blockIdx.x == 0 && S.plan.flags && P.dev_status) atomicOr(P.dev_status, S.plan.flags);
  if (S.plan.ntiles == 0) return;  // uniform

  if (tid == 0) {
    for (int s = 0; s < kPages; ++s) {
      mbar_init(smem_u32(&S.full[s]), 1);
      mbar_init(smem_u32(&S.empty[s]), 2);  // the two worker warps (one per group) that read the page
    }
    for (int g = 0; g < 2; ++g) mbar_init(smem_u32(&S.afull[g]), 4);  // the four warps of the group
    for (int s = 0; s < kDStages; ++s) {
      mbar_init(smem_u32(&S.dfull[s]), 2);  // both MMA threads commit
      mbar_init(smem_u32(&S.dempty[s]), 4);
    }
    for (int i = 0; i < kKeyRing; ++i) {
      mbar_init(smem_u32(&S.kfull[i]), kWorkerWarps);  // every worker warp, once per tile
      mbar_init(smem_u32(&S.kempty[i]), 1);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(smem_u32(&S.rfull[i]), 1);
      mbar_init(smem_u32(&S.rempty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&S.qfull[i]), 1);
      mbar_init(smem_u32(&S.qempty[i]), kQEmptyCount);
    }
    mbar_init(smem_u32(&S.drain), 2);
    mbar_init_fence();
    fence_proxy_async_smem();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(&S.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  {
    int32_t qflags = 0;
    if constexpr (kFmt == CSA_RECORD_MXFP4)
      prep_first_query_fp4(P, S, S.plan.b0, &qflags);
    else
      prep_first_query<kH>(P, S, S.plan.b0, &qflags);
    fence_proxy_async_smem();  // the MMA reads the query through the async proxy
    if (qflags) atomicOr(&S.status, qflags);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) mbar_arrive(smem_u32(&S.qfull[0]));

  if (warp == kWarpIssuer) {
    role_issuer<kFmt>(P, S);
  } else if (warp == kWarpMma) {
    if ((tid & 31) == 0) role_mma<kFmt>(P, S, 0);
  } else if (warp == kWarpMma2) {
    if ((tid & 31) == 0) role_mma<kFmt>(P, S, 1);
  } else if (warp == kWarpWalker) {
    walk_pages<kTP, Smem, Cursor64>(P, S);
  } else if (warp < kWarpSelect) {
    role_worker<kTopk, kFmt>(P, S);
  } else if (kTopk) {
    role_select<kFmt, kShort>(P, S);
  } else if (warp == kWarpSelect) {
    if constexpr (kFmt == CSA_RECORD_MXFP4)
      prep_segments_fp4(P, S);
    else
      prep_segments<kH, kTP>(P, S);
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

}  // namespace w64
}  // namespace csa
