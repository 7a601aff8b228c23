// csa_select.cuh — block-level top-k building blocks over 64-bit ranking keys.
//
// A candidate is one 64-bit key: the high word is an order-preserving image of
// the fp32 value (logit or score), the low word the bitwise complement of the
// record's logical position. Larger key = better candidate, and equal values
// rank the lower position first, which is the order the top-k returns
// (value descending, position ascending). Keys of distinct positions are
// distinct, so "the k-th largest key" is always well defined.
//
// All helpers run on a group of NT threads (a multiple of 32) that share a
// named barrier `bar`; `gtid` is the thread's index inside the group.
#pragma once

#include <cstdint>

#include "csa_ptx.cuh"

namespace csa {

__device__ __forceinline__ uint32_t float_key(float f) {
  if (f == 0.0f) f = 0.0f;  // -0 and +0 rank alike
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_float(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

__device__ __forceinline__ uint64_t make_key(float v, int32_t position) {
  return (static_cast<uint64_t>(float_key(v)) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(position));
}

__device__ __forceinline__ int32_t key_position(uint64_t key) {
  return static_cast<int32_t>(~static_cast<uint32_t>(key));
}

__device__ __forceinline__ float key_value(uint64_t key) { return key_float(static_cast<uint32_t>(key >> 32)); }

// Shared scratch of one selecting group.
constexpr int kCutCandidates = 8;  // thresholds tried per sampled cut

constexpr int kHistBins = 512;  // bins of the widest histogram cut
struct SelectShared {
  uint32_t hist[kHistBins];
  uint32_t bcast[4];
  uint32_t gather;    // compaction cursor
  uint32_t n;         // live candidates in the buffer
  uint64_t tau;       // admission threshold: a key must exceed it
  uint64_t cut[kCutCandidates];        // candidate thresholds of a sampled cut, descending
  uint32_t cut_count[kCutCandidates];  // keys >= each
  uint32_t part[2][8];                 // per-warp partials of a histogram cut (up to 8 warps)
  uint32_t pick[3];                    // its boundary bin, keys above it, keys in it
};

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Returns T such that between `kk` and `max_keep` of keys[0, n) are >= T
// (1 <= kk <= max_keep, kk <= n, keys distinct); with max_keep == kk, T is the
// kk-th largest key. MSB-first radix select with 8-bit digits: after each digit,
// the keys whose prefix is above the boundary digit are in, those below are out,
// and it stops as soon as taking the boundary group whole keeps at most
// max_keep keys.
template <int NT>
__device__ uint64_t select_kth(const uint64_t* keys, int n, int kk, int max_keep, SelectShared* ss, int bar,
                               int gtid) {
  const int lane = gtid & 31;
  const int warp = gtid >> 5;
  uint64_t prefix = 0, mask = 0;
  int need = kk;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int j = gtid; j < 256; j += NT) ss->hist[j] = 0;
    named_bar_sync(bar, NT);
    for (int base = 0; base < n; base += NT) {
      const int i = base + gtid;
      uint32_t d = 256;
      if (i < n) {
        const uint64_t key = keys[i];
        if ((key & mask) == prefix) d = static_cast<uint32_t>(key >> shift) & 255u;
      }
      const uint32_t peers = __match_any_sync(0xFFFFFFFFu, d);
      if (d < 256 && lane == __ffs(peers) - 1) atomicAdd(&ss->hist[d], static_cast<uint32_t>(__popc(peers)));
    }
    named_bar_sync(bar, NT);
    if (warp == 0) {
      // lane l holds digits 255-8l ... 248-8l (descending)
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = ss->hist[255 - 8 * lane - j];
        sum += c[j];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      const uint32_t excl = incl - sum;
      const bool here = excl < static_cast<uint32_t>(need) && static_cast<uint32_t>(need) <= incl;
      if (here) {
        uint32_t acc = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (acc + c[j] >= static_cast<uint32_t>(need)) {
            ss->bcast[0] = 255 - 8 * lane - j;
            ss->bcast[1] = acc;
            ss->bcast[2] = c[j];
            break;
          }
          acc += c[j];
        }
      }
    }
    named_bar_sync(bar, NT);
    const uint32_t digit = ss->bcast[0];
    const int above = static_cast<int>(ss->bcast[1]);
    const int group = static_cast<int>(ss->bcast[2]);
    need -= above;
    prefix |= static_cast<uint64_t>(digit) << shift;
    mask |= static_cast<uint64_t>(0xFFu) << shift;
    // keys >= prefix: (kk - need) above the group, plus the group itself
    if ((kk - need) + group <= max_keep) return prefix;
  }
  return prefix;
}

// Keeps the keys >= T of keys[0, n) (in some order) at the front of `keys`,
// using `scratch` (room for `cap` keys). Returns their count, at most `cap`
// (more only if the caller broke the distinct-key precondition). One shared
// atomic per warp and round.
template <int NT>
__device__ int compact_ge(uint64_t* keys, int n, uint64_t T, uint64_t* scratch, int cap, SelectShared* ss,
                          int bar, int gtid) {
  if (gtid == 0) ss->gather = 0;
  named_bar_sync(bar, NT);
  for (int base = 0; base < n; base += NT) {
    const int i = base + gtid;
    const uint64_t key = i < n ? keys[i] : 0ull;
    const bool take = i < n && key >= T;
    const uint32_t ballot = __ballot_sync(0xFFFFFFFFu, take);
    uint32_t p = 0;
    if ((gtid & 31) == 0 && ballot) p = atomicAdd(&ss->gather, static_cast<uint32_t>(__popc(ballot)));
    p = __shfl_sync(0xFFFFFFFFu, p, 0) + __popc(ballot & lanemask_lt());
    if (take && p < static_cast<uint32_t>(cap)) scratch[p] = key;
  }
  named_bar_sync(bar, NT);
  const int m = min(static_cast<int>(ss->gather), cap);
  for (int i = gtid; i < m; i += NT) keys[i] = scratch[i];
  named_bar_sync(bar, NT);
  return m;
}

// Sample-guided cut. Tries to find a T with kk <= #(keys[0, n) >= T) <= max_keep
// and, when it does, moves the keys >= T to the front of `keys` (through
// `scratch`, room for max(NS / 2, max_keep) keys) and returns T with their count
// in *kept; otherwise it returns 0 and leaves `keys` alone (the caller falls
// back to select_kth). The candidate thresholds are value words with a zero
// position word, T = v << 32, so "key >= T" is "value word >= v" and every test
// below is a 32-bit compare.
//
// NS evenly spaced samples, one per thread of the first NS / 32 warps, are
// sorted inside each warp (bitonic, by shuffles) and ranked across warps by
// binary search in the other warps' sorted lists; the sample of rank r has
// about (r + 1) * n / NS keys at or above it, so the samples whose rank
// predicts a count between kk and max_keep give kCutCandidates thresholds.
// One pass counts the keys at or above each; the highest threshold whose count
// lies in the window wins, and a block-wide scan of each thread's own count
// places the kept keys without atomics. Keys are nonzero.
template <int NT, int NS>
__device__ uint64_t cut_sampled(uint64_t* keys, int n, int kk, int max_keep, uint64_t* scratch, int* kept,
                                SelectShared* ss, int bar, int gtid) {
  static_assert(NS % 32 == 0 && NS <= NT && NS <= 256, "one sample per thread of the first NS");
  constexpr int kC = kCutCandidates, kW = NS / 32;
  const int lane = gtid & 31, warp = gtid >> 5;
  uint32_t* sorted = reinterpret_cast<uint32_t*>(scratch);  // kW lists of 32 value words, descending
  if (gtid < kC) ss->cut_count[gtid] = 0;
  if (gtid < NS) {
    uint32_t x = static_cast<uint32_t>(keys[static_cast<int>((static_cast<int64_t>(gtid) * n) / NS)] >> 32);
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
      for (int st = size >> 1; st > 0; st >>= 1) {
        const uint32_t y = __shfl_xor_sync(0xFFFFFFFFu, x, st);
        const bool keep_max = ((lane & st) == 0) == ((lane & size) == 0);
        x = keep_max ? max(x, y) : min(x, y);
      }
    }
    sorted[32 * warp + lane] = x;
  }
  named_bar_sync(bar, NT);
  const int lo = max(0, (kk * NS + n - 1) / n - 1);
  const int hi = max(lo, min(NS - 1, (max_keep * NS) / n - 1));
  if (gtid < NS) {
    const uint32_t x = sorted[32 * warp + lane];
    int r = lane;  // equal words: earlier warps rank above, later ones below
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      if (w == warp) continue;
      const uint32_t* L = sorted + 32 * w;
      int a = 0;
#pragma unroll
      for (int step = 16; step > 0; step >>= 1) {
        const uint32_t v = L[a + step - 1];
        if (w < warp ? v >= x : v > x) a += step;
      }
      if (a == 31 && (w < warp ? L[31] >= x : L[31] > x)) a = 32;
      r += a;
    }
#pragma unroll
    for (int c = 0; c < kC; ++c)
      if (r == lo + ((hi - lo) * c) / (kC - 1)) ss->cut[c] = static_cast<uint64_t>(x) << 32;
  }
  named_bar_sync(bar, NT);
  uint32_t T[kC], cnt[kC];
#pragma unroll
  for (int c = 0; c < kC; ++c) {
    T[c] = static_cast<uint32_t>(ss->cut[c] >> 32);
    cnt[c] = 0;
  }
  const uint32_t* words = reinterpret_cast<const uint32_t*>(keys) + 1;  // value words, stride 2
  int i = gtid;
  for (; i + 3 * NT < n; i += 4 * NT) {
    uint32_t x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) x[u] = words[2 * (i + u * NT)];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int c = 0; c < kC; ++c) cnt[c] += x[u] >= T[c] ? 1u : 0u;
  }
  for (; i < n; i += NT) {
    const uint32_t x = words[2 * i];
#pragma unroll
    for (int c = 0; c < kC; ++c) cnt[c] += x >= T[c] ? 1u : 0u;
  }
#pragma unroll
  for (int c = 0; c < kC; ++c) {
    const uint32_t sum = __reduce_add_sync(0xFFFFFFFFu, cnt[c]);
    if (lane == 0 && sum) atomicAdd(&ss->cut_count[c], sum);
  }
  named_bar_sync(bar, NT);
  // thresholds descend with c, so counts ascend: the first count >= kk decides
  uint32_t best = 0, mine = 0, total = 0;
  bool found = false;
#pragma unroll
  for (int c = 0; c < kC; ++c) {
    const uint32_t m = ss->cut_count[c];
    if (!found && m >= static_cast<uint32_t>(kk)) {
      found = true;
      if (m <= static_cast<uint32_t>(max_keep)) {
        best = T[c];
        mine = cnt[c];
        total = m;
      }
    }
  }
  if (best == 0) return 0ull;  // uniform
  uint32_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) ss->hist[warp] = incl;
  named_bar_sync(bar, NT);
  uint32_t p = incl - mine;
  for (int w = 0; w < warp; ++w) p += ss->hist[w];
  i = gtid;
  for (; i + 3 * NT < n; i += 4 * NT) {
    uint64_t x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) x[u] = keys[i + u * NT];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (static_cast<uint32_t>(x[u] >> 32) >= best) scratch[p++] = x[u];
  }
  for (; i < n; i += NT) {
    const uint64_t x = keys[i];
    if (static_cast<uint32_t>(x >> 32) >= best) scratch[p++] = x;
  }
  named_bar_sync(bar, NT);
  for (int j = gtid; j < static_cast<int>(total); j += NT) keys[j] = scratch[j];
  named_bar_sync(bar, NT);
  *kept = static_cast<int>(total);
  return static_cast<uint64_t>(best) << 32;
}

// Histogram cut with the keys held in registers. Tries to find a value word T
// with kk <= #(keys[0, n) >= T << 32) <= max_keep and, when it does, compacts
// those keys in place to the front of `keys`, sets ss->n to their count and
// ss->tau so that later keys must be >= T << 32, and returns true. Returns false,
// with `keys` untouched, only when ties of value words make every such T
// impossible (the caller then selects on whole keys). n <= KPT * NT.
//
// Thread g holds keys g, g + NT, ... in registers for the whole cut, so the
// compaction may overwrite the buffer in any order. The value words span
// [lo, hi]; a round spreads the words of a window [base, base + NB * 2^s) over
// NB bins of width 2^s (NB = 256 or 512), scans the bin counts from the top and
// finds the bin holding the kk-th key. If every key from that bin up fits in
// max_keep, the bin's lower edge is T; otherwise the next round zooms into that
// bin with bins NB times narrower. Four rounds at most; the first usually
// decides, because the window starts at the keys' own range (a segment's first
// cut spans logits of both signs: 512 bins then decide in one round more often
// than 256; measured on the long ragged batch, 177.6 against 178.9 us per step).
template <int NT, int KPT, int NB = 256>
__device__ bool cut_hist(uint64_t* keys, int n, int kk, int max_keep, SelectShared* ss, int bar, int gtid) {
  static_assert((NT == 128 || NT == 256) && (NB == 256 || NB == 512) && NB <= kHistBins, "whole bins per thread");
  constexpr int BPT = NB / NT;
  constexpr int kBits = NB == 256 ? 8 : 9;
  constexpr int NW = NT / 32;
  const int lane = gtid & 31, warp = gtid >> 5;
  uint64_t k[KPT];
  uint32_t lo = 0xFFFFFFFFu, hi = 0;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const int i = gtid + NT * j;
    k[j] = i < n ? keys[i] : 0ull;  // keys are nonzero: 0 marks an empty register
    if (i < n) {
      const uint32_t v = static_cast<uint32_t>(k[j] >> 32);
      lo = min(lo, v);
      hi = max(hi, v);
    }
  }
  lo = __reduce_min_sync(0xFFFFFFFFu, lo);
  hi = __reduce_max_sync(0xFFFFFFFFu, hi);
  if (lane == 0) {
    ss->part[0][warp] = lo;
    ss->part[1][warp] = hi;
  }
#pragma unroll
  for (int j = 0; j < BPT; ++j) ss->hist[BPT * gtid + j] = 0;
  named_bar_sync(bar, NT);
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    lo = min(lo, ss->part[0][w]);
    hi = max(hi, ss->part[1][w]);
  }
  uint32_t base = lo;
  int s = (32 - kBits) - __clz(hi - lo);  // NB bins of width 2^s cover [lo, hi]
  s = s < 0 ? 0 : s;
  uint32_t need = static_cast<uint32_t>(kk), room = static_cast<uint32_t>(max_keep), T = 0;
  while (true) {
    // keys above the window were taken in an earlier round, keys below it dropped
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const uint32_t v = static_cast<uint32_t>(k[j] >> 32);
      if (k[j] != 0ull && v >= base) {
        const uint32_t d = (v - base) >> s;
        if (d < static_cast<uint32_t>(NB)) atomicAdd(&ss->hist[d], 1u);
      }
    }
    named_bar_sync(bar, NT);
    // thread g reads bins 255 - BPT g - j, j < BPT (descending), and clears them
    // for the next round; the scan below is over those groups
    uint32_t c[BPT], sum = 0;
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
      c[j] = ss->hist[NB - 1 - BPT * gtid - j];
      ss->hist[NB - 1 - BPT * gtid - j] = 0;
      sum += c[j];
    }
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += x;
    }
    if (lane == 31) ss->part[0][warp] = incl;
    named_bar_sync(bar, NT);
    uint32_t excl = incl - sum;
    for (int w = 0; w < warp; ++w) excl += ss->part[0][w];
    if (excl < need && need <= excl + sum) {  // one thread: the kk-th key is in one of its bins
      uint32_t acc = excl;
#pragma unroll
      for (int j = 0; j < BPT; ++j) {
        if (acc < need && need <= acc + c[j]) {
          ss->pick[0] = NB - 1 - BPT * gtid - j;
          ss->pick[1] = acc;
          ss->pick[2] = c[j];
        }
        acc += c[j];
      }
    }
    named_bar_sync(bar, NT);
    const uint32_t d = ss->pick[0], above = ss->pick[1], cnt = ss->pick[2];
    if (above + cnt <= room) {
      T = base + (d << s);
      break;
    }
    if (s == 0) return false;  // uniform: one value word holds too many keys
    need -= above;
    room -= above;
    base += d << s;
    s = s >= kBits ? s - kBits : 0;
  }
  // compaction in place: exclusive scan of each thread's kept count
  uint32_t mine = 0;
#pragma unroll
  for (int j = 0; j < KPT; ++j) mine += (k[j] != 0ull && static_cast<uint32_t>(k[j] >> 32) >= T) ? 1u : 0u;
  uint32_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) ss->part[1][warp] = incl;
  named_bar_sync(bar, NT);
  uint32_t p = incl - mine, total = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const uint32_t c = ss->part[1][w];
    p += w < warp ? c : 0u;
    total += c;
  }
#pragma unroll
  for (int j = 0; j < KPT; ++j)
    if (k[j] != 0ull && static_cast<uint32_t>(k[j] >> 32) >= T) keys[p++] = k[j];
  if (gtid == 0) {
    ss->n = total;
    ss->tau = (static_cast<uint64_t>(T) << 32) - 1;  // T >= lo > 0: no value word is 0
  }
  return true;
}

// Every thread offers two keys (`take_a`, `take_b`); accepted keys are appended
// to buf at ss->n with one shared atomic per warp. The caller's group barrier
// makes ss->n current.
__device__ __forceinline__ void append_keys2(uint64_t* buf, uint64_t a, bool take_a, uint64_t b, bool take_b,
                                             SelectShared* ss) {
  const uint32_t ba = __ballot_sync(0xFFFFFFFFu, take_a);
  const uint32_t bb = __ballot_sync(0xFFFFFFFFu, take_b);
  const uint32_t na = __popc(ba);
  uint32_t base = 0;
  if ((threadIdx.x & 31) == 0 && (ba | bb)) base = atomicAdd(&ss->n, na + static_cast<uint32_t>(__popc(bb)));
  base = __shfl_sync(0xFFFFFFFFu, base, 0);
  const uint32_t lt = lanemask_lt();
  if (take_a) buf[base + __popc(ba & lt)] = a;
  if (take_b) buf[base + na + __popc(bb & lt)] = b;
}

// Every thread offers at most one key (`take`); accepted keys are appended to
// buf at ss->n. Ends with a group barrier, after which ss->n is current.
__device__ __forceinline__ void append_key(uint64_t* buf, uint64_t key, bool take, SelectShared* ss) {
  const uint32_t ballot = __ballot_sync(0xFFFFFFFFu, take);
  uint32_t base = 0;
  if ((threadIdx.x & 31) == 0 && ballot) base = atomicAdd(&ss->n, static_cast<uint32_t>(__popc(ballot)));
  base = __shfl_sync(0xFFFFFFFFu, base, 0);
  if (take) buf[base + __popc(ballot & lanemask_lt())] = key;
}

// Cuts the buffer down when it holds more than `limit` keys: to the keys >= T
// for a T that keeps between kk and max_keep of them (exactly the kk best when
// max_keep == kk), and raises the admission threshold to T. Any such T is a
// valid threshold: at least kk keys seen so far are >= T, so no key below T can
// be among the kk best. The sampled cut is tried first when the window is
// open; `scratch` holds max(NS, max_keep) keys. Group-uniform. Kept out of
// line: cuts are rare, and one copy of their code leaves more of the
// instruction cache to the loops that run every tile.
template <int NT, int NS>
__device__ __noinline__ void shrink_if_above(uint64_t* buf, uint64_t* scratch, int limit, int kk, int max_keep, SelectShared* ss,
                                int bar, int gtid) {
  const int n = static_cast<int>(ss->n);
  if (n <= limit || n <= kk) return;
  uint64_t T = 0;
  int m = 0;
  if (max_keep > kk) T = cut_sampled<NT, NS>(buf, n, kk, max_keep, scratch, &m, ss, bar, gtid);
  if (T == 0) {
    T = select_kth<NT>(buf, n, kk, max_keep, ss, bar, gtid);
    m = compact_ge<NT>(buf, n, T, scratch, max_keep, ss, bar, gtid);
  }
  if (gtid == 0) {
    ss->n = static_cast<uint32_t>(m);
    ss->tau = T ? T - 1 : 0;  // admit keys > T - 1, i.e. >= T; later keys are new (distinct)
  }
  named_bar_sync(bar, NT);
}

// shrink_if_above for a buffer of at most KPT * NT keys: the histogram cut in
// registers, with the exact radix selection as its fallback.
template <int NT, int KPT, int NB = 256>
__device__ __noinline__ void shrink_if_above_reg(uint64_t* buf, uint64_t* scratch, int limit, int kk, int max_keep,
                                                 SelectShared* ss, int bar, int gtid) {
  const int n = static_cast<int>(ss->n);
  if (n <= limit || n <= kk) return;
  if (!cut_hist<NT, KPT, NB>(buf, n, kk, max_keep, ss, bar, gtid)) {
    const uint64_t T = select_kth<NT>(buf, n, kk, max_keep, ss, bar, gtid);
    const int m = compact_ge<NT>(buf, n, T, scratch, max_keep, ss, bar, gtid);
    if (gtid == 0) {
      ss->n = static_cast<uint32_t>(m);
      ss->tau = T ? T - 1 : 0;
    }
  }
  named_bar_sync(bar, NT);
}

// Sorts keys[0, m) in descending order; m is a power of two.
template <int NT>
__device__ void bitonic_sort_desc(uint64_t* keys, int m, int bar, int gtid) {
  for (int size = 2; size <= m; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = gtid; t < (m >> 1); t += NT) {
        const int lo = 2 * t - (t & (stride - 1));
        const int hi = lo + stride;
        const uint64_t a = keys[lo], b = keys[hi];
        const bool desc = (lo & size) == 0;
        if (desc ? (a < b) : (a > b)) {
          keys[lo] = b;
          keys[hi] = a;
        }
      }
      named_bar_sync(bar, NT);
    }
  }
}

// Orders (a, b) descending when desc, ascending otherwise.
__device__ __forceinline__ void cex(uint64_t& a, uint64_t& b, bool desc) {
  if (desc ? (a < b) : (a > b)) {
    const uint64_t x = a;
    a = b;
    b = x;
  }
}

// Bitonic sort of keys[0, m) into descending order, E consecutive keys per
// thread in registers (the first m / E threads, whole warps): strides below E
// inside a thread, strides from E to 16E by shuffles within the warp, longer
// strides through shared memory with one barrier each. m is a power of two,
// 32E <= m <= E * NT.
template <int NT, int E>
__device__ void sort_regs_desc(uint64_t* keys, int m, int bar, int gtid) {
  const int t = gtid;
  const bool act = t < m / E;
  uint64_t v[E];
#pragma unroll
  for (int i = 0; i < E; ++i) v[i] = act ? keys[E * t + i] : 0ull;
  for (int size = 2; size <= m; size <<= 1) {
    int st = size >> 1;
    if (st >= 32 * E) {
      if (act) {
#pragma unroll
        for (int i = 0; i < E; ++i) keys[E * t + i] = v[i];
      }
      named_bar_sync(bar, NT);
      for (; st >= 32 * E; st >>= 1) {
        for (int u = t; u < (m >> 1); u += NT) {
          const int lo = 2 * u - (u & (st - 1));
          uint64_t x = keys[lo], y = keys[lo + st];
          cex(x, y, (lo & size) == 0);
          keys[lo] = x;
          keys[lo + st] = y;
        }
        named_bar_sync(bar, NT);
      }
      if (act) {
#pragma unroll
        for (int i = 0; i < E; ++i) v[i] = keys[E * t + i];
      }
    }
    for (; st >= E; st >>= 1) {  // partner thread t ^ (st / E), same warp
      const int ts = st / E;
      const bool keep_max = ((t & ts) == 0) == (((E * t) & size) == 0);
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const uint64_t pv = __shfl_xor_sync(0xFFFFFFFFu, v[i], ts);
        v[i] = keep_max ? (v[i] > pv ? v[i] : pv) : (v[i] < pv ? v[i] : pv);
      }
    }
#pragma unroll
    for (int sc = E / 2; sc > 0; sc >>= 1) {  // inside the thread
      if (sc <= st) {
#pragma unroll
        for (int i = 0; i < E; ++i)
          if ((i & sc) == 0) cex(v[i], v[i + sc], (((E * t + i) & size) == 0));
      }
    }
  }
  if (act) {
#pragma unroll
    for (int i = 0; i < E; ++i) keys[E * t + i] = v[i];
  }
  named_bar_sync(bar, NT);
}

// Sorts keys[0, n) into descending order by rank: the keys are counted into NB
// bins of equal width over their value words (bin 0 the highest), scattered by
// bin into tmp (n entries), and each key's place is its bin's offset plus the
// number of keys of its bin that order before it (greater, or equal and
// scattered earlier). A few barriers instead of a sorting network's dependent
// stages; a bin's keys compare only among themselves. Returns false, having
// moved nothing, when some bin holds more than kRankCrowd keys (many equal or
// nearly equal values), where a sorting network is cheaper. hist and cur are
// NB-entry arrays (after the scatter, cur is each bin's end), red holds
// 2 * NT / 32 words.
constexpr int kRankCrowd = 48;
template <int NT, int NB>
__device__ bool rank_sort_desc(uint64_t* keys, int n, uint64_t* tmp, uint32_t* hist, uint32_t* cur, uint32_t* red,
                               int bar, int gtid) {
  static_assert(NB % NT == 0 && NT % 32 == 0, "whole bins per thread");
  constexpr int NW = NT / 32, BPT = NB / NT;
  const int lane = gtid & 31, warp = gtid >> 5;
  uint32_t lo = 0xFFFFFFFFu, hi = 0;
  for (int i = gtid; i < n; i += NT) {
    const uint32_t v = static_cast<uint32_t>(keys[i] >> 32);
    lo = min(lo, v);
    hi = max(hi, v);
  }
  lo = __reduce_min_sync(0xFFFFFFFFu, lo);
  hi = __reduce_max_sync(0xFFFFFFFFu, hi);
  if (lane == 0) {
    red[warp] = lo;
    red[NW + warp] = hi;
  }
#pragma unroll
  for (int j = 0; j < BPT; ++j) hist[BPT * gtid + j] = 0;
  named_bar_sync(bar, NT);
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    lo = min(lo, red[w]);
    hi = max(hi, red[NW + w]);
  }
  constexpr int kBits = NB == 256 ? 8 : NB == 512 ? 9 : NB == 1024 ? 10 : 11;
  static_assert(NB == (1 << kBits), "NB is 256, 512, 1024 or 2048");
  const int s = hi > lo ? max(0, 32 - kBits - __clz(hi - lo)) : 0;  // (hi - lo) >> s < NB
  auto bin_of = [&](uint64_t key) {
    return static_cast<uint32_t>(NB - 1) - ((static_cast<uint32_t>(key >> 32) - lo) >> s);
  };
  for (int i = gtid; i < n; i += NT) atomicAdd(&hist[bin_of(keys[i])], 1u);
  named_bar_sync(bar, NT);
  // exclusive scan over the bins (highest values first) and the fullest bin
  uint32_t c[BPT], sum = 0, most = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    c[j] = hist[BPT * gtid + j];
    sum += c[j];
    most = max(most, c[j]);
  }
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += x;
  }
  most = __reduce_max_sync(0xFFFFFFFFu, most);
  if (lane == 31) red[warp] = incl;  // lo and hi were read before the last barrier
  if (lane == 0) red[NW + warp] = most;
  named_bar_sync(bar, NT);
  uint32_t before = 0;
  most = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    before += w < warp ? red[w] : 0u;
    most = max(most, red[NW + w]);
  }
  if (most > static_cast<uint32_t>(kRankCrowd)) return false;  // uniform
  uint32_t run = before + incl - sum;
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    cur[BPT * gtid + j] = run;
    run += c[j];
  }
  named_bar_sync(bar, NT);
  for (int i = gtid; i < n; i += NT) {
    const uint64_t key = keys[i];
    tmp[atomicAdd(&cur[bin_of(key)], 1u)] = key;
  }
  named_bar_sync(bar, NT);
  for (int p = gtid; p < n; p += NT) {
    const uint64_t key = tmp[p];
    const uint32_t d = bin_of(key), b1 = cur[d], b0 = b1 - hist[d];
    uint32_t r = 0;
#pragma unroll 4
    for (uint32_t j = b0; j < b1; ++j) {
      const uint64_t o = tmp[j];
      r += (o > key || (o == key && j < static_cast<uint32_t>(p))) ? 1u : 0u;
    }
    keys[b0 + r] = key;
  }
  named_bar_sync(bar, NT);
  return true;
}

// Sorts keys[0, n) in descending order in place; keys[n, m) are overwritten with
// zero padding, where m is the power of two >= max(n, 64) (the buffer must hold
// m keys). Up to 8 * NT keys are sorted in registers (sort_regs_desc).
template <int NT>
__device__ void sort_prefix_desc(uint64_t* keys, int n, int bar, int gtid) {
  int m = 64;
  while (m < n) m <<= 1;
  for (int j = n + gtid; j < m; j += NT) keys[j] = 0ull;
  named_bar_sync(bar, NT);
  if (m <= 2 * NT)
    sort_regs_desc<NT, 2>(keys, m, bar, gtid);
  else if (m <= 4 * NT)
    sort_regs_desc<NT, 4>(keys, m, bar, gtid);
  else if (m <= 8 * NT)
    sort_regs_desc<NT, 8>(keys, m, bar, gtid);
  else
    bitonic_sort_desc<NT>(keys, m, bar, gtid);
}

}  // namespace csa
