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
struct SelectShared {
  uint32_t hist[256];
  uint32_t bcast[4];
  uint32_t gather;    // compaction cursor
  uint32_t n;         // live candidates in the buffer
  uint64_t tau;       // admission threshold: a key must exceed it
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
// (more only if the caller broke the distinct-key precondition).
template <int NT>
__device__ int compact_ge(uint64_t* keys, int n, uint64_t T, uint64_t* scratch, int cap, SelectShared* ss,
                          int bar, int gtid) {
  if (gtid == 0) ss->gather = 0;
  named_bar_sync(bar, NT);
  for (int i = gtid; i < n; i += NT) {
    const uint64_t key = keys[i];
    if (key >= T) {
      const uint32_t p = atomicAdd(&ss->gather, 1u);
      if (p < static_cast<uint32_t>(cap)) scratch[p] = key;
    }
  }
  named_bar_sync(bar, NT);
  const int m = min(static_cast<int>(ss->gather), cap);
  for (int i = gtid; i < m; i += NT) keys[i] = scratch[i];
  named_bar_sync(bar, NT);
  return m;
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
// be among the kk best. Group-uniform.
template <int NT>
__device__ void shrink_if_above(uint64_t* buf, uint64_t* scratch, int limit, int kk, int max_keep, SelectShared* ss,
                                int bar, int gtid) {
  const int n = static_cast<int>(ss->n);
  if (n <= limit || n <= kk) return;
  const uint64_t T = select_kth<NT>(buf, n, kk, max_keep, ss, bar, gtid);
  const int m = compact_ge<NT>(buf, n, T, scratch, max_keep, ss, bar, gtid);
  if (gtid == 0) {
    ss->n = static_cast<uint32_t>(m);
    ss->tau = T ? T - 1 : 0;  // admit keys > T - 1, i.e. >= T; later keys are new (distinct)
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

}  // namespace csa
