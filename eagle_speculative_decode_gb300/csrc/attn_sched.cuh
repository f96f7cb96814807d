// Work partition shared by the decode attention kernels (attention.cu, attention_tc.cu).
#pragma once
#include "common.cuh"

namespace e3 {

// The unit partition of one launch: pre[b] = units of one kv head of sequences < b (a
// table chain_begin wrote for this step before any later kernel of the round started);
// CTA c owns units [start(c), start(c + 1)) of the Hkv * pre[B] units in (sequence,
// kv head, unit) order.
struct AttnSched {
  const int *pre;
  int B, Hkv, grid;
  long long total;
  __device__ long long start(int c) const { return total * c / grid; }
  __device__ int cta_of(long long u) const {
    int c = (int)(u * grid / total);
    while (c + 1 < grid && start(c + 1) <= u) ++c;
    while (c > 0 && start(c) > u) --c;
    return c;
  }
  // sequence b whose units hold u: the largest b with Hkv * pre[b] <= u
  __device__ int seq_of(long long u) const {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((long long)Hkv * pre[mid] <= u) lo = mid;
      else hi = mid - 1;
    }
    return lo;
  }
};

// A run of units [r0, r1) of pair (b, kvh) inside one CTA's share; pair units nu.
struct AttnSeg {
  int b, kvh, r0, r1, nu;
  long long pair_u0;  // first unit of the pair
};

__device__ __forceinline__ AttnSeg attn_seg(const AttnSched &S, long long u, long long u_end) {
  AttnSeg s;
  s.b = S.seq_of(u);
  s.nu = S.pre[s.b + 1] - S.pre[s.b];
  const long long off = u - (long long)S.Hkv * S.pre[s.b];
  s.kvh = (int)(off / s.nu);
  s.r0 = (int)(off - (long long)s.kvh * s.nu);
  s.pair_u0 = u - s.r0;
  s.r1 = (int)min((long long)s.nu, (long long)s.r0 + (u_end - u));
  return s;
}

}  // namespace e3
