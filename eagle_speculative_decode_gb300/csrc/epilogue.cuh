// Device code shared by the CUDA-core GEMV (gemv.cu) and the tensor-core GEMM
// (gemm_tc.cu): logical row maps, warp reductions, activation staging and the fused
// epilogues of every projection mode.
#pragma once

#include <math.h>

#include "common.cuh"

namespace e3 {

// Weight matrix (0: w0, 1: w1, 2: w2) and row of logical row lr of a mode.
struct RowRef {
  int m;
  size_t row;
};

template <int MODE>
__device__ __forceinline__ RowRef row_ref(const GemvParams &p, int lr) {
  if constexpr (MODE == GM_GATEUP) {
    return {lr & 1, (size_t)(lr >> 1)};
  } else if constexpr (MODE == GM_QKV) {
    const int d = p.head_dim, R = p.rope_dims;
    const int qr = p.n_head * d, kr = p.n_head_kv * d;
    if (lr < qr + kr) {
      const bool isq = lr < qr;
      const int rr = isq ? lr : lr - qr;
      const int head = rr / d, li = rr - head * d;
      // RoPE partners (i, i + R/2) sit on adjacent logical rows 2i, 2i + 1.
      const int dim = li < R ? ((li & 1) ? (li >> 1) + (R >> 1) : (li >> 1)) : li;
      return {isq ? 0 : 1, (size_t)head * d + dim};
    }
    return {2, (size_t)(lr - qr - kr)};
  } else {
    return {0, (size_t)lr};
  }
}

__device__ __forceinline__ const uint16_t *bf16_row(const GemvParams &p, RowRef r) {
  const uint16_t *base = r.m == 0 ? p.w0 : (r.m == 1 ? p.w1 : p.w2);
  return base + r.row * (size_t)p.K;
}

// INT4 weights: w0..w2 hold the packed codes, sz0..sz2 the (scale, zero) rows.
__device__ __forceinline__ const unsigned char *q4_codes(const GemvParams &p, RowRef r) {
  const uint16_t *base = r.m == 0 ? p.w0 : (r.m == 1 ? p.w1 : p.w2);
  return reinterpret_cast<const unsigned char *>(base) + r.row * (size_t)(p.K >> 1);
}

__device__ __forceinline__ const uint32_t *q4_sz(const GemvParams &p, RowRef r) {
  const uint32_t *base = r.m == 0 ? p.sz0 : (r.m == 1 ? p.sz1 : p.sz2);
  return base + r.row * (size_t)p.sz_stride;
}

template <int N>
struct Log2 {
  static constexpr int value = (N >= 32) ? 5 : (N >= 16) ? 4 : (N >= 8) ? 3 : (N >= 4) ? 2 : (N >= 2) ? 1 : 0;
};

// Reduce N = 2^S values held by every lane across the warp.  Afterwards lane l holds
// the warp total of value index idx(l) = bits 4..(5-S) of l read as an S-bit number;
// lanes whose low (5-S) bits are zero are the designated writers.
template <int N>
__device__ __forceinline__ float warp_reduce_multi(float (&v)[N], int lane) {
  static_assert(N >= 1 && N <= 32 && (N & (N - 1)) == 0, "1..32 values, a power of two");
#pragma unroll
  for (int cnt = N, o = 16; cnt > 1; cnt >>= 1, o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < cnt / 2; ++i) {
      const float send = upper ? v[i] : v[i + cnt / 2];
      const float keep = upper ? v[i + cnt / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float r = v[0];
#pragma unroll
  for (int o = 16 >> Log2<N>::value; o >= 1; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  return r;
}

template <int N>
__device__ __forceinline__ int warp_reduce_index(int lane) {
  int idx = 0;
#pragma unroll
  for (int s = 0; s < Log2<N>::value; ++s) idx = (idx << 1) | ((lane >> (4 - s)) & 1);
  return idx;
}

template <int N>
__device__ __forceinline__ bool warp_reduce_writer(int lane) {
  return (lane & ((1 << (5 - Log2<N>::value)) - 1)) == 0;
}

// ------------------------------------------------------------------ x staging
template <int MODE>
struct ModeTraits {
  static constexpr bool kBf16X = MODE == GM_ENCODE;  // x kept as the caller's bf16
  static constexpr int kHalves = MODE == GM_QKV ? 2 : 1;  // separately normalised K halves
  static constexpr bool kNorm = MODE == GM_QKV || MODE == GM_GATEUP || MODE == GM_LMHEAD;
  static constexpr int kUnit = (MODE == GM_QKV || MODE == GM_GATEUP) ? 2 : 1;  // row pairing
};

__device__ __forceinline__ float sq8(float4 a, float4 b) {
  return a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w + b.x * b.x + b.y * b.y + b.z * b.z +
         b.w * b.w;
}
__device__ __forceinline__ float4 mul4(float4 a, float w0, float w1, float w2, float w3) {
  return make_float4(a.x * w0, a.y * w1, a.z * w2, a.w * w3);
}

// Writes x[m, k] (times the norm gain where the op normalises) into shared memory and
// accumulates this thread's share of sum(x^2) per item and K half into ss.
template <int NB, int MODE>
__device__ void stage_x(const GemvParams &p, unsigned char *xmem, float (&ss)[NB][ModeTraits<MODE>::kHalves]) {
  using T = ModeTraits<MODE>;
  const int K = p.K, KV = K >> 3, tid = threadIdx.x;
#pragma unroll
  for (int m = 0; m < NB; ++m)
#pragma unroll
    for (int h = 0; h < T::kHalves; ++h) ss[m][h] = 0.f;
  for (int m = 0; m < NB; ++m) {
    const bool live = m < p.items;
    const int item = p.item0 + m;
    if constexpr (T::kBf16X) {
      uint4 *xb = reinterpret_cast<uint4 *>(xmem) + (size_t)m * KV;
      const uint4 *src = reinterpret_cast<const uint4 *>(p.xb + (size_t)item * K);
      for (int kv = tid; kv < KV; kv += kGemvThreads) xb[kv] = live ? src[kv] : make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    float4 *x0 = reinterpret_cast<float4 *>(xmem) + (size_t)(m * 2) * KV;
    float4 *x1 = x0 + KV;
    if (!live) {
      for (int kv = tid; kv < KV; kv += kGemvThreads) {
        x0[kv] = make_float4(0.f, 0.f, 0.f, 0.f);
        x1[kv] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      continue;
    }
    // up to VU vectors of a thread are loaded before any of them is stored, so that their
    // round trips overlap (K = 12288 gives each thread three)
    constexpr int VU = 3;
    if constexpr (MODE == GM_O || MODE == GM_DOWN) {
      const float4 *src = reinterpret_cast<const float4 *>(p.xf + (size_t)item * K);
      for (int kv0 = tid; kv0 < KV; kv0 += VU * kGemvThreads) {
        float4 a[VU], b[VU];
#pragma unroll
        for (int u = 0; u < VU; ++u) {
          const int kv = kv0 + u * kGemvThreads;
          if (kv < KV) {
            a[u] = src[2 * kv];
            b[u] = src[2 * kv + 1];
          }
        }
#pragma unroll
        for (int u = 0; u < VU; ++u) {
          const int kv = kv0 + u * kGemvThreads;
          if (kv < KV) {
            x0[kv] = a[u];
            x1[kv] = b[u];
          }
        }
      }
    } else if constexpr (MODE == GM_GATEUP || MODE == GM_LMHEAD) {
      const float4 *src = reinterpret_cast<const float4 *>(p.xf + (size_t)item * K);
      const uint4 *wn = reinterpret_cast<const uint4 *>(p.norm0);
      for (int kv0 = tid; kv0 < KV; kv0 += VU * kGemvThreads) {
        float4 a[VU], b[VU];
        uint4 w[VU];
#pragma unroll
        for (int u = 0; u < VU; ++u) {
          const int kv = kv0 + u * kGemvThreads;
          if (kv < KV) {
            a[u] = src[2 * kv];
            b[u] = src[2 * kv + 1];
            w[u] = wn[kv];
          }
        }
#pragma unroll
        for (int u = 0; u < VU; ++u) {
          const int kv = kv0 + u * kGemvThreads;
          if (kv < KV) {
            ss[m][0] += sq8(a[u], b[u]);
            x0[kv] = mul4(a[u], bf_lo(w[u].x), bf_hi(w[u].x), bf_lo(w[u].y), bf_hi(w[u].y));
            x1[kv] = mul4(b[u], bf_lo(w[u].z), bf_hi(w[u].z), bf_lo(w[u].w), bf_hi(w[u].w));
          }
        }
      }
    }
  }
  if constexpr (MODE == GM_QKV) {
    // [embed(tok) * w_in ; g * w_hid]; the two RMSNorm scales come later.  An item's
    // embedding row is known only once its token is loaded, so the pairs of a group of
    // items are resolved together and every global load of the group is issued before any
    // shared-memory store: two dependent round trips per group instead of several per item.
    const int n = p.n_embd, NV = n >> 3;
    constexpr int MB = NB < 4 ? NB : 4;
    const uint4 *wi = reinterpret_cast<const uint4 *>(p.norm0);
    const uint4 *wh = reinterpret_cast<const uint4 *>(p.norm1);
#pragma unroll
    for (int m0 = 0; m0 < NB; m0 += MB) {
      const uint4 *er[MB];
      const float4 *gr[MB];
#pragma unroll
      for (int mm = 0; mm < MB; ++mm) {
        const int m = m0 + mm;
        er[mm] = nullptr;
        gr[mm] = nullptr;
        if (m < p.items) {
          const PairItem it = resolve_pair(p.pairs, p.item0 + m, n);
          int tok = it.tok;
          if (tok < 0 || tok >= p.target_vocab) {
            // only rows whose K/V are kept (or the chain's q) may report a bad token
            if (tid == 0 && (it.write_kv || p.row_base == 0)) set_status(p.status, EAGLE3_DEV_BAD_TOKEN);
            tok = 0;
          }
          er[mm] = reinterpret_cast<const uint4 *>(p.embed + (size_t)tok * n);
          gr[mm] = reinterpret_cast<const float4 *>(it.g);
        }
      }
      for (int kv = tid; kv < NV; kv += kGemvThreads) {
        uint4 u[MB];
        float4 a[MB], b[MB];
#pragma unroll
        for (int mm = 0; mm < MB; ++mm) {
          if (er[mm]) {
            u[mm] = er[mm][kv];
            a[mm] = gr[mm][2 * kv];
            b[mm] = gr[mm][2 * kv + 1];
          }
        }
        const uint4 w = wi[kv], hw = wh[kv];
#pragma unroll
        for (int mm = 0; mm < MB; ++mm) {
          const int m = m0 + mm;
          if (!er[mm]) continue;
          float4 *x0 = reinterpret_cast<float4 *>(xmem) + (size_t)(m * 2) * KV;
          float4 *x1 = x0 + KV;
          const float4 ea = make_float4(bf_lo(u[mm].x), bf_hi(u[mm].x), bf_lo(u[mm].y), bf_hi(u[mm].y));
          const float4 eb = make_float4(bf_lo(u[mm].z), bf_hi(u[mm].z), bf_lo(u[mm].w), bf_hi(u[mm].w));
          ss[m][0] += sq8(ea, eb);
          x0[kv] = mul4(ea, bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y));
          x1[kv] = mul4(eb, bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w));
          ss[m][T::kHalves - 1] += sq8(a[mm], b[mm]);
          x0[NV + kv] = mul4(a[mm], bf_lo(hw.x), bf_hi(hw.x), bf_lo(hw.y), bf_hi(hw.y));
          x1[NV + kv] = mul4(b[mm], bf_lo(hw.z), bf_hi(hw.z), bf_lo(hw.w), bf_hi(hw.w));
        }
      }
    }
  }
}

// The x vectors this thread uses, k = 8 (tid + kGemvThreads j) for j < XRV, computed
// straight into registers (the launches whose x fits there keep no copy of x in shared
// memory, which leaves the whole ring budget to the weights); the same values and RMSNorm
// sums as stage_x.  All global loads of the thread are issued before any use.
template <int NB, int MODE, int XRV>
__device__ __forceinline__ void stage_x_regs(const GemvParams &p, float (&xr)[XRV][NB][8],
                                             float (&ss)[NB][ModeTraits<MODE>::kHalves]) {
  using T = ModeTraits<MODE>;
  constexpr int H = T::kHalves;
  const int K = p.K, KV = K >> 3, tid = threadIdx.x;
#pragma unroll
  for (int m = 0; m < NB; ++m)
#pragma unroll
    for (int h = 0; h < H; ++h) ss[m][h] = 0.f;
  if constexpr (MODE == GM_QKV) {
    // [embed(tok) * w_in ; g * w_hid]: e vectors kv < NV, g vectors kv >= NV
    const int n = p.n_embd, NV = n >> 3;
    const uint4 *er[NB];
    const float4 *gr[NB];
#pragma unroll
    for (int m = 0; m < NB; ++m) {
      er[m] = nullptr;
      gr[m] = nullptr;
      if (m < p.items) {
        const PairItem it = resolve_pair(p.pairs, p.item0 + m, n);
        int tok = it.tok;
        if (tok < 0 || tok >= p.target_vocab) {
          // only rows whose K/V are kept (or the chain's q) may report a bad token
          if (tid == 0 && (it.write_kv || p.row_base == 0)) set_status(p.status, EAGLE3_DEV_BAD_TOKEN);
          tok = 0;
        }
        er[m] = reinterpret_cast<const uint4 *>(p.embed + (size_t)tok * n);
        gr[m] = reinterpret_cast<const float4 *>(it.g);
      }
    }
    const uint4 *wi = reinterpret_cast<const uint4 *>(p.norm0);
    const uint4 *wh = reinterpret_cast<const uint4 *>(p.norm1);
#pragma unroll
    for (int j = 0; j < XRV; ++j) {
      const int kv = tid + j * kGemvThreads;
#pragma unroll
      for (int m = 0; m < NB; ++m) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
        if (kv < KV && er[m]) {
          if (kv < NV) {
            const uint4 u = er[m][kv];
            a = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
          } else {
            a = gr[m][2 * (kv - NV)];
            b = gr[m][2 * (kv - NV) + 1];
          }
        }
        xr[j][m][0] = a.x; xr[j][m][1] = a.y; xr[j][m][2] = a.z; xr[j][m][3] = a.w;
        xr[j][m][4] = b.x; xr[j][m][5] = b.y; xr[j][m][6] = b.z; xr[j][m][7] = b.w;
      }
    }
#pragma unroll
    for (int j = 0; j < XRV; ++j) {
      const int kv = tid + j * kGemvThreads;
      const bool eh = kv < NV;
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (kv < KV) w = eh ? wi[kv] : wh[kv - NV];
#pragma unroll
      for (int m = 0; m < NB; ++m) {
        float4 a, b;
        if (eh) {
          const uint32_t u0 = __float_as_uint(xr[j][m][0]), u1 = __float_as_uint(xr[j][m][1]);
          const uint32_t u2 = __float_as_uint(xr[j][m][2]), u3 = __float_as_uint(xr[j][m][3]);
          a = make_float4(bf_lo(u0), bf_hi(u0), bf_lo(u1), bf_hi(u1));
          b = make_float4(bf_lo(u2), bf_hi(u2), bf_lo(u3), bf_hi(u3));
        } else {
          a = make_float4(xr[j][m][0], xr[j][m][1], xr[j][m][2], xr[j][m][3]);
          b = make_float4(xr[j][m][4], xr[j][m][5], xr[j][m][6], xr[j][m][7]);
        }
        if (kv < KV) ss[m][eh ? 0 : H - 1] += sq8(a, b);
        const float4 xa = mul4(a, bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y));
        const float4 xb = mul4(b, bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w));
        xr[j][m][0] = xa.x; xr[j][m][1] = xa.y; xr[j][m][2] = xa.z; xr[j][m][3] = xa.w;
        xr[j][m][4] = xb.x; xr[j][m][5] = xb.y; xr[j][m][6] = xb.z; xr[j][m][7] = xb.w;
      }
    }
  } else if constexpr (T::kBf16X) {
    // the encode: the caller's bf16 features as they are
#pragma unroll
    for (int j = 0; j < XRV; ++j) {
      const int kv = tid + j * kGemvThreads;
#pragma unroll
      for (int m = 0; m < NB; ++m) {
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if (kv < KV && m < p.items) u = reinterpret_cast<const uint4 *>(p.xb + (size_t)(p.item0 + m) * K)[kv];
        xr[j][m][0] = bf_lo(u.x); xr[j][m][1] = bf_hi(u.x); xr[j][m][2] = bf_lo(u.y); xr[j][m][3] = bf_hi(u.y);
        xr[j][m][4] = bf_lo(u.z); xr[j][m][5] = bf_hi(u.z); xr[j][m][6] = bf_lo(u.w); xr[j][m][7] = bf_hi(u.w);
      }
    }
  } else {
    // float32 activations: attention output / act as they are, x1 / gsum times the norm gain
    constexpr bool kNormed = MODE == GM_GATEUP || MODE == GM_LMHEAD;
#pragma unroll
    for (int j = 0; j < XRV; ++j) {
      const int kv = tid + j * kGemvThreads;
#pragma unroll
      for (int m = 0; m < NB; ++m) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
        if (kv < KV && m < p.items) {
          const float4 *src = reinterpret_cast<const float4 *>(p.xf + (size_t)(p.item0 + m) * K);
          a = __ldcg(src + 2 * kv);
          b = __ldcg(src + 2 * kv + 1);
        }
        xr[j][m][0] = a.x; xr[j][m][1] = a.y; xr[j][m][2] = a.z; xr[j][m][3] = a.w;
        xr[j][m][4] = b.x; xr[j][m][5] = b.y; xr[j][m][6] = b.z; xr[j][m][7] = b.w;
      }
    }
    if constexpr (kNormed) {
      const uint4 *wn = reinterpret_cast<const uint4 *>(p.norm0);
#pragma unroll
      for (int j = 0; j < XRV; ++j) {
        const int kv = tid + j * kGemvThreads;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (kv < KV) w = wn[kv];
#pragma unroll
        for (int m = 0; m < NB; ++m) {
          const float4 a = make_float4(xr[j][m][0], xr[j][m][1], xr[j][m][2], xr[j][m][3]);
          const float4 b = make_float4(xr[j][m][4], xr[j][m][5], xr[j][m][6], xr[j][m][7]);
          ss[m][0] += sq8(a, b);
          const float4 xa = mul4(a, bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y));
          const float4 xb = mul4(b, bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w));
          xr[j][m][0] = xa.x; xr[j][m][1] = xa.y; xr[j][m][2] = xa.z; xr[j][m][3] = xa.w;
          xr[j][m][4] = xb.x; xr[j][m][5] = xb.y; xr[j][m][6] = xb.z; xr[j][m][7] = xb.w;
        }
      }
    }
  }
}

// x vector kv of item m as 8 floats.
template <int MODE>
__device__ __forceinline__ void load_x8(const unsigned char *xmem, int KV, int m, int kv, float (&x)[8]) {
  if constexpr (ModeTraits<MODE>::kBf16X) {
    const uint4 u = reinterpret_cast<const uint4 *>(xmem)[(size_t)m * KV + kv];
    x[0] = bf_lo(u.x); x[1] = bf_hi(u.x); x[2] = bf_lo(u.y); x[3] = bf_hi(u.y);
    x[4] = bf_lo(u.z); x[5] = bf_hi(u.z); x[6] = bf_lo(u.w); x[7] = bf_hi(u.w);
  } else {
    const float4 *xs = reinterpret_cast<const float4 *>(xmem);
    const float4 a = xs[(size_t)(m * 2) * KV + kv], b = xs[(size_t)(m * 2 + 1) * KV + kv];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

__device__ __forceinline__ float dot8(const uint4 w, const float (&x)[8], float a) {
  a = fmaf(bf_lo(w.x), x[0], a); a = fmaf(bf_hi(w.x), x[1], a);
  a = fmaf(bf_lo(w.y), x[2], a); a = fmaf(bf_hi(w.y), x[3], a);
  a = fmaf(bf_lo(w.z), x[4], a); a = fmaf(bf_hi(w.z), x[5], a);
  a = fmaf(bf_lo(w.w), x[6], a); a = fmaf(bf_hi(w.w), x[7], a);
  return a;
}

// ---------------------------------------------------------------- epilogues
__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

// Last CTA of an lm_head launch: decode each item's winning (logit, row) key, map the
// draft id through d2t and write the step's tokens; the slots are left at zero.
__device__ __forceinline__ void lmhead_finalize(const GemvParams &p, int item0, int items, int tid,
                                                int nthreads) {
  for (int m = tid; m < items; m += nthreads) {
    const int item = item0 + m;
    const unsigned long long key = atomicExch(p.am_slot + item, 0ull);
    uint32_t id;
    long long tgt;  // no d2t: the draft ids are target ids
    const bool bad = !argmax_ids(key, p.d2t, p.draft_vocab, p.target_vocab, id, tgt);
    if (bad) set_status(p.status, EAGLE3_DEV_BAD_TOKEN);
    // without a status word (the context-free entry point) the row itself carries the error
    const bool valid = (!p.gamma_eff || p.step < p.gamma_eff[item]) && !(bad && !p.status);
    const size_t o = (size_t)item * p.gamma + p.step;
    p.draft_tok[o] = valid ? (int32_t)tgt : -1;
    if (p.draft_id) p.draft_id[o] = valid ? (int32_t)id : -1;
    if (p.next_tok) p.next_tok[item] = (int32_t)tgt;
  }
}

// Row stride (floats) of the accumulator tile accs[row][item].  Wide tiles (the tensor-core
// GEMM) pad it to an odd stride so that walking rows hits distinct banks; they also walk
// rows fastest so that the global writes of one item are contiguous.
template <int NB>
struct AccStride {
  static constexpr int value = NB >= 16 ? NB + 1 : NB;
  static constexpr bool kRowsFast = NB >= 16;
};

// Global row of local row r: tiles of TR rows dealt round robin over the CTAs.
template <int TR>
__device__ __forceinline__ int tile_row(int r) {
  return ((r / TR) * (int)gridDim.x + (int)blockIdx.x) * TR + (r % TR);
}

template <int NB, int MODE, int TR>
__device__ void epilogue(const GemvParams &p, const float *accs, int nrows) {
  const int tid = threadIdx.x;
  constexpr int AS = AccStride<NB>::value;
  constexpr bool kRowsFast = AccStride<NB>::kRowsFast;
  const int live = p.items < NB ? p.items : NB;
  if constexpr (MODE == GM_ENCODE || MODE == GM_O || MODE == GM_DOWN) {
    for (int idx = tid; idx < nrows * NB; idx += kGemvThreads) {
      const int m = kRowsFast ? idx / nrows : idx % NB, r = kRowsFast ? idx % nrows : idx / NB;
      if (m >= live) {
        if (kRowsFast) break;
        continue;
      }
      const int item = p.item0 + m, row = tile_row<TR>(r);
      float v = accs[r * AS + m];
      if constexpr (MODE != GM_ENCODE) v += p.res[(size_t)item * p.rows + row];
      p.out_f[(size_t)item * p.rows + row] = v;
      if constexpr (MODE == GM_DOWN) {
        if (p.dbg_f) p.dbg_f[(size_t)item * p.dbg_stride_b + p.dbg_off + row] = v;
      }
    }
  } else if constexpr (MODE == GM_GATEUP) {
    const int npairs = nrows >> 1;
    for (int idx = tid; idx < npairs * NB; idx += kGemvThreads) {
      const int m = kRowsFast ? idx / npairs : idx % NB, pr = kRowsFast ? idx % npairs : idx / NB;
      if (m >= live) {
        if (kRowsFast) break;
        continue;
      }
      const int item = p.item0 + m;
      const float gate = accs[(2 * pr) * AS + m], up = accs[(2 * pr + 1) * AS + m];
      p.out_f[(size_t)item * p.n_ff + (tile_row<TR>(2 * pr) >> 1)] = silu_f(gate) * up;
    }
  } else if constexpr (MODE == GM_QKV) {
    const int d = p.head_dim, R = p.rope_dims, half = R >> 1;
    const int qr = p.n_head * d, kr = p.n_head_kv * d;
    const int npairs = nrows >> 1;
    for (int idx = tid; idx < npairs * NB; idx += kGemvThreads) {
      const int m = kRowsFast ? idx / npairs : idx % NB, pr = kRowsFast ? idx % npairs : idx / NB;
      if (m >= live) {
        if (kRowsFast) break;
        continue;
      }
      const int item = p.item0 + m;
      const int lr = p.row_base + tile_row<TR>(2 * pr);  // even logical row
      float a = accs[(2 * pr) * AS + m], b = accs[(2 * pr + 1) * AS + m];
      const PairItem it = resolve_pair(p.pairs, item, p.n_embd);
      const int region = lr < qr ? 0 : (lr < qr + kr ? 1 : 2);
      const int rr = region == 0 ? lr : (region == 1 ? lr - qr : lr - qr - kr);
      const int head = rr / d, li = rr - head * d;
      int dim0 = li, dim1 = li + 1;
      if (region < 2 && li < R) {
        dim0 = li >> 1;
        dim1 = dim0 + half;
        int pos = it.pos;
        if (pos < 0 || pos >= p.max_cache_len) pos = 0;
        const float2 cs = p.rope[(size_t)pos * half + dim0];
        const float ra = a * cs.x - b * cs.y;
        const float rb = b * cs.x + a * cs.y;
        a = ra;
        b = rb;
      }
      if (region == 0) {
        float *q = p.out_f + (size_t)item * qr + (size_t)head * d;
        q[dim0] = a;
        q[dim1] = b;
      } else if (it.write_kv && p.kv_stage) {
        // quantized KV: float32 into the staging buffer, kv_quant writes the blocks
        float *stg = p.kv_stage + ((size_t)item * 2 + (region - 1)) * kr + (size_t)head * d;
        stg[dim0] = a;
        stg[dim1] = b;
      } else if (it.write_kv) {
        const int pos = it.pos;
        if (pos < 0 || pos >= p.max_cache_len) {
          set_status(p.status, EAGLE3_DEV_BAD_POSITION);
          continue;
        }
        const int pg = p.page_table[(size_t)it.b * p.max_pages + pos / p.page_size];
        if (pg < 0 || pg >= p.num_pages) {
          set_status(p.status, EAGLE3_DEV_BAD_PAGE);
          continue;
        }
        uint16_t *pool = region == 1 ? p.k_pool : p.v_pool;
        uint16_t *dst = pool + (((size_t)pg * p.n_head_kv + head) * p.page_size + pos % p.page_size) * d;
        dst[dim0] = f2bf(a);
        dst[dim1] = f2bf(b);
      }
    }
  } else if constexpr (MODE == GM_LMHEAD) {
    // Per item: best (logit, lowest row) over this CTA's rows, then a global 64-bit
    // atomicMax of (order key << 32 | ~row); the last CTA decodes and applies d2t.
    __shared__ unsigned long long best_sh[kGemvWarps];
    __shared__ int last_sh;
    if constexpr (kRowsFast) {
      // wide tiles: one warp per item, no block barriers per item
      const int lane = tid & 31;
      for (int m = tid >> 5; m < live; m += kGemvWarps) {
        const int item = p.item0 + m;
        unsigned long long best = 0ull;
        for (int r = lane; r < nrows; r += 32) {
          const float v = accs[r * AS + m];
          const int row = tile_row<TR>(r);
          if (p.dbg_f) p.dbg_f[(size_t)item * p.dbg_stride_b + p.dbg_off + row] = v;
          const unsigned long long key =
              ((unsigned long long)float_order_key(v) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)row);
          best = key > best ? key : best;
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
          const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
          best = other > best ? other : best;
        }
        if (lane == 0 && nrows > 0) atomicMax(p.am_slot + item, best);
      }
      __threadfence();  // every warp's maxima land before this CTA is counted
      consumer_sync();
    }
    for (int m = 0; m < (kRowsFast ? 0 : p.items); ++m) {
      const int item = p.item0 + m;
      unsigned long long best = 0ull;
      for (int r = tid; r < nrows; r += kGemvThreads) {
        const float v = accs[r * AS + m];
        const int row = tile_row<TR>(r);
        if (p.dbg_f) p.dbg_f[(size_t)item * p.dbg_stride_b + p.dbg_off + row] = v;
        const unsigned long long key =
            ((unsigned long long)float_order_key(v) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)row);
        best = key > best ? key : best;
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other > best ? other : best;
      }
      if ((tid & 31) == 0) best_sh[tid >> 5] = best;
      consumer_sync();
      if (tid == 0) {
        unsigned long long b = 0ull;
        for (int w = 0; w < kGemvWarps; ++w) b = best_sh[w] > b ? best_sh[w] : b;
        if (nrows > 0) atomicMax(p.am_slot + item, b);
      }
      consumer_sync();
    }
    // deferred: the launch's completion publishes the maxima to the kernel that decodes them
    if (p.am_defer) return;
    if (tid == 0) {
      __threadfence();
      const unsigned prev = atomicAdd(p.am_count, 1u);
      last_sh = (prev == gridDim.x - 1) ? 1 : 0;
    }
    consumer_sync();
    if (last_sh) {
      __threadfence();
      lmhead_finalize(p, p.item0, p.items, tid, kGemvThreads);
      if (tid == 0) *p.am_count = 0u;
    }
  }
}

}  // namespace e3
