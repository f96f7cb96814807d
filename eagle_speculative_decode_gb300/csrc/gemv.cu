// Weight-streaming GEMV for the drafter's projections at small batch (items <= 8).
//
// y[item, row] = sum_k W[row, k] * x[item, k] with bf16 weights in [out, in] row-major
// and float32 activations/accumulators, fused with the op that feeds x (RMSNorm of the
// layer input, of x1 or of gsum; the embedding gather; the 2n concat) and the op that
// consumes y (partial RoPE + bf16 KV append, residual adds, SwiGLU, argmax + d2t).
// Ops follow "memra_engine/eagle.rs", module doc "Op-sequence".
//
// Data movement (one CTA per SM): the CTA owns a contiguous, balanced range of row
// pairs.  A producer warp streams those rows, SR whole rows per stage (<= 32 KB), with
// bulk copies (cp.async.bulk, TMA) into an NSTAGE-deep shared-memory ring guarded by
// mbarriers.  It starts before the kernel waits on its predecessor (programmatic
// dependent launch), so the next weights are already in flight while the previous
// kernel drains.  Eight consumer warps stage x (normalised where the op says so) in
// shared memory (float32 in two float4 planes -- elements 0-3 and 4-7 of each 8-element
// vector, conflict-free LDS.128 -- or as the caller's bf16 for the encode), then, per
// stage, each thread takes 16-byte vectors k = 8 * (tid + 256 j) of all SR rows, so every
// x vector it loads serves SR rows; single-item launches keep their x vectors in
// registers.  RMSNorm is applied after the dot product: the GEMV runs on x * w_norm and
// the per-item scale 1 / sqrt(mean(x^2) + eps), reduced while x is staged, multiplies the
// row sums, so no block-wide reduction stands between the dependency wait and the first
// FMA.  A stage's per-row sums are reduced within the warp and kept per warp; the eight
// warp partials are added in a fixed order before the epilogue (deterministic).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace e3 {

template <int MODE>
__device__ __forceinline__ const uint16_t *row_ptr(const GemvParams &p, int lr) {
  const size_t K = (size_t)p.K;
  if constexpr (MODE == GM_GATEUP) {
    return ((lr & 1) ? p.w1 : p.w0) + (size_t)(lr >> 1) * K;
  } else if constexpr (MODE == GM_QKV) {
    const int d = p.head_dim, R = p.rope_dims;
    const int qr = p.n_head * d, kr = p.n_head_kv * d;
    if (lr < qr + kr) {
      const bool isq = lr < qr;
      const uint16_t *base = isq ? p.w0 : p.w1;
      const int rr = isq ? lr : lr - qr;
      const int head = rr / d, li = rr - head * d;
      // RoPE partners (i, i + R/2) sit on adjacent logical rows 2i, 2i + 1.
      const int dim = li < R ? ((li & 1) ? (li >> 1) + (R >> 1) : (li >> 1)) : li;
      return base + ((size_t)head * d + dim) * K;
    }
    return p.w2 + (size_t)(lr - qr - kr) * K;
  } else {
    return p.w0 + (size_t)lr * K;
  }
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
    if constexpr (MODE == GM_O || MODE == GM_DOWN) {
      const float4 *src = reinterpret_cast<const float4 *>(p.xf + (size_t)item * K);
      for (int kv = tid; kv < KV; kv += kGemvThreads) {
        x0[kv] = src[2 * kv];
        x1[kv] = src[2 * kv + 1];
      }
    } else if constexpr (MODE == GM_GATEUP || MODE == GM_LMHEAD) {
      const float4 *src = reinterpret_cast<const float4 *>(p.xf + (size_t)item * K);
      const uint4 *wn = reinterpret_cast<const uint4 *>(p.norm0);
      for (int kv = tid; kv < KV; kv += kGemvThreads) {
        const float4 a = src[2 * kv], b = src[2 * kv + 1];
        const uint4 w = wn[kv];
        ss[m][0] += sq8(a, b);
        x0[kv] = mul4(a, bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y));
        x1[kv] = mul4(b, bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w));
      }
    } else if constexpr (MODE == GM_QKV) {
      // [embed(tok) * w_in ; g * w_hid]; the two RMSNorm scales come later
      const int n = p.n_embd, NV = n >> 3;
      const PairItem it = resolve_pair(p.pairs, item, n);
      int tok = it.tok;
      if (tok < 0 || tok >= p.target_vocab) {
        // only rows whose K/V are kept (or the chain's q) may report a bad token
        if (tid == 0 && (it.write_kv || p.row_base == 0)) set_status(p.status, EAGLE3_DEV_BAD_TOKEN);
        tok = 0;
      }
      const uint4 *er = reinterpret_cast<const uint4 *>(p.embed + (size_t)tok * n);
      const float4 *gr = reinterpret_cast<const float4 *>(it.g);
      const uint4 *wi = reinterpret_cast<const uint4 *>(p.norm0);
      const uint4 *wh = reinterpret_cast<const uint4 *>(p.norm1);
      for (int kv = tid; kv < NV; kv += kGemvThreads) {
        const uint4 u = er[kv];
        const float4 ea = make_float4(bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y));
        const float4 eb = make_float4(bf_lo(u.z), bf_hi(u.z), bf_lo(u.w), bf_hi(u.w));
        const uint4 w = wi[kv];
        ss[m][0] += sq8(ea, eb);
        x0[kv] = mul4(ea, bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y));
        x1[kv] = mul4(eb, bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w));
        const float4 a = gr[2 * kv], b = gr[2 * kv + 1];
        const uint4 hw = wh[kv];
        ss[m][T::kHalves - 1] += sq8(a, b);
        x0[NV + kv] = mul4(a, bf_lo(hw.x), bf_hi(hw.x), bf_lo(hw.y), bf_hi(hw.y));
        x1[NV + kv] = mul4(b, bf_lo(hw.z), bf_hi(hw.z), bf_lo(hw.w), bf_hi(hw.w));
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

template <int NB, int MODE>
__device__ void epilogue(const GemvParams &p, const float *accs, int row0, int nrows) {
  const int tid = threadIdx.x;
  if constexpr (MODE == GM_ENCODE || MODE == GM_O || MODE == GM_DOWN) {
    for (int idx = tid; idx < nrows * NB; idx += kGemvThreads) {
      const int m = idx % NB, r = idx / NB;
      if (m >= p.items) continue;
      const int item = p.item0 + m, row = row0 + r;
      float v = accs[r * NB + m];
      if constexpr (MODE != GM_ENCODE) v += p.res[(size_t)item * p.rows + row];
      p.out_f[(size_t)item * p.rows + row] = v;
      if constexpr (MODE == GM_DOWN) {
        if (p.dbg_f) p.dbg_f[(size_t)item * p.dbg_stride_b + p.dbg_off + row] = v;
      }
    }
  } else if constexpr (MODE == GM_GATEUP) {
    const int npairs = nrows >> 1;
    for (int idx = tid; idx < npairs * NB; idx += kGemvThreads) {
      const int m = idx % NB, pr = idx / NB;
      if (m >= p.items) continue;
      const int item = p.item0 + m;
      const float gate = accs[(2 * pr) * NB + m], up = accs[(2 * pr + 1) * NB + m];
      p.out_f[(size_t)item * p.n_ff + ((row0 >> 1) + pr)] = silu_f(gate) * up;
    }
  } else if constexpr (MODE == GM_QKV) {
    const int d = p.head_dim, R = p.rope_dims, half = R >> 1;
    const int qr = p.n_head * d, kr = p.n_head_kv * d;
    const int npairs = nrows >> 1;
    for (int idx = tid; idx < npairs * NB; idx += kGemvThreads) {
      const int m = idx % NB, pr = idx / NB;
      if (m >= p.items) continue;
      const int item = p.item0 + m;
      const int lr = p.row_base + row0 + 2 * pr;  // even logical row
      float a = accs[(2 * pr) * NB + m], b = accs[(2 * pr + 1) * NB + m];
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
    for (int m = 0; m < p.items; ++m) {
      const int item = p.item0 + m;
      unsigned long long best = 0ull;
      for (int r = tid; r < nrows; r += kGemvThreads) {
        const float v = accs[r * NB + m];
        const int row = row0 + r;
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
    if (tid == 0) {
      __threadfence();
      const unsigned prev = atomicAdd(p.am_count, 1u);
      last_sh = (prev == gridDim.x - 1) ? 1 : 0;
    }
    consumer_sync();
    if (last_sh) {
      __threadfence();
      for (int m = tid; m < p.items; m += kGemvThreads) {
        const int item = p.item0 + m;
        const unsigned long long key = atomicExch(p.am_slot + item, 0ull);
        uint32_t id = 0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull);
        if (id >= (uint32_t)p.draft_vocab) {
          set_status(p.status, EAGLE3_DEV_BAD_TOKEN);
          id = 0;
        }
        long long tgt = (long long)id + p.d2t[id];
        if (tgt < 0 || tgt >= p.target_vocab) {
          set_status(p.status, EAGLE3_DEV_BAD_TOKEN);
          tgt = 0;
        }
        const bool valid = p.step < p.gamma_eff[item];
        const size_t o = (size_t)item * p.gamma + p.step;
        p.draft_tok[o] = valid ? (int32_t)tgt : -1;
        if (p.draft_id) p.draft_id[o] = valid ? (int32_t)id : -1;
        if (p.next_tok) p.next_tok[item] = (int32_t)tgt;
      }
      if (tid == 0) *p.am_count = 0u;
    }
  }
}

// -------------------------------------------------------------------- kernel
constexpr int kStageBytes = 32 * 1024;
// Single-item launches with K <= 6 * 256 * 8 = 12288 keep x in registers: 6 vectors of 8
// floats per thread (larger K reads x from shared memory).
constexpr int kXRegVecs = 6;
constexpr int kGemvCtaThreads = kGemvThreads + 32;  // 8 consumer warps + 1 producer warp

struct GemvSmem {
  int x_bytes, ring_off, stage_bytes, part_off, accs_off, red_off, scale_off, bar_off, flag_off,
      total;
};

__host__ __device__ inline GemvSmem gemv_smem_layout(int NB, int SR, int H, int xbytes_per_elem,
                                                     int K, int nstage, int max_rows) {
  GemvSmem L;
  L.x_bytes = NB * K * xbytes_per_elem;
  L.stage_bytes = SR * K * 2;
  L.ring_off = L.x_bytes;
  L.part_off = L.ring_off + nstage * L.stage_bytes;
  L.accs_off = L.part_off + max_rows * kGemvWarps * H * NB * 4;
  L.red_off = L.accs_off + max_rows * NB * 4;
  L.scale_off = L.red_off + kGemvWarps * NB * H * 4;
  L.bar_off = (L.scale_off + NB * H * 4 + 15) / 16 * 16;
  L.flag_off = L.bar_off + 2 * nstage * 8;
  L.total = L.flag_off + 16;
  return L;
}

template <int NB, int SR, int MODE>
__global__ void __launch_bounds__(kGemvCtaThreads, 1) gemv_kernel(const GemvParams p) {
  using T = ModeTraits<MODE>;
  constexpr int H = T::kHalves;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.K, KV = K >> 3;
  // rows are handed out in units of 2 where the epilogue pairs rows (RoPE, SwiGLU)
  const int nunits = p.rows / T::kUnit;
  const int ub = (int)((long long)blockIdx.x * nunits / gridDim.x);
  const int ue = (int)((long long)(blockIdx.x + 1) * nunits / gridDim.x);
  const int row0 = T::kUnit * ub, nrows = T::kUnit * (ue - ub);
  const int max_rows = T::kUnit * ((nunits + gridDim.x - 1) / gridDim.x);
  const int nst = p.nstage;
  const GemvSmem L = gemv_smem_layout(NB, SR, H, T::kBf16X ? 2 : 4, K, nst, max_rows);
  const int n_stages = (nrows + SR - 1) / SR;
  const int NVH = H == 2 ? (p.n_embd >> 3) : KV;  // first vector of the second K half

  unsigned char *xmem = smem;
  unsigned char *ring = smem + L.ring_off;
  float *part = reinterpret_cast<float *>(smem + L.part_off);  // [max_rows][warps][H][NB]
  float *accs = reinterpret_cast<float *>(smem + L.accs_off);  // [max_rows][NB]
  float *red = reinterpret_cast<float *>(smem + L.red_off);    // [warps][NB * H]
  float *scale = reinterpret_cast<float *>(smem + L.scale_off);  // [NB * H]
  const uint32_t full0 = smem_addr(smem + L.bar_off);
  const uint32_t empty0 = full0 + 8 * nst;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.flag_off);

  if (tid == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, kGemvWarps);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  pdl_trigger();

  if (warp == kGemvWarps) {
    // ------------------------------------------------------------ producer warp
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      const uint32_t row_bytes = (uint32_t)K * 2u;
      int issued = 0;
      for (int st = 0; st < n_stages; ++st) {
        const int slot = st % nst;
        if (st >= nst && !mbar_wait(empty0 + 8 * slot, ((st / nst) - 1) & 1, abort_flag, p.status))
          break;
        const int rows_here = min(SR, nrows - st * SR);
        mbar_expect_tx(full0 + 8 * slot, (uint32_t)rows_here * row_bytes);
        const uint32_t dst = smem_addr(ring + (size_t)slot * L.stage_bytes);
        for (int r = 0; r < rows_here; ++r)
          bulk_g2s(dst + r * row_bytes, row_ptr<MODE>(p, p.row_base + row0 + st * SR + r), row_bytes,
                   full0 + 8 * slot, pol);
        issued = st + 1;
      }
      // Never leave copies in flight into shared memory: wait for the last stages issued.
      for (int st = max(0, issued - nst); st < issued; ++st)
        mbar_wait(full0 + 8 * (st % nst), (st / nst) & 1, abort_flag, p.status);
    }
    return;
  }

  // ------------------------------------------------------------ consumer warps
  pdl_wait();
  float ss[NB][H];
  stage_x<NB, MODE>(p, xmem, ss);
  consumer_sync();
  const bool xreg = (NB == 1) && (KV <= kXRegVecs * kGemvThreads);
  float xr[NB == 1 ? kXRegVecs : 1][8];
  if (xreg) {
#pragma unroll
    for (int j = 0; j < (NB == 1 ? kXRegVecs : 0); ++j) {
      const int kv = tid + j * kGemvThreads;
      if (kv < KV) {
        load_x8<MODE>(xmem, KV, 0, kv, xr[j]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) xr[j][i] = 0.f;
      }
    }
  }

  for (int st = 0; st < n_stages; ++st) {
    const int slot = st % nst;
    const bool ok = mbar_wait(full0 + 8 * slot, (st / nst) & 1, abort_flag, p.status);
    float acc[H][SR][NB];
#pragma unroll
    for (int h = 0; h < H; ++h)
#pragma unroll
      for (int r = 0; r < SR; ++r)
#pragma unroll
        for (int m = 0; m < NB; ++m) acc[h][r][m] = 0.f;
    if (ok) {
      const unsigned char *stage = ring + (size_t)slot * L.stage_bytes;
      const int rows_here = min(SR, nrows - st * SR);
      auto fma_rows = [&](int kv, const float (&x)[8], int m, float (&a)[SR][NB]) {
#pragma unroll
        for (int r = 0; r < SR; ++r)
          if (r < rows_here) {
            const uint4 w = *reinterpret_cast<const uint4 *>(stage + ((size_t)r * K + (size_t)kv * 8) * 2);
            a[r][m] = dot8(w, x, a[r][m]);
          }
      };
      if (xreg) {
#pragma unroll
        for (int j = 0; j < (NB == 1 ? kXRegVecs : 0); ++j) {
          const int kv = tid + j * kGemvThreads;
          if (kv < KV) {
            if (H == 1 || kv < NVH)
              fma_rows(kv, xr[j], 0, acc[0]);
            else
              fma_rows(kv, xr[j], 0, acc[H - 1]);
          }
        }
      } else {
        // several items: each weight vector is loaded and widened once, then used for
        // every item
        for (int kv = tid; kv < KV; kv += kGemvThreads) {
          float wf[SR][8];
#pragma unroll
          for (int r = 0; r < SR; ++r) {
            uint4 w = make_uint4(0u, 0u, 0u, 0u);
            if (r < rows_here) w = *reinterpret_cast<const uint4 *>(stage + ((size_t)r * K + (size_t)kv * 8) * 2);
            wf[r][0] = bf_lo(w.x); wf[r][1] = bf_hi(w.x); wf[r][2] = bf_lo(w.y); wf[r][3] = bf_hi(w.y);
            wf[r][4] = bf_lo(w.z); wf[r][5] = bf_hi(w.z); wf[r][6] = bf_lo(w.w); wf[r][7] = bf_hi(w.w);
          }
          const int h = (H == 1 || kv < NVH) ? 0 : H - 1;
#pragma unroll
          for (int m = 0; m < NB; ++m) {
            float x[8];
            load_x8<MODE>(xmem, KV, m, kv, x);
#pragma unroll
            for (int r = 0; r < SR; ++r) {
              float a0 = 0.f;
#pragma unroll
              for (int i = 0; i < 8; ++i) a0 = fmaf(wf[r][i], x[i], a0);
              if (h == 0)
                acc[0][r][m] += a0;
              else
                acc[H - 1][r][m] += a0;
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * slot);
    // per-warp partial of every (half, row, item) of this stage
    constexpr int N = H * SR * NB;
    float v[N];
#pragma unroll
    for (int h = 0; h < H; ++h)
#pragma unroll
      for (int r = 0; r < SR; ++r)
#pragma unroll
        for (int m = 0; m < NB; ++m) v[(h * SR + r) * NB + m] = acc[h][r][m];
    const float tot = warp_reduce_multi<N>(v, lane);
    if (warp_reduce_writer<N>(lane)) {
      const int idx = warp_reduce_index<N>(lane);
      const int m = idx % NB, r = (idx / NB) % SR, h = idx / (NB * SR);
      const int lrow = st * SR + r;
      if (lrow < nrows) part[(((size_t)lrow * kGemvWarps + warp) * H + h) * NB + m] = tot;
    }
  }
  // RMSNorm scales 1 / sqrt(mean(x^2) + eps) per item and K half
  if constexpr (T::kNorm) {
    float v[NB * H];
#pragma unroll
    for (int m = 0; m < NB; ++m)
#pragma unroll
      for (int h = 0; h < H; ++h) v[m * H + h] = ss[m][h];
    const float tot = warp_reduce_multi<NB * H>(v, lane);
    if (warp_reduce_writer<NB * H>(lane)) red[warp * NB * H + warp_reduce_index<NB * H>(lane)] = tot;
  }
  consumer_sync();
  if constexpr (T::kNorm) {
    if (tid < NB * H) {
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < kGemvWarps; ++w) t += red[w * NB * H + tid];
      const float len = (float)(K / H);
      scale[tid] = rsqrtf(t / len + p.eps);
    }
    consumer_sync();
  }
  for (int e = tid; e < nrows * NB; e += kGemvThreads) {
    const int r = e / NB, m = e - r * NB;
    float y = 0.f;
#pragma unroll
    for (int h = 0; h < H; ++h) {
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kGemvWarps; ++w) sum += part[(((size_t)r * kGemvWarps + w) * H + h) * NB + m];
      y += T::kNorm ? sum * scale[m * H + h] : sum;
    }
    accs[e] = y;
  }
  consumer_sync();
  epilogue<NB, MODE>(p, accs, row0, nrows);
}

// ------------------------------------------------------------------ launcher
// Rows per ring stage: whole rows up to kStageBytes, at most 8, at most 32 / (NB * H) so
// that a stage's sums fit one warp reduction, and fewer if that keeps >= 4 stages.
template <int MODE>
static int stage_rows(int K, int NB, int max_rows) {
  using T = ModeTraits<MODE>;
  int sr = kStageBytes / (2 * K);
  if (sr < 1) sr = 1;
  if (sr > 8) sr = 8;
  if (sr > 32 / (NB * T::kHalves)) sr = 32 / (NB * T::kHalves);
  int p2 = 1;
  while (p2 * 2 <= sr) p2 *= 2;
  while (p2 > 1) {
    const GemvSmem L = gemv_smem_layout(NB, p2, T::kHalves, T::kBf16X ? 2 : 4, K, 0, max_rows);
    const long long room = (long long)kGemvSmemLimit - L.total - 64;
    if (room / (p2 * K * 2 + 16) >= 4) break;
    p2 >>= 1;
  }
  return p2;
}

template <int NB, int SR, int MODE>
static cudaError_t launch_one(GemvParams p, int grid, int max_rows, cudaStream_t st, bool pdl) {
  using T = ModeTraits<MODE>;
  const GemvSmem L0 = gemv_smem_layout(NB, SR, T::kHalves, T::kBf16X ? 2 : 4, p.K, 0, max_rows);
  const long long room = (long long)kGemvSmemLimit - L0.total - 64;
  int nst = (int)(room / (SR * p.K * 2 + 16));
  if (nst > 8) nst = 8;
  if (nst < 2) return cudaErrorInvalidValue;
  p.nstage = nst;
  const GemvSmem L = gemv_smem_layout(NB, SR, T::kHalves, T::kBf16X ? 2 : 4, p.K, nst, max_rows);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemvCtaThreads);
  cfg.dynamicSmemBytes = (size_t)L.total;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemv_kernel<NB, SR, MODE>, p);
}

template <int NB, int MODE>
static cudaError_t dispatch_sr(const GemvParams &p, int grid, cudaStream_t st, bool pdl) {
  using T = ModeTraits<MODE>;
  const int nunits = p.rows / T::kUnit;
  if (grid > nunits) grid = nunits;
  if (grid < 1) grid = 1;
  const int max_rows = T::kUnit * ((nunits + grid - 1) / grid);
  constexpr int SRMAX = 32 / (NB * T::kHalves) >= 8 ? 8 : 32 / (NB * T::kHalves);
  switch (stage_rows<MODE>(p.K, NB, max_rows)) {
    case 1: return launch_one<NB, 1, MODE>(p, grid, max_rows, st, pdl);
    case 2: return launch_one<NB, (SRMAX >= 2 ? 2 : 1), MODE>(p, grid, max_rows, st, pdl);
    case 4: return launch_one<NB, (SRMAX >= 4 ? 4 : 1), MODE>(p, grid, max_rows, st, pdl);
    default: return launch_one<NB, SRMAX, MODE>(p, grid, max_rows, st, pdl);
  }
}

template <int MODE>
static cudaError_t dispatch_nb(const GemvParams &p, int nb, int grid, cudaStream_t st, bool pdl) {
  switch (nb) {
    case 1: return dispatch_sr<1, MODE>(p, grid, st, pdl);
    case 2: return dispatch_sr<2, MODE>(p, grid, st, pdl);
    case 4: return dispatch_sr<4, MODE>(p, grid, st, pdl);
    case 8: return dispatch_sr<8, MODE>(p, grid, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

template <int NB, int MODE>
static cudaError_t prepare_nb() {
  using T = ModeTraits<MODE>;
  constexpr int SRMAX = 32 / (NB * T::kHalves) >= 8 ? 8 : 32 / (NB * T::kHalves);
  const int lim = (int)kGemvSmemLimit;
  cudaError_t e = cudaFuncSetAttribute(gemv_kernel<NB, 1, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemv_kernel<NB, (SRMAX >= 2 ? 2 : 1), MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemv_kernel<NB, (SRMAX >= 4 ? 4 : 1), MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemv_kernel<NB, SRMAX, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  return e;
}

template <int MODE>
static cudaError_t prepare_mode() {
  cudaError_t e = prepare_nb<1, MODE>();
  if (e == cudaSuccess) e = prepare_nb<2, MODE>();
  if (e == cudaSuccess) e = prepare_nb<4, MODE>();
  if (e == cudaSuccess) e = prepare_nb<8, MODE>();
  return e;
}

// Raise every instantiation's dynamic shared memory limit once, outside any capture.
cudaError_t gemv_prepare() {
  cudaError_t e = prepare_mode<GM_ENCODE>();
  if (e == cudaSuccess) e = prepare_mode<GM_QKV>();
  if (e == cudaSuccess) e = prepare_mode<GM_O>();
  if (e == cudaSuccess) e = prepare_mode<GM_GATEUP>();
  if (e == cudaSuccess) e = prepare_mode<GM_DOWN>();
  if (e == cudaSuccess) e = prepare_mode<GM_LMHEAD>();
  return e;
}

int gemv_items_per_launch(int mode, int K, int items) {
  // x of one launch lives in shared memory: NB * K * (2 or 4) bytes <= kGemvMaxXBytes.
  const size_t eb = mode == GM_ENCODE ? 2 : 4;
  int nb = 8;
  while (nb > 1 && (size_t)nb * K * eb > kGemvMaxXBytes) nb >>= 1;
  while (nb > 1 && nb / 2 >= items) nb >>= 1;
  return nb;
}

cudaError_t gemv_launch(const GemvParams &p, int grid, cudaStream_t st, bool pdl) {
  const int nb = gemv_items_per_launch(p.mode, p.K, p.items);
  if (p.items > nb || p.items < 1) return cudaErrorInvalidValue;
  switch (p.mode) {
    case GM_ENCODE: return dispatch_nb<GM_ENCODE>(p, nb, grid, st, pdl);
    case GM_QKV: return dispatch_nb<GM_QKV>(p, nb, grid, st, pdl);
    case GM_O: return dispatch_nb<GM_O>(p, nb, grid, st, pdl);
    case GM_GATEUP: return dispatch_nb<GM_GATEUP>(p, nb, grid, st, pdl);
    case GM_DOWN: return dispatch_nb<GM_DOWN>(p, nb, grid, st, pdl);
    case GM_LMHEAD: return dispatch_nb<GM_LMHEAD>(p, nb, grid, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace e3
