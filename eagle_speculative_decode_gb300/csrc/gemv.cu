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
// shared memory as float32 in two float4 planes (elements 0-3 and 4-7 of each 8-element
// vector: conflict-free LDS.128), then, per stage, each thread takes 16-byte vectors
// k = 8 * (warp * 32 + lane + 256 j) of all SR rows, so every x vector it loads serves
// SR rows.  A stage's per-row sums are reduced within the warp and kept per warp; the
// eight warp partials are added in a fixed order before the epilogue (deterministic).
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

// Block-wide sum of one float per thread; result valid in every thread.
__device__ __forceinline__ float block_sum(float v, float *scratch) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  consumer_sync();
  if (lane == 0) scratch[warp] = v;
  consumer_sync();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kGemvWarps; ++w) t += scratch[w];
  return t;
}

// ------------------------------------------------------------------ x staging
// Writes x[m, k] into the two float4 planes xs[(m * 2 + plane) * KV + kv].
template <int NB, int MODE>
__device__ void stage_x(const GemvParams &p, float4 *xs, float *scratch) {
  const int K = p.K, KV = K >> 3, tid = threadIdx.x;
  for (int m = 0; m < NB; ++m) {
    float4 *x0 = xs + (size_t)(m * 2) * KV;
    float4 *x1 = x0 + KV;
    const bool live = m < p.items;
    if (!live) {
      for (int kv = tid; kv < KV; kv += kGemvThreads) {
        x0[kv] = make_float4(0.f, 0.f, 0.f, 0.f);
        x1[kv] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      continue;
    }
    const int item = p.item0 + m;
    if constexpr (MODE == GM_ENCODE) {
      const uint4 *src = reinterpret_cast<const uint4 *>(p.xb + (size_t)item * K);
      for (int kv = tid; kv < KV; kv += kGemvThreads) {
        const uint4 u = src[kv];
        x0[kv] = make_float4(bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y));
        x1[kv] = make_float4(bf_lo(u.z), bf_hi(u.z), bf_lo(u.w), bf_hi(u.w));
      }
    } else if constexpr (MODE == GM_O || MODE == GM_DOWN) {
      const float4 *src = reinterpret_cast<const float4 *>(p.xf + (size_t)item * K);
      for (int kv = tid; kv < KV; kv += kGemvThreads) {
        x0[kv] = src[2 * kv];
        x1[kv] = src[2 * kv + 1];
      }
    } else if constexpr (MODE == GM_GATEUP || MODE == GM_LMHEAD) {
      // RMSNorm(x) * w over K = n_embd.
      const float4 *src = reinterpret_cast<const float4 *>(p.xf + (size_t)item * K);
      float ss = 0.f;
      for (int kv = tid; kv < KV; kv += kGemvThreads) {
        const float4 a = src[2 * kv], b = src[2 * kv + 1];
        ss += a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w + b.x * b.x + b.y * b.y + b.z * b.z +
              b.w * b.w;
      }
      ss = block_sum(ss, scratch);
      const float sc = rsqrtf(ss / (float)K + p.eps);
      const uint4 *wn = reinterpret_cast<const uint4 *>(p.norm0);
      for (int kv = tid; kv < KV; kv += kGemvThreads) {
        const float4 a = src[2 * kv], b = src[2 * kv + 1];
        const uint4 w = wn[kv];
        x0[kv] = make_float4(a.x * sc * bf_lo(w.x), a.y * sc * bf_hi(w.x), a.z * sc * bf_lo(w.y),
                             a.w * sc * bf_hi(w.y));
        x1[kv] = make_float4(b.x * sc * bf_lo(w.z), b.y * sc * bf_hi(w.z), b.z * sc * bf_lo(w.w),
                             b.w * sc * bf_hi(w.w));
      }
    } else if constexpr (MODE == GM_QKV) {
      // [RMSNorm(embed(tok)) * w_in ; RMSNorm(g) * w_hid], K = 2 n.
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
      float se = 0.f, sg = 0.f;
      for (int kv = tid; kv < NV; kv += kGemvThreads) {
        const uint4 u = er[kv];
        const float e[8] = {bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y),
                            bf_lo(u.z), bf_hi(u.z), bf_lo(u.w), bf_hi(u.w)};
#pragma unroll
        for (int i = 0; i < 8; ++i) se += e[i] * e[i];
        const float4 a = gr[2 * kv], b = gr[2 * kv + 1];
        sg += a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w + b.x * b.x + b.y * b.y + b.z * b.z +
              b.w * b.w;
      }
      se = block_sum(se, scratch);
      sg = block_sum(sg, scratch + kGemvWarps);
      const float sce = rsqrtf(se / (float)n + p.eps);
      const float scg = rsqrtf(sg / (float)n + p.eps);
      const uint4 *wi = reinterpret_cast<const uint4 *>(p.norm0);
      const uint4 *wh = reinterpret_cast<const uint4 *>(p.norm1);
      for (int kv = tid; kv < NV; kv += kGemvThreads) {
        const uint4 u = er[kv];
        const uint4 w = wi[kv];
        x0[kv] = make_float4(bf_lo(u.x) * sce * bf_lo(w.x), bf_hi(u.x) * sce * bf_hi(w.x),
                             bf_lo(u.y) * sce * bf_lo(w.y), bf_hi(u.y) * sce * bf_hi(w.y));
        x1[kv] = make_float4(bf_lo(u.z) * sce * bf_lo(w.z), bf_hi(u.z) * sce * bf_hi(w.z),
                             bf_lo(u.w) * sce * bf_lo(w.w), bf_hi(u.w) * sce * bf_hi(w.w));
        const float4 a = gr[2 * kv], b = gr[2 * kv + 1];
        const uint4 h = wh[kv];
        x0[NV + kv] = make_float4(a.x * scg * bf_lo(h.x), a.y * scg * bf_hi(h.x),
                                  a.z * scg * bf_lo(h.y), a.w * scg * bf_hi(h.y));
        x1[NV + kv] = make_float4(b.x * scg * bf_lo(h.z), b.y * scg * bf_hi(h.z),
                                  b.z * scg * bf_lo(h.w), b.w * scg * bf_hi(h.w));
      }
    }
  }
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
  int x_bytes, ring_off, stage_bytes, part_off, accs_off, scratch_off, bar_off, flag_off, total;
};

__host__ __device__ inline GemvSmem gemv_smem_layout(int NB, int SR, int K, int nstage, int max_rows) {
  GemvSmem L;
  L.x_bytes = NB * K * 4;
  L.stage_bytes = SR * K * 2;
  L.ring_off = L.x_bytes;
  L.part_off = L.ring_off + nstage * L.stage_bytes;
  L.accs_off = L.part_off + max_rows * kGemvWarps * NB * 4;
  L.scratch_off = L.accs_off + max_rows * NB * 4;
  L.bar_off = (L.scratch_off + 2 * kGemvWarps * 4 + 15) / 16 * 16;
  L.flag_off = L.bar_off + 2 * nstage * 8;
  L.total = L.flag_off + 16;
  return L;
}

template <int NB, int SR, int MODE>
__global__ void __launch_bounds__(kGemvCtaThreads, 1) gemv_kernel(const GemvParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.K, KV = K >> 3;
  // rows are handed out in units of 2 where the epilogue pairs rows (RoPE, SwiGLU)
  constexpr int UNIT = (MODE == GM_QKV || MODE == GM_GATEUP) ? 2 : 1;
  const int nunits = p.rows / UNIT;
  const int ub = (int)((long long)blockIdx.x * nunits / gridDim.x);
  const int ue = (int)((long long)(blockIdx.x + 1) * nunits / gridDim.x);
  const int row0 = UNIT * ub, nrows = UNIT * (ue - ub);
  const int max_rows = UNIT * ((nunits + gridDim.x - 1) / gridDim.x);
  const int nst = p.nstage;
  const GemvSmem L = gemv_smem_layout(NB, SR, K, nst, max_rows);
  const int n_stages = (nrows + SR - 1) / SR;

  float4 *xs = reinterpret_cast<float4 *>(smem);
  unsigned char *ring = smem + L.ring_off;
  float *part = reinterpret_cast<float *>(smem + L.part_off);     // [max_rows][warps][NB]
  float *accs = reinterpret_cast<float *>(smem + L.accs_off);     // [max_rows][NB]
  float *scratch = reinterpret_cast<float *>(smem + L.scratch_off);
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
  stage_x<NB, MODE>(p, xs, scratch);
  consumer_sync();
  float xr[NB == 1 ? kXRegVecs : 1][8];
  const bool xreg = (NB == 1) && (KV <= kXRegVecs * kGemvThreads);
  if (xreg) {
#pragma unroll
    for (int j = 0; j < (NB == 1 ? kXRegVecs : 0); ++j) {
      const int kv = tid + j * kGemvThreads;
      const float4 a = kv < KV ? xs[kv] : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 c = kv < KV ? xs[KV + kv] : make_float4(0.f, 0.f, 0.f, 0.f);
      xr[j][0] = a.x; xr[j][1] = a.y; xr[j][2] = a.z; xr[j][3] = a.w;
      xr[j][4] = c.x; xr[j][5] = c.y; xr[j][6] = c.z; xr[j][7] = c.w;
    }
  }

  for (int st = 0; st < n_stages; ++st) {
    const int slot = st % nst;
    const bool ok = mbar_wait(full0 + 8 * slot, (st / nst) & 1, abort_flag, p.status);
    float acc[SR][NB];
#pragma unroll
    for (int r = 0; r < SR; ++r)
#pragma unroll
      for (int m = 0; m < NB; ++m) acc[r][m] = 0.f;
    if (ok) {
      const unsigned char *stage = ring + (size_t)slot * L.stage_bytes;
      const int rows_here = min(SR, nrows - st * SR);
      if (xreg) {
        // x of this thread's vectors is held in registers across all stages
#pragma unroll
        for (int j = 0; j < (NB == 1 ? kXRegVecs : 0); ++j) {
          const int kv = tid + j * kGemvThreads;
          if (kv < KV) {
#pragma unroll
            for (int r = 0; r < SR; ++r) {
              if (r < rows_here) {
                const uint4 w = *reinterpret_cast<const uint4 *>(stage + ((size_t)r * K + (size_t)kv * 8) * 2);
                float a = acc[r][0];
                a = fmaf(bf_lo(w.x), xr[j][0], a); a = fmaf(bf_hi(w.x), xr[j][1], a);
                a = fmaf(bf_lo(w.y), xr[j][2], a); a = fmaf(bf_hi(w.y), xr[j][3], a);
                a = fmaf(bf_lo(w.z), xr[j][4], a); a = fmaf(bf_hi(w.z), xr[j][5], a);
                a = fmaf(bf_lo(w.w), xr[j][6], a); a = fmaf(bf_hi(w.w), xr[j][7], a);
                acc[r][0] = a;
              }
            }
          }
        }
      } else {
        for (int kv = tid; kv < KV; kv += kGemvThreads) {
          float4 xa[NB], xb[NB];
#pragma unroll
          for (int m = 0; m < NB; ++m) {
            xa[m] = xs[(size_t)(m * 2) * KV + kv];
            xb[m] = xs[(size_t)(m * 2 + 1) * KV + kv];
          }
#pragma unroll
          for (int r = 0; r < SR; ++r) {
            if (r < rows_here) {
              const uint4 w = *reinterpret_cast<const uint4 *>(stage + ((size_t)r * K + (size_t)kv * 8) * 2);
              const float w0 = bf_lo(w.x), w1 = bf_hi(w.x), w2 = bf_lo(w.y), w3 = bf_hi(w.y);
              const float w4 = bf_lo(w.z), w5 = bf_hi(w.z), w6 = bf_lo(w.w), w7 = bf_hi(w.w);
#pragma unroll
              for (int m = 0; m < NB; ++m) {
                float a = acc[r][m];
                a = fmaf(w0, xa[m].x, a); a = fmaf(w1, xa[m].y, a);
                a = fmaf(w2, xa[m].z, a); a = fmaf(w3, xa[m].w, a);
                a = fmaf(w4, xb[m].x, a); a = fmaf(w5, xb[m].y, a);
                a = fmaf(w6, xb[m].z, a); a = fmaf(w7, xb[m].w, a);
                acc[r][m] = a;
              }
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * slot);
    // per-warp partial of every (row, item) of this stage
    constexpr int N = SR * NB;
    float v[N];
#pragma unroll
    for (int r = 0; r < SR; ++r)
#pragma unroll
      for (int m = 0; m < NB; ++m) v[r * NB + m] = acc[r][m];
    const float tot = warp_reduce_multi<N>(v, lane);
    if (warp_reduce_writer<N>(lane)) {
      const int idx = warp_reduce_index<N>(lane);
      const int r = idx / NB, m = idx - r * NB;
      const int lrow = st * SR + r;
      if (lrow < nrows) part[((size_t)lrow * kGemvWarps + warp) * NB + m] = tot;
    }
  }
  consumer_sync();
  for (int e = tid; e < nrows * NB; e += kGemvThreads) {
    const int r = e / NB, m = e - r * NB;
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kGemvWarps; ++w) sum += part[((size_t)r * kGemvWarps + w) * NB + m];
    accs[e] = sum;
  }
  consumer_sync();
  epilogue<NB, MODE>(p, accs, row0, nrows);
}

// ------------------------------------------------------------------ launcher
// Rows per ring stage: whole rows up to kStageBytes, at most 8, and at most 32 / NB so
// that a stage's (row, item) sums fit one warp reduction.
static int stage_rows(int K, int NB) {
  int sr = kStageBytes / (2 * K);
  if (sr < 1) sr = 1;
  if (sr > 8) sr = 8;
  if (sr > 32 / NB) sr = 32 / NB;
  int p2 = 1;
  while (p2 * 2 <= sr) p2 *= 2;
  return p2;
}

template <int NB, int SR, int MODE>
static cudaError_t launch_one(GemvParams p, int grid, cudaStream_t st, bool pdl) {
  constexpr int UNIT = (MODE == GM_QKV || MODE == GM_GATEUP) ? 2 : 1;
  const int nunits = p.rows / UNIT;
  if (grid > nunits) grid = nunits;
  if (grid < 1) grid = 1;
  const int max_rows = UNIT * ((nunits + grid - 1) / grid);
  const GemvSmem L0 = gemv_smem_layout(NB, SR, p.K, 0, max_rows);
  const long long room = (long long)kGemvSmemLimit - L0.total - 64;
  int nst = (int)(room / (SR * p.K * 2 + 16));
  if (nst > 8) nst = 8;
  if (nst < 2) return cudaErrorInvalidValue;
  p.nstage = nst;
  const GemvSmem L = gemv_smem_layout(NB, SR, p.K, nst, max_rows);
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
  switch (stage_rows(p.K, NB)) {
    case 1: return launch_one<NB, 1, MODE>(p, grid, st, pdl);
    case 2: return launch_one<NB, 2, MODE>(p, grid, st, pdl);
    case 4: return launch_one<NB, 4, MODE>(p, grid, st, pdl);
    default: return launch_one<NB, (NB <= 4 ? 8 : 4), MODE>(p, grid, st, pdl);
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
  cudaError_t e = cudaSuccess;
  const int lim = (int)kGemvSmemLimit;
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_kernel<NB, 1, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_kernel<NB, 2, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_kernel<NB, 4, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  if (NB <= 4 && e == cudaSuccess)
    e = cudaFuncSetAttribute(gemv_kernel<NB, (NB <= 4 ? 8 : 4), MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
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

int gemv_items_per_launch(int K, int items) {
  // x of one launch lives in shared memory: NB * K * 4 bytes <= kGemvMaxXBytes.
  int nb = 8;
  while (nb > 1 && (size_t)nb * K * 4 > kGemvMaxXBytes) nb >>= 1;
  while (nb > 1 && nb / 2 >= items) nb >>= 1;
  return nb;
}

cudaError_t gemv_launch(const GemvParams &p, int grid, cudaStream_t st, bool pdl) {
  const int nb = gemv_items_per_launch(p.K, p.items);
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
