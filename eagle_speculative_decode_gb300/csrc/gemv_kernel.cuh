// Weight-streaming GEMV for the drafter's projections at small batch (items <= 8), as a
// template shared by the bf16 instantiations (gemv.cu) and the INT4 ones (gemv_q4.cu).
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
// kernel drains.  Sixteen consumer warps stage x (normalised where the op says so) in
// shared memory (float32 in two float4 planes -- elements 0-3 and 4-7 of each 8-element
// vector, conflict-free LDS.128 -- or as the caller's bf16 for the encode), then, per
// stage, each thread takes 16-byte vectors k = 8 * (tid + 512 j) of all SR rows, so every
// x vector it loads serves SR rows; single-item launches keep their x vectors in
// registers.  RMSNorm is applied after the dot product: the GEMV runs on x * w_norm and
// the per-item scale 1 / sqrt(mean(x^2) + eps), reduced while x is staged, multiplies the
// row sums, so no block-wide reduction stands between the dependency wait and the first
// FMA.  A stage's per-row sums are reduced within the warp and kept per warp; the sixteen
// warp partials are added in a fixed order before the epilogue (deterministic).
//
// INT4 weights (Q4): a row is K / 2 bytes of 4-bit codes (byte j: code of k = 2j in the
// low nibble, k = 2j + 1 in the high one) and, per group of 128 k, a (scale, zero) pair of
// bf16, w = scale * (code - 8) + zero.  The producer copies both parts of each row.  A
// consumer thread takes the same 8-element k vector as in the bf16 case (4 code bytes):
// each code becomes the float 128 + code by a byte permute under the exponent of 128 and
// code - 8 by one exact packed add, the dot product with x runs on packed two-lane FMAs,
// and the group's affine map is applied to the 8-element partial:
// scale * sum((code - 8) x) + zero * sum(x).
#pragma once
#include <math.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "internal.h"

namespace e3 {

// -------------------------------------------------------------------- kernel
constexpr int kStageBytes = 32 * 1024;
// Single-item launches with K <= 3 * 512 * 8 = 12288 keep x in registers: up to 3 vectors
// of 8 floats per thread (larger K reads x from shared memory).
constexpr int kXRegVecs = 3;
constexpr int kGemvCtaThreads = kGemvThreads + 32;  // 16 consumer warps + 1 producer warp

struct GemvSmem {
  int x_bytes, ring_off, stage_bytes, part_off, accs_off, red_off, scale_off, bar_off, flag_off,
      total;
};

// Bytes of one weight row in the ring: bf16, or INT4 codes + the padded (scale, zero) row.
__host__ __device__ inline int gemv_row_bytes(bool q4, int K, int sz_stride) {
  return q4 ? K / 2 + sz_stride * 4 : K * 2;
}

__host__ __device__ inline GemvSmem gemv_smem_layout(int NB, int SR, int H, int xbytes_per_elem,
                                                     int K, int nstage, int max_rows, int row_bytes) {
  GemvSmem L;
  L.x_bytes = NB * K * xbytes_per_elem;
  L.stage_bytes = SR * row_bytes;
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

// Eight INT4 codes of one 32-bit word as the floats code - 8, in the pair order
// (0, 2), (4, 6), (1, 3), (5, 7) of their k offsets: 0x43_0c_00_00 reads as 128 + c
// exactly (c < 16 stays below the exponent field), minus 136 (exact integers).
__device__ __forceinline__ void q4_to_f32x2(uint32_t w, float2 (&f)[4]) {
  const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
  const float2 bias = make_float2(-136.f, -136.f);
  f[0] = make_float2(__uint_as_float(__byte_perm(lo, 0x43000000u, 0x7044)),
                     __uint_as_float(__byte_perm(lo, 0x43000000u, 0x7144)));
  f[1] = make_float2(__uint_as_float(__byte_perm(lo, 0x43000000u, 0x7244)),
                     __uint_as_float(__byte_perm(lo, 0x43000000u, 0x7344)));
  f[2] = make_float2(__uint_as_float(__byte_perm(hi, 0x43000000u, 0x7044)),
                     __uint_as_float(__byte_perm(hi, 0x43000000u, 0x7144)));
  f[3] = make_float2(__uint_as_float(__byte_perm(hi, 0x43000000u, 0x7244)),
                     __uint_as_float(__byte_perm(hi, 0x43000000u, 0x7344)));
#pragma unroll
  for (int i = 0; i < 4; ++i) f[i] = __fadd2_rn(f[i], bias);
}

// x of one 8-element k vector in the pair order of q4_to_f32x2, and its sum.
__device__ __forceinline__ void q4_x_pairs(const float (&x)[8], float2 (&xq)[4], float &xs) {
  xq[0] = make_float2(x[0], x[2]);
  xq[1] = make_float2(x[4], x[6]);
  xq[2] = make_float2(x[1], x[3]);
  xq[3] = make_float2(x[5], x[7]);
  xs = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
}

// a + scale * sum_i (code_i - 8) x_i + zero * xs, i.e. a + sum_i w_i x_i.
__device__ __forceinline__ float q4_dot(const float2 (&f)[4], const float2 (&xq)[4], float xs, uint32_t sz,
                                        float a) {
  float2 d = __fmul2_rn(f[0], xq[0]);
  d = __ffma2_rn(f[1], xq[1], d);
  d = __ffma2_rn(f[2], xq[2], d);
  d = __ffma2_rn(f[3], xq[3], d);
  return fmaf(bf_lo(sz), d.x + d.y, fmaf(bf_hi(sz), xs, a));
}

template <int NB, int SR, int MODE, bool Q4>
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
  const int szw = Q4 ? p.sz_stride : 0;  // (scale, zero) pairs per row
  const GemvSmem L = gemv_smem_layout(NB, SR, H, T::kBf16X ? 2 : 4, K, nst, max_rows, gemv_row_bytes(Q4, K, szw));
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
      const uint32_t row_bytes = (uint32_t)(Q4 ? K / 2 : K * 2), sz_bytes = (uint32_t)szw * 4u;
      int issued = 0;
      for (int st = 0; st < n_stages; ++st) {
        const int slot = st % nst;
        if (st >= nst && !mbar_wait(empty0 + 8 * slot, ((st / nst) - 1) & 1, abort_flag, p.status))
          break;
        const int rows_here = min(SR, nrows - st * SR);
        mbar_expect_tx(full0 + 8 * slot, (uint32_t)rows_here * (row_bytes + sz_bytes));
        const uint32_t dst = smem_addr(ring + (size_t)slot * L.stage_bytes);
        for (int r = 0; r < rows_here; ++r) {
          const RowRef rr = row_ref<MODE>(p, p.row_base + row0 + st * SR + r);
          if constexpr (Q4) {
            // codes, then the row's (scale, zero) pairs after the stage's SR code rows
            bulk_g2s(dst + r * row_bytes, q4_codes(p, rr), row_bytes, full0 + 8 * slot, pol);
            bulk_g2s(dst + SR * row_bytes + r * sz_bytes, q4_sz(p, rr), sz_bytes, full0 + 8 * slot, pol);
          } else {
            bulk_g2s(dst + r * row_bytes, bf16_row(p, rr), row_bytes, full0 + 8 * slot, pol);
          }
        }
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
  constexpr int XRV = NB == 1 ? kXRegVecs : 1;
  float xr[Q4 ? 1 : XRV][8];              // bf16 weights: x as loaded
  float2 xq[Q4 ? XRV : 1][4];             // INT4 weights: x in code pair order, and its sums
  float xsum[Q4 ? XRV : 1];
  if (xreg) {
#pragma unroll
    for (int j = 0; j < (NB == 1 ? kXRegVecs : 0); ++j) {
      const int kv = tid + j * kGemvThreads;
      float x[8];
      if (kv < KV) {
        load_x8<MODE>(xmem, KV, 0, kv, x);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = 0.f;
      }
      if constexpr (Q4) {
        q4_x_pairs(x, xq[j], xsum[j]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) xr[j][i] = x[i];
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
      // INT4: the 4 code bytes of k vector kv and its group's (scale, zero) in row r
      const uint32_t *szs = reinterpret_cast<const uint32_t *>(stage + (size_t)SR * (K >> 1));
      auto q4_rows = [&](int kv, const float2 (&x2)[4], float xs, int m, float (&a)[SR][NB]) {
#pragma unroll
        for (int r = 0; r < SR; ++r)
          if (r < rows_here) {
            const uint32_t w = *reinterpret_cast<const uint32_t *>(stage + (size_t)r * (K >> 1) + (size_t)kv * 4);
            float2 f[4];
            q4_to_f32x2(w, f);
            a[r][m] = q4_dot(f, x2, xs, szs[(size_t)r * szw + (kv >> 4)], a[r][m]);
          }
      };
      if (xreg && Q4) {
#pragma unroll
        for (int j = 0; j < (NB == 1 && Q4 ? kXRegVecs : 0); ++j) {
          const int kv = tid + j * kGemvThreads;
          if (kv < KV) {
            if (H == 1 || kv < NVH)
              q4_rows(kv, xq[j], xsum[j], 0, acc[0]);
            else
              q4_rows(kv, xq[j], xsum[j], 0, acc[H - 1]);
          }
        }
      } else if (Q4) {
        // several items: each row's codes are decoded once, then used for every item
        for (int kv = tid; kv < KV; kv += kGemvThreads) {
          float2 wf[SR][4];
          uint32_t wsz[SR];
#pragma unroll
          for (int r = 0; r < SR; ++r) {
            uint32_t w = 0x88888888u;  // code 8 = weight zero: rows past the stage's end
            wsz[r] = 0u;
            if (r < rows_here) {
              w = *reinterpret_cast<const uint32_t *>(stage + (size_t)r * (K >> 1) + (size_t)kv * 4);
              wsz[r] = szs[(size_t)r * szw + (kv >> 4)];
            }
            q4_to_f32x2(w, wf[r]);
          }
          const int h = (H == 1 || kv < NVH) ? 0 : H - 1;
#pragma unroll
          for (int m = 0; m < NB; ++m) {
            float x[8], xs;
            float2 x2[4];
            load_x8<MODE>(xmem, KV, m, kv, x);
            q4_x_pairs(x, x2, xs);
#pragma unroll
            for (int r = 0; r < SR; ++r) {
              const float a0 = q4_dot(wf[r], x2, xs, wsz[r], 0.f);
              if (h == 0)
                acc[0][r][m] += a0;
              else
                acc[H - 1][r][m] += a0;
            }
          }
        }
      } else if (xreg) {
#pragma unroll
        for (int j = 0; j < (NB == 1 && !Q4 ? kXRegVecs : 0); ++j) {
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
// Most rows per ring stage: a stage's sums fit one warp reduction (32 / (NB * halves)),
// at most 8, and for INT4 with several items at most 2 / (NB / 2) so that the per-row sums
// and the decoded codes of a stage stay in registers (one item keeps 8 rows: the stage's
// fixed cost then spreads over more rows, which measured faster despite a few spilled
// registers).
template <int NB, int MODE, bool Q4>
constexpr int sr_max() {
  constexpr int a = 32 / (NB * ModeTraits<MODE>::kHalves) >= 8 ? 8 : 32 / (NB * ModeTraits<MODE>::kHalves);
  constexpr int q = NB == 1 ? 8 : (NB == 2 ? 2 : 1);
  return Q4 ? (a < q ? a : q) : a;
}

// Rows per ring stage: whole rows up to kStageBytes, at most 8, at most 32 / (NB * H) so
// that a stage's sums fit one warp reduction, and fewer if that keeps >= 4 stages.
template <int MODE, bool Q4>
static int stage_rows(int K, int NB, int max_rows, int row_bytes) {
  using T = ModeTraits<MODE>;
  int sr = kStageBytes / row_bytes;
  if (sr < 1) sr = 1;
  if (sr > 8) sr = 8;
  if (sr > 32 / (NB * T::kHalves)) sr = 32 / (NB * T::kHalves);
  if (Q4 && NB > 1 && sr > (NB == 2 ? 2 : 1)) sr = NB == 2 ? 2 : 1;
  int p2 = 1;
  while (p2 * 2 <= sr) p2 *= 2;
  while (p2 > 1) {
    const GemvSmem L = gemv_smem_layout(NB, p2, T::kHalves, T::kBf16X ? 2 : 4, K, 0, max_rows, row_bytes);
    const long long room = (long long)kGemvSmemLimit - L.total - 64;
    if (room / (p2 * row_bytes + 16) >= 4) break;
    p2 >>= 1;
  }
  return p2;
}

template <int NB, int SR, int MODE, bool Q4>
static cudaError_t launch_one(GemvParams p, int grid, int max_rows, cudaStream_t st, bool pdl) {
  using T = ModeTraits<MODE>;
  const int rb = gemv_row_bytes(Q4, p.K, p.sz_stride);
  const GemvSmem L0 = gemv_smem_layout(NB, SR, T::kHalves, T::kBf16X ? 2 : 4, p.K, 0, max_rows, rb);
  const long long room = (long long)kGemvSmemLimit - L0.total - 64;
  int nst = (int)(room / (SR * rb + 16));
  if (nst > 8) nst = 8;
  if (nst < 2) return cudaErrorInvalidValue;
  p.nstage = nst;
  const GemvSmem L = gemv_smem_layout(NB, SR, T::kHalves, T::kBf16X ? 2 : 4, p.K, nst, max_rows, rb);
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
  return cudaLaunchKernelEx(&cfg, gemv_kernel<NB, SR, MODE, Q4>, p);
}

template <int NB, int MODE, bool Q4>
static cudaError_t dispatch_sr(const GemvParams &p, int grid, cudaStream_t st, bool pdl) {
  using T = ModeTraits<MODE>;
  const int nunits = p.rows / T::kUnit;
  if (grid > nunits) grid = nunits;
  if (grid < 1) grid = 1;
  const int max_rows = T::kUnit * ((nunits + grid - 1) / grid);
  constexpr int SRMAX = sr_max<NB, MODE, Q4>();
  switch (stage_rows<MODE, Q4>(p.K, NB, max_rows, gemv_row_bytes(Q4, p.K, p.sz_stride))) {
    case 1: return launch_one<NB, 1, MODE, Q4>(p, grid, max_rows, st, pdl);
    case 2: return launch_one<NB, (SRMAX >= 2 ? 2 : 1), MODE, Q4>(p, grid, max_rows, st, pdl);
    case 4: return launch_one<NB, (SRMAX >= 4 ? 4 : 1), MODE, Q4>(p, grid, max_rows, st, pdl);
    default: return launch_one<NB, SRMAX, MODE, Q4>(p, grid, max_rows, st, pdl);
  }
}

template <int MODE, bool Q4>
static cudaError_t dispatch_nb(const GemvParams &p, int nb, int grid, cudaStream_t st, bool pdl) {
  switch (nb) {
    case 1: return dispatch_sr<1, MODE, Q4>(p, grid, st, pdl);
    case 2: return dispatch_sr<2, MODE, Q4>(p, grid, st, pdl);
    case 4: return dispatch_sr<4, MODE, Q4>(p, grid, st, pdl);
    case 8: return dispatch_sr<8, MODE, Q4>(p, grid, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

template <int NB, int MODE, bool Q4>
static cudaError_t prepare_nb() {
  using T = ModeTraits<MODE>;
  constexpr int SRMAX = sr_max<NB, MODE, Q4>();
  const int lim = (int)kGemvSmemLimit;
  cudaError_t e = cudaFuncSetAttribute(gemv_kernel<NB, 1, MODE, Q4>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemv_kernel<NB, (SRMAX >= 2 ? 2 : 1), MODE, Q4>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemv_kernel<NB, (SRMAX >= 4 ? 4 : 1), MODE, Q4>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemv_kernel<NB, SRMAX, MODE, Q4>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  return e;
}

template <int MODE, bool Q4>
static cudaError_t prepare_mode() {
  cudaError_t e = prepare_nb<1, MODE, Q4>();
  if (e == cudaSuccess) e = prepare_nb<2, MODE, Q4>();
  if (e == cudaSuccess) e = prepare_nb<4, MODE, Q4>();
  if (e == cudaSuccess) e = prepare_nb<8, MODE, Q4>();
  return e;
}


}  // namespace e3
