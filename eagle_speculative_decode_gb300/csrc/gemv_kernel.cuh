// Weight-streaming GEMV for the drafter's projections at small batch (items <= 8), as a
// template shared by the bf16 instantiations (gemv.cu) and the INT4 ones (gemv_q4.cu).
//
// y[item, row] = sum_k W[row, k] * x[item, k] with bf16 weights in [out, in] row-major
// and float32 activations/accumulators, fused with the op that feeds x (RMSNorm of the
// layer input, of x1 or of gsum; the embedding gather; the 2n concat) and the op that
// consumes y (partial RoPE + bf16 KV append, residual adds, SwiGLU, argmax + d2t).
// Ops follow "memra_engine/eagle.rs", module doc "Op-sequence".
//
// Data movement (one CTA per SM): rows are dealt to the CTAs in tiles of whole stages
// (pairs kept together), round robin, so that the SMs stream neighbouring parts of the
// weights at any moment.  A producer warp streams a CTA's rows, SR whole rows per stage
// (<= 32 KB), with bulk copies (cp.async.bulk, TMA) into a shared-memory ring of about
// 128 KB guarded by mbarriers.  It starts before the kernel waits on its predecessor (programmatic
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
// scale * sum((code - 8) x) + zero * sum(x).  Single-item INT4 launches with K a multiple
// of 2048 use the tensor-core variant below (gemv_q4_mma_kernel) instead.
#pragma once
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "epilogue.cuh"
#include "internal.h"

namespace e3 {

// -------------------------------------------------------------------- kernel
constexpr int kStageBytes = 32 * 1024;
// x vectors (8 k each) per item and thread that a launch keeps in registers: about 64
// registers of x in all (a bf16 vector takes 8, an INT4 one 9 with its sum), and no more
// than K = 3 * 512 * 8 = 12288 needs.  A launch whose K / 8 exceeds 512 times this reads x
// from shared memory per row instead.
__host__ __device__ constexpr int gemv_xreg_vecs(int nb, bool q4) {
  return nb == 1 ? 3 : nb == 2 ? 3 : nb == 4 ? 2 : 1;
}
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

// A launch's rows are dealt to the CTAs in tiles of TR rows, round robin (tile t to CTA
// t % grid), so that at any moment the SMs stream neighbouring parts of the weight
// matrices; the DRAM serves that faster than one distant contiguous range per SM.  Local
// row r of CTA b is row ((r / TR) * grid + b) * TR + r % TR; only the last tile of the
// launch can be partial, and it is the last tile of its CTA.
__host__ __device__ inline int tiles_max_rows(int rows, int TR, int grid) {
  const int nt = (rows + TR - 1) / TR;
  return (nt + grid - 1) / grid * TR;
}
__host__ __device__ inline int tiles_rows_of(int rows, int TR, int grid, int b) {
  const int nt = (rows + TR - 1) / TR;
  if (b >= nt) return 0;
  const int mine = (nt - b + grid - 1) / grid;
  const int last = b + (mine - 1) * grid;
  const int tail = rows - last * TR;
  return (mine - 1) * TR + (tail < TR ? tail : TR);
}
// The largest per-CTA row count over the tile sizes the GEMV uses (1 to 16 rows).
__host__ __device__ inline int tiles_max_rows_bound(int rows, int grid) {
  int m = 0;
  for (int tr = 1; tr <= 16; tr <<= 1) {
    const int v = tiles_max_rows(rows, tr, grid);
    m = v > m ? v : m;
  }
  return m;
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

// Tail shared by the GEMV kernels: the RMSNorm scale 1 / sqrt(mean(x^2) + eps) per item and
// K half from the consumers' shares ss, the per-warp row sums in part ([warps][H][NB][rows],
// rows prs apart: the threads that each add up one row read consecutive words, free of bank
// conflicts) added in warp order and scaled, then the mode's epilogue on the finished rows.
template <int NB, int MODE, int TR>
__device__ __forceinline__ void gemv_finish(const GemvParams &p, const float (&ss)[NB][ModeTraits<MODE>::kHalves],
                                            const float *part, int prs, float *accs, float *red, float *scale,
                                            int nrows) {
  using T = ModeTraits<MODE>;
  constexpr int H = T::kHalves;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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
      const float len = (float)(p.K / H);
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
      for (int w = 0; w < kGemvWarps; ++w) sum += part[(((size_t)w * H + h) * NB + m) * prs + r];
      y += T::kNorm ? sum * scale[m * H + h] : sum;
    }
    accs[e] = y;
  }
  consumer_sync();
  epilogue<NB, MODE, TR>(p, accs, nrows);
}

// A chain step's q/k/v whose previous lm_head left its argmax in the slots: CTA 0 writes
// that step's draft tokens and ids (its other CTAs decode the token themselves).
template <int MODE>
__device__ __forceinline__ void chain_prev_outputs(const GemvParams &p) {
  if constexpr (MODE == GM_QKV) {
    if (p.pairs.kind == PAIR_CHAIN && p.pairs.step_key && blockIdx.x == 0 && (int)threadIdx.x < p.items)
      chain_step_outputs(p.pairs.step_key, p.pairs.step - 1, p.item0 + (int)threadIdx.x, p.gamma, p.gamma_eff, p.d2t,
                         p.draft_vocab, p.target_vocab, p.draft_tok, p.draft_id, p.next_tok, p.status);
  }
}

template <int NB, int SR, int MODE, bool Q4>
__global__ void __launch_bounds__(kGemvCtaThreads, 1) gemv_kernel(const GemvParams p) {
  using T = ModeTraits<MODE>;
  constexpr int H = T::kHalves;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.K, KV = K >> 3;
  // rows are handed out in units of 2 where the epilogue pairs rows (RoPE, SwiGLU)
  // tiles of whole stages that keep row pairs (RoPE, SwiGLU) together
  constexpr int TR = SR >= T::kUnit ? SR : T::kUnit;
  const int nrows = tiles_rows_of(p.rows, TR, gridDim.x, blockIdx.x);
  const int max_rows = tiles_max_rows(p.rows, TR, gridDim.x);
  const int nst = p.nstage;
  const int szw = Q4 ? p.sz_stride : 0;  // (scale, zero) pairs per row
  constexpr int XRV = gemv_xreg_vecs(NB, Q4);
  const bool xreg = KV <= XRV * kGemvThreads;
  // several items with x in registers: x goes straight to registers, none in shared memory
  const bool xdirect = xreg && NB > 1;
  const GemvSmem L = gemv_smem_layout(NB, SR, H, xdirect ? 0 : (T::kBf16X ? 2 : 4), K, nst, max_rows,
                                      gemv_row_bytes(Q4, K, szw));
  const int n_stages = (nrows + SR - 1) / SR;
  const int NVH = H == 2 ? (p.n_embd >> 3) : KV;  // first vector of the second K half

  unsigned char *xmem = smem;
  unsigned char *ring = smem + L.ring_off;
  float *part = reinterpret_cast<float *>(smem + L.part_off);  // [warps][H][NB][max_rows]
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
          const RowRef rr = row_ref<MODE>(p, p.row_base + tile_row<TR>(st * SR + r));
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
  chain_prev_outputs<MODE>(p);
  float ss[NB][H];
  // x in registers: XRV 8-element vectors per item and thread (k = 8 (tid + 512 j)), so that
  // every weight vector read from the ring serves all items without x being re-read from
  // shared memory per row (with several items that re-read, not HBM, would set the pace);
  // such launches compute their x straight into registers.  Launches whose x does not fit
  // the register budget stage it in shared memory and read it per row.
  float xr[XRV][NB][8];                    // bf16 weights: x as computed
  float2 xq[Q4 ? XRV : 1][NB][4];          // INT4 weights: x in code pair order,
  float xsum[Q4 ? XRV : 1][NB];            // and its sums
  if (xdirect) {
    stage_x_regs<NB, MODE, XRV>(p, xr, ss);
  } else {
    stage_x<NB, MODE>(p, xmem, ss);
    consumer_sync();
    if (xreg) {
#pragma unroll
      for (int j = 0; j < XRV; ++j) {
        const int kv = tid + j * kGemvThreads;
#pragma unroll
        for (int m = 0; m < NB; ++m) {
          if (kv < KV) {
            load_x8<MODE>(xmem, KV, m, kv, xr[j][m]);
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) xr[j][m][i] = 0.f;
          }
        }
      }
    }
  }
  if constexpr (Q4) {
    if (xreg) {
#pragma unroll
      for (int j = 0; j < XRV; ++j)
#pragma unroll
        for (int m = 0; m < NB; ++m) q4_x_pairs(xr[j][m], xq[j][m], xsum[j][m]);
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
      // bf16: weight vector kv of every row of the stage against each item's x in registers
      auto fma_rows = [&](int kv, int j, float (&a)[SR][NB]) {
#pragma unroll
        for (int r = 0; r < SR; ++r)
          if (r < rows_here) {
            const uint4 w = *reinterpret_cast<const uint4 *>(stage + ((size_t)r * K + (size_t)kv * 8) * 2);
#pragma unroll
            for (int m = 0; m < NB; ++m) a[r][m] = dot8(w, xr[j][m], a[r][m]);
          }
      };
      // INT4: the 4 code bytes of k vector kv and its group's (scale, zero) in row r, decoded
      // once and used for every item
      const uint32_t *szs = reinterpret_cast<const uint32_t *>(stage + (size_t)SR * (K >> 1));
      auto q4_rows = [&](int kv, int j, float (&a)[SR][NB]) {
#pragma unroll
        for (int r = 0; r < SR; ++r)
          if (r < rows_here) {
            const uint32_t w = *reinterpret_cast<const uint32_t *>(stage + (size_t)r * (K >> 1) + (size_t)kv * 4);
            const uint32_t sz = szs[(size_t)r * szw + (kv >> 4)];
            float2 f[4];
            q4_to_f32x2(w, f);
#pragma unroll
            for (int m = 0; m < NB; ++m)
              a[r][m] = q4_dot(f, xq[Q4 ? j : 0][m], xsum[Q4 ? j : 0][m], sz, a[r][m]);
          }
      };
      if (xreg && Q4) {
#pragma unroll
        for (int j = 0; j < (Q4 ? XRV : 0); ++j) {
          const int kv = tid + j * kGemvThreads;
          if (kv < KV) {
            if (H == 1 || kv < NVH)
              q4_rows(kv, j, acc[0]);
            else
              q4_rows(kv, j, acc[H - 1]);
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
        for (int j = 0; j < (Q4 ? 0 : XRV); ++j) {
          const int kv = tid + j * kGemvThreads;
          if (kv < KV) {
            if (H == 1 || kv < NVH)
              fma_rows(kv, j, acc[0]);
            else
              fma_rows(kv, j, acc[H - 1]);
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
      if (lrow < nrows) part[(((size_t)warp * H + h) * NB + m) * max_rows + lrow] = tot;
    }
  }
  gemv_finish<NB, MODE, TR>(p, ss, part, max_rows, accs, red, scale, nrows);
}

// ------------------------------------- INT4, one item, on the tensor cores (mma.sync)
// Single-item INT4 launches with K a multiple of 2048 run the dot products as warp-level
// m16n8k16 fp16 MMAs.  The CUDA-core INT4 path spends several instructions per weight on
// decoding and multiply-adds and is bound by instruction issue; here 16 weight rows are
// the A operand and one MMA does 256 multiply-adds of a warp.  A code word becomes fp16
// pairs with one AND-OR each (0x64 is the exponent of 1024, whose 10-bit mantissa holds a
// nibble in bits 0-3 as 1024 + c and in bits 4-7 as 1024 + 16 c; one shift brings bytes 1
// and 3 down) and then c - 8 exactly by one packed fp16 add or multiply-add, which runs on
// the FMA pipe while the AND-ORs fill the ALU pipe.  The activations enter as three fp16
// parts x s = x0 + x1 + x2 in columns 0-2 of the n = 8 B operand, s a power of two per
// 128-input group that puts the group's largest |x| s in [2^14, 2^15) (no overflow, and
// the parts keep float32 accuracy); products are exact and the accumulators float32.  The
// row sums take scale / s * acc + zero * sum(x) per group.  The MMA reads its operands
// from registers, so the decoded codes feed it directly (a tcgen05 MMA would need them
// stored to shared or tensor memory first).
//
// A stage is one tile of 16 whole rows: their codes, their (scale, zero) rows and a 16-byte
// header giving the tile-local row of each of the 16 slots.  The producer ranks the tile's
// rows by their place in memory and copies each run of consecutive rows with one bulk copy
// (one or two runs per tile: all rows, or the two halves of RoPE / gate-up pairs), since
// many small copies stream far below the rate of a few large ones.  Warp w takes inputs
// [w K / 16, (w + 1) K / 16) of every row; lane (g, q) of the MMA fragments loads the 16
// bytes (32 codes) of rows g and g + 8 at inputs 128 G + 32 q of each of its groups G.  The
// order of the 16 inputs of one MMA is free as long as A and B follow the same one, and the
// B fragments are laid out in shared memory once per launch in that order, at
// xfrag[mma * 12 + 4 * part + q].
struct MmaSmem {
  int xfrag_off, gsum_off, ring_off, stage, part_off, accs_off, red_off, scale_off, bar_off, flag_off, total;
};

__host__ __device__ inline MmaSmem mma_smem_layout(int H, int K, int sz_stride, int nstage, int max_rows) {
  MmaSmem L;
  L.xfrag_off = K * 4;                  // float32 x planes (stage_x) first
  L.gsum_off = L.xfrag_off + K * 6;     // K / 16 MMAs x 12 lanes x 8 bytes
  L.ring_off = (L.gsum_off + (K / 128) * 16 + 127) / 128 * 128;
  L.stage = 16 * (K / 2) + 16 * sz_stride * 4 + 16;
  L.part_off = L.ring_off + nstage * L.stage;
  L.accs_off = L.part_off + max_rows * kGemvWarps * H * 4;
  L.red_off = L.accs_off + max_rows * 4;
  L.scale_off = L.red_off + kGemvWarps * H * 4;
  L.bar_off = (L.scale_off + H * 4 + 15) / 16 * 16;
  L.flag_off = L.bar_off + 2 * nstage * 8;
  L.total = L.flag_off + 16;
  return L;
}

// (lo, hi) -> fp16 pair, round to nearest even.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t u) {
  float2 f;
  asm("{\n .reg .f16 l, h;\n mov.b32 {l, h}, %2;\n cvt.f32.f16 %0, l;\n cvt.f32.f16 %1, h;\n}\n"
      : "=f"(f.x), "=f"(f.y)
      : "r"(u));
  return f;
}

// Three fp16 parts of (a, b), each the rounding of what the previous ones left.
__device__ __forceinline__ void split3_f16x2(float a, float b, uint32_t &p0, uint32_t &p1, uint32_t &p2) {
  p0 = pack_f16x2(a, b);
  float2 f = f16x2_to_f32x2(p0);
  a -= f.x;
  b -= f.y;
  p1 = pack_f16x2(a, b);
  f = f16x2_to_f32x2(p1);
  a -= f.x;
  b -= f.y;
  p2 = pack_f16x2(a, b);
}

// Eight INT4 codes of one 32-bit word as fp16 pairs c - 8 (exact), in the pair order
// (0, 4), (1, 5), (2, 6), (3, 7) of their k offsets.
__device__ __forceinline__ void q4_to_f16x2(uint32_t w, uint32_t (&r)[4]) {
  constexpr uint32_t e = 0x64006400u;              // 1024, 1024
  constexpr uint32_t lo_bias = 0xE408E408u;        // -1032, -1032
  constexpr uint32_t sixteenth = 0x2C002C00u;      // 1/16, 1/16
  constexpr uint32_t hi_bias = 0xD480D480u;        // -72, -72
  const uint32_t w8 = w >> 8;
  uint32_t t0 = (w & 0x000F000Fu) | e, t1 = (w & 0x00F000F0u) | e;    // 1024 + c, 1024 + 16 c
  uint32_t t2 = (w8 & 0x000F000Fu) | e, t3 = (w8 & 0x00F000F0u) | e;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r[0]) : "r"(t0), "r"(lo_bias));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r[1]) : "r"(t1), "r"(sixteenth), "r"(hi_bias));
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r[2]) : "r"(t2), "r"(lo_bias));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r[3]) : "r"(t3), "r"(sixteenth), "r"(hi_bias));
}

// d += A B for one m16n8k16 fp16 tile (A rows g / g + 8 in a0 a2 / a1 a3, B column g in
// b0 b1), float32 accumulators.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The B fragments and the per-group (sum(x), 1 / s) from the float32 x planes that
// stage_x wrote.  Vector v (inputs 8v .. 8v + 7) is word v % 4 of lane q = (v / 4) % 4 in
// group v / 16 (whose 16 vectors sit on 16 consecutive lanes, K being a multiple of 2048);
// its pairs (0, 4) .. (3, 7) are the B rows of MMAs 2 (v % 4) and 2 (v % 4) + 1.
__device__ __forceinline__ void mma_stage_b(const unsigned char *xmem, int K, uint2 *xfrag, float2 *gsum) {
  const int KV = K >> 3, lane = threadIdx.x & 31;
  const float4 *xa = reinterpret_cast<const float4 *>(xmem), *xb = xa + KV;
  for (int v = threadIdx.x; v < KV; v += kGemvThreads) {
    const float4 lo = xa[v], hi = xb[v];
    float mx = fmaxf(fmaxf(fmaxf(fabsf(lo.x), fabsf(lo.y)), fmaxf(fabsf(lo.z), fabsf(lo.w))),
                     fmaxf(fmaxf(fabsf(hi.x), fabsf(hi.y)), fmaxf(fabsf(hi.z), fabsf(hi.w))));
    float sum = ((lo.x + lo.y) + (lo.z + lo.w)) + ((hi.x + hi.y) + (hi.z + hi.w));
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      sum += __shfl_xor_sync(0xffffffffu, sum, o);
    }
    // s = 2^(141 - E) for a group maximum in [2^(E - 127), 2^(E - 126)): max * s in
    // [2^14, 2^15); exponents clamped to the normal range (an all-zero group takes s = 1)
    const int E = (int)((__float_as_uint(mx) >> 23) & 0xFFu);
    int es = E == 0 ? 127 : 268 - E;
    es = es < 1 ? 1 : (es > 253 ? 253 : es);
    const float sc = __uint_as_float((uint32_t)es << 23), inv = __uint_as_float((uint32_t)(254 - es) << 23);
    uint32_t p0[4], p1[4], p2[4];
    split3_f16x2(lo.x * sc, hi.x * sc, p0[0], p1[0], p2[0]);
    split3_f16x2(lo.y * sc, hi.y * sc, p0[1], p1[1], p2[1]);
    split3_f16x2(lo.z * sc, hi.z * sc, p0[2], p1[2], p2[2]);
    split3_f16x2(lo.w * sc, hi.w * sc, p0[3], p1[3], p2[3]);
    const int grp = v >> 4, q = (v >> 2) & 3, i = v & 3;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      uint2 *dst = xfrag + (size_t)(grp * 8 + 2 * i + t) * 12 + q;
      dst[0] = make_uint2(p0[2 * t], p0[2 * t + 1]);
      dst[4] = make_uint2(p1[2 * t], p1[2 * t + 1]);
      dst[8] = make_uint2(p2[2 * t], p2[2 * t + 1]);
    }
    if ((lane & 15) == 0) gsum[grp] = make_float2(sum, inv);
  }
}

template <int MODE, int NG>
__global__ void __launch_bounds__(kGemvCtaThreads, 1) gemv_q4_mma_kernel(const GemvParams p) {
  using T = ModeTraits<MODE>;
  constexpr int H = T::kHalves;
  constexpr int TR = 16;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = NG * 2048, CP = K / 2, SP = p.sz_stride * 4;  // NG 128-input groups per warp
  const int nrows = tiles_rows_of(p.rows, TR, gridDim.x, blockIdx.x);
  const int max_rows = tiles_max_rows(p.rows, TR, gridDim.x);
  const int nst = p.nstage;
  const MmaSmem L = mma_smem_layout(H, K, p.sz_stride, nst, max_rows);
  const int ntiles = (nrows + TR - 1) / TR;

  unsigned char *ring = smem + L.ring_off;
  uint2 *xfrag = reinterpret_cast<uint2 *>(smem + L.xfrag_off);
  float2 *gsum = reinterpret_cast<float2 *>(smem + L.gsum_off);
  float *part = reinterpret_cast<float *>(smem + L.part_off);  // [warps][H][max_rows]
  float *accs = reinterpret_cast<float *>(smem + L.accs_off);
  float *red = reinterpret_cast<float *>(smem + L.red_off);
  float *scale = reinterpret_cast<float *>(smem + L.scale_off);
  const uint32_t full0 = smem_addr(smem + L.bar_off);
  const uint32_t empty0 = full0 + 8 * nst;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.flag_off);
  const int hdr_off = 16 * CP + 16 * SP;  // slot -> tile-local row, 0xFF for none

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
    // lane r handles row r of the tile: its place in memory, its rank in memory order, and
    // (where it starts a run of consecutive rows) the bulk copies of the run
    const uint64_t pol = l2_evict_first_policy();
    int issued = 0;
    for (int st = 0; st < ntiles; ++st) {
      const int slot = st % nst;
      if (st >= nst) {
        int ok = 1;
        if (lane == 0) ok = mbar_wait(empty0 + 8 * slot, ((st / nst) - 1) & 1, abort_flag, p.status) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
      const int rows_here = min(TR, nrows - st * TR);
      unsigned char *stg = ring + (size_t)slot * L.stage;
      const bool live = lane < rows_here;
      RowRef rr = {0, 0};
      if (live) rr = row_ref<MODE>(p, p.row_base + tile_row<TR>(st * TR + lane));
      const unsigned long long key = live ? (((unsigned long long)rr.m << 40) | (unsigned long long)rr.row) : ~0ull;
      int pos = 0;  // rank of this row in memory order (keys of live rows are distinct)
#pragma unroll
      for (int j = 0; j < TR; ++j) pos += __shfl_sync(0xffffffffu, key, j) < key ? 1 : 0;
      if (live) stg[hdr_off + pos] = (unsigned char)lane;
      else if (lane < TR) stg[hdr_off + lane] = 0xFF;  // slots rows_here .. TR - 1 hold no row
      __syncwarp();
      const int prev = live && pos > 0 ? stg[hdr_off + pos - 1] : 0;
      const unsigned long long kprev = __shfl_sync(0xffffffffu, key, prev);
      const bool start = live && (pos == 0 || kprev + 1 != key);
      const unsigned starts = __reduce_or_sync(0xffffffffu, start ? (1u << pos) : 0u);
      const uint32_t full = full0 + 8 * slot, dst = smem_addr(stg);
      if (lane == 0) mbar_expect_tx(full, (uint32_t)rows_here * (uint32_t)(CP + SP));
      __syncwarp();
      if (start) {
        const unsigned later = starts & ~((2u << pos) - 1u);
        const int len = (later ? __ffs(later) - 1 : rows_here) - pos;
        bulk_g2s(dst + pos * CP, q4_codes(p, rr), (uint32_t)(len * CP), full, pol);
        bulk_g2s(dst + 16 * CP + pos * SP, q4_sz(p, rr), (uint32_t)(len * SP), full, pol);
      }
      issued = st + 1;
    }
    // Never leave copies in flight into shared memory: wait for the last stages issued.
    if (lane == 0)
      for (int st = max(0, issued - nst); st < issued; ++st)
        mbar_wait(full0 + 8 * (st % nst), (st / nst) & 1, abort_flag, p.status);
    return;
  }

  // ------------------------------------------------------------ consumer warps
  pdl_wait();
  chain_prev_outputs<MODE>(p);
  float ss[1][H];
  stage_x<1, MODE>(p, smem, ss);
  consumer_sync();
  mma_stage_b(smem, K, xfrag, gsum);
  consumer_sync();

  const int g = lane >> 2, q = lane & 3;
  // warps 0-7 cover the first K half, 8-15 the second (K = 2 n_embd where there are two)
  const int h = H == 2 && warp >= kGemvWarps / 2 ? 1 : 0;
  // The warp's B fragments and part sums are the same for every tile: up to two groups
  // per warp they stay in registers (lanes of columns 3-7 hold zeros); with more, the B
  // fragments of a group are loaded from shared memory when the group is processed.
  constexpr bool kBReg = NG <= 2;
  constexpr int NBR = kBReg ? NG : 1;
  uint32_t bx[NBR][8], by[NBR][8];
  auto load_b = [&](int G, uint32_t (&x)[8], uint32_t (&y)[8]) {
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const uint2 v = lane < 12 ? xfrag[(size_t)(G * 8 + m) * 12 + lane] : make_uint2(0u, 0u);
      x[m] = v.x;
      y[m] = v.y;
    }
  };
  float S[NG], inv_s[NG];  // sum(x) on lanes of column 0 (q = 0), else 0; 1 / s
#pragma unroll
  for (int j = 0; j < NG; ++j) {
    const int G = warp * NG + j;
    if constexpr (kBReg) load_b(G, bx[j], by[j]);
    const float2 gs = gsum[G];
    S[j] = q == 0 ? gs.x : 0.f;
    inv_s[j] = gs.y;
  }
  const int a_off = g * CP + warp * NG * 64 + q * 16, b_off = a_off + 8 * CP;
  const int sa_off = 16 * CP + g * SP + warp * NG * 4, sb_off = sa_off + 8 * SP;

  for (int st = 0; st < ntiles; ++st) {
    const int slot = st % nst;
    const bool ok = mbar_wait(full0 + 8 * slot, (st / nst) & 1, abort_flag, p.status);
    float tt[4] = {0.f, 0.f, 0.f, 0.f};
    int ra_row = 0xFF, rb_row = 0xFF;
    if (ok) {
      const unsigned char *stg = ring + (size_t)slot * L.stage;
      ra_row = stg[hdr_off + g];
      rb_row = stg[hdr_off + g + 8];
#pragma unroll
      for (int j = 0; j < NG; ++j) {
        // lane (g, q): 32 codes of rows g and g + 8 at inputs 128 G + 32 q
        const uint4 ca = *reinterpret_cast<const uint4 *>(stg + a_off + j * 64);
        const uint4 cb = *reinterpret_cast<const uint4 *>(stg + b_off + j * 64);
        const uint32_t sa = *reinterpret_cast<const uint32_t *>(stg + sa_off + j * 4);
        const uint32_t sb = *reinterpret_cast<const uint32_t *>(stg + sb_off + j * 4);
        // two accumulator chains (MMAs of even / odd t)
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t wa[4] = {ca.x, ca.y, ca.z, ca.w}, wb[4] = {cb.x, cb.y, cb.z, cb.w};
        const int jb = kBReg ? j : 0;
        if constexpr (!kBReg) load_b(warp * NG + j, bx[0], by[0]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t da[4], db[4];
          q4_to_f16x2(wa[i], da);
          q4_to_f16x2(wb[i], db);
          mma_16816(acc0, da[0], db[0], da[1], db[1], bx[jb][2 * i], by[jb][2 * i]);
          mma_16816(acc1, da[2], db[2], da[3], db[3], bx[jb][2 * i + 1], by[jb][2 * i + 1]);
        }
        const float fa = bf_lo(sa) * inv_s[j], fb = bf_lo(sb) * inv_s[j];
        tt[0] = fmaf(fa, acc0[0] + acc1[0], fmaf(bf_hi(sa), S[j], tt[0]));
        tt[1] = fmaf(fa, acc0[1] + acc1[1], tt[1]);
        tt[2] = fmaf(fb, acc0[2] + acc1[2], fmaf(bf_hi(sb), S[j], tt[2]));
        tt[3] = fmaf(fb, acc0[3] + acc1[3], tt[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * slot);
    // the tile's rows are complete: add the part columns and the four k-pair lanes
    float v0 = tt[0] + tt[1], v1 = tt[2] + tt[3];
    v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
    v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
    v0 += __shfl_xor_sync(0xffffffffu, v0, 2);
    v1 += __shfl_xor_sync(0xffffffffu, v1, 2);
    if (q == 0) {
#pragma unroll
      for (int hh = 0; hh < H; ++hh) {
        if (ra_row < TR) part[((size_t)warp * H + hh) * max_rows + st * TR + ra_row] = hh == h ? v0 : 0.f;
        if (rb_row < TR) part[((size_t)warp * H + hh) * max_rows + st * TR + rb_row] = hh == h ? v1 : 0.f;
      }
    }
  }
  gemv_finish<1, MODE, TR>(p, ss, part, max_rows, accs, red, scale, nrows);
}

// ------------------------------------------------------------------ launcher
// Ring depth: about 128 KB of weights in flight per SM (at least two stages).  Measured on
// the batch-1 chain: 64 KB 169.5, 96 KB 151.2, 128 KB 147.8 us per step, and the earlier
// room-limited ring (~200 KB) 152.3.
constexpr int kRingBytes = 128 * 1024;
inline int ring_stages_cap(int stage_bytes) {
  const int n = kRingBytes / stage_bytes;
  return n < 2 ? 2 : (n > 8 ? 8 : n);
}

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
// Whether a launch of several items keeps x in registers (then it has no copy of x in
// shared memory; one item still stages x there).
inline bool gemv_xreg(int K, int NB, bool q4) { return NB > 1 && K / 8 <= gemv_xreg_vecs(NB, q4) * kGemvThreads; }

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
    const GemvSmem L = gemv_smem_layout(NB, p2, T::kHalves, gemv_xreg(K, NB, Q4) ? 0 : (T::kBf16X ? 2 : 4), K, 0,
                                        max_rows, row_bytes);
    const long long room = (long long)kGemvSmemLimit - L.total - 64;
    if (room / (p2 * row_bytes + 16) >= 4) break;
    p2 >>= 1;
  }
  return p2;
}

template <int NB, int SR, int MODE, bool Q4>
static cudaError_t launch_one(GemvParams p, int grid, cudaStream_t st, bool pdl) {
  using T = ModeTraits<MODE>;
  constexpr int TR = SR >= T::kUnit ? SR : T::kUnit;
  grid = std::max(1, std::min(grid, (p.rows + TR - 1) / TR));
  const int max_rows = tiles_max_rows(p.rows, TR, grid);
  const int rb = gemv_row_bytes(Q4, p.K, p.sz_stride);
  const int xb = gemv_xreg(p.K, NB, Q4) ? 0 : (T::kBf16X ? 2 : 4);
  const GemvSmem L0 = gemv_smem_layout(NB, SR, T::kHalves, xb, p.K, 0, max_rows, rb);
  const long long room = (long long)kGemvSmemLimit - L0.total - 64;
  int nst = (int)(room / (SR * rb + 16));
  nst = std::min(nst, ring_stages_cap(SR * rb));
  if (nst < 2) return cudaErrorInvalidValue;
  p.nstage = nst;
  const GemvSmem L = gemv_smem_layout(NB, SR, T::kHalves, xb, p.K, nst, max_rows, rb);
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
  const int max_rows = tiles_max_rows_bound(p.rows, grid);
  constexpr int SRMAX = sr_max<NB, MODE, Q4>();
  switch (stage_rows<MODE, Q4>(p.K, NB, max_rows, gemv_row_bytes(Q4, p.K, p.sz_stride))) {
    case 1: return launch_one<NB, 1, MODE, Q4>(p, grid, st, pdl);
    case 2: return launch_one<NB, (SRMAX >= 2 ? 2 : 1), MODE, Q4>(p, grid, st, pdl);
    case 4: return launch_one<NB, (SRMAX >= 4 ? 4 : 1), MODE, Q4>(p, grid, st, pdl);
    default: return launch_one<NB, SRMAX, MODE, Q4>(p, grid, st, pdl);
  }
}

// Ring stages of the INT4 tensor-core GEMV for this launch (0: it does not apply: one item
// only, K a multiple of 2048, and x, its fragments and two whole-row tiles must fit in
// shared memory).  As many stages as fit, up to kQ4MmaMaxStages: the consumers hold a
// stage for about a thousand cycles of decoding and MMAs, so the ring must cover that as
// well as the DRAM latency.
constexpr int kQ4MmaMaxStages = 6;

template <int MODE>
static int q4_mma_stages(const GemvParams &p, int grid) {
  using T = ModeTraits<MODE>;
  if (T::kBf16X || p.K % 2048 || p.K > 4 * 2048 || p.items != 1) return 0;
  const int gr = std::max(1, std::min(grid, (p.rows + 15) / 16));
  const MmaSmem L0 = mma_smem_layout(T::kHalves, p.K, p.sz_stride, 0, tiles_max_rows(p.rows, 16, gr));
  const long long room = (long long)kGemvSmemLimit - L0.total - 64;
  int nst = (int)(room / (L0.stage + 16));
  nst = std::min(nst, kQ4MmaMaxStages);
  return nst >= 2 ? nst : 0;
}

template <int MODE>
static cudaError_t launch_q4_mma(GemvParams p, int grid, int nst, cudaStream_t st, bool pdl) {
  using T = ModeTraits<MODE>;
  grid = std::max(1, std::min(grid, (p.rows + 15) / 16));
  p.nstage = nst;
  const MmaSmem L = mma_smem_layout(T::kHalves, p.K, p.sz_stride, nst, tiles_max_rows(p.rows, 16, grid));
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
  switch (p.K / 2048) {
    case 1: return cudaLaunchKernelEx(&cfg, gemv_q4_mma_kernel<MODE, 1>, p);
    case 2: return cudaLaunchKernelEx(&cfg, gemv_q4_mma_kernel<MODE, 2>, p);
    case 3: return cudaLaunchKernelEx(&cfg, gemv_q4_mma_kernel<MODE, 3>, p);
    case 4: return cudaLaunchKernelEx(&cfg, gemv_q4_mma_kernel<MODE, 4>, p);
    default: return cudaErrorInvalidValue;
  }
}

template <int MODE, bool Q4>
static cudaError_t dispatch_nb(const GemvParams &p, int nb, int grid, cudaStream_t st, bool pdl) {
  if constexpr (Q4 && !ModeTraits<MODE>::kBf16X) {
    const int nst = nb == 1 ? q4_mma_stages<MODE>(p, grid) : 0;
    if (nst) return launch_q4_mma<MODE>(p, grid, nst, st, pdl);
  }
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
  if constexpr (Q4 && !ModeTraits<MODE>::kBf16X) {
    const int lim = (int)kGemvSmemLimit;
    const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
    if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_q4_mma_kernel<MODE, 1>, a, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_q4_mma_kernel<MODE, 2>, a, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_q4_mma_kernel<MODE, 3>, a, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_q4_mma_kernel<MODE, 4>, a, lim);
  }
  if (e == cudaSuccess) e = prepare_nb<2, MODE, Q4>();
  if (e == cudaSuccess) e = prepare_nb<4, MODE, Q4>();
  if (e == cudaSuccess) e = prepare_nb<8, MODE, Q4>();
  return e;
}


}  // namespace e3
