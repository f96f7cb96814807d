// GQA decode attention over the paged drafter KV cache (bf16 rows) on the tensor cores.
// The same operation as attention.cu ("memra_engine/eagle.rs", ``attn``: for each sequence
// b and q head h, softmax over keys 0..len-1 of (q . k) / sqrt(d), then sum of p * v) and
// the same persistent stream-K schedule over units of U keys (attn_sched.cuh).
//
// Per unit (U <= 64 keys of one (sequence, kv head) pair, K and V rows brought into shared
// memory by 128-byte-swizzled tensor-map boxes, 64 dims x U rows each):
//  * scores: warp w takes keys 8w .. 8w + 7 against all dims with warp-level
//    mma.sync.m16n8k16 bf16 MMAs.  The A operand is q in three exact bf16 parts
//    (q = q0 + q1 + q2, float32's 24 bits), rows r = 4 p + h for part p of head h (rows of
//    part 3 and of heads >= G are zero); the B operand is the keys' bf16 rows.  A head's
//    score is the sum of its three part rows: products are exact and sums float32.
//  * softmax: per-warp maxima and sums meet in shared memory; every thread keeps each
//    head's running max (log2 domain) and sum.
//  * values: the probabilities p, again in three bf16 parts (rows 4 q + h), go to shared
//    memory; warp w takes dims [w d / 8, (w + 1) d / 8) over all the unit's keys, B = the
//    value rows (ldmatrix with transpose), accumulating float32 in registers.
// At the end of a pair's run of units the three part rows are added; a pair whose units
// all fall to this CTA is written out at once, otherwise its (max, sum, weighted V) is
// published and the last contributing CTA merges the contributions in CTA order, as in
// attention.cu.  Every mbarrier wait is bounded, and no copy is left in flight when the
// CTA finishes.
#include <cuda.h>
#include <math.h>

#include "attn_sched.cuh"
#include "common.cuh"
#include "internal.h"

namespace e3 {

// 2-D bf16 tensor map, box of 64 columns x box_rows rows, 128-byte swizzle (gemm_tc.cu).
bool tc_make_map(CUtensorMap *map, const void *base, int rows, int cols, int box_rows);

constexpr int kAtcWarps = 8;                         // consumer warps
constexpr int kAtcThreads = kAtcWarps * 32;
constexpr int kAtcCtaThreads = kAtcThreads + 32;     // + one producer warp
constexpr int kAtcStages = 3;
constexpr int kAtcMaxU = 64;                         // keys per unit: 8 per consumer warp
constexpr int kAtcScratch = 12 * 1024;               // cross-CTA merge scratch

struct AttnTcArgs {
  AttnParams p;
  CUtensorMap kmap;  // K pool as [num_pages * H_kv * page_size][d] bf16, box 64 x U, 128B swizzle
  CUtensorMap vmap;  // V pool, the same
};

template <int D, int G>
struct AtcShape {
  static constexpr int kUnitBytes = kAtcMaxU * D * 2;            // K (or V) of a full unit
  static constexpr int kStage = 2 * kUnitBytes;
  static constexpr int PS = kAtcMaxU + 8;                          // P row stride (bf16), padded
  static constexpr int kP = 16 * PS * 2;                           // one P buffer
  static constexpr int kRingOff = 0;
  static constexpr int kPOff = kAtcStages * kStage;                // two P buffers
  static constexpr int kRedOff = kPOff + 2 * kP;                   // max / sum exchange [2][2][8][4]
  static constexpr int kScrOff = kRedOff + 2 * 2 * kAtcWarps * 4 * 4;
  static constexpr int kBarOff = kScrOff + kAtcScratch;
  static constexpr int kSmem = kBarOff + 2 * kAtcStages * 8 + 16 + 1024;  // + alignment slack
  static_assert(kSmem <= 227 * 1024, "attention shared memory");
  static constexpr int NT = D / 64;                                // PV n-tiles of 8 dims per warp
  static constexpr int kMaxContrib = (kAtcScratch - 64) / (G * 12 + 4);
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ void atc_tma_load(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar,
                                             uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t &r0, uint32_t &r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// d += a * b, m16n8k16, bf16 operands, float32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// x split into three bf16 parts x0 + x1 + x2 (both differences exact); part p of x.
__device__ __forceinline__ uint16_t bf16_part(float x, int p) {
  const uint16_t u0 = f2bf(x);
  if (p == 0) return u0;
  const float r1 = x - bf1(u0);
  const uint16_t u1 = f2bf(r1);
  if (p == 1) return u1;
  return f2bf(r1 - bf1(u1));
}
// Shared-memory address of 16-byte chunk c (8 dims) of row r in a unit laid out as
// 128-byte-swizzled boxes of 64 dims x U rows (chunk cc of a row at cc ^ (row % 8)).
__device__ __forceinline__ uint32_t atc_chunk(uint32_t base, int U, int r, int c) {
  return base + (uint32_t)((c >> 3) * U * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

template <int D, int G>
__global__ void __launch_bounds__(kAtcCtaThreads, 1) attn_tc_kernel(const __grid_constant__ AttnTcArgs args) {
  using S = AtcShape<D, G>;
  constexpr int NT = S::NT, PS = S::PS;
  const AttnParams &p = args.p;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  float *red = reinterpret_cast<float *>(smem + S::kRedOff);  // [buf][max, sum][warp][head]
  unsigned char *scr = smem + S::kScrOff;
  const uint32_t full0 = smem_addr(smem + S::kBarOff);
  const uint32_t empty0 = full0 + 8 * kAtcStages;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kBarOff + 2 * kAtcStages * 8);
  __shared__ int last_sh;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = p.n_head, Hkv = p.n_head_kv, ps = p.page_size, U = p.unit_keys;
  AttnSched sch;
  sch.pre = p.unit_pre;
  sch.B = p.batch;
  sch.Hkv = Hkv;
  sch.total = (long long)Hkv * sch.pre[p.batch];
  sch.grid = (int)min((long long)gridDim.x, sch.total);
  const int cta = blockIdx.x;
  const long long u_begin = cta < sch.grid ? sch.start(cta) : 0, u_end = cta < sch.grid ? sch.start(cta + 1) : 0;

  if (tid == 0) {
    for (int i = 0; i < kAtcStages; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, kAtcWarps);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  // the P buffers' rows of part 3 and of heads >= G stay zero
  for (int i = tid; i < 2 * S::kP / 4; i += kAtcCtaThreads) reinterpret_cast<uint32_t *>(smem + S::kPOff)[i] = 0u;
  __syncthreads();
  pdl_trigger();
  if (u_begin >= u_end) {  // a CTA beyond the unit count: nothing to do
    pdl_wait();
    return;
  }

  // keys of sequence b: the estimate before gamma_eff is read (committed + step + 1) fixes
  // the unit partition; the final length (after the wait) trims the last unit.
  auto est_len = [&](int b) {
    const int L = p.kv_len[b];
    int len = L + p.step + 1;
    if (len > p.max_cache_len) len = p.max_cache_len;
    return len < 1 ? 1 : len;
  };
  auto final_len = [&](int b) {
    const int L = p.kv_len[b];
    const int ge = p.gamma_eff ? p.gamma_eff[b] : p.step + 1;
    int len2 = L + min(p.step, max(ge - 1, 0)) + 1;
    if (L < 0 || len2 > p.max_cache_len) len2 = min(max(len2, 1), p.max_cache_len);
    return min(est_len(b), len2);
  };

  if (warp == kAtcWarps) {
    // ---------------------------------------------------------- producer warp
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      bool waited = false;
      int g = 0;
      bool ok = true;
      for (long long u = u_begin; u < u_end && ok;) {
        const AttnSeg sg = attn_seg(sch, u, u_end);
        u += sg.r1 - sg.r0;
        const int L = p.kv_len[sg.b], est = est_len(sg.b);
        const int32_t *pt = p.page_table + (size_t)sg.b * p.max_pages;
        for (int r = sg.r0; r < sg.r1; ++r) {
          const int k0 = r * U;
          int k1 = min(k0 + U, est);
          if (k1 > L) {  // this unit holds keys written by the chain: wait for them
            if (!waited) {
              pdl_wait();
              waited = true;
            }
            k1 = min(k1, final_len(sg.b));
          }
          if (k1 <= k0) continue;  // trimmed away: the consumers skip it too
          const int slot = g % kAtcStages;
          if (g >= kAtcStages && !mbar_wait(empty0 + 8 * slot, ((g / kAtcStages) - 1) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const int pg = pt[k0 / ps];
          const uint32_t bytes = (uint32_t)(2 * U * D * 2);
          mbar_expect_tx(full0 + 8 * slot, bytes);
          if (pg < 0 || pg >= p.num_pages) {
            // keep the ring in step: complete the stage without data (consumers skip it)
            set_status(p.status, EAGLE3_DEV_BAD_PAGE);
            asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(full0 + 8 * slot), "r"(bytes) : "memory");
          } else {
            // the unit's U rows: one 64-dim box of K and of V per 64 dims
            const int row = (pg * Hkv + sg.kvh) * ps + k0 % ps;
            const uint32_t kdst = smem_addr(smem + (size_t)slot * S::kStage);
            const uint32_t vdst = kdst + (uint32_t)(U * D * 2);
#pragma unroll
            for (int bx = 0; bx < D / 64; ++bx) {
              atc_tma_load(kdst + (uint32_t)(bx * U * 128), &args.kmap, bx * 64, row, full0 + 8 * slot, pol);
              atc_tma_load(vdst + (uint32_t)(bx * U * 128), &args.vmap, bx * 64, row, full0 + 8 * slot, pol);
            }
          }
          ++g;
        }
      }
      // no copy may still be in flight when the CTA moves on
      for (int i = max(0, g - kAtcStages); i < g; ++i)
        mbar_wait(full0 + 8 * (i % kAtcStages), (i / kAtcStages) & 1, abort_flag, p.status);
      if (!waited) pdl_wait();
    }
    __syncwarp();
    return;
  }

  // ------------------------------------------------------------ consumer warps
  pdl_wait();
  const float qscale = rsqrtf((float)D) * 1.4426950408889634f;
  const int gq = lane >> 2, qq = lane & 3;   // mma fragment coordinates
  const int hA = gq & 3;                     // head of this thread's fragment rows
  const int pA0 = gq >> 2, pA1 = 2 + (gq >> 2);  // parts of rows gq and gq + 8
  const bool rowA = hA < G;
  const uint32_t pbase0 = smem_addr(smem + S::kPOff);
  int g = 0;
  for (long long u = u_begin; u < u_end;) {
    const AttnSeg sg = attn_seg(sch, u, u_end);
    u += sg.r1 - sg.r0;
    const int b = sg.b, kvh = sg.kvh;
    const int est = est_len(b), fin = final_len(b), L = p.kv_len[b];
    const int32_t *pt = p.page_table + (size_t)b * p.max_pages;
    // q of the kv head's G query heads as the QK A operand, one fragment per 16 dims:
    // rows gq (part pA0) and gq + 8 (part pA1; part 3 is zero), head hA
    uint32_t qa[D / 16][4];
    {
      const float *qh = p.q + (size_t)b * H * D + (size_t)(kvh * G + (rowA ? hA : 0)) * D;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const float2 lo = rowA ? __ldcg(reinterpret_cast<const float2 *>(qh + ks * 16 + 2 * qq)) : make_float2(0.f, 0.f);
        const float2 hi = rowA ? __ldcg(reinterpret_cast<const float2 *>(qh + ks * 16 + 8 + 2 * qq)) : make_float2(0.f, 0.f);
        const float x0 = lo.x * qscale, x1 = lo.y * qscale, x2 = hi.x * qscale, x3 = hi.y * qscale;
        auto pack = [](uint16_t a, uint16_t c) { return (uint32_t)a | ((uint32_t)c << 16); };
        qa[ks][0] = pack(bf16_part(x0, pA0), bf16_part(x1, pA0));
        qa[ks][2] = pack(bf16_part(x2, pA0), bf16_part(x3, pA0));
        if (pA1 < 3) {
          qa[ks][1] = pack(bf16_part(x0, pA1), bf16_part(x1, pA1));
          qa[ks][3] = pack(bf16_part(x2, pA1), bf16_part(x3, pA1));
        } else {
          qa[ks][1] = 0u;
          qa[ks][3] = 0u;
        }
      }
    }
    float m_run[G], l_run[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m_run[h] = -INFINITY;
      l_run[h] = 0.f;
    }
    float oacc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) oacc[nt][i] = 0.f;

    for (int r = sg.r0; r < sg.r1; ++r) {
      const int k0 = r * U;
      int k1 = min(k0 + U, est);
      if (k1 > L) k1 = min(k1, fin);
      if (k1 <= k0) continue;
      const int n = k1 - k0;
      const int slot = g % kAtcStages, buf = g & 1;
      const bool ok = mbar_wait(full0 + 8 * slot, (g / kAtcStages) & 1, abort_flag, p.status);
      ++g;
      const int pg = pt[k0 / ps];
      const bool have = __all_sync(0xffffffffu, ok) && pg >= 0 && pg < p.num_pages;
      const uint32_t kbase = smem_addr(smem + (size_t)slot * S::kStage);
      const uint32_t vbase = kbase + (uint32_t)(U * D * 2);
      const uint32_t pbuf = pbase0 + (uint32_t)(buf * S::kP);
      float *rmax = red + buf * 2 * kAtcWarps * 4, *rsum = rmax + kAtcWarps * 4;

      // ---- scores of keys 8 warp .. +7 (this warp's n-tile)
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
      const int kw = 8 * warp;
      if (have && kw < n) {
        // four independent accumulator chains over the k-steps, added at the end
        constexpr int NC = D / 16 >= 4 ? 4 : D / 16;
        float sc[NC][4];
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
          for (int i = 0; i < 4; ++i) sc[c][i] = 0.f;
        const int krow = kw + (lane & 7);  // ldmatrix row address of lanes 0-15
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t b0, b1;
          ldsm_x2(atc_chunk(kbase, U, krow, 2 * ks + ((lane >> 3) & 1)), b0, b1);
          mma_bf16(sc[ks % NC], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
        }
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
          for (int i = 0; i < 4; ++i) sacc[i] += sc[c][i];
      }
      // a head's score = its part rows 0 and 2 (this lane) + part row 1 (lane + 16)
      const float up0 = __shfl_down_sync(0xffffffffu, sacc[0], 16);
      const float up1 = __shfl_down_sync(0xffffffffu, sacc[1], 16);
      const int key0 = kw + 2 * qq;
      const bool own = lane < 16 && rowA && have;  // lanes holding a head's scores
      float s0 = own && key0 < n ? sacc[0] + sacc[2] + up0 : -INFINITY;
      float s1 = own && key0 + 1 < n ? sacc[1] + sacc[3] + up1 : -INFINITY;
      float wm = fmaxf(s0, s1);
      wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, 1));
      wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, 2));
      if (lane < 16 && qq == 0 && rowA) rmax[warp * 4 + hA] = wm;
      asm volatile("bar.sync 1, 256;" ::: "memory");
      float m_new[G], corr[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float m = m_run[h];
#pragma unroll
        for (int w = 0; w < kAtcWarps; ++w) m = fmaxf(m, rmax[w * 4 + h]);
        m_new[h] = m;
        corr[h] = m == -INFINITY ? 1.f : exp2f(m_run[h] - m);
        m_run[h] = m;
      }
      // ---- probabilities of this lane's two keys, in three bf16 parts, into P rows 4 part + head
      {
        float mh = m_new[0];
#pragma unroll
        for (int h = 1; h < G; ++h)
          if (hA == h) mh = m_new[h];
        const float p0 = (s0 == -INFINITY) ? 0.f : exp2f(s0 - mh);
        const float p1 = (s1 == -INFINITY) ? 0.f : exp2f(s1 - mh);
        if (lane < 16 && rowA && kw < U) {
#pragma unroll
          for (int part = 0; part < 3; ++part) {
            const uint32_t v = (uint32_t)bf16_part(p0, part) | ((uint32_t)bf16_part(p1, part) << 16);
            *reinterpret_cast<uint32_t *>(smem + S::kPOff + buf * S::kP + ((4 * part + hA) * PS + key0) * 2) = v;
          }
        }
        float ps2 = p0 + p1;
        ps2 += __shfl_xor_sync(0xffffffffu, ps2, 1);
        ps2 += __shfl_xor_sync(0xffffffffu, ps2, 2);
        if (lane < 16 && qq == 0 && rowA) rsum[warp * 4 + hA] = ps2;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kAtcWarps; ++w) sum += rsum[w * 4 + h];
        l_run[h] = l_run[h] * corr[h] + sum;
      }
      // ---- values: this warp's dims over all the unit's keys
      {
        float ch = corr[0];
#pragma unroll
        for (int h = 1; h < G; ++h)
          if (hA == h) ch = corr[h];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) oacc[nt][i] *= ch;
      }
      if (have) {
        const int c0 = warp * (D / 64);  // first 8-dim chunk of this warp's dims
        for (int kb = 0; kb < U; kb += 16) {
          // A: P rows 0-15 x keys kb .. kb + 15 (four 8x8 tiles)
          uint32_t pa[4];
          {
            const int m = lane >> 3, rr = lane & 7;
            const int prow = (m & 1) * 8 + rr, pcol = kb + (m >> 1) * 8;
            ldsm_x4(pbuf + (uint32_t)((prow * PS + pcol) * 2), pa);
          }
          const int m = lane >> 3, rr = lane & 7;
          const int vrow = kb + (m & 1) * 8 + rr;
          if constexpr (NT == 1) {
            // B: value rows kb .. kb + 15 of this warp's 8 dims (transposed tiles)
            uint32_t b0, b1;
            ldsm_x2_t(atc_chunk(vbase, U, vrow, c0), b0, b1);
            mma_bf16(oacc[0], pa[0], pa[1], pa[2], pa[3], b0, b1);
          } else {
#pragma unroll
            for (int nt = 0; nt < NT; nt += 2) {
              // B: value rows kb .. kb + 15, dims of n-tiles nt and nt + 1 (transposed tiles)
              uint32_t vb[4];
              ldsm_x4_t(atc_chunk(vbase, U, vrow, c0 + nt + (m >> 1)), vb);
              mma_bf16(oacc[nt], pa[0], pa[1], pa[2], pa[3], vb[0], vb[1]);
              mma_bf16(oacc[nt + 1], pa[0], pa[1], pa[2], pa[3], vb[2], vb[3]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * slot);
    }

    // ---- end of this CTA's units of pair (b, kvh): a head's weighted V = its part rows
    const bool whole = sg.r0 == 0 && sg.r1 == sg.nu;
    float *out = p.out + (size_t)b * H * D + (size_t)kvh * G * D;
    const int mine = cta * 2 + (sch.start(cta) >= sg.pair_u0 ? 0 : 1);  // partial slot
    float lh = l_run[0], mh = m_run[0];
#pragma unroll
    for (int h = 1; h < G; ++h)
      if (hA == h) {
        lh = l_run[h];
        mh = m_run[h];
      }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float u0 = __shfl_down_sync(0xffffffffu, oacc[nt][0], 16);
      const float u1 = __shfl_down_sync(0xffffffffu, oacc[nt][1], 16);
      if (lane < 16 && rowA) {
        const int dim = warp * (D / 8) + nt * 8 + 2 * qq;
        const float o0 = oacc[nt][0] + oacc[nt][2] + u0, o1 = oacc[nt][1] + oacc[nt][3] + u1;
        if (whole) {
          const float inv = 1.0f / lh;
          *reinterpret_cast<float2 *>(out + (size_t)hA * D + dim) = make_float2(o0 * inv, o1 * inv);
        } else {
          *reinterpret_cast<float2 *>(p.part_o + (size_t)mine * G * D + (size_t)hA * D + dim) = make_float2(o0, o1);
        }
      }
    }
    if (!whole && tid == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) p.part_ml[(size_t)mine * G + h] = make_float2(m_run[h], l_run[h]);
    }
    if (whole) continue;

    // ---- a pair shared with other CTAs: the last of them merges, in CTA order
    const int pair = b * Hkv + kvh;
    const long long pu0 = sg.pair_u0, pu1 = sg.pair_u0 + sg.nu;
    const int c_first = sch.cta_of(pu0), c_last = sch.cta_of(pu1 - 1);
    __threadfence();
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (tid == 0) {
      const unsigned prev = atomicAdd(p.count + pair, 1u);
      last_sh = prev == (unsigned)(c_last - c_first) ? 1 : 0;
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (!last_sh) continue;
    __threadfence();
    const int nc = c_last - c_first + 1;
    float2 *ml_s = reinterpret_cast<float2 *>(scr);        // [nc][G]
    float *w_s = reinterpret_cast<float *>(ml_s + nc * G);  // [nc][G]
    int *slot_s = reinterpret_cast<int *>(w_s + nc * G);    // [nc]
    float2 *ML = reinterpret_cast<float2 *>((reinterpret_cast<uintptr_t>(slot_s + nc) + 7) & ~(uintptr_t)7);  // [G]
    for (int i = tid; i < nc; i += kAtcThreads) {
      const int c2 = c_first + i;
      slot_s[i] = c2 * 2 + (sch.start(c2) >= pu0 ? 0 : 1);
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    for (int i = tid; i < nc * G; i += kAtcThreads) ml_s[i] = __ldcg(&p.part_ml[(size_t)slot_s[i / G] * G + i % G]);
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (tid < G) {
      float M = -INFINITY;
      for (int q = 0; q < nc; ++q) M = fmaxf(M, ml_s[q * G + tid].x);
      float Ls = 0.f;
      for (int q = 0; q < nc; ++q)
        if (ml_s[q * G + tid].x != -INFINITY) Ls += ml_s[q * G + tid].y * exp2f(ml_s[q * G + tid].x - M);
      ML[tid] = make_float2(M, 1.0f / Ls);
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    for (int i = tid; i < nc * G; i += kAtcThreads) {
      const float2 ml = ml_s[i];
      const int gg = i % G;
      w_s[i] = ml.x == -INFINITY ? 0.f : exp2f(ml.x - ML[gg].x) * ML[gg].y;
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    const float4 *po = reinterpret_cast<const float4 *>(p.part_o);
    float4 *out4 = reinterpret_cast<float4 *>(out);
    for (int f = tid; f < G * D / 4; f += kAtcThreads) {
      const int gg = (f * 4) / D;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      int q = 0;
      for (; q + 8 <= nc; q += 8) {
        float4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = __ldcg(po + (size_t)slot_s[q + k] * (G * D / 4) + f);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float w = w_s[(q + k) * G + gg];
          o.x = fmaf(w, v[k].x, o.x); o.y = fmaf(w, v[k].y, o.y);
          o.z = fmaf(w, v[k].z, o.z); o.w = fmaf(w, v[k].w, o.w);
        }
      }
      for (; q < nc; ++q) {
        const float4 v = __ldcg(po + (size_t)slot_s[q] * (G * D / 4) + f);
        const float w = w_s[q * G + gg];
        o.x = fmaf(w, v.x, o.x); o.y = fmaf(w, v.y, o.y);
        o.z = fmaf(w, v.z, o.z); o.w = fmaf(w, v.w, o.w);
      }
      out4[f] = o;
    }
    if (tid == 0) p.count[pair] = 0u;
    asm volatile("bar.sync 1, 256;" ::: "memory");  // the scratch is free again
  }
}

// ------------------------------------------------------------------ host side
// bf16 KV with 16 <= U <= 64 keys per unit (a multiple of 16), G <= 4 and d in {64, 128, 256}
bool attn_tc_supported(int head_dim, int group, int unit_keys) {
  return (head_dim == 64 || head_dim == 128 || head_dim == 256) && (group == 1 || group == 2 || group == 4) &&
         unit_keys >= 16 && unit_keys <= kAtcMaxU && unit_keys % 16 == 0;
}

template <int D, int G>
static cudaError_t attn_tc_launch_dg(const AttnParams &p, int num_sms, cudaStream_t st, bool pdl) {
  using S = AtcShape<D, G>;
  AttnTcArgs a;
  memset(&a, 0, sizeof(a));
  a.p = p;
  const int rows = p.num_pages * p.n_head_kv * p.page_size;
  if (!tc_make_map(&a.kmap, p.k_pool, rows, D, p.unit_keys) || !tc_make_map(&a.vmap, p.v_pool, rows, D, p.unit_keys))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms < S::kMaxContrib ? num_sms : S::kMaxContrib);
  cfg.blockDim = dim3(kAtcCtaThreads);
  cfg.dynamicSmemBytes = S::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_tc_kernel<D, G>, a);
}

#define E3_ATC_ALL(X) X(64, 1) X(64, 2) X(64, 4) X(128, 1) X(128, 2) X(128, 4) X(256, 1) X(256, 2) X(256, 4)

cudaError_t attn_tc_prepare() {
  cudaError_t e = cudaSuccess;
#define E3_ATC_PREP(DD, GG)                                                                             \
  if (e == cudaSuccess)                                                                                 \
    e = cudaFuncSetAttribute(attn_tc_kernel<DD, GG>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             AtcShape<DD, GG>::kSmem);
  E3_ATC_ALL(E3_ATC_PREP)
#undef E3_ATC_PREP
  return e;
}

cudaError_t attn_tc_launch(const AttnParams &p, int num_sms, cudaStream_t st, bool pdl) {
  const int G = p.n_head / p.n_head_kv;
  if (p.batch < 1 || p.kv_q || !p.unit_pre || !attn_tc_supported(p.head_dim, G, p.unit_keys))
    return cudaErrorInvalidValue;
#define E3_ATC_CASE(DD, GG) \
  if (p.head_dim == DD && G == GG) return attn_tc_launch_dg<DD, GG>(p, num_sms, st, pdl);
  E3_ATC_ALL(E3_ATC_CASE)
#undef E3_ATC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace e3
