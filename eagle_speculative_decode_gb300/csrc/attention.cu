// GQA decode attention over the paged drafter KV cache, bf16 or quantized (q8_0 K, q5_1
// V; a K block's scale multiplies the partial dot once, V = d * code + m with the p * m
// terms summed apart).
//
// For each sequence b and q head h (kv head h / G, G = n_head / n_head_kv): softmax over
// the keys 0..len-1 of (q . k) / sqrt(d), then sum of p * v ("memra_engine/eagle.rs",
// ``attn``: fa_decode with scale 1/sqrt(head_dim); the new key is appended first).
//
// Persistent stream-K schedule: the keys of every (sequence, kv head) pair are cut into
// units of U consecutive positions inside one page (U = min(64-ish run, the largest power
// of two dividing the page size)), and one CTA per SM takes an equal share of all units in
// (sequence, kv head, unit) order, so ragged lengths and any batch fill the GPU evenly.
// Inside a CTA, a producer warp streams the K rows and V rows of each unit -- contiguous
// in the paged pool -- with bulk copies (TMA) into a 3-stage shared-memory ring guarded by
// mbarriers, across pair boundaries without a pause.  Units below the committed length
// were written before the chain started, so they are requested before the kernel waits
// on its predecessor (programmatic dependent launch); for the others, the lengths and the
// page-table entry (also fixed before the chain) are read before that wait, so only the
// copy itself follows it.
//
// Eight consumer warps take UNR keys per lane group of each unit (a key of d = 256 dims
// spans a warp, 8 dims = 16 bytes per lane; smaller heads put several keys in a warp).
// The UNR x G partial scores are reduced across the lane group in one transposed
// reduction: each lane ends with one full score and takes its exponential, and the
// probabilities are broadcast for the V update.  An online softmax per head keeps the
// running max (log2 domain), sum and weighted V.  At the end of a pair's run of units the
// CTA merges its lane groups in shared memory; a pair whose units all fall to this CTA is
// written out at once, otherwise its (max, sum, weighted V) is published and the last
// contributing CTA merges the contributions in CTA order.
#include <cuda_fp16.h>
#include <math.h>

#include "attn_sched.cuh"
#include "common.cuh"
#include "internal.h"

namespace e3 {

constexpr int kAttnWarps = 8;                          // consumer warps
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kAttnCtaThreads = kAttnThreads + 32;     // + one producer warp
constexpr int kAttnStages = 3;

template <int X>
struct ILog2 {
  static constexpr int value = X <= 1 ? 0 : 1 + ILog2<X / 2>::value;
};
template <>
struct ILog2<1> {
  static constexpr int value = 0;
};

template <int D, int G, bool KVQ>
struct AttnShape {
  // bytes of one key's K and V row: bf16, or q8_0 / q5_1 blocks of 32 values
  static constexpr int KR = KVQ ? D / 32 * 34 : D * 2;
  static constexpr int VR = KVQ ? D / 32 * 24 : D * 2;
  static constexpr int LPK = D / 8;             // lanes per key (a segment of the warp)
  static constexpr int KPW = 32 / LPK;          // keys per warp pass
  static constexpr int NP = kAttnWarps * KPW;   // lane groups per CTA
  // keys per lane group per unit; UNR * G partial scores fit one segment reduction
  static constexpr int UNR = (LPK / G) < 8 ? (LPK / G < 1 ? 1 : LPK / G) : 8;
  static constexpr int N = UNR * G;
  static constexpr int SH = ILog2<LPK>::value - ILog2<N>::value;  // lane bits below a score index
  static constexpr int LOG_G = ILog2<G>::value;
  static constexpr int CH = NP * UNR;                     // keys per unit at most (one pass of all warps)
  static constexpr size_t kStage = (size_t)CH * (KR + VR);  // K and V rows of a unit
  static constexpr size_t kAcc = (size_t)NP * G * D * 4;    // lane-group partial V sums
  static constexpr size_t kRing = kAttnStages * kStage;
  static constexpr size_t kBar = kRing + kAcc;              // mbarriers and flags
  static constexpr size_t kSmem = kBar + 2 * kAttnStages * 8 + 16;
  static_assert(kSmem <= 227 * 1024, "attention shared memory");
  // merge scratch in the lane-group area: (max, sum), weight and slot per contributor
  static constexpr int kMaxContrib = (int)((kAcc - 64) / (G * 12 + 4));
};

// Reduce N values held by each lane across a segment of LPK lanes (N <= LPK, both powers
// of two).  Afterwards lane li of the segment holds the segment total of value index
// li >> (log2 LPK - log2 N).
template <int N, int LPK>
__device__ __forceinline__ float seg_reduce_multi(float (&v)[N], int li) {
#pragma unroll
  for (int cnt = N, o = LPK / 2; cnt > 1; cnt >>= 1, o >>= 1) {
    const bool upper = (li & o) != 0;
#pragma unroll
    for (int i = 0; i < cnt / 2; ++i) {
      const float send = upper ? v[i] : v[i + cnt / 2];
      const float keep = upper ? v[i + cnt / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o, LPK);
    }
  }
  float r = v[0];
#pragma unroll
  for (int o = LPK / (2 * N); o >= 1; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o, LPK);
  return r;
}

// Four bytes of w as floats without the conversion unit: a byte placed under the exponent
// of 2^23 (0x4B0000xx) reads as 2^23 + byte exactly, so one byte permute and one add give
// the value.  Signed bytes are first offset by 128 (w ^ 0x80808080), then 2^23 + 128 is
// subtracted; both results are exact integers.
template <bool SIGNED>
__device__ __forceinline__ void bytes_to_f32x2(uint32_t w, float2 *f) {
  constexpr float kBias = SIGNED ? -8388736.0f : -8388608.0f;
  if (SIGNED) w ^= 0x80808080u;
  const float2 bias = make_float2(kBias, kBias);
  f[0] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540)),
                                __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7541))), bias);
  f[1] = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7542)),
                                __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7543))), bias);
}

__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t u) { return make_float2(bf_lo(u), bf_hi(u)); }

// Bit i (i < 4) of x moved to bit 4 of byte i: x * 0x00204081 puts bit i at 8i + 7(j - i)
// for each j; only j = i lands on a multiple of 8 and no two terms share a bit (no carry).
__device__ __forceinline__ uint32_t spread4_to_bit4(uint32_t x) {
  return ((x * 0x00204081u) & 0x01010101u) << 4;
}

template <int D, int G, bool KVQ>
__global__ void __launch_bounds__(kAttnCtaThreads, 1) attn_decode_kernel(const AttnParams p) {
  using S = AttnShape<D, G, KVQ>;
  constexpr int KR = S::KR, VR = S::VR;
  constexpr int LPK = S::LPK, KPW = S::KPW, NP = S::NP, UNR = S::UNR, N = S::N, SH = S::SH;
  constexpr int LOG_G = S::LOG_G, CH = S::CH;
  extern __shared__ __align__(128) unsigned char smem[];
  float *sm_acc = reinterpret_cast<float *>(smem + S::kRing);  // [NP][G][D] lane-group partials
  const uint32_t full0 = smem_addr(smem + S::kBar);
  const uint32_t empty0 = full0 + 8 * kAttnStages;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kBar + 2 * kAttnStages * 8);
  __shared__ float2 sm_ml[NP][G];
  __shared__ int last_sh;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = lane / LPK, li = lane - grp * LPK;
  const int H = p.n_head, Hkv = p.n_head_kv, ps = p.page_size, U = p.unit_keys;
  AttnSched sch;
  sch.pre = p.unit_pre;
  sch.B = p.batch;
  sch.Hkv = Hkv;
  sch.total = (long long)Hkv * sch.pre[p.batch];
  // every active CTA owns at least one unit (a CTA beyond the unit count has none)
  sch.grid = (int)min((long long)gridDim.x, sch.total);
  const int cta = blockIdx.x;
  const long long u_begin = cta < sch.grid ? sch.start(cta) : 0, u_end = cta < sch.grid ? sch.start(cta + 1) : 0;

  if (tid == 0) {
    for (int i = 0; i < kAttnStages; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, kAttnWarps);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
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

  if (warp == kAttnWarps) {
    // ---------------------------------------------------------- producer warp
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      bool waited = false;
      int g = 0;  // ring stage counter
      bool ok = true;
      for (long long u = u_begin; u < u_end && ok;) {
        const AttnSeg sg = attn_seg(sch, u, u_end);
        u += sg.r1 - sg.r0;
        // the lengths and the page table were fixed before the chain started: only the
        // copies of units holding keys the chain writes wait for the previous kernel
        const int L = p.kv_len[sg.b], est = est_len(sg.b), fin = final_len(sg.b);
        const int32_t *pt = p.page_table + (size_t)sg.b * p.max_pages;
        for (int r = sg.r0; r < sg.r1; ++r) {
          const int k0 = r * U;
          int k1 = min(k0 + U, est);
          const bool fresh = k1 > L;  // this unit holds keys written by the chain
          if (fresh) k1 = min(k1, fin);
          if (k1 <= k0) continue;  // trimmed away: the consumers skip it too
          const int slot = g % kAttnStages;
          if (g >= kAttnStages && !mbar_wait(empty0 + 8 * slot, ((g / kAttnStages) - 1) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const int pg = pt[k0 / ps];
          if (fresh && !waited) {
            pdl_wait();
            waited = true;
          }
          // bf16 rows: the unit's valid keys; quantized rows: the whole unit (sizes stay
          // multiples of 16 bytes; the slots past the valid keys are in the same page)
          const int nk = KVQ ? U : k1 - k0;
          const uint32_t kbytes = (uint32_t)nk * KR, vbytes = (uint32_t)nk * VR;
          mbar_expect_tx(full0 + 8 * slot, kbytes + vbytes);
          if (pg < 0 || pg >= p.num_pages) {
            // keep the ring in step: complete the stage without data (consumers skip it)
            set_status(p.status, EAGLE3_DEV_BAD_PAGE);
            asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(full0 + 8 * slot), "r"(kbytes + vbytes) : "memory");
          } else {
            const size_t row = ((size_t)pg * Hkv + sg.kvh) * ps + k0 % ps;
            const uint32_t dst = smem_addr(smem + (size_t)slot * S::kStage);
            bulk_g2s(dst, p.k_pool + row * KR, kbytes, full0 + 8 * slot, pol);
            bulk_g2s(dst + (uint32_t)(CH * KR), p.v_pool + row * VR, vbytes, full0 + 8 * slot, pol);
          }
          ++g;
        }
      }
      // no copy may still be in flight when the CTA moves on
      for (int i = max(0, g - kAttnStages); i < g; ++i)
        mbar_wait(full0 + 8 * (i % kAttnStages), (i / kAttnStages) & 1, abort_flag, p.status);
      if (!waited) pdl_wait();
    }
    __syncwarp();
    return;
  }

  // ------------------------------------------------------------ consumer warps
  bool waited = false;  // q is written by the previous kernel: wait before the first read
  const float qscale = rsqrtf((float)D) * 1.4426950408889634f;
  // Score index of this lane after the segment reduction: (key u_me, head g_me).
  const int idx_me = li >> SH;
  const int g_me = idx_me & (G - 1), u_me = idx_me >> LOG_G;
  const int part = warp * KPW + grp;
  int g = 0;
  for (long long u = u_begin; u < u_end;) {
    const AttnSeg sg = attn_seg(sch, u, u_end);
    u += sg.r1 - sg.r0;
    const int b = sg.b, kvh = sg.kvh;
    const int est = est_len(b), fin = final_len(b), L = p.kv_len[b];
    const int32_t *pt = p.page_table + (size_t)b * p.max_pages;
    if (!waited) {
      pdl_wait();
      waited = true;
    }
    // q, the running weighted V and the K / V values are float pairs: every multiply-add
    // of the loop is a packed two-lane FMA
    float2 qv[G][4];
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      const float4 *qp = reinterpret_cast<const float4 *>(p.q + (size_t)b * H * D + (size_t)(kvh * G + gg) * D + li * 8);
      const float4 a = __ldcg(qp), c = __ldcg(qp + 1);
      qv[gg][0] = make_float2(a.x * qscale, a.y * qscale);
      qv[gg][1] = make_float2(a.z * qscale, a.w * qscale);
      qv[gg][2] = make_float2(c.x * qscale, c.y * qscale);
      qv[gg][3] = make_float2(c.z * qscale, c.w * qscale);
    }
    float m_me = -INFINITY, l_me = 0.f;  // running max (log2 domain) and sum of head g_me
    float2 acc[G][4];                    // running weighted V of this lane's 8 dims, every head
    float accm[G];                       // quantized V: running sum of p * m (block minimum)
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      accm[gg] = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[gg][i] = make_float2(0.f, 0.f);
    }

    for (int r = sg.r0; r < sg.r1; ++r) {
      const int k0 = r * U;
      int k1 = min(k0 + U, est);
      if (k1 > L) k1 = min(k1, fin);
      if (k1 <= k0) continue;
      const int n = k1 - k0;
      const int slot = g % kAttnStages;
      const int pg = pt[k0 / ps];
      const bool ok = mbar_wait(full0 + 8 * slot, (g / kAttnStages) & 1, abort_flag, p.status);
      ++g;
      const bool have = ok && pg >= 0 && pg < p.num_pages;
      const unsigned char *kst = smem + (size_t)slot * S::kStage;
      const unsigned char *vst = kst + (size_t)CH * KR;
      // keys of this lane group: kk = warp * KPW * UNR + uu * KPW + grp
      unsigned vmask = 0u;
      float part_s[N];
#pragma unroll
      for (int uu = 0; uu < UNR; ++uu) {
        const int kk = warp * KPW * UNR + uu * KPW + grp;
        const bool v = have && kk < n;
        vmask |= v ? (1u << uu) : 0u;
        float2 kf[4];
        float kscale = 1.f;
        if constexpr (KVQ) {
          // q8_0: this lane's 8 codes of block li / 4 (2-byte aligned: four 16-bit loads);
          // the block scale multiplies the partial dot once
          const unsigned char *blk = kst + (size_t)kk * KR + (li >> 2) * 34;
          const uint16_t *c16 = reinterpret_cast<const uint16_t *>(blk + 2 + 8 * (li & 3));
          uint32_t w0 = 0u, w1 = 0u;
          if (v) {
            w0 = __byte_perm(c16[0], c16[1], 0x5410);
            w1 = __byte_perm(c16[2], c16[3], 0x5410);
          }
          bytes_to_f32x2<true>(w0, kf);
          bytes_to_f32x2<true>(w1, kf + 2);
          kscale = v ? __half2float(*reinterpret_cast<const __half *>(blk)) : 0.f;
        } else {
          uint4 ku = make_uint4(0u, 0u, 0u, 0u);
          if (v) ku = *reinterpret_cast<const uint4 *>(kst + (size_t)kk * KR + li * 16);
          kf[0] = bf16x2_to_f32x2(ku.x); kf[1] = bf16x2_to_f32x2(ku.y);
          kf[2] = bf16x2_to_f32x2(ku.z); kf[3] = bf16x2_to_f32x2(ku.w);
        }
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          float2 d2 = __fmul2_rn(qv[gg][0], kf[0]);
#pragma unroll
          for (int i = 1; i < 4; ++i) d2 = __ffma2_rn(qv[gg][i], kf[i], d2);
          const float d = d2.x + d2.y;
          part_s[uu * G + gg] = KVQ ? d * kscale : d;
        }
      }
      const bool vld = (vmask >> u_me) & 1u;
      const float red = seg_reduce_multi<N, LPK>(part_s, li);  // every lane takes part
      const float sc = vld ? red : -INFINITY;
      // block max and sum over the keys of head g_me (lanes differing in the key bits)
      float bm = sc;
#pragma unroll
      for (int o = 1 << (SH + LOG_G); o < LPK; o <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o, LPK));
      const float m_new = fmaxf(m_me, bm);
      const float corr = m_new == -INFINITY ? 1.f : exp2f(m_me - m_new);
      const float pr = vld ? exp2f(sc - m_new) : 0.f;
      float psum = pr;
#pragma unroll
      for (int o = 1 << (SH + LOG_G); o < LPK; o <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o, LPK);
      l_me = l_me * corr + psum;
      m_me = m_new;
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        const float c = __shfl_sync(0xffffffffu, corr, gg << SH, LPK);
        const float2 c2 = make_float2(c, c);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[gg][i] = __fmul2_rn(acc[gg][i], c2);
        if constexpr (KVQ) accm[gg] *= c;
      }
#pragma unroll
      for (int uu = 0; uu < UNR; ++uu) {
        const int kk = warp * KPW * UNR + uu * KPW + grp;
        const bool vv = (vmask >> uu) & 1u;
        float2 vf[4];
        float vd = 1.f, vm = 0.f;
        if constexpr (KVQ) {
          // q5_1: this lane's 8 codes of block li / 4 -- 4 bits from one 8-byte load (low
          // nibbles for values 0-15 of the block, high for 16-31) and the fifth bit from qh;
          // v = d * code + m, with p * m summed apart (all 8 values share the block)
          const unsigned char *blk = vst + (size_t)kk * VR + (li >> 2) * 24;
          const int e = 8 * (li & 3);
          uint2 qs = make_uint2(0u, 0u);
          unsigned qh = 0u;
          if (vv) {
            qs = *reinterpret_cast<const uint2 *>(blk + 8 + (e & 15));
            qh = *reinterpret_cast<const unsigned *>(blk + 4);
            vd = __half2float(*reinterpret_cast<const __half *>(blk));
            vm = __half2float(*reinterpret_cast<const __half *>(blk + 2));
          } else {
            vd = 0.f;
          }
          const int sh = e >= 16 ? 4 : 0;
          const uint32_t hb = qh >> e;  // fifth bits of values e .. e + 7
          const uint32_t w0 = ((qs.x >> sh) & 0x0F0F0F0Fu) | spread4_to_bit4(hb & 15u);
          const uint32_t w1 = ((qs.y >> sh) & 0x0F0F0F0Fu) | spread4_to_bit4((hb >> 4) & 15u);
          bytes_to_f32x2<false>(w0, vf);
          bytes_to_f32x2<false>(w1, vf + 2);
        } else {
          uint4 vu = make_uint4(0u, 0u, 0u, 0u);
          if (vv) vu = *reinterpret_cast<const uint4 *>(vst + (size_t)kk * VR + li * 16);
          vf[0] = bf16x2_to_f32x2(vu.x); vf[1] = bf16x2_to_f32x2(vu.y);
          vf[2] = bf16x2_to_f32x2(vu.z); vf[3] = bf16x2_to_f32x2(vu.w);
        }
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          const float pg2 = __shfl_sync(0xffffffffu, pr, (uu * G + gg) << SH, LPK);
          const float pw = KVQ ? pg2 * vd : pg2;
          const float2 pw2 = make_float2(pw, pw);
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[gg][i] = __ffma2_rn(pw2, vf[i], acc[gg][i]);
          if constexpr (KVQ) accm[gg] = fmaf(pg2, vm, accm[gg]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * slot);
    }

    // ---- end of this CTA's units of pair (b, kvh): merge the lane groups
    asm volatile("bar.sync 1, 256;" ::: "memory");  // the previous pair's reads of sm_acc are done
    if (u_me == 0 && (li & ((1 << SH) - 1)) == 0) sm_ml[part][g_me] = make_float2(m_me, l_me);
#pragma unroll
    for (int gg = 0; gg < G; ++gg)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float mm = KVQ ? accm[gg] : 0.f;
        *reinterpret_cast<float2 *>(sm_acc + ((size_t)part * G + gg) * D + li * 8 + 2 * i) =
            make_float2(acc[gg][i].x + mm, acc[gg][i].y + mm);
      }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    const bool whole = sg.r0 == 0 && sg.r1 == sg.nu;
    float *out = p.out + (size_t)b * H * D + (size_t)kvh * G * D;
    // this CTA's (max, sum, weighted V) of the pair: in place in sm_acc lane group 0 and
    // sm_ml, or written out when no other CTA holds units of the pair
    const int mine = cta * 2 + (sch.start(cta) >= sg.pair_u0 ? 0 : 1);  // partial slot
    for (int e = tid; e < G * D; e += kAttnThreads) {
      const int gg = e / D, dim = e - gg * D;
      float M = -INFINITY;
#pragma unroll
      for (int q = 0; q < NP; ++q) M = fmaxf(M, sm_ml[q][gg].x);
      float Ls = 0.f, O = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int q = 0; q < NP; ++q) {
          const float2 ml = sm_ml[q][gg];
          const float w = exp2f(ml.x - M);
          Ls += ml.y * w;
          O += sm_acc[((size_t)q * G + gg) * D + dim] * w;
        }
      }
      if (whole) {
        out[e] = O / Ls;
      } else {
        p.part_o[(size_t)mine * G * D + e] = O;
        if (dim == 0) p.part_ml[(size_t)mine * G + gg] = make_float2(M, Ls);
      }
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
    // Weights first: every contributor's (max, sum) and slot into shared memory (the lane-
    // group area is free now), w = exp2(m - M) / L per (contributor, head); then each
    // thread sums float4 slices over the contributors, 8 loads at a time.
    const int nc = c_last - c_first + 1;
    float2 *ml_s = reinterpret_cast<float2 *>(sm_acc);   // [nc][G]
    float *w_s = reinterpret_cast<float *>(ml_s + nc * G); // [nc][G]
    int *slot_s = reinterpret_cast<int *>(w_s + nc * G);   // [nc]
    float2 *ML = reinterpret_cast<float2 *>((reinterpret_cast<uintptr_t>(slot_s + nc) + 7) & ~(uintptr_t)7);  // [G]
    for (int i = tid; i < nc; i += kAttnThreads) {
      const int c2 = c_first + i;
      slot_s[i] = c2 * 2 + (sch.start(c2) >= pu0 ? 0 : 1);
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    for (int i = tid; i < nc * G; i += kAttnThreads) ml_s[i] = __ldcg(&p.part_ml[(size_t)slot_s[i / G] * G + i % G]);
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
    for (int i = tid; i < nc * G; i += kAttnThreads) {
      const float2 ml = ml_s[i];
      const int gg = i % G;
      w_s[i] = ml.x == -INFINITY ? 0.f : exp2f(ml.x - ML[gg].x) * ML[gg].y;
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    const float4 *po = reinterpret_cast<const float4 *>(p.part_o);
    float4 *out4 = reinterpret_cast<float4 *>(out);
    for (int f = tid; f < G * D / 4; f += kAttnThreads) {
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
  }
}

// Keys per unit: the run of one pass of all warps, cut to the largest power of two that
// divides the page size (a unit never crosses a page).  Quantized rows are copied a whole
// unit at a time, so a unit's K and V bytes must be multiples of 16; 0 when they are not.
template <int D, int G, bool KVQ>
static int attn_unit_keys_dg(int page_size) {
  using S = AttnShape<D, G, KVQ>;
  int u = S::CH;
  while (u > 1 && page_size % u) u >>= 1;
  if (KVQ && (((size_t)u * S::KR) % 16 || ((size_t)u * S::VR) % 16)) return 0;
  return u;
}

template <int D, int G, bool KVQ>
static cudaError_t attn_launch_dg(const AttnParams &p, int num_sms, cudaStream_t st, bool pdl) {
  using S = AttnShape<D, G, KVQ>;
  if (p.unit_keys < 1 || p.unit_keys != attn_unit_keys_dg<D, G, KVQ>(p.page_size)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  // one CTA per SM; no more contributors per pair than the merge scratch holds
  cfg.gridDim = dim3(num_sms < S::kMaxContrib ? num_sms : S::kMaxContrib);
  cfg.blockDim = dim3(kAttnCtaThreads);
  cfg.dynamicSmemBytes = S::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_decode_kernel<D, G, KVQ>, p);
}

template <int D, int G>
static cudaError_t attn_prepare_dg() {
  cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<D, G, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)AttnShape<D, G, false>::kSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_decode_kernel<D, G, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)AttnShape<D, G, true>::kSmem);
  return e;
}

bool attn_supported(int head_dim, int group) {
  return (head_dim == 64 || head_dim == 128 || head_dim == 256) &&
         (group == 1 || group == 2 || group == 4 || group == 8);
}

#define E3_ATTN_ALL(X) \
  X(64, 1) X(64, 2) X(64, 4) X(64, 8) X(128, 1) X(128, 2) X(128, 4) X(128, 8) X(256, 1) X(256, 2) X(256, 4) X(256, 8)

cudaError_t attn_prepare() {
  cudaError_t e = attn_tc_prepare();
#define E3_PREP(DD, GG) \
  if (e == cudaSuccess) e = attn_prepare_dg<DD, GG>();
  E3_ATTN_ALL(E3_PREP)
#undef E3_PREP
  return e;
}

int attn_unit_keys(int head_dim, int group, int page_size, int kv_q) {
#define E3_UNIT(DD, GG)                                                                 \
  if (head_dim == DD && group == GG)                                                   \
    return kv_q ? attn_unit_keys_dg<DD, GG, true>(page_size) : attn_unit_keys_dg<DD, GG, false>(page_size);
  E3_ATTN_ALL(E3_UNIT)
#undef E3_UNIT
  return 0;
}

cudaError_t attn_launch(const AttnParams &p, int num_sms, cudaStream_t st, bool pdl) {
  const int G = p.n_head / p.n_head_kv;
  if (p.batch < 1 || p.unit_keys < 1 || !p.unit_pre) return cudaErrorInvalidValue;
  if (p.tc && !p.kv_q && attn_tc_supported(p.head_dim, G, p.unit_keys)) return attn_tc_launch(p, num_sms, st, pdl);
#define E3_ATTN_CASE(DD, GG)                                                             \
  if (p.head_dim == DD && G == GG)                                                      \
    return p.kv_q ? attn_launch_dg<DD, GG, true>(p, num_sms, st, pdl) : attn_launch_dg<DD, GG, false>(p, num_sms, st, pdl);
  E3_ATTN_ALL(E3_ATTN_CASE)
#undef E3_ATTN_CASE
  return cudaErrorInvalidValue;
}

}  // namespace e3
