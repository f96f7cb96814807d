// Split-KV GQA decode attention over the paged bf16 drafter KV cache.
//
// For each sequence b and q head h (kv head h / G, G = n_head / n_head_kv): softmax over
// the keys 0..len-1 of (q . k) / sqrt(d), then sum of p * v ("memra_engine/eagle.rs",
// ``attn``: fa_decode with scale 1/sqrt(head_dim); the new key is appended first).
//
// One CTA per (split, kv head, sequence): the G query heads that share a kv head are
// served from one read of each K/V vector.  A producer warp streams the split's keys in
// runs of up to 64 consecutive positions inside one page -- the K rows and the V rows of
// a run are contiguous in the paged pool -- with bulk copies (TMA) into a 3-stage
// shared-memory ring guarded by mbarriers.  Runs below the committed length were written
// before the chain started, so they are requested before the kernel waits on its
// predecessor (programmatic dependent launch).  Eight consumer warps take UNR keys per
// lane group of each run (a key of d = 256 dims spans a warp, 8 dims = 16 bytes per
// lane; smaller heads put several keys in a warp).  The UNR x G partial scores are
// reduced across the lane group in one transposed reduction: each lane ends with one full
// score and takes its exponential, and the probabilities are broadcast for the V update.
// An online softmax per head keeps the running max (log2 domain), sum and weighted V.
// The CTA merges its lane groups in shared memory; with more than one split the last CTA
// of a (sequence, kv head) to finish merges the splits' partials.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace e3 {

constexpr int kAttnWarps = 8;                          // consumer warps
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kAttnCtaThreads = kAttnThreads + 32;     // + one producer warp
constexpr int kMaxAttnSplits = 64;
constexpr int kAttnStages = 3;

template <int X>
struct ILog2 {
  static constexpr int value = X <= 1 ? 0 : 1 + ILog2<X / 2>::value;
};
template <>
struct ILog2<1> {
  static constexpr int value = 0;
};

template <int D, int G>
struct AttnShape {
  static constexpr int LPK = D / 8;             // lanes per key (a segment of the warp)
  static constexpr int KPW = 32 / LPK;          // keys per warp pass
  static constexpr int NP = kAttnWarps * KPW;   // lane groups per CTA
  // keys per lane group per block; UNR * G partial scores fit one segment reduction
  static constexpr int UNR = (LPK / G) < 8 ? (LPK / G < 1 ? 1 : LPK / G) : 8;
  static constexpr int N = UNR * G;
  static constexpr int SH = ILog2<LPK>::value - ILog2<N>::value;  // lane bits below a score index
  static constexpr int LOG_G = ILog2<G>::value;
  static constexpr int CH = NP * UNR;                     // keys per run (one pass of all warps)
  static constexpr size_t kStage = (size_t)2 * CH * D * 2;  // K and V rows of a run, bf16
  static constexpr size_t kAcc = (size_t)NP * G * D * 4;    // lane-group partial V sums
  static constexpr size_t kRing = kAttnStages * kStage;
  static constexpr size_t kSmem = (kRing > kAcc ? kRing : kAcc) + 2 * kAttnStages * 8 + 16;
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

template <int D, int G>
__global__ void __launch_bounds__(kAttnCtaThreads, 1) attn_decode_kernel(const AttnParams p) {
  using S = AttnShape<D, G>;
  constexpr int LPK = S::LPK, KPW = S::KPW, NP = S::NP, UNR = S::UNR, N = S::N, SH = S::SH;
  constexpr int LOG_G = S::LOG_G, CH = S::CH;
  extern __shared__ __align__(128) unsigned char smem[];
  // ring of runs; after the last run the same memory holds the lane-group partials
  float *sm_acc = reinterpret_cast<float *>(smem);  // [NP][G][D]
  const size_t bar_off = (S::kRing > S::kAcc ? S::kRing : S::kAcc);
  const uint32_t full0 = smem_addr(smem + bar_off);
  const uint32_t empty0 = full0 + 8 * kAttnStages;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + bar_off + 2 * kAttnStages * 8);
  __shared__ float2 sm_ml[NP][G];
  __shared__ int last_sh;

  const int s = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = lane / LPK, li = lane - grp * LPK;
  const int H = p.n_head, Hkv = p.n_head_kv, ps = p.page_size;
  const int32_t *pt = p.page_table + (size_t)b * p.max_pages;

  // Key range of this split, from the length before gamma_eff is known (committed + step).
  const int L = p.kv_len[b];
  int len = L + p.step + 1;
  if (len > p.max_cache_len) len = p.max_cache_len;
  if (len < 1) len = 1;
  const int chunk = (len + p.splits - 1) / p.splits;
  const int k0 = min(s * chunk, len);
  const int k1_est = min(len, k0 + chunk);
  const int run_max = min(CH, ps);  // a run never crosses a page

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

  // run boundaries: [pos, pos + n), n = min(run_max, page end - pos, k1 - pos)
  auto run_len = [&](int pos, int k1) { return min(min(run_max, (pos / ps + 1) * ps - pos), k1 - pos); };
  auto final_k1 = [&]() {
    const int ge = p.gamma_eff ? p.gamma_eff[b] : p.step + 1;
    int len2 = L + min(p.step, max(ge - 1, 0)) + 1;
    if (L < 0 || len2 > p.max_cache_len) len2 = min(max(len2, 1), p.max_cache_len);
    return min(k1_est, len2);
  };

  if (warp == kAttnWarps) {
    // ---------------------------------------------------------- producer warp
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      bool waited = false;
      int k1 = k1_est, r = 0;
      for (int pos = k0; pos < k1; ++r) {
        int n = run_len(pos, k1);
        if (!waited && (pos + n > L || L < 0)) {  // this run holds keys written by the chain
          pdl_wait();
          waited = true;
          k1 = final_k1();
          if (pos >= k1) break;
          n = run_len(pos, k1);
        }
        const int slot = r % kAttnStages;
        if (r >= kAttnStages && !mbar_wait(empty0 + 8 * slot, ((r / kAttnStages) - 1) & 1, abort_flag, p.status))
          break;
        const int pg = pt[pos / ps];
        const uint32_t bytes = (uint32_t)n * D * 2u;
        mbar_expect_tx(full0 + 8 * slot, 2u * bytes);
        if (pg < 0 || pg >= p.num_pages) {
          // keep the ring in step: complete the stage without data (consumers skip it)
          set_status(p.status, EAGLE3_DEV_BAD_PAGE);
          asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(full0 + 8 * slot), "r"(2u * bytes) : "memory");
        } else {
          const size_t off = (((size_t)pg * Hkv + kvh) * ps + pos % ps) * D;
          const uint32_t dst = smem_addr(smem + (size_t)slot * S::kStage);
          bulk_g2s(dst, p.k_pool + off, bytes, full0 + 8 * slot, pol);
          bulk_g2s(dst + (uint32_t)(CH * D * 2), p.v_pool + off, bytes, full0 + 8 * slot, pol);
        }
        pos += n;
      }
      // no copy may still be in flight when the CTA moves on
      for (int i = max(0, r - kAttnStages); i < r; ++i)
        mbar_wait(full0 + 8 * (i % kAttnStages), (i / kAttnStages) & 1, abort_flag, p.status);
      if (!waited) pdl_wait();
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- consumer warps
    pdl_wait();
    const int k1 = final_k1();
    const float qscale = rsqrtf((float)D) * 1.4426950408889634f;
    float qv[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float4 *qp = reinterpret_cast<const float4 *>(p.q + (size_t)b * H * D + (size_t)(kvh * G + g) * D + li * 8);
      const float4 a = qp[0], c = qp[1];
      qv[g][0] = a.x * qscale; qv[g][1] = a.y * qscale; qv[g][2] = a.z * qscale; qv[g][3] = a.w * qscale;
      qv[g][4] = c.x * qscale; qv[g][5] = c.y * qscale; qv[g][6] = c.z * qscale; qv[g][7] = c.w * qscale;
    }
    // Score index of this lane after the segment reduction: (key u_me, head g_me).
    const int idx_me = li >> SH;
    const int g_me = idx_me & (G - 1), u_me = idx_me >> LOG_G;
    float m_me = -INFINITY, l_me = 0.f;  // running max (log2 domain) and sum of head g_me
    float acc[G][8];                     // running weighted V of this lane's 8 dims, every head
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[g][i] = 0.f;

    int r = 0;
    for (int pos = k0; pos < k1; ++r) {
      const int n = run_len(pos, k1);
      const int slot = r % kAttnStages;
      const bool ok = mbar_wait(full0 + 8 * slot, (r / kAttnStages) & 1, abort_flag, p.status);
      const int pg = pt[pos / ps];
      const bool have = ok && pg >= 0 && pg < p.num_pages;
      const unsigned char *kst = smem + (size_t)slot * S::kStage;
      const unsigned char *vst = kst + (size_t)CH * D * 2;
      // keys of this lane group: kk = warp * KPW * UNR + u * KPW + grp
      unsigned vmask = 0u;
      float part_s[N];
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const int kk = warp * KPW * UNR + u * KPW + grp;
        const bool v = have && kk < n;
        vmask |= v ? (1u << u) : 0u;
        uint4 ku = make_uint4(0u, 0u, 0u, 0u);
        if (v) ku = *reinterpret_cast<const uint4 *>(kst + ((size_t)kk * D + li * 8) * 2);
        const float kf[8] = {bf_lo(ku.x), bf_hi(ku.x), bf_lo(ku.y), bf_hi(ku.y),
                             bf_lo(ku.z), bf_hi(ku.z), bf_lo(ku.w), bf_hi(ku.w)};
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float d = 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) d = fmaf(qv[g][i], kf[i], d);
          part_s[u * G + g] = d;
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
      for (int g = 0; g < G; ++g) {
        const float c = __shfl_sync(0xffffffffu, corr, g << SH, LPK);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[g][i] *= c;
      }
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const int kk = warp * KPW * UNR + u * KPW + grp;
        uint4 vu = make_uint4(0u, 0u, 0u, 0u);
        if ((vmask >> u) & 1u) vu = *reinterpret_cast<const uint4 *>(vst + ((size_t)kk * D + li * 8) * 2);
        const float vf[8] = {bf_lo(vu.x), bf_hi(vu.x), bf_lo(vu.y), bf_hi(vu.y),
                             bf_lo(vu.z), bf_hi(vu.z), bf_lo(vu.w), bf_hi(vu.w)};
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pg2 = __shfl_sync(0xffffffffu, pr, (u * G + g) << SH, LPK);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[g][i] = fmaf(pg2, vf[i], acc[g][i]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * slot);
      pos += n;
    }
    // the ring is reused for the partials only after every warp is done with it
    asm volatile("bar.sync 1, 256;" ::: "memory");
    const int part = warp * KPW + grp;
    if (u_me == 0 && (li & ((1 << SH) - 1)) == 0) sm_ml[part][g_me] = make_float2(m_me, l_me);
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int i = 0; i < 8; ++i) sm_acc[((size_t)part * G + g) * D + li * 8 + i] = acc[g][i];
  }
  __syncthreads();

  const size_t slot = ((size_t)b * Hkv + kvh) * p.splits + s;
  for (int e = tid; e < G * D; e += kAttnCtaThreads) {
    const int g = e / D, dim = e - g * D;
    float M = -INFINITY;
#pragma unroll
    for (int q = 0; q < NP; ++q) M = fmaxf(M, sm_ml[q][g].x);
    float Ls = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int q = 0; q < NP; ++q) {
        const float2 ml = sm_ml[q][g];
        const float w = exp2f(ml.x - M);
        Ls += ml.y * w;
        O += sm_acc[((size_t)q * G + g) * D + dim] * w;
      }
    }
    if (p.splits == 1) {
      p.out[(size_t)b * H * D + (size_t)(kvh * G + g) * D + dim] = O / Ls;
    } else {
      p.part_o[(slot * G + g) * D + dim] = O;
      if (dim == 0) p.part_ml[slot * G + g] = make_float2(M, Ls);
    }
  }
  if (p.splits == 1) return;

  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(p.count + (size_t)b * Hkv + kvh, 1u);
    last_sh = (prev == (unsigned)p.splits - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!last_sh) return;
  __threadfence();
  // Merge the splits: weights w[q][g] = exp2(m_q - M_g) / L_g first (all splits loaded in
  // parallel), then every thread sums float4 slices over the splits, 8 loads at a time.
  __shared__ float2 ml_all[kMaxAttnSplits][G];
  __shared__ float wsm[kMaxAttnSplits][G];
  __shared__ float2 ML[G];
  const size_t slot0 = ((size_t)b * Hkv + kvh) * p.splits;
  for (int i = tid; i < p.splits * G; i += kAttnCtaThreads)
    ml_all[i / G][i % G] = __ldcg(&p.part_ml[slot0 * G + i]);
  __syncthreads();
  if (tid < G) {
    float M = -INFINITY;
    for (int q = 0; q < p.splits; ++q) M = fmaxf(M, ml_all[q][tid].x);
    float Ls = 0.f;
    for (int q = 0; q < p.splits; ++q)
      if (ml_all[q][tid].x != -INFINITY) Ls += ml_all[q][tid].y * exp2f(ml_all[q][tid].x - M);
    ML[tid] = make_float2(M, 1.0f / Ls);
  }
  __syncthreads();
  for (int i = tid; i < p.splits * G; i += kAttnCtaThreads) {
    const int q = i / G, g = i % G;
    const float2 ml = ml_all[q][g];
    wsm[q][g] = ml.x == -INFINITY ? 0.f : exp2f(ml.x - ML[g].x) * ML[g].y;
  }
  __syncthreads();
  const float4 *po = reinterpret_cast<const float4 *>(p.part_o) + slot0 * (G * D / 4);
  float4 *out4 = reinterpret_cast<float4 *>(p.out + (size_t)b * H * D + (size_t)kvh * G * D);
  for (int f = tid; f < G * D / 4; f += kAttnCtaThreads) {
    const int g = (f * 4) / D;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    int q = 0;
    for (; q + 8 <= p.splits; q += 8) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldcg(po + (size_t)(q + u) * (G * D / 4) + f);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float w = wsm[q + u][g];
        o.x = fmaf(w, v[u].x, o.x); o.y = fmaf(w, v[u].y, o.y);
        o.z = fmaf(w, v[u].z, o.z); o.w = fmaf(w, v[u].w, o.w);
      }
    }
    for (; q < p.splits; ++q) {
      const float4 v = __ldcg(po + (size_t)q * (G * D / 4) + f);
      const float w = wsm[q][g];
      o.x = fmaf(w, v.x, o.x); o.y = fmaf(w, v.y, o.y);
      o.z = fmaf(w, v.z, o.z); o.w = fmaf(w, v.w, o.w);
    }
    out4[f] = o;
  }
  if (tid == 0) p.count[(size_t)b * Hkv + kvh] = 0u;
}

template <int D, int G>
static cudaError_t attn_launch_dg(const AttnParams &p, int B, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits, p.n_head_kv, B);
  cfg.blockDim = dim3(kAttnCtaThreads);
  cfg.dynamicSmemBytes = AttnShape<D, G>::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_decode_kernel<D, G>, p);
}

template <int D, int G>
static cudaError_t attn_prepare_dg() {
  return cudaFuncSetAttribute(attn_decode_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)AttnShape<D, G>::kSmem);
}

bool attn_supported(int head_dim, int group) {
  return (head_dim == 64 || head_dim == 128 || head_dim == 256) &&
         (group == 1 || group == 2 || group == 4 || group == 8);
}

#define E3_ATTN_ALL(X) \
  X(64, 1) X(64, 2) X(64, 4) X(64, 8) X(128, 1) X(128, 2) X(128, 4) X(128, 8) X(256, 1) X(256, 2) X(256, 4) X(256, 8)

cudaError_t attn_prepare() {
  cudaError_t e = cudaSuccess;
#define E3_PREP(DD, GG) \
  if (e == cudaSuccess) e = attn_prepare_dg<DD, GG>();
  E3_ATTN_ALL(E3_PREP)
#undef E3_PREP
  return e;
}

cudaError_t attn_launch(const AttnParams &p, int B, cudaStream_t st, bool pdl) {
  const int G = p.n_head / p.n_head_kv;
  if (p.splits < 1 || p.splits > kMaxAttnSplits) return cudaErrorInvalidValue;
#define E3_ATTN_CASE(DD, GG) \
  if (p.head_dim == DD && G == GG) return attn_launch_dg<DD, GG>(p, B, st, pdl);
  E3_ATTN_ALL(E3_ATTN_CASE)
#undef E3_ATTN_CASE
  return cudaErrorInvalidValue;
}

}  // namespace e3
