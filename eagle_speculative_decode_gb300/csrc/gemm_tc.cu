// bf16 instantiations of the tensor-core GEMM (gemm_tc.cuh), the GEMM entry points, the
// tensor maps and the activation prep kernel; INT4 instantiations are in gemm_tc_q4.cu.
#include "gemm_tc.cuh"

namespace e3 {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix with a (64 x box_rows) box and
// 128-byte swizzle.
bool tc_make_map(CUtensorMap *map, const void *base, int rows, int cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn || !base || (reinterpret_cast<uintptr_t>(base) & 15u) || cols % 64 || rows < 1) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kTcK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D tensor map over INT4 code rows ([rows][K / 2] bytes): a box of one k-tile's codes
// (32 bytes) by box_rows rows, no swizzle.
bool tc_make_code_map(CUtensorMap *map, const void *base, int rows, int K, int box_rows) {
  auto fn = encode_fn();
  if (!fn || !base || (reinterpret_cast<uintptr_t>(base) & 15u) || K % 128 || rows < 1) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K / 2, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K / 2};
  cuuint32_t box[2] = {(cuuint32_t)kTcK / 2, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Items per tile: the smallest of 16, 32, 64 (128 for the one-part encode) that holds M;
// more items take several item tiles.
int tc_tile_items(int M, int mode) {
  const int cap = mode == GM_ENCODE ? TcMode<GM_ENCODE>::kMaxN : TcMode<GM_QKV>::kMaxN;
  int n = 16;
  while (n < M && n < cap) n *= 2;
  return n;
}

cudaError_t tc_launch(const TcLaunch &L, cudaStream_t st, bool pdl) {
  if (L.s0) return tc_q4_launch(L, st, pdl);  // INT4 weights (the encode's fc stays bf16)
  switch (L.p.mode) {
    case GM_ENCODE: return tc_launch_mode<GM_ENCODE, false>(L, st, pdl);
    case GM_QKV: return tc_launch_mode<GM_QKV, false>(L, st, pdl);
    case GM_O: return tc_launch_mode<GM_O, false>(L, st, pdl);
    case GM_GATEUP: return tc_launch_mode<GM_GATEUP, false>(L, st, pdl);
    case GM_DOWN: return tc_launch_mode<GM_DOWN, false>(L, st, pdl);
    case GM_LMHEAD: return tc_launch_mode<GM_LMHEAD, false>(L, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t tc_prepare() {
  if (!encode_fn()) return cudaErrorNotSupported;
  cudaError_t e = tc_prepare_mode<GM_ENCODE, false>();
  if (e == cudaSuccess) e = tc_prepare_mode<GM_QKV, false>();
  if (e == cudaSuccess) e = tc_prepare_mode<GM_O, false>();
  if (e == cudaSuccess) e = tc_prepare_mode<GM_GATEUP, false>();
  if (e == cudaSuccess) e = tc_prepare_mode<GM_DOWN, false>();
  if (e == cudaSuccess) e = tc_prepare_mode<GM_LMHEAD, false>();
  if (e == cudaSuccess) e = tc_q4_prepare();
  return e;
}

// ------------------------------------------------------------------ activation prep
constexpr int kPrepIters = 8;  // 8-element vectors per thread: K up to 8 * 256 * 8 = 16384
// x (times the norm gain where the op normalises) split into three bf16 parts
// x0 = bf16(x), x1 = bf16(x - x0), x2 = bf16(x - x0 - x1) -- both differences are exact
// in float32 and x0 + x1 + x2 carries x's 24 significant bits -- and the sum of squares
// per item and K half for the deferred RMSNorm scale; for INT4 weights also the sum of x
// over each 128-wide group (gsum [item][K / 128], the zero points' term).  One CTA per
// item.
template <int MODE>
__global__ void __launch_bounds__(256) tc_prep_kernel(const GemvParams p, uint16_t *x0, uint16_t *x1,
                                                      uint16_t *x2, float *sumsq, float *gsum) {
  using T = ModeTraits<MODE>;
  constexpr int H = T::kHalves;
  __shared__ float red[8][H];
  pdl_trigger();
  pdl_wait();
  const int item = blockIdx.x, tid = threadIdx.x;
  const int K = p.K, KV = K >> 3;
  float ss[H];
#pragma unroll
  for (int h = 0; h < H; ++h) ss[h] = 0.f;
  uint4 *d0 = reinterpret_cast<uint4 *>(x0 + (size_t)item * K);
  uint4 *d1 = reinterpret_cast<uint4 *>(x1 + (size_t)item * K);
  uint4 *d2 = reinterpret_cast<uint4 *>(x2 + (size_t)item * K);
  auto pack = [](const uint16_t (&u)[8]) {
    return make_uint4(u[0] | ((uint32_t)u[1] << 16), u[2] | ((uint32_t)u[3] << 16),
                      u[4] | ((uint32_t)u[5] << 16), u[6] | ((uint32_t)u[7] << 16));
  };
  // the sum of x over vector kv's 128-wide group, from the 16 lanes that hold the group
  // (every lane of the warp takes part; inactive ones add zeros and do not write)
  const int GS = K >> 7;
  auto group_sum = [&](int kv, bool act, const float (&x)[8]) {
    float v = 0.f;
    if (act) v = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (act && (tid & 15) == 0) gsum[(size_t)item * GS + (kv >> 4)] = v;
  };
  auto put = [&](int kv, const float (&x)[8]) {
    uint16_t u0[8], u1[8], u2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      u0[i] = f2bf(x[i]);
      const float r1 = x[i] - bf1(u0[i]);
      u1[i] = f2bf(r1);
      u2[i] = f2bf(r1 - bf1(u1[i]));
    }
    d0[kv] = pack(u0);
    d1[kv] = pack(u1);
    d2[kv] = pack(u2);
  };
  if constexpr (MODE == GM_QKV) {
    const int n = p.n_embd, NV = n >> 3;
    const PairItem itm = resolve_pair(p.pairs, item, n);
    int tok = itm.tok;
    if (tok < 0 || tok >= p.target_vocab) {
      if (tid == 0 && (itm.write_kv || p.row_base == 0)) set_status(p.status, EAGLE3_DEV_BAD_TOKEN);
      tok = 0;
    }
    const uint4 *er = reinterpret_cast<const uint4 *>(p.embed + (size_t)tok * n);
    const float4 *gr = reinterpret_cast<const float4 *>(itm.g);
    const uint4 *wi = reinterpret_cast<const uint4 *>(p.norm0);
    const uint4 *wh = reinterpret_cast<const uint4 *>(p.norm1);
    // every load of this thread first (all in flight together), then convert and store
    constexpr int kIt = kPrepIters / 2;
    uint4 ue[kIt], uw[kIt], uh[kIt];
    float4 ga[kIt], gb[kIt];
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
      const int kv = tid + it * 256;
      if (kv < NV) {
        ue[it] = __ldg(er + kv);
        uw[it] = __ldg(wi + kv);
        uh[it] = __ldg(wh + kv);
        ga[it] = __ldcg(gr + 2 * kv);
        gb[it] = __ldcg(gr + 2 * kv + 1);
      }
    }
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
      const int kv = tid + it * 256;
      if (tid - (tid & 31) + it * 256 >= NV) break;  // the whole warp is past the end
      const bool act = kv < NV;
      if (!act) {
        const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (gsum) {
          group_sum(kv, false, z);
          group_sum(NV + kv, false, z);
        }
        continue;
      }
      const uint4 u = ue[it], w = uw[it];
      const float e[8] = {bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y), bf_lo(u.z), bf_hi(u.z), bf_lo(u.w), bf_hi(u.w)};
      const float wf[8] = {bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y), bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w)};
      float x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ss[0] += e[i] * e[i];
        x[i] = e[i] * wf[i];
      }
      put(kv, x);
      if (gsum) group_sum(kv, true, x);
      const float4 a = ga[it], b = gb[it];
      const uint4 hw = uh[it];
      const float g[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      const float hf[8] = {bf_lo(hw.x), bf_hi(hw.x), bf_lo(hw.y), bf_hi(hw.y), bf_lo(hw.z), bf_hi(hw.z), bf_lo(hw.w), bf_hi(hw.w)};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ss[H - 1] += g[i] * g[i];
        x[i] = g[i] * hf[i];
      }
      put(NV + kv, x);
      if (gsum) group_sum(NV + kv, true, x);
    }
  } else {
    const float4 *src = reinterpret_cast<const float4 *>(p.xf + (size_t)item * K);
    const uint4 *wn = reinterpret_cast<const uint4 *>(p.norm0);
    // every load of this thread first (all in flight together), then convert and store
    float4 va[kPrepIters], vb[kPrepIters];
    uint4 vw[kPrepIters];
#pragma unroll
    for (int it = 0; it < kPrepIters; ++it) {
      const int kv = tid + it * 256;
      if (kv < KV) {
        va[it] = __ldcg(src + 2 * kv);
        vb[it] = __ldcg(src + 2 * kv + 1);
        if constexpr (T::kNorm) vw[it] = __ldg(wn + kv);
      }
    }
#pragma unroll
    for (int it = 0; it < kPrepIters; ++it) {
      const int kv = tid + it * 256;
      if (tid - (tid & 31) + it * 256 >= KV) break;  // the whole warp is past the end
      if (kv >= KV) {
        const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (gsum) group_sum(kv, false, z);
        continue;
      }
      const float4 a = va[it], b = vb[it];
      float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      if constexpr (T::kNorm) {
        const uint4 w = vw[it];
        const float wf[8] = {bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y), bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w)};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          ss[0] += x[i] * x[i];
          x[i] *= wf[i];
        }
      }
      put(kv, x);
      if (gsum) group_sum(kv, true, x);
    }
  }
  if constexpr (T::kNorm) {
#pragma unroll
    for (int h = 0; h < H; ++h) {
      float v = ss[h];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if ((tid & 31) == 0) red[tid >> 5][h] = v;
    }
    __syncthreads();
    if (tid < H) {
      float t = 0.f;
      for (int w = 0; w < 8; ++w) t += red[w][tid];
      sumsq[(size_t)item * H + tid] = t;
    }
  }
}

cudaError_t tc_prep_launch(const GemvParams &p, int M, uint16_t *x0, uint16_t *x1, uint16_t *x2,
                           float *sumsq, float *gsum, cudaStream_t st, bool pdl) {
  if (p.K > kPrepIters * 256 * 8 || p.K % 8 || (gsum && p.K % 128)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(M);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  switch (p.mode) {
    case GM_QKV: return cudaLaunchKernelEx(&cfg, tc_prep_kernel<GM_QKV>, p, x0, x1, x2, sumsq, gsum);
    case GM_O: return cudaLaunchKernelEx(&cfg, tc_prep_kernel<GM_O>, p, x0, x1, x2, sumsq, gsum);
    case GM_GATEUP: return cudaLaunchKernelEx(&cfg, tc_prep_kernel<GM_GATEUP>, p, x0, x1, x2, sumsq, gsum);
    case GM_DOWN: return cudaLaunchKernelEx(&cfg, tc_prep_kernel<GM_DOWN>, p, x0, x1, x2, sumsq, gsum);
    case GM_LMHEAD: return cudaLaunchKernelEx(&cfg, tc_prep_kernel<GM_LMHEAD>, p, x0, x1, x2, sumsq, gsum);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace e3
