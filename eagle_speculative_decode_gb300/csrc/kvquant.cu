// Quantized drafter KV append: q8_0 keys and q5_1 values in blocks of 32 values
// ("memra_engine/eagle.rs", Eagle3Scratch: the drafter KV uses the q8_0-K / q5_1-V layout
// of the trunk KV, 34- and 24-byte blocks, head_dim % 32 == 0).
//
// The q/k/v projection (GEMV or tensor-core GEMM) leaves the float32 k (after RoPE) and v
// of every item in a staging buffer; this kernel quantizes them.  One warp per block of
// 32 values of one (item, K or V, kv head): lane i holds value i, the warp reduces the
// block's max |x| (q8_0) or min and max (q5_1), lane 0 writes the header and every lane
// its code, through the page table at the item's position.  Codes are decided in float32
// with the stored fp16 scale: d = fp16(max|x| / 127), code = rint(x / d) clamped to
// [-127, 127] (q8_0); d = fp16((max - min) / 31), m = fp16(min), code = rint((x - m) / d)
// clamped to [0, 31] (q5_1); all codes 0 when d = 0.
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace e3 {

constexpr int kQuantWarps = 8;

__global__ void __launch_bounds__(kQuantWarps * 32) kv_quant_kernel(const GemvParams p, int items, int k_row,
                                                                     int v_row) {
  pdl_trigger();
  pdl_wait();  // the staged k / v come from the projection just before
  const int lane = threadIdx.x & 31;
  const int d = p.head_dim, nb = d / 32, hkv = p.n_head_kv;
  const int kr = hkv * d;
  const long long total = (long long)items * 2 * hkv * nb;
  const long long w = (long long)blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
  if (w >= total) return;  // whole warps only
  const int blk = (int)(w % nb);
  const int head = (int)((w / nb) % hkv);
  const int kind = (int)((w / ((long long)nb * hkv)) % 2);  // 0: K, 1: V
  const int item = (int)(w / ((long long)nb * hkv * 2));

  const PairItem it = resolve_pair(p.pairs, item, p.n_embd);
  if (!it.write_kv) return;
  const int pos = it.pos;
  if (pos < 0 || pos >= p.max_cache_len) {
    if (lane == 0) set_status(p.status, EAGLE3_DEV_BAD_POSITION);
    return;
  }
  const int pg = p.page_table[(size_t)it.b * p.max_pages + pos / p.page_size];
  if (pg < 0 || pg >= p.num_pages) {
    if (lane == 0) set_status(p.status, EAGLE3_DEV_BAD_PAGE);
    return;
  }
  const float x = __ldcg(p.kv_stage + ((size_t)item * 2 + kind) * kr + (size_t)head * d + blk * 32 + lane);
  const size_t slot = ((size_t)pg * hkv + head) * p.page_size + pos % p.page_size;
  if (kind == 0) {
    unsigned char *blkp = reinterpret_cast<unsigned char *>(p.k_pool) + slot * k_row + (size_t)blk * 34;
    float amax = fabsf(x);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const __half d16 = __float2half_rn(__fdiv_rn(amax, 127.0f));
    const float df = __half2float(d16);
    int code = 0;
    if (df > 0.f) code = max(-127, min(127, (int)rintf(__fdiv_rn(x, df))));
    if (lane == 0) *reinterpret_cast<__half *>(blkp) = d16;
    blkp[2 + lane] = (unsigned char)(signed char)code;
  } else {
    unsigned char *blkp = reinterpret_cast<unsigned char *>(p.v_pool) + slot * v_row + (size_t)blk * 24;
    float mn = x, mx = x;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    const __half d16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 31.0f));
    const __half m16 = __float2half_rn(mn);
    const float df = __half2float(d16), mf = __half2float(m16);
    int code = 0;
    if (df > 0.f) code = max(0, min(31, (int)rintf(__fdiv_rn(__fsub_rn(x, mf), df))));
    const unsigned qh = __ballot_sync(0xffffffffu, (code >> 4) & 1);
    const int hi = __shfl_down_sync(0xffffffffu, code, 16);  // code of value lane + 16
    if (lane == 0) {
      *reinterpret_cast<__half *>(blkp) = d16;
      *reinterpret_cast<__half *>(blkp + 2) = m16;
      *reinterpret_cast<unsigned *>(blkp + 4) = qh;
    }
    if (lane < 16) blkp[8 + lane] = (unsigned char)((code & 15) | ((hi & 15) << 4));
  }
}

cudaError_t kv_quant_launch(const GemvParams &p, int items, int k_row, int v_row, cudaStream_t st,
                            bool pdl) {
  if (items <= 0) return cudaSuccess;
  const long long warps = (long long)items * 2 * p.n_head_kv * (p.head_dim / 32);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((warps + kQuantWarps - 1) / kQuantWarps));
  cfg.blockDim = dim3(kQuantWarps * 32);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kv_quant_kernel, p, items, k_row, v_row);
}

}  // namespace e3
