// Bookkeeping kernels of a speculative round: chain begin/end, rewind, the greedy accept
// walk and the boundary updates of rebuild and prefill.  All integer work except two
// row copies of the boundary feature.
#include "common.cuh"
#include "internal.h"

namespace e3 {

static cudaLaunchConfig_t small_cfg(int grid, int block, cudaStream_t st, bool pdl,
                                    cudaLaunchAttribute *attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cfg;
}

// Records the round start and the per-sequence chain length, and plans the attention
// work of every draft step.  gamma_eff follows the capacity rule:
// kv_len + gamma_eff + 1 <= max_cache_len.  Plan: pre[j][b] = sum over sequences b' < b of
// ceil(len_j(b') / U), len_j = clamp(kv_len + j + 1, 1, max_cache_len), pre[j][B] the
// total (the attention's unit partition).  One CTA; it does not signal its dependents
// early, so every later kernel of the round starts after it has finished.
__global__ void __launch_bounds__(1024) chain_begin_kernel(int B, int gamma, unsigned flags,
                                                           int max_cache_len, const int32_t *kv_len,
                                                           int32_t *round_start, int32_t *geff,
                                                           int32_t *geff_out, int *status, int U,
                                                           int32_t *pre, unsigned long long *slots,
                                                           int n_slots) {
  pdl_wait();
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
  // argmax slots of a chain whose steps leave their maxima there (zero before the first)
  for (int i = tid; slots && i < n_slots; i += nt) slots[i] = 0ull;
  for (int b = tid; b < B; b += nt) {
    const int L = kv_len[b];
    int ge = gamma;
    if (L < 0 || L + gamma + 1 > max_cache_len) {
      if ((flags & EAGLE3_SHRINK_GAMMA) && L >= 0 && max_cache_len - L - 1 >= 1) {
        ge = max_cache_len - L - 1;
      } else {
        ge = 0;
        set_status(status, EAGLE3_DEV_BAD_LENGTH);
      }
    }
    round_start[b] = L < 0 ? 0 : L;
    geff[b] = ge;
    if (geff_out) geff_out[b] = ge;
  }
  if (!pre || U < 1) return;
  __shared__ int wsum[32];
  const int per = (B + nt - 1) / nt;  // consecutive sequences per thread
  auto units = [&](int b, int j) {
    int len = kv_len[b] + j + 1;
    if (len > max_cache_len) len = max_cache_len;
    if (len < 1) len = 1;
    return (len + U - 1) / U;
  };
  for (int j = 0; j < gamma; ++j) {
    int32_t *row = pre + (size_t)j * (B + 1);
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int b = tid * per + i;
      if (b < B) local += units(b, j);
    }
    // exclusive scan of the per-thread sums across the block
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = lane < nt / 32 ? wsum[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += v;
      }
      if (lane < nt / 32) wsum[lane] = w;  // inclusive prefix over warps
    }
    __syncthreads();
    int run = incl - local + (warp > 0 ? wsum[warp - 1] : 0);
    for (int i = 0; i < per; ++i) {
      const int b = tid * per + i;
      if (b < B) {
        row[b] = run;
        run += units(b, j);
      }
    }
    if (tid == nt - 1) row[B] = run;  // the last thread ends at the total
    __syncthreads();
  }
}

__global__ void chain_end_kernel(int B, int32_t *kv_len, const int32_t *round_start,
                                 const int32_t *geff, ChainLast last) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) {
    // the last step's tokens, where its lm_head left the argmax in the slots
    if (last.slot)
      chain_step_outputs(last.slot, last.gamma - 1, b, last.gamma, geff, last.d2t, last.draft_vocab,
                         last.target_vocab, last.draft_tok, last.draft_id, nullptr, last.status);
    kv_len[b] = round_start[b] + geff[b];
  }
}

__global__ void rewind_kernel(int B, int32_t *kv_len, const int32_t *round_start) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) kv_len[b] = round_start[b];
}

// n = leading matches of target_pred[b, i] with draft_tok[b, i]; bonus = target_pred[b, n].
__global__ void accept_kernel(int B, int gamma, const int32_t *draft_tok, const int32_t *target_pred,
                              const int32_t *gamma_eff, int32_t *n_acc, int32_t *bonus) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  int ge = gamma_eff ? gamma_eff[b] : gamma;
  ge = ge < 0 ? 0 : (ge > gamma ? gamma : ge);
  const int32_t *d = draft_tok + (size_t)b * gamma;
  const int32_t *y = target_pred + (size_t)b * (gamma + 1);
  int n = 0;
  while (n < ge && y[n] == d[n]) ++n;
  n_acc[b] = n;
  bonus[b] = y[n];
}

// New boundary (fc v_n, bonus) and kv_len += n + 1.
__global__ void rebuild_finish_kernel(int B, int gamma, int n_embd, const float *enc_g,
                                      const int32_t *n_acc, const int32_t *bonus, float *bnd_g,
                                      int32_t *bnd_tok, int32_t *kv_len, int max_cache_len,
                                      int *status) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.y;
  int n = n_acc[b];
  if (n < 0 || n > gamma) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, EAGLE3_DEV_BAD_LENGTH);
    n = n < 0 ? 0 : gamma;
  }
  const float *src = enc_g + ((size_t)b * (gamma + 1) + n) * n_embd;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_embd; i += gridDim.x * blockDim.x)
    bnd_g[(size_t)b * n_embd + i] = src[i];
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    bnd_tok[b] = bonus[b];
    int L = kv_len[b] + n + 1;
    if (L > max_cache_len) {
      set_status(status, EAGLE3_DEV_BAD_LENGTH);
      L = max_cache_len;
    }
    kv_len[b] = L;
  }
}

__global__ void prefill_finish_kernel(int b, int n_embd, int kv_len_value, const float *enc_last,
                                      const int32_t *next_tok, float *bnd_g, int32_t *bnd_tok,
                                      int32_t *kv_len) {
  pdl_trigger();
  pdl_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_embd; i += gridDim.x * blockDim.x)
    bnd_g[(size_t)b * n_embd + i] = enc_last[i];
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    bnd_tok[b] = next_tok[b];
    kv_len[b] = kv_len_value;
  }
}

// Residual of checkpoints with norm_before_residual: out[b] = RMSNorm(g[b]) * w (w the
// bf16 hidden_norm gain), one CTA per sequence.
__global__ void __launch_bounds__(256) res_norm_kernel(int n, float eps, const float *g, const uint16_t *w,
                                                       float *out) {
  __shared__ float part[8];
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, tid = threadIdx.x;
  const float *x = g + (size_t)b * n;
  float s = 0.f;
  for (int i = tid; i < n; i += 256) s = fmaf(x[i], x[i], s);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((tid & 31) == 0) part[tid >> 5] = s;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) t += part[i];  // the same order in every thread
  const float scale = rsqrtf(t / (float)n + eps);
  for (int i = tid; i < n; i += 256) out[(size_t)b * n + i] = x[i] * scale * bf1(w[i]);
}

cudaError_t launch_res_norm(int B, int n, float eps, const float *g, const uint16_t *w, float *out,
                            cudaStream_t st) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = small_cfg(B, 256, st, true, attr);
  return cudaLaunchKernelEx(&cfg, res_norm_kernel, n, eps, g, w, out);
}

// Self-test of the bounded wait every kernel uses on its mbarriers: one thread waits on a
// barrier that nothing completes, so the wait gives up, raises EAGLE3_DEV_TIMEOUT in
// *status and sets the CTA's abort flag; a second wait then returns at once.  Nothing is
// in flight on the barrier, so the kernel ends normally and the context stays usable.
__global__ void wait_selftest_kernel(int *status, int *result) {
  __shared__ __align__(8) unsigned long long bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool first = mbar_wait(smem_addr(&bar), 0, &abort_flag, status);
    const bool second = mbar_wait(smem_addr(&bar), 0, &abort_flag, status);
    result[0] = (first ? 1 : 0) | (second ? 2 : 0) | (abort_flag ? 4 : 0);
  }
}

cudaError_t launch_wait_selftest(int *status, int *result, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(status, result);
  return cudaGetLastError();
}

cudaError_t launch_chain_begin(int B, int gamma, unsigned flags, int max_cache_len,
                               const int32_t *kv_len, int32_t *round_start, int32_t *geff,
                               int32_t *geff_out, int *status, int unit_keys, int32_t *unit_pre,
                               unsigned long long *slots, int n_slots, cudaStream_t st) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = small_cfg(1, 1024, st, false, attr);
  return cudaLaunchKernelEx(&cfg, chain_begin_kernel, B, gamma, flags, max_cache_len, kv_len,
                            round_start, geff, geff_out, status, unit_keys, unit_pre, slots, n_slots);
}

cudaError_t launch_chain_end(int B, int32_t *kv_len, const int32_t *round_start,
                             const int32_t *geff, const ChainLast &last, cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = small_cfg((B + 127) / 128, 128, st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, chain_end_kernel, B, kv_len, round_start, geff, last);
}

// The bookkeeping kernels are launched as programmatic dependents of whatever kernel
// precedes them on the stream (each waits for it before touching data), so their launch
// overlaps the previous kernel's tail.
cudaError_t launch_rewind(int B, int32_t *kv_len, const int32_t *round_start, cudaStream_t st) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = small_cfg((B + 127) / 128, 128, st, true, attr);
  return cudaLaunchKernelEx(&cfg, rewind_kernel, B, kv_len, round_start);
}

cudaError_t launch_accept(int B, int gamma, const int32_t *draft_tok, const int32_t *target_pred,
                          const int32_t *gamma_eff, int32_t *n_acc, int32_t *bonus,
                          cudaStream_t st) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = small_cfg((B + 127) / 128, 128, st, true, attr);
  return cudaLaunchKernelEx(&cfg, accept_kernel, B, gamma, draft_tok, target_pred, gamma_eff, n_acc,
                            bonus);
}

cudaError_t launch_rebuild_finish(int B, int gamma, int n_embd, const float *enc_g,
                                  const int32_t *n_acc, const int32_t *bonus, float *bnd_g,
                                  int32_t *bnd_tok, int32_t *kv_len, int max_cache_len,
                                  int *status, cudaStream_t st) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = small_cfg(1, 256, st, true, attr);
  cfg.gridDim = dim3((n_embd + 1023) / 1024, B);
  return cudaLaunchKernelEx(&cfg, rebuild_finish_kernel, B, gamma, n_embd, enc_g, n_acc, bonus, bnd_g,
                            bnd_tok, kv_len, max_cache_len, status);
}

cudaError_t launch_prefill_finish(int b, int n_embd, int kv_len_value, const float *enc_last,
                                  const int32_t *next_tok, float *bnd_g, int32_t *bnd_tok,
                                  int32_t *kv_len, cudaStream_t st) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = small_cfg((n_embd + 1023) / 1024, 256, st, true, attr);
  return cudaLaunchKernelEx(&cfg, prefill_finish_kernel, b, n_embd, kv_len_value, enc_last, next_tok,
                            bnd_g, bnd_tok, kv_len);
}

}  // namespace e3
