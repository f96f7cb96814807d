// eagle3_lmhead_argmax_noalloc: the fused final-RMSNorm + lm_head + argmax + d2t kernel
// of the draft chain, callable without a context and without any device allocation.
//
// The kernel needs scratch beyond its inputs and outputs: one 64-bit argmax slot per row
// of x and an arrival counter that lets the last CTA finish the reduction.  Inside a
// context that scratch is carved from the caller's workspace.  Here it lives in the
// file-scope array below, which every GPU that loads the library holds until the process
// exits.  The launch itself is the same kernel the chain uses.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kNoAllocMaxRows = 64;

// [0, 64): argmax slots (u64); [64]: arrival counter (u32, padded to 8 bytes).
static __device__ __align__(256) unsigned long long g_lmhead_scratch[kNoAllocMaxRows + 1];

// The kernel marks a row valid when its step (0 here) is below this per-row chain length.
static __device__ __align__(16) int32_t g_lmhead_rows_valid[kNoAllocMaxRows] = {
    1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1,
    1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1,
    1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1};

constexpr int kMaxDevices = 64;

struct DeviceScratch {
  bool ready = false;
  unsigned long long *scratch = nullptr;
  int32_t *rows_valid = nullptr;
  int num_sms = 0;
};

std::mutex g_mu;
DeviceScratch g_dev[kMaxDevices];

// Device addresses of the two arrays on the current device; looked up once per device.
// (In host code the arrays' names are only host-side stand-ins, not device addresses.)
int scratch_for_current_device(DeviceScratch *out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return EAGLE3_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceScratch &d = g_dev[dev];
  if (!d.ready) {
    void *a = nullptr, *b = nullptr;
    if (cudaGetSymbolAddress(&a, g_lmhead_scratch) != cudaSuccess) return EAGLE3_ERR_CUDA;
    if (cudaGetSymbolAddress(&b, g_lmhead_rows_valid) != cudaSuccess) return EAGLE3_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return EAGLE3_ERR_CUDA;
    if (e3::gemv_prepare() != cudaSuccess) return EAGLE3_ERR_CUDA;
    d.scratch = static_cast<unsigned long long *>(a);
    d.rows_valid = static_cast<int32_t *>(b);
    d.ready = true;
  }
  *out = d;
  return EAGLE3_OK;
}

bool aligned16(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int eagle3_lmhead_argmax_noalloc(const uint16_t *lm_head, const uint16_t *final_norm,
                                            const int64_t *d2t, const float *x, int rows,
                                            int n_embd, int draft_vocab, int target_vocab,
                                            float rms_eps, int32_t *draft_id, int32_t *target_id,
                                            float *logits, eagle3_stream_t stream) {
  if (rows < 1 || rows > kNoAllocMaxRows) return EAGLE3_ERR_INVALID_ARG;
  if (n_embd <= 0 || n_embd % 8 || 4 * (size_t)n_embd > e3::kGemvMaxXBytes) return EAGLE3_ERR_INVALID_ARG;
  if (draft_vocab <= 0 || draft_vocab % 2 || target_vocab <= 0 || !(rms_eps >= 0.f))
    return EAGLE3_ERR_INVALID_ARG;
  if (!aligned16(lm_head) || !aligned16(final_norm) || !aligned16(x) || !d2t || !target_id)
    return EAGLE3_ERR_INVALID_ARG;
  if (logits && !aligned16(logits)) return EAGLE3_ERR_INVALID_ARG;
  DeviceScratch d;
  const int rc = scratch_for_current_device(&d);
  if (rc != EAGLE3_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // slots and counter must start at zero; a call that was cut short may have left values
  if (cudaMemsetAsync(d.scratch, 0, sizeof(unsigned long long) * (kNoAllocMaxRows + 1), st) !=
      cudaSuccess)
    return EAGLE3_ERR_CUDA;

  e3::GemvParams p;
  memset(&p, 0, sizeof(p));
  p.mode = e3::GM_LMHEAD;
  p.rows = draft_vocab;
  p.K = n_embd;
  p.n_embd = n_embd;
  p.draft_vocab = draft_vocab;
  p.target_vocab = target_vocab;
  p.eps = rms_eps;
  p.w0 = lm_head;
  p.norm0 = final_norm;
  p.xf = x;
  p.am_slot = d.scratch;
  p.am_count = reinterpret_cast<unsigned int *>(d.scratch + kNoAllocMaxRows);
  p.d2t = d2t;
  p.draft_tok = target_id;
  p.draft_id = draft_id;
  p.gamma_eff = d.rows_valid;
  p.gamma = 1;
  p.step = 0;
  p.dbg_f = logits;
  p.dbg_stride_b = draft_vocab;
  p.dbg_off = 0;
  const int nb = e3::gemv_items_per_launch(p, rows, d.num_sms);
  for (int i0 = 0; i0 < rows; i0 += nb) {
    p.item0 = i0;
    p.items = rows - i0 < nb ? rows - i0 : nb;
    if (e3::gemv_launch(p, d.num_sms, st, false) != cudaSuccess) return EAGLE3_ERR_CUDA;
  }
  return EAGLE3_OK;
}
