// INT4-weight instantiations of the weight-streaming GEMV (gemv_kernel.cuh): the chain's
// q/k/v, o, gate/up, down and lm_head projections (and the k/v-only teacher forcing) of a
// drafter whose weights are 4-bit codes with a bf16 (scale, zero) per 128-wide k group.
// The fc encode keeps bf16 weights.
#include "gemv_kernel.cuh"

namespace e3 {

cudaError_t gemv_q4_prepare() {
  cudaError_t e = prepare_mode<GM_QKV, true>();
  if (e == cudaSuccess) e = prepare_mode<GM_O, true>();
  if (e == cudaSuccess) e = prepare_mode<GM_GATEUP, true>();
  if (e == cudaSuccess) e = prepare_mode<GM_DOWN, true>();
  if (e == cudaSuccess) e = prepare_mode<GM_LMHEAD, true>();
  return e;
}

cudaError_t gemv_q4_launch(const GemvParams &p, int nb, int grid, cudaStream_t st, bool pdl) {
  if (p.K % 128 || p.sz_stride < p.K / 128 || p.sz_stride % 4) return cudaErrorInvalidValue;
  switch (p.mode) {
    case GM_QKV: return dispatch_nb<GM_QKV, true>(p, nb, grid, st, pdl);
    case GM_O: return dispatch_nb<GM_O, true>(p, nb, grid, st, pdl);
    case GM_GATEUP: return dispatch_nb<GM_GATEUP, true>(p, nb, grid, st, pdl);
    case GM_DOWN: return dispatch_nb<GM_DOWN, true>(p, nb, grid, st, pdl);
    case GM_LMHEAD: return dispatch_nb<GM_LMHEAD, true>(p, nb, grid, st, pdl);
    default: return cudaErrorInvalidValue;  // the encode has bf16 weights
  }
}

}  // namespace e3
