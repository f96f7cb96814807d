// INT4-weight instantiations of the tensor-core GEMM (gemm_tc.cuh): the projections of a
// drafter whose weights are 4-bit codes with a bf16 (scale, zero) per 128-wide k group,
// decoded to bf16 in shared memory by the epilogue warps.  The fc encode keeps bf16.
#include "gemm_tc.cuh"

namespace e3 {

cudaError_t tc_q4_launch(const TcLaunch &L, cudaStream_t st, bool pdl) {
  switch (L.p.mode) {
    case GM_QKV: return tc_launch_mode<GM_QKV, true>(L, st, pdl);
    case GM_O: return tc_launch_mode<GM_O, true>(L, st, pdl);
    case GM_GATEUP: return tc_launch_mode<GM_GATEUP, true>(L, st, pdl);
    case GM_DOWN: return tc_launch_mode<GM_DOWN, true>(L, st, pdl);
    case GM_LMHEAD: return tc_launch_mode<GM_LMHEAD, true>(L, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t tc_q4_prepare() {
  cudaError_t e = tc_prepare_mode<GM_QKV, true>();
  if (e == cudaSuccess) e = tc_prepare_mode<GM_O, true>();
  if (e == cudaSuccess) e = tc_prepare_mode<GM_GATEUP, true>();
  if (e == cudaSuccess) e = tc_prepare_mode<GM_DOWN, true>();
  if (e == cudaSuccess) e = tc_prepare_mode<GM_LMHEAD, true>();
  return e;
}

}  // namespace e3
