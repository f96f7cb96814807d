// bf16 instantiations of the weight-streaming GEMV (gemv_kernel.cuh) and the GEMV entry
// points; INT4 launches are forwarded to gemv_q4.cu.
#include <algorithm>

#include "gemv_kernel.cuh"

namespace e3 {

// Raise every instantiation's dynamic shared memory limit once, outside any capture.
cudaError_t gemv_prepare() {
  cudaError_t e = prepare_mode<GM_ENCODE, false>();
  if (e == cudaSuccess) e = prepare_mode<GM_QKV, false>();
  if (e == cudaSuccess) e = prepare_mode<GM_O, false>();
  if (e == cudaSuccess) e = prepare_mode<GM_GATEUP, false>();
  if (e == cudaSuccess) e = prepare_mode<GM_DOWN, false>();
  if (e == cudaSuccess) e = prepare_mode<GM_LMHEAD, false>();
  if (e == cudaSuccess) e = gemv_q4_prepare();
  return e;
}

int gemv_items_per_launch(const GemvParams &p, int items, int grid) {
  // x of one launch lives in shared memory (NB * K * (2 or 4) bytes <= kGemvMaxXBytes), and
  // so do the per-warp row sums of the CTA's rows (max_rows * warps * halves * NB floats):
  // NB halves until both fit with a two-stage ring of single rows.
  const int eb = p.mode == GM_ENCODE ? 2 : 4;
  const int H = p.mode == GM_QKV ? 2 : 1;
  const int unit = (p.mode == GM_QKV || p.mode == GM_GATEUP) ? 2 : 1;
  const int nunits = p.rows / unit;
  const int g = std::max(1, std::min(grid, nunits));
  const int max_rows = tiles_max_rows_bound(p.rows, g);
  const int rb = gemv_row_bytes(p.sz0 != nullptr, p.K, p.sz_stride);
  auto fits = [&](int nb) {
    if ((size_t)nb * p.K * eb > kGemvMaxXBytes) return false;
    const GemvSmem L = gemv_smem_layout(nb, 1, H, eb, p.K, 2, max_rows, rb);
    return (size_t)L.total + 64 <= kGemvSmemLimit;
  };
  int nb = 8;
  while (nb > 1 && !fits(nb)) nb >>= 1;
  while (nb > 1 && nb / 2 >= items) nb >>= 1;
  return nb;
}

cudaError_t gemv_launch(const GemvParams &p, int grid, cudaStream_t st, bool pdl) {
  const int nb = gemv_items_per_launch(p, p.items, grid);
  if (p.items > nb || p.items < 1) return cudaErrorInvalidValue;
  if (p.sz0) return gemv_q4_launch(p, nb, grid, st, pdl);  // INT4 weights
  switch (p.mode) {
    case GM_ENCODE: return dispatch_nb<GM_ENCODE, false>(p, nb, grid, st, pdl);
    case GM_QKV: return dispatch_nb<GM_QKV, false>(p, nb, grid, st, pdl);
    case GM_O: return dispatch_nb<GM_O, false>(p, nb, grid, st, pdl);
    case GM_GATEUP: return dispatch_nb<GM_GATEUP, false>(p, nb, grid, st, pdl);
    case GM_DOWN: return dispatch_nb<GM_DOWN, false>(p, nb, grid, st, pdl);
    case GM_LMHEAD: return dispatch_nb<GM_LMHEAD, false>(p, nb, grid, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace e3
