// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace e3 {

// Largest float32 activation block (items * K * 4 bytes) one GEMV launch keeps in
// shared memory.
constexpr size_t kGemvMaxXBytes = 128 * 1024;
// Dynamic shared memory ceiling of a GEMV CTA (x + weight ring + row sums + barriers).
constexpr size_t kGemvSmemLimit = 224 * 1024;

cudaError_t gemv_prepare();
int gemv_items_per_launch(const GemvParams &p, int items, int grid);
cudaError_t gemv_launch(const GemvParams &p, int grid, cudaStream_t st, bool pdl);
// INT4-weight instantiations (gemv_q4.cu); nb items per launch as gemv_items_per_launch.
cudaError_t gemv_q4_prepare();
cudaError_t gemv_q4_launch(const GemvParams &p, int nb, int grid, cudaStream_t st, bool pdl);

// Tensor-core GEMM (gemm_tc.cu): weights [rows, K] against M activation rows.
constexpr size_t kTcSmemLimit = 220 * 1024;
struct TcLaunch {
  GemvParams p;                 // mode, rows, row_base, K and the epilogue's parameters
  int M;                        // activation rows (items)
  const void *a0, *a1, *a2;     // weight matrices of the mode (see gemm_tc.cu)
  int a0_rows, a1_rows, a2_rows;
  const uint16_t *b0, *b1, *b2; // activations bf16 [M, K]: one part (encode) or three
  const uint32_t *s0, *s1, *s2; // INT4 weights: (scale, zero) rows of a0 / a1 / a2 (a* are
                                // then code rows of K / 2 bytes); null for bf16 weights
  int sz_stride;                // INT4: pairs per (scale, zero) row
  const float *gsum;            // INT4: [M][K / 128] sums of x per 128-wide group
  const float *sumsq;           // [M][halves] (norm modes)
  float *part;                  // split-K partials
  size_t part_elems;
  unsigned *tile_cnt;           // split-K counters (zero between launches)
  size_t tile_cnt_elems;
  int num_sms;
  int schedule;                 // TC_SCHED_*: how the tiles are split over the SMs
};
// eagle3_set_tc_schedule's values
constexpr int TC_SCHED_AUTO = 0, TC_SCHED_STREAM_K = 1, TC_SCHED_CLUSTER = 2;
// eagle3_set_attention's values
constexpr int ATTN_CUDA_CORES = 0, ATTN_TENSOR_CORES = 1;
cudaError_t tc_prepare();
int tc_tile_items(int M, int mode);
cudaError_t tc_launch(const TcLaunch &L, cudaStream_t st, bool pdl);
// INT4-weight instantiations (gemm_tc_q4.cu)
cudaError_t tc_q4_prepare();
cudaError_t tc_q4_launch(const TcLaunch &L, cudaStream_t st, bool pdl);
cudaError_t tc_prep_launch(const GemvParams &p, int M, uint16_t *x0, uint16_t *x1, uint16_t *x2,
                           float *sumsq, float *gsum, cudaStream_t st, bool pdl);

bool attn_supported(int head_dim, int group);
cudaError_t attn_prepare();
int attn_unit_keys(int head_dim, int group, int page_size, int kv_q);
cudaError_t kv_quant_launch(const GemvParams &p, int items, int k_row, int v_row, cudaStream_t st,
                            bool pdl);
cudaError_t attn_launch(const AttnParams &p, int num_sms, cudaStream_t st, bool pdl);
// Tensor-core variant for bf16 KV (attention_tc.cu): d 64 / 128 / 256, G <= 4, units of
// 16..64 keys (a multiple of 16).
bool attn_tc_supported(int head_dim, int group, int unit_keys);
cudaError_t attn_tc_prepare();
cudaError_t attn_tc_launch(const AttnParams &p, int num_sms, cudaStream_t st, bool pdl);

// Small bookkeeping kernels (small.cu).
// slots / n_slots: the chain's per-step argmax slots, zeroed first (null: none)
cudaError_t launch_chain_begin(int B, int gamma, unsigned flags, int max_cache_len,
                               const int32_t *kv_len, int32_t *round_start, int32_t *geff,
                               int32_t *geff_out, int *status, int unit_keys, int32_t *unit_pre,
                               unsigned long long *slots, int n_slots, cudaStream_t st);
// The last step of a chain whose lm_head left its argmax in the slots (slot null: its
// lm_head decoded it itself).
struct ChainLast {
  const unsigned long long *slot;  // [B] of the last step
  int gamma, draft_vocab, target_vocab;
  const int64_t *d2t;
  int32_t *draft_tok, *draft_id;
  int *status;
};
cudaError_t launch_chain_end(int B, int32_t *kv_len, const int32_t *round_start,
                             const int32_t *geff, const ChainLast &last, cudaStream_t st, bool pdl);
cudaError_t launch_rewind(int B, int32_t *kv_len, const int32_t *round_start, cudaStream_t st);
cudaError_t launch_wait_selftest(int *status, int *result, cudaStream_t st);
cudaError_t launch_res_norm(int B, int n, float eps, const float *g, const uint16_t *w, float *out,
                            cudaStream_t st);
cudaError_t launch_accept(int B, int gamma, const int32_t *draft_tok, const int32_t *target_pred,
                          const int32_t *gamma_eff, int32_t *n_acc, int32_t *bonus,
                          cudaStream_t st);
cudaError_t launch_rebuild_finish(int B, int gamma, int n_embd, const float *enc_g,
                                  const int32_t *n_acc, const int32_t *bonus, float *bnd_g,
                                  int32_t *bnd_tok, int32_t *kv_len, int max_cache_len,
                                  int *status, cudaStream_t st);
cudaError_t launch_prefill_finish(int b, int n_embd, int kv_len_value, const float *enc_last,
                                  const int32_t *next_tok, float *bnd_g, int32_t *bnd_tok,
                                  int32_t *kv_len, cudaStream_t st);

}  // namespace e3
