// Device helpers and launch-parameter structs shared by the EAGLE-3 drafter kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/eagle3.h"

namespace e3 {

constexpr int kGemvThreads = 512;  // GEMV consumer threads (16 warps)
constexpr int kGemvWarps = kGemvThreads / 32;

// ------------------------------------------------------------------ PDL (griddepcontrol)
// Programmatic dependent launch: a kernel may start while its predecessor drains.  Code
// before pdl_wait() touches only constant data (weights); pdl_trigger() lets the next
// kernel in the stream be scheduled early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------------- loads
// Streaming 16-byte weight load: read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Hint the L2 to fetch [p, p + bytes) (bytes a multiple of 16, p 16-byte aligned).
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// bf16 pair in a 32-bit word -> two floats (exact widening).
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ float bf1(uint16_t u) { return __uint_as_float(((uint32_t)u) << 16); }

// float -> bf16 bits, round to nearest even (finite inputs).
__device__ __forceinline__ uint16_t f2bf(float f) {
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

__device__ __forceinline__ void set_status(int *status, int bit) {
  if (status) atomicOr(status, bit);
}

// ------------------------------------------------------- mbarrier + bulk copies (TMA)
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: gives up after ~1 s of polling, raises EAGLE3_DEV_TIMEOUT and the CTA's
// abort flag so that every later wait of the CTA returns at once.
constexpr uint32_t kWaitLimit = 1u << 21;
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          int *status) {
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (i > 64) __nanosleep(64);
  }
  *abort_flag = 1;
  set_status(status, EAGLE3_DEV_TIMEOUT);
  return false;
}
// One bulk copy global -> shared (16-byte aligned, size a multiple of 16) completing on bar.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}
// L2 policy for data read once per step (weights): evict first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// Barrier among the consumer threads of a GEMV CTA (the producer warp is not in it).
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kGemvThreads) : "memory"); }

// Order-preserving map of a float to uint32 (larger float -> larger key); -0 -> +0.
__device__ __forceinline__ uint32_t float_order_key(float f) {
  if (f == 0.0f) f = 0.0f;
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ------------------------------------------------------------------ item sources
// A GEMV "item" is one activation row.  For the layer-input modes an item is a
// (token, g, position) triple whose meaning depends on who launches the kernel.
enum PairKind : int {
  PAIR_CHAIN = 0,    // item = sequence b, draft step j
  PAIR_REBUILD = 1,  // item = (b, i), i = 0..gamma
  PAIR_PREFILL = 2,  // item = position p of one sequence
};

struct PairSource {
  int kind;
  int step;                  // chain: j
  int gamma;                 // chain / rebuild: gamma
  int seq;                   // prefill: the sequence
  int pos0;                  // prefill: position of item 0
  int tok_stride;            // prefill: row stride of tokens
  const int32_t *bnd_tok;    // chain j == 0, rebuild i == 0
  const float *bnd_g;        // [B, n]
  const int32_t *step_tok;   // chain j > 0: token of this step per b [B]
  // chain j > 0 with the argmax left in its slot: the winning (order key, ~row) of step
  // j - 1 per b, decoded here (step_tok is then not read)
  const unsigned long long *step_key;
  const int64_t *d2t;        // draft id -> target id offsets (null: the ids are target ids)
  int draft_vocab, target_vocab;
  const float *step_g;       // chain j > 0: g of this step [B, n]
  const int32_t *draft_tok;  // rebuild: [B, gamma]
  const float *enc_g;        // rebuild: [B, gamma + 1, n]; prefill: [items, n]
  const int32_t *tokens;     // prefill: [*, tok_stride]
  const int32_t *kv_len;     // [B]
  const int32_t *gamma_eff;  // chain: [B]
  const int32_t *n_acc;      // rebuild: [B]
};

struct PairItem {
  int b;
  int tok;
  const float *g;
  int pos;
  bool write_kv;
};

// The draft id and target id of an argmax slot's winning key (order key << 32 | ~row);
// false when either is out of range.
__device__ __forceinline__ bool argmax_ids(unsigned long long key, const int64_t *d2t, int draft_vocab,
                                           int target_vocab, uint32_t &id, long long &tgt) {
  id = 0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull);
  if (id >= (uint32_t)draft_vocab) {
    id = 0;
    tgt = 0;
    return false;
  }
  tgt = d2t ? (long long)id + d2t[id] : (long long)id;
  if (tgt < 0 || tgt >= target_vocab) {
    tgt = 0;
    return false;
  }
  return true;
}

// A chain's step whose lm_head left its argmax in the step's slots (am_defer): thread t
// writes item t's draft token and id of that step and the next step's token, as
// lmhead_finalize does; run by the kernel after it (the next step's q/k/v, or the chain
// end for the last step) once that lm_head has completed.
__device__ __forceinline__ void chain_step_outputs(const unsigned long long *slot, int step, int item, int gamma,
                                                   const int32_t *gamma_eff, const int64_t *d2t, int draft_vocab,
                                                   int target_vocab, int32_t *draft_tok, int32_t *draft_id,
                                                   int32_t *next_tok, int *status) {
  uint32_t id;
  long long tgt;
  if (!argmax_ids(slot[item], d2t, draft_vocab, target_vocab, id, tgt)) set_status(status, EAGLE3_DEV_BAD_TOKEN);
  const bool valid = !gamma_eff || step < gamma_eff[item];
  const size_t o = (size_t)item * gamma + step;
  draft_tok[o] = valid ? (int32_t)tgt : -1;
  if (draft_id) draft_id[o] = valid ? (int32_t)id : -1;
  if (next_tok) next_tok[item] = (int32_t)tgt;
}

__device__ __forceinline__ PairItem resolve_pair(const PairSource &s, int item, int n_embd) {
  PairItem it;
  if (s.kind == PAIR_CHAIN) {
    it.b = item;
    if (s.step == 0) {
      it.tok = s.bnd_tok[item];
      it.g = s.bnd_g + (size_t)item * n_embd;
    } else {
      if (s.step_key) {
        uint32_t id;
        long long tgt;
        it.tok = argmax_ids(s.step_key[item], s.d2t, s.draft_vocab, s.target_vocab, id, tgt) ? (int)tgt : -1;
      } else {
        it.tok = s.step_tok[item];
      }
      it.g = s.step_g + (size_t)item * n_embd;
    }
    it.pos = s.kv_len[item] + s.step;
    it.write_kv = s.step < s.gamma_eff[item];
  } else if (s.kind == PAIR_REBUILD) {
    const int b = item / (s.gamma + 1), i = item % (s.gamma + 1);
    it.b = b;
    if (i == 0) {
      it.tok = s.bnd_tok[b];
      it.g = s.bnd_g + (size_t)b * n_embd;
    } else {
      it.tok = s.draft_tok[(size_t)b * s.gamma + (i - 1)];
      it.g = s.enc_g + ((size_t)b * (s.gamma + 1) + (i - 1)) * n_embd;
    }
    it.pos = s.kv_len[b] + i;
    it.write_kv = i <= s.n_acc[b];
  } else {
    it.b = s.seq;
    const int p = s.pos0 + item;
    it.tok = s.tokens[(size_t)s.seq * s.tok_stride + p + 1];
    it.g = s.enc_g + (size_t)item * n_embd;
    it.pos = p;
    it.write_kv = true;
  }
  return it;
}

// ----------------------------------------------------------------- GEMV params
enum GemvMode : int {
  GM_ENCODE = 0,  // x = aux (bf16 [items, 3n]); y -> out_f [items, rows]
  GM_QKV = 1,     // x = [RMS(embed) w_in ; RMS(g) w_hid]; rows: q | k | v (row_base skips q)
  GM_O = 2,       // x = attention output; y + g -> x1
  GM_GATEUP = 3,  // x = RMS(x1) w_post; rows interleave gate/up; silu(gate) * up -> act
  GM_DOWN = 4,    // x = act; y + x1 -> gsum (next g)
  GM_LMHEAD = 5,  // x = RMS(gsum) w_final; argmax + d2t
};

struct GemvParams {
  int mode;
  int rows;       // logical rows handled by this launch
  int row_base;   // first logical row (QKV: q_rows to skip q)
  int K;          // input width
  int items;      // active items in this launch (<= NB)
  int item0;      // global index of item 0
  int n_embd, n_head, n_head_kv, head_dim, rope_dims, n_ff, draft_vocab, target_vocab;
  float eps;
  // weights: bf16 rows, or (sz0 non-null) INT4 code rows of K / 2 bytes with the
  // (scale, zero) bf16 pairs of each 128-wide k group in sz rows of sz_stride pairs
  const uint16_t *w0, *w1, *w2;
  const uint32_t *sz0, *sz1, *sz2;
  int sz_stride;
  const uint16_t *norm0, *norm1;
  const uint16_t *embed;
  // plain inputs
  const uint16_t *xb;  // bf16 [items, K] (encode)
  const float *xf;     // f32 [items, K] (o: attention output, down: act, gateup: x1, lmhead: gsum)
  const float *res;    // residual [items, n] (o: g of the step, down: x1)
  PairSource pairs;
  // outputs
  float *out_f;        // encode: g; qkv: q; o: x1; gateup: act; down: gsum
  float *dbg_f;        // down: g_dbg [B, gamma, n] ; lmhead: logits_dbg [B, gamma, V_d]
  int dbg_stride_b;    // elements between batch rows of dbg (gamma * n or gamma * V_d)
  int dbg_off;         // element offset of this step in a batch row (j * n or j * V_d)
  // KV
  uint16_t *k_pool, *v_pool;  // bf16 rows, or the quantized pools' bytes (kv_quant)
  float *kv_stage;            // non-null: quantized KV -- the q/k/v epilogue leaves float32
                              // k (after RoPE) and v here, [item][K, V][n_head_kv * head_dim]
  const int32_t *page_table;
  int num_pages, max_pages, page_size, max_cache_len;
  const float2 *rope;  // [max_cache_len][rope_dims / 2] (cos, sin)
  // argmax
  unsigned long long *am_slot;  // [max_batch]
  unsigned int *am_count;       // arrival counter of the launch's CTAs
  const int64_t *d2t;
  int32_t *draft_tok;   // [B, gamma]
  int32_t *draft_id;    // [B, gamma] or null
  int32_t *next_tok;    // [B] token of the next step
  const int32_t *gamma_eff;
  int gamma, step;
  int *status;
  int nstage;           // stages in the weight ring (set by the launcher)
  // lm_head of a chain whose next q/k/v decodes the argmax: the CTAs only fold their
  // maxima into am_slot (no arrival count, no last-CTA decode)
  int am_defer;
};

// ----------------------------------------------------------------- attention
struct AttnParams {
  const float *q;          // [B, H * d]
  float *out;              // [B, H * d]
  const unsigned char *k_pool, *v_pool;  // rows of k_row / v_row bytes (bf16 or q8_0 / q5_1)
  const int32_t *page_table;
  const int32_t *kv_len;   // [B]
  const int32_t *gamma_eff;
  int step;
  int num_pages, max_pages, page_size, max_cache_len;
  int n_head, n_head_kv, head_dim;
  int batch;               // sequences B
  int kv_q;                // 0: bf16 rows; 1: q8_0 K / q5_1 V rows
  int tc;                  // bf16 rows: 1 = the tensor-core kernel (attention_tc.cu)
  int unit_keys;           // keys per work unit (divides the page size)
  const int32_t *unit_pre; // [B + 1] unit prefix of this step (round plan)
  float *part_o;           // [2 * CTAs, G, d] shared pairs' weighted V sums
  float2 *part_ml;         // [2 * CTAs, G] their (max, sum)
  unsigned int *count;     // [B, H_kv]
  int *status;
};

}  // namespace e3
