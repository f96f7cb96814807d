// C ABI of the EAGLE-3 drafter draft round: argument validation, workspace layout,
// the round state machine and kernel orchestration (direct launches or a CUDA graph of
// the gamma-step chain).  See include/eagle3.h for the contract of every entry point.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "common.cuh"
#include "internal.h"

using namespace e3;

namespace {

constexpr int kPrefillChunk = 512;   // prompt positions encoded per prefill chunk
constexpr int kSplitSlots = 4096;    // attention partial slots (two per CTA) and pair counters
constexpr int kMaxGraphs = 16;

struct Layout {
  size_t rope, q, attn_o, part_o, part_ml, attn_cnt, x1, act, gwork, tokwork, am_slot, am_cnt, am_steps,
      round_start, geff, status, genc, xp0, xp1, xp2, sumsq, gsum, tc_part, tc_cnt, attn_plan, kv_stage, gres,
      total;
  size_t tc_items, tc_k, tc_part_elems;
};

constexpr int kTcMinItems = 3;       // batched projections use the tensor-core GEMM from here
constexpr size_t kTcCounters = 32768;  // (row tile, item tile) arrival counters: the
                                       // target head of verify has ~2000 row tiles
constexpr int kTcEncodeChunk = 2048;  // encode rows per tensor-core launch
constexpr int kTcPrepMaxK = 16384;    // widest float32 input the activation split handles

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool cfg_valid(const eagle3_config *c) {
  if (!c) return false;
  if (c->n_embd <= 0 || c->n_embd % 8) return false;
  if (c->n_head <= 0 || c->n_head_kv <= 0 || c->n_head % c->n_head_kv) return false;
  if (!attn_supported(c->head_dim, c->n_head / c->n_head_kv)) return false;
  if (c->rope_dims < 0 || c->rope_dims % 2 || c->rope_dims > c->head_dim) return false;
  if (!(c->rope_theta > 0.f) || !(c->rms_eps >= 0.f)) return false;
  if (c->n_ff <= 0 || c->n_ff % 8) return false;
  if (c->draft_vocab % 2 || (c->head_dim * c->n_head_kv) % 2) return false;  // GEMV row pairs
  if (c->draft_vocab <= 0 || c->target_vocab <= 0) return false;
  if (c->max_batch <= 0 || c->max_gamma <= 0 || c->max_gamma > 64) return false;
  if (c->max_cache_len <= 1 || c->page_size <= 0) return false;
  // one GEMV launch must hold one item's activations in shared memory
  const size_t kmax = (size_t)std::max(std::max(3 * c->n_embd, 2 * c->n_embd),
                                       std::max(c->n_ff, c->n_head * c->head_dim));
  if (kmax * 4 > kGemvMaxXBytes) return false;
  if ((size_t)c->max_batch * c->n_head_kv > (size_t)kSplitSlots) return false;
  if (c->kv_format != EAGLE3_KV_BF16 && c->kv_format != EAGLE3_KV_Q8_0_Q5_1) return false;
  if (c->flags & ~EAGLE3_CKPT_NORM_BEFORE_RESIDUAL) return false;
  if (c->weight_format != EAGLE3_W_BF16 && c->weight_format != EAGLE3_W_INT4_G128) return false;
  if (c->weight_format == EAGLE3_W_INT4_G128 &&
      (c->n_embd % 128 || (c->n_head * c->head_dim) % 128 || c->n_ff % 128))
    return false;
  if (c->kv_format == EAGLE3_KV_Q8_0_Q5_1 && c->head_dim % 32) return false;
  if (attn_unit_keys(c->head_dim, c->n_head / c->n_head_kv, c->page_size, c->kv_format) < 1) return false;
  return true;
}

// Bytes of one K / V row of the paged pools (one position of one kv head).
void kv_rows(const eagle3_config &c, size_t *k_row, size_t *v_row) {
  if (c.kv_format == EAGLE3_KV_Q8_0_Q5_1) {
    *k_row = (size_t)c.head_dim / 32 * 34;
    *v_row = (size_t)c.head_dim / 32 * 24;
  } else {
    *k_row = *v_row = (size_t)c.head_dim * 2;
  }
}

Layout make_layout(const eagle3_config &c) {
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = align_up(off, 256);
    off = o + std::max<size_t>(bytes, 1);
    return o;
  };
  const size_t B = c.max_batch, n = c.n_embd, hd = (size_t)c.n_head * c.head_dim;
  const size_t G = c.n_head / c.n_head_kv;
  L.rope = take((size_t)c.max_cache_len * (c.rope_dims / 2) * sizeof(float2));
  L.q = take(B * hd * 4);
  L.attn_o = take(B * hd * 4);
  L.part_o = take((size_t)kSplitSlots * G * c.head_dim * 4);
  L.part_ml = take((size_t)kSplitSlots * G * sizeof(float2));
  L.attn_cnt = take(B * c.n_head_kv * 4);
  L.x1 = take(B * n * 4);
  L.act = take(B * (size_t)c.n_ff * 4);
  L.gwork = take(B * n * 4);
  L.tokwork = take(B * 4);
  L.am_slot = take(B * (c.max_gamma + 1) * 8);  // one per chain item or verify row
  L.am_cnt = take(64 * 4);
  L.am_steps = take(B * c.max_gamma * 8);  // per chain step and item (GEMV chains)
  L.round_start = take(B * 4);
  L.geff = take(B * 4);
  L.status = take(4);
  L.genc = take(std::max<size_t>(B * (c.max_gamma + 1), kPrefillChunk) * n * 4);
  // tensor-core path: the three bf16 parts of x, norm sums, split-K partials and counters
  L.tc_items = std::max<size_t>(B * (c.max_gamma + 1), kPrefillChunk);
  L.tc_k = std::max(std::max<size_t>(2 * n, (size_t)c.n_ff), hd);
  L.xp0 = take(L.tc_items * L.tc_k * 2);
  L.xp1 = take(L.tc_items * L.tc_k * 2);
  L.xp2 = take(L.tc_items * L.tc_k * 2);
  L.sumsq = take(L.tc_items * 2 * 4);
  // INT4 weights: each item's sum of x over every 128-wide group of a projection's input
  L.gsum = take(c.weight_format == EAGLE3_W_INT4_G128 ? L.tc_items * (L.tc_k / 128) * 4 : 0);
  L.tc_part_elems = (size_t)2 * 160 * 128 * 256;
  L.tc_part = take(L.tc_part_elems * 4);
  L.tc_cnt = take(kTcCounters * 4);
  L.attn_plan = take((size_t)c.max_gamma * (B + 1) * 4);  // attention unit prefix per step
  // quantized KV: the projection's float32 k / v before kv_quant writes the blocks
  L.kv_stage = take(c.kv_format == EAGLE3_KV_Q8_0_Q5_1 ? L.tc_items * 2 * c.n_head_kv * c.head_dim * 4 : 0);
  L.gres = take(c.flags & EAGLE3_CKPT_NORM_BEFORE_RESIDUAL ? B * n * 4 : 0);  // normed residual
  L.total = align_up(off, 256);
  return L;
}

struct GraphKey {
  int B, gamma, splits;
  unsigned flags;
  const void *ptrs[12];
  int ints[3];
  bool operator==(const GraphKey &o) const {
    if (B != o.B || gamma != o.gamma || splits != o.splits || flags != o.flags) return false;
    for (int i = 0; i < 12; ++i)
      if (ptrs[i] != o.ptrs[i]) return false;
    for (int i = 0; i < 3; ++i)
      if (ints[i] != o.ints[i]) return false;
    return true;
  }
};

struct GraphEntry {
  GraphKey key;
  cudaGraphExec_t exec;
  unsigned long long last_use;
  unsigned long long kernels;
};

}  // namespace

struct eagle3_ctx {
  eagle3_config c;
  eagle3_weights w;
  char *ws;
  size_t ws_bytes;
  Layout L;
  float2 *rope;
  float *q, *attn_o, *part_o, *x1, *act, *gwork, *genc;
  float2 *part_ml;
  unsigned *attn_cnt, *am_cnt;
  unsigned long long *am_slot, *am_steps;
  int32_t *tokwork, *round_start, *geff;
  int *status;
  int num_sms;
  int graph_mode;
  int round_open;
  int open_B;
  int rebuild_ok;
  cudaStream_t last_stream;
  cudaStream_t cap_stream;
  std::vector<GraphEntry> graphs;
  unsigned long long use_clock;
  // measurement: kernels launched (graph replays count their kernels) and optional
  // events recorded after each kernel of a direct-mode chain
  unsigned long long launches;
  cudaEvent_t *ev;
  int ev_cap, ev_used;
  std::vector<int> ev_label;
  std::vector<cudaEvent_t> ev_pool;
  // tensor-core path
  int tc_ok, tc_min_items, tc_sched;
  int attn_mode;  // ATTN_*: which decode attention kernel runs (bf16 KV)
  // attention work units (keys per unit) and the round's unit prefix tables
  int unit_keys;
  int32_t *attn_plan;
  // KV storage format: bf16, or q8_0 K / q5_1 V written by kv_quant from kv_stage
  int kv_q, k_row, v_row;
  float *kv_stage;
  float *gres;  // norm_before_residual: RMSNorm(g) * hidden_norm of the step, [B, n]
  int q4;       // INT4 projection weights (EAGLE3_W_INT4_G128)
  uint16_t *xp0, *xp1, *xp2;  // the three bf16 parts of x
  float *gsum;                // INT4: sums of x per 128-wide group (tensor-core path)
  float *sumsq, *tc_part;
  unsigned *tc_cnt;
};

namespace {

int cuda_err(cudaError_t e) { return e == cudaSuccess ? EAGLE3_OK : EAGLE3_ERR_CUDA; }

bool kv_valid(const eagle3_ctx *ctx, const eagle3_kv *kv) {
  if (!kv || !aligned16(kv->k_pool) || !aligned16(kv->v_pool) || !kv->page_table || !kv->kv_len)
    return false;
  if (kv->num_pages <= 0 || kv->max_pages_per_seq <= 0) return false;
  if ((long long)kv->max_pages_per_seq * ctx->c.page_size < ctx->c.max_cache_len) return false;
  return true;
}

GemvParams base_params(const eagle3_ctx *ctx) {
  GemvParams p;
  std::memset(&p, 0, sizeof(p));
  const eagle3_config &c = ctx->c;
  p.n_embd = c.n_embd;
  p.n_head = c.n_head;
  p.n_head_kv = c.n_head_kv;
  p.head_dim = c.head_dim;
  p.rope_dims = c.rope_dims;
  p.n_ff = c.n_ff;
  p.draft_vocab = c.draft_vocab;
  p.target_vocab = c.target_vocab;
  p.eps = c.rms_eps;
  p.embed = ctx->w.embed;
  p.rope = ctx->rope;
  p.max_cache_len = c.max_cache_len;
  p.page_size = c.page_size;
  p.status = ctx->status;
  return p;
}

void set_kv(GemvParams &p, const eagle3_kv *kv) {
  p.k_pool = static_cast<uint16_t *>(kv->k_pool);
  p.v_pool = static_cast<uint16_t *>(kv->v_pool);
  p.page_table = kv->page_table;
  p.num_pages = kv->num_pages;
  p.max_pages = kv->max_pages_per_seq;
}

// Phase labels of the measurement events (eagle3_phase_event_label).
enum PhaseLabel : int {
  PH_START = 0, PH_QKV = 1, PH_ATTN = 2, PH_O = 3, PH_GATEUP = 4, PH_DOWN = 5, PH_LMHEAD = 6,
  PH_ENCODE = 7, PH_KV = 8, PH_SMALL = 9,
};

int gemv_label(int mode) {
  switch (mode) {
    case GM_ENCODE: return PH_ENCODE;
    case GM_QKV: return PH_QKV;
    case GM_O: return PH_O;
    case GM_GATEUP: return PH_GATEUP;
    case GM_DOWN: return PH_DOWN;
    default: return PH_LMHEAD;
  }
}

void record_event(eagle3_ctx *ctx, cudaStream_t st, int label) {
  if (ctx->ev && ctx->ev_used < ctx->ev_cap) {
    cudaEventRecord(ctx->ev[ctx->ev_used], st);
    ctx->ev_label[ctx->ev_used++] = label;
  }
}

// Book-keeping after every kernel launch.
cudaError_t launched(eagle3_ctx *ctx, cudaStream_t st, cudaError_t e, int label) {
  if (e == cudaSuccess) {
    ++ctx->launches;
    record_event(ctx, st, label);
  }
  return e;
}

// Tensor-core GEMM of one projection over `items` activation rows: x split into three bf16
// parts (not for the encode, whose features are bf16 already), then the tcgen05 kernel.
cudaError_t tc_items(eagle3_ctx *ctx, const GemvParams &p, int items, cudaStream_t st, bool pdl) {
  const eagle3_config &c = ctx->c;
  TcLaunch L;
  std::memset(&L, 0, sizeof(L));
  L.p = p;
  L.p.item0 = 0;
  L.p.items = items;
  L.M = items;
  L.sumsq = ctx->sumsq;
  L.part = ctx->tc_part;
  L.part_elems = ctx->L.tc_part_elems;
  L.tile_cnt = ctx->tc_cnt;
  L.tile_cnt_elems = kTcCounters;
  L.num_sms = ctx->num_sms;
  L.schedule = ctx->tc_sched;
  if (p.sz0) {  // INT4 weights: a* are code rows
    L.s0 = p.sz0;
    L.s1 = p.sz1;
    L.s2 = p.sz2;
    L.sz_stride = p.sz_stride;
    L.gsum = ctx->gsum;
  }
  const int n = c.n_embd, qr = c.n_head * c.head_dim, kr = c.n_head_kv * c.head_dim;
  switch (p.mode) {
    case GM_ENCODE: L.a0 = ctx->w.fc; L.a0_rows = n; break;
    case GM_QKV:
      L.a0 = ctx->w.q; L.a0_rows = qr;
      L.a1 = ctx->w.k; L.a1_rows = kr;
      L.a2 = ctx->w.v; L.a2_rows = kr;
      break;
    case GM_O: L.a0 = ctx->w.o; L.a0_rows = n; break;
    case GM_GATEUP:
      L.a0 = ctx->w.gate; L.a0_rows = c.n_ff;
      L.a1 = ctx->w.up; L.a1_rows = c.n_ff;
      break;
    case GM_DOWN: L.a0 = ctx->w.down; L.a0_rows = n; break;
    default: L.a0 = p.w0; L.a0_rows = p.rows; break;  // the draft lm_head, or verify's target head
  }
  const int label = (p.mode == GM_QKV && p.row_base > 0) ? PH_KV : gemv_label(p.mode);
  if (p.mode == GM_ENCODE) {
    // bf16 features straight from the caller's rows, in chunks of kTcEncodeChunk items
    for (int i0 = 0; i0 < items; i0 += kTcEncodeChunk) {
      L.M = std::min(kTcEncodeChunk, items - i0);
      L.p.items = L.M;
      L.p.out_f = p.out_f + (size_t)i0 * p.rows;
      L.b0 = p.xb + (size_t)i0 * p.K;
      cudaError_t e = launched(ctx, st, tc_launch(L, st, pdl), label);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  } else {
    cudaError_t e = launched(
        ctx, st, tc_prep_launch(p, items, ctx->xp0, ctx->xp1, ctx->xp2, ctx->sumsq, p.sz0 ? ctx->gsum : nullptr, st, pdl),
        PH_SMALL);
    if (e != cudaSuccess) return e;
    L.b0 = ctx->xp0;
    L.b1 = ctx->xp1;
    L.b2 = ctx->xp2;
  }
  return launched(ctx, st, tc_launch(L, st, pdl), label);
}

bool use_tc(const eagle3_ctx *ctx, const GemvParams &p, int items) {
  if (!ctx->tc_ok || items < ctx->tc_min_items) return false;
  if (p.sz0 && (!ctx->gsum || p.K % 128)) return false;  // INT4: the group sums' buffer and whole groups
  // k/v-only teacher forcing of a few pairs (rebuild) with bf16 weights: the 4-8-item
  // GEMV measured faster (INT4 takes the tensor cores: its several-item GEMV is slower)
  if (p.mode == GM_QKV && p.row_base > 0 && items <= 8 && !p.sz0) return false;
  if (p.mode != GM_ENCODE && (size_t)items > ctx->L.tc_items) return false;
  if (p.mode != GM_ENCODE && p.K > kTcPrepMaxK) return false;  // the activation split's limit
  return true;
}

// A q/k/v (or k/v-only) projection over `items` pairs; with quantized KV the epilogue
// stages float32 k / v and kv_quant writes the q8_0 / q5_1 blocks.
cudaError_t gemv_items(eagle3_ctx *ctx, GemvParams p, int items, cudaStream_t st, bool pdl);
cudaError_t qkv_items(eagle3_ctx *ctx, GemvParams p, int items, cudaStream_t st, bool pdl) {
  p.kv_stage = ctx->kv_stage;
  cudaError_t e = gemv_items(ctx, p, items, st, pdl);
  if (e == cudaSuccess && ctx->kv_q)
    e = launched(ctx, st, kv_quant_launch(p, items, ctx->k_row, ctx->v_row, st, true), PH_SMALL);
  return e;
}

// Launch a GEMV over `items` activation rows in as many launches as shared memory needs.
cudaError_t gemv_items(eagle3_ctx *ctx, GemvParams p, int items, cudaStream_t st, bool pdl) {
  if (use_tc(ctx, p, items)) return tc_items(ctx, p, items, st, pdl);
  const int nb = gemv_items_per_launch(p, items, ctx->num_sms);
  const int label = (p.mode == GM_QKV && p.row_base > 0) ? PH_KV : gemv_label(p.mode);
  for (int i0 = 0; i0 < items; i0 += nb) {
    p.item0 = i0;
    p.items = std::min(nb, items - i0);
    cudaError_t e = launched(ctx, st, gemv_launch(p, ctx->num_sms, st, pdl), label);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t enqueue_encode(eagle3_ctx *ctx, const uint16_t *aux, int M, float *g, cudaStream_t st,
                           bool pdl) {
  if (M <= 0) return cudaSuccess;
  GemvParams p = base_params(ctx);
  p.mode = GM_ENCODE;
  p.rows = ctx->c.n_embd;
  p.K = 3 * ctx->c.n_embd;
  p.w0 = ctx->w.fc;
  p.xb = aux;
  p.out_f = g;
  return gemv_items(ctx, p, M, st, pdl);
}

// (scale, zero) pairs per INT4 weight row: one per 128 inputs, rounded up to 4 (16 bytes).
int q4_sz_stride(int K) { return (K / 128 + 3) / 4 * 4; }

// Weight operands of a projection (p.K set): bf16 rows, or INT4 codes with their
// (scale, zero) rows.
void set_weights(const eagle3_ctx *ctx, GemvParams &p, const uint16_t *w0, const uint32_t *s0,
                 const uint16_t *w1 = nullptr, const uint32_t *s1 = nullptr, const uint16_t *w2 = nullptr,
                 const uint32_t *s2 = nullptr) {
  p.w0 = w0;
  p.w1 = w1;
  p.w2 = w2;
  if (ctx->q4) {
    p.sz0 = s0;
    p.sz1 = s1;
    p.sz2 = s2;
    p.sz_stride = q4_sz_stride(p.K);
  }
}

void kv_only_params(const eagle3_ctx *ctx, const eagle3_kv *kv, GemvParams &p) {
  const eagle3_config &c = ctx->c;
  set_kv(p, kv);
  p.mode = GM_QKV;
  p.row_base = c.n_head * c.head_dim;
  p.rows = 2 * c.n_head_kv * c.head_dim;
  p.K = 2 * c.n_embd;
  set_weights(ctx, p, ctx->w.q, ctx->w.q_sz, ctx->w.k, ctx->w.k_sz, ctx->w.v, ctx->w.v_sz);
  p.norm0 = ctx->w.in_norm;
  p.norm1 = ctx->w.hidden_norm;
}

struct ChainArgs {
  int B, gamma, splits;
  unsigned flags;
  const eagle3_kv *kv;
  const eagle3_boundary *bnd;
  int32_t *draft_tok, *draft_id, *gamma_eff;
  float *logits_dbg, *g_dbg;
};

// Whether a chain of B sequences runs its q/k/v and its lm_head on the GEMV (then the
// lm_head's argmax is decoded by the kernel after it).
bool chain_defers_argmax(const eagle3_ctx *ctx, int B) {
  const eagle3_config &c = ctx->c;
  GemvParams q = base_params(ctx);
  q.mode = GM_QKV;
  q.K = 2 * c.n_embd;
  q.sz0 = ctx->q4 ? ctx->w.q_sz : nullptr;
  GemvParams l = base_params(ctx);
  l.mode = GM_LMHEAD;
  l.K = c.n_embd;
  l.sz0 = ctx->q4 ? ctx->w.lm_head_sz : nullptr;
  return !use_tc(ctx, q, B) && !use_tc(ctx, l, B);
}

cudaError_t enqueue_chain(eagle3_ctx *ctx, const ChainArgs &a, cudaStream_t st) {
  const eagle3_config &c = ctx->c;
  const int n = c.n_embd, qr = c.n_head * c.head_dim, kr = c.n_head_kv * c.head_dim;
  const bool pdl = true;
  record_event(ctx, st, PH_START);
  // Chains whose q/k/v and lm_head both run on the GEMV leave each step's argmax in a slot
  // of the step: the lm_head CTAs fold their maxima in and leave, the next step's q/k/v
  // decodes the token (and writes the step's outputs), the chain end the last step's.
  const bool defer = chain_defers_argmax(ctx, a.B);
  const int ss = c.max_batch;  // slot row stride
  cudaError_t e = launched(ctx, st,
                           launch_chain_begin(a.B, a.gamma, a.flags, c.max_cache_len, a.kv->kv_len,
                                              ctx->round_start, ctx->geff, a.gamma_eff,
                                              ctx->status, ctx->unit_keys, ctx->attn_plan,
                                              defer ? ctx->am_steps : nullptr, a.gamma * ss, st),
                           PH_SMALL);
  if (e != cudaSuccess) return e;
  for (int j = 0; j < a.gamma; ++j) {
    // q/k/v + RoPE + KV append
    GemvParams p = base_params(ctx);
    set_kv(p, a.kv);
    p.mode = GM_QKV;
    p.rows = qr + 2 * kr;
    p.row_base = 0;
    p.K = 2 * n;
    set_weights(ctx, p, ctx->w.q, ctx->w.q_sz, ctx->w.k, ctx->w.k_sz, ctx->w.v, ctx->w.v_sz);
    p.norm0 = ctx->w.in_norm;
    p.norm1 = ctx->w.hidden_norm;
    p.pairs.kind = PAIR_CHAIN;
    p.pairs.step = j;
    p.pairs.gamma = a.gamma;
    p.pairs.bnd_tok = a.bnd->tok;
    p.pairs.bnd_g = a.bnd->g;
    p.pairs.step_tok = ctx->tokwork;
    p.pairs.step_g = ctx->gwork;
    p.pairs.kv_len = a.kv->kv_len;
    p.pairs.gamma_eff = ctx->geff;
    if (defer && j > 0) {
      p.pairs.step_key = ctx->am_steps + (size_t)(j - 1) * ss;
      p.pairs.d2t = ctx->w.d2t;
      p.pairs.draft_vocab = c.draft_vocab;
      p.pairs.target_vocab = c.target_vocab;
      // the previous step's outputs (written by CTA 0)
      p.d2t = ctx->w.d2t;
      p.draft_tok = a.draft_tok;
      p.draft_id = a.draft_id;
      p.next_tok = ctx->tokwork;
      p.gamma_eff = ctx->geff;
      p.gamma = a.gamma;
    }
    p.out_f = ctx->q;
    if ((e = qkv_items(ctx, p, a.B, st, pdl)) != cudaSuccess) return e;

    // attention
    AttnParams ap;
    std::memset(&ap, 0, sizeof(ap));
    ap.q = ctx->q;
    ap.out = ctx->attn_o;
    ap.k_pool = static_cast<const unsigned char *>(a.kv->k_pool);
    ap.v_pool = static_cast<const unsigned char *>(a.kv->v_pool);
    ap.kv_q = ctx->kv_q;
    ap.tc = ctx->attn_mode == ATTN_TENSOR_CORES;
    ap.page_table = a.kv->page_table;
    ap.kv_len = a.kv->kv_len;
    ap.gamma_eff = ctx->geff;
    ap.step = j;
    ap.num_pages = a.kv->num_pages;
    ap.max_pages = a.kv->max_pages_per_seq;
    ap.page_size = c.page_size;
    ap.max_cache_len = c.max_cache_len;
    ap.n_head = c.n_head;
    ap.n_head_kv = c.n_head_kv;
    ap.head_dim = c.head_dim;
    ap.batch = a.B;
    ap.unit_keys = ctx->unit_keys;
    ap.unit_pre = ctx->attn_plan + (size_t)j * (a.B + 1);
    ap.part_o = ctx->part_o;
    ap.part_ml = ctx->part_ml;
    ap.count = ctx->attn_cnt;
    ap.status = ctx->status;
    if ((e = launched(ctx, st, attn_launch(ap, ctx->num_sms, st, pdl), PH_ATTN)) != cudaSuccess) return e;

    // o_proj + residual: the pre-norm g of this step, or RMSNorm(g) * hidden_norm for
    // checkpoints with norm_before_residual
    const float *g_step = j == 0 ? a.bnd->g : ctx->gwork;
    if (ctx->gres) {
      if ((e = launched(ctx, st, launch_res_norm(a.B, n, c.rms_eps, g_step, ctx->w.hidden_norm, ctx->gres, st),
                        PH_SMALL)) != cudaSuccess)
        return e;
      g_step = ctx->gres;
    }
    p = base_params(ctx);
    p.mode = GM_O;
    p.rows = n;
    p.K = qr;
    set_weights(ctx, p, ctx->w.o, ctx->w.o_sz);
    p.xf = ctx->attn_o;
    p.res = g_step;
    p.out_f = ctx->x1;
    if ((e = gemv_items(ctx, p, a.B, st, pdl)) != cudaSuccess) return e;

    // post-attention RMSNorm + gate/up + SiLU * up
    p = base_params(ctx);
    p.mode = GM_GATEUP;
    p.rows = 2 * c.n_ff;
    p.K = n;
    set_weights(ctx, p, ctx->w.gate, ctx->w.gate_sz, ctx->w.up, ctx->w.up_sz);
    p.xf = ctx->x1;
    p.norm0 = ctx->w.post_norm;
    p.out_f = ctx->act;
    if ((e = gemv_items(ctx, p, a.B, st, pdl)) != cudaSuccess) return e;

    // down + fused-add residual -> gsum, the next g
    p = base_params(ctx);
    p.mode = GM_DOWN;
    p.rows = n;
    p.K = c.n_ff;
    set_weights(ctx, p, ctx->w.down, ctx->w.down_sz);
    p.xf = ctx->act;
    p.res = ctx->x1;
    p.out_f = ctx->gwork;
    p.dbg_f = a.g_dbg;
    p.dbg_stride_b = a.gamma * n;
    p.dbg_off = j * n;
    if ((e = gemv_items(ctx, p, a.B, st, pdl)) != cudaSuccess) return e;

    // final RMSNorm + lm_head + argmax + d2t
    p = base_params(ctx);
    p.mode = GM_LMHEAD;
    p.rows = c.draft_vocab;
    p.K = n;
    set_weights(ctx, p, ctx->w.lm_head, ctx->w.lm_head_sz);
    p.xf = ctx->gwork;
    p.norm0 = ctx->w.final_norm;
    p.am_slot = defer ? ctx->am_steps + (size_t)j * ss : ctx->am_slot;
    p.am_count = ctx->am_cnt;
    p.am_defer = defer ? 1 : 0;
    p.d2t = ctx->w.d2t;
    p.draft_tok = a.draft_tok;
    p.draft_id = a.draft_id;
    p.next_tok = ctx->tokwork;
    p.gamma_eff = ctx->geff;
    p.gamma = a.gamma;
    p.step = j;
    p.dbg_f = a.logits_dbg;
    p.dbg_stride_b = a.gamma * c.draft_vocab;
    p.dbg_off = j * c.draft_vocab;
    if ((e = gemv_items(ctx, p, a.B, st, pdl)) != cudaSuccess) return e;
  }
  ChainLast last;
  std::memset(&last, 0, sizeof(last));
  if (defer) {
    last.slot = ctx->am_steps + (size_t)(a.gamma - 1) * ss;
    last.gamma = a.gamma;
    last.draft_vocab = c.draft_vocab;
    last.target_vocab = c.target_vocab;
    last.d2t = ctx->w.d2t;
    last.draft_tok = a.draft_tok;
    last.draft_id = a.draft_id;
    last.status = ctx->status;
  }
  return launched(ctx, st, launch_chain_end(a.B, a.kv->kv_len, ctx->round_start, ctx->geff, last, st, pdl),
                  PH_SMALL);
}

GraphKey chain_key(const ChainArgs &a) {
  GraphKey k;
  std::memset(&k, 0, sizeof(k));
  k.B = a.B;
  k.gamma = a.gamma;
  k.splits = a.splits;
  k.flags = a.flags;
  const void *p[12] = {a.kv->k_pool, a.kv->v_pool, a.kv->page_table, a.kv->kv_len, a.bnd->g,
                       a.bnd->tok, a.draft_tok, a.draft_id, a.gamma_eff, a.logits_dbg, a.g_dbg,
                       nullptr};
  for (int i = 0; i < 12; ++i) k.ptrs[i] = p[i];
  k.ints[0] = a.kv->num_pages;
  k.ints[1] = a.kv->max_pages_per_seq;
  return k;
}

// Forget every captured chain (after the work already enqueued on the last stream).
void drop_graphs(eagle3_ctx *ctx) {
  if (ctx->graphs.empty()) return;
  cudaStreamSynchronize(ctx->last_stream);
  for (auto &g : ctx->graphs) cudaGraphExecDestroy(g.exec);
  ctx->graphs.clear();
}

cudaError_t run_chain_graph(eagle3_ctx *ctx, const ChainArgs &a, cudaStream_t st) {
  const GraphKey key = chain_key(a);
  for (auto &g : ctx->graphs) {
    if (g.key == key) {
      g.last_use = ++ctx->use_clock;
      const cudaError_t e = cudaGraphLaunch(g.exec, st);
      if (e == cudaSuccess) ctx->launches += g.kernels;
      return e;
    }
  }
  if (!ctx->cap_stream) {
    cudaError_t e = cudaStreamCreateWithFlags(&ctx->cap_stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaStreamBeginCapture(ctx->cap_stream, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) return e;
  const unsigned long long before = ctx->launches;
  cudaEvent_t *ev_saved = ctx->ev;
  ctx->ev = nullptr;  // no measurement events inside a graph
  const cudaError_t e_enq = enqueue_chain(ctx, a, ctx->cap_stream);
  ctx->ev = ev_saved;
  const unsigned long long kernels = ctx->launches - before;
  ctx->launches = before;
  cudaGraph_t graph = nullptr;
  e = cudaStreamEndCapture(ctx->cap_stream, &graph);
  if (e_enq != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    return e_enq;
  }
  if (e != cudaSuccess) return e;
  cudaGraphExec_t exec = nullptr;
  e = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) return e;
  if ((int)ctx->graphs.size() >= kMaxGraphs) {
    auto old = std::min_element(ctx->graphs.begin(), ctx->graphs.end(),
                                [](const GraphEntry &x, const GraphEntry &y) { return x.last_use < y.last_use; });
    cudaGraphExecDestroy(old->exec);
    ctx->graphs.erase(old);
  }
  ctx->graphs.push_back(GraphEntry{key, exec, ++ctx->use_clock, kernels});
  e = cudaGraphLaunch(exec, st);
  if (e == cudaSuccess) ctx->launches += kernels;
  return e;
}

}  // namespace

// =========================================================================== C ABI

extern "C" {

int eagle3_version(void) { return (1 << 16) | 0; }

const char *eagle3_error_string(int code) {
  switch (code) {
    case EAGLE3_OK: return "ok";
    case EAGLE3_ERR_INVALID_ARG: return "invalid argument";
    case EAGLE3_ERR_CAPACITY: return "kv_len + gamma + 1 exceeds max_cache_len";
    case EAGLE3_ERR_STATE: return "call out of order for the round state";
    case EAGLE3_ERR_CUDA: return "CUDA error";
    case EAGLE3_ERR_DEVICE: return "device status word set";
    case EAGLE3_ERR_UNSUPPORTED: return "unsupported geometry";
    default: return "unknown error";
  }
}

int eagle3_selftest_bounded_wait(int *device_status, int *device_result, eagle3_stream_t stream) {
  if (!device_status || !device_result) return EAGLE3_ERR_INVALID_ARG;
  return cuda_err(launch_wait_selftest(device_status, device_result, reinterpret_cast<cudaStream_t>(stream)));
}

int eagle3_kv_row_bytes(const eagle3_config *cfg, size_t *k_row, size_t *v_row) {
  if (!cfg_valid(cfg) || !k_row || !v_row) return EAGLE3_ERR_INVALID_ARG;
  kv_rows(*cfg, k_row, v_row);
  return EAGLE3_OK;
}

size_t eagle3_workspace_bytes(const eagle3_config *cfg) {
  if (!cfg_valid(cfg)) return 0;
  return make_layout(*cfg).total;
}

int eagle3_plan_gamma(int kv_len, int gamma, int max_cache_len, unsigned flags, int *gamma_eff) {
  if (!gamma_eff || gamma < 1 || kv_len < 0 || max_cache_len < 1) return EAGLE3_ERR_INVALID_ARG;
  if ((long long)kv_len + gamma + 1 <= max_cache_len) {
    *gamma_eff = gamma;
    return EAGLE3_OK;
  }
  if (!(flags & EAGLE3_SHRINK_GAMMA)) return EAGLE3_ERR_CAPACITY;
  const long long g = (long long)max_cache_len - kv_len - 1;
  if (g < 1) return EAGLE3_ERR_CAPACITY;
  *gamma_eff = (int)g;
  return EAGLE3_OK;
}

int eagle3_init(const eagle3_config *cfg, const eagle3_weights *w, void *workspace,
                size_t workspace_bytes, eagle3_stream_t stream, eagle3_ctx **out) {
  if (!out) return EAGLE3_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !w || !workspace) return EAGLE3_ERR_INVALID_ARG;
  if (!cfg_valid(cfg)) return EAGLE3_ERR_UNSUPPORTED;
  const void *wp[] = {w->fc, w->in_norm, w->hidden_norm, w->q, w->k, w->v, w->o, w->post_norm,
                      w->gate, w->up, w->down, w->final_norm, w->lm_head, w->embed, w->d2t};
  if (cfg->weight_format == EAGLE3_W_INT4_G128) {
    const void *sp[] = {w->q_sz, w->k_sz, w->v_sz, w->o_sz, w->gate_sz, w->up_sz, w->down_sz, w->lm_head_sz};
    for (const void *p : sp)
      if (!aligned16(p)) return EAGLE3_ERR_INVALID_ARG;
  }
  for (const void *p : wp)
    if (!aligned16(p)) return EAGLE3_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return EAGLE3_ERR_INVALID_ARG;
  const Layout L = make_layout(*cfg);
  if (workspace_bytes < L.total) return EAGLE3_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  // d2t: every draft id must map to a distinct target id in range.
  std::vector<int64_t> d2t(cfg->draft_vocab);
  if (cudaMemcpy(d2t.data(), w->d2t, d2t.size() * sizeof(int64_t), cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return EAGLE3_ERR_CUDA;
  {
    std::vector<int64_t> t(d2t.size());
    for (size_t i = 0; i < d2t.size(); ++i) {
      t[i] = (int64_t)i + d2t[i];
      if (t[i] < 0 || t[i] >= cfg->target_vocab) return EAGLE3_ERR_INVALID_ARG;
    }
    std::sort(t.begin(), t.end());
    for (size_t i = 1; i < t.size(); ++i)
      if (t[i] == t[i - 1]) return EAGLE3_ERR_INVALID_ARG;
  }

  eagle3_ctx *ctx = new (std::nothrow) eagle3_ctx();
  if (!ctx) return EAGLE3_ERR_INVALID_ARG;
  ctx->c = *cfg;
  ctx->w = *w;
  ctx->ws = static_cast<char *>(workspace);
  ctx->ws_bytes = workspace_bytes;
  ctx->L = L;
  char *b = ctx->ws;
  ctx->rope = reinterpret_cast<float2 *>(b + L.rope);
  ctx->q = reinterpret_cast<float *>(b + L.q);
  ctx->attn_o = reinterpret_cast<float *>(b + L.attn_o);
  ctx->part_o = reinterpret_cast<float *>(b + L.part_o);
  ctx->part_ml = reinterpret_cast<float2 *>(b + L.part_ml);
  ctx->attn_cnt = reinterpret_cast<unsigned *>(b + L.attn_cnt);
  ctx->x1 = reinterpret_cast<float *>(b + L.x1);
  ctx->act = reinterpret_cast<float *>(b + L.act);
  ctx->gwork = reinterpret_cast<float *>(b + L.gwork);
  ctx->tokwork = reinterpret_cast<int32_t *>(b + L.tokwork);
  ctx->am_slot = reinterpret_cast<unsigned long long *>(b + L.am_slot);
  ctx->am_cnt = reinterpret_cast<unsigned *>(b + L.am_cnt);
  ctx->am_steps = reinterpret_cast<unsigned long long *>(b + L.am_steps);
  ctx->round_start = reinterpret_cast<int32_t *>(b + L.round_start);
  ctx->geff = reinterpret_cast<int32_t *>(b + L.geff);
  ctx->status = reinterpret_cast<int *>(b + L.status);
  ctx->genc = reinterpret_cast<float *>(b + L.genc);
  ctx->attn_plan = reinterpret_cast<int32_t *>(b + L.attn_plan);
  ctx->unit_keys = attn_unit_keys(cfg->head_dim, cfg->n_head / cfg->n_head_kv, cfg->page_size, cfg->kv_format);
  ctx->kv_q = cfg->kv_format == EAGLE3_KV_Q8_0_Q5_1 ? 1 : 0;
  {
    size_t kr = 0, vr = 0;
    kv_rows(*cfg, &kr, &vr);
    ctx->k_row = (int)kr;
    ctx->v_row = (int)vr;
  }
  ctx->kv_stage = ctx->kv_q ? reinterpret_cast<float *>(b + L.kv_stage) : nullptr;
  ctx->q4 = cfg->weight_format == EAGLE3_W_INT4_G128 ? 1 : 0;
  ctx->gres = (cfg->flags & EAGLE3_CKPT_NORM_BEFORE_RESIDUAL) ? reinterpret_cast<float *>(b + L.gres) : nullptr;
  ctx->xp0 = reinterpret_cast<uint16_t *>(b + L.xp0);
  ctx->xp1 = reinterpret_cast<uint16_t *>(b + L.xp1);
  ctx->xp2 = reinterpret_cast<uint16_t *>(b + L.xp2);
  ctx->sumsq = reinterpret_cast<float *>(b + L.sumsq);
  ctx->gsum = ctx->q4 ? reinterpret_cast<float *>(b + L.gsum) : nullptr;
  ctx->tc_part = reinterpret_cast<float *>(b + L.tc_part);
  ctx->tc_cnt = reinterpret_cast<unsigned *>(b + L.tc_cnt);
  ctx->graph_mode = 1;
  ctx->last_stream = st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      gemv_prepare() != cudaSuccess || attn_prepare() != cudaSuccess) {
    delete ctx;
    return EAGLE3_ERR_CUDA;
  }

  // The tensor-core path needs 64-aligned K dims, 128-row q / k / v blocks that hold whole
  // heads (or whole heads that hold whole 128-row tiles) and a driver with tensor maps.
  {
    const int n = cfg->n_embd, d = cfg->head_dim;
    const int qr = cfg->n_head * d, kr = cfg->n_head_kv * d;
    const bool geo = n % 64 == 0 && cfg->n_ff % 64 == 0 && qr % 128 == 0 && kr % 128 == 0 &&
                     qr % 64 == 0 && (d % 128 == 0 || 128 % d == 0) && cfg->n_ff % 64 == 0;
    ctx->tc_ok = geo && tc_prepare() == cudaSuccess ? 1 : 0;
    ctx->tc_min_items = kTcMinItems;
    ctx->tc_sched = TC_SCHED_AUTO;
    ctx->attn_mode = ATTN_CUDA_CORES;
  }

  // RoPE table: angle p * theta^(-2i/R) in double, stored as float32 (cos, sin).
  const int half = cfg->rope_dims / 2;
  if (half > 0) {
    std::vector<float2> tab((size_t)cfg->max_cache_len * half);
    for (int i = 0; i < half; ++i) {
      const double inv = std::pow((double)cfg->rope_theta, -2.0 * i / cfg->rope_dims);
      for (int p = 0; p < cfg->max_cache_len; ++p) {
        const double a = (double)p * inv;
        tab[(size_t)p * half + i] = make_float2((float)std::cos(a), (float)std::sin(a));
      }
    }
    if (cudaMemcpy(ctx->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) !=
        cudaSuccess) {
      delete ctx;
      return EAGLE3_ERR_CUDA;
    }
  }
  // Counters and argmax slots start at zero and are returned to zero by their users.
  cudaError_t e = cudaMemsetAsync(b + L.attn_cnt, 0, (size_t)cfg->max_batch * cfg->n_head_kv * 4, st);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(b + L.am_slot, 0, (size_t)cfg->max_batch * (cfg->max_gamma + 1) * 8, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(b + L.am_cnt, 0, 64 * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(b + L.status, 0, 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(b + L.tc_cnt, 0, kTcCounters * 4, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    delete ctx;
    return EAGLE3_ERR_CUDA;
  }
  *out = ctx;
  return EAGLE3_OK;
}

int eagle3_destroy(eagle3_ctx *ctx) {
  if (!ctx) return EAGLE3_ERR_INVALID_ARG;
  for (auto &g : ctx->graphs) cudaGraphExecDestroy(g.exec);
  for (cudaEvent_t e : ctx->ev_pool) cudaEventDestroy(e);
  if (ctx->cap_stream) cudaStreamDestroy(ctx->cap_stream);
  delete ctx;
  return EAGLE3_OK;
}

int eagle3_set_graph_mode(eagle3_ctx *ctx, int enabled) {
  if (!ctx) return EAGLE3_ERR_INVALID_ARG;
  ctx->graph_mode = enabled ? 1 : 0;
  return EAGLE3_OK;
}

int eagle3_set_tc_min_items(eagle3_ctx *ctx, int min_items) {
  if (!ctx || min_items < 0) return EAGLE3_ERR_INVALID_ARG;
  const int v = min_items == 0 ? kTcMinItems : min_items;
  if (v != ctx->tc_min_items) {
    ctx->tc_min_items = v;
    drop_graphs(ctx);
  }
  return EAGLE3_OK;
}

int eagle3_set_tc_schedule(eagle3_ctx *ctx, int schedule) {
  if (!ctx || schedule < TC_SCHED_AUTO || schedule > TC_SCHED_CLUSTER) return EAGLE3_ERR_INVALID_ARG;
  if (schedule != ctx->tc_sched) {
    ctx->tc_sched = schedule;
    drop_graphs(ctx);
  }
  return EAGLE3_OK;
}

int eagle3_set_attention(eagle3_ctx *ctx, int mode) {
  if (!ctx || mode < ATTN_CUDA_CORES || mode > ATTN_TENSOR_CORES) return EAGLE3_ERR_INVALID_ARG;
  if (mode != ctx->attn_mode) {
    ctx->attn_mode = mode;
    drop_graphs(ctx);
  }
  return EAGLE3_OK;
}

int eagle3_encode(eagle3_ctx *ctx, const uint16_t *aux, int M, float *g, eagle3_stream_t stream) {
  if (!ctx || M < 0) return EAGLE3_ERR_INVALID_ARG;
  if (M == 0) return EAGLE3_OK;
  if (!aligned16(aux) || !aligned16(g)) return EAGLE3_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  ctx->last_stream = st;
  return cuda_err(enqueue_encode(ctx, aux, M, g, st, true));
}

int eagle3_prefill(eagle3_ctx *ctx, int B, const int32_t *tokens, int P_max,
                   const int32_t *next_tok, const int32_t *prompt_len_host, const uint16_t *aux,
                   const eagle3_kv *kv, eagle3_boundary *bnd, eagle3_stream_t stream) {
  if (!ctx || B < 1 || B > ctx->c.max_batch || P_max < 1) return EAGLE3_ERR_INVALID_ARG;
  if (!tokens || !next_tok || !prompt_len_host || !aligned16(aux)) return EAGLE3_ERR_INVALID_ARG;
  if (!kv_valid(ctx, kv) || !bnd || !aligned16(bnd->g) || !bnd->tok) return EAGLE3_ERR_INVALID_ARG;
  if (ctx->round_open) return EAGLE3_ERR_STATE;
  for (int b = 0; b < B; ++b) {
    const int P = prompt_len_host[b];
    if (P < 1 || P > P_max) return EAGLE3_ERR_INVALID_ARG;
    if (P > ctx->c.max_cache_len) return EAGLE3_ERR_CAPACITY;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  ctx->last_stream = st;
  const int n = ctx->c.n_embd;
  const size_t aux_row = (size_t)3 * n;
  cudaError_t e = cudaSuccess;
  for (int b = 0; b < B && e == cudaSuccess; ++b) {
    const int P = prompt_len_host[b];
    for (int p0 = 0; p0 < P && e == cudaSuccess; p0 += kPrefillChunk) {
      const int cnt = std::min(kPrefillChunk, P - p0);
      e = enqueue_encode(ctx, aux + ((size_t)b * P_max + p0) * aux_row, cnt, ctx->genc, st, true);
      if (e != cudaSuccess) break;
      const int pairs = std::min(cnt, P - 1 - p0);
      if (pairs > 0) {
        GemvParams p = base_params(ctx);
        kv_only_params(ctx, kv, p);
        p.pairs.kind = PAIR_PREFILL;
        p.pairs.seq = b;
        p.pairs.pos0 = p0;
        p.pairs.tok_stride = P_max;
        p.pairs.tokens = tokens;
        p.pairs.enc_g = ctx->genc;
        e = qkv_items(ctx, p, pairs, st, true);
        if (e != cudaSuccess) break;
      }
      if (p0 + cnt == P)
        e = launched(ctx, st,
                     launch_prefill_finish(b, n, P - 1, ctx->genc + (size_t)(P - 1 - p0) * n,
                                           next_tok, bnd->g, bnd->tok, kv->kv_len, st),
                     PH_SMALL);
    }
  }
  ctx->rebuild_ok = 0;
  return cuda_err(e);
}

int eagle3_draft_chain(eagle3_ctx *ctx, int B, int gamma, unsigned flags,
                       const int32_t *kv_len_host, const eagle3_kv *kv,
                       const eagle3_boundary *bnd, int32_t *draft_tok, int32_t *draft_id,
                       int32_t *gamma_eff, float *logits_dbg, float *g_dbg,
                       eagle3_stream_t stream) {
  if (!ctx || B < 1 || B > ctx->c.max_batch) return EAGLE3_ERR_INVALID_ARG;
  if (gamma < 1 || gamma > ctx->c.max_gamma) return EAGLE3_ERR_INVALID_ARG;
  if (!kv_len_host || !kv_valid(ctx, kv) || !bnd || !aligned16(bnd->g) || !bnd->tok || !draft_tok)
    return EAGLE3_ERR_INVALID_ARG;
  if ((logits_dbg && !aligned16(logits_dbg)) || (g_dbg && !aligned16(g_dbg)))
    return EAGLE3_ERR_INVALID_ARG;
  if (flags & ~EAGLE3_SHRINK_GAMMA) return EAGLE3_ERR_INVALID_ARG;
  if (ctx->round_open) return EAGLE3_ERR_STATE;
  for (int b = 0; b < B; ++b) {
    int ge = 0;
    const int r = eagle3_plan_gamma(kv_len_host[b], gamma, ctx->c.max_cache_len, flags, &ge);
    if (r == EAGLE3_ERR_INVALID_ARG) return EAGLE3_ERR_INVALID_ARG;
    if (r != EAGLE3_OK) return EAGLE3_ERR_CAPACITY;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  ctx->last_stream = st;
  ChainArgs a;
  a.B = B;
  a.gamma = gamma;
  a.flags = flags;
  a.splits = 1;  // the attention's partition is planned on the device each round
  a.kv = kv;
  a.bnd = bnd;
  a.draft_tok = draft_tok;
  a.draft_id = draft_id;
  a.gamma_eff = gamma_eff;
  a.logits_dbg = logits_dbg;
  a.g_dbg = g_dbg;
  const cudaError_t e = ctx->graph_mode ? run_chain_graph(ctx, a, st) : enqueue_chain(ctx, a, st);
  if (e != cudaSuccess) return EAGLE3_ERR_CUDA;
  ctx->round_open = 1;
  ctx->open_B = B;
  ctx->rebuild_ok = 0;
  return EAGLE3_OK;
}

int eagle3_rewind(eagle3_ctx *ctx, int B, const eagle3_kv *kv, eagle3_stream_t stream) {
  if (!ctx || !kv || !kv->kv_len) return EAGLE3_ERR_INVALID_ARG;
  if (!ctx->round_open) return EAGLE3_ERR_STATE;
  if (B != ctx->open_B) return EAGLE3_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  ctx->last_stream = st;
  const cudaError_t e = launched(ctx, st, launch_rewind(B, kv->kv_len, ctx->round_start, st), PH_SMALL);
  if (e != cudaSuccess) return EAGLE3_ERR_CUDA;
  ctx->round_open = 0;
  ctx->rebuild_ok = 1;
  return EAGLE3_OK;
}

int eagle3_accept(eagle3_ctx *ctx, int B, int gamma, const int32_t *draft_tok,
                  const int32_t *target_pred, const int32_t *gamma_eff, int32_t *n_acc,
                  int32_t *bonus, eagle3_stream_t stream) {
  if (!ctx || B < 1 || B > ctx->c.max_batch || gamma < 1 || gamma > ctx->c.max_gamma)
    return EAGLE3_ERR_INVALID_ARG;
  if (!draft_tok || !target_pred || !n_acc || !bonus) return EAGLE3_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  ctx->last_stream = st;
  return cuda_err(launched(ctx, st,
                           launch_accept(B, gamma, draft_tok, target_pred, gamma_eff, n_acc, bonus, st),
                           PH_SMALL));
}

int eagle3_verify_greedy(eagle3_ctx *ctx, int B, int gamma, const uint16_t *target_lm_head,
                         const uint16_t *target_norm, float target_rms_eps, const float *hidden,
                         const int32_t *draft_tok, const int32_t *gamma_eff, int32_t *target_pred,
                         int32_t *n_acc, int32_t *bonus, float *logits_dbg, eagle3_stream_t stream) {
  if (!ctx || B < 1 || B > ctx->c.max_batch || gamma < 1 || gamma > ctx->c.max_gamma)
    return EAGLE3_ERR_INVALID_ARG;
  if (!aligned16(target_lm_head) || !aligned16(target_norm) || !aligned16(hidden)) return EAGLE3_ERR_INVALID_ARG;
  if (!draft_tok || !target_pred || !n_acc || !bonus || (logits_dbg && !aligned16(logits_dbg)))
    return EAGLE3_ERR_INVALID_ARG;
  const eagle3_config &c = ctx->c;
  if (c.target_vocab % 2 || !(target_rms_eps >= 0.f)) return EAGLE3_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  ctx->last_stream = st;
  // the lm_head + argmax kernels of the chain with the target's head: no d2t (ids are
  // target ids), every row valid, one output per window row
  GemvParams p = base_params(ctx);
  p.mode = GM_LMHEAD;
  p.rows = c.target_vocab;
  p.K = c.n_embd;
  p.w0 = target_lm_head;
  p.xf = hidden;
  p.norm0 = target_norm;
  p.eps = target_rms_eps;
  p.am_slot = ctx->am_slot;
  p.am_count = ctx->am_cnt;
  p.d2t = nullptr;
  p.draft_vocab = c.target_vocab;
  p.draft_tok = target_pred;
  p.gamma = 1;
  p.step = 0;
  p.dbg_f = logits_dbg;
  p.dbg_stride_b = c.target_vocab;
  p.dbg_off = 0;
  cudaError_t e = gemv_items(ctx, p, B * (gamma + 1), st, true);
  if (e == cudaSuccess)
    e = launched(ctx, st, launch_accept(B, gamma, draft_tok, target_pred, gamma_eff, n_acc, bonus, st),
                 PH_SMALL);
  return cuda_err(e);
}

int eagle3_rebuild_after_verify(eagle3_ctx *ctx, int B, int gamma, const int32_t *n_acc,
                                const int32_t *draft_tok, const int32_t *bonus,
                                const uint16_t *verify_aux, const eagle3_kv *kv,
                                eagle3_boundary *bnd, eagle3_stream_t stream) {
  if (!ctx || B < 1 || B > ctx->c.max_batch || gamma < 1 || gamma > ctx->c.max_gamma)
    return EAGLE3_ERR_INVALID_ARG;
  if (!n_acc || !draft_tok || !bonus || !aligned16(verify_aux)) return EAGLE3_ERR_INVALID_ARG;
  if (!kv_valid(ctx, kv) || !bnd || !aligned16(bnd->g) || !bnd->tok) return EAGLE3_ERR_INVALID_ARG;
  if (ctx->round_open || !ctx->rebuild_ok) return EAGLE3_ERR_STATE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  ctx->last_stream = st;
  const int n = ctx->c.n_embd;
  const int M = B * (gamma + 1);
  cudaError_t e = enqueue_encode(ctx, verify_aux, M, ctx->genc, st, true);
  if (e == cudaSuccess) {
    GemvParams p = base_params(ctx);
    kv_only_params(ctx, kv, p);
    p.pairs.kind = PAIR_REBUILD;
    p.pairs.gamma = gamma;
    p.pairs.bnd_tok = bnd->tok;
    p.pairs.bnd_g = bnd->g;
    p.pairs.draft_tok = draft_tok;
    p.pairs.enc_g = ctx->genc;
    p.pairs.kv_len = kv->kv_len;
    p.pairs.n_acc = n_acc;
    e = qkv_items(ctx, p, M, st, true);
  }
  if (e == cudaSuccess)
    e = launched(ctx, st,
                 launch_rebuild_finish(B, gamma, n, ctx->genc, n_acc, bonus, bnd->g, bnd->tok,
                                       kv->kv_len, ctx->c.max_cache_len, ctx->status, st),
                 PH_SMALL);
  if (e != cudaSuccess) return EAGLE3_ERR_CUDA;
  ctx->rebuild_ok = 0;
  return EAGLE3_OK;
}

unsigned long long eagle3_launch_count(const eagle3_ctx *ctx) { return ctx ? ctx->launches : 0ull; }

int eagle3_profile_begin(eagle3_ctx *ctx, int max_events) {
  if (!ctx || max_events < 2 || max_events > (1 << 16)) return EAGLE3_ERR_INVALID_ARG;
  for (cudaEvent_t e : ctx->ev_pool) cudaEventDestroy(e);
  ctx->ev_pool.assign(max_events, nullptr);
  for (int i = 0; i < max_events; ++i)
    if (cudaEventCreate(&ctx->ev_pool[i]) != cudaSuccess) {
      for (int j = 0; j < i; ++j) cudaEventDestroy(ctx->ev_pool[j]);
      ctx->ev_pool.clear();
      ctx->ev = nullptr;
      return EAGLE3_ERR_CUDA;
    }
  ctx->ev = ctx->ev_pool.data();
  ctx->ev_cap = max_events;
  ctx->ev_used = 0;
  ctx->ev_label.assign(max_events, -1);
  return EAGLE3_OK;
}

int eagle3_profile_end(eagle3_ctx *ctx, int *n_events) {
  if (!ctx || !n_events) return EAGLE3_ERR_INVALID_ARG;
  *n_events = ctx->ev_used;
  ctx->ev = nullptr;
  if (ctx->ev_used > 0 && cudaEventSynchronize(ctx->ev_pool[ctx->ev_used - 1]) != cudaSuccess)
    return EAGLE3_ERR_CUDA;
  return EAGLE3_OK;
}

int eagle3_profile_interval(const eagle3_ctx *ctx, int i, int *label, float *ms) {
  if (!ctx || !label || !ms || i < 1 || i >= ctx->ev_used) return EAGLE3_ERR_INVALID_ARG;
  *label = ctx->ev_label[i];
  if (cudaEventElapsedTime(ms, ctx->ev_pool[i - 1], ctx->ev_pool[i]) != cudaSuccess)
    return EAGLE3_ERR_CUDA;
  return EAGLE3_OK;
}

int eagle3_get_status(eagle3_ctx *ctx, int *device_status) {
  if (!ctx || !device_status) return EAGLE3_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(ctx->last_stream) != cudaSuccess) return EAGLE3_ERR_CUDA;
  int s = 0;
  if (cudaMemcpy(&s, ctx->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return EAGLE3_ERR_CUDA;
  *device_status = s;
  if (s != 0) {
    if (cudaMemset(ctx->status, 0, sizeof(int)) != cudaSuccess) return EAGLE3_ERR_CUDA;
    return EAGLE3_ERR_DEVICE;
  }
  return EAGLE3_OK;
}

}  // extern "C"
