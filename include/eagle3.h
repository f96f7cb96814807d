/*
 * eagle3.h -- C ABI of the EAGLE-3 drafter draft round for greedy speculative decoding,
 * GB300 (sm_103a).  Library: libeagle3.so (eagle_speculative_decode_gb300/).
 *
 * What the library computes (sources are cited as page title + section):
 *   - "memra_engine/eagle.rs" (docs.rs source page), module doc "Op-sequence": the fc
 *     encode g = fc . [aux_1; aux_15; aux_28] and one draft step: embed, RMSNorm of the
 *     embedding and of g, the 2*n_embd concat, q/k/v projections, partial NeoX RoPE,
 *     GQA attention over the drafter KV cache, o_proj + residual (pre-norm g),
 *     post-attention RMSNorm, SwiGLU MLP, fused-add residual (gsum, fed back as the next
 *     g), final RMSNorm, lm_head, argmax and target_id = draft_id + d2t[draft_id]
 *     (``d2t_map``); ``generate_spec_eagle`` steps 2 and 4: the chain of gamma steps and
 *     the greedy accept-prefix walk.
 *   - "feat(eagle3): Qwen3 EAGLE-3 drafter forward pass (single-step + chain rollout)",
 *     PR body: prefill_prompt / prefill_batched, draft_chain, chain_round (rewind leaves
 *     a round side-effect free), rebuild_after_verify; review comment: the k + 1
 *     capacity rule (start 97, k 3, max 100 must be refused or k shrunk).
 *   - "Add the Eagle3Speculator module for speculative decoding", PR body: the drafter
 *     pairs target hidden state t with token t + 1; after verify the draft cache is
 *     reseeded from verify's features paired with the corrected token.
 *
 * State of one sequence (committed tokens t_0..t_N, target features a_0..a_{N-1}):
 *   drafter KV holds pairs (fc a_p, t_{p+1}) at positions p = 0..N-2, kv_len = N - 1, and
 *   the boundary is (g = fc a_{N-1} as float32 [n_embd], tok = t_N).
 *
 * Conventions, all entry points:
 *   - Every buffer is caller-owned.  Weights, KV pools, page tables, boundary and output
 *     buffers are DEVICE pointers; arguments named *_host are HOST pointers.  bf16 data is
 *     passed as uint16_t bit patterns.  Device pointers must be 16-byte aligned.
 *   - Calls are asynchronous on the given stream and make no host<->device
 *     synchronisation, except eagle3_init (one upload of the RoPE table and a check of
 *     d2t) and eagle3_get_status.
 *   - Return 0 (EAGLE3_OK) or a negative error code.  On an error return nothing has
 *     been enqueued and no state has changed, except EAGLE3_ERR_CUDA where a launch
 *     failed part-way.
 *   - Device-side range checks (token ids, page ids, positions) never fault: the access
 *     is skipped and a bit is set in a device status word read by eagle3_get_status.
 *   - A context is used from one host thread at a time.
 */
#ifndef EAGLE3_H
#define EAGLE3_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *eagle3_stream_t;

#define EAGLE3_OK 0
#define EAGLE3_ERR_INVALID_ARG (-1) /* null/misaligned pointer, bad shape, gamma out of range, bad d2t */
#define EAGLE3_ERR_CAPACITY (-2)    /* kv_len + gamma + 1 > max_cache_len without EAGLE3_SHRINK_GAMMA */
#define EAGLE3_ERR_STATE (-3)       /* call out of order: chain while a round is open, rebuild before rewind */
#define EAGLE3_ERR_CUDA (-4)        /* a CUDA call or launch failed */
#define EAGLE3_ERR_DEVICE (-5)      /* the device status word is non-zero (eagle3_get_status) */
#define EAGLE3_ERR_UNSUPPORTED (-6) /* geometry outside what the kernels are built for */

/* Device status bits (eagle3_get_status). */
#define EAGLE3_DEV_BAD_TOKEN 1      /* token id outside [0, target_vocab) */
#define EAGLE3_DEV_BAD_PAGE 2       /* page id outside [0, num_pages) */
#define EAGLE3_DEV_BAD_POSITION 4   /* KV position outside [0, max_cache_len) */
#define EAGLE3_DEV_BAD_LENGTH 8     /* kv_len or prompt length out of range */
#define EAGLE3_DEV_TIMEOUT 16       /* a bounded on-chip wait gave up (the kernel returned) */

/* Drafter KV storage formats (eagle3_config.kv_format).
 *   EAGLE3_KV_BF16:       each K and V element as bf16.
 *   EAGLE3_KV_Q8_0_Q5_1:  the quantized drafter KV of "memra_engine/eagle.rs"
 *                         (Eagle3Scratch): K in q8_0 and V in q5_1 blocks of 32 values,
 *                         34 and 24 bytes per block; needs head_dim % 32 == 0.  Block
 *                         bytes (fp16 little endian):
 *                           q8_0: fp16 d | 32 int8 codes, x = d * code;
 *                           q5_1: fp16 d | fp16 m | uint32 whose bit i is bit 4 of code i |
 *                                 byte j = (code j & 15) | (code j+16 & 15) << 4, x = d * code + m.
 *                         Codes: d = fp16(max|x| / 127), code = rint(x / d) (q8_0);
 *                         d = fp16((max - min) / 31), m = fp16(min), code = rint((x - m) / d)
 *                         clamped to [0, 31] (q5_1); float32 arithmetic; all codes 0 when d = 0. */
#define EAGLE3_KV_BF16 0
#define EAGLE3_KV_Q8_0_Q5_1 1

/* Drafter weight formats (eagle3_config.weight_format).
 *   EAGLE3_W_BF16:       every matrix bf16 [out, in].
 *   EAGLE3_W_INT4_G128:  the per-step projections q, k, v, o, gate, up, down and lm_head
 *                        as 4-bit weights ("Add a weight-stationary INT4 GEMM for small M",
 *                        the stack of the Eagle3Speculator PR): a matrix [out, in] is
 *                        codes, uint8 [out, in / 2] with the code of in-index 2j in the low
 *                        nibble of byte j and 2j + 1 in the high nibble, and sz, bf16 pairs
 *                        (scale, zero) [out, sz_stride(in)] for the groups of 128 in-indices,
 *                        sz_stride(in) = in / 128 rounded up to a multiple of 4 (the pad is
 *                        unused); w = scale * (code - 8) + zero.  fc, the norm gains and the
 *                        embedding stay bf16.  Needs n_embd, n_head * head_dim and n_ff
 *                        multiples of 128.  Single-item launches whose input width is a
 *                        multiple of 2048 run on warp-level tensor-core MMAs (mma.sync) fed
 *                        by codes decoded in registers; launches of several items, and other
 *                        widths, run on the CUDA-core GEMV (one launch streams the weights
 *                        once for up to 8 items). */
#define EAGLE3_W_BF16 0
#define EAGLE3_W_INT4_G128 1

/* Checkpoint flags (eagle3_config.flags) of the EAGLE-3 layer's op sequence
 * ("memra_engine/eagle.rs", module doc: this checkpoint has norm_before_residual,
 * norm_before_fc, fc_norm and norm_output all false, and its residual is the PRE-norm g).
 *   EAGLE3_CKPT_NORM_BEFORE_RESIDUAL: the attention residual is the normed
 *   RMSNorm(g) * hidden_norm instead of g (x1 = o_proj(attn) + RMSNorm(g) * hidden_norm).
 * The other three flags are not supported (eagle3_config_from_json refuses them). */
#define EAGLE3_CKPT_NORM_BEFORE_RESIDUAL 1u

/* eagle3_draft_chain flags. */
#define EAGLE3_SHRINK_GAMMA 1u      /* shrink gamma per sequence to max_cache_len - kv_len - 1 */

/* Drafter geometry and capacity limits.
 * Kernels are built for head_dim in {64, 128, 256}, n_head / n_head_kv in {1, 2, 4, 8},
 * n_embd, n_ff multiples of 8 and rope_dims even, <= head_dim. */
typedef struct {
  int n_embd;          /* hidden size n                                     (4096)   */
  int n_head;          /* query heads H                                     (16)     */
  int n_head_kv;       /* key/value heads H_kv                              (4)      */
  int head_dim;        /* d                                                 (256)    */
  int rope_dims;       /* leading dims of each head that RoPE rotates       (64)     */
  float rope_theta;    /* RoPE base                                         (1e7)    */
  float rms_eps;       /* RMSNorm epsilon                                   (1e-6)   */
  int n_ff;            /* MLP width F                                       (12288)  */
  int draft_vocab;     /* lm_head rows V_d                                  (32000)  */
  int target_vocab;    /* embedding rows V_t, range of d2t-mapped ids       (248320) */
  int max_batch;       /* largest B of any call                                      */
  int max_gamma;       /* largest chain length                                       */
  int max_cache_len;   /* KV positions per sequence (0 .. max_cache_len - 1)         */
  int page_size;       /* KV positions per page                                      */
  unsigned flags;      /* EAGLE3_CKPT_* checkpoint flags, 0 for the eagle.rs checkpoint      */
  int kv_format;       /* EAGLE3_KV_BF16 (default) or EAGLE3_KV_Q8_0_Q5_1; quantized pools
                        * are read a page-aligned run of keys at a time, so that run's K and
                        * V bytes must be multiples of 16 (head_dim 64: page_size % 4 == 0;
                        * head_dim 128: even page_size; head_dim 256: any page_size)     */
  int weight_format;   /* EAGLE3_W_BF16 (default) or EAGLE3_W_INT4_G128                    */
} eagle3_config;

/* Drafter weights: bf16, PyTorch Linear layout [out, in] row-major, device memory,
 * owned by the caller and left unchanged.  Shapes: fc [n, 3n]; q [H d, 2n];
 * k, v [H_kv d, 2n]; o [n, H d]; gate, up [F, n]; down [n, F]; lm_head [V_d, n];
 * embed [V_t, n] (the target's token embedding, indexed by target id); the four
 * RMSNorm gains [n].  d2t: int64 [V_d], target_id = draft_id + d2t[draft_id].
 * With EAGLE3_W_INT4_G128 the eight projection pointers hold the codes and the *_sz
 * pointers their (scale, zero) rows (see the format above); otherwise the *_sz pointers
 * are ignored.  Every pointer 16-byte aligned. */
typedef struct {
  const uint16_t *fc, *in_norm, *hidden_norm, *q, *k, *v, *o, *post_norm, *gate, *up, *down,
      *final_norm, *lm_head, *embed;
  const int64_t *d2t;
  const uint32_t *q_sz, *k_sz, *v_sz, *o_sz, *gate_sz, *up_sz, *down_sz, *lm_head_sz;
} eagle3_weights;

/* Paged drafter KV cache, device memory owned by the caller.
 *   k_pool, v_pool: [num_pages, n_head_kv, page_size] rows of eagle3_kv_row_bytes bytes:
 *                   bf16 [head_dim] per row, or head_dim / 32 q8_0 (K) / q5_1 (V) blocks;
 *                   16-byte aligned.
 *   page_table:     int32 [B, max_pages_per_seq]; position p of sequence b lives in page
 *                   page_table[b, p / page_size] at slot p % page_size.  The caller
 *                   reserves max_cache_len positions per sequence up front.
 *   kv_len:         int32 [B], committed length of each sequence (device copy). */
typedef struct {
  void *k_pool, *v_pool;
  const int32_t *page_table;
  int num_pages;
  int max_pages_per_seq;
  int32_t *kv_len;
} eagle3_kv;

/* Boundary of each sequence: g float32 [B, n] (= fc a_{N-1}) and tok int32 [B] (= t_N). */
typedef struct {
  float *g;
  int32_t *tok;
} eagle3_boundary;

typedef struct eagle3_ctx eagle3_ctx;

/* Library version, (major << 16) | minor. */
int eagle3_version(void);

/* Static description of an error code. */
const char *eagle3_error_string(int code);

/* Device workspace a context needs for cfg, in bytes; 0 if cfg is invalid or
 * unsupported.  Host-only arithmetic. */
size_t eagle3_workspace_bytes(const eagle3_config *cfg);

/* Bytes of one K row and one V row of the paged pools (one position of one kv head) for
 * cfg's kv_format: 2 * head_dim each for bf16; head_dim / 32 * 34 (K) and
 * head_dim / 32 * 24 (V) for q8_0 / q5_1.  Returns EAGLE3_ERR_INVALID_ARG for an invalid
 * cfg or null outputs.  Host-only arithmetic. */
int eagle3_kv_row_bytes(const eagle3_config *cfg, size_t *k_row, size_t *v_row);

/* Self-test of the device-side failure path: launches one small kernel whose thread waits
 * on an mbarrier that nothing completes.  The bounded wait gives up (about a second at
 * most), ORs EAGLE3_DEV_TIMEOUT into *device_status (device int32, caller-zeroed) and sets
 * the CTA's abort flag, after which a second wait returns at once; *device_result (device
 * int32) receives bit 0 = first wait succeeded, bit 1 = second wait succeeded, bit 2 =
 * abort flag set (4 expected).  The kernel exits normally, so the context stays usable.
 * Asynchronous on stream.  EAGLE3_ERR_INVALID_ARG for null pointers. */
int eagle3_selftest_bounded_wait(int *device_status, int *device_result, eagle3_stream_t stream);

/* Rotary width of a drafter config ("memra_engine/eagle.rs", EagleConfig::rope_dim_count
 * and its tests on the eagle3-qwen35-9b config): an explicit rotary dim count (has_rotary_dim,
 * even, 2..head_dim) wins over a fraction of head_dim (has_factor), which wins over the full
 * width; a fraction outside (0, 1] or one that does not give a whole, even number of dims
 * takes the full width, never a rotation wider than the head.  Returns 0 for an odd or
 * non-positive head_dim.  Host-only arithmetic. */
int eagle3_resolve_rope_dims(int head_dim, int has_rotary_dim, int rotary_dim, int has_factor,
                             float factor);

/* Drafter shape from the text of a checkpoint's config.json ("memra_engine/eagle.rs",
 * EagleConfig::from_json_str): n_embd (hidden_size), n_head (num_attention_heads), n_head_kv
 * (num_key_value_heads), head_dim, n_ff (intermediate_size), draft_vocab
 * (draft_vocab_size), target_vocab (vocab_size), rope_dims (eagle3_resolve_rope_dims of
 * rotary_dim and partial_rotary_factor, found top-level or under rope_parameters),
 * rope_theta (default 10000), rms_eps (rms_norm_eps, default 1e-6) and flags
 * (norm_before_residual).  max_batch, max_gamma, max_cache_len, page_size and kv_format are
 * left as the caller set them.  EAGLE3_ERR_INVALID_ARG when a required key is missing or
 * not a positive integer, or the aux-layer list is malformed; EAGLE3_ERR_UNSUPPORTED when
 * norm_before_fc, fc_norm or norm_output is true or the aux-layer list does not hold three
 * ids (fc takes three features).  cfg is written only on success.  Host-only. */
int eagle3_config_from_json(const char *json, eagle3_config *cfg);

/* Capacity rule ("feat(eagle3) ...", review comment on rebuild_after_verify committing
 * k + 1 entries): a chain of gamma drafts at committed length kv_len needs
 * kv_len + gamma + 1 <= max_cache_len.  Writes the allowed chain length to *gamma_eff and
 * returns EAGLE3_OK, or returns EAGLE3_ERR_CAPACITY (with EAGLE3_SHRINK_GAMMA in flags the
 * chain shrinks to max_cache_len - kv_len - 1, refused below 1), or EAGLE3_ERR_INVALID_ARG
 * for gamma < 1 or kv_len < 0.  Host-only arithmetic. */
int eagle3_plan_gamma(int kv_len, int gamma, int max_cache_len, unsigned flags, int *gamma_eff);

/* Create a context.  workspace: device buffer of eagle3_workspace_bytes(cfg) bytes,
 * 256-byte aligned, owned by the caller and used by this context only until
 * eagle3_destroy.  Validates cfg and the weight pointers, checks on the host that d2t
 * maps every draft id to a distinct target id in [0, target_vocab) (a blocking copy of
 * d2t), and uploads the RoPE table (angles in double, stored as float32 cos/sin).  The
 * context object itself lives in host memory and is freed by eagle3_destroy. */
int eagle3_init(const eagle3_config *cfg, const eagle3_weights *w, void *workspace,
                size_t workspace_bytes, eagle3_stream_t stream, eagle3_ctx **out);

/* Release the host context (the workspace stays the caller's). */
int eagle3_destroy(eagle3_ctx *ctx);

/* Encode ("memra_engine/eagle.rs", Eagle3Draft::encode): g[m] = fc . concat(aux[m, 0],
 * aux[m, 1], aux[m, 2]) for m < M.  aux: bf16 [M, 3, n] device; g: float32 [M, n] device.
 * M >= 0 (M = 0 does nothing). */
int eagle3_encode(eagle3_ctx *ctx, const uint16_t *aux, int M, float *g, eagle3_stream_t stream);

/* Teacher-forced prefill ("feat(eagle3) ...", PR body: prefill_prompt / prefill_batched).
 * For each sequence b with prompt t_0..t_{P-1} (P = prompt_len_host[b], 1 <= P <= P_max),
 * target features a_0..a_{P-1} and the target's greedy next token t_P:
 * writes the KV pairs (fc a_p, t_{p+1}) at positions p = 0..P-2, sets kv_len[b] = P - 1
 * and the boundary (fc a_{P-1}, t_P).
 *   tokens:   int32 [B, P_max] device, row b holds t_0..t_{P-1}
 *   next_tok: int32 [B] device, t_P
 *   aux:      bf16 [B, P_max, 3, n] device
 *   prompt_len_host: int32 [B] host; P <= max_cache_len is required. */
int eagle3_prefill(eagle3_ctx *ctx, int B, const int32_t *tokens, int P_max,
                   const int32_t *next_tok, const int32_t *prompt_len_host, const uint16_t *aux,
                   const eagle3_kv *kv, eagle3_boundary *bnd, eagle3_stream_t stream);

/* Draft chain ("memra_engine/eagle.rs", generate_spec_eagle step 2; "feat(eagle3) ...",
 * PR body: draft_chain): gamma draft steps from the boundary of each sequence at
 * positions kv_len[b] + j.  Step 0 embeds bnd->tok with g = bnd->g; step j > 0 embeds the
 * previous step's target id with the previous step's gsum.  Opens a round: the
 * speculative KV entries are written at kv_len .. kv_len + gamma_eff - 1 and kv_len
 * advances by gamma_eff; eagle3_rewind closes the round.  The boundary is not modified.
 *   kv_len_host: int32 [B] host mirror of kv_len, used for the capacity check.
 *   draft_tok:   int32 [B, gamma] device, target ids d_1..d_gamma (-1 past gamma_eff).
 *   draft_id, gamma_eff, logits_dbg (float32 [B, gamma, V_d]), g_dbg (float32
 *   [B, gamma, n]): optional device outputs, NULL to skip.
 * Refused with EAGLE3_ERR_CAPACITY unless kv_len + gamma + 1 <= max_cache_len for every
 * sequence, or EAGLE3_SHRINK_GAMMA is set (then gamma_eff = max_cache_len - kv_len - 1). */
int eagle3_draft_chain(eagle3_ctx *ctx, int B, int gamma, unsigned flags,
                       const int32_t *kv_len_host, const eagle3_kv *kv,
                       const eagle3_boundary *bnd, int32_t *draft_tok, int32_t *draft_id,
                       int32_t *gamma_eff, float *logits_dbg, float *g_dbg,
                       eagle3_stream_t stream);

/* Rewind ("feat(eagle3) ...", PR body: chain_round rewinds the speculative KV): restore
 * kv_len[b] to its value at the start of the open round.  Committed entries, the page
 * table and the boundary are untouched.  EAGLE3_ERR_STATE if no round is open. */
int eagle3_rewind(eagle3_ctx *ctx, int B, const eagle3_kv *kv, eagle3_stream_t stream);

/* Greedy accept walk ("memra_engine/eagle.rs", generate_spec_eagle step 4):
 * n_acc[b] = number of leading i with target_pred[b, i] == draft_tok[b, i] (i < gamma_eff),
 * bonus[b] = target_pred[b, n_acc[b]].  target_pred: int32 [B, gamma + 1] device, the
 * target's greedy token after each verify position; gamma_eff may be NULL (= gamma). */
int eagle3_accept(eagle3_ctx *ctx, int B, int gamma, const int32_t *draft_tok,
                  const int32_t *target_pred, const int32_t *gamma_eff, int32_t *n_acc,
                  int32_t *bonus, eagle3_stream_t stream);

/* Greedy verify on the target side ("Add the Eagle3Speculator module for speculative
 * decoding", PR body: target_verify returns the greedy argmax target id of every window
 * position; "memra_engine/eagle.rs", generate_spec_eagle steps 3-4).  For sequence b and
 * window position i = 0..gamma:
 *   target_pred[b, i] = argmax over v < target_vocab of
 *                       (target_lm_head . (RMSNorm(hidden[b, i]) * target_norm))[v],
 * the lowest id among equal maxima (RMSNorm with target_rms_eps), then the accept walk of
 * eagle3_accept writes n_acc and bonus.
 *   target_lm_head: bf16 [target_vocab, n_embd] row-major, device, 16-byte aligned.
 *   target_norm:    bf16 [n_embd], the target's final-norm gain.
 *   hidden:         float32 [B, gamma + 1, n_embd], the target's last hidden states at
 *                   the window positions (before its final norm), 16-byte aligned.
 *   draft_tok [B, gamma], gamma_eff [B] or NULL: as eagle3_accept.
 *   target_pred:    int32 [B, gamma + 1] out; n_acc, bonus: int32 [B] out.
 *   logits_dbg:     float32 [B, gamma + 1, target_vocab] or NULL.
 * Every window row is computed whatever gamma_eff (the head is read once either way).
 * Uses the context's argmax scratch, so it runs on the context's stream order like the
 * other calls; it changes no round state.  EAGLE3_ERR_INVALID_ARG for B or gamma out of
 * range, a null or misaligned pointer, an odd target_vocab or a negative eps. */
int eagle3_verify_greedy(eagle3_ctx *ctx, int B, int gamma, const uint16_t *target_lm_head,
                         const uint16_t *target_norm, float target_rms_eps, const float *hidden,
                         const int32_t *draft_tok, const int32_t *gamma_eff, int32_t *target_pred,
                         int32_t *n_acc, int32_t *bonus, float *logits_dbg, eagle3_stream_t stream);

/* Rebuild after verify ("feat(eagle3) ...", PR body: rebuild_after_verify; "Add the
 * Eagle3Speculator module", PR body): with verify features v_i (target features at the
 * verify positions N + i, bf16 [B, gamma + 1, 3, n] device) writes the pairs at
 * kv_len + i for i = 0..n_acc[b]: pair 0 = (old boundary g, old boundary tok), pair i >= 1
 * = (fc v_{i-1}, draft_tok[b, i-1]); then kv_len += n_acc + 1 and the boundary becomes
 * (fc v_{n_acc}, bonus).  Requires the round to be rewound first (EAGLE3_ERR_STATE).
 * n_acc, draft_tok, bonus: device int32 from the chain and eagle3_accept. */
int eagle3_rebuild_after_verify(eagle3_ctx *ctx, int B, int gamma, const int32_t *n_acc,
                                const int32_t *draft_tok, const int32_t *bonus,
                                const uint16_t *verify_aux, const eagle3_kv *kv,
                                eagle3_boundary *bnd, eagle3_stream_t stream);

/* Synchronise the context's last stream and read the device status word (0 = clean);
 * returns EAGLE3_ERR_DEVICE when it is non-zero.  Clears the word.  Not for hot loops. */
int eagle3_get_status(eagle3_ctx *ctx, int *device_status);

/* Launch mode of eagle3_draft_chain: 1 (default) replays a CUDA graph of the gamma
 * steps captured per (B, gamma, flags, buffer set); 0 launches the kernels directly. */
int eagle3_set_graph_mode(eagle3_ctx *ctx, int enabled);

/* Smallest number of activation rows (items) for which a projection runs on the tensor
 * cores (tcgen05, the weights read once for up to 128 items per tile) instead of the
 * CUDA-core weight-streaming GEMV.  0 restores the default (3); a value above every batch
 * keeps all projections on the GEMV.  The tensor-core path needs a geometry whose K dims
 * are multiples of 64 and whose q / k / v blocks are whole 128-row tiles; otherwise the
 * GEMV is used whatever the threshold.  Takes effect for later calls (a captured chain
 * graph is re-captured).  Returns EAGLE3_ERR_INVALID_ARG for a negative value. */
int eagle3_set_tc_min_items(eagle3_ctx *ctx, int min_items);

/* How a tensor-core projection spreads its 128-row tiles over the SMs.  0 (the default)
 * chooses per launch: cluster split-K when there are few tiles -- each tile split along K
 * over a thread-block cluster of 2..8 CTAs whose partial sums meet in distributed shared
 * memory, every rank finishing its share of the tile's columns -- if that keeps at least
 * 60% of the SMs busy; persistent stream-K otherwise (equal shares of all k-tiles per
 * SM, a shared tile finished by its last contributor from partials published in L2).
 * 1 always uses stream-K; 2 uses cluster split-K wherever 2..8 CTAs per tile fit on the
 * GPU at once, whatever the fill.  Both give the same results up to the float32
 * summation order of the partial sums.  Takes effect for later calls (a captured chain
 * graph is re-captured).  Returns EAGLE3_ERR_INVALID_ARG for another value. */
int eagle3_set_tc_schedule(eagle3_ctx *ctx, int schedule);

/* Which kernel runs the decode attention over a bf16 KV cache.  0 (the default): the
 * CUDA-core kernel (packed float32 FMAs).  1: the tensor-core kernel -- QK and PV on
 * warp-level bf16 MMAs, q and the probabilities split into three exact bf16 parts so the
 * arithmetic keeps float32 accuracy -- wherever it applies (head_dim 64, 128 or 256; at
 * most 4 q heads per kv head; attention units of 16 to 64 keys, i.e. a page size that is
 * a multiple of 16), the CUDA-core kernel otherwise.  A quantized KV cache always uses the
 * CUDA-core kernel.  Both give the same results up to the float32 summation order; on
 * the drafter's long contexts the CUDA-core kernel is the faster one.  Takes effect for
 * later calls (a captured chain graph is re-captured).  Returns EAGLE3_ERR_INVALID_ARG for
 * another value. */
int eagle3_set_attention(eagle3_ctx *ctx, int mode);

/* ---- measurement (no counterpart on the pages; used by the benchmark) ----------------- */

/* Number of kernels this context has launched since eagle3_init (a graph replay counts
 * every kernel in the graph).  Host-only. */
unsigned long long eagle3_launch_count(const eagle3_ctx *ctx);

/* Kernel timing.  eagle3_profile_begin creates max_events CUDA events (host calls, no
 * device memory) and from then on every directly launched call (graph mode off) records
 * one event on its stream after each of its kernels (eagle3_draft_chain also records one
 * before its first kernel), until max_events are used.  An event between two kernels
 * removes their launch overlap, so use this to time kernels, not whole rounds. */
int eagle3_profile_begin(eagle3_ctx *ctx, int max_events);

/* Stop recording, wait for the last recorded event, and return how many were recorded. */
int eagle3_profile_end(eagle3_ctx *ctx, int *n_events);

/* For recorded event i >= 1: *ms = time from event i-1 to event i, and *label = the kernel
 * launched between them: 0 = start marker, 1 = q/k/v GEMV, 2 = attention, 3 = o_proj
 * GEMV, 4 = gate/up GEMV, 5 = down GEMV, 6 = lm_head GEMV + argmax, 7 = encode GEMV,
 * 8 = k/v-only GEMV (prefill, rebuild), 9 = bookkeeping kernel. */
int eagle3_profile_interval(const eagle3_ctx *ctx, int i, int *label, float *ms);

/* ---- lm_head argmax without any allocation ------------------------------------------
 * The pages have no counterpart: this entry point exists for callers that cannot allocate
 * device memory when they need the result -- for example code that runs while a CUDA
 * graph is being captured (cudaMalloc is not allowed there) or a runtime whose memory plan
 * is fixed at start-up and that therefore cannot provide a context workspace.
 *
 * Computes, for each of `rows` float32 vectors x[r] (device, [rows, n_embd]), what the
 * draft chain's lm_head step computes, on the chain's CUDA-core GEMV kernel (the chain
 * itself runs its lm_head on that kernel for one or two rows and on the tensor cores from
 * three rows on): logits = lm_head . (RMSNorm(x[r]) * final_norm), draft_id[r] = the
 * argmax (lowest index on ties), target_id[r] = draft_id[r] + d2t[draft_id[r]].  Same
 * weights and layouts as eagle3_weights; draft_id and logits ([rows, draft_vocab]) may be
 * NULL; target_id is required.  Every buffer is caller-owned device memory.  There is no
 * context and so no status word: a row whose target id falls outside [0, target_vocab)
 * (a d2t table that was never validated) gets -1 in target_id and draft_id instead.  The
 * inputs must be finite; a NaN in x or the weights is not detected.
 *
 * The kernel's scratch (one argmax slot per row and an arrival counter) lives in a static
 * device array inside the library, so the call allocates nothing: it is limited to
 * rows <= 64 (larger requests return EAGLE3_ERR_INVALID_ARG), and every GPU that loads the
 * library holds that array (about 520 bytes) until the process exits.  The first call on a
 * device looks the array's device address up; make that first call before any stream
 * capture.  All calls share the array, which keeps the last call's contents (each call
 * clears it on its stream before use).  Each device has its own copy of the array, so
 * calls race only when they overlap on the same device (issued on different streams, or
 * from different host threads without ordering); serialise those.
 * Returns EAGLE3_OK, EAGLE3_ERR_INVALID_ARG or EAGLE3_ERR_CUDA. */
int eagle3_lmhead_argmax_noalloc(const uint16_t *lm_head, const uint16_t *final_norm,
                                 const int64_t *d2t, const float *x, int rows, int n_embd,
                                 int draft_vocab, int target_vocab, float rms_eps,
                                 int32_t *draft_id, int32_t *target_id, float *logits,
                                 eagle3_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* EAGLE3_H */
