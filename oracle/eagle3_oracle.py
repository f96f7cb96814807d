"""CPU oracle of the EAGLE-3 drafter draft round -- TEST INFRASTRUCTURE, not product.

Only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference legs
of ``bench.py`` may import this module.  The product path (the CUDA library and its
Python binding) never calls it, and this module imports nothing from the product.

It is the plain definition of what the drafter computes, written in float64 numpy:
bf16 weights are widened exactly, every product and sum is float64, and the only
rounding the method itself prescribes -- the drafter KV cache stored as bf16 -- is
applied at the point where entries are stored.  No blocking, fusion or reordering.

Sources (page title, section):
  * "memra_engine/eagle.rs" (docs.rs source page): module doc "Op-sequence" (the
    authority on one draft step), ``Eagle3Draft::encode``, ``draft_token``, ``attn``,
    ``d2t_map``, and ``generate_spec_eagle`` steps 1-5 (round loop, greedy accept walk,
    EAGLE token/hidden alignment comment).
  * "feat(eagle3): Qwen3 EAGLE-3 drafter forward pass (single-step + chain rollout)":
    PR body (draft_step, prefill_prompt, draft_chain, chain_round,
    rebuild_after_verify) and the review comment on the k + 1 capacity rule.
  * "Add the Eagle3Speculator module for speculative decoding": PR body (shifted
    pairing of hidden state t with token t + 1; reseeding the draft cache after verify).

Readings where the pages are silent or disagree (the plainest one the rest of the pages
support):
  * RoPE is NeoX rotate-half over the first ``rope_dims`` dims, frequencies
    theta^(-2i/rope_dims); the remaining dims pass through.
  * q head h reads kv head h // (n_head / n_head_kv); scale 1/sqrt(head_dim); the new
    key is appended before attending.
  * RMSNorm multiplies the gain directly: x / sqrt(mean(x^2) + eps) * w.
  * argmax takes the lowest index among equal maxima.
  * State of a sequence with committed tokens t_0..t_N and target features
    a_0..a_{N-1}: KV pairs (a_p, t_{p+1}) at positions p = 0..N-2, kv_len L = N-1,
    boundary (g = fc a_{N-1}, tok = t_N).

Parity status: every function below is pinned by tests/test_oracle_pins.py against
closed forms, special cases and page-fixed values; none is "parity unpinned".
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


class CapacityError(ValueError):
    """A chain of gamma drafts would not leave room for the all-accepted rebuild."""


# ----------------------------------------------------------------------------- bf16

def widen_bf16(bits) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact: bf16 is the top half of a float32)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even (values inside
    bf16's normal range).  bf16 keeps 7 of float64's 52 fraction bits."""
    a = np.ascontiguousarray(x, dtype=np.float64)
    u = a.view(np.uint64)
    drop = np.uint64(45)
    lsb = (u >> drop) & np.uint64(1)
    half_minus_one = np.uint64((1 << 44) - 1)
    r = (u + half_minus_one + lsb) & ~np.uint64((1 << 45) - 1)
    return r.view(np.float64)


# ----------------------------------------------------------------------- elementary

def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """Llama RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * w."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def rope_neox(x: np.ndarray, pos: int, rope_dims: int, theta: float) -> np.ndarray:
    """Partial NeoX RoPE on x[..., head_dim] at position pos: for i < rope_dims/2 the pair
    (x_i, x_{i+rope_dims/2}) is rotated by the angle pos * theta^(-2i/rope_dims);
    dims >= rope_dims are returned unchanged ("memra_engine/eagle.rs", ``attn``:
    rope_neox with rope_dim_count 64 of head_dim 256)."""
    half = rope_dims // 2
    i = np.arange(half, dtype=np.float64)
    ang = float(pos) * np.power(float(theta), -2.0 * i / rope_dims)
    c, s = np.cos(ang), np.sin(ang)
    out = np.array(x, dtype=np.float64, copy=True)
    a = x[..., :half]
    b = x[..., half:rope_dims]
    out[..., :half] = a * c - b * s
    out[..., half:rope_dims] = b * c + a * s
    return out


def gqa_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """Decode attention of one query position.  q [H, d]; k, v [T, H_kv, d].
    Head h attends with kv head h // (H / H_kv); scores scaled by 1/sqrt(d); softmax
    over all T keys (no mask needed: every cached key precedes the query)."""
    n_head, d = q.shape
    group = n_head // k.shape[1]
    out = np.empty((n_head, d), dtype=np.float64)
    for h in range(n_head):
        kh = k[:, h // group, :]
        vh = v[:, h // group, :]
        s = (kh @ q[h]) / np.sqrt(d)
        p = np.exp(s - s.max())
        out[h] = (p @ vh) / p.sum()
    return out


def silu(x: np.ndarray) -> np.ndarray:
    """x * sigmoid(x)."""
    return x / (1.0 + np.exp(-x))


def argmax_first(x: np.ndarray) -> int:
    """Index of the maximum; the lowest index among equal maxima."""
    return int(np.argmax(x))


# ------------------------------------------------------------- quantized drafter KV
# "memra_engine/eagle.rs", ``Eagle3Scratch``: the drafter KV uses the q8_0-K / q5_1-V
# quantized layout of the trunk KV, blocks of 32 values (head_dim % 32 == 0), 34 and 24
# bytes per block.  The page names the formats and sizes only; the encodings below are
# the plain reading of those names and sizes: per block, q8_0 keeps an
# fp16 scale and 32 signed 8-bit codes, q5_1 an fp16 scale, an fp16 minimum and 32
# unsigned 5-bit codes.  Codes are decided in float32 on the values as the kernel holds
# them (float32), with the stored (fp16) scale: the same precision on both sides.

QK = 32                   # values per block
Q8_0_BLOCK_BYTES = 34     # fp16 d + 32 x int8
Q5_1_BLOCK_BYTES = 24     # fp16 d + fp16 m + uint32 fifth bits + 16 bytes of 4-bit codes


def _blocks(x) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32)
    if x.shape[-1] % QK:
        raise ValueError("the last axis must be a multiple of 32")
    return x.reshape(x.shape[:-1] + (x.shape[-1] // QK, QK))


def quantize_q8_0(x):
    """Per block of 32: d = fp16(max|x| / 127); code = clamp(rint(x / d), -127, 127),
    all codes 0 when d = 0.  Returns (d as float16 [..., nb], codes int8 [..., nb, 32])."""
    xb = _blocks(x)
    amax = np.max(np.abs(xb), axis=-1)
    d16 = (amax / np.float32(127)).astype(np.float16)
    d = d16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(d > 0, np.clip(np.rint(xb / np.where(d > 0, d, np.float32(1))), -127, 127), 0)
    return d16, q.astype(np.int8)


def dequantize_q8_0(d16, codes) -> np.ndarray:
    """x = d * code (exact in float32: an 11-bit scale times an 8-bit code)."""
    v = d16.astype(np.float32)[..., None] * codes.astype(np.float32)
    return v.reshape(v.shape[:-2] + (v.shape[-2] * QK,))


def quantize_q5_1(x):
    """Per block of 32: d = fp16((max - min) / 31), m = fp16(min);
    code = clamp(rint((x - m) / d), 0, 31), all codes 0 when d = 0.
    Returns (d float16 [..., nb], m float16 [..., nb], codes uint8 [..., nb, 32])."""
    xb = _blocks(x)
    mn = np.min(xb, axis=-1)
    mx = np.max(xb, axis=-1)
    d16 = ((mx - mn) / np.float32(31)).astype(np.float16)
    m16 = mn.astype(np.float16)
    d = d16.astype(np.float32)[..., None]
    m = m16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(d > 0, np.clip(np.rint((xb - m) / np.where(d > 0, d, np.float32(1))), 0, 31), 0)
    return d16, m16, q.astype(np.uint8)


def dequantize_q5_1(d16, m16, codes) -> np.ndarray:
    """x = d * code + m in float32 (the product is exact; one rounding for the sum)."""
    v = d16.astype(np.float32)[..., None] * codes.astype(np.float32) + m16.astype(np.float32)[..., None]
    return v.astype(np.float32).reshape(v.shape[:-2] + (v.shape[-2] * QK,))


def pack_q8_0(d16, codes) -> np.ndarray:
    """Block bytes: fp16 d (little endian), then the 32 int8 codes in element order."""
    d16 = np.asarray(d16, dtype=np.float16)
    out = np.empty(d16.shape + (Q8_0_BLOCK_BYTES,), dtype=np.uint8)
    out[..., 0:2] = d16[..., None].view(np.uint8).reshape(d16.shape + (2,))
    out[..., 2:] = np.asarray(codes, dtype=np.int8).view(np.uint8)
    return out


def unpack_q8_0(blocks):
    b = np.asarray(blocks, dtype=np.uint8)
    d16 = np.ascontiguousarray(b[..., 0:2]).view(np.float16)[..., 0]
    return d16, np.ascontiguousarray(b[..., 2:]).view(np.int8)


def pack_q5_1(d16, m16, codes) -> np.ndarray:
    """Block bytes: fp16 d, fp16 m, uint32 whose bit i is bit 4 of code i, then byte j =
    (code j & 15) | (code (j + 16) & 15) << 4 for j = 0..15."""
    d16 = np.asarray(d16, dtype=np.float16)
    m16 = np.asarray(m16, dtype=np.float16)
    q = np.asarray(codes, dtype=np.uint32)
    out = np.empty(d16.shape + (Q5_1_BLOCK_BYTES,), dtype=np.uint8)
    out[..., 0:2] = d16[..., None].view(np.uint8).reshape(d16.shape + (2,))
    out[..., 2:4] = m16[..., None].view(np.uint8).reshape(m16.shape + (2,))
    qh = np.sum(((q >> 4) & 1) << np.arange(QK, dtype=np.uint32), axis=-1).astype(np.uint32)
    out[..., 4:8] = qh[..., None].view(np.uint8).reshape(qh.shape + (4,))
    out[..., 8:] = ((q[..., :16] & 15) | ((q[..., 16:] & 15) << 4)).astype(np.uint8)
    return out


def unpack_q5_1(blocks):
    b = np.asarray(blocks, dtype=np.uint8)
    d16 = np.ascontiguousarray(b[..., 0:2]).view(np.float16)[..., 0]
    m16 = np.ascontiguousarray(b[..., 2:4]).view(np.float16)[..., 0]
    qh = np.ascontiguousarray(b[..., 4:8]).view(np.uint32)[..., 0]
    lo = b[..., 8:].astype(np.uint32)
    nib = np.concatenate([lo & 15, lo >> 4], axis=-1)
    hi = (qh[..., None] >> np.arange(QK, dtype=np.uint32)) & 1
    return d16, m16, (nib | (hi << 4)).astype(np.uint8)


KV_FORMATS = ("bf16", "q8_0/q5_1")

# ------------------------------------------------------------- INT4 drafter weights
# The stack of "Add the Eagle3Speculator module for speculative decoding" includes "Add a
# weight-stationary INT4 GEMM for small M"; the page names nothing more.  The format read
# here: per output row, 4-bit codes two to a byte (in-index 2j in the low nibble of byte
# j, 2j + 1 in the high one) and, for each group of 128 in-indices, a bf16 (scale, zero)
# pair stored as one uint32 (scale in the low half); w = scale * (code - 8) + zero.

INT4_GROUP = 128


def dequantize_int4(codes, sz, in_dim: int) -> np.ndarray:
    """float64 [out, in] of INT4 codes uint8 [out, in / 2] and (scale, zero) uint32 rows."""
    c = np.asarray(codes, dtype=np.uint8)
    q = np.empty((c.shape[0], in_dim), dtype=np.float64)
    q[:, 0::2] = c & 15
    q[:, 1::2] = c >> 4
    groups = in_dim // INT4_GROUP
    pairs = np.asarray(sz, dtype=np.uint32)[:, :groups]
    scale = widen_bf16((pairs & 0xFFFF).astype(np.uint16))
    zero = widen_bf16((pairs >> 16).astype(np.uint16))
    g = np.arange(in_dim) // INT4_GROUP
    return scale[:, g] * (q - 8.0) + zero[:, g]


def store_k(x, kv_format: str) -> np.ndarray:
    """Value of a K vector as the cache holds it (float64 of the stored form)."""
    if kv_format == "bf16":
        return round_bf16(x)
    return dequantize_q8_0(*quantize_q8_0(np.asarray(x, dtype=np.float64).astype(np.float32))).astype(np.float64)


def store_v(x, kv_format: str) -> np.ndarray:
    """Value of a V vector as the cache holds it (float64 of the stored form)."""
    if kv_format == "bf16":
        return round_bf16(x)
    return dequantize_q5_1(*quantize_q5_1(np.asarray(x, dtype=np.float64).astype(np.float32))).astype(np.float64)


# --------------------------------------------------------------------------- drafter

class Drafter:
    """float64 view of the drafter weights (one decoder layer + fc + lm_head + d2t)."""

    def __init__(self, geom, bits: dict, d2t, kv_format: str = "bf16",
                 norm_before_residual: bool = False, int4: dict | None = None):
        """norm_before_residual: the checkpoint flag of "memra_engine/eagle.rs" (module
        doc, false for its checkpoint, whose attention residual is the pre-norm g); when
        true the residual is the normed RMSNorm(g) * hidden_norm instead."""
        if kv_format not in KV_FORMATS:
            raise ValueError(f"kv_format must be one of {KV_FORMATS}")
        if kv_format != "bf16" and geom.head_dim % QK:
            raise ValueError("quantized KV needs head_dim % 32 == 0")
        self.geom = geom
        self.kv_format = kv_format
        self.norm_before_residual = bool(norm_before_residual)
        self.w = {name: widen_bf16(b) for name, b in bits.items() if name != "embed"}
        for name, (codes, sz) in (int4 or {}).items():  # INT4 projections, dequantized
            self.w[name] = dequantize_int4(codes, sz, 2 * codes.shape[1])
        self._embed_bits = bits["embed"]
        self.d2t = np.asarray(d2t, dtype=np.int64)

    def embed(self, tok: int) -> np.ndarray:
        """Row of the target-vocab embedding table (EAGLE-3 shares the target's)."""
        return widen_bf16(self._embed_bits[int(tok)])

    def d2t_map(self, draft_id: int) -> int:
        """target_id = draft_id + d2t[draft_id] ("memra_engine/eagle.rs", ``d2t_map``)."""
        return int(draft_id + self.d2t[draft_id])


def encode(dr: Drafter, aux_bits) -> np.ndarray:
    """g = fc . concat(aux_0, aux_1, aux_2) for every leading index of aux [..., 3, n]
    ("memra_engine/eagle.rs", ``Eagle3Draft::encode``; aux in ascending-layer order)."""
    a = widen_bf16(aux_bits)
    cat = a.reshape(a.shape[:-2] + (a.shape[-2] * a.shape[-1],))
    return cat @ dr.w["fc"].T


def layer_input(dr: Drafter, tok: int, g: np.ndarray) -> np.ndarray:
    """cat = [RMSNorm(embed(tok), input_layernorm) ; RMSNorm(g, hidden_norm)]  [2n]."""
    eps = dr.geom.rms_eps
    e_n = rms_norm(dr.embed(tok), dr.w["in_norm"], eps)
    g_n = rms_norm(np.asarray(g, dtype=np.float64), dr.w["hidden_norm"], eps)
    return np.concatenate([e_n, g_n])


def kv_projection(dr: Drafter, tok: int, g: np.ndarray, pos: int):
    """K (after RoPE) and V of the pair (g, tok) at position pos before storage, float64
    [H_kv, d] each ("memra_engine/eagle.rs", Op-sequence: k/v projections of the
    concatenated normed inputs, RoPE on k).  A one-layer drafter's KV at a position depends
    on nothing else."""
    geo = dr.geom
    cat = layer_input(dr, tok, g)
    k = (dr.w["k"] @ cat).reshape(geo.n_head_kv, geo.head_dim)
    v = (dr.w["v"] @ cat).reshape(geo.n_head_kv, geo.head_dim)
    return rope_neox(k, pos, geo.rope_dims, geo.rope_theta), v


def kv_entry(dr: Drafter, tok: int, g: np.ndarray, pos: int):
    """kv_projection as the cache stores it (bf16, or the q8_0 / q5_1 blocks)."""
    k, v = kv_projection(dr, tok, g, pos)
    return store_k(k, dr.kv_format), store_v(v, dr.kv_format)


def kv_projections(dr: Drafter, toks, gs: np.ndarray, positions):
    """kv_projection for many pairs at once: the same definition with the projections of
    all pairs done as one matrix product (rows are independent; a library matmul step)."""
    geo = dr.geom
    eps = geo.rms_eps
    toks = np.asarray(toks)
    e = np.stack([dr.embed(t) for t in toks])
    cat = np.concatenate([rms_norm(e, dr.w["in_norm"], eps),
                          rms_norm(np.asarray(gs, dtype=np.float64), dr.w["hidden_norm"], eps)], axis=1)
    k = (cat @ dr.w["k"].T).reshape(len(toks), geo.n_head_kv, geo.head_dim)
    v = (cat @ dr.w["v"].T).reshape(len(toks), geo.n_head_kv, geo.head_dim)
    k = np.stack([rope_neox(k[i], int(p), geo.rope_dims, geo.rope_theta)
                  for i, p in enumerate(positions)]) if len(toks) else k
    return k, v


def kv_entries(dr: Drafter, toks, gs: np.ndarray, positions):
    """kv_entry for many pairs at once (kv_projections, then storage)."""
    k, v = kv_projections(dr, toks, gs, positions)
    return store_k(k, dr.kv_format), store_v(v, dr.kv_format)


@dataclass
class StepOut:
    logits: np.ndarray      # [draft_vocab]
    g_next: np.ndarray      # gsum, the pre-norm residual fed back as the next g
    k: np.ndarray           # [H_kv, d] stored form of the entry appended at pos
    v: np.ndarray
    draft_id: int
    target_id: int
    x1: np.ndarray          # o_proj output + residual
    attn: np.ndarray        # attention output [H * d]
    k_raw: np.ndarray = None  # this step's k (after RoPE) and v before storage
    v_raw: np.ndarray = None


def layer_after_attention(dr: Drafter, g: np.ndarray, attn: np.ndarray):
    """o_proj + residual (pre-norm g), post-attention RMSNorm, SwiGLU MLP, fused-add
    residual, final RMSNorm and lm_head ("memra_engine/eagle.rs", Op-sequence)."""
    w, eps = dr.w, dr.geom.rms_eps
    res = rms_norm(g, w["hidden_norm"], eps) if dr.norm_before_residual else g
    x1 = w["o"] @ attn + res
    z = rms_norm(x1, w["post_norm"], eps)
    act = silu(w["gate"] @ z) * (w["up"] @ z)
    gsum = w["down"] @ act + x1
    logits = w["lm_head"] @ rms_norm(gsum, w["final_norm"], eps)
    return x1, gsum, logits


def draft_step(dr: Drafter, prev_tok: int, g: np.ndarray, k_cache: np.ndarray,
               v_cache: np.ndarray, pos: int, new_kv=None) -> StepOut:
    """One T=1 draft step at position pos over a cache holding positions 0..pos-1
    ("memra_engine/eagle.rs", Op-sequence and ``draft_token`` / ``attn``).

    new_kv: optional (k, v) stored form to append at pos instead of this step's own.
    Where a stored form is decided by rounding (a quantization code on a boundary) more
    than one form is valid; a caller can evaluate the step on the form another
    implementation stored, after checking it against k_raw / v_raw."""
    geo = dr.geom
    if k_cache.shape[0] != pos:
        raise ValueError("cache must hold exactly the positions before pos")
    g = np.asarray(g, dtype=np.float64)
    cat = layer_input(dr, prev_tok, g)
    q = (dr.w["q"] @ cat).reshape(geo.n_head, geo.head_dim)
    q = rope_neox(q, pos, geo.rope_dims, geo.rope_theta)
    k_raw, v_raw = kv_projection(dr, prev_tok, g, pos)
    if new_kv is None:
        k_new, v_new = store_k(k_raw, dr.kv_format), store_v(v_raw, dr.kv_format)
    else:
        k_new, v_new = (np.asarray(x, dtype=np.float64) for x in new_kv)
    k_all = np.concatenate([k_cache, k_new[None]], axis=0)
    v_all = np.concatenate([v_cache, v_new[None]], axis=0)
    attn = gqa_attention(q, k_all, v_all).reshape(-1)
    x1, gsum, logits = layer_after_attention(dr, g, attn)
    did = argmax_first(logits)
    return StepOut(logits, gsum, k_new, v_new, did, dr.d2t_map(did), x1, attn, k_raw, v_raw)


# ---------------------------------------------------------------- sequence state

@dataclass
class SeqState:
    """Committed drafter state of one sequence."""
    k: np.ndarray           # [L, H_kv, d] stored form (bf16-valued or quantized blocks)
    v: np.ndarray
    g: np.ndarray           # boundary feature fc . a_{N-1}   [n]
    tok: int                # boundary token t_N (target id)
    k_raw: np.ndarray = None  # [L, H_kv, d] the same entries before storage (float64)
    v_raw: np.ndarray = None

    @property
    def kv_len(self) -> int:
        return int(self.k.shape[0])

    def copy(self) -> "SeqState":
        return SeqState(self.k.copy(), self.v.copy(), self.g.copy(), int(self.tok),
                        None if self.k_raw is None else self.k_raw.copy(),
                        None if self.v_raw is None else self.v_raw.copy())


def _empty_kv(geo):
    return np.zeros((0, geo.n_head_kv, geo.head_dim), dtype=np.float64)


def prefill(dr: Drafter, tokens, next_tok: int, aux_bits) -> SeqState:
    """Teacher-forced prefill from a prompt t_0..t_{P-1}, its target features
    a_0..a_{P-1} and the target's greedy next token t_P: writes the pairs
    (fc a_p, t_{p+1}) at positions p = 0..P-2 and sets the boundary (fc a_{P-1}, t_P)
    ("feat(eagle3) ... drafter forward pass", PR body: prefill_prompt; "Add the
    Eagle3Speculator module", PR body: hidden state t paired with token t + 1)."""
    tokens = np.asarray(tokens)
    n_prompt = tokens.shape[0]
    if n_prompt < 1:
        raise ValueError("empty prompt")
    genc = encode(dr, aux_bits)
    geo = dr.geom
    if n_prompt > 1:
        k_raw, v_raw = kv_projections(dr, tokens[1:n_prompt], genc[:n_prompt - 1],
                                      np.arange(n_prompt - 1))
    else:
        k_raw, v_raw = _empty_kv(geo), _empty_kv(geo)
    return SeqState(store_k(k_raw, dr.kv_format), store_v(v_raw, dr.kv_format),
                    genc[n_prompt - 1].copy(), int(next_tok), k_raw, v_raw)


def plan_gamma(kv_len: int, gamma: int, max_cache_len: int, shrink: bool) -> int:
    """Chain length allowed at committed length kv_len.  A fully accepted round commits
    gamma + 1 entries, so kv_len + gamma + 1 must fit in max_cache_len; otherwise the
    request is refused, or gamma shrinks to max_cache_len - kv_len - 1 when asked
    (review comment on "feat(eagle3) ... drafter forward pass": start 97, k 3, max 100
    drafts but overflows the rebuild).  A shrunk gamma below 1 is refused."""
    if gamma < 1:
        raise ValueError("gamma must be >= 1")
    if kv_len + gamma + 1 <= max_cache_len:
        return gamma
    if not shrink:
        raise CapacityError(f"kv_len {kv_len} + gamma {gamma} + 1 > {max_cache_len}")
    g_eff = max_cache_len - kv_len - 1
    if g_eff < 1:
        raise CapacityError(f"no room for a draft at kv_len {kv_len}")
    return g_eff


@dataclass
class ChainOut:
    draft_tok: list          # target ids d_1..d_gamma
    draft_id: list           # draft-vocab ids
    logits: list             # per step [draft_vocab]
    g: list                  # per step g_next
    spec_k: np.ndarray       # [gamma, H_kv, d] entries written at L..L+gamma-1
    spec_v: np.ndarray
    steps: list = field(default_factory=list)


def draft_chain(dr: Drafter, st: SeqState, gamma: int, stepper=None) -> ChainOut:
    """gamma autoregressive draft steps from the boundary (g, tok) at positions
    L..L+gamma-1.  Step j > 0 uses the previous step's target id and g_next
    ("memra_engine/eagle.rs", ``generate_spec_eagle`` step 2; "feat(eagle3) ...",
    PR body: draft_chain).  The committed state is not modified: the speculative
    entries are returned separately, which is what the rewind restores.
    ``stepper(j, step_out)`` may return a different token to feed the next step (used
    to follow another implementation's choice where two logits are nearly tied)."""
    k_all, v_all = st.k.copy(), st.v.copy()
    g, prev = st.g.copy(), int(st.tok)
    out = ChainOut([], [], [], [], None, None)
    base = st.kv_len
    for j in range(gamma):
        so = draft_step(dr, prev, g, k_all, v_all, base + j)
        k_all = np.concatenate([k_all, so.k[None]], axis=0)
        v_all = np.concatenate([v_all, so.v[None]], axis=0)
        out.draft_tok.append(so.target_id)
        out.draft_id.append(so.draft_id)
        out.logits.append(so.logits)
        out.g.append(so.g_next)
        out.steps.append(so)
        nxt = so.target_id
        if stepper is not None:
            nxt = stepper(j, so)
        prev, g = int(nxt), so.g_next
    out.spec_k, out.spec_v = k_all[base:], v_all[base:]
    return out


def draft_chain_stateless(dr: Drafter, committed_pairs, boundary_g, boundary_tok,
                          gamma: int) -> ChainOut:
    """Same chain with no cache: at every step all K/V are recomputed from the pair
    list (tok, g, position) -- the "cached draft chain matching the stateless
    recompute" check of "Add the Eagle3Speculator module", PR body."""
    geo = dr.geom
    pairs = list(committed_pairs)
    base = len(pairs)
    g, prev = np.asarray(boundary_g, dtype=np.float64), int(boundary_tok)
    out = ChainOut([], [], [], [], None, None)
    for j in range(gamma):
        pos = base + j
        spec_pairs = pairs + [(prev, g, pos)]
        ks, vs = zip(*[kv_entry(dr, t, gg, p) for (t, gg, p) in spec_pairs])
        k_all, v_all = np.stack(ks), np.stack(vs)
        cat = layer_input(dr, prev, g)
        q = rope_neox((dr.w["q"] @ cat).reshape(geo.n_head, geo.head_dim), pos,
                      geo.rope_dims, geo.rope_theta)
        attn = gqa_attention(q, k_all, v_all).reshape(-1)
        _, gsum, logits = layer_after_attention(dr, g, attn)
        did = argmax_first(logits)
        tid = dr.d2t_map(did)
        out.draft_tok.append(tid)
        out.draft_id.append(did)
        out.logits.append(logits)
        out.g.append(gsum)
        pairs = spec_pairs
        prev, g = tid, gsum
    out.spec_k = np.stack([kv_entry(dr, t, gg, p)[0] for (t, gg, p) in pairs[base:]])
    out.spec_v = np.stack([kv_entry(dr, t, gg, p)[1] for (t, gg, p) in pairs[base:]])
    return out


def accept(draft_tok, target_pred, gamma_eff: int | None = None):
    """Greedy accept-prefix walk: n = number of leading i with target_pred[i] ==
    draft_tok[i] (stopping at the first mismatch); bonus = target_pred[n]
    ("memra_engine/eagle.rs", ``generate_spec_eagle`` step 4)."""
    g_eff = len(draft_tok) if gamma_eff is None else int(gamma_eff)
    n = 0
    while n < g_eff and int(target_pred[n]) == int(draft_tok[n]):
        n += 1
    return n, int(target_pred[n])


def target_verify(head_bits, norm_bits, hidden, eps: float, rows_per_block: int = 8192):
    """Greedy verify on the target side ("Add the Eagle3Speculator module for speculative
    decoding", PR body: target_verify returns, for every window position, the greedy
    argmax target id; "memra_engine/eagle.rs", ``generate_spec_eagle`` steps 3-4: argmax
    of the target logits at each position).  logits = head . (RMSNorm(h) * norm) for each
    hidden row h; ids = the first maximum of each row.  The head is widened to float64
    rows_per_block vocabulary rows at a time (memory only: each logit is its own dot
    product).  Returns (logits [..., V], ids [...] int64)."""
    h = np.asarray(hidden, dtype=np.float64)
    lead = h.shape[:-1]
    x = rms_norm(h.reshape(-1, h.shape[-1]), widen_bf16(norm_bits), eps)
    head = np.asarray(head_bits)
    V = head.shape[0]
    logits = np.empty((x.shape[0], V), dtype=np.float64)
    for r0 in range(0, V, rows_per_block):
        logits[:, r0:r0 + rows_per_block] = x @ widen_bf16(head[r0:r0 + rows_per_block]).T
    ids = np.array([argmax_first(l) for l in logits], dtype=np.int64)
    return logits.reshape(lead + (V,)), ids.reshape(lead)


def rebuild_after_verify(dr: Drafter, st: SeqState, n_acc: int, draft_tok, bonus: int,
                         verify_aux_bits) -> SeqState:
    """Teacher-force the accepted prefix into the committed KV and set the next
    boundary.  verify_aux[i] are the target features at positions N+i (i = 0..gamma).
    Pairs written at L+i, i = 0..n: i = 0 is the old boundary (g, tok); i >= 1 is
    (fc v_{i-1}, d_i).  New kv_len L+n+1; new boundary (fc v_n, bonus)
    ("feat(eagle3) ...", PR body: rebuild_after_verify; "Add the Eagle3Speculator
    module", PR body: reseed from verify's features paired with the corrected token)."""
    L = st.kv_len
    venc = encode(dr, np.asarray(verify_aux_bits)[: n_acc + 1])
    pairs = [(int(st.tok), st.g)] + [(int(draft_tok[i - 1]), venc[i - 1])
                                     for i in range(1, n_acc + 1)]
    kr, vr = zip(*[kv_projection(dr, t, gg, L + i) for i, (t, gg) in enumerate(pairs)])
    kr, vr = np.stack(kr), np.stack(vr)
    k_raw = None if st.k_raw is None else np.concatenate([st.k_raw, kr])
    v_raw = None if st.v_raw is None else np.concatenate([st.v_raw, vr])
    return SeqState(np.concatenate([st.k, store_k(kr, dr.kv_format)]),
                    np.concatenate([st.v, store_v(vr, dr.kv_format)]),
                    venc[n_acc].copy(), int(bonus), k_raw, v_raw)
