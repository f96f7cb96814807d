"""Seeded synthetic inputs for the EAGLE-3 drafter draft round.

Everything here is random data or bookkeeping about random data: drafter weights,
auxiliary target features, prompt tokens, page tables and imposed accept patterns.
None of the drafter's arithmetic lives in this module.  The CUDA path and the CPU
oracle both take their inputs from these functions, so they see identical bits.

Random numbers come from numpy's SFC64 generator, one independent stream per
(seed, tensor, 4 Mi-element chunk), so results do not depend on the thread count
and any tensor can be regenerated on its own.  bf16 values are produced by
round-to-nearest-even of float32 samples and are returned as uint16 bit patterns.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_CHUNK = 1 << 22


@dataclass(frozen=True)
class Geometry:
    """Drafter geometry: one Llama-style decoder layer fed by an fc encoder."""
    n_embd: int
    n_head: int
    n_head_kv: int
    head_dim: int
    rope_dims: int
    rope_theta: float
    rms_eps: float
    n_ff: int
    draft_vocab: int
    target_vocab: int
    n_aux: int = 3

    @property
    def q_rows(self) -> int:
        return self.n_head * self.head_dim

    @property
    def kv_rows(self) -> int:
        return self.n_head_kv * self.head_dim


# Small drafter used for exhaustive parity: n_embd 256, 4 q heads / 1 kv head of 64,
# RoPE on the first 16 dims at theta 1e7, n_ff 768, draft vocab 1024 -> target 4096.
TINY = Geometry(n_embd=256, n_head=4, n_head_kv=1, head_dim=64, rope_dims=16,
                rope_theta=1e7, rms_eps=1e-6, n_ff=768, draft_vocab=1024,
                target_vocab=4096)

# Drafter of the eagle.rs page (memra_engine, tensor list and config fixture):
# hidden 4096, 16 q / 4 kv heads of 256, partial RoPE 64/256 at theta 1e7,
# n_ff 12288, draft vocab 32000 mapped into a 248320-entry target vocab.
FULL = Geometry(n_embd=4096, n_head=16, n_head_kv=4, head_dim=256, rope_dims=64,
                rope_theta=1e7, rms_eps=1e-6, n_ff=12288, draft_vocab=32000,
                target_vocab=248320)

# Small drafter whose q / k / v blocks are whole 128-row tiles (8:2 GQA of 64-wide
# heads), so that batched projections take the tensor-core GEMM at test sizes.
SMALL = Geometry(n_embd=256, n_head=8, n_head_kv=2, head_dim=64, rope_dims=16,
                 rope_theta=1e7, rms_eps=1e-6, n_ff=768, draft_vocab=1024,
                 target_vocab=4096)

GEOMETRIES = {"tiny": TINY, "small": SMALL, "full": FULL}

# Tensor order fixes the per-tensor sub-seed.
WEIGHT_NAMES = ("fc", "in_norm", "hidden_norm", "q", "k", "v", "o", "post_norm",
                "gate", "up", "down", "final_norm", "lm_head", "embed")
NORM_NAMES = ("in_norm", "hidden_norm", "post_norm", "final_norm")


def weight_shapes(geom: Geometry) -> dict[str, tuple[int, ...]]:
    """[out, in] row-major shapes of every drafter tensor (PyTorch Linear layout)."""
    n, f = geom.n_embd, geom.n_ff
    return {
        "fc": (n, geom.n_aux * n),
        "in_norm": (n,),
        "hidden_norm": (n,),
        "q": (geom.q_rows, 2 * n),
        "k": (geom.kv_rows, 2 * n),
        "v": (geom.kv_rows, 2 * n),
        "o": (n, geom.q_rows),
        "post_norm": (n,),
        "gate": (f, n),
        "up": (f, n),
        "down": (n, f),
        "final_norm": (n,),
        "lm_head": (geom.draft_vocab, n),
        "embed": (geom.target_vocab, n),
    }


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 samples to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def _stream(seed: int, key: tuple[int, ...]) -> np.random.Generator:
    return np.random.Generator(np.random.SFC64(np.random.SeedSequence(seed, spawn_key=key)))


def normal_bf16(shape, seed: int, key: tuple[int, ...], std: float = 1.0,
                mean: float = 0.0, threads: int | None = None) -> np.ndarray:
    """bf16 bits of mean + std * N(0, 1), generated chunk-parallel and reproducibly."""
    total = int(np.prod(shape))
    out = np.empty(total, dtype=np.uint16)
    n_chunks = (total + _CHUNK - 1) // _CHUNK
    std32, mean32 = np.float32(std), np.float32(mean)

    def fill(c: int) -> None:
        lo, hi = c * _CHUNK, min(total, (c + 1) * _CHUNK)
        z = _stream(seed, key + (c,)).standard_normal(hi - lo, dtype=np.float32)
        if std32 != np.float32(1.0):
            z *= std32
        if mean32 != np.float32(0.0):
            z += mean32
        out[lo:hi] = f32_to_bf16_bits(z)

    workers = threads or min(32, os.cpu_count() or 1)
    if n_chunks <= 1 or workers <= 1:
        for c in range(n_chunks):
            fill(c)
    else:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out.reshape(shape)


def make_d2t(geom: Geometry, seed: int) -> np.ndarray:
    """Draft-to-target offsets: a sorted random draft_vocab-subset S of the target
    vocab, d2t[i] = S[i] - i (int64), so target ids are distinct and increasing."""
    rng = _stream(seed, (100,))
    s = np.sort(rng.choice(geom.target_vocab, size=geom.draft_vocab, replace=False))
    return (s.astype(np.int64) - np.arange(geom.draft_vocab, dtype=np.int64))


@dataclass
class DrafterWeights:
    geom: Geometry
    bits: dict[str, np.ndarray]          # name -> uint16 bf16 bits, [out, in] row-major
    d2t: np.ndarray                      # int64 [draft_vocab]
    seed: int = 0
    gains: str = "one_plus"
    extra: dict = field(default_factory=dict)
    # INT4 projections: name -> (codes uint8 [out, in / 2], sz uint32 [out, stride]) where
    # sz packs bf16 (scale, zero) as scale | zero << 16; `bits` then omits those names
    int4: dict | None = None


def make_weights(geom: Geometry, seed: int = 0, gains: str = "one_plus",
                 std: float = 0.02, skip: tuple[str, ...] = ()) -> DrafterWeights:
    """Seeded drafter weights.  Linear and embedding weights are N(0, std).  RMSNorm
    gains are 1 + N(0, std) ("one_plus") or literally N(0, std) ("literal")."""
    if gains not in ("one_plus", "literal"):
        raise ValueError(gains)
    shapes = weight_shapes(geom)
    bits: dict[str, np.ndarray] = {}
    for idx, name in enumerate(WEIGHT_NAMES):
        if name in skip:
            continue
        mean = 1.0 if (name in NORM_NAMES and gains == "one_plus") else 0.0
        bits[name] = normal_bf16(shapes[name], seed, (idx,), std=std, mean=mean)
    return DrafterWeights(geom, bits, make_d2t(geom, seed), seed, gains)


def make_target_head(geom: Geometry, seed: int, std: float = 0.02):
    """Synthetic target output head for the verify step: lm_head bf16 bits
    [target_vocab, n_embd] ~ N(0, std) and final-norm gains 1 + N(0, std)."""
    head = normal_bf16((geom.target_vocab, geom.n_embd), seed, (300,), std=std)
    norm = normal_bf16((geom.n_embd,), seed, (301,), std=std, mean=1.0)
    return head, norm


def make_hidden(shape_prefix: tuple[int, ...], geom: Geometry, seed: int,
                stream: int = 0) -> np.ndarray:
    """Synthetic target last hidden states: float32 (bf16-valued) N(0, 1), shape
    prefix + (n_embd,)."""
    bits = normal_bf16(tuple(shape_prefix) + (geom.n_embd,), seed, (400, stream))
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


INT4_NAMES = ("q", "k", "v", "o", "gate", "up", "down", "lm_head")
INT4_GROUP = 128


def int4_sz_stride(in_dim: int) -> int:
    """(scale, zero) pairs per INT4 row: in / 128 rounded up to a multiple of 4."""
    return (in_dim // INT4_GROUP + 3) // 4 * 4


def make_int4_weights(geom: Geometry, seed: int = 0, std: float = 0.02) -> DrafterWeights:
    """Seeded drafter with INT4 projections (a random-init INT4 model, not a quantized bf16
    one): codes uniform in 0..15; per 128-wide group a bf16 scale std / 4.6 * exp(0.2 N)
    (code - 8 has standard deviation about 4.6) and a bf16 zero scale / 2 + N(0, std / 10),
    which centres the weights (code - 8 has mean -1/2); padding pairs are zero.  fc, the
    norm gains and the embedding are bf16 as in make_weights."""
    base = make_weights(geom, seed, skip=INT4_NAMES, std=std)
    shapes = weight_shapes(geom)
    int4 = {}
    for idx, name in enumerate(INT4_NAMES):
        out_dim, in_dim = shapes[name]
        rng = _stream(seed, (500, idx))
        codes = rng.integers(0, 256, size=(out_dim, in_dim // 2), dtype=np.uint8)
        groups = in_dim // INT4_GROUP
        scale = (np.float32(std / 4.6) * np.exp(np.float32(0.2) * rng.standard_normal((out_dim, groups),
                                                                                     dtype=np.float32)))
        zero = np.float32(0.5) * scale + np.float32(std / 10) * rng.standard_normal((out_dim, groups),
                                                                                     dtype=np.float32)
        sz = np.zeros((out_dim, int4_sz_stride(in_dim)), dtype=np.uint32)
        sz[:, :groups] = f32_to_bf16_bits(scale).astype(np.uint32) | \
            (f32_to_bf16_bits(zero).astype(np.uint32) << np.uint32(16))
        int4[name] = (codes, sz)
    base.int4 = int4
    return base


def make_aux(shape_prefix: tuple[int, ...], geom: Geometry, seed: int,
             stream: int = 0) -> np.ndarray:
    """Auxiliary target features N(0, 1) in bf16, shape prefix + (n_aux, n_embd)."""
    return normal_bf16(tuple(shape_prefix) + (geom.n_aux, geom.n_embd), seed, (200, stream))


def make_tokens(shape, geom: Geometry, seed: int, stream: int = 0) -> np.ndarray:
    """Uniform target-vocab token ids (int32)."""
    return _stream(seed, (300, stream)).integers(0, geom.target_vocab, size=shape,
                                                 dtype=np.int64).astype(np.int32)


def ragged_lengths(batch: int, lo: int, hi: int, seed: int, stream: int = 0) -> np.ndarray:
    """Per-sequence lengths uniform in [lo, hi] (int32)."""
    return _stream(seed, (400, stream)).integers(lo, hi + 1, size=batch).astype(np.int32)


def page_table(batch: int, pages_per_seq: int, seed: int | None = None) -> np.ndarray:
    """Page table [batch, pages_per_seq] over a pool of batch*pages_per_seq pages.
    With a seed the physical pages are a random permutation (non-contiguous pages);
    without one they are laid out in order."""
    total = batch * pages_per_seq
    ids = np.arange(total, dtype=np.int32)
    if seed is not None:
        ids = _stream(seed, (500,)).permutation(total).astype(np.int32)
    return ids.reshape(batch, pages_per_seq)


def imposed_accept_lengths(batch: int, gamma: int, seed: int, stream: int = 0,
                           p_accept: float | None = None) -> np.ndarray:
    """Accept lengths n_b in [0, gamma]: uniform, or the run length of independent
    per-token accepts with probability p_accept (stopping at the first miss)."""
    rng = _stream(seed, (600, stream))
    if p_accept is None:
        return rng.integers(0, gamma + 1, size=batch).astype(np.int32)
    u = rng.random((batch, gamma))
    miss = u >= p_accept
    first = np.where(miss.any(axis=1), miss.argmax(axis=1), gamma)
    return first.astype(np.int32)


def impose_target_predictions(draft_tok: np.ndarray, n_acc: np.ndarray, geom: Geometry,
                              seed: int, stream: int = 0) -> np.ndarray:
    """Target predictions y[b, 0..gamma] that accept exactly n_acc[b] leading drafts:
    y[b, i] = draft[b, i] for i < n, y[b, n] a random id != draft[b, n] (when n < gamma),
    remaining entries random."""
    b_, g_ = draft_tok.shape
    rng = _stream(seed, (700, stream))
    y = rng.integers(0, geom.target_vocab, size=(b_, g_ + 1), dtype=np.int64).astype(np.int32)
    for b in range(b_):
        n = int(n_acc[b])
        y[b, :n] = draft_tok[b, :n]
        if n < g_ and y[b, n] == draft_tok[b, n]:
            y[b, n] = (int(draft_tok[b, n]) + 1) % geom.target_vocab
    return y
