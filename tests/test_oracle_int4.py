"""Pins of the oracle's INT4 drafter weights (CPU only): the format w = scale * (code - 8)
+ zero with 4-bit codes two to a byte (low nibble first) and one bf16 (scale, zero) pair
per 128 inputs, checked on hand-written bytes, group boundaries, ignored padding, and a
drafter whose INT4 weights equal a bf16 drafter's values (identical chains)."""
import numpy as np

from eagle_speculative_decode_gb300 import synth
from oracle import eagle3_oracle as O


def pair(scale_bits, zero_bits):
    return np.uint32(scale_bits | (zero_bits << 16))


def test_hand_written_row():
    # one row of 256 inputs: group 0 scale 2.0 (0x4000), zero 1.0 (0x3F80); group 1 scale
    # 0.5 (0x3F00), zero -3.0 (0xC040); the two pad pairs hold garbage
    codes = np.zeros((1, 128), np.uint8)
    codes[0, 0] = 0x4A          # k0 = 10, k1 = 4
    codes[0, 1] = 0xF0          # k2 = 0, k3 = 15
    codes[0, 2] = 0x88          # k4 = k5 = 8
    codes[0, 63] = 0x18         # k126 = 8, k127 = 1   (last pair of group 0)
    codes[0, 64] = 0x9F         # k128 = 15, k129 = 9  (first pair of group 1)
    codes[0, 127] = 0x07        # k254 = 7, k255 = 0
    sz = np.array([[pair(0x4000, 0x3F80), pair(0x3F00, 0xC040), 0xDEADBEEF, 0x7FC07FC0]], np.uint32)
    w = O.dequantize_int4(codes, sz, 256)
    want = {0: 2 * (10 - 8) + 1, 1: 2 * (4 - 8) + 1, 2: 2 * (0 - 8) + 1, 3: 2 * (15 - 8) + 1,
            4: 1.0, 5: 1.0, 126: 1.0, 127: 2 * (1 - 8) + 1,
            128: 0.5 * (15 - 8) - 3, 129: 0.5 * (9 - 8) - 3, 254: 0.5 * (7 - 8) - 3, 255: 0.5 * (0 - 8) - 3}
    for k, v in want.items():
        assert w[0, k] == v, (k, w[0, k], v)
    # every other code is 0: w = zero - 8 scale in its group
    assert w[0, 10] == 1.0 - 16 and w[0, 200] == -3.0 - 4
    assert np.all(np.isfinite(w))        # the NaN-pattern pad pair is never read


def test_code_eight_is_the_zero_point_and_the_grid():
    rng = np.random.default_rng(0)
    sz = synth.make_int4_weights(synth.TINY, seed=1).int4["o"][1]
    codes = np.full((sz.shape[0], 128), 0x88, np.uint8)
    w = O.dequantize_int4(codes, sz, 256)
    zero = O.widen_bf16((sz[:, :2] >> 16).astype(np.uint16))
    assert np.array_equal(w[:, :128], np.repeat(zero[:, :1], 128, axis=1))
    assert np.array_equal(w[:, 128:], np.repeat(zero[:, 1:2], 128, axis=1))
    c = rng.integers(0, 256, size=(4, 128), dtype=np.uint8)
    w = O.dequantize_int4(c, sz[:4], 256)
    scale = O.widen_bf16((sz[:4, :2] & 0xFFFF).astype(np.uint16))
    q = (w - np.repeat(zero[:4], 128, axis=1)) / np.repeat(scale, 128, axis=1) + 8
    assert np.allclose(q, np.rint(q), atol=1e-9) and q.min() >= 0 and q.max() <= 15


def test_synthetic_int4_statistics_and_padding():
    shapes = synth.weight_shapes(synth.FULL)
    assert [synth.int4_sz_stride(shapes[n][1]) for n in ("q", "o", "gate", "down", "lm_head")] == \
        [64, 32, 32, 96, 32]
    t = synth.make_int4_weights(synth.TINY, seed=2)
    c, s = t.int4["q"]               # in 512: 4 groups, stride 4
    assert s.shape[1] == 4
    c, s = t.int4["gate"]            # in 256: 2 groups padded to 4
    assert s.shape[1] == 4 and np.all(s[:, 2:] == 0)
    w = O.dequantize_int4(c, s, 256)
    assert 0.015 < float(np.std(w)) < 0.025
    assert "q" not in t.bits and "fc" in t.bits and "embed" in t.bits


def test_int4_drafter_equals_the_bf16_drafter_of_the_same_values():
    """Codes and pairs chosen so that every weight is exactly a bf16 value: a drafter given
    them as INT4 and one given the same values as bf16 bits draft the same chain."""
    g = synth.TINY
    base = synth.make_weights(g, seed=4)
    rng = np.random.default_rng(5)
    shapes = synth.weight_shapes(g)
    int4, bits = {}, dict(base.bits)
    for name in synth.INT4_NAMES:
        out_dim, in_dim = shapes[name]
        codes = rng.integers(0, 256, size=(out_dim, in_dim // 2), dtype=np.uint8)
        groups = in_dim // 128
        sz = np.zeros((out_dim, synth.int4_sz_stride(in_dim)), np.uint32)
        sz[:, :groups] = pair(0x3C00, 0xBB00)   # scale 2^-7, zero -2^-9: exact in bf16 sums
        int4[name] = (codes, sz)
        w = O.dequantize_int4(codes, sz, in_dim)
        bits[name] = synth.f32_to_bf16_bits(w.astype(np.float32))
        assert np.array_equal(O.widen_bf16(bits[name]), w)
    d_int4 = O.Drafter(g, {k: v for k, v in base.bits.items()}, base.d2t, int4=int4)
    d_bf16 = O.Drafter(g, bits, base.d2t)
    toks = synth.make_tokens(12, g, seed=6)
    aux = synth.make_aux((11,), g, seed=7)
    s1 = O.prefill(d_int4, toks[:11], int(toks[11]), aux)
    s2 = O.prefill(d_bf16, toks[:11], int(toks[11]), aux)
    c1, c2 = O.draft_chain(d_int4, s1, 4), O.draft_chain(d_bf16, s2, 4)
    assert c1.draft_tok == c2.draft_tok
    assert all(np.array_equal(a, b) for a, b in zip(c1.logits, c2.logits))
