"""Pins of the oracle's quantized drafter KV (q8_0 keys, q5_1 values), CPU only.

The page ("memra_engine/eagle.rs", Eagle3Scratch) fixes the formats' names, the 32-value
blocks and their sizes (34 and 24 bytes; head_dim % 32 == 0).  These tests tie the
oracle's encoders to those facts, to hand-written block bytes (tests/golden), to closed
forms (values on the grid come back exactly; the error of a code is at most half a step)
and to brute force (every code is the nearest representable value)."""
import os

import numpy as np
import pytest

from eagle_speculative_decode_gb300 import synth
from oracle import eagle3_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_quant_blocks.txt")


def test_block_sizes_follow_the_page():
    # 34 / 24 bytes per 32 values; a 256-wide head token is 8 blocks: 272 + 192 bytes
    assert O.QK == 32 and O.Q8_0_BLOCK_BYTES == 34 and O.Q5_1_BLOCK_BYTES == 24
    x = np.random.default_rng(0).standard_normal(256).astype(np.float32)
    assert O.pack_q8_0(*O.quantize_q8_0(x)).size == 272
    assert O.pack_q5_1(*O.quantize_q5_1(x)).size == 192
    with pytest.raises(ValueError):
        O.quantize_q8_0(np.zeros(48, np.float32))


def test_golden_block_bytes():
    n = 0
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        fmt, d, m, codes, exp = line.split()
        c = np.array([int(x) for x in codes.split(",")])
        d16 = np.array(int(d, 16), dtype=np.uint16).view(np.float16)
        if fmt == "q8_0":
            got = O.pack_q8_0(d16, c.astype(np.int8))
            assert got.tobytes().hex() == exp
            d2, c2 = O.unpack_q8_0(got)
            assert d2 == d16 and np.array_equal(c2, c)
        else:
            m16 = np.array(int(m, 16), dtype=np.uint16).view(np.float16)
            got = O.pack_q5_1(d16, m16, c.astype(np.uint8))
            assert got.tobytes().hex() == exp
            d2, m2, c2 = O.unpack_q5_1(got)
            assert d2 == d16 and m2 == m16 and np.array_equal(c2, c)
        n += 1
    assert n == 4


def test_q8_0_grid_values_round_trip_exactly():
    rng = np.random.default_rng(1)
    codes = rng.integers(-127, 128, size=(5, 32))
    codes[:, 0] = 127                      # the block maximum sits on the top code
    d = np.float32(2.0 ** -6)              # exact in fp16; amax / 127 = d exactly
    x = (codes * d).astype(np.float32)
    d16, q = O.quantize_q8_0(x.reshape(-1))
    assert np.all(d16.astype(np.float32) == d)
    assert np.array_equal(q.reshape(5, 32), codes)
    assert np.array_equal(O.dequantize_q8_0(d16, q), x.reshape(-1))


def test_q5_1_grid_values_round_trip_exactly():
    rng = np.random.default_rng(2)
    codes = rng.integers(0, 32, size=(4, 32))
    codes[:, 0], codes[:, 1] = 0, 31       # min and max on the end codes
    d, m = np.float32(0.125), np.float32(-1.5)
    x = (codes * d + m).astype(np.float32)
    d16, m16, q = O.quantize_q5_1(x.reshape(-1))
    assert np.all(d16.astype(np.float32) == d) and np.all(m16.astype(np.float32) == m)
    assert np.array_equal(q.reshape(4, 32), codes)
    assert np.array_equal(O.dequantize_q5_1(d16, m16, q), x.reshape(-1))


def test_codes_are_the_nearest_representable_values():
    """Brute force over every code: no other code is strictly closer (ties may go either
    way only at exact half steps)."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((64, 32)) * rng.uniform(0.01, 10, size=(64, 1))).astype(np.float32)
    d16, q = O.quantize_q8_0(x.reshape(-1))
    d = d16.astype(np.float64)[:, None]
    grid = d[:, :, None] * np.arange(-127, 128)[None, None, :]          # [blocks, 1, codes]
    err_all = np.abs(x.astype(np.float64)[:, :, None] - grid)
    err_q = np.abs(x.astype(np.float64) - d * q.astype(np.float64))
    assert np.all(err_q <= err_all.min(axis=-1) + 1e-12 * np.abs(x))
    assert np.all(err_q <= d / 2 * (1 + 1e-6))

    d16, m16, q = O.quantize_q5_1(x.reshape(-1))
    d = d16.astype(np.float64)[:, None]
    m = m16.astype(np.float64)[:, None]
    grid = d[:, :, None] * np.arange(32)[None, None, :] + m[:, :, None]
    err_all = np.abs(x.astype(np.float64)[:, :, None] - grid)
    err_q = np.abs(x.astype(np.float64) - (d * q.astype(np.float64) + m))
    assert np.all(err_q <= err_all.min(axis=-1) + 1e-6 * np.abs(x) + 1e-7)


def test_degenerate_blocks():
    z = np.zeros(64, np.float32)
    d16, q = O.quantize_q8_0(z)
    assert np.all(d16 == 0) and np.all(q == 0) and np.all(O.dequantize_q8_0(d16, q) == 0)
    c = np.full(32, 0.3, np.float32)       # constant block: no range for q5_1
    d16, m16, q = O.quantize_q5_1(c)
    assert np.all(d16 == 0) and np.all(q == 0)
    assert np.all(O.dequantize_q5_1(d16, m16, q) == np.float32(np.float16(0.3)))


def test_q8_0_is_odd_symmetric():
    x = np.random.default_rng(4).standard_normal(128).astype(np.float32)
    d1, q1 = O.quantize_q8_0(x)
    d2, q2 = O.quantize_q8_0(-x)
    assert np.array_equal(d1, d2) and np.array_equal(q1, -q2)


def test_store_paths_and_cache_equivalences_under_quantized_kv():
    """kv_entries (batched) equals kv_entry (one by one) and the cached chain equals the
    stateless recompute when the cache holds quantized blocks; stored values are the
    quantizer's round trip of the float32 k / v."""
    g = synth.TINY
    wts = synth.make_weights(g, seed=9)
    dr = O.Drafter(g, wts.bits, wts.d2t, kv_format="q8_0/q5_1")
    toks = synth.make_tokens(6, g, seed=10)
    gs = O.encode(dr, synth.make_aux((6,), g, seed=11))
    kb, vb = O.kv_entries(dr, toks, gs, np.arange(6))
    for i in range(6):
        k1, v1 = O.kv_entry(dr, int(toks[i]), gs[i], i)
        assert np.array_equal(k1, kb[i]) and np.array_equal(v1, vb[i])
    # every stored K block is on its own q8_0 grid; V on its q5_1 grid
    for row in kb.reshape(-1, 32):
        d16, q = O.quantize_q8_0(row.astype(np.float32))
        assert np.array_equal(O.dequantize_q8_0(d16, q), row.astype(np.float32))
    ptoks = synth.make_tokens(10, g, seed=12)
    aux = synth.make_aux((9,), g, seed=13)
    st = O.prefill(dr, ptoks[:9], int(ptoks[9]), aux)
    genc = O.encode(dr, aux)
    pairs = [(int(ptoks[p + 1]), genc[p], p) for p in range(8)]
    out = O.draft_chain(dr, st, 3)
    ref = O.draft_chain_stateless(dr, pairs, st.g, st.tok, 3)
    assert out.draft_tok == ref.draft_tok
    assert np.array_equal(out.spec_k, ref.spec_k) and np.array_equal(out.spec_v, ref.spec_v)


def test_quantized_format_needs_blocks_of_32():
    import dataclasses
    g = dataclasses.replace(synth.TINY, head_dim=48)
    wts = synth.make_weights(synth.TINY, seed=0)
    with pytest.raises(ValueError):
        O.Drafter(g, wts.bits, wts.d2t, kv_format="q8_0/q5_1")




def test_parity_decoder_reads_packed_rows():
    """The parity tests decode the GPU's pool rows with the oracle's unpackers: packed
    rows of several blocks decode to the oracle's stored values."""
    from parity import kv_values
    x = np.random.default_rng(5).standard_normal((3, 2, 128))
    kraw = O.pack_q8_0(*O.quantize_q8_0(x.astype(np.float32))).reshape(3, 2, -1)
    vraw = O.pack_q5_1(*O.quantize_q5_1(x.astype(np.float32))).reshape(3, 2, -1)
    assert kraw.shape[-1] == 4 * 34 and vraw.shape[-1] == 4 * 24
    assert np.array_equal(kv_values(kraw, "q8_0/q5_1", "k"), O.store_k(x, "q8_0/q5_1"))
    assert np.array_equal(kv_values(vraw, "q8_0/q5_1", "v"), O.store_v(x, "q8_0/q5_1"))


def test_validity_check_accepts_own_encoding_and_rejects_planted_errors():
    """assert_quant_valid (the GPU parity bar for stored blocks) is not vacuous: the
    oracle's own bytes pass; a code moved by one away from a boundary, a scale two fp16
    steps off, or a wrong minimum fail; at an exact code boundary either neighbour passes."""
    from parity import assert_quant_valid
    rng = np.random.default_rng(6)
    x = rng.standard_normal((8, 64))
    kb = O.pack_q8_0(*O.quantize_q8_0(x.astype(np.float32))).reshape(8, -1)
    vb = O.pack_q5_1(*O.quantize_q5_1(x.astype(np.float32))).reshape(8, -1)
    assert_quant_valid(kb, x, "k", "own K")
    assert_quant_valid(vb, x, "v", "own V")

    def planted(blocks, which, fn):
        b = blocks.copy()
        fn(b.reshape(-1, 34 if which == "k" else 24))
        with pytest.raises(AssertionError):
            assert_quant_valid(b, x, which, "planted")

    d16, _ = O.quantize_q8_0(x.astype(np.float32))
    t = x.reshape(-1, 32) / d16.astype(np.float64).reshape(-1)[:, None]
    blk, i = np.argwhere((np.abs(t - np.rint(t)) < 0.3) & (np.abs(t) < 120))[0]

    def bump_code(flat):
        flat[blk, 2 + i] = (int(flat[blk, 2 + i]) + 1) & 0xff

    def bump_scale(flat):
        h = int(flat[3, 0:2].view(np.uint16)[0])
        flat[3, 0:2] = np.array([h + 2], dtype=np.uint16).view(np.uint8)

    def bump_min(flat):
        h = int(flat[5, 2:4].view(np.uint16)[0])
        flat[5, 2:4] = np.array([h + 3], dtype=np.uint16).view(np.uint8)

    planted(kb, "k", bump_code)
    planted(kb, "k", bump_scale)
    planted(vb, "v", bump_min)
    # a value exactly half-way between two q8_0 codes: either neighbour is valid
    y = np.zeros(32)
    y[0] = 127.0 * 0.25           # scale 0.25 exactly
    y[1] = 10.5 * 0.25            # on the boundary between codes 10 and 11
    for c in (10, 11):
        codes = np.zeros(32, np.int8)
        codes[0], codes[1] = 127, c
        assert_quant_valid(O.pack_q8_0(np.float16(0.25), codes), y, "k", f"tie code {c}")
    codes[1] = 12
    with pytest.raises(AssertionError):
        assert_quant_valid(O.pack_q8_0(np.float16(0.25), codes), y, "k", "two codes off")


def test_step_on_its_own_stored_entry_and_raw_state():
    """draft_step given its own stored entry as new_kv is the same step; prefill and
    rebuild keep the unstored k / v whose storage is the state's KV."""
    g = synth.TINY
    wts = synth.make_weights(g, seed=9)
    dr = O.Drafter(g, wts.bits, wts.d2t, kv_format="q8_0/q5_1")
    ptoks = synth.make_tokens(12, g, seed=14)
    aux = synth.make_aux((11,), g, seed=15)
    st = O.prefill(dr, ptoks[:11], int(ptoks[11]), aux)
    assert np.array_equal(O.store_k(st.k_raw, dr.kv_format), st.k)
    assert np.array_equal(O.store_v(st.v_raw, dr.kv_format), st.v)
    a = O.draft_step(dr, st.tok, st.g, st.k, st.v, st.kv_len)
    b = O.draft_step(dr, st.tok, st.g, st.k, st.v, st.kv_len, new_kv=(a.k, a.v))
    assert np.array_equal(a.logits, b.logits) and np.array_equal(a.g_next, b.g_next)
    assert np.array_equal(O.store_k(a.k_raw, dr.kv_format), a.k)
    # a different appended entry changes the step (the override is used)
    c = O.draft_step(dr, st.tok, st.g, st.k, st.v, st.kv_len, new_kv=(a.k, a.v * 0.5))
    assert not np.array_equal(a.g_next, c.g_next)
    vaux = synth.make_aux((4,), g, seed=16)
    st2 = O.rebuild_after_verify(dr, st, 2, [int(ptoks[1]), int(ptoks[2]), int(ptoks[3])], 7, vaux)
    assert st2.kv_len == st.kv_len + 3
    assert np.array_equal(O.store_k(st2.k_raw, dr.kv_format), st2.k)
    assert np.array_equal(O.store_v(st2.v_raw, dr.kv_format), st2.v)
