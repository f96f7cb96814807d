"""Pins of the CPU oracle against closed forms, special cases and page-fixed values.

Each test fixes one fact that a plausible mistake in the oracle would break: a dropped
term, a wrong sign or index, a transposed operand, a swapped role, an off-by-one in the
position or pairing bookkeeping.  No expected value here is computed by re-calling the
oracle routine under test.
"""
import math
import os

import numpy as np
import pytest

from eagle_speculative_decode_gb300 import synth
from oracle import eagle3_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- helpers

def bits_exact(x) -> np.ndarray:
    """bf16 bits of values that bf16 represents exactly (asserted)."""
    x32 = np.asarray(x, dtype=np.float32)
    u = x32.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


MICRO = synth.Geometry(n_embd=8, n_head=2, n_head_kv=1, head_dim=4, rope_dims=2,
                       rope_theta=1e7, rms_eps=1e-6, n_ff=8, draft_vocab=8,
                       target_vocab=16)


def micro_drafter(**over):
    """Hand-built drafter on MICRO with exactly representable weights.  Defaults are
    zeros (so each test switches on only the paths it pins) and unit gains."""
    g = MICRO
    n, f = g.n_embd, g.n_ff
    w = {
        "fc": np.zeros((n, 3 * n)), "in_norm": np.ones(n), "hidden_norm": np.ones(n),
        "q": np.zeros((g.q_rows, 2 * n)), "k": np.zeros((g.kv_rows, 2 * n)),
        "v": np.zeros((g.kv_rows, 2 * n)), "o": np.zeros((n, g.q_rows)),
        "post_norm": np.ones(n), "gate": np.zeros((f, n)), "up": np.zeros((f, n)),
        "down": np.zeros((n, f)), "final_norm": np.ones(n),
        "lm_head": np.eye(g.draft_vocab, n), "embed": np.zeros((g.target_vocab, n)),
    }
    w.update(over)
    d2t = over.get("d2t", np.arange(g.draft_vocab, dtype=np.int64))  # id -> 2*id
    bits = {k: bits_exact(v) for k, v in w.items() if k != "d2t"}
    return O.Drafter(g, bits, d2t)


def random_tiny(seed=1, gains="one_plus"):
    wts = synth.make_weights(synth.TINY, seed=seed, gains=gains)
    return wts, O.Drafter(synth.TINY, wts.bits, wts.d2t)


# -------------------------------------------------------------------------- bf16

def test_widen_bf16_known_bit_patterns():
    cases = {0x3F80: 1.0, 0xBF80: -1.0, 0x4000: 2.0, 0x3FC0: 1.5, 0x0000: 0.0,
             0x4049: 3.140625, 0x0080: 2.0 ** -126, 0x0001: 2.0 ** -133,
             0x7F7F: (2 - 2.0 ** -7) * 2.0 ** 127, 0xC2F7: -123.5}
    got = O.widen_bf16(np.array(list(cases), dtype=np.uint16))
    assert got.dtype == np.float64
    np.testing.assert_array_equal(got, np.array(list(cases.values())))


def test_round_bf16_ties_to_even_and_carries():
    e = 2.0 ** -8  # half of bf16's unit in the last place at 1.0
    cases = [(1.0, 1.0), (1 + e, 1.0), (1 + 3 * e, 1 + 2.0 ** -6),
             (1 + e + 2.0 ** -40, 1 + 2.0 ** -7), (1 + 2.0 ** -9, 1.0),
             (-(1 + 3 * e), -(1 + 2.0 ** -6)), (255.5, 256.0), (2 - e, 2.0),
             (0.0, 0.0), (3.0, 3.0), (1e-3, 0.00099945068359375)]
    for x, want in cases:
        assert O.round_bf16(np.array([x]))[0] == want, x


def test_round_bf16_is_nearest_representable():
    x = np.random.default_rng(0).standard_normal(20000) * 10.0 ** np.random.default_rng(1).integers(-6, 6, 20000)
    r = O.round_bf16(x)
    # representable: float32 with the low 16 bits clear
    r32 = r.astype(np.float32)
    assert np.all(r32.astype(np.float64) == r)
    assert np.all((r32.view(np.uint32) & 0xFFFF) == 0)
    # within half an ulp (2^-8 relative) and idempotent, monotone
    assert np.all(np.abs(x - r) <= np.abs(x) * 2.0 ** -8)
    np.testing.assert_array_equal(O.round_bf16(r), r)
    xs = np.sort(x)
    assert np.all(np.diff(O.round_bf16(xs)) >= 0)


# ----------------------------------------------------------------------- RMSNorm

def test_rms_norm_closed_forms():
    eps = 1e-6
    c = np.full(8, 3.0)
    np.testing.assert_allclose(O.rms_norm(c, np.full(8, 2.0), eps), 2 * 3 / math.sqrt(9 + eps),
                               rtol=1e-15)
    x = np.array([3.0, 4.0, 0.0, 0.0])          # mean square 25/4 -> rms 2.5
    np.testing.assert_allclose(O.rms_norm(x, np.ones(4), 0.0), [1.2, 1.6, 0.0, 0.0], rtol=1e-15)
    # the gain multiplies (Llama), it is not 1 + w
    np.testing.assert_array_equal(O.rms_norm(x, np.zeros(4), eps), np.zeros(4))
    np.testing.assert_allclose(O.rms_norm(x, np.array([1.0, -2.0, 5.0, 1.0]), 0.0),
                               [1.2, -3.2, 0.0, 0.0], rtol=1e-15)
    np.testing.assert_array_equal(O.rms_norm(np.zeros(5), np.ones(5), eps), np.zeros(5))


def test_rms_norm_unit_rms_and_row_independence():
    eps = 1e-6
    x = np.random.default_rng(3).standard_normal((4, 256)) * np.array([[1e-2], [1.0], [7.0], [300.0]])
    y = O.rms_norm(x, np.ones(256), eps)
    ms = np.mean(x * x, axis=1)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), np.sqrt(ms / (ms + eps)), rtol=1e-12)
    np.testing.assert_allclose(O.rms_norm(x[2], np.ones(256), eps), y[2], rtol=1e-15)


# -------------------------------------------------------------------------- RoPE

def test_rope_identity_at_position_zero_and_tail_untouched():
    x = np.random.default_rng(4).standard_normal((3, 64))
    np.testing.assert_array_equal(O.rope_neox(x, 0, 16, 1e7), x)
    y = O.rope_neox(x, 12345, 16, 1e7)
    np.testing.assert_array_equal(y[:, 16:], x[:, 16:])
    assert not np.allclose(y[:, :16], x[:, :16])


def test_rope_neox_pairing_sign_and_frequency():
    R, theta = 64, 1e7
    e0 = np.zeros(256)
    e0[0] = 1.0
    y = O.rope_neox(e0, 1, R, theta)            # pair (0, 32), frequency 1
    want = np.zeros(256)
    want[0], want[32] = math.cos(1.0), math.sin(1.0)
    np.testing.assert_allclose(y, want, atol=1e-15)
    e32 = np.zeros(256)
    e32[32] = 1.0
    y = O.rope_neox(e32, 1, R, theta)
    want = np.zeros(256)
    want[0], want[32] = -math.sin(1.0), math.cos(1.0)
    np.testing.assert_allclose(y, want, atol=1e-15)
    # pair i = 1 turns at theta^(-2/R) = 10^(-7/32) ~ 0.6043 rad per position (not 10^(-7/128))
    e1 = np.zeros(256)
    e1[1] = 1.0
    y = O.rope_neox(e1, 5, R, theta)
    w1 = 10.0 ** (-7.0 / 32.0)
    np.testing.assert_allclose([y[1], y[33]], [math.cos(5 * w1), math.sin(5 * w1)], atol=1e-14)
    # the last pair (31, 63) turns at theta^(-62/64)
    e31 = np.zeros(256)
    e31[31] = 1.0
    y = O.rope_neox(e31, 1000, R, theta)
    w31 = 10.0 ** (-7.0 * 62.0 / 64.0)
    np.testing.assert_allclose([y[31], y[63]], [math.cos(1000 * w31), math.sin(1000 * w31)], atol=1e-14)


def test_rope_preserves_pair_norms_and_relative_position():
    rng = np.random.default_rng(5)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    R = 16
    y = O.rope_neox(q, 777, R, 1e7)
    for i in range(R // 2):
        np.testing.assert_allclose(math.hypot(y[i], y[i + R // 2]),
                                   math.hypot(q[i], q[i + R // 2]), rtol=1e-13)
    a = O.rope_neox(q, 10, R, 1e7) @ O.rope_neox(k, 3, R, 1e7)
    b = O.rope_neox(q, 10 + 4000, R, 1e7) @ O.rope_neox(k, 3 + 4000, R, 1e7)
    np.testing.assert_allclose(a, b, rtol=1e-9)


# --------------------------------------------------------------------- attention

def test_attention_single_key_returns_value_exactly():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((16, 256))
    k = rng.standard_normal((1, 4, 256))
    v = rng.standard_normal((1, 4, 256))
    out = O.gqa_attention(q, k, v)
    for h in range(16):
        np.testing.assert_array_equal(out[h], v[0, h // 4])


def test_attention_two_keys_closed_form_scale():
    # d = 4: q.k1 = 2 -> scaled score 2/sqrt(4) = 1; q.k2 = 0.  p1 = sigmoid(1).
    q = np.array([[2.0, 0.0, 0.0, 0.0]])
    k = np.array([[[1.0, 0.0, 0.0, 0.0]], [[0.0, 5.0, 0.0, 0.0]]])
    v = np.array([[[1.0, 0.0, 0.0, 0.0]], [[0.0, 1.0, 0.0, 0.0]]])
    out = O.gqa_attention(q, k, v)
    np.testing.assert_allclose(out[0], [0.7310585786300049, 0.2689414213699951, 0, 0], rtol=1e-15)


def test_attention_equal_keys_average_values_and_gqa_mapping():
    rng = np.random.default_rng(7)
    T = 9
    k = np.repeat(rng.standard_normal((1, 2, 8)), T, axis=0)
    v = rng.standard_normal((T, 2, 8))
    q = rng.standard_normal((8, 8))
    out = O.gqa_attention(q, k, v)
    for h in range(8):   # heads 0-3 read kv head 0, heads 4-7 kv head 1 (contiguous groups)
        np.testing.assert_allclose(out[h], v[:, h // 4].mean(axis=0), rtol=1e-13)
    # permuting the keys changes nothing
    k2 = rng.standard_normal((T, 2, 8))
    perm = rng.permutation(T)
    np.testing.assert_allclose(O.gqa_attention(q, k2, v), O.gqa_attention(q, k2[perm], v[perm]),
                               rtol=1e-13)


def test_silu_and_argmax_special_values():
    ln3 = math.log(3.0)
    np.testing.assert_allclose(O.silu(np.array([0.0, ln3, -ln3])), [0.0, 0.75 * ln3, -0.25 * ln3],
                               rtol=1e-15, atol=0)
    assert O.argmax_first(np.array([1.0, 5.0, 2.0, 5.0])) == 1
    assert O.argmax_first(np.array([-3.0, -3.0])) == 0


# ------------------------------------------------------------- encode / layer wiring

def test_encode_concatenates_aux_in_order():
    g = synth.TINY
    n = g.n_embd
    wts, dr = random_tiny()
    aux = synth.make_aux((5,), g, seed=2)
    a = O.widen_bf16(aux)
    for i in range(3):
        fc = np.zeros((n, 3 * n))
        fc[:, i * n:(i + 1) * n] = np.eye(n)
        dr.w["fc"] = fc
        np.testing.assert_array_equal(O.encode(dr, aux), a[:, i, :])


def test_layer_zero_o_and_gate_passes_g_to_lm_head():
    g_vec = np.array([1.0, -2.0, 3.0, 0.5, 8.0, -6.0, 2.0, 4.0])
    wfin = np.array([1.0, 1.0, 1.0, 1.0, 0.25, 1.0, 1.0, 1.0])
    d2t = np.array([3, 3, 3, 3, 3, 3, 3, 1], dtype=np.int64)
    dr = micro_drafter(final_norm=wfin, d2t=d2t)
    so = O.draft_step(dr, 3, g_vec, np.zeros((0, 1, 4)), np.zeros((0, 1, 4)), 0)
    np.testing.assert_array_equal(so.x1, g_vec)          # W_o = 0: x1 is the pre-norm g
    np.testing.assert_array_equal(so.g_next, g_vec)      # W_gate = 0: gsum = x1
    rms = math.sqrt(np.mean(g_vec ** 2) + 1e-6)          # mean square 135.25/8
    np.testing.assert_allclose(so.logits, g_vec * wfin / rms, rtol=1e-14)
    # g * w_final = [1, -2, 3, .5, 2, -6, 2, 4]: the maximum 4 sits at draft id 7
    assert so.draft_id == 7
    assert so.target_id == 8                              # 7 + d2t[7]


def test_layer_single_key_attention_o_proj_and_residual():
    """First position (empty cache): attention returns v for every q head; x1 = W_o . attn + g.
    W_v picks the first 4 entries of the embedding half of the concat."""
    n = MICRO.n_embd
    emb = np.zeros((16, n))
    emb[5] = 2.0                                          # constant row -> normalised ~ w_in
    w_in = np.array([1.0, 2.0, -1.0, 0.5, 1.0, 1.0, 1.0, 1.0])
    wv = np.zeros((4, 2 * n))
    wv[:, :4] = np.eye(4)
    wo = np.eye(n)                                        # head 0 -> x1[0:4], head 1 -> x1[4:8]
    g_vec = np.array([0.5, 0.25, -1.0, 2.0, 1.0, -3.0, 0.0, 1.5])
    dr = micro_drafter(embed=emb, in_norm=w_in, v=wv, o=wo)
    so = O.draft_step(dr, 5, g_vec, np.zeros((0, 1, 4)), np.zeros((0, 1, 4)), 0)
    scale = 2.0 / math.sqrt(4.0 + 1e-6)
    v_exp = O.round_bf16(w_in[:4] * scale)                # the value is stored as bf16
    np.testing.assert_array_equal(so.v[0], v_exp)
    np.testing.assert_allclose(so.attn, np.concatenate([v_exp, v_exp]), rtol=0, atol=0)
    np.testing.assert_allclose(so.x1, np.concatenate([v_exp, v_exp]) + g_vec, rtol=1e-15)
    np.testing.assert_allclose(so.g_next, so.x1, rtol=0)


def test_layer_hidden_half_uses_hidden_norm_of_g():
    """W_v reading the second half of the concat sees RMSNorm(g) * hidden_norm."""
    n = MICRO.n_embd
    wv = np.zeros((4, 2 * n))
    wv[:, n:n + 4] = np.eye(4)
    w_hid = np.array([2.0, 1.0, 1.0, 0.5, 1.0, 1.0, 1.0, 1.0])
    g_vec = np.array([3.0, 4.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0])   # mean square 25/8
    dr = micro_drafter(hidden_norm=w_hid, v=wv, embed=np.ones((16, n)))
    so = O.draft_step(dr, 0, g_vec, np.zeros((0, 1, 4)), np.zeros((0, 1, 4)), 0)
    rms = math.sqrt(25.0 / 8.0 + 1e-6)
    np.testing.assert_array_equal(so.v[0], O.round_bf16(np.array([6.0, 4.0, 0.0, 0.0]) / rms))


def test_layer_swiglu_roles_and_fused_residual():
    """W_o = 0 -> x1 = g; gate = I, up = 2 I, down = I: gsum = silu(z) * 2z + g with
    z = RMSNorm(g) * post_norm.  Swapping the gate and up roles would give silu(2z) * z."""
    n = MICRO.n_embd
    g_vec = np.full(n, 2.0)
    w_post = np.array([0.5, 1.0, -1.0, 2.0, 0.0, 1.0, 0.25, 1.0])
    dr = micro_drafter(post_norm=w_post, gate=np.eye(n), up=2 * np.eye(n), down=np.eye(n))
    so = O.draft_step(dr, 0, g_vec, np.zeros((0, 1, 4)), np.zeros((0, 1, 4)), 0)
    z = w_post * (2.0 / math.sqrt(4.0 + 1e-6))
    want = z / (1 + np.exp(-z)) * 2 * z + g_vec
    np.testing.assert_allclose(so.g_next, want, rtol=1e-14)
    assert not np.allclose(so.g_next, (2 * z) / (1 + np.exp(-2 * z)) * z + g_vec)
    # lm_head = I: the logits are the final RMSNorm of gsum (not of x1)
    np.testing.assert_allclose(so.logits, want / math.sqrt(np.mean(want ** 2) + 1e-6), rtol=1e-13)


def test_rope_applies_to_q_and_k_not_v():
    """q and k rows read the same concat entry; at position p the stored k is (cos, sin)
    rotated, v is not, and q . k of the same position is rotation invariant."""
    n = MICRO.n_embd
    wq = np.zeros((8, 2 * n))
    wq[0, 0] = 1.0
    wq[4, 0] = 1.0
    wk = np.zeros((4, 2 * n))
    wk[0, 0] = 1.0
    wv = np.zeros((4, 2 * n))
    wv[0, 0] = 1.0
    emb = np.ones((16, n))
    dr = micro_drafter(q=wq, k=wk, v=wv, embed=emb)
    cache = np.zeros((3, 1, 4))
    so = O.draft_step(dr, 1, np.ones(n), cache, cache, 3)
    c0 = 1.0 / math.sqrt(1.0 + 1e-6)
    np.testing.assert_array_equal(so.k[0], O.round_bf16(np.array([c0 * math.cos(3.0), c0 * math.sin(3.0), 0, 0])))
    np.testing.assert_array_equal(so.v[0], O.round_bf16(np.array([c0, 0, 0, 0])))


# ------------------------------------------------------------ page-fixed values

def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [l.split() for l in f if l.strip() and not l.startswith("#")]


def test_full_geometry_matches_page_tensor_list_and_config():
    rows = _golden_lines("drafter_geometry.txt")
    shapes = synth.weight_shapes(synth.FULL)
    cfg = {r[1]: r[2] for r in rows if r[0] == "config"}
    g = synth.FULL
    for r in rows:
        if r[0] == "tensor" and r[1] in shapes:
            assert shapes[r[1]] == tuple(int(x) for x in r[2:]), r[1]
    assert int(cfg["hidden_size"]) == g.n_embd
    assert int(cfg["num_attention_heads"]) == g.n_head
    assert int(cfg["num_key_value_heads"]) == g.n_head_kv
    assert int(cfg["head_dim"]) == g.head_dim
    assert int(cfg["intermediate_size"]) == g.n_ff
    assert int(cfg["draft_vocab_size"]) == g.draft_vocab
    assert int(cfg["vocab_size"]) == g.target_vocab
    assert float(cfg["rope_theta"]) == g.rope_theta
    assert float(cfg["rms_norm_eps"]) == g.rms_eps
    assert int(float(cfg["partial_rotary_factor"]) * g.head_dim) == int(cfg["rope_dims"]) == g.rope_dims
    d2t_len = [int(r[2]) for r in rows if r[:2] == ["tensor", "d2t"]][0]
    assert d2t_len == g.draft_vocab
    n_bytes = 2 * sum(int(np.prod(s)) for k, s in shapes.items() if k != "embed")
    assert abs(n_bytes / 1e9 - float(cfg["draft_gb_approx"])) < 0.05


def test_capacity_boundary_rule():
    for start, k, mx, plain, shrunk in _golden_lines("capacity_boundary.txt"):
        start, k, mx = int(start), int(k), int(mx)
        if plain == "refuse":
            with pytest.raises(O.CapacityError):
                O.plan_gamma(start, k, mx, shrink=False)
        else:
            assert O.plan_gamma(start, k, mx, shrink=False) == int(plain)
        if shrunk == "refuse":
            with pytest.raises(O.CapacityError):
                O.plan_gamma(start, k, mx, shrink=True)
        else:
            assert O.plan_gamma(start, k, mx, shrink=True) == int(shrunk)


# ------------------------------------------------------------- accept walk

def test_accept_walk_cases():
    d = [11, 12, 13]
    assert O.accept(d, [11, 12, 13, 99]) == (3, 99)       # all accepted: bonus is y_gamma
    assert O.accept(d, [11, 5, 13, 99]) == (1, 5)         # stop at the first mismatch
    assert O.accept(d, [7, 12, 13, 99]) == (0, 7)         # later matches do not count
    assert O.accept(d, [11, 12, 13, 99], gamma_eff=2) == (2, 13)


# ------------------------------------------------- state bookkeeping on TINY

def _history(dr, seed, n_prompt):
    g = synth.TINY
    toks = synth.make_tokens((n_prompt + 1,), g, seed)
    aux = synth.make_aux((n_prompt,), g, seed)
    return toks, aux


def test_cached_chain_equals_stateless_recompute():
    wts, dr = random_tiny(seed=3)
    toks, aux = _history(dr, 11, 9)
    st = O.prefill(dr, toks[:9], int(toks[9]), aux)
    assert st.kv_len == 8
    genc = O.encode(dr, aux)
    pairs = [(int(toks[p + 1]), genc[p], p) for p in range(8)]
    a = O.draft_chain(dr, st, 4)
    b = O.draft_chain_stateless(dr, pairs, st.g, st.tok, 4)
    assert a.draft_tok == b.draft_tok and a.draft_id == b.draft_id
    for la, lb in zip(a.logits, b.logits):
        np.testing.assert_allclose(la, lb, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(a.spec_k, b.spec_k)
    np.testing.assert_array_equal(a.spec_v, b.spec_v)


def test_prefill_of_one_token_has_empty_cache_and_first_step_attends_one_key():
    wts, dr = random_tiny(seed=4)
    toks, aux = _history(dr, 12, 1)
    st = O.prefill(dr, toks[:1], int(toks[1]), aux)
    assert st.kv_len == 0 and st.tok == int(toks[1])
    np.testing.assert_allclose(st.g, O.widen_bf16(aux[0]).reshape(-1) @ dr.w["fc"].T, rtol=1e-12)
    ch = O.draft_chain(dr, st, 1)
    # one key: the attention output is that key's value for every q head
    so = ch.steps[0]
    group = dr.geom.n_head // dr.geom.n_head_kv
    for h in range(dr.geom.n_head):
        np.testing.assert_array_equal(so.attn.reshape(dr.geom.n_head, -1)[h], so.v[h // group])


def test_chain_leaves_committed_state_untouched():
    wts, dr = random_tiny(seed=5)
    toks, aux = _history(dr, 13, 7)
    st = O.prefill(dr, toks[:7], int(toks[7]), aux)
    snap = st.copy()
    O.draft_chain(dr, st, 3)
    np.testing.assert_array_equal(st.k, snap.k)
    np.testing.assert_array_equal(st.v, snap.v)
    np.testing.assert_array_equal(st.g, snap.g)
    assert st.tok == snap.tok


@pytest.mark.parametrize("n_acc", [0, 1, 3])
def test_rebuild_equals_prefill_over_extended_history(n_acc):
    g = synth.TINY
    wts, dr = random_tiny(seed=6)
    P, gamma = 10, 3
    toks, aux = _history(dr, 14, P)
    st = O.prefill(dr, toks[:P], int(toks[P]), aux)
    ch = O.draft_chain(dr, st, gamma)
    vaux = synth.make_aux((gamma + 1,), g, seed=14, stream=1)
    bonus = 1234
    new = O.rebuild_after_verify(dr, st, n_acc, ch.draft_tok, bonus, vaux)
    assert new.kv_len == st.kv_len + n_acc + 1
    ext_tok = list(toks[:P + 1]) + ch.draft_tok[:n_acc]
    ext_aux = np.concatenate([aux, vaux[:n_acc + 1]])
    ref = O.prefill(dr, np.array(ext_tok), bonus, ext_aux)
    assert ref.kv_len == new.kv_len and ref.tok == new.tok == bonus
    np.testing.assert_allclose(new.g, ref.g, rtol=1e-12)
    np.testing.assert_array_equal(new.k, ref.k)
    np.testing.assert_array_equal(new.v, ref.v)
    # position L (pair 0) equals the chain's own first speculative entry
    np.testing.assert_array_equal(new.k[st.kv_len], ch.spec_k[0])


class SyntheticTarget:
    """Deterministic stand-in for the target model: its greedy next token and its
    auxiliary features are functions of the token history alone.  To give the
    accept walk something to accept, two histories in three take the drafter's own
    first proposal from a prefill over that history."""

    def __init__(self, dr, seed):
        self.dr, self.seed = dr, seed

    @staticmethod
    def _key(hist):
        # tuple-of-int hashing is deterministic in CPython (no per-process salt)
        return hash(tuple(int(t) for t in hist)) & ((1 << 62) - 1)

    def aux(self, hist):
        key = self._key(hist) % (1 << 31)
        return synth.make_aux((), self.dr.geom, self.seed, stream=key)

    def next_token(self, hist):
        key = self._key(hist)
        if (key >> 20) % 3 == 0:
            return int(key % self.dr.geom.target_vocab)
        auxs = np.stack([self.aux(hist[:p + 1]) for p in range(len(hist) - 1)])
        st2 = O.prefill(self.dr, np.array(hist[:-1]), hist[-1], auxs)
        return int(O.draft_chain(self.dr, st2, 1).draft_tok[0])


def test_speculative_loop_reproduces_target_greedy_stream():
    """"Add the Eagle3Speculator module" (tests: the full shifted speculative loop reproduces
    greedy decoding); "memra_engine/eagle.rs" module doc (greedy spec decode is exact)."""
    wts, dr = random_tiny(seed=7)
    tgt = SyntheticTarget(dr, seed=21)
    prompt = [int(t) for t in synth.make_tokens((6,), dr.geom, 22)]
    gamma, rounds = 3, 5
    # plain greedy stream of the target
    hist = list(prompt)
    for _ in range(rounds * (gamma + 1) + 1):
        hist.append(tgt.next_token(hist))
    greedy = hist[len(prompt):]
    # speculative loop
    hist = list(prompt)
    aux = np.stack([tgt.aux(hist[:p + 1]) for p in range(len(hist))])
    first = tgt.next_token(hist)
    st = O.prefill(dr, np.array(hist), first, aux)
    hist.append(first)
    accepted = 0
    for _ in range(rounds):
        ch = O.draft_chain(dr, st, gamma)
        ver = [hist + ch.draft_tok[:i] for i in range(gamma + 1)]
        y = [tgt.next_token(h) for h in ver]
        vaux = np.stack([tgt.aux(h) for h in ver])
        n, bonus = O.accept(ch.draft_tok, y)
        accepted += n
        st = O.rebuild_after_verify(dr, st, n, ch.draft_tok, bonus, vaux)
        hist = hist + ch.draft_tok[:n] + [bonus]
        assert st.kv_len == len(hist) - 2 and st.tok == hist[-1]
    out = hist[len(prompt):]
    assert out == greedy[:len(out)]
    assert accepted > 0


def test_batched_kv_entries_equal_one_by_one():
    wts, dr = random_tiny(seed=8)
    toks = synth.make_tokens((9,), dr.geom, 30)
    gs = O.encode(dr, synth.make_aux((9,), dr.geom, 30))
    pos = np.array([0, 1, 5, 17, 18, 40, 41, 90, 99])
    kb, vb = O.kv_entries(dr, toks, gs, pos)
    for i in range(9):
        k1, v1 = O.kv_entry(dr, int(toks[i]), gs[i], int(pos[i]))
        assert np.max(np.abs(kb[i] - k1)) <= 2.0 ** -8 * np.max(np.abs(k1))
        assert np.max(np.abs(vb[i] - v1)) <= 2.0 ** -8 * np.max(np.abs(v1))


def test_norm_before_residual_flag_uses_the_normed_g():
    """With the checkpoint flag norm_before_residual the attention residual is
    RMSNorm(g) * hidden_norm: with W_o = 0 and W_gate = 0, x1 = gsum = the normed g.  A g
    of equal-magnitude entries normalises to its signs (eps 1e-6 changes the scale by
    about 5e-7 relative at magnitude 1); gains of 2 on dims 0 and 5 double those dims."""
    dr = micro_drafter(hidden_norm=np.array([2.0, 1, 1, 1, 1, 2.0, 1, 1]))
    dr.norm_before_residual = True
    g_vec = np.array([1.0, -1.0, 1.0, 1.0, -1.0, -1.0, 1.0, 1.0])
    so = O.draft_step(dr, 3, g_vec, np.zeros((0, 1, 4)), np.zeros((0, 1, 4)), 0)
    want = np.array([2.0, -1.0, 1.0, 1.0, -1.0, -2.0, 1.0, 1.0]) / math.sqrt(1.0 + 1e-6)
    np.testing.assert_allclose(so.x1, want, rtol=1e-15)
    np.testing.assert_array_equal(so.g_next, so.x1)
    dr.norm_before_residual = False
    so = O.draft_step(dr, 3, g_vec, np.zeros((0, 1, 4)), np.zeros((0, 1, 4)), 0)
    np.testing.assert_array_equal(so.x1, g_vec)
