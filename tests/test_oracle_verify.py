"""Pins of the oracle's target-side greedy verify (CPU only): the argmax of the target
head over RMSNorm'd hidden states ("Add the Eagle3Speculator module for speculative
decoding", PR body: target_verify returns the greedy argmax id of every window position).
Closed forms: with eps 0 a constant hidden row normalises to the norm gains exactly, so
each logit is a hand-computable weighted row sum of the head."""
import numpy as np

from eagle_speculative_decode_gb300 import synth
from oracle import eagle3_oracle as O


def bf(x):
    return synth.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def test_constant_row_logits_are_gain_weighted_row_sums():
    n = 4
    head = np.array([[0.5, 0.5, 0.0, 0.0],     # sum 1.0
                     [1.0, 1.0, 1.0, 0.0],     # 3.0  <- the maximum
                     [0.0, 0.0, 0.0, 2.0],     # 2.0
                     [1.0, 0.5, 0.5, 0.5]])    # 2.5
    h = np.full((1, n), -7.0)                 # a negative constant: RMSNorm gives -1
    logits, ids = O.target_verify(bf(head), bf(np.ones(n)), h, eps=0.0)
    assert np.array_equal(logits[0], -np.array([1.0, 3.0, 2.0, 2.5]))
    assert ids[0] == 0                         # -1.0 is the largest of the negated sums
    logits, ids = O.target_verify(bf(head), bf(np.ones(n)), -h, eps=0.0)
    assert ids[0] == 1 and logits[0, 1] == 3.0


def test_norm_gain_multiplies_and_ties_take_the_lowest_id():
    head = np.array([[0.0, 1.0], [1.0, 0.0], [1.0, 0.0]])
    h = np.ones((1, 2))
    _, ids = O.target_verify(bf(head), bf([2.0, 1.0]), h, eps=0.0)
    assert ids[0] == 1                         # gain 2 on dim 0 favours rows 1 and 2: lowest
    _, ids = O.target_verify(bf(head), bf([1.0, 2.0]), h, eps=0.0)
    assert ids[0] == 0
    _, ids = O.target_verify(bf(head), bf([1.0, 1.0]), h, eps=0.0)
    assert ids[0] == 0                         # a three-way tie


def test_shapes_scale_invariance_and_blocking():
    g = synth.TINY
    head, norm = synth.make_target_head(g, seed=1)
    hid = synth.make_hidden((3, 4), g, seed=2)
    logits, ids = O.target_verify(head, norm, hid, eps=0.0)
    assert logits.shape == (3, 4, g.target_vocab) and ids.shape == (3, 4)
    l3, i3 = O.target_verify(head, norm, 3.0 * hid, eps=0.0)
    assert np.array_equal(i3, ids) and np.allclose(l3, logits, rtol=1e-12, atol=1e-12)
    lb, ib = O.target_verify(head, norm, hid, eps=0.0, rows_per_block=7)
    assert np.array_equal(ib, ids) and np.allclose(lb, logits, rtol=1e-12, atol=1e-12)
    # brute force on one row: the id is the index of the largest dot product
    x = hid[1, 2].astype(np.float64)
    x = x / np.sqrt(np.mean(x * x)) * O.widen_bf16(norm)
    dots = [float(np.dot(O.widen_bf16(head[v]), x)) for v in range(g.target_vocab)]
    assert ids[1, 2] == max(range(g.target_vocab), key=lambda v: (dots[v], -v))


def test_verify_then_accept_reproduces_the_greedy_walk():
    """Drafts equal to the verify ids on a prefix are accepted exactly that far, and the
    bonus is the target's id at the first disagreement."""
    g = synth.TINY
    head, norm = synth.make_target_head(g, seed=3)
    hid = synth.make_hidden((1, 5), g, seed=4)
    _, ids = O.target_verify(head, norm, hid, eps=1e-6)
    y = ids[0]
    for n in range(5):
        d = y[:4].copy()
        if n < 4:
            d[n] = (d[n] + 1) % g.target_vocab
        assert O.accept(d, y, 4) == (n, int(y[n]))
