"""GPU parity of the target-side greedy verify (eagle3_verify_greedy) against the CPU
oracle: the argmax of a target head over the RMSNorm'd hidden states of every window row
(the margin rule of the chain: bit-exact ids where the oracle's top-2 margin exceeds 1e-2,
otherwise within 1e-2 of the maximum), the logits within the float tolerance, and the
accept walk on the GPU's ids.  Covers the CUDA-core GEMV (one or two rows), the tensor-core
GEMM (three rows and more, several item tiles), gamma_eff below gamma, and the full target
vocabulary (248320 rows)."""
import numpy as np
import pytest
import torch

from eagle_speculative_decode_gb300 import synth
from eagle_speculative_decode_gb300.runtime import DraftModel
from oracle import eagle3_oracle as O
from parity import MARGIN, assert_close, top2_margin

pytestmark = pytest.mark.gpu


def _drafts_with_prefix(y, n_match, vocab, seed):
    """Drafts that agree with the ids y on the first n_match positions, then disagree."""
    rng = np.random.default_rng(seed)
    B, W = y.shape
    gamma = W - 1
    d = rng.integers(0, vocab, size=(B, gamma)).astype(np.int32)
    for b in range(B):
        n = int(n_match[b])
        d[b, :n] = y[b, :n]
        if n < gamma and d[b, n] == y[b, n]:
            d[b, n] = (d[b, n] + 1) % vocab
    return d


def _check(seq, model, head, norm, hid, gamma_eff, eps, seed, rows=None):
    g = model.geom
    dev = model.device
    B, W = hid.shape[0], hid.shape[1]
    gamma = W - 1
    logits_o, ids_o = O.target_verify(head, norm, hid if rows is None else hid[rows[:, 0], rows[:, 1]], eps)
    # drafts: build them from the oracle ids so that accept lengths cover 0..gamma
    n_match = np.random.default_rng(seed).integers(0, gamma + 1, size=B)
    y_ref = np.zeros((B, W), np.int64)
    if rows is None:
        y_ref = ids_o
    draft = _drafts_with_prefix(y_ref, n_match, g.target_vocab, seed)
    t_head = torch.from_numpy(head.view(np.int16)).to(dev)
    t_norm = torch.from_numpy(norm.view(np.int16)).to(dev)
    t_hid = torch.from_numpy(np.ascontiguousarray(hid)).to(dev)
    t_draft = torch.from_numpy(draft).to(dev)
    t_ge = torch.from_numpy(gamma_eff.astype(np.int32)).to(dev) if gamma_eff is not None else None
    pred, n_acc, bonus, lg = seq.verify_greedy(t_head, t_norm, t_hid, t_draft, t_ge,
                                               target_rms_eps=eps, logits=True)
    torch.cuda.synchronize()
    assert model.status() == 0
    pred = pred.cpu().numpy()
    lg = lg.cpu().numpy()
    sel = [(b, i) for b in range(B) for i in range(W)] if rows is None else [tuple(r) for r in rows]
    for k, (b, i) in enumerate(sel):
        lo = logits_o[b, i] if rows is None else logits_o[k]
        io = int(ids_o[b, i] if rows is None else ids_o[k])
        assert_close(lg[b, i], lo, f"target logits b{b} i{i}")
        if top2_margin(lo) > MARGIN:
            assert pred[b, i] == io, f"b{b} i{i}: GPU id {pred[b, i]} vs oracle {io}"
        else:
            assert lo[pred[b, i]] >= lo.max() - MARGIN
    ge = gamma_eff if gamma_eff is not None else np.full(B, gamma)
    na, bo = n_acc.cpu().numpy(), bonus.cpu().numpy()
    for b in range(B):
        assert (na[b], bo[b]) == O.accept(draft[b], pred[b], int(ge[b]))
    return pred, na


@pytest.fixture(scope="module")
def tiny(built_lib):
    g = synth.TINY
    wts = synth.make_weights(g, seed=0)
    model = DraftModel(wts, max_batch=8, max_gamma=8, max_cache_len=64, page_size=16)
    head, norm = synth.make_target_head(g, seed=50)
    yield g, model, head, norm
    model.close()


@pytest.mark.parametrize("B,gamma", [(1, 1), (2, 3), (8, 8)])
def test_verify_gemv_path(tiny, B, gamma):
    """The small drafter keeps every projection on the CUDA-core GEMV."""
    g, model, head, norm = tiny
    seq = model.new_state(B)
    hid = synth.make_hidden((B, gamma + 1), g, seed=51 + B)
    _, na = _check(seq, model, head, norm, hid, None, g.rms_eps, seed=B)
    assert na.max() <= gamma


def test_verify_gamma_eff_stops_the_walk(tiny):
    g, model, head, norm = tiny
    B, gamma = 4, 5
    seq = model.new_state(B)
    hid = synth.make_hidden((B, gamma + 1), g, seed=60)
    ge = np.array([5, 3, 1, 2])
    _check(seq, model, head, norm, hid, ge, 1e-5, seed=61)


@pytest.fixture(scope="module")
def small(built_lib):
    g = synth.SMALL
    wts = synth.make_weights(g, seed=30)
    model = DraftModel(wts, max_batch=40, max_gamma=4, max_cache_len=64, page_size=16)
    head, norm = synth.make_target_head(g, seed=70)
    yield g, model, head, norm
    model.close()


@pytest.mark.parametrize("B,gamma", [(1, 2), (5, 4), (40, 4)])
def test_verify_tensor_core_path(small, B, gamma):
    """3 to 200 rows on the tensor cores: item tiles of 16 to 64 columns, several item
    tiles at 200 rows, 32 row tiles of the 4096-row head."""
    g, model, head, norm = small
    seq = model.new_state(B)
    hid = synth.make_hidden((B, gamma + 1), g, seed=71 + B)
    _check(seq, model, head, norm, hid, None, g.rms_eps, seed=72 + B)


def test_verify_full_target_vocab(built_lib):
    """The eagle.rs geometry's target vocabulary (248320 rows x 4096): batch 1, gamma 3
    (four rows, every one compared), and batch 64, gamma 3 (256 rows, 24 sampled rows
    compared; accept results checked for all)."""
    g = synth.FULL
    wts = synth.make_weights(g, seed=0, skip=("fc", "q", "k", "v", "o", "gate", "up", "down", "lm_head"))
    shapes = synth.weight_shapes(g)
    for name in ("fc", "q", "k", "v", "o", "gate", "up", "down", "lm_head"):
        wts.bits[name] = np.zeros(shapes[name], np.uint16)
    head = wts.bits["embed"]                      # a target with tied embeddings
    norm = synth.normal_bf16((g.n_embd,), 80, (301,), std=0.02, mean=1.0)
    model = DraftModel(wts, max_batch=64, max_gamma=3, max_cache_len=64, page_size=64)
    try:
        seq = model.new_state(1)
        hid = synth.make_hidden((1, 4), g, seed=81)
        _check(seq, model, head, norm, hid, None, g.rms_eps, seed=82)
        seq = model.new_state(64)
        hid = synth.make_hidden((64, 4), g, seed=83)
        rng = np.random.default_rng(84)
        rows = np.stack([rng.integers(0, 64, 24), rng.integers(0, 4, 24)], axis=1)
        _check(seq, model, head, norm, hid, None, g.rms_eps, seed=85, rows=rows)
    finally:
        model.close()
