"""GPU parity of the batched (tensor-core) projections on a small drafter whose q / k / v
blocks are whole 128-row tiles (n_embd 256, 8:2 GQA, head 64): item tiles of 16 to 256
columns with ragged tails, two item tiles in one launch (a 300-token prefill chunk), and
full rounds at batch 20 and 40, element by element against the CPU oracle -- under both
tile schedules: stream-K (partials through L2, the last contributor finishes a tile) and
cluster split-K (partials through distributed shared memory, each rank finishes its
share of the columns), which the automatic choice would not take at this size."""
import numpy as np
import pytest
import torch

from eagle_speculative_decode_gb300 import synth
from eagle_speculative_decode_gb300.runtime import DraftModel
from oracle import eagle3_oracle as O
from parity import check_state, gpu_prefill, oracle_prefill, run_round

pytestmark = pytest.mark.gpu
G = synth.SMALL


@pytest.fixture(scope="module")
def small(built_lib):
    wts = synth.make_weights(G, seed=30)
    model = DraftModel(wts, max_batch=40, max_gamma=4, max_cache_len=320, page_size=16)
    dr = O.Drafter(G, wts.bits, wts.d2t)
    yield wts, model, dr
    model.close()


def _prompt(batch, lens, seed):
    P_max = int(max(lens))
    toks = synth.make_tokens((batch, P_max + 1), G, seed)
    aux = synth.make_aux((batch, P_max), G, seed)
    return toks, aux


STREAM_K, CLUSTER = 1, 2


@pytest.fixture(params=[STREAM_K, CLUSTER], ids=["stream_k", "cluster"])
def schedule(request, small):
    small[1].set_tc_schedule(request.param)
    yield request.param
    small[1].set_tc_schedule(0)


@pytest.mark.parametrize("sched", [STREAM_K, CLUSTER], ids=["stream_k", "cluster"])
@pytest.mark.parametrize("rows", [3, 16, 20, 37, 64, 100, 256, 300])
def test_tc_encode_exact_integer_case(small, rows, sched):
    """fc in {-1, 0, 1} * 2^-4 and integer features: the tensor-core sums are exact in
    float32, so every output equals the oracle bit for bit -- a check of the operand
    layouts (swizzle, descriptors, item tiles) independent of rounding."""
    wts, model, dr = small
    rng = np.random.default_rng(rows)
    fc = (rng.integers(-1, 2, size=(G.n_embd, 3 * G.n_embd)) * 2.0 ** -4).astype(np.float32)
    aux = rng.integers(-8, 9, size=(rows, 3, G.n_embd)).astype(np.float32)
    fc_bits = (fc.view(np.uint32) >> 16).astype(np.uint16)
    aux_bits = (aux.view(np.uint32) >> 16).astype(np.uint16)
    bits = dict(wts.bits)
    bits["fc"] = fc_bits
    m2 = DraftModel(synth.DrafterWeights(G, bits, wts.d2t), max_batch=2, max_gamma=2,
                    max_cache_len=16, page_size=16)
    m2.set_tc_schedule(sched)
    try:
        got = m2.encode(torch.from_numpy(aux_bits.view(np.int16)).to(m2.device)).cpu().numpy()
    finally:
        m2.close()
    want = O.encode(O.Drafter(G, bits, wts.d2t), aux_bits)
    assert np.array_equal(got.astype(np.float64), want)


def test_tc_rounds_batch20_random_pages(small, schedule):
    wts, model, dr = small
    B = 20
    lens = synth.ragged_lengths(B, 1, 60, seed=31)
    toks, aux = _prompt(B, lens, seed=32)
    pages_per_seq = (model.max_cache_len + model.page_size - 1) // model.page_size
    pt = synth.page_table(B, pages_per_seq, seed=33)
    seq = model.new_state(B, page_table=pt)
    gpu_prefill(seq, model, toks, aux, lens)
    torch.cuda.synchronize()
    states = oracle_prefill(dr, toks, aux, lens)
    check_state(seq, states, "prefill")
    for r in range(2):
        n = synth.imposed_accept_lengths(B, 4, seed=34 + r)
        states = run_round(model, dr, seq, states, 4, n, seed=34 + r)[0]


def test_tc_rounds_batch40_long_prompts(small, schedule):
    """Prompts up to 300 tokens: each prefill chunk is one launch over two item tiles."""
    wts, model, dr = small
    B = 40
    lens = synth.ragged_lengths(B, 200, 300, seed=41)
    lens[0] = 300
    toks, aux = _prompt(B, lens, seed=42)
    seq = model.new_state(B)
    gpu_prefill(seq, model, toks, aux, lens)
    torch.cuda.synchronize()
    states = oracle_prefill(dr, toks, aux, lens)
    check_state(seq, states, "prefill")
    n = synth.imposed_accept_lengths(B, 3, seed=43)
    run_round(model, dr, seq, states, 3, n, seed=43)
