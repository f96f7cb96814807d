"""GPU parity of the drafter with a quantized KV cache (q8_0 keys, q5_1 values, blocks of
32 values), through the C ABI, against the CPU oracle run with the same format.

Every stored block must be a valid encoding of the oracle's unstored k / v: the oracle's
own bytes, except that a code or header field within float32 rounding of a boundary may
take either neighbour.  Because such a code may differ, the chain is checked step by
step: the oracle runs each step on the implementation's inputs to it (previous g and
token, the stored KV decoded) and the step's ids (margin rule), logits and g are compared;
accept lengths and positions are bit-exact.  Covered: the small drafter through the CUDA-core
GEMV (one sequence, ragged batch with non-contiguous pages, the graph and direct launch
paths), the tensor-core projections at batch 20 (quantization of the staged k / v of a
whole item tile), and the full geometry at batch 1 with a 512-token prompt."""
import numpy as np
import pytest
import torch

from eagle_speculative_decode_gb300 import synth
from eagle_speculative_decode_gb300.runtime import DraftModel
from oracle import eagle3_oracle as O
from parity import (assert_quant_valid, check_state, gpu_prefill, oracle_prefill, run_round,
                    with_kv_format)

pytestmark = pytest.mark.gpu
FMT = "q8_0/q5_1"


def _prompt(g, batch, lens, seed):
    P_max = int(max(lens))
    toks = synth.make_tokens((batch, P_max + 1), g, seed)
    aux = synth.make_aux((batch, P_max), g, seed)
    return toks, aux


def _rounds(model, dr, seq, toks, aux, lens, gamma, seeds):
    gpu_prefill(seq, model, toks, aux, lens)
    torch.cuda.synchronize()
    states = oracle_prefill(dr, toks, aux, lens)
    check_state(seq, states, "prefill")
    for s in seeds:
        n = synth.imposed_accept_lengths(seq.B, gamma, seed=s)
        states = run_round(model, dr, seq, states, gamma, n, seed=s)[0]
    return states


@pytest.fixture(scope="module")
def tiny(built_lib):
    g = synth.TINY
    wts = synth.make_weights(g, seed=0)
    model = DraftModel(wts, max_batch=8, max_gamma=8, max_cache_len=100, page_size=16, kv_format=FMT)
    dr = O.Drafter(g, wts.bits, wts.d2t, kv_format=FMT)
    yield g, wts, model, dr
    model.close()


def test_pool_rows_are_quantized_blocks(tiny):
    g, wts, model, dr = tiny
    seq = model.new_state(1)
    assert seq.k_pool.dtype == torch.uint8
    assert seq.k_pool.shape[-1] == g.head_dim // 32 * 34
    assert seq.v_pool.shape[-1] == g.head_dim // 32 * 24


def test_single_sequence_rounds(tiny):
    g, wts, model, dr = tiny
    lens = np.array([32])
    toks, aux = _prompt(g, 1, lens, seed=1)
    seq = model.new_state(1)
    _rounds(model, dr, seq, toks, aux, lens, 3, [10, 11, 12])


@pytest.mark.parametrize("graphs", [True, False])
def test_ragged_batch_random_pages(tiny, graphs):
    g, wts, model, dr = tiny
    model.set_graph_mode(graphs)
    try:
        lens = np.array([5, 32, 17, 1])
        toks, aux = _prompt(g, 4, lens, seed=2)
        pages_per_seq = (model.max_cache_len + model.page_size - 1) // model.page_size
        seq = model.new_state(4, page_table=synth.page_table(4, pages_per_seq, seed=3))
        _rounds(model, dr, seq, toks, aux, lens, 4, [20, 21, 22])
    finally:
        model.set_graph_mode(True)


def test_prefill_blocks_are_the_oracle_bytes_off_boundaries(tiny):
    """The prefill's stored blocks against the oracle's own encoding of its unstored k / v:
    byte-identical except where a code or a header field sits within float32 rounding of
    a boundary, and valid encodings everywhere."""
    g, wts, model, dr = tiny
    lens = np.array([40])
    toks, aux = _prompt(g, 1, lens, seed=5)
    seq = model.new_state(1)
    gpu_prefill(seq, model, toks, aux, lens)
    torch.cuda.synchronize()
    st = oracle_prefill(dr, toks, aux, lens)[0]
    kr, vr = seq.kv_entries(0, 0, st.kv_len)
    nb = g.head_dim // 32
    ko = O.pack_q8_0(*O.quantize_q8_0(st.k_raw.astype(np.float32)))
    vo = O.pack_q5_1(*O.quantize_q5_1(st.v_raw.astype(np.float32)))
    same_k = int(np.sum(np.all(kr.reshape(-1, nb, 34) == ko.reshape(-1, nb, 34), axis=-1)))
    same_v = int(np.sum(np.all(vr.reshape(-1, nb, 24) == vo.reshape(-1, nb, 24), axis=-1)))
    total = st.kv_len * g.n_head_kv * nb
    assert same_k >= 0.98 * total and same_v >= 0.98 * total, (same_k, same_v, total)
    assert_quant_valid(kr, st.k_raw, "k", "prefill K")
    assert_quant_valid(vr, st.v_raw, "v", "prefill V")


@pytest.fixture(scope="module")
def small(built_lib):
    g = synth.SMALL
    wts = synth.make_weights(g, seed=30)
    model = DraftModel(wts, max_batch=24, max_gamma=4, max_cache_len=320, page_size=16, kv_format=FMT)
    dr = O.Drafter(g, wts.bits, wts.d2t, kv_format=FMT)
    yield g, wts, model, dr
    model.close()


def test_tc_rounds_batch20_random_pages(small):
    g, wts, model, dr = small
    B = 20
    lens = synth.ragged_lengths(B, 1, 200, seed=31)
    toks, aux = _prompt(g, B, lens, seed=32)
    pages_per_seq = (model.max_cache_len + model.page_size - 1) // model.page_size
    seq = model.new_state(B, page_table=synth.page_table(B, pages_per_seq, seed=33))
    _rounds(model, dr, seq, toks, aux, lens, 4, [34, 35])


def test_full_geometry_batch1_prompt512(full_drafter):
    g = synth.FULL
    wts, dr = full_drafter
    dr = with_kv_format(dr, FMT)
    model = DraftModel(wts, max_batch=1, max_gamma=3, max_cache_len=1024, page_size=64, kv_format=FMT)
    try:
        lens = np.array([512])
        toks, aux = _prompt(g, 1, lens, seed=101)
        seq = model.new_state(1)
        _rounds(model, dr, seq, toks, aux, lens, 3, [110, 111])
    finally:
        model.close()
