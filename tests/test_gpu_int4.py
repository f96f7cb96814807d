"""GPU parity of the drafter with INT4 projection weights (4-bit codes, a bf16 (scale,
zero) per 128 inputs; fc, norms and embedding bf16) against the oracle dequantizing the
same codes: full rounds through the C ABI on the small drafter (one item per launch with x
in registers, and 2 to 8 items per launch: the ragged batch and the prefill's k/v-only
projections), with CUDA graphs and with direct launches; batched rounds on a small drafter
whose projections take the tensor cores (the codes decoded to bf16 in shared memory, each
128-wide group's sums scaled in the epilogue) under both tile schedules, and on the
CUDA-core GEMV for comparison; and on the eagle.rs geometry at batch 1 / prompt 512 /
gamma 3 (the benchmark's configuration) and a batch of 8 (tensor cores)."""
import numpy as np
import pytest
import torch

from eagle_speculative_decode_gb300 import synth
from eagle_speculative_decode_gb300.runtime import DraftModel
from oracle import eagle3_oracle as O
from parity import check_state, gpu_prefill, oracle_prefill, run_round

pytestmark = pytest.mark.gpu


def _rounds(g, model, dr, lens, gamma, seeds, seed, pages=True):
    B = len(lens)
    P_max = int(max(lens))
    toks = synth.make_tokens((B, P_max + 1), g, seed)
    aux = synth.make_aux((B, P_max), g, seed)
    pt = None
    if pages:
        pt = synth.page_table(B, (model.max_cache_len + model.page_size - 1) // model.page_size, seed=seed + 1)
    seq = model.new_state(B, page_table=pt)
    gpu_prefill(seq, model, toks, aux, lens)
    torch.cuda.synchronize()
    states = oracle_prefill(dr, toks, aux, lens)
    check_state(seq, states, "prefill")
    for s in seeds:
        n = synth.imposed_accept_lengths(B, gamma, seed=s)
        states = run_round(model, dr, seq, states, gamma, n, seed=s)[0]


@pytest.fixture(scope="module")
def tiny(built_lib):
    g = synth.TINY
    wts = synth.make_int4_weights(g, seed=7)
    model = DraftModel(wts, max_batch=8, max_gamma=4, max_cache_len=100, page_size=16)
    dr = O.Drafter(g, wts.bits, wts.d2t, int4=wts.int4)
    yield g, model, dr
    model.close()


def test_int4_single_sequence(tiny):
    g, model, dr = tiny
    _rounds(g, model, dr, np.array([40]), 3, [10, 11, 12], seed=13, pages=False)


@pytest.mark.parametrize("graphs", [True, False])
def test_int4_ragged_batch(tiny, graphs):
    g, model, dr = tiny
    model.set_graph_mode(graphs)
    try:
        _rounds(g, model, dr, np.array([5, 33, 17, 1, 60, 2, 9]), 4, [20, 21], seed=22)
    finally:
        model.set_graph_mode(True)


@pytest.fixture(scope="module")
def small_q4(built_lib):
    g = synth.SMALL
    wts = synth.make_int4_weights(g, seed=8)
    model = DraftModel(wts, max_batch=20, max_gamma=4, max_cache_len=160, page_size=16)
    dr = O.Drafter(g, wts.bits, wts.d2t, int4=wts.int4)
    yield g, model, dr
    model.close()


@pytest.mark.parametrize("path", ["tc_stream_k", "tc_cluster", "gemv"])
def test_int4_batched_projections(small_q4, path):
    """Batch 20 (and prefills of up to 100 positions): 3 or more items per projection run
    on the tensor cores unless the threshold keeps them on the GEMV."""
    g, model, dr = small_q4
    if path == "gemv":
        model.set_tc_min_items(1 << 20)
    else:
        model.set_tc_schedule(1 if path == "tc_stream_k" else 2)
    try:
        _rounds(g, model, dr, synth.ragged_lengths(20, 1, 100, seed=70), 4, [71, 72], seed=73)
    finally:
        model.set_tc_min_items(0)
        model.set_tc_schedule(0)


def test_int4_full_geometry(built_lib):
    g = synth.FULL
    wts = synth.make_int4_weights(g, seed=0)
    dr = O.Drafter(g, wts.bits, wts.d2t, int4=wts.int4)
    model = DraftModel(wts, max_batch=8, max_gamma=3, max_cache_len=1024, page_size=64)
    try:
        _rounds(g, model, dr, np.array([512]), 3, [110, 111], seed=101, pages=False)
        _rounds(g, model, dr, synth.ragged_lengths(8, 64, 256, seed=120), 3, [130], seed=121)
    finally:
        model.close()
