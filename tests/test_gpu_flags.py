"""GPU parity of the checkpoint flag norm_before_residual (attention residual =
RMSNorm(g) * hidden_norm instead of g) against the oracle with the same flag: full rounds on
the CUDA-core GEMV (small drafter) and on the tensor cores (batch 20), through the C ABI."""
import numpy as np
import pytest
import torch

from eagle_speculative_decode_gb300 import binding as Bd
from eagle_speculative_decode_gb300 import synth
from eagle_speculative_decode_gb300.runtime import DraftModel
from oracle import eagle3_oracle as O
from parity import check_state, gpu_prefill, oracle_prefill, run_round

pytestmark = pytest.mark.gpu
FLAG = Bd.EAGLE3_CKPT_NORM_BEFORE_RESIDUAL


def _rounds(g, model, dr, B, lens, gamma, seeds, seed):
    P_max = int(max(lens))
    toks = synth.make_tokens((B, P_max + 1), g, seed)
    aux = synth.make_aux((B, P_max), g, seed)
    pages = (model.max_cache_len + model.page_size - 1) // model.page_size
    seq = model.new_state(B, page_table=synth.page_table(B, pages, seed=seed + 1))
    gpu_prefill(seq, model, toks, aux, lens)
    torch.cuda.synchronize()
    states = oracle_prefill(dr, toks, aux, lens)
    check_state(seq, states, "prefill")
    for s in seeds:
        n = synth.imposed_accept_lengths(B, gamma, seed=s)
        states = run_round(model, dr, seq, states, gamma, n, seed=s)[0]


def test_norm_before_residual_gemv(built_lib):
    g = synth.TINY
    wts = synth.make_weights(g, seed=3)
    model = DraftModel(wts, max_batch=4, max_gamma=4, max_cache_len=100, page_size=16, flags=FLAG)
    try:
        dr = O.Drafter(g, wts.bits, wts.d2t, norm_before_residual=True)
        _rounds(g, model, dr, 3, np.array([20, 7, 33]), 4, [90, 91], seed=92)
        # the flag changes the chain: the same weights without it draft other logits
        assert O.Drafter(g, wts.bits, wts.d2t).norm_before_residual is False
    finally:
        model.close()


def test_norm_before_residual_tensor_cores(built_lib):
    g = synth.SMALL
    wts = synth.make_weights(g, seed=31)
    model = DraftModel(wts, max_batch=20, max_gamma=3, max_cache_len=160, page_size=16, flags=FLAG)
    try:
        dr = O.Drafter(g, wts.bits, wts.d2t, norm_before_residual=True)
        _rounds(g, model, dr, 20, synth.ragged_lengths(20, 1, 60, seed=93), 3, [94], seed=95)
    finally:
        model.close()
