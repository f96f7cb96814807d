"""GPU parity at the long-context configurations of the drafter (the eagle.rs geometry:
n_embd 4096, 16:4 GQA with head_dim 256, RoPE 64/256 at theta 1e7, draft vocab 32000 ->
target vocab 248320), through the C ABI, against the CPU oracle, at their full sizes:

  * batch 4, context 32768 each, gamma 7, paged KV with page size 64 on shuffled pages,
    rewind + rebuild every round: 16 rounds with the bf16 cache, 4 with q8_0 K / q5_1 V;
  * batch 8, ragged contexts uniform in 512..8192, gamma 5, accept lengths uniform in
    0..gamma, 4 rounds.

The oracle prefills some sequences in full (sequence 0 of the first case; the longest and
the shortest of the second) and follows them through every round end to end: chain ids
under the margin rule, logits, g and speculative KV per step (step by step on the stored
blocks with the quantized cache), rewind, the accept walk and the rebuilt entries and
boundary; at the end their whole committed cache is compared again, so drift over many
rounds would show.  Every other sequence is checked at a seeded sample of 256 prefill
positions (a one-layer drafter's KV entry depends only on its own pair and position) and,
every round, on each entry the rebuild writes, its new boundary and length, and the accept
walk.  The attention runs at these sizes over about ten stream-K contributors per
(sequence, kv head) pair, and the RoPE table spans all 32K positions."""
import numpy as np
import pytest
import torch

from eagle_speculative_decode_gb300 import synth
from eagle_speculative_decode_gb300.runtime import DraftModel
from oracle import eagle3_oracle as O
from parity import (Tracked, assert_close, check_prefill_sampled, check_rebuild_tracked, check_state,
                    gpu_prefill, oracle_prefill, run_round, stored_state, with_kv_format)

pytestmark = pytest.mark.gpu
G = synth.FULL
PAGE = 64
SAMPLES = 256


def _inputs(B, lens, seed):
    P_max = int(max(lens))
    toks = synth.make_tokens((B, P_max + 1), G, seed)
    aux = synth.make_aux((B, P_max), G, seed)
    return toks, aux


def _run_case(full_drafter, lens, gamma, rounds, follow, prefilled, toks, aux, seed, kv_format):
    wts, dr0 = full_drafter
    dr = with_kv_format(dr0, kv_format)
    B = len(lens)
    max_cache = int(lens.max()) + (gamma + 1) * rounds + 64
    max_cache = (max_cache + PAGE - 1) // PAGE * PAGE
    model = DraftModel(wts, max_batch=B, max_gamma=gamma, max_cache_len=max_cache, page_size=PAGE,
                       kv_format=kv_format)
    try:
        seq = model.new_state(B, page_table=synth.page_table(B, max_cache // PAGE, seed=seed))
        gpu_prefill(seq, model, toks, aux, lens)
        torch.cuda.synchronize()
        states = {b: stored_state(prefilled[b], kv_format) for b in follow}
        check_state(seq, states, "prefill")
        # the other sequences: sampled prefill entries; every boundary
        rng = np.random.default_rng(seed + 1)
        g_last = O.encode(dr, aux[np.arange(B), lens - 1])
        tracked = {}
        for b in range(B):
            if b not in states:
                check_prefill_sampled(seq, dr, toks, aux, lens, b, SAMPLES, rng, kv_format)
            tracked[b] = Tracked(int(lens[b]) - 1, g_last[b], int(toks[b, lens[b]]))
        assert_close(seq.g.cpu().numpy(), g_last, "prefill boundaries", max_abs=1e-3, rel_l2=1e-5)
        assert np.array_equal(seq.tok.cpu().numpy(), toks[np.arange(B), lens])
        d2t_image = set((np.arange(G.draft_vocab) + wts.d2t).tolist())
        report = []
        for r in range(rounds):
            n = synth.imposed_accept_lengths(B, gamma, seed=seed + 10 + r)
            kv_lo = min(st.kv_len for st in states.values())
            states, out, na, bo, vaux, _ = run_round(model, dr, seq, states, gamma, n, seed=seed + 10 + r,
                                                     kv_lo=kv_lo, stepwise=True, report=report)
            dt = out["draft_tok"].cpu().numpy()
            assert set(dt.ravel().tolist()) <= d2t_image
            venc = O.encode(dr, vaux)
            for b in range(B):
                if b in states:
                    tracked[b] = Tracked(states[b].kv_len, states[b].g, states[b].tok)
                else:
                    tracked[b] = check_rebuild_tracked(seq, dr, b, tracked[b], dt[b], int(na[b]), int(bo[b]),
                                                       venc[b], kv_format)
        rep = np.array([x[2:] for x in report])
        print(f"\n{kv_format} B{B} gamma {gamma}: {len(report)} chain steps, max-abs error per step: "
              f"logits median {np.median(rep[:, 0]):.2e} max {rep[:, 0].max():.2e}; "
              f"g median {np.median(rep[:, 1]):.2e} max {rep[:, 1].max():.2e}")
        # the whole committed cache of the followed sequences after all rounds
        check_state(seq, states, f"after {rounds} rounds")
        assert model.status() == 0
    finally:
        model.close()


@pytest.fixture(scope="module")
def ctx32k(full_drafter):
    """Batch 4 at context 32768: prompts, features, and sequence 0 prefilled by the oracle
    (its raw k / v serve both cache formats)."""
    _, dr = full_drafter
    B, P = 4, 32768
    lens = np.full(B, P, np.int32)
    toks, aux = _inputs(B, lens, seed=500)
    prefilled = oracle_prefill(dr, toks, aux, lens, which=[0])
    return lens, toks, aux, prefilled


def test_batch4_context32768_gamma7_16_rounds(full_drafter, ctx32k):
    lens, toks, aux, prefilled = ctx32k
    _run_case(full_drafter, lens, 7, 16, [0], prefilled, toks, aux, seed=510, kv_format="bf16")


def test_batch4_context32768_gamma7_quantized_kv(full_drafter, ctx32k):
    lens, toks, aux, prefilled = ctx32k
    _run_case(full_drafter, lens, 7, 4, [0], prefilled, toks, aux, seed=540, kv_format="q8_0/q5_1")


def test_batch8_ragged_512_8192_gamma5(full_drafter):
    _, dr = full_drafter
    B = 8
    lens = synth.ragged_lengths(B, 512, 8192, seed=600)
    toks, aux = _inputs(B, lens, seed=601)
    follow = sorted({int(np.argmax(lens)), int(np.argmin(lens))})
    prefilled = oracle_prefill(dr, toks, aux, lens, which=follow)
    _run_case(full_drafter, lens, 5, 4, follow, prefilled, toks, aux, seed=610, kv_format="bf16")
