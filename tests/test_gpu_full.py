"""GPU parity on the full drafter geometry (n_embd 4096, q 4096x8192, k/v 1024x8192,
16:4 GQA with head_dim 256, RoPE 64/256 at theta 1e7, n_ff 12288, draft vocab 32000 ->
target vocab 248320), through the C ABI, against the CPU oracle.

Sizes where the oracle runs the whole path in seconds are compared element by element
(batch 1 with a 512-token prompt, the benchmark's headline configuration; a ragged
batch of 8).  At the batch-64 / 2048-context size the benchmark also times, the oracle
checks what it can compute one by one (prefill and rebuild KV entries at sampled and at
all rebuilt positions, the first speculative entry of every chain, accept walks) plus two
sampled sequences end to end.
"""
import numpy as np
import pytest
import torch

from eagle_speculative_decode_gb300 import synth
from eagle_speculative_decode_gb300.runtime import DraftModel
from oracle import eagle3_oracle as O
from parity import (assert_close, assert_close_bf16, bf16_bits_to_f64, check_state, gpu_prefill,
                    oracle_prefill, run_round)

pytestmark = pytest.mark.gpu
G = synth.FULL


@pytest.fixture(scope="module")
def full(full_drafter):
    return full_drafter


def _prompt(batch, lens, seed):
    P_max = int(max(lens))
    toks = synth.make_tokens((batch, P_max + 1), G, seed)
    aux = synth.make_aux((batch, P_max), G, seed)
    return toks, aux


def test_batch1_prompt512_gamma3_rounds(full):
    """The headline configuration, every output compared, two rounds."""
    wts, dr = full
    model = DraftModel(wts, max_batch=1, max_gamma=3, max_cache_len=1024, page_size=64)
    try:
        lens = np.array([512])
        toks, aux = _prompt(1, lens, seed=101)
        seq = model.new_state(1)
        gpu_prefill(seq, model, toks, aux, lens)
        torch.cuda.synchronize()
        states = oracle_prefill(dr, toks, aux, lens)
        check_state(seq, states, "prefill")
        for r, n in enumerate([3, 1]):
            states = run_round(model, dr, seq, states, 3, np.array([n]), seed=110 + r)[0]
    finally:
        model.close()


@pytest.mark.parametrize("attention", [0, 1], ids=["attn_cuda_cores", "attn_tensor_cores"])
def test_ragged_batch8_gamma5_random_pages(full, attention):
    """Ragged prompts (shortened from the 512-8192 range so that the oracle runs every
    position), gamma 5, accept lengths uniform in 0..gamma, non-contiguous pages; under
    both decode attention kernels (head 256, 4 q heads per kv head, 64-key units)."""
    wts, dr = full
    B, gamma, ps, max_cache = 8, 5, 64, 1024
    model = DraftModel(wts, max_batch=B, max_gamma=gamma, max_cache_len=max_cache, page_size=ps)
    model.set_attention(attention)
    try:
        lens = synth.ragged_lengths(B, 64, 384, seed=120)
        toks, aux = _prompt(B, lens, seed=121)
        pt = synth.page_table(B, max_cache // ps, seed=122)
        seq = model.new_state(B, page_table=pt)
        gpu_prefill(seq, model, toks, aux, lens)
        torch.cuda.synchronize()
        states = oracle_prefill(dr, toks, aux, lens)
        check_state(seq, states, "prefill")
        for r in range(2):
            n = synth.imposed_accept_lengths(B, gamma, seed=130 + r)
            states = run_round(model, dr, seq, states, gamma, n, seed=130 + r)[0]
    finally:
        model.close()


def test_batch64_context2048_sampled(full):
    """Batch 64 at context 2048, gamma 3 (the benchmark's batched launch configuration)."""
    wts, dr = full
    B, gamma, ps, P = 64, 3, 64, 2048
    model = DraftModel(wts, max_batch=B, max_gamma=gamma, max_cache_len=2048 + 64, page_size=ps)
    try:
        lens = np.full(B, P, np.int32)
        toks, aux = _prompt(B, lens, seed=140)
        pt = synth.page_table(B, (2048 + 64) // ps, seed=141)
        seq = model.new_state(B, page_table=pt)
        gpu_prefill(seq, model, toks, aux, lens)
        torch.cuda.synchronize()
        rng = np.random.default_rng(142)
        # prefill KV entries at sampled (sequence, position) pairs, one by one
        bs = rng.integers(0, B, 48)
        ps_ = rng.integers(0, P - 1, 48)
        for b, p in zip(bs, ps_):
            g_p = O.encode(dr, aux[b, p])
            k, v = O.kv_entry(dr, int(toks[b, p + 1]), g_p, int(p))
            kg, vg = seq.kv_entries(int(b), int(p), int(p) + 1)
            assert_close_bf16(bf16_bits_to_f64(kg[0]), k, f"prefill K b{b} p{p}")
            assert_close_bf16(bf16_bits_to_f64(vg[0]), v, f"prefill V b{b} p{p}")
        # boundary of every sequence
        g_all = seq.g.cpu().numpy()
        want = O.encode(dr, aux[np.arange(B), lens - 1])
        assert_close(g_all, want, "boundary g", max_abs=1e-3, rel_l2=1e-5)
        assert np.array_equal(seq.tok.cpu().numpy(), toks[np.arange(B), lens])
        # two sampled sequences end to end (the oracle prefills them in full)
        states = oracle_prefill(dr, toks, aux, lens, which=[3, 57])
        n = synth.imposed_accept_lengths(B, gamma, seed=143, p_accept=0.6)
        new_states, out, na, bo, vaux, ties = run_round(model, dr, seq, states, gamma, n, seed=143,
                                                        kv_lo=P - 2)
        # every sequence: first speculative entry = the boundary pair at position L,
        # and the rebuilt entries L..L+n are the pairs the rebuild rule names
        dt = out["draft_tok"].cpu().numpy()
        assert np.all((dt >= 0) & (dt < G.target_vocab))
        d2t_image = set((np.arange(G.draft_vocab) + wts.d2t).tolist())
        assert set(dt.ravel().tolist()) <= d2t_image
        L = lens - 1
        kv_len = seq.kv_len.cpu().numpy()
        assert np.array_equal(kv_len, L + na + 1)
        venc = O.encode(dr, vaux)
        for b in rng.choice(B, 16, replace=False):
            b = int(b)
            pairs = [(int(toks[b, lens[b]]), want[b])] + \
                    [(int(dt[b, i - 1]), venc[b, i - 1]) for i in range(1, int(na[b]) + 1)]
            kg, vg = seq.kv_entries(b, int(L[b]), int(L[b]) + len(pairs))
            for i, (t, gg) in enumerate(pairs):
                k, v = O.kv_entry(dr, t, gg, int(L[b]) + i)
                assert_close_bf16(bf16_bits_to_f64(kg[i]), k, f"rebuilt K b{b} i{i}")
                assert_close_bf16(bf16_bits_to_f64(vg[i]), v, f"rebuilt V b{b} i{i}")
            assert_close(seq.g[b].cpu().numpy(), venc[b, int(na[b])], f"new boundary b{b}",
                         max_abs=1e-3, rel_l2=1e-5)
            assert int(seq.tok[b].item()) == int(bo[b])
    finally:
        model.close()
