"""The speculative loop on the GPU, through the C ABI, on the small drafter (n_embd 256,
4:1 GQA, head 64, draft vocab 1024 -> 4096).

* Lossless loop ("Add the Eagle3Speculator module for speculative decoding", PR body: the
  shifted speculative loop reproduces greedy decoding; "memra_engine/eagle.rs",
  ``generate_spec_eagle``: greedy output identical): draft_chain -> rewind -> target
  predictions -> accept -> rebuild_after_verify against a synthetic deterministic target,
  with nothing imposed: the stream the loop emits (accepted drafts + bonus of every round)
  must be the target's own greedy stream.  The target's next token after a history is
  the oracle drafter's first draft from that history's state (so drafts are often
  accepted), except where a hash of the history picks another token (so they are also
  rejected).
* No host synchronisation ("feat(eagle3) ... drafter forward pass", review comments on
  the per-token device-to-host copy and stream sync): a whole round is enqueued behind a
  kernel that keeps the stream busy, and every call returns while the stream is still
  busy; the round's outputs are then checked against the oracle.
"""
import time

import numpy as np
import pytest
import torch

from eagle_speculative_decode_gb300 import synth
from eagle_speculative_decode_gb300.runtime import DraftModel
from oracle import eagle3_oracle as O
from parity import check_state, gpu_prefill, oracle_chain_following, oracle_prefill

pytestmark = pytest.mark.gpu
G = synth.TINY


@pytest.fixture(scope="module")
def tiny(built_lib):
    wts = synth.make_weights(G, seed=0)
    dr = O.Drafter(G, wts.bits, wts.d2t)
    return wts, dr


def _fnv(tokens) -> int:
    h = 0xCBF29CE484222325
    for t in tokens:
        h = ((h ^ (int(t) & 0xFFFFFFFF)) * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


class SyntheticTarget:
    """A deterministic greedy target over token histories t_0..t_N.  Its features at
    position p are a fixed seeded draw (they depend on the position only)."""

    def __init__(self, dr, aux_all):
        self.dr, self.aux_all = dr, aux_all

    def state_after(self, st: O.SeqState, tokens_after) -> O.SeqState:
        """Drafter state of the history extended by tokens_after (each token commits the
        previous boundary and becomes the new one)."""
        for t in tokens_after:
            N = st.kv_len + 1                     # the boundary token's position
            st = O.rebuild_after_verify(self.dr, st, 0, [], int(t), self.aux_all[N:N + 1])
        return st

    def next_token(self, history, st: O.SeqState) -> int:
        """Greedy next token after `history`, whose drafter state is st."""
        h = _fnv(history)
        if h % 10 < 3:
            return int((h >> 20) % G.target_vocab)
        return O.draft_step(self.dr, int(st.tok), st.g, st.k, st.v, st.kv_len).target_id


def test_lossless_loop_reproduces_target_greedy_stream(tiny):
    wts, dr = tiny
    P, gamma, want_tokens = 16, 3, 60
    max_cache = 128
    aux_all = synth.make_aux((max_cache + 8,), G, seed=900)
    prompt = synth.make_tokens((P,), G, seed=901)
    target = SyntheticTarget(dr, aux_all)
    # the target's own greedy stream, token by token, from the state of the prompt
    # t_0..t_{P-1} (boundary t_{P-1}); st0 is then the state after its first token t_P
    hist = list(prompt)
    st_prompt = O.prefill(dr, prompt[:P - 1], int(prompt[P - 1]), aux_all[:P - 1])
    st0 = target.state_after(st_prompt, [target.next_token(hist, st_prompt)])
    ref, st = [st0.tok], st0
    while len(ref) < want_tokens + gamma + 2:
        nxt = target.next_token(hist + ref, st)
        st = target.state_after(st, [nxt])
        ref.append(nxt)

    model = DraftModel(wts, max_batch=1, max_gamma=gamma, max_cache_len=max_cache, page_size=16)
    try:
        seq = model.new_state(1)
        toks = np.array([list(prompt) + [st0.tok]], dtype=np.int32)
        gpu_prefill(seq, model, toks, aux_all[None, :P], np.array([P]))
        dev = model.device
        emitted, committed = [st0.tok], st0       # target-side view of the committed history
        accepted_rounds, rounds = 0, 0
        while len(emitted) < want_tokens:
            out = seq.draft_chain(gamma)
            seq.rewind()
            d = out["draft_tok"].cpu().numpy()[0]
            # the target's prediction after each prefix of the drafts
            y, s = [], committed
            for i in range(gamma + 1):
                y.append(target.next_token(hist + emitted + list(d[:i]), s))
                if i < gamma:
                    s = target.state_after(s, [d[i]])
            n_acc, bonus = seq.accept(out["draft_tok"], torch.tensor([y], dtype=torch.int32, device=dev),
                                      out["gamma_eff"])
            N = committed.kv_len + 1
            vaux = torch.from_numpy(aux_all[N:N + gamma + 1][None].view(np.int16)).to(dev)
            seq.rebuild_after_verify(n_acc, out["draft_tok"], bonus, vaux)
            n, b = int(n_acc.item()), int(bonus.item())
            assert (n, b) == O.accept(d, y)
            new = [int(t) for t in d[:n]] + [b]
            emitted += new
            committed = target.state_after(committed, new)
            accepted_rounds += n > 0
            rounds += 1
        torch.cuda.synchronize()
        assert emitted[:want_tokens] == ref[:want_tokens]
        assert accepted_rounds >= rounds // 4, f"only {accepted_rounds} of {rounds} rounds accepted a draft"
        # the GPU's committed drafter state is the target-side state of the emitted history
        check_state(seq, {0: committed}, "after the loop")
        assert model.status() == 0
    finally:
        model.close()


def test_round_enqueues_without_host_sync(tiny):
    wts, dr = tiny
    B, gamma = 2, 3
    model = DraftModel(wts, max_batch=B, max_gamma=gamma, max_cache_len=100, page_size=16)
    try:
        lens = np.array([24, 11])
        toks = synth.make_tokens((B, 25), G, seed=910)
        aux = synth.make_aux((B, 24), G, seed=911)
        dev = model.device
        seq = model.new_state(B)
        gpu_prefill(seq, model, toks, aux, lens)
        # capture the chain's graph once (a capture is set-up, not the steady state)
        out = seq.draft_chain(gamma)
        seq.rewind()
        torch.cuda.synchronize()
        states = oracle_prefill(dr, toks, aux, lens)
        y = torch.from_numpy(synth.make_tokens((B, gamma + 1), G, seed=912)).to(dev)
        vaux = torch.from_numpy(synth.make_aux((B, gamma + 1), G, seed=913).view(np.int16)).to(dev)
        n_acc = torch.empty(B, dtype=torch.int32, device=dev)
        bonus = torch.empty(B, dtype=torch.int32, device=dev)
        stream = torch.cuda.current_stream()
        # keep the stream busy for ~0.5 s (a kernel that spins on the clock and returns)
        torch.cuda._sleep(int(1.0e9))
        t0 = time.perf_counter()
        out = seq.draft_chain(gamma, out=out)
        busy_after_chain = not stream.query()
        seq.rewind()
        seq.accept(out["draft_tok"], y, out["gamma_eff"], n_acc=n_acc, bonus=bonus)
        # n_acc_host only advances the wrapper's host mirror of kv_len (read by the next
        # chain's capacity check); giving it a placeholder keeps the wrapper from reading
        # n_acc back, and the mirror is refreshed after the synchronisation below
        seq.rebuild_after_verify(n_acc, out["draft_tok"], bonus, vaux, n_acc_host=np.zeros(B, np.int32))
        enqueue_s = time.perf_counter() - t0
        busy_after_round = not stream.query()
        assert busy_after_chain and busy_after_round, "a call waited for the device"
        assert enqueue_s < 0.3, f"enqueueing the round took {enqueue_s:.3f} s"
        torch.cuda.synchronize()
        seq.kv_len_host = seq.kv_len.cpu().numpy()
        # the round's results against the oracle
        dt = out["draft_tok"].cpu().numpy()
        di = out["draft_id"].cpu().numpy()
        na, bo = n_acc.cpu().numpy(), bonus.cpu().numpy()
        yh = y.cpu().numpy()
        new_states = {}
        for b, st in states.items():
            oracle_chain_following(dr, st, gamma, di[b], dt[b])
            assert (na[b], bo[b]) == O.accept(dt[b], yh[b], gamma)
            new_states[b] = O.rebuild_after_verify(dr, st, int(na[b]), dt[b], int(bo[b]),
                                                   vaux[b].cpu().numpy().view(np.uint16))
        check_state(seq, new_states, "round behind a busy stream")
        assert model.status() == 0
    finally:
        model.close()
