"""eagle3_lmhead_argmax_noalloc: the lm_head + argmax + d2t kernel for callers that cannot
allocate device memory (for instance code running under CUDA graph capture, or a runtime
whose memory plan is fixed before the first call).  Its scratch lives in a static device
array inside the library.  Checked through the C ABI, on two calls in a row, against the
draft chain's own outputs for the same rows (the chain kept on the same CUDA-core GEMV)
and against the oracle's lm_head . (RMSNorm(x) * final_norm) with its argmax and d2t map.
Collected last on purpose."""
import numpy as np
import pytest
import torch

from eagle_speculative_decode_gb300 import binding as Bd
from eagle_speculative_decode_gb300 import synth
from eagle_speculative_decode_gb300.runtime import DraftModel
from oracle import eagle3_oracle as O
from parity import MARGIN, assert_close, gpu_prefill, top2_margin

pytestmark = pytest.mark.gpu
G = synth.TINY


def _call(model, x, rows, ids, tgt, logits, d2t=None):
    w = model.w
    Bd.eagle3_lmhead_argmax_noalloc(
        w["lm_head"].data_ptr(), w["final_norm"].data_ptr(),
        (model.d2t if d2t is None else d2t).data_ptr(), x.data_ptr(), rows, G.n_embd,
        G.draft_vocab, G.target_vocab, G.rms_eps,
        None if ids is None else ids.data_ptr(), tgt.data_ptr(),
        None if logits is None else logits.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_lmhead_matches_chain_and_oracle(built_lib):
    wts = synth.make_weights(G, seed=5)
    B, gamma = 9, 2  # 9 rows: more than one launch of the kernel per call
    model = DraftModel(wts, max_batch=B, max_gamma=gamma, max_cache_len=64, page_size=16)
    try:
        # the chain's lm_head on the same CUDA-core GEMV as the entry point (3+ rows would
        # otherwise take the tensor-core GEMM, whose float32 sums round differently)
        model.set_tc_min_items(B + 1)
        lens = synth.ragged_lengths(B, 3, 20, seed=6)
        P_max = int(lens.max())
        toks = synth.make_tokens((B, P_max + 1), G, seed=7)
        aux = synth.make_aux((B, P_max), G, seed=8)
        seq = model.new_state(B)
        gpu_prefill(seq, model, toks, aux, lens)
        out = seq.draft_chain(gamma, debug=True)
        torch.cuda.synchronize()
        dev = model.device
        for j in range(gamma):  # two calls in a row, each checked
            x = out["g"][:, j, :].contiguous()
            ids = torch.full((B,), -7, dtype=torch.int32, device=dev)
            tgt = torch.full((B,), -7, dtype=torch.int32, device=dev)
            logits = torch.empty(B, G.draft_vocab, dtype=torch.float32, device=dev)
            _call(model, x, B, ids, tgt, logits)
            torch.cuda.synchronize()
            got_ids, got_tgt = ids.cpu().numpy(), tgt.cpu().numpy()
            got_logits = logits.cpu().numpy()
            # same kernel, same rows: identical to the chain's own step
            assert np.array_equal(got_ids, out["draft_id"][:, j].cpu().numpy())
            assert np.array_equal(got_tgt, out["draft_tok"][:, j].cpu().numpy())
            assert_close(got_logits, out["logits"][:, j].cpu().numpy(), f"logits vs chain, step {j}")
            # the oracle on the same rows
            want, want_ids = O.target_verify(wts.bits["lm_head"], wts.bits["final_norm"],
                                             x.cpu().numpy().astype(np.float64), G.rms_eps)
            assert_close(got_logits, want, f"logits vs oracle, step {j}")
            dr = O.Drafter(G, wts.bits, wts.d2t)
            for r in range(B):
                if top2_margin(want[r]) > MARGIN:
                    assert got_ids[r] == want_ids[r], f"row {r}: {got_ids[r]} vs oracle {want_ids[r]}"
                else:
                    assert want[r, got_ids[r]] >= want[r].max() - MARGIN
                assert got_tgt[r] == dr.d2t_map(int(got_ids[r]))
        seq.rewind()
        # more rows than the static scratch holds are refused
        big = torch.zeros(65, G.n_embd, dtype=torch.float32, device=dev)
        t65 = torch.zeros(65, dtype=torch.int32, device=dev)
        with pytest.raises(Bd.Eagle3Error) as ei:
            _call(model, big, 65, None, t65, None)
        assert ei.value.code == Bd.EAGLE3_ERR_INVALID_ARG
        # a d2t table mapping every id past the target vocabulary: the kernel's own range
        # check marks each row -1 (there is no status word to raise)
        bad_d2t = torch.full((G.draft_vocab,), G.target_vocab, dtype=torch.int64, device=dev)
        x = out["g"][:, 0, :].contiguous()
        ids = torch.zeros(B, dtype=torch.int32, device=dev)
        tgt = torch.zeros(B, dtype=torch.int32, device=dev)
        _call(model, x, B, ids, tgt, None, d2t=bad_d2t)
        torch.cuda.synchronize()
        assert np.all(ids.cpu().numpy() == -1) and np.all(tgt.cpu().numpy() == -1)
        # and the next call with the valid table is correct again
        _call(model, x, B, ids, tgt, None)
        torch.cuda.synchronize()
        assert np.array_equal(tgt.cpu().numpy(), out["draft_tok"][:, 0].cpu().numpy())
    finally:
        model.close()
