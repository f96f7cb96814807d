"""eagle3_lmhead_argmax_noalloc: the lm_head + argmax + d2t kernel for callers that cannot
allocate device memory (for instance code running under CUDA graph capture, or a runtime
whose memory plan is fixed before the first call).  Its scratch lives in a static device
array inside the library.  Checked through the C ABI against the draft chain's own
outputs for the same rows, on two calls in a row.  Collected last on purpose."""
import numpy as np
import pytest
import torch

from eagle_speculative_decode_gb300 import binding as Bd
from eagle_speculative_decode_gb300 import synth
from eagle_speculative_decode_gb300.runtime import DraftModel
from parity import assert_close, gpu_prefill

pytestmark = pytest.mark.gpu
G = synth.TINY


def test_noalloc_lmhead_matches_draft_chain(built_lib):
    wts = synth.make_weights(G, seed=5)
    B, gamma = 9, 2  # 9 rows: more than one launch of the kernel per call
    model = DraftModel(wts, max_batch=B, max_gamma=gamma, max_cache_len=64, page_size=16)
    try:
        lens = synth.ragged_lengths(B, 3, 20, seed=6)
        P_max = int(lens.max())
        toks = synth.make_tokens((B, P_max + 1), G, seed=7)
        aux = synth.make_aux((B, P_max), G, seed=8)
        seq = model.new_state(B)
        gpu_prefill(seq, model, toks, aux, lens)
        out = seq.draft_chain(gamma, debug=True)
        torch.cuda.synchronize()
        dev = model.device
        w = model.w
        for j in range(gamma):  # two calls in a row, each checked
            x = out["g"][:, j, :].contiguous()
            ids = torch.full((B,), -7, dtype=torch.int32, device=dev)
            tgt = torch.full((B,), -7, dtype=torch.int32, device=dev)
            logits = torch.empty(B, G.draft_vocab, dtype=torch.float32, device=dev)
            Bd.eagle3_lmhead_argmax_noalloc(
                w["lm_head"].data_ptr(), w["final_norm"].data_ptr(), model.d2t.data_ptr(),
                x.data_ptr(), B, G.n_embd, G.draft_vocab, G.target_vocab, G.rms_eps,
                ids.data_ptr(), tgt.data_ptr(), logits.data_ptr(),
                torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            assert np.array_equal(ids.cpu().numpy(), out["draft_id"][:, j].cpu().numpy())
            assert np.array_equal(tgt.cpu().numpy(), out["draft_tok"][:, j].cpu().numpy())
            assert_close(logits.cpu().numpy(), out["logits"][:, j].cpu().numpy(), f"logits step {j}")
        seq.rewind()
        # more rows than the static scratch holds are refused
        big = torch.zeros(65, G.n_embd, dtype=torch.float32, device=dev)
        t65 = torch.zeros(65, dtype=torch.int32, device=dev)
        with pytest.raises(Bd.Eagle3Error) as ei:
            Bd.eagle3_lmhead_argmax_noalloc(
                w["lm_head"].data_ptr(), w["final_norm"].data_ptr(), model.d2t.data_ptr(),
                big.data_ptr(), 65, G.n_embd, G.draft_vocab, G.target_vocab, G.rms_eps,
                None, t65.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
        assert ei.value.code == Bd.EAGLE3_ERR_INVALID_ARG
    finally:
        model.close()
