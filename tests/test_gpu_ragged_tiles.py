"""GPU parity on a drafter whose row counts leave partial tiles: n_embd 2048 (every
single-item INT4 projection, down included, runs on the tensor-core GEMV, whose tiles are
16 whole rows) and a draft vocabulary of 3002 rows (3002 = 187 x 16 + 10, and 3002 = 750 x
4 + 2 for the bf16 GEMV's four-row tiles), so that the last tile of the lm_head launch holds
fewer rows than a stage and sits on one CTA of the round robin.  Full rounds through the
C ABI against the oracle, bf16 and INT4 weights, one sequence (single-item launches) and a
ragged batch of 5 (several items per launch)."""
import numpy as np
import pytest

from eagle_speculative_decode_gb300 import synth
from eagle_speculative_decode_gb300.runtime import DraftModel
from oracle import eagle3_oracle as O
from test_gpu_int4 import _rounds

pytestmark = pytest.mark.gpu

RAGGED = synth.Geometry(n_embd=2048, n_head=8, n_head_kv=2, head_dim=256, rope_dims=64,
                        rope_theta=1e7, rms_eps=1e-6, n_ff=2048, draft_vocab=3002,
                        target_vocab=8192)


@pytest.mark.parametrize("weights", ["bf16", "int4"])
def test_partial_last_tiles(built_lib, weights):
    g = RAGGED
    assert g.draft_vocab % 16 and g.draft_vocab % 4
    if weights == "int4":
        wts = synth.make_int4_weights(g, seed=41)
        dr = O.Drafter(g, wts.bits, wts.d2t, int4=wts.int4)
    else:
        wts = synth.make_weights(g, seed=41)
        dr = O.Drafter(g, wts.bits, wts.d2t)
    model = DraftModel(wts, max_batch=5, max_gamma=3, max_cache_len=192, page_size=32)
    try:
        _rounds(g, model, dr, np.array([96]), 3, [140, 141], seed=142, pages=False)
        _rounds(g, model, dr, synth.ragged_lengths(5, 8, 150, seed=143), 3, [144], seed=145)
    finally:
        model.close()
