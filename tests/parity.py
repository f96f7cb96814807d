"""Shared helpers of the GPU-vs-oracle parity tests.

The bar (from the drafter's accuracy requirement): token ids, accept lengths, KV
positions and rewind state bit-exact, provided the oracle's top-2 logit margin exceeds
1e-2 (on a closer call the GPU's id must be within 1e-2 of the oracle's maximum and the
oracle then follows the GPU's choice); float outputs (g, logits, KV) within max-abs 2e-2
and relative L2 1e-2.
"""
from __future__ import annotations

import numpy as np

from oracle import eagle3_oracle as O

MARGIN = 1e-2
MAX_ABS = 2e-2
REL_L2 = 1e-2


def bf16_bits_to_f64(bits) -> np.ndarray:
    return O.widen_bf16(np.asarray(bits).view(np.uint16))


def assert_close(got, want, what: str, max_abs=MAX_ABS, rel_l2=REL_L2):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, f"{what}: shape {got.shape} vs {want.shape}"
    err = np.abs(got - want)
    ma = float(err.max()) if err.size else 0.0
    denom = float(np.linalg.norm(want)) or 1.0
    rl = float(np.linalg.norm(got - want)) / denom
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert ma <= max_abs and rl <= rel_l2, f"{what}: max-abs {ma:.3e}, rel-L2 {rl:.3e}"
    return ma, rl


def top2_margin(logits: np.ndarray) -> float:
    s = np.sort(logits)
    return float(s[-1] - s[-2])


class ChainFollower:
    """Stepper for oracle.draft_chain that checks the GPU's choice at each step and
    feeds the GPU's token forward (so a near tie cannot desynchronise the chains)."""

    def __init__(self, dr: O.Drafter, gpu_ids, gpu_toks):
        self.dr = dr
        self.gpu_ids = [int(x) for x in gpu_ids]
        self.gpu_toks = [int(x) for x in gpu_toks]
        self.ties = 0

    def __call__(self, j: int, so) -> int:
        gid = self.gpu_ids[j]
        if top2_margin(so.logits) > MARGIN:
            assert gid == so.draft_id, f"step {j}: GPU id {gid} vs oracle {so.draft_id}"
        else:
            self.ties += 1
            assert so.logits[gid] >= so.logits.max() - MARGIN, f"step {j}: GPU id {gid} not near max"
        assert self.gpu_toks[j] == self.dr.d2t_map(gid), f"step {j}: d2t of {gid}"
        return self.gpu_toks[j]


def oracle_chain_following(dr, st, gamma, gpu_ids, gpu_toks):
    f = ChainFollower(dr, gpu_ids, gpu_toks)
    ch = O.draft_chain(dr, st, gamma, stepper=f)
    return ch, f
