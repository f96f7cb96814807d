"""Shared helpers of the GPU-vs-oracle parity tests.

The bar (from the drafter's accuracy requirement): token ids, accept lengths, KV
positions and rewind state bit-exact, provided the oracle's top-2 logit margin exceeds
1e-2 (on a closer call the GPU's id must be within 1e-2 of the oracle's maximum and the
oracle then follows the GPU's choice); float outputs (g, logits, KV) within max-abs 2e-2
and relative L2 1e-2.
"""
from __future__ import annotations

import copy

import numpy as np
import torch

from eagle_speculative_decode_gb300 import binding as Bd
from eagle_speculative_decode_gb300 import synth
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


def bf16_ulp(x) -> np.ndarray:
    """Unit in the last place of bf16 at |x| (8 significant bits)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, 2.0 ** (e - 7), 2.0 ** -133)


def assert_close_bf16(got, want, what: str, max_abs=MAX_ABS, rel_l2=REL_L2):
    """Values stored as bf16 (the KV cache): each element within max(max_abs, one bf16 ulp
    of the oracle's value) -- where the float32 and float64 results straddle a rounding
    boundary the two stored values differ by one ulp -- and relative L2 within rel_l2."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, f"{what}: shape {got.shape} vs {want.shape}"
    err = np.abs(got - want)
    bound = np.maximum(max_abs, bf16_ulp(want) * 1.0000001)
    bad = err > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond max(2e-2, 1 ulp); worst {float(err.max()):.3e}"
    denom = float(np.linalg.norm(want)) or 1.0
    rl = float(np.linalg.norm(got - want)) / denom
    assert rl <= rel_l2, f"{what}: rel-L2 {rl:.3e}"


def kv_values(raw, kv_format: str, which: str) -> np.ndarray:
    """Stored K (which "k") or V rows as float64 [..., H_kv, d], decoded with the oracle's
    unpackers."""
    raw = np.asarray(raw)
    if kv_format == "bf16":
        return bf16_bits_to_f64(raw)
    if which == "k":
        d16, q = O.unpack_q8_0(raw.reshape(raw.shape[:-1] + (-1, O.Q8_0_BLOCK_BYTES)))
        return O.dequantize_q8_0(d16, q).astype(np.float64)
    d16, m16, q = O.unpack_q5_1(raw.reshape(raw.shape[:-1] + (-1, O.Q5_1_BLOCK_BYTES)))
    return O.dequantize_q5_1(d16, m16, q).astype(np.float64)


QUANT_REL = 1e-5   # float32 vs float64 k / v inputs to the quantizer, relative to the block's max |x|


def _f16_bracket(x, eps_abs):
    """The fp16 values that x moved by at most eps_abs can round to (nearest even)."""
    lo = np.asarray(x - eps_abs, dtype=np.float32).astype(np.float16).astype(np.float64)
    hi = np.asarray(x + eps_abs, dtype=np.float32).astype(np.float16).astype(np.float64)
    return lo, hi


def assert_quant_valid(raw, x, which: str, what: str, rel=QUANT_REL):
    """The stored q8_0 (which "k") / q5_1 ("v") blocks `raw` are a valid encoding of the
    oracle's unstored values x [..., d] when the implementation's float32 inputs may differ
    from x by delta = rel * max|x| of the block: every header field and every code must be
    one that some input within delta of x produces under the encoding's rule.  Away from
    rounding boundaries that is exactly the oracle's encoding; at a boundary either
    neighbour is accepted (where several results are correct, check that the one given is
    valid)."""
    raw = np.asarray(raw, dtype=np.uint8)
    x = np.asarray(x, dtype=np.float64)
    xb = x.reshape(-1, O.QK)
    delta = rel * np.abs(xb).max(axis=-1) + 1e-7                     # [blocks]
    if which == "k":
        d16, q = O.unpack_q8_0(raw.reshape(-1, O.Q8_0_BLOCK_BYTES))
        d = d16.astype(np.float64)
        s = np.abs(xb).max(axis=-1) / 127.0
        lo, hi = _f16_bracket(s, delta / 127.0)
        bad_h = (d < lo) | (d > hi)
        assert not bad_h.any(), f"{what}: q8_0 scale outside its rounding bracket in {int(bad_h.sum())} blocks"
        dd = np.where(d > 0, d, 1.0)[:, None]
        t_lo = (xb - delta[:, None]) / dd
        t_hi = (xb + delta[:, None]) / dd
        c_lo = np.clip(np.rint(t_lo), -127, 127)
        c_hi = np.clip(np.rint(t_hi), -127, 127)
        code = q.astype(np.float64)
    else:
        d16, m16, q = O.unpack_q5_1(raw.reshape(-1, O.Q5_1_BLOCK_BYTES))
        d, m = d16.astype(np.float64), m16.astype(np.float64)
        s = (xb.max(axis=-1) - xb.min(axis=-1)) / 31.0
        lo, hi = _f16_bracket(s, 2 * delta / 31.0)
        mlo, mhi = _f16_bracket(xb.min(axis=-1), delta)
        bad_h = (d < lo) | (d > hi) | (m < mlo) | (m > mhi)
        assert not bad_h.any(), f"{what}: q5_1 scale / minimum outside their rounding brackets in {int(bad_h.sum())} blocks"
        dd = np.where(d > 0, d, 1.0)[:, None]
        t_lo = (xb - delta[:, None] - m[:, None]) / dd
        t_hi = (xb + delta[:, None] - m[:, None]) / dd
        c_lo = np.clip(np.rint(t_lo), 0, 31)
        c_hi = np.clip(np.rint(t_hi), 0, 31)
        code = q.astype(np.float64)
    zero = (d == 0)[:, None]
    c_lo = np.where(zero, 0, c_lo)
    c_hi = np.where(zero, 0, c_hi)
    bad = (code < c_lo) | (code > c_hi)
    assert not bad.any(), f"{what}: {int(bad.sum())} codes not a nearest code of any input within delta"
    n_edge = int(np.sum(c_lo != c_hi))
    assert n_edge <= max(4, code.size // 100), f"{what}: {n_edge} codes on boundaries (delta too wide?)"


def assert_bf16_valid(bits, x, what: str, rel=QUANT_REL):
    """Stored bf16 values `bits` [..., d] are a valid rounding of the oracle's unstored
    values x when the implementation's float32 inputs may differ from x by delta = rel *
    max|x| of the row: each must lie between the roundings of x - delta and x + delta.
    Away from a rounding boundary that is exactly the oracle's own bf16 value."""
    got = bf16_bits_to_f64(bits)
    x = np.asarray(x, dtype=np.float64)
    delta = rel * np.abs(x).max(axis=-1, keepdims=True) + 1e-7
    lo, hi = O.round_bf16(x - delta), O.round_bf16(x + delta)
    bad = (got < lo) | (got > hi)
    assert not bad.any(), f"{what}: {int(bad.sum())} values not a rounding of any input within delta"
    # not vacuous: a value lies within delta of a rounding boundary with probability about
    # 2 delta / ulp (bf16's ulp scales with the value, so small values often do); far more
    # brackets than that would mean delta lets wrong values through
    n_edge = int(np.sum(lo != hi))
    expect = float(np.minimum(1.0, 2 * delta / bf16_ulp(x)).sum())
    assert n_edge <= 2 * expect + 8, f"{what}: {n_edge} values on boundaries, about {expect:.0f} expected"


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


def with_kv_format(dr: O.Drafter, kv_format: str) -> O.Drafter:
    """The same oracle drafter (its widened weights shared, not copied) storing its KV in
    another format."""
    if kv_format not in O.KV_FORMATS:
        raise ValueError(kv_format)
    d = copy.copy(dr)
    d.kv_format = kv_format
    return d


def stored_state(st: O.SeqState, kv_format: str) -> O.SeqState:
    """A prefilled oracle state with its entries stored in another KV format (the raw
    float64 k / v are the same in every format)."""
    return O.SeqState(O.store_k(st.k_raw, kv_format), O.store_v(st.v_raw, kv_format), st.g.copy(),
                      int(st.tok), st.k_raw.copy(), st.v_raw.copy())


# ----------------------------------------------------------------- round driver
def upload_prompt(model, toks, aux, lens):
    dev = model.device
    P_max = aux.shape[1]
    t = torch.from_numpy(np.ascontiguousarray(toks[:, :P_max])).to(dev)
    nxt = torch.from_numpy(np.ascontiguousarray(toks[np.arange(len(lens)), lens])).to(dev)
    a = torch.from_numpy(aux.view(np.int16)).to(dev)
    return t, nxt, a


def gpu_prefill(seq, model, toks, aux, lens):
    t, nxt, a = upload_prompt(model, toks, aux, lens)
    seq.prefill(t, nxt, lens, a)


def oracle_prefill(dr, toks, aux, lens, which=None):
    which = range(len(lens)) if which is None else which
    return {b: O.prefill(dr, toks[b, :lens[b]], int(toks[b, lens[b]]), aux[b, :lens[b]]) for b in which}


def check_state(seq, states: dict, what, kv_lo=0):
    kv_len = seq.kv_len.cpu().numpy()
    g = seq.g.cpu().numpy()
    tok = seq.tok.cpu().numpy()
    for b, st in states.items():
        assert kv_len[b] == st.kv_len, f"{what}: kv_len[{b}] {kv_len[b]} vs {st.kv_len}"
        assert tok[b] == st.tok, f"{what}: tok[{b}]"
        assert_close(g[b], st.g, f"{what}: boundary g[{b}]", max_abs=1e-3, rel_l2=1e-5)
        if st.kv_len > kv_lo:
            k, v = seq.kv_entries(b, kv_lo, st.kv_len)
            fmt = seq.model.kv_format
            if fmt == "bf16":
                assert_close_bf16(bf16_bits_to_f64(k), st.k[kv_lo:], f"{what}: K[{b}]")
                assert_close_bf16(bf16_bits_to_f64(v), st.v[kv_lo:], f"{what}: V[{b}]")
            else:
                assert_quant_valid(k, st.k_raw[kv_lo:], "k", f"{what}: K[{b}]")
                assert_quant_valid(v, st.v_raw[kv_lo:], "v", f"{what}: V[{b}]")


def check_chain_stepwise(seq, dr, b, st, g_eff, out, di, dt, report=None) -> int:
    """Chain of sequence b step by step: step j of the oracle runs on the implementation's
    inputs to that step (its boundary or previous g, its previous token, its stored KV
    decoded, including the entry it appended at this step), since a stored value on a
    rounding boundary -- a quantization code, or a bf16 value one ulp away -- may validly
    differ between the two, and over a long chain such a difference moves later steps by
    more than float noise.  Each appended entry must be a valid encoding of the oracle's
    k / v of the step (assert_quant_valid / assert_bf16_valid); ids follow the margin
    rule; logits and g are compared with the float tolerance.  `report`, a list, receives
    (b, j, max-abs error of the logits, of g) per step."""
    fmt = seq.model.kv_format
    L = st.kv_len
    kraw, vraw = seq.kv_entries(b, 0, L + g_eff)
    kd = kv_values(kraw, fmt, "k")
    vd = kv_values(vraw, fmt, "v")
    logits = out["logits"][b, :g_eff].cpu().numpy()
    gdbg = out["g"][b, :g_eff].cpu().numpy().astype(np.float64)
    g_in, tok_in, ties = st.g, int(st.tok), 0
    for j in range(g_eff):
        pos = L + j
        so = O.draft_step(dr, tok_in, g_in, kd[:pos], vd[:pos], pos, new_kv=(kd[pos], vd[pos]))
        if fmt == "bf16":
            assert_bf16_valid(kraw[pos], so.k_raw, f"spec K b{b} j{j}")
            assert_bf16_valid(vraw[pos], so.v_raw, f"spec V b{b} j{j}")
        else:
            assert_quant_valid(kraw[pos], so.k_raw, "k", f"spec K b{b} j{j}")
            assert_quant_valid(vraw[pos], so.v_raw, "v", f"spec V b{b} j{j}")
        gid = int(di[b, j])
        if top2_margin(so.logits) > MARGIN:
            assert gid == so.draft_id, f"b{b} step {j}: GPU id {gid} vs oracle {so.draft_id}"
        else:
            ties += 1
            assert so.logits[gid] >= so.logits.max() - MARGIN, f"b{b} step {j}: GPU id {gid} not near max"
        assert int(dt[b, j]) == dr.d2t_map(gid), f"b{b} step {j}: d2t of {gid}"
        if report is not None:
            report.append((b, j, float(np.abs(logits[j] - so.logits).max()),
                           float(np.abs(gdbg[j] - so.g_next).max())))
        assert_close(logits[j], so.logits, f"logits b{b} j{j}")
        assert_close(gdbg[j], so.g_next, f"g b{b} j{j}")
        g_in, tok_in = gdbg[j], int(dt[b, j])
    return ties


def run_round(model, dr, seq, states: dict, gamma, n_imposed, seed, flags=0, kv_lo=0, stepwise=False,
              report=None):
    """One full round on the GPU and, for the sequences in `states`, the oracle: chain
    (ids with the margin rule, logits, g, speculative KV), rewind (kv_len, committed
    bytes, boundary), accept against imposed target predictions, rebuild.  The chain is
    compared end to end (the oracle's own cache and g), or step by step on the stored
    entries (check_chain_stepwise) with a quantized cache or when `stepwise` is set."""
    geo = model.geom
    Bn = seq.B
    out = seq.draft_chain(gamma, flags=flags, debug=True)
    torch.cuda.synchronize()
    dt = out["draft_tok"].cpu().numpy()
    di = out["draft_id"].cpu().numpy()
    ge = out["gamma_eff"].cpu().numpy()
    L_all = seq._round_start_host.copy()
    assert np.array_equal(seq.kv_len.cpu().numpy(), L_all + ge)
    ties = 0
    for b, st in states.items():
        g_eff = O.plan_gamma(st.kv_len, gamma, model.max_cache_len, bool(flags & Bd.EAGLE3_SHRINK_GAMMA))
        assert ge[b] == g_eff
        assert np.all(dt[b, g_eff:] == -1)
        if model.kv_format != "bf16" or stepwise:
            ties += check_chain_stepwise(seq, dr, b, st, g_eff, out, di, dt, report)
            continue
        ch, f = oracle_chain_following(dr, st, g_eff, di[b, :g_eff], dt[b, :g_eff])
        ties += f.ties
        assert np.all(dt[b, g_eff:] == -1)
        logits = out["logits"][b, :g_eff].cpu().numpy()
        gdbg = out["g"][b, :g_eff].cpu().numpy()
        for j in range(g_eff):
            assert_close(logits[j], ch.logits[j], f"logits b{b} j{j}")
            assert_close(gdbg[j], ch.g[j], f"g b{b} j{j}")
        k, v = seq.kv_entries(b, st.kv_len, st.kv_len + g_eff)
        assert_close_bf16(bf16_bits_to_f64(k), ch.spec_k, f"spec K b{b}")
        assert_close_bf16(bf16_bits_to_f64(v), ch.spec_v, f"spec V b{b}")
    # rewind: kv_len back, committed bytes and boundary untouched
    snap = {b: seq.kv_entries(b, max(0, st.kv_len - 64), st.kv_len) for b, st in states.items()}
    g_snap, tok_snap = seq.g.clone(), seq.tok.clone()
    seq.rewind()
    torch.cuda.synchronize()
    assert np.array_equal(seq.kv_len.cpu().numpy(), L_all)
    for b, st in states.items():
        k, v = seq.kv_entries(b, max(0, st.kv_len - 64), st.kv_len)
        assert np.array_equal(k, snap[b][0]) and np.array_equal(v, snap[b][1])
    assert torch.equal(seq.g, g_snap) and torch.equal(seq.tok, tok_snap)
    # accept against imposed target predictions
    y = synth.impose_target_predictions(np.where(dt < 0, 0, dt), np.minimum(n_imposed, ge), geo, seed)
    dev = model.device
    n_acc, bonus = seq.accept(out["draft_tok"], torch.from_numpy(y).to(dev), out["gamma_eff"])
    torch.cuda.synchronize()
    na, bo = n_acc.cpu().numpy(), bonus.cpu().numpy()
    for b in range(Bn):
        assert (na[b], bo[b]) == O.accept(dt[b], y[b], int(ge[b]))
    vaux = synth.make_aux((Bn, gamma + 1), geo, seed, stream=9)
    seq.rebuild_after_verify(n_acc, out["draft_tok"], bonus, torch.from_numpy(vaux.view(np.int16)).to(dev))
    torch.cuda.synchronize()
    new_states = {b: O.rebuild_after_verify(dr, st, int(na[b]), dt[b], int(bo[b]), vaux[b])
                  for b, st in states.items()}
    check_state(seq, new_states, "rebuild", kv_lo=kv_lo)
    assert seq.model.status() == 0
    return new_states, out, na, bo, vaux, ties


# ------------------------------------------------- long contexts: sampled and tracked checks
def compare_entries(got_k, got_v, k_raw, v_raw, kv_format, what):
    """Stored K / V rows of the implementation against the oracle's unstored k / v: bf16
    per R16 (one ulp), quantized blocks per R21 (a valid encoding)."""
    if kv_format == "bf16":
        assert_close_bf16(bf16_bits_to_f64(got_k), O.store_k(k_raw, "bf16"), f"{what} K")
        assert_close_bf16(bf16_bits_to_f64(got_v), O.store_v(v_raw, "bf16"), f"{what} V")
    else:
        assert_quant_valid(got_k, k_raw, "k", f"{what} K")
        assert_quant_valid(got_v, v_raw, "v", f"{what} V")


def check_prefill_sampled(seq, dr, toks, aux, lens, b, n_samples, rng, kv_format):
    """Prefill entries of sequence b at a seeded sample of positions: each entry depends
    only on its own (aux_p, t_{p+1}, p), so the oracle computes the sampled ones alone.
    Returns the sampled positions."""
    P = int(lens[b])
    if P < 2:
        return np.zeros(0, np.int64)
    pos = np.sort(rng.choice(P - 1, size=min(n_samples, P - 1), replace=False))
    g_p = O.encode(dr, aux[b, pos])
    kr, vr = O.kv_projections(dr, toks[b, pos + 1], g_p, pos)
    got_k, got_v = seq.kv_entries_at(b, pos)
    compare_entries(got_k, got_v, kr, vr, kv_format, f"prefill b{b} sampled")
    return pos


class Tracked:
    """What the oracle knows of a sequence it did not prefill in full: the committed
    length and the boundary (g, token).  Enough to check every entry a rebuild writes and
    the boundary it leaves, without the sequence's whole cache."""

    def __init__(self, L: int, g: np.ndarray, tok: int):
        self.L, self.g, self.tok = int(L), np.asarray(g, dtype=np.float64), int(tok)


def check_rebuild_tracked(seq, dr, b, tr: Tracked, dt_row, n: int, bonus: int, venc_b, kv_format):
    """The entries rebuild_after_verify wrote for sequence b at L..L+n -- pair 0 = the old
    boundary (g, token), pair i = (fc v_{i-1}, d_i) -- and the new boundary (fc v_n, bonus)
    and length L+n+1.  Returns the updated tracker."""
    toks = [tr.tok] + [int(dt_row[i - 1]) for i in range(1, n + 1)]
    gs = np.stack([tr.g] + [venc_b[i - 1] for i in range(1, n + 1)])
    pos = np.arange(tr.L, tr.L + n + 1)
    kr, vr = O.kv_projections(dr, toks, gs, pos)
    got_k, got_v = seq.kv_entries_at(b, pos)
    compare_entries(got_k, got_v, kr, vr, kv_format, f"rebuilt b{b}")
    assert int(seq.kv_len[b].item()) == tr.L + n + 1
    assert_close(seq.g[b].cpu().numpy(), venc_b[n], f"new boundary g b{b}", max_abs=1e-3, rel_l2=1e-5)
    assert int(seq.tok[b].item()) == int(bonus)
    return Tracked(tr.L + n + 1, venc_b[n], bonus)
