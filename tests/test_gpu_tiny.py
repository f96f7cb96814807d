"""GPU parity of the whole round on the small drafter (n_embd 256, 4:1 GQA, head 64,
RoPE 16/64, draft vocab 1024 -> 4096), through the C ABI, against the CPU oracle:
prefill, chain, rewind, accept and rebuild, element by element, over several rounds,
ragged batches, non-contiguous pages and the capacity boundary; the rounds under both
decode attention kernels (tensor-core and CUDA-core)."""
import numpy as np
import pytest
import torch

from eagle_speculative_decode_gb300 import binding as Bd
from eagle_speculative_decode_gb300 import synth
from eagle_speculative_decode_gb300.runtime import DraftModel
from oracle import eagle3_oracle as O
from parity import check_state, gpu_prefill, oracle_prefill, run_round

pytestmark = pytest.mark.gpu
G = synth.TINY


@pytest.fixture(scope="module")
def tiny(built_lib):
    wts = synth.make_weights(G, seed=0)
    model = DraftModel(wts, max_batch=8, max_gamma=8, max_cache_len=100, page_size=16)
    dr = O.Drafter(G, wts.bits, wts.d2t)
    yield wts, model, dr
    model.close()


def _prompt(batch, lens, seed, P_max=None):
    P_max = P_max or int(max(lens))
    toks = synth.make_tokens((batch, P_max + 1), G, seed)
    aux = synth.make_aux((batch, P_max), G, seed)
    return toks, aux, P_max


@pytest.fixture(params=[0, 1], ids=["attn_cuda_cores", "attn_tensor_cores"])
def attention(request, tiny):
    tiny[1].set_attention(request.param)
    yield request.param
    tiny[1].set_attention(0)


def _round(model, dr, seq, states, gamma, n_imposed, seed, flags=0):
    return run_round(model, dr, seq, states, gamma, n_imposed, seed, flags)[0]


def test_single_sequence_rounds(tiny, attention):
    wts, model, dr = tiny
    lens = np.array([32])
    toks, aux, _ = _prompt(1, lens, seed=1)
    seq = model.new_state(1)
    gpu_prefill(seq, model, toks, aux, lens)
    torch.cuda.synchronize()
    states = oracle_prefill(dr, toks, aux, lens)
    check_state(seq, states, "prefill")
    for r, n in enumerate([2, 0, 3]):
        states = _round(model, dr, seq, states, 3, np.array([n]), seed=10 + r)


def test_ragged_batch_random_pages(tiny, attention):
    wts, model, dr = tiny
    lens = np.array([5, 32, 17, 1])
    toks, aux, _ = _prompt(4, lens, seed=2)
    pages_per_seq = (model.max_cache_len + model.page_size - 1) // model.page_size
    pt = synth.page_table(4, pages_per_seq, seed=3)
    seq = model.new_state(4, page_table=pt)
    gpu_prefill(seq, model, toks, aux, lens)
    torch.cuda.synchronize()
    states = oracle_prefill(dr, toks, aux, lens)
    check_state(seq, states, "prefill")
    for r in range(3):
        n = synth.imposed_accept_lengths(4, 4, seed=20 + r)
        states = _round(model, dr, seq, states, 4, n, seed=20 + r)


def test_capacity_boundary_start_97_gamma_3_max_100(tiny):
    """The review's worked case: start 97, k 3, max 100 must be refused, or drafted with
    k shrunk to 2, after which an all-accepted rebuild ends exactly at 100."""
    wts, model, dr = tiny
    lens = np.array([98])
    toks, aux, _ = _prompt(1, lens, seed=4)
    seq = model.new_state(1)
    gpu_prefill(seq, model, toks, aux, lens)
    torch.cuda.synchronize()
    states = oracle_prefill(dr, toks, aux, lens)
    assert states[0].kv_len == 97
    with pytest.raises(Bd.Eagle3Error) as ei:
        seq.draft_chain(3)
    assert ei.value.code == Bd.EAGLE3_ERR_CAPACITY
    assert seq.kv_len.cpu().item() == 97          # refused: nothing enqueued
    states = _round(model, dr, seq, states, 3, np.array([3]), seed=5, flags=Bd.EAGLE3_SHRINK_GAMMA)
    assert states[0].kv_len == 100 and seq.kv_len.cpu().item() == 100


def test_graph_and_direct_launch_agree(tiny):
    wts, model, dr = tiny
    lens = np.array([20, 9])
    toks, aux, _ = _prompt(2, lens, seed=6)
    outs = []
    for graph in (True, False, True):
        model.set_graph_mode(graph)
        seq = model.new_state(2)
        gpu_prefill(seq, model, toks, aux, lens)
        o = seq.draft_chain(5, debug=True)
        torch.cuda.synchronize()
        outs.append({k: v.cpu().numpy() for k, v in o.items()})
        seq.rewind()
    model.set_graph_mode(True)
    for o in outs[1:]:
        for k in outs[0]:
            assert np.array_equal(outs[0][k], o[k]), k


def test_encode_exact_integer_case(tiny):
    """fc in {-1, 0, 1} * 2^-4 and integer features: every partial sum is exact in
    float32, so the GPU must equal the oracle bit for bit."""
    wts, model, dr = tiny
    rng = np.random.default_rng(7)
    fc = (rng.integers(-1, 2, size=(G.n_embd, 3 * G.n_embd)) * 2.0 ** -4).astype(np.float32)
    aux = rng.integers(-8, 9, size=(5, 3, G.n_embd)).astype(np.float32)
    fc_bits = (fc.view(np.uint32) >> 16).astype(np.uint16)
    aux_bits = (aux.view(np.uint32) >> 16).astype(np.uint16)
    bits = dict(wts.bits)
    bits["fc"] = fc_bits
    m2 = DraftModel(synth.DrafterWeights(G, bits, wts.d2t), max_batch=2, max_gamma=2,
                    max_cache_len=16, page_size=16)
    try:
        got = m2.encode(torch.from_numpy(aux_bits.view(np.int16)).to(m2.device)).cpu().numpy()
    finally:
        m2.close()
    want = O.encode(O.Drafter(G, bits, wts.d2t), aux_bits)
    assert np.array_equal(got.astype(np.float64), want)


def test_state_machine_and_argument_errors(tiny):
    wts, model, dr = tiny
    lens = np.array([10])
    toks, aux, _ = _prompt(1, lens, seed=8)
    seq = model.new_state(1)
    gpu_prefill(seq, model, toks, aux, lens)
    dev = model.device
    dummy = torch.zeros(1, 4, dtype=torch.int32, device=dev)
    vaux = torch.zeros(1, 4, 3, G.n_embd, dtype=torch.int16, device=dev)
    with pytest.raises(Bd.Eagle3Error) as ei:            # no round open
        seq.rewind()
    assert ei.value.code == Bd.EAGLE3_ERR_STATE
    with pytest.raises(Bd.Eagle3Error) as ei:            # rebuild before any chain/rewind
        seq.rebuild_after_verify(dummy[:, 0], dummy[:, :3], dummy[:, 0], vaux, n_acc_host=[0])
    assert ei.value.code == Bd.EAGLE3_ERR_STATE
    with pytest.raises(Bd.Eagle3Error) as ei:            # gamma above max_gamma
        seq.draft_chain(9)
    assert ei.value.code == Bd.EAGLE3_ERR_INVALID_ARG
    out = seq.draft_chain(3)
    with pytest.raises(Bd.Eagle3Error) as ei:            # a round is already open
        seq.draft_chain(3)
    assert ei.value.code == Bd.EAGLE3_ERR_STATE
    with pytest.raises(Bd.Eagle3Error) as ei:            # rebuild before rewind
        seq.rebuild_after_verify(dummy[:, 0], out["draft_tok"], dummy[:, 0], vaux, n_acc_host=[0])
    assert ei.value.code == Bd.EAGLE3_ERR_STATE
    seq.rewind()
    with pytest.raises(Bd.Eagle3Error) as ei:            # null verify features
        Bd.eagle3_rebuild_after_verify(model.ctx, 1, 3, dummy.data_ptr(), out["draft_tok"].data_ptr(),
                                       dummy.data_ptr(), 0, seq.kv, seq.bnd)
    assert ei.value.code == Bd.EAGLE3_ERR_INVALID_ARG
    assert model.status() == 0


def test_out_of_range_token_sets_status_without_fault(tiny):
    wts, model, dr = tiny
    lens = np.array([6])
    toks, aux, _ = _prompt(1, lens, seed=9)
    seq = model.new_state(1)
    gpu_prefill(seq, model, toks, aux, lens)
    seq.tok.fill_(G.target_vocab + 5)
    seq.draft_chain(2)
    torch.cuda.synchronize()
    st = model.status()
    assert st & Bd.EAGLE3_DEV_BAD_TOKEN
    assert model.status() == 0                            # reading clears the word
    seq.rewind()


def test_bounded_wait_times_out_and_the_context_stays_usable(tiny):
    """The device failure path without a fault: a wait that nothing completes gives up,
    raises EAGLE3_DEV_TIMEOUT in the status word and the abort flag (a second wait returns
    at once); afterwards the same process still runs a round with parity."""
    wts, model, dr = tiny
    status = torch.zeros(1, dtype=torch.int32, device=model.device)
    result = torch.zeros(1, dtype=torch.int32, device=model.device)
    Bd.eagle3_selftest_bounded_wait(status.data_ptr(), result.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert int(status.item()) == Bd.EAGLE3_DEV_TIMEOUT
    assert int(result.item()) == 4      # first wait gave up, second returned at once, abort set
    lens = np.array([9])
    toks, aux, _ = _prompt(1, lens, seed=77)
    seq = model.new_state(1)
    gpu_prefill(seq, model, toks, aux, lens)
    torch.cuda.synchronize()
    states = oracle_prefill(dr, toks, aux, lens)
    _round(model, dr, seq, states, 3, np.array([2]), seed=78)
    assert model.status() == 0


@pytest.mark.parametrize("kv_format", ["bf16", "q8_0/q5_1"])
def test_out_of_range_page_sets_status_without_fault(built_lib, kv_format):
    """A page-table entry past the pool: every kernel that would touch that page (the
    k/v append of prefill and chain, the quantizer, the attention's copies) skips it and
    raises EAGLE3_DEV_BAD_PAGE; pages in range are still written, and reading the status
    clears it."""
    wts = synth.make_weights(G, seed=0)
    model = DraftModel(wts, max_batch=2, max_gamma=4, max_cache_len=64, page_size=16, kv_format=kv_format)
    try:
        pages = (model.max_cache_len + model.page_size - 1) // model.page_size
        pt = synth.page_table(1, pages)
        seq = model.new_state(1, page_table=pt)
        bad = seq.page_table.clone()
        bad[0, 1] = seq.num_pages + 3               # positions 16..31 map past the pool
        seq.page_table.copy_(bad)
        lens = np.array([24])
        toks, aux, _ = _prompt(1, lens, seed=11)
        gpu_prefill(seq, model, toks, aux, lens)
        torch.cuda.synchronize()
        assert model.status() & Bd.EAGLE3_DEV_BAD_PAGE
        assert model.status() == 0
        seq.draft_chain(2)                          # attention reads the bad page: skipped
        torch.cuda.synchronize()
        assert model.status() & Bd.EAGLE3_DEV_BAD_PAGE
        seq.rewind()
        # the entries of the first page were written normally
        dr = O.Drafter(G, wts.bits, wts.d2t, kv_format=kv_format)
        st = oracle_prefill(dr, toks, aux, lens)[0]
        k, v = seq.kv_entries(0, 0, 16)
        if kv_format == "bf16":
            assert np.max(np.abs(O.widen_bf16(k) - st.k[:16])) < 0.1
        else:
            from parity import assert_quant_valid
            assert_quant_valid(k, st.k_raw[:16], "k", "first page K")
    finally:
        model.close()
