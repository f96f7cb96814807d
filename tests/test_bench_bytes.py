"""The benchmark's algorithmic byte counts (the roofline's numerator) against the figures
the drafter's tensor list fixes ("memra_engine/eagle.rs", the tensor table: fc
[4096, 12288], q [4096, 8192], k and v [1024, 8192], o [4096, 4096], gate and up
[12288, 4096], down [4096, 12288], lm_head [32000, 4096], all bf16; K/V of 4 kv heads x 256
per position): 698,351,616 weight bytes per draft step, 100,663,296 fc bytes per round,
4 KB of bf16 K/V per position, and the tiny drafter's 2,228,224 weight bytes per step."""
import bench
from eagle_speculative_decode_gb300 import synth


def _weight_bytes(g, weights="bf16"):
    mb = lambda rows, K: bench.matrix_bytes(rows, K, weights)  # noqa: E731
    n, F = g.n_embd, g.n_ff
    return (mb(g.q_rows + 2 * g.kv_rows, 2 * n) + mb(n, g.q_rows) + mb(2 * F, n) + mb(n, F)
            + mb(g.draft_vocab, n))


def test_weight_bytes_per_step():
    assert _weight_bytes(synth.FULL) == 698_351_616
    assert _weight_bytes(synth.TINY) == 2_228_224


def test_phase_bytes_carry_each_weight_once_per_step():
    """Beyond the weights, a step's bytes are the per-sequence activations and KV (linear in
    the batch) plus the norm gains (a constant): the weights are not counted per sequence."""
    g = synth.FULL
    extra = [sum(bench.phase_bytes(g, B, 0).values()) - _weight_bytes(g) for B in (1, 2, 3, 64)]
    per_seq = extra[1] - extra[0]
    assert per_seq > 0 and extra[2] - extra[1] == per_seq
    assert extra[3] == extra[0] + 63 * per_seq
    assert 0 < extra[0] - per_seq < 64 * 1024  # the gains: a few n-wide bf16 vectors


def test_kv_bytes_per_position():
    g = synth.FULL
    assert bench.kv_bytes_per_position(g, "bf16") == 4096
    # q8_0 keys (34 bytes per 32 values) and q5_1 values (24 bytes per 32 values)
    assert bench.kv_bytes_per_position(g, "q8_0/q5_1") == 1024 // 32 * (34 + 24) == 1856
    # the attention phase reads ctx_len positions per sequence
    a0 = bench.phase_bytes(g, 4, 0)["attn"]
    a1 = bench.phase_bytes(g, 4, 1000)["attn"]
    assert a1 - a0 == 4 * 1000 * 4096


def test_round_adds_the_fc_encode_and_kv_only_projection():
    g = synth.FULL
    B, gamma = 1, 3
    chain = gamma * sum(bench.phase_bytes(g, B, 512).values())
    rebuild = bench.round_bytes(g, B, gamma, 512) - chain
    fc = 100_663_296
    kv_only = bench.matrix_bytes(2 * g.kv_rows, 2 * g.n_embd)
    assert fc == 3 * 4096 * 4096 * 2 and kv_only == 33_554_432
    assert rebuild == fc + kv_only + B * (gamma + 1) * (3 * 4096 * 2 + 4096 * 4)


def test_int4_matrix_bytes():
    # 4-bit codes (K / 2 bytes) plus one bf16 (scale, zero) pair per 128 inputs, padded to
    # a multiple of 4 pairs
    assert bench.matrix_bytes(32000, 4096, "int4") == 32000 * (2048 + 32 * 4)
    assert bench.matrix_bytes(10, 384, "int4") == 10 * (192 + 4 * 4)   # 3 groups -> 4 pairs
    full = _weight_bytes(synth.FULL, "int4")
    assert full < _weight_bytes(synth.FULL) // 3
