"""Drafter configuration from a checkpoint config.json (eagle3_config_from_json) and the
rotary-width rule (eagle3_resolve_rope_dims), on the host, no GPU.

tests/golden/drafter_config.json carries the values of the eagle3-qwen35-9b config that
"memra_engine/eagle.rs" prints in its draft_rope_width_tests (partial_rotary_factor 0.25
both top-level and under rope_parameters, head_dim 256, no rotary_dim, rope_theta 1e7
under rope_parameters, aux layers [1, 15, 28]).  The variants and the expected widths are
the page's own cases: 64 as declared; 64 with the factor only nested; 256 with no
declaration; 32 when an explicit rotary_dim 32 sits beside the factor; 256 for the
malformed factors 2.0 and 0.0."""
import os

import pytest

from eagle_speculative_decode_gb300 import binding as Bd
from eagle_speculative_decode_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "drafter_config.json")
TOP = '\n  "partial_rotary_factor": 0.25,'
NESTED = '\n    "partial_rotary_factor": 0.25,'


def fixture():
    return open(GOLDEN).read()


def edited(src, old, new):
    assert old in src, f"fixture drifted: {old!r} not found"
    return src.replace(old, new)


def test_fixture_gives_the_page_geometry(built_lib):
    c = Bd.eagle3_config_from_json(fixture())
    g = synth.FULL
    got = (c.n_embd, c.n_head, c.n_head_kv, c.head_dim, c.rope_dims, c.n_ff, c.draft_vocab,
           c.target_vocab)
    assert got == (g.n_embd, g.n_head, g.n_head_kv, g.head_dim, g.rope_dims, g.n_ff, g.draft_vocab,
                   g.target_vocab)
    assert c.rope_theta == 1e7 and abs(c.rms_eps - 1e-6) < 1e-12 and c.flags == 0


def test_batch_and_cache_fields_are_left_alone(built_lib):
    c = Bd.Config(max_batch=8, max_gamma=5, max_cache_len=4096, page_size=64,
                  kv_format=Bd.EAGLE3_KV_Q8_0_Q5_1)
    Bd.eagle3_config_from_json(fixture(), c)
    assert (c.max_batch, c.max_gamma, c.max_cache_len, c.page_size, c.kv_format) == \
        (8, 5, 4096, 64, Bd.EAGLE3_KV_Q8_0_Q5_1)
    assert Bd.eagle3_workspace_bytes(c) > 0


@pytest.mark.parametrize("variant,width", [
    ("as_declared", 64),
    ("nested_only", 64),
    ("undeclared", 256),
    ("explicit_32", 32),
    ("factor_2", 256),
    ("factor_0", 256),
])
def test_rope_width_cases_of_the_page(built_lib, variant, width):
    src = fixture()
    if variant == "nested_only":
        src = edited(src, TOP, "")
    elif variant == "undeclared":
        src = edited(edited(src, TOP, ""), NESTED, "")
        assert "partial_rotary_factor" not in src
    elif variant == "explicit_32":
        src = edited(src, TOP, TOP + '\n  "rotary_dim": 32,')
    elif variant == "factor_2":
        src = src.replace('"partial_rotary_factor": 0.25', '"partial_rotary_factor": 2.0')
    elif variant == "factor_0":
        src = src.replace('"partial_rotary_factor": 0.25', '"partial_rotary_factor": 0.0')
    assert Bd.eagle3_config_from_json(src).rope_dims == width


def test_resolve_rule_directly(built_lib):
    r = Bd.eagle3_resolve_rope_dims
    assert r(256, None, 0.25) == 64
    assert r(256, 32, 0.25) == 32          # explicit wins
    assert r(256, None, None) == 256       # full width
    assert r(256, None, 1.0) == 256
    assert r(256, None, 2.0) == 256 and r(256, None, 0.0) == 256 and r(256, None, -0.5) == 256
    assert r(256, None, 0.3) == 256        # 76.8 dims: not whole, malformed
    assert r(64, None, 0.25) == 16
    assert r(256, 512, None) == 256        # wider than the head: not usable, full width
    assert r(256, 33, 0.25) == 64          # odd explicit count: not usable, the factor decides
    assert r(0, None, None) == 0


def test_defaults_flags_and_refusals(built_lib):
    src = fixture()
    no_theta = edited(src, '    "rope_theta": 10000000,\n', "")
    assert Bd.eagle3_config_from_json(no_theta).rope_theta == 10000.0
    no_eps = edited(src, '\n  "rms_norm_eps": 1e-06,', "")
    assert abs(Bd.eagle3_config_from_json(no_eps).rms_eps - 1e-6) < 1e-12
    nbr = edited(src, '\n  "model_type": "llama",', '\n  "model_type": "llama",\n  "norm_before_residual": true,')
    assert Bd.eagle3_config_from_json(nbr).flags == Bd.EAGLE3_CKPT_NORM_BEFORE_RESIDUAL
    for flag in ("norm_before_fc", "fc_norm", "norm_output"):
        on = edited(src, '\n  "model_type": "llama",', f'\n  "model_type": "llama",\n  "{flag}": true,')
        with pytest.raises(Bd.Eagle3Error) as ei:
            Bd.eagle3_config_from_json(on)
        assert ei.value.code == Bd.EAGLE3_ERR_UNSUPPORTED
        off = edited(src, '\n  "model_type": "llama",', f'\n  "model_type": "llama",\n  "{flag}": false,')
        assert Bd.eagle3_config_from_json(off).flags == 0
    two_aux = edited(src, "[1, 15, 28]", "[1, 28]")
    with pytest.raises(Bd.Eagle3Error) as ei:
        Bd.eagle3_config_from_json(two_aux)
    assert ei.value.code == Bd.EAGLE3_ERR_UNSUPPORTED
    for key in ("hidden_size", "head_dim", "vocab_size", "draft_vocab_size"):
        broken = src.replace(f'"{key}"', f'"x_{key}"')
        with pytest.raises(Bd.Eagle3Error) as ei:
            Bd.eagle3_config_from_json(broken)
        assert ei.value.code == Bd.EAGLE3_ERR_INVALID_ARG
