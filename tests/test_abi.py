"""The C-ABI library on the host, no GPU: libeagle3.so builds for sm_103a, loads, exports
every function include/eagle3.h declares, and its host-only entry points (version, error
strings, workspace and KV row sizes, config validation, the capacity rule) answer as the
header states.  Nothing here launches a kernel."""
import ctypes
import os
import re

import pytest

from eagle_speculative_decode_gb300 import binding as Bd
from eagle_speculative_decode_gb300 import synth

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "eagle3.h")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "capacity_boundary.txt")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(eagle3_[a-z0-9_]+)\s*\(", src)))


def _cfg(g=synth.FULL, **kw):
    c = dict(n_embd=g.n_embd, n_head=g.n_head, n_head_kv=g.n_head_kv, head_dim=g.head_dim,
             rope_dims=g.rope_dims, rope_theta=g.rope_theta, rms_eps=g.rms_eps, n_ff=g.n_ff,
             draft_vocab=g.draft_vocab, target_vocab=g.target_vocab, max_batch=64, max_gamma=8,
             max_cache_len=8192, page_size=64, flags=0, kv_format=Bd.EAGLE3_KV_BF16)
    c.update(kw)
    return Bd.Config(**c)


def test_header_functions_are_exported(built_lib):
    names = _declared()
    assert len(names) >= 20
    assert set(names) == set(Bd.EXPORTED), set(names) ^ set(Bd.EXPORTED)
    for n in names:
        assert isinstance(getattr(built_lib, n), ctypes._CFuncPtr), n


def test_version_and_error_strings(built_lib):
    v = Bd.eagle3_version()
    assert v >> 16 >= 1
    for code in (Bd.EAGLE3_OK, Bd.EAGLE3_ERR_INVALID_ARG, Bd.EAGLE3_ERR_CAPACITY, Bd.EAGLE3_ERR_STATE,
                 Bd.EAGLE3_ERR_CUDA, Bd.EAGLE3_ERR_DEVICE, Bd.EAGLE3_ERR_UNSUPPORTED):
        s = Bd.error_string(code)
        assert isinstance(s, str) and s
    assert Bd.error_string(Bd.EAGLE3_OK) != Bd.error_string(Bd.EAGLE3_ERR_CAPACITY)


def test_kv_row_bytes_per_format(built_lib):
    d = synth.FULL.head_dim
    assert Bd.eagle3_kv_row_bytes(_cfg()) == (2 * d, 2 * d)
    # q8_0 K: 34 bytes per 32 values; q5_1 V: 24 bytes per 32 values
    assert Bd.eagle3_kv_row_bytes(_cfg(kv_format=Bd.EAGLE3_KV_Q8_0_Q5_1)) == (d // 32 * 34, d // 32 * 24)
    t = synth.TINY
    assert Bd.eagle3_kv_row_bytes(_cfg(t, kv_format=Bd.EAGLE3_KV_Q8_0_Q5_1)) == (68, 48)


def test_invalid_configs_are_refused(built_lib):
    assert Bd.eagle3_workspace_bytes(_cfg()) > 0
    assert Bd.eagle3_workspace_bytes(_cfg(kv_format=Bd.EAGLE3_KV_Q8_0_Q5_1)) > 0
    assert Bd.eagle3_workspace_bytes(_cfg(flags=Bd.EAGLE3_CKPT_NORM_BEFORE_RESIDUAL)) > 0
    for bad in (dict(kv_format=2), dict(kv_format=-1), dict(flags=2), dict(flags=0x80000000), dict(n_head=15), dict(max_gamma=0),
                dict(max_gamma=65), dict(page_size=0), dict(max_cache_len=1), dict(n_embd=4100),
                dict(rope_dims=3), dict(rope_theta=0.0), dict(draft_vocab=0)):
        assert Bd.eagle3_workspace_bytes(_cfg(**bad)) == 0, bad
        with pytest.raises(Bd.Eagle3Error) as ei:
            Bd.eagle3_kv_row_bytes(_cfg(**bad))
        assert ei.value.code == Bd.EAGLE3_ERR_INVALID_ARG


def test_quantized_kv_unit_alignment(built_lib):
    """A quantized attention unit (the keys of one page copied at once) must be a whole
    number of 16-byte chunks: at head_dim 64 a q8_0 row is 68 bytes, so units of 4 keys
    (page sizes divisible by 4) are needed; bf16 rows (128 bytes) take any page size."""
    t = synth.TINY
    q = Bd.EAGLE3_KV_Q8_0_Q5_1
    for ps in (1, 2, 6):
        assert Bd.eagle3_workspace_bytes(_cfg(t, page_size=ps)) > 0
        assert Bd.eagle3_workspace_bytes(_cfg(t, page_size=ps, kv_format=q)) == 0, ps
    for ps in (4, 12, 16, 64):
        assert Bd.eagle3_workspace_bytes(_cfg(t, page_size=ps, kv_format=q)) > 0, ps
    # head_dim 256: 272- and 192-byte rows are whole chunks at any unit
    assert Bd.eagle3_workspace_bytes(_cfg(page_size=1, kv_format=q)) > 0


def test_capacity_rule_matches_the_worked_case(built_lib):
    n = 0
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        start, k, mx, plain, shrink = line.split()
        for flags, want in ((0, plain), (Bd.EAGLE3_SHRINK_GAMMA, shrink)):
            if want == "refuse":
                with pytest.raises(Bd.Eagle3Error) as ei:
                    Bd.eagle3_plan_gamma(int(start), int(k), int(mx), flags)
                assert ei.value.code == Bd.EAGLE3_ERR_CAPACITY
            else:
                assert Bd.eagle3_plan_gamma(int(start), int(k), int(mx), flags) == int(want)
        n += 1
    assert n >= 6
    with pytest.raises(Bd.Eagle3Error):
        Bd.eagle3_plan_gamma(-1, 3, 100)
    with pytest.raises(Bd.Eagle3Error):
        Bd.eagle3_plan_gamma(0, 0, 100)


def test_header_is_plain_c(tmp_path):
    """include/eagle3.h compiles as C99 with warnings as errors: the boundary has no C++
    types, and every declaration is referenced once."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    names = _declared()
    src = tmp_path / "use_header.c"
    src.write_text('#include "eagle3.h"\nvoid *const eagle3_all[] = {\n' +
                   ",\n".join(f"  (void *){n}" for n in names) + "\n};\n")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-Wno-pedantic", "-I",
                        os.path.dirname(HEADER), "-c", str(src), "-o", str(tmp_path / "o.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_context_knobs_refuse_a_null_context(built_lib):
    """The host-only setters check their context before anything else (no GPU needed)."""
    for call in (lambda: Bd.eagle3_set_tc_schedule(0, 0), lambda: Bd.eagle3_set_attention(0, 0),
                 lambda: Bd.eagle3_set_tc_min_items(0, 3),
                 lambda: Bd.eagle3_set_graph_mode(0, True)):
        with pytest.raises(Bd.Eagle3Error) as ei:
            call()
        assert ei.value.code == Bd.EAGLE3_ERR_INVALID_ARG
