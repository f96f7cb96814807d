"""The benchmark's table of profiled DRAM traffic (the bench line's roofline.traffic) against
the committed profile summaries: every entry lists kernel sources that exist, carries a
sha256 digest that one of the summaries under profiles/ cites (so each figure can be traced
to the ncu command that produced it), and a byte count within a few percent of the
algorithmic bytes of the launch it covers (traffic well above them would mean re-reads)."""
import glob
import os
import re

import bench
from eagle_speculative_decode_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "eagle_speculative_decode_gb300", "csrc")


def _summaries() -> str:
    return "\n".join(open(f).read() for f in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))))


def test_entries_name_existing_sources_and_a_cited_digest():
    text = _summaries()
    assert bench.PROFILED_TRAFFIC
    for key, e in bench.PROFILED_TRAFFIC.items():
        for f in e["sources"]:
            assert os.path.isfile(os.path.join(CSRC, f)), (key, f)
        assert re.fullmatch(r"[0-9a-f]{64}", e["sha256"]), key
        # summaries cite the digest in full or by its first eight hex digits
        assert e["sha256"] in text or e["sha256"][:8] in text, key


def test_traffic_close_to_the_algorithmic_bytes():
    g = synth.FULL
    lm = g.draft_vocab * g.n_embd * 2  # the lm_head weights streamed once per launch
    kv = {"bf16": 2 * g.n_head_kv * g.head_dim * 2, "q8_0/q5_1": g.n_head_kv * (g.head_dim // 32) * (34 + 24)}
    contexts = {"c4": 64 * 2057, "c5": 4 * 32780}  # keys attended per launch (mean contexts)
    for key, e in bench.PROFILED_TRAFFIC.items():
        cfg, kind = key[0], key[1]
        if kind == "lmhead":
            algo = lm
        else:
            fmt = key[2] if len(key) > 2 else "bf16"
            algo = contexts[cfg] * kv[fmt]
        assert 1.0 <= e["bytes"] / algo <= 1.05, (key, e["bytes"], algo)
