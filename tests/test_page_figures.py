"""The pages' printed figures are consistent with their own operands, and the benchmark's byte
accounting (unique bytes read once against bytes read through every block table) gives the
ratio the pages' read-once argument rests on: members x prefix against one prefix."""
import json
import os

import numpy as np

import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "page_figures.json")


def _near(x, printed, rel):
    return abs(x - printed) <= rel * abs(printed)


def test_printed_ratios_follow_from_their_operands():
    g = json.load(open(GOLDEN))
    t = g["prefix_traffic"]
    assert _near(t["paged_bytes"] / t["read_once_bytes"], t["printed_ratio"], 0.02)
    k = g["prefix_kernel_time"]
    assert _near(k["paged_s"] / k["read_once_s"], k["printed_ratio"], 0.01)
    h = g["tuning_headroom"]
    assert _near(1.0 / h["fraction_of_limit"], h["printed_bound"], 0.005)
    a = g["amdahl"]
    assert _near(1.0 / ((1 - a["f"]) + a["f"] / a["s"]), a["printed"], 0.02)
    s = g["gain_share"]
    share = (s["cascade_tok_s"] - s["paged_tok_s"]) / (s["granikv_tok_s"] - s["paged_tok_s"])
    assert _near(share, s["printed_share"], 0.005)
    r = g["admission_ramp"]
    assert _near((r["ramp_ps1_s"] - r["ramp_ps128_s"]) / r["intervals"] * 1e3, r["printed_ms"], 0.02)
    d = g["headline_gap"]
    assert _near((d["ps1_ms"] / d["ps128_ms"] - 1) * 100, d["printed_pct"], 0.002)
    # the pages' own traffic pair is not exactly one prefix per request: 256 x 37 MB is 9.5 GB
    assert t["requests"] * t["read_once_bytes"] / t["paged_bytes"] > 1.05


def test_byte_accounting_counts_a_shared_prefix_once():
    """unique_kv_bytes counts each stored slot once and paged_kv_bytes counts every request's
    whole context: with 256 members of a 4096-token prefix and one private token each, their
    ratio is (256 x 4097) / (4096 + 256), computed here by hand."""
    c = workloads.make_case("agent", 2, batch=256, prefix_len=4096, private_range=(1, 1), tables_only=True)
    tb = c.kv_token_bytes()
    assert workloads.paged_kv_bytes(c) == 256 * 4097 * tb
    assert workloads.unique_kv_bytes(c) == (4096 + 256) * tb
    assert np.isclose(workloads.paged_kv_bytes(c) / workloads.unique_kv_bytes(c), 256 * 4097 / 4352)
    # nested: the root once, each block's segment once, each request's private tokens once
    n = workloads.make_case("agent", 2, batch=16, prefix_len=512, private_range=(1, 1), nested=(4, 256),
                            tables_only=True)
    assert workloads.unique_kv_bytes(n) == (512 + 4 * 256 + 16) * tb
