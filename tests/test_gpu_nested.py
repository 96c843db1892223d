"""GPU parity for nested prefix groups (a tree of shared beginnings): each level's own
segment is read once for every request below it, and a request merges the partials of
every read-once level on its path with its suffix splits.  Compared with the fp64 oracle's
plain attention over each request's block table, at the tolerances of the other parity
tests; the launch forms and the token-flat lowering must agree bit for bit."""
import dataclasses

import numpy as np
import pytest

import oracle
import workloads
from gpu_util import TOL, max_err, run_case
from oracle_pins import _three_level_tables

pytestmark = pytest.mark.gpu

NESTED = [
    ("agent", dict(name="agent", batch=24, prefix_len=600, private_range=(1, 300), nested=(4, 500))),
    ("agent-ps1", dict(name="agent", batch=10, prefix_len=300, private_range=(1, 200), nested=(3, 170),
                       page_size=1)),
    ("agent-ps64-unaligned", dict(name="agent", batch=14, prefix_len=700, private_range=(1, 260),
                                  nested=(3, 650), page_size=64)),
    ("fp8", dict(name="fp8_large", batch=16, prefix_len=1024, private_range=(1, 400), nested=(3, 600))),
    ("fp8-d64", dict(name="fp8_large", batch=9, prefix_len=256, private_range=(1, 150), nested=(2, 300),
                     head_dim=64)),
    ("agent-d64-g8", dict(name="agent", batch=8, prefix_len=320, private_range=(1, 120), nested=(3, 200),
                          head_dim=64, num_q_heads=64)),
    ("fp32", dict(name="tiny", batch=7, prefix_len=100, private_range=(1, 90), nested=(3, 70))),
    ("one-split-each", dict(name="agent", batch=20, prefix_len=512, private_range=(1, 1), nested=(4, 256))),
    ("one-subgroup", dict(name="fp8_large", batch=6, prefix_len=300, private_range=(1, 500), nested=(1, 900))),
]


def _make(kw, seed=3):
    kw = dict(kw)
    return workloads.make_case(kw.pop("name"), seed, **kw)


def _check(case, out):
    ref_o, ref_lse = oracle.attend_all(case)
    tol = TOL[case.workload.kv_dtype]
    o, lse = out
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert max_err(o, ref_o) <= tol and max_err(lse, ref_lse) <= tol


@pytest.mark.parametrize("label,kw", NESTED, ids=[c[0] for c in NESTED])
@pytest.mark.parametrize("branch", ["dense", "cascade", "mixed"])
def test_nested_matches_oracle(label, kw, branch):
    case = _make(kw)
    G = case.workload.num_q_heads // case.workload.num_kv_heads
    # mixed: the root (every request) dense, the subgroups cascade
    thr = {"dense": 1, "cascade": 1 << 20, "mixed": case.batch * G}[branch]
    _check(case, run_case(case, threshold=thr))


def test_nested_forms_and_lowering_bit_identical(monkeypatch):
    """Sequential and concurrent dependent launches, the forked prefix stream and the
    token-flat lowering give the same bits on nested groups (a one-split request of several
    levels merges in its suffix CTA or through its counter)."""
    for kw in (NESTED[0][1], NESTED[3][1], dict(NESTED[7][1], private_range=(1, 80))):
        case = _make(kw, seed=8)
        outs = []
        for form in ("1", "2", "2"):
            monkeypatch.setenv("PSP_PDL_FORM", form)
            outs.append(run_case(case))
        monkeypatch.delenv("PSP_PDL_FORM")
        outs.append(run_case(case, token_flat=True))
        outs.append(run_case(case, concurrent=True))
        for o, l in outs[1:]:
            assert np.array_equal(o, outs[0][0]) and np.array_equal(l, outs[0][1]), kw["name"]
        _check(case, outs[0])


def _with_pools(case, seed):
    """The case with seeded random queries and a fully written bf16 pool."""
    w = case.workload
    n = case.num_pages * case.page_size
    q = workloads._encode(workloads.normal_f32((case.batch, w.num_q_heads, w.head_dim), seed, 1), w.q_dtype)
    k = workloads._encode(workloads.normal_f32((n, w.num_kv_heads, w.head_dim), seed, 2), w.kv_dtype)
    v = workloads._encode(workloads.normal_f32((n, w.num_kv_heads, w.head_dim), seed, 3), w.kv_dtype)
    shape = (case.num_pages, case.page_size, w.num_kv_heads, w.head_dim)
    return dataclasses.replace(case, q=q, k_pool=k.reshape(shape), v_pool=v.reshape(shape))


def test_three_levels_match_oracle():
    """Hand-built three-level tree plus a side branch: requests merge one, two or three
    levels; every branch mix, both launch forms."""
    case = _with_pools(_three_level_tables(num_q_heads=8, num_kv_heads=2, head_dim=64), 12)
    for thr in (1, 1 << 20, 16):
        _check(case, run_case(case, threshold=thr))
        _check(case, run_case(case, threshold=thr, concurrent=True))


def test_nested_paged_levels_match_oracle():
    """Built-in read-once minimums on a tree whose root segment is short: the root is paged
    and so is every level below it (the plan is the plan without sharing); with a long root
    and short subgroup segments only the root is read once."""
    short_root = _make(dict(name="agent", batch=12, prefix_len=200, private_range=(1, 100), nested=(2, 2048)))
    long_root = _make(dict(name="agent", batch=12, prefix_len=2048, private_range=(1, 100), nested=(3, 200)))
    for case in (short_root, long_root):
        _check(case, run_case(case, read_once=None))


@pytest.mark.parametrize("name,n_sub,seg", [("fp8_large", 16, 2048), ("agent", 64, 1024)])
def test_nested_full_size_sampled(name, n_sub, seg):
    """The benchmark's nested batches (256 requests, 4096-token root, one segment per block,
    suffixes U[128, 1024]) under the built-in dispatcher and with every level read once:
    1,024 sampled rows plus the longest and shortest requests against the oracle."""
    case = workloads.make_case(name, 17, batch=256, prefix_len=4096, private_range=(128, 1024),
                               nested=(n_sub, seg))
    w = case.workload
    rng = np.random.default_rng(5)
    bb = np.concatenate([rng.integers(0, case.batch, 1024), np.repeat([np.argmax(case.kv_len),
                                                                       np.argmin(case.kv_len)], w.num_q_heads)])
    hh = np.concatenate([rng.integers(0, w.num_q_heads, 1024), np.tile(np.arange(w.num_q_heads), 2)])
    ref_o, ref_lse = oracle.attend(case, bb, hh)
    tol = TOL[w.kv_dtype]
    for read_once in (None, dict(read_once_min_tokens=-1, read_once_min_mib=-1)):
        o, lse = run_case(case, read_once=read_once)
        assert max_err(o[bb, hh], ref_o) <= tol and max_err(lse[bb, hh], ref_lse) <= tol


def test_random_trees_match_oracle():
    """Random trees of shared beginnings on the GPU, cycling cache types, page sizes and
    dispatcher thresholds, against the oracle."""
    cells = [("agent", 16, 1), ("fp8_large", 16, 16), ("tiny", 16, 1 << 20), ("agent", 64, 40),
             ("fp8_large", 1, 1), ("agent", 32, 1 << 20), ("fp8_large", 64, 64), ("agent", 16, 16)]
    for i, (name, ps, thr) in enumerate(cells):
        spec = workloads.random_tree_spec(200 + i, batch=14, max_seg=500)
        heads = dict(num_q_heads=16, num_kv_heads=4) if name != "tiny" else {}
        case = workloads.make_tree_case(name, i, page_size=ps, private_range=(1, 300), **heads, **spec)
        _check(case, run_case(case, threshold=thr))


def test_deep_chain_matches_oracle():
    """A chain of 24 nested levels (one request leaving at each level, the last two at the
    deepest): requests merge up to 24 levels of prefix partials with their suffix."""
    case = workloads.make_tree_case("agent", 6, parents=[-1] + list(range(23)),
                                    seg_lens=[64 + 8 * g for g in range(24)],
                                    request_groups=list(range(24)) + [-1, 23], page_size=16,
                                    num_q_heads=16, num_kv_heads=4, private_range=(1, 200))
    for thr in (1, 1 << 20):
        _check(case, run_case(case, threshold=thr))
        _check(case, run_case(case, threshold=thr, concurrent=True))
