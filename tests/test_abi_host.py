"""Host-side checks of the C ABI (no GPU): exported symbols, configuration and
batch validation, and the integer plan against the oracle, bit for bit."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import paged_shared_prefix_gb300 as psp
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NUM_SMS = 152


def declared_functions():
    text = open(os.path.join(ROOT, "include", "psp.h")).read()
    return sorted(set(re.findall(r"^PSP_API\s+[\w\s\*]+?\b(psp_\w+)\(", text, flags=re.M)))


def test_library_exports_every_declared_function():
    names = declared_functions()
    assert len(names) >= 15
    lib = ctypes.CDLL(psp.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/psp.h but not exported"
    assert set(names) == set(psp.EXPORTED), "binding and header disagree"


def test_header_documents_every_environment_override():
    import glob
    header = open(os.path.join(ROOT, "include", "psp.h")).read()
    section = header[header.index("Environment overrides"):header.index("#ifndef PSP_H_")]
    documented = set(re.findall(r"\bPSP_[A-Z_]+[A-Z]\b", section))
    read = set()
    for path in glob.glob(os.path.join(ROOT, "paged_shared_prefix_gb300", "csrc", "*.c*")):
        read |= set(re.findall(r'(?:getenv|env_int)\("(PSP_[A-Z_]+)"', open(path).read()))
    assert read and read == documented, (sorted(read - documented), sorted(documented - read))


def test_version_and_status_strings():
    assert "sm_103a" in psp.version()
    for code in psp.STATUS_NAMES:
        assert psp.psp_status_string(code)


def _create_status(**over):
    base = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, q_dtype=1, kv_dtype=1, o_dtype=1,
                page_size=16, num_pages=100, num_sms=NUM_SMS, dense_threshold=0, flags=0)
    base.update(over)
    cfg = psp.psp_config(**base)
    h = ctypes.c_void_p()
    st = psp.psp_create(ctypes.byref(cfg), ctypes.byref(h))
    if st == 0:
        psp.psp_destroy(h)
    return st


@pytest.mark.parametrize("over,expect", [
    ({}, 0),
    (dict(num_q_heads=24), -2),            # G = 3 is not built
    (dict(num_q_heads=30), -1),            # not a multiple of Hkv
    (dict(head_dim=96), -2),
    (dict(page_size=24), -2),              # not a power of two: refused, never coerced
    (dict(page_size=2048), -2),
    (dict(page_size=1), 0),
    (dict(page_size=128), 0),
    (dict(q_dtype=2), -2),                 # fp8 queries are not supported
    (dict(kv_dtype=0), -2),                # fp32 KV with bf16 Q
    (dict(kv_dtype=0, q_dtype=0, o_dtype=0), 0),
    (dict(kv_dtype=2), 0),
    (dict(o_dtype=2), -2),
    (dict(num_pages=0), -1),
    (dict(flags=4), -1),
    (dict(flags=1), 0),
])
def test_create_validation(over, expect):
    assert _create_status(**over) == expect


NO_MINIMUM = dict(read_once_min_tokens=-1, read_once_min_mib=-1)  # every shared prefix read once


def _lib_plan(case, threshold=0, num_sms=NUM_SMS, **read_once):
    step = psp.DecodeStep.for_case(case, num_sms=num_sms, dense_threshold=threshold, **read_once)
    step.plan_case(case)
    return step


PLAN_FIELDS = ["suffix_start", "suffix_len", "suffix_page_indptr", "suffix_page_indices",
               "split_indptr", "split_begin", "split_end", "group_shared_len", "group_page_indptr",
               "group_page_indices", "group_m_eff", "group_branch", "group_row_blocks",
               "group_chunk_indptr", "chunk_begin", "chunk_end", "req_level_indptr", "req_level_group"]


def _check_plan_matches_oracle(case, threshold=0, num_sms=NUM_SMS, **read_once):
    step = _lib_plan(case, threshold, num_sms, **read_once)
    info = step.plan_info()
    params = {k: info[k] for k, _ in oracle.PlanParams._fields_}
    ref = oracle.plan(case, params)
    for f in PLAN_FIELDS:
        got = step.plan_query(f)
        want = np.asarray(ref[f], np.int32)
        assert np.array_equal(got, want), f"{f}: library {got[:12]} oracle {want[:12]}"
    indptr, _ = oracle.expand_kv_indices(case)
    assert np.array_equal(step.plan_query("kv_indptr"), indptr)
    assert info["num_splits"] == len(ref["split_begin"])
    assert info["num_chunks"] == len(ref["chunk_begin"])
    assert info["suffix_tokens"] == int(ref["suffix_len"].sum())
    assert info["kv_indices_len"] == int(case.kv_len.sum())
    assert info["workspace_bytes"] > 0
    step.close()
    return info, ref


def _table_cases():
    out = []
    for name in ("tiny", "llama8b_noshare", "agent", "short_prefix", "fp8_large"):
        out.append((f"{name}-full", dict(name=name)))
    for ps in (1, 16, 128):
        out.append((f"llama-ps{ps}", dict(name="llama8b_noshare", page_size=ps)))
    out += [
        ("agent-ps1", dict(name="agent", page_size=1, batch=40)),
        ("agent-ps128-unaligned", dict(name="agent", page_size=128, prefix_len=1000, batch=20)),
        ("prefix-2003-ps16", dict(name="agent", prefix_len=2003, batch=9, private_range=(1, 50))),
        ("prefix-shorter-than-page", dict(name="agent", prefix_len=10, batch=5, page_size=16)),
        ("agent-ps32", dict(name="agent", page_size=32, batch=33)),
        ("agent-ps1024", dict(name="agent", page_size=1024, batch=12, prefix_len=4096)),
        ("one-request", dict(name="short_prefix", batch=1)),
        ("single-token-suffixes", dict(name="fp8_large", batch=64, private_range=(1, 1))),
    ]
    return out


@pytest.mark.parametrize("label,kw", _table_cases(), ids=[c[0] for c in _table_cases()])
def test_plan_matches_oracle(label, kw):
    kw = dict(kw)
    name = kw.pop("name")
    case = workloads.make_case(name, 3, tables_only=True, **kw)
    _check_plan_matches_oracle(case)                       # built-in read-once minimums
    _check_plan_matches_oracle(case.without_sharing())
    _check_plan_matches_oracle(case, threshold=1, **NO_MINIMUM)        # every group dense
    _check_plan_matches_oracle(case, threshold=1 << 20, **NO_MINIMUM)  # every group cascade
    _check_plan_matches_oracle(case, num_sms=7)
    _check_plan_matches_oracle(case, num_sms=7, **NO_MINIMUM)


def test_plan_identical_across_page_sizes():
    plans = []
    for ps in (1, 16, 128):
        case = workloads.make_case("llama8b_noshare", 1, page_size=ps, tables_only=True)
        step = _lib_plan(case)
        plans.append([step.plan_query(f).tolist() for f in ("split_indptr", "split_begin", "split_end")])
    assert plans[0] == plans[1] == plans[2]


def _multi_group_case():
    """Three prefix groups of different lengths plus ungrouped requests, one pool."""
    import dataclasses
    rng = np.random.default_rng(5)
    ps, B = 16, 23
    groups = np.array([-1, 0, 0, 1, 2, 1, 0, -1, 2, 2, 1, 0, 0, -1, 1, 2, 0, 1, 1, 2, -1, 0, 2], np.int32)
    gl = np.array([160, 37, 512], np.int32)
    priv = rng.integers(1, 300, B)
    kv_len = np.where(groups >= 0, gl[np.maximum(groups, 0)], 0) + priv
    n_pages = 4000
    perm = rng.permutation(n_pages)
    pos = 0
    shared = []
    for g in range(3):
        n = gl[g] // ps
        shared.append(perm[pos:pos + n])
        pos += n
    tables = []
    for b in range(B):
        g = groups[b]
        pre = shared[g] if g >= 0 else np.zeros(0, np.int64)
        need = -(-int(kv_len[b]) // ps) - len(pre)
        tables.append(np.concatenate([pre, perm[pos:pos + need]]))
        pos += need
    indptr = np.concatenate([[0], np.cumsum([len(t) for t in tables])]).astype(np.int32)
    base = workloads.make_case("agent", 0, batch=B, tables_only=True)
    return dataclasses.replace(base, num_pages=n_pages, kv_len=kv_len.astype(np.int32),
                               page_indptr=indptr, page_indices=np.concatenate(tables).astype(np.int32),
                               prefix_group=groups, group_prefix_len=gl)


def test_plan_multi_group_matches_oracle():
    case = _multi_group_case()
    for thr in (0, 1, 40, 1 << 20):
        for ro in ({}, NO_MINIMUM, dict(read_once_min_tokens=100, read_once_min_mib=-1)):
            info, ref = _check_plan_matches_oracle(case, threshold=thr, **ro)
    assert info["num_groups"] == 3
    # a 100-token minimum: the 37-token group (two full pages, 32 shared tokens) takes the paged branch
    assert list(ref["group_branch"]) == [2 if thr <= 28 else 1, 3, 2 if thr <= 24 else 1]


def _nested_cases():
    import sys
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    from oracle_pins import _three_level_tables
    out = [("three-level-ps16", _three_level_tables(head_dim=64))]
    for ps in (1, 16, 64):
        out.append((f"two-level-ps{ps}", workloads.make_case(
            "agent", 7, batch=40, prefix_len=1500, private_range=(1, 300), page_size=ps, nested=(5, 700),
            tables_only=True)))
    out.append(("two-level-one-block", workloads.make_case(
        "fp8_large", 2, batch=12, prefix_len=2048, private_range=(1, 64), nested=(1, 2048), tables_only=True)))
    out.append(("two-level-empty-segments", workloads.make_case(
        "agent", 3, batch=9, prefix_len=300, private_range=(1, 40), nested=(3, 0), tables_only=True)))
    out.append(("two-level-short-root", workloads.make_case(
        "agent", 5, batch=30, prefix_len=40, private_range=(1, 50), nested=(3, 1200), tables_only=True)))
    # a chain of 24 levels, one request leaving at each level
    out.append(("chain-24", workloads.make_tree_case(
        "agent", 6, parents=[-1] + list(range(23)), seg_lens=[64 + 8 * g for g in range(24)],
        request_groups=list(range(24)) + [-1, 23], page_size=16, tables_only=True)))
    return out


@pytest.mark.parametrize("label,case", _nested_cases(), ids=[c[0] for c in _nested_cases()])
def test_plan_nested_matches_oracle(label, case):
    """Nested groups: the library's plan equals the oracle's field by field (levels included)
    under the built-in read-once minimums, none, every group dense or cascade, and a small GPU."""
    for thr, ro, sms in ((0, {}, NUM_SMS), (0, NO_MINIMUM, NUM_SMS), (1, NO_MINIMUM, NUM_SMS),
                         (1 << 20, NO_MINIMUM, NUM_SMS), (0, NO_MINIMUM, 7),
                         (0, dict(read_once_min_tokens=100, read_once_min_mib=-1), NUM_SMS)):
        info, ref = _check_plan_matches_oracle(case, threshold=thr, num_sms=sms, **ro)
        assert info["num_groups"] == case.num_groups


@pytest.mark.parametrize("ps", [1, 16, 64])
def test_plan_random_trees_match_oracle(ps):
    """Random trees of shared beginnings (up to six groups, zero-length segments, requests
    outside any group): the library's plan equals the oracle's under several dispatcher
    settings."""
    for seed in range(12):
        spec = workloads.random_tree_spec(100 + seed, batch=20, max_seg=600)
        case = workloads.make_tree_case("agent", seed, page_size=ps, tables_only=True, **spec)
        for thr, ro, sms in ((0, {}, NUM_SMS), (0, NO_MINIMUM, NUM_SMS), (40, NO_MINIMUM, 7),
                             (0, dict(read_once_min_tokens=100, read_once_min_mib=-1), NUM_SMS)):
            _check_plan_matches_oracle(case, threshold=thr, num_sms=sms, **ro)


def test_plan_all_roots_equals_no_parents():
    """group_parent of all -1 plans exactly like no group_parent array."""
    import dataclasses
    case = _multi_group_case()
    roots = dataclasses.replace(case, group_parent=np.full(case.num_groups, -1, np.int32))
    for ro in ({}, NO_MINIMUM):
        a, b = _lib_plan(case, **ro), _lib_plan(roots, **ro)
        for f in PLAN_FIELDS:
            assert np.array_equal(a.plan_query(f), b.plan_query(f)), f
        a.close()
        b.close()


def test_nested_invalid_trees_rejected_like_the_oracle():
    import dataclasses
    import sys
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    from oracle_pins import _three_level_tables
    t = _three_level_tables(head_dim=64)
    bad_cases = [
        ("parent after child", dataclasses.replace(t, group_parent=np.array([-1, 0, 3, 0], np.int32)), -1),
        ("own parent", dataclasses.replace(t, group_parent=np.array([-1, 1, 1, 0], np.int32)), -1),
        ("parent below -1", dataclasses.replace(t, group_parent=np.array([-2, 0, 1, 0], np.int32)), -1),
        ("child shorter than parent", dataclasses.replace(t, group_prefix_len=np.array([64, 128, 120, 96], np.int32)), -1),
    ]
    for b, idx, label in ((5, 5, "leaves group 1's segment"), (1, 2, "leaves the root pages"),
                          (4, 17, "leaves group 2's own segment"), (2, 1, "first member of group 1 leaves the root"),
                          (3, 10, "second member of group 1 leaves its segment")):
        pi = t.page_indices.copy()
        pi[t.page_indptr[b] + idx] = 99
        bad_cases.append((f"request {b} {label}", dataclasses.replace(t, page_indices=pi), -5))
    pi = t.page_indices.copy()
    pi[t.page_indptr[5] + 6] = 1000       # out of range inside a shared page of a later member
    bad_cases.append(("out of range in a nested shared page", dataclasses.replace(t, page_indices=pi), -3))
    for label, case, code in bad_cases:
        assert _status_of_plan(case) == code, label
        assert _oracle_status(case) == code, label


def _status_of_plan(case):
    step = psp.DecodeStep.for_case(case, num_sms=NUM_SMS)
    b, keep = step.make_case_batch(case)
    st = psp.psp_plan(step.handle, ctypes.byref(b))
    step.close()
    return st


def _oracle_status(case):
    try:
        oracle.plan(case, dict(num_sms=NUM_SMS, dense_threshold=1024, tile_tokens=64, split_min_tiles=4,
                               split_ctas_per_sm=4, prefix_rows_dense=128, prefix_rows_cascade=64,
                               prefix_min_tiles=4, prefix_ctas_per_sm=1))
    except oracle.OracleError as e:
        return e.code
    return 0


def test_invalid_batches_rejected_like_the_oracle():
    import dataclasses
    c = workloads.make_case("agent", 1, batch=5, prefix_len=64, private_range=(1, 40), tables_only=True)
    bad_cases = []
    pi = c.page_indices.copy()
    pi[-1] = c.num_pages
    bad_cases.append(("page id == num_pages", dataclasses.replace(c, page_indices=pi), -3))
    pi = c.page_indices.copy()
    pi[3] = -1
    bad_cases.append(("negative page id", dataclasses.replace(c, page_indices=pi), -3))
    kl = c.kv_len.copy()
    kl[1] += 16
    bad_cases.append(("kv_len beyond its pages", dataclasses.replace(c, kv_len=kl), -4))
    kl = c.kv_len.copy()
    kl[2] = 0
    bad_cases.append(("empty context", dataclasses.replace(c, kv_len=kl), -4))
    pi = c.page_indices.copy()
    b1 = c.page_indptr[1]
    pi[b1], pi[-1] = pi[-1], pi[b1]
    bad_cases.append(("members disagree", dataclasses.replace(c, page_indices=pi), -5))
    pg = c.prefix_group.copy()
    pg[0] = 1
    bad_cases.append(("group id out of range", dataclasses.replace(c, prefix_group=pg), -1))
    bad_cases.append(("prefix longer than a context",
                      dataclasses.replace(c, group_prefix_len=np.array([int(c.kv_len.min()) + 1], np.int32)), -5))
    # out of range inside a later member's shared pages: reported as out of range, not as a
    # prefix mismatch (the library compares those pages instead of range-checking them twice)
    pi = c.page_indices.copy()
    pi[c.page_indptr[2]] = c.num_pages + 7
    bad_cases.append(("out of range in a shared page of the third member", dataclasses.replace(c, page_indices=pi), -3))
    pi = c.page_indices.copy()
    pi[c.page_indptr[2]] = -2
    bad_cases.append(("negative id in a shared page of the third member", dataclasses.replace(c, page_indices=pi), -3))
    for label, case, code in bad_cases:
        assert _status_of_plan(case) == code, label
        assert _oracle_status(case) == code, label


@pytest.mark.parametrize("threads", ["1", "3", "8"])
def test_large_batch_mismatch_found_with_planning_threads(threads, monkeypatch):
    """A batch large enough for the threaded page comparison: the plan equals the oracle's,
    and a member that leaves its group's pages is reported (the first in request order, as
    the error names it) however many threads compare."""
    import dataclasses
    monkeypatch.setenv("PSP_PLAN_THREADS", threads)
    case = workloads.make_case("fp8_large", 1, batch=256, prefix_len=8192, private_range=(1, 64), tables_only=True)
    assert case.page_indptr[-1] >= 1 << 17
    _check_plan_matches_oracle(case)
    for bad_bs in ([250], [77, 200], [3, 130, 254]):
        pi = case.page_indices.copy()
        for b in bad_bs:
            pi[case.page_indptr[b] + 100] = case.num_pages - 1 - b
        bad = dataclasses.replace(case, page_indices=pi)
        step = psp.DecodeStep.for_case(bad, num_sms=NUM_SMS)
        b, keep = step.make_case_batch(bad)
        assert psp.psp_plan(step.handle, ctypes.byref(b)) == -5
        assert f"request {bad_bs[0]} " in psp.psp_last_error(step.handle).decode()
        step.close()
        assert _oracle_status(bad) == -5


def test_sm_count_override_and_nvtx_ranges():
    """PSP_NUM_SMS sizes the partition when the configuration leaves num_sms at 0 (no device
    is queried: this host has none), and PSP_NVTX=1 plans the same step with its NVTX ranges."""
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    code = (
        "import sys; sys.path[:0] = [%r, %r]\n"
        "import json, workloads, paged_shared_prefix_gb300 as psp\n"
        "case = workloads.make_case('agent', 3, batch=20, prefix_len=1024, private_range=(1, 300), tables_only=True)\n"
        "step = psp.DecodeStep.for_case(case, num_sms=0)\n"
        "step.plan_case(case)\n"
        "print(json.dumps({'info': step.plan_info(), 'split': step.plan_query('split_end').tolist()}))\n"
        % (here, os.path.dirname(here)))
    outs = []
    for extra in ({"PSP_NUM_SMS": "37"}, {"PSP_NUM_SMS": "37", "PSP_NVTX": "1"}):
        env = dict(os.environ, **extra)
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, r.stderr[-2000:]
        outs.append(r.stdout.strip().splitlines()[-1])
    import json
    got = json.loads(outs[0])
    assert got["info"]["num_sms"] == 37
    assert outs[0] == outs[1]
    case = workloads.make_case("agent", 3, batch=20, prefix_len=1024, private_range=(1, 300), tables_only=True)
    step = _lib_plan(case, num_sms=37)
    assert step.plan_query("split_end").tolist() == got["split"]
    step.close()


def test_sizes_past_int32_are_refused():
    """Contexts whose lengths sum past 2^31 - 1 tokens are refused before anything is planned
    (the token-flat offsets are int32), and so is a pool of more than 2^31 - 1 slots."""
    ps, L, B = 1024, (1 << 30) + 5, 2          # 2 x (2^30 + 5) tokens > 2^31 - 1
    n = -(-L // ps)
    step = psp.DecodeStep(1, 1, 64, "bf16", "bf16", "bf16", ps, n, num_sms=NUM_SMS)
    ok, keep1 = step.make_batch(np.array([L], np.int32), np.array([0, n], np.int32), np.arange(n, dtype=np.int32))
    assert psp.psp_plan(step.handle, ctypes.byref(ok)) == 0
    kv = np.array([L] * B, np.int32)
    indptr = np.array([0, n, 2 * n], np.int32)
    pages = np.concatenate([np.arange(n), np.arange(n)]).astype(np.int32)
    b, keep = step.make_batch(kv, indptr, pages)
    assert psp.psp_plan(step.handle, ctypes.byref(b)) == -1
    assert "int32" in psp.psp_last_error(step.handle).decode()
    step.close()
    assert _create_status(page_size=1024, num_pages=(1 << 21) + 1) == -1   # 2^31 + 1024 slots


def test_calls_before_plan_report_no_plan():
    step = psp.DecodeStep(8, 2, 64, "f32", "f32", "f32", 16, 64, num_sms=NUM_SMS)
    n = ctypes.c_size_t(0)
    assert psp.psp_workspace_size(step.handle, ctypes.byref(n)) == -6
    t = psp.psp_tensors()
    assert psp.psp_run(step.handle, ctypes.byref(t), None) == -6
    assert psp.psp_upload(step.handle, None, 0, None) == -6
    info = psp.psp_plan_info()
    assert psp.psp_plan_info_get(step.handle, ctypes.byref(info)) == -6
    step.close()


def test_plan_query_capacity_and_empty_batch():
    case = workloads.make_case("tiny", 0, tables_only=True)
    step = _lib_plan(case)
    need = ctypes.c_size_t(0)
    small = np.zeros(1, np.int32)
    st = psp.psp_plan_query(step.handle, 3, small.ctypes.data, 4, ctypes.byref(need))
    assert st == -11 and need.value == 4 * len(step.plan_query("suffix_page_indices"))
    assert psp.psp_plan_query(step.handle, 99, None, 0, None) == -1
    step.plan(np.zeros(0, np.int32), np.zeros(1, np.int32), np.zeros(0, np.int32))
    assert step.plan_info()["num_splits"] == 0
    step.close()


def _random_batch(rng, ps, n_pages, max_b=24):
    """A seeded random batch: 0-3 prefix groups (unaligned prefix lengths, some shorter
    than a page), ungrouped requests, suffixes of 1-700 tokens, pages drawn without
    replacement from a pool of n_pages."""
    import dataclasses
    B = int(rng.integers(1, max_b + 1))
    ng = int(rng.integers(0, 4))
    gl = rng.integers(0, 900, ng).astype(np.int32)
    groups = rng.integers(-1, ng, B).astype(np.int32) if ng else np.full(B, -1, np.int32)
    priv = rng.integers(1, 701, B)
    if rng.random() < 0.2:
        priv[:] = 1
    pre_len = gl[np.maximum(groups, 0)] if ng else np.zeros(B, np.int32)
    kv_len = (np.where(groups >= 0, pre_len, 0) + priv).astype(np.int32)
    perm = rng.permutation(n_pages)
    pos = 0
    shared = []
    for g in range(ng):
        n = int(gl[g]) // ps
        shared.append(perm[pos:pos + n])
        pos += n
    tables = []
    for b in range(B):
        g = int(groups[b])
        pre = shared[g] if g >= 0 else np.zeros(0, np.int64)
        need = -(-int(kv_len[b]) // ps) - len(pre)
        tables.append(np.concatenate([pre, perm[pos:pos + need]]))
        pos += need
    assert pos <= n_pages
    indptr = np.concatenate([[0], np.cumsum([len(t) for t in tables])]).astype(np.int32)
    base = workloads.make_case("agent", 0, batch=B, page_size=ps, tables_only=True)
    return dataclasses.replace(base, num_pages=n_pages, kv_len=kv_len, page_indptr=indptr,
                               page_indices=np.concatenate(tables).astype(np.int32), prefix_group=groups,
                               group_prefix_len=gl)


@pytest.mark.parametrize("ps", [1, 16, 128])
def test_replans_on_one_handle_match_oracle(ps):
    # one handle plans a sequence of random batches that grow and shrink; every plan must
    # match the oracle's exactly (nothing of an earlier plan may leak into a later one)
    rng = np.random.default_rng([11, ps])
    n_pages = 40000 // ps + 64
    first = _random_batch(rng, ps, n_pages)
    step = psp.DecodeStep.for_case(first, num_sms=NUM_SMS)
    for i in range(12):
        case = first if i == 0 else _random_batch(rng, ps, n_pages)
        step.plan_case(case)
        info = step.plan_info()
        ref = oracle.plan(case, {k: info[k] for k, _ in oracle.PlanParams._fields_})
        for f in PLAN_FIELDS:
            assert np.array_equal(step.plan_query(f), np.asarray(ref[f], np.int32)), (ps, i, f)
        assert info["num_splits"] == len(ref["split_begin"]) and info["num_chunks"] == len(ref["chunk_begin"])
        assert info["num_groups"] == case.num_groups
    step.close()


def test_plan_log_line_records_the_step():
    # PSP_LOG=1 (read at psp_create): one "psp_step {json}" line per plan on stderr with the
    # shapes, index and block-table lengths and the dispatcher's choice per group
    import json
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    code = (
        "import sys; sys.path[:0] = [%r, %r]\n"
        "import json, workloads, paged_shared_prefix_gb300 as psp\n"
        "from test_abi_host import _multi_group_case\n"
        "case = _multi_group_case()\n"
        "step = psp.DecodeStep.for_case(case, num_sms=152, dense_threshold=26, read_once_min_tokens=-1,\n"
        "                               read_once_min_mib=-1)\n"
        "step.plan_case(case)\n"
        "info = step.plan_info()\n"
        "print(json.dumps({'info': info, 'm_eff': step.plan_query('group_m_eff').tolist(),\n"
        "                  'branch': step.plan_query('group_branch').tolist(),\n"
        "                  'pages': int(case.page_indptr[-1])}))\n" % (here, os.path.dirname(here)))
    env = dict(os.environ, PSP_LOG="1")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stderr.splitlines() if ln.startswith("psp_step ")]
    assert len(lines) == 1
    rec = json.loads(lines[0][len("psp_step "):])
    want = json.loads(r.stdout.strip().splitlines()[-1])
    info = want["info"]
    for k in ("kv_indices_len", "suffix_tokens", "shared_tokens", "num_splits", "num_chunks", "suffix_ctas",
              "prefix_dense_ctas", "prefix_cascade_ctas", "dense_threshold", "num_sms", "workspace_bytes"):
        assert rec[k] == info[k], k
    assert rec["batch"] == info["batch_size"] and rec["page_table_len"] == want["pages"]
    assert rec["coerced"] is False and rec["kv_dtype"] == "bf16" and rec["page_size"] == 16
    names = {0: "none", 1: "cascade", 2: "dense", 3: "paged"}
    assert [g["m_eff"] for g in rec["groups"]] == want["m_eff"]
    assert [g["branch"] for g in rec["groups"]] == [names[b] for b in want["branch"]]
    assert {g["branch"] for g in rec["groups"]} == {"dense", "cascade"}
    assert [g["parent"] for g in rec["groups"]] == [-1, -1, -1]
    # a nested batch records each group's parent
    code_nested = code.replace("case = _multi_group_case()",
                               "case = workloads.make_case('agent', 2, batch=12, prefix_len=300, "
                               "private_range=(1, 40), nested=(3, 200), tables_only=True)")
    r = subprocess.run([sys.executable, "-c", code_nested], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    rec = json.loads([ln for ln in r.stderr.splitlines() if ln.startswith("psp_step ")][0][len("psp_step "):])
    assert [g["parent"] for g in rec["groups"]] == [-1, 0, 0, 0]
    assert [g["members"] for g in rec["groups"]] == [12, 4, 4, 4]
    # without the variable nothing is written
    r = subprocess.run([sys.executable, "-c", code], env={k: v for k, v in os.environ.items() if k != "PSP_LOG"},
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "psp_step" not in r.stderr


SUFFIX_FIELDS = ["suffix_start", "suffix_len", "suffix_page_indptr", "suffix_page_indices", "split_indptr",
                 "split_begin", "split_end"]


def test_paged_branch_shares_nothing():
    # a group whose prefix is too short, or saves too little, to be read once takes the paged
    # branch: nothing is shared and every per-request array is the plan without the group
    cases = [
        (workloads.make_case("short_prefix", 2, tables_only=True), {}),           # 512 tokens < 1024
        (workloads.make_case("agent", 2, batch=8, prefix_len=2048, tables_only=True), {}),  # 7 x 2048 x 4 KiB < 64 MiB
        (workloads.make_case("agent", 2, batch=40, prefix_len=1024, tables_only=True),
         dict(read_once_min_tokens=1025, read_once_min_mib=-1)),
    ]
    for case, ro in cases:
        step = _lib_plan(case, **ro)
        alone = _lib_plan(case.without_sharing())
        for f in SUFFIX_FIELDS:
            assert np.array_equal(step.plan_query(f), alone.plan_query(f)), f
        assert list(step.plan_query("group_branch")) == [psp.BRANCH_PAGED]
        assert list(step.plan_query("group_shared_len")) == [0]
        assert list(step.plan_query("group_chunk_indptr")) == [0, 0]
        G = case.workload.num_q_heads // case.workload.num_kv_heads
        assert list(step.plan_query("group_m_eff")) == [case.batch * G]
        info = step.plan_info()
        assert info["shared_tokens"] == 0 and info["prefix_dense_ctas"] == 0 and info["prefix_cascade_ctas"] == 0
        _check_plan_matches_oracle(case, **ro)
        step.close()
        alone.close()


def test_read_once_minimums_at_their_boundaries():
    # shared tokens equal to the minimum are read once, one token more is the paged branch
    case = workloads.make_case("agent", 4, batch=40, prefix_len=1024, tables_only=True)
    for min_tokens, want in ((1024, psp.BRANCH_DENSE), (1025, psp.BRANCH_PAGED)):
        step = _lib_plan(case, read_once_min_tokens=min_tokens, read_once_min_mib=-1)
        assert list(step.plan_query("group_branch")) == [want]
        step.close()
    # 257 members sharing 64 tokens of 4 KiB save 256 x 64 x 4096 bytes = exactly 64 MiB
    case = workloads.make_case("agent", 4, batch=257, prefix_len=64, private_range=(1, 20), tables_only=True)
    assert case.kv_token_bytes() == 4096
    for min_mib, want in ((64, psp.BRANCH_DENSE), (65, psp.BRANCH_PAGED)):
        step = _lib_plan(case, read_once_min_tokens=-1, read_once_min_mib=min_mib)
        assert list(step.plan_query("group_branch")) == [want]
        info = step.plan_info()
        assert info["read_once_min_mib"] == min_mib and info["token_bytes"] == 4096
        _check_plan_matches_oracle(case, read_once_min_tokens=-1, read_once_min_mib=min_mib)
        step.close()
    # the built-in minimums as reported
    step = _lib_plan(case)
    info = step.plan_info()
    assert (info["read_once_min_tokens"], info["read_once_min_mib"]) == (1024, 64)
    step.close()
