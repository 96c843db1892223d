"""GPU parity: the CUDA decode step against the fp64 oracle on the same seeded
inputs, through the C ABI.

Small cases (every output row compared) span several 64-token tiles and
ragged tails for each workload shape; full-size workloads compare every row
(2,048 sampled rows plus the extremes on the 32,768-row fp8 batch) in the
launch configuration the benchmark times.  Tolerances are the
max |O_gpu - O_oracle| bounds of the target: 2e-3 (fp32 KV), 1.5e-2 (bf16
KV), 6e-2 (fp8 KV); LSE uses the same bound.  Indexing outputs are bit-exact.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_shared_prefix_gb300 as psp
import workloads
from gpu_util import READ_ONCE_ALWAYS, TOL, device_tensors, max_err, run_case

pytestmark = pytest.mark.gpu

SMALL = [
    ("tiny", dict()),
    ("tiny-seed7", dict(name="tiny", seed=7)),
    ("llama", dict(name="llama8b_noshare", batch=4, private_range=(100, 700))),
    ("agent", dict(name="agent", batch=12, prefix_len=256, private_range=(1, 300))),
    ("short_prefix", dict(name="short_prefix", batch=8, private_range=(1, 400))),
    ("fp8_large", dict(name="fp8_large", batch=6, prefix_len=1024, private_range=(1, 300))),
    ("agent-d64", dict(name="agent", batch=5, prefix_len=128, private_range=(1, 200), head_dim=64)),
    ("fp8-d64", dict(name="fp8_large", batch=4, prefix_len=192, private_range=(1, 150), head_dim=64)),
    ("fp32-d128", dict(name="tiny", head_dim=128, private_range=(1, 200))),
    ("agent-g1", dict(name="agent", batch=7, prefix_len=64, private_range=(1, 100), num_q_heads=8)),
    ("agent-g8", dict(name="agent", batch=4, prefix_len=80, private_range=(1, 100), num_q_heads=64)),
    ("fp8-g2", dict(name="fp8_large", batch=5, prefix_len=96, private_range=(1, 70), num_q_heads=16)),
]


def _make(kw):
    kw = dict(kw)
    name = kw.pop("name", None)
    seed = kw.pop("seed", 0)
    return workloads.make_case(name, seed, **kw)


@pytest.mark.parametrize("label,kw", SMALL, ids=[s[0] for s in SMALL])
@pytest.mark.parametrize("branch", ["dense", "cascade"])
def test_small_matches_oracle(label, kw, branch):
    kw = dict(kw)
    kw.setdefault("name", label)
    case = _make(kw)
    thr = 1 if branch == "dense" else 1 << 20
    o, lse = run_case(case, threshold=thr)
    ref_o, ref_lse = oracle.attend_all(case)
    tol = TOL[case.workload.kv_dtype]
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert max_err(o, ref_o) <= tol
    assert max_err(lse, ref_lse) <= tol


def test_page_sizes_and_layouts_bit_identical():
    outs = []
    for ps in (1, 16, 128):
        for layout in ("scatter", "contiguous"):
            case = workloads.make_case("llama8b_noshare", 2, batch=3, private_range=(200, 900), page_size=ps,
                                       layout=layout)
            outs.append(run_case(case))
    case = workloads.make_case("llama8b_noshare", 2, batch=3, private_range=(200, 900), page_size=16,
                               layout="block128")
    outs.append(run_case(case))
    for o, l in outs[1:]:
        assert np.array_equal(o, outs[0][0]) and np.array_equal(l, outs[0][1])
    ref_o, ref_lse = oracle.attend_all(case)
    assert max_err(outs[0][0], ref_o) <= TOL["bf16"]


@pytest.mark.parametrize("name", ["llama8b_noshare", "fp8_large"])
def test_every_page_size_bit_identical(name):
    """Every supported page size gives the same bits: pages smaller than a 16-token sub-tile
    (one table entry per row), pages holding whole sub-tiles (one entry per sub-tile) and a
    page larger than any context; suffixes that end mid-page, with and without a shared prefix."""
    kw = dict(batch=3, private_range=(1, 700)) if name == "llama8b_noshare" else dict(
        batch=4, prefix_len=0, private_range=(1, 700))
    outs = [run_case(workloads.make_case(name, 4, page_size=ps, **kw)) for ps in (1, 2, 4, 8, 16, 32, 256, 1024)]
    for o, l in outs[1:]:
        assert np.array_equal(o, outs[0][0]) and np.array_equal(l, outs[0][1])
    case = workloads.make_case(name, 4, page_size=16, **kw)
    ref_o, ref_lse = oracle.attend_all(case)
    tol = TOL[case.workload.kv_dtype]
    assert max_err(outs[0][0], ref_o) <= tol and max_err(outs[0][1], ref_lse) <= tol


@pytest.mark.parametrize("ps", [2, 4, 8, 32, 256])
@pytest.mark.parametrize("name", ["agent", "fp8_large"])
def test_shared_prefix_at_other_page_sizes(name, ps):
    """Shared-prefix steps at page sizes the other tests leave out (the dense kernel's
    per-page boxes of 2-8 tokens, a prefix tail kept private by large pages) against the
    oracle, dense and cascade."""
    case = workloads.make_case(name, 5, batch=12, prefix_len=600, private_range=(1, 300), page_size=ps)
    tol = TOL[case.workload.kv_dtype]
    ref_o, ref_lse = oracle.attend_all(case)
    for thr in (1, 1 << 20):
        o, lse = run_case(case, threshold=thr)
        assert max_err(o, ref_o) <= tol and max_err(lse, ref_lse) <= tol, (thr, max_err(o, ref_o))


def test_token_flat_lowering_bit_identical():
    for name, kw in (("agent", dict(batch=6, prefix_len=160, private_range=(1, 200))),
                     ("fp8_large", dict(batch=4, prefix_len=128, private_range=(1, 150))),
                     ("tiny", {})):
        case = workloads.make_case(name, 4, **kw)
        a = run_case(case)
        b = run_case(case, token_flat=True)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]), name


def test_contiguous_prefix_bit_identical():
    """A prefix whose pages are physically consecutive is fetched in whole-tile boxes; the
    results must equal, bit for bit, those of the same batch with its pages scattered."""
    for name, kw in (("agent", dict(batch=20, prefix_len=1000, private_range=(1, 200))),
                     ("fp8_large", dict(batch=12, prefix_len=700, private_range=(1, 300)))):
        for ps in (16, 64):
            outs = []
            for layout in ("scatter", "contiguous", "block128"):
                case = workloads.make_case(name, 6, page_size=ps, layout=layout, **kw)
                outs.append(run_case(case))
            for o, l in outs[1:]:
                assert np.array_equal(o, outs[0][0]) and np.array_equal(l, outs[0][1]), (name, ps)
            ref_o, ref_lse = oracle.attend_all(case)
            tol = TOL[case.workload.kv_dtype]
            assert max_err(outs[0][0], ref_o) <= tol and max_err(outs[0][1], ref_lse) <= tol


def test_launch_forms_bit_identical(monkeypatch):
    """The sequential and the concurrent dependent-launch forms merge a one-split request's
    row on different paths (in its suffix CTA, or through its counter by whichever part
    arrives last, at a moment set by timing); the result must not depend on the path."""
    for name, kw in (("agent", dict(batch=24, prefix_len=1024, private_range=(1, 300))),
                     ("fp8_large", dict(batch=16, prefix_len=512, private_range=(1, 400)))):
        case = workloads.make_case(name, 5, **kw)
        outs = []
        for form in ("1", "2", "2"):
            monkeypatch.setenv("PSP_PDL_FORM", form)
            outs.append(run_case(case))
        for o, l in outs[1:]:
            assert np.array_equal(o, outs[0][0]) and np.array_equal(l, outs[0][1]), name
        ref_o, ref_lse = oracle.attend_all(case)
        tol = TOL[case.workload.kv_dtype]
        assert max_err(outs[0][0], ref_o) <= tol and max_err(outs[0][1], ref_lse) <= tol


def test_expand_kv_indices_bit_exact():
    for ps in (1, 16, 128):
        case = workloads.make_case("agent", 1, batch=9, prefix_len=300, private_range=(1, 500), page_size=ps)
        step = psp.DecodeStep.for_case(case)
        step.plan_case(case)
        ws = torch.empty(step.workspace_size(), dtype=torch.uint8, device="cuda:0")
        step.upload(ws)
        n = step.plan_info()["kv_indices_len"]
        out = torch.full((n + 7,), -7, dtype=torch.int32, device="cuda:0")
        step.expand_kv_indices(out)
        torch.cuda.synchronize()
        indptr, idx = oracle.expand_kv_indices(case)
        got = out.cpu().numpy()
        assert np.array_equal(got[:n], idx) and np.all(got[n:] == -7)
        assert np.array_equal(step.plan_query("kv_indptr"), indptr)
        step.close()


def test_shared_equals_per_request_paged():
    case = workloads.make_case("agent", 5, batch=16, prefix_len=512, private_range=(1, 256))
    a = run_case(case)
    b = run_case(case.without_sharing())
    ref_o, ref_lse = oracle.attend_all(case)
    for o, l in (a, b):
        assert max_err(o, ref_o) <= TOL["bf16"] and max_err(l, ref_lse) <= TOL["bf16"]


def test_edge_cases():
    # empty suffix: a context that ends exactly at the page-aligned shared prefix
    case = workloads.make_case("agent", 6, batch=5, prefix_len=128, private_lengths=[0, 3, 0, 17, 64])
    o, lse = run_case(case)
    ro, rl = oracle.attend_all(case)
    assert max_err(o, ro) <= TOL["bf16"] and max_err(lse, rl) <= TOL["bf16"]
    # prefix shorter than one page: nothing shared, everything is suffix
    case = workloads.make_case("agent", 6, batch=4, prefix_len=9, private_range=(1, 30))
    o, lse = run_case(case)
    ro, rl = oracle.attend_all(case)
    assert max_err(o, ro) <= TOL["bf16"]
    # one-token contexts
    case = workloads.make_case("llama8b_noshare", 6, batch=5, private_lengths=[1, 1, 2, 1, 3])
    o, lse = run_case(case)
    ro, rl = oracle.attend_all(case)
    assert max_err(o, ro) <= TOL["bf16"] and max_err(lse, rl) <= TOL["bf16"]
    # unaligned prefix at page size 128 (tail of the prefix stays private)
    case = workloads.make_case("fp8_large", 6, batch=4, prefix_len=300, private_range=(1, 90), page_size=128)
    o, lse = run_case(case)
    ro, rl = oracle.attend_all(case)
    assert max_err(o, ro) <= TOL["fp8_e4m3"] and max_err(lse, rl) <= TOL["fp8_e4m3"]


def test_empty_batch_then_replan():
    """A batch of no requests plans, uploads and runs (nothing is launched and the device
    status stays clear); the same handle then plans and runs a real batch correctly."""
    case = workloads.make_case("agent", 9, batch=6, prefix_len=160, private_range=(1, 90))
    tens = device_tensors(case)
    step = psp.DecodeStep.for_case(case, **READ_ONCE_ALWAYS)
    z = np.zeros(0, np.int32)
    step.plan(z, np.zeros(1, np.int32), z)
    ws = torch.empty(max(step.workspace_size(), 256), dtype=torch.uint8, device="cuda:0")
    step.upload(ws)
    w = case.workload
    o = torch.full((case.batch, w.num_q_heads, w.head_dim), float("nan"), dtype=torch.bfloat16, device="cuda:0")
    lse = torch.full((case.batch, w.num_q_heads), float("nan"), dtype=torch.float32, device="cuda:0")
    step.set_kernel_timing(True)
    step.run(tens["q"], tens["k_pool"], tens["v_pool"], o, lse)
    torch.cuda.synchronize()
    assert step.kernel_times() == []
    assert step.device_status() == 0
    assert torch.isnan(lse).all()  # nothing was written
    step.plan_case(case)
    ws = torch.empty(step.workspace_size(), dtype=torch.uint8, device="cuda:0")
    step.upload(ws)
    step.run(tens["q"], tens["k_pool"], tens["v_pool"], o, lse)
    torch.cuda.synchronize()
    assert step.device_status() == 0
    assert len(step.kernel_times()) >= 1
    ro, rl = oracle.attend_all(case)
    assert max_err(o.float().cpu().numpy(), ro) <= TOL["bf16"]
    assert max_err(lse.cpu().numpy(), rl) <= TOL["bf16"]
    step.close()


def test_step_host_matches_run():
    case = workloads.make_case("agent", 8, batch=10, prefix_len=192, private_range=(1, 200))
    w = case.workload
    (o_ref, l_ref), step, ws = run_case(case, return_step=True)
    tens = device_tensors(case)
    q_host = torch.from_numpy(case.q.view(np.int16)).pin_memory()
    o_host = torch.empty((case.batch, w.num_q_heads, w.head_dim), dtype=torch.int16).pin_memory()
    l_host = torch.empty((case.batch, w.num_q_heads), dtype=torch.float32).pin_memory()
    o_dev = torch.empty((case.batch, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda:0")
    l_dev = torch.empty((case.batch, w.num_q_heads), dtype=torch.float32, device="cuda:0")
    q_dev = torch.empty_like(tens["q"])
    batch, keep = step.make_case_batch(case)
    dev = step.tensors(q_dev, tens["k_pool"], tens["v_pool"], o_dev, l_dev)
    step.step_host(batch, q_host, o_host, l_host, dev, ws)
    o = o_host.view(torch.bfloat16).float().double().numpy()
    assert np.array_equal(o, o_ref) and np.array_equal(l_host.double().numpy(), l_ref)
    step.close()


def test_kernel_timing_reports_launches():
    case = workloads.make_case("agent", 9, batch=8, prefix_len=256, private_range=(1, 200))
    tens = device_tensors(case)
    step = psp.DecodeStep.for_case(case, dense_threshold=1, **READ_ONCE_ALWAYS)
    step.plan_case(case)
    ws = torch.empty(step.workspace_size(), dtype=torch.uint8, device="cuda:0")
    step.upload(ws)
    w = case.workload
    o = torch.empty((case.batch, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda:0")
    step.set_kernel_timing(True)
    step.run(tens["q"], tens["k_pool"], tens["v_pool"], o)
    torch.cuda.synchronize()
    names = [n for n, _ in step.kernel_times()]
    assert names == ["prefix_dense", "suffix_splitkv"]
    assert all(t > 0 for _, t in step.kernel_times())
    step.close()


# ---------------------------------------------------------------- full size

FULL = [("llama8b_noshare", 16), ("agent", 16), ("short_prefix", 16), ("fp8_large", 16),
        ("tiny", 16), ("llama8b_noshare", 1), ("llama8b_noshare", 128)]


def _sample_rows(case, n, seed=0):
    rng = np.random.default_rng(seed)
    B, Hq = case.batch, case.workload.num_q_heads
    rows = rng.choice(B * Hq, size=min(n, B * Hq), replace=False)
    # always include the longest and the shortest request
    L = case.kv_len
    extra = [int(np.argmax(L)) * Hq, int(np.argmin(L)) * Hq + Hq - 1]
    rows = np.unique(np.concatenate([rows, extra]))
    return rows // Hq, rows % Hq


@pytest.mark.parametrize("name,ps", FULL, ids=[f"{n}-ps{p}" for n, p in FULL])
def test_full_size_rows(name, ps):
    # every (request, query head) row on the four smaller workloads; 2,048 sampled rows
    # plus the longest and shortest requests on the 512-request fp8 batch (32,768 rows)
    case = workloads.make_case(name, 0, page_size=ps)
    o, lse = run_case(case)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    tol = TOL[case.workload.kv_dtype]
    if case.batch * case.workload.num_q_heads <= 8192:
        ro, rl = oracle.attend_all(case)
        assert max_err(o, ro) <= tol
        assert max_err(lse, rl) <= tol
    else:
        bb, hh = _sample_rows(case, 2048)
        ro, rl = oracle.attend(case, bb, hh)
        assert max_err(o[bb, hh], ro) <= tol
        assert max_err(lse[bb, hh], rl) <= tol


def test_full_size_page_sizes_bit_identical():
    outs = [run_case(workloads.make_case("llama8b_noshare", 0, page_size=ps)) for ps in (1, 16, 128)]
    for o, l in outs[1:]:
        assert np.array_equal(o, outs[0][0]) and np.array_equal(l, outs[0][1])


def test_full_size_paged_comparator_matches():
    # the read-once step and the per-request paged step against the oracle, every row
    case = workloads.make_case("agent", 0)
    a = run_case(case)
    b = run_case(case.without_sharing())
    ro, rl = oracle.attend_all(case)
    for o, l in (a, b):
        assert max_err(o, ro) <= TOL["bf16"] and max_err(l, rl) <= TOL["bf16"]


def test_bounded_wait_reports_timeout_instead_of_hanging():
    case = workloads.make_case("tiny", 0)
    step = psp.DecodeStep.for_case(case)
    step.plan_case(case)
    ws = torch.empty(step.workspace_size(), dtype=torch.uint8, device="cuda:0")
    step.upload(ws)
    torch.cuda.synchronize()
    assert step.device_status() == 0
    step.wait_selftest(2000)
    torch.cuda.synchronize()
    code = step.device_status(raise_on_timeout=False)
    assert code & 0xff == 1 and code >> 8 == 99
    # the context stays usable and a fresh upload clears the word
    step.upload(ws)
    o, lse = run_case(case)
    ref_o, _ = oracle.attend_all(case)
    assert max_err(o, ref_o) <= TOL["f32"]
    assert step.device_status() == 0
    step.close()


DENSE = [
    ("rows-2-blocks", dict(name="agent", batch=80, prefix_len=384, private_range=(1, 64))),
    ("rows-exact-256", dict(name="agent", batch=64, prefix_len=256, private_range=(1, 32))),
    ("rows-400", dict(name="agent", batch=100, prefix_len=320, private_range=(1, 32))),
    ("partial-tile", dict(name="agent", batch=40, prefix_len=208, private_range=(1, 40))),
    ("long-prefix", dict(name="agent", batch=33, prefix_len=2048 + 64, private_range=(1, 30))),
    ("ps128", dict(name="agent", batch=20, prefix_len=640, private_range=(1, 200), page_size=128)),
    ("ps1", dict(name="agent", batch=20, prefix_len=300, private_range=(1, 100), page_size=1)),
    ("g8", dict(name="agent", batch=24, prefix_len=512, private_range=(1, 50), num_q_heads=64)),
    ("fp8-2-blocks", dict(name="fp8_large", batch=20, prefix_len=640, private_range=(1, 60))),
    ("fp8-3-tiles", dict(name="fp8_large", batch=40, prefix_len=448, private_range=(1, 30))),
    ("fp8-partial-tile", dict(name="fp8_large", batch=9, prefix_len=336, private_range=(1, 30))),
    ("fp8-g4-ps1", dict(name="fp8_large", batch=12, prefix_len=256, private_range=(1, 40), num_q_heads=32,
                        page_size=1)),
]


@pytest.mark.parametrize("label,kw", DENSE, ids=[d[0] for d in DENSE])
def test_dense_prefix_matches_oracle(label, kw):
    case = _make(kw)
    tol = TOL[case.workload.kv_dtype]
    o, lse = run_case(case, threshold=1)
    ref_o, ref_lse = oracle.attend_all(case)
    assert max_err(o, ref_o) <= tol and max_err(lse, ref_lse) <= tol
    # the token-flat lowering reads the same tokens: bit-identical
    o2, lse2 = run_case(case, threshold=1, token_flat=True)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    # different SM counts change the prefix chunking; the result stays within tolerance
    o3, lse3 = run_case(case, threshold=1, num_sms=37)
    assert max_err(o3, ref_o) <= tol and max_err(lse3, ref_lse) <= tol


CONCURRENT = [
    ("tiny", dict(name="tiny")),
    ("agent-dense", dict(name="agent", batch=40, prefix_len=512, private_range=(1, 300)), 1),
    ("agent-cascade", dict(name="agent", batch=12, prefix_len=256, private_range=(1, 300)), 1 << 20),
    ("fp8-dense", dict(name="fp8_large", batch=20, prefix_len=640, private_range=(1, 600)), 1),
    ("multi-split", dict(name="short_prefix", batch=6, private_range=(800, 2000)), 0),
    ("empty-suffix", dict(name="agent", batch=5, prefix_len=128, private_lengths=[0, 3, 0, 17, 64]), 1),
]


@pytest.mark.parametrize("spec", CONCURRENT, ids=[c[0] for c in CONCURRENT])
def test_concurrent_prefix_matches_oracle(spec):
    label, kw = spec[0], spec[1]
    thr = spec[2] if len(spec) > 2 else 0
    case = _make(kw)
    tol = TOL[case.workload.kv_dtype]
    ref_o, ref_lse = oracle.attend_all(case)
    for num_sms in (0, 11):   # 11 SMs: many splits per request, counters exercised
        o, lse = run_case(case, threshold=thr, concurrent=True, num_sms=num_sms)
        assert max_err(o, ref_o) <= tol and max_err(lse, ref_lse) <= tol, (label, num_sms)
    # a second step through the same workspace: the counters reset themselves
    (o1, l1), step, ws = run_case(case, threshold=thr, concurrent=True, return_step=True)
    tens = device_tensors(case)
    w = case.workload
    o2 = torch.empty((case.batch, w.num_q_heads, w.head_dim),
                     dtype=torch.float32 if w.o_dtype == "f32" else torch.bfloat16, device="cuda:0")
    l2 = torch.empty((case.batch, w.num_q_heads), dtype=torch.float32, device="cuda:0")
    step.run(tens["q"], tens["k_pool"], tens["v_pool"], o2, l2, tens["k_scale"], tens["v_scale"])
    torch.cuda.synchronize()
    assert max_err(o2.float().cpu().double().numpy(), ref_o) <= tol
    assert max_err(l2.cpu().double().numpy(), ref_lse) <= tol
    step.close()


def _multi_group_full_case():
    """Three prefix groups (160, 37 and 512 tokens; 8, 6 and 6 members) plus ungrouped
    requests in one pool, with every slot of the pool holding finite random K/V."""
    from test_abi_host import _multi_group_case
    tables = _multi_group_case()
    full = workloads.make_case("agent", 3, batch=tables.batch)
    w = full.workload
    shape = (tables.num_pages, tables.page_size, w.num_kv_heads, w.head_dim)
    k = workloads.bf16_bits_from_f32(workloads.normal_f32(shape, 21, 1))
    v = workloads.bf16_bits_from_f32(workloads.normal_f32(shape, 21, 2))
    return dataclasses.replace(tables, q=full.q, k_pool=k, v_pool=v, k_scale=None, v_scale=None)


@pytest.mark.gpu
def test_multi_group_mixed_branches_match_oracle():
    # M_eff = 32, 24, 24 (G = 4): threshold 30 sends group 0 to the dense kernel and
    # groups 1 and 2 to the cascade kernel in the same step, then the suffix kernel
    case = _multi_group_full_case()
    ref_o, ref_lse = oracle.attend_all(case)
    tol = TOL[case.workload.kv_dtype]
    tens = device_tensors(case)
    for thr, kw in ((30, {}), (1, {}), (1 << 20, {}), (30, dict(concurrent=True)), (30, dict(token_flat=True))):
        o, lse = run_case(case, threshold=thr, tensors=tens, **kw)
        assert np.isfinite(o).all() and np.isfinite(lse).all(), (thr, kw)
        assert max_err(o, ref_o) <= tol and max_err(lse, ref_lse) <= tol, (thr, kw, max_err(o, ref_o))


def _fp8_growing_scores_case():
    """e4m3 suffixes whose first 128 keys per request are zero: the first tile's scores are
    all 0, so a later tile's maximum exceeds the first reference by more than 2^8 and the
    tensor-core suffix kernel must move its reference max and rescale O^T mid-sequence.
    Lengths give 1-11 tiles (ragged tails; more tiles than ring stages)."""
    case = workloads.make_case("fp8_large", 11, batch=4, prefix_len=0, private_lengths=[700, 130, 1300, 257])
    ps = case.page_size
    k = case.k_pool.reshape(-1, case.workload.num_kv_heads, case.workload.head_dim)
    for b in range(case.batch):
        pages = case.page_indices[case.page_indptr[b]:case.page_indptr[b + 1]]
        t = np.arange(min(128, int(case.kv_len[b])))
        k[pages[t // ps] * ps + t % ps] = 0  # e4m3 code 0 is +0
    return case


@pytest.mark.gpu
def test_fp8_suffix_rescale_and_long_splits(monkeypatch):
    case = _fp8_growing_scores_case()
    ref_o, ref_lse = oracle.attend_all(case)
    tol = TOL["fp8_e4m3"]
    tens = device_tensors(case)
    # default partition (256-token splits here: every request is merged through its
    # counter), then one split per request (direct merge, up to 11 tiles per CTA)
    for min_tiles in (None, "64"):
        if min_tiles:
            monkeypatch.setenv("PSP_SPLIT_MIN_TILES", min_tiles)
        o, lse = run_case(case, tensors=tens)
        assert np.isfinite(o).all() and np.isfinite(lse).all(), min_tiles
        assert max_err(o, ref_o) <= tol and max_err(lse, ref_lse) <= tol, (min_tiles, max_err(o, ref_o))



def test_paged_branch_equals_the_plan_without_the_group():
    # the built-in read-once minimums send the short-prefix batch (512 shared tokens) down the
    # paged branch: its step is the step of the same batch without the group, bit for bit
    case = workloads.make_case("short_prefix", 0)
    (o, lse), step, ws = run_case(case, read_once=None, return_step=True)
    assert list(step.plan_query("group_branch")) == [psp.BRANCH_PAGED]
    assert step.plan_info()["prefix_dense_ctas"] == 0
    step.close()
    o2, lse2 = run_case(case.without_sharing(), read_once=None)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    ro, rl = oracle.attend_all(case)
    assert max_err(o, ro) <= TOL["bf16"] and max_err(lse, rl) <= TOL["bf16"]
    # and the headline batches read their prefixes once under the same minimums
    for name in ("agent", "fp8_large"):
        c = workloads.make_case(name, 0, tables_only=True)
        s = psp.DecodeStep.for_case(c)
        s.plan_case(c)
        assert list(s.plan_query("group_branch")) == [psp.BRANCH_DENSE]
        s.close()


def test_outputs_and_workspace_guard_bands():
    """Canary words before and after O, LSE and the workspace stay untouched by a step (nested
    groups, e4m3 and bf16, both launch forms, the token-flat lowering): no kernel writes
    outside its buffers."""
    from gpu_util import device_tensors
    for name, kw, flags in (("fp8_large", dict(batch=12, prefix_len=700, private_range=(1, 400), nested=(3, 300)), {}),
                            ("agent", dict(batch=10, prefix_len=520, private_range=(1, 300)), dict(token_flat=True)),
                            ("agent", dict(batch=10, prefix_len=520, private_range=(1, 300)), dict(concurrent=True))):
        case = workloads.make_case(name, 9, **kw)
        w = case.workload
        tens = device_tensors(case)
        step = psp.DecodeStep.for_case(case, **flags, read_once_min_tokens=-1, read_once_min_mib=-1)
        step.plan_case(case)
        guard = 4096  # bytes on each side (a multiple of 256, so alignment is kept)
        nws = step.workspace_size()
        ws_all = torch.full((nws + 2 * guard,), 0x5A, dtype=torch.uint8, device="cuda:0")
        ws = ws_all[guard:guard + nws]
        step.upload(ws)
        n_o = case.batch * w.num_q_heads * w.head_dim
        o_all = torch.full((n_o + 2 * guard // 2,), -7.0, dtype=torch.bfloat16, device="cuda:0")
        o = o_all[guard // 2:guard // 2 + n_o].view(case.batch, w.num_q_heads, w.head_dim)
        n_l = case.batch * w.num_q_heads
        l_all = torch.full((n_l + 2 * guard // 4,), -7.0, dtype=torch.float32, device="cuda:0")
        lse = l_all[guard // 4:guard // 4 + n_l].view(case.batch, w.num_q_heads)
        step.run(tens["q"], tens["k_pool"], tens["v_pool"], o, lse, tens["k_scale"], tens["v_scale"])
        torch.cuda.synchronize()
        assert step.device_status() == 0
        assert bool((ws_all[:guard] == 0x5A).all()) and bool((ws_all[guard + nws:] == 0x5A).all()), name
        assert bool((o_all[:guard // 2] == -7.0).all()) and bool((o_all[guard // 2 + n_o:] == -7.0).all()), name
        assert bool((l_all[:guard // 4] == -7.0).all()) and bool((l_all[guard // 4 + n_l:] == -7.0).all()), name
        ref_o, ref_lse = oracle.attend_all(case)
        tol = TOL[w.kv_dtype]
        assert max_err(o.float().cpu().double().numpy(), ref_o) <= tol
        assert max_err(lse.cpu().double().numpy(), ref_lse) <= tol
        step.close()
