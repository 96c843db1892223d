"""psp_run_noalloc: the decode step for callers that cannot allocate device
memory (an engine whose KV pool and weights already hold nearly all of HBM, a
plugin callback that must not allocate, a latency-critical loop).  It must give
the same result as psp_run with a caller workspace, call after call, while the
library's static scratch keeps the previous call's contents.

Kept in a file that pytest collects last, so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_shared_prefix_gb300 as psp
import workloads
from gpu_util import READ_ONCE_ALWAYS, TOL, device_tensors, max_err, run_case

pytestmark = pytest.mark.gpu


def _fresh_outputs(case):
    w = case.workload
    dt = torch.float32 if w.o_dtype == "f32" else torch.bfloat16
    o = torch.full((case.batch, w.num_q_heads, w.head_dim), float("nan"), dtype=dt, device="cuda:0")
    lse = torch.full((case.batch, w.num_q_heads), float("nan"), dtype=torch.float32, device="cuda:0")
    return o, lse


NOALLOC_CASES = [
    ("agent", dict(batch=24, prefix_len=512, private_range=(1, 300)), {}),
    ("fp8_large", dict(batch=10, prefix_len=384, private_range=(1, 200)), {}),
    ("tiny", dict(), {}),
    # the token-flat indices lie past the zeroed region of the scratch
    ("agent", dict(batch=12, prefix_len=256, private_range=(1, 300)), dict(token_flat=True)),
    # the concurrent flag is ignored on this path (one stream, no side stream to create)
    ("fp8_large", dict(batch=8, prefix_len=320, private_range=(1, 200)), dict(token_flat=True, concurrent=True)),
    # nested groups: per-request part lists in the scratch
    ("agent", dict(batch=16, prefix_len=300, private_range=(1, 200), nested=(3, 260)), {}),
]


@pytest.mark.parametrize("name,kw,flags", NOALLOC_CASES,
                         ids=["agent", "fp8", "tiny", "agent-token-flat", "fp8-concurrent-token-flat", "agent-nested"])
def test_noalloc_matches_workspace_run_twice(name, kw, flags):
    case = workloads.make_case(name, 3, **kw)
    ref_o, ref_lse = run_case(case, **flags)        # psp_run with a caller workspace
    tens = device_tensors(case)
    step = psp.DecodeStep.for_case(case, **flags, **READ_ONCE_ALWAYS)
    step.plan_case(case)
    tol = TOL[case.workload.kv_dtype]
    for _ in range(2):                             # the second call reuses the scratch as left
        o, lse = _fresh_outputs(case)
        step.run_noalloc(tens["q"], tens["k_pool"], tens["v_pool"], o, lse, tens["k_scale"], tens["v_scale"])
        torch.cuda.synchronize()
        assert step.device_status() == 0
        got_o = o.float().cpu().double().numpy()
        got_lse = lse.cpu().double().numpy()
        assert max_err(got_o, ref_o) <= tol and max_err(got_lse, ref_lse) <= tol
    o_ref, _ = oracle.attend_all(case)
    assert max_err(got_o, o_ref) <= tol
    step.close()


def test_noalloc_rejected_call_leaves_the_binding():
    # an fp8 call without scales is rejected before anything is copied; the handle's own
    # workspace stays bound, so psp_run on it still gives the workspace result
    case = workloads.make_case("fp8_large", 4, batch=6, prefix_len=256, private_range=(1, 120))
    (ref_o, ref_lse), step, ws = run_case(case, return_step=True)
    tens = device_tensors(case)
    o, lse = _fresh_outputs(case)
    t = step.tensors(tens["q"], tens["k_pool"], tens["v_pool"], o, lse, None, None)
    assert psp.psp_run_noalloc(step.handle, ctypes.byref(t), None) == -1   # PSP_ERR_INVALID_ARGUMENT
    step.run(tens["q"], tens["k_pool"], tens["v_pool"], o, lse, tens["k_scale"], tens["v_scale"])
    torch.cuda.synchronize()
    assert step.device_status() == 0
    assert np.array_equal(o.float().cpu().double().numpy(), ref_o)
    step.close()


def test_noalloc_rejects_a_plan_larger_than_the_scratch():
    case = workloads.make_case("fp8_large", 0, batch=4096, tables_only=True)
    step = psp.DecodeStep.for_case(case)
    step.plan_case(case)
    assert step.workspace_size() > 64 << 20
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda:0")
    t = step.tensors(dummy, dummy, dummy, dummy)
    st = psp.psp_run_noalloc(step.handle, ctypes.byref(t), None)
    assert st == -7                                # PSP_ERR_WORKSPACE, nothing launched
    assert b"static scratch" in psp.psp_last_error(step.handle)
    step.close()
