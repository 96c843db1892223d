"""Helpers for the GPU tests: run one decode step of a generated case through
the C ABI and return host arrays."""
from __future__ import annotations

import numpy as np
import torch

import paged_shared_prefix_gb300 as psp

TOL = {"f32": 2e-3, "bf16": 1.5e-2, "fp8_e4m3": 6e-2}

# The kernel parity tests read every shared prefix once, whatever its size, so that the prefix
# kernels run on their small cases; the dispatcher's built-in read-once minimums have tests of
# their own (read_once=None keeps them).
READ_ONCE_ALWAYS = dict(read_once_min_tokens=-1, read_once_min_mib=-1)


def device_tensors(case, dev="cuda:0"):
    def t(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return dict(q=t(case.q), k_pool=t(case.k_pool), v_pool=t(case.v_pool), k_scale=t(case.k_scale),
                v_scale=t(case.v_scale))


def run_case(case, *, threshold=0, token_flat=False, tensors=None, num_sms=0, return_step=False,
             concurrent=False, read_once=READ_ONCE_ALWAYS):
    """One step on cuda:0; returns (O float64 [B, Hq, d], LSE float64 [B, Hq])."""
    w = case.workload
    dev = torch.device("cuda:0")
    tens = tensors or device_tensors(case)
    step = psp.DecodeStep.for_case(case, num_sms=num_sms, dense_threshold=threshold, token_flat=token_flat,
                                   concurrent=concurrent, **(read_once or {}))
    step.plan_case(case)
    ws = torch.empty(step.workspace_size(), dtype=torch.uint8, device=dev)
    step.upload(ws)
    o = torch.full((case.batch, w.num_q_heads, w.head_dim), float("nan"),
                   dtype=torch.float32 if w.o_dtype == "f32" else torch.bfloat16, device=dev)
    lse = torch.full((case.batch, w.num_q_heads), float("nan"), dtype=torch.float32, device=dev)
    step.run(tens["q"], tens["k_pool"], tens["v_pool"], o, lse, tens["k_scale"], tens["v_scale"])
    torch.cuda.synchronize()
    status = step.device_status()
    assert status == 0, f"device status {status}"
    out = (o.float().cpu().double().numpy(), lse.cpu().double().numpy())
    if return_step:
        return out, step, ws
    step.close()
    return out


def max_err(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))))
