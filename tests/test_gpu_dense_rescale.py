"""GPU parity of the shared-prefix kernels when the running maximum of the
scores has to move in the middle of the prefix.

The dense tensor-core kernel keeps a lazily updated reference maximum per row:
the reference moves (and the accumulated output is rescaled in tensor memory)
only when a tile's maximum exceeds it by more than 2^8 in the base-2 exponent,
i.e. by more than 8 ln 2 ~= 5.55 in natural-log units of q.k / sqrt(d).  With
Q, K ~ N(0, 1) that never happens, so these cases build prefixes whose scores
jump: keys that are zero (or scaled down) over most of the prefix and at full
scale later, with the queries scaled up.  Each case first checks, from the
decoded inputs alone, that the construction crosses the bound, then compares
the GPU step with the fp64 oracle (max |dO|, |dLSE| within the dtype's
tolerance) in the default partition and with many prefix chunks (num_sms=37).

A second family gives every query row the same direction (scaled per row) and
plants one key along it, so that every row's score jump lies just below the
bound (e4m3 probabilities up to 2^7.5, inside e4m3's 448, without a rescale)
or just above it (a rescale in every row).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import TOL, max_err, run_case

pytestmark = pytest.mark.gpu

LN2 = float(np.log(2.0))


def _decode_pool(case) -> np.ndarray:
    """K pool as float64 [slots, Hkv, d] (codes decoded, fp8 scale applied)."""
    w = case.workload
    k = case.k_pool.reshape(-1, w.num_kv_heads, w.head_dim)
    if w.kv_dtype == "bf16":
        return (k.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if w.kv_dtype == "fp8_e4m3":
        vals = torch.from_numpy(np.ascontiguousarray(k)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        return vals * case.k_scale.astype(np.float64)[None, :, None]
    return k.astype(np.float64)


def _decode_q(case) -> np.ndarray:
    return (case.q.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _prefix_slots(case) -> np.ndarray:
    ps = case.page_size
    n_sh = int(case.group_prefix_len[0]) // ps
    pages = case.page_indices[case.page_indptr[0]:case.page_indptr[0] + n_sh].astype(np.int64)
    t = np.arange(n_sh * ps)
    return pages[t // ps] * ps + t % ps


def _largest_jump(case, window=64) -> float:
    """Largest amount, in natural-log units, by which the maximum score of a window of
    the shared prefix exceeds the running maximum of the windows before it, over all
    (request, query head) rows."""
    w = case.workload
    G = w.num_q_heads // w.num_kv_heads
    k = _decode_pool(case)[_prefix_slots(case)]          # [P, Hkv, d]
    q = _decode_q(case)                                   # [B, Hq, d]
    P = k.shape[0]
    best = -np.inf
    for h in range(w.num_kv_heads):
        s = q[:, h * G:(h + 1) * G, :].reshape(-1, w.head_dim) @ k[:, h, :].T / np.sqrt(w.head_dim)
        run = np.full(s.shape[0], -np.inf)
        for a in range(0, P, window):
            m = s[:, a:a + window].max(axis=1)
            if a > 0:
                best = max(best, float(np.max(m - run)))
            run = np.maximum(run, m)
    return best


def _scale_bf16_bits(bits: np.ndarray, factor: float) -> np.ndarray:
    x = (bits.astype(np.uint32) << 16).view(np.float32) * np.float32(factor)
    return workloads.bf16_bits_from_f32(x)


def _aligned_queries(case, seed: int, norm: float):
    """Replaces every query row by c_row * u, with u = norm / sqrt(d) * (random signs):
    every element of a row has the same magnitude, so the e4m3 kernels' per-row query
    quantisation (scale amax / 448) is exact and the scores carry no quantisation error;
    c_row in [0.75, 1.25] makes the rows differ.  Returns (u as stored for c = 1, c)."""
    w = case.workload
    rng = np.random.default_rng([seed, 99])
    u = norm / np.sqrt(w.head_dim) * rng.choice([-1.0, 1.0], size=w.head_dim)
    c = rng.uniform(0.75, 1.25, size=(case.batch, w.num_q_heads))
    case.q = workloads.bf16_bits_from_f32((c[..., None] * u[None, None, :]).astype(np.float32))
    return _decode_q(case)[0, 0] / c[0, 0], c


def _quiet_values(case):
    """Scales every value by 1/4 (bf16, exact) or 1/8 (e4m3, through the per-head scale).
    A peaked softmax makes O close to one value row; small values keep the bf16 rounding
    of O and the e4m3 rounding of the probabilities inside the absolute tolerance."""
    if case.workload.kv_dtype == "bf16":
        case.v_pool = _scale_bf16_bits(case.v_pool, 0.25)
    else:
        case.v_scale = (case.v_scale * np.float32(0.125)).astype(np.float32)


def _store_keys(case, slots, kvec):
    """Writes the float key kvec [d] (all KV heads) at the given pool slots, encoded."""
    w = case.workload
    kflat = case.k_pool.reshape(-1, w.num_kv_heads, w.head_dim)
    rows = np.broadcast_to(kvec.astype(np.float32), (w.num_kv_heads, w.head_dim))
    if w.kv_dtype == "bf16":
        kflat[slots] = workloads.bf16_bits_from_f32(rows.copy())
    else:
        codes = np.clip(rows / case.k_scale[:, None], -448.0, 448.0).astype(np.float32)
        kflat[slots] = workloads.fp8_codes_from_f32(codes)


def _jump_case(kv_dtype: str, where: str, seed: int):
    """Shared prefix of 1024 tokens, 64 requests x 4 query heads per KV head (M_eff 256:
    both 128-row query tiles of a dense block).  `where` = "early": the first 192 prefix
    tokens are quiet; "last": all but the last 64 are.  Then the first windows after the
    quiet part jump by far more than the bound.
    bf16: queries scaled by 8; quiet keys are zero ("early") or scaled by 1/16 ("last").
    e4m3 (whose kernels quantise each query row to e4m3, an error proportional to the
    score): every query row is c_row * u, quiet keys are zero, and a few keys after the
    quiet part lie along u with a score of ~10 c_row (natural units), where the error of
    the quantised query averages out over the 128 elements."""
    name = "agent" if kv_dtype == "bf16" else "fp8_large"
    case = workloads.make_case(name, seed, batch=64, prefix_len=1024, private_range=(1, 200),
                               num_q_heads=32, num_kv_heads=8)
    slots = _prefix_slots(case)
    w = case.workload
    kflat = case.k_pool.reshape(-1, w.num_kv_heads, w.head_dim)
    quiet = slots[:192] if where == "early" else slots[:-64]
    _quiet_values(case)
    if kv_dtype == "bf16":
        case.q = _scale_bf16_bits(case.q, 8.0)
        if where == "last":
            kflat[quiet] = _scale_bf16_bits(kflat[quiet], 1.0 / 16.0)
        else:
            kflat[quiet] = 0
        return case
    u, _ = _aligned_queries(case, seed, 6.0)
    kflat[quiet] = 0  # e4m3 code 0 is +0
    alpha = 10.0 * np.sqrt(w.head_dim) / float(u @ u)
    loud = slots[[200, 230, 300, 517]] if where == "early" else slots[[-60, -33, -2]]
    _store_keys(case, loud, alpha * u)
    return case


JUMPS = [(dt, where, seed) for dt in ("bf16", "fp8_e4m3") for where, seed in (("early", 1), ("last", 2))]


@pytest.mark.parametrize("kv_dtype,where,seed", JUMPS, ids=[f"{d}-{w}" for d, w, _ in JUMPS])
def test_dense_prefix_rescales_mid_prefix(kv_dtype, where, seed):
    case = _jump_case(kv_dtype, where, seed)
    jump = _largest_jump(case)
    assert jump > 8 * LN2 + 2.0, f"construction does not cross the lazy-rescale bound: {jump}"
    ref_o, ref_lse = oracle.attend_all(case)
    tol = TOL[kv_dtype]
    for num_sms in (0, 37):
        for thr in (1, 1 << 20):   # dense branch, then the cascade branch on the same step
            o, lse = run_case(case, threshold=thr, num_sms=num_sms)
            assert np.isfinite(o).all() and np.isfinite(lse).all(), (num_sms, thr)
            assert max_err(o, ref_o) <= tol, (num_sms, thr, max_err(o, ref_o))
            assert max_err(lse, ref_lse) <= tol, (num_sms, thr, max_err(lse, ref_lse))


def _near_bound_case(kv_dtype: str, target_log2: float, seed: int):
    """Every query row is c_row * u (|u| = 6, c_row in [0.75, 1.25]), the first 512 prefix
    keys are zero (scores exactly 0) and prefix token 700 holds a key along u whose score
    is target_log2 * c_row in base-2 units; the rest of the prefix stays N(0, 1), with
    scores well below it.  The lazy maximum then holds at 0 and that token's probability
    is 2^(target_log2 * c_row) while that stays below the bound."""
    name = "agent" if kv_dtype == "bf16" else "fp8_large"
    case = workloads.make_case(name, seed, batch=64, prefix_len=1024, private_range=(1, 100),
                               num_q_heads=32, num_kv_heads=8)
    w = case.workload
    u, c = _aligned_queries(case, seed, 6.0)
    _quiet_values(case)
    slots = _prefix_slots(case)
    case.k_pool.reshape(-1, w.num_kv_heads, w.head_dim)[slots[:512]] = 0
    alpha = target_log2 * LN2 * np.sqrt(w.head_dim) / float(u @ u)
    _store_keys(case, slots[[700]], alpha * u)
    return case, c


NEAR = [(dt, t) for dt in ("bf16", "fp8_e4m3") for t in (6.0, 11.0)]


@pytest.mark.parametrize("kv_dtype,target", NEAR, ids=[f"{d}-{t}" for d, t in NEAR])
def test_dense_prefix_probabilities_near_the_bound(kv_dtype, target):
    # target 6.0: with c_row up to 1.25 the planted score reaches 7.5 < 8 (no rescale, e4m3
    # probabilities up to 2^7.5 ~ 181); target 11.0: every row's score passes the bound (>= 8.25)
    case, c = _near_bound_case(kv_dtype, target, 5)
    w = case.workload
    k = _decode_pool(case)[_prefix_slots(case)]
    u = _decode_q(case)[0, 0] / c[0, 0]
    s = k[:, 0, :] @ u / np.sqrt(w.head_dim) / LN2   # base-2 scores of the direction u (c = 1)
    assert np.all(s[:512] == 0.0)
    assert abs(s[700] - target) < 0.35, s[700]
    others = np.delete(s, 700)
    assert s[700] - others.max() > 1.0
    if target < 8:
        assert s[700] * c.max() < 8.0
    else:
        assert s[700] * c.min() > 8.0
    ref_o, ref_lse = oracle.attend_all(case)
    tol = TOL[kv_dtype]
    for num_sms in (0, 37):
        o, lse = run_case(case, threshold=1, num_sms=num_sms)
        assert np.isfinite(o).all() and np.isfinite(lse).all()
        assert max_err(o, ref_o) <= tol, (num_sms, max_err(o, ref_o))
        assert max_err(lse, ref_lse) <= tol, (num_sms, max_err(lse, ref_lse))
