"""Checks that pin the fp64 oracle to things other than itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with a library routine (torch decoders, torch SDPA in fp64),
a closed form, an invariance the pages state, or a worked example printed on
the pages.  ``tests/test_oracle_pins.py`` runs them on the real oracle;
``tests/test_oracle_mutations.py`` runs them on deliberately broken copies
and requires every copy to fail at least one pin.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# partition constants used by the pins (any valid set; the library reports its own)
PLAN_PARAMS = dict(num_sms=16, dense_threshold=1024, tile_tokens=64, split_min_tiles=2,
                   split_ctas_per_sm=2, prefix_rows_dense=128, prefix_rows_cascade=64,
                   prefix_min_tiles=2, prefix_ctas_per_sm=1)


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------ library decoders

def torch_decode(arr: np.ndarray, dtype: str, scale=None) -> torch.Tensor:
    """Decode stored values with torch's own dtype conversions (independent of the oracle)."""
    if dtype == "f32":
        t = torch.from_numpy(np.ascontiguousarray(arr)).double()
    elif dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).double()
    elif dtype == "fp8_e4m3":
        t = torch.from_numpy(np.ascontiguousarray(arr)).view(torch.float8_e4m3fn).double()
    else:
        raise ValueError(dtype)
    if scale is not None:
        t = t * torch.from_numpy(np.asarray(scale, np.float64)).reshape(-1, 1)
    return t


def sdpa_rows(case, b: int):
    """torch SDPA (fp64) over request b's contiguous logical K/V: O [Hq, d], LSE [Hq]."""
    w = case.workload
    rows = case.logical_rows[b]
    k = torch_decode(case.k_logical[rows], w.kv_dtype, case.k_scale)   # [L, Hkv, d]
    v = torch_decode(case.v_logical[rows], w.kv_dtype, case.v_scale)
    q = torch_decode(case.q[b], w.q_dtype)                              # [Hq, d]
    G = w.num_q_heads // w.num_kv_heads
    kr = k.permute(1, 0, 2).repeat_interleave(G, dim=0)                 # [Hq, L, d]
    vr = v.permute(1, 0, 2).repeat_interleave(G, dim=0)
    o = F.scaled_dot_product_attention(q[:, None, :], kr, vr)[:, 0, :]
    scores = torch.einsum("hd,hld->hl", q, kr) / math.sqrt(w.head_dim)
    lse = torch.logsumexp(scores, dim=-1)
    return o.numpy(), lse.numpy()


def _small_cases():
    return [
        workloads.make_case("tiny", 3, keep_logical=True),
        workloads.make_case("llama8b_noshare", 5, batch=2, private_range=(30, 160),
                            keep_logical=True),
        workloads.make_case("short_prefix", 7, batch=3, prefix_len=48, private_range=(1, 90),
                            keep_logical=True),
        workloads.make_case("fp8_large", 11, batch=2, prefix_len=32, private_range=(1, 70),
                            keep_logical=True),
    ]


# ---------------------------------------------------------------------- pins

def pin_fp8_decode_all_codes(orc):
    """Every e4m3 code against torch.float8_e4m3fn -> float64 (NaN codes stay NaN)."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch_decode(codes, "fp8_e4m3").numpy()
    got = np.array([orc.decode_fp8(int(c)) for c in codes])
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "fp8 NaN codes"
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok]), "fp8 decode"


def pin_bf16_decode_all_patterns(orc):
    """Every bf16 bit pattern against torch.bfloat16 -> float64."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch_decode(pats, "bf16").numpy()
    sample = np.concatenate([np.arange(0, 65536, 97), [0x0000, 0x8000, 0x0001, 0x7F80, 0xFF80,
                                                       0x7FC0, 0x3F80, 0xBF80, 0x007F, 0x0080]])
    got = np.array([orc.decode_bf16(int(p)) for p in sample])
    exp = ref[sample]
    assert np.array_equal(np.isnan(got), np.isnan(exp))
    ok = ~np.isnan(exp)
    assert np.array_equal(got[ok], exp[ok]), "bf16 decode"


def pin_sdpa_fp64(orc):
    """Oracle O and LSE equal torch SDPA (fp64) on contiguous K/V, GQA by repetition."""
    for case in _small_cases():
        o, lse = orc.attend_all(case)
        for b in range(case.batch):
            ro, rl = sdpa_rows(case, b)
            assert np.max(np.abs(o[b] - ro)) <= 1e-12, (case.workload.name, b, "O")
            assert np.max(np.abs(lse[b] - rl)) <= 1e-12, (case.workload.name, b, "LSE")


def pin_closed_forms(orc):
    """Q = 0 gives the mean of V and LSE = ln L; one token gives V_0; constant V gives it back;
    a dominant score selects its token's V."""
    base = workloads.make_case("tiny", 1, keep_logical=True)
    w = base.workload
    # Q = 0
    import dataclasses
    zq = dataclasses.replace(base, q=np.zeros_like(base.q))
    o, lse = orc.attend_all(zq)
    for b in range(base.batch):
        v = torch_decode(base.v_logical[base.logical_rows[b]], w.kv_dtype).numpy()  # [L, Hkv, d]
        G = w.num_q_heads // w.num_kv_heads
        for hq in range(w.num_q_heads):
            mean = v[:, hq // G, :].mean(axis=0)
            assert np.max(np.abs(o[b, hq] - mean)) <= 1e-12, "Q=0 mean"
            assert abs(lse[b, hq] - math.log(base.kv_len[b])) <= 1e-12, "Q=0 LSE"
    # one context token
    one = workloads.make_case("tiny", 2, prefix_len=0, private_lengths=[1, 1, 1, 1],
                              keep_logical=True)
    o, lse = orc.attend_all(one)
    G = w.num_q_heads // w.num_kv_heads
    for b in range(one.batch):
        v = torch_decode(one.v_logical[one.logical_rows[b]], "f32").numpy()[0]
        k = torch_decode(one.k_logical[one.logical_rows[b]], "f32").numpy()[0]
        qb = torch_decode(one.q[b], "f32").numpy()
        for hq in range(w.num_q_heads):
            assert np.array_equal(o[b, hq], v[hq // G]), "single token O"
            s = float(np.dot(qb[hq], k[hq // G])) / math.sqrt(w.head_dim)
            assert abs(lse[b, hq] - s) <= 1e-12, "single token LSE"
    # constant V
    vc = np.where(np.isnan(base.v_pool), base.v_pool, np.float32(0.375))
    cv = dataclasses.replace(base, v_pool=vc)
    o, _ = orc.attend_all(cv)
    assert np.max(np.abs(o - 0.375)) <= 1e-14, "constant V"
    # dominant score: key of one token made parallel to the query of head 0
    b, j = 1, 7
    kp = base.k_pool.copy().reshape(base.num_pages * base.page_size, w.num_kv_heads, w.head_dim)
    pages = base.page_indices[base.page_indptr[b]:base.page_indptr[b + 1]]
    slot = pages[j // base.page_size] * base.page_size + j % base.page_size
    kp[slot, 0, :] = 12.0 * base.q[b, 0, :]
    dom = dataclasses.replace(base, k_pool=kp.reshape(base.k_pool.shape))
    o, _ = orc.attend(dom, [b], [0])
    vp = base.v_pool.reshape(-1, w.num_kv_heads, w.head_dim)
    assert np.max(np.abs(o[0] - vp[slot, 0].astype(np.float64))) <= 1e-9, "dominant token"


def _permute_pool(case, seed: int):
    """Same logical step with the physical pages shuffled (remapped block tables)."""
    import dataclasses
    perm = np.random.default_rng(seed).permutation(case.num_pages)   # old id -> new id
    kp = np.empty_like(case.k_pool)
    vp = np.empty_like(case.v_pool)
    kp[perm] = case.k_pool
    vp[perm] = case.v_pool
    return dataclasses.replace(case, k_pool=kp, v_pool=vp,
                               page_indices=perm[case.page_indices].astype(np.int32))


def pin_paging_invariance(orc):
    """Page size (1, 16, 128), physical permutation and index layout leave O and LSE
    bit-for-bit unchanged (the runbook page: paging leaves results identical)."""
    outs = []
    for ps in (1, 16, 128):
        c = workloads.make_case("llama8b_noshare", 4, batch=3, private_range=(60, 330),
                                page_size=ps)
        outs.append(orc.attend_all(c))
        p = _permute_pool(c, 99)
        op = orc.attend_all(p)
        assert np.array_equal(op[0], outs[-1][0]) and np.array_equal(op[1], outs[-1][1]), \
            f"permutation at ps={ps}"
    for o, l in outs[1:]:
        assert np.array_equal(o, outs[0][0]) and np.array_equal(l, outs[0][1]), "page size"
    for layout in ("contiguous", "block128"):
        c = workloads.make_case("llama8b_noshare", 4, batch=3, private_range=(60, 330),
                                page_size=16, layout=layout)
        o, l = orc.attend_all(c)
        assert np.array_equal(o, outs[0][0]) and np.array_equal(l, outs[0][1]), layout
    # shared prefix: reading the prefix through every block table is the same tokens
    c = workloads.make_case("agent", 2, batch=3, prefix_len=80, private_range=(5, 70),
                            num_q_heads=8, num_kv_heads=2)
    a = orc.attend_all(c)
    n = orc.attend_all(c.without_sharing())
    assert np.array_equal(a[0], n[0]) and np.array_equal(a[1], n[1]), "sharing"


def pin_merge_identity(orc):
    """Prefix-part and suffix-part results merged by log-sum-exp equal full attention;
    an empty part is the identity of the merge."""
    for case in (workloads.make_case("tiny", 5),
                 workloads.make_case("fp8_large", 3, batch=2, prefix_len=48,
                                     private_range=(1, 60))):
        w = case.workload
        B, Hq = case.batch, w.num_q_heads
        bb, hh = np.meshgrid(np.arange(B), np.arange(Hq), indexing="ij")
        bb, hh = bb.reshape(-1), hh.reshape(-1)
        L = case.kv_len[bb]
        cut = np.minimum(L, (w.prefix_len // case.page_size) * case.page_size)
        full = orc.attend(case, bb, hh)
        pre = orc.attend(case, bb, hh, np.zeros_like(cut), cut)
        suf = orc.attend(case, bb, hh, cut, L)
        o, lse = orc.merge(pre[0], pre[1], suf[0], suf[1])
        assert np.max(np.abs(o - full[0])) <= 1e-12, "merge O"
        assert np.max(np.abs(lse - full[1])) <= 1e-12, "merge LSE"
        # split elsewhere too: first third / rest
        third = L // 3
        a = orc.attend(case, bb, hh, np.zeros_like(third), third)
        r = orc.attend(case, bb, hh, third, L)
        o, lse = orc.merge(a[0], a[1], r[0], r[1])
        assert np.max(np.abs(o - full[0])) <= 1e-12 and np.max(np.abs(lse - full[1])) <= 1e-12
        empty = orc.attend(case, bb, hh, np.zeros_like(L), np.zeros_like(L))
        assert np.all(empty[1] == -np.inf) and np.all(empty[0] == 0.0)
        o, lse = orc.merge(empty[0], empty[1], full[0], full[1])
        assert np.array_equal(o, full[0]) and np.array_equal(lse, full[1]), "empty part"


def pin_kv_indices(orc):
    """Hand-written example; length = sum of context lengths at every page size; the
    indices of a no-sharing step are exactly the non-poisoned pool slots, once each."""
    g = golden("kv_indices_hand.json")

    class T:
        pass
    t = T()
    t.kv_len = np.array(g["kv_len"], np.int32)
    t.page_indptr = np.array(g["page_indptr"], np.int32)
    t.page_indices = np.array(g["page_indices"], np.int32)
    t.page_size = g["page_size"]
    t.num_pages = g["num_pages"]
    ip, idx = orc.expand_kv_indices(t)
    assert ip.tolist() == g["kv_indptr"] and idx.tolist() == g["kv_indices"], "hand example"
    for ps in (1, 16, 128):
        c = workloads.make_case("llama8b_noshare", 6, batch=3, private_range=(1, 300),
                                page_size=ps, num_q_heads=4, num_kv_heads=2, head_dim=16)
        ip, idx = orc.expand_kv_indices(c)
        assert ip[-1] == int(c.kv_len.sum()) == idx.shape[0], "length B x L"
        assert np.unique(idx).shape[0] == idx.shape[0], "distinct slots"
        first = torch_decode(c.k_pool.reshape(-1, 2 * 16)[:, 0].copy(), c.workload.kv_dtype)
        live = np.flatnonzero(~np.isnan(first.numpy()))
        assert np.array_equal(np.sort(idx), live), "indices = stored slots"


def pin_block_aligned_prefix(orc):
    """2,003-token prefix at block 16: 125 shared blocks, 3 tokens private; waste < block."""
    g = golden("block_aligned_prefix.json")
    ps = g["page_size"]
    c = workloads.make_case("agent", 8, batch=3, prefix_len=g["prefix_tokens"],
                            private_range=(1, 40), page_size=ps, num_q_heads=4,
                            num_kv_heads=2, head_dim=16)
    p = orc.plan(c, PLAN_PARAMS)
    assert p["group_page_indptr"][1] == g["shared_pages"], "shared blocks"
    assert p["group_shared_len"][0] == g["shared_pages"] * ps
    for b in range(c.batch):
        assert p["suffix_start"][b] == g["shared_pages"] * ps
        assert p["suffix_len"][b] == c.kv_len[b] - g["shared_pages"] * ps
        priv = p["suffix_len"][b] - (c.kv_len[b] - g["prefix_tokens"])
        assert priv == g["unshared_prefix_tokens"], "unshared prefix tokens"
        pages = c.page_indptr[b + 1] - c.page_indptr[b]
        assert 0 <= pages * ps - c.kv_len[b] <= g["max_internal_waste_tokens"], "waste"


def pin_dispatcher(orc):
    """M_eff = members x GQA group; M_eff >= threshold selects the dense branch."""
    g = golden("dispatcher.json")
    for cs in g["cases"]:
        c = workloads.make_case("agent", 0, batch=cs["batch"], prefix_len=64,
                                private_range=(1, 3), num_q_heads=cs["num_q_heads"],
                                num_kv_heads=cs["num_kv_heads"], head_dim=8)
        p = orc.plan(c, dict(PLAN_PARAMS, dense_threshold=g["threshold_a100"]))
        assert p["group_m_eff"][0] == cs["m_eff"]
        want = {"dense": 2, "cascade": 1}[cs["branch"]]
        assert p["group_branch"][0] == want


def pin_paged_branch(orc):
    """A prefix too short, or saving too few bytes, to be read once is planned as not shared:
    every per-request array equals the plan of the same batch without the group and the group
    shares nothing.  Hand-computed boundaries of the read-once test ((members - 1) x shared
    tokens x bytes per token against the minimum; 4096 bytes per token here: 8 KV heads x
    d = 128 x 2 bytes x K and V): at either minimum exactly the prefix is read once."""
    arrays = ("suffix_start", "suffix_len", "suffix_page_indptr", "suffix_page_indices", "split_indptr",
              "split_begin", "split_end")
    base = dict(PLAN_PARAMS, dense_threshold=1)
    c = workloads.make_case("agent", 4, batch=40, prefix_len=1024, tables_only=True)
    assert c.kv_token_bytes() == 4096
    alone = orc.plan(c.without_sharing(), base)
    paged = orc.plan(c, dict(base, read_once_min_tokens=1025))
    assert paged["group_branch"][0] == 3 and paged["group_shared_len"][0] == 0
    assert len(paged["chunk_begin"]) == 0
    for f in arrays:
        assert np.array_equal(paged[f], alone[f]), f
    once = orc.plan(c, dict(base, read_once_min_tokens=1024))
    assert once["group_branch"][0] == 2 and once["group_shared_len"][0] == 1024
    assert np.all(once["suffix_start"] == 1024)
    # 257 members x 64 shared tokens: 256 x 64 x 4096 B = 64 MiB saved, exactly the minimum
    c = workloads.make_case("agent", 4, batch=257, prefix_len=64, private_range=(1, 20), tables_only=True)
    assert orc.plan(c, dict(base, read_once_min_mib=64))["group_branch"][0] == 2
    assert orc.plan(c, dict(base, read_once_min_mib=65))["group_branch"][0] == 3
    # 2 members x 8192 tokens: the one other member's re-read, 8192 x 4096 B = 32 MiB, is saved
    c = workloads.make_case("agent", 4, batch=2, prefix_len=8192, private_range=(1, 20), tables_only=True)
    assert orc.plan(c, dict(base, read_once_min_mib=32))["group_branch"][0] == 2
    assert orc.plan(c, dict(base, read_once_min_mib=33))["group_branch"][0] == 3


def pin_partition(orc):
    """Splits tile each suffix exactly, in order, in equal tile-aligned chunks except the
    last; prefix chunks tile the shared prefix; the partition is the same at every page
    size (it is defined in tokens)."""
    ref = None
    for ps in (1, 16, 128):
        c = workloads.make_case("llama8b_noshare", 9, batch=5, private_range=(1, 900),
                                page_size=ps, num_q_heads=4, num_kv_heads=2, head_dim=16)
        p = orc.plan(c, PLAN_PARAMS)
        tile = PLAN_PARAMS["tile_tokens"]
        lens = set()
        for b in range(c.batch):
            s0, s1 = p["split_indptr"][b], p["split_indptr"][b + 1]
            beg, end = p["split_begin"][s0:s1], p["split_end"][s0:s1]
            S = p["suffix_len"][b]
            assert S == c.kv_len[b] and p["suffix_start"][b] == 0
            assert beg[0] == 0 and end[-1] == S and np.all(beg[1:] == end[:-1]) and np.all(end > beg)
            assert np.all(beg % tile == 0)
            lens.update((end[:-1] - beg[:-1]).tolist())
            assert np.all(end - beg <= (end[0] - beg[0]) if s1 - s0 > 1 else True)
        assert len(lens) <= 1, "equal chunks"
        key = (p["split_indptr"].tolist(), p["split_begin"].tolist(), p["split_end"].tolist())
        ref = ref or key
        assert key == ref, "partition depends on page size"
    c = workloads.make_case("agent", 4, batch=6, prefix_len=1000, private_range=(1, 50),
                            num_q_heads=8, num_kv_heads=2, head_dim=16)
    p = orc.plan(c, dict(PLAN_PARAMS, dense_threshold=8))
    c0, c1 = p["group_chunk_indptr"][0], p["group_chunk_indptr"][1]
    beg, end = p["chunk_begin"][c0:c1], p["chunk_end"][c0:c1]
    assert beg[0] == 0 and end[-1] == p["group_shared_len"][0] == 992
    assert np.all(beg[1:] == end[:-1]) and np.all(end > beg)
    assert p["group_row_blocks"][0] == -(-p["group_m_eff"][0] // PLAN_PARAMS["prefix_rows_dense"])


def pin_validation(orc):
    """Invalid block tables and groups are rejected, never coerced."""
    import dataclasses
    from oracle import OracleError
    c = workloads.make_case("agent", 1, batch=3, prefix_len=64, private_range=(1, 40),
                            num_q_heads=4, num_kv_heads=2, head_dim=16)

    def rejects(case, code):
        try:
            orc.plan(case, PLAN_PARAMS)
        except OracleError as e:
            assert e.code == code, (e.code, code)
            return
        raise AssertionError(f"accepted an invalid step (expected {code})")

    bad = c.page_indices.copy()
    bad[-1] = c.num_pages
    rejects(dataclasses.replace(c, page_indices=bad), -3)
    kl = c.kv_len.copy()
    kl[0] += 16
    rejects(dataclasses.replace(c, kv_len=kl), -4)
    bad = c.page_indices.copy()
    b1 = c.page_indptr[1]
    bad[b1], bad[-1] = bad[-1], bad[b1]     # member 1 no longer shares page 0
    rejects(dataclasses.replace(c, page_indices=bad), -5)
    pg = c.prefix_group.copy()
    pg[0] = 3
    rejects(dataclasses.replace(c, prefix_group=pg), -1)
    gl = np.array([int(c.kv_len.min()) + 1], np.int32)
    rejects(dataclasses.replace(c, group_prefix_len=gl), -5)


def _three_level_tables(num_q_heads=4, num_kv_heads=2, head_dim=16):
    """Hand-built block tables of a three-level tree at page size 16 (ids fixed here, nothing
    generated): group 0 = 64 tokens (4 pages) shared by all six requests, group 1 = 256 tokens
    under it for requests 2-5, group 2 = 328 tokens under group 1 for requests 4 and 5 (20 full
    pages, 8 tokens private), and group 3 = 96 tokens under group 0 for request 1 alone."""
    import dataclasses
    ps = 16
    root = [40, 41, 42, 43]
    mid = root + list(range(50, 62))
    leaf = mid + [62, 63, 64, 65]
    side = root + [70, 71]
    tables = [root + [1, 2], side + [3, 4], mid + [5], mid + [6, 7], leaf + [80, 8, 9], leaf + [81, 10]]
    kv_len = np.array([64 + 20, 96 + 30, 256 + 16, 256 + 17, 328 + 28, 328 + 9], np.int32)
    for b, t in enumerate(tables):
        assert len(t) == -(-int(kv_len[b]) // ps)
    base = workloads.make_case("agent", 0, batch=6, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                               head_dim=head_dim, tables_only=True)
    return dataclasses.replace(
        base, page_size=ps, num_pages=100, kv_len=kv_len,
        page_indptr=np.concatenate([[0], np.cumsum([len(t) for t in tables])]).astype(np.int32),
        page_indices=np.concatenate(tables).astype(np.int32),
        prefix_group=np.array([0, 3, 1, 1, 2, 2], np.int32),
        group_prefix_len=np.array([64, 256, 328, 96], np.int32),
        group_parent=np.array([-1, 0, 1, 0], np.int32))


def _covered_once(p, b, kv_len):
    """Token coverage of request b by its levels' prefix chunks and its suffix splits."""
    cover = np.zeros(int(kv_len), np.int64)
    for l in range(p["req_level_indptr"][b], p["req_level_indptr"][b + 1]):
        g = p["req_level_group"][l]
        for c in range(p["group_chunk_indptr"][g], p["group_chunk_indptr"][g + 1]):
            cover[p["chunk_begin"][c]:p["chunk_end"][c]] += 1
    s0 = p["suffix_start"][b]
    for s in range(p["split_indptr"][b], p["split_indptr"][b + 1]):
        cover[s0 + p["split_begin"][s]:s0 + p["split_end"][s]] += 1
    return cover


def pin_nested_prefix(orc):
    """Nested groups (a tree of shared beginnings, each level read once for every request
    below it): the members of a group are its own requests and its descendants' (M_eff
    counted by hand), each request merges the read-once levels on its path from the root in
    order, every context token is covered exactly once by those levels' chunks and the
    request's splits, the merged parts equal full attention (and torch SDPA on contiguous
    K/V), a level below a paged level is paged, and bad trees are rejected."""
    import dataclasses
    from oracle import OracleError
    params = dict(PLAN_PARAMS, dense_threshold=8, read_once_min_tokens=-1, read_once_min_mib=-1)
    t = _three_level_tables()
    p = orc.plan(t, params)
    assert list(p["group_m_eff"]) == [12, 8, 4, 2], "members counted through descendants (G = 2)"
    assert list(p["group_branch"]) == [2, 2, 1, 1]
    assert list(p["group_shared_len"]) == [64, 192, 64, 32], "own segments only"
    assert list(p["suffix_start"]) == [64, 96, 256, 256, 320, 320]
    assert p["req_level_indptr"].tolist() == [0, 1, 3, 5, 7, 10, 13]
    assert p["req_level_group"].tolist() == [0, 0, 3, 0, 1, 0, 1, 0, 1, 2, 0, 1, 2]
    g2 = p["group_page_indices"][p["group_page_indptr"][2]:p["group_page_indptr"][3]]
    assert g2.tolist() == [40, 41, 42, 43] + list(range(50, 66)), "whole prefix, root first"
    for b in range(t.batch):
        assert np.all(_covered_once(p, b, t.kv_len[b]) == 1), b
    # a short root segment (64 tokens) under a 100-token minimum: the root is paged and so is
    # every level below it, the 192-token segment of group 1 too; the plan is then the plan
    # without sharing
    paged = orc.plan(t, dict(params, read_once_min_tokens=100))
    alone = orc.plan(t.without_sharing(), dict(params, read_once_min_tokens=100))
    assert list(paged["group_branch"]) == [3, 3, 3, 3]
    for f in ("suffix_start", "suffix_len", "split_indptr", "split_begin", "split_end"):
        assert np.array_equal(paged[f], alone[f]), f
    # a 40-token minimum: the 32-token side segment (group 3) alone is paged
    part = orc.plan(t, dict(params, read_once_min_tokens=40))
    assert list(part["group_branch"]) == [2, 2, 1, 3] and part["suffix_start"][1] == 64

    # values: the generator's two-level tree, parts merged in plan order = full attention
    for kv in ("bf16", "fp8_e4m3"):
        c = workloads.make_case("agent", 11, batch=7, prefix_len=100, private_range=(1, 90), page_size=16,
                                num_q_heads=4, num_kv_heads=2, head_dim=16, kv_dtype=kv, nested=(3, 70),
                                keep_logical=True)
        p = orc.plan(c, dict(params, tile_tokens=16, prefix_min_tiles=1, split_min_tiles=1))
        assert p["group_m_eff"].tolist() == [14] + [2 * int(np.sum(c.prefix_group == k)) for k in (1, 2, 3)]
        for b in range(c.batch):
            assert np.all(_covered_once(p, b, c.kv_len[b]) == 1), b
            hh = np.arange(4)
            bb = np.full(4, b)
            ranges = []
            for l in range(p["req_level_indptr"][b], p["req_level_indptr"][b + 1]):
                g = p["req_level_group"][l]
                ranges += [(p["chunk_begin"][k], p["chunk_end"][k])
                           for k in range(p["group_chunk_indptr"][g], p["group_chunk_indptr"][g + 1])]
            s0 = p["suffix_start"][b]
            ranges += [(s0 + p["split_begin"][s], s0 + p["split_end"][s])
                       for s in range(p["split_indptr"][b], p["split_indptr"][b + 1])]
            o, lse = orc.attend(c, bb, hh, np.full(4, ranges[0][0]), np.full(4, ranges[0][1]))
            for lo, hi in ranges[1:]:
                po, pl = orc.attend(c, bb, hh, np.full(4, lo), np.full(4, hi))
                o, lse = orc.merge(o, lse, po, pl)
            full = orc.attend(c, bb, hh)
            assert np.max(np.abs(o - full[0])) <= 1e-12 and np.max(np.abs(lse - full[1])) <= 1e-12
            so, sl = sdpa_rows(c, b)
            assert np.max(np.abs(full[0] - so)) <= 1e-12 and np.max(np.abs(full[1] - sl)) <= 1e-12

    # random trees (up to six groups, zero-length segments, requests outside any group): every
    # token covered once, a member's levels are the read-once groups on its path in order, and
    # full attention over the paged layout equals torch SDPA on the contiguous logical rows
    for seed in range(4):
        spec = workloads.random_tree_spec(seed)
        c = workloads.make_tree_case("agent", seed, page_size=16, num_q_heads=4, num_kv_heads=2, head_dim=16,
                                     **spec)
        p = orc.plan(c, dict(params, tile_tokens=16, prefix_min_tiles=1, split_min_tiles=1))
        for b in range(c.batch):
            assert np.all(_covered_once(p, b, c.kv_len[b]) == 1), (seed, b)
            path, g = [], int(c.prefix_group[b])
            while g >= 0:
                path.insert(0, g)
                g = int(c.group_parent[g])
            levels = p["req_level_group"][p["req_level_indptr"][b]:p["req_level_indptr"][b + 1]].tolist()
            assert levels == [a for a in path if p["group_branch"][a] in (1, 2)], (seed, b)
        full = orc.attend_all(c)
        for b in range(c.batch):
            so, sl = sdpa_rows(c, b)
            assert np.max(np.abs(full[0][b] - so)) <= 1e-12 and np.max(np.abs(full[1][b] - sl)) <= 1e-12

    def rejects(case, code):
        try:
            orc.plan(case, params)
        except OracleError as e:
            assert e.code == code, (e.code, code)
            return
        raise AssertionError(f"accepted an invalid tree (expected {code})")

    rejects(dataclasses.replace(t, group_parent=np.array([-1, 0, 3, 0], np.int32)), -1)   # parent after child
    rejects(dataclasses.replace(t, group_parent=np.array([-1, 1, 1, 0], np.int32)), -1)   # own parent
    rejects(dataclasses.replace(t, group_prefix_len=np.array([64, 128, 120, 96], np.int32)), -1)  # shorter than parent
    bad = t.page_indices.copy()
    bad[t.page_indptr[5] + 5] = 99          # request 5 leaves group 1's segment
    rejects(dataclasses.replace(t, page_indices=bad), -5)
    bad = t.page_indices.copy()
    bad[t.page_indptr[1] + 2] = 98          # request 1 leaves the root's pages
    rejects(dataclasses.replace(t, page_indices=bad), -5)
    bad = t.page_indices.copy()
    bad[t.page_indptr[4] + 17] = 97         # request 4 leaves group 2's own segment
    rejects(dataclasses.replace(t, page_indices=bad), -5)


ALL_PINS = [pin_paged_branch, pin_fp8_decode_all_codes, pin_bf16_decode_all_patterns, pin_sdpa_fp64,
            pin_closed_forms, pin_paging_invariance, pin_merge_identity, pin_kv_indices,
            pin_block_aligned_prefix, pin_dispatcher, pin_partition, pin_validation, pin_nested_prefix]
