"""Plants plausible mistakes in copies of the oracle (on the CPU) and requires the pin
battery to catch every one of them."""
import os
import shutil

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, original text, planted mistake)
MUTATIONS = [
    ("gqa_head_map", "h = hq / G;", "h = hq % Hkv;"),
    ("drop_softmax_scale", "s[j] = acc * inv_sqrt_d;", "s[j] = acc;"),
    ("slot_offset", "return (int64_t)page * ps + t % ps;", "return (int64_t)page * ps + (t + 1) % ps;"),
    ("fp8_k_scale_dropped", "acc += qv[i] * (elem(k_pool, base + i, kv_dtype) * ks);",
     "acc += qv[i] * elem(k_pool, base + i, kv_dtype);"),
    ("lse_without_log_l", "lse_out[r] = m + log(l);", "lse_out[r] = m;"),
    ("fp8_subnormal_exponent", "ldexp((double)mantissa / 8.0, 1 - 7)", "ldexp((double)mantissa / 8.0, -7)"),
    ("bf16_shift", "((uint32_t)bits) << 16;", "((uint32_t)bits) << 15;"),
    ("merge_weight_swapped", "w2 * o2[(int64_t)r * d + i];", "w1 * o2[(int64_t)r * d + i];"),
    ("prefix_pages_rounded_up", "n_sh = group_prefix_len[a] / ps;", "n_sh = (group_prefix_len[a] + ps - 1) / ps;"),
    ("paged_saving_counts_every_member", "int64_t saved = (int64_t)(members[g] - 1) * shared * pp->token_bytes;",
     "int64_t saved = (int64_t)members[g] * shared * pp->token_bytes;"),
    ("paged_minimum_tokens_inclusive", "shared < pp->read_once_min_tokens;", "shared <= pp->read_once_min_tokens;"),
    ("paged_members_keep_their_prefix",
     "if (leaf < 0 || !member_of(group_parent, leaf, a) || !read_once(out->group_branch[a])) continue;",
     "if (leaf < 0 || !member_of(group_parent, leaf, a) || out->group_branch[a] == OR_BRANCH_NONE) continue;"),
    ("nested_segment_start_dropped", "out->chunk_begin[nc] = (int32_t)(seg0 + lo);", "out->chunk_begin[nc] = (int32_t)(lo);"),
    ("nested_members_only_direct", "if (leaf < 0 || !member_of(group_parent, leaf, g)) continue;",
     "if (leaf != g) continue;"),
    ("nested_paged_not_inherited", "if (below_paged || too_short || too_little)", "if (too_short || too_little)"),
    ("nested_no_grandparents", "for (int g = leaf; g >= 0; g = parent_of(group_parent, g))",
     "for (int g = leaf; g >= 0; g = (g == leaf) ? parent_of(group_parent, g) : -1)"),
    ("nested_segment_counts_whole_prefix",
     "shared_pages(group_prefix_len, g, ps) - shared_pages(group_prefix_len, par, ps) : 0;",
     "shared_pages(group_prefix_len, g, ps) : 0;"),
    ("nested_shared_len_whole_prefix", "out->group_shared_len[g] = (int32_t)(n_sh * ps - seg0);",
     "out->group_shared_len[g] = (int32_t)(n_sh * ps);"),
    ("v_from_k_pool", "out[i] += w * (elem(v_pool, base + i, kv_dtype) * vs);",
     "out[i] += w * (elem(k_pool, base + i, kv_dtype) * vs);"),
    ("q_row_transposed", "qv[i] = elem(q, ((int64_t)b * Hq + hq) * d + i, q_dtype);",
     "qv[i] = elem(q, ((int64_t)hq * 1 + b) * d + i, q_dtype);"),
    ("m_eff_without_group", "int64_t m_eff = (int64_t)members[g] * G;", "int64_t m_eff = (int64_t)members[g];"),
    ("threshold_strict", "(m_eff >= pp->dense_threshold)", "(m_eff > pp->dense_threshold)"),
    ("split_off_by_one", "out->split_end[ns] = (int32_t)(hi < S ? hi : S);",
     "out->split_end[ns] = (int32_t)(hi < S ? hi - 1 : S);"),
    ("page_range_unchecked", "if (page_indices[i] < 0 || page_indices[i] >= num_pages) return OR_ERANGE;",
     "if (page_indices[i] < 0) return OR_ERANGE;"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(name, old, new, tmp_path):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
    src = tmp_path / "oracle_mut.c"
    src.write_text(text.replace(old, new))
    lib = oracle.build(force=True, src=str(src), out=str(tmp_path / "liboracle_mut.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
        except Exception as e:  # a crash-free error path also counts as detection
            caught.append(f"{pin.__name__}:{type(e).__name__}")
    assert caught, f"no pin caught mutation {name}"
