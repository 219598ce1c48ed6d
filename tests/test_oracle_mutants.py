"""Planted mistakes in the oracle, each caught by a pin of test_oracle.py.

Every mutant edits ONE expression of the oracle's own source text (a dropped
term, a wrong sign, index or comparison, a transposed operand), compiles the
edited function beside the original and swaps it into the oracle module for
the duration of the check.  The pins named for the mutant then run against the
mutated oracle; at least one of them has to fail.  This is what makes the pins
a check of the oracle and not of themselves: a pin that passed for every
mutant would pin nothing.

All of it runs on the CPU; nothing here touches the CUDA library.
"""
import inspect
import textwrap

import pytest

from oracle import xattn_oracle as O
import test_oracle as P


def _each(fn, *cases):
    def run():
        for c in cases:
            fn(*c)
    return run


PINS = {
    "cu_seq_lens": P.test_cu_seq_lens_worked_example,
    "block_table": P.test_block_table_worked_example,
    "policy_arithmetic": P.test_bsa_policy_arithmetic,
    "ring": P.test_ring_buffer_arithmetic_and_schedule,
    "gather_history": P.test_gather_history_follows_block_table,
    "store_pool": P.test_store_chunk_builds_the_sequence_pool,
    "store_skip": P.test_store_chunk_skips_unallocated_pages,
    "scores_brute": _each(P.test_scores_bruteforce,
                          *[(m, S, lh, lq) for m in ("antidiag", "diag")
                            for S, lh, lq in ((2, 8, 8), (4, 16, 8), (3, 0, 9))]),
    "antidiagonal": P.test_antidiagonal_is_the_antidiagonal_of_the_token_product,
    "stride_one": P.test_stride_one_reduces_to_plain_scaled_qk,
    "stat_merge": _each(P.test_three_stage_merge_equals_one_shot, *[(s,) for s in range(4)]),
    "block_invariants": _each(P.test_block_sum_invariants, *[(s,) for s in range(3)]),
    "uniform_closed_form": P.test_block_sums_uniform_scores_closed_form,
    "sampled_qblocks": P.test_block_sums_of_sampled_query_blocks_match_full,
    "select_brute": _each(P.test_threshold_select_bruteforce, *[(s,) for s in range(40)]),
    "select_edges": P.test_threshold_select_edge_cases,
    "round_half_even": P.test_quantization_is_round_half_even,
    "vote": P.test_vote_hand_cases,
    "textbook": P.test_attention_textbook_loops,
    "single_key": P.test_single_key_attention,
    "split_merge": _each(P.test_split_kv_lse_merge_equals_unsplit, *[(s,) for s in range(3)]),
    "empty_merge": P.test_lse_merge_with_empty_parts,
    "chunk_textbook": P.test_chunk_attention_head_matches_textbook_loops,
    "estimate_request": P.test_estimate_request_reads_each_heads_group_through_the_pages,
    "attend_request": P.test_attend_request_sampled_rows_and_partial_selection,
    "tau_one": P.test_tau_one_is_full_causal_attention,
    "per_kv_select": P.test_per_kv_head_selection_hand_cases,
    "per_kv_union": _each(P.test_majority_vote_is_inside_the_union_of_per_kv_head_sets,
                          *[(s,) for s in range(6)]),
    "per_kv_attend": P.test_attention_with_pages_per_kv_head,
    "est_scale": P.test_default_estimation_scale_hand_values,
    "est_scale_bs": P.test_estimation_scale_decides_block_sums_and_selection,
    "sampled_brute": _each(P.test_sampled_estimation_bruteforce, (1,), (2,), (4,)),
    "sampled_reduce": P.test_sampled_estimation_reductions,
}

# (oracle function, exact source fragment, its mistaken replacement, pins that must catch it)
MUTANTS = [
    # indexing ([PAGED])
    ("cu_seq_lens", "out[-1] + int(n)", "int(n)", ["cu_seq_lens"]),
    ("request_index", "int(cu[r + 1] - cu[r])", "int(cu[r + 1])", ["cu_seq_lens"]),
    ("paged_location", "[t // page_size]", "[t % page_size]", ["block_table", "gather_history"]),
    ("paged_location", "return page, t % page_size", "return page, t // page_size",
     ["block_table", "gather_history"]),
    ("pages_after_append", "cache_len + 1 + page_size - 1", "cache_len + page_size - 1",
     ["block_table"]),
    ("gather_history", "pool[p, off, kvh]", "pool[p, off, 0]", ["gather_history", "tau_one"]),
    ("store_chunk", "kh_len + t,", "t,", ["store_pool", "store_skip"]),
    ("store_chunk", "out[p, off] = chunk_kv[:, t]", "out[p, off] = chunk_kv[:, 0]",
     ["store_pool", "store_skip"]),
    # estimation scores ([BSA] Steps 1-2)
    ("stride_reshape", "groups[:, ::-1, :]", "groups[:, :, ::-1]",
     ["scores_brute", "antidiagonal"]),
    ("estimation_scores", "Kr = stride_reshape(K, stride, reverse=False)",
     "Kr = stride_reshape(K, stride, reverse=True)", ["scores_brute", "antidiagonal"]),
    ("estimation_scores", "s = scale * (Qr @ Kr.T)", "s = Qr @ Kr.T",
     ["scores_brute", "stride_one"]),
    ("estimation_scores", "s[:, ch:][b > a] = NEG_INF", "s[:, ch:][b >= a] = NEG_INF",
     ["scores_brute", "stride_one"]),
    ("estimation_scores", "a = row0 + np.arange(rq)", "a = np.arange(rq)", ["sampled_qblocks"]),
    ("estimation_scores", "ch = k_hist.shape[0] // stride", "ch = k_hist.shape[0]",
     ["scores_brute", "stride_one"]),
    # softmax statistics and block sums ([SYNC] three stages)
    ("softmax_stats", "np.exp(s[fin] - m[fin, None])", "np.exp(s[fin])",
     ["stat_merge", "block_invariants"]),
    ("merge_stats", "ls[:, fin] * w[:, fin]", "ls[:, fin]", ["stat_merge"]),
    ("merge_stats", "m = np.max(ms, axis=0)", "m = np.min(ms, axis=0)", ["stat_merge"]),
    ("normalized_block_sums", "/ l[fin, None]", "", ["block_invariants", "uniform_closed_form"]),
    ("normalized_block_sums", ".sum(axis=(1, 3))", ".mean(axis=(1, 3))",
     ["block_invariants", "uniform_closed_form"]),
    ("block_sums_chunked", "s[:, a:b]", "s[:, a:b + 1]", ["stat_merge"]),
    ("block_sums_qblocks", "q[qb * block:(qb + 1) * block]", "q[qb * rb:(qb + 1) * rb * 2]",
     ["sampled_qblocks"]),
    # selection ([BSA] Steps 3-4)
    ("quantize_block_sums", "np.rint(", "np.floor(", ["round_half_even"]),
    ("threshold_select_row", "float(before) < R", "float(before) <= R",
     ["select_brute", "select_edges"]),
    ("threshold_select_row", "(-int(q[j]), j)", "(-int(q[j]), -j)",
     ["select_brute", "select_edges"]),
    ("threshold_select_row", "return q > 0", "return q >= 0", ["select_brute", "select_edges"]),
    ("threshold_select_row",
     "keep[j] = float(before) < R\n        before += int(q[j])",
     "before += int(q[j])\n        keep[j] = float(before) < R",
     ["select_brute", "select_edges"]),
    ("threshold_select_row", "R = float(tau) * float(total)", "R = float(total)",
     ["select_brute", "select_edges"]),
    ("gqa_vote", "per_kv = m.any(axis=1)", "per_kv = m.all(axis=1)", ["vote"]),
    ("gqa_vote", "count * den > num * num_kv_heads * qb",
     "count * den >= num * num_kv_heads * qb", ["vote"]),
    ("gqa_vote", "count = per_kv.sum(axis=(0, 1))", "count = m.sum(axis=(0, 1, 2))", ["vote"]),
    ("gqa_vote", "reshape(num_kv_heads, G, qb, kb_hist)", "reshape(G, num_kv_heads, qb, kb_hist)",
     ["vote"]),
    ("gqa_vote", "keep[0] = True", "keep[0] = keep[0]", ["vote"]),
    ("gqa_vote", "mask[:, :, :kb_hist]", "mask[:, :, -kb_hist:]", ["vote"]),
    ("select_request", "int(bt_row[j])", "int(j)", ["tau_one"]),
    ("per_kv_head_select", "mask[g * G:(g + 1) * G]", "mask[g::num_kv_heads]",
     ["per_kv_select", "per_kv_union"]),
    ("per_kv_head_select", "gqa_vote(mask[g * G:(g + 1) * G], 1,",
     "gqa_vote(mask[g * G:(g + 1) * G], G,", ["per_kv_select", "per_kv_union"]),
    ("density", "return selected / available", "return available / selected",
     ["policy_arithmetic"]),
    # attention and the merge ([BSA] compute_chunked_prefill)
    ("attention_with_lse", "logits = scale * (q @ k.T)", "logits = q @ k.T",
     ["textbook", "single_key"]),
    ("attention_with_lse", "lse[fin] = m[fin] + np.log(l)", "lse[fin] = np.log(l)",
     ["textbook", "single_key"]),
    ("attention_with_lse", "o[fin] = (p @ v) / l[:, None]", "o[fin] = p @ v",
     ["textbook", "split_merge"]),
    ("causal_visible", "np.arange(lk)[None, :] <= np.arange(lq)[:, None]",
     "np.arange(lk)[None, :] < np.arange(lq)[:, None]", ["chunk_textbook"]),
    ("causal_visible", "np.arange(lk)[None, :] <= np.arange(lq)[:, None]",
     "np.arange(lk)[:, None] <= np.arange(lq)[None, :]", ["chunk_textbook"]),
    ("lse_merge", "o2[fin] * w2[:, None]", "o2[fin] * w1[:, None]", ["split_merge"]),
    ("lse_merge", "lse[fin] = mx[fin] + np.log(s)", "lse[fin] = np.log(s)",
     ["split_merge", "empty_merge"]),
    ("lse_merge", "w1 = np.exp(lse1[fin] - lse[fin])", "w1 = np.exp(lse[fin] - lse1[fin])",
     ["split_merge", "empty_merge"]),
    ("bsa_chunk_attention_head", "np.ones((lq, k_sel.shape[0]), dtype=bool)",
     "np.zeros((lq, k_sel.shape[0]), dtype=bool)", ["chunk_textbook"]),
    ("estimate_request", "kvh = h // G", "kvh = h % Hkv", ["estimate_request"]),
    ("attend_request", "h = kvh * G + g", "h = g * Hkv + kvh", ["attend_request", "tau_one"]),
    ("attend_request", "np.arange(lq)[None, :] <= rows[:, None]",
     "np.arange(lq)[None, :] <= np.arange(len(rows))[:, None]", ["attend_request"]),
    ("attend_request", "np.arange(lq)[None, :] <= rows[:, None]",
     "np.arange(lq)[None, :] < rows[:, None]", ["attend_request", "tau_one"]),
    ("attend_request_per_kv", "pages_per_kv[g], G, 1,", "pages_per_kv[0], G, 1,",
     ["per_kv_attend"]),
    ("attend_request_per_kv", "pool_k[:, :, g:g + 1], pool_v[:, :, g:g + 1]",
     "pool_k[:, :, 0:1], pool_v[:, :, 0:1]", ["per_kv_attend"]),
    # the estimation scale reading (1/(sqrt(D) * S))
    ("default_estimation_scale", "math.sqrt(head_dim) * stride", "math.sqrt(head_dim)",
     ["est_scale", "est_scale_bs"]),
    ("default_estimation_scale", "math.sqrt(head_dim) * stride", "math.sqrt(head_dim * stride)",
     ["est_scale", "est_scale_bs"]),
    ("default_estimation_scale", "math.sqrt(head_dim) * stride", "head_dim * stride",
     ["est_scale", "est_scale_bs"]),
    # sampled estimation ([BSA] 性能分析, 优化方向 2)
    ("sampled_block_sums_one_head", "w = np.where(col < ch, rb / samples, 1.0)",
     "w = np.where(col < ch, 1.0, 1.0)", ["sampled_brute", "sampled_reduce"]),
    ("sampled_block_sums_one_head", "((col % rb) < samples)", "((col % rb) <= samples)",
     ["sampled_brute", "sampled_reduce"]),
    ("sampled_block_sums_one_head", "(col >= ch) |", "(col < 0) |",
     ["sampled_brute", "sampled_reduce"]),
    ("sampled_block_sums_one_head", "p[fin] /= l[fin, None]", "p[fin] /= p.shape[1]",
     ["sampled_brute", "sampled_reduce"]),
    # layer ring ([PLAN] Phases 1.1 and 4)
    ("ring_slot", "layer % num_buffers", "layer // num_buffers", ["ring"]),
    ("ring_schedule", "if l + num_buffers < num_layers", "if l + num_buffers <= num_layers",
     ["ring"]),
    ("ring_schedule", "(\"load\", l + num_buffers, ring_slot(l, num_buffers))",
     "(\"load\", l + num_buffers, ring_slot(l + 1, num_buffers))", ["ring"]),
    ("layer_slot_bytes", "* elem_bytes", "", ["ring"]),
]


def _mutant(name, old, new):
    src = textwrap.dedent(inspect.getsource(getattr(O, name)))
    assert src.count(old) == 1, f"{name}: fragment {old!r} is not unique in the source"
    ns = dict(vars(O))
    exec(compile(src.replace(old, new), f"<mutant of {name}>", "exec"), ns)
    return ns[name]


@pytest.mark.parametrize("name,old,new,pins", MUTANTS,
                         ids=[f"{m[0]}:{i}" for i, m in enumerate(MUTANTS)])
def test_planted_mistake_fails_a_pin(monkeypatch, name, old, new, pins):
    monkeypatch.setattr(O, name, _mutant(name, old, new))
    caught = []
    for pin in pins:
        try:
            PINS[pin]()
        except (NameError, TypeError, AttributeError, SyntaxError):
            raise                       # a broken mutant, not a caught one
        except Exception:               # an assertion, or an index the mistake ran past
            caught.append(pin)
    assert caught, f"no pin among {pins} fails when {name} has {old!r} -> {new!r}"


def test_unmutated_oracle_passes_every_listed_pin():
    """The harness itself: with no mistake planted, every pin passes, so a
    failure above comes from the mutant."""
    for pin in sorted({p for m in MUTANTS for p in m[3]}):
        PINS[pin]()
