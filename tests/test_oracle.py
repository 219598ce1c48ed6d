"""Pins of the float64 oracle against what the pages and the mathematics fix.

None of these re-types an oracle formula: each checks a worked example printed
on the pages, a closed form, an invariant, a special case that reduces to a
textbook routine, or brute force over explicit loops on tiny inputs.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import xattn_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Worked examples printed on the pages
# ---------------------------------------------------------------------------


def test_cu_seq_lens_worked_example():
    g = _golden("paged_attention_examples.json")["varlen"]
    cu_q = O.cu_seq_lens(g["q_lens"])
    cu_k = O.cu_seq_lens(g["k_lens"])
    assert cu_q.tolist() == g["cu_seq_lens_q"]
    assert cu_k.tolist() == g["cu_seq_lens_k"]
    assert max(g["q_lens"]) == g["max_length_q"]
    assert max(g["k_lens"]) == g["max_length_k"]
    assert O.request_index(cu_q) == g["q_request_index"]
    assert O.request_index(cu_k) == g["k_request_index"]
    assert cu_q[-1] == g["q_shape_tokens"] and cu_k[-1] == g["k_shape_tokens"]


def test_block_table_worked_example():
    g = _golden("paged_attention_examples.json")["decode"]
    bt = g["block_table"]
    ps = g["page_size"]
    for s, n in enumerate(g["cache_seqlens"]):
        # the rows hold the pages of the cached tokens plus the appended one
        pages = sorted({O.paged_location(bt, s, t, ps)[0] for t in range(n + 1)},
                       key=lambda p: bt[s].index(p))
        assert pages == g["cache_pages_of_seq"][s]
        assert O.pages_after_append(n, ps) == g["pages_after_append"][s]
    # token 69 of sequence 2 sits at offset 5 of its third page (physical 6)
    assert O.paged_location(bt, 2, 69, ps) == (6, 5)
    assert O.paged_location(bt, 1, 31, ps) == (0, 31)
    assert O.paged_location(bt, 1, 32, ps) == (1, 0)
    with pytest.raises(IndexError):
        O.paged_location(bt, 0, 32, ps)          # -1: unallocated page


def test_bsa_policy_arithmetic():
    g = _golden("bsa_policy_arithmetic.json")
    r = g["reshaped_block_size"]
    assert r["block_size"] // r["stride"] == r["expected"]
    d = g["density_stats"]
    dens = O.density(d["total_selected_blocks"], d["total_available_blocks"])
    assert round(dens, 2) == d["overall_density_2dp"]
    lg = g["debug_log"]
    assert round(100 * O.density(lg["selected"], lg["available"]), 1) == lg["chunk_density_pct_1dp"]
    assert g["cli_threshold"]["flag"] / 10 == g["cli_threshold"]["value"]


def test_ring_buffer_arithmetic_and_schedule():
    g = _golden("layerwise_ring_arithmetic.json")
    b = O.layer_slot_bytes(g["max_tokens"], g["kv_heads"], g["head_dim"], g["elem_bytes"])
    assert b == g["slot_mib"] * 2 ** 20
    assert g["num_kv_buffers"] * b == g["ring_gib"] * 2 ** 30
    assert g["all_layers"] * b == g["all_layers_mib"] * 2 ** 20
    ev = O.ring_schedule(8, g["num_kv_buffers"])
    comp = [s for kind, l, s in ev if kind == "compute"]
    assert comp == g["schedule_4_buffers_8_layers_compute_slots"]
    # every layer is loaded exactly once, before it is computed, and a slot is
    # reloaded only after the layer that used it has been computed
    loaded, slot_owner, done = {}, {}, set()
    for kind, l, s in ev:
        if kind == "load":
            assert l not in loaded
            prev = slot_owner.get(s)
            assert prev is None or prev in done
            loaded[l] = s
            slot_owner[s] = l
        else:
            assert loaded[l] == s and slot_owner[s] == l
            done.add(l)
    assert len(done) == 8
    assert sorted(loaded) == list(range(8))   # no load of a layer that does not exist


# ---------------------------------------------------------------------------
# Stride-reshaped scores: brute force and special cases
# ---------------------------------------------------------------------------


def _brute_scores(q, kh, kc, S, scale, mode):
    """Explicit loops over (a, b, i, d); masked cells are None."""
    K = np.concatenate([kh, kc], axis=0)
    rq, c, ch = q.shape[0] // S, K.shape[0] // S, kh.shape[0] // S
    out = [[None] * c for _ in range(rq)]
    for a in range(rq):
        for b in range(c):
            if b >= ch and (b - ch) > a:
                continue
            acc = 0.0
            for i in range(S):
                qi = S * a + (S - 1 - i if mode == "antidiag" else i)
                for d in range(q.shape[1]):
                    acc += q[qi, d] * K[S * b + i, d]
            out[a][b] = acc * scale
    return out


@pytest.mark.parametrize("mode", ["antidiag", "diag"])
@pytest.mark.parametrize("S,lh,lq", [(2, 8, 8), (4, 16, 8), (3, 0, 9)])
def test_scores_bruteforce(mode, S, lh, lq):
    rng = np.random.default_rng(7 + S + lh)
    D = 3
    q = rng.standard_normal((lq, D))
    kh = rng.standard_normal((lh, D))
    kc = rng.standard_normal((lq, D))
    s = O.estimation_scores(q, kh, kc, S, 0.37, mode)
    ref = _brute_scores(q, kh, kc, S, 0.37, mode)
    for a in range(s.shape[0]):
        for b in range(s.shape[1]):
            if ref[a][b] is None:
                assert s[a, b] == -np.inf
            else:
                assert abs(s[a, b] - ref[a][b]) < 1e-12


def test_antidiagonal_is_the_antidiagonal_of_the_token_product():
    """Each reshaped score is the trace of the left-right flipped S x S block of
    the token-level product Q K^T (its anti-diagonal), not its diagonal."""
    rng = np.random.default_rng(3)
    S, D, L = 4, 5, 16
    q = rng.standard_normal((L, D))
    k = rng.standard_normal((L, D))
    s = O.estimation_scores(q, k[:0], k, S, 1.0, "antidiag")
    full = q @ k.T
    for a in range(L // S):
        for b in range(a + 1):
            blk = full[S * a:S * a + S, S * b:S * b + S]
            assert abs(s[a, b] - np.trace(np.fliplr(blk))) < 1e-12
            assert abs(s[a, b] - np.trace(blk)) > 1e-9 or a == b == 0


def test_stride_one_reduces_to_plain_scaled_qk():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((6, 4))
    kh = rng.standard_normal((4, 4))
    kc = rng.standard_normal((6, 4))
    s = O.estimation_scores(q, kh, kc, 1, 0.5)
    ref = 0.5 * q @ np.concatenate([kh, kc]).T
    ref[:, 4:][np.triu(np.ones((6, 6), dtype=bool), 1)] = -np.inf
    assert np.array_equal(np.isinf(s), np.isinf(ref))
    assert np.allclose(s[np.isfinite(s)], ref[np.isfinite(ref)], atol=1e-13)


# ---------------------------------------------------------------------------
# Softmax statistics and block sums
# ---------------------------------------------------------------------------


def _rand_problem(seed, lh=32, lq=16, D=4, S=4, block=8):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((lq, D)) * 2, rng.standard_normal((lh, D)),
            rng.standard_normal((lq, D)), S, block)


@pytest.mark.parametrize("seed", range(4))
def test_three_stage_merge_equals_one_shot(seed):
    q, kh, kc, S, block = _rand_problem(seed)
    s = O.estimation_scores(q, kh, kc, S, 0.3)
    m1, l1 = O.softmax_stats(s)
    rng = np.random.default_rng(100 + seed)
    c = s.shape[1]
    cuts = sorted(rng.choice(np.arange(1, c), size=3, replace=False).tolist())
    edges = [0] + cuts + [c]
    chunks = list(zip(edges[:-1], edges[1:]))
    bs_c, (m2, l2) = O.block_sums_chunked(q, kh, kc, S, block, 0.3, chunks)
    bs_1 = O.block_sums_one_head(q, kh, kc, S, block, 0.3)
    assert np.array_equal(m1, m2)
    assert np.allclose(l1, l2, rtol=1e-12)
    assert np.allclose(bs_c, bs_1, rtol=1e-12, atol=0)
    # direct definition of the normaliser, written as a sum over cells
    for a in range(s.shape[0]):
        vals = [math.exp(x - m1[a]) for x in s[a] if np.isfinite(x)]
        assert abs(sum(vals) - l1[a]) < 1e-12 * l1[a]


@pytest.mark.parametrize("seed", range(3))
def test_block_sum_invariants(seed):
    q, kh, kc, S, block = _rand_problem(seed, lh=48, lq=24, S=4, block=8)
    bs = O.block_sums_one_head(q, kh, kc, S, block, 0.6)
    br = block // S
    qb, kb = bs.shape
    kbh = kh.shape[0] // block
    assert np.all(bs >= 0)
    assert np.allclose(bs.sum(axis=1), br, rtol=1e-12)   # each softmax row sums to 1
    for i in range(qb):
        for j in range(kb - kbh):
            if j > i:
                assert bs[i, kbh + j] == 0.0            # future blocks of the chunk


def test_block_sums_uniform_scores_closed_form():
    """q = 0 makes every visible score equal, so P is uniform over the visible
    columns of each row: the block sum is sum over rows of (visible in block /
    visible in row)."""
    S, block, D = 2, 4, 3
    lh, lq = 8, 8
    q = np.zeros((lq, D))
    kh = np.ones((lh, D))
    kc = np.ones((lq, D))
    bs = O.block_sums_one_head(q, kh, kc, S, block, 1.0)
    br, ch = block // S, lh // S
    rq = lq // S
    exp = np.zeros_like(bs)
    for a in range(rq):
        vis = [b for b in range(ch + rq) if b < ch or b - ch <= a]
        for b in vis:
            exp[a // br, b // br] += 1.0 / len(vis)
    assert np.allclose(bs, exp, rtol=1e-14, atol=1e-15)


def test_default_estimation_scale_hand_values():
    """The estimation logit scale, read as 1/(sqrt(D) * stride) (the BSA page
    passes an unnamed `scale` to its block-sum step, select_blocks Step 2):
    values worked out by hand for the two head sizes of the workloads."""
    assert O.default_estimation_scale(128, 8) == pytest.approx(0.011048543456039806, rel=1e-15)
    assert O.default_estimation_scale(128, 16) == pytest.approx(0.005524271728019903, rel=1e-15)
    assert O.default_estimation_scale(64, 16) == 0.0078125       # 1 / (8 * 16)
    assert O.default_estimation_scale(4, 2) == 0.25              # 1 / (2 * 2)


def test_estimation_scale_decides_block_sums_and_selection():
    """One reshaped row (S = 2, D = 4, one KV block per reshaped column) whose
    antidiagonal products are 8, 0 and 4 by construction: with the default
    scale 1/(2*2) the scores are 2, 0, 1, so the block sums are
    e^2, 1, e over e^2 + e + 1 (closed form), and tau = 0.7 keeps blocks 0 and
    2 (0.665 < 0.7 <= 0.910).  A scale without the stride factor (0.5) or with
    sqrt(D*S) would keep block 0 alone."""
    S, block, D = 2, 2, 4
    scale = O.default_estimation_scale(D, S)
    q = np.zeros((2, D))
    q[1, 0] = 4.0                      # row a = 0 reads q[1] with key phase 0
    kh = np.zeros((4, D))
    kh[0, 0] = 2.0                     # history column 0: 4 * 2 = 8
    kc = np.zeros((2, D))
    kc[0, 0] = 1.0                     # current column 0 (visible from row 0): 4
    bs = O.block_sums_one_head(q, kh, kc, S, block, scale)
    e = math.e
    z = e * e + e + 1.0
    assert np.allclose(bs, [[e * e / z, 1.0 / z, e / z]], rtol=1e-14, atol=0)
    keep = O.threshold_select_row(bs[0].astype(np.float32), 0.7)
    assert keep.tolist() == [True, False, True]


def _sampled_bruteforce(q, kh, kc, S, block, scale, samples):
    """Explicit loops over rows and columns of the sampled estimate: the
    antidiagonal score of every visible cell, history cells outside a block's
    first `samples` reshaped columns left out, the others weighted Br/samples."""
    rb = block // S
    rq, ch, cc = q.shape[0] // S, kh.shape[0] // S, kc.shape[0] // S
    K = np.concatenate([kh, kc])
    out = np.zeros((rq // rb, (ch + cc) // rb))
    for a in range(rq):
        cells = []
        for b in range(ch + cc):
            if b < ch and b % rb >= samples:
                continue
            if b >= ch and b - ch > a:
                continue
            sc = scale * sum(float(q[S * a + S - 1 - i] @ K[S * b + i]) for i in range(S))
            cells.append((b, sc, rb / samples if b < ch else 1.0))
        m = max(c[1] for c in cells)
        tot = sum(wt * math.exp(sc - m) for _, sc, wt in cells)
        for b, sc, wt in cells:
            out[a // rb, b // rb] += wt * math.exp(sc - m) / tot
    return out


@pytest.mark.parametrize("samples", [1, 2, 4])
def test_sampled_estimation_bruteforce(samples):
    q, kh, kc, S, block = _rand_problem(31 + samples, lh=48, lq=16, S=2, block=8)
    got = O.sampled_block_sums_one_head(q, kh, kc, S, block, 0.4, samples)
    want = _sampled_bruteforce(q, kh, kc, S, block, 0.4, samples)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-14)
    assert np.allclose(got.sum(axis=1), block // S, rtol=1e-12)   # rows still sum to Br


def test_sampled_estimation_reductions():
    """All samples -> the full estimate; keys constant within each history block
    -> every sample size gives the full estimate (each sampled cell then equals
    the cells it stands for)."""
    q, kh, kc, S, block = _rand_problem(9, lh=64, lq=16, S=4, block=16)
    rb = block // S
    full = O.block_sums_one_head(q, kh, kc, S, block, 0.3)
    assert np.allclose(O.sampled_block_sums_one_head(q, kh, kc, S, block, 0.3, rb), full,
                       rtol=1e-13, atol=0)
    # one key per block, repeated: every reshaped column of a block scores alike
    rng = np.random.default_rng(10)
    kb = rng.standard_normal((kh.shape[0] // block, kh.shape[1]))
    kconst = np.repeat(kb, block, axis=0)
    full = O.block_sums_one_head(q, kconst, kc, S, block, 0.3)
    for samples in (1, 2, 3):
        got = O.sampled_block_sums_one_head(q, kconst, kc, S, block, 0.3, samples)
        assert np.allclose(got, full, rtol=1e-12, atol=1e-15)


def test_block_sums_of_sampled_query_blocks_match_full():
    q, kh, kc, S, block = _rand_problem(5, lh=32, lq=32, S=4, block=8)
    full = O.block_sums_one_head(q, kh, kc, S, block, 0.45)
    part = O.block_sums_qblocks(q, kh, kc, S, block, 0.45, [0, 2, 3])
    assert np.allclose(part, full[[0, 2, 3]], rtol=1e-13, atol=0)


# ---------------------------------------------------------------------------
# Threshold selection (find_blocks_chunked) by brute force
# ---------------------------------------------------------------------------


def _brute_select(q, tau):
    """Smallest set whose integer mass reaches R = fl(tau*T); among those of that
    size the heaviest, ties to the lowest indices."""
    n = len(q)
    T = int(sum(int(x) for x in q))
    if tau >= 1.0:
        return {j for j in range(n) if q[j] > 0}
    R = float(tau) * float(T)
    for k in range(0, n + 1):
        best = None
        for sub in itertools.combinations(range(n), k):
            mass = sum(int(q[j]) for j in sub)
            if float(mass) >= R:
                key = (-mass, sub)
                if best is None or key < best:
                    best = key
        if best is not None:
            return set(best[1])
    return set(range(n))


@pytest.mark.parametrize("seed", range(40))
def test_threshold_select_bruteforce(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 15))          # rows of up to 14 blocks
    # mix of continuous values, exact ties and zeros, like block sums
    v = rng.exponential(1.0, n).astype(np.float32)
    if n > 3:
        v[rng.integers(0, n)] = v[rng.integers(0, n)]
        v[rng.integers(0, n)] = 0.0
    tau = float(rng.choice([0.1, 0.5, 0.9, 0.95, 0.999, 1.0]))
    got = O.threshold_select_row(v, tau)
    q = O.quantize_block_sums(v)
    exp = _brute_select(q, tau)
    assert set(np.nonzero(got)[0].tolist()) == exp


def test_threshold_select_edge_cases():
    v = np.array([0.5, 2.0, 0.25, 0.0, 2.0], dtype=np.float32)
    assert O.threshold_select_row(v, 1e-12).tolist() == [False, True, False, False, False]
    assert O.threshold_select_row(v, 1.0).tolist() == [True, True, True, False, True]
    assert not O.threshold_select_row(np.zeros(4, np.float32), 0.9).any()
    # 2^-33 is below the fixed-point resolution: massless at every threshold
    tiny = np.array([1.0, 2.0 ** -34], dtype=np.float32)
    assert O.threshold_select_row(tiny, 1.0).tolist() == [True, False]
    # tau = 0.5 on [1,1,1,1]: two blocks reach half the mass exactly
    assert O.threshold_select_row(np.ones(4, np.float32), 0.5).tolist() == [True, True, False, False]


def test_quantization_is_round_half_even():
    # 3 * 2^-33 and 2^-33 sit exactly halfway between fixed-point steps
    v = np.array([2.0 ** -33, 3 * 2.0 ** -33, 5 * 2.0 ** -33], dtype=np.float32)
    assert O.quantize_block_sums(v).tolist() == [0, 2, 2]


# ---------------------------------------------------------------------------
# GQA vote
# ---------------------------------------------------------------------------


def test_vote_hand_cases():
    # H=4, Hkv=2 (G=2), Qb=2, Kb=5 (kb_hist=4, one current block)
    m = np.zeros((4, 2, 5), dtype=bool)
    # block 1: head 0 (kv 0) in qb 0, head 3 (kv 1) in qb 0 and 1 -> 3 of 4 votes
    m[0, 0, 1] = True
    m[3, 0, 1] = m[3, 1, 1] = True
    # block 2: exactly half of the votes -> not kept (strictly > 0.5)
    m[1, 0, 2] = m[1, 1, 2] = True
    # both heads of kv 0 choosing block 2 in the same qb counts once (any)
    m[0, 0, 2] = True
    # current-chunk column never takes part
    m[:, :, 4] = True
    sel = O.gqa_vote(m, 2, 4)
    assert sel.tolist() == [0, 1, 3]          # 0 and 3 forced (sink, last)
    assert O.gqa_vote(m, 2, 4, force=False).tolist() == [1]
    # other vote ratios num/den over the same counts (block 1: 3 of 4, block 2: 2 of 4)
    assert O.gqa_vote(m, 2, 4, force=False, vote=(0, 1)).tolist() == [1, 2]  # any vote
    assert O.gqa_vote(m, 2, 4, force=False, vote=(1, 4)).tolist() == [1, 2]  # > 1 of 4
    assert O.gqa_vote(m, 2, 4, force=False, vote=(3, 4)).tolist() == []      # > 3 of 4
    assert O.gqa_vote(m, 2, 4, force=False, vote=(1, 1)).tolist() == []
    assert O.gqa_vote(m, 2, 4, vote=(1, 1)).tolist() == [0, 3]                # forced only
    # G = 1: the mask votes as it is
    m1 = np.zeros((2, 3, 6), dtype=bool)
    m1[:, :2, 2] = True                        # 4 of 6 votes
    m1[0, :, 3] = True                         # 3 of 6 votes: not kept
    assert O.gqa_vote(m1, 2, 6, force=False).tolist() == [2]
    assert O.gqa_vote(m1, 2, 0).tolist() == []
    assert O.gqa_vote(m1, 2, 1).tolist() == [0]


def test_per_kv_head_selection_hand_cases():
    # H=4, Hkv=2 (G=2), Qb=2, 5 history blocks
    m = np.zeros((4, 2, 5), dtype=bool)
    m[0, 0, 1] = m[1, 1, 1] = True     # kv 0: block 1 in both query blocks (two heads)
    m[2, 0, 2] = True                  # kv 1: block 2 in one query block of two
    m[3, :, 3] = True                  # kv 1: block 3 in both
    got = O.per_kv_head_select(m, 2, 5)
    assert [g.tolist() for g in got] == [[0, 1, 4], [0, 3, 4]]
    got = O.per_kv_head_select(m, 2, 5, force=False, vote=(0, 1))
    assert [g.tolist() for g in got] == [[1], [2, 3]]


@pytest.mark.parametrize("seed", range(6))
def test_majority_vote_is_inside_the_union_of_per_kv_head_sets(seed):
    """A block with more than half of all (KV head, query block) votes has more
    than half of some KV head's own votes (pigeonhole), so the vote across KV
    heads never keeps a block that every per-KV-head selection drops."""
    rng = np.random.default_rng(seed)
    Hkv, G, qb, kb = 4, 2, 3, 9
    m = rng.random((Hkv * G, qb, kb)) < rng.uniform(0.1, 0.6)
    vote = O.gqa_vote(m, Hkv, kb, force=False)
    union = set().union(*[set(g.tolist()) for g in O.per_kv_head_select(m, Hkv, kb, force=False)])
    assert set(vote.tolist()) <= union


def test_attention_with_pages_per_kv_head():
    """Each group attends over its own pages: equal to the one-head chunk
    attention over that group's selected tokens, and to attend_request when all
    groups hold the same pages."""
    rng = np.random.default_rng(23)
    H, Hkv, D, block = 4, 2, 4, 8
    lh, lq = 32, 16
    q, k_all, v_all, perm, pool_k, pool_v = _paged_sequence(rng, H, Hkv, D, lh, lq, block)
    kc, vc = k_all[:, lh:], v_all[:, lh:]
    sel = [[0, 3], [1, 2, 3]]
    pages = [[int(perm[j]) for j in s] for s in sel]
    o, lse = O.attend_request_per_kv(q, kc, vc, pool_k, pool_v, pages, H, Hkv, 0.5)
    G = H // Hkv
    for h in range(H):
        g = h // G
        toks = np.concatenate([np.arange(j * block, (j + 1) * block) for j in sel[g]])
        ro, rl = O.bsa_chunk_attention_head(q[h], k_all[g, toks], v_all[g, toks], kc[g], vc[g],
                                            0.5)
        assert np.allclose(o[h], ro, atol=1e-12) and np.allclose(lse[h], rl, atol=1e-12)
    same = [pages[1], pages[1]]
    o2, l2 = O.attend_request_per_kv(q, kc, vc, pool_k, pool_v, same, H, Hkv, 0.5)
    o3, l3 = O.attend_request(q, kc, vc, pool_k, pool_v, pages[1], H, Hkv, 0.5)
    assert np.allclose(o2, o3, atol=1e-13) and np.allclose(l2, l3, atol=1e-13)


# ---------------------------------------------------------------------------
# Attention and the LSE merge
# ---------------------------------------------------------------------------


def _textbook_attention(q, k, v, scale, visible):
    o = np.zeros((q.shape[0], v.shape[1]))
    lse = np.zeros(q.shape[0])
    for i in range(q.shape[0]):
        logits = [scale * float(np.dot(q[i], k[j])) for j in range(k.shape[0]) if visible[i, j]]
        idx = [j for j in range(k.shape[0]) if visible[i, j]]
        if not idx:
            lse[i] = -np.inf
            continue
        z = sum(math.exp(x) for x in logits)
        for x, j in zip(logits, idx):
            o[i] += math.exp(x) / z * v[j]
        lse[i] = math.log(z)
    return o, lse


def test_attention_textbook_loops():
    rng = np.random.default_rng(11)
    q, k, v = rng.standard_normal((5, 3)), rng.standard_normal((7, 3)), rng.standard_normal((7, 2))
    vis = rng.random((5, 7)) < 0.7
    vis[2] = False
    o, lse = O.attention_with_lse(q, k, v, 0.8, vis)
    o2, lse2 = _textbook_attention(q, k, v, 0.8, vis)
    assert np.allclose(o, o2, atol=1e-12)
    assert np.array_equal(np.isinf(lse), np.isinf(lse2))
    fin = np.isfinite(lse)
    assert np.allclose(lse[fin], lse2[fin], atol=1e-12)
    assert np.all(o[2] == 0)


def test_single_key_attention():
    q = np.array([[1.0, 2.0]])
    k = np.array([[0.5, -1.0]])
    v = np.array([[3.0, 4.0, 5.0]])
    o, lse = O.attention_with_lse(q, k, v, 2.0)
    assert np.allclose(o, v) and abs(lse[0] - 2.0 * (0.5 - 2.0)) < 1e-15


@pytest.mark.parametrize("seed", range(3))
def test_split_kv_lse_merge_equals_unsplit(seed):
    rng = np.random.default_rng(seed)
    q, k, v = rng.standard_normal((6, 4)), rng.standard_normal((20, 4)), rng.standard_normal((20, 4))
    cut = int(rng.integers(1, 19))
    o, lse = O.attention_with_lse(q, k, v, 0.5)
    o1, l1 = O.attention_with_lse(q, k[:cut], v[:cut], 0.5)
    o2, l2 = O.attention_with_lse(q, k[cut:], v[cut:], 0.5)
    om, lm = O.lse_merge(o1, l1, o2, l2)
    assert np.allclose(om, o, atol=1e-12) and np.allclose(lm, lse, atol=1e-12)
    # merge order does not matter
    om2, lm2 = O.lse_merge(o2, l2, o1, l1)
    assert np.allclose(om2, o, atol=1e-12) and np.allclose(lm2, lse, atol=1e-12)


def test_lse_merge_with_empty_parts():
    o1 = np.array([[1.0, 2.0], [0.0, 0.0]])
    l1 = np.array([0.3, -np.inf])
    o2 = np.zeros((2, 2))
    l2 = np.array([-np.inf, -np.inf])
    om, lm = O.lse_merge(o1, l1, o2, l2)
    assert np.allclose(om[0], o1[0]) and lm[0] == 0.3
    assert np.all(om[1] == 0) and lm[1] == -np.inf


def test_history_then_causal_merge_equals_one_shot():
    """The pages' split form (non-causal history part, causal current part,
    merge) equals the one-shot attention over the union."""
    rng = np.random.default_rng(9)
    lq, lh, D = 8, 12, 4
    q = rng.standard_normal((lq, D))
    kh, vh = rng.standard_normal((lh, D)), rng.standard_normal((lh, D))
    kc, vc = rng.standard_normal((lq, D)), rng.standard_normal((lq, D))
    o1, l1 = O.attention_with_lse(q, kh, vh, 0.7)
    o2, l2 = O.attention_with_lse(q, kc, vc, 0.7, O.causal_visible(lq, lq))
    om, lm = O.lse_merge(o1, l1, o2, l2)
    o, lse = O.bsa_chunk_attention_head(q, kh, vh, kc, vc, 0.7)
    assert np.allclose(om, o, atol=1e-12) and np.allclose(lm, lse, atol=1e-12)


# ---------------------------------------------------------------------------
# Whole chunk: threshold 1.0 reduces to full causal attention
# ---------------------------------------------------------------------------


def test_chunk_attention_head_matches_textbook_loops():
    """One head of the chunk attention against explicit loops whose visibility
    is spelled out key by key: every selected history key, then current key j
    for query i only when j <= i (the aligned causal diagonal)."""
    rng = np.random.default_rng(13)
    lq, lh, D = 6, 5, 3
    q = rng.standard_normal((lq, D))
    kh, vh = rng.standard_normal((lh, D)), rng.standard_normal((lh, D))
    kc, vc = rng.standard_normal((lq, D)), rng.standard_normal((lq, D))
    vis = np.zeros((lq, lh + lq), dtype=bool)
    for i in range(lq):
        for j in range(lh):
            vis[i, j] = True
        for j in range(i + 1):
            vis[i, lh + j] = True
    ref_o, ref_l = _textbook_attention(q, np.concatenate([kh, kc]), np.concatenate([vh, vc]),
                                       0.6, vis)
    o, lse = O.bsa_chunk_attention_head(q, kh, vh, kc, vc, 0.6)
    assert np.allclose(o, ref_o, atol=1e-12) and np.allclose(lse, ref_l, atol=1e-12)
    # query 0 with no history sees exactly its own key: O = v_0
    o0, l0 = O.bsa_chunk_attention_head(q, kh[:0], vh[:0], kc, vc, 0.6)
    assert np.allclose(o0[0], vc[0], atol=1e-15)
    assert abs(l0[0] - 0.6 * float(np.dot(q[0], kc[0]))) < 1e-14


def _paged_sequence(rng, H, Hkv, D, lh, lq, block):
    """A sequence [history; chunk] of one request, its keys/values laid out in a
    pool whose pages are a permutation of the logical blocks."""
    Lt = lh + lq
    q = rng.standard_normal((H, lq, D)) * 0.5
    k_all = rng.standard_normal((Hkv, Lt, D)) * 0.5
    v_all = rng.standard_normal((Hkv, Lt, D))
    npg = Lt // block
    perm = rng.permutation(npg)
    pool_k = np.zeros((npg, block, Hkv, D))
    pool_v = np.zeros((npg, block, Hkv, D))
    for j in range(npg):
        for t in range(block):
            for kvh in range(Hkv):
                pool_k[perm[j], t, kvh] = k_all[kvh, j * block + t]
                pool_v[perm[j], t, kvh] = v_all[kvh, j * block + t]
    return q, k_all, v_all, perm, pool_k, pool_v


def test_estimate_request_reads_each_heads_group_through_the_pages():
    """The block sums of a request, read through a permuted page pool, equal the
    per-head block sums over the contiguous sequence, query head h using KV
    head floor(h / G) ([BSA] Step 1 repeats each KV head over its G query
    heads)."""
    rng = np.random.default_rng(17)
    H, Hkv, D, S, block = 6, 2, 4, 4, 8
    lh, lq = 24, 16
    q, k_all, _, perm, pool_k, _ = _paged_sequence(rng, H, Hkv, D, lh, lq, block)
    bs = O.estimate_request(q, k_all[:, lh:], pool_k, perm, lh, H, Hkv, S, block, 0.4)
    G = H // Hkv
    for h in range(H):
        ref = O.block_sums_one_head(q[h], k_all[h // G, :lh], k_all[h // G, lh:], S, block, 0.4)
        assert np.allclose(bs[h], ref, rtol=1e-13, atol=0)
    # the KV heads differ, so a head mapped to the wrong group is visible
    assert not np.allclose(bs[0], bs[G])


def test_attend_request_sampled_rows_and_partial_selection():
    """attend_request on a subset of query rows equals those rows of the full
    call, and with a partial page selection each head equals the one-head
    chunk attention over the selected pages' tokens, gathered from the
    contiguous sequence."""
    rng = np.random.default_rng(19)
    H, Hkv, D, block = 4, 2, 4, 8
    lh, lq = 32, 16
    q, k_all, v_all, perm, pool_k, pool_v = _paged_sequence(rng, H, Hkv, D, lh, lq, block)
    sel = [0, 2, 3]                              # logical history blocks kept
    pages = [int(perm[j]) for j in sel]
    kc, vc = k_all[:, lh:], v_all[:, lh:]
    o, lse = O.attend_request(q, kc, vc, pool_k, pool_v, pages, H, Hkv, 0.5)
    G = H // Hkv
    toks = np.concatenate([np.arange(j * block, (j + 1) * block) for j in sel])
    for h in range(H):
        ro, rl = O.bsa_chunk_attention_head(q[h], k_all[h // G, toks], v_all[h // G, toks],
                                            kc[h // G], vc[h // G], 0.5)
        assert np.allclose(o[h], ro, atol=1e-12) and np.allclose(lse[h], rl, atol=1e-12)
    rows = [0, 5, 15]
    o2, l2 = O.attend_request(q, kc, vc, pool_k, pool_v, pages, H, Hkv, 0.5, rows=rows)
    assert np.allclose(o2, o[:, rows], atol=1e-13) and np.allclose(l2, lse[:, rows], atol=1e-13)


def test_tau_one_is_full_causal_attention():
    """FullAttentionPolicy equivalence: with tau = 1 every history block with
    positive mass is kept by every head, so the vote keeps all of them and the
    chunk output equals dense causal attention over [history; chunk]."""
    rng = np.random.default_rng(21)
    H, Hkv, D, S, block = 4, 2, 8, 4, 8
    lh, lq = 32, 16
    Lt = lh + lq
    q_all = rng.standard_normal((H, Lt, D)) * 0.5
    k_all = rng.standard_normal((Hkv, Lt, D)) * 0.5
    v_all = rng.standard_normal((Hkv, Lt, D))
    # page pool in a permuted order
    npg = Lt // block
    perm = rng.permutation(npg)
    pool_k = np.zeros((npg, block, Hkv, D))
    pool_v = np.zeros((npg, block, Hkv, D))
    for j in range(npg):
        pool_k[perm[j]] = k_all[:, j * block:(j + 1) * block].transpose(1, 0, 2)
        pool_v[perm[j]] = v_all[:, j * block:(j + 1) * block].transpose(1, 0, 2)
    q = q_all[:, lh:]
    kc, vc = k_all[:, lh:], v_all[:, lh:]
    bs = O.estimate_request(q, kc, pool_k, perm, lh, H, Hkv, S, block,
                            O.default_estimation_scale(D, S))
    mask, sel, pages = O.select_request(bs.astype(np.float32), 1.0, Hkv, lh // block, perm)
    assert sel.tolist() == list(range(lh // block))
    assert pages.tolist() == perm[:lh // block].tolist()
    o, lse = O.attend_request(q, kc, vc, pool_k, pool_v, pages, H, Hkv, 1 / math.sqrt(D))
    G = H // Hkv
    for h in range(H):
        vis = np.arange(Lt)[None, :] <= (lh + np.arange(lq))[:, None]
        ref_o, ref_l = _textbook_attention(q[h], k_all[h // G], v_all[h // G],
                                           1 / math.sqrt(D), vis)
        assert np.allclose(o[h], ref_o, atol=1e-12)
        assert np.allclose(lse[h], ref_l, atol=1e-12)


def test_gather_history_follows_block_table():
    rng = np.random.default_rng(2)
    pool = rng.standard_normal((5, 4, 2, 3))
    bt = [3, 0, 4]
    rows = O.gather_history(pool, bt, 10, 1)
    assert np.array_equal(rows[0:4], pool[3, :, 1])
    assert np.array_equal(rows[4:8], pool[0, :, 1])
    assert np.array_equal(rows[8:10], pool[4, :2, 1])


# ---------------------------------------------------------------------------
# Planted mistakes must be caught by the pins above
# ---------------------------------------------------------------------------


def test_planted_mistakes_are_caught(monkeypatch):
    """Swap the antidiagonal for the diagonal reading, or drop the current-chunk
    mask, and the brute-force / closed-form pins fail."""
    q, kh, kc, S, block = _rand_problem(1, lh=8, lq=8, S=2, block=4)
    ref = _brute_scores(q, kh, kc, S, 0.37, "antidiag")
    wrong = O.estimation_scores(q, kh, kc, S, 0.37, "diag")
    diffs = [abs(wrong[a, b] - ref[a][b]) for a in range(len(ref))
             for b in range(len(ref[0])) if ref[a][b] is not None]
    assert max(diffs) > 1e-6
    s_nomask = O.estimation_scores(q, np.concatenate([kh, kc]), kc[:0], S, 0.37,
                                   include_current=False)
    assert np.isfinite(s_nomask).all() and not np.isfinite(
        O.estimation_scores(q, kh, kc, S, 0.37)).all()


def test_store_chunk_builds_the_sequence_pool():
    """Storing every chunk of a sequence, in order, into an empty pool gives the
    pool the input recipe lays out directly (logical page j of the sequence on
    physical page perm[j]): two independent statements of the same placement."""
    from xattention_block_sparse_gb300 import inputs as I
    rng = np.random.default_rng(11)
    Hkv, L, D, Bk, chunk = 2, 512, 8, 64, 128
    kv = rng.integers(1, 1 << 15, size=(Hkv, L, D)).astype(np.uint16)
    P = L // Bk + 2
    perm = rng.permutation(P).astype(np.int32)
    want = I._pages_from_seq(kv, Bk, perm, P)
    pool = np.zeros_like(want)
    for c in range(L // chunk):
        pool = O.store_chunk(pool, perm, c * chunk, kv[:, c * chunk:(c + 1) * chunk])
    assert np.array_equal(pool, want)


def test_store_chunk_skips_unallocated_pages():
    Hkv, D, Bk = 1, 4, 64
    pool = np.full((3, Bk, Hkv, D), 7.0)
    kv = np.arange(Hkv * 2 * Bk * D, dtype=np.float64).reshape(Hkv, 2 * Bk, D)
    out = O.store_chunk(pool, np.array([2, -1, 0]), Bk, kv)  # positions 64..191
    assert np.array_equal(out[0], kv[:, Bk:].transpose(1, 0, 2))   # block 2 -> page 0
    assert (out[1] == 7.0).all() and (out[2] == 7.0).all()         # block 1 is -1: skipped
