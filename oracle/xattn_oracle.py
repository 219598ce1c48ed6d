"""Float64 CPU oracle of XAttention block-sparse attention for chunked prefill.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA library.

Every function is the plain definition written out in float64 NumPy, in the
order the pages give the steps, with no blocking or fusion of its own.
Sources (page title, then section):

  [BSA]  "XAttention BSA Policy 设计文档" (nano-vllm docs/xattn_bsa_policy_design.md)
         -- 核心算法 1 select_blocks Steps 1-4, 核心算法 2 compute_chunked_prefill,
            参数配置, Density 统计 API
  [SYNC] "XAttention Offload Stream Synchronization Fix"
         (nano-vllm docs/xattn_offload_stream_sync_fix.md)
         -- 技术细节 "三阶段 KV Chunking 流程", 测试结果
  [PLAN] "Task Plan: Layerwise Offload Refactoring" (nano-vllm task_plan.md)
         -- Phase 1.1 ring buffer layout, Phase 1.2 per-block KV store,
            Phase 4 ring-buffer schedule
  [PAGED] "Atenção paginada" (transformers docs paged_attention.md)
         -- Caminho Varlen "Mecanismo de indexação"/"Exemplo",
            Caminho de decodificação "Exemplo"

Readings taken where the pages are silent (each is also a documented reading
of the library): antidiagonal stride reshape; estimation scale
1/(sqrt(D)*stride); current chunk included in estimation with a causal mask
at reshaped granularity (diagonal cell kept); threshold rule on block sums
quantised to 2^-32 with (value desc, index asc) order; vote restricted to
history blocks; sink and last history block forced after the vote.

Parity status: the antidiagonal reading of the stride reshape is
"parity unpinned" by the pages (they print no score values); it is pinned
only by brute force against its own definition, by the S=1 reduction to a
plain Q.K^T, and by the threshold = 1.0 reduction to full attention.
"""
from __future__ import annotations

import math

import numpy as np

NEG_INF = -np.inf

# ---------------------------------------------------------------------------
# Indexing conventions  [PAGED]
# ---------------------------------------------------------------------------


def cu_seq_lens(lengths) -> np.ndarray:
    """Cumulative sequence lengths with a leading 0 ([PAGED], Caminho Varlen,
    "Mecanismo de indexação": cu_seq_lens_q/k)."""
    out = [0]
    for n in lengths:
        out.append(out[-1] + int(n))
    return np.asarray(out, dtype=np.int64)


def request_index(cu) -> list:
    """Request id of every packed token, from cumulative lengths ([PAGED],
    Caminho Varlen, "Exemplo": Q/K request index)."""
    ids = []
    for r in range(len(cu) - 1):
        ids.extend([r] * int(cu[r + 1] - cu[r]))
    return ids


def paged_location(block_table, seq: int, t: int, page_size: int):
    """(physical page, offset) of token t of sequence seq ([PAGED], Caminho de
    decodificação, "Mecanismo de indexação": block_table rows hold the physical
    pages of a request; -1 marks an unallocated page)."""
    page = int(block_table[seq][t // page_size])
    if page < 0:
        raise IndexError(f"token {t} of sequence {seq} is in an unallocated page")
    return page, t % page_size


def pages_after_append(cache_len: int, page_size: int) -> int:
    """Pages a sequence needs once one more token is appended ([PAGED], Caminho
    de decodificação, "Exemplo": 30+1 fits one 32-token page, 32+1 needs two)."""
    return (cache_len + 1 + page_size - 1) // page_size


def gather_history(pool, block_table_row, n_tokens: int, kvh: int) -> np.ndarray:
    """History rows [n_tokens, D] of KV head kvh, read token by token through the
    block table from a pool laid out [pages, page_size, Hkv, D] ([BSA] Step 1:
    a K block arrives as [1, block_size, num_kv_heads, head_dim])."""
    page_size = pool.shape[1]
    rows = np.empty((n_tokens, pool.shape[3]), dtype=np.float64)
    for t in range(n_tokens):
        p, off = paged_location([block_table_row], 0, t, page_size)
        rows[t] = pool[p, off, kvh]
    return rows


def store_chunk(pool, block_table_row, kh_len: int, chunk_kv) -> np.ndarray:
    """The pool after a chunk's keys (or values) are stored ([PLAN] Phase 1.2,
    offload_layer_kv_async: a prefill's K/V go block by block into the cache
    blocks named by its block ids).  chunk_kv [Hkv, n, D] holds tokens at
    positions kh_len .. kh_len + n - 1 of the request; each lands at the
    [PAGED] location of its position.  A position whose page is unallocated
    (-1) is left out.  pool: [pages, page_size, Hkv, D]; returns a copy."""
    out = np.array(pool, copy=True)
    page_size = pool.shape[1]
    for t in range(chunk_kv.shape[1]):
        try:
            p, off = paged_location([block_table_row], 0, kh_len + t, page_size)
        except IndexError:
            continue
        out[p, off] = chunk_kv[:, t]
    return out


# ---------------------------------------------------------------------------
# Estimation  [BSA] Steps 1-2, [SYNC] three-stage KV chunking
# ---------------------------------------------------------------------------


def stride_reshape(x: np.ndarray, stride: int, reverse: bool) -> np.ndarray:
    """[L, D] -> [L/stride, stride*D].  Row a is the concatenation over
    i = 0..stride-1 of x[stride*a + i] (or x[stride*a + stride-1-i] when
    ``reverse``).  [BSA] Step 1 "flat_group_gemm_fuse_reshape" produces scores
    of shape [B, H, Q/s, K/s]; the reversed query order makes each score the
    sum along the anti-diagonal of a stride x stride cell (XAttention's
    antidiagonal scoring; the pages do not spell it out)."""
    L, D = x.shape
    assert L % stride == 0
    groups = x.reshape(L // stride, stride, D)
    if reverse:
        groups = groups[:, ::-1, :]
    return groups.reshape(L // stride, stride * D)


def estimation_scores(q, k_hist, k_cur, stride: int, scale: float,
                      mode: str = "antidiag", include_current: bool = True, row0: int = 0):
    """Reshaped scores s[a, b] of one query head, with masked cells at -inf.

    q: [Lq, D] query chunk; k_hist: [Lh, D] history keys (all visible:
    [BSA] Step 2 passes is_causal=False); k_cur: [Lq, D] current-chunk keys,
    appended after the history ([SYNC] Pass 1/Pass 2 "当前 chunk").  Current
    column b (chunk-local) is visible from reshaped row a iff b <= a.
    mode "antidiag": s = scale * sum_i q[S a + S-1-i] . k[S b + i];
    mode "diag":     s = scale * sum_i q[S a + i]     . k[S b + i].
    ``row0`` is the reshaped index of q's first row when q is a slice of the
    chunk (the causal test then uses the row's index in the whole chunk)."""
    keys = [k_hist] + ([k_cur] if include_current else [])
    K = np.concatenate(keys, axis=0) if len(keys) > 1 else keys[0]
    Qr = stride_reshape(q, stride, reverse=(mode == "antidiag"))
    Kr = stride_reshape(K, stride, reverse=False)
    s = scale * (Qr @ Kr.T)
    if include_current:
        ch = k_hist.shape[0] // stride
        rq = Qr.shape[0]
        a = row0 + np.arange(rq)[:, None]
        b = np.arange(k_cur.shape[0] // stride)[None, :]
        s[:, ch:][b > a] = NEG_INF
    return s


def softmax_stats(s: np.ndarray):
    """One-shot row statistics: m = max over visible cells, l = sum exp(s - m).
    A row with no visible cell has m = -inf and l = 0."""
    m = np.max(s, axis=-1)
    l = np.zeros_like(m)
    fin = np.isfinite(m)
    l[fin] = np.sum(np.exp(s[fin] - m[fin, None]), axis=-1)
    return m, l


def partial_stats(s_chunk: np.ndarray):
    """[SYNC] Stage 1 softmax_compute_partial_stats: (m_i, l_i) of one KV chunk."""
    return softmax_stats(s_chunk)


def merge_stats(parts):
    """[SYNC] Stage 2 merge_softmax_stats: m = max_i m_i,
    l = sum_i l_i * exp(m_i - m)."""
    ms = np.stack([p[0] for p in parts])
    ls = np.stack([p[1] for p in parts])
    m = np.max(ms, axis=0)
    l = np.zeros_like(m)
    fin = np.isfinite(m)
    w = np.zeros_like(ms)
    w[:, fin] = np.exp(ms[:, fin] - m[None, fin])
    l[fin] = np.sum(ls[:, fin] * w[:, fin], axis=0)
    return m, l


def normalized_block_sums(s: np.ndarray, m, l, rblock: int) -> np.ndarray:
    """[SYNC] Stage 3 softmax_normalize_and_block_sum / [BSA] Step 2
    softmax_fuse_block_sum: P = exp(s - m)/l, summed over rblock x rblock cells
    (reshaped_block_size = block_size / stride).  Returns [Qb, Kb]."""
    rq, c = s.shape
    assert rq % rblock == 0 and c % rblock == 0
    p = np.zeros_like(s)
    fin = np.isfinite(m)
    p[fin] = np.exp(s[fin] - m[fin, None]) / l[fin, None]
    return p.reshape(rq // rblock, rblock, c // rblock, rblock).sum(axis=(1, 3))


def block_sums_one_head(q, k_hist, k_cur, stride, block, scale, mode="antidiag",
                        include_current=True):
    """Block sums [Qb, Kb_h + Kb_c] of one query head (one-shot statistics)."""
    s = estimation_scores(q, k_hist, k_cur, stride, scale, mode, include_current)
    m, l = softmax_stats(s)
    return normalized_block_sums(s, m, l, block // stride)


def block_sums_qblocks(q, k_hist, k_cur, stride, block, scale, qblocks, mode="antidiag"):
    """Rows ``qblocks`` of block_sums_one_head, computed from those query blocks
    alone: softmax statistics are per reshaped row, so a row needs only its own
    scores.  Returns [len(qblocks), Kb_h + Kb_c]."""
    rb = block // stride
    out = []
    for qb in qblocks:
        s = estimation_scores(q[qb * block:(qb + 1) * block], k_hist, k_cur, stride, scale,
                              mode, row0=qb * rb)
        m, l = softmax_stats(s)
        out.append(normalized_block_sums(s, m, l, rb)[0])
    return np.stack(out)


def block_sums_chunked(q, k_hist, k_cur, stride, block, scale, col_chunks,
                       mode="antidiag"):
    """The three stages of [SYNC] over explicit column chunks (lists of column
    ranges of the reshaped score matrix): partial stats per chunk, merge, then
    normalise + block-sum with the merged stats."""
    s = estimation_scores(q, k_hist, k_cur, stride, scale, mode)
    parts = [partial_stats(s[:, a:b]) for a, b in col_chunks]
    m, l = merge_stats(parts)
    return normalized_block_sums(s, m, l, block // stride), (m, l)


def sampled_block_sums_one_head(q, k_hist, k_cur, stride, block, scale, samples,
                                mode="antidiag"):
    """Block sums estimated from a sample of each history block's keys ([BSA]
    性能分析, 优化方向 2: estimate from part of the K blocks; the chunked
    policy page's Phase 1 loads samples_per_chunk tokens of each history
    chunk).  Reading: of each history block only its first `samples` reshaped
    columns (samples * stride tokens) are scored; each sampled cell stands for
    block/stride / samples cells of its block, so it carries the weight
    w = (block/stride) / samples in the row's softmax sum and in the block's
    sum; the current chunk's columns are all scored (weight 1).  With
    samples = block/stride this is block_sums_one_head.  Returns [Qb, Kb]."""
    rb = block // stride
    assert 1 <= samples <= rb
    s = estimation_scores(q, k_hist, k_cur, stride, scale, mode)
    ch = k_hist.shape[0] // stride
    col = np.arange(s.shape[1])
    sampled = (col >= ch) | ((col % rb) < samples)     # history: first `samples` of a block
    w = np.where(col < ch, rb / samples, 1.0)
    s = np.where(sampled[None, :], s, NEG_INF)
    m = np.max(s, axis=-1)
    p = np.zeros_like(s)
    fin = np.isfinite(m)
    p[fin] = w[None, :] * np.exp(s[fin] - m[fin, None])
    l = p.sum(axis=-1)
    p[fin] /= l[fin, None]
    rq, c = s.shape
    return p.reshape(rq // rb, rb, c // rb, rb).sum(axis=(1, 3))


# ---------------------------------------------------------------------------
# Selection  [BSA] Steps 3-4
# ---------------------------------------------------------------------------

FIX_SHIFT = 32


def quantize_block_sums(v32: np.ndarray) -> np.ndarray:
    """Fixed-point block mass: round-half-even(v * 2^32) as int64.  v is the
    fp32 block sum; v * 2^32 is exact in float64, so the integer is unique."""
    v = np.asarray(v32, dtype=np.float32).astype(np.float64)
    return np.rint(v * float(2 ** FIX_SHIFT)).astype(np.int64)


def threshold_select_row(v32_row: np.ndarray, tau: float) -> np.ndarray:
    """[BSA] Step 3 find_blocks_chunked on one (head, query-block) row: keep the
    shortest prefix of blocks, in descending mass order, whose mass reaches
    tau * (row total).  Exact rule: with integer masses q_j and T = sum q_j,
    R = fl64(tau * T); walking j in (q_j desc, j asc) order, block j is kept
    iff the integer mass of the blocks before it is < R.  tau >= 1 keeps every
    block with q_j > 0."""
    q = quantize_block_sums(v32_row)
    n = q.shape[0]
    keep = np.zeros(n, dtype=bool)
    if tau >= 1.0:
        return q > 0
    total = int(q.sum())
    R = float(tau) * float(total)
    order = sorted(range(n), key=lambda j: (-int(q[j]), j))
    before = 0
    for j in order:
        keep[j] = float(before) < R
        before += int(q[j])
    return keep


def threshold_select(v32: np.ndarray, tau: float) -> np.ndarray:
    """find_blocks_chunked over a [H, Qb, Kb] block-sum tensor -> bool mask."""
    out = np.zeros(v32.shape, dtype=bool)
    for idx in np.ndindex(*v32.shape[:-1]):
        out[idx] = threshold_select_row(v32[idx], tau)
    return out


def gqa_vote(mask: np.ndarray, num_kv_heads: int, kb_hist: int, force: bool = True,
             vote=(1, 2)):
    """[BSA] Step 4 GQA-aware aggregation + majority voting on a [H, Qb, Kb]
    mask.  Any query head of a KV-head group selects for the group (with one
    head per group the mask is used as it is); a history block survives when
    it is voted for by more than vote = num/den of the (KV head, query block)
    pairs -- the pages' vote_ratio > 0.5 is (1, 2); then, with `force`, the
    first (sink) and last history block are always added.  Only the history
    columns j < kb_hist take part: the current chunk is always attended
    causally.  Returns ascending logical block ids."""
    H, qb, _ = mask.shape
    G = H // num_kv_heads
    if kb_hist == 0:
        return np.zeros(0, dtype=np.int64)
    m = mask[:, :, :kb_hist].reshape(num_kv_heads, G, qb, kb_hist)
    per_kv = m.any(axis=1)
    count = per_kv.sum(axis=(0, 1))
    num, den = vote
    keep = count * den > num * num_kv_heads * qb   # count / total > num / den, in integers
    if force:
        keep[0] = True
        keep[kb_hist - 1] = True
    return np.nonzero(keep)[0].astype(np.int64)


def per_kv_head_select(mask: np.ndarray, num_kv_heads: int, kb_hist: int, force: bool = True,
                       vote=(1, 2)):
    """One block set per KV head, the selection [BSA] Step 4 sets beside the vote
    across KV heads ("为什么使用 Majority Voting?").  Reading: KV head g keeps
    history block j when more than num/den of its query blocks chose it, any
    query head of its group counting for the block; sink and last forced.  It
    is the vote above restricted to one KV head.  Returns one ascending id
    array per KV head."""
    G = mask.shape[0] // num_kv_heads
    return [gqa_vote(mask[g * G:(g + 1) * G], 1, kb_hist, force=force, vote=vote)
            for g in range(num_kv_heads)]


def density(selected: int, available: int) -> float:
    """[BSA] Density 统计 API: selected / available history blocks."""
    return selected / available if available else 0.0


# ---------------------------------------------------------------------------
# Attention  [BSA] compute_chunked_prefill
# ---------------------------------------------------------------------------


def attention_with_lse(q, k, v, scale: float, visible=None):
    """Softmax attention with log-sum-exp per query row (the flash_attn_with_lse
    contract of [BSA] compute_chunked_prefill).  Rows with no visible key give
    O = 0 and LSE = -inf."""
    logits = scale * (q @ k.T)
    if visible is not None:
        logits = np.where(visible, logits, NEG_INF)
    m = np.max(logits, axis=-1) if logits.shape[-1] else np.full(q.shape[0], NEG_INF)
    o = np.zeros((q.shape[0], v.shape[1]), dtype=np.float64)
    lse = np.full(q.shape[0], NEG_INF)
    fin = np.isfinite(m)
    if np.any(fin):
        p = np.exp(logits[fin] - m[fin, None])
        l = p.sum(axis=-1)
        o[fin] = (p @ v) / l[:, None]
        lse[fin] = m[fin] + np.log(l)
    return o, lse


def causal_visible(lq: int, lk: int) -> np.ndarray:
    """Causal mask of a query chunk against its own keys (same length, aligned
    diagonal): query i sees key j iff j <= i ([BSA] step 2, causal=True)."""
    assert lq == lk
    return np.arange(lk)[None, :] <= np.arange(lq)[:, None]


def lse_merge(o1, lse1, o2, lse2):
    """merge_attention_outputs ([BSA] compute_chunked_prefill steps 1 and 3):
    lse = log(exp(lse1) + exp(lse2)) computed around the max;
    o = o1 * exp(lse1 - lse) + o2 * exp(lse2 - lse).  Two empty parts
    (both -inf) merge to O = 0, LSE = -inf."""
    mx = np.maximum(lse1, lse2)
    lse = np.full_like(mx, NEG_INF)
    o = np.zeros_like(o1)
    fin = np.isfinite(mx)
    s = np.exp(lse1[fin] - mx[fin]) + np.exp(lse2[fin] - mx[fin])
    lse[fin] = mx[fin] + np.log(s)
    w1 = np.exp(lse1[fin] - lse[fin])
    w2 = np.exp(lse2[fin] - lse[fin])
    o[fin] = o1[fin] * w1[:, None] + o2[fin] * w2[:, None]
    return o, lse


def bsa_chunk_attention_head(q, k_sel, v_sel, k_cur, v_cur, scale: float):
    """One head of [BSA] compute_chunked_prefill, one-shot over the union of keys:
    every selected history token (non-causal) plus the current chunk's tokens
    j <= i.  Equal, up to rounding, to the pages' split form (history partial,
    current causal partial, merged by lse_merge)."""
    lq = q.shape[0]
    K = np.concatenate([k_sel, k_cur], axis=0)
    V = np.concatenate([v_sel, v_cur], axis=0)
    vis = np.concatenate([np.ones((lq, k_sel.shape[0]), dtype=bool),
                          causal_visible(lq, k_cur.shape[0])], axis=1)
    return attention_with_lse(q, K, V, scale, vis)


# ---------------------------------------------------------------------------
# Whole chunk, as the library's entry points see it
# ---------------------------------------------------------------------------


def estimate_request(q, k_cur, pool_k, bt_row, kh_len, H, Hkv, stride, block, scale,
                     mode="antidiag"):
    """Block sums [H, Qb, Kb_h + Kb_c] of one request of one chunk.
    q: [H, Lq, D]; k_cur: [Hkv, Lq, D]; history through the block table."""
    G = H // Hkv
    out = []
    hist = [gather_history(pool_k, bt_row, kh_len, kvh) for kvh in range(Hkv)]
    for h in range(H):
        kvh = h // G          # [BSA] Step 1: repeat_interleave(num_groups, dim=1)
        out.append(block_sums_one_head(q[h], hist[kvh], k_cur[kvh], stride, block,
                                       scale, mode))
    return np.stack(out)


def select_request(bs32, tau, Hkv, kb_hist, bt_row, vote=(1, 2), force=True):
    """Threshold selection + vote of one request: (mask, sel_idx, sel_page)."""
    mask = threshold_select(bs32, tau)
    sel = gqa_vote(mask, Hkv, kb_hist, force=force, vote=vote)
    pages = np.asarray([int(bt_row[j]) for j in sel], dtype=np.int64)
    return mask, sel, pages


def attend_request(q, k_cur, v_cur, pool_k, pool_v, sel_pages, H, Hkv, scale,
                   rows=None):
    """Attention output [H, Lq, D] and LSE [H, Lq] of one request over the
    selected pages (ascending logical order) plus the causal current chunk.
    ``rows`` restricts the query rows computed (sampling for large shapes)."""
    G = H // Hkv
    lq = q.shape[1]
    rows = np.arange(lq) if rows is None else np.asarray(rows)
    D = q.shape[2]
    o = np.zeros((H, len(rows), D))
    lse = np.zeros((H, len(rows)))
    for kvh in range(Hkv):
        if len(sel_pages):
            ks = np.concatenate([pool_k[p, :, kvh, :] for p in sel_pages], axis=0)
            vs = np.concatenate([pool_v[p, :, kvh, :] for p in sel_pages], axis=0)
        else:
            ks = np.zeros((0, D))
            vs = np.zeros((0, D))
        for g in range(G):
            h = kvh * G + g
            K = np.concatenate([ks, k_cur[kvh]], axis=0)
            V = np.concatenate([vs, v_cur[kvh]], axis=0)
            vis = np.concatenate(
                [np.ones((len(rows), ks.shape[0]), dtype=bool),
                 np.arange(lq)[None, :] <= rows[:, None]], axis=1)
            o[h], lse[h] = attention_with_lse(q[h, rows], K, V, scale, vis)
    return o, lse


def attend_request_per_kv(q, k_cur, v_cur, pool_k, pool_v, pages_per_kv, H, Hkv, scale,
                          rows=None):
    """attend_request with its own selected pages for each KV head
    (per_kv_head_select): the query heads of group g attend over the pages in
    pages_per_kv[g] and the causal current chunk."""
    G = H // Hkv
    outs = [attend_request(q[g * G:(g + 1) * G], k_cur[g:g + 1], v_cur[g:g + 1],
                           pool_k[:, :, g:g + 1], pool_v[:, :, g:g + 1], pages_per_kv[g], G, 1,
                           scale, rows) for g in range(Hkv)]
    return (np.concatenate([o for o, _ in outs], axis=0),
            np.concatenate([l for _, l in outs], axis=0))


def default_estimation_scale(head_dim: int, stride: int) -> float:
    """Reading: the pages pass an unnamed scale; 1/(sqrt(D)*stride) is the usual
    1/sqrt(D) logit scale averaged over the stride products of a cell."""
    return 1.0 / (math.sqrt(head_dim) * stride)


# ---------------------------------------------------------------------------
# Ring-buffer schedule  [PLAN]
# ---------------------------------------------------------------------------


def ring_slot(layer: int, num_buffers: int) -> int:
    """[PLAN] Phase 4: layer l computes from ring slot l mod N."""
    return layer % num_buffers


def ring_schedule(num_layers: int, num_buffers: int):
    """[PLAN] Phase 4 ring schedule as an event list: preload the first N
    layers, then after computing layer l reload its slot with layer l+N.
    Returns [("load"|"compute", layer, slot), ...] in issue order."""
    ev = [("load", l, ring_slot(l, num_buffers)) for l in range(min(num_buffers, num_layers))]
    for l in range(num_layers):
        ev.append(("compute", l, ring_slot(l, num_buffers)))
        if l + num_buffers < num_layers:
            ev.append(("load", l + num_buffers, ring_slot(l, num_buffers)))
    return ev


def layer_slot_bytes(max_tokens: int, kv_heads: int, head_dim: int, elem_bytes: int = 2):
    """[PLAN] Phase 1.1: bytes of one layer's K (or V) ring slot."""
    return max_tokens * kv_heads * head_dim * elem_bytes
