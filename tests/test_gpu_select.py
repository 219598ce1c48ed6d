"""xattn_select on synthetic block sums of many row lengths, against the oracle's
selection on the same fp32 values ("XAttention BSA Policy 设计文档", select_blocks
Step 3 find_blocks_chunked and Step 4 majority voting).

Rows of up to 1024 blocks are sorted by one warp each; longer rows by a whole
CTA.  The cases put every sort width of both paths under test, with ties
(equal block sums: the lower block index goes first), zero blocks and a
threshold of 1."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import xattn_oracle as O
from xattention_block_sparse_gb300 import xattn as X

from gpu_common import dev

pytestmark = pytest.mark.gpu


def _block_sums(rng, H, qb, kb, br, ties):
    """Rows shaped like block sums (non-negative, each row adding up to about
    Br), with runs of equal values and exact zeros."""
    v = rng.gamma(0.6, 1.0, size=(H, qb, kb))
    v[rng.random(v.shape) < 0.1] = 0.0
    v = v / np.maximum(v.sum(-1, keepdims=True), 1e-30) * br
    v = v.astype(np.float32)
    if ties:  # repeat a few values inside every row
        for h in range(H):
            for q in range(qb):
                idx = rng.choice(kb, size=min(kb, 6), replace=False)
                v[h, q, idx] = v[h, q, idx[0]]
    return v


def _run(H, Hkv, Bk, q_blocks, kh_blocks, tau, seed, vote=(1, 2), force=True, ties=True):
    rng = np.random.default_rng(seed)
    br = 16
    B = len(q_blocks)
    bt_stride = max(max(kh_blocks), 1)
    P = sum(kh_blocks) + 1
    perm = rng.permutation(P).astype(np.int32)
    bt = np.full((B, bt_stride), -1, dtype=np.int32)
    off = 0
    for r, n in enumerate(kh_blocks):
        bt[r, :n] = perm[off:off + n]
        off += n
    BT = torch.from_numpy(bt).to(dev())
    prob = X.Problem(H, Hkv, 128, 8, Bk, [n * Bk for n in q_blocks], [n * Bk for n in kh_blocks],
                     BT, P)
    rows = [_block_sums(rng, H, qb, qb + kb, br, ties) for qb, kb in zip(q_blocks, kh_blocks)]
    flat = np.concatenate([r.reshape(-1) for r in rows])
    assert flat.size == X.xattn_block_sums_count(prob)
    bs = torch.from_numpy(flat).to(dev())
    ws = torch.empty(X.xattn_workspace_size(prob), dtype=torch.uint8, device=dev())
    mask = torch.full((flat.size,), 7, dtype=torch.uint8, device=dev())
    sel_idx = torch.full((B, bt_stride), -5, dtype=torch.int32, device=dev())
    sel_page = torch.full((B, bt_stride), -5, dtype=torch.int32, device=dev())
    n_sel = torch.zeros(B, dtype=torch.int32, device=dev())
    X.xattn_select(prob, bs, tau, ws, mask, sel_idx, sel_page, n_sel, vote=vote,
                   force_sink_last=force)
    torch.cuda.synchronize()
    assert X.xattn_device_error() == 0
    gm, gs, gp, gn = (mask.cpu().numpy(), sel_idx.cpu().numpy(), sel_page.cpu().numpy(),
                      n_sel.cpu().numpy())
    for r, (qb, kb) in enumerate(zip(q_blocks, kh_blocks)):
        m_ref, s_ref, p_ref = O.select_request(rows[r], tau, Hkv, kb, bt[r], vote=vote,
                                               force=force)
        off = X.xattn_block_sums_offset(prob, r)
        m_gpu = gm[off:off + rows[r].size].reshape(rows[r].shape)
        assert np.array_equal(m_gpu.astype(bool), m_ref), f"request {r}: mask"
        assert gn[r] == len(s_ref), f"request {r}: n_sel {gn[r]} vs {len(s_ref)}"
        assert np.array_equal(gs[r, :gn[r]], s_ref), f"request {r}: selected ids"
        assert np.array_equal(gp[r, :gn[r]], p_ref), f"request {r}: pages"


@pytest.mark.parametrize("tau", [0.5, 0.9, 1.0])
def test_warp_sorted_rows_of_every_width(tau):
    # rows of 1..1024 blocks: each of the 1, 2, 4, 8, 16 and 32 keys-per-lane sorts,
    # ragged lengths inside them, requests of 0 history blocks
    _run(16, 8, 128, [1, 2, 3, 4, 2, 8, 16, 5], [0, 31, 60, 120, 250, 500, 1008, 3], tau,
         seed=11)


@pytest.mark.parametrize("H,Hkv", [(4, 4), (12, 4), (24, 2)])
def test_warp_sorted_rows_group_sizes(H, Hkv):
    # group sizes 1, 3 and 12 (more rows than a CTA's warps)
    _run(H, Hkv, 128, [3, 2, 1], [40, 0, 300], 0.8, seed=12)


def test_long_rows_take_the_cta_sort():
    # one row longer than a warp sorts: the launch goes through the CTA-wide sort
    _run(8, 4, 128, [2, 3], [1100, 200], 0.9, seed=13)


def test_vote_ratios_on_warp_path():
    _run(16, 8, 128, [4, 8], [100, 700], 0.6, seed=14, vote=(3, 4), force=False)
    _run(16, 8, 128, [4, 8], [100, 700], 0.6, seed=15, vote=(0, 1), force=True)


@pytest.mark.parametrize("per_kv", [False, True])
def test_no_history_and_no_mask_selects_nothing(per_kv):
    """A call whose requests have no history block and that asks for no mask
    (a sequence's first chunk) has empty selections: n_sel is zero for every
    row, the lists are left as they were, and the same call with a mask gives
    the same counts -- the mask it writes comes from the full kernel."""
    H, Hkv, Bk = 4, 2, 128
    q_blocks = [4, 2]
    B = len(q_blocks)
    rng = np.random.default_rng(11)
    BT = torch.full((B, 4), -1, dtype=torch.int32, device=dev())
    prob = X.Problem(H, Hkv, 128, 8, Bk, [n * Bk for n in q_blocks], [0] * B, BT, 1)
    flat = np.concatenate([_block_sums(rng, H, qb, qb, 16, False).reshape(-1) for qb in q_blocks])
    bs = torch.from_numpy(flat).to(dev())
    ws = torch.empty(X.xattn_workspace_size(prob), dtype=torch.uint8, device=dev())
    rows = B * Hkv if per_kv else B
    shape = (B, Hkv, 4) if per_kv else (B, 4)
    select = X.xattn_select_per_kv_head if per_kv else X.xattn_select
    for mask in (None, torch.full((flat.size,), 7, dtype=torch.uint8, device=dev())):
        sel_idx = torch.full(shape, -5, dtype=torch.int32, device=dev())
        sel_page = torch.full(shape, -5, dtype=torch.int32, device=dev())
        n_sel = torch.full(shape[:-1], 9, dtype=torch.int32, device=dev())
        select(prob, bs, 0.9, ws, mask, sel_idx, sel_page, n_sel)
        torch.cuda.synchronize()
        assert X.xattn_device_error() == 0
        assert n_sel.numel() == rows and torch.all(n_sel == 0)
        assert torch.all(sel_idx == -5) and torch.all(sel_page == -5)
        if mask is not None:
            assert torch.all((mask == 0) | (mask == 1))  # written by the kernel
