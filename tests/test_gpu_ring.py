"""The 128K config (Qwen3-4B-like: 32 Q / 8 KV heads, stride 16) through the
4-slot layer ring fed from pinned host memory on a side stream.

Eight synthetic layers (two wraps of the ring) run chunks 0, 1, 2 and 31 of a
131072-token context; layers 0 and 5 are checked against the float64 oracle:
block sums on sampled query blocks of sampled heads, the selection on every
row (bit-exact, oracle applied to the GPU's block sums), attention on sampled
query rows over the GPU's selection.  A slot read before its copy landed, or
reused before its layer finished, shows up as wrong keys in these checks."""
import math
import time

import numpy as np
import pytest
import torch

from oracle import xattn_oracle as O
from xattention_block_sparse_gb300 import inputs as I
from xattention_block_sparse_gb300 import runner as RN
from xattention_block_sparse_gb300 import xattn as X

from gpu_common import check_attention, check_block_sums, check_selection, dev

pytestmark = pytest.mark.gpu


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def test_q4b_128k_layer_ring_parity():
    cfg = I.CONFIGS["q4b_128k"]
    d = dev()
    H, Hkv, D, S, Bk, L, chunk = cfg.H, cfg.Hkv, cfg.D, cfg.stride, cfg.block, cfg.L, cfg.chunk
    G = H // Hkv
    P = L // Bk
    tau = cfg.taus[0]
    layers = [I.make_ring_layer(l, d) for l in range(cfg.layers)]
    ring = RN.LayerRing(cfg.ring_slots, P, Bk, Hkv, D, d)
    BT = torch.arange(P, dtype=torch.int32, device=d)[None]
    chunks = [0, 1, 2, L // chunk - 1]
    problems = {c: RN.ring_problem(H, Hkv, D, S, Bk, L, chunk, c, BT, P) for c in chunks}
    bufs = RN.ChunkBuffers.for_problems(list(problems.values()), d, with_mask=True)
    outs = [(torch.zeros((H, L, D), dtype=torch.bfloat16, device=d),
             torch.zeros((H, L), dtype=torch.float32, device=d)) for _ in layers]
    stream = torch.cuda.Stream(device=d)
    check_layers = (0, 5)
    cap = {}

    def on_layer(c):
        def f(l, b):
            if l in check_layers:
                stream.synchronize()
                n = X.xattn_block_sums_count(problems[c])
                cap[(l, c)] = dict(bs=b.block_sums[:n].cpu().numpy().copy(),
                                   mask=b.mask[:n].cpu().numpy().copy(),
                                   sel=b.sel_idx[0].cpu().numpy().copy(),
                                   pages=b.sel_page[0].cpu().numpy().copy(),
                                   n_sel=int(b.n_sel[0].item()))
        return f

    timing = {}
    for c in chunks:
        t0 = time.perf_counter()
        RN.ring_prefill_chunk(ring, layers, c, chunk, H, Hkv, D, S, Bk, tau, bufs, problems[c],
                              outs, stream, on_layer=on_layer(c))
        torch.cuda.synchronize()
        timing[c] = time.perf_counter() - t0
    assert X.xattn_device_error() == 0
    print("ring chunk wall times (s, with checks):", {c: round(t, 3) for c, t in timing.items()},
          "H2D GB:", round(ring.bytes_copied / 1e9, 2))

    rng = np.random.default_rng(7)
    scale = O.default_estimation_scale(D, S)
    br = Bk // S
    bt_row = np.arange(P)
    for l in check_layers:
        kh_all = layers[l].k_host
        vh_all = layers[l].v_host
        for c in chunks:
            t0, t1 = c * chunk, (c + 1) * chunk
            n_hist = t0 // Bk
            qb_n = chunk // Bk
            got = cap[(l, c)]
            bs32 = got["bs"].reshape(H, qb_n, n_hist + qb_n)
            heads = sorted({0, int(rng.integers(1, H - 1)), H - 1})
            qblocks = sorted({0, qb_n - 1, int(rng.integers(1, qb_n - 1))})
            for h in heads:
                kvh = h // G
                pool_k = _f64(kh_all[:, :, kvh:kvh + 1, :])
                hist = O.gather_history(pool_k, bt_row, t0, 0)
                kc = pool_k[n_hist:n_hist + qb_n, :, 0, :].reshape(chunk, D)
                q = _f64(layers[l].q[h, t0:t1])
                ref = O.block_sums_qblocks(q, hist, kc, S, Bk, scale, qblocks)
                check_block_sums(bs32[h, qblocks], ref, br, f"layer {l} chunk {c} head {h}")
            sel, pages = check_selection(bs32, got["mask"].reshape(bs32.shape), got["sel"],
                                         got["pages"], got["n_sel"], tau, Hkv, n_hist, bt_row,
                                         f"layer {l} chunk {c}")
            rows = sorted({0, chunk - 1, *rng.integers(0, chunk, 6).tolist()})
            og, lg = outs[l]
            for kvh in sorted({h // G for h in heads}):
                pk = _f64(kh_all[:, :, kvh:kvh + 1, :])
                pv = _f64(vh_all[:, :, kvh:kvh + 1, :])
                kc = pk[n_hist:n_hist + qb_n, :, 0, :].reshape(chunk, D)[None]
                vc = pv[n_hist:n_hist + qb_n, :, 0, :].reshape(chunk, D)[None]
                q = _f64(layers[l].q[kvh * G:(kvh + 1) * G, t0:t1])
                o_ref, l_ref = O.attend_request(q, kc, vc, pk, pv, pages, G, 1,
                                                1 / math.sqrt(D), rows=rows)
                idx = t0 + np.asarray(rows)
                o_g = _f64(og[kvh * G:(kvh + 1) * G][:, idx])
                l_g = lg[kvh * G:(kvh + 1) * G][:, idx].cpu().numpy()
                check_attention(o_g, l_g, o_ref, l_ref, f"layer {l} chunk {c} kv head {kvh}")


def test_ring_reused_selection_parity():
    """Layer 0's selection shared by the later layers ("XAttention BSA Policy
    设计文档", 性能分析, 优化方向 1): layer 0 estimates and selects; layers 1
    and 2 attend over layer 0's pages with their own queries, keys and values.
    Their outputs must equal the oracle's attention of each layer over layer 0's
    selected pages (and layer 0's selection the oracle's on its block sums).
    The 128K recipe at 16K tokens, three layers through two ring slots."""
    cfg = I.CONFIGS["q4b_128k"]
    d = dev()
    H, Hkv, D, S, Bk, chunk = cfg.H, cfg.Hkv, cfg.D, cfg.stride, cfg.block, cfg.chunk
    L = 4 * chunk
    G = H // Hkv
    P = L // Bk
    tau = cfg.taus[0]
    layers = [I.make_ring_layer(l, d, L=L) for l in range(3)]
    ring = RN.LayerRing(2, P, Bk, Hkv, D, d)
    BT = torch.arange(P, dtype=torch.int32, device=d)[None]
    chunks = [1, 3]
    problems = {c: RN.ring_problem(H, Hkv, D, S, Bk, L, chunk, c, BT, P) for c in chunks}
    bufs = RN.ChunkBuffers.for_problems(list(problems.values()), d, with_mask=True)
    outs = [(torch.zeros((H, L, D), dtype=torch.bfloat16, device=d),
             torch.zeros((H, L), dtype=torch.float32, device=d)) for _ in layers]
    stream = torch.cuda.Stream(device=d)
    cap = {}

    def on_layer(c):
        def f(l, b):
            if l == 0:
                stream.synchronize()
                n = X.xattn_block_sums_count(problems[c])
                cap[c] = dict(bs=b.block_sums[:n].cpu().numpy().copy(),
                              mask=b.mask[:n].cpu().numpy().copy(),
                              sel=b.sel_idx[0].cpu().numpy().copy(),
                              pages=b.sel_page[0].cpu().numpy().copy(),
                              n_sel=int(b.n_sel[0].item()))
        return f

    for c in chunks:
        RN.ring_prefill_chunk(ring, layers, c, chunk, H, Hkv, D, S, Bk, tau, bufs, problems[c],
                              outs, stream, on_layer=on_layer(c), reuse_selection=True)
    torch.cuda.synchronize()
    assert X.xattn_device_error() == 0
    rng = np.random.default_rng(5)
    bt_row = np.arange(P)
    for c in chunks:
        t0, t1 = c * chunk, (c + 1) * chunk
        n_hist, qb_n = t0 // Bk, chunk // Bk
        got = cap[c]
        bs32 = got["bs"].reshape(H, qb_n, n_hist + qb_n)
        _, pages = check_selection(bs32, got["mask"].reshape(bs32.shape), got["sel"],
                                   got["pages"], got["n_sel"], tau, Hkv, n_hist, bt_row,
                                   f"layer 0 chunk {c}")
        rows = sorted({0, chunk - 1, *rng.integers(0, chunk, 6).tolist()})
        for l in (1, 2):
            og, lg = outs[l]
            for kvh in (0, Hkv - 1):
                pk = _f64(layers[l].k_host[:, :, kvh:kvh + 1, :])
                pv = _f64(layers[l].v_host[:, :, kvh:kvh + 1, :])
                kc = pk[n_hist:n_hist + qb_n, :, 0, :].reshape(chunk, D)[None]
                vc = pv[n_hist:n_hist + qb_n, :, 0, :].reshape(chunk, D)[None]
                q = _f64(layers[l].q[kvh * G:(kvh + 1) * G, t0:t1])
                o_ref, l_ref = O.attend_request(q, kc, vc, pk, pv, pages, G, 1,
                                                1 / math.sqrt(D), rows=rows)
                idx = t0 + np.asarray(rows)
                check_attention(_f64(og[kvh * G:(kvh + 1) * G][:, idx]),
                                lg[kvh * G:(kvh + 1) * G][:, idx].cpu().numpy(), o_ref, l_ref,
                                f"layer {l} chunk {c} kv head {kvh}")
