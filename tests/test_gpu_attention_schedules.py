"""bsa_chunk_attention on its own, on shapes that drive each of its schedules:

* stream-K with a unit split over many CTAs (the merge of more than five
  parts, from global memory),
* stream-K with units split over two or three CTAs (the merge that keeps the
  last CTA's own part in tensor memory),
* a ragged last unit (128 rows: no second query tile), head_dim 64 with
  64-key tiles,
* one whole unit per CTA (a small launch),
* waves of whole units, one per CTA per wave, then stream-K ranges sized so
  that every CTA carries the same total (more units than CTAs, none longer
  than a fair share): one and two waves on one request, one wave over two
  requests of different history lengths -- each also run as plain stream-K
  (XATTN_ATTN_SCHEDULE chooses; by default waves run only when the keys and
  values exceed twice L2).

Every case uses a hand-made selection (a random ascending subset of the
history pages, pages permuted in the pool) and compares sampled rows of every
head -- including the first and last row of each 128-row tile -- with the
float64 oracle."""
import math

import numpy as np
import pytest
import torch

from oracle import xattn_oracle as O
from xattention_block_sparse_gb300 import inputs as I
from xattention_block_sparse_gb300 import xattn as X

from gpu_common import check_attention, dev, to_dev_bf16

pytestmark = pytest.mark.gpu

CASES = {
    # name: H, Hkv, D, block, stride, lq, history pages, selected pages
    "one_unit_over_many_ctas": (2, 1, 128, 128, 8, 256, 96, 96),
    "units_over_two_or_three_ctas": (32, 8, 128, 128, 8, 512, 60, 45),
    "ragged_last_unit": (4, 2, 128, 128, 8, 640, 12, 7),
    "head_dim_64_block_64": (2, 2, 64, 64, 8, 384, 150, 150),
    "whole_units": (16, 8, 128, 128, 8, 4096, 8, 3),
    "one_wave_then_stream_k": (32, 8, 128, 128, 8, 1536, 200, 150),
    "two_waves_then_stream_k": (32, 8, 128, 128, 8, 2816, 200, 150),
}
WAVE_CASES = ("one_wave_then_stream_k", "two_waves_then_stream_k")



def _bits_to_f64(bits):
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("name,schedule",
                         [(n, None) for n in CASES if n not in WAVE_CASES]
                         + [(n, sch) for n in WAVE_CASES for sch in ("waves", "streamk")])
def test_attention_schedule_parity(monkeypatch, name, schedule):
    if schedule is not None:
        monkeypatch.setenv("XATTN_ATTN_SCHEDULE", schedule)
    H, Hkv, D, Bk, S, lq, n_hist, n_sel = CASES[name]
    d = dev()
    rng = np.random.default_rng(100 + list(CASES).index(name))
    P = n_hist + 4
    q = I.bf16_round(rng.standard_normal((H, lq, D), dtype=np.float32))
    kc = I.bf16_round(rng.standard_normal((Hkv, lq, D), dtype=np.float32))
    vc = I.bf16_round(rng.standard_normal((Hkv, lq, D), dtype=np.float32))
    kp = I.bf16_round(rng.standard_normal((P, Bk, Hkv, D), dtype=np.float32))
    vp = I.bf16_round(rng.standard_normal((P, Bk, Hkv, D), dtype=np.float32))
    perm = rng.permutation(P).astype(np.int32)
    bt = perm[None, :n_hist].copy()
    logical = np.sort(rng.choice(n_hist, size=n_sel, replace=False))
    pages = bt[0, logical]

    BT = torch.from_numpy(bt).to(d)
    prob = X.Problem(H, Hkv, D, S, Bk, [lq], [n_hist * Bk], BT, P)
    ws = torch.empty(max(X.xattn_workspace_size(prob), 256), dtype=torch.uint8, device=d)
    sel_page = torch.full((1, bt.shape[1]), -7, dtype=torch.int32, device=d)
    sel_page[0, :n_sel] = torch.from_numpy(pages.astype(np.int32)).to(d)
    n_sel_t = torch.tensor([n_sel], dtype=torch.int32, device=d)
    O_ = torch.zeros((H, lq, D), dtype=torch.bfloat16, device=d)
    LSE = torch.zeros((H, lq), dtype=torch.float32, device=d)
    scale = 1.0 / math.sqrt(D)
    X.bsa_chunk_attention(prob, to_dev_bf16(q), to_dev_bf16(kc), to_dev_bf16(vc), to_dev_bf16(kp),
                          to_dev_bf16(vp), sel_page, n_sel_t, scale, ws, O_, LSE)
    torch.cuda.synchronize()
    assert X.xattn_device_error() == 0

    edges = {e for m in range(0, lq, 128) for e in (m, m + 1, m + 126, m + 127)}
    rows = sorted({r for r in edges if r < lq} | set(rng.integers(0, lq, 16).tolist()))
    o_ref, l_ref = O.attend_request(_bits_to_f64(q), _bits_to_f64(kc), _bits_to_f64(vc),
                                    _bits_to_f64(kp), _bits_to_f64(vp), pages, H, Hkv, scale,
                                    rows=rows)
    idx = np.asarray(rows)
    og = O_.float().cpu().numpy()[:, idx].astype(np.float64)
    lg = LSE.cpu().numpy()[:, idx]
    check_attention(og, lg, o_ref, l_ref, name)


@pytest.mark.parametrize("schedule", ["waves", "streamk"])
def test_wave_over_two_requests(monkeypatch, schedule):
    """Two requests (1024 and 512 query rows; 260 and 220 history pages, 200
    and 180 selected): 192 units, the wave crossing from the first request's
    units into the second's."""
    monkeypatch.setenv("XATTN_ATTN_SCHEDULE", schedule)
    H, Hkv, D, Bk, S = 32, 8, 128, 128, 8
    q_lens, n_hist, n_sel = [1024, 512], [260, 220], [200, 180]
    d = dev()
    rng = np.random.default_rng(77)
    tot = sum(q_lens)
    P = sum(n_hist) + 5
    q = I.bf16_round(rng.standard_normal((H, tot, D), dtype=np.float32))
    kc = I.bf16_round(rng.standard_normal((Hkv, tot, D), dtype=np.float32))
    vc = I.bf16_round(rng.standard_normal((Hkv, tot, D), dtype=np.float32))
    kp = I.bf16_round(rng.standard_normal((P, Bk, Hkv, D), dtype=np.float32))
    vp = I.bf16_round(rng.standard_normal((P, Bk, Hkv, D), dtype=np.float32))
    perm = rng.permutation(P).astype(np.int32)
    W = max(n_hist)
    bt = np.full((2, W), -1, dtype=np.int32)
    bt[0, :n_hist[0]] = perm[:n_hist[0]]
    bt[1, :n_hist[1]] = perm[n_hist[0]:n_hist[0] + n_hist[1]]
    pages = [bt[r, np.sort(rng.choice(n_hist[r], size=n_sel[r], replace=False))]
             for r in range(2)]
    prob = X.Problem(H, Hkv, D, S, Bk, q_lens, [n * Bk for n in n_hist],
                     torch.from_numpy(bt).to(d), P)
    ws = torch.empty(max(X.xattn_workspace_size(prob), 256), dtype=torch.uint8, device=d)
    sel_page = torch.full((2, W), -7, dtype=torch.int32, device=d)
    for r in range(2):
        sel_page[r, :n_sel[r]] = torch.from_numpy(pages[r].astype(np.int32)).to(d)
    n_sel_t = torch.tensor(n_sel, dtype=torch.int32, device=d)
    O_ = torch.zeros((H, tot, D), dtype=torch.bfloat16, device=d)
    LSE = torch.zeros((H, tot), dtype=torch.float32, device=d)
    scale = 1.0 / math.sqrt(D)
    X.bsa_chunk_attention(prob, to_dev_bf16(q), to_dev_bf16(kc), to_dev_bf16(vc), to_dev_bf16(kp),
                          to_dev_bf16(vp), sel_page, n_sel_t, scale, ws, O_, LSE)
    torch.cuda.synchronize()
    assert X.xattn_device_error() == 0
    og_all, lg_all = O_.float().cpu().numpy(), LSE.cpu().numpy()
    q0 = 0
    for r in range(2):
        lq = q_lens[r]
        edges = {e for m in range(0, lq, 128) for e in (m, m + 127)}
        rows = sorted({x for x in edges if x < lq} | set(rng.integers(0, lq, 12).tolist()))
        sl = slice(q0, q0 + lq)
        o_ref, l_ref = O.attend_request(_bits_to_f64(q[:, sl]), _bits_to_f64(kc[:, sl]),
                                        _bits_to_f64(vc[:, sl]), _bits_to_f64(kp),
                                        _bits_to_f64(vp), pages[r], H, Hkv, scale, rows=rows)
        idx = q0 + np.asarray(rows)
        check_attention(og_all[:, idx].astype(np.float64), lg_all[:, idx], o_ref, l_ref,
                        f"request {r}")
        q0 += lq


@pytest.mark.parametrize("schedule,span", [(None, "page"), ("streamk", "page"),
                                           (None, "second_half"), ("streamk", "second_half")])
def test_attention_logit_jumps(monkeypatch, schedule, span):
    """Keys whose logits sit far above or below the rest: every query carries
    a shared direction u, and the keys of some selected pages (all 128 of
    them, or only the second 64) carry +-beta u, which moves their logits by
    the boost below (in nats); so do 40 keys in the middle of the current
    chunk (+60 nats), which rows reach on their causal diagonal.  The kernel
    takes exponentials against the row max as it stood when last raised; a
    64-key half whose values climb 2^64 above it (62 nats = 89 in base 2) is
    finished by the retake -- with nothing of the tile stored yet, or after
    the first half's P was stored and must be rescaled -- one that climbs
    less is accepted as is (30 and 45 nats), and keys far below it underflow
    to zero as they should.  Rows of every 128-row tile's edges and random
    rows against the float64 oracle."""
    if schedule is not None:
        monkeypatch.setenv("XATTN_ATTN_SCHEDULE", schedule)
    H, Hkv, D, Bk, S, lq, n_hist = 4, 2, 128, 128, 8, 512, 40
    boost = {3: 30.0, 12: 62.0, 20: 0.0, 25: -62.0, 30: 45.0, 36: 70.0}
    d = dev()
    rng = np.random.default_rng(4242)
    P = n_hist + 3
    G = H // Hkv
    u = rng.standard_normal((Hkv, D))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    alpha = 8.0
    q = rng.standard_normal((H, lq, D)) + alpha * np.repeat(u, G, axis=0)[:, None, :]
    kc = rng.standard_normal((Hkv, lq, D))
    vc = rng.standard_normal((Hkv, lq, D))
    kp = rng.standard_normal((P, Bk, Hkv, D))
    vp = rng.standard_normal((P, Bk, Hkv, D))
    perm = rng.permutation(P).astype(np.int32)
    bt = perm[None, :n_hist].copy()
    rows_of_page = slice(0, Bk) if span == "page" else slice(Bk // 2, Bk)
    for lp, b in boost.items():
        beta = b * math.sqrt(D) / alpha
        kp[bt[0, lp], rows_of_page] += beta * u[None, :, :]
    kc[:, 300:340] += (60.0 * math.sqrt(D) / alpha) * u[:, None, :]
    q, kc, vc, kp, vp = (I.bf16_round(a.astype(np.float32)) for a in (q, kc, vc, kp, vp))
    pages = bt[0, :]

    prob = X.Problem(H, Hkv, D, S, Bk, [lq], [n_hist * Bk], torch.from_numpy(bt).to(d), P)
    ws = torch.empty(max(X.xattn_workspace_size(prob), 256), dtype=torch.uint8, device=d)
    sel_page = torch.from_numpy(pages.astype(np.int32))[None, :].to(d)
    n_sel_t = torch.tensor([n_hist], dtype=torch.int32, device=d)
    O_ = torch.zeros((H, lq, D), dtype=torch.bfloat16, device=d)
    LSE = torch.zeros((H, lq), dtype=torch.float32, device=d)
    scale = 1.0 / math.sqrt(D)
    X.bsa_chunk_attention(prob, to_dev_bf16(q), to_dev_bf16(kc), to_dev_bf16(vc), to_dev_bf16(kp),
                          to_dev_bf16(vp), sel_page, n_sel_t, scale, ws, O_, LSE)
    torch.cuda.synchronize()
    assert X.xattn_device_error() == 0

    edges = {e for m in range(0, lq, 128) for e in (m, m + 1, m + 126, m + 127)}
    rows = sorted(edges | set(rng.integers(0, lq, 16).tolist()))
    o_ref, l_ref = O.attend_request(_bits_to_f64(q), _bits_to_f64(kc), _bits_to_f64(vc),
                                    _bits_to_f64(kp), _bits_to_f64(vp), pages, H, Hkv, scale,
                                    rows=rows)
    # the boosted pages dominate: the largest LSE is near the top boost
    assert l_ref.max() > 60.0
    idx = np.asarray(rows)
    check_attention(O_.float().cpu().numpy()[:, idx].astype(np.float64), LSE.cpu().numpy()[:, idx],
                    o_ref, l_ref, "logit jumps")
