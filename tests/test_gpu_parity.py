"""GPU-vs-oracle parity of the whole chunked-prefill path, through the C-ABI.

Block sums within 1e-3 relative; the oracle's selection applied to the GPU's
block sums equals the GPU's mask, block ids and pages bit for bit; attention
output within 2e-2 max-abs and LSE within 1e-3 against the oracle over the
same selection."""
import math

import numpy as np
import pytest
import torch

from oracle import xattn_oracle as O
from xattention_block_sparse_gb300 import inputs as I
from xattention_block_sparse_gb300 import runner as RN
from xattention_block_sparse_gb300 import xattn as X

from gpu_common import (SequenceCase, check_attention, check_block_sums, check_selection, dev,
                        record_flips, to_dev_bf16)

pytestmark = pytest.mark.gpu


def test_tiny_all_chunks_full_parity():
    case = SequenceCase("tiny")
    tau = case.cfg.taus[0]
    n = case.L // case.chunk
    O_, LSE, cap = case.run(tau, capture=range(n))
    for c in range(n):
        case.check_chunk(c, cap[c], O_, LSE, tau)


def test_tiny_ragged_chunk_of_one_block():
    """Chunks of one 64-token block: a query tile shorter than the CTA tile
    and reshaped rows fewer than one GEMM tile."""
    case = SequenceCase("tiny", L=512, chunk=64)
    tau = 0.9
    n = case.L // case.chunk
    O_, LSE, cap = case.run(tau, capture=range(n))
    for c in range(n):
        case.check_chunk(c, cap[c], O_, LSE, tau)


def test_tiny_tau_one_is_dense_causal_attention():
    """threshold 1.0 keeps every history block (FullAttentionPolicy): the output
    equals dense causal attention over the whole prefix."""
    case = SequenceCase("tiny")
    O_, LSE, cap = case.run(1.0, capture=range(4))
    q, k, v, _, _ = case.oracle_inputs()
    for c in range(4):
        assert cap[c]["n_sel"] == c * case.chunk // case.cfg.block
    L, D = case.L, case.cfg.D
    for h in range(case.cfg.H):
        vis = np.arange(L)[None, :] <= np.arange(L)[:, None]
        o_ref, l_ref = O.attention_with_lse(q[h], k[0], v[0], 1 / math.sqrt(D), vis)
        check_attention(O_[h], LSE[h], o_ref, l_ref, f"head {h}")


def test_q06b_4k_all_chunks_full_parity():
    case = SequenceCase("q06b_4k")
    tau = 0.9
    n = case.L // case.chunk
    O_, LSE, cap = case.run(tau, capture=range(n))
    for c in range(n):
        case.check_chunk(c, cap[c], O_, LSE, tau)


@pytest.mark.parametrize("tau", [0.9, 0.95])
def test_q06b_32k_sampled_parity(tau):
    """Full 32K context in 4096-token chunks through the permuted page pool;
    block sums on sampled query blocks, selection on every row, attention on
    sampled query rows (first, last and spread)."""
    case = SequenceCase("q06b_32k")
    n = case.L // case.chunk
    chunks = [0, 1, n - 1]
    O_, LSE, cap = case.run(tau, capture=chunks)
    rng = np.random.default_rng(0)
    for c in chunks:
        qblocks = sorted({0, case.chunk // case.cfg.block - 1,
                          int(rng.integers(1, case.chunk // case.cfg.block - 1))})
        rows = sorted({0, case.chunk - 1, *rng.integers(0, case.chunk, 14).tolist()})
        case.check_chunk(c, cap[c], O_, LSE, tau, qblocks=qblocks, rows=rows)


def test_varlen_batch_parity():
    wl = I.make_workload("varlen")
    cfg = wl.cfg
    call = wl.calls[0]
    d = dev()
    Q, K, V = to_dev_bf16(wl.q_bits), to_dev_bf16(wl.k_bits), to_dev_bf16(wl.v_bits)
    KP, VP = to_dev_bf16(wl.kpool_bits), to_dev_bf16(wl.vpool_bits)
    BT = torch.from_numpy(wl.block_table).to(d)
    prob = X.Problem(cfg.H, cfg.Hkv, cfg.D, cfg.stride, cfg.block, call.q_lens, call.kh_lens, BT,
                     KP.shape[0])
    bufs = RN.ChunkBuffers.for_problems([prob], d, with_mask=True)
    tot = sum(call.q_lens)
    O_ = torch.empty((cfg.H, tot, cfg.D), dtype=torch.bfloat16, device=d)
    LSE = torch.empty((cfg.H, tot), dtype=torch.float32, device=d)
    tau = cfg.taus[0]
    RN.prefill_chunk(prob, Q, K, V, KP, VP, tau, bufs, O_, LSE)
    torch.cuda.synchronize()
    assert X.xattn_device_error() == 0
    bs_all = bufs.block_sums.cpu().numpy()
    mask_all = bufs.mask.cpu().numpy()
    sel_all, page_all = bufs.sel_idx.cpu().numpy(), bufs.sel_page.cpu().numpy()
    nsel = bufs.n_sel.cpu().numpy()
    Og, Lg = O_.float().cpu().numpy(), LSE.cpu().numpy()
    q, k, v = wl.f64("q"), wl.f64("k"), wl.f64("v")
    kp, vp = wl.f64("kpool"), wl.f64("vpool")
    scale = O.default_estimation_scale(cfg.D, cfg.stride)
    br = cfg.block // cfg.stride
    G = cfg.H // cfg.Hkv
    rng = np.random.default_rng(1)
    for r in range(3):
        q0, q1 = int(call.cu_q[r]), int(call.cu_q[r + 1])
        kh = call.kh_lens[r]
        kbh, qb_n = kh // cfg.block, (q1 - q0) // cfg.block
        off = X.xattn_block_sums_offset(prob, r)
        bs = bs_all[off:off + cfg.H * qb_n * (kbh + qb_n)].reshape(cfg.H, qb_n, kbh + qb_n)
        mk = mask_all[off:off + bs.size].reshape(bs.shape)
        qblocks = sorted({0, qb_n - 1, int(rng.integers(0, qb_n))})
        for h in range(cfg.H):
            hist = O.gather_history(kp, wl.block_table[r], kh, h // G)
            ref = O.block_sums_qblocks(q[h, q0:q1], hist, k[h // G, q0:q1], cfg.stride,
                                       cfg.block, scale, qblocks)
            check_block_sums(bs[h, qblocks], ref, br, f"request {r} head {h}")
        sel, pages = check_selection(bs, mk, sel_all[r], page_all[r], int(nsel[r]), tau,
                                     cfg.Hkv, kbh, wl.block_table[r], f"request {r}")
        rows = sorted({0, q1 - q0 - 1, *rng.integers(0, q1 - q0, 10).tolist()})
        o_ref, l_ref = O.attend_request(q[:, q0:q1], k[:, q0:q1], v[:, q0:q1], kp, vp, pages,
                                        cfg.H, cfg.Hkv, 1 / math.sqrt(cfg.D), rows=rows)
        idx = q0 + np.asarray(rows)
        check_attention(Og[:, idx], Lg[:, idx], o_ref, l_ref, f"request {r}")
    assert nsel[0] == 0  # no history, no selection


def test_lse_merge_matches_oracle():
    rng = np.random.default_rng(4)
    rows, D = 1000, 128
    o1, o2 = rng.standard_normal((rows, D)), rng.standard_normal((rows, D))
    l1, l2 = rng.standard_normal(rows) * 3, rng.standard_normal(rows) * 3
    l1[:5] = -np.inf
    l2[3:8] = -np.inf
    d = dev()
    t = lambda a: torch.from_numpy(a.astype(np.float32)).to(d)
    oo = torch.empty((rows, D), dtype=torch.float32, device=d)
    lo = torch.empty(rows, dtype=torch.float32, device=d)
    X.lse_merge(t(o1), t(l1), t(o2), t(l2), oo, lo)
    ob = torch.empty((rows, D), dtype=torch.bfloat16, device=d)
    lb = torch.empty(rows, dtype=torch.float32, device=d)
    X.lse_merge(t(o1), t(l1), t(o2), t(l2), ob, lb)
    torch.cuda.synchronize()
    f32 = lambda a: a.astype(np.float32).astype(np.float64)
    o_ref, l_ref = O.lse_merge(f32(o1), f32(l1), f32(o2), f32(l2))
    assert np.abs(oo.cpu().numpy() - o_ref).max() < 1e-5
    assert np.abs(ob.float().cpu().numpy() - o_ref).max() < 2e-2
    lg = lo.cpu().numpy()
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(lg), fin)
    assert np.abs(lg[fin] - l_ref[fin]).max() < 1e-5
    # in place: o_out aliases o1, lse_out aliases lse1
    a, la = t(o1), t(l1)
    X.lse_merge(a, la, t(o2), t(l2), a, la)
    torch.cuda.synchronize()
    assert np.abs(a.cpu().numpy() - o_ref).max() < 1e-5
    assert np.abs(la.cpu().numpy()[fin] - l_ref[fin]).max() < 1e-5


def test_unallocated_page_is_reported_not_trapped():
    """A block-table entry of -1 inside the history is recorded in the device
    error word; kernels skip the page and the context stays usable."""
    case = SequenceCase("tiny")
    X.xattn_device_error()  # clear
    bt = case.BT.clone()
    bt[0, 1] = -1
    prob = X.Problem(case.cfg.H, case.cfg.Hkv, case.cfg.D, case.cfg.stride, case.cfg.block,
                     [case.chunk], [2 * case.chunk], bt, case.KP.shape[0],
                     q_head_stride=case.L * case.cfg.D, kv_head_stride=case.L * case.cfg.D,
                     lse_head_stride=case.L)
    bufs = RN.ChunkBuffers.for_problems([prob], dev())
    O_ = torch.empty((case.cfg.H, case.L, case.cfg.D), dtype=torch.bfloat16, device=dev())
    LSE = torch.empty((case.cfg.H, case.L), dtype=torch.float32, device=dev())
    t0 = 2 * case.chunk
    X.xattn_device_error(clear=True)  # clear anything an earlier test left
    RN.prefill_chunk(prob, case.Q[:, t0:], case.K[:, t0:], case.V[:, t0:], case.KP, case.VP, 0.9,
                     bufs, O_[:, t0:], LSE[:, t0:])
    code = X.xattn_device_error(clear=False)
    assert code == -3
    assert X.xattn_last_device_error() == -3  # read and reset
    assert X.xattn_device_error() == 0
    assert torch.isfinite(LSE[:, t0:]).all()


def test_stream_ordering_side_stream_copy():
    """History pages are written on a side stream and published with an event;
    the compute stream waits on the event before estimation (the ordering the
    stream-sync page prescribes).  Results equal a run with the pool already
    resident."""
    case = SequenceCase("tiny")
    d = dev()
    c = 3
    t0 = c * case.chunk
    ref = {}
    prob = case.seq.problems[c]
    host_k = case.KP.cpu().pin_memory()
    host_v = case.VP.cpu().pin_memory()
    for mode in ("resident", "side"):
        kp = torch.zeros_like(case.KP)
        vp = torch.zeros_like(case.VP)
        bufs = RN.ChunkBuffers.for_problems([prob], d, with_mask=True)
        O_ = torch.zeros((case.cfg.H, case.L, case.cfg.D), dtype=torch.bfloat16, device=d)
        LSE = torch.zeros((case.cfg.H, case.L), dtype=torch.float32, device=d)
        if mode == "resident":
            kp.copy_(case.KP)
            vp.copy_(case.VP)
        torch.cuda.synchronize()
        side, comp = torch.cuda.Stream(), torch.cuda.Stream()
        if mode == "side":
            ev = torch.cuda.Event()
            with torch.cuda.stream(side):
                kp.copy_(host_k, non_blocking=True)
                vp.copy_(host_v, non_blocking=True)
                ev.record(side)
            comp.wait_event(ev)
        with torch.cuda.stream(comp):
            RN.prefill_chunk(prob, case.Q[:, t0:], case.K[:, t0:], case.V[:, t0:], kp, vp, 0.9,
                             bufs, O_[:, t0:], LSE[:, t0:], stream=comp)
        torch.cuda.synchronize()
        n = int(bufs.n_sel[0].item())
        ref[mode] = (bufs.block_sums.cpu().numpy(), bufs.sel_idx[0, :n].cpu().numpy(),
                     O_.float().cpu().numpy())
    assert np.array_equal(ref["resident"][0], ref["side"][0])
    assert np.array_equal(ref["resident"][1], ref["side"][1])
    assert np.array_equal(ref["resident"][2], ref["side"][2])


@pytest.mark.parametrize("vote,force", [((0, 1), False), ((1, 4), True), ((3, 4), False),
                                        ((1, 1), True)])
def test_selection_vote_parameters(vote, force):
    """Vote ratio num/den and sink/last forcing of xattn_select, bit-exact against
    the oracle's selection on the GPU's own block sums (a partial threshold, so
    the votes differ between blocks)."""
    case = SequenceCase("q06b_4k")
    cfg = case.cfg
    c, tau = 3, 0.6
    p, b = case.seq.problems[c], case.seq.bufs
    t0 = c * case.chunk
    X.xattn_estimate(p, case.Q[:, t0:], case.K[:, t0:], case.KP,
                     RN.estimation_scale(cfg.D, cfg.stride), b.workspace, b.block_sums)
    X.xattn_select(p, b.block_sums, tau, b.workspace, b.mask, b.sel_idx, b.sel_page, b.n_sel,
                   vote=vote, force_sink_last=force)
    torch.cuda.synchronize()
    assert X.xattn_device_error() == 0
    n = X.xattn_block_sums_count(p)
    kbh, qb_n = t0 // cfg.block, case.chunk // cfg.block
    bs32 = b.block_sums[:n].cpu().numpy().reshape(cfg.H, qb_n, kbh + qb_n)
    mk = b.mask[:n].cpu().numpy().reshape(bs32.shape)
    check_selection(bs32, mk, b.sel_idx[0].cpu().numpy(), b.sel_page[0].cpu().numpy(),
                    int(b.n_sel[0].item()), tau, cfg.Hkv, kbh, case.wl.block_table[0],
                    f"vote {vote} force {force}", vote=vote, force=force)
    if vote == (1, 4):  # the oracle's own block sums, for the flip report
        q, k, _, kp, _ = case.oracle_inputs()
        ref = O.estimate_request(q[:, t0:t0 + case.chunk], k[:, t0:t0 + case.chunk], kp,
                                 case.wl.block_table[0], t0, cfg.H, cfg.Hkv, cfg.stride,
                                 cfg.block, O.default_estimation_scale(cfg.D, cfg.stride))
        check_block_sums(bs32, ref, cfg.block // cfg.stride, "q06b_4k chunk 3")
        record_flips(f"q06b_4k tau {tau} chunk {c} (vote (1, 2))", ref, mk, tau, cfg.Hkv, kbh,
                     O.gqa_vote(mk.astype(bool), cfg.Hkv, kbh))


@pytest.mark.parametrize("out_direct", [True, False])
def test_prefill_from_host_matches_device_resident_run(out_direct):
    """SequencePrefill.run_from_host (copies of later chunks overlapped with the
    compute of earlier ones; outputs written into the host buffers by the
    attention, or read back chunk by chunk) gives exactly the O and LSE of the
    run on device-resident inputs: a chunk that computed before its inputs or
    history pages landed, or a read-back before the chunk finished, would
    differ."""
    case = SequenceCase("q06b_4k")
    O_dev, L_dev, _ = case.run(0.9)
    pin = lambda t: t.cpu().pin_memory()
    host = {"q": pin(case.Q), "k": pin(case.K), "v": pin(case.V), "kpool": pin(case.KP),
            "vpool": pin(case.VP)}
    host["o"] = torch.zeros((case.cfg.H, case.L, case.cfg.D), dtype=torch.bfloat16).pin_memory()
    host["lse"] = torch.zeros((case.cfg.H, case.L), dtype=torch.float32).pin_memory()
    devb = {k: torch.full_like(t, 0, device=dev()) for k, t in host.items()}
    stream = torch.cuda.Stream(device=dev())
    h2d, d2h = torch.cuda.Stream(device=dev()), torch.cuda.Stream(device=dev())
    for _ in range(2):  # twice: the second run reuses every buffer
        case.seq.run_from_host(host, devb, 0.9, stream, h2d, d2h, out_direct=out_direct)
    stream.synchronize()
    assert X.xattn_device_error() == 0
    assert np.array_equal(host["o"].float().numpy(), O_dev)
    assert np.array_equal(host["lse"].numpy(), L_dev)


@pytest.mark.parametrize("Hkv,D,Bk", [(8, 128, 128), (1, 64, 64)])
def test_store_kv_writes_each_chunk_block_to_its_page(Hkv, D, Bk):
    """xattn_store_kv on a two-request varlen chunk equals the oracle's store
    bit for bit: every chunk block lands on the page its position names in the
    block table; history pages and pages no block names keep their contents; a
    -1 entry records XATTN_EPAGE and leaves that block unwritten."""
    d = dev()
    rng = np.random.default_rng(7 + D)
    q_lens, kh_lens = [2 * Bk, 3 * Bk], [Bk, 0]
    tot = sum(q_lens)
    P = 12
    kc = rng.integers(0, 1 << 16, size=(Hkv, tot, D), dtype=np.uint16)
    vc = rng.integers(0, 1 << 16, size=(Hkv, tot, D), dtype=np.uint16)
    perm = rng.permutation(P).astype(np.int32)
    bt = np.full((2, 4), -1, dtype=np.int32)
    bt[0, :3] = perm[:3]           # block 0 is history: not written
    bt[1, :3] = perm[3:6]
    bt[1, 1] = -1                  # unallocated: recorded, skipped
    sentinel = np.uint16(0x7E7E)
    kp = np.full((P, Bk, Hkv, D), sentinel, dtype=np.uint16)
    vp = kp.copy()
    as_dev = lambda a: torch.from_numpy(a.view(np.int16)).to(d).view(torch.bfloat16)
    KC, VC, KP, VP = as_dev(kc), as_dev(vc), as_dev(kp), as_dev(vp)
    prob = X.Problem(8 * Hkv, Hkv, D, 8, Bk, q_lens, kh_lens, torch.from_numpy(bt).to(d), P)
    X.xattn_store_kv(prob, KC, VC, KP, VP)
    torch.cuda.synchronize()
    assert X.xattn_last_device_error() == -3  # XATTN_EPAGE
    want_k, want_v = kp, vp
    q0 = 0
    for r in range(2):  # the oracle's store, request after request
        q1 = q0 + q_lens[r]
        want_k = O.store_chunk(want_k, bt[r], kh_lens[r], kc[:, q0:q1])
        want_v = O.store_chunk(want_v, bt[r], kh_lens[r], vc[:, q0:q1])
        q0 = q1
    got_k = KP.view(torch.int16).cpu().numpy().view(np.uint16)
    got_v = VP.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got_k, want_k)
    assert np.array_equal(got_v, want_v)


@pytest.mark.parametrize("out_direct", [True, False])
def test_prefill_from_host_with_kv_store_matches_prefilled_pool(out_direct):
    """run_from_host(store_kv=True) copies only Q, K, V and builds the pools on
    the device, chunk by chunk, from the sequence's own keys and values (the
    outputs copied back, or written into the host buffers by the attention):
    its O and LSE equal those of the run on the prefilled pools, and the pools
    end equal to them.  The device pools start as NaN, so a history page read
    before it was stored would show."""
    case = SequenceCase("q06b_4k")
    O_dev, L_dev, _ = case.run(0.9)
    pin = lambda t: t.cpu().pin_memory()
    host = {"q": pin(case.Q), "k": pin(case.K), "v": pin(case.V)}
    host["o"] = torch.zeros((case.cfg.H, case.L, case.cfg.D), dtype=torch.bfloat16).pin_memory()
    host["lse"] = torch.zeros((case.cfg.H, case.L), dtype=torch.float32).pin_memory()
    devb = {k: torch.zeros_like(t, device=dev()) for k, t in host.items()}
    for name, ref in (("kpool", case.KP), ("vpool", case.VP)):
        devb[name] = torch.full_like(ref, float("nan"))
    stream = torch.cuda.Stream(device=dev())
    h2d, d2h = torch.cuda.Stream(device=dev()), torch.cuda.Stream(device=dev())
    for _ in range(2):
        case.seq.run_from_host(host, devb, 0.9, stream, h2d, d2h, store_kv=True,
                               out_direct=out_direct)
    stream.synchronize()
    assert X.xattn_device_error() == 0
    assert np.array_equal(host["o"].float().numpy(), O_dev)
    assert np.array_equal(host["lse"].numpy(), L_dev)
    assert torch.equal(devb["kpool"].view(torch.int16), case.KP.view(torch.int16))
    assert torch.equal(devb["vpool"].view(torch.int16), case.VP.view(torch.int16))


@pytest.mark.parametrize("H,Hkv,D,Bk,S", [(3, 1, 128, 128, 8), (2, 2, 64, 64, 8),
                                           (5, 5, 128, 128, 16)])
def test_odd_group_sizes_full_path(H, Hkv, D, Bk, S):
    """Query heads per KV head odd (3 and 1): the score GEMM takes its
    one-CTA-per-tile form (sibling heads pair up only for even groups).  One
    chunk with history in a permuted pool: every block sum of every head
    against the oracle, the selection against the oracle on the GPU's block
    sums, sampled attention rows against the oracle."""
    d = dev()
    rng = np.random.default_rng(500 + H * 10 + Hkv)
    lq, kh = 4 * Bk, 6 * Bk
    P = kh // Bk + 3
    q = I.bf16_round(rng.standard_normal((H, lq, D), dtype=np.float32))
    kc = I.bf16_round(rng.standard_normal((Hkv, lq, D), dtype=np.float32))
    vc = I.bf16_round(rng.standard_normal((Hkv, lq, D), dtype=np.float32))
    kp32 = rng.standard_normal((P, Bk, Hkv, D), dtype=np.float32)
    kp32[2, 5] *= 4.0  # a few peaked keys so the selection keeps part of the history
    kp32[4, 17] *= 4.0
    kp = I.bf16_round(kp32)
    vp = I.bf16_round(rng.standard_normal((P, Bk, Hkv, D), dtype=np.float32))
    bt = rng.permutation(P).astype(np.int32)[None, : kh // Bk].copy()
    prob = X.Problem(H, Hkv, D, S, Bk, [lq], [kh], torch.from_numpy(bt).to(d), P)
    bufs = RN.ChunkBuffers.for_problems([prob], d, with_mask=True)
    O_ = torch.empty((H, lq, D), dtype=torch.bfloat16, device=d)
    LSE = torch.empty((H, lq), dtype=torch.float32, device=d)
    tau = 0.9
    RN.prefill_chunk(prob, to_dev_bf16(q), to_dev_bf16(kc), to_dev_bf16(vc), to_dev_bf16(kp),
                     to_dev_bf16(vp), tau, bufs, O_, LSE)
    torch.cuda.synchronize()
    assert X.xattn_device_error() == 0
    f64 = lambda b: (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    qd, kcd, vcd, kpd, vpd = f64(q), f64(kc), f64(vc), f64(kp), f64(vp)
    kbh, qb = kh // Bk, lq // Bk
    bs = bufs.block_sums[: H * qb * (kbh + qb)].cpu().numpy().reshape(H, qb, kbh + qb)
    ref = O.estimate_request(qd, kcd, kpd, bt[0], kh, H, Hkv, S, Bk,
                             O.default_estimation_scale(D, S))
    check_block_sums(bs, ref, Bk // S, f"H={H} Hkv={Hkv}")
    mk = bufs.mask[: bs.size].cpu().numpy().reshape(bs.shape)
    record_flips(f"H={H} Hkv={Hkv} D={D} S={S} tau {tau}", ref, mk, tau, Hkv, kbh,
                 bufs.sel_idx[0, : int(bufs.n_sel[0].item())].cpu().numpy())
    sel, pages = check_selection(bs, mk, bufs.sel_idx[0].cpu().numpy(),
                                 bufs.sel_page[0].cpu().numpy(), int(bufs.n_sel[0].item()), tau,
                                 Hkv, kbh, bt[0], f"H={H} Hkv={Hkv}")
    rows = sorted({0, Bk - 1, Bk, lq - 1, *rng.integers(0, lq, 10).tolist()})
    o_ref, l_ref = O.attend_request(qd, kcd, vcd, kpd, vpd, pages, H, Hkv, 1 / math.sqrt(D),
                                    rows=rows)
    idx = np.asarray(rows)
    check_attention(O_.float().cpu().numpy()[:, idx], LSE.cpu().numpy()[:, idx], o_ref, l_ref,
                    f"H={H} Hkv={Hkv}")
