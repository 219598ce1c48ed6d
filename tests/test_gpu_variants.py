"""GPU parity of the library's variants of the chunk path, through the C-ABI.

* xattn_estimate_seq (keys in token order) against xattn_estimate (keys from
  the pool pages): the same block sums bit for bit, for head-major and
  token-major key layouts, a chunked sequence and the varlen batch.
* k_cur / v_cur given as a [tokens, Hkv, D] view (kv_token_stride): the
  same outputs as the packed [Hkv, tokens, D] copy.
* one block set per KV head (xattn_select_per_kv_head ->
  bsa_chunk_attention_per_kv_head): the selection bit-exact against the
  oracle's per-KV-head selection on the GPU's block sums, the attention
  within the usual bands of the oracle over each KV head's own pages.
"""
import math

import numpy as np
import pytest
import torch

from oracle import xattn_oracle as O
from xattention_block_sparse_gb300 import inputs as I
from xattention_block_sparse_gb300 import runner as RN
from xattention_block_sparse_gb300 import xattn as X

from gpu_common import SequenceCase, check_attention, check_block_sums, dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _estimate_both(prob, Q, Kc, KP, k_seq, starts, hs, ts, scale):
    bufs = RN.ChunkBuffers.for_problems([prob], dev())
    n = X.xattn_block_sums_count(prob)
    X.xattn_estimate(prob, Q, Kc, KP, scale, bufs.workspace, bufs.block_sums)
    a = bufs.block_sums[:n].clone()
    bufs.block_sums.fill_(float("nan"))
    X.xattn_estimate_seq(prob, Q, k_seq, starts, scale, bufs.workspace, bufs.block_sums,
                         head_stride=hs, token_stride=ts)
    b = bufs.block_sums[:n].clone()
    torch.cuda.synchronize()
    assert X.xattn_device_error() == 0
    return a, b


@pytest.mark.parametrize("name", ["tiny", "q06b_4k"])
def test_estimate_seq_equals_paged_estimate_every_chunk(name):
    case = SequenceCase(name)
    cfg = case.cfg
    scale = RN.estimation_scale(cfg.D, cfg.stride)
    Kt = case.K.permute(1, 0, 2).contiguous()   # [L, Hkv, D]: token-major keys
    for c in range(case.L // case.chunk):
        p, t0 = case.seq.problems[c], c * case.chunk
        a, b = _estimate_both(p, case.Q[:, t0:], case.K[:, t0:], case.KP, case.K, [0],
                              case.K.stride(0), 0, scale)
        assert torch.equal(a, b), f"{name} chunk {c}: head-major keys"
        _, b2 = _estimate_both(p, case.Q[:, t0:], case.K[:, t0:], case.KP, Kt, [0],
                               cfg.D, cfg.Hkv * cfg.D, scale)
        assert torch.equal(a, b2), f"{name} chunk {c}: token-major keys"


def test_estimate_seq_equals_paged_estimate_varlen():
    """Three requests (history 0, 16384, 65536 tokens): each request's keys,
    history then chunk, are laid one after another in a [Hkv, tokens, D]
    buffer with a gap between requests."""
    wl = I.make_workload("varlen")
    cfg, call = wl.cfg, wl.calls[0]
    d = dev()
    Q, Kc = to_dev_bf16(wl.q_bits), to_dev_bf16(wl.k_bits)
    KP = to_dev_bf16(wl.kpool_bits)
    BT = torch.from_numpy(wl.block_table).to(d)
    prob = X.Problem(cfg.H, cfg.Hkv, cfg.D, cfg.stride, cfg.block, call.q_lens, call.kh_lens, BT,
                     KP.shape[0])
    parts, starts, pos = [], [], 0
    for r in range(call.B):
        nh = call.kh_lens[r] // cfg.block
        hist = KP[BT[r, :nh].long()].permute(2, 0, 1, 3).reshape(cfg.Hkv, -1, cfg.D)
        q0, q1 = int(call.cu_q[r]), int(call.cu_q[r + 1])
        gap = torch.zeros((cfg.Hkv, 3 * cfg.stride, cfg.D), dtype=torch.bfloat16, device=d)
        parts += [gap, hist, Kc[:, q0:q1]]
        pos += gap.shape[1]
        starts.append(pos)
        pos += hist.shape[1] + (q1 - q0)
    kseq = torch.cat(parts, dim=1).contiguous()
    a, b = _estimate_both(prob, Q, Kc, KP, kseq, starts, kseq.stride(0), 0,
                          RN.estimation_scale(cfg.D, cfg.stride))
    assert torch.equal(a, b)


def test_token_major_current_chunk_matches_packed():
    """k_cur / v_cur as [tokens, Hkv, D] views (kv_head_stride = D,
    kv_token_stride = Hkv * D) give exactly the block sums, selection, O and
    LSE of the packed [Hkv, tokens, D] copies, and xattn_store_kv writes the
    same pages from them."""
    case = SequenceCase("q06b_4k")
    cfg = case.cfg
    c, t0 = 2, 2 * case.chunk
    Kt = case.K.permute(1, 0, 2).contiguous()
    Vt = case.V.permute(1, 0, 2).contiguous()
    res = []
    for tm in (False, True):
        if tm:
            p = X.Problem(cfg.H, cfg.Hkv, cfg.D, cfg.stride, cfg.block, [case.chunk], [t0],
                          case.BT, case.KP.shape[0], q_head_stride=case.L * cfg.D,
                          kv_head_stride=cfg.D, lse_head_stride=case.L,
                          kv_token_stride=cfg.Hkv * cfg.D)
            kc, vc = Kt[t0:], Vt[t0:]
        else:
            p = case.seq.problems[c]
            kc, vc = case.K[:, t0:], case.V[:, t0:]
        bufs = RN.ChunkBuffers.for_problems([p], dev(), with_mask=True)
        O_ = torch.zeros((cfg.H, case.L, cfg.D), dtype=torch.bfloat16, device=dev())
        LSE = torch.zeros((cfg.H, case.L), dtype=torch.float32, device=dev())
        RN.prefill_chunk(p, case.Q[:, t0:], kc, vc, case.KP, case.VP, 0.9, bufs, O_[:, t0:],
                         LSE[:, t0:])
        kp, vp = torch.zeros_like(case.KP), torch.zeros_like(case.VP)
        X.xattn_store_kv(p, kc, vc, kp, vp)
        torch.cuda.synchronize()
        assert X.xattn_device_error() == 0
        n = int(bufs.n_sel[0].item())
        res.append((bufs.block_sums.clone(), bufs.sel_page[0, :n].clone(), O_, LSE, kp, vp))
    for x, y in zip(res[0], res[1]):
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y)


def _per_kv_case(case, c, tau, vote=(1, 2)):
    """Chunk c of a SequenceCase with one block set per KV head: returns the
    GPU's block sums, mask, per-KV-head selection, O and LSE."""
    cfg = case.cfg
    p, t0 = case.seq.problems[c], c * case.chunk
    bufs = RN.ChunkBuffers.for_problems([p], dev(), with_mask=True)
    W = p.bt_stride
    bufs.sel_idx = torch.full((cfg.Hkv, W), -7, dtype=torch.int32, device=dev())
    bufs.sel_page = torch.full((cfg.Hkv, W), -7, dtype=torch.int32, device=dev())
    bufs.n_sel = torch.full((cfg.Hkv,), -7, dtype=torch.int32, device=dev())
    O_ = torch.zeros((cfg.H, case.L, cfg.D), dtype=torch.bfloat16, device=dev())
    LSE = torch.zeros((cfg.H, case.L), dtype=torch.float32, device=dev())
    RN.estimate_select(p, case.Q[:, t0:], case.K[:, t0:], case.KP, tau, bufs,
                       k_seq=case.seq.key_seq(case.K), per_kv_head=True)
    if vote != (1, 2):  # re-select with another ratio over the same block sums
        X.xattn_select_per_kv_head(p, bufs.block_sums, tau, bufs.workspace, bufs.mask,
                                   bufs.sel_idx, bufs.sel_page, bufs.n_sel, vote=vote)
    RN.attend(p, case.Q[:, t0:], case.K[:, t0:], case.V[:, t0:], case.KP, case.VP, bufs,
              O_[:, t0:], LSE[:, t0:], per_kv_head=True)
    torch.cuda.synchronize()
    assert X.xattn_device_error() == 0
    n = X.xattn_block_sums_count(p)
    kbh, qb = t0 // cfg.block, case.chunk // cfg.block
    bs = bufs.block_sums[:n].cpu().numpy().reshape(cfg.H, qb, kbh + qb)
    mk = bufs.mask[:n].cpu().numpy().reshape(bs.shape).astype(bool)
    sel = [bufs.sel_idx[k, :int(bufs.n_sel[k])].cpu().numpy() for k in range(cfg.Hkv)]
    pages = [bufs.sel_page[k, :int(bufs.n_sel[k])].cpu().numpy() for k in range(cfg.Hkv)]
    return bs, mk, sel, pages, O_.float().cpu().numpy(), LSE.cpu().numpy()


@pytest.mark.parametrize("tau,vote", [(0.9, (1, 2)), (0.6, (1, 2)), (0.6, (0, 1))])
def test_per_kv_head_selection_and_attention_q06b_4k(tau, vote):
    case = SequenceCase("q06b_4k")
    cfg = case.cfg
    q, k, v, kp, vp = case.oracle_inputs()
    bt_row = case.wl.block_table[0]
    rng = np.random.default_rng(11)
    for c in (1, 3):
        t0, t1 = c * case.chunk, (c + 1) * case.chunk
        kbh = t0 // cfg.block
        bs, mk, sel, pages, Og, Lg = _per_kv_case(case, c, tau, vote)
        # threshold masks and the per-KV-head vote against the oracle on the GPU's sums
        want_mask = O.threshold_select(bs, tau)
        assert np.array_equal(want_mask, mk), f"chunk {c}: mask"
        want = O.per_kv_head_select(want_mask, cfg.Hkv, kbh, vote=vote)
        for kvh in range(cfg.Hkv):
            assert np.array_equal(sel[kvh], want[kvh]), f"chunk {c} kv {kvh}: ids"
            assert np.array_equal(pages[kvh], bt_row[want[kvh]]), f"chunk {c} kv {kvh}: pages"
        # attention of every KV head's group over its own pages
        rows = sorted({0, case.chunk - 1, *rng.integers(0, case.chunk, 12).tolist()})
        o_ref, l_ref = O.attend_request_per_kv(q[:, t0:t1], k[:, t0:t1], v[:, t0:t1], kp, vp,
                                               [bt_row[w] for w in want], cfg.H, cfg.Hkv,
                                               1 / math.sqrt(cfg.D), rows=rows)
        idx = t0 + np.asarray(rows)
        check_attention(Og[:, idx], Lg[:, idx], o_ref, l_ref, f"chunk {c}")


def test_per_kv_head_varlen():
    """The varlen batch with a selection per KV head: three requests x eight KV
    heads run as 24 groups in one attention launch."""
    wl = I.make_workload("varlen")
    cfg, call = wl.cfg, wl.calls[0]
    d = dev()
    Q, K, V = to_dev_bf16(wl.q_bits), to_dev_bf16(wl.k_bits), to_dev_bf16(wl.v_bits)
    KP, VP = to_dev_bf16(wl.kpool_bits), to_dev_bf16(wl.vpool_bits)
    BT = torch.from_numpy(wl.block_table).to(d)
    prob = X.Problem(cfg.H, cfg.Hkv, cfg.D, cfg.stride, cfg.block, call.q_lens, call.kh_lens, BT,
                     KP.shape[0])
    bufs = RN.ChunkBuffers.for_problems([prob], d, with_mask=True)
    W = prob.bt_stride
    bufs.sel_idx = torch.full((call.B, cfg.Hkv, W), -7, dtype=torch.int32, device=d)
    bufs.sel_page = torch.full((call.B, cfg.Hkv, W), -7, dtype=torch.int32, device=d)
    bufs.n_sel = torch.full((call.B, cfg.Hkv), -7, dtype=torch.int32, device=d)
    tot = sum(call.q_lens)
    O_ = torch.empty((cfg.H, tot, cfg.D), dtype=torch.bfloat16, device=d)
    LSE = torch.empty((cfg.H, tot), dtype=torch.float32, device=d)
    tau = 0.6
    RN.prefill_chunk(prob, Q, K, V, KP, VP, tau, bufs, O_, LSE, per_kv_head=True)
    torch.cuda.synchronize()
    assert X.xattn_device_error() == 0
    q, k, v = wl.f64("q"), wl.f64("k"), wl.f64("v")
    kp, vp = wl.f64("kpool"), wl.f64("vpool")
    bs_all, mask_all = bufs.block_sums.cpu().numpy(), bufs.mask.cpu().numpy()
    sel_all, page_all = bufs.sel_idx.cpu().numpy(), bufs.sel_page.cpu().numpy()
    nsel = bufs.n_sel.cpu().numpy()
    Og, Lg = O_.float().cpu().numpy(), LSE.cpu().numpy()
    rng = np.random.default_rng(3)
    for r in range(call.B):
        q0, q1 = int(call.cu_q[r]), int(call.cu_q[r + 1])
        kbh, qb = call.kh_lens[r] // cfg.block, (q1 - q0) // cfg.block
        off = X.xattn_block_sums_offset(prob, r)
        bs = bs_all[off:off + cfg.H * qb * (kbh + qb)].reshape(cfg.H, qb, kbh + qb)
        mk = mask_all[off:off + bs.size].reshape(bs.shape).astype(bool)
        want_mask = O.threshold_select(bs, tau)
        assert np.array_equal(want_mask, mk), f"request {r}: mask"
        want = O.per_kv_head_select(want_mask, cfg.Hkv, kbh)
        for kvh in range(cfg.Hkv):
            n = int(nsel[r, kvh])
            assert np.array_equal(sel_all[r, kvh, :n], want[kvh]), f"request {r} kv {kvh}"
            assert np.array_equal(page_all[r, kvh, :n], wl.block_table[r][want[kvh]])
        rows = sorted({0, q1 - q0 - 1, *rng.integers(0, q1 - q0, 8).tolist()})
        o_ref, l_ref = O.attend_request_per_kv(
            q[:, q0:q1], k[:, q0:q1], v[:, q0:q1], kp, vp,
            [wl.block_table[r][w] for w in want], cfg.H, cfg.Hkv, 1 / math.sqrt(cfg.D),
            rows=rows)
        idx = q0 + np.asarray(rows)
        check_attention(Og[:, idx], Lg[:, idx], o_ref, l_ref, f"request {r}")


def test_one_shot_estimate_matches_kv_chunked_estimation():
    """GPU-only mode against the offload mode ("XAttention Offload Stream
    Synchronization Fix", 测试结果, Density 对齐验证): the library estimates over
    the whole resident history in one launch; the offload path takes softmax
    statistics per KV chunk, merges them and then normalises (the oracle's
    block_sums_chunked, four KV chunks).  The two agree to the block-sum
    tolerance, and the selections made from them are compared (density and
    flips, for information) on the seeded 4K and sparse 32K-shaped inputs."""
    from gpu_common import FLIPS
    for name, c, L in (("q06b_4k", 3, None), ("q06b_32k_sparse", 1, 8192)):
        case = SequenceCase(name, L=L)
        cfg = case.cfg
        tau = 0.9
        _, _, cap = case.run(tau, capture=[c])
        q, k, _, kp, _ = case.oracle_inputs()
        t0, t1 = c * case.chunk, (c + 1) * case.chunk
        kbh, qb = t0 // cfg.block, case.chunk // cfg.block
        bs = cap[c]["bs"].reshape(cfg.H, qb, kbh + qb)
        scale = O.default_estimation_scale(cfg.D, cfg.stride)
        ncol = (t1) // cfg.stride
        cuts = np.linspace(0, ncol, 5).astype(int)
        chunks = [(int(a), int(b)) for a, b in zip(cuts[:-1], cuts[1:])]
        G = cfg.H // cfg.Hkv
        ref = []
        for h in range(cfg.H):
            hist = O.gather_history(kp, case.wl.block_table[0], t0, h // G)
            full, _ = O.block_sums_chunked(q[h, t0:t1], hist, k[h // G, t0:t1], cfg.stride,
                                           cfg.block, scale, chunks)
            ref.append(full)
        ref = np.stack(ref)
        check_block_sums(bs, ref, cfg.block // cfg.stride, f"{name} chunk {c}")
        chunked = O.select_request(ref.astype(np.float32), tau, cfg.Hkv, kbh,
                                   case.wl.block_table[0])[1]
        gpu = cap[c]["sel"][:cap[c]["n_sel"]]
        FLIPS.append((f"{name} chunk {c}: GPU one-shot density {len(gpu) / kbh:.4f} vs "
                      f"KV-chunked oracle {len(chunked) / kbh:.4f}",
                      int((O.threshold_select(ref.astype(np.float32), tau)
                           != cap[c]["mask"].reshape(bs.shape).astype(bool)).sum()),
                      int(bs.size), len(set(gpu.tolist()) ^ set(chunked.tolist()))))


def _sampled_ref(q, hist, kcur, S, Bk, scale, samples):
    """The library's rule: a request's history is sampled when its sampled
    columns, rounded up to 128, are fewer than its history's columns."""
    kbh = hist.shape[0] // Bk
    hc = -(-kbh * samples // 128) * 128
    if hc < hist.shape[0] // S:
        return O.sampled_block_sums_one_head(q, hist, kcur, S, Bk, scale, samples)
    return O.block_sums_one_head(q, hist, kcur, S, Bk, scale)


@pytest.mark.parametrize("samples", [4, 8])
def test_sampled_estimation_matches_oracle_q06b_4k(samples):
    """xattn_estimate_sampled against the oracle's sampled estimate (chunks 2
    and 3 sample their history; chunk 1's 8 blocks are estimated in full), and
    the selection from the sampled block sums bit-exact."""
    case = SequenceCase("q06b_4k")
    cfg = case.cfg
    q, k, _, kp, _ = case.oracle_inputs()
    scale = RN.estimation_scale(cfg.D, cfg.stride)
    br = cfg.block // cfg.stride
    G = cfg.H // cfg.Hkv
    for c in (1, 2, 3):
        p, t0 = case.seq.problems[c], c * case.chunk
        t1 = t0 + case.chunk
        b = case.seq.bufs
        X.xattn_estimate_sampled(p, case.Q[:, t0:], case.K, [0], samples, scale, b.workspace,
                                 b.block_sums)
        X.xattn_select(p, b.block_sums, 0.9, b.workspace, b.mask, b.sel_idx, b.sel_page,
                       b.n_sel)
        torch.cuda.synchronize()
        assert X.xattn_device_error() == 0
        kbh, qb = t0 // cfg.block, case.chunk // cfg.block
        n = X.xattn_block_sums_count(p)
        bs = b.block_sums[:n].cpu().numpy().reshape(cfg.H, qb, kbh + qb)
        ref = np.stack([_sampled_ref(q[h, t0:t1], k[h // G, :t0], k[h // G, t0:t1], cfg.stride,
                                     cfg.block, scale, samples) for h in range(cfg.H)])
        check_block_sums(bs, ref, br, f"samples {samples} chunk {c}")
        from gpu_common import check_selection
        check_selection(bs, b.mask[:n].cpu().numpy().reshape(bs.shape), b.sel_idx[0].cpu().numpy(),
                        b.sel_page[0].cpu().numpy(), int(b.n_sel[0].item()), 0.9, cfg.Hkv, kbh,
                        case.wl.block_table[0], f"samples {samples} chunk {c}")


def test_sampled_estimation_token_major_keys_and_varlen():
    """Stride 16 (Br = 8, half of each block sampled) with keys laid out
    [tokens, Hkv, D] as in a layer-ring slot, two requests whose key ranges
    start at block multiples with a gap between them."""
    d = dev()
    rng = np.random.default_rng(61)
    H, Hkv, D, S, Bk = 8, 2, 128, 16, 128
    q_lens, kh_lens = [512, 256], [20 * Bk, 36 * Bk]
    starts = [Bk, 2 * Bk + kh_lens[0] + q_lens[0]]
    tot_k = starts[1] + kh_lens[1] + q_lens[1]
    qq = I.bf16_round(rng.standard_normal((H, sum(q_lens), D), dtype=np.float32))
    kt = I.bf16_round(rng.standard_normal((tot_k, Hkv, D), dtype=np.float32))
    Q, KT = to_dev_bf16(qq), to_dev_bf16(kt)
    # (the estimate reads no block table; the problem still describes the pool)
    BT = torch.zeros((2, 40), dtype=torch.int32, device=d)
    prob = X.Problem(H, Hkv, D, S, Bk, q_lens, kh_lens, BT, 1)
    bufs = RN.ChunkBuffers.for_problems([prob], d)
    scale = RN.estimation_scale(D, S)
    X.xattn_estimate_sampled(prob, Q, KT, starts, 4, scale, bufs.workspace, bufs.block_sums,
                             head_stride=D, token_stride=Hkv * D)
    torch.cuda.synchronize()
    assert X.xattn_device_error() == 0
    f64 = lambda b: (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    qd, kd = f64(qq), f64(kt)
    bs_all = bufs.block_sums.cpu().numpy()
    G = H // Hkv
    q0 = 0
    for r in range(2):
        lq, kh, st = q_lens[r], kh_lens[r], starts[r]
        kbh, qb = kh // Bk, lq // Bk
        off = X.xattn_block_sums_offset(prob, r)
        bs = bs_all[off:off + H * qb * (kbh + qb)].reshape(H, qb, kbh + qb)
        ref = np.stack([_sampled_ref(qd[h, q0:q0 + lq], kd[st:st + kh, h // G],
                                     kd[st + kh:st + kh + lq, h // G], S, Bk, scale, 4)
                        for h in range(H)])
        check_block_sums(bs, ref, Bk // S, f"request {r}")
        q0 += lq


def test_chunk_captured_in_a_cuda_graph_replays_the_same_bits():
    """Every entry point of a chunk (estimate in token order, select, attend)
    enqueues only stream work after its host checks, so the chunk can be
    captured once in a CUDA graph and replayed: the replays give exactly the
    eager call's block sums, selection, O and LSE (the bench times its steps
    this way)."""
    case = SequenceCase("q06b_4k")
    cfg = case.cfg
    c, t0 = 3, 3 * case.chunk
    p = case.seq.problems[c]
    stream = torch.cuda.Stream(device=dev())

    def outputs():
        n = int(case.seq.bufs.n_sel[0].item())
        return (case.seq.bufs.block_sums.clone(), case.seq.bufs.sel_page[0, :n].clone(),
                O_[:, t0:].clone(), LSE[:, t0:].clone())

    O_ = torch.zeros((cfg.H, case.L, cfg.D), dtype=torch.bfloat16, device=dev())
    LSE = torch.zeros((cfg.H, case.L), dtype=torch.float32, device=dev())
    with torch.cuda.stream(stream):
        case.seq.run_chunk(c, case.Q, case.K, case.V, case.KP, case.VP, 0.9, O_, LSE, stream)
    torch.cuda.synchronize()
    want = outputs()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
        case.seq.run_chunk(c, case.Q, case.K, case.V, case.KP, case.VP, 0.9, O_, LSE, stream)
    for _ in range(2):
        O_.zero_()
        LSE.zero_()
        case.seq.bufs.block_sums.zero_()
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        assert X.xattn_device_error() == 0
        for a, b in zip(want, outputs()):
            assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                               b.view(torch.int16) if b.dtype == torch.bfloat16 else b)


def test_estimate_started_during_the_previous_attention_gives_the_same_bits():
    """A chunk's estimate may start while the previous chunk's attention is
    still finishing (it is launched as a programmatic dependent and waits for
    the attention only at its end).  The 32K-shaped sparse sequence (8K, two
    chunks; whole-unit and stream-K attention) and the 4K one run once with the
    host synchronising after every chunk -- no overlap possible -- and once
    back to back, eagerly and as one CUDA graph: the block sums, selections, O
    and LSE must be the same bits."""
    for name, L in (("q06b_4k", None), ("q06b_32k_sparse", 8192)):
        case = SequenceCase(name, L=L)
        cfg = case.cfg
        stream = torch.cuda.Stream(device=dev())
        runs = []
        for mode in ("synced", "back_to_back", "graph"):
            O_ = torch.zeros((cfg.H, case.L, cfg.D), dtype=torch.bfloat16, device=dev())
            LSE = torch.zeros((cfg.H, case.L), dtype=torch.float32, device=dev())
            sels = []

            def chunks():
                for c in range(len(case.seq.problems)):
                    case.seq.run_chunk(c, case.Q, case.K, case.V, case.KP, case.VP, 0.9, O_,
                                       LSE, stream)
                    if mode == "synced":
                        torch.cuda.synchronize()
                        n = int(case.seq.bufs.n_sel[0].item())
                        sels.append(case.seq.bufs.sel_page[0, :n].clone())

            if mode == "graph":
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                    chunks()
                O_.zero_()
                LSE.zero_()
                with torch.cuda.stream(stream):
                    g.replay()
            else:
                with torch.cuda.stream(stream):
                    chunks()
            torch.cuda.synchronize()
            assert X.xattn_device_error() == 0
            runs.append((O_.view(torch.int16).clone(), LSE.clone(),
                         case.seq.bufs.block_sums.clone(), sels))
        ref = runs[0]
        for other in runs[1:]:
            assert torch.equal(ref[0], other[0]), f"{name}: O differs"
            assert torch.equal(ref[1], other[1]), f"{name}: LSE differs"
            assert torch.equal(ref[2], other[2]), f"{name}: block sums differ"
        # the last chunk's selection of the back-to-back run equals the synced one
        n = int(case.seq.bufs.n_sel[0].item())
        assert torch.equal(case.seq.bufs.sel_page[0, :n], ref[3][-1])


def test_host_fed_prefill_replayed_from_a_cuda_graph():
    """The host-fed prefill (copies on two side streams, the KV store, the
    three calls per chunk, the read-back) captured once as a CUDA graph -- the
    way the bench's end-to-end leg times it -- and replayed: every replay moves
    the inputs in and the outputs out again, and the host O and LSE equal the
    device-resident run's."""
    case = SequenceCase("q06b_4k")
    O_dev, L_dev, _ = case.run(0.9)
    pin = lambda t: t.cpu().pin_memory()
    host = {"q": pin(case.Q), "k": pin(case.K), "v": pin(case.V)}
    host["o"] = torch.zeros((case.cfg.H, case.L, case.cfg.D), dtype=torch.bfloat16).pin_memory()
    host["lse"] = torch.zeros((case.cfg.H, case.L), dtype=torch.float32).pin_memory()
    devb = {k: torch.zeros_like(t, device=dev()) for k, t in host.items()}
    for name, ref in (("kpool", case.KP), ("vpool", case.VP)):
        devb[name] = torch.zeros_like(ref)
    stream = torch.cuda.Stream(device=dev())
    h2d, d2h = torch.cuda.Stream(device=dev()), torch.cuda.Stream(device=dev())
    case.seq.run_from_host(host, devb, 0.9, stream, h2d, d2h, store_kv=True)  # warm-up
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
        case.seq.run_from_host(host, devb, 0.9, stream, h2d, d2h, store_kv=True)
    torch.cuda.synchronize()
    for _ in range(2):
        host["o"].zero_()
        host["lse"].zero_()
        for name in ("q", "k", "v", "o", "lse", "kpool", "vpool"):
            devb[name].zero_()  # nothing may survive from the previous replay
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        assert X.xattn_device_error() == 0
        assert np.array_equal(host["o"].float().numpy(), O_dev)
        assert np.array_equal(host["lse"].numpy(), L_dev)


def test_attention_writes_pinned_host_outputs():
    """bsa_chunk_attention with o and lse in page-locked host memory (whole
    tensors, and windows of them at a token offset, as the host-fed prefill
    passes them) writes exactly the bits it writes into device buffers; the
    per-KV-head entry point too.  Pageable host memory is refused with
    XATTN_EINVAL before anything is launched."""
    import ctypes
    case = SequenceCase("q06b_4k")
    cfg, H, L, D = case.cfg, case.cfg.H, case.L, case.cfg.D
    # chunks 0 .. 2 on the device, then chunk 3's attention both ways
    seq, b = case.seq, case.seq.bufs
    O_d = torch.zeros((H, L, D), dtype=torch.bfloat16, device=dev())
    L_d = torch.zeros((H, L), dtype=torch.float32, device=dev())
    for c in range(4):
        seq.run_chunk(c, case.Q, case.K, case.V, case.KP, case.VP, 0.9, O_d, L_d, None)
    torch.cuda.synchronize()
    c = 3
    t0 = c * case.chunk
    p = seq.problems[c]
    scale = 1.0 / np.sqrt(D)
    O_h = torch.full((H, L, D), 7.0, dtype=torch.bfloat16).pin_memory()
    L_h = torch.full((H, L), 7.0, dtype=torch.float32).pin_memory()
    args = (p, case.Q[:, t0:], case.K[:, t0:], case.V[:, t0:], case.KP, case.VP, b.sel_page,
            b.n_sel, scale, b.workspace)
    X.bsa_chunk_attention(*args, O_h[:, t0:], L_h[:, t0:])
    torch.cuda.synchronize()
    assert X.xattn_device_error() == 0
    assert torch.equal(O_h[:, t0:].view(torch.int16), O_d[:, t0:].cpu().view(torch.int16))
    assert torch.equal(L_h[:, t0:], L_d[:, t0:].cpu())
    assert torch.all(O_h[:, :t0] == 7.0) and torch.all(L_h[:, :t0] == 7.0)  # nothing else
    # the per-KV-head entry point on the selection of every KV head
    sel_kv = b.sel_page.repeat_interleave(cfg.Hkv, 0)[None].reshape(1, cfg.Hkv, -1).contiguous()
    n_kv = b.n_sel.repeat_interleave(cfg.Hkv, 0)[None].reshape(1, cfg.Hkv).contiguous()
    O_h2 = torch.zeros_like(O_h).pin_memory()
    L_h2 = torch.zeros_like(L_h).pin_memory()
    O_d2, L_d2 = torch.zeros_like(O_d), torch.zeros_like(L_d)
    for o_, l_ in ((O_d2, L_d2), (O_h2, L_h2)):
        X.bsa_chunk_attention_per_kv_head(p, *args[1:6], sel_kv, n_kv, scale, b.workspace,
                                          o_[:, t0:], l_[:, t0:])
    torch.cuda.synchronize()
    assert X.xattn_device_error() == 0
    assert torch.equal(O_h2[:, t0:].view(torch.int16), O_d2[:, t0:].cpu().view(torch.int16))
    assert torch.equal(L_h2[:, t0:], L_d2[:, t0:].cpu())
    # pageable host memory: the binding refuses it, and so does the library
    pageable_o = torch.zeros((H, L, D), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        X.bsa_chunk_attention(*args, pageable_o, L_h)
    lib = X.load_library()
    vp = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.bsa_chunk_attention(p.ref(), vp(case.Q[:, t0:]), vp(case.K[:, t0:]),
                                 vp(case.V[:, t0:]), vp(case.KP), vp(case.VP), vp(b.sel_page),
                                 vp(b.n_sel), float(scale), vp(b.workspace),
                                 b.workspace.numel(), vp(pageable_o), vp(L_h),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == -1  # XATTN_EINVAL
    torch.cuda.synchronize()
    assert torch.all(pageable_o == 0)


def test_pipelined_host_fed_prefills_give_each_its_own_results():
    """HostFedPipeline: three prefills (inputs A, B, A; B's queries are A's with
    head_dim reversed) through two device buffer sets, the next one's copies
    overlapping the current one's compute, each into host outputs of its own:
    every one equals the device-resident run of its inputs, bit for bit --
    eagerly, and replayed from one CUDA graph of the three."""
    case = SequenceCase("q06b_4k")
    cfg, L = case.cfg, case.L
    Qb = case.Q.flip(-1).contiguous()
    refs = {}
    for tag, Q in (("A", case.Q), ("B", Qb)):
        O_ = torch.empty((cfg.H, L, cfg.D), dtype=torch.bfloat16, device=dev())
        LSE = torch.empty((cfg.H, L), dtype=torch.float32, device=dev())
        case.seq.run(Q, case.K, case.V, case.KP, case.VP, 0.9, O_, LSE)
        torch.cuda.synchronize()
        refs[tag] = (O_.cpu(), LSE.cpu())
    pin = lambda t: t.cpu().pin_memory()
    ins = {"A": {"q": pin(case.Q), "k": pin(case.K), "v": pin(case.V)},
           "B": {"q": pin(Qb), "k": pin(case.K), "v": pin(case.V)}}
    order = ["A", "B", "A"]
    hosts = []
    for tag in order:
        h = dict(ins[tag])
        h["o"] = torch.zeros((cfg.H, L, cfg.D), dtype=torch.bfloat16).pin_memory()
        h["lse"] = torch.zeros((cfg.H, L), dtype=torch.float32).pin_memory()
        hosts.append(h)
    sets = []
    for _ in range(2):
        d = {k: torch.zeros_like(ins["A"][k], device=dev()) for k in ("q", "k", "v")}
        d["o"] = torch.zeros((cfg.H, L, cfg.D), dtype=torch.bfloat16, device=dev())
        d["lse"] = torch.zeros((cfg.H, L), dtype=torch.float32, device=dev())
        sets.append(d)
    for name, ref in (("kpool", case.KP), ("vpool", case.VP)):
        pool = torch.full_like(ref, float("nan"))
        for d in sets:
            d[name] = pool
    stream = torch.cuda.Stream(device=dev())
    h2d, d2h = torch.cuda.Stream(device=dev()), torch.cuda.Stream(device=dev())

    def many():
        pipe = RN.HostFedPipeline(case.seq, sets, stream, h2d, d2h, store_kv=True)
        for h in hosts:
            pipe.submit(h, 0.9)
        pipe.join()

    def check():
        assert X.xattn_device_error() == 0
        for tag, h in zip(order, hosts):
            assert torch.equal(h["o"].view(torch.int16), refs[tag][0].view(torch.int16)), tag
            assert torch.equal(h["lse"], refs[tag][1]), tag

    with torch.cuda.stream(stream):
        many()
    stream.synchronize()
    check()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
        many()
    torch.cuda.synchronize()
    for h in hosts:
        h["o"].zero_()
        h["lse"].zero_()
    for d in sets:
        for k in ("q", "k", "v", "o", "lse"):
            d[k].zero_()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    check()
