"""Host logic of SequencePrefill.run_from_host on the CPU: the cross-stream
order of the host-fed chunked prefill, checked with recording stand-ins for
CUDA streams and events ("XAttention Offload Stream Synchronization Fix",
修复方案: every consumer waits on the event of the copy it reads; "Task Plan:
Layerwise Offload Refactoring", Phase 1.2: a chunk's K/V stored into its
pages, the next chunk's history).

The library calls are replaced by recorders, so no kernel and no copy runs;
the test checks, on CUDA's happens-before order rebuilt from the log:

  * chunk c's estimate follows the host-to-device copies of its Q and K (and,
    with prefilled pools, of both pools when it has history);
  * its KV store and its attention follow the copy of its V;
  * with the store, the estimate of chunk c + 1 follows chunk c's store;
  * O and LSE copied to the host only after its attention, or, the other
    way, written by the attention straight into the host buffers;
  * the side streams start after the work already on the compute stream,
    and the returned event follows every attention, read-back and store.
"""
import pytest
import torch

import fake_streams as FS
from xattention_block_sparse_gb300 import build as B
from xattention_block_sparse_gb300 import runner as RN
from xattention_block_sparse_gb300 import xattn as X


class _Pool:
    """A device pool stand-in whose bulk copy is logged on the current stream."""

    def __init__(self, log, name):
        self.log, self.name = log, name

    def copy_(self, src, non_blocking=False):
        self.log.append(("copy", FS.CURRENT[0], (self.name, 0)))


@pytest.fixture(scope="module")
def built():
    B.build()
    X.load_library()


def _run(monkeypatch, store_kv, n_chunks=3, out_direct=False):
    log, _ = FS.install(monkeypatch)
    H, Hkv, D, S, Bk, chunk = 2, 1, 64, 8, 64, 64
    L = chunk * n_chunks
    bt = torch.arange(L // Bk, dtype=torch.int32)[None]
    seq = RN.SequencePrefill(H, Hkv, D, S, Bk, L, chunk, bt, L // Bk)
    chunk_of = {id(p): c for c, p in enumerate(seq.problems)}
    host = {n: torch.zeros(s) for n, s in (("q", (H, L, D)), ("k", (Hkv, L, D)),
                                           ("v", (Hkv, L, D)), ("o", (H, L, D)), ("lse", (H, L)))}
    dev = {n: torch.zeros_like(t) for n, t in host.items()}
    dev["kpool"], dev["vpool"] = _Pool(log, "kpool"), _Pool(log, "vpool")
    if not store_kv:
        host["kpool"], host["vpool"] = object(), object()
    names = {id(t): n for n, t in list(host.items()) + list(dev.items())}

    def copy_window(dst, src, t0, t1, stream=None):
        assert t1 - t0 == chunk
        log.append(("copy", stream, (names[id(dst)], t0 // chunk)))

    outputs = {}

    def rec(kind):
        def f(p, *a, **k):
            stream = a[-1] if a else k.get("stream")
            log.append((kind, stream, chunk_of[id(p)]))
            if kind == "attend":  # o, lse come before the stream
                outputs[chunk_of[id(p)]] = tuple(names[id(t._base)] + ":" + (
                    "host" if t._base is host[n] else "dev") for t, n in zip(a[-3:-1], ("o", "lse")))
        return f

    monkeypatch.setattr(X, "copy_window_async", copy_window)
    for kind, fn in (("estimate", "xattn_estimate"), ("estimate", "xattn_estimate_seq"),
                     ("select", "xattn_select"),
                     ("attend", "bsa_chunk_attention"), ("store", "xattn_store_kv")):
        monkeypatch.setattr(X, fn, rec(kind))
    compute, h2d, d2h = (FS.Stream(log, n) for n in ("compute", "h2d", "d2h"))
    log.append(("earlier work", compute, None))
    back = seq.run_from_host(host, dev, 0.9, compute, h2d, d2h, store_kv=store_kv,
                             out_direct=out_direct)
    return log, back, (compute, h2d, d2h), n_chunks, outputs


def _index(log, kind, payload):
    hits = [i for i, op in enumerate(log) if op[0] == kind and op[2] == payload]
    assert len(hits) == 1, (kind, payload, hits)
    return hits[0]


@pytest.mark.parametrize("out_direct", [True, False])
@pytest.mark.parametrize("store_kv", [True, False])
def test_host_fed_prefill_orders_every_consumer_after_its_copy(built, monkeypatch, store_kv,
                                                               out_direct):
    log, back, (compute, h2d, side), n, outputs = _run(monkeypatch, store_kv,
                                                       out_direct=out_direct)
    before = FS.happens_before(log)
    end = FS.record_index(log, back)
    for c in range(n):
        est, att = _index(log, "estimate", c), _index(log, "attend", c)
        assert log[est][1] is compute and log[att][1] is compute
        for name in ("q", "k"):
            assert before(_index(log, "copy", (name, c)), est)
        # the estimate reads the keys of the whole prefix in token order
        for c2 in range(c):
            assert before(_index(log, "copy", ("k", c2)), est)
        assert before(_index(log, "copy", ("v", c)), att)
        assert before(est, _index(log, "select", c)) and before(_index(log, "select", c), att)
        assert before(att, end)
        if out_direct:
            assert outputs[c] == ("o:host", "lse:host")
            assert not any(op[0] == "copy" and op[2] == (name, c) for op in log
                           for name in ("o", "lse"))
        else:
            assert outputs[c] == ("o:dev", "lse:dev")
            for name in ("o", "lse"):
                rb = _index(log, "copy", (name, c))
                assert log[rb][1] is side and before(att, rb) and before(rb, end)
        if store_kv:
            st = _index(log, "store", c)
            assert log[st][1] is compute
            assert before(_index(log, "copy", ("v", c)), st) and before(st, att)
            if c + 1 < n:
                assert before(st, _index(log, "estimate", c + 1))
        elif c > 0:
            for pool in ("kpool", "vpool"):
                assert before(_index(log, "copy", (pool, 0)), est)
    assert any(op[0] == "store" for op in log) == store_kv
    first = _index(log, "earlier work", None)
    for s in (h2d, side):
        ops = [i for i, op in enumerate(log) if op[1] is s and op[0] != "record"]
        assert all(before(first, i) for i in ops)


def test_estimate_does_not_wait_for_its_v(built, monkeypatch):
    """Q and K are all the estimate reads: its wait ends at the K copy, so the
    V copy of the same chunk can still be in flight (the copies are issued
    Q, K, V)."""
    log, _, _, n, _ = _run(monkeypatch, True)
    before = FS.happens_before(log)
    for c in range(n):
        assert not before(_index(log, "copy", ("v", c)), _index(log, "estimate", c))


def test_a_missing_wait_is_caught(built, monkeypatch):
    """The check has teeth: without the compute stream's waits, chunk 1's
    estimate no longer follows its copies."""
    log, _, (compute, _, _), _, _ = _run(monkeypatch, True)
    log2 = [op for op in log if not (op[0] == "wait" and op[1] is compute)]
    before = FS.happens_before(log2)
    assert not before(_index(log2, "copy", ("k", 1)), _index(log2, "estimate", 1))


def test_pipelined_prefills_overlap_copies_and_reuse_buffers_in_order(built, monkeypatch):
    """HostFedPipeline, three prefills through two device buffer sets: the
    second prefill's inputs may cross while the first one computes (no order
    between them), the third one's inputs overwrite the first one's set only
    after the first one's last attention, and its outputs only after the first
    one's last read-back; within every prefill, each chunk still follows the
    copies it reads, and the prefills' compute stays in order."""
    log, _ = FS.install(monkeypatch)
    H, Hkv, D, S, Bk, chunk, n = 2, 1, 64, 8, 64, 64, 3
    L = chunk * n
    bt = torch.arange(L // Bk, dtype=torch.int32)[None]
    seq = RN.SequencePrefill(H, Hkv, D, S, Bk, L, chunk, bt, L // Bk)
    chunk_of = {id(p): c for c, p in enumerate(seq.problems)}
    host = {nm: torch.zeros(s) for nm, s in (("q", (H, L, D)), ("k", (Hkv, L, D)),
                                             ("v", (Hkv, L, D)), ("o", (H, L, D)),
                                             ("lse", (H, L)))}
    sets = [{nm: torch.zeros_like(t) for nm, t in host.items()} for _ in range(2)]
    for st in sets:
        st["kpool"], st["vpool"] = _Pool(log, "kpool"), _Pool(log, "vpool")
    names = {id(t): nm for nm, t in host.items()}
    for i, st in enumerate(sets):
        names.update({id(t): f"{nm}{i}" for nm, t in st.items() if torch.is_tensor(t)})
    current = [0]  # the prefill being enqueued

    def copy_window(dst, src, t0, t1, stream=None):
        nm = names[id(dst)] if dst is not host.get("o") and dst is not host.get("lse") \
            else names[id(src)] + ">host"
        log.append(("copy", stream, (current[0], nm, t0 // chunk)))

    def rec(kind):
        def f(p, *a, **k):
            stream = a[-1] if a else k.get("stream")
            log.append((kind, stream, (current[0], chunk_of[id(p)])))
        return f

    monkeypatch.setattr(X, "copy_window_async", copy_window)
    for kind, fn in (("estimate", "xattn_estimate_seq"), ("select", "xattn_select"),
                     ("attend", "bsa_chunk_attention"), ("store", "xattn_store_kv")):
        monkeypatch.setattr(X, fn, rec(kind))
    compute, h2d, d2h = (FS.Stream(log, nm) for nm in ("compute", "h2d", "d2h"))
    pipe = RN.HostFedPipeline(seq, sets, compute, h2d, d2h, store_kv=True)
    for i in range(3):
        current[0] = i
        pipe.submit(host, 0.9)
    before = FS.happens_before(log)
    idx = lambda kind, payload: _index(log, kind, payload)
    s = lambda i: i % 2
    for i in range(3):
        for c in range(n):
            est, att = idx("estimate", (i, c)), idx("attend", (i, c))
            assert before(idx("copy", (i, f"k{s(i)}", c)), est)
            assert before(idx("copy", (i, f"q{s(i)}", c)), est)
            assert before(idx("copy", (i, f"v{s(i)}", c)), att)
            assert before(att, idx("copy", (i, f"o{s(i)}>host", c)))
    # early waits: chunk c + 1's keys are waited for before chunk c's attention
    for i in range(3):
        for c in range(n - 1):
            assert before(idx("copy", (i, f"k{s(i)}", c + 1)), idx("attend", (i, c)))
    # consecutive prefills: compute in order, copies free to overlap
    assert before(idx("attend", (0, n - 1)), idx("estimate", (1, 0)))
    assert not before(idx("attend", (0, 0)), idx("copy", (1, "q1", 0)))
    assert not before(idx("copy", (0, "o0>host", n - 1)), idx("estimate", (1, 0)))
    # the third prefill reuses set 0: inputs after the first one's compute,
    # outputs after its read-back
    assert before(idx("attend", (0, n - 1)), idx("copy", (2, "q0", 0)))
    assert before(idx("copy", (0, "o0>host", n - 1)), idx("attend", (2, 0)))
    assert before(idx("copy", (0, "lse0>host", n - 1)), idx("attend", (2, 0)))


def test_pipeline_refuses_shared_pools_copied_from_the_host(built, monkeypatch):
    """Pools copied in from the host by every prefill cannot be shared by the
    two buffer sets: the next prefill's copy would overwrite what the current
    one reads."""
    FS.install(monkeypatch)
    H, Hkv, D, S, Bk, chunk = 2, 1, 64, 8, 64, 64
    bt = torch.arange(2, dtype=torch.int32)[None]
    seq = RN.SequencePrefill(H, Hkv, D, S, Bk, 2 * chunk, chunk, bt, 2)
    pool = torch.zeros(1)
    sets = [{"kpool": pool, "vpool": pool}, {"kpool": pool, "vpool": pool}]
    streams = [FS.Stream([], nm) for nm in ("c", "h", "d")]
    with pytest.raises(ValueError):
        RN.HostFedPipeline(seq, sets, *streams, store_kv=False)
    RN.HostFedPipeline(seq, sets, *streams, store_kv=True)  # built on the device: fine
