"""Host logic of the layer ring on the CPU: the event discipline of runner.LayerRing
and ring_prefill_chunk, checked with recording stand-ins for CUDA streams and
events ("Task Plan: Layerwise Offload Refactoring", Phase 4 ring schedule;
"XAttention Offload Stream Synchronization Fix", 修复方案 / Event 同步机制).

From the log of waits and records the test rebuilds CUDA's happens-before
order and checks:

  * the compute of layer l runs after the copy of layer l into its slot;
  * a slot is refilled only after the compute of the layer it held finished;
  * loads and computes come in the order of the ring schedule;
  * at each compute the slot holds that layer's pages (the copies run
    synchronously here, so the contents are those the schedule put there).

No kernel runs: the chunk's compute is replaced by a recorder.
"""
import pytest
import torch

import fake_streams as FS
from oracle import xattn_oracle as O
from xattention_block_sparse_gb300 import runner as RN


class _Layer:
    def __init__(self, l, P, Bk, Hkv, D, H, L):
        g = torch.Generator().manual_seed(l)
        self.k_host = torch.randn((P, Bk, Hkv, D), generator=g).to(torch.bfloat16)
        self.v_host = torch.randn((P, Bk, Hkv, D), generator=g).to(torch.bfloat16)
        self.q = torch.zeros((H, L, D), dtype=torch.bfloat16)


def _loads(ops, ring):
    """(layer, index of its start record, index of its ready record) per load."""
    return [(layer, FS.record_index(ops, start), FS.record_index(ops, ready))
            for layer, start, ready, _ in ring.log]


@pytest.mark.parametrize("num_layers,num_slots", [(8, 4), (5, 2), (3, 4)])
def test_ring_event_discipline(monkeypatch, num_layers, num_slots):
    log, _ = FS.install(monkeypatch)
    P, Bk, Hkv, D, H = 8, 4, 2, 2, 4
    chunk, c = 8, 2
    L = P * Bk
    n_load = (c * chunk + chunk) // Bk
    layers = [_Layer(l, P, Bk, Hkv, D, H, L) for l in range(num_layers)]
    ring = RN.LayerRing(num_slots, P, Bk, Hkv, D, "cpu")
    compute = FS.Stream(log, "compute")

    def fake_prefill(problem, q, kc, vc, kp, vp, tau, bufs, o, lse, stream=None, k_seq=None):
        l = len([op for op in log if op[0] == "compute"])
        assert torch.equal(kp[:n_load], layers[l].k_host[:n_load])   # the slot holds layer l
        assert torch.equal(vp[:n_load], layers[l].v_host[:n_load])
        assert stream is compute and FS.CURRENT[0] is compute
        log.append(("compute", stream, l))

    monkeypatch.setattr(RN, "prefill_chunk", fake_prefill)
    outs = [(torch.zeros((H, L, D)), torch.zeros((H, L))) for _ in layers]
    RN.ring_prefill_chunk(ring, layers, c, chunk, H, Hkv, D, 2, Bk, 0.9, None, None, outs,
                          compute)

    before = FS.happens_before(log)
    loads = _loads(log, ring)
    comp = {op[2]: i for i, op in enumerate(log) if op[0] == "compute"}
    assert sorted(comp) == list(range(num_layers))
    for layer, si, ri in loads:
        assert before(ri, comp[layer]), f"layer {layer} computed before its copy landed"
        prev = layer - num_slots
        if prev >= 0:
            assert before(comp[prev], si), f"slot of layer {prev} refilled before its compute"
    # issue order of loads and computes = the ring schedule of the task plan
    issued = sorted([(si, "load", layer) for layer, si, _ in loads] +
                    [(i, "compute", l) for l, i in comp.items()])
    want = [(k, l) for k, l, _ in O.ring_schedule(num_layers, num_slots)]
    assert [(k, l) for _, k, l in issued] == want
    assert [ring.slot(l) for l in range(num_layers)] == [O.ring_slot(l, num_slots)
                                                        for l in range(num_layers)]


def test_a_refill_without_the_done_wait_is_caught(monkeypatch):
    """The check above has teeth: drop the copy stream's wait on the slot's
    done event and a refill no longer follows the compute it overwrites."""
    log, _ = FS.install(monkeypatch)
    ring = RN.LayerRing(2, 4, 4, 1, 2, "cpu")
    monkeypatch.setattr(ring.copy_stream, "wait_event", lambda ev: None)
    compute = FS.Stream(log, "compute")
    layers = [_Layer(l, 4, 4, 1, 2, 1, 16) for l in range(3)]
    monkeypatch.setattr(RN, "prefill_chunk",
                        lambda *a, stream=None, **k: log.append(("compute", stream, None)))
    outs = [(torch.zeros((1, 16, 2)), torch.zeros((1, 16))) for _ in layers]
    RN.ring_prefill_chunk(ring, layers, 1, 4, 1, 1, 2, 2, 4, 0.9, None, None, outs, compute)
    before = FS.happens_before(log)
    comp0 = next(i for i, op in enumerate(log) if op[0] == "compute")
    layer, si, _ = _loads(log, ring)[2]
    assert layer == 2 and not before(comp0, si)


def test_reused_selection_estimates_once_per_chunk(monkeypatch):
    """With the selection shared across layers, layer 0 runs estimate + select +
    attention and every later layer only attention, on the same buffers (the
    sel_page / n_sel layer 0 wrote); the ring's order is unchanged."""
    log, _ = FS.install(monkeypatch)
    P, Bk, Hkv, D, H, chunk, c, nl = 8, 4, 1, 2, 2, 8, 1, 6
    layers = [_Layer(l, P, Bk, Hkv, D, H, P * Bk) for l in range(nl)]
    ring = RN.LayerRing(4, P, Bk, Hkv, D, "cpu")
    compute = FS.Stream(log, "compute")
    bufs = object()
    seen = []

    def full(problem, q, kc, vc, kp, vp, tau, b, o, lse, stream=None, k_seq=None):
        seen.append(b)
        log.append(("full", stream, len([op for op in log if op[0] in ("full", "attend")])))

    def attend_only(problem, q, kc, vc, kp, vp, b, o, lse, softmax_scale=None, stream=None):
        seen.append(b)
        log.append(("attend", stream, len([op for op in log if op[0] in ("full", "attend")])))

    monkeypatch.setattr(RN, "prefill_chunk", full)
    monkeypatch.setattr(RN, "attend", attend_only)
    outs = [(torch.zeros((H, P * Bk, D)), torch.zeros((H, P * Bk))) for _ in layers]
    RN.ring_prefill_chunk(ring, layers, c, chunk, H, Hkv, D, 2, Bk, 0.9, bufs, None, outs,
                          compute, reuse_selection=True)
    kinds = [(op[0], op[2]) for op in log if op[0] in ("full", "attend")]
    assert kinds == [("full", 0)] + [("attend", l) for l in range(1, nl)]
    assert all(b is bufs for b in seen)
    before = FS.happens_before(log)
    comp = {op[2]: i for i, op in enumerate(log) if op[0] in ("full", "attend")}
    for layer, si, ri in _loads(log, ring):
        assert before(ri, comp[layer])
        if layer >= 4:
            assert before(comp[layer - 4], si)
