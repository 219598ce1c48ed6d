"""Host logic of the layer ring on the CPU: the event discipline of runner.LayerRing
and ring_prefill_chunk, checked with recording stand-ins for CUDA streams and
events ("Task Plan: Layerwise Offload Refactoring", Phase 4 ring schedule;
"XAttention Offload Stream Synchronization Fix", 修复方案 / Event 同步机制).

The stand-ins log every stream wait and event record in issue order.  From the
log the test rebuilds the happens-before order CUDA gives those calls (program
order on each stream; a wait on an event orders the waiting stream after the
work before the event's latest record) and checks:

  * the compute of layer l runs after the copy of layer l into its slot;
  * a slot is refilled only after the compute of the layer it held finished;
  * loads and computes come in the order of the ring schedule;
  * at each compute the slot holds that layer's pages (the copies run
    synchronously here, so the contents are those the schedule put there).

No kernel runs: the chunk's compute is replaced by a recorder.
"""
import itertools

import pytest
import torch

from oracle import xattn_oracle as O
from xattention_block_sparse_gb300 import runner as RN

_ids = itertools.count()


class _Log:
    def __init__(self):
        self.ops = []          # (kind, stream, payload)


class _Stream:
    def __init__(self, log, name):
        self.log, self.name = log, name

    def wait_event(self, ev):
        self.log.ops.append(("wait", self, ev))

    def wait_stream(self, other):
        ev = _Event(self.log)
        ev.record(other)
        self.wait_event(ev)


class _Event:
    def __init__(self, log, enable_timing=False):
        self.log, self.id = log, next(_ids)

    def record(self, stream=None):
        self.log.ops.append(("record", stream if stream is not None else _current[0], self))


_current = [None]


class _StreamCtx:
    def __init__(self, s):
        self.s = s

    def __enter__(self):
        self.prev, _current[0] = _current[0], self.s

    def __exit__(self, *a):
        _current[0] = self.prev


class _Layer:
    def __init__(self, l, P, Bk, Hkv, D, H, L):
        g = torch.Generator().manual_seed(l)
        self.k_host = torch.randn((P, Bk, Hkv, D), generator=g).to(torch.bfloat16)
        self.v_host = torch.randn((P, Bk, Hkv, D), generator=g).to(torch.bfloat16)
        self.q = torch.zeros((H, L, D), dtype=torch.bfloat16)


def _happens_before(ops):
    """Edges of CUDA's order over the logged ops: program order per stream, and
    record -> wait for the latest record of the waited event before the wait."""
    n = len(ops)
    preds = [set() for _ in range(n)]
    last_on = {}
    last_record = {}
    for i, (kind, s, x) in enumerate(ops):
        if s in last_on:
            preds[i].add(last_on[s])
        last_on[s] = i
        if kind == "record":
            last_record[x] = i
        elif kind == "wait" and x in last_record:
            preds[i].add(last_record[x])
    reach = []
    for i in range(n):
        r = set()
        for p in preds[i]:
            r.add(p)
            r |= reach[p]
        reach.append(r)
    return lambda a, b: a in reach[b]          # does op a happen before op b?


@pytest.mark.parametrize("num_layers,num_slots", [(8, 4), (5, 2), (3, 4)])
def test_ring_event_discipline(monkeypatch, num_layers, num_slots):
    log = _Log()
    monkeypatch.setattr(torch.cuda, "Stream", lambda device=None: _Stream(log, f"s{next(_ids)}"))
    monkeypatch.setattr(torch.cuda, "Event", lambda enable_timing=False: _Event(log))
    default = _Stream(log, "default")
    monkeypatch.setattr(torch.cuda, "current_stream", lambda device=None: default)
    monkeypatch.setattr(torch.cuda, "stream", _StreamCtx)

    P, Bk, Hkv, D, H = 8, 4, 2, 2, 4
    chunk, c = 8, 2
    L = P * Bk
    n_load = (c * chunk + chunk) // Bk
    layers = [_Layer(l, P, Bk, Hkv, D, H, L) for l in range(num_layers)]
    ring = RN.LayerRing(num_slots, P, Bk, Hkv, D, "cpu")
    compute = _Stream(log, "compute")

    def fake_prefill(problem, q, kc, vc, kp, vp, tau, bufs, o, lse, stream=None):
        l = len([op for op in log.ops if op[0] == "compute"])
        assert torch.equal(kp[:n_load], layers[l].k_host[:n_load])   # the slot holds layer l
        assert torch.equal(vp[:n_load], layers[l].v_host[:n_load])
        assert stream is compute and _current[0] is compute
        log.ops.append(("compute", stream, l))

    monkeypatch.setattr(RN, "prefill_chunk", fake_prefill)
    outs = [(torch.zeros((H, L, D)), torch.zeros((H, L))) for _ in layers]
    RN.ring_prefill_chunk(ring, layers, c, chunk, H, Hkv, D, 2, Bk, 0.9, None, None, outs,
                          compute)

    ops = log.ops
    before = _happens_before(ops)
    # each load is bracketed by two records on the copy stream: start, ready
    loads = []                                    # (layer, start index, ready index)
    for layer, start, ready, _ in ring.log:
        si = max(i for i, op in enumerate(ops) if op[0] == "record" and op[2] is start)
        ri = max(i for i, op in enumerate(ops) if op[0] == "record" and op[2] is ready)
        loads.append((layer, si, ri))
    comp = {op[2]: i for i, op in enumerate(ops) if op[0] == "compute"}
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
    log = _Log()
    monkeypatch.setattr(torch.cuda, "Stream", lambda device=None: _Stream(log, f"s{next(_ids)}"))
    monkeypatch.setattr(torch.cuda, "Event", lambda enable_timing=False: _Event(log))
    default = _Stream(log, "default")
    monkeypatch.setattr(torch.cuda, "current_stream", lambda device=None: default)
    monkeypatch.setattr(torch.cuda, "stream", _StreamCtx)
    ring = RN.LayerRing(2, 4, 4, 1, 2, "cpu")
    monkeypatch.setattr(ring.copy_stream, "wait_event", lambda ev: None)
    compute = _Stream(log, "compute")
    layers = [_Layer(l, 4, 4, 1, 2, 1, 16) for l in range(3)]
    monkeypatch.setattr(RN, "prefill_chunk",
                        lambda *a, stream=None, **k: log.ops.append(("compute", stream, None)))
    outs = [(torch.zeros((1, 16, 2)), torch.zeros((1, 16))) for _ in layers]
    RN.ring_prefill_chunk(ring, layers, 1, 4, 1, 1, 2, 2, 4, 0.9, None, None, outs, compute)
    before = _happens_before(log.ops)
    comp0 = next(i for i, op in enumerate(log.ops) if op[0] == "compute")
    layer2_start = ring.log[2][1]
    si = max(i for i, op in enumerate(log.ops) if op[0] == "record" and op[2] is layer2_start)
    assert ring.log[2][0] == 2 and not before(comp0, si)
