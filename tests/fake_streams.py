"""Recording stand-ins for CUDA streams and events, for CPU tests of the host
code that orders work across streams.

``install(monkeypatch)`` replaces torch.cuda.Stream / Event / current_stream /
stream with objects that append every wait and record to one log, in issue
order; ``happens_before(ops)`` rebuilds the order CUDA gives those calls:
program order on each stream, and a wait on an event orders the waiting
stream after the work issued before that event's latest record.  Other
callers log their own operations as ("name", stream, payload) tuples into the
same list, which places them in that order too."""
import itertools

import torch

_ids = itertools.count()


class Stream:
    def __init__(self, log, name):
        self.log, self.name = log, name

    def wait_event(self, ev):
        self.log.append(("wait", self, ev))

    def wait_stream(self, other):
        ev = Event(self.log)
        ev.record(other)
        self.wait_event(ev)

    def __repr__(self):
        return f"<stream {self.name}>"


class Event:
    def __init__(self, log, enable_timing=False):
        self.log, self.id = log, next(_ids)

    def record(self, stream=None):
        self.log.append(("record", stream if stream is not None else CURRENT[0], self))


CURRENT = [None]


class _StreamCtx:
    def __init__(self, s):
        self.s = s

    def __enter__(self):
        self.prev, CURRENT[0] = CURRENT[0], self.s

    def __exit__(self, *a):
        CURRENT[0] = self.prev


def install(monkeypatch):
    """Patch torch.cuda's stream and event types; returns (log, default stream)."""
    log = []
    default = Stream(log, "default")
    CURRENT[0] = default
    monkeypatch.setattr(torch.cuda, "Stream", lambda device=None: Stream(log, f"s{next(_ids)}"))
    monkeypatch.setattr(torch.cuda, "Event", lambda enable_timing=False: Event(log))
    monkeypatch.setattr(torch.cuda, "current_stream", lambda device=None: default)
    monkeypatch.setattr(torch.cuda, "stream", _StreamCtx)
    return log, default


def happens_before(ops):
    """Returns before(a, b): does logged op a happen before logged op b?"""
    preds = [set() for _ in ops]
    last_on, last_record = {}, {}
    for i, (kind, s, x) in enumerate(ops):
        if s in last_on:
            preds[i].add(last_on[s])
        last_on[s] = i
        if kind == "record":
            last_record[x] = i
        elif kind == "wait" and x in last_record:
            preds[i].add(last_record[x])
    reach = []
    for i in range(len(ops)):
        r = set()
        for p in preds[i]:
            r.add(p)
            r |= reach[p]
        reach.append(r)
    return lambda a, b: a in reach[b]


def record_index(ops, ev):
    """Index of the latest record of event ev in the log."""
    return max(i for i, op in enumerate(ops) if op[0] == "record" and op[2] is ev)
