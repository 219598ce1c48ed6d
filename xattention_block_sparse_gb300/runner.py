"""Chunked-prefill driver over the libxattn entry points.

Per chunk: xattn_estimate -> xattn_select -> bsa_chunk_attention, all on one
stream ("XAttention BSA Policy 设计文档": select_blocks then
compute_chunked_prefill; "XAttention Offload Stream Synchronization Fix":
estimation, selection and attention share the compute stream).  torch only
provides device memory and the stream; every step runs in libxattn kernels.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

from . import xattn as X


@dataclass
class ChunkBuffers:
    """Scratch and outputs of one chunk call, sized for the largest call."""
    workspace: torch.Tensor
    block_sums: torch.Tensor
    mask: torch.Tensor | None
    sel_idx: torch.Tensor
    sel_page: torch.Tensor
    n_sel: torch.Tensor

    @staticmethod
    def for_problems(problems, device, with_mask=False):
        ws = max(X.xattn_workspace_size(p) for p in problems)
        nbs = max(X.xattn_block_sums_count(p) for p in problems)
        B = max(p.B for p in problems)
        bt = max(max(p.bt_stride, 1) for p in problems)
        return ChunkBuffers(
            torch.empty(max(ws, 256), dtype=torch.uint8, device=device),
            torch.empty(max(nbs, 1), dtype=torch.float32, device=device),
            torch.empty(max(nbs, 1), dtype=torch.uint8, device=device) if with_mask else None,
            torch.empty((B, bt), dtype=torch.int32, device=device),
            torch.empty((B, bt), dtype=torch.int32, device=device),
            torch.empty(B, dtype=torch.int32, device=device),
        )


def estimation_scale(head_dim: int, stride: int) -> float:
    return 1.0 / (math.sqrt(head_dim) * stride)


@dataclass
class KeySeq:
    """Keys of every request in logical token order (xattn_estimate_seq):
    request r's history and current keys are tokens [starts[r], ...) of
    `keys`, with element strides between heads and between tokens."""
    keys: object
    starts: list
    head_stride: int
    token_stride: int = 0
    samples: int = 0          # > 0: score the first `samples` reshaped columns of each
                              # history block only (xattn_estimate_sampled)


def estimate_select(problem, q, k_cur, k_pool, tau, bufs: ChunkBuffers, est_scale=None,
                    stream=None, k_seq: KeySeq | None = None, per_kv_head=False):
    """Steps 1 and 2 of a chunk: estimation, then the block selection (sel_page,
    n_sel in bufs).  Reads Q and the keys -- the chunk's K and the history
    pages, or the same keys in logical order when k_seq is given; not V.
    per_kv_head: one block set per KV head instead of the vote across them."""
    D = problem.c.head_dim
    est_scale = estimation_scale(D, problem.c.stride) if est_scale is None else est_scale
    if k_seq is not None and k_seq.samples:
        X.xattn_estimate_sampled(problem, q, k_seq.keys, k_seq.starts, k_seq.samples, est_scale,
                                 bufs.workspace, bufs.block_sums, stream,
                                 head_stride=k_seq.head_stride, token_stride=k_seq.token_stride)
    elif k_seq is not None:
        X.xattn_estimate_seq(problem, q, k_seq.keys, k_seq.starts, est_scale, bufs.workspace,
                             bufs.block_sums, stream, head_stride=k_seq.head_stride,
                             token_stride=k_seq.token_stride)
    else:
        X.xattn_estimate(problem, q, k_cur, k_pool, est_scale, bufs.workspace, bufs.block_sums,
                         stream)
    select = X.xattn_select_per_kv_head if per_kv_head else X.xattn_select
    select(problem, bufs.block_sums, tau, bufs.workspace, bufs.mask, bufs.sel_idx,
           bufs.sel_page, bufs.n_sel, stream)


def attend(problem, q, k_cur, v_cur, k_pool, v_pool, bufs: ChunkBuffers, o, lse,
           softmax_scale=None, stream=None, per_kv_head=False):
    """Step 3 of a chunk: attention over the selected pages and the causal chunk."""
    D = problem.c.head_dim
    softmax_scale = 1.0 / math.sqrt(D) if softmax_scale is None else softmax_scale
    att = X.bsa_chunk_attention_per_kv_head if per_kv_head else X.bsa_chunk_attention
    att(problem, q, k_cur, v_cur, k_pool, v_pool, bufs.sel_page, bufs.n_sel, softmax_scale,
        bufs.workspace, o, lse, stream)


def prefill_chunk(problem, q, k_cur, v_cur, k_pool, v_pool, tau, bufs: ChunkBuffers, o, lse,
                  est_scale=None, softmax_scale=None, stream=None, k_seq: KeySeq | None = None,
                  per_kv_head=False):
    """One chunk of XAttention BSA prefill: estimate, select, attend."""
    estimate_select(problem, q, k_cur, k_pool, tau, bufs, est_scale, stream, k_seq, per_kv_head)
    attend(problem, q, k_cur, v_cur, k_pool, v_pool, bufs, o, lse, softmax_scale, stream,
           per_kv_head)


class SequencePrefill:
    """Chunked prefill of one sequence of length L in chunks of `chunk` tokens.

    Q [H, L, D], K/V [Hkv, L, D] (current-chunk views are windows of these),
    pools [P, Bk, Hkv, D] and block_table [1, P] as device tensors.  Chunk c
    queries tokens [c*chunk, (c+1)*chunk) and reads history [0, c*chunk)
    through the block table for its attention.  The estimation reads the keys
    [0, (c+1)*chunk) of K in token order (xattn_estimate_seq), or, with
    est_from_pages, the history pages and the chunk's K (xattn_estimate): the
    two give the same bits.  per_kv_head selects one block set per KV head;
    est_samples > 0 estimates each history block from its first est_samples
    reshaped columns (xattn_estimate_sampled)."""

    def __init__(self, H, Hkv, D, stride, block, L, chunk, block_table, num_pages,
                 with_mask=False, est_from_pages=False, per_kv_head=False, est_samples=0):
        self.H, self.Hkv, self.D, self.L, self.chunk = H, Hkv, D, L, chunk
        self.est_from_pages = est_from_pages
        self.est_samples = est_samples
        self.per_kv_head = per_kv_head
        self.problems = [
            X.Problem(H, Hkv, D, stride, block, [chunk], [c * chunk], block_table, num_pages,
                      q_head_stride=L * D, kv_head_stride=L * D, lse_head_stride=L)
            for c in range(L // chunk)]
        self.bufs = ChunkBuffers.for_problems(self.problems, block_table.device, with_mask)
        if per_kv_head:  # selections per (request, KV head)
            dev = block_table.device
            self.bufs.sel_idx = torch.empty((Hkv, L // block), dtype=torch.int32, device=dev)
            self.bufs.sel_page = torch.empty((Hkv, L // block), dtype=torch.int32, device=dev)
            self.bufs.n_sel = torch.empty(Hkv, dtype=torch.int32, device=dev)

    def key_seq(self, K):
        return None if self.est_from_pages else KeySeq(K, [0], K.stride(0),
                                                       samples=self.est_samples)

    def run_chunk(self, c, Q, K, V, kpool, vpool, tau, O, LSE, stream=None):
        t0 = c * self.chunk
        prefill_chunk(self.problems[c], Q[:, t0:], K[:, t0:], V[:, t0:], kpool, vpool, tau,
                      self.bufs, O[:, t0:], LSE[:, t0:], stream=stream, k_seq=self.key_seq(K),
                      per_kv_head=self.per_kv_head)

    def run(self, Q, K, V, kpool, vpool, tau, O, LSE, stream=None, on_chunk=None):
        for c in range(len(self.problems)):
            self.run_chunk(c, Q, K, V, kpool, vpool, tau, O, LSE, stream)
            if on_chunk is not None:
                on_chunk(c, self.bufs)

    def run_from_host(self, host, dev, tau, stream, h2d_stream, d2h_stream, store_kv=False,
                      out_direct=False):
        """The whole prefill from pinned host memory, copies overlapped with
        compute.  Chunk c computes on `stream` once the copies it reads have
        landed (an event) ([SYNC] 修复方案: every consumer waits on the event of
        the copy it reads).

        Inputs: on `h2d_stream`, chunk by chunk, Q and K (all the estimate
        reads) then V (read by the attention only).

        Outputs: O and LSE go device -> host on `d2h_stream` once the chunk is
        done.  out_direct=True instead has the attention write them straight
        into the pinned host buffers (bsa_chunk_attention takes page-locked
        host memory): nothing is copied, but the kernel's row stores then cross
        the host link as it runs.

        store_kv=False: the page pools are inputs, copied on `h2d_stream` after
        chunk 0's Q, K, V (one copy each: a chunk's history pages are scattered
        through the pool by the block table); chunk 0 runs while they come in.
        store_kv=True: the pools are built on the device.  Before chunk c's
        attention, xattn_store_kv writes its K and V into the pages the block
        table gives their positions ("Task Plan: Layerwise Offload
        Refactoring", Phase 1.2), which is the history chunk c + 1 reads.  With
        a block table that maps every position of the sequence, the pools end
        up equal to a prefilled pool of the same sequence, so the results are
        too.

        host, dev: dicts of tensors 'q', 'k', 'v', 'o', 'lse' (and 'kpool',
        'vpool' on the device; on the host too unless store_kv), host pinned,
        same shapes.  Work is enqueued after whatever `stream` already holds;
        the side streams start from that point too.  Returns the event recorded
        on `stream` once every output is on the host."""
        return self._host_fed(host, dev, tau, stream, h2d_stream, d2h_stream, store_kv,
                              out_direct, None, None, True)

    def _host_fed(self, host, dev, tau, stream, h2d_stream, d2h_stream, store_kv, out_direct,
                  inputs_after, outputs_after, join, early_waits=False):
        """run_from_host's work.  inputs_after / outputs_after: events after
        which the device inputs (q, k, v) / outputs (o, lse) may be overwritten
        (None: once `stream` has done what it holds).  join: `stream` waits for
        the read-backs and the event it then records is returned; otherwise
        (event after the last attention on `stream`, event after the last
        read-back on `d2h_stream`).  early_waits: chunk c + 1's wait for its
        keys goes before chunk c's attention, so that its estimate follows that
        attention with nothing in between and may start in its tail (a
        programmatic dependent launch); for callers whose copies run well
        ahead of the compute (HostFedPipeline)."""
        import torch
        start = torch.cuda.Event()
        start.record(stream)
        h2d_stream.wait_event(inputs_after if inputs_after is not None else start)
        d2h_stream.wait_event(start)
        n = len(self.problems)
        ready, ready_v = [], []

        def chunk_inputs(c):
            t0, t1 = c * self.chunk, (c + 1) * self.chunk
            for name in ("q", "k", "v"):  # one 2-D copy each: a row per head
                X.copy_window_async(dev[name], host[name], t0, t1, h2d_stream)
                if name != "q":
                    ev = torch.cuda.Event()
                    ev.record(h2d_stream)
                    (ready if name == "k" else ready_v).append(ev)

        with torch.cuda.stream(h2d_stream):
            chunk_inputs(0)
            if not store_kv:
                dev["kpool"].copy_(host["kpool"], non_blocking=True)
                dev["vpool"].copy_(host["vpool"], non_blocking=True)
            for c in range(1, n):
                chunk_inputs(c)
        out = host if out_direct else dev
        for c in range(n):
            t0, t1 = c * self.chunk, (c + 1) * self.chunk
            p = self.problems[c]
            q, k, v = dev["q"][:, t0:], dev["k"][:, t0:], dev["v"][:, t0:]
            if not early_waits or c == 0:
                stream.wait_event(ready[c])  # K of chunks 0..c have landed (one copy stream)
            estimate_select(p, q, k, dev["kpool"], tau, self.bufs, stream=stream,
                            k_seq=self.key_seq(dev["k"]), per_kv_head=self.per_kv_head)
            stream.wait_event(ready_v[c])
            if c == 0 and outputs_after is not None:  # the previous read-back of o, lse
                stream.wait_event(outputs_after)
            if store_kv:  # the history of chunk c + 1, before anything reads it
                X.xattn_store_kv(p, k, v, dev["kpool"], dev["vpool"], stream)
            if early_waits and c + 1 < n:
                stream.wait_event(ready[c + 1])
            attend(p, q, k, v, dev["kpool"], dev["vpool"], self.bufs, out["o"][:, t0:],
                   out["lse"][:, t0:], stream=stream, per_kv_head=self.per_kv_head)
            if not out_direct:
                done = torch.cuda.Event()
                done.record(stream)
                d2h_stream.wait_event(done)
                X.copy_window_async(host["o"], dev["o"], t0, t1, d2h_stream)
                X.copy_window_async(host["lse"], dev["lse"], t0, t1, d2h_stream)
        side_done = torch.cuda.Event()
        side_done.record(d2h_stream)
        if not join:
            compute_done = torch.cuda.Event()
            compute_done.record(stream)
            return compute_done, side_done
        stream.wait_event(side_done)
        back = torch.cuda.Event()
        back.record(stream)
        return back


class HostFedPipeline:
    """Prefills of a stream of same-shaped sequences fed from pinned host
    memory, through two device buffer sets in turn: the next prefill's Q, K, V
    cross the host link while the current one computes, and the current one's
    O and LSE come back while the next one computes.  Each prefill is
    `SequencePrefill.run_from_host`'s (chunks ordered after the copies they
    read by events); what changes is only when its copies may start: its
    inputs once the prefill two back has finished reading that buffer set,
    its outputs once that prefill's read-back has left it.  The compute of
    consecutive prefills stays in order on `stream` (they share the
    sequence's workspace and page pools).

    seq: a SequencePrefill; dev_sets: two dicts of device tensors as
    run_from_host's `dev`.  The page pools may be shared when they are built
    on the device (store_kv: a prefill's stores run on `stream`, after the
    previous prefill's attentions); pools copied from the host need a pair
    per set."""

    def __init__(self, seq, dev_sets, stream, h2d_stream, d2h_stream, store_kv=True,
                 out_direct=False):
        if len(dev_sets) != 2:
            raise ValueError("HostFedPipeline takes two device buffer sets")
        if not store_kv and any(dev_sets[0][k] is dev_sets[1][k] for k in ("kpool", "vpool")):
            # the next prefill's pool copy would overwrite the pools this one reads
            raise ValueError("HostFedPipeline with pools copied from the host needs a pool "
                             "pair per buffer set")
        self.seq, self.dev_sets = seq, dev_sets
        self.stream, self.h2d, self.d2h = stream, h2d_stream, d2h_stream
        self.store_kv, self.out_direct = store_kv, out_direct
        import torch
        # both sets are free once `stream` has done what it holds now
        ready = torch.cuda.Event()
        ready.record(stream)
        self.in_free = [ready, ready]   # set s's inputs no longer read
        self.out_free = [ready, ready]  # set s's outputs read back
        self.n = 0

    def submit(self, host, tau):
        """Enqueue one prefill of `host` (run_from_host's dict); returns the
        event after which its O and LSE are on the host."""
        s = self.n % 2
        self.n += 1
        compute_done, side_done = self.seq._host_fed(
            host, self.dev_sets[s], tau, self.stream, self.h2d, self.d2h, self.store_kv,
            self.out_direct, self.in_free[s], self.out_free[s], False, early_waits=True)
        self.in_free[s], self.out_free[s] = compute_done, side_done
        return side_done

    def join(self):
        """`stream` waits for every read-back submitted so far."""
        for ev in self.out_free:
            self.stream.wait_event(ev)


class LayerRing:
    """N-slot ring of per-layer KV page pools fed from pinned host memory.

    "Task Plan: Layerwise Offload Refactoring", Phase 1.1 / Phase 4: slot
    l mod N holds layer l; the first N layers are preloaded, and the slot of
    layer l is reloaded with layer l+N once layer l's compute has finished.
    Copies run on one side stream; the compute stream waits on the slot's
    `ready` event before use and records its `done` event after, the event
    discipline of "XAttention Offload Stream Synchronization Fix" (修复方案,
    Event 同步机制) that keeps estimation from reading a slot still in flight."""

    def __init__(self, num_slots, pages, block, Hkv, D, device):
        self.N = num_slots
        shape = (num_slots, pages, block, Hkv, D)
        self.k = torch.empty(shape, dtype=torch.bfloat16, device=device)
        self.v = torch.empty(shape, dtype=torch.bfloat16, device=device)
        self.copy_stream = torch.cuda.Stream(device=device)
        self.ready = [None] * num_slots
        self.done = [torch.cuda.Event() for _ in range(num_slots)]
        self.owner = [None] * num_slots
        self.log = []  # (layer, start event, ready event, bytes) per load
        cur = torch.cuda.current_stream(device)
        for e in self.done:  # every slot starts free
            e.record(cur)

    def slot(self, layer):
        return layer % self.N

    def load(self, layer, host_k, host_v, n_pages):
        """Queue the copy of the first n_pages pages of `layer` into its slot."""
        s = self.slot(layer)
        start = torch.cuda.Event(enable_timing=True)
        ready = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.copy_stream):
            self.copy_stream.wait_event(self.done[s])
            start.record(self.copy_stream)
            if n_pages > 0:
                self.k[s, :n_pages].copy_(host_k[:n_pages], non_blocking=True)
                self.v[s, :n_pages].copy_(host_v[:n_pages], non_blocking=True)
            ready.record(self.copy_stream)
        self.ready[s] = ready
        self.owner[s] = layer
        self.log.append((layer, start, ready, 2 * n_pages * host_k[0].numel() * 2))

    @property
    def bytes_copied(self):
        return sum(x[3] for x in self.log)

    def acquire(self, layer, stream):
        s = self.slot(layer)
        assert self.owner[s] == layer, "slot holds another layer"
        stream.wait_event(self.ready[s])
        return self.k[s], self.v[s]

    def release(self, layer, stream):
        self.done[self.slot(layer)].record(stream)


def ring_problem(H, Hkv, D, stride, block, L, chunk, c, block_table, num_pages):
    """The problem of chunk c in the layer ring: history [0, c*chunk) through
    the block table, the chunk's own K/V read where the ring slot holds them --
    its pages, [tokens, Hkv, D] (heads D apart, tokens Hkv*D apart)."""
    return X.Problem(H, Hkv, D, stride, block, [chunk], [c * chunk], block_table, num_pages,
                     q_head_stride=L * D, kv_head_stride=D, lse_head_stride=L,
                     kv_token_stride=Hkv * D)


def ring_prefill_chunk(ring, layers, c, chunk, H, Hkv, D, stride, block, tau, bufs, problem,
                       outs, stream, on_layer=None, compute_events=None, reuse_selection=False):
    """Chunk c of every layer through the ring: history pages [0, c*chunk/block)
    of each layer are loaded into its slot, the current chunk's K/V are the
    next chunk/block pages of the same host cache (copied in the same load).
    The slot holds the layer's pages in logical order (an identity block
    table), so the chunk's K/V are read in place as a [tokens, Hkv, D] view
    (`problem` from ring_problem) and the estimation reads the slot's keys
    [0, (c+1)*chunk) in token order (xattn_estimate_seq).

    reuse_selection: only layer 0 estimates and selects; every later layer
    attends over the pages layer 0 selected ("XAttention BSA Policy 设计文档",
    性能分析, 优化方向 1: share the estimate across layers).  The page ids
    stay valid because every slot lays its layer out under one block table."""
    n_hist = c * chunk // block
    n_load = n_hist + chunk // block
    L = len(layers)
    for l in range(min(ring.N, L)):
        ring.load(l, layers[l].k_host, layers[l].v_host, n_load)
    for l in range(L):
        kp, vp = ring.acquire(l, stream)
        if compute_events is not None:  # starts after the slot wait
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
        with torch.cuda.stream(stream):
            # the chunk's K/V: its pages of the slot, [tokens, Hkv, D] in place
            kc, vc = kp[n_hist:n_load], vp[n_hist:n_load]
            q = layers[l].q[:, c * chunk:]
            o, lse = outs[l]
            if reuse_selection and l > 0:
                attend(problem, q, kc, vc, kp, vp, bufs, o[:, c * chunk:], lse[:, c * chunk:],
                       stream=stream)
            else:
                prefill_chunk(problem, q, kc, vc, kp, vp, tau, bufs, o[:, c * chunk:],
                              lse[:, c * chunk:], stream=stream,
                              k_seq=KeySeq(kp, [0], D, Hkv * D))
            if compute_events is not None:
                e1.record(stream)
                compute_events.append((e0, e1))
            if on_layer is not None:
                on_layer(l, bufs)
        ring.release(l, stream)
        if l + ring.N < L:
            ring.load(l + ring.N, layers[l + ring.N].k_host, layers[l + ring.N].v_host, n_load)
