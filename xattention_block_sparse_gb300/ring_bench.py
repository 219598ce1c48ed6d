"""Timing of the 128K layer ring: chunked prefill of 8 layers through 4 KV slots
fed from pinned host memory on a side stream.

    python -m xattention_block_sparse_gb300.ring_bench [--chunks 28,29,30,31]
                                                       [--reuse-selection]

For each chunk, every layer's history (and current chunk) pages are copied
host -> device into slot (layer mod 4) while the compute stream works on the
other slots; the compute stream waits on the slot's ready event.  Reports,
as one JSON line, the compute time with the event waits excluded (CUDA events
on the compute stream, the first recorded after each wait), the copy time and
bandwidth of the side stream, the wall time, and the overlap
1 - (wall - compute) / copy.  Inputs are the seeded device-drawn layers of the
128K config.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from xattention_block_sparse_gb300 import inputs as I  # noqa: E402
from xattention_block_sparse_gb300 import runner as RN  # noqa: E402
from xattention_block_sparse_gb300 import xattn as X  # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--chunks", default="28,29,30,31")
    ap.add_argument("--layers", type=int, default=None)
    ap.add_argument("--reuse-selection", action="store_true",
                    help="estimate and select on layer 0 only; later layers reuse its pages")
    a = ap.parse_args()
    from __graft_entry__ import build
    build()
    cfg = I.CONFIGS["q4b_128k"]
    d = torch.device("cuda:0")
    H, Hkv, D, S, Bk, L, chunk = cfg.H, cfg.Hkv, cfg.D, cfg.stride, cfg.block, cfg.L, cfg.chunk
    P = L // Bk
    nl = a.layers or cfg.layers
    layers = [I.make_ring_layer(l, d) for l in range(nl)]
    ring = RN.LayerRing(cfg.ring_slots, P, Bk, Hkv, D, d)
    BT = torch.arange(P, dtype=torch.int32, device=d)[None]
    chunks = [int(x) for x in a.chunks.split(",")]
    problems = {c: RN.ring_problem(H, Hkv, D, S, Bk, L, chunk, c, BT, P) for c in chunks}
    bufs = RN.ChunkBuffers.for_problems(list(problems.values()), d)
    outs = [(torch.empty((H, L, D), dtype=torch.bfloat16, device=d),
             torch.empty((H, L), dtype=torch.float32, device=d)) for _ in layers]
    stream = torch.cuda.Stream(device=d)
    tau = cfg.taus[0]
    RN.ring_prefill_chunk(ring, layers, chunks[0], chunk, H, Hkv, D, S, Bk, tau, bufs,
                          problems[chunks[0]], outs, stream,
                          reuse_selection=a.reuse_selection)  # warm-up
    torch.cuda.synchronize()
    per_chunk = []
    for c in chunks:
        ring.log.clear()
        comp = []
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        w0.record(stream)
        ring.copy_stream.wait_stream(stream)
        RN.ring_prefill_chunk(ring, layers, c, chunk, H, Hkv, D, S, Bk, tau, bufs, problems[c],
                              outs, stream, compute_events=comp,
                              reuse_selection=a.reuse_selection)
        w1.record(stream)
        torch.cuda.synchronize()
        per_chunk.append({
            "chunk": c,
            "compute_ms": sum(a.elapsed_time(b) for a, b in comp),
            "copy_ms": sum(st.elapsed_time(en) for _, st, en, _ in ring.log),
            "wall_ms": w0.elapsed_time(w1),
            "h2d_bytes": ring.bytes_copied,
        })
    assert X.xattn_device_error() == 0
    comp = sum(p["compute_ms"] for p in per_chunk)
    copy = sum(p["copy_ms"] for p in per_chunk)
    wall = sum(p["wall_ms"] for p in per_chunk)
    byts = sum(p["h2d_bytes"] for p in per_chunk)
    tokens = chunk * len(chunks)
    print(json.dumps({
        "workload": (f"q4b_128k: {H} Q / {Hkv} KV heads, head_dim {D}, stride {S}, chunks "
                     f"{chunks} of {chunk} tokens at 128K context, {nl} layers through "
                     f"{cfg.ring_slots} ring slots, tau {tau}"
                     + (", layer 0's selection reused by every layer" if a.reuse_selection
                        else "")),
        "compute_ms": comp, "copy_ms": copy, "wall_ms": wall,
        "h2d_GB": byts / 1e9, "h2d_GBps": byts / 1e9 / (copy / 1e3) if copy else None,
        "overlap": 1.0 - (wall - comp) / copy if copy else None,
        # layer-tokens per second: every layer prefills the same chunk tokens
        "layer_tokens_per_s_compute": tokens * nl / (comp / 1e3),
        "layer_tokens_per_s_wall": tokens * nl / (wall / 1e3),
        "per_chunk": per_chunk,
    }))


if __name__ == "__main__":
    main()
