"""Density of the block-aggregation variants the XAttention BSA pages compare.

[BSA] 核心算法 1, Step 4 ("为什么使用 Majority Voting?") weighs three ways of
turning the per-head threshold masks into one block set per chunk: any()
over all heads (density close to 100%), all() (too aggressive), and the
majority vote (> 50% of the KV-head x query-block votes) the method keeps;
it quotes per-head density 20-35%, any() ~100% and the vote ~45% on its
model.  All three are the library's vote rule with another ratio
num/den: keep block j when votes_j * den > num * (Hkv * Qb), with

  any()    = (0, 1)          one vote is enough;
  majority = (1, 2)          the pages' rule;
  all()    = (N - 1, N)      N > Hkv * Qb, so only votes_j = Hkv * Qb passes.

A fourth variant, one block set per KV head (each KV head's own majority
over its query blocks, no vote across KV heads), is the reading this file
takes of a per-KV-head selection; its density is the mean over KV heads.
Every variant forces the sink and last history blocks, as Step 4 does.

The test checks the order the definitions imply on a seeded workload of the
input recipe; ``python tests/test_aggregation_density.py <workload> [L]``
prints the table of densities per chunk from the oracle.
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from oracle import xattn_oracle as O  # noqa: E402
from xattention_block_sparse_gb300 import inputs as I  # noqa: E402

VARIANTS = ("per_head", "any", "per_kv_head", "majority", "all")


def chunk_densities(wl, c, tau):
    """Densities of chunk c of a chunked workload, one per variant."""
    cfg = wl.cfg
    chunk = wl.calls[c].q_lens[0]
    t0, t1 = c * chunk, (c + 1) * chunk
    kbh = t0 // cfg.block
    q, k = wl.f64("q"), wl.f64("k")
    bs = O.estimate_request(q[:, t0:t1], k[:, t0:t1], wl.f64("kpool"), wl.block_table[0], t0,
                            cfg.H, cfg.Hkv, cfg.stride, cfg.block,
                            O.default_estimation_scale(cfg.D, cfg.stride))
    mask = O.threshold_select(bs.astype(np.float32), tau)
    qb = mask.shape[1]
    out = {"per_head": float(mask[:, :, :kbh].mean())}
    n_all = cfg.Hkv * qb + 1
    for name, vote in (("any", (0, 1)), ("majority", (1, 2)), ("all", (n_all - 1, n_all))):
        out[name] = O.density(len(O.gqa_vote(mask, cfg.Hkv, kbh, vote=vote)), kbh)
    per_kv = [len(s) for s in O.per_kv_head_select(mask, cfg.Hkv, kbh)]
    out["per_kv_head"] = O.density(sum(per_kv), kbh * cfg.Hkv)
    return out


def test_variant_densities_follow_the_vote_ratio():
    wl = I.make_workload("q06b_4k")
    for c in range(1, len(wl.calls)):
        d = chunk_densities(wl, c, 0.6)
        assert 0.0 < d["all"] <= d["majority"] <= d["any"] <= 1.0
        assert d["per_kv_head"] <= d["any"]
        assert d["per_head"] <= d["any"]
        # sink and last are forced, so no variant falls below 2 blocks
        kbh = c * wl.calls[c].q_lens[0] // wl.cfg.block
        assert d["all"] >= min(2, kbh) / kbh


if __name__ == "__main__":
    name = sys.argv[1] if len(sys.argv) > 1 else "q06b_4k"
    L = int(sys.argv[2]) if len(sys.argv) > 2 and sys.argv[2] else None
    taus = [float(t) for t in sys.argv[3].split(",")] if len(sys.argv) > 3 else [0.9]
    wl = I.make_workload(name, L=L)
    for tau in taus:
        print(f"{name} L={L or wl.cfg.L} tau={tau}")
        print("chunk " + " ".join(f"{v:>11}" for v in VARIANTS))
        for c in range(1, len(wl.calls)):
            d = chunk_densities(wl, c, tau)
            print(f"{c:5d} " + " ".join(f"{d[v]:11.4f}" for v in VARIANTS), flush=True)
