"""Seeded synthetic inputs for XAttention block-sparse chunked prefill.

This module draws random tensors and lays them out; it holds none of the
method's arithmetic (no scores, softmax, selection or attention).  Both the
CUDA path (tests, bench) and the float64 oracle (tests) consume what it
produces, so the two sides always see the same bf16 values.

Shapes follow the workloads the XAttention BSA pages describe: Qwen3-0.6B /
Qwen3-4B-like attention layers (16/8 and 32/8 heads, head_dim 128) at 4K to
128K context, chunked prefill with 128-token KV pages addressed through a
block_table, and a varlen batch addressed through cu_seq_lens.

Recipe (all configs):
  * numpy PCG64, seed = 1000 + config index, one child generator per tensor
    in the order Q, K, V, extras (needles / page permutation / bias);
  * values drawn in fp32 and rounded to bf16 with round-to-nearest-even;
    the oracle reads exactly those bf16 values widened to float64;
  * RoPE, where a config asks for it, is the NeoX rotate-half form with
    theta = 1e6 at absolute positions 0..L-1, applied in fp32 before the
    bf16 rounding (it is part of the synthetic workload, not of the method);
  * heavy key blocks (q06b_32k_sparse): in every run of `heavy_every` blocks
    one seeded block is heavy; per KV head a direction u (unit, seeded) is
    added as a*u to every query of the group and to every key of the heavy
    blocks, after RoPE, with a^2 / sqrt(D) = heavy_boost, so a heavy key's
    logit gains about heavy_boost.  This concentrates attention the way the
    pages' needle-in-a-haystack runs do, without their data.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "CONFIGS",
    "Workload",
    "ChunkCall",
    "make_workload",
    "bf16_round",
    "bf16_bits_to_f64",
    "chunk_calls",
]


# --------------------------------------------------------------------------
# bf16 helpers (storage format only)
# --------------------------------------------------------------------------

def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest-even); returns the uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = (bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float64 exactly."""
    u32 = bits.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def _rope_neox(x: np.ndarray, theta: float) -> np.ndarray:
    """x: [heads, L, D] fp32 at absolute positions 0..L-1 (NeoX rotate-half)."""
    _, L, D = x.shape
    half = D // 2
    inv = theta ** (-np.arange(half, dtype=np.float64) * 2.0 / D)
    ang = np.arange(L, dtype=np.float64)[:, None] * inv[None, :]
    cos = np.cos(ang).astype(np.float32)
    sin = np.sin(ang).astype(np.float32)
    x1 = x[..., :half]
    x2 = x[..., half:]
    out = np.empty_like(x)
    out[..., :half] = x1 * cos - x2 * sin
    out[..., half:] = x2 * cos + x1 * sin
    return out


# --------------------------------------------------------------------------
# Configurations
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class Config:
    index: int
    name: str
    H: int
    Hkv: int
    D: int
    stride: int
    block: int
    taus: tuple
    # chunked single sequence: total length and chunk length
    L: int = 0
    chunk: int = 0
    # varlen batch (one chunk per request)
    q_lens: tuple = ()
    kh_lens: tuple = ()
    pool_pages: int = 0
    bt_width: int = 0
    rope: bool = False
    needles: int = 0
    sink: bool = False
    local_bias: bool = False
    layers: int = 1
    ring_slots: int = 0
    # heavy key blocks: one seeded block in every `heavy_every` blocks carries a
    # shared direction that every query also carries (logit boost heavy_boost)
    heavy_every: int = 0
    heavy_boost: float = 0.0


CONFIGS = {
    "tiny": Config(1, "tiny", H=2, Hkv=1, D=64, stride=8, block=64, taus=(0.9,),
                   L=1024, chunk=256, needles=3),
    "q06b_4k": Config(2, "q06b_4k", H=16, Hkv=8, D=128, stride=8, block=128, taus=(0.9,),
                      L=4096, chunk=1024, rope=True),
    "q06b_32k": Config(3, "q06b_32k", H=16, Hkv=8, D=128, stride=8, block=128,
                       taus=(0.9, 0.95), L=32768, chunk=4096, rope=True),
    "q4b_128k": Config(4, "q4b_128k", H=32, Hkv=8, D=128, stride=16, block=128, taus=(0.9,),
                       L=131072, chunk=4096, rope=True, sink=True, local_bias=True,
                       layers=8, ring_slots=4),
    "varlen": Config(5, "varlen", H=16, Hkv=8, D=128, stride=8, block=128, taus=(0.9,),
                     q_lens=(8192, 3072, 1024), kh_lens=(0, 16384, 65536),
                     pool_pages=640, bt_width=512),
    # the 32K shapes with attention concentrated on a few key blocks, so that
    # tau = 0.9 keeps about a tenth of the history (the density the stream-sync
    # page measures for Qwen3-0.6B at 32K, ~9.8%)
    "q06b_32k_sparse": Config(6, "q06b_32k_sparse", H=16, Hkv=8, D=128, stride=8, block=128,
                              taus=(0.9,), L=32768, chunk=4096, rope=True, heavy_every=12,
                              heavy_boost=6.0),
}


# --------------------------------------------------------------------------
# Workload containers
# --------------------------------------------------------------------------

@dataclass
class ChunkCall:
    """One invocation of the hot path: B requests, each a query chunk plus history.

    q_tok0[r] is the first token of request r's query chunk inside the packed
    q/k_cur/v_cur token axis (the packed axis may be a window of a longer
    sequence: token offset tok_base into the full tensors)."""
    q_lens: list
    kh_lens: list
    tok_base: int                 # offset of the packed token axis into Q/Kc/Vc
    block_table: np.ndarray       # int32 [B, bt_width]

    @property
    def B(self) -> int:
        return len(self.q_lens)

    @property
    def cu_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)

    @property
    def cu_kh(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.kh_lens)]).astype(np.int32)


@dataclass
class Workload:
    cfg: Config
    # bf16 bit patterns
    q_bits: np.ndarray            # [H, Ltot, D]
    k_bits: np.ndarray            # [Hkv, Ltot, D]   current-chunk K (packed)
    v_bits: np.ndarray            # [Hkv, Ltot, D]
    kpool_bits: np.ndarray        # [P, Bk, Hkv, D]
    vpool_bits: np.ndarray        # [P, Bk, Hkv, D]
    block_table: np.ndarray       # int32 [B, W]
    calls: list = field(default_factory=list)

    def f64(self, name: str) -> np.ndarray:
        return bf16_bits_to_f64(getattr(self, name + "_bits"))


def _children(seed: int, n: int = 4):
    ss = np.random.SeedSequence(seed)
    return [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(n)]


def _normal(rng, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32)


def _pages_from_seq(kv_bits: np.ndarray, block: int, perm: np.ndarray, P: int) -> np.ndarray:
    """Scatter a [Hkv, L, D] sequence into a [P, Bk, Hkv, D] pool: logical page j
    of the sequence lands on physical page perm[j]."""
    Hkv, L, D = kv_bits.shape
    npg = L // block
    pool = np.zeros((P, block, Hkv, D), dtype=np.uint16)
    seq = kv_bits.reshape(Hkv, npg, block, D).transpose(1, 2, 0, 3)  # [npg, Bk, Hkv, D]
    pool[perm[:npg]] = seq
    return pool


def make_workload(name: str, layer: int = 0, L: int | None = None,
                  chunk: int | None = None) -> Workload:
    """Build the seeded synthetic inputs of one config (one layer).

    ``L``/``chunk`` may shrink a chunked config (used for quick tests of the
    same recipe); the default is the config's own size."""
    cfg = CONFIGS[name]
    seed = 1000 + cfg.index + 7919 * layer
    g_q, g_k, g_v, g_x = _children(seed)
    H, Hkv, D, Bk = cfg.H, cfg.Hkv, cfg.D, cfg.block

    if cfg.q_lens:                          # varlen batch, one chunk per request
        q_lens = list(cfg.q_lens)
        kh_lens = list(cfg.kh_lens)
        Lq = sum(q_lens)
        q = _normal(g_q, (H, Lq, D))
        k = _normal(g_k, (Hkv, Lq, D))
        v = _normal(g_v, (Hkv, Lq, D))
        P, W = cfg.pool_pages, cfg.bt_width
        perm = g_x.permutation(P).astype(np.int32)
        hist_k = _normal(g_x, (P, Bk, Hkv, D))
        hist_v = _normal(g_x, (P, Bk, Hkv, D))
        bt = np.full((len(q_lens), W), -1, dtype=np.int32)
        used = 0
        for r, kh in enumerate(kh_lens):
            n = kh // Bk
            bt[r, :n] = perm[used:used + n]
            used += n
        # pages nobody references stay filled with noise: a wrong page id
        # reads plausible values, so only exact indexing passes parity
        wl = Workload(cfg, bf16_round(q), bf16_round(k), bf16_round(v),
                      bf16_round(hist_k), bf16_round(hist_v), bt)
        wl.calls = [ChunkCall(q_lens, kh_lens, 0, bt)]
        return wl

    L = L or cfg.L
    chunk = chunk or cfg.chunk
    assert L % chunk == 0 and chunk % Bk == 0
    q = _normal(g_q, (H, L, D))
    k = _normal(g_k, (Hkv, L, D))
    v = _normal(g_v, (Hkv, L, D))
    if cfg.needles:
        pos = g_x.choice(L, size=cfg.needles, replace=False)
        k[:, pos, :] *= 4.0
    if cfg.rope:
        q = _rope_neox(q, 1e6)
        k = _rope_neox(k, 1e6)
    if cfg.local_bias:
        nwin = (L + 1023) // 1024
        u = (0.5 * _normal(g_x, (Hkv, nwin, D))).astype(np.float32)
        G = H // Hkv
        win = np.arange(L) // 1024
        k += u[:, win, :]
        q += np.repeat(u, G, axis=0)[:, win, :]
    if cfg.sink:
        k[:, 0:4, :] *= 3.0
    if cfg.heavy_every:
        nblk = L // Bk
        starts = np.arange(0, nblk, cfg.heavy_every)
        span = np.minimum(cfg.heavy_every, nblk - starts)
        heavy = starts + (g_x.random(len(starts)) * span).astype(np.int64)
        u = _normal(g_x, (Hkv, D)).astype(np.float64)
        u /= np.linalg.norm(u, axis=1, keepdims=True)
        a = np.sqrt(cfg.heavy_boost * np.sqrt(D))
        G = H // Hkv
        q += np.repeat((a * u).astype(np.float32), G, axis=0)[:, None, :]
        tok = (heavy[:, None] * Bk + np.arange(Bk)[None, :]).reshape(-1)
        k[:, tok, :] += (a * u).astype(np.float32)[:, None, :]
    P = L // Bk
    perm = g_x.permutation(P).astype(np.int32)
    kb, vb = bf16_round(k), bf16_round(v)
    wl = Workload(cfg, bf16_round(q), kb, vb,
                  _pages_from_seq(kb, Bk, perm, P), _pages_from_seq(vb, Bk, perm, P),
                  perm[None, :].copy())
    wl.calls = chunk_calls(L, chunk, wl.block_table)
    return wl


def chunk_calls(L: int, chunk: int, block_table: np.ndarray) -> list:
    """Chunked prefill of one sequence: chunk c has queries [c*chunk, (c+1)*chunk)
    and history tokens [0, c*chunk) read through the block_table."""
    return [ChunkCall([chunk], [c * chunk], c * chunk, block_table)
            for c in range(L // chunk)]


# --------------------------------------------------------------------------
# Long-context layer stack (the 128K config): drawn on the device
# --------------------------------------------------------------------------

@dataclass
class RingLayer:
    """One synthetic layer of the 128K config.

    q        device bf16 [H, L, D]
    k_host   pinned host bf16 [P, Bk, Hkv, D]   the layer's KV cache in host
    v_host   pinned host bf16 [P, Bk, Hkv, D]   memory, pages in logical order
    """
    q: object
    k_host: object
    v_host: object


def make_ring_layer(layer: int, device, L: int | None = None) -> RingLayer:
    """Seeded inputs of one layer of the 128K config (Qwen3-4B-like: 32 Q / 8 KV
    heads, head_dim 128).  The tensors (1 GB of q per layer at 128K) are drawn
    with torch's counter-based generator on the device, seed 1004 + 7919*layer,
    in the order q, k, v, window bias; values fp32 -> RoPE (NeoX, theta 1e6)
    -> local-window bias u ~ N(0, 0.5^2) per (1024-token window, KV head) added
    to q and k -> sink keys 0..3 scaled x3 -> bf16 (round to nearest even).
    The KV cache goes to pinned host memory in page layout (the history a
    layer-ring slot is filled from); q stays on the device."""
    import torch

    cfg = CONFIGS["q4b_128k"]
    L = L or cfg.L
    H, Hkv, D, Bk = cfg.H, cfg.Hkv, cfg.D, cfg.block
    gen = torch.Generator(device=device)
    gen.manual_seed(1000 + cfg.index + 7919 * layer)

    def rope(x):
        half = D // 2
        inv = 1e6 ** (-torch.arange(half, device=device, dtype=torch.float64) * 2.0 / D)
        ang = torch.arange(L, device=device, dtype=torch.float64)[:, None] * inv[None, :]
        cos, sin = torch.cos(ang).float(), torch.sin(ang).float()
        x1, x2 = x[..., :half], x[..., half:]
        return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], dim=-1)

    q = rope(torch.randn((H, L, D), generator=gen, device=device))
    k = rope(torch.randn((Hkv, L, D), generator=gen, device=device))
    v = torch.randn((Hkv, L, D), generator=gen, device=device)
    nwin = (L + 1023) // 1024
    u = 0.5 * torch.randn((Hkv, nwin, D), generator=gen, device=device)
    win = torch.arange(L, device=device) // 1024
    k += u[:, win, :]
    q += u.repeat_interleave(H // Hkv, dim=0)[:, win, :]
    k[:, 0:4, :] *= 3.0
    qb = q.to(torch.bfloat16)
    del q

    def to_host_pages(x):
        pages = x.to(torch.bfloat16).reshape(Hkv, L // Bk, Bk, D).permute(1, 2, 0, 3)
        host = torch.empty(pages.shape, dtype=torch.bfloat16, pin_memory=True)
        host.copy_(pages)
        return host

    return RingLayer(qb, to_host_pages(k), to_host_pages(v))
