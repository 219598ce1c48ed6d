"""Helpers shared by the GPU parity tests: upload seeded inputs, run the chunked
prefill through the C-ABI and compare with the float64 oracle."""
from __future__ import annotations

import math

import numpy as np
import torch

from oracle import xattn_oracle as O
from xattention_block_sparse_gb300 import inputs as I
from xattention_block_sparse_gb300 import runner as RN
from xattention_block_sparse_gb300 import xattn as X

# Acceptance bands (block sums relative with an absolute floor tied to the row
# mass; attention output max-abs; LSE absolute).
BS_RTOL = 1e-3
BS_ATOL_PER_BR = 1e-6
O_ATOL = 2e-2
LSE_ATOL = 1e-3

# For information only: the oracle's own selection (on its float64 block sums)
# against the GPU's, per checked chunk -- (what, mask entries that differ,
# mask entries compared, history blocks selected by one side only or None when
# only sampled rows were estimated).  conftest.py prints them after the run.
FLIPS = []


def record_flips(what, ref_bs, gpu_mask, tau, Hkv=None, kbh=None, gpu_sel=None):
    """Flip count of the oracle's threshold masks on its own block sums against
    the GPU's masks on the same rows, and, given every row, of the vote."""
    own = O.threshold_select(np.asarray(ref_bs, dtype=np.float32), tau)
    mask_flips = int((own != np.asarray(gpu_mask, dtype=bool)).sum())
    sel_flips = None
    if gpu_sel is not None:
        sel = O.gqa_vote(own, Hkv, kbh)
        sel_flips = len(set(sel.tolist()) ^ set(np.asarray(gpu_sel).tolist()))
    FLIPS.append((what, mask_flips, int(own.size), sel_flips))


def dev():
    if not torch.cuda.is_available():
        raise RuntimeError("GPU test run without a CUDA device")
    return torch.device("cuda:0")


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev()).view(
        torch.bfloat16)


def check_block_sums(gpu, ref, br, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    err = np.abs(gpu - ref)
    tol = BS_RTOL * np.abs(ref) + BS_ATOL_PER_BR * br
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} block sums out of tolerance; worst "
                           f"{err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    return float((err / np.maximum(np.abs(ref), 1e-30)).max())


def check_selection(bs32, gpu_mask, gpu_sel, gpu_pages, n_sel, tau, Hkv, kbh, bt_row, what="",
                    vote=(1, 2), force=True):
    """The oracle's selection applied to the GPU's own block sums must equal the
    GPU's mask, selected block ids and pages bit for bit."""
    mask, sel, pages = O.select_request(bs32, tau, Hkv, kbh, bt_row, vote=vote, force=force)
    if gpu_mask is not None:
        diff = mask != gpu_mask.astype(bool)
        assert not diff.any(), f"{what}: mask differs in {diff.sum()} entries"
    assert n_sel == len(sel), f"{what}: n_sel {n_sel} vs oracle {len(sel)}"
    assert np.array_equal(gpu_sel[:n_sel], sel), f"{what}: selected ids differ"
    assert np.array_equal(gpu_pages[:n_sel], pages), f"{what}: selected pages differ"
    return sel, pages


def check_attention(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    o_err = np.abs(np.asarray(o_gpu, np.float64) - o_ref).max()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse_gpu), fin), f"{what}: LSE finiteness differs"
    l_err = np.abs(np.asarray(lse_gpu, np.float64)[fin] - lse_ref[fin]).max() if fin.any() else 0
    assert o_err <= O_ATOL, f"{what}: O max-abs error {o_err:.3e}"
    assert l_err <= LSE_ATOL, f"{what}: LSE abs error {l_err:.3e}"
    return float(o_err), float(l_err)


class SequenceCase:
    """A chunked single-sequence workload on the GPU, with per-chunk captures."""

    def __init__(self, name, L=None, chunk=None, layer=0):
        self.wl = I.make_workload(name, layer=layer, L=L, chunk=chunk)
        cfg = self.wl.cfg
        self.cfg = cfg
        self.L = self.wl.q_bits.shape[1]
        self.chunk = chunk or cfg.chunk
        d = dev()
        self.Q = to_dev_bf16(self.wl.q_bits)
        self.K = to_dev_bf16(self.wl.k_bits)
        self.V = to_dev_bf16(self.wl.v_bits)
        self.KP = to_dev_bf16(self.wl.kpool_bits)
        self.VP = to_dev_bf16(self.wl.vpool_bits)
        self.BT = torch.from_numpy(self.wl.block_table).to(d)
        self.seq = RN.SequencePrefill(cfg.H, cfg.Hkv, cfg.D, cfg.stride, cfg.block, self.L,
                                      self.chunk, self.BT, self.KP.shape[0], with_mask=True)

    def run(self, tau, capture=()):
        cap = {}
        H, L, D = self.cfg.H, self.L, self.cfg.D
        O_ = torch.empty((H, L, D), dtype=torch.bfloat16, device=dev())
        LSE = torch.empty((H, L), dtype=torch.float32, device=dev())

        def on_chunk(c, bufs):
            if c in capture:
                p = self.seq.problems[c]
                n = X.xattn_block_sums_count(p)
                cap[c] = dict(bs=bufs.block_sums[:n].cpu().numpy().copy(),
                              mask=bufs.mask[:n].cpu().numpy().copy(),
                              sel=bufs.sel_idx[0].cpu().numpy().copy(),
                              pages=bufs.sel_page[0].cpu().numpy().copy(),
                              n_sel=int(bufs.n_sel[0].item()))

        self.seq.run(self.Q, self.K, self.V, self.KP, self.VP, tau, O_, LSE, on_chunk=on_chunk)
        torch.cuda.synchronize()
        assert X.xattn_device_error() == 0
        return O_.float().cpu().numpy(), LSE.cpu().numpy(), cap

    def oracle_inputs(self):
        return (self.wl.f64("q"), self.wl.f64("k"), self.wl.f64("v"), self.wl.f64("kpool"),
                self.wl.f64("vpool"))

    def check_chunk(self, c, cap, O_gpu, LSE_gpu, tau, qblocks=None, rows=None):
        cfg = self.cfg
        q, k, v, kp, vp = self.oracle_inputs()
        t0, t1 = c * self.chunk, (c + 1) * self.chunk
        kh = t0
        kbh = kh // cfg.block
        qb_n = self.chunk // cfg.block
        bs32 = cap["bs"].reshape(cfg.H, qb_n, kbh + qb_n)
        br = cfg.block // cfg.stride
        scale = O.default_estimation_scale(cfg.D, cfg.stride)
        G = cfg.H // cfg.Hkv
        bt_row = self.wl.block_table[0]
        # estimation
        refs = []
        for h in range(cfg.H):
            kvh = h // G
            hist = O.gather_history(kp, bt_row, kh, kvh)
            if qblocks is None:
                ref = O.block_sums_one_head(q[h, t0:t1], hist, k[kvh, t0:t1], cfg.stride,
                                            cfg.block, scale)
                check_block_sums(bs32[h], ref, br, f"chunk {c} head {h}")
            else:
                ref = O.block_sums_qblocks(q[h, t0:t1], hist, k[kvh, t0:t1], cfg.stride,
                                           cfg.block, scale, qblocks)
                check_block_sums(bs32[h, qblocks], ref, br, f"chunk {c} head {h}")
            refs.append(ref)
        gmask = cap["mask"].reshape(bs32.shape)
        if qblocks is None:
            record_flips(f"{self.wl.cfg.name} tau {tau} chunk {c}", np.stack(refs), gmask, tau,
                         cfg.Hkv, kbh, cap["sel"][:cap["n_sel"]])
        else:
            record_flips(f"{self.wl.cfg.name} tau {tau} chunk {c} (sampled query blocks)",
                         np.stack(refs), gmask[:, qblocks], tau)
        # selection on the GPU's block sums
        sel, pages = check_selection(bs32, cap["mask"].reshape(bs32.shape), cap["sel"],
                                     cap["pages"], cap["n_sel"], tau, cfg.Hkv, kbh, bt_row,
                                     f"chunk {c}")
        # attention over that selection
        o_ref, l_ref = O.attend_request(q[:, t0:t1], k[:, t0:t1], v[:, t0:t1], kp, vp, pages,
                                        cfg.H, cfg.Hkv, 1 / math.sqrt(cfg.D), rows=rows)
        sl = slice(t0, t1) if rows is None else (t0 + np.asarray(rows))
        check_attention(O_gpu[:, sl], LSE_gpu[:, sl], o_ref, l_ref, f"chunk {c}")
        return len(sel), kbh
