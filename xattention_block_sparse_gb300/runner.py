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


def prefill_chunk(problem, q, k_cur, v_cur, k_pool, v_pool, tau, bufs: ChunkBuffers, o, lse,
                  est_scale=None, softmax_scale=None, stream=None):
    """One chunk of XAttention BSA prefill: estimate, select, attend."""
    D = problem.c.head_dim
    est_scale = estimation_scale(D, problem.c.stride) if est_scale is None else est_scale
    softmax_scale = 1.0 / math.sqrt(D) if softmax_scale is None else softmax_scale
    X.xattn_estimate(problem, q, k_cur, k_pool, est_scale, bufs.workspace, bufs.block_sums,
                     stream)
    X.xattn_select(problem, bufs.block_sums, tau, bufs.workspace, bufs.mask, bufs.sel_idx,
                   bufs.sel_page, bufs.n_sel, stream)
    X.bsa_chunk_attention(problem, q, k_cur, v_cur, k_pool, v_pool, bufs.sel_page, bufs.n_sel,
                          softmax_scale, o, lse, stream)


class SequencePrefill:
    """Chunked prefill of one sequence of length L in chunks of `chunk` tokens.

    Q [H, L, D], K/V [Hkv, L, D] (current-chunk views are windows of these),
    pools [P, Bk, Hkv, D] and block_table [1, P] as device tensors.  Chunk c
    queries tokens [c*chunk, (c+1)*chunk) and reads history [0, c*chunk)
    through the block table."""

    def __init__(self, H, Hkv, D, stride, block, L, chunk, block_table, num_pages,
                 with_mask=False):
        self.H, self.Hkv, self.D, self.L, self.chunk = H, Hkv, D, L, chunk
        self.problems = [
            X.Problem(H, Hkv, D, stride, block, [chunk], [c * chunk], block_table, num_pages,
                      q_head_stride=L * D, kv_head_stride=L * D, lse_head_stride=L)
            for c in range(L // chunk)]
        self.bufs = ChunkBuffers.for_problems(self.problems, block_table.device, with_mask)

    def run_chunk(self, c, Q, K, V, kpool, vpool, tau, O, LSE, stream=None):
        t0 = c * self.chunk
        prefill_chunk(self.problems[c], Q[:, t0:], K[:, t0:], V[:, t0:], kpool, vpool, tau,
                      self.bufs, O[:, t0:], LSE[:, t0:], stream=stream)

    def run(self, Q, K, V, kpool, vpool, tau, O, LSE, stream=None, on_chunk=None):
        for c in range(len(self.problems)):
            self.run_chunk(c, Q, K, V, kpool, vpool, tau, O, LSE, stream)
            if on_chunk is not None:
                on_chunk(c, self.bufs)
