"""xattn_select_noalloc: selection for callers that cannot allocate device memory.

A serving process that hands all free HBM to its KV-page pool and weights at
start-up, or a C caller with no caching allocator, cannot give the library a
scratch workspace on the prefill path.  For them xattn_select_noalloc keeps
its vote counters in a fixed device array inside the library.  It must select
exactly what xattn_select selects with a caller workspace (selection is
integer work: the match is bit for bit), call after call, although every call
reuses the same array.
"""
import ctypes

import numpy as np
import pytest

from xattention_block_sparse_gb300 import xattn as X


def _fake_problem(q_lens, kh_lens, W):
    class BT:
        dtype = "torch.int32"

        def dim(self):
            return 2

        def stride(self, i):
            return (W, 1)[i]

        def data_ptr(self):
            return 0x10000

    return X.Problem(16, 8, 128, 8, 128, q_lens, kh_lens, BT(), 4096)


def test_noalloc_rejects_sizes_beyond_its_array():
    """num_requests * bt_stride above the fixed capacity is refused on the host,
    before anything is enqueued (no device is touched)."""
    from xattention_block_sparse_gb300 import build as B
    B.build()
    lib = X.load_library()
    W = X.XATTN_NOALLOC_MAX_COUNTERS // 2 + 1
    p = _fake_problem([128, 128], [128, 128], W)
    fake = ctypes.c_void_p(0x10000)
    st = lib.xattn_select_noalloc(p.ref(), fake, 0.9, 1, 2, 1, None, fake, fake, fake, None)
    assert st == -6  # XATTN_EWORKSPACE


@pytest.mark.gpu
def test_noalloc_select_matches_workspace_select_on_consecutive_calls():
    import torch

    import __graft_entry__
    from xattention_block_sparse_gb300 import inputs as I
    from xattention_block_sparse_gb300 import runner as RN

    __graft_entry__.build()
    lib = X.load_library()
    dev = torch.device("cuda:0")
    wl = I.make_workload("q06b_4k")
    cfg = wl.cfg
    up = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).to(dev).view(
        torch.bfloat16)
    Q, K, KP = up(wl.q_bits), up(wl.k_bits), up(wl.kpool_bits)
    BT = torch.from_numpy(wl.block_table).to(dev)
    seq = RN.SequencePrefill(cfg.H, cfg.Hkv, cfg.D, cfg.stride, cfg.block, cfg.L, cfg.chunk, BT,
                             KP.shape[0], with_mask=True)
    bufs = seq.bufs
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # two calls in a row: the first votes for every block of chunk 3, the second
    # keeps only some blocks of chunk 2 -- votes left over in the shared array
    # from the first call would make the second keep them all
    for c, tau in ((3, 0.9), (2, 0.25)):
        p = seq.problems[c]
        t0 = c * cfg.chunk
        X.xattn_estimate(p, Q[:, t0:], K[:, t0:], KP, RN.estimation_scale(cfg.D, cfg.stride),
                         bufs.workspace, bufs.block_sums)
        n = X.xattn_block_sums_count(p)
        X.xattn_select(p, bufs.block_sums, tau, bufs.workspace, bufs.mask, bufs.sel_idx,
                       bufs.sel_page, bufs.n_sel)
        torch.cuda.synchronize()
        want = (bufs.mask[:n].cpu().numpy().copy(), int(bufs.n_sel[0].item()),
                bufs.sel_idx[0].cpu().numpy().copy(), bufs.sel_page[0].cpu().numpy().copy())
        mask2 = torch.full((n,), 7, dtype=torch.uint8, device=dev)
        idx2 = torch.full_like(bufs.sel_idx, -9)
        page2 = torch.full_like(bufs.sel_page, -9)
        nsel2 = torch.full_like(bufs.n_sel, -9)
        st = lib.xattn_select_noalloc(p.ref(), ptr(bufs.block_sums), ctypes.c_double(tau), 1, 2,
                                      1, ptr(mask2), ptr(idx2), ptr(page2), ptr(nsel2), stream)
        assert st == 0, X.STATUS.get(st, st)
        torch.cuda.synchronize()
        k = int(nsel2[0].item())
        assert k == want[1]
        assert np.array_equal(mask2.cpu().numpy(), want[0])
        assert np.array_equal(idx2[0, :k].cpu().numpy(), want[2][:k])
        assert np.array_equal(page2[0, :k].cpu().numpy(), want[3][:k])
        if tau < 0.5:
            assert k < c * cfg.chunk // cfg.block  # a partial selection
    assert X.xattn_device_error() == 0
