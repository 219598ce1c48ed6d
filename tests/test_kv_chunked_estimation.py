"""KV-chunked estimation selects what one-shot estimation selects.

"XAttention Offload Stream Synchronization Fix" (测试结果, Density 对齐验证)
compares the offload mode, whose estimation takes softmax statistics per KV
chunk and merges them, with a GPU-only mode that processes all KV at once,
and puts their ~3% density gap down to the two ways of accumulating KV.  The
merge is exact arithmetic (m = max m_i, l = sum l_i e^(m_i - m)), so on the
same inputs the two ways give the same block sums up to rounding, and the
same selection.  This test shows it on a seeded 4K workload with the KV
history cut into the pages' 4096-token estimation chunks scaled down to
1024 tokens; the pages' gap compares two different models."""
import numpy as np

from oracle import xattn_oracle as O
from xattention_block_sparse_gb300 import inputs as I


def test_kv_chunked_statistics_select_the_one_shot_blocks():
    wl = I.make_workload("q06b_4k")
    cfg = wl.cfg
    c, chunk = 3, cfg.chunk
    t0, t1 = c * chunk, (c + 1) * chunk
    q, k, kp = wl.f64("q"), wl.f64("k"), wl.f64("kpool")
    scale = O.default_estimation_scale(cfg.D, cfg.stride)
    G = cfg.H // cfg.Hkv
    ncol = (t1) // cfg.stride
    per = 1024 // cfg.stride                       # reshaped columns per KV chunk
    cols = [(a, min(a + per, ncol)) for a in range(0, ncol, per)]
    one, chunked = [], []
    for h in range(cfg.H):
        hist = O.gather_history(kp, wl.block_table[0], t0, h // G)
        one.append(O.block_sums_one_head(q[h, t0:t1], hist, k[h // G, t0:t1], cfg.stride,
                                         cfg.block, scale))
        chunked.append(O.block_sums_chunked(q[h, t0:t1], hist, k[h // G, t0:t1], cfg.stride,
                                            cfg.block, scale, cols)[0])
    one, chunked = np.stack(one), np.stack(chunked)
    assert len(cols) == 4
    assert np.allclose(one, chunked, rtol=1e-12, atol=0)
    kbh = t0 // cfg.block
    for tau in (0.5, 0.8, 0.9):
        m1, s1, _ = O.select_request(one.astype(np.float32), tau, cfg.Hkv, kbh, wl.block_table[0])
        m2, s2, _ = O.select_request(chunked.astype(np.float32), tau, cfg.Hkv, kbh,
                                     wl.block_table[0])
        assert np.array_equal(m1, m2) and np.array_equal(s1, s2)
