"""bsa_chunk_attention on its own, on shapes that drive each of its schedules:

* stream-K with a unit split over many CTAs (the merge of more than five
  parts, from global memory),
* stream-K with units split over two or three CTAs (the merge that keeps the
  last CTA's own part in tensor memory),
* a ragged last unit (128 rows: no second query tile), head_dim 64 with
  64-key tiles,
* one whole unit per CTA (a small launch).

Every case uses a hand-made selection (a random ascending subset of the
history pages, pages permuted in the pool) and compares sampled rows of every
head -- including the first and last row of each 128-row tile -- with the
float64 oracle."""
import math

import numpy as np
import pytest
import torch

from oracle import xattn_oracle as O
from xattention_block_sparse_gb300 import inputs as I
from xattention_block_sparse_gb300 import xattn as X

from gpu_common import check_attention, dev, to_dev_bf16

pytestmark = pytest.mark.gpu

CASES = {
    # name: H, Hkv, D, block, stride, lq, history pages, selected pages
    "one_unit_over_many_ctas": (2, 1, 128, 128, 8, 256, 96, 96),
    "units_over_two_or_three_ctas": (32, 8, 128, 128, 8, 512, 60, 45),
    "ragged_last_unit": (4, 2, 128, 128, 8, 640, 12, 7),
    "head_dim_64_block_64": (2, 2, 64, 64, 8, 384, 150, 150),
    "whole_units": (16, 8, 128, 128, 8, 4096, 8, 3),
}


def _bits_to_f64(bits):
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("name", list(CASES))
def test_attention_schedule_parity(name):
    H, Hkv, D, Bk, S, lq, n_hist, n_sel = CASES[name]
    d = dev()
    rng = np.random.default_rng(100 + list(CASES).index(name))
    P = n_hist + 4
    q = I.bf16_round(rng.standard_normal((H, lq, D), dtype=np.float32))
    kc = I.bf16_round(rng.standard_normal((Hkv, lq, D), dtype=np.float32))
    vc = I.bf16_round(rng.standard_normal((Hkv, lq, D), dtype=np.float32))
    kp = I.bf16_round(rng.standard_normal((P, Bk, Hkv, D), dtype=np.float32))
    vp = I.bf16_round(rng.standard_normal((P, Bk, Hkv, D), dtype=np.float32))
    perm = rng.permutation(P).astype(np.int32)
    bt = perm[None, :n_hist].copy()
    logical = np.sort(rng.choice(n_hist, size=n_sel, replace=False))
    pages = bt[0, logical]

    BT = torch.from_numpy(bt).to(d)
    prob = X.Problem(H, Hkv, D, S, Bk, [lq], [n_hist * Bk], BT, P)
    ws = torch.empty(max(X.xattn_workspace_size(prob), 256), dtype=torch.uint8, device=d)
    sel_page = torch.full((1, bt.shape[1]), -7, dtype=torch.int32, device=d)
    sel_page[0, :n_sel] = torch.from_numpy(pages.astype(np.int32)).to(d)
    n_sel_t = torch.tensor([n_sel], dtype=torch.int32, device=d)
    O_ = torch.zeros((H, lq, D), dtype=torch.bfloat16, device=d)
    LSE = torch.zeros((H, lq), dtype=torch.float32, device=d)
    scale = 1.0 / math.sqrt(D)
    X.bsa_chunk_attention(prob, to_dev_bf16(q), to_dev_bf16(kc), to_dev_bf16(vc), to_dev_bf16(kp),
                          to_dev_bf16(vp), sel_page, n_sel_t, scale, ws, O_, LSE)
    torch.cuda.synchronize()
    assert X.xattn_device_error() == 0

    edges = {e for m in range(0, lq, 128) for e in (m, m + 1, m + 126, m + 127)}
    rows = sorted({r for r in edges if r < lq} | set(rng.integers(0, lq, 16).tolist()))
    o_ref, l_ref = O.attend_request(_bits_to_f64(q), _bits_to_f64(kc), _bits_to_f64(vc),
                                    _bits_to_f64(kp), _bits_to_f64(vp), pages, H, Hkv, scale,
                                    rows=rows)
    idx = np.asarray(rows)
    og = O_.float().cpu().numpy()[:, idx].astype(np.float64)
    lg = LSE.cpu().numpy()[:, idx]
    check_attention(og, lg, o_ref, l_ref, name)
