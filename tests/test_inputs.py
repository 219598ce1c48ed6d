"""The seeded input generator: bf16 rounding, determinism and paging layout."""
import numpy as np
import torch

from xattention_block_sparse_gb300 import inputs as I


def test_bf16_round_matches_torch_rne():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(10000).astype(np.float32),
                        np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -2.5, 0.0, 65504.0],
                                 dtype=np.float32)])
    ours = I.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert ours[-6:-3].tolist() == [0x3F80, 0x3F80, 0x3F82]   # ties to even
    back = I.bf16_bits_to_f64(ours)
    assert np.array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16)
                          .to(torch.float64).numpy())


def test_workload_is_deterministic_and_paged_correctly():
    a = I.make_workload("tiny")
    b = I.make_workload("tiny")
    assert np.array_equal(a.q_bits, b.q_bits) and np.array_equal(a.kpool_bits, b.kpool_bits)
    cfg = a.cfg
    assert a.q_bits.shape == (cfg.H, cfg.L, cfg.D)
    assert a.k_bits.shape == (cfg.Hkv, cfg.L, cfg.D)
    bt = a.block_table[0]
    # logical page j of the sequence sits at physical page bt[j]
    for j in range(cfg.L // cfg.block):
        for kvh in range(cfg.Hkv):
            assert np.array_equal(a.kpool_bits[bt[j], :, kvh, :],
                                  a.k_bits[kvh, j * cfg.block:(j + 1) * cfg.block, :])
    assert sorted(bt.tolist()) == list(range(cfg.L // cfg.block))
    calls = a.calls
    assert [c.kh_lens[0] for c in calls] == [0, 256, 512, 768]
    assert [c.tok_base for c in calls] == [0, 256, 512, 768]


def test_varlen_block_table_layout():
    w = I.make_workload("varlen")
    bt = w.block_table
    assert bt.shape == (3, 512)
    assert (bt[0] == -1).all()
    assert (bt[1, :128] >= 0).all() and (bt[1, 128:] == -1).all()
    assert (bt[2] >= 0).all()
    used = np.concatenate([bt[1, :128], bt[2]])
    assert len(set(used.tolist())) == 640
    c = w.calls[0]
    assert c.cu_q.tolist() == [0, 8192, 11264, 12288]
    assert c.cu_kh.tolist() == [0, 0, 16384, 81920]
