"""Host-side checks of libxattn that need no GPU: the library builds and loads,
exports every entry point include/xattn.h declares, sizes its workspace as
documented, and rejects invalid problems before touching CUDA.

Every call below fails argument validation, which happens before any CUDA
runtime call, so nothing here can reach a device."""
import ctypes
import os
import re

import numpy as np
import pytest

from xattention_block_sparse_gb300 import build as B
from xattention_block_sparse_gb300 import xattn as X

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return X.load_library()


def _declared():
    src = open(os.path.join(ROOT, "include", "xattn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:size_t|xattn_status|const char \*)\s*(\w+)\s*\(",
                                 src, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert "xattn_estimate" in names and "bsa_chunk_attention" in names and "lse_merge" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(X.EXPORTED)


class _FakeBT:
    """Stands in for a device block table: only data_ptr/stride are read, and
    only by validation that fails first."""

    def __init__(self, B, W):
        self.dtype = "torch.int32"
        self._s = (W, 1)

    def dim(self):
        return 2

    def stride(self, i):
        return self._s[i]

    def data_ptr(self):
        return 0x10000


def _prob(q_lens, kh_lens, H=16, Hkv=8, D=128, S=8, Bk=128, W=512, pages=1024, **kw):
    return X.Problem(H, Hkv, D, S, Bk, q_lens, kh_lens, _FakeBT(len(q_lens), W), pages, **kw)


def test_workspace_and_block_sum_sizes(lib):
    # one 4096-token chunk with 28672 history tokens (last chunk of the 32K case)
    p = _prob([4096], [28672])
    H, rq, ncol = 16, 4096 // 8, 32768 // 8
    bpart = H * rq * (ncol // 16) * 4    # one float per (reshaped row, KV block of Br = 16)
    tstat = H * rq * (ncol // 128) * 8
    al = lambda x: (x + 255) // 256 * 256
    counts = al(al(bpart) + tstat)
    est = al(counts + (8 * 512 + 1) * 4)  # vote counters of every (request, KV head) +
                                          # the finishing counter
    # the attention's block (at the end of the caller's buffer): partials of
    # 160 CTAs x 2 slots x 256 rows, then two part counters per 256-row unit
    part_lse = al(160 * 2 * 256 * 128 * 4)
    att_cnt = al(part_lse + 160 * 2 * 256 * 4)
    attn = al(att_cnt + 16 * 16 * 2 * 4)
    expect = est + attn + 256  # + the slack that aligns the attention block
    assert X.xattn_workspace_size(p) == expect
    assert X.xattn_block_sums_count(p) == H * 32 * 256
    # varlen batch: slabs packed request after request
    v = _prob([8192, 3072, 1024], [0, 16384, 65536])
    sizes = [16 * 64 * 64, 16 * 24 * (128 + 24), 16 * 8 * (512 + 8)]
    assert X.xattn_block_sums_count(v) == sum(sizes)
    assert [X.xattn_block_sums_offset(v, r) for r in range(3)] == [0, sizes[0], sizes[0] + sizes[1]]


@pytest.mark.parametrize("kw", [
    dict(q_lens=[100], kh_lens=[0]),                 # not a multiple of the block
    dict(q_lens=[128], kh_lens=[64]),
    dict(q_lens=[128], kh_lens=[0], H=6, Hkv=4),     # H % Hkv
    dict(q_lens=[128], kh_lens=[0], D=96),           # head_dim not built
    dict(q_lens=[128], kh_lens=[0], S=3),            # block % stride
    dict(q_lens=[128], kh_lens=[0], S=64),           # block/stride < 8
    dict(q_lens=[128], kh_lens=[0], S=32),           # block/stride = 4 < 8
    dict(q_lens=[128], kh_lens=[128 * 600], W=512),  # history beyond the table row
    dict(q_lens=[128] * 65, kh_lens=[0] * 65),       # too many requests
    dict(q_lens=[128], kh_lens=[0], q_head_stride=100),  # head stride too small
    dict(q_lens=[128], kh_lens=[128 * 8200], W=9000),    # > 8192 blocks in a row
    dict(q_lens=[128], kh_lens=[0], kv_token_stride=100),  # token stride not 16-byte
    dict(q_lens=[128], kh_lens=[0], kv_token_stride=64),   # token stride below head_dim
    dict(q_lens=[256], kh_lens=[0], kv_head_stride=128 * 8,  # views of k_cur overlap
         kv_token_stride=128 * 4),
])
def test_invalid_problems_rejected(lib, kw):
    p = _prob(**kw)
    assert X.xattn_workspace_size(p) == 0
    fake = ctypes.c_void_p(0x10000)
    st = lib.xattn_estimate(p.ref(), fake, fake, fake, 0.1, fake, 1 << 40, fake, None)
    assert st in (-1, -5), st
    st = lib.bsa_chunk_attention(p.ref(), fake, fake, fake, fake, fake, fake, fake, 0.1, fake,
                                 1 << 40, fake, fake, None)
    assert st in (-1, -5), st


def test_entry_point_argument_errors(lib):
    p = _prob([1024], [1024])
    fake = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10002)
    # null outputs, bad threshold, unaligned pointers, small workspace
    assert lib.xattn_estimate(p.ref(), fake, fake, fake, 0.1, fake, 1 << 40, None, None) == -1
    assert lib.xattn_estimate(p.ref(), odd, fake, fake, 0.1, fake, 1 << 40, fake, None) == -2
    assert lib.xattn_estimate(p.ref(), fake, fake, fake, float("nan"), fake, 1 << 40, fake,
                              None) == -1
    assert lib.xattn_estimate(p.ref(), fake, fake, fake, 0.1, fake, 16, fake, None) == -6
    for tau in (0.0, -1.0, float("nan"), float("inf")):
        assert lib.xattn_select(p.ref(), fake, tau, 1, 2, 1, fake, 1 << 40, None, fake, fake, fake,
                                None) == -1
    assert lib.xattn_select(p.ref(), fake, 0.9, 1, 2, 1, fake, 16, None, fake, fake, fake,
                            None) == -6
    for num, den, force in ((1, 0, 1), (-1, 2, 1), (3, 2, 1), (1, 2, 2)):  # bad vote / force
        assert lib.xattn_select(p.ref(), fake, 0.9, num, den, force, fake, 1 << 40, None, fake,
                                fake, fake, None) == -1
        assert lib.xattn_select_noalloc(p.ref(), fake, 0.9, num, den, force, None, fake, fake,
                                        fake, None) == -1
    assert lib.bsa_chunk_attention(p.ref(), fake, fake, fake, fake, fake, fake, fake, 0.1, fake,
                                   1 << 40, odd, fake, None) == -2
    assert lib.bsa_chunk_attention(p.ref(), fake, fake, fake, fake, fake, fake, fake, 0.1, fake,
                                   16, fake, fake, None) == -6
    assert lib.bsa_chunk_attention(p.ref(), fake, fake, fake, fake, fake, fake, fake, 0.1, None,
                                   1 << 40, fake, fake, None) == -1
    assert lib.lse_merge(fake, fake, fake, fake, 10, 6, fake, 0, fake, None) == -1
    assert lib.lse_merge(fake, fake, fake, fake, -1, 128, fake, 0, fake, None) == -1
    assert lib.lse_merge(odd, fake, fake, fake, 10, 128, fake, 0, fake, None) == -2
    assert lib.lse_merge(None, None, None, None, 0, 128, None, 0, None, None) == 0
    assert lib.xattn_status_string(-3) == b"page id outside the pool"
    # the 2-D window copy checks its geometry before touching CUDA
    assert lib.xattn_copy_rows_async(fake, 100, fake, 100, 200, 4, 1, None) == -1  # pitch < width
    assert lib.xattn_copy_rows_async(fake, 256, fake, 256, 128, -1, 1, None) == -1
    assert lib.xattn_copy_rows_async(None, 256, fake, 256, 128, 4, 0, None) == -1
    assert lib.xattn_copy_rows_async(None, 256, None, 256, 0, 4, 0, None) == 0    # nothing to copy
    # the KV store: null pools, unaligned pointers, a block table row too short for the chunk
    assert lib.xattn_store_kv(p.ref(), fake, fake, None, fake, None) == -1
    assert lib.xattn_store_kv(p.ref(), fake, odd, fake, fake, None) == -2
    short = _prob([1024], [1024], W=15)  # 8 history + 8 chunk blocks need 16 entries
    assert lib.xattn_store_kv(short.ref(), fake, fake, fake, fake, None) == -1
    assert lib.xattn_store_kv(_prob([1024], [0], pages=0).ref(), fake, fake, fake, fake,
                              None) == -1  # no pool pages


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(FileNotFoundError):
        X.load_library(str(tmp_path / "nope.so"))


def test_sequence_prefill_chunk_problems(lib):
    """SequencePrefill's per-chunk problems on the host: chunk c queries tokens
    [c*chunk, (c+1)*chunk) with c*chunk history tokens, heads strided over the
    whole sequence, and one set of buffers sized for the largest chunk (the
    last, whose history is longest)."""
    import torch
    from xattention_block_sparse_gb300 import runner as RN
    H, Hkv, D, S, Bk, L, chunk = 16, 8, 128, 8, 128, 32768, 4096
    bt = torch.arange(L // Bk, dtype=torch.int32)[None, :]
    seq = RN.SequencePrefill(H, Hkv, D, S, Bk, L, chunk, bt, L // Bk)
    assert len(seq.problems) == L // chunk
    for c, p in enumerate(seq.problems):
        assert (p.B, p.bt_stride) == (1, L // Bk)
        assert (p.c.q_head_stride, p.c.kv_head_stride, p.c.lse_head_stride) == (L * D, L * D, L)
        assert (p.q_lens, p.kh_lens) == ([chunk], [c * chunk])
    sizes = [X.xattn_workspace_size(p) for p in seq.problems]
    assert sizes == sorted(sizes) and sizes[0] > 0
    assert seq.bufs.workspace.numel() == sizes[-1]
    assert seq.bufs.block_sums.numel() == X.xattn_block_sums_count(seq.problems[-1])
    assert tuple(seq.bufs.sel_page.shape) == (1, L // Bk) and seq.bufs.mask is None


class _DevT:
    """A GPU-tensor stand-in for the binding's checks: the checks raise before
    any library call, so its pointer is never used."""

    is_cuda = True
    shape = (4, 128)

    def __init__(self, dtype, n=16):
        self.dtype, self._n = dtype, n

    def data_ptr(self):
        return 0x20000

    def numel(self):
        return self._n

    def element_size(self):
        return 1


def test_binding_refuses_host_tensors_and_wrong_types(lib):
    """A host tensor handed to a kernel would be read as device memory, and a
    wrong element type as garbage: the binding stops both before the call."""
    import torch
    p = _prob([1024], [0])
    bf, f32, i32 = _DevT("torch.bfloat16"), _DevT("torch.float32"), _DevT("torch.int32")
    ws = _DevT("torch.uint8")
    with pytest.raises(ValueError, match="CUDA tensor"):
        X.xattn_estimate(p, torch.zeros(4, dtype=torch.bfloat16), bf, bf, 0.1, ws, f32)
    with pytest.raises(TypeError, match="q: element type"):
        X.xattn_estimate(p, f32, bf, bf, 0.1, ws, f32)
    with pytest.raises(TypeError, match="block_sums"):
        X.xattn_estimate(p, bf, bf, bf, 0.1, ws, bf)
    with pytest.raises(TypeError, match="sel_page"):
        X.xattn_select(p, f32, 0.9, ws, None, i32, f32, i32)
    with pytest.raises(TypeError, match="o: element type"):
        X.bsa_chunk_attention(p, bf, bf, bf, bf, bf, i32, i32, 0.1, ws, f32, f32)
    with pytest.raises(TypeError, match="lse_out"):
        X.lse_merge(f32, f32, f32, f32, bf, bf)
    with pytest.raises(ValueError, match="CUDA tensor"):
        X.xattn_store_kv(p, bf, bf, torch.zeros(4, dtype=torch.bfloat16), bf)


def test_runner_estimation_scale_equals_the_oracle_reading():
    """The product path's estimation scale (runner.estimation_scale, what the
    bench and the prefill driver pass to xattn_estimate) and the oracle's
    reading (default_estimation_scale, what the parity tests pass) are written
    out separately; they must agree on every workload's head size and stride,
    or the parity tests would pass while the bench selects with another scale."""
    from oracle import xattn_oracle as O
    from xattention_block_sparse_gb300 import inputs as I
    from xattention_block_sparse_gb300 import runner as RN
    for cfg in I.CONFIGS.values():
        assert RN.estimation_scale(cfg.D, cfg.stride) == O.default_estimation_scale(
            cfg.D, cfg.stride), cfg.name


def test_sampled_estimation_argument_checks(lib):
    """xattn_estimate_sampled refuses sample counts it has no kernel for and
    key ranges that do not start on a block, before touching the GPU."""
    import ctypes as C
    p = _prob([1024], [4096])
    starts = (C.c_int64 * 1)(0)
    fake = C.c_void_p(0x10000)
    # Br = 16: 4 and 8 are built; 2, 3 and 16 are not
    for bad in (2, 3, 16):
        assert lib.xattn_estimate_sampled(p.ref(), fake, fake, 128 * 5120, 0, starts, bad,
                                          0.01, fake, 1 << 30, fake, None) == -5
    assert lib.xattn_estimate_sampled(p.ref(), fake, fake, 128 * 5120, 0, starts, 0, 0.01, fake,
                                      1 << 30, fake, None) == -1
    off = (C.c_int64 * 1)(64)  # a multiple of the stride, not of the block
    assert lib.xattn_estimate_sampled(p.ref(), fake, fake, 128 * 5120, 0, off, 4, 0.01, fake,
                                      1 << 30, fake, None) == -1
