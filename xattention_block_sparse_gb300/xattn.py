"""ctypes binding of libxattn (include/xattn.h), same names as the C ABI.

Argument marshalling only: tensors are passed as raw pointers of torch CUDA
tensors and every step runs in the library's kernels.  The library must have
been built (``__graft_entry__.build()`` or ``python -m
xattention_block_sparse_gb300.build``); a missing library raises, there is no
other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(os.path.abspath(os.environ["XATTN_BUILD_DIR"]) if os.environ.get(
    "XATTN_BUILD_DIR") else os.path.join(_PKG, "_build"), "libxattn.so")

XATTN_MAX_REQUESTS = 64
XATTN_MAX_BLOCKS_PER_ROW = 8192
XATTN_NOALLOC_MAX_COUNTERS = 262144

STATUS = {0: "XATTN_OK", -1: "XATTN_EINVAL", -2: "XATTN_EALIGN", -3: "XATTN_EPAGE",
          -4: "XATTN_ECUDA", -5: "XATTN_EUNSUPPORTED", -6: "XATTN_EWORKSPACE",
          -7: "XATTN_ETIMEOUT"}

EXPORTED = ["xattn_workspace_size", "xattn_block_sums_count", "xattn_block_sums_offset",
            "xattn_estimate", "xattn_estimate_seq", "xattn_estimate_sampled", "xattn_select",
            "xattn_select_per_kv_head",
            "xattn_select_noalloc", "bsa_chunk_attention", "bsa_chunk_attention_per_kv_head",
            "lse_merge", "xattn_store_kv",
            "xattn_device_error", "xattn_last_device_error", "xattn_copy_rows_async",
            "xattn_status_string"]


class XattnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class xattn_problem(ctypes.Structure):
    _fields_ = [
        ("num_requests", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("stride", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("cu_seqlens_q", ctypes.POINTER(ctypes.c_int32)),
        ("cu_seqlens_kh", ctypes.POINTER(ctypes.c_int32)),
        ("block_table", ctypes.c_void_p),
        ("bt_stride", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("q_head_stride", ctypes.c_int64),
        ("kv_head_stride", ctypes.c_int64),
        ("lse_head_stride", ctypes.c_int64),
        ("kv_token_stride", ctypes.c_int64),
    ]


_lib = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Open libxattn (once) and declare its signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise FileNotFoundError(
            f"libxattn not built ({p} missing): run __graft_entry__.build() first")
    lib = ctypes.CDLL(p)
    P = ctypes.POINTER(xattn_problem)
    vp, i32, i64, f32, f64, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                  ctypes.c_float, ctypes.c_double, ctypes.c_size_t)
    sig = {
        "xattn_workspace_size": (sz, [P]),
        "xattn_block_sums_count": (sz, [P]),
        "xattn_block_sums_offset": (sz, [P, i32]),
        "xattn_estimate": (ctypes.c_int, [P, vp, vp, vp, f32, vp, sz, vp, vp]),
        "xattn_estimate_seq": (ctypes.c_int, [P, vp, vp, i64, i64, ctypes.POINTER(i64), f32, vp,
                                               sz, vp, vp]),
        "xattn_estimate_sampled": (ctypes.c_int, [P, vp, vp, i64, i64, ctypes.POINTER(i64), i32,
                                                   f32, vp, sz, vp, vp]),
        "xattn_select": (ctypes.c_int, [P, vp, f64, i32, i32, i32, vp, sz, vp, vp, vp, vp, vp]),
        "xattn_select_per_kv_head": (ctypes.c_int, [P, vp, f64, i32, i32, i32, vp, sz, vp, vp, vp,
                                                     vp, vp]),
        "xattn_select_noalloc": (ctypes.c_int, [P, vp, f64, i32, i32, i32, vp, vp, vp, vp, vp]),
        "bsa_chunk_attention": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, f32, vp, sz, vp, vp,
                                                vp]),
        "bsa_chunk_attention_per_kv_head": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, f32, vp,
                                                            sz, vp, vp, vp]),
        "lse_merge": (ctypes.c_int, [vp, vp, vp, vp, i64, i32, vp, i32, vp, vp]),
        "xattn_store_kv": (ctypes.c_int, [P, vp, vp, vp, vp, vp]),
        "xattn_device_error": (ctypes.c_int, [vp, ctypes.POINTER(i32), i32]),
        "xattn_last_device_error": (ctypes.c_int, [vp, ctypes.POINTER(i32)]),
        "xattn_copy_rows_async": (ctypes.c_int, [vp, i64, vp, i64, i64, i64, i32, vp]),
        "xattn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


# ---------------------------------------------------------------------------
# Problem description
# ---------------------------------------------------------------------------


class Problem:
    """Host-side xattn_problem plus the host arrays it points to.

    q_lens / kh_lens: per-request query-chunk and history token counts;
    block_table: DEVICE int32 tensor [B, bt_stride] (or None without history);
    strides are element strides between heads of q/o, k_cur/v_cur and lse, and
    between tokens of k_cur/v_cur (None: head_dim, the [Hkv, tokens, D] layout)."""

    def __init__(self, num_heads, num_kv_heads, head_dim, stride, block_size, q_lens, kh_lens,
                 block_table=None, num_pages=0, q_head_stride=None, kv_head_stride=None,
                 lse_head_stride=None, kv_token_stride=None):
        self.q_lens = [int(x) for x in q_lens]
        self.kh_lens = [int(x) for x in kh_lens]
        B = len(self.q_lens)
        self.cu_q = np.zeros(B + 1, dtype=np.int32)
        self.cu_kh = np.zeros(B + 1, dtype=np.int32)
        self.cu_q[1:] = np.cumsum(self.q_lens)
        self.cu_kh[1:] = np.cumsum(self.kh_lens)
        tot = int(self.cu_q[-1])
        self.block_table = block_table
        bt_ptr, bt_stride = None, 0
        if block_table is not None:
            assert block_table.dtype.__str__().endswith("int32") and block_table.dim() == 2
            assert block_table.stride(1) == 1
            bt_ptr, bt_stride = block_table.data_ptr(), block_table.stride(0)
        self.c = xattn_problem(
            B, num_heads, num_kv_heads, head_dim, stride, block_size,
            self.cu_q.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            self.cu_kh.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            bt_ptr, bt_stride, num_pages,
            q_head_stride if q_head_stride is not None else tot * head_dim,
            kv_head_stride if kv_head_stride is not None else tot * head_dim,
            lse_head_stride if lse_head_stride is not None else tot,
            kv_token_stride if kv_token_stride is not None else 0)

    @property
    def B(self):
        return self.c.num_requests

    @property
    def bt_stride(self):
        return self.c.bt_stride

    def ref(self):
        return ctypes.byref(self.c)


_BF16, _F32, _I32, _U8 = "torch.bfloat16", "torch.float32", "torch.int32", "torch.uint8"


def _dev(t, what, *dtypes):
    """Device pointer of tensor t, after checking that it lives on a GPU and has
    one of the element types the header gives for the argument: a host
    pointer handed to a kernel would be read as device memory.  None passes
    through (the library answers XATTN_EINVAL where it needs the pointer)."""
    if t is None:
        return None
    if not getattr(t, "is_cuda", False):
        raise ValueError(f"{what}: a CUDA tensor is required (the kernels read it on the GPU)")
    if dtypes and str(t.dtype) not in dtypes:
        raise TypeError(f"{what}: element type {t.dtype}, expected {' or '.join(dtypes)}")
    return ctypes.c_void_p(t.data_ptr())


def _out(t, what, *dtypes):
    """Address of an attention output: a CUDA tensor, or a pinned CPU tensor
    that the kernel writes over the host link (the library resolves its device
    alias and refuses pageable memory)."""
    if t is not None and not getattr(t, "is_cuda", False):
        if not t.is_pinned():
            raise ValueError(f"{what}: a CUDA tensor or a pinned CPU tensor is required")
        if dtypes and str(t.dtype) not in dtypes:
            raise TypeError(f"{what}: element type {t.dtype}, expected {' or '.join(dtypes)}")
        return ctypes.c_void_p(t.data_ptr())
    return _dev(t, what, *dtypes)


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(status, what):
    if status != 0:
        raise XattnError(status, what)


# ---------------------------------------------------------------------------
# Entry points (same names as the C ABI)
# ---------------------------------------------------------------------------


def xattn_workspace_size(problem: Problem) -> int:
    return int(load_library().xattn_workspace_size(problem.ref()))


def xattn_block_sums_count(problem: Problem) -> int:
    return int(load_library().xattn_block_sums_count(problem.ref()))


def xattn_block_sums_offset(problem: Problem, r: int) -> int:
    return int(load_library().xattn_block_sums_offset(problem.ref(), r))


def xattn_estimate(problem, q, k_cur, k_pool, scale, workspace, block_sums, stream=None):
    st = load_library().xattn_estimate(problem.ref(), _dev(q, "q", _BF16),
                                       _dev(k_cur, "k_cur", _BF16), _dev(k_pool, "k_pool", _BF16),
                                       float(scale), _dev(workspace, "workspace"),
                                       workspace.numel() * workspace.element_size(),
                                       _dev(block_sums, "block_sums", _F32), _stream(stream))
    _check(st, "xattn_estimate")


def xattn_estimate_seq(problem, q, k_seq, k_seq_starts, scale, workspace, block_sums,
                       stream=None, head_stride=None, token_stride=0):
    """xattn_estimate over keys in logical token order: request r's history and
    current keys are tokens [k_seq_starts[r], ...) of k_seq.  k_seq is a
    [Hkv, tokens, D] tensor unless head_stride / token_stride say otherwise."""
    starts = np.ascontiguousarray(np.asarray(k_seq_starts, dtype=np.int64))
    hs = k_seq.stride(0) if head_stride is None else int(head_stride)
    st = load_library().xattn_estimate_seq(problem.ref(), _dev(q, "q", _BF16),
                                           _dev(k_seq, "k_seq", _BF16), hs, int(token_stride),
                                           starts.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                           float(scale), _dev(workspace, "workspace"),
                                           workspace.numel() * workspace.element_size(),
                                           _dev(block_sums, "block_sums", _F32), _stream(stream))
    _check(st, "xattn_estimate_seq")


def xattn_estimate_sampled(problem, q, k_seq, k_seq_starts, samples, scale, workspace,
                           block_sums, stream=None, head_stride=None, token_stride=0):
    """xattn_estimate_seq scoring only the first `samples` reshaped columns of
    each history block (each weighted Br/samples)."""
    starts = np.ascontiguousarray(np.asarray(k_seq_starts, dtype=np.int64))
    hs = k_seq.stride(0) if head_stride is None else int(head_stride)
    st = load_library().xattn_estimate_sampled(
        problem.ref(), _dev(q, "q", _BF16), _dev(k_seq, "k_seq", _BF16), hs, int(token_stride),
        starts.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), int(samples), float(scale),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _dev(block_sums, "block_sums", _F32), _stream(stream))
    _check(st, "xattn_estimate_sampled")


def xattn_select(problem, block_sums, threshold, workspace, mask, sel_idx, sel_page, n_sel,
                 stream=None, vote=(1, 2), force_sink_last=True):
    """vote = (num, den): a history block is selected when its votes exceed
    num/den of the (KV head, query block) pairs; (1, 2) is the strict majority."""
    st = load_library().xattn_select(problem.ref(), _dev(block_sums, "block_sums", _F32),
                                     float(threshold),
                                     int(vote[0]), int(vote[1]), int(bool(force_sink_last)),
                                     _dev(workspace, "workspace"),
                                     workspace.numel() * workspace.element_size(),
                                     _dev(mask, "mask", _U8), _dev(sel_idx, "sel_idx", _I32),
                                     _dev(sel_page, "sel_page", _I32), _dev(n_sel, "n_sel", _I32),
                                     _stream(stream))
    _check(st, "xattn_select")


def xattn_select_per_kv_head(problem, block_sums, threshold, workspace, mask, sel_idx, sel_page,
                             n_sel, stream=None, vote=(1, 2), force_sink_last=True):
    """One block set per KV head: sel_idx / sel_page [B, Hkv, bt_stride], n_sel
    [B, Hkv]; KV head k keeps a block its own query blocks vote for by more
    than num/den."""
    st = load_library().xattn_select_per_kv_head(
        problem.ref(), _dev(block_sums, "block_sums", _F32), float(threshold), int(vote[0]),
        int(vote[1]), int(bool(force_sink_last)), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _dev(mask, "mask", _U8),
        _dev(sel_idx, "sel_idx", _I32), _dev(sel_page, "sel_page", _I32),
        _dev(n_sel, "n_sel", _I32), _stream(stream))
    _check(st, "xattn_select_per_kv_head")


def xattn_select_noalloc(problem, block_sums, threshold, mask, sel_idx, sel_page, n_sel,
                         stream=None, vote=(1, 2), force_sink_last=True):
    """xattn_select without a workspace, for callers that cannot allocate device
    memory on the prefill path; its vote counters live in a fixed array inside
    the library (one per GPU), so calls that overlap on the GPU race."""
    st = load_library().xattn_select_noalloc(problem.ref(),
                                             _dev(block_sums, "block_sums", _F32),
                                             float(threshold), int(vote[0]), int(vote[1]),
                                             int(bool(force_sink_last)),
                                             _dev(mask, "mask", _U8),
                                             _dev(sel_idx, "sel_idx", _I32),
                                             _dev(sel_page, "sel_page", _I32),
                                             _dev(n_sel, "n_sel", _I32), _stream(stream))
    _check(st, "xattn_select_noalloc")


def bsa_chunk_attention(problem, q, k_cur, v_cur, k_pool, v_pool, sel_page, n_sel, softmax_scale,
                        workspace, o, lse, stream=None):
    st = load_library().bsa_chunk_attention(problem.ref(), _dev(q, "q", _BF16),
                                            _dev(k_cur, "k_cur", _BF16),
                                            _dev(v_cur, "v_cur", _BF16),
                                            _dev(k_pool, "k_pool", _BF16),
                                            _dev(v_pool, "v_pool", _BF16),
                                            _dev(sel_page, "sel_page", _I32),
                                            _dev(n_sel, "n_sel", _I32), float(softmax_scale),
                                            _dev(workspace, "workspace"),
                                            workspace.numel() * workspace.element_size(),
                                            _out(o, "o", _BF16), _out(lse, "lse", _F32),
                                            _stream(stream))
    _check(st, "bsa_chunk_attention")


def bsa_chunk_attention_per_kv_head(problem, q, k_cur, v_cur, k_pool, v_pool, sel_page, n_sel,
                                    softmax_scale, workspace, o, lse, stream=None):
    """bsa_chunk_attention over a selection per KV head (sel_page [B, Hkv,
    bt_stride], n_sel [B, Hkv])."""
    st = load_library().bsa_chunk_attention_per_kv_head(
        problem.ref(), _dev(q, "q", _BF16), _dev(k_cur, "k_cur", _BF16),
        _dev(v_cur, "v_cur", _BF16), _dev(k_pool, "k_pool", _BF16), _dev(v_pool, "v_pool", _BF16),
        _dev(sel_page, "sel_page", _I32), _dev(n_sel, "n_sel", _I32), float(softmax_scale),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _out(o, "o", _BF16), _out(lse, "lse", _F32), _stream(stream))
    _check(st, "bsa_chunk_attention_per_kv_head")


def lse_merge(o1, lse1, o2, lse2, o_out, lse_out, stream=None):
    rows, d = o1.shape[0], o1.shape[-1]
    bf16 = 1 if str(o_out.dtype).endswith("bfloat16") else 0
    st = load_library().lse_merge(_dev(o1, "o1", _F32), _dev(lse1, "lse1", _F32),
                                  _dev(o2, "o2", _F32), _dev(lse2, "lse2", _F32), rows, d,
                                  _dev(o_out, "o_out", _BF16, _F32), bf16,
                                  _dev(lse_out, "lse_out", _F32), _stream(stream))
    _check(st, "lse_merge")


def xattn_device_error(stream=None, clear: bool = True) -> int:
    code = ctypes.c_int32(0)
    st = load_library().xattn_device_error(_stream(stream), ctypes.byref(code), 1 if clear else 0)
    _check(st, "xattn_device_error")
    return int(code.value)


def xattn_last_device_error(stream=None) -> int:
    code = ctypes.c_int32(0)
    st = load_library().xattn_last_device_error(_stream(stream), ctypes.byref(code))
    _check(st, "xattn_last_device_error")
    return int(code.value)


def xattn_store_kv(problem, k_cur, v_cur, k_pool, v_pool, stream=None):
    """Write the chunk's K/V (views with the problem's kv_head_stride and
    kv_token_stride) into the pool pages the block table gives their positions."""
    st = load_library().xattn_store_kv(problem.ref(), _dev(k_cur, "k_cur", _BF16),
                                       _dev(v_cur, "v_cur", _BF16),
                                       _dev(k_pool, "k_pool", _BF16),
                                       _dev(v_pool, "v_pool", _BF16), _stream(stream))
    _check(st, "xattn_store_kv")


def copy_window_async(dst, src, t0, t1, stream=None):
    """dst[:, t0:t1] = src[:, t0:t1] for [rows, L, ...] tensors on opposite sides
    (one side pinned host, the other device), as one 2-D copy on `stream`."""
    to_device = 1 if dst.is_cuda else 0
    if dst.is_cuda == src.is_cuda:
        raise ValueError("copy_window_async copies between host and device")
    if dst.shape != src.shape or not dst.is_contiguous() or not src.is_contiguous():
        raise ValueError("copy_window_async wants two contiguous tensors of one shape")
    row = dst[0].numel() * dst.element_size()          # bytes of one leading row
    per_t = dst[0, 0].numel() * dst.element_size()     # bytes of one token
    off = t0 * per_t
    st = load_library().xattn_copy_rows_async(
        ctypes.c_void_p(dst.data_ptr() + off), row, ctypes.c_void_p(src.data_ptr() + off), row,
        (t1 - t0) * per_t, dst.shape[0], to_device, _stream(stream))
    _check(st, "xattn_copy_rows_async")


def xattn_status_string(status: int) -> str:
    return load_library().xattn_status_string(status).decode()
