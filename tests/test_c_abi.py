"""The C ABI used from C: include/xattn.h compiles as strict C99, a C program
that takes the address of every entry point links against libxattn.so with no
undefined symbol, and its host-side calls (sizes, validation, status strings)
give what the Python binding gives.

Only calls that return before any CUDA runtime call are made, so this runs
on a machine without a GPU."""
import os
import re
import shutil
import subprocess

import pytest

from xattention_block_sparse_gb300 import build as B
from xattention_block_sparse_gb300 import xattn as X

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "xattn.h")


def _declared():
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:size_t|xattn_status|const char \*)\s*(\w+)\s*\(",
                                 src, flags=re.M)))


PROGRAM_HEAD = r"""
#include <stdio.h>
#include "xattn.h"

typedef void (*any_fn)(void);
"""

PROGRAM_MAIN = r"""
int main(void) {
  /* two requests: 1024 queries over 2048 history tokens, 512 queries alone */
  const int32_t cu_q[3] = {0, 1024, 1536};
  const int32_t cu_kh[3] = {0, 2048, 2048};
  xattn_problem p;
  size_t i;
  p.num_requests = 2; p.num_heads = 16; p.num_kv_heads = 8; p.head_dim = 128;
  p.stride = 8; p.block_size = 128;
  p.cu_seqlens_q = cu_q; p.cu_seqlens_kh = cu_kh;
  p.block_table = (const int32_t *)0x10000;   /* device pointer: never read on the host */
  p.bt_stride = 64; p.num_pages = 256;
  p.q_head_stride = 1536 * 128; p.kv_head_stride = 1536 * 128; p.lse_head_stride = 1536;
  p.kv_token_stride = 0;

  for (i = 0; i < sizeof(entry_points) / sizeof(entry_points[0]); ++i)
    if (!entry_points[i]) return 2;

  printf("workspace %zu\n", xattn_workspace_size(&p));
  printf("block_sums %zu\n", xattn_block_sums_count(&p));
  printf("offset1 %zu\n", xattn_block_sums_offset(&p, 1));
  printf("estimate_null_q %d\n",
         (int)xattn_estimate(&p, NULL, NULL, NULL, 0.01f, NULL, 0, NULL, NULL));
  printf("select_bad_vote %d\n",
         (int)xattn_select(&p, NULL, 0.9, 3, 2, 1, NULL, 0, NULL, NULL, NULL, NULL, NULL));
  printf("merge_null %d\n",
         (int)lse_merge(NULL, NULL, NULL, NULL, 4, 128, NULL, 1, NULL, NULL));
  p.head_dim = 96;
  printf("workspace_bad_dim %zu\n", xattn_workspace_size(&p));
  printf("estimate_bad_dim %d\n",
         (int)xattn_estimate(&p, NULL, NULL, NULL, 0.01f, NULL, 0, NULL, NULL));
  printf("status %s\n", xattn_status_string(XATTN_EPAGE));
  return 0;
}
"""


def _program():
    names = _declared()
    table = ",\n".join(f"  (any_fn){n}" for n in names)
    return PROGRAM_HEAD + f"static const any_fn entry_points[] = {{\n{table}\n}};\n" + PROGRAM_MAIN


@pytest.fixture(scope="module")
def c_run():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    so = B.build()
    libdir = os.path.dirname(so)
    d = os.path.join(libdir, "c_abi_check")     # in-tree build folder, git-ignored
    os.makedirs(d, exist_ok=True)
    src = os.path.join(d, "prog.c")
    with open(src, "w") as f:
        f.write(_program())
    exe = os.path.join(d, "prog")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), src, "-L", libdir, "-lxattn",
           f"-Wl,-rpath,{libdir}", "-Wl,--unresolved-symbols=report-all", "-o", exe]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    out = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stdout + out.stderr
    return dict(line.split(" ", 1) for line in out.stdout.strip().splitlines())


def test_header_compiles_as_c99_and_every_entry_point_links(c_run):
    names = _declared()
    for core in ("xattn_workspace_size", "xattn_estimate", "xattn_select", "bsa_chunk_attention",
                 "lse_merge", "xattn_store_kv", "xattn_last_device_error"):
        assert core in names
    assert set(names) == set(X.EXPORTED)


def test_c_caller_sees_the_bindings_sizes(c_run):
    prob = X.Problem(16, 8, 128, 8, 128, [1024, 512], [2048, 0], _FakeBT(), 256,
                     q_head_stride=1536 * 128, kv_head_stride=1536 * 128, lse_head_stride=1536)
    assert int(c_run["workspace"]) == X.xattn_workspace_size(prob) > 0
    assert int(c_run["block_sums"]) == X.xattn_block_sums_count(prob)
    # request 0: 16 heads x 8 query blocks x (16 + 8) blocks precede request 1
    assert int(c_run["offset1"]) == 16 * 8 * 24
    assert int(c_run["block_sums"]) == 16 * 8 * 24 + 16 * 4 * 4


def test_c_caller_gets_validation_errors_before_any_launch(c_run):
    assert int(c_run["estimate_null_q"]) == -1        # XATTN_EINVAL
    assert int(c_run["select_bad_vote"]) == -1        # vote_num > vote_den, null outputs
    assert int(c_run["merge_null"]) == -1
    assert int(c_run["workspace_bad_dim"]) == 0       # invalid problem: size 0
    assert int(c_run["estimate_bad_dim"]) == -5       # XATTN_EUNSUPPORTED
    assert c_run["status"].strip()


class _FakeBT:
    """A device block table stand-in: only its pointer and row pitch are read."""
    dtype = "torch.int32"

    def dim(self):
        return 2

    def stride(self, i):
        return (64, 1)[i]

    def data_ptr(self):
        return 0x10000
