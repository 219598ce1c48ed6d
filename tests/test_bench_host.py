"""Host arithmetic of bench.py, on the CPU: the algorithmic work counts behind
the roofline figures, the clock-record parsing behind the throttle check, and
the source-hash guard on the committed DRAM traffic."""
import itertools

import pytest

import bench
from xattention_block_sparse_gb300 import inputs as I


class _Cfg:
    def __init__(self, H, Hkv, D, stride, block):
        self.H, self.Hkv, self.D, self.stride, self.block = H, Hkv, D, stride, block


@pytest.mark.parametrize("S,Bk,chunk,c", [(2, 4, 8, 0), (2, 4, 8, 3), (4, 8, 16, 2)])
def test_chunk_work_counts_by_enumeration(S, Bk, chunk, c):
    """Reshaped cells and attention FLOPs counted cell by cell and key by key:
    every history cell of every reshaped row, current cells b' <= a; every
    selected history key and current keys j <= i."""
    cfg = _Cfg(H=3, Hkv=1, D=5, stride=S, block=Bk)
    Lh, Lc = c * chunk, chunk
    n_sel = Lh // Bk - (1 if Lh >= 2 * Bk else 0)          # a partial selection
    cells = 0
    for a, b in itertools.product(range(Lc // S), range((Lh + Lc) // S)):
        cells += b < Lh // S or (b - Lh // S) <= a
    keys = sum(n_sel * Bk + (i + 1) for i in range(Lc))
    w = bench.chunk_work(cfg, c, chunk, n_sel)
    assert w["cells"] == cfg.H * cells
    assert w["f_est"] == 2 * S * cfg.D * cfg.H * cells      # S*D multiply-adds per cell
    assert w["f_att"] == 4 * cfg.H * cfg.D * keys           # QK^T and PV, 2 flops each
    # key bytes: each KV head's keys once (history and chunk), bf16
    assert w["b_est"] == 2 * cfg.Hkv * cfg.D * (Lh + Lc) + 2 * cfg.H * Lc * cfg.D


def test_workload_totals_match_the_scope_tables():
    """Sums over the chunks of a whole prefill, against the per-config totals
    computed independently for the scope table: 32K config F_A1 = 2.75e11 and
    5.37e8 bytes of fp32 scores per pass (now never stored), dense-equivalent
    attention 3.85e12 + 5.50e11; 128K config F_A1 = 4.40e12, 4.30e9 score bytes,
    dense attention 1.41e14."""
    def totals(name):
        cfg = I.CONFIGS[name]
        n = cfg.L // cfg.chunk
        ws = [bench.chunk_work(cfg, c, cfg.chunk, c * cfg.chunk // cfg.block) for c in range(n)]
        hist = sum(4 * cfg.H * cfg.D * cfg.chunk * c * cfg.chunk for c in range(n))
        return (sum(w["f_est"] for w in ws), 4 * sum(w["cells"] for w in ws),
                hist, sum(w["f_att"] for w in ws) - hist)

    f1, sb, fh, fc = totals("q06b_32k")
    assert f1 == pytest.approx(2.75e11, rel=5e-3) and sb == pytest.approx(5.37e8, rel=5e-3)
    assert fh == pytest.approx(3.85e12, rel=5e-3) and fc == pytest.approx(5.50e11, rel=5e-3)
    f1, sb, fh, fc = totals("q4b_128k")
    assert f1 == pytest.approx(4.40e12, rel=5e-3) and sb == pytest.approx(4.30e9, rel=5e-3)
    assert fh + fc == pytest.approx(1.41e14, rel=5e-3)


class _Proc:
    def __init__(self, out):
        self.out = out

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.out, ""


def test_clock_record_parsing(monkeypatch):
    monkeypatch.setattr(bench.time, "sleep", lambda s: None)
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.idx = 0
    cs.proc = _Proc("0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                    "0, 2070, 2070, 1150.0, 0x4, Not Active, Not Active, Not Active, Active\n"
                    "0, 1800, 2070, 1390.5, 0x8, Active, Not Active, Not Active, Active\n"
                    "garbage line\n")
    r = cs.stop()
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0 and r["samples"] == 3
    assert r["reasons"] == ["hw_slowdown", "sw_power_cap"]
    cs.proc = None
    assert cs.stop()["sm_mhz"] is None


def test_traffic_is_reported_only_for_the_profiled_source():
    files = ("attention.cu", "tc_common.cuh", "common.cuh")
    sha = bench.source_sha(files)
    assert len(sha) == 16
    assert bench.traffic_for(files, "no_such_kernel") is None
    # a capture line whose hash is not the current source's is ignored
    real = bench.traffic_for(files, "attn_tc_kernel")
    with open(bench.os.path.join(bench.ROOT, "profiles", "traffic.txt")) as f:
        lines = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    listed = {(p[0], p[1]) for p in lines}
    assert (real is not None) == (("attn_tc_kernel", sha) in listed)
