"""Host-side pieces of bench.py that need no GPU: the staleness check of the
committed DRAM-traffic figure."""
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _copy_sources(tmp_path):
    src = os.path.join(ROOT, "nvfp4_mixture_experts_top_gb300", "csrc")
    dst = tmp_path / "nvfp4_mixture_experts_top_gb300" / "csrc"
    dst.mkdir(parents=True)
    for fn in ("gemm_w4a4.cu", "gemm_w4a16.cu", "common.cuh", "workitems.cuh"):
        shutil.copy(os.path.join(src, fn), dst / fn)
    return dst


def test_kernel_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    dst = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench._kernel_hash("w4a4")
    f = dst / "gemm_w4a4.cu"
    text = f.read_text()
    f.write_text("// a new comment line\n" + text.replace("\n", "\n   ", 3) + "\n/* trailing\n block */\n")
    assert bench._kernel_hash("w4a4") == h0
    f.write_text(text.replace("constexpr int KC = 256;", "constexpr int KC = 512;"))
    assert bench._kernel_hash("w4a4") != h0


def test_committed_traffic_matches_the_current_sources():
    """profiles/traffic.json was taken from the kernels as they are now, so
    the bench reports its figures rather than null."""
    for wl_, mode in (("decode_c16", "w4a4"), ("decode_b512", "w4a4"), ("decode_c16", "mxw4a4"),
                      ("decode_c16", "w4a16")):
        assert bench._traffic(wl_, mode) is not None, (wl_, mode)
