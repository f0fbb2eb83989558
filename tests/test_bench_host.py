"""Host logic of bench.py that needs no GPU: the captured-traffic lookup
reports DRAM bytes only for the kernel sources the capture was taken on."""
import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _digest():
    h = hashlib.sha256()
    for f in ("gemm.cu", "gemm_pair.cu", "common.cuh", "layout.cuh"):
        with open(os.path.join(ROOT, "nvfp4_mixture_experts_route_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def test_traffic_only_for_unchanged_sources(monkeypatch):
    entry = {"kernel": "grouped_gemm_kernel<3, 32>", "bytes": 123, "sources": _digest()}
    monkeypatch.setattr(bench, "NCU_TRAFFIC", {"decode_b8": entry})
    assert bench._traffic("decode_b8", "grouped_gemm_kernel<3, 32>") == 123
    assert bench._traffic("decode_b8", "grouped_gemm_kernel<1>") is None
    assert bench._traffic("decode_b64_zipf", "grouped_gemm_kernel<3, 32>") is None
    monkeypatch.setattr(bench, "NCU_TRAFFIC", {"decode_b8": dict(entry, sources="0" * 64)})
    assert bench._traffic("decode_b8", "grouped_gemm_kernel<3, 32>") is None


def test_recorded_traffic_matches_the_sources():
    """The committed captures were taken on the committed kernel sources, so
    the bench line carries their traffic (not null)."""
    for name, t in bench.NCU_TRAFFIC.items():
        assert t["sources"] == _digest(), name
        assert bench._traffic(name, t["kernel"]) == t["bytes"]
