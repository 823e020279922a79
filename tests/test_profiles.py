"""The committed ncu summaries describe the committed kernels.

bench.py reports a GEMM's DRAM traffic per launch only from a summary taken on
the same kernel source and launch order (else null).  These checks keep the
summaries in step with the sources: a kernel or launch-order change without a
fresh capture fails here instead of silently nulling the bench's figure.
"""
import hashlib
import os
import re

import pytest

import bench
from communication_overlap_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "communication_overlap_gb300", "csrc")
PROFILES = os.path.join(ROOT, "profiles")


def _sha16(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


GEMM_SUMMARIES = sorted(
    f[len("signaled_gemm_"):-len("_ncu.md")] for f in os.listdir(PROFILES)
    if f.startswith("signaled_gemm_") and f.endswith("_ncu.md"))


def test_every_benchmarked_workload_with_taller_bands_has_a_summary():
    assert {"alltoall", "allreduce", "reducescatter", "wave_pattern"} <= set(GEMM_SUMMARIES)


@pytest.mark.parametrize("name", GEMM_SUMMARIES)
def test_gemm_traffic_summary_matches_source_and_launch_order(name):
    w = W.WORKLOADS[name]
    traffic = bench.traffic_from_profile(w, os.path.join(CSRC, "gemm.cu"))
    assert traffic is not None, f"profiles/signaled_gemm_{name}_ncu.md is stale"
    # at least the compulsory reads of A and B, and not absurdly more
    a_b = (w.M * w.K + max(1, w.n_experts) * w.K * w.N) * 2
    assert 0.5 * a_b < traffic < 4 * (a_b + w.M * w.N * 2)


def test_consumer_and_reorder_summary_matches_sources():
    txt = open(os.path.join(PROFILES, "consumer_reorder_kernels_ncu.md")).read()
    for src in ("comm.cu", "reorder.cu"):
        m = re.search(r"source_sha256_16 %s: ([0-9a-f]{16})" % re.escape(src), txt)
        assert m, src
        assert m.group(1) == _sha16(os.path.join(CSRC, src)), f"{src} changed since its capture"
