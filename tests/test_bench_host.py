"""bench.py's host logic that needs no GPU: how a committed ncu summary becomes the
`roofline.traffic` figure of a bench line."""
import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _setup(tmp_path, monkeypatch, body: str, src_text: bytes = b"kernel source"):
    (tmp_path / "profiles").mkdir()
    src = tmp_path / "k.cu"
    src.write_bytes(src_text)
    sha = hashlib.sha256(src_text).hexdigest()
    (tmp_path / "profiles" / "gemv1_gpt-oss-decode.md").write_text(
        body.replace("SHA", sha))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return str(src)


def test_per_expert_traffic_scales_with_active_experts(tmp_path, monkeypatch):
    src = _setup(tmp_path, monkeypatch, "traffic_bytes_per_active_expert: 2.5e7\n"
                 "traffic_workloads: gpt-oss-decode@T=1 gpt-oss-decode@T=8\n"
                 "source_sha256: SHA\n")
    assert bench.profile_traffic("gemv1", "gpt-oss-decode@T=1", 4, src) == 1e8
    # the smaller-expert capture itself (@E= dropped) and another listed batch
    assert bench.profile_traffic("gemv1", "gpt-oss-decode@T=1@E=16", 4, src) == 1e8
    assert bench.profile_traffic("gemv1", "gpt-oss-decode@T=8", 28, src) == 7e8
    # a batch the summary does not stand for
    assert bench.profile_traffic("gemv1", "gpt-oss-decode@T=32", 81, src) is None


def test_per_launch_traffic_only_for_its_own_workload(tmp_path, monkeypatch):
    src = _setup(tmp_path, monkeypatch, "traffic_bytes_per_launch: 1.5e9\nsource_sha256: SHA\n")
    assert bench.profile_traffic("gemv1", "gpt-oss-decode", 128, src) == 1.5e9
    assert bench.profile_traffic("gemv1", "gpt-oss-decode@T=8", 28, src) is None


def test_changed_kernel_source_voids_the_traffic(tmp_path, monkeypatch):
    src = _setup(tmp_path, monkeypatch, "traffic_bytes_per_active_expert: 2.5e7\n"
                 "traffic_workloads: gpt-oss-decode@T=1\nsource_sha256: SHA\n")
    with open(src, "ab") as f:
        f.write(b"// edited")
    assert bench.profile_traffic("gemv1", "gpt-oss-decode@T=1", 4, src) is None
    # and a kernel without a summary has none
    assert bench.profile_traffic("gemm1", "gpt-oss-decode@T=1", 4, src) is None


def test_included_header_edit_voids_the_traffic(tmp_path, monkeypatch):
    """The pinned hash covers the headers a kernel file includes from its directory: an edit
    to a kernel body kept in a header voids the figure; one to another file does not."""
    src = _setup(tmp_path, monkeypatch, "traffic_bytes_per_launch: 1.5e9\nsource_sha256: SHA\n",
                 b'#include "k_dev.cuh"\n#include <cstdint>\n')
    (tmp_path / "k_dev.cuh").write_bytes(b"device code")
    (tmp_path / "other.cuh").write_bytes(b"unrelated")
    txt = (tmp_path / "profiles" / "gemv1_gpt-oss-decode.md").read_text()
    (tmp_path / "profiles" / "gemv1_gpt-oss-decode.md").write_text(
        txt.replace(hashlib.sha256(b'#include "k_dev.cuh"\n#include <cstdint>\n').hexdigest(),
                    bench.source_hash(src)))
    assert bench.profile_traffic("gemv1", "gpt-oss-decode", 128, src) == 1.5e9
    (tmp_path / "other.cuh").write_bytes(b"edited")
    assert bench.profile_traffic("gemv1", "gpt-oss-decode", 128, src) == 1.5e9
    (tmp_path / "k_dev.cuh").write_bytes(b"device code, edited")
    assert bench.profile_traffic("gemv1", "gpt-oss-decode", 128, src) is None


def test_committed_summaries_parse():
    """Every committed summary that bench.py may read names a source hash and a traffic
    figure in one of the two forms."""
    prof = os.path.join(ROOT, "profiles")
    for name in os.listdir(prof):
        if not (name.startswith("gemm") or name.startswith("gemv")):
            continue
        txt = open(os.path.join(prof, name)).read()
        assert "source_sha256:" in txt, name
        assert ("traffic_bytes_per_launch:" in txt or
                ("traffic_bytes_per_active_expert:" in txt and "traffic_workloads:" in txt)), name
