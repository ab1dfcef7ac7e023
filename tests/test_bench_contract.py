"""The bench's recorded DRAM traffic belongs to the kernel source in the tree.

`bench.py` reports `roofline.traffic` from ncu captures only while the
attention kernel's device source hashes to the value the capture was taken
with.  These checks keep the committed figures and the committed kernel
together: a kernel change without a new capture fails here instead of
silently turning the figure into null.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    sys.path.insert(0, ROOT)
    import bench

    return bench


def test_every_profiled_traffic_entry_matches_the_kernel_source():
    bench = _bench()
    current = bench.attn_kernel_source_sha256()
    assert bench.PROFILED_TRAFFIC, "no ncu traffic figure recorded"
    for key, entry in bench.PROFILED_TRAFFIC.items():
        assert entry["kernel_source_sha256"] == current, f"{key}: captured on another kernel source"
        assert entry["dram_bytes_per_launch"] > 0
        src = entry["source"]
        path = os.path.join(ROOT, src[src.index("profiles/"):].split()[0])
        assert os.path.exists(path), f"{key}: {path} missing"
        with open(path) as f:
            assert current in f.read(), f"{key}: {path} does not name the kernel source it summarises"


def test_default_workload_has_a_traffic_figure():
    """The default line's workload (the 2M-token sequence, FUSED) carries one."""
    bench = _bench()
    assert ("seq2m", "fused") in bench.PROFILED_TRAFFIC


def test_kernel_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    bench = _bench()
    src = open(bench.ATTN_SRC).read()
    ptx = open(os.path.join(os.path.dirname(bench.ATTN_SRC), "sm103_ptx.cuh")).read()
    (tmp_path / "sm103_ptx.cuh").write_text(ptx)
    current = bench.attn_kernel_source_sha256()
    f = tmp_path / "attn_fwd.cu"
    monkeypatch.setattr(bench, "ATTN_SRC", str(f))
    f.write_text("// a new comment line\n\n" + src.replace("{\n", "{  // trailing note\n", 3))
    assert bench.attn_kernel_source_sha256() == current
    f.write_text("static int extra_device_symbol;\n" + src)
    assert bench.attn_kernel_source_sha256() != current
