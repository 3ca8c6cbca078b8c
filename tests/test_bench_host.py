"""bench.py's host logic on the CPU: every workload it times or profiles has a
spec, the kernel-source digest ignores comments and whitespace but not code,
and the committed DRAM-traffic record parses into the workloads it names."""
import os
import shutil

import bench


def test_every_workload_has_a_spec():
    for group in (bench.STEP_WORKLOADS, bench.NEXT_WORKLOADS):
        assert len(group) == len(set(group))
    names = list(bench.STEP_WORKLOADS) + list(bench.NEXT_WORKLOADS) + list(bench.PROFILE_CASES)
    for name in names:
        spec = bench.workload_spec(name)
        assert spec["op"] in {"sum", "axis", "reduce", "cumsum", "rcumsum"}, name
        assert all(isinstance(d, int) and d > 0 for d in spec["shape"]), name
        if "dim" in spec:
            assert 0 <= spec["dim"] < len(spec["shape"]), name


def test_source_digest_ignores_comments_not_code(tmp_path, monkeypatch):
    root = tmp_path / "repo"
    shutil.copytree(os.path.join(bench.ROOT, "reduction_scan_primitives_gb300", "csrc"),
                    root / "reduction_scan_primitives_gb300" / "csrc")
    monkeypatch.setattr(bench, "ROOT", str(root))
    base = bench.source_digest()
    f = root / "reduction_scan_primitives_gb300" / "csrc" / "lr_device.cuh"
    text = f.read_text()
    f.write_text("// a new comment line\n" + text.replace("\n", "\n  ", 1) + "/* and a block */\n")
    assert bench.source_digest() == base
    f.write_text(text + "\nconstexpr int kProbeOnly = 1;\n")
    assert bench.source_digest() != base


def test_recorded_traffic_names_bench_workloads():
    path = os.path.join(bench.ROOT, "profiles", "dram_traffic.txt")
    known = set(bench.STEP_WORKLOADS) | set(bench.NEXT_WORKLOADS)
    rows = [line.split() for line in open(path) if line.strip() and not line.startswith("#")]
    assert rows
    for parts in rows:
        assert len(parts) == 5, parts
        workload, nbytes, digest, case, scale = parts
        assert workload in known, workload
        assert int(nbytes) > 0 and len(digest) == 16 and scale.startswith("x")
        assert case in bench.PROFILE_CASES or case in known, case
