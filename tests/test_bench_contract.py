"""The JSON line of bench.py's reference arm (the oracle timed on the host
cores) carries every key of the benchmark contract, for the voxelizer and
for farthest point sampling, and the profile lookup keys on device code only.
No GPU needed: the reference arm runs the oracle alone."""

from __future__ import annotations

import io
import json
import os
import shutil
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


def _reference_line(**kw):
    args = {"workload": "tiny", "steps": 2, "warmup": 1, "gpus": 1, "batch": 1, "op": "voxelize"}
    args.update(kw)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(type("A", (), args)(), 0, 1)
    lines = [ln for ln in buf.getvalue().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


@pytest.mark.parametrize("op,workload", [("voxelize", "tiny"), ("voxelize", "kitti"), ("fps", "lidar65k")])
def test_reference_line_has_every_contract_key(op, workload):
    d = _reference_line(op=op, workload=workload)
    assert KEYS <= set(d), KEYS - set(d)
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "Mpoints/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 2 and d["warmup"] == 1
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_profile_lookup_keys_on_device_code(tmp_path, monkeypatch):
    # A committed summary names the SHA-256 of the kernel's sources (the
    # shared device header and the kernel's file) up to their host-side
    # markers, comments left out: host edits and comment edits keep the
    # summary, device-code edits in either file void it.
    src_dir = tmp_path / "lidar_point_cloud_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    prof = tmp_path / "profiles"
    prof.mkdir()
    texts = {}
    for name in bench.KERNEL_SOURCES["pv_voxelize_kernel"]:
        src = os.path.join(ROOT, "lidar_point_cloud_gb300", "csrc", name)
        texts[name] = open(src, "rb").read()
        assert bench.HOST_SIDE_MARKER in texts[name]
        shutil.copy(src, src_dir / name)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.kernel_sha()
    (prof / "pv_voxelize_kernel_probe.md").write_text(
        f"# probe\n\n- dram_bytes_per_launch: `1234`\n- kernel_source_sha256: `{sha}`\n")
    assert bench.profiled_traffic("probe") == 1234
    for name, text in texts.items():
        cut = text.index(bench.HOST_SIDE_MARKER)
        (src_dir / name).write_bytes(text + b"\nstatic int host_side_edit = 0;\n")
        assert bench.profiled_traffic("probe") == 1234
        (src_dir / name).write_bytes(text[:cut] + b"// a comment in the device code\n" + text[cut:])
        assert bench.profiled_traffic("probe") == 1234
        (src_dir / name).write_bytes(text[:cut] + b"static __device__ int device_side_edit;\n" + text[cut:])
        assert bench.profiled_traffic("probe") is None
        (src_dir / name).write_bytes(text)
        assert bench.profiled_traffic("probe") == 1234
