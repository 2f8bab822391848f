"""bench.py's reference arm (the fp64 oracle timed on the host cores) prints
one JSON line with the contract's keys, on the same workload, metric and unit
as the GPU arm."""
import json
import types

import bench


def test_reference_arm_prints_one_contract_line(capsys):
    args = types.SimpleNamespace(steps=1, warmup=0, gpus=1)
    assert bench.run_reference(args) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference"
    assert rec["metric"] == bench.METRIC and rec["unit"] == bench.UNIT
    assert rec["higher_is_better"] is True and rec["n_gpus"] == 1
    assert rec["steps"] == 1 and rec["warmup"] == 0
    assert rec["config"]["workload"] == "ref2va-1doc-S20423"
    assert rec["value"] > 0 and rec["ms_per_step"] > 0
    cpu = rec["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == rec["value"] and cpu["sample"]
    e2e = rec["e2e"]
    assert e2e["value"] == rec["value"] and e2e["unit"] == rec["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    # the value is the sampled rows' algorithmic FLOPs over the sampled time
    assert rec["value"] * 1e12 * rec["ms_per_step"] * 1e-3 > 4 * 128 * 20423 * 512


def test_kernel_code_hash_ignores_comments_only(tmp_path):
    # the recorded DRAM traffic stays valid across comment edits, not code edits
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    c = tmp_path / "c.cu"
    a.write_text("// header\n__global__ void k(int* p) {\n  p[0] = 1;  // store\n}\n")
    b.write_text("// a different header\n\n__global__ void k(int* p) {\n  p[0] = 1;\n}\n")
    c.write_text("// header\n__global__ void k(int* p) {\n  p[0] = 2;  // store\n}\n")
    assert bench.kernel_code_hash(str(a)) == bench.kernel_code_hash(str(b))
    assert bench.kernel_code_hash(str(a)) != bench.kernel_code_hash(str(c))
