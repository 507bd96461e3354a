"""bench.py pieces that need no GPU: the reference arm (the oracle timed on the host) prints
one JSON line in the contract's shape, and the workload table holds what the docs state."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("workload,unit", [("c0", "TOPS"), ("d1", "tok/s")])
def test_reference_arm_prints_one_contract_line(workload, unit):
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", workload, "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == unit and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    for key in ("metric", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "config", "dtype"):
        assert key in d, key


def test_workloads_match_the_documented_shapes():
    sys.path.insert(0, ROOT)
    from w4a8_block_quantized_gb300 import synth
    shapes = {k: [(s.M, s.K, s.N) for s in synth.workload(k)[1]] for k in synth.WORKLOADS}
    assert shapes["c0"] == [(128, 1024, 1024)]
    assert shapes["c1"] == [(512, 1024, 3072)] and synth.workload("c1")[1][0].bias
    assert shapes["c2"] == [(512, 2048, 6144), (512, 6144, 2048)]
    assert shapes["c3"] == [(512, 2048, 2048), (512, 2048, 1024), (512, 2048, 1024), (512, 2048, 2048),
                            (512, 2048, 6144), (512, 2048, 6144), (512, 6144, 2048)]
    assert shapes["c4"] == [(8192, 4096, 14336), (8192, 14336, 4096)]
    assert all(M == 1 for k in ("d1", "d3", "d4") for M, _, _ in shapes[k])
    assert [(K, N) for _, K, N in shapes["d3"]] == [(K, N) for _, K, N in shapes["c3"]]
    # the decode workloads' weights at 4.5 bits per weight
    s = synth.workload("d4")[1][0]
    assert synth.weight_bytes(s) == s.N * s.K // 2 + 4 * s.N * (s.K // 64)


def test_cpu_baseline_object():
    """The GPU line's `cpu_baseline`: the oracle on all host cores over a stated sample, the CPU
    model and core count, and the single-thread build's figure beside it."""
    sys.path.insert(0, ROOT)
    import bench
    from w4a8_block_quantized_gb300 import synth
    _, specs = synth.workload("c0")
    lin = [{"host": synth.make_linear(s), "spec": s} for s in specs]
    c = bench.cpu_baseline(lin, specs, 1.0)
    assert c["kind"] == "oracle" and c["unit"] == "TOPS" and c["value"] > 0
    assert c["cores"] >= 1 and c["nproc"] == os.cpu_count() and c["cpu"]
    assert "rows" in c["sample"] and c["seconds"] > 0
    one = c["one_core"]
    assert one["unit"] == "TOPS" and 0 < one["value"] and "rows" in one["sample"]
    # one thread cannot outrun the whole pool by much (timing noise aside)
    assert one["value"] <= 2 * c["value"]


def test_traffic_record_follows_every_source_of_its_kernel(tmp_path, monkeypatch):
    """The recorded DRAM bytes are reported only while every listed source file (the kernel's
    .cu file and the headers it includes) is byte-identical to the one captured."""
    sys.path.insert(0, ROOT)
    import bench
    (tmp_path / "profiles").mkdir()
    (tmp_path / "k.cu").write_text("kernel\n")
    (tmp_path / "h.cuh").write_text("header\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    entry = {"kernel": "k", "sources": ["k.cu", "h.cuh"], "dram_bytes_per_launch": 1234}
    entry["sha256"] = bench.sources_sha256(entry["sources"])
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"c1": entry}))
    assert bench.recorded_traffic("c1") == 1234
    assert bench.recorded_traffic("c2") is None
    (tmp_path / "h.cuh").write_text("header changed\n")
    assert bench.recorded_traffic("c1") is None
    (tmp_path / "h.cuh").write_text("header\n")
    assert bench.recorded_traffic("c1") == 1234
    (tmp_path / "h.cuh").unlink()
    assert bench.recorded_traffic("c1") is None


def test_committed_traffic_record_lists_the_included_headers():
    """Each entry of the committed record lists its kernel's .cu file and every in-tree header
    that file includes, directly or through another header."""
    import re
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for e in rec.values():
        srcs = e["sources"]
        todo, seen = [srcs[0]], set()
        while todo:
            p = todo.pop()
            if p in seen:
                continue
            seen.add(p)
            with open(os.path.join(ROOT, p)) as f:
                for inc in re.findall(r'#include "([^"]+)"', f.read()):
                    todo.append(os.path.join(os.path.dirname(p), inc))
        assert seen == set(srcs), (e["kernel"], sorted(seen ^ set(srcs)))


def test_fused_step_bytes_by_hand():
    """The fused step's byte counts for the pp512 linear (M 512, K 1024, N 3072, bias), term by
    term: x 2 MiB, packed weights 1.5 MiB, fp16 scales and zeros 192 KiB, bias 12 KiB, y 6 MiB;
    token records 2 B per element + 16 B per 64 elements + 4 B per row, weight records 1 B per
    weight + 16 B and a 4-byte scale per 64 (3072 rows, already a multiple of 128)."""
    sys.path.insert(0, ROOT)
    import bench
    M, K, N = 512, 1024, 3072
    x, wq, sz, bias, y = 4 * M * K, N * K // 2, 2 * 2 * N * (K // 64), 4 * N, 4 * M * N
    tok = 2 * M * K + 16 * M * (K // 64) + 4 * M
    wrec = N * K + 16 * N * (K // 64) + 4 * N * (K // 64)
    alg, des = bench.fused_step_bytes(M, K, N, True)
    assert alg == x + wq + sz + bias + y == 10170368
    assert des == (x + tok) + (wq + sz + wrec) + (tok + wrec + bias + y)
    # rows padded to 128 in the weight records; no bias
    alg2, des2 = bench.fused_step_bytes(1, 128, 130, False)
    assert alg2 == 4 * 128 + 130 * 64 + 2 * 2 * 130 * 2 + 4 * 130
    assert des2 - alg2 == 2 * (2 * 128 + 16 * 2 + 4) + 2 * (256 * 128 + 256 * 2 * 16 + 256 * 2 * 4)
