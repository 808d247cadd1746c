"""Host-side legs of bench.py that need no GPU: the CPU baseline (the oracle
on a bounded sample, or the full join for a small workload) and the roofline
arithmetic helpers."""
import json

import numpy as np

import bench
import datagen


def test_cpu_baseline_full_and_sampled():
    x = datagen.generate(1, n=1500)
    full = bench.cpu_baseline(x, 0.6, None)          # 1500 rows: the whole join
    assert full["full_join_s_kind"] == "measured" and "full join" in full["sample"]
    part = bench.cpu_baseline(x, 0.6, 100)
    assert part["full_join_s_kind"] == "extrapolated" and part["sample"].startswith("100 random query rows")
    for r in (full, part):
        assert r["kind"] == "oracle" and r["cores"] >= 1 and r["value"] > 0 and r["cpu_model"]
        json.dumps(r)


def test_sample_rows_bounds():
    assert bench.sample_rows(20_000, 16, bench.CPU_SAMPLE_COORD_OPS) == 20_000
    n = bench.sample_rows(5_000_000, 16, bench.CPU_SAMPLE_COORD_OPS)
    assert 64 <= n < 5_000_000 and abs(n * 5_000_000 * 16 - bench.CPU_SAMPLE_COORD_OPS) < 5_000_000 * 16


def test_fp32_peak_counts_two_flops_per_lane():
    assert abs(bench.fp32_peak_tflops(152, 2070.0) - 152 * 128 * 2.07e9 * 2 / 1e12) < 1e-9


def test_reference_arm_prints_one_line(capsys, monkeypatch):
    class A:
        config, steps, warmup, ref_step_rows = 1, 1, 0, 50
        n = None
        batch_bytes, shard, refine = bench.DEFAULT_BATCH_BYTES, False, "cuda"
    bench.run_reference(A, 1, 0)
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["unit"] == bench.UNIT and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_code_sha_ignores_comments_not_code(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("int f() {\n    return 1;  // one\n}\n")
    b = tmp_path / "b.cu"
    b.write_text("// a comment\nint f() {\n\n    return 1;\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f() {\n    return 2;\n}\n")
    assert bench.code_sha(str(a)) == bench.code_sha(str(b)) != bench.code_sha(str(c))
