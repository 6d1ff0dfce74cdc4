"""Host logic of bench.py that needs no GPU: the ncu summary and the traffic lookup."""
import bench

HEADER = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size",'
          '"Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"\n')


def row(i, name, metric, unit, value):
    return (f'"{i}","1","python","h","{name}","1","7","(192, 1, 1)","(152, 1, 1)","0","10.3","",'
            f'"{metric}","{unit}","{value}"\n')


W = "void zbk::(anonymous namespace)::gemm_pair_kernel<true, true, 3, 2>(CUtensorMap, CUtensorMap, KParams)"
B = "void zbk::(anonymous namespace)::gemm_pair_kernel<false, true, 0, 2>(CUtensorMap, CUtensorMap, KParams)"
F = "void zbk::(anonymous namespace)::gemm_pair_kernel<false, false, 1, 2>(CUtensorMap, CUtensorMap, KParams)"
R = "void zbk::(anonymous namespace)::rmsnorm_bwd_kernel<2>(const unsigned short *, int)"
# the form ncu's CSV prints on the GB300 box: bools as 0 / 1, anonymous namespaces as "unnamed>"
B_NCU = "void unnamed>::gemm_pair_kernel<0, 1, 2, 2>(CUtensorMap_st, CUtensorMap_st, unnamed>::KParams)"


def test_labels_of_ncu_names():
    assert bench.kernel_label(B_NCU) == "gemm_pair_kernel B (SwiGLU backward epilogue)"
    assert bench.kernel_label(W) == "gemm_pair_kernel W (float32 TMA reduce-add epilogue)"
    assert bench.kernel_label("void <unnamed>::dgamma_final_kernel(<unnamed>::GammaBatch)") == "dgamma_final_kernel"


def test_summary_shares_and_gemm_traffic(tmp_path):
    csv = tmp_path / "l.csv"
    lines = ["==PROF== Connected to process\n", HEADER]
    launches = [(0, F, 100.0, 10.0, 1.0), (1, B, 200.0, 20.0, 2.0), (2, W, 600.0, 30.0, 40.0), (3, R, 100.0, 5.0, 5.0)]
    for i, name, us, rd_mb, wr_mb in launches:
        lines.append(row(i, name, "gpu__time_duration.sum", "ns", f"{1000 * us:,.0f}"))
        lines.append(row(i, name, "dram__bytes_read.sum", "Mbyte", rd_mb))
        lines.append(row(i, name, "dram__bytes_write.sum", "byte", int(wr_mb * 1e6)))
    csv.write_text("".join(lines))
    text = bench.summarize_ncu(str(csv), "ncu ... python bench.py", "t", bw_flops=4.6e9)
    assert "| gemm_pair_kernel W (float32 TMA reduce-add epilogue) | 1 | 0.60 | 60.0 % | 30.0 | 40.0 |" in text
    assert "| rmsnorm_bwd_kernel<2> | 1 | 0.10 | 10.0 % |" in text
    assert "| **total** | 4 | 1.00 | 100 % |" in text
    # B and W GEMM launches only: (20 + 2 + 30 + 40) MB over 4.6 GFLOP
    assert "B/W GEMM DRAM bytes per algorithmic FLOP: 2.000000e-02" in text
    rec = bench.gemm_traffic_record(str(csv), "ncu ... python bench.py", 4.6e9)
    assert abs(rec["dram_bytes_per_unit"] - 2e-2) < 1e-12 and rec["launches"] == 2
    assert rec["source_sha256"] == bench.gemm_source_sha()


def test_traffic_lookup_needs_matching_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "gemm_source_sha", lambda: "abc")
    assert bench.profiled_gemm_traffic("w", "per-microbatch")[0] is None
    (prof / "gemm_traffic_w.json").write_text('{"dram_bytes_per_unit": 1.5e-4, "source_sha256": "abc"}')
    assert bench.profiled_gemm_traffic("w", "per-microbatch")[0] == 1.5e-4
    assert bench.profiled_gemm_traffic("w", "flush")[0] is None
    (prof / "gemm_traffic_w.json").write_text('{"dram_bytes_per_unit": 1.5e-4, "source_sha256": "old"}')
    assert bench.profiled_gemm_traffic("w", "per-microbatch")[0] is None


def test_summary_of_several_logs(tmp_path):
    """Captures taken in chunks (ids restart at 0 in each log) add up launch by launch."""
    paths = []
    for f in range(2):
        csv = tmp_path / f"c{f}.csv"
        csv.write_text(HEADER + row(0, W, "gpu__time_duration.sum", "ns", "1000") +
                       row(0, W, "dram__bytes_read.sum", "byte", "2000000") +
                       row(0, W, "dram__bytes_write.sum", "byte", "0"))
        paths.append(str(csv))
    text = bench.summarize_ncu(",".join(paths), "cmd", "t", bw_flops=1e9)
    assert "| gemm_pair_kernel W (float32 TMA reduce-add epilogue) | 2 | 0.00 | 100.0 % | 2.0 | 0.0 |" in text
    assert "B/W GEMM DRAM bytes per algorithmic FLOP: 4.000000e-03" in text


def test_reference_arm_json_line():
    """`bench.py --impl reference` (the float64 oracle on the host cores) prints one JSON line
    with the contract's keys, on the same metric and unit as the GPU arm."""
    import json
    import subprocess
    import sys

    out = subprocess.run([sys.executable, bench.__file__, "--impl", "reference", "--workload", "tiny_stage",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["higher_is_better"] is True and d["value"] > 0 and d["steps"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "tiny_stage"
    # the same workload description as the GPU arm's line, plus how it was sampled
    for key, val in bench.WORKLOADS["tiny_stage"].items():
        assert d["config"][key] == val, key
    assert d["config"]["sample_tokens_per_step"] > 0


def test_row_traffic_record(tmp_path):
    """Row-kernel DRAM bytes per algorithmic byte, from the B/W row launches of a capture only."""
    csv = tmp_path / "r.csv"
    lines = [HEADER]
    for i, (name, rd, wr) in enumerate([(R, 6.0, 2.0), (W, 100.0, 100.0),
                                        ("void <unnamed>::dgamma_final_kernel(<unnamed>::GammaBatch, const float *)",
                                         1.0, 1.0)]):
        lines.append(row(i, name, "gpu__time_duration.sum", "ns", "1000"))
        lines.append(row(i, name, "dram__bytes_read.sum", "Mbyte", rd))
        lines.append(row(i, name, "dram__bytes_write.sum", "Mbyte", wr))
    csv.write_text("".join(lines))
    rec = bench.row_traffic_record(str(csv), "cmd", 5e6)
    assert rec["launches"] == 2 and abs(rec["dram_bytes_per_unit"] - 2.0) < 1e-12
    assert rec["source_sha256"] == bench.row_source_sha()


def test_attention_roofline_record():
    import bench

    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "measured"}
    ab = {"flops": 343.7e9 * 4, "ms": 1.4, "launches": 4}
    rec = bench.attention_roofline(ab, peaks, "bf16_tflops_sustained")
    assert rec["bound"] == "tensor" and rec["unit"] == "TFLOP/s"
    assert abs(rec["achieved"] - 343.7e9 * 4 / 1.4e-3 / 1e12) < 1e-9
    assert abs(rec["frac"] - rec["achieved"] / 1700.0) < 1e-12
    assert rec["ms_per_launch"] == 0.35
    assert bench.attention_roofline({"flops": 0.0, "ms": 0.0, "launches": 0}, peaks, "bf16_tflops") is None
