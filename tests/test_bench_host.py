"""Host-side logic of bench.py, on the CPU: the roofline arithmetic of every
kernel class and the DRAM-traffic record (averaging an ncu capture, keyed by
a hash of the kernel sources so that a stale figure reads as null).  No GPU
and no library calls."""
import importlib.util
import json
import os

import pytest

import synth

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture()
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


PEAKS = {"hbm_gbs": 6000.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "sm_max_mhz": 2000.0,
         "source": "test"}


def k(work, ms):
    return {"work_per_launch": work, "avg_launch_ms": ms, "launches_per_step": 1.0, "ms_per_step": ms}


def test_hbm_roofline_is_bytes_over_time(bench):
    w = synth.WORKLOADS["gpt2_124m_B4_T64_fp32"]
    r = bench.roofline_for("adamw", k(3.0e9, 0.5), PEAKS, w)  # 3 GB in 0.5 ms = 6000 GB/s
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(6000.0)
    assert r["frac"] == pytest.approx(1.0)
    assert r["frac_of_nominal"] == pytest.approx(6000.0 / 7700.0)  # beside it: the 7.7 TB/s datasheet figure


def test_fp32_matmul_peak_is_tf32_from_bf16(bench):
    w = synth.WORKLOADS["gpt2_124m_B4_T64_fp32"]
    r = bench.roofline_for("gemm", k(2.0e12, 10.0), PEAKS, w)  # 2 TFLOP in 10 ms = 200 TFLOP/s
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(200.0)
    assert r["peak"] == pytest.approx(1800.0 * 1.1 / 2.25)


def test_fp32_matmul_peak_is_the_measured_tf32_rate_when_present(bench):
    w = synth.WORKLOADS["gpt2_124m_B4_T64_fp32"]
    peaks = dict(PEAKS, tf32_tflops=900.0, tf32_source="test")
    r = bench.roofline_for("gemm", k(2.0e12, 10.0), peaks, w)  # 200 TFLOP/s
    assert r["peak"] == 900.0
    assert r["frac"] == pytest.approx(200.0 / 900.0)
    # three MMAs per 3xTF32 product: the ceiling is a third of the peak
    assert r["frac_of_3xtf32_ceiling"] == pytest.approx(600.0 / 900.0)


def test_bf16_matmul_peak_is_the_sustained_bf16_rate(bench):
    # kernels timed inside a long graph-replayed step: the sustained figure,
    # with the burst fraction beside it
    w = synth.WORKLOADS["gpt2_124m_B16_T1024_bf16"]
    r = bench.roofline_for("gemm", k(1.4e12, 1.0), PEAKS, w)
    assert r["peak"] == 1400.0 and r["frac"] == pytest.approx(1.0)
    assert r["frac_of_burst"] == pytest.approx(1400.0 / 1800.0)
    # without a sustained figure, the burst one
    peaks = {kk: v for kk, v in PEAKS.items() if kk != "bf16_tflops_sustained"}
    r = bench.roofline_for("gemm", k(1.8e12, 1.0), peaks, w)
    assert r["peak"] == 1800.0 and r["frac"] == pytest.approx(1.0)


def test_attention_bounds(bench):
    # fp32 with head size 16 (the tiny model): CUDA cores, against the FP32
    # FMA issue rate, 148 SMs x 128 lanes x 2 FLOPs x clock
    w = synth.WORKLOADS["tiny_L2_C64"]
    r = bench.roofline_for("attn_bwd", k(1.0e9, 1.0), PEAKS, w)
    assert r["bound"] == "alu"
    assert r["peak"] == pytest.approx(148 * 128 * 2 * 2000e6 / 1e12)
    assert r["achieved"] == pytest.approx(1.0)
    # fp32 with head size 64 and T <= 64: 3xTF32 tcgen05 products
    w = synth.WORKLOADS["gpt2_124m_B4_T64_fp32"]
    peaks = dict(PEAKS, tf32_tflops=900.0, tf32_source="test")
    r = bench.roofline_for("attn_fwd", k(3.0e11, 1.0), peaks, w)  # 300 TFLOP/s
    assert r["bound"] == "tensor" and r["peak"] == 900.0
    assert r["frac_of_3xtf32_ceiling"] == pytest.approx(1.0)
    # bf16 with head size 64 and T % 128 == 0: the tensor-core kernels
    w = synth.WORKLOADS["gpt2_124m_B16_T1024_bf16"]
    r = bench.roofline_for("attn_fwd", k(1.0e9, 1.0), PEAKS, w)
    assert r["bound"] == "tensor" and r["peak"] == 1400.0


def write_capture(path, launches):
    """An ncu --csv launch list: one row per (launch, metric)."""
    lines = ['"ID","Kernel Name","Metric Name","Metric Unit","Metric Value"']
    for i, (name, rd, wr) in enumerate(launches):
        lines.append(f'"{i}","{name}","dram__bytes_read.sum","Mbyte","{rd}"')
        lines.append(f'"{i}","{name}","dram__bytes_write.sum","Kbyte","{wr}"')
    with open(path, "w") as fh:
        fh.write("==PROF== a line ncu prints first\n" + "\n".join(lines) + "\n")


def test_traffic_record_averages_matmul_launches_and_goes_stale(bench, tmp_path, monkeypatch):
    os.makedirs(tmp_path / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = {"v": "aaaa"}
    monkeypatch.setattr(bench, "kernel_source_sha", lambda kind: sha["v"])
    cap = tmp_path / "cap.csv"
    write_capture(cap, [("tc::gemm_tf32x3_kernel(...)", "10", "2000"),
                        ("tc::gemm_tf32x3_persistent_kernel(...)", "30", "0"),
                        ("adamw_kernel(...)", "999", "999")])
    w = synth.WORKLOADS["gpt2_124m_B4_T64_fp32"]
    assert bench.record_traffic(str(cap), w) == 0
    rec = json.load(open(tmp_path / "profiles" / "roofline_traffic.json"))[w.name]["gemm"]
    # (10 MB + 2 MB) and (30 MB + 0) over the two matmul launches; AdamW is not a matmul
    assert rec["launches_captured"] == 2
    assert rec["dram_bytes_per_launch"] == pytest.approx((12e6 + 30e6) / 2)
    assert bench.recorded_traffic("gemm", w) == pytest.approx(21e6)
    sha["v"] = "bbbb"  # the kernel sources changed since the capture
    assert bench.recorded_traffic("gemm", w) is None
    assert bench.recorded_traffic("gemm", synth.WORKLOADS["gpt2_124m_B16_T1024_bf16"]) is None


def test_attention_traffic_is_per_layer_op(bench, tmp_path, monkeypatch):
    # one timed attention-backward launch is a layer's op: the (-lse log2 e,
    # -D) pass, dK/dV and dQ, so the record sums the kernels' means; a
    # capture window that cuts a layer's op in two does not bias it
    os.makedirs(tmp_path / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_sha", lambda kind: "cccc")
    cap = tmp_path / "cap.csv"
    write_capture(cap, [("tca::attn_bwd_dkv_tc_kernel(...)", "100", "20000"),  # window starts mid-op
                        ("tca::attn_bwd_dq_tc_kernel(...)", "100", "8000"),
                        ("void tca::attn_bwd_ld_bf16_kernel<8>(...)", "50", "0"),
                        ("tca::attn_bwd_dkv_tc_kernel(...)", "104", "20000"),
                        ("tca::attn_bwd_dq_tc_kernel(...)", "100", "8000"),
                        ("tca::attn_fwd_tc_kernel(...)", "77", "1000"),
                        ("tcb::gemm_bf16_kernel<256, 0, 2>(...)", "999", "0")])
    w = synth.WORKLOADS["gpt2_124m_B16_T1024_bf16"]
    assert bench.record_traffic(str(cap), w, "attn_bwd") == 0
    assert bench.recorded_traffic("attn_bwd", w) == pytest.approx(50e6 + 122e6 + 108e6)
    assert bench.record_traffic(str(cap), w, "attn_fwd") == 0
    assert bench.recorded_traffic("attn_fwd", w) == pytest.approx(78e6)
    peaks = dict(PEAKS)
    r = bench.roofline_for("attn_bwd", k(1.0e9, 1.0), peaks, w)
    assert r["traffic"] == pytest.approx(280e6)


def test_oracle_one_thread_sample_runs_in_a_child_with_one_thread(bench):
    # the cpu_baseline's one-thread figure: a child process with
    # OMP_NUM_THREADS=1 times the oracle and reports one core
    rec = bench.oracle_one_thread(synth.WORKLOADS["tiny_L2_C64"], seconds=0.2)
    assert rec is not None
    assert rec["cores"] == 1 and rec["unit"] == "tokens/s" and rec["value"] > 0
