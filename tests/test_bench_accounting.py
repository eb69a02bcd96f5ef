"""Host logic of bench.py, on the CPU.

- Algorithmic bytes: the byte count the bench divides by time for each
  configuration equals the totals the workload table prints for it (codes
  N*K, scales 4N, bias 4N when present, x 2MK, y 2MN), so a changed shape,
  a dropped bias or a miscounted term fails here.
- The stored DRAM traffic of a kernel is used only while the kernel's source
  is the one it was taken on.
- The parser of the ncu launch CSV that writes that record.
"""
import json
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import synthetic  # noqa: E402


def _bytes(case):
    return bench.call_bytes(case["m"], case["n"], case["k"], with_bias=case["bias"] is not None)


@pytest.mark.parametrize("name,total", [
    ("tiny_gemv", 1_060_864),        # 1 x 1024 x 1024
    ("outlier_gemv", 16_809_984),    # 1 x 4096 x 4096, no bias
    ("fp16_template", 4_452_352),    # 22 x 1024 x 4096
])
def test_config_bytes_match_the_workload_table(name, total):
    assert _bytes(synthetic.case(name)) == total


def test_skinny_sweep_bytes_match_the_workload_table():
    # K = 4096, N = 14336: 58,834,944 + 36,864 M, and 58,871,808 at M = 1
    n, k = 14336, 4096
    for m in (1,) + synthetic.SKINNY_M:
        assert bench.call_bytes(m, n, k) == 58_834_944 + 36_864 * m
    assert bench.call_bytes(1, n, k) == 58_871_808
    assert bench.call_bytes(32, n, k) == 60_014_592


def test_down_orientation_bytes_match_the_workload_table():
    # the 58.7 MB weight as [4096 x 14336] at M = 1
    (_, n, k), = [s for s in synthetic.DECODE_STACK if s[0] == "down"]
    assert (n, k) == (4096, 14336)
    assert bench.call_bytes(1, n, k) == 58_789_888


def test_decode_stack_codes_per_pass():
    # seven matrices, 218,103,808 code bytes a pass; three passes a step
    assert sum(n * k for (_, n, k) in synthetic.DECODE_STACK) == 218_103_808
    calls = bench.step_calls()
    assert len(calls) == 21 and [m for (m, _, _, _) in calls[::7]] == list(synthetic.DECODE_STACK_M)
    codes = sum(n * k for (_, _, n, k) in calls)
    assert codes == 3 * 218_103_808
    # everything else a step moves is small next to the codes (scales, bias,
    # activations and outputs of 21 calls)
    assert 0 < bench.step_bytes() - codes < 8_000_000


def _fake_root(tmp_path):
    src = os.path.join(ROOT, "fp8_weight_only_gb300", "csrc")
    dst = tmp_path / "fp8_weight_only_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in ("skinny.cu", "gemv.cu", "fp8w_device.cuh"):
        shutil.copy(os.path.join(src, f), dst / f)
    (tmp_path / "profiles").mkdir()
    return tmp_path


NCU_HEADER = ["ID", "Process ID", "Process Name", "Host Name", "Kernel Name", "Context", "Stream", "Block Size",
              "Grid Size", "Device", "CC", "Section Name", "Metric Name", "Metric Unit", "Metric Value"]


def _ncu_rows(launch_id, kernel, read, write):
    base = [str(launch_id), "1", "python3", "127.0.0.1", kernel, "1", "7", "(640, 1, 1)", "(112, 1, 1)", "0", "10.3",
            "Command line profiler metrics"]
    return [base + ["dram__bytes_read.sum", "byte", "{:,}".format(read)],
            base + ["dram__bytes_write.sum", "byte", "{:,}".format(write)]]


def test_record_traffic_then_stored_traffic(tmp_path, monkeypatch):
    root = _fake_root(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    skinny = "void fp8w::skinny_kernel<32, true, 0, 1>(CUtensorMap, CUtensorMap, const float *)"
    gemv = "gemv_kernel<2, true, true, 0>(const unsigned short *, const unsigned char *)"
    rows = [NCU_HEADER]
    rows += _ncu_rows(0, skinny, 31_000_000, 500_000)
    rows += _ncu_rows(1, gemv, 26_000_000, 10_000)
    rows += _ncu_rows(2, skinny, 32_000_000, 500_000)
    csv_path = tmp_path / "traffic.csv"
    with open(csv_path, "w") as f:
        f.write("==PROF== a line ncu prints before the table\n")
        for r in rows:
            f.write(",".join('"%s"' % c for c in r) + "\n")
    bench.record_traffic(str(csv_path))
    with open(root / "profiles" / "dram_traffic_decode_stack.json") as f:
        rec = json.load(f)
    assert rec["command"] == bench.TRAFFIC_COMMAND
    k = rec["kernels"]
    assert set(k) == {"fp8w::skinny_kernel<32, true, 0, 1>", "fp8w::gemv_kernel<2, true, true, 0>"}
    assert k["fp8w::skinny_kernel<32, true, 0, 1>"]["launches"] == 2
    assert k["fp8w::skinny_kernel<32, true, 0, 1>"]["dram_bytes_per_launch"] == 32_000_000
    assert k["fp8w::gemv_kernel<2, true, true, 0>"]["dram_bytes_per_launch"] == 26_010_000
    # read back while the sources are unchanged ...
    got, why = bench.stored_traffic("fp8w::skinny_kernel<32, true, 0, 1>")
    assert got == 32_000_000 and why.startswith("ncu dram__bytes_read.sum + dram__bytes_write.sum")
    # ... and refused once the kernel's source differs from the one measured
    with open(root / "fp8_weight_only_gb300" / "csrc" / "skinny.cu", "a") as f:
        f.write("\n")
    got, why = bench.stored_traffic("fp8w::skinny_kernel<32, true, 0, 1>")
    assert got is None and "changed" in why
    # the GEMV's record is untouched by an edit of the other kernel
    got, _ = bench.stored_traffic("fp8w::gemv_kernel<2, true, true, 0>")
    assert got == 26_010_000
    # a shared header changes both
    with open(root / "fp8_weight_only_gb300" / "csrc" / "fp8w_device.cuh", "a") as f:
        f.write("\n")
    assert bench.stored_traffic("fp8w::gemv_kernel<2, true, true, 0>")[0] is None


def test_stored_traffic_without_a_record(tmp_path, monkeypatch):
    root = _fake_root(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    got, why = bench.stored_traffic("fp8w::skinny_kernel<32, 1, 0, 1>")
    assert got is None and "no stored" in why
