"""The bench's roofline arithmetic, on the CPU: the algorithmic bytes per kernel, the
scaling of the committed DRAM-traffic lines and their guard on the kernel source, and the
fraction of the measured peak that the JSON line reports."""

import hashlib
import os
import shutil

import pytest

import bench


def _w(name):
    return bench.WORKLOADS[name]


def test_algorithmic_bytes_of_the_walks_at_32k():
    # compulsory tensors of each kernel, once: x, dy, dx, y are T*H*P bf16; B, C, dB, dC
    # T*G*N bf16; raw_dt and d_raw_dt T*H fp32
    T, H, P, N = 32768, 80, 64, 128
    act, bc, raw = T * H * P * 2, T * N * 2, T * H * 4
    w = _w("mamba2.8b_32k")
    assert bench.kernel_model("tc_bwd_dxdb", w) == ("hbm", float(3 * act + 3 * bc + 2 * raw), "byte")
    assert bench.kernel_model("tc_bwd_dc", w) == ("hbm", float(2 * act + 3 * bc + raw), "byte")
    assert bench.kernel_model("tc_fwd_walk", w) == ("hbm", float(2 * act + 2 * bc + raw), "byte")
    assert bench.kernel_model("tc_bwd_dxdb", w)[1] == 1052770304.0
    assert bench.kernel_model("no_such_kernel", w) == (None, None, None)


def test_step_bytes_count_each_tensor_once():
    w = _w("genomics_2m")
    T, H, P, N = 2097152, 16, 64, 64
    fwd_b, _, _, _ = bench.algorithmic(w)
    # x and y, B and C, raw_dt, the final state
    assert fwd_b == 2 * T * H * P * 2 + 2 * T * N * 2 + T * H * 4 + H * P * N * 4


def test_traffic_lines_scale_with_tokens_and_heads():
    w = _w("mamba2.8b_32k")
    per_token = None
    for line in open(os.path.join(bench.ROOT, "profiles", "dram_traffic_walks.txt")):
        p = line.split()
        if line.startswith("#") or len(p) < 6 or p[0] != "tc_bwd_dxdb" or int(p[5]) != 128:
            continue
        per_token, heads = float(p[1]), float(p[4])
        src_ok = hashlib.sha256(open(os.path.join(bench.ROOT, p[2]), "rb").read()).hexdigest() == p[3]
    assert per_token is not None
    got = bench.measured_traffic("tc_bwd_dxdb", w)
    if not src_ok:
        assert got is None
    else:
        assert got == pytest.approx(per_token * 32768 * 80 / heads)
        # within 1.5x of the algorithmic bytes: the capture measured this kernel
        assert 1.0 <= got / bench.kernel_model("tc_bwd_dxdb", w)[1] <= 1.5


def test_traffic_line_is_dropped_once_the_source_changes(tmp_path, monkeypatch):
    root = tmp_path / "repo"
    (root / "profiles").mkdir(parents=True)
    shutil.copy(os.path.join(bench.ROOT, "profiles", "dram_traffic_walks.txt"), root / "profiles")
    src = "state_space_model_ssd_gb300/csrc/ssd_tc.cu"
    (root / os.path.dirname(src)).mkdir(parents=True)
    shutil.copy(os.path.join(bench.ROOT, src), root / src)
    monkeypatch.setattr(bench, "ROOT", str(root))
    w = _w("mamba2.8b_32k")
    before = bench.measured_traffic("tc_bwd_dc", w)
    with open(root / src, "a") as f:
        f.write("\n// edited\n")
    assert bench.measured_traffic("tc_bwd_dc", w) is None
    assert before is None or before > 0


def test_roofline_fraction_is_algorithmic_bytes_over_time_over_peak():
    w = _w("mamba2.8b_32k")
    peaks = {"hbm_gbs": 6790.7}
    # 10 launches, 5.7 ms in all: 0.57 ms each
    rec = bench.roofline_record("tc_bwd_dxdb", {"tc_bwd_dxdb": (10, 5.7)}, w, peaks,
                                "measured", {})
    amount = bench.kernel_model("tc_bwd_dxdb", w)[1]
    assert rec["bound"] == "hbm" and rec["unit"] == "GB/s"
    assert rec["achieved"] == pytest.approx(amount / 0.57e-3 / 1e9)
    assert rec["frac"] == pytest.approx(rec["achieved"] / 6790.7)
    assert rec["avg_launch_ms"] == pytest.approx(0.57)
    assert bench.roofline_record("tc_bwd_dxdb", {}, w, peaks, "measured", {}) is None
