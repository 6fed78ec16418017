"""Host logic of bench.py that needs no GPU: the roofline record, the
pointer to the committed DRAM-traffic captures, and the reference arm."""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _prof(ms_gemm=24.0, ms_attn=3.0):
    return {
        "gemm_tc": {"launches": 32, "ms": 2 * ms_gemm, "flops": 84e12,
                    "bytes": 2.6e10},
        "attn_bwd_dkdv": {"launches": 2, "ms": 2 * ms_attn, "flops": 3.3e12,
                          "bytes": 6e8},
        "rmsnorm": {"launches": 0, "ms": 0.0, "flops": 0.0, "bytes": 0.0},
    }


PEAKS = {"bf16_tflops": 1907.0, "bf16_tflops_sustained": 1714.4,
         "hbm_gbs": 6796.9}


def test_roofline_picks_the_dominant_family_and_divides_per_launch():
    roof, kernels = bench.roofline(_prof(), 2, PEAKS, "measured")
    assert roof["kernel"] == "gemm_tc" and roof["bound"] == "tensor"
    per_launch_s = 24.0 * 2 / 32 / 1e3
    assert abs(roof["achieved"] - 84e12 / 32 / per_launch_s / 1e12) < 1e-6
    # timed over well under a second: the burst peak is the denominator
    assert abs(roof["frac"] - roof["achieved"] / 1907.0) < 1e-12
    assert abs(roof["frac_sustained"] - roof["achieved"] / 1714.4) < 1e-12
    assert "rmsnorm" not in kernels   # families without launches are dropped
    assert abs(sum(k["share"] for k in kernels.values()) - 1.0) < 1e-12


def test_traffic_points_at_the_single_launch_captures():
    # no per-launch traffic figure for a step of differently shaped GEMMs;
    # the note names the committed summary of the single-launch captures
    roof, _ = bench.roofline(_prof(), 2, PEAKS, "measured")
    assert roof["traffic"] is None
    path = roof["traffic_source"].split(" ")[0]
    assert os.path.exists(os.path.join(ROOT, path))
    text = open(os.path.join(ROOT, path), encoding="utf-8").read()
    assert "--clock-control none" in text and "-c 1" in text


def test_reference_arm_maps_no_product_library():
    # the oracle arm counts its FLOPs with the oracle's own accountant: after
    # a full run of the arm, libtp.so is not mapped into the process
    import subprocess
    code = (
        "import sys, json; sys.argv = ['bench.py', '--impl', 'reference', "
        "'--workload', 'mlp_gelu_bf16', '--steps', '1', '--warmup', '0']\n"
        "import bench; bench.main()\n"
        "maps = open('/proc/self/maps').read()\n"
        "print('LIBTP' if 'libtp.so' in maps else 'CLEAN')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = r.stdout.strip().splitlines()
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert lines[-1] == "CLEAN"


def test_oracle_flop_count_equals_the_library_accountant(tp):
    # the two counts agree bit for bit on every workload's bench sample and
    # on the full workloads
    from megatron_tensor_transformer_gate_gb300 import inputs as I
    for name in ("layer_bf16", "mlp_swiglu_bf16", "mlp_gelu_bf16",
                 "attn_gqa_bf16"):
        cfg = I.workload(name)
        for c in (cfg, bench.cpu_sample_cfg(cfg)):
            assert bench.oracle_flops_per_step(c) == bench.flops_per_step(c)
