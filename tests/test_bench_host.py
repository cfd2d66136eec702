"""bench.py's host logic on CPU: algorithmic work per weight format, the
kernel-source hash behind the DRAM traffic records, and the reference arm's
JSON line (the oracle on a token sample)."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402

E, H, I = 4, 256, 128
OFFSETS = np.array([0, 2, 2, 5, 6])  # expert 1 has no rows: three active experts


def work(fp8=False, nvfp4=False):
    return bench.algorithmic_work(dict(E=E, H=H, I=I, fp8=fp8, nvfp4=nvfp4), OFFSETS)


def test_bf16_work():
    w = work()
    assert w["active_experts"] == 3 and w["rows"] == 6
    assert w["fc1_bytes"] == 3 * (2 * I) * H * 2
    assert w["fc2_bytes"] == 3 * H * I * 2
    assert w["fc1_flops"] == 2.0 * 6 * H * 2 * I
    assert w["fc2_flops"] == 2.0 * 6 * I * H


def test_fp8_formats_are_told_apart():
    per_channel = work(fp8=True)
    block = work(fp8="block")
    # E4M3 codes plus one fp32 scale per output channel ...
    assert per_channel["fc1_bytes"] == 3 * ((2 * I) * H + 2 * I * 4)
    assert per_channel["fc2_bytes"] == 3 * (H * I + H * 4)
    # ... or per 128 x 128 tile
    assert block["fc1_bytes"] == 3 * ((2 * I) * H + (2 * I // 128) * (H // 128) * 4)
    assert block["fc2_bytes"] == 3 * (H * I + (H // 128) * (I // 128) * 4)
    assert block["fc1_flops"] == per_channel["fc1_flops"] == work()["fc1_flops"]


def test_nvfp4_work():
    w = work(nvfp4=True)
    # half a byte per code, one E4M3 scale per 16 codes, one fp32 per matrix
    assert w["fc1_bytes"] == 3 * ((2 * I) * H // 2 + (2 * I) * H // 16 + 4)
    assert w["fc2_bytes"] == 3 * (H * I // 2 + H * I // 16 + 4)


def test_kernel_source_sha_follows_the_kernel_file():
    shas = {w: bench.kernel_source_sha(w) for w in workloads.CONFIGS}
    assert len(set(shas.values())) == 3        # gemm_tc.cu, gemm_nvfp4.cu, gemm_fp8b.cu
    assert shas["c2_decode_balanced"] == shas["c5_prefill"] == shas["c8_prefill_fp8"]
    assert shas["c7_decode_fp8_block"] == shas["c9_prefill_fp8_block"]
    assert shas["c6_decode_nvfp4"] not in (shas["c2_decode_balanced"], shas["c7_decode_fp8_block"])
    assert all(len(v) == 12 for v in shas.values())
    assert bench.kernel_source_sha("c2_decode_balanced") == shas["c2_decode_balanced"]


def test_traffic_records_are_keyed_on_the_current_source():
    assert bench.read_traffic("ffn", "no_such_workload") is None
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    for ln in open(path):
        parts = ln.split()
        if ln.startswith("#") or len(parts) < 4:
            continue
        kernel, wl, sha, nbytes = parts[:4]
        got = bench.read_traffic(kernel, wl)
        # a record is used only while it matches the kernel's source
        assert got == (float(nbytes) if sha == bench.kernel_source_sha(wl) else None)


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "c1_tiny", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "c1_tiny" and d["higher_is_better"] is True


@pytest.mark.parametrize("name", sorted(workloads.CONFIGS))
def test_every_workload_has_a_cpu_sample_size(name):
    assert bench.auto_cpu_tokens(name) >= 1
