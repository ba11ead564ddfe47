"""The bench's reference arm (the CPU oracle timed on the host cores) runs without a GPU
and prints one JSON line with the keys the measurement contract asks for."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--steps", "1", "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert "smaller than L2" in d["config"]["l2"]  # tiny: said so, not claimed otherwise


def test_traffic_record_is_void_once_the_kernel_sources_change(tmp_path, monkeypatch):
    """roofline.traffic comes from a recorded ncu capture only while the hashed kernel sources
    are the ones it was taken on; other shapes get none."""
    import hashlib
    import shutil

    sys.path.insert(0, ROOT)
    import bench
    from sparse_moe_layer_12_b300 import inputs as I

    csrc = os.path.join(ROOT, "sparse_moe_layer_12_b300", "csrc")
    root = tmp_path / "repo"
    shutil.copytree(csrc, root / "sparse_moe_layer_12_b300" / "csrc")
    (root / "profiles").mkdir()
    rec = {}
    for key, srcs in (("bf16", ["expert_gemm.cu", "moe_device.cuh"]), ("fp8", ["expert_gemm_fp8.cu", "moe_device.cuh"]),
                      ("fp8_pow2", ["expert_gemm_mx.cu", "moe_device.cuh"])):
        h = hashlib.sha256()
        for name in srcs:
            h.update((root / "sparse_moe_layer_12_b300" / "csrc" / name).read_bytes())
        rec[key] = {"bytes_per_launch": float(len(key)), "sources": srcs, "sources_sha256": h.hexdigest()}
    (root / "profiles" / "expert_ffn_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench._traffic(I.CONFIGS["v3"]) == 4.0
    assert bench._traffic(I.CONFIGS["v3fp8"]) == 3.0
    assert bench._traffic(I.CONFIGS["v3fp8p2"]) == 8.0
    assert bench._traffic(I.CONFIGS["mid"]) is None
    assert bench._traffic(I.CONFIGS["v3fp8"].with_(T=1024)) is None
    with open(root / "sparse_moe_layer_12_b300" / "csrc" / "expert_gemm_mx.cu", "a") as f:
        f.write("\n// changed\n")
    assert bench._traffic(I.CONFIGS["v3fp8p2"]) is None
    assert bench._traffic(I.CONFIGS["v3"]) == 4.0
