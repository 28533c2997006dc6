"""`bench.py --impl reference` on the CPU: the fp64 oracle timed as it stands.

The pages ship no runnable program, so the oracle is the reference arm. These
checks run it as the driver does (a subprocess, small K and W) and read its
one JSON line: the same metric, unit, config and direction as the GPU arm,
`impl: reference`, a `cpu_baseline` that describes this run, and an `e2e`
that moves no bytes. Under a launcher, ranks other than 0 exit 0 without
work or output. A warm-up below 3 is refused.
"""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, "bench.py"] + args, cwd=ROOT, env=e,
                          capture_output=True, text=True, timeout=600)


def _line(stdout):
    lines = [l for l in stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, stdout
    return json.loads(lines[0])


def test_reference_arm_default_workload_is_the_video_vae_conv3d():
    r = _run(["--impl", "reference", "--steps", "3", "--warmup", "3"])
    assert r.returncode == 0, r.stderr
    d = _line(r.stdout)
    assert d["impl"] == "reference"
    assert d["config"]["workload"] == "conv3d_f16_1x128x5x128x240_oc128_k3p1s1"
    # a step is a seeded sample of n outputs: value = n/total of the
    # layer's FLOP per step time
    n, total = [int(v) for v in d["cpu_baseline"]["sample"].split(" outputs")[0].split(" of ")]
    flop = 2 * 128 * 5 * 128 * 240 * 128 * 27 * n / total
    assert abs(d["value"] - flop / (d["ms_per_step"] * 1e-3) / 1e12) <= 0.02 * d["value"]


def test_reference_arm_prints_one_contract_line():
    r = _run(["--impl", "reference", "--steps", "3", "--warmup", "3",
              "--workload", "detection_stem"])
    assert r.returncode == 0, r.stderr
    d = _line(r.stdout)
    assert d["impl"] == "reference"
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    # one step = one whole-layer oracle call: value = FLOP / step time
    assert d["config"]["workload"] == "conv2d_f32_1x3x640x640_oc32_k3p1s2_relu"
    flop = 2 * 32 * 320 * 320 * 3 * 9
    assert abs(d["value"] - flop / (d["ms_per_step"] * 1e-3) / 1e12) <= 0.02 * d["value"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_workload_keeps_its_config():
    r = _run(["--impl", "reference", "--steps", "3", "--warmup", "3",
              "--workload", "text_line_batch"])
    assert r.returncode == 0, r.stderr
    d = _line(r.stdout)
    assert d["impl"] == "reference"
    assert d["config"]["workload"] == "conv2d_f32_16x64x12x80_oc128_k3p1s1_relu"
    assert d["value"] > 0
    assert d["cpu_baseline"]["sample"].startswith("whole layer")   # 2.27 GFLOP: whole calls


def test_reference_arm_samples_the_large_layers():
    # the video-VAE Convolution3D (135.9 GFLOP): each step times the same
    # seeded sample of outputs, and the line says so
    r = _run(["--impl", "reference", "--steps", "3", "--warmup", "3",
              "--workload", "video_vae_conv3d_f16"])
    assert r.returncode == 0, r.stderr
    d = _line(r.stdout)
    assert d["config"]["workload"] == "conv3d_f16_1x128x5x128x240_oc128_k3p1s1"
    assert "outputs per step" in d["cpu_baseline"]["sample"]
    assert d["value"] > 0 and d["ms_per_step"] < 5000


def test_reference_arm_non_zero_rank_is_silent():
    r = _run(["--impl", "reference", "--steps", "3", "--warmup", "3"],
             env={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr
    assert not [l for l in r.stdout.splitlines() if l.strip().startswith("{")]


def test_warmup_below_three_is_refused():
    r = _run(["--impl", "reference", "--steps", "3", "--warmup", "2"])
    assert r.returncode != 0
    assert "warmup" in r.stderr
