"""bench.py's JSON line (reference arm, on CPU): one line with the keys the
benchmark contract asks for."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["unit"] == "us/call" and d["higher_is_better"] is False and d["steps"] == 3
    assert d["config"]["workload"] == "wan_32760x40x128"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["value"] > 0


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "2"], capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert r.returncode != 0


def test_config_sweep_names_every_configuration():
    # the default bench line times every workload of the five configurations
    # and their variants, plus the next rows' workloads
    sys.path.insert(0, ROOT)
    import bench
    from diffusion_transformer_qk_gb300 import inputs as I

    names = [bench.sweep_entry_name(n, o) for n, o in bench.CONFIG_SWEEP]
    assert len(set(names)) == len(names)
    known = set(I.WORKLOADS) | set(I.ADALN_WORKLOADS) | set(I.GN_WORKLOADS)
    assert all(n in known for n, _ in bench.CONFIG_SWEEP)
    assert set(I.WORKLOADS) <= {n for n, _ in bench.CONFIG_SWEEP}
    assert set(I.ADALN_WORKLOADS) | set(I.GN_WORKLOADS) <= {n for n, _ in bench.CONFIG_SWEEP}
    wan = [I.WORKLOADS[n].with_(**o) for n, o in bench.CONFIG_SWEEP if n.startswith("wan")]
    assert {(w.cos_layout, w.cos_dtype, w.rope_style) for w in wan} >= {
        (lay, cd, st) for lay in ("per_head_expanded",) for cd in ("fp32", "bf16")
        for st in ("interleaved", "rotate_half")}
    flux = [I.WORKLOADS[n].with_(**o) for n, o in bench.CONFIG_SWEEP if n.startswith("flux")]
    assert {(w.dtype, w.single_launch) for w in flux} == {(d, s) for d in ("bf16", "fp16") for s in (False, True)}
