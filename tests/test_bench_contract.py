"""bench.py's reference arm (the fp64 oracle on the host cores) prints the one JSON line the
benchmark contract asks for; ranks other than 0 print nothing and exit 0.  CPU only."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra):
    env = dict(os.environ, **env_extra)
    # a short sequence keeps the oracle sample to a second or two
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--n", "1024", "--steps", "1",
                           "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_json_line():
    r = _run({})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["metric"].startswith("attention backward TFLOP/s")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] and d["config"]["Nq"] == 1024


def test_reference_arm_other_ranks_are_silent():
    r = _run({"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def _bench_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_bench_parity_of_one_group():
    """The bench's CPU leg runs the oracle on one group of the run's own inputs and reports the
    GPU gradients' error against it; here the 'GPU' gradients are the oracle's own (rounded to
    16 bits), then one with a planted error."""
    import torch
    from attn_bwd_gb300 import inputs
    from oracle import attn_ref
    bench = _bench_module()
    sh = inputs.Shape(1, 4, 1, 96, 96, 32, 1, "bf16")
    q, k, v, do = inputs.draw(sh, 5)
    ref = attn_ref.backward(q, k, v, do, sh.softmax_scale, sh.causal)
    grads = [torch.from_numpy(ref[n]).to(torch.bfloat16) for n in ("dq", "dk", "dv")]
    base, par = bench.run_cpu_baseline(sh, (q, k, v, do, *grads))
    assert base["kind"] == "oracle" and base["value"] > 0 and base["cores"] >= 1
    assert set(par) == {"dq", "dk", "dv"} and all(0 <= r < 0.5 for r in par.values()), par
    bad = grads[0].clone()
    bad[0, 1, 7, 3] += 0.05 * float(bad.float().abs().max())
    _, par2 = bench.run_cpu_baseline(sh, (q, k, v, do, bad, grads[1], grads[2]))
    assert par2["dq"] > 1.0 and par2["dk"] == par["dk"]
    base3, none = bench.run_cpu_baseline(sh)
    assert none is None and base3["value"] > 0
