"""bench.py's reference arm (the oracle timed on the host cores) prints one JSON line with the
contract's keys; warm-up below 3 is refused.  CPU only: the reference arm needs no GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, timeout=600):
    return subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True, text=True,
                          timeout=timeout)


def test_reference_arm_prints_one_contract_line():
    r = _run("--impl", "reference", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key, typ in (("metric", str), ("value", float), ("unit", str), ("n_gpus", int), ("steps", int),
                     ("warmup", int), ("ms_per_step", float), ("higher_is_better", bool), ("scaling", str),
                     ("dtype", str), ("data", str), ("config", dict), ("cpu_baseline", dict), ("e2e", dict)):
        assert isinstance(d[key], typ), key
    assert d["value"] > 0 and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert isinstance(cb["cpu_model"], str) and cb["cpu_model"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_warmup_below_three_is_refused():
    r = _run("--impl", "reference", "--steps", "1", "--warmup", "1", timeout=300)
    assert r.returncode != 0 and "warmup" in r.stderr


def test_tensor_sha256_is_the_bit_pattern_digest():
    import hashlib

    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    import bench
    t = torch.tensor([[1.0, -2.5], [3.0, 0.125]], dtype=torch.bfloat16)
    raw = t.view(torch.int16).numpy().astype("<i2").tobytes()
    assert bench.tensor_sha256(t) == hashlib.sha256(raw).hexdigest()
    f = torch.arange(6, dtype=torch.float32).reshape(2, 3)
    assert bench.tensor_sha256(f) == hashlib.sha256(np.arange(6, dtype="<f4").tobytes()).hexdigest()
    assert bench.tensor_sha256(f.t()) != bench.tensor_sha256(f)     # row-major bytes of the view
