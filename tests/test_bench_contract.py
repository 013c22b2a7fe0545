"""bench.py contract checks that need no GPU: the reference arm's JSON line and the
binding names the GPU arm calls."""
import json
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_calls_only_exported_names():
    import sparse_attention_speculative_gb300 as vsd
    src = open(os.path.join(ROOT, "bench.py")).read()
    names = set(re.findall(r"(?<![/\w\"])vsd\.(\w+)", src))
    missing = sorted(n for n in names if not hasattr(vsd, n))
    assert not missing, "bench.py uses names the package does not export: %s" % missing


def test_reference_arm_prints_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_p512_d64", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1]
    res = json.loads(line)
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in res, key
    assert res["impl"] == "reference"
    assert res["value"] > 0
    assert res["cpu_baseline"]["kind"] == "oracle" and res["cpu_baseline"]["cores"] >= 1
    assert res["e2e"]["h2d_bytes_per_step"] == 0 and res["e2e"]["value"] == res["value"]
    assert res["config"]["workload"] == "tiny_p512_d64"


def test_reference_arm_under_torchrun_prints_once():
    """Two ranks launched as the multi-GPU contract launches them: rank 0 alone runs the
    oracle and prints one JSON line, the other rank exits 0 without work."""
    import socket
    with socket.socket() as s_:
        s_.bind(("127.0.0.1", 0))
        port = s_.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port",
                        str(port), os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--workload", "tiny_p512_d64", "--steps", "1",
                        "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["value"] > 0


def test_algorithmic_bytes_match_the_configuration_table():
    """The bytes the benchmark divides by, against the figures the configurations are
    stated with: the Qwen3-8B 32K layer (verification 142.7 MB: K/V 134.2 + logits 8.4 +
    q/out, plus the 1 MB of partials it also writes; one draft step 8.4 MB) and the
    36-layer loop (per iteration 41.1 GB of verification, 0.30 GB of selection, 2.42 GB
    per draft step)."""
    sys.path.insert(0, ROOT)
    import bench
    from sparse_attention_speculative_gb300.workloads import LOOP_36L, QWEN3_8B_32K

    w = QWEN3_8B_32K
    prefix = list(w.prefix())
    vb, sb, spb = bench.iteration_bytes(w, prefix, [w.k] * w.B,
                                        [[2 + i] * w.B for i in range(w.gamma)])
    assert abs(vb / 1e6 - (142.7 + 1.05)) < 0.5
    assert all(abs(x / 1e6 - 8.4) < 0.1 for x in spb)
    w = LOOP_36L
    prefix = list(w.prefix())
    vb, sb, spb = bench.iteration_bytes(w, prefix, [w.k] * w.B,
                                        [[2 + i] * w.B for i in range(w.gamma)])
    L = w.layers
    assert abs(L * vb / 1e9 - 41.1) / 41.1 < 0.01
    assert abs(L * sb / 1e9 - 0.30) / 0.30 < 0.02
    assert all(abs(L * x / 1e9 - 2.42) / 2.42 < 0.01 for x in spb)


def test_loop_run_bytes_follow_the_growing_prefix():
    """A decode run's bytes: the first iteration is the configuration's iteration at P
    (plus the appends), and every iteration's prefix is the previous one plus the
    accepted drafts plus one."""
    sys.path.insert(0, ROOT)
    import bench
    from sparse_attention_speculative_gb300.workloads import LOOP_36L as w
    acc = [[(i + b) % (w.gamma + 1) for b in range(w.B)] for i in range(w.iterations)]
    run = bench.loop_run_bytes(w, acc)
    assert len(run) == w.iterations
    vb, sb, spb = bench.iteration_bytes(w, list(w.prefix()), [w.k] * w.B,
                                        [[acc[0][b] + 2 + i for b in range(w.B)]
                                         for i in range(w.gamma)])
    assert run[0]["verify"] == w.layers * vb and run[0]["select"] == w.layers * sb
    assert run[0]["sparse"] == w.layers * sum(spb)
    # appends: (R + gamma) rows of K and V per sequence and KV head, read and written
    assert run[0]["append"] == w.layers * 4 * w.B * (w.R + w.gamma) * w.Hkv * w.d * 2
    for i in range(1, w.iterations):
        assert run[i]["prefix"] == [p + a + 1 for p, a in zip(run[i - 1]["prefix"], acc[i - 1])]
    assert run[-1]["verify"] > run[0]["verify"]


def test_bench_defaults_to_the_decode_loop():
    src = open(os.path.join(ROOT, "bench.py")).read()
    assert 'default="qwen3_8b_36layer_loop"' in src
