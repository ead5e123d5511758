"""Host-side checks of bench.py: the algorithmic accounting behind its roofline figures,
the single-GPU rule of the GPU arm, and the config both arms print."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_accounting_of_the_tiny_workload():
    import bench
    from workloads import mla as W
    p = W.config_tiny()
    alg = bench.algorithmic(p)
    keys = 37 + 70                                  # causal, one query at the end of each cache
    assert alg["keys"] == keys
    assert alg["kv_bytes"] == keys * 2 * (64 + 16)
    pages = 3 + 5
    assert alg["decode_bytes"] == alg["kv_bytes"] + 4 * pages
    w = 2 * (4 * 64 * 32 + 4 * 32 * 64)
    assert alg["total_bytes"] == alg["decode_bytes"] + w + 2 * 4 * 48 * 2 + 2 * 4 * 32 * 2
    flops = 2 * 4 * keys * 80 + 2 * 4 * keys * 64 + 2 * 2 * 4 * 64 * 32 + 2 * 2 * 4 * 32 * 64
    assert alg["flops"] == flops


def _bench(*argv, env=None):
    e = dict(os.environ)
    e.update(env or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *argv], capture_output=True,
                       text=True, env=e, timeout=300)
    return r


def test_gpu_arm_refuses_more_than_one_gpu():
    # no device is touched: the refusal comes before torch or the library is imported
    r = _bench("--gpus", "2", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["n_gpus"] == 2 and "single GPU only" in line["unavailable"]
    r = _bench("--steps", "1", "--warmup", "3", env={"WORLD_SIZE": "4", "RANK": "1"})
    assert r.returncode == 0 and r.stdout.strip() == ""      # only rank 0 prints


def test_both_arms_describe_the_workload_alike():
    import argparse

    import bench
    from workloads import mla as W
    p = W.config_tiny()
    a = argparse.Namespace(num_splits=0)
    assert bench.config_of(p, a) == bench.config_of(p, a)
    cfg = bench.config_of(p, a)
    assert cfg["global_batch"] == 2 and cfg["query_tokens"] == 2 and cfg["num_splits"] == "auto"
