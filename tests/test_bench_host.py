"""Host-side checks (no GPU) of bench.py's contract: the reference arm's JSON line, the
config both arms share, the rule that the timed inputs do not fit in L2, and the source
hash that ties a committed ncu summary to the kernel it was taken on."""
import contextlib
import io
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from scaled_dot_product_sdpa_gb300.configs import WORKLOADS  # noqa: E402

LINE_KEYS = {"metric", "value", "unit", "impl", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
             "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


@pytest.fixture(autouse=True)
def _single_process(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)


def run_reference(workload, steps=1):
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        bench.main(["--impl", "reference", "--workload", workload, "--steps", str(steps), "--warmup", "0"])
    lines = [json.loads(x) for x in out.getvalue().splitlines() if x.startswith("{")]
    assert len(lines) == 1, out.getvalue()
    return lines[0]


def test_reference_arm_prints_one_contract_line():
    d = run_reference("caseA")
    assert LINE_KEYS <= set(d), LINE_KEYS - set(d)
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["warmup"] == 3  # the contract's minimum is enforced
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOPS" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["vs_baseline"] is None and d["data"] == "synthetic" and d["dtype"] == "f64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and "heads" in cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_both_arms_share_the_config():
    d = run_reference("caseA")
    assert d["config"] == bench.workload_config(WORKLOADS["caseA"], 1)
    assert d["config"]["workload"] == "caseA"


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_timed_inputs_exceed_l2(name):
    w = WORKLOADS[name]
    assert bench.n_rotating_sets(w) * w.bytes() > 2 * bench.L2_BYTES


def test_source_hash_ignores_comments_only():
    code = "int a = 1;  // first\n/* block\n comment */\nint b = a + 2;\n\n"
    assert bench._code_only(code) == "int a = 1;\nint b = a + 2;"
    assert bench._code_only(code.replace("first", "changed")) == bench._code_only(code)
    assert bench._code_only(code.replace("a + 2", "a + 3")) != bench._code_only(code)


def test_source_hash_covers_each_kernel_family():
    hashes = {k: bench.kernel_source_hash(k) for k in ("fwd", "decode", "bwd")}
    assert all(len(h) == 16 for h in hashes.values())
    assert len(set(hashes.values())) == 3
