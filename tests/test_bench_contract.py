"""bench.py's contract on the host (no GPU): the reference arm's JSON line and
the committed ncu summaries the bench reads its roofline traffic from.

Every summary under profiles/ that carries a source_sha256 names the kernel
source it was captured on; the hash (comments and whitespace stripped) must
be that of the source as it stands, so that no figure in profiles/ describes
a kernel that has changed since."""

import json
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

# profile file prefix -> kernel source
SOURCES = {
    "conv": "gate_conv.cu",
    "kv_proj_gate": "kv_proj.cu",
    "gather_fp8": "lookup.cu",
    "lookup": "lookup.cu",
    "ngram_lookup": "lookup.cu",
}
WORKLOADS = ("fp8x8", "prefill8k", "decode256x4", "uva32g", "tiny")


def hashed_profiles():
    out = []
    for name in sorted(os.listdir(os.path.join(ROOT, "profiles"))):
        text = open(os.path.join(ROOT, "profiles", name)).read()
        m = re.search(r"^source_sha256: `([0-9a-f]{16})`", text, flags=re.M)
        if m:
            out.append((name, m.group(1), text))
    return out


def test_reference_arm_prints_one_contract_line():
    res = subprocess.run(
        [sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "2",
         "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_profiles_name_their_source_and_bytes():
    profiles = hashed_profiles()
    assert len(profiles) >= 8
    for name, _, text in profiles:
        stem = name[:-3]
        kernel = next((k for k in sorted(SOURCES, key=len, reverse=True)
                       if stem.startswith(k + "_") and stem[len(k) + 1:] in WORKLOADS), None)
        assert kernel is not None, f"{name}: no kernel/workload in its name"
        m = re.search(r"^(dram|link)_bytes_per_launch: `(\d+)`", text, flags=re.M)
        assert m and int(m.group(2)) > 0, f"{name}: no bytes per launch"
        assert "--clock-control none" in text, f"{name}: ncu without --clock-control none"


@pytest.mark.parametrize("name,digest", [(n, h) for n, h, _ in hashed_profiles()])
def test_profiles_match_the_current_sources(name, digest):
    stem = name[:-3]
    kernel = next(k for k in sorted(SOURCES, key=len, reverse=True) if stem.startswith(k + "_"))
    src = os.path.join(ROOT, "hashed_gram_embedding_gb300", "csrc", SOURCES[kernel])
    assert digest == bench.source_hash(src), (
        f"{name} was captured on another version of {SOURCES[kernel]}: capture it again")


def test_ncu_traffic_reads_the_roofline_summaries():
    assert bench.ncu_traffic("kv_proj_gate", "fp8x8") > 0
    assert bench.ncu_traffic("kv_proj_gate", "prefill8k") > 0
    assert bench.ncu_traffic("lookup", "uva32g", "link_bytes_per_launch") > 0
    assert bench.ncu_traffic("lookup", "no_such_workload") is None


def test_source_hash_ignores_comments_and_whitespace(tmp_path):
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    a.write_text("int f() { return 1; }  // one\n/* block */\n")
    b.write_text("int f()\n{\n  return 1;\n}\n")
    assert bench.source_hash(str(a)) == bench.source_hash(str(b))
    b.write_text("int f() { return 2; }\n")
    assert bench.source_hash(str(a)) != bench.source_hash(str(b))
