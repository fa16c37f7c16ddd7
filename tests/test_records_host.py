"""The committed DRAM traffic records (profiles/dram_traffic.json) that the
bench reports as `roofline.traffic`: well formed, and taken on the current
code of every kernel whose line reports one.  A kernel change without a new
capture fails here instead of silently turning the bench's `traffic` to
null.  The cross K/V fill's record predates the current shared headers and
is documented as reading null, so it is only checked for its form.
"""
import importlib.util
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_for_records",
                                                  os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.fixture(scope="module")
def records():
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        return json.load(f)["records"]


def test_records_are_well_formed(records):
    seen = set()
    for r in records:
        assert isinstance(r["workload"], str) and isinstance(r["kernel"], str)
        assert len(r["code_sha"]) == 16 and int(r["code_sha"], 16) >= 0
        assert isinstance(r["dram_bytes_per_launch"], int) and r["dram_bytes_per_launch"] > 0
        alg = r.get("algorithmic_bytes_per_launch")
        assert alg is None or (isinstance(alg, int) and alg > 0)
        key = (r["workload"], r["kernel"])
        assert key not in seen, f"two records for {key}"
        seen.add(key)


CURRENT = [
    # workload, traffic key, sources the bench hashes for it
    ("whisper_large_b32", "cross", "DECODE_SOURCES"),
    ("whisper_large_b32", "self+append", "DECODE_SOURCES"),
    ("qwen3_asr_gqa_b16", "gqa", "DECODE_SOURCES"),
    ("whisper_tiny_b64_beam5", "cross", "DECODE_SOURCES"),
    ("whisper_tiny_b64_beam5", "self+append+reorder", "DECODE_SOURCES"),
    ("qwen3_asr_prefill_b8", "prefill_attn", "PREFILL_SOURCES"),
    ("whisper_large_encoder_b8", "asr_encoder_attn", "PREFILL_SOURCES"),
    ("whisper_large_prefill_b32", "asr_mha_prefill", "PREFILL_SOURCES"),
]


@pytest.mark.parametrize("workload,kernel,sources", CURRENT)
def test_record_matches_the_current_code(bench, records, workload, kernel, sources):
    rec = [r for r in records if r["workload"] == workload and r["kernel"] == kernel]
    assert len(rec) == 1, f"no record for {workload} / {kernel}"
    sha = bench.code_sha(getattr(bench, sources))
    assert rec[0]["code_sha"] == sha, (
        f"{workload} / {kernel}: record taken on {rec[0]['code_sha']}, code is {sha}: "
        "capture the kernel's DRAM bytes again")
    # and the bench reads it back
    assert bench.recorded_traffic(getattr(bench, sources), workload, kernel) == \
        rec[0]["dram_bytes_per_launch"]
