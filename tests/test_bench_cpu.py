"""Host logic of bench.py that needs no GPU: the reference arm's JSON line (the
fp64 oracle timed on the host cores) and the rule that a committed ncu summary's
DRAM traffic is reported only while the kernel sources still hash to the value
it was taken on."""
import io
import json
import os
import sys
from contextlib import redirect_stdout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def run_json(argv):
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.main(argv) in (0, None)
    return json.loads(buf.getvalue().strip().splitlines()[-1])


def test_reference_arm_line_on_the_tiny_workload():
    line = run_json(["--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3"])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "GB/s"
    assert line["value"] > 0 and line["steps"] == 3 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["dtype"] == "f64" and line["config"]["accumulate"] == "fp64"
    assert line["higher_is_better"] is True and line["vs_baseline"] is None
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert line["config"]["workload"].startswith("tiny: B=2")


def test_warmup_below_three_is_refused():
    import pytest
    with pytest.raises(SystemExit):
        bench.main(["--impl", "reference", "--workload", "tiny", "--warmup", "2"])


def test_profiled_traffic_follows_the_source_hash(tmp_path):
    files = ["decode.cuh", "decode_common.cuh"]
    good = tmp_path / "good.md"
    good.write_text("source_files: %s\nsource_sha256: %s\ndram_bytes_per_launch: 12345\n"
                    % (" ".join(files), bench.kernel_source_hash(files)))
    assert bench.profiled_traffic(str(good)) == 12345
    stale = tmp_path / "stale.md"
    stale.write_text("source_files: %s\nsource_sha256: 0000000000000000\ndram_bytes_per_launch: 12345\n"
                     % " ".join(files))
    assert bench.profiled_traffic(str(stale)) is None
    assert bench.profiled_traffic(str(tmp_path / "missing.md")) is None
    # a different file list hashes differently
    assert bench.kernel_source_hash(files) != bench.kernel_source_hash(files[:1])


def test_committed_profiles_name_existing_sources():
    for path in list(bench.PROFILE_SUMMARIES.values()) + [bench.MLA_PROFILE_SUMMARY]:
        text = open(path).read()
        names = [l for l in text.splitlines() if l.startswith("source_files:")]
        assert names, path
        for f in names[0].split()[1:]:
            assert os.path.exists(os.path.join(ROOT, "paged_kv_gqa_table_gb300", "csrc", f)), (path, f)


def test_l2_note_states_the_cold_clean_flush():
    from paged_kv_gqa_table_gb300 import synth
    case = synth.decode_case(seed=0, **synth.WORKLOADS["tiny"])
    cfg = bench.workload_config(case, "tiny")
    assert cfg["l2"] == bench.L2_NOTE and "256 MiB written" in cfg["l2"] and "read" in cfg["l2"]
    assert bench.workload_config(case, "tiny", flushed=False, accumulate="fp64")["accumulate"] == "fp64"


def test_headline_is_the_largest_single_gpu_decode_configuration():
    # The default workload (no --workload) is the GQA-6, D = 256 vLLM-layout
    # step, the largest decode configuration; the others are per_config lines.
    from paged_kv_gqa_table_gb300 import synth
    assert bench.HEADLINE == "gqa6_d256_vllm_decode"
    sizes = {n: synth.kv_bytes(synth.decode_case(seed=0, **synth.WORKLOADS[n]))
             for n in ("llama3_8b_decode", "long_context_decode", "gqa6_d256_vllm_decode")}
    assert max(sizes, key=sizes.get) == bench.HEADLINE
    assert {"llama3_8b_decode", "long_context_decode", "mla_prefill_h16"} <= set(bench.PER_CONFIG)


def test_profiled_field_follows_the_source_hash(tmp_path):
    files = ["decode.cuh"]
    good = tmp_path / "good.md"
    good.write_text("source_files: %s\nsource_sha256: %s\ndram_bytes_per_launch: 1\ndram_throughput_pct: 87.5\n"
                    % (" ".join(files), bench.kernel_source_hash(files)))
    assert bench.profiled_field(str(good), "dram_throughput_pct") == 87.5
    assert bench.profiled_field(str(good), "tensor_pipe_pct") is None
    stale = tmp_path / "stale.md"
    stale.write_text("source_files: decode.cuh\nsource_sha256: 0\ndram_bytes_per_launch: 1\n"
                     "dram_throughput_pct: 87.5\n")
    assert bench.profiled_field(str(stale), "dram_throughput_pct") is None
