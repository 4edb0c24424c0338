"""The ncu traffic figures bench.py reports are keyed to the sources they were captured on:
every record must match its kernel's current sources, and each profile summary must name
that source hash, so a kernel changed without a new capture shows up here (and the bench
reports null traffic for it) instead of passing off old counters."""
import re
from pathlib import Path

import bench

ROOT = Path(__file__).resolve().parents[1]

# profile summary -> the kernel key whose traffic it records
PROFILES = {
    "chain_seq_b256_v128256.md": "chain_seq",
    "chain_stream_b256_v128256.md": "chain_stats",
    "block_row_b256_v128256.md": "block_fused",
    "tree_walk_cluster_b32_n64_v32000.md": "tree_walk",
    "tree_rr_b32_n64_v32000.md": "tree_rr",
}


def test_every_record_matches_its_sources():
    for kernel, rec in bench.NCU_TRAFFIC.items():
        assert kernel in bench.KERNEL_SOURCES, kernel
        for f in bench.KERNEL_SOURCES[kernel]:
            assert (ROOT / "speculative_decoding_token_temperature_gb300" / "csrc" / f).is_file(), f
        assert rec["src_sha"] == bench.kernel_source_sha(kernel), (kernel, rec["src_sha"])
        assert rec["bytes"] > 0


def test_profile_summaries_name_the_recorded_hash_and_bytes():
    for name, kernel in PROFILES.items():
        text = (ROOT / "profiles" / name).read_text()
        rec = bench.NCU_TRAFFIC[kernel]
        assert rec["src_sha"] in text, (name, rec["src_sha"])
        # the summary states the recorded traffic in MB with two decimals (read + written)
        mb = [float(x) for x in re.findall(r"(\d+\.\d\d) MB read", text)]
        assert mb, name
        assert any(abs(m * 1e6 - rec["bytes"]) < 0.02 * rec["bytes"] for m in mb), (name, mb, rec["bytes"])
        assert "--clock-control none" in text, name


def test_recorded_traffic_only_for_its_workload_and_rule():
    for kernel, rec in bench.NCU_TRAFFIC.items():
        assert bench.recorded_traffic(kernel, rec["workload"], rec["rule"]) == rec["bytes"]
        assert bench.recorded_traffic(kernel, rec["workload"] + "_other", rec["rule"]) is None
        assert bench.recorded_traffic(kernel, rec["workload"], rec["rule"] + "_other") is None
    assert bench.recorded_traffic("no_such_kernel", "chain_b256_v128256", "chain") is None
