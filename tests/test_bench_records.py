"""The ncu traffic figures bench.py reports are keyed to the sources they were captured on:
a record whose kernel sources changed since its capture is reported as null traffic, never
as a figure of the current kernel, and each profile summary names the source hash of the
traffic it records."""
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


def test_records_name_existing_sources_and_stale_ones_read_null():
    for kernel, rec in bench.NCU_TRAFFIC.items():
        assert kernel in bench.KERNEL_SOURCES, kernel
        for f in bench.KERNEL_SOURCES[kernel]:
            assert (ROOT / "speculative_decoding_token_temperature_gb300" / "csrc" / f).is_file(), f
        assert rec["bytes"] > 0
        current = rec["src_sha"] == bench.kernel_source_sha(kernel)
        got = bench.recorded_traffic(kernel, rec["workload"], rec["rule"])
        assert got == (rec["bytes"] if current else None), (kernel, rec["src_sha"], got)


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
        if rec["src_sha"] == bench.kernel_source_sha(kernel):
            assert bench.recorded_traffic(kernel, rec["workload"], rec["rule"]) == rec["bytes"]
        assert bench.recorded_traffic(kernel, rec["workload"] + "_other", rec["rule"]) is None
        assert bench.recorded_traffic(kernel, rec["workload"], rec["rule"] + "_other") is None
    assert bench.recorded_traffic("no_such_kernel", "chain_b256_v128256", "chain") is None
