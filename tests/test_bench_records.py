"""The ncu traffic figures bench.py reports are keyed to the sources they were captured on:
a record whose kernel sources changed since its capture is reported as null traffic, never
as a figure of the current kernel, and each profile summary names the source hash of the
traffic it records."""
import re
from pathlib import Path

import bench

ROOT = Path(__file__).resolve().parents[1]



def _summaries_of(kernel):
    """The committed profile summaries that cite this kernel's source hash."""
    key = f'kernel_source_sha("{kernel}")'
    return [(p.name, p.read_text()) for p in sorted((ROOT / "profiles").iterdir())
            if p.is_file() and key in p.read_text()]


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
    """Every traffic record has a profile summary that names its source hash and states the
    recorded traffic (MB read, two decimals) and the ncu command's --clock-control none."""
    for kernel, rec in bench.NCU_TRAFFIC.items():
        found = []
        for name, text in _summaries_of(kernel):
            mb = [float(x) for x in re.findall(r"(\d+\.\d\d) MB read", text)]
            if rec["src_sha"] in text and any(abs(m * 1e6 - rec["bytes"]) < 0.02 * rec["bytes"] for m in mb):
                assert "--clock-control none" in text, name
                found.append(name)
        assert found, (kernel, rec["src_sha"], rec["bytes"])


def test_recorded_traffic_only_for_its_workload_and_rule():
    for kernel, rec in bench.NCU_TRAFFIC.items():
        if rec["src_sha"] == bench.kernel_source_sha(kernel):
            assert bench.recorded_traffic(kernel, rec["workload"], rec["rule"]) == rec["bytes"]
        assert bench.recorded_traffic(kernel, rec["workload"] + "_other", rec["rule"]) is None
        assert bench.recorded_traffic(kernel, rec["workload"], rec["rule"] + "_other") is None
    assert bench.recorded_traffic("no_such_kernel", "chain_b256_v128256", "chain") is None
