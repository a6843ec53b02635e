"""The committed DRAM-traffic records under profiles/ describe the kernel
sources as they stand.

bench.py reports a kernel's measured DRAM traffic from these records only
while the record's source hash matches the kernel's current sources (else
it reports null).  This test fails as soon as a kernel source changes
without a fresh capture, so a stale record cannot go unnoticed."""
import glob
import json
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
RECORDS = sorted(glob.glob(os.path.join(ROOT, "profiles", "*_traffic.json")))


def test_records_exist():
    names = {os.path.basename(p) for p in RECORDS}
    assert {"scan_long_bf16_traffic.json", "linattn_bf16_traffic.json"} <= names


@pytest.mark.parametrize("path", RECORDS, ids=[os.path.basename(p) for p in RECORDS])
def test_record_matches_current_kernel_sources(path):
    rec = json.load(open(path))
    kernel = rec["kernel"].split("<")[0]
    assert sorted(rec["kernel_sources"]) == sorted(bench.KERNEL_SOURCES[kernel])
    assert rec["kernel_source_sha"] == bench.kernel_source_hash(kernel), (
        f"{os.path.basename(path)} was captured on older sources of {kernel}: re-capture it")


@pytest.mark.parametrize("path", RECORDS, ids=[os.path.basename(p) for p in RECORDS])
def test_record_is_consistent(path):
    rec = json.load(open(path))
    per = (rec["dram_bytes_read"] + rec["dram_bytes_write"]) / rec["head_tokens"]
    assert per == pytest.approx(rec["dram_bytes_per_head_token"], rel=1e-9)
    assert rec["passes"] == 1
    # no re-reads: within a few percent of the algorithmic bytes (writes may stay in L2)
    assert 0.5 * rec["algorithmic_bytes_per_head_token"] < per <= 1.05 * rec["algorithmic_bytes_per_head_token"]
