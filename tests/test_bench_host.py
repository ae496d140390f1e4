"""Host logic of bench.py that needs no GPU: the roofline's `traffic` comes
from the committed ncu record only while the kernel source still hashes to
the capture's, and is null once the kernel has changed."""
import hashlib
import json
import os
import shutil

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "dsa_sparse_attention_paged_gb300", "csrc")
RECORD = os.path.join(ROOT, "profiles", "logits_fused_hist_c2.json")


def _sha(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def test_traffic_record_matches_the_committed_kernel():
    with open(RECORD) as f:
        rec = json.load(f)
    assert rec["dram_bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
    srcs = [os.path.join(CSRC, "logits.cu"), os.path.join(CSRC, "dsa_device.cuh")]
    if _sha(srcs) != rec["source_sha256"]:
        # the kernel changed after the capture: the bench must report null
        assert bench.traffic_record(srcs[0]) is None
    else:
        assert bench.traffic_record(srcs[0]) == float(rec["dram_bytes_per_launch"])


def test_traffic_record_is_null_for_a_changed_kernel(tmp_path):
    shutil.copy(os.path.join(CSRC, "logits.cu"), tmp_path / "logits.cu")
    shutil.copy(os.path.join(CSRC, "dsa_device.cuh"), tmp_path / "dsa_device.cuh")
    assert bench.traffic_record(str(tmp_path / "logits.cu")) == bench.traffic_record(
        os.path.join(CSRC, "logits.cu"))
    with open(tmp_path / "dsa_device.cuh", "a") as f:
        f.write("\n// changed\n")
    assert bench.traffic_record(str(tmp_path / "logits.cu")) is None


def test_traffic_record_missing_source_is_null(tmp_path):
    assert bench.traffic_record(str(tmp_path / "logits.cu")) is None
