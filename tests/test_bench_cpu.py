"""Host logic of the benchmark that needs no GPU: the algorithmic byte counts
the roofline divides by, and the rule that a stored DRAM-traffic figure is
dropped once the kernel source it was measured on changes."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from dsa_inputs import WORKLOADS  # noqa: E402


def test_indexer_bytes_at_128k_by_hand():
    """131,072 index keys of 64 BF16 (16 MiB), 131,072 fp32 scores written
    (512 KiB), plus one query's qI (2 KiB) and head weights (64 B)."""
    ab = bench.algorithmic_bytes(WORKLOADS["decode_128k"])
    assert ab["indexer"] == 131072 * 128 + 131072 * 4 + 16 * 64 * 2 + 16 * 4 == 17303616


def test_step_bytes_at_128k_by_hand():
    """The step adds the scores read back, the 2,048 selected K and V rows of
    2 FP16 heads (1 KiB per token), q, the output and the index rows."""
    wl = WORKLOADS["decode_128k"]
    ab = bench.algorithmic_bytes(wl)
    kv = 2048 * 2 * 256 * 2
    small = 16 * 64 * 2 + 16 * 4 + 24 * 128 * 2 * 2 + 2048 * 4 * 2
    assert ab["kv"] == kv
    assert ab["step"] == 131072 * 128 + 131072 * 4 * 2 + kv + small


def test_int8_kv_rows_carry_their_scales():
    ab = bench.algorithmic_bytes(WORKLOADS["decode_256k_int8"])
    # one sequence, 2,048 unique rows, 2 heads x (128 codes + 4-byte scale), K and V
    assert ab["kv"] == 2048 * 2 * (128 + 4) * 2


def test_append_bytes_by_hand():
    # per token: read kI 128 B + 2 heads x 2 x 256 B; write the same (16-bit)
    assert bench.append_bytes(1, 1, 2, "bf16", "bf16") == 2 * (128 + 2 * 2 * 256)
    # INT8: each K / V row becomes 128 code bytes and a 4-byte scale
    assert bench.append_bytes(1, 1, 2, "bf16", "int8") == (128 + 1024) + (128 + 2 * 2 * 132)
    assert bench.append_bytes(4, 8, 2, "fp16", "fp16") == 32 * bench.append_bytes(1, 1, 2, "fp16", "fp16")


def test_traffic_figure_is_dropped_when_the_source_changes(monkeypatch):
    name = "decode_128k"
    assert bench.indexer_traffic(name) == bench.INDEXER_TRAFFIC[name]
    monkeypatch.setattr(bench, "TRAFFIC_SOURCE_SHA", "0" * 16)
    assert bench.indexer_traffic(name) is None


def test_whole_job_value_counts_every_rank():
    assert bench.whole_job_value(1, 8, 2.0) == pytest.approx(4000.0)
    assert bench.whole_job_value(4, 8, 2.0) == pytest.approx(16000.0)
