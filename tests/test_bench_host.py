"""bench.py's host-side helpers on the CPU: the committed DRAM record is used
only while the node kernel's sources are unchanged, peaks fall back when no
measurement file exists, seeds differ per rank and per workload, and the
oracle's sample arrays keep the library's layout."""
import json

import numpy as np
import torch

import bench
from draft_verification_row_gb300 import workloads as W


def test_traffic_record_valid_only_for_its_sources(tmp_path, monkeypatch):
    rec = {"dram_bytes_per_inner_node": 7.0e5, "kernel_source_sha256": bench.kernel_sha()}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.recorded_traffic() == (7.0e5, 7.0e5)
    rec["kernel_source_sha256"] = "0" * 64  # the sources changed since
    path.write_text(json.dumps(rec))
    assert bench.recorded_traffic() == (None, 7.0e5)
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.json"))
    assert bench.recorded_traffic() == (None, None)


def test_row_counts_of_a_trie():
    """Two requests, K=3 drafts: request 0 (L_b = 2) has drafts 0 and 1
    sharing their first token; request 1 has L_b = 0."""
    tokens = torch.tensor([[[5, 6], [5, 7], [9, 1]], [[0, 0], [0, 0], [0, 0]]], dtype=torch.int32)
    lengths = torch.tensor([2, 0], dtype=torch.int32)
    inner, leaves = bench.trie_nodes(tokens, lengths, 3)
    # request 0: root, (5), (9) inner; leaves (5,6), (5,7), (9,1).  request 1: the root is its leaf
    assert (inner, leaves) == (3, 4)
    assert bench.table_rows(lengths, 3) == (2 + 3 * 3) + 1
    assert bench.table_rows(lengths, 3, greedy=True) == (1 + 3 * 2) + 1

    class B:
        V, dtype = 10, "bf16"
    assert bench.row_bytes_of(B, inner, leaves) == (7 + 3) * 20
    assert bench.row_bytes_of(B, inner, leaves, greedy=True, ended_at_leaf=2) == (3 + 2) * 20


def test_first_drafts_keeps_the_first_k():
    batch = W.make("multidraft-B32-K4-L4-V32000-f32", "cpu", B=3, V=37)
    b1 = bench.first_drafts(batch, 1)
    assert b1.K == 1 and b1.target.shape == (3, 1, 5, batch.stride) and b1.target.is_contiguous()
    assert torch.equal(b1.tokens[:, 0], batch.tokens[:, 0]) and torch.equal(b1.sample_u[:, 0], batch.sample_u[:, 0])
    assert bench.first_drafts(batch, 4) is batch


def test_kernel_sha_covers_the_node_kernel_sources():
    names = {p.split("/")[-1] for p in bench.KERNEL_SRCS}
    assert names == {"sdv_stream.cu", "sdv_device.cuh", "sdv_internal.h"}
    assert bench.kernel_sha() == bench.kernel_sha() and len(bench.kernel_sha()) == 64


def test_peaks_fall_back_without_a_measurement(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (6800.0, "fallback")
    assert bench.measured_bf16_peak() == (1900.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6000.0, "bf16_tflops": 1800.0}))
    assert bench.measured_peaks() == (6000.0, "measured")
    assert bench.measured_bf16_peak() == (1800.0, "measured")


def test_rank_seeds():
    a = bench.rank_seed(W.HEADLINE, 0)
    assert a == W.WORKLOADS[W.HEADLINE]["seed"] and bench.rank_seed(W.HEADLINE, 1) != a
    assert bench.rank_seed(W.LM_HEAD_HEADLINE, 0) == W.LM_HEAD_WORKLOADS[W.LM_HEAD_HEADLINE]["seed"]


def test_sample_arrays_keep_the_layout():
    batch = W.make(W.HEADLINE, "cpu", B=5, K=2, L=2, V=67)
    a = bench.sample_arrays(batch, [1, 3])
    assert a["target"].dtype == np.int16 and a["target"].shape == (2, 2, 3, batch.stride)
    np.testing.assert_array_equal(a["target"], batch.target[[1, 3]].view(torch.int16).numpy())
    np.testing.assert_array_equal(a["lengths"], batch.lengths[[1, 3]].numpy())
    p, dt = bench.oracle_sample(batch, "multidraft", [1, 3], a)
    assert p == int(batch.lengths[[1, 3]].sum()) * batch.K and dt > 0
