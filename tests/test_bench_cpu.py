"""Host logic of bench.py (no GPU): the algorithmic bytes it divides by for
every kind of call, the append workloads it builds, and the traffic record
it reports only for the current kernel sources."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from decode_attention_preallocated_gb300 import workloads as W  # noqa: E402


def test_bytes_count_the_filled_prefix_only():
    inp = W.dense_inputs(2, 1, 8, 2, 128, 1000, [300, 17], 1, False)
    assert bench.algorithmic_bytes(inp) == (300 + 17) * 2 * 128 * 2 * 2
    i8 = W.dense_inputs(2, 1, 8, 2, 128, 1000, [300, 17], 1, False, int8=True)
    assert bench.algorithmic_bytes(i8) == (300 + 17) * 2 * (128 * 2 + 8)


def test_paged_bytes_equal_the_flat_bytes():
    flat = W.dense_inputs(3, 2, 8, 2, 128, 640, [640, 5, 333], 2, True)
    paged = W.paged_inputs(3, 2, 8, 2, 128, 64, 10, [640, 5, 333], 2, True)
    assert bench.algorithmic_bytes(paged) == bench.algorithmic_bytes(flat)


def test_gather_bytes_count_listed_cells():
    inp = W.gather_inputs(1, 2, 8, 2, 128, 500, 40, 8, seed=3)
    inp.idx[0, 0, :5] = -1
    valid = 2 * 40 - 5
    assert bench.algorithmic_bytes(inp) == valid * 2 * 128 * 2 * 2


def test_append_inputs_and_bytes():
    base = W.workload("mtp_verify", seed=1)
    inp = bench.append_inputs("mtp_verify", 1, "cpu")
    n = base.q.shape[1]
    assert inp.k_new.shape == (1, n, 4, 256) and inp.v_new.shape == inp.k_new.shape
    assert inp.kv_lengths.tolist() == [L - n for L in base.kv_lengths.tolist()]
    assert inp.lengths_host == [L - n for L in base.lengths_host]
    # the prefix read including the new rows, plus the new rows read and written
    want = bench.kv_bytes(base.lengths_host, 4, 256, 2) + 2 * bench.kv_bytes([n], 4, 256, 2)
    assert bench.algorithmic_bytes(inp) == want
    assert bench.make_inputs("append_mtp_verify", 1, "cpu").k_new.shape == inp.k_new.shape


def test_traffic_record_follows_the_kernel_sources(tmp_path, monkeypatch):
    # a record taken on the current kernel sources is reported; one taken on
    # other sources is not
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = tmp_path / "decode_attention_preallocated_gb300"
    os.symlink(os.path.join(ROOT, "decode_attention_preallocated_gb300"), src)
    (prof / "traffic_ragged.txt").write_text(
        "kernel_sources: %s\ndram_bytes_per_launch: 123\n" % bench.kernel_source_hash())
    assert bench.recorded_traffic("ragged") == 123.0
    (prof / "traffic_ragged.txt").write_text(
        "kernel_sources: 0000000000000000\ndram_bytes_per_launch: 123\n")
    assert bench.recorded_traffic("ragged") is None


def test_oracle_timing_whole_call_and_scaled_sample():
    # whole call, and a one-sequence sample scaled by the batch's bytes
    inp = W.dense_inputs(3, 2, 8, 2, 128, 300, [300, 100, 200], 4, True)
    us, how = bench.oracle_us(inp, 1)
    assert us > 0 and how == "whole call"
    us1, how1 = bench.oracle_us(inp, 1, 0.0)
    assert us1 > 0 and how1 == "1 of 3 sequences, scaled by bytes"
    g = W.gather_inputs(1, 1, 8, 2, 128, 400, 64, 8, seed=2)
    assert bench.oracle_us(g, 2)[0] > 0


def test_baseline_config_tags_name_the_five_workloads():
    assert [n for _, n in bench.BASELINE_CONFIGS] == list(W.WORKLOADS)
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()


def test_int8_gather_bytes_count_codes_and_scales():
    inp = W.gather_inputs(1, 2, 8, 2, 128, 500, 40, 8, seed=3, int8=True)
    inp.idx[0, 1, :3] = -1
    assert bench.algorithmic_bytes(inp) == (2 * 40 - 3) * 2 * (128 * 2 + 8)


def test_masked_bytes_count_visible_chunks():
    inp = W.dense_inputs(2, 2, 8, 2, 128, 200, [200, 70], 5, False)
    inp.mask = torch.full((2, 2, 200), -float("inf"))
    inp.mask[0, 0, 3] = 0.0          # chunk 0 of sequence 0
    inp.mask[0, 1, 40] = 1.0         # chunk 1 of sequence 0
    inp.mask[0, 1, 41] = 1.0         # (same chunk)
    inp.mask[1, 0, 65] = 0.0         # chunk 2 of sequence 1 (length 70)
    inp.mask[1, 1, 100] = 0.0        # past the length: not counted
    assert bench.algorithmic_bytes(inp) == 3 * 32 * 2 * 128 * 2 * 2


def test_oracle_call_serves_every_named_kind():
    # dense, int8, gather, int8 gather and masked inputs all reach the oracle
    small = [W.dense_inputs(2, 2, 8, 2, 128, 100, [100, 40], 6, True),
             W.dense_inputs(1, 1, 8, 2, 128, 100, [77], 6, False, int8=True),
             W.gather_inputs(1, 1, 8, 2, 128, 300, 40, 8, seed=6),
             W.gather_inputs(1, 1, 8, 2, 128, 300, 40, 8, seed=6, int8=True)]
    m = W.dense_inputs(1, 1, 8, 2, 128, 100, [100], 6, False)
    m.mask = torch.zeros((1, 1, 100))
    m.mask[0, 0, 50:] = -float("inf")
    small.append(m)
    for inp in small:
        out = bench.oracle_call(inp, slice(0, 1))
        assert out.shape == (1,) + tuple(inp.q.shape[1:])
