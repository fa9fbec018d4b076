"""The benchmark's algorithmic work (the numerators of its roofline
fractions) against the oracle's closed forms, on the CPU.

bench.py counts prefill FLOPs as 4 * d * |visible pairs| * H and decode bytes
as K and V of the attended keys plus q, k, v, o.  Here the pair count comes
from the oracle's visible_pair_count (pinned to brute-force enumeration of
the mask) and the attended keys from its cache_len (the pages' C(T)), so a
slip in either of bench.py's formulas fails."""

import numpy as np
import pytest

import bench
import oracle
import workloads


def test_prefill_flops_match_visible_pairs():
    w = workloads.WORKLOADS["multipage_prefill_bf16"]
    pairs = oracle.visible_pair_count(w.m, w.n, w.m + w.T)
    assert bench.prefill_flops(w) == 4 * w.head_dim * pairs * w.heads * w.batch
    # 1.468 TFLOP per layer for the 32K-row, 40-page workload
    assert abs(bench.prefill_flops(w) / 1e12 - 1.468) < 5e-4


def test_single_page_decode_bytes_match_cache_len():
    w = workloads.WORKLOADS["single_page_bf16"]
    elt = 2
    # step t appends output t, then attends C(t + 1) = m + min(n, t + 1) keys
    keys = np.mean([oracle.cache_len(w.m, w.n, t + 1) for t in range(w.T)])
    per_head = w.head_dim * elt * (2 * keys + 4)     # K, V rows; q, k, v, o
    assert bench.single_page_bytes_per_decode(w) == pytest.approx(
        w.batch * w.heads * per_head, rel=1e-12)


def test_batched_decode_bytes_match_cache_len():
    w = workloads.WORKLOADS["batched_decode_bf16"]
    m_list = [256 + (29 * b) % 1793 for b in range(w.batch)]   # ragged, one per sequence
    t_b = 4096                                     # ring full
    elt = 2
    keys = sum(oracle.cache_len(m, w.n, t_b + 1) for m in m_list)
    want = w.heads * w.head_dim * elt * (2 * keys + 4 * len(m_list))
    assert bench.batched_step_bytes(m_list, w) == want


def test_job_throughput_is_whole_job():
    # tokens of all ranks over the slowest rank's time
    assert bench.job_throughput(6000, 4, 20.0) == pytest.approx(4 * 6000 / 0.020)
