"""The bytes the bench divides by: the logit rows each rule must read, for
every workload, against counts written out from the workloads' shapes."""

import functools

import numpy as np
import pytest

from speculative_decoding_verify_sample_gb300 import synth


@functools.lru_cache(maxsize=None)
def inputs(name):
    return synth.make_inputs(name)


def test_llama3_reads_every_target_and_draft_row():
    inp = inputs("llama3")
    assert synth.rows_needed(inp) == (32 * 5, 32 * 4)


def test_greedy_reads_no_draft_row():
    inp = inputs("greedy")
    assert synth.rows_needed(inp) == (256 * 5, 0)


def test_dsv3_reads_draft_rows_of_sampled_requests_only():
    inp = inputs("dsv3_mtp")
    sampled = int(np.sum(np.asarray(inp["temperature"]) > 0))
    assert synth.rows_needed(inp) == (512 * 2, sampled)
    assert 0.7 * 512 < sampled < 0.8 * 512


def test_ragged_reads_rows_up_to_each_draft_length():
    inp = inputs("ragged")
    n = np.asarray(inp["draft_len"])
    assert synth.rows_needed(inp) == (int(np.sum(n + 1)), int(np.sum(n)))


def test_onehot_reads_no_draft_logits():
    """The one-hot rule takes q(x) = 1: no draft rows, whatever the temperature."""
    inp = synth.onehot_case(5, 128, 4, 128256, "bf16", temperature=0.7, greedy_frac=0.25)
    assert inp.get("draft") is None
    assert synth.rows_needed(inp) == (128 * 5, 0)


@pytest.mark.parametrize("name", ["llama3", "greedy", "dsv3_mtp", "ragged"])
def test_required_bytes_match_the_row_counts(name):
    import bench
    inp = inputs(name)
    rt, rd = synth.rows_needed(inp)
    elt = 2 if inp["dtype"] == "bf16" else 4
    assert bench.required_bytes(inp) == (rt + rd) * inp["V"] * elt
