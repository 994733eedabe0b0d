"""Pins for oracle.split: partition-size invariance against the unsplit oracle and
torch's log-sum-exp; empty partitions carry no weight."""

import numpy as np
import pytest
import torch

from oracle import attention, split


@pytest.mark.parametrize("ctx,part", [(1, 16), (37, 16), (512, 64), (1000, 512), (1000, 4096), (300, 7)])
def test_partition_invariance(ctx, part):
    rng = np.random.default_rng(ctx + part)
    q = rng.normal(size=(8, 32))
    K = rng.normal(size=(ctx, 2, 32))
    V = rng.normal(size=(ctx, 2, 32))
    whole = attention.decode_attention_contiguous(q, K, V, 0.2)
    np.testing.assert_allclose(split.decode_attention_split(q, K, V, 0.2, part), whole, rtol=0, atol=1e-13)


def test_partials_give_the_global_log_sum_exp():
    rng = np.random.default_rng(9)
    q = rng.normal(size=(1, 16))
    K = rng.normal(size=(100, 1, 16))
    V = rng.normal(size=(100, 1, 16))
    m, l, _ = split.partition_partials(q, K, V, 0.5, 30)
    assert m.shape == (4, 1)
    scores = torch.from_numpy(K[:, 0, :] @ q[0] * 0.5)
    lse = torch.logsumexp(scores, dim=0).item()
    assert abs(np.log(np.sum(l[:, 0] * np.exp(m[:, 0]))) - lse) < 1e-12


def test_empty_partitions_are_ignored():
    m = np.array([[1.0], [-np.inf]])
    l = np.array([[2.0], [0.0]])
    o = np.array([[[3.0, 4.0]], [[0.0, 0.0]]])
    assert np.array_equal(split.merge_partials(m, l, o), np.array([[3.0, 4.0]]))
    assert np.array_equal(split.merge_partials(np.full((2, 1), -np.inf), np.zeros((2, 1)), np.zeros((2, 1, 2))),
                          np.zeros((1, 2)))
