"""Data-parallel gradient averaging on a linear model, in fp64 (oracle; test infrastructure).

Source: "Data parallelism", "Why averaging gradients is exactly large-batch
training": with the loss a mean over the batch, the gradient of the whole batch
is the average of the shards' mean gradients when every shard has the same
number of examples; with unequal (token) counts, summing the per-token losses
on each rank, summing the counts across ranks and dividing once recovers the
global mean, while averaging the ranks' means does not.

Model: prediction x . w, loss per example 0.5 (x . w - y)^2, so the gradient of
one example is (x . w - y) x.
"""
from __future__ import annotations

import numpy as np


def example_grads(X: np.ndarray, y: np.ndarray, w: np.ndarray) -> np.ndarray:
    """One gradient row per example, fp64."""
    resid = X @ w - y
    return resid[:, None] * X


def batch_mean_grad(X, y, w) -> np.ndarray:
    """Gradient of the mean loss over all examples (the large-batch gradient)."""
    return example_grads(X, y, w).mean(axis=0)


def shard_mean_grads(shards, w) -> list[np.ndarray]:
    """Each rank's gradient of its own mean loss."""
    return [example_grads(X, y, w).mean(axis=0) for X, y in shards]


def shard_sum_grads(shards, w) -> list[np.ndarray]:
    """Each rank's gradient of its summed (not averaged) loss."""
    return [example_grads(X, y, w).sum(axis=0) for X, y in shards]


def mean_of_means(shards, w) -> np.ndarray:
    g = shard_mean_grads(shards, w)
    return sum(g) / len(g)


def sum_then_divide_once(shards, w) -> np.ndarray:
    total_count = sum(X.shape[0] for X, _ in shards)
    return sum(shard_sum_grads(shards, w)) / total_count
