"""Host-side helpers for running the head data-parallel over whole pairs.

Per-sequence means never cross pairs, so a batch of P pairs splits into
contiguous blocks of pairs, one per rank.  Each rank runs the three entry
points on its own rows with n_pairs = P_rank.  orpo_loss then returns the mean
over its P_rank pairs, and its cotangent carries 1/P_rank.  To make the sum
over ranks equal the single-device result, scale each rank's loss and
cotangent g by P_rank / P before the backward.  After that, all-reducing dW
(and the five metric sums) across ranks gives the global values; dh rows stay
on the rank that owns them.
"""

from __future__ import annotations

import numpy as np


def pair_range(n_pairs: int, rank: int, world: int):
    """[p0, p1): the contiguous block of pairs owned by `rank`."""
    if not (0 <= rank < world) or n_pairs < world:
        raise ValueError("need 0 <= rank < world <= n_pairs")
    return rank * n_pairs // world, (rank + 1) * n_pairs // world


def shard_pairs(seq_id, n_pairs: int, rank: int, world: int):
    """Rows, renumbered sequence ids and pair count of the rank's shard.

    Padding rows (seq_id = -1) are not carried.  Returns (rows, local_seq_id,
    local_pairs, scale) where scale = local_pairs / n_pairs multiplies the
    rank's loss and cotangent.
    """
    seq_id = np.asarray(seq_id)
    p0, p1 = pair_range(n_pairs, rank, world)
    rows = np.where((seq_id >= 2 * p0) & (seq_id < 2 * p1))[0]
    local = (seq_id[rows] - 2 * p0).astype(np.int32)
    return rows, local, p1 - p0, (p1 - p0) / n_pairs
