"""Host logic of the benchmark's pipelined end-to-end leg (no GPU): how the
units are cut into chunks, each one bkv_round on its own unit range."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

MB = 1 << 20


@pytest.mark.parametrize("U,step_mb,max_chunks,want", [
    (112, 265, 4, 4),    # Qwen3-4B one layer: 157 MB in + 121 MB out
    (112, 265, 8, 8),
    (112, 265, 32, 16),  # at least 16 MB per chunk
    (2, 0.4, 4, 1),      # the tiny workload stays one round
    (3, 265, 8, 3),      # never more chunks than units
    (24, 57, 4, 3),
])
def test_chunk_count(U, step_mb, max_chunks, want):
    cuts = bench.e2e_chunk_cuts(U, int(step_mb * MB), max_chunks)
    assert len(cuts) - 1 == want


@pytest.mark.parametrize("U", [1, 2, 7, 24, 112, 113, 5120])
@pytest.mark.parametrize("max_chunks", [1, 3, 4, 8])
def test_chunks_partition_the_units(U, max_chunks):
    cuts = bench.e2e_chunk_cuts(U, 10 ** 12, max_chunks)
    assert cuts[0] == 0 and cuts[-1] == U
    sizes = [b - a for a, b in zip(cuts, cuts[1:])]
    assert all(s >= 1 for s in sizes)              # no empty round
    assert max(sizes) - min(sizes) <= 1            # near-equal chunks
