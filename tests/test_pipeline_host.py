"""Host logic of attention_step_host (no GPU): how the B*H heads are cut
into chunks, and the checks on an explicit list of chunk sizes."""
import pytest
import torch

import exact_attention_97_gb300 as fa
from exact_attention_97_gb300.pipeline import chunk_bounds


@pytest.mark.parametrize("n", [1, 2, 5, 7, 16, 100, 256, 1000])
@pytest.mark.parametrize("chunks", [1, 2, 3, 6, 16, 40])
@pytest.mark.parametrize("ramp", [False, True])
def test_chunk_bounds_cover_every_head_once(n, chunks, ramp):
    b = chunk_bounds(n, chunks, ramp)
    assert b[0] == 0 and b[-1] == n
    assert len(b) - 1 == min(chunks, n)
    assert all(b[i + 1] > b[i] for i in range(len(b) - 1))  # no empty chunk


def test_ramped_chunks_are_smaller_at_both_ends():
    b = chunk_bounds(256, 16, True)
    sizes = [b[i + 1] - b[i] for i in range(16)]
    assert sizes[0] < sizes[1] < sizes[2] and sizes[-1] < sizes[-2] < sizes[-3]


@pytest.mark.parametrize("sizes", [[3, 3, 3], [5, 5, 1], [0, 10], [10, -1, 1], []])
def test_explicit_chunk_sizes_must_cover_the_heads(sizes):
    q = torch.zeros(2, 5, 16, 64, dtype=torch.bfloat16)  # 10 heads
    with pytest.raises(ValueError):
        fa.attention_step_host(q, q, q, q, chunks=sizes)
