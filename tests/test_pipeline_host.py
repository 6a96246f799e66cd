"""Host-side logic of the schedules (combine_ep_route_topk_gb300.pipeline):
rank splits, round rank offsets and the micro-batch group checks.  CPU only:
nothing here launches a kernel."""
import pytest
import torch

from combine_ep_route_topk_gb300 import pipeline as pl


def test_split_by_ranks_even_and_uneven_counts():
    offs = [0, 3, 3, 10, 12, 20]  # R = 5
    assert pl.split_by_ranks(offs, 2) == [(0, 2), (2, 5)]
    assert pl.split_by_ranks(offs, 5) == [(i, i + 1) for i in range(5)]
    assert pl.split_by_ranks(offs, 8) == [(0, 1), (1, 2), (2, 3), (3, 4), (4, 5)]


def test_round_rank_offsets_clip_each_rank_to_the_round():
    offs = [0, 5, 5, 12, 20]
    assert pl.round_rank_offsets(offs, 0, 8) == [0, 5, 5, 8, 8]
    assert pl.round_rank_offsets(offs, 8, 16) == [0, 0, 0, 4, 8]
    assert pl.round_rank_offsets(offs, 16, 20) == [0, 0, 0, 0, 4]
    # every token of every round belongs to exactly one rank
    T = 8
    for t0 in range(0, 20, T):
        r = pl.round_rank_offsets(offs, t0, min(20, t0 + T))
        assert r[0] == 0 and r[-1] == min(20, t0 + T) - t0
        assert all(a <= b for a, b in zip(r, r[1:]))


@pytest.mark.parametrize("groups", [
    [(0, 2), (3, 4)],          # gap
    [(0, 2), (1, 4)],          # overlap
    [(1, 4)],                  # does not start at 0
    [(0, 3)],                  # does not end at R
    [(0, 0), (0, 4)],          # empty group
    [],
])
def test_micro_batch_groups_must_tile_the_ranks(groups):
    ro = torch.tensor([0, 2, 4, 6, 8], dtype=torch.int32)
    with pytest.raises(ValueError):
        pl.make_micro_batches(torch.zeros(8, 4), torch.zeros(8, 8, dtype=torch.bfloat16), ro, 2,
                              0, torch.zeros(8, 8, dtype=torch.bfloat16), rank_groups=groups)
