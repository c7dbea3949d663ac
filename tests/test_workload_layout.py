"""Host checks of the seeded workload layouts (no GPU): modality tags and
image numbers (the per-image keep pools) agree with each layout's stated
structure, and inputs are pure functions of their seeds."""
import torch

from oracle import sprint_oracle as orc
from workload import WORKLOADS, image_layout, prefix_inputs, prefix_layout


def sizes(ids):
    return torch.bincount(ids.long()).tolist()


def test_image_numbers_follow_the_layouts():
    w = WORKLOADS["prefix-32k"]
    ids = image_layout(w)
    assert sizes(ids) == [16 * 1024] + [1024] * 16      # 16 text spans, 16 images
    w = WORKLOADS["prefix-4k"]
    assert sizes(image_layout(w)) == [1024, 1024, 1024, 1024]  # three adjacent images
    w = WORKLOADS["sequential-64-blocks"]
    for b in (0, 63):
        assert sizes(image_layout(w, block=b)) == [1024 + 32 * b, 1024]
    w = WORKLOADS["batch-16x8k"]
    for s in range(16):
        ids, tags = image_layout(w, s), prefix_layout(w, s)
        assert torch.equal(ids > 0, tags > 0)
        assert all(n == 256 for n in sizes(ids)[1:])    # every image a 256-token slot
        # numbered in position order
        first = [int((ids == j).nonzero()[0]) for j in range(1, int(ids.max()) + 1)]
        assert first == sorted(first)


def test_image_runs_match_the_oracle_where_images_are_separate():
    # prefix-32k's images are separated by text, so maximal image runs (the
    # oracle's helper) and the layout's image numbers coincide
    w = WORKLOADS["prefix-32k"]
    assert image_layout(w).long().tolist() == list(orc.image_pool_ids(prefix_layout(w)))


def test_inputs_are_seeded():
    w = WORKLOADS["tiny-256"]
    a, b = prefix_inputs(w), prefix_inputs(w)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    c = prefix_inputs(w, seq=1)
    assert not torch.equal(a["K"], c["K"])
