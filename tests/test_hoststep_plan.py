"""Host-side plan of the host-buffer step (no GPU): how sequences are cut
into stream groups, and how many groups are chosen."""
import numpy as np
import pytest

import workloads as wl
from paged_prefix_reuse_gb300.step import HostStep


@pytest.mark.parametrize("groups", [1, 2, 3, 4, 7])
def test_partition_covers_the_prefill_sequences_in_order(groups):
    rng = np.random.default_rng(groups)
    lens = rng.integers(0, 300, size=13)
    lens[[2, 3]] = 0  # sequences without new tokens
    cu = np.concatenate([[0], np.cumsum(lens), np.cumsum(lens)[-1] + np.arange(1, 6)])  # + 5 decode tokens
    parts = HostStep.partition(cu, 13, 5, groups)
    pre = [p for p in parts if p[0] == "prefill"]
    assert parts[-1] == ("decode", 13, 18)
    assert len(pre) <= groups
    # contiguous, in order, every prefill token in exactly one group, no empty group
    assert pre[0][1] == 0 and pre[-1][2] == 13
    for (_, a0, b0), (_, a1, b1) in zip(pre, pre[1:]):
        assert b0 == a1
    assert all(cu[b] > cu[a] for _, a, b in pre)
    # balance: no group exceeds its share by more than one sequence's tokens
    share = cu[13] / len(pre)
    assert all(cu[b] - cu[a] <= share + lens.max() for _, a, b in pre)


def test_partition_without_prefill_or_decode():
    assert HostStep.partition([0, 1, 2, 3], 0, 3, 4) == [("decode", 0, 3)]
    assert HostStep.partition([0, 5, 9], 2, 0, 1) == [("prefill", 0, 2)]
    assert HostStep.partition([0, 0, 0], 2, 0, 2) == []


def test_auto_groups_follow_the_prefix_cta_count():
    # one group per 152 prefix-attention CTAs, at most four
    assert HostStep.auto_groups(wl.make_config(2), wl.make_config(2).num_prefill) == 1  # 128 CTAs
    w4 = wl.make_config(4)
    assert HostStep.auto_groups(w4, w4.num_prefill) == 2  # 320 CTAs
    w3 = wl.make_config(3)
    assert HostStep.auto_groups(w3, w3.num_prefill) == 4
    assert HostStep.auto_groups(w3, 0) == 1
