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


def test_plan_keeps_whole_sequences_while_groups_do_not_outnumber_them():
    cu = [0, 50, 120, 121, 122]
    assert HostStep.plan(cu, 2, 2, 2) == [(k, a, b, None, None) for k, a, b in HostStep.partition(cu, 2, 2, 2)]


@pytest.mark.parametrize("groups", [5, 8, 9])
def test_plan_cuts_long_sequences_into_aligned_chunks(groups):
    lens = [2048, 0, 600, 1300]
    cu = np.concatenate([[0], np.cumsum(lens), [sum(lens) + 1, sum(lens) + 2]])  # + 2 decode tokens
    plan = HostStep.plan(cu, 4, 2, groups)
    assert plan[-1] == ("decode", 4, 6, None, None)
    pre = plan[:-1]
    # every new token of every prefill sequence in exactly one chunk, in order
    seen = []
    for kind, a, b, c0, c1 in pre:
        assert kind == "prefill" and b == a + 1 and c0 < c1
        assert c0 % 256 == 0 and (c1 % 256 == 0 or c1 == lens[a])
        seen += [(a, t) for t in range(c0, c1)]
    assert seen == [(s, t) for s in range(4) for t in range(lens[s])]
    per = -(-groups // 3)  # three sequences have new tokens
    for s in (0, 2, 3):
        assert len([1 for _, a, _, _, _ in pre if a == s]) <= per


def test_auto_groups_follow_the_prefix_cta_count():
    # one group per 152 prefix-attention CTAs, or per sequence of at least 76, at most sixteen
    assert HostStep.auto_groups(wl.make_config(2), wl.make_config(2).num_prefill) == 1  # 128 CTAs
    w4 = wl.make_config(4)
    assert HostStep.auto_groups(w4, w4.num_prefill) == 4  # 320 CTAs, four sequences of 80
    w3 = wl.make_config(3)
    assert HostStep.auto_groups(w3, w3.num_prefill) == 4
    assert HostStep.auto_groups(w3, 0) == 1
    w5 = wl.make_config(5)
    assert HostStep.auto_groups(w5, w5.num_prefill) == 13  # 2048 CTAs
    cu5 = np.asarray(w5.cu_seqlens_q)
    assert len(HostStep.plan(cu5, w5.num_prefill, 0, 13)) == 16  # four sequences in four chunks of 512
