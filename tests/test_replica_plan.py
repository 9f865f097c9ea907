"""The redundant-expert plan (moe_plan_replicas, a host function of the C ABI;
no GPU): popular experts get extra copies (ai.flicky.cc 3.5), each extra copy
going to the expert with the highest load per copy."""
import itertools

import numpy as np
import pytest
import torch

from mixture_experts_layer_87_b300 import build, capi


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return capi.lib()


def _plan(counts, n_extra):
    first, copies, slot_expert = capi.moe_plan_replicas(torch.tensor(counts, dtype=torch.int32), n_extra)
    return first.numpy(), copies.numpy(), slot_expert.numpy()


def test_plan_tables_are_consistent():
    rng = np.random.default_rng(3)
    for _ in range(20):
        E = int(rng.integers(1, 40))
        counts = rng.integers(0, 500, E)
        n_extra = int(rng.integers(0, 50))
        first, copies, slot_expert = _plan(counts, n_extra)
        assert (copies >= 1).all() and copies.sum() == E + n_extra
        assert first[0] == 0 and (np.diff(first) == copies[:-1]).all()
        for e in range(E):
            assert (slot_expert[first[e]:first[e] + copies[e]] == e).all()


def test_no_extra_copies_is_the_identity():
    first, copies, slot_expert = _plan([5, 0, 9, 3], 0)
    np.testing.assert_array_equal(first, [0, 1, 2, 3])
    np.testing.assert_array_equal(copies, 1)
    np.testing.assert_array_equal(slot_expert, [0, 1, 2, 3])


def test_plan_minimises_the_heaviest_copy_load():
    """Against every way of handing out the extra copies (brute force on small
    cases): the plan's largest load per copy, max counts[e] / copies[e], is the
    smallest possible."""
    rng = np.random.default_rng(4)
    for _ in range(30):
        E = int(rng.integers(1, 5))
        counts = rng.integers(0, 60, E)
        n_extra = int(rng.integers(0, 5))
        _, copies, _ = _plan(counts, n_extra)
        got = max(c / n for c, n in zip(counts, copies))
        best = min(max(c / (1 + x) for c, x in zip(counts, extra))
                   for extra in itertools.product(range(n_extra + 1), repeat=E) if sum(extra) == n_extra)
        assert got == pytest.approx(best, rel=0, abs=1e-12)


def test_heaviest_expert_gets_the_first_copy_and_ties_go_low():
    _, copies, _ = _plan([10, 40, 40, 5], 1)
    np.testing.assert_array_equal(copies, [1, 2, 1, 1])
    _, copies, _ = _plan([10, 40, 40, 5], 3)     # 40/2, 40/2, 10, 5 -> next goes to expert 1 (20 vs 20: lower)
    np.testing.assert_array_equal(copies, [1, 3, 2, 1])


def test_plan_rejects_bad_arguments():
    with pytest.raises(capi.MoEError):
        capi.moe_plan_replicas(torch.tensor([1, -2, 3], dtype=torch.int32), 1)
    with pytest.raises(capi.MoEError):
        capi.moe_plan_replicas(torch.tensor([1, 2], dtype=torch.int32), -1)
