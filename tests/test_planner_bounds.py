"""The partitioner's list schedule against the optimum on tiny instances.

CoDec, "workload balancing", assigns the sub-tasks of a plan to the m
thread-block slots with a list schedule and cites Graham's bound: any list
schedule ends within (2 - 1/m) of the optimal makespan. Taking the tasks
largest first (as the planner does) tightens that to 4/3 - 1/(3m) (Graham,
1969). Here the optimum comes from brute force over all m^n assignments
(n <= 8 tasks, m <= 4 slots), not from any schedule."""
import itertools

import numpy as np
import pytest


def brute_force_opt(costs, m):
    """Smallest makespan over every assignment of the tasks to m slots."""
    n = len(costs)
    if n == 0:
        return 0.0
    A = np.array(list(itertools.product(range(m), repeat=n)), dtype=np.int64)   # [m^n, n]
    loads = np.stack([(np.where(A == s, costs[None, :], 0.0)).sum(axis=1) for s in range(m)], axis=1)
    return float(loads.max(axis=1).min())


def _instances():
    rng = np.random.default_rng(20260601)
    out = []
    for n in range(1, 9):
        for m in range(1, 5):
            out.append((rng.uniform(0.1, 10.0, size=n), m))            # real costs
            out.append((rng.integers(1, 6, size=n).astype(float), m))   # many ties
    return out


@pytest.mark.parametrize("case", range(64))
def test_list_schedule_within_graham_bounds(lib, case):
    costs, m = _instances()[case]
    slot, mk = lib.list_schedule(costs, m)
    # a valid assignment whose largest load is the reported makespan
    assert slot.shape == costs.shape and np.all((slot >= 0) & (slot < m))
    loads = np.bincount(slot, weights=costs, minlength=m)
    assert abs(loads.max() - mk) <= 1e-9 * max(1.0, mk)
    opt = brute_force_opt(costs, m)
    assert mk <= (2.0 - 1.0 / m) * opt * (1 + 1e-12)          # any list schedule
    assert mk <= (4.0 / 3.0 - 1.0 / (3.0 * m)) * opt * (1 + 1e-12)   # largest first


@pytest.mark.parametrize("case", range(0, 64, 5))
def test_list_schedule_is_largest_first_greedy(lib, case):
    """Replaying the tasks largest first (lower index first among equal
    costs), each one went to a least-loaded slot, the lowest index among
    equally loaded ones."""
    costs, m = _instances()[case]
    slot, _ = lib.list_schedule(costs, m)
    order = sorted(range(len(costs)), key=lambda i: (-costs[i], i))
    load = np.zeros(m)
    for i in order:
        best = int(np.argmin(load))     # first index of the minimum
        assert slot[i] == best
        load[best] += costs[i]


@pytest.mark.parametrize("m", [2, 3, 4])
def test_list_schedule_tight_example(lib, m):
    """Graham's instance on which largest-first meets its bound: two tasks
    each of 2m-1 .. m+1 and three of m. Largest first ends at 4m - 1, the
    optimum is 3m."""
    costs = [float(c) for c in range(2 * m - 1, m, -1) for _ in range(2)] + [float(m)] * 3
    costs = np.array(costs)
    if len(costs) <= 8:
        assert brute_force_opt(costs, m) == 3 * m
    _, mk = lib.list_schedule(costs, m)
    assert mk == 4 * m - 1
    assert mk / (3 * m) == pytest.approx(4.0 / 3.0 - 1.0 / (3.0 * m))


def test_list_schedule_rejects_bad_input(lib):
    with pytest.raises(lib.PstError):
        lib.list_schedule([1.0, -1.0], 2)
    with pytest.raises(lib.PstError):
        lib.list_schedule([1.0], 0)
    slot, mk = lib.list_schedule([], 3)
    assert slot.size == 0 and mk == 0.0


@pytest.mark.parametrize("n_tok,chunk,sms", [(8192, 1024, 20), (8192, 1536, 20), (8192, 1536, 7),
                                             (9000, 4096, 3), (20000, 2560, 152)])
def test_predicted_makespan_is_the_list_schedule_of_one_launch(lib, n_tok, chunk, sms):
    """A plan whose items all belong to one tensor-core launch is dispatched
    largest first onto the SMs, one block each: its predicted makespan is the
    list schedule (above) of its items' C_est. One node of n_tok tokens seen
    by 64 queries x 4 q-heads per kv head (256 rows: tensor cores, P rounded
    once), 8 kv heads, uniform chunks; the chunk lengths come from the plan,
    the costs from the cost model's own estimate."""
    n_pages = (n_tok + 15) // 16
    t = lib.tree_build([n_tok], [-1], [0, n_pages], list(range(n_pages)), None, 16, n_pages)
    p = lib.plan_create(t, [0] * 64, 32, 8, 128, "bf16", split_policy="uniform", fixed_chunk=chunk, num_sms=sms)
    st, ex = p.stats(), p.export()
    assert st["n_cc_items"] == 0
    lens = np.diff(ex["chunk_tok_ptr"])
    costs = [lib.cost_estimate(1, 256, int(n)) for n in lens for _ in range(8)]
    assert st["n_tc_items"] == len(costs)
    _, mk = lib.list_schedule(costs, sms)
    assert st["predicted_makespan_us"] == pytest.approx(mk, rel=1e-12)
