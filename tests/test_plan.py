"""Properties of the split-KV planner (host twin of the device planner; CPU only)."""
import numpy as np
import pytest

from mla_latent_kv_17_gb300 import build as mbuild
from mla_latent_kv_17_gb300 import inputs, ops
from planview import parse

OVH = {"bf16": 2, "fp8": 3}  # per-piece overhead in tiles, as the planner charges it per cache layout
MIN = 2  # shortest piece the planner makes
TILE = 128  # tokens per planner tile


@pytest.fixture(scope="module", autouse=True)
def _built():
    mbuild.build()


def check_plan(seq_lens, H=128, topk=0, num_sms=148, kv="bf16"):
    B = len(seq_lens)
    ovh = OVH[kv]
    p = parse(ops.plan_host(seq_lens if topk == 0 else None, B, H, topk, num_sms, kv_dtype=kv), B, H)
    lens = [topk if topk else max(0, int(x)) for x in seq_lens]
    units = p["units"]
    assert units == max(1, num_sms // 2)
    ub = p["unit_begin"]
    assert ub[0] == 0 and ub[-1] == p["n_items"] and np.all(np.diff(ub) >= 0)
    assert p["n_items"] <= p["max_items"] == B + units
    items = p["items"]
    # coverage: each request's pieces tile [0, len) exactly once, in order, on tile bounds
    per_req = {b: [] for b in range(B)}
    for b, t0, t1, slot in items:
        per_req[int(b)].append((int(t0), int(t1), int(slot)))
    slots = []
    for b in range(B):
        pcs = per_req[b]
        assert len(pcs) == p["num_splits"][b] >= 1
        if lens[b] == 0:
            assert pcs == [(0, 0, -1)]
            continue
        pos = 0
        for t0, t1, _ in pcs:
            assert t0 == pos and t1 > t0 and t0 % TILE == 0
            pos = t1
        assert pos == lens[b]
        if len(pcs) == 1:
            assert pcs[0][2] == -1 and p["split_base"][b] == -1
        else:
            s = [x[2] for x in pcs]
            assert s == list(range(p["split_base"][b], p["split_base"][b] + len(pcs)))
            slots += s
    assert sorted(slots) == list(range(len(slots))) and len(slots) == p["n_partials"]
    assert p["n_partials"] <= p["max_partials"]
    # items are grouped by unit in order, and each unit's load stays near the budget: at most
    # one folded short run (< MIN tiles) and one extra piece overhead beyond it
    assert np.all(np.diff(p["item_unit"]) >= 0)
    for u in range(units):
        assert np.all(p["item_unit"][ub[u]:ub[u + 1]] == u)
    cost = np.zeros(units, dtype=np.int64)
    for u in range(units):
        for i in range(ub[u], ub[u + 1]):
            b, t0, t1, _ = items[i]
            if t1 > t0:
                cost[u] += (t1 - t0 + TILE - 1) // TILE + ovh
    assert np.all(cost <= p["per"] + MIN + 2 * ovh), (cost.max(), p["per"])
    # pieces are never shorter than MIN tiles unless the whole request is
    for b in range(B):
        pcs = per_req[b]
        if len(pcs) > 1:
            assert all((t1 - t0 + TILE - 1) // TILE >= MIN for t0, t1, _ in pcs)
    return p, cost


@pytest.mark.parametrize("name", list(inputs.WORKLOADS))
def test_workload_plans(name):
    sl = inputs.workload_seq_lens(name).tolist()
    topk = 2048 if "sparse" in name else 0
    p, cost = check_plan(sl, topk=topk)
    tiles = sum(((topk or L) + TILE - 1) // TILE for L in sl)
    ub, items = p["unit_begin"], p["items"]
    load = [sum((t1 - t0 + TILE - 1) // TILE for _, t0, t1, _ in items[ub[u]:ub[u + 1]])
            for u in range(p["units"])]
    # the busiest unit carries at most its share plus two folded short runs
    assert max(load) <= p["per"] + 2 * (MIN - 1), (max(load), p["per"])
    assert sum(load) == tiles


@pytest.mark.parametrize("name", ["dsv3_dense_b64_h128_l1k_8k", "fp8_ragged_b128_h128_lognormal", "long_dense_b4_h128_l128k"])
def test_fp8_plans_charge_more_per_piece(name):
    # the same invariants with the FP8 records' piece overhead; the budget grows with it
    sl = inputs.workload_seq_lens(name).tolist()
    p2, _ = check_plan(sl)
    p3, _ = check_plan(sl, kv="fp8")
    assert p3["per"] >= p2["per"]
    assert p3["n_items"] <= p2["n_items"]


def test_edge_lengths():
    check_plan([1, 63, 64, 65, 0, 128, 129])
    check_plan([0])
    check_plan([0, 0, 0])
    check_plan([1])
    check_plan([131072] * 4)
    check_plan([5] * 300)                   # more requests than units
    check_plan(list(range(0, 5000, 37)))


@pytest.mark.parametrize("num_sms", [2, 3, 8, 148, 152])
def test_sm_counts(num_sms):
    rng = np.random.default_rng(num_sms)
    check_plan(rng.integers(0, 9000, size=37).tolist(), num_sms=num_sms)


def test_sparse_plan_uses_topk():
    p, _ = check_plan([10, 100000, 3], topk=2048)
    assert p["topk"] == 2048


def test_long_requests_are_split_and_short_batches_are_not():
    p, _ = check_plan([131072] * 4)
    assert all(n > 1 for n in p["num_splits"])
    p, _ = check_plan([256])
    assert p["num_splits"][0] == 1 and p["n_partials"] == 0


def test_plan_is_deterministic():
    sl = inputs.workload_seq_lens("dsv3_dense_b64_h128_l1k_8k").tolist()
    a = ops.plan_host(sl, 64, 128, 0, 148)
    b = ops.plan_host(sl, 64, 128, 0, 148)
    assert np.array_equal(a, b)


def test_random_plans_hold_every_invariant():
    # mixtures of empty, single-token, page-edge, ordinary and very long requests, over
    # request counts from 1 to 700 and several SM counts: coverage, slots, unit order and
    # per-unit load bound all hold (check_plan)
    r = np.random.default_rng(2024)
    for trial in range(150):
        B = int(r.choice([1, 2, 3, 7, 64, 128, 300, 700]))
        kind = r.integers(0, 5, size=B)
        lens = np.where(kind == 0, 0,
               np.where(kind == 1, 1,
               np.where(kind == 2, 64 * r.integers(1, 40, size=B),
               np.where(kind == 3, r.integers(2, 9000, size=B), r.integers(30000, 140000, size=B)))))
        num_sms = int(r.choice([2, 20, 132, 148, 152]))
        check_plan(lens.astype(np.int32), H=int(r.choice([16, 64, 128])), num_sms=num_sms)


def test_uniform_topk_batches_fit_one_unit_per_request():
    # top-k lists cost the same for every request: with no more requests than units each
    # request gets a unit of its own (no partials, no merge); with many more, they are split
    p, _ = check_plan([65536] * 64, topk=2048)
    assert p["n_partials"] == 0 and all(n == 1 for n in p["num_splits"])
    assert p["per"] == 2048 // TILE + OVH["bf16"]
    p, _ = check_plan([65536] * 4, topk=2048)
    assert p["n_partials"] > 0
