"""Pins of the oracle's routing layout (counts, mask, slots) to what the pages fix.

* The lesson-14 exercise's routing table (tests/golden/lesson14_routing_table.json).
* Conservation: the expert queues hold N*K entries minus the masked ones
  (lesson 14, "practice task" assertion; DeepEP V1 guide 6.3 on -1 slots).
* Per-rank deduplication: a token reaches a rank once even if several of its
  experts live there ("DeepEP Ascend deep dive", "Two Transfers").
* Slots: an independent formulation (a stable sort of (expert, token, k)
  triples) and brute force over every routing of tiny problems.
"""
import itertools
import json
import os

import numpy as np
import pytest

import epinputs as ei
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _sorted_slots(idx, E, R):
    """Slots by a stable sort: an independent formulation of the definition."""
    N, K = idx.shape
    L = E // R
    flat = idx.reshape(-1).astype(np.int64)
    valid = (flat >= 0) & (flat < E)
    pos = np.nonzero(valid)[0]                       # (t, k) in lexicographic order
    order = np.argsort(flat[pos], kind="stable")     # by expert, ties keep (t, k) order
    expert_slot = np.full(N * K, -1, np.int64)
    expert_slot[pos[order]] = np.arange(len(pos))
    # ranks: dedup (t, r) pairs, then stable sort by rank
    t_of = pos // K
    r_of = flat[pos] // L
    pairs = np.unique(np.stack([r_of, t_of], 1), axis=0)   # sorted by (r, t)
    rank_slot = np.full((N, R), -1, np.int64)
    rank_slot[pairs[:, 1], pairs[:, 0]] = np.arange(len(pairs))
    return expert_slot.reshape(N, K), rank_slot


def test_lesson14_table():
    g = json.load(open(os.path.join(GOLDEN, "lesson14_routing_table.json")))
    idx = np.array(g["topk_idx"], np.int32)
    o = oracle.layout(idx, g["E"], g["R"])
    assert o["status"] == 0
    assert int(o["num_tokens_per_expert"].sum()) == g["conserved_total"]
    for key in ["num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank",
                "expert_offset", "rank_offset", "expert_slot", "rank_slot"]:
        assert o[key].tolist() == g[key], key


@pytest.mark.parametrize("c", [1, 2, 3, 4, 5])
def test_invariants_on_configs(c):
    cfg = ei.WORKLOADS[c]
    idx, _ = ei.make_routing(cfg, 0)
    E, R, N, K = cfg.E, cfg.R, cfg.N, cfg.K
    L = E // R
    o = oracle.layout(idx, E, R)
    assert o["status"] == 0
    pe, pr = o["num_tokens_per_expert"], o["num_tokens_per_rank"]
    mask = o["is_token_in_rank"].astype(bool)
    n_masked = int((idx == -1).sum())
    # conservation
    assert int(pe.sum()) == N * K - n_masked
    assert np.array_equal(pe, np.bincount(idx[idx >= 0], minlength=E))
    # per-rank dedup: mask[t, r] iff some expert of t is on r; count once
    ref_mask = np.zeros((N, R), bool)
    for k in range(K):
        v = idx[:, k] >= 0
        ref_mask[np.nonzero(v)[0], idx[v, k] // L] = True
    assert np.array_equal(mask, ref_mask)
    assert np.array_equal(pr, mask.sum(0))
    assert np.all(pr <= pe.reshape(R, L).sum(1))
    assert np.all(pr <= N)
    # offsets are exclusive prefix sums
    assert np.array_equal(o["expert_offset"], np.concatenate([[0], np.cumsum(pe)]))
    assert np.array_equal(o["rank_offset"], np.concatenate([[0], np.cumsum(pr)]))
    # slots: bijections onto [0, D_e) and [0, D_r)
    es = o["expert_slot"]
    assert np.array_equal(np.sort(es[es >= 0]), np.arange(pe.sum()))
    assert np.all((es >= 0) == (idx >= 0))
    rs = o["rank_slot"]
    assert np.array_equal(np.sort(rs[rs >= 0]), np.arange(pr.sum()))
    assert np.array_equal(rs >= 0, mask)
    # slots equal the stable-sort formulation
    es2, rs2 = _sorted_slots(idx, E, R)
    assert np.array_equal(es, es2)
    assert np.array_equal(rs, rs2)
    # each slot lies inside its expert's / rank's range, in token order
    e_of = np.where(idx >= 0, idx, 0)
    assert np.all((es < 0) | ((es >= o["expert_offset"][e_of]) & (es < o["expert_offset"][e_of + 1])))


def _brute(idx, E, R):
    """The definition, counted literally: slot = offset + #earlier entries with the same key."""
    N, K = idx.shape
    L = E // R
    entries = [(t, k, int(idx[t, k])) for t in range(N) for k in range(K)]
    valid = [(t, k, e) for (t, k, e) in entries if 0 <= e < E]
    per_expert = [sum(1 for (_, _, e) in valid if e == x) for x in range(E)]
    in_rank = [[any(0 <= int(idx[t, k]) < E and int(idx[t, k]) // L == r for k in range(K))
                for r in range(R)] for t in range(N)]
    per_rank = [sum(in_rank[t][r] for t in range(N)) for r in range(R)]
    eslot = [[-1] * K for _ in range(N)]
    for (t, k, e) in valid:
        before = sum(1 for (t2, k2, e2) in valid if e2 < e) + \
            sum(1 for (t2, k2, e2) in valid if e2 == e and (t2, k2) < (t, k))
        eslot[t][k] = before
    rslot = [[-1] * R for _ in range(N)]
    for t in range(N):
        for r in range(R):
            if in_rank[t][r]:
                rslot[t][r] = sum(per_rank[:r]) + sum(in_rank[t2][r] for t2 in range(t))
    return per_expert, per_rank, in_rank, eslot, rslot


@pytest.mark.parametrize("N,K,R", [(3, 2, 1), (3, 2, 2), (3, 2, 4), (2, 3, 2), (1, 4, 4)])
def test_brute_force_tiny(N, K, R):
    """Every routing in {-1..3}^(N*K) with E=4 (5^6 = 15,625 cases for N=3, K=2)."""
    E = 4
    for combo in itertools.product(range(-1, E), repeat=N * K):
        idx = np.array(combo, np.int32).reshape(N, K)
        o = oracle.layout(idx, E, R)
        pe, pr, mask, es, rs = _brute(idx, E, R)
        assert o["num_tokens_per_expert"].tolist() == pe
        assert o["num_tokens_per_rank"].tolist() == pr
        assert o["is_token_in_rank"].astype(bool).tolist() == mask
        assert o["expert_slot"].tolist() == es, combo
        assert o["rank_slot"].tolist() == rs, combo


def test_duplicate_experts_in_a_row():
    # The generator never repeats an expert within a row; the oracle still
    # gives each (t, k) its own row and keeps one copy per rank.
    idx = np.array([[3, 3, 1], [1, -1, 3]], np.int32)
    o = oracle.layout(idx, 4, 2)
    assert o["num_tokens_per_expert"].tolist() == [0, 2, 0, 3]
    assert o["expert_slot"].tolist() == [[2, 3, 0], [1, -1, 4]]
    assert o["num_tokens_per_rank"].tolist() == [2, 2]


def test_bad_indices_are_masked_and_flagged():
    idx = np.array([[0, 4], [-2, 1], [2, -1]], np.int32)
    o = oracle.layout(idx, 4, 2)
    assert o["status"] & oracle.BAD_INDEX
    assert o["num_tokens_per_expert"].tolist() == [1, 1, 1, 0]
    assert o["expert_slot"].tolist() == [[0, -1], [-1, 1], [2, -1]]
    assert o["is_token_in_rank"].tolist() == [[1, 0], [1, 0], [0, 1]]


def test_empty_and_all_masked():
    o = oracle.layout(np.zeros((0, 4), np.int32), 8, 4)
    assert o["num_tokens_per_expert"].sum() == 0 and o["rank_offset"].tolist() == [0] * 5
    idx = np.full((5, 3), -1, np.int32)
    o = oracle.layout(idx, 8, 4)
    assert o["status"] == 0
    assert np.all(o["expert_slot"] == -1) and np.all(o["rank_slot"] == -1)
    assert o["expert_offset"].tolist() == [0] * 9
