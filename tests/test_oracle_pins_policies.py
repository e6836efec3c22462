"""Pins of the oracle's overflow policies, expert-choice routing and
sequence-level statistics against facts that do not come from the oracle:
hand-worked cases (tests/golden), an independent algorithm, closed forms and
invariants.

Pages: "MoE notes" (chiang97912.github.io), section Expert capacity (full
expert -> next candidate; all full -> the token skips the layer);
mkbk-pku.cn MoE notes, capacity section (drop, second-choice re-routing,
padding to capacity); heavensheep.xyz MoE notes, Routing Function (expert
choose token) and Training (sequence-level balance)."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, rest = line.split(None, 1)
        rows[key] = rest
    return rows


def _groups(text, dtype=int):
    return np.array([[dtype(v) for v in g.split()] for g in text.split("|")])


# ------------------------------------------------------------ f2: overflow

def test_overflow_hand_worked_example():
    g = _golden("overflow_example.txt")
    cand = _groups(g["candidates"])
    for priority, key in ((0, "token_order_slot"), (1, "rank_order_slot")):
        r = oracle.capacity_policy(cand, k=1, E=3, C=1, priority=priority)
        np.testing.assert_array_equal(r["slot"], _groups(g[key]), err_msg=key)
        np.testing.assert_array_equal(r["offsets"], [0, 1, 2, 3])


def _fixed_point(cand, k, C, E, priority):
    """A second algorithm for the same policy, written independently of the
    sequential walk: iterate each expert's fill position (the position, in the
    priority order, of the candidate that took its last row) until it stops
    changing; a candidate is available iff it comes no later than that
    position. Returns rank-in-expert of kept candidates, -1 otherwise."""
    T, n = cand.shape
    pos = (lambda t, j: t * n + j) if priority == 0 else (lambda t, j: j * T + t)
    order = sorted(((t, j) for t in range(T) for j in range(n)), key=lambda a: pos(*a))
    inf = T * n
    fill = np.full(E, inf)
    for _ in range(10 * T * n + 10):
        tried = np.zeros((T, n), bool)
        for t in range(T):
            need = k
            for j in range(n):
                if need == 0:
                    break
                tried[t, j] = True
                if pos(t, j) <= fill[cand[t, j]]:
                    need -= 1
        rank = -np.ones((T, n), int)
        cnt = np.zeros(E, int)
        new = np.full(E, inf)
        for t, j in order:
            if tried[t, j]:
                e = cand[t, j]
                rank[t, j] = cnt[e]
                if cnt[e] == C - 1:
                    new[e] = pos(t, j)
                cnt[e] += 1
        if (new == fill).all():
            return np.where(rank < C, rank, -1)
        fill = new
    raise AssertionError("fixed point did not settle")


@pytest.mark.parametrize("priority", [0, 1])
def test_overflow_matches_fixed_point_algorithm(priority):
    rng = np.random.default_rng(11 + priority)
    for _ in range(120):
        T = int(rng.integers(1, 40))
        E = int(rng.integers(2, 8))
        k = int(rng.integers(1, min(3, E) + 1))
        n = int(rng.integers(k, E + 1))
        C = int(rng.integers(1, T * k // E + 3))
        w = rng.random(E) ** 3 + 0.02
        cand = np.stack([rng.choice(E, n, replace=False, p=w / w.sum()) for _ in range(T)])
        r = oracle.capacity_policy(cand, k, E, C, priority=priority)
        rank = _fixed_point(cand, k, C, E, priority)
        kept_rows = np.where(rank >= 0, r["offsets"][cand] + rank, -1)
        np.testing.assert_array_equal(r["slot"], kept_rows)


def test_overflow_invariants_and_padding():
    rng = np.random.default_rng(5)
    T, E, k, n, C = 300, 6, 2, 4, 70
    w = np.array([8, 4, 2, 1, 1, 1], float)
    cand = np.stack([rng.choice(E, n, replace=False, p=w / w.sum()) for _ in range(T)])
    for priority in (0, 1):
        r = oracle.capacity_policy(cand, k, E, C, priority=priority)
        kept_per_token = (r["slot"] >= 0).sum(1)
        assert kept_per_token.max() <= k
        assert (r["kept"] <= C).all()
        assert r["kept"].sum() == (r["slot"] >= 0).sum()
        np.testing.assert_array_equal(r["counts"], np.bincount(cand[:, :k].ravel(), minlength=E))
        # every token short of k experts found every candidate it did not keep full
        full = r["kept"] == C
        for t in np.nonzero(kept_per_token < k)[0]:
            assert all(full[cand[t, j]] for j in range(n) if r["slot"][t, j] < 0)
        # re-routing keeps at least as many as dropping
        drop = oracle.capacity_policy(cand[:, :k], k, E, C, priority=priority)
        assert (r["slot"] >= 0).sum() >= (drop["slot"] >= 0).sum()
        # padding: same rows per expert, blocks of exactly C rows
        rp = oracle.capacity_policy(cand, k, E, C, priority=priority, pad=True)
        np.testing.assert_array_equal(rp["offsets"], np.arange(E + 1) * C)
        np.testing.assert_array_equal(rp["kept"], r["kept"])
        same = (rp["slot"] >= 0) == (r["slot"] >= 0)
        assert same.all()
        for e in range(E):
            assert (rp["row_token"][e * C + r["kept"][e]:(e + 1) * C] == -1).all()
            np.testing.assert_array_equal(
                rp["row_token"][e * C:e * C + r["kept"][e]],
                r["row_token"][r["offsets"][e]:r["offsets"][e + 1]])


def test_overflow_special_cases():
    rng = np.random.default_rng(9)
    T, E, k = 64, 8, 2
    cand = np.stack([rng.permutation(E)[:4] for _ in range(T)])
    # no limit: nothing is re-routed, the first k candidates are all kept
    r = oracle.capacity_policy(cand, k, E, C=T, priority=0)
    assert (r["slot"][:, :k] >= 0).all() and (r["slot"][:, k:] < 0).all()
    # one candidate per choice, token order: plain dropping (the pinned drop capacity)
    r = oracle.capacity_policy(cand[:, :k], k, E, C=9, priority=0)
    ref = oracle.capacity(cand[:, :k], E, 9)
    np.testing.assert_array_equal(r["slot"], ref["slot"])
    # rank order without re-routing = token-order dropping over the list
    # of choices laid out rank by rank (one choice per list entry)
    r = oracle.capacity_policy(cand[:, :k], k, E, C=9, priority=1)
    flat = cand[:, :k].T.reshape(-1, 1)
    ref = oracle.capacity(flat, E, 9)
    np.testing.assert_array_equal((r["slot"] >= 0).T.reshape(-1), ref["slot"][:, 0] >= 0)


def test_select_candidates_order_and_gates():
    rng = np.random.default_rng(3)
    T, E, k, n = 50, 9, 2, 5
    s = rng.integers(0, 4, (T, E)).astype(np.float32)  # many ties
    p = rng.random((T, E)).astype(np.float32)
    ids, w = oracle.select_candidates(s, p, k, n, renorm=True)
    for t in range(T):
        order = np.lexsort((np.arange(E), -s[t].astype(np.float64)))[:n]
        np.testing.assert_array_equal(ids[t], order)
    ids2, w2 = oracle.select(s, p, k, renorm=True)
    np.testing.assert_array_equal(ids[:, :k], ids2)
    np.testing.assert_allclose(w[:, :k].sum(1), 1.0, rtol=0, atol=1e-12)
    pj = p[np.arange(T)[:, None], ids].astype(np.float64)
    np.testing.assert_allclose(w / w[:, :1], pj / pj[:, :1], rtol=1e-12)
    _, wr = oracle.select_candidates(s, p, k, n, renorm=False)
    np.testing.assert_array_equal(wr, pj)


# -------------------------------------------------------- f3: expert choice

def test_expert_choice_hand_worked_example():
    g = _golden("expert_choice_example.txt")
    p = np.stack([np.array(g["p0"].split(), np.float32), np.array(g["p1"].split(), np.float32)], 1)
    r = oracle.expert_choice(p, 2)
    np.testing.assert_array_equal(r["row_token"], [int(v) for v in g["row_token"].split()])
    np.testing.assert_array_equal(r["tok_row"], _groups(g["tok_row"]))
    np.testing.assert_array_equal(r["row_w"], p[r["row_token"], [0, 0, 1, 1]])


def test_expert_choice_brute_force_and_invariants():
    rng = np.random.default_rng(21)
    for T, E, C in [(40, 4, 10), (33, 7, 5), (16, 3, 16), (25, 5, 1)]:
        p = rng.integers(0, 6, (T, E)).astype(np.float32) / 8  # ties
        r = oracle.expert_choice(p, C)
        for e in range(E):
            order = np.lexsort((np.arange(T), -p[:, e].astype(np.float64)))
            chosen = np.sort(order[:C])
            np.testing.assert_array_equal(r["row_token"][e * C:(e + 1) * C], chosen)
            rest = np.setdiff1d(np.arange(T), chosen)
            if rest.size:
                assert p[chosen, e].min() >= p[rest, e].max()
            for i, t in enumerate(chosen):
                assert r["tok_row"][t, e] == e * C + i
        assert ((r["tok_row"] >= 0).sum(0) == C).all()


def test_expert_choice_full_capacity_is_the_dense_mixture():
    """With C = T every expert takes every token, so the layer output is the
    dense softmax mixture sum_e p_e E_e(x) ("MoE notes": y = sum_i G(x)_i E_i(x)
    with G the full softmax), written here as an explicit dense loop."""
    rng = np.random.default_rng(4)
    T, d, E, F = 6, 5, 3, 4
    x = rng.normal(size=(T, d)).astype(np.float32)
    W1 = rng.normal(size=(E, F, d)).astype(np.float32)
    W2 = rng.normal(size=(E, d, F)).astype(np.float32)
    z = rng.normal(size=(T, E))
    p = (np.exp(z) / np.exp(z).sum(1, keepdims=True)).astype(np.float32)
    r = oracle.expert_choice(p, T)
    O = np.zeros((E * T, d))
    for e in range(E):
        rows = r["row_token"][e * T:(e + 1) * T]
        O[e * T:(e + 1) * T] = oracle.expert_ffn(x[rows], W1[e], W2[e], oracle.RELU)
    y = oracle.combine_expert_choice(r["tok_row"], p, O)
    dense = np.zeros((T, d))
    for t in range(T):
        for e in range(E):
            h = np.maximum(W1[e].astype(np.float64) @ x[t].astype(np.float64), 0.0)
            dense[t] += float(p[t, e]) * (W2[e].astype(np.float64) @ h)
    np.testing.assert_allclose(y, dense, rtol=1e-12, atol=1e-12)


# ------------------------------------------------ f4: sequence-level stats

def test_seq_stats_hand_worked_example():
    g = _golden("seq_stats_example.txt")
    offs = np.array(g["offsets"].split(), np.int32)
    ids = np.array(g["ids"].split(), np.int32).reshape(-1, 1)
    p = np.array(g["p"].split(), np.float32).reshape(-1, 2)
    r = oracle.seq_aux_stats(p, ids, 1, offs)
    np.testing.assert_allclose(r["aux"], [float(v) for v in g["aux"].split()], rtol=1e-12)
    assert r["mean"] == pytest.approx(float(g["mean"]), rel=1e-12)
    np.testing.assert_allclose(r["f"][1], [1 / 3, 2 / 3], rtol=1e-12)


def test_seq_stats_one_sequence_is_the_batch_statistic_and_uniform_is_one():
    rng = np.random.default_rng(8)
    T, E, k = 96, 6, 2
    z = rng.normal(size=(T, E))
    p = (np.exp(z) / np.exp(z).sum(1, keepdims=True)).astype(np.float32)
    ids = np.stack([rng.permutation(E)[:3] for _ in range(T)]).astype(np.int32)
    r = oracle.seq_aux_stats(p, ids, k, [0, T])
    b = oracle.aux_stats(p, ids[:, :k], np.ones((T, k), np.float32), E)
    np.testing.assert_allclose(r["f"][0], b["f"], rtol=1e-12)
    np.testing.assert_allclose(r["P"][0], b["P"], rtol=1e-12)
    assert r["aux"][0] == pytest.approx(b["aux"], rel=1e-12)
    # uniform inside every sequence: token t's row is a fixed vector rotated by
    # t mod E and it chooses experts t, t+1 (mod E); sequences are multiples of E
    base = np.array([0.4, 0.25, 0.15, 0.1, 0.06, 0.04])
    pu = np.stack([np.roll(base, t % E) for t in range(T)]).astype(np.float32)
    iu = np.stack([[(t) % E, (t + 1) % E] for t in range(T)]).astype(np.int32)
    r = oracle.seq_aux_stats(pu, iu, 2, [0, 12, 48, 48, 96])
    np.testing.assert_allclose(r["aux"], [1, 1, 0, 1], rtol=1e-6)
    assert r["mean"] == pytest.approx(1.0, rel=1e-6)
