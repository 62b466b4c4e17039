"""Checks that pin the oracle to facts fixed outside itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` (the real one, or a copy with a planted
mistake) and raises AssertionError when the oracle disagrees with the fact it pins.  The
facts come from the pages (worked example, printed depths, the losslessness theorem and
its corollaries), from the Philox publication (known-answer vectors), or from textbook
routines (numpy argmax, scipy logsumexp, a chi-squared test).

Sources (page title -- section):
  [SD] "7.6 Speculative Decoding: Draft Models, Medusa, EAGLE & Lookahead"
  [MS] "Medusa, EAGLE and self-speculation"
  [HB] "Speculative Decoding: Draft Models, EAGLE, and How to Actually Use It"
"""
from __future__ import annotations

import itertools
import os

import numpy as np
from scipy import special, stats

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _softmax(l, T):
    l = np.asarray(l, np.float64) / T
    m = np.max(l)
    e = np.exp(l - m)
    return e / e.sum()


# --------------------------------------------------------------------------------------
# Philox4x32-10 known-answer vectors (SC'11 reference implementation)
# --------------------------------------------------------------------------------------
def pin_philox_kat(orc):
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        lines = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert lines
    for ln in lines:
        v = [int(x, 16) for x in ln]
        out = orc.philox4x32_10(v[0:4], v[4:6])
        assert list(out) == v[6:10], (ln, [hex(x) for x in out])


def pin_uniform_definition(orc):
    """u = (word0 >> 8) * 2^-24 of Philox at counter (4i + purpose, b, off lo, off hi)."""
    rng = np.random.RandomState(7)
    for _ in range(200):
        seed = int(rng.randint(0, 2**62)) * 3 + 1
        off = int(rng.randint(0, 2**62))
        b, i, pur = int(rng.randint(0, 2**20)), int(rng.randint(0, 2**10)), int(rng.randint(0, 2))
        w = orc.philox4x32_10([(i << 2) | pur, b, off & 0xFFFFFFFF, off >> 32],
                              [seed & 0xFFFFFFFF, seed >> 32])
        u = orc.uniform(seed, off, b, i, pur)
        assert u == (int(w[0]) >> 8) * 2.0**-24
        assert 0.0 <= u <= 1.0 - 2.0**-24


# --------------------------------------------------------------------------------------
# P1: brute-force losslessness [SD "The proof that this is exact"; HB "The Algorithm"]
# --------------------------------------------------------------------------------------
def _tiny_model(prefix, V, salt, scale, mask_frac=0.0):
    """Deterministic prefix-dependent logits of a toy language model."""
    h = salt
    for t in prefix:
        h = (h * 1000003 + 7919 * (t + 1)) % (2**32)
    rs = np.random.RandomState(h)
    l = rs.normal(0.0, scale, V)
    if mask_frac > 0:
        masked = rs.rand(V) < mask_frac
        if masked.all():
            masked[rs.randint(V)] = False
        l[masked] = -np.inf
    return l


def speculative_law(orc, V, gamma, L, T, salt_p=11, salt_q=23, mask_p=0.0):
    """Law of the first L emitted tokens when rounds of the oracle's enumeration mode are
    composed, drafts drawn from the toy draft model; prefixes are merged so the work stays
    polynomial."""
    law = {}
    frontier = {(): 1.0}
    while frontier:
        nxt = {}
        for y, w in frontier.items():
            if len(y) >= L:
                law[y[:L]] = law.get(y[:L], 0.0) + w
                continue
            for x in itertools.product(range(V), repeat=gamma):
                qx = 1.0
                for i in range(gamma):
                    qx *= _softmax(_tiny_model(y + x[:i], V, salt_q, 1.5), T)[x[i]]
                if qx == 0.0:
                    continue
                t_rows = [_tiny_model(y + x[:i], V, salt_p, 1.5, mask_p) for i in range(gamma + 1)]
                d_rows = [_tiny_model(y + x[:i], V, salt_q, 1.5) for i in range(gamma)]
                P = orc.exact_probs(np.array(t_rows), np.array(d_rows).reshape(gamma, V),
                                    np.array(x, np.int32), T)
                for k in range(gamma + 1):
                    for j in range(V):
                        if P[k, j] > 0.0:
                            z = y + tuple(x[:k]) + (j,)
                            nxt[z] = nxt.get(z, 0.0) + w * qx * P[k, j]
        frontier = nxt
    return law


def target_law(V, L, T, salt_p=11, mask_p=0.0):
    law = {}
    for s in itertools.product(range(V), repeat=L):
        pr = 1.0
        for l in range(L):
            pr *= _softmax(_tiny_model(s[:l], V, salt_p, 1.5, mask_p), T)[s[l]]
        law[s] = pr
    return law


def pin_bruteforce_lossless(orc, cases=((3, 2, 3, 0.8, 0.0), (2, 3, 4, 1.3, 0.0),
                                        (4, 1, 2, 1.0, 0.3), (5, 2, 2, 0.7, 0.25))):
    for V, gamma, L, T, mask in cases:
        got = speculative_law(orc, V, gamma, L, T, mask_p=mask)
        want = target_law(V, L, T, mask_p=mask)
        keys = set(got) | set(want)
        err = max(abs(got.get(k, 0.0) - want.get(k, 0.0)) for k in keys)
        assert err < 1e-12, (V, gamma, L, T, mask, err)
        assert abs(sum(got.values()) - 1.0) < 1e-12


# --------------------------------------------------------------------------------------
# P2: chi-squared test of the Philox-driven sampler against p [SD "The rule"]
# --------------------------------------------------------------------------------------
def _chi2_rows(V, gamma):
    rs = np.random.RandomState(4242)
    # rows for absolute positions 0..gamma+1 (target) and 0..gamma (draft); the toy model
    # is position-dependent but prefix-independent, so the law of (y0, y1) is p0 x p1
    t = rs.normal(0, 1.3, (gamma + 2, V))
    d = t[: gamma + 1] + rs.normal(0, 1.0, (gamma + 1, V))
    return t.astype(np.float32), d.astype(np.float32)


def pin_chi2_sampler(orc, trials=1_000_000, V=5, gamma=2, T=0.9, seed=0xC0FFEE, alpha=1e-3):
    t, d = _chi2_rows(V, gamma)
    p = [_softmax(t[l], T) for l in range(gamma + 2)]
    q = [_softmax(d[l], T) for l in range(gamma + 1)]
    rng = np.random.RandomState(99)

    def drafts(start):
        cols = []
        for i in range(gamma):
            cdf = np.cumsum(q[start + i])
            cols.append(np.minimum(np.searchsorted(cdf, rng.rand(trials), side="right"), V - 1))
        return np.stack(cols, 1).astype(np.int32)

    def rows(a, start, n):
        return np.broadcast_to(a[start:start + n][None], (trials, n, V))

    x1 = drafts(0)
    acc1, out1, _ = orc.verify_sample(rows(t, 0, gamma + 1), rows(d, 0, gamma), x1, T, seed, 0)
    y0 = out1[:, 0]
    # second token: from this round when it emitted >= 2 tokens, else from a second round
    # that starts at position 1 with fresh uniforms (offset 1)
    x2 = drafts(1)
    acc2, out2, _ = orc.verify_sample(rows(t, 1, gamma + 1), rows(d, 1, gamma), x2, T, seed, 1)
    y1 = np.where(acc1 >= 1, out1[:, 1], out2[:, 0])
    assert (acc1 >= 0).all() and (acc1 <= gamma).all()
    obs0 = np.bincount(y0, minlength=V)
    _, pv0 = stats.chisquare(obs0, p[0] * trials)
    obs01 = np.bincount(y0 * V + y1, minlength=V * V)
    _, pv01 = stats.chisquare(obs01, np.outer(p[0], p[1]).ravel() * trials)
    assert pv0 > alpha, ("first token", pv0, obs0 / trials, p[0])
    assert pv01 > alpha, ("first two tokens", pv01)


# --------------------------------------------------------------------------------------
# P3: q == p accepts every draft (u < 1 = p/q) [SD "The rule"]
# --------------------------------------------------------------------------------------
def pin_identical_rows_accept_all(orc):
    rs = np.random.RandomState(3)
    for gamma, V, T in ((1, 7, 1.0), (4, 50, 0.7), (8, 33, 1.3)):
        B = 500
        t = rs.normal(0, 2.0, (B, gamma + 1, V)).astype(np.float32)
        d = t[:, :gamma, :].copy()
        x = np.stack([[rs.choice(V, p=_softmax(d[b, i], T)) for i in range(gamma)]
                      for b in range(B)]).astype(np.int32)
        acc, out, _ = orc.verify_sample(t, d, x, T, 1234, 0)
        assert (acc == gamma).all(), np.bincount(acc)
        assert (out[:, :gamma] == x).all()


# --------------------------------------------------------------------------------------
# P4: point masses reduce sampling to greedy [SD "Extending to a chain": temperature 0]
# --------------------------------------------------------------------------------------
def pin_one_hot_equals_greedy(orc):
    rs = np.random.RandomState(5)
    B, gamma, V = 400, 5, 40
    a = rs.randint(0, V, (B, gamma + 1))
    x = np.where(rs.rand(B, gamma) < 0.7, a[:, :gamma], rs.randint(0, V, (B, gamma)))
    t = np.full((B, gamma + 1, V), -np.inf, np.float32)
    d = np.full((B, gamma, V), -np.inf, np.float32)
    for b in range(B):
        for i in range(gamma + 1):
            t[b, i, a[b, i]] = rs.normal()
        for i in range(gamma):
            d[b, i, x[b, i]] = rs.normal()
    acc_s, out_s, _ = orc.verify_sample(t, d, x.astype(np.int32), 1.0, 77, 0)
    acc_g, out_g = orc.verify_greedy(t, x.astype(np.int32))
    assert (acc_s == acc_g).all() and (out_s == out_g).all()


def pin_one_hot_draft_accept_prob(orc):
    """q one-hot on x*: P(accept) = p(x*) exactly, residual = p off x*, renormalised."""
    rs = np.random.RandomState(6)
    for V in (2, 5, 17):
        t = rs.normal(0, 1.5, (2, V))
        xs = int(rs.randint(V))
        d = np.full((1, V), -np.inf)
        d[0, xs] = 0.0
        P = orc.exact_probs(t, d, np.array([xs], np.int32), 1.0)
        p0 = _softmax(t[0], 1.0)
        assert abs(P[1].sum() - p0[xs]) < 1e-15
        res = p0.copy()
        res[xs] = 0.0
        res /= res.sum()
        assert np.max(np.abs(P[0] - (1 - p0[xs]) * res)) < 1e-15


# --------------------------------------------------------------------------------------
# P5: structural invariants of a sampling round [SD "Extending to a chain"]
# --------------------------------------------------------------------------------------
def pin_round_invariants(orc):
    rs = np.random.RandomState(8)
    for gamma, V in ((1, 3), (3, 11), (6, 64)):
        B = 300
        t = rs.normal(0, 2, (B, gamma + 1, V)).astype(np.float32)
        d = (t[:, :gamma] + rs.normal(0, 1.0, (B, gamma, V))).astype(np.float32)
        x = rs.randint(0, V, (B, gamma)).astype(np.int32)
        acc, out, _ = orc.verify_sample(t, d, x, 1.0, 5, 3)
        assert ((acc >= 0) & (acc <= gamma)).all()
        for b in range(B):
            k = acc[b]
            assert (out[b, :k] == x[b, :k]).all()
            assert 0 <= out[b, k] < V
            assert (out[b, k + 1:] == -1).all()


# --------------------------------------------------------------------------------------
# P6: the worked p/q example [HB "The Algorithm"]
# --------------------------------------------------------------------------------------
def pin_worked_example(orc):
    with open(os.path.join(GOLDEN, "worked_example_accept.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    # two-token vocabulary per position: index 0 is the drafted token, index 1 "the rest"
    qs = [float(r[2]) for r in rows]
    ps = [float(r[3]) for r in rows]
    printed = [float(r[4]) for r in rows]
    gamma = len(rows)
    t = np.log(np.array([[p, 1 - p] for p in ps] + [[0.5, 0.5]]))
    d = np.log(np.array([[q, 1 - q] for q in qs]))
    P = orc.exact_probs(t, d, np.zeros(gamma, np.int32), 1.0)
    reach = [P[k:].sum() for k in range(gamma + 1)]
    for i in range(gamma):
        cond = reach[i + 1] / reach[i]
        assert abs(cond - min(1.0, ps[i] / qs[i])) < 1e-12
        assert round(cond, 2) == printed[i], (i, cond, printed[i])
    # "accepted [A, B], rejected C": the correction after rejecting C never re-emits C,
    # because the residual (p - q)+ is zero where the draft over-covered
    assert P[2, 0] == 0.0 and P[2, 1] > 0.0


# --------------------------------------------------------------------------------------
# P7: alpha = sum min(p, q) = 1 - TV(p, q) [SD Exercise 2c] and E[tokens] per round
#     (1 - alpha^(gamma+1)) / (1 - alpha) = 3.36 at alpha 0.8, k = 4 [HB "The Algorithm"]
# --------------------------------------------------------------------------------------
def pin_acceptance_rate(orc):
    rs = np.random.RandomState(9)
    for V in (2, 4, 9):
        t = rs.normal(0, 1.2, (2, V))
        d = rs.normal(0, 1.2, (1, V))
        p, q = _softmax(t[0], 1.0), _softmax(d[0], 1.0)
        acc = sum(q[x] * orc.exact_probs(t, d, np.array([x], np.int32), 1.0)[1].sum()
                  for x in range(V))
        assert abs(acc - np.minimum(p, q).sum()) < 1e-14
        assert abs(acc - (1.0 - 0.5 * np.abs(p - q).sum())) < 1e-14
    gamma, alpha = 4, 0.8
    p, q = np.array([0.9, 0.1]), np.array([0.7, 0.3])  # sum min(p, q) = 0.8
    t = np.log(np.tile(p, (gamma + 1, 1)))
    d = np.log(np.tile(q, (gamma, 1)))
    E = 0.0
    for x in itertools.product(range(2), repeat=gamma):
        w = np.prod([q[xi] for xi in x])
        P = orc.exact_probs(t, d, np.array(x, np.int32), 1.0)
        E += w * sum((k + 1) * P[k].sum() for k in range(gamma + 1))
    assert abs(E - (1 - alpha ** (gamma + 1)) / (1 - alpha)) < 1e-12
    assert round(E, 2) == 3.36


# --------------------------------------------------------------------------------------
# P8: greedy = longest prefix matching a textbook argmax [SD "Extending to a chain";
#     MS speculative_greedy]
# --------------------------------------------------------------------------------------
def _bf16_bits_from_float(a):
    """Round-to-nearest-even fp32 -> bf16 bit patterns (test-side helper)."""
    u = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return r


def pin_greedy_textbook(orc):
    rs = np.random.RandomState(10)
    for gamma, V, dt in ((1, 5, "f32"), (4, 37, "bf16"), (6, 300, "f32"), (3, 1, "f32")):
        B = 300
        # small integers -> many exact ties, so the lowest-index rule is exercised
        vals = rs.randint(-3, 4, (B, gamma + 1, V)).astype(np.float32)
        a = np.argmax(vals, axis=-1)  # numpy: first occurrence of the maximum
        x = np.where(rs.rand(B, gamma) < 0.75, a[:, :gamma], rs.randint(0, V, (B, gamma)))
        x = x.astype(np.int32)
        nan_rows = rs.rand(B) < 0.05
        vals[nan_rows, rs.randint(0, gamma + 1), rs.randint(0, V)] = np.nan
        bad_tok = (rs.rand(B) < 0.03) & (gamma > 0)
        x[bad_tok, 0] = V + 3
        logits = _bf16_bits_from_float(vals) if dt == "bf16" else vals
        acc, out = orc.verify_greedy(logits, x)
        for b in range(B):
            if nan_rows[b] or bad_tok[b]:
                assert acc[b] == -1 and (out[b] == -1).all()
                continue
            n = 0
            while n < gamma and x[b, n] == a[b, n]:
                n += 1
            assert acc[b] == n
            assert list(out[b, :n]) == list(x[b, :n]) and out[b, n] == a[b, n]
            assert (out[b, n + 1:] == -1).all()


# --------------------------------------------------------------------------------------
# P9: trees -- the printed depths [SD "Tree Attention"], a chain tree equals greedy, and
#     brute force over root paths [SD Exercise 5]
# --------------------------------------------------------------------------------------
def pin_tree_printed_depths(orc):
    with open(os.path.join(GOLDEN, "tree_depths.txt")) as f:
        kv = {ln.split()[0]: [int(v) for v in ln.split()[1:]] for ln in f
              if ln.strip() and not ln.startswith("#")}
    parents, depths = kv["parents"], kv["depths"]
    N, V = len(parents), 8
    # one sequence per node v: only the path root -> v matches, so accepted_len = depth(v)
    B = N
    t = np.zeros((B, N, V), np.float32)
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        for u in range(N):
            t[b, u, (u + 1) % V] = 5.0  # argmax of node u is (u + 1) % V
        on_path = set()
        w = b
        while w != -1:
            on_path.add(w)
            w = parents[w]
        for u in range(1, N):
            want = (parents[u] + 1) % V
            tokens[b, u] = want if u in on_path else (want + 1) % V
    acc, out, path, _ = orc.verify_tree_greedy(t, parents, tokens, max(depths))
    assert list(acc) == depths
    for b in range(B):
        assert path[b, depths[b]] == b


def pin_chain_tree_equals_greedy(orc):
    rs = np.random.RandomState(12)
    for gamma, V in ((1, 4), (5, 23), (7, 100)):
        B = 200
        vals = rs.randint(-2, 3, (B, gamma + 1, V)).astype(np.float32)
        a = np.argmax(vals, axis=-1)
        x = np.where(rs.rand(B, gamma) < 0.8, a[:, :gamma], rs.randint(0, V, (B, gamma)))
        x = x.astype(np.int32)
        parent = [-1] + list(range(gamma))
        tokens = np.concatenate([np.zeros((B, 1), np.int32), x], 1)
        acc_t, out_t, path_t, _ = orc.verify_tree_greedy(vals, parent, tokens, gamma)
        acc_g, out_g = orc.verify_greedy(vals, x)
        assert (acc_t == acc_g).all() and (out_t == out_g).all()
        for b in range(B):
            assert list(path_t[b, :acc_t[b] + 1]) == list(range(acc_t[b] + 1))


def random_tree(rs, N):
    parent = [-1] + [int(rs.randint(0, v)) for v in range(1, N)]
    return parent


def pin_tree_bruteforce(orc):
    rs = np.random.RandomState(13)
    for N, V, dup in ((1, 3, False), (2, 2, False), (9, 3, True), (30, 5, True), (64, 50, False)):
        B = 150
        parent = random_tree(rs, N)
        depth = [0] * N
        for v in range(1, N):
            depth[v] = depth[parent[v]] + 1
        D = max(depth)
        vals = rs.randint(-2, 3, (B, N, V)).astype(np.float32)
        a = np.argmax(vals, axis=-1)
        tokens = rs.randint(0, V, (B, N)).astype(np.int32)
        for b in range(B):
            for v in range(1, N):
                if rs.rand() < 0.6:
                    tokens[b, v] = a[b, parent[v]]
        acc, out, path, flags = orc.verify_tree_greedy(vals, parent, tokens, D)
        for b in range(B):
            ok = []
            for v in range(N):  # a node is accepted iff every edge on its root path matches
                w, good = v, True
                while w != 0:
                    good &= tokens[b, w] == a[b, parent[w]]
                    w = parent[w]
                ok.append(good)
            cands = [v for v in range(N) if ok[v]]
            best = min(cands, key=lambda v: (-depth[v], v))
            chain = []
            w = best
            while w != -1:
                chain.append(w)
                w = parent[w]
            chain = chain[::-1]
            assert acc[b] == depth[best]
            assert list(path[b, :len(chain)]) == chain and (path[b, len(chain):] == -1).all()
            assert list(out[b, :depth[best]]) == [tokens[b, w] for w in chain[1:]]
            assert out[b, depth[best]] == a[b, best]
            # Exercise 5's greedy walk takes the first matching child at each node
            node, walk = 0, [0]
            while True:
                nxt = [c for c in range(N) if parent[c] == node and tokens[b, c] == a[b, node]]
                if not nxt:
                    break
                node = nxt[0]
                walk.append(node)
            assert bool(flags[b] & 1) == (walk != chain)
    # a malformed or too-deep tree invalidates every sequence
    vals = np.zeros((2, 3, 4), np.float32)
    toks = np.zeros((2, 3), np.int32)
    for par, D in (([-1, 0, 2], 2), ([0, 0, 1], 2), ([-1, 0, 1], 1)):
        acc, out, path, _ = orc.verify_tree_greedy(vals, par, toks, D)
        assert (acc == -1).all() and (out == -1).all() and (path == -1).all()


# --------------------------------------------------------------------------------------
# Token-tree sampling: multi-round rejection [SD "Tree Attention", the paragraph on
# SpecInfer's rule].  The rule is lossless for a drafter that draws each node's children
# from q at that node, with or without replacement.
# --------------------------------------------------------------------------------------
def _draw_law(q, k, without_replacement):
    """Every ordered k-tuple of tokens a drafter draws from q, with its probability."""
    V = len(q)
    for xs in itertools.product(range(V), repeat=k):
        pr, left, used = 1.0, 1.0, set()
        for x in xs:
            if without_replacement:
                if x in used or left <= 0.0:
                    pr = 0.0
                    break
                pr *= q[x] / left
                left -= q[x]
                used.add(x)
            else:
                pr *= q[x]
        if pr > 0.0:
            yield xs, pr


def tree_round_law(orc, y, parent, V, T, wor, salt_p=11, salt_q=23, mask_p=0.0):
    """Law of the tokens one tree round emits after prefix y, averaged over the drafter's
    draws of every node's children and over the rule's uniforms (enumeration mode)."""
    N = len(parent)
    children = [[c for c in range(N) if parent[c] == v] for v in range(N)]

    def path_tokens(v, tok):
        out = []
        while v != 0:
            out.append(tok[v])
            v = parent[v]
        return tuple(reversed(out))

    assignments = [({}, 1.0)]
    for v in range(N):  # parents before children: path(v) is known when v's children are drawn
        if not children[v]:
            continue
        grown = []
        for tok, pr in assignments:
            q = _softmax(_tiny_model(y + path_tokens(v, tok), V, salt_q, 1.5), T)
            for xs, pq in _draw_law(q, len(children[v]), wor):
                t2 = dict(tok)
                t2.update(zip(children[v], xs))
                grown.append((t2, pr * pq))
        assignments = grown
    law = {}
    for tok, pr in assignments:
        tokens = [0] + [tok[c] for c in range(1, N)]
        t_rows = [_tiny_model(y + path_tokens(v, tok), V, salt_p, 1.5, mask_p) for v in range(N)]
        d_rows = [_tiny_model(y + path_tokens(v, tok), V, salt_q, 1.5) for v in range(N)]
        P = orc.exact_probs_tree(np.array(t_rows), np.array(d_rows), parent, tokens, T, wor)
        for v in range(N):
            for j in range(V):
                if P[v, j] > 0.0:
                    z = path_tokens(v, tok) + (j,)
                    law[z] = law.get(z, 0.0) + pr * P[v, j]
    return law


def pin_tree_sample_lossless(orc, cases=(([-1, 0, 0], 3, 3, 0.8, False, 0.0),
                                         ([-1, 0, 0], 3, 3, 0.8, True, 0.0),
                                         ([-1, 0, 0, 0], 4, 2, 1.1, True, 0.25),
                                         ([-1, 0, 0, 0], 3, 2, 1.0, True, 0.0),
                                         ([-1, 0, 0, 1], 3, 3, 0.9, False, 0.3),
                                         ([-1, 0, 1, 1, 0], 3, 3, 1.2, True, 0.0))):
    """Composed rounds of the tree rule emit exactly the target model's law (< 1e-12)."""
    for parent, V, L, T, wor, mask in cases:
        got, frontier = {}, {(): 1.0}
        while frontier:
            nxt = {}
            for y, w in frontier.items():
                if len(y) >= L:
                    got[y[:L]] = got.get(y[:L], 0.0) + w
                    continue
                for z, pz in tree_round_law(orc, y, parent, V, T, wor, mask_p=mask).items():
                    nxt[y + z] = nxt.get(y + z, 0.0) + w * pz
            frontier = nxt
        want = target_law(V, L, T, mask_p=mask)
        keys = set(got) | set(want)
        err = max(abs(got.get(k, 0.0) - want.get(k, 0.0)) for k in keys)
        assert err < 1e-12, (parent, V, L, T, wor, mask, err)


def _children_draws(rs, q, n, k, without_replacement):
    """n independent drafter draws of k ordered children from q ([n, k] tokens)."""
    if not without_replacement:
        return rs.choice(len(q), size=(n, k), p=q).astype(np.int32)
    # Gumbel keys: sorting log q + G gives sequential sampling without replacement
    with np.errstate(divide="ignore"):
        keys = np.log(q)[None, :] + rs.gumbel(size=(n, len(q)))
    return np.argsort(-keys, axis=1)[:, :k].astype(np.int32)


def pin_tree_sample_chi2(orc, trials=200_000, V=5, T=0.9, alpha=1e-3):
    """The Philox-driven tree sampler: over many rounds (fresh drafter draws and uniforms)
    the first emitted token follows p at the root and, after child c is accepted, the
    second follows p at c (chi-squared at alpha)."""
    rs = np.random.RandomState(4343)
    parent = [-1, 0, 0, 0]
    t_rows = rs.normal(0, 1.5, (4, V)).astype(np.float32)
    d_rows = rs.normal(0, 1.5, (4, V)).astype(np.float32)
    t_rows[0, 1] = -np.inf  # a token the target never emits
    p = [_softmax(t_rows[v].astype(np.float64), T) for v in range(4)]
    q0 = _softmax(d_rows[0].astype(np.float64), T)
    target = np.ascontiguousarray(np.broadcast_to(t_rows, (trials, 4, V)))
    draft = np.ascontiguousarray(np.broadcast_to(d_rows, (trials, 4, V)))
    for wor in (False, True):
        toks = np.zeros((trials, 4), np.int32)
        toks[:, 1:] = _children_draws(rs, q0, trials, 3, wor)
        acc, out, path, _ = orc.verify_tree_sample(target, draft, parent, toks, 1, T, seed=77,
                                                   offset=int(wor), without_replacement=wor)
        assert ((acc == 0) | (acc == 1)).all()
        live = p[0] > 0
        cnt = np.bincount(out[:, 0], minlength=V)
        assert (cnt[~live] == 0).all()
        assert stats.chisquare(cnt[live], trials * p[0][live]).pvalue > alpha
        for c in (1, 2, 3):  # the bonus after child c
            sel = path[:, 1] == c
            cnt = np.bincount(out[sel, 1], minlength=V)
            assert stats.chisquare(cnt, sel.sum() * p[c]).pvalue > alpha


def pin_chain_tree_sample_equals_chain(orc):
    """On a chain-shaped tree the tree rule is the chain rule, uniforms included: the same
    tokens, lengths and flags, bit for bit, in both sibling modes."""
    rs = np.random.RandomState(31)
    for gamma, V, T in ((1, 7, 1.0), (4, 40, 0.8), (6, 100, 1.3)):
        B = 96
        t = rs.normal(0, 2, (B, gamma + 1, V)).astype(np.float32)
        d = (t[:, :gamma] + rs.normal(0, 1, (B, gamma, V))).astype(np.float32)
        t[rs.rand(B, gamma + 1, V) < 0.1] = -np.inf
        t[:, :, 0] = 0.0  # every row keeps a finite entry
        x = np.array([[rs.choice(V, p=_softmax(d[b, i].astype(np.float64), T))
                       for i in range(gamma)] for b in range(B)], np.int32)
        acc, out, flags = orc.verify_sample(t, d, x, T, seed=5, offset=3)
        parent = [-1] + list(range(gamma))
        dd = np.concatenate([d, np.zeros((B, 1, V), np.float32)], axis=1)  # leaf row unused
        toks = np.concatenate([np.zeros((B, 1), np.int32), x], axis=1)
        for wor in (False, True):
            acc2, out2, path2, flags2 = orc.verify_tree_sample(t, dd, parent, toks, gamma, T, 5, 3,
                                                               without_replacement=wor)
            assert (acc2 == acc).all() and (out2 == out).all() and (flags2 == flags).all()
            for b in range(B):
                assert list(path2[b, :acc[b] + 1]) == list(range(acc[b] + 1))


def pin_tree_sample_invariants(orc):
    """Outputs of random trees: a root path of parent-child steps, its node tokens, one
    final token with positive weight, -1 padding; bad input gives -1."""
    rs = np.random.RandomState(57)
    for N, V in ((1, 3), (6, 4), (20, 9), (40, 30)):
        B = 60
        parent = random_tree(rs, N)
        depth = [0] * N
        for v in range(1, N):
            depth[v] = depth[parent[v]] + 1
        D = max(depth)
        t = rs.normal(0, 2, (B, N, V)).astype(np.float32)
        d = rs.normal(0, 2, (B, N, V)).astype(np.float32)
        t[rs.rand(B, N, V) < 0.2] = -np.inf
        t[:, :, V - 1] = 1.0
        toks = rs.randint(0, V, (B, N)).astype(np.int32)
        for wor in (False, True):
            acc, out, path, _ = orc.verify_tree_sample(t, d, parent, toks, D, 0.9, 11, 0, wor)
            for b in range(B):
                k = acc[b]
                assert 0 <= k <= D and path[b, 0] == 0 and (path[b, k + 1:] == -1).all()
                for s in range(1, k + 1):
                    assert parent[path[b, s]] == path[b, s - 1]
                    assert out[b, s - 1] == toks[b, path[b, s]]
                assert 0 <= out[b, k] < V and np.isfinite(t[b, path[b, k], out[b, k]])
                assert (out[b, k + 1:] == -1).all()
    t = np.zeros((3, 3, 4), np.float32)
    d = np.zeros((3, 3, 4), np.float32)
    t[0, 0, 1] = np.nan          # the root's target row
    d[1, 0, :] = -np.inf         # the draft row of a reached node with children
    toks = np.zeros((3, 3), np.int32)
    toks[2, 1] = 4               # a token out of range
    acc, out, path, _ = orc.verify_tree_sample(t, d, [-1, 0, 0], toks, 1, 1.0, 0)
    assert (acc == -1).all() and (out == -1).all() and (path == -1).all()
    # a row the walk never reads cannot matter: node 1's token has p = 0 at the root, so
    # node 1 is always rejected and its child, node 2, never reached
    t = rs.normal(0, 1, (40, 4, 6)).astype(np.float32)
    d = rs.normal(0, 1, (40, 4, 6)).astype(np.float32)
    t[:, 0, 3] = -np.inf
    toks = np.tile(np.array([0, 3, 1, 2], np.int32), (40, 1))
    ref = orc.verify_tree_sample(t, d, [-1, 0, 1, 0], toks, 2, 1.0, 9)
    t[:, 2, :] = np.nan
    d[:, 2, :] = np.nan
    d[:, 1, :] = np.nan  # node 1 has a child but is never reached
    got = orc.verify_tree_sample(t, d, [-1, 0, 1, 0], toks, 2, 1.0, 9)
    assert all((a == b).all() for a, b in zip(ref, got)) and (ref[0] >= 0).all()


# --------------------------------------------------------------------------------------
# Prompt-lookup (n-gram) drafting [MS lookup_draft; SD Exercise 4 ngram_draft]
# --------------------------------------------------------------------------------------
def pin_ngram_worked_examples(orc):
    """Drafts worked by hand from the pages' definitions (tests/golden)."""
    with open(os.path.join(GOLDEN, "ngram_draft_examples.txt")) as f:
        cases = [ln.rstrip("\n") for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(cases) >= 10
    for ln in cases:
        head, hist, want = (s.split() for s in ln.split("|"))
        n, k, pad = (int(x) for x in head)
        h = np.array([[int(x) for x in hist]], np.int32)
        drafts, count = orc.ngram_draft(h, [h.shape[1]], n, k, pad)
        want = [int(x) for x in want]
        assert count[0] == len(want) and list(drafts[0, :len(want)]) == want, (ln, drafts, count)
        assert (drafts[0, len(want):] == -1).all()


def pin_ngram_bruteforce(orc):
    """On random small-alphabet histories (ragged lengths, padded rows): the draft is the
    continuation of the latest earlier occurrence of the tail -- every later start in the
    search range fails to match -- and nothing is proposed without one (unless padded)."""
    rs = np.random.RandomState(61)
    for n, k, pad, alpha in ((1, 4, 1, 3), (1, 5, 0, 8), (2, 4, 0, 3), (3, 4, 0, 2), (4, 7, 1, 2)):
        B, T = 300, 40
        h = rs.randint(0, alpha, (B, T)).astype(np.int32)
        L = rs.randint(0, T + 1, B).astype(np.int32)
        drafts, count = orc.ngram_draft(h, L, n, k, pad)
        for b in range(B):
            seq = list(h[b, :L[b]])
            starts = [i for i in range(0, len(seq) - n) if seq[i:i + n] == seq[len(seq) - n:]]
            if starts:
                i = max(starts)
                cont = seq[i + n:i + n + k]
            else:
                cont = []
            if pad and seq:
                cont = cont + [seq[-1]] * (k - len(cont))
            assert count[b] == len(cont) and list(drafts[b, :len(cont)]) == cont, (b, seq)
            assert (drafts[b, len(cont):] == -1).all()


# --------------------------------------------------------------------------------------
# P10: row max / log-sum-exp against scipy's logsumexp [SD apply_temperature]
# --------------------------------------------------------------------------------------
def pin_row_stats(orc):
    rs = np.random.RandomState(14)
    for V, T in ((1, 1.0), (7, 0.7), (1000, 1.3), (4099, 0.5)):
        l = rs.normal(0, 3, (3, 4, V)).astype(np.float32)
        l[0, 1, : V // 2] = -np.inf
        m, lse, valid = orc.row_stats(l, T)
        ref = special.logsumexp(l.astype(np.float64) / T, axis=-1)
        assert valid.all()
        assert np.max(np.abs(lse - ref) / np.maximum(np.abs(ref), 1)) < 1e-13
        assert np.array_equal(m, np.max(l.astype(np.float64), -1) / T)
    l = np.zeros((1, 3, 4), np.float32)
    l[0, 0, 1] = np.nan
    l[0, 1, :] = -np.inf
    l[0, 2, 2] = np.inf
    _, _, valid = orc.row_stats(l, 1.0)
    assert not valid.any()


# --------------------------------------------------------------------------------------
# Typical acceptance [SD "Medusa" paragraph and the note on typical acceptance: accept a
# draft whose target probability exceeds a threshold scaled by the step's entropy].  The
# rule's form is a reading (threshold min(epsilon, delta exp(-H)); parity of the constants
# unpinned); these pins fix what does not depend on the constants.
# --------------------------------------------------------------------------------------
def _typical_case(rows, T=1.0):
    """Target [1, len(rows), V] from logit rows; draft i = the argmax of row i (finite)."""
    t = np.stack([np.asarray(r, np.float64) for r in rows])[None].astype(np.float32)
    x = np.array([[int(np.argmax(r)) for r in rows[:-1]]], np.int32)
    return t, x


def pin_typical_entropy(orc):
    """The entropy the rule reads is the textbook one: ln V for a uniform row, 0 for a
    one-hot row, scipy.stats.entropy (natural log) of softmax(t / T) for random and
    partly masked rows.  epsilon = 0 makes the threshold 0, so every row is read."""
    V, T = 37, 0.8
    rs = np.random.RandomState(71)
    hot = np.full(V, -np.inf)
    hot[5] = 0.0
    masked = rs.randn(V) * 2
    masked[rs.rand(V) < 0.4] = -np.inf
    masked[3] = 1.0
    rows = [np.zeros(V), hot, rs.randn(V) * 3, masked, rs.randn(V)]
    t, x = _typical_case(rows, T)
    acc, out, flags, H = orc.verify_typical(t, x, T, 0.0, 0.3, 5, 0)
    assert acc[0] == len(rows) - 1, acc
    want = [np.log(V), 0.0] + [stats.entropy(_softmax(t[0, i], T)) for i in range(2, len(rows))]
    assert np.allclose(H[0], want, rtol=1e-12, atol=1e-12), (H[0], want)


def pin_typical_threshold_closed_forms(orc):
    """Uniform rows (p(x) = 1/V, H = ln V, threshold min(epsilon, delta / V)) and one-hot
    rows (p(x) = 1, H = 0, threshold min(epsilon, delta)): the first draft is accepted
    exactly on the side of each closed-form threshold; equality rejects (strict >)."""
    V, G = 40, 3
    uni = [np.zeros(V)] * (G + 1)
    t, x = _typical_case(uni)
    for eps, delta, accept in ((1.0, 0.99, True), (1.0, 1.01, False), (0.99 / V, 100.0, True),
                               (1.01 / V, 100.0, False)):
        acc, _, _, _ = orc.verify_typical(t, x, 1.0, eps, delta, 3, 0)
        assert (acc[0] == G) == accept and (acc[0] == 0) == (not accept), (eps, delta, acc)
    hot = np.full(V, -np.inf)
    hot[7] = 2.0
    t, x = _typical_case([hot] * (G + 1))
    for eps, delta, want in ((1.0, 1.0, 0), (0.5, 2.0, G), (2.0, 0.999, G), (1.0, 5.0, 0)):
        acc, out, _, _ = orc.verify_typical(t, x, 1.0, eps, delta, 3, 0)
        assert acc[0] == want and out[0, want] == 7, (eps, delta, acc, out)


def pin_typical_zero_threshold(orc):
    """epsilon = 0: a draft is accepted exactly when its logit is finite, so the prefix
    ends at the first draft the target rules out (a -inf logit)."""
    rs = np.random.RandomState(72)
    B, G, V = 400, 5, 23
    t = (rs.randn(B, G + 1, V) * 2).astype(np.float32)
    t[rs.rand(B, G + 1, V) < 0.3] = -np.inf
    t[:, :, 0] = 0.0  # every row stays a distribution
    x = rs.randint(0, V, (B, G)).astype(np.int32)
    acc, out, _, _ = orc.verify_typical(t, x, 1.0, 0.0, 0.5, 9, 0)
    for b in range(B):
        dead = [i for i in range(G) if t[b, i, x[b, i]] == -np.inf]
        k = dead[0] if dead else G
        assert acc[b] == k and list(out[b, :k]) == list(x[b, :k]), (b, acc[b], k)
        assert np.isfinite(t[b, k, out[b, k]]) and (out[b, k + 1:] == -1).all()


def pin_typical_draw_law(orc, trials=200_000, V=5, G=2, T=0.9, alpha=1e-3):
    """The token at the stop is drawn from p at the stop row: with every draft rejected
    (threshold min(2, 1e30 e^-H) = 2 > any probability) the first token's law is p_0; with
    every draft accepted (epsilon = 0, finite rows) the bonus's law is p_gamma (chi-squared
    over Philox draws)."""
    t, _ = _chi2_rows(V, G)
    rows = np.ascontiguousarray(np.broadcast_to(t[:G + 1][None], (trials, G + 1, V)))
    x = np.zeros((trials, G), np.int32)
    for eps, delta, k in ((2.0, 1e30, 0), (0.0, 0.5, G)):
        acc, out, _, _ = orc.verify_typical(rows, x, T, eps, delta, 0xBEEF, 0)
        assert (acc == k).all(), (eps, np.unique(acc))
        obs = np.bincount(out[:, k], minlength=V)
        _, pv = stats.chisquare(obs, _softmax(t[k], T) * trials)
        assert pv > alpha, (k, pv, obs / trials)


def pin_typical_lazy_rows(orc):
    """Rows are read up to the stop: a NaN row past it leaves the result unchanged, a NaN
    row the rule reads, or a draft token out of range, gives -1."""
    rs = np.random.RandomState(73)
    G, V = 4, 30
    t = (rs.randn(1, G + 1, V) * 2).astype(np.float32)
    x = np.zeros((1, G), np.int32)
    t[0, 0, 0] = -np.inf  # the first draft is ruled out: the stop is row 0
    acc, out, _, _ = orc.verify_typical(t, x, 1.0, 0.0, 0.3, 4, 0)
    assert acc[0] == 0
    t2 = t.copy()
    t2[0, 2, 5] = np.nan
    acc2, out2, _, H2 = orc.verify_typical(t2, x, 1.0, 0.0, 0.3, 4, 0)
    assert acc2[0] == 0 and (out2 == out).all() and np.isnan(H2[0, 1:]).all()
    t3 = t.copy()
    t3[0, 0, 9] = np.nan
    acc3, out3, _, _ = orc.verify_typical(t3, x, 1.0, 0.0, 0.3, 4, 0)
    assert acc3[0] == -1 and (out3 == -1).all()
    acc4, _, _, _ = orc.verify_typical(t, np.full((1, G), V, np.int32), 1.0, 0.0, 0.3, 4, 0)
    assert acc4[0] == -1


ALL_PINS = [
    pin_philox_kat, pin_uniform_definition, pin_bruteforce_lossless, pin_chi2_sampler,
    pin_identical_rows_accept_all, pin_one_hot_equals_greedy, pin_one_hot_draft_accept_prob,
    pin_round_invariants, pin_worked_example, pin_acceptance_rate, pin_greedy_textbook,
    pin_tree_printed_depths, pin_chain_tree_equals_greedy, pin_tree_bruteforce, pin_row_stats,
    pin_tree_sample_lossless, pin_tree_sample_chi2, pin_chain_tree_sample_equals_chain,
    pin_tree_sample_invariants, pin_ngram_worked_examples, pin_ngram_bruteforce,
    pin_typical_entropy, pin_typical_threshold_closed_forms, pin_typical_zero_threshold,
    pin_typical_draw_law, pin_typical_lazy_rows,
]
