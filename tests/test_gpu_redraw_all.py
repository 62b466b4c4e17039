"""Every marked sequence is redone: inputs built so that EVERY sequence's decision sits about
1e-9 (relative) from its boundary -- far inside the fp32 windows, far outside the
double-float error -- so every sequence is marked, and far more per call than any fixed
number of re-draw slots.  Each case must match the oracle on every sequence, with the
status words reporting marked == redone and no timeout.

The rule that decides those sequences: "7.6 Speculative Decoding: Draft Models, Medusa,
EAGLE & Lookahead", "The rule" (accept iff u q(x) < p(x); the residual (p - q)+; the bonus
from p) and "Extending to a chain of gamma draft tokens"; the inverse-CDF draw of reading R3.

The logits are fp32 so that a row can be tuned finely: a row's boundary is placed by a
small "tuning" token whose mass sets the row's total.  Uniforms come from the oracle's
Philox (pinned to the SC'11 known-answer vectors), never from the CUDA path.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verify_spec_gb300 as sv
from speculative_decoding_verify_spec_gb300 import binding
from parity_util import oracle_sample, oracle_tree_sample

pytestmark = pytest.mark.gpu
DEV = "cuda"
ETA = 1e-9          # the planted margin, relative to the row's total
NEG = -np.inf


def f32(x) -> float:
    return float(np.float32(x))


def tuned_draw_row(V, u, rng, exclude=()):
    """fp32 logits of one row whose inverse-CDF draw with uniform u lands ETA (relative,
    either side at random) from the boundary after its first token: tokens j0 < j1 < j2
    carry weights 1, ~(1/u - 1)(1 - 1e-5) and the rest of the mass (the tuning token); a
    few background tokens at -30 sit before j0; every other logit is -inf.  Positions in
    `exclude` are left alone (the caller sets them).  Returns (row, (j0, j1, j2))."""
    row = np.full(V, NEG, np.float32)
    free = np.setdiff1d(np.arange(V), np.asarray(exclude, dtype=np.int64))
    j0, j1, j2 = np.sort(rng.choice(free[(free > 8) & (free < V - 8)], 3, replace=False))
    bg = rng.choice(free[free < j0], min(4, int((free < j0).sum())), replace=False)
    row[bg] = -30.0
    row[j0] = 0.0
    c_j0 = float(np.exp(row[:j0 + 1].astype(np.float64)).sum())  # the prefix through j0
    s = rng.choice([-1.0, 1.0])
    R = c_j0 / (u - s * ETA)           # u R - C_j0 = s ETA R
    rest = R - c_j0
    t1 = np.float32(np.log(rest * (1 - 1e-5)))
    row[j1] = t1
    c = rest - float(np.exp(np.float64(t1)))
    assert c > 0
    row[j2] = np.float32(np.log(c))
    return row, (int(j0), int(j1), int(j2))


def tuned_accept_rows(V, u0, x, rng):
    """fp32 (target, draft) logits of one position whose accept test u0 q(x) < p(x) sits ETA
    (relative, either side) from its threshold: the draft row N(0, 1); the target row the
    same except at x (shifted so p(x) / q(x) ~ u0) and at one tuning token j2 whose draft
    logit is -inf."""
    d = rng.standard_normal(V).astype(np.float32)
    j2 = int(rng.choice(np.setdiff1d(np.arange(V), [x])))
    d[j2] = NEG
    t = d.copy()
    s = rng.choice([-1.0, 1.0])
    rho = u0 * (1 + s * ETA)  # the planted p(x) / q(x)
    ed = np.exp(d.astype(np.float64))
    Sd, ex = float(ed.sum()), float(ed[x])
    S0 = Sd - ex
    tx0 = np.log(rho * ex * S0 / (Sd - rho * ex))
    tx = np.float32(tx0 + 1e-5)
    if float(tx) <= tx0:
        tx = np.nextafter(tx, np.float32(np.inf))
    t[x] = tx
    etx = float(np.exp(np.float64(tx)))
    c = etx * Sd / (ex * rho) - S0 - etx  # S_t = S0 + e^tx + c makes p / q = rho
    assert c > 0
    t[j2] = np.float32(np.log(c))
    return t, d


def chain_batch(B, V, seed, offset, rng, kind_of=lambda b: b % 3):
    """gamma = 2, T = 1, fp32.  Sequence b of kind kind_of(b) (b % 3 by default):
      0  accepted drafts (target = draft on rows 0, 1), the bonus draw on row 2 tuned;
      1  row 0 rejected for certain (q one-hot on x0, p(x0) ~ e^-40), the residual draw on
         row 0 tuned (the residual is p without x0);
      2  the accept test of row 0 tuned (then row 1 accepted, a plain bonus draw)."""
    G = 2
    t = rng.standard_normal((B, G + 1, V)).astype(np.float32)
    d = t[:, :G].copy()
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    for b in range(B):
        kind = kind_of(b)
        if kind == 0:
            t[b, G], _ = tuned_draw_row(V, oracle.uniform(seed, offset, b, G, 1), rng)
        elif kind == 1:
            row, (_, _, j2) = tuned_draw_row(V, oracle.uniform(seed, offset, b, 0, 1), rng)
            x0 = int(rng.integers(j2 + 1, V))
            row[x0] = -40.0
            t[b, 0] = row
            d[b, 0] = NEG
            d[b, 0, x0] = 0.0
            x[b, 0] = x0
        else:
            t[b, 0], d[b, 0] = tuned_accept_rows(V, oracle.uniform(seed, offset, b, 0, 0), int(x[b, 0]), rng)
    return t, d, x


def target_only_batch(B, V, seed, offset, rng):
    """gamma = 2, T = 1, fp32, for typical acceptance and one-hot sampling: draft x0 has
    probability 0 (a -inf logit), so both rules stop at row 0 and draw from p_0 (p_0 without
    x0, which has no mass anyway); the draw on row 0 is tuned."""
    G = 2
    t = rng.standard_normal((B, G + 1, V)).astype(np.float32)
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    for b in range(B):
        row, (j0, j1, j2) = tuned_draw_row(V, oracle.uniform(seed, offset, b, 0, 1), rng)
        x0 = int(rng.choice(np.nonzero(np.isneginf(row))[0]))  # a token with no mass
        row[x0] = NEG
        t[b, 0] = row
        x[b, 0] = x0
    return t, x


SEED, OFFSET = 0x5EED + 11, 7
B, V = 576, 3000  # 192 sequences of each kind; V not a multiple of any tile


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def check_status(ws, mode, rows, want_min):
    marked, redone, status, marks = binding.call_status(ws, mode, B, rows, V, binding.FP32)
    assert status == 0
    assert redone == marked == int((marks != 0).sum())
    assert marked >= want_min, (marked, want_min)
    return marked


@pytest.fixture(scope="module")
def chain():
    rng = np.random.default_rng(2024)
    t, d, x = chain_batch(B, V, SEED, OFFSET, rng)
    o_acc, o_out, o_flags = oracle_sample(t, d, x, 1.0, SEED, OFFSET)
    assert (o_flags != 0).mean() > 0.95  # the oracle sees every planted margin as near
    return t, d, x, o_acc, o_out


def test_chain_sampling_redoes_every_marked_sequence(chain):
    t, d, x, o_acc, o_out = chain
    ws = torch.empty(sv.spec_verify_workspace_size(binding.MODE_SAMPLE, B, 2, V, binding.FP32),
                     dtype=torch.uint8, device=DEV)
    for rep in range(2):  # twice: the lists and counters start again every call
        acc, out = sv.spec_verify_sample(cuda(t), cuda(d), cuda(x), 1.0, SEED, OFFSET, workspace=ws)
        assert (acc.cpu().numpy() == o_acc).all()
        assert (out.cpu().numpy() == o_out).all()
        check_status(ws, binding.MODE_SAMPLE, 2, int(0.95 * B))


def test_lazy_and_tree_sampling_rewalk_every_marked_sequence(chain):
    t, d, x, o_acc, o_out = chain
    ws = torch.empty(sv.spec_verify_workspace_size(binding.MODE_SAMPLE_LAZY, B, 2, V, binding.FP32),
                     dtype=torch.uint8, device=DEV)
    acc, out = sv.spec_verify_sample_lazy(cuda(t), cuda(d), cuda(x), 1.0, SEED, OFFSET, workspace=ws)
    assert (acc.cpu().numpy() == o_acc).all()
    assert (out.cpu().numpy() == o_out).all()
    check_status(ws, binding.MODE_SAMPLE_LAZY, 2, 64)
    # the same rounds as a chain-shaped tree (node v's parent is v - 1, its token x_{v-1})
    N = 3
    parent = np.array([-1, 0, 1], np.int32)
    tokens = np.concatenate([np.zeros((B, 1), np.int32), x], axis=1)
    dt = np.concatenate([d, np.zeros((B, 1, V), np.float32)], axis=1)  # the leaf's draft row is never read
    ot = oracle_tree_sample(t, dt, parent, tokens, 2, 1.0, SEED, OFFSET)
    assert (ot[0] == o_acc).all() and (ot[1] == o_out).all()
    ws2 = torch.empty(sv.spec_verify_workspace_size(binding.MODE_TREE_SAMPLE, B, N, V, binding.FP32),
                      dtype=torch.uint8, device=DEV)
    acc, out, path = sv.spec_verify_tree_sample(cuda(t), cuda(dt), cuda(parent), cuda(tokens), 2, 1.0, SEED,
                                                OFFSET, workspace=ws2)
    assert (acc.cpu().numpy() == ot[0]).all()
    assert (out.cpu().numpy() == ot[1]).all()
    assert (path.cpu().numpy() == ot[2]).all()
    check_status(ws2, binding.MODE_TREE_SAMPLE, N, 64)


def test_target_only_rules_redraw_every_marked_sequence():
    rng = np.random.default_rng(77)
    t, x = target_only_batch(B, V, SEED, OFFSET, rng)
    orc = oracle.default()
    eps, dlt = 0.1, 0.3
    o_acc, o_out, o_flags, _ = orc.verify_typical(t, x, 1.0, eps, dlt, SEED, OFFSET)
    assert (o_acc == 0).all() and (o_flags != 0).mean() > 0.95
    ws = torch.empty(sv.spec_verify_workspace_size(binding.MODE_TYPICAL, B, 2, V, binding.FP32),
                     dtype=torch.uint8, device=DEV)
    acc, out = sv.spec_verify_typical(cuda(t), cuda(x), 1.0, eps, dlt, SEED, OFFSET, workspace=ws)
    assert (acc.cpu().numpy() == o_acc).all()
    assert (out.cpu().numpy() == o_out).all()
    check_status(ws, binding.MODE_TYPICAL, 2, int(0.95 * B))
    # one-hot q on x: p(x0) = 0 rejects at row 0; the residual p_0 without x0 is p_0
    d1 = np.full_like(t[:, :2], NEG)
    np.put_along_axis(d1, x[:, :, None].astype(np.int64), 0.0, axis=2)
    s_acc, s_out, _ = oracle_sample(t, d1, x, 1.0, SEED, OFFSET)
    assert (s_acc == 0).all() and (s_out == o_out).all()
    ws2 = torch.empty(sv.spec_verify_workspace_size(binding.MODE_SAMPLE_ONEHOT, B, 2, V, binding.FP32),
                      dtype=torch.uint8, device=DEV)
    acc, out = sv.spec_verify_sample_onehot(cuda(t), cuda(x), 1.0, SEED, OFFSET, workspace=ws2)
    assert (acc.cpu().numpy() == s_acc).all()
    assert (out.cpu().numpy() == s_out).all()
    check_status(ws2, binding.MODE_SAMPLE_ONEHOT, 2, int(0.95 * B))


def test_single_sequence_call_redoes_its_marked_sequence():
    """B = 1 with few tiles runs as one kernel of one CTA (its stages and the re-draw in
    one launch): each kind of near-boundary decision, planted for sequence 0, is marked,
    redone and equals the oracle; the four-kernel path on a batch of two agrees on it."""
    rng = np.random.default_rng(77)
    for kind in (0, 1, 2):
        for rep in range(3):
            off = OFFSET + 100 * kind + rep
            t, d, x = chain_batch(2, V, SEED, off, rng, kind_of=lambda b: kind)
            o_acc, o_out, _ = oracle_sample(t[:1], d[:1], x[:1], 1.0, SEED, off)
            ws = torch.empty(sv.spec_verify_workspace_size(binding.MODE_SAMPLE, 1, 2, V, binding.FP32),
                             dtype=torch.uint8, device=DEV)
            acc, out = sv.spec_verify_sample(cuda(t[:1]), cuda(d[:1]), cuda(x[:1]), 1.0, SEED, off, workspace=ws)
            assert (acc.cpu().numpy() == o_acc).all() and (out.cpu().numpy() == o_out).all(), (kind, rep)
            marked, redone, status, marks = binding.call_status(ws, binding.MODE_SAMPLE, 1, 2, V, binding.FP32)
            assert status == 0 and marked == redone == 1 and marks[0] != 0, (kind, rep, marked, redone)
            acc2, out2 = sv.spec_verify_sample(cuda(t), cuda(d), cuda(x), 1.0, SEED, off)
            assert torch.equal(acc2[:1], acc) and torch.equal(out2[:1], out)
