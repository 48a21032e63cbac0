"""Pins for the fp64 CPU oracle: the pages' worked examples, closed forms,
invariants and finite differences. None of these compares the oracle with a
retyped copy of itself.

Sources:
  * tutorial page "research-attention", section 03: single-row demo (scores
    [1,2,0,3], tile size 2) with its printed state after the first tile and its
    printed result;
  * LLaMA 3 notes page "Flash Attention", the 4-token d=2 example (Q=K=V=X,
    scale 1/sqrt(2)) with its printed softmax row, denominator, numerators and
    outputs of tokens 0 and 1;
  * tutorial section 02 (the recurrence, "one division at the end") and
    section 04 (L = m + log l);
  * blog page "Flash Attention 原理与实现", section "Backward 的 Tiling 策略"
    (the gradient products), checked by central finite differences.
"""
import json
import math
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from oracle.online_softmax import tiled_row

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- worked examples

def test_tutorial_single_row_full_attention():
    """The demo row as full attention: q=[1,0], k_j=[s_j,0], scale 1, so every
    query row has scores [1,2,0,3]; the page prints [0.795176, 2.200684]."""
    g = _golden("tutorial_single_row.json")
    s = np.array(g["scores"])
    N = len(s)
    q = np.tile([1.0, 0.0], (N, 1))[None, None]
    k = np.stack([s, np.zeros(N)], axis=1)[None, None]
    v = np.array(g["values"])[None, None]
    o, lse = oracle.attention_fwd(q, k, v, scale=1.0, causal=False)
    half_ulp = 0.5 * 10.0 ** (-g["printed_output_decimals"])
    for i in range(N):
        assert np.max(np.abs(o[0, 0, i] - np.array(g["printed_output"]))) <= half_ulp
    # L is the log of the one-shot denominator: sum_j e^{s_j}
    assert abs(lse[0, 0, 0] - math.log(sum(math.exp(x) for x in s))) < 1e-12


def test_tutorial_recurrence_states_and_result():
    g = _golden("tutorial_single_row.json")
    o, L, states = tiled_row(g["scores"], g["values"], g["tile"])
    half_ulp = 0.5 * 10.0 ** (-g["state_decimals"])
    st = states[0]
    assert st.m == g["state_after_first_tile"]["m"]
    assert abs(st.l - g["state_after_first_tile"]["l"]) <= half_ulp
    assert np.max(np.abs(np.array(st.u) - g["state_after_first_tile"]["u"])) <= half_ulp
    assert np.max(np.abs(np.array(o) - g["printed_output"])) <= half_ulp
    # the page's own check: tiled vs one-shot within 1e-12
    s = np.array(g["scores"])
    q = np.tile([1.0, 0.0], (4, 1))[None, None]
    k = np.stack([s, np.zeros(4)], axis=1)[None, None]
    o_ref, lse_ref = oracle.attention_fwd(q, k, np.array(g["values"])[None, None], 1.0)
    assert np.max(np.abs(np.array(o) - o_ref[0, 0, 0])) < g["tiled_vs_one_shot_bound"]
    assert abs(L - lse_ref[0, 0, 0]) < 1e-12


def test_llama_notes_four_tokens():
    g = _golden("llama_notes_four_tokens.json")
    X = np.array(g["X"])
    scale = 1.0 / math.sqrt(X.shape[1])
    x4 = X[None, None]
    o, lse = oracle.attention_fwd(x4, x4, x4, scale)
    o, lse = o[0, 0], lse[0, 0]
    assert np.max(np.abs(o[0] - g["output_token0"])) <= g["tol_outputs"]
    assert np.max(np.abs(o[1] - g["output_token1"])) <= g["tol_outputs"]
    P = oracle.softmax_probs(X, X, scale)
    assert np.max(np.abs(P[0] - g["softmax_row0"])) <= g["tol_softmax"]
    # the page's denominator and numerators carry no max shift: den = e^L, num = O * den
    den0 = math.exp(lse[0])
    assert abs(den0 - g["denominator_row0"]) <= g["tol_sums"]
    assert np.max(np.abs(o[0] * den0 - g["numerators_row0"])) <= g["tol_sums"]
    den1 = math.exp(lse[1])
    assert np.max(np.abs(o[1] * den1 - g["numerators_row1"])) <= g["tol_sums"]
    # "symmetric queries give symmetric outputs" (summary of the same section)
    assert np.max(np.abs(o[1] - o[0][::-1])) < 1e-12


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("seed", [0, 1])
def test_every_tile_size_matches_one_shot(seed):
    """Tutorial section 03: tiling yields the same exact attention for any block size."""
    r = _rng(seed)
    N, d = 13, 3
    q = r.standard_normal((1, 1, N, d))
    k = r.standard_normal((1, 1, N, d)) * 3.0
    v = r.standard_normal((1, 1, N, d))
    for causal in (False, True):
        o_ref, lse_ref = oracle.attention_fwd(q, k, v, 0.7, causal)
        for i in range(N):
            s = [0.7 * float(np.dot(q[0, 0, i], k[0, 0, j])) if (not causal or j <= i) else -math.inf
                 for j in range(N)]
            for tile in range(1, N + 1):
                o_t, L_t, _ = tiled_row(s, v[0, 0].tolist(), tile)
                assert np.max(np.abs(np.array(o_t) - o_ref[0, 0, i])) < 1e-12
                assert abs(L_t - lse_ref[0, 0, i]) < 1e-12


def test_fully_masked_leading_tile_keeps_state():
    """A tile that is all -inf before any finite score leaves (m, l, u) at its start."""
    o, L, states = tiled_row([-math.inf, -math.inf, 0.5, 1.5], [[1, 0], [0, 1], [2, 0], [0, 2]], 2)
    assert states[0].m == -math.inf and states[0].l == 0.0 and states[0].u == [0.0, 0.0]
    w = np.exp(np.array([0.5, 1.5]) - 1.5)
    ref = (w[0] * np.array([2, 0]) + w[1] * np.array([0, 2])) / w.sum()
    assert np.max(np.abs(np.array(o) - ref)) < 1e-15


def test_probability_rows_sum_to_one_and_mask():
    r = _rng(3)
    N, d = 37, 8
    q, k = r.standard_normal((N, d)), r.standard_normal((N, d))
    for causal in (False, True):
        P = oracle.softmax_probs(q, k, 0.4, causal)
        assert np.max(np.abs(P.sum(axis=1) - 1.0)) < 1e-12
        assert (P >= 0).all()
        if causal:
            assert np.all(P[np.triu_indices(N, 1)] == 0.0)
            assert np.all(P[np.tril_indices(N)] > 0.0)


def test_key_permutation_permutes_probability_columns_only():
    r = _rng(4)
    N, d = 20, 5
    q, k, v = (r.standard_normal((1, 1, N, d)) for _ in range(3))
    perm = r.permutation(N)
    o1, l1 = oracle.attention_fwd(q, k, v, 0.5)
    o2, l2 = oracle.attention_fwd(q, k[:, :, perm], v[:, :, perm], 0.5)
    assert np.max(np.abs(o1 - o2)) < 1e-12 and np.max(np.abs(l1 - l2)) < 1e-12
    P1 = oracle.softmax_probs(q[0, 0], k[0, 0], 0.5)
    P2 = oracle.softmax_probs(q[0, 0], k[0, 0, perm], 0.5)
    assert np.max(np.abs(P1[:, perm] - P2)) < 1e-15


def test_batch_and_head_independence():
    """Heads never mix: each (b, h) slice equals the same slice computed alone."""
    r = _rng(5)
    q, k, v, dO = (r.standard_normal((2, 3, 9, 4)) for _ in range(4))
    o, lse = oracle.attention_fwd(q, k, v, 0.6, True)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dO, 0.6, True)
    for b in range(2):
        for h in range(3):
            sl = (slice(b, b + 1), slice(h, h + 1))
            o1, l1 = oracle.attention_fwd(q[sl], k[sl], v[sl], 0.6, True)
            g1 = oracle.attention_bwd(q[sl], k[sl], v[sl], dO[sl], 0.6, True)
            assert np.array_equal(o1[0, 0], o[b, h]) and np.array_equal(l1[0, 0], lse[b, h])
            for a, full in zip(g1, (dq, dk, dv)):
                assert np.array_equal(a[0, 0], full[b, h])


# ---------------------------------------------------------------- closed forms

def test_single_key_returns_value():
    r = _rng(6)
    q, k, v = (r.standard_normal((1, 2, 1, 6)) for _ in range(3))
    o, lse = oracle.attention_fwd(q, k, v, 0.3)
    assert np.array_equal(o, v)
    assert np.max(np.abs(lse - 0.3 * np.sum(q * k, axis=-1))) < 1e-15


def test_causal_first_row_sees_only_itself():
    r = _rng(7)
    q, k, v = (r.standard_normal((1, 1, 11, 4)) for _ in range(3))
    o, lse = oracle.attention_fwd(q, k, v, 0.9, True)
    assert np.array_equal(o[0, 0, 0], v[0, 0, 0])
    assert abs(lse[0, 0, 0] - 0.9 * np.dot(q[0, 0, 0], k[0, 0, 0])) < 1e-15


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_average_values(causal):
    r = _rng(8)
    N, d = 17, 3
    q = np.zeros((1, 1, N, d))
    k, v, dO = (r.standard_normal((1, 1, N, d)) for _ in range(3))
    o, lse = oracle.attention_fwd(q, k, v, 1.0, causal)
    _, _, dv = oracle.attention_bwd(q, k, v, dO, 1.0, causal)
    for i in range(N):
        n = i + 1 if causal else N
        assert np.max(np.abs(o[0, 0, i] - v[0, 0, :n].mean(axis=0))) < 1e-14
        assert abs(lse[0, 0, i] - math.log(n)) < 1e-14
    for j in range(N):
        if causal:
            ref = sum(dO[0, 0, i] / (i + 1) for i in range(j, N))
        else:
            ref = dO[0, 0].sum(axis=0) / N
        assert np.max(np.abs(dv[0, 0, j] - ref)) < 1e-13


def test_constant_score_shift_moves_lse_only():
    """Adding c to every score of a row: P and O unchanged, L grows by c
    (tutorial section 02: a common base leaves the ratio unchanged)."""
    r = _rng(9)
    N, d, c = 12, 4, 2.5
    q, k, v = (r.standard_normal((1, 1, N, d)) for _ in range(3))
    scale = 0.5
    q2 = np.concatenate([q, np.full((1, 1, N, 1), c / scale)], axis=-1)
    k2 = np.concatenate([k, np.ones((1, 1, N, 1))], axis=-1)
    for causal in (False, True):
        o1, l1 = oracle.attention_fwd(q, k, v, scale, causal)
        v2 = np.concatenate([v, np.zeros((1, 1, N, 1))], axis=-1)
        o2, l2 = oracle.attention_fwd(q2, k2, v2, scale, causal)
        assert np.max(np.abs(o1 - o2[..., :d])) < 1e-13
        assert np.max(np.abs(l2 - l1 - c)) < 1e-12


def test_large_scores_stay_finite():
    """Scores near 1e4: max subtraction keeps every exp argument <= 0 (blog,
    pitfalls item 4; tutorial section 02)."""
    r = _rng(10)
    q = r.standard_normal((1, 1, 16, 4)) * 100
    k = r.standard_normal((1, 1, 16, 4)) * 100
    v, dO = r.standard_normal((1, 1, 16, 4)), r.standard_normal((1, 1, 16, 4))
    o, lse = oracle.attention_fwd(q, k, v, 1.0, False)
    g = oracle.attention_bwd(q, k, v, dO, 1.0, False)
    assert np.abs(lse).max() > 1e3
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert all(np.isfinite(x).all() for x in g)
    # every output is a convex combination of value rows
    assert (o <= v.max(axis=2, keepdims=True) + 1e-12).all()
    assert (o >= v.min(axis=2, keepdims=True) - 1e-12).all()


# ---------------------------------------------------------------- backward

def _loss(q, k, v, dO, scale, causal):
    o, _ = oracle.attention_fwd(q, k, v, scale, causal)
    return float(np.sum(o * dO))


@pytest.mark.parametrize("N", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("d", [1, 2, 4])
@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_central_differences(N, d, causal):
    r = _rng(100 + 10 * N + d)
    q, k, v, dO = (r.standard_normal((1, 1, N, d)) for _ in range(4))
    scale = 0.8
    grads = oracle.attention_bwd(q, k, v, dO, scale, causal)
    h = 1e-6
    for which, g in zip(range(3), grads):
        num = np.zeros_like(g)
        base = [q, k, v]
        for idx in np.ndindex(g.shape):
            plus = [x.copy() for x in base]
            minus = [x.copy() for x in base]
            plus[which][idx] += h
            minus[which][idx] -= h
            num[idx] = (_loss(*plus, dO, scale, causal) - _loss(*minus, dO, scale, causal)) / (2 * h)
        err = np.max(np.abs(num - g)) / max(1.0, np.max(np.abs(g)))
        assert err <= 1e-6, (which, err)


def test_gradient_sum_rules():
    """Softmax rows sum to 1, so each row of dS sums to 0: sum_j dK_j = 0 and
    sum_j dV_j = sum_i dO_i."""
    r = _rng(11)
    q, k, v, dO = (r.standard_normal((2, 2, 33, 6)) for _ in range(4))
    for causal in (False, True):
        _, dk, dv = oracle.attention_bwd(q, k, v, dO, 0.4, causal)
        assert np.max(np.abs(dk.sum(axis=2))) < 1e-12
        assert np.max(np.abs(dv.sum(axis=2) - dO.sum(axis=2))) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_against_torch_autograd_fp64(causal):
    """An independent route: torch's fp64 softmax/matmul and autograd."""
    torch = pytest.importorskip("torch")
    r = _rng(12)
    B, H, N, d = 2, 3, 40, 16
    q, k, v, dO = (r.standard_normal((B, H, N, d)) for _ in range(4))
    scale = 1 / math.sqrt(d)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    s = torch.matmul(tq, tk.transpose(-1, -2)) * scale
    if causal:
        s = s.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), float("-inf"))
    o_t = torch.matmul(torch.softmax(s, dim=-1), tv)
    o_t.backward(torch.tensor(dO))
    o, lse = oracle.attention_fwd(q, k, v, scale, causal)
    grads = oracle.attention_bwd(q, k, v, dO, scale, causal)
    assert np.max(np.abs(o - o_t.detach().numpy())) < 1e-12
    assert np.max(np.abs(lse - torch.logsumexp(s, dim=-1).detach().numpy())) < 1e-12
    for g, t in zip(grads, (tq, tk, tv)):
        assert np.max(np.abs(g - t.grad.numpy())) < 1e-11


# ---------------------------------------------------------------- Nq queries, Nk keys

def _square_with_prefix(r, Nq, Nk, d):
    """A square Nk x Nk problem whose last Nq query rows are the Nq x Nk one;
    the leading rows get zero upstream gradient, so they add nothing to dK, dV."""
    q = r.standard_normal((1, 2, Nq, d))
    k, v = (r.standard_normal((1, 2, Nk, d)) for _ in range(2))
    dO = r.standard_normal((1, 2, Nq, d))
    q_full = np.concatenate([r.standard_normal((1, 2, Nk - Nq, d)), q], axis=2)
    dO_full = np.concatenate([np.zeros((1, 2, Nk - Nq, d)), dO], axis=2)
    return q, k, v, dO, q_full, dO_full


@pytest.mark.parametrize("Nq,Nk", [(1, 9), (4, 9), (9, 9), (7, 20)])
def test_kv_bottom_right_causal_is_the_last_rows_of_the_square_problem(Nq, Nk):
    """Bottom-right alignment means exactly this: the Nq queries are the last
    Nq rows of the causal Nk x Nk problem on the same keys."""
    r = _rng(40 + Nq + Nk)
    q, k, v, dO, q_full, dO_full = _square_with_prefix(r, Nq, Nk, 3)
    o, lse = oracle.attention_fwd_kv(q, k, v, 0.7, True)
    o_sq, lse_sq = oracle.attention_fwd(q_full, k, v, 0.7, True)
    assert np.max(np.abs(o - o_sq[:, :, Nk - Nq:])) < 1e-13
    assert np.max(np.abs(lse - lse_sq[:, :, Nk - Nq:])) < 1e-13
    dq, dk, dv = oracle.attention_bwd_kv(q, k, v, dO, 0.7, True)
    dq_sq, dk_sq, dv_sq = oracle.attention_bwd(q_full, k, v, dO_full, 0.7, True)
    assert np.max(np.abs(dq - dq_sq[:, :, Nk - Nq:])) < 1e-12
    assert np.max(np.abs(dk - dk_sq)) < 1e-12 and np.max(np.abs(dv - dv_sq)) < 1e-12


def test_kv_single_query_decode_sees_every_key():
    r = _rng(41)
    q = r.standard_normal((1, 1, 1, 4))
    k, v = (r.standard_normal((1, 1, 13, 4)) for _ in range(2))
    oc, lc = oracle.attention_fwd_kv(q, k, v, 0.5, True)
    on, ln = oracle.attention_fwd_kv(q, k, v, 0.5, False)
    assert np.max(np.abs(oc - on)) < 1e-15 and np.max(np.abs(lc - ln)) < 1e-15
    s = 0.5 * (k[0, 0] @ q[0, 0, 0])
    w = np.exp(s - s.max())
    assert np.max(np.abs(on[0, 0, 0] - (w / w.sum()) @ v[0, 0])) < 1e-14


@pytest.mark.parametrize("Nq,Nk,causal", [(3, 5, True), (3, 5, False), (5, 3, False), (2, 2, True)])
def test_kv_gradients_match_central_differences(Nq, Nk, causal):
    r = _rng(200 + 10 * Nq + Nk)
    q = r.standard_normal((1, 1, Nq, 2))
    k, v = (r.standard_normal((1, 1, Nk, 2)) for _ in range(2))
    dO = r.standard_normal((1, 1, Nq, 2))
    grads = oracle.attention_bwd_kv(q, k, v, dO, 0.9, causal)
    h = 1e-6

    def loss(qq, kk, vv):
        return float(np.sum(oracle.attention_fwd_kv(qq, kk, vv, 0.9, causal)[0] * dO))

    for which, g in enumerate(grads):
        for idx in np.ndindex(g.shape):
            plus = [q.copy(), k.copy(), v.copy()]
            minus = [q.copy(), k.copy(), v.copy()]
            plus[which][idx] += h
            minus[which][idx] -= h
            num = (loss(*plus) - loss(*minus)) / (2 * h)
            assert abs(num - g[idx]) <= 1e-6 * max(1.0, np.abs(g).max())


# ---------------------------------------------------------------- sampled-row entry points

@pytest.mark.parametrize("causal", [False, True])
def test_sampled_rows_match_full(causal):
    r = _rng(13)
    N, d = 70, 8
    q, k, v, dO = (r.standard_normal((1, 1, N, d)) for _ in range(4))
    o, lse = oracle.attention_fwd(q, k, v, 0.35, causal)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dO, 0.35, causal)
    rows = [0, 1, 17, 42, 69]
    o_r, l_r, dq_r = oracle.query_rows(q[0, 0], k[0, 0], v[0, 0], dO[0, 0], rows, 0.35, causal)
    assert np.max(np.abs(o_r - o[0, 0, rows])) < 1e-13
    assert np.max(np.abs(l_r - lse[0, 0, rows])) < 1e-13
    assert np.max(np.abs(dq_r - dq[0, 0, rows])) < 1e-13
    keys = [0, 5, 33, 69]
    dk_r, dv_r = oracle.key_rows(q[0, 0], k[0, 0], v[0, 0], dO[0, 0], keys, 0.35, causal)
    assert np.max(np.abs(dk_r - dk[0, 0, keys])) < 1e-12
    assert np.max(np.abs(dv_r - dv[0, 0, keys])) < 1e-12


# ---------------------------------------------------------------- planted mistakes

MUTATIONS = {
    "dK without scale": ("dkj[c] += scale * dSij * qi[c];", "dkj[c] += dSij * qi[c];"),
    "dS with wrong sign of D": ("p[j] * (dPij - Di)", "p[j] * (dPij + Di)"),
    "dV transposed operand": ("dvj[c] += p[j] * doi[c];", "dvj[c] += p[j] * qi[c];"),
    "causal sees one key too many": ("const int n = i + 1 + (Nk - Nq);", "const int n = i + 2 + (Nk - Nq);"),
    "causal aligned top-left": ("const int n = i + 1 + (Nk - Nq);", "const int n = i + 1;"),
    "L without the max": ("return m + log(l);", "return log(l);"),
    "softmax not normalised": ("for (int j = 0; j < nk; ++j) p[j] /= l;", ""),
}


class _Lib:
    """ctypes view of a (possibly mutated) oracle build."""

    def __init__(self, so):
        import ctypes
        self.P = ctypes.c_void_p
        self.lib = ctypes.CDLL(so)
        self.lib.oracle_fwd.argtypes = [self.P] * 5 + [ctypes.c_int] * 4 + [ctypes.c_double, ctypes.c_int]
        self.lib.oracle_bwd.argtypes = [self.P] * 7 + [ctypes.c_int] * 4 + [ctypes.c_double, ctypes.c_int]
        self.lib.oracle_fwd_kv.argtypes = [self.P] * 5 + [ctypes.c_int] * 5 + [ctypes.c_double, ctypes.c_int]

    def fwd(self, q, k, v, scale, causal):
        B, H, N, d = q.shape
        o = np.empty_like(q); lse = np.empty(q.shape[:3])
        self.lib.oracle_fwd(*(x.ctypes.data_as(self.P) for x in (q, k, v, o, lse)), B, H, N, d, scale, int(causal))
        return o, lse

    def fwd_kv(self, q, k, v, scale, causal):
        B, H, Nq, d = q.shape
        Nk = k.shape[2]
        o = np.empty_like(q); lse = np.empty(q.shape[:3])
        self.lib.oracle_fwd_kv(*(x.ctypes.data_as(self.P) for x in (q, k, v, o, lse)), B, H, Nq, Nk, d, scale,
                               int(causal))
        return o, lse

    def bwd(self, q, k, v, dO, scale, causal):
        B, H, N, d = q.shape
        g = [np.empty_like(q) for _ in range(3)]
        self.lib.oracle_bwd(*(x.ctypes.data_as(self.P) for x in (q, k, v, dO, *g)), B, H, N, d, scale, int(causal))
        return g


def _pins_hold(lib):
    """The forward pins (tutorial row with its L, causal row 0) and the
    finite-difference pin of the backward, run against ``lib``."""
    g = _golden("tutorial_single_row.json")
    s = np.array(g["scores"])
    q = np.tile([1.0, 0.0], (4, 1))[None, None]
    k = np.stack([s, np.zeros(4)], axis=1)[None, None]
    o, lse = lib.fwd(q, k, np.array(g["values"])[None, None], 1.0, False)
    if np.max(np.abs(o[0, 0, 0] - g["printed_output"])) > 5e-7:
        return False
    if abs(lse[0, 0, 0] - math.log(np.exp(s).sum())) > 1e-12:
        return False
    r = _rng(14)
    q, k, v, dO = (r.standard_normal((1, 1, 5, 3)) for _ in range(4))
    o, lse = lib.fwd(q, k, v, 0.8, True)
    if not np.array_equal(o[0, 0, 0], v[0, 0, 0]) or abs(lse[0, 0, 0] - 0.8 * q[0, 0, 0] @ k[0, 0, 0]) > 1e-14:
        return False
    # bottom-right causal alignment: the kv problem is the tail of the square one
    qf = r.standard_normal((1, 1, 7, 3))
    kf, vf = r.standard_normal((1, 1, 7, 3)), r.standard_normal((1, 1, 7, 3))
    o_kv, _ = lib.fwd_kv(np.ascontiguousarray(qf[:, :, 4:]), kf, vf, 0.8, True)
    if np.max(np.abs(o_kv - lib.fwd(qf, kf, vf, 0.8, True)[0][:, :, 4:])) > 1e-12:
        return False
    h = 1e-6
    for causal in (False, True):
        grads = lib.bwd(q, k, v, dO, 0.8, causal)
        for which in range(3):
            for idx in np.ndindex(q.shape):
                plus = [q.copy(), k.copy(), v.copy()]
                minus = [q.copy(), k.copy(), v.copy()]
                plus[which][idx] += h
                minus[which][idx] -= h
                num = (np.sum(lib.fwd(*plus, 0.8, causal)[0] * dO)
                       - np.sum(lib.fwd(*minus, 0.8, causal)[0] * dO)) / (2 * h)
                if abs(num - grads[which][idx]) > 1e-6 * max(1.0, np.abs(grads[which]).max()):
                    return False
    return True


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_planted_mistakes_are_caught():
    """The pins hold for the real oracle, and each plausible slip planted in a
    copy of its source (a dropped factor, a wrong sign, a transposed operand, an
    off-by-one mask, a lost term) makes at least one of them fail."""
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert _pins_hold(_Lib(oracle.build()))
    with tempfile.TemporaryDirectory() as tmp:
        for n, (name, (old, new)) in enumerate(MUTATIONS.items()):
            assert old in src, name
            path = os.path.join(tmp, f"mutant{n}.c")
            with open(path, "w") as f:
                f.write(src.replace(old, new))
            so = path[:-2] + ".so"
            subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                                   path, "-o", so, "-lm"])
            assert not _pins_hold(_Lib(so)), name


# ---------------------------------------------------------------- dropout

def test_philox_known_answers():
    """The oracle's Philox4x32-10 reproduces the generator's published
    known-answer vectors (tests/golden/philox4x32_10_known_answers.json)."""
    g = _golden("philox4x32_10_known_answers.json")
    for vec in g["vectors"]:
        ctr = [int(x, 16) for x in vec["counter"]]
        key = [int(x, 16) for x in vec["key"]]
        want = [int(x, 16) for x in vec["output"]]
        assert list(oracle.philox4x32_10(ctr, key)) == want


def _curand():
    import ctypes
    import ctypes.util
    for name in ("libcurand.so", "libcurand.so.10", ctypes.util.find_library("curand"),
                 "/usr/local/cuda/lib64/libcurand.so"):
        if not name:
            continue
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    return None


def test_philox_matches_curand_host_generator():
    """cuRAND's host-side Philox4_32_10 generator (legacy ordering) emits, for
    seed s, the blocks f(counter = (0, 0, i, 0), key = (s_lo, s_hi)) for
    i = 0, 1, ...; an implementation independent of the oracle's."""
    import ctypes
    lib = _curand()
    if lib is None:
        pytest.skip("no cuRAND library")
    gen = ctypes.c_void_p()
    if lib.curandCreateGeneratorHost(ctypes.byref(gen), 161) != 0:  # CURAND_RNG_PSEUDO_PHILOX4_32_10
        pytest.skip("cuRAND host generator unavailable")
    try:
        assert lib.curandSetGeneratorOrdering(gen, 103) == 0  # CURAND_ORDERING_PSEUDO_LEGACY
        for seed in (0, 1, 0x0123456789ABCDEF, 0xFFFFFFFF00000001):
            assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
            assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(0)) == 0
            buf = (ctypes.c_uint * 64)()
            assert lib.curandGenerate(gen, buf, 64) == 0
            key = [seed & 0xFFFFFFFF, seed >> 32]
            for i in range(16):
                assert list(buf[4 * i:4 * i + 4]) == list(oracle.philox4x32_10([0, 0, i, 0], key)), (seed, i)
    finally:
        lib.curandDestroyGenerator(gen)


def test_dropout_mask_layout_and_rate():
    """The mask is the documented byte of the documented Philox call, does not
    depend on the problem's shape, and keeps about 1 - t/256 of the entries."""
    seed, off, t = 0x9E3779B97F4A7C15, 7, 77
    m = oracle.dropout_mask(seed, off, t, 5, 64, 96)
    for (i, j) in [(0, 0), (1, 2), (3, 95), (17, 40), (63, 63)]:
        w = oracle.philox4x32_10([j // 4, i // 4, 5, off], [seed & 0xFFFFFFFF, seed >> 32])
        assert m[i, j] == int(((int(w[i % 4]) >> (8 * (j % 4))) & 0xFF) >= t)
    assert np.array_equal(oracle.dropout_mask(seed, off, t, 5, 20, 30), m[:20, :30])
    big = np.stack([oracle.dropout_mask(seed, off, t, h, 256, 256) for h in range(4)])
    keep = 1.0 - t / 256.0
    sigma = math.sqrt(keep * (1 - keep) / big.size)
    assert abs(big.mean() - keep) < 5 * sigma
    assert not np.array_equal(big[0], big[1])                                  # heads differ
    assert not np.array_equal(oracle.dropout_mask(seed, off + 1, t, 5, 64, 96), m)  # offsets differ
    assert oracle.dropout_mask(seed, off, 0, 5, 64, 96).all()                  # t = 0 keeps everything


def test_dropout_with_zero_probability_is_plain_attention():
    r = _rng(40)
    q, dO = (r.standard_normal((1, 2, 9, 5)) for _ in range(2))
    k, v = (r.standard_normal((1, 2, 13, 5)) for _ in range(2))
    for causal in (False, True):
        o, lse = oracle.attention_fwd_kv(q, k, v, 0.7, causal)
        od, lsed = oracle.attention_fwd_dropout_kv(q, k, v, 0.7, causal, 11, 0, 0)
        assert np.max(np.abs(od - o)) < 1e-14 and np.max(np.abs(lsed - lse)) == 0
        g = oracle.attention_bwd_kv(q, k, v, dO, 0.7, causal)
        gd = oracle.attention_bwd_dropout_kv(q, k, v, dO, 0.7, causal, 11, 0, 0)
        for a, b in zip(g, gd):
            assert np.max(np.abs(a - b)) < 1e-13


def test_dropout_is_unbiased():
    """E[O] over masks equals the undropped O: the kept entries are scaled by
    256 / (256 - t). Mean over 2000 seeds, checked to 5 standard errors."""
    r = _rng(41)
    q, k, v = (r.standard_normal((1, 1, 3, 4)) for _ in range(3))
    o, _ = oracle.attention_fwd(q, k, v, 0.9, False)
    t = 64
    samples = np.stack([oracle.attention_fwd_dropout_kv(q, k, v, 0.9, False, s, 3, t)[0] for s in range(2000)])
    se = samples.std(axis=0) / math.sqrt(len(samples))
    assert np.all(np.abs(samples.mean(axis=0) - o) < 5 * se + 1e-12)


def test_dropout_backward_finite_differences():
    """With the mask fixed by (seed, offset, t), the dropout forward is a smooth
    function of Q, K, V; the oracle's dropout backward matches central
    differences of sum(O * dO), dropped entries' -P*D terms included."""
    r = _rng(42)
    q, dO = (r.standard_normal((1, 1, 6, 3)) for _ in range(2))
    k, v = (r.standard_normal((1, 1, 8, 3)) for _ in range(2))
    h, args = 1e-6, (0.8, True, 1234, 5, 90)
    assert oracle.dropout_mask(1234, 5, 90, 0, 6, 8).min() == 0  # some entries are dropped
    grads = oracle.attention_bwd_dropout_kv(q, k, v, dO, *args)
    for which, x in enumerate((q, k, v)):
        for idx in np.ndindex(x.shape):
            xs = [q.copy(), k.copy(), v.copy()]
            xs[which][idx] += h
            up = np.sum(oracle.attention_fwd_dropout_kv(*xs, *args)[0] * dO)
            xs[which][idx] -= 2 * h
            dn = np.sum(oracle.attention_fwd_dropout_kv(*xs, *args)[0] * dO)
            assert abs((up - dn) / (2 * h) - grads[which][idx]) < 1e-6 * max(1.0, np.abs(grads[which]).max())


DROPOUT_MUTATIONS = {
    "Philox multiplier swapped": ("(uint64_t)0xD2511F53u * c[0]", "(uint64_t)0xCD9E8D57u * c[0]"),
    "Philox key schedule dropped": ("    k[0] += 0x9E3779B9u;\n", ""),
    "kept entries not rescaled": ("o[c] += p[j] * inv_keep * vj[c];", "o[c] += p[j] * vj[c];"),
    "dropped entries lose -P D": ("const double dSij = p[j] * (dPij - Di);\n          const double pdij",
                                  "const double dSij = z ? p[j] * (dPij - Di) : 0.0;\n          const double pdij"),
    "dV with the undropped P": ("dvj[c] += pdij * doi[c];", "dvj[c] += p[j] * doi[c];"),
    "dP mask not applied": ("const double dPij = z ? dot(doi, vh + (size_t)j * d, d) * inv_keep : 0.0;",
                            "const double dPij = dot(doi, vh + (size_t)j * d, d) * inv_keep;"),
}


def _dropout_pins_hold(so):
    """The dropout pins above, run against a (possibly mutated) oracle build."""
    import ctypes
    P, i, dbl, u32, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_uint32, ctypes.c_uint64
    lib = ctypes.CDLL(so)
    lib.oracle_philox4x32_10.argtypes = [P, P, P]
    lib.oracle_fwd_dropout_kv.argtypes = [P, P, P, P, P, i, i, i, i, i, dbl, i, u64, u32, i]
    lib.oracle_bwd_dropout_kv.argtypes = [P, P, P, P, P, P, P, i, i, i, i, i, dbl, i, u64, u32, i]

    def fwd(q, k, v, scale, causal, seed, off, t):
        o = np.empty_like(q); lse = np.empty(q.shape[:3])
        lib.oracle_fwd_dropout_kv(*(x.ctypes.data_as(P) for x in (q, k, v, o, lse)), *q.shape[:3], k.shape[2],
                                  q.shape[3], scale, int(causal), seed, off, t)
        return o

    def bwd(q, k, v, dO, scale, causal, seed, off, t):
        g = [np.empty_like(q), np.empty_like(k), np.empty_like(v)]
        lib.oracle_bwd_dropout_kv(*(x.ctypes.data_as(P) for x in (q, k, v, dO, *g)), *q.shape[:3], k.shape[2],
                                  q.shape[3], scale, int(causal), seed, off, t)
        return g

    for vec in _golden("philox4x32_10_known_answers.json")["vectors"]:
        c = np.array([int(x, 16) for x in vec["counter"]], dtype=np.uint32)
        kk = np.array([int(x, 16) for x in vec["key"]], dtype=np.uint32)
        out = np.empty(4, dtype=np.uint32)
        lib.oracle_philox4x32_10(c.ctypes.data_as(P), kk.ctypes.data_as(P), out.ctypes.data_as(P))
        if list(out) != [int(x, 16) for x in vec["output"]]:
            return False
    r = _rng(41)
    q, k, v = (r.standard_normal((1, 1, 3, 4)) for _ in range(3))
    o, _ = oracle.attention_fwd(q, k, v, 0.9, False)
    samples = np.stack([fwd(q, k, v, 0.9, False, s, 3, 64) for s in range(2000)])
    if not np.all(np.abs(samples.mean(axis=0) - o) < 5 * samples.std(axis=0) / math.sqrt(2000) + 1e-12):
        return False
    r = _rng(42)
    q, dO = (r.standard_normal((1, 1, 6, 3)) for _ in range(2))
    k, v = (r.standard_normal((1, 1, 8, 3)) for _ in range(2))
    h, args = 1e-6, (0.8, True, 1234, 5, 90)
    grads = bwd(q, k, v, dO, *args)
    for which, x in enumerate((q, k, v)):
        for idx in np.ndindex(x.shape):
            xs = [q.copy(), k.copy(), v.copy()]
            xs[which][idx] += h
            up = np.sum(fwd(*xs, *args) * dO)
            xs[which][idx] -= 2 * h
            dn = np.sum(fwd(*xs, *args) * dO)
            if abs((up - dn) / (2 * h) - grads[which][idx]) > 1e-6 * max(1.0, np.abs(grads[which]).max()):
                return False
    return True


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_planted_dropout_mistakes_are_caught():
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert _dropout_pins_hold(oracle.build())
    with tempfile.TemporaryDirectory() as tmp:
        for n, (name, (old, new)) in enumerate(DROPOUT_MUTATIONS.items()):
            assert src.count(old) == 1, name
            path = os.path.join(tmp, f"dmutant{n}.c")
            with open(path, "w") as f:
                f.write(src.replace(old, new))
            so = path[:-2] + ".so"
            subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                                   path, "-o", so, "-lm"])
            assert not _dropout_pins_hold(so), name
