"""Pins for the backward oracle (`oracle/bptt.py`): what the definition of a gradient fixes.

The gradients are those of the scalar loss L = sum_t <d_o_t, o_t> + <d_S, S_T> through the
forward recurrence, so central finite differences of that forward pass pin every one of them
(the forward recurrence in numpy fp64, itself pinned against the C oracle and the pages by
`tests/test_oracle_pins.py`).  A closed form pins the decay-free additive case ("From
Attention to Learned Memory", sec. 1-2: o_t = (S0 + sum_{j<=t} k_j v_j^T)^T q_t), and planted
mistakes in the backward show that the pins catch them.
"""
import numpy as np
import pytest

import oracle
from oracle.bptt import backward_arrays, backward_seq


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def inputs(seed, T, dk, dv, per_channel):
    r = rng(seed)
    q = r.standard_normal((T, dk))
    k = r.standard_normal((T, dk))
    v = r.standard_normal((T, dv))
    beta = r.uniform(0.1, 0.9, T)
    g = -r.uniform(0.05, 0.6, (T, dk) if per_channel else T)
    S0 = r.standard_normal((dk, dv)) * 0.3
    do = r.standard_normal((T, dv))
    dS = r.standard_normal((dk, dv))
    return dict(q=q, k=k, v=v, beta=beta, g=g, S0=S0), do, dS


def loss(x, do, dS, **kw):
    o, S = oracle.recurrence_py(x["q"], x["k"], x["v"], x["beta"], x["g"], x["S0"], **kw)
    return float(np.sum(do * o) + np.sum(dS * S))


def finite_differences(x, do, dS, h=1e-6, **kw):
    """Central differences of the loss w.r.t. every element of every input."""
    fd = {}
    for name, arr in x.items():
        grad = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            xp = {n: a.copy() for n, a in x.items()}
            xm = {n: a.copy() for n, a in x.items()}
            xp[name][idx] += h
            xm[name][idx] -= h
            grad[idx] = (loss(xp, do, dS, **kw) - loss(xm, do, dS, **kw)) / (2 * h)
        fd[name] = grad
    return fd


def assert_grads_match(r, fd):
    for ours, theirs in (("dq", "q"), ("dk", "k"), ("dv", "v"), ("dbeta", "beta"), ("dg", "g"),
                         ("dS0", "S0")):
        ref = fd[theirs]
        tol = 1e-6 * max(1.0, float(np.max(np.abs(ref))))
        np.testing.assert_allclose(r[ours], ref, rtol=0, atol=tol, err_msg=ours)


CASES = [(pc, dr, l2) for pc in (False, True) for dr in (True, False) for l2 in (True, False)]


def pin_finite_differences(mutant=0):
    for per_channel, delta_rule, l2norm in CASES:
        x, do, dS = inputs(5 + per_channel + 2 * delta_rule + 4 * l2norm, 6, 4, 3, per_channel)
        fd = finite_differences(x, do, dS, l2norm=l2norm, delta_rule=delta_rule)
        r = backward_seq(x["q"], x["k"], x["v"], x["beta"], x["g"], x["S0"], do, dS,
                         l2norm=l2norm, delta_rule=delta_rule, mutant=mutant)
        assert_grads_match(r, fd)


def test_finite_differences():
    """Every gradient of one sequence equals central differences of the forward recurrence:
    scalar and per-channel gates, delta rule and additive write, with and without the L2
    normalisation."""
    pin_finite_differences()


@pytest.mark.parametrize("mutant", [1, 2, 3])
def test_planted_mistakes_fail_the_finite_differences(mutant):
    """Dropping the prediction's path into dk, taking the forget gate's gradient against the
    written state, or leaving out the normalisation's projection each fail the pin."""
    with pytest.raises(AssertionError):
        pin_finite_differences(mutant)


def test_additive_decay_free_closed_form():
    """No decay, additive write: o_t = (S0 + sum_{j<=t} beta_j k^_j v_j^T)^T q^_t and
    S_T = S0 + sum_j beta_j k^_j v_j^T, so dv_j = beta_j (sum_{t>=j} (q^_t . k^_j) do_t
    + dS^T k^_j) and dS0 = sum_t q^_t do_t^T + dS."""
    x, do, dS = inputs(31, 9, 5, 4, False)
    x["g"][:] = 0.0
    r = backward_seq(x["q"], x["k"], x["v"], x["beta"], x["g"], x["S0"], do, dS,
                     delta_rule=False)
    kn = x["k"] / np.sqrt(np.sum(x["k"] ** 2, axis=1, keepdims=True) + oracle.L2_EPS)
    qn = x["q"] / np.sqrt(np.sum(x["q"] ** 2, axis=1, keepdims=True) + oracle.L2_EPS) / np.sqrt(5)
    scores = np.tril(qn @ kn.T)                                  # [t, j]
    np.testing.assert_allclose(r["dv"], x["beta"][:, None] * (scores.T @ do + kn @ dS), rtol=0,
                               atol=1e-12)
    np.testing.assert_allclose(r["dS0"], qn.T @ do + dS, rtol=0, atol=1e-12)


def test_ragged_gqa_pool_composition():
    """The batch form: GQA sums the key head's gradients over its value heads, each sequence
    starts from its own slot, and an empty sequence passes d_state through unchanged.
    Checked against finite differences of the whole batch's loss on sampled elements."""
    r = rng(71)
    HK, HV, dk, dv = 1, 2, 4, 3
    lens = [5, 0, 4]
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T = int(offs[-1])
    slots = np.array([2, 0, 3])
    q = r.standard_normal((T, HK, dk))
    k = r.standard_normal((T, HK, dk))
    v = r.standard_normal((T, HV, dv))
    beta = r.uniform(0.1, 0.9, (T, HV))
    g = -r.uniform(0.05, 0.6, (T, HV, dk))
    pool = r.standard_normal((4, HV, dk, dv)) * 0.3
    d_o = r.standard_normal((T, HV, dv))
    d_state = r.standard_normal((4, HV, dk, dv))
    out = backward_arrays(offsets=offs, slot_idx=slots, q=q, k=k, v=v, beta=beta, g=g, pool=pool,
                          d_o=d_o, d_state=d_state)

    def batch_loss(q, k, v, beta, g, pool):
        total = 0.0
        for b in range(3):
            s, e = offs[b], offs[b + 1]
            for h in range(HV):
                o, S = oracle.recurrence_py(q[s:e, h // 2], k[s:e, h // 2], v[s:e, h],
                                            beta[s:e, h], g[s:e, h], pool[slots[b], h])
                total += np.sum(d_o[s:e, h] * o) + np.sum(d_state[slots[b], h] * S)
        return total

    args = dict(q=q, k=k, v=v, beta=beta, g=g, pool=pool)
    names = {"q": "dq", "k": "dk", "v": "dv", "beta": "dbeta", "g": "dg", "pool": "d_state0"}
    h = 1e-6
    for name, arr in args.items():
        for idx in list(np.ndindex(arr.shape))[::7]:
            if name == "pool" and idx[0] not in (2, 0, 3):
                continue
            ap = {n: a.copy() for n, a in args.items()}
            am = {n: a.copy() for n, a in args.items()}
            ap[name][idx] += h
            am[name][idx] -= h
            fd = (batch_loss(**ap) - batch_loss(**am)) / (2 * h)
            assert abs(out[names[name]][idx] - fd) <= 1e-6 * max(1.0, abs(fd)), (name, idx)
    # the empty sequence's slot: the state passes through, so does its gradient
    np.testing.assert_array_equal(out["d_state0"][0], d_state[0])
