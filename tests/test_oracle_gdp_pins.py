"""Pins for the Gated DeltaProduct oracle ("Linear attention visualized", Gated Delta Product
section): n_h transitions per token, each with its own key, value and gate; the previous
state decays once, before the first; the query reads after the last.

Each pin raises AssertionError on a mismatch; `runner` is the oracle's GDP recurrence
(optionally a planted-mistake build), so the pins also show that they catch the mistakes
a substep loop invites (`test_gdp_mutants_are_caught`).
"""
import functools

import numpy as np
import pytest

import oracle


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def gdp_runner(mutant=0):
    return functools.partial(oracle.run_gdp_arrays, mutant=mutant, nthreads=2)


def one_token_seq(runner, q, k, v, beta, g, S0, **kw):
    """One sequence, one head: q [T, dk], k [T, n_h, dk], v [T, n_h, dv], beta [T, n_h],
    g [T] (scalar) or [T, dk].  Returns (o [T, dv], S [dk, dv])."""
    T = q.shape[0]
    per_channel = g.ndim == 2
    o, pool = runner(offsets=[0, T], slot_idx=[0], q=q[:, None, :], k=k[:, :, None, :],
                     v=v[:, :, None, :], beta=beta[:, :, None],
                     g=(g[:, None, :] if per_channel else g[:, None]), per_channel=per_channel,
                     pool=S0[None, None], **kw)
    return o[:, 0, :], pool[0, 0]


def exact_orthonormal_keys(r, n, dk):
    """n mutually orthonormal keys exactly representable in fp32: four entries of +-1/2 on
    disjoint supports."""
    assert 4 * n <= dk
    perm = r.permutation(dk)
    k = np.zeros((n, dk), np.float32)
    for j in range(n):
        k[j, perm[4 * j:4 * j + 4]] = r.choice([-0.5, 0.5], 4)
    return k


def pin_virtual_sequence(runner):
    """The page's construction: GDP equals Gated DeltaNet over the virtual sequence
    m = t * n_h + j with k~_m = k_{t,j}, v~_m = v_{t,j}, beta~_m = beta_{t,j}, decay a_t at
    j = 0 and 1 after, query q_t at j = n_h - 1 and 0 before; every n_h-th output is kept.
    Ragged batch, GQA, pool slots, both gate kinds."""
    r = rng(61)
    HK, HV, dk, dv, n_h = 2, 4, 8, 6, 3
    lens = [4, 0, 6]
    T = sum(lens)
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    q = r.standard_normal((T, HK, dk)).astype(np.float32)
    k = r.standard_normal((T, n_h, HK, dk)).astype(np.float32)
    v = r.standard_normal((T, n_h, HV, dv)).astype(np.float32)
    beta = r.uniform(0.1, 0.9, (T, n_h, HV)).astype(np.float32)
    pool = r.standard_normal((5, HV, dk, dv)) * 0.3
    slots = np.array([3, 0, 1])
    for per_channel in (False, True):
        g = (-r.uniform(0.01, 0.6, (T, HV, dk) if per_channel else (T, HV))).astype(np.float32)
        o, P = runner(offsets=offs, slot_idx=slots, q=q, k=k, v=v, beta=beta, g=g,
                      per_channel=per_channel, pool=pool)
        qv = np.zeros((T, n_h, HK, dk), np.float32)
        qv[:, n_h - 1] = q
        gv = np.zeros((T, n_h) + g.shape[1:], np.float32)
        gv[:, 0] = g
        ov, Pv = runner(offsets=offs * n_h, slot_idx=slots, q=qv.reshape(T * n_h, HK, dk),
                        k=k.reshape(T * n_h, 1, HK, dk), v=v.reshape(T * n_h, 1, HV, dv),
                        beta=beta.reshape(T * n_h, 1, HV), g=gv.reshape((T * n_h,) + g.shape[1:]),
                        per_channel=per_channel, pool=pool)
        np.testing.assert_allclose(o, ov.reshape(T, n_h, HV, dv)[:, n_h - 1], rtol=0, atol=1e-12)
        np.testing.assert_allclose(P, Pv, rtol=0, atol=1e-12)


def pin_decay_once_per_token(runner):
    """With every gate beta = 0 nothing is written: S_T = Diag(exp(sum_t g_t)) S_0 and
    o_t = S_t^T (s q^_t) -- the state decays once per token, not once per substep."""
    r = rng(62)
    T, n_h, dk, dv = 5, 3, 8, 6
    q = r.standard_normal((T, dk)).astype(np.float32)
    k = r.standard_normal((T, n_h, dk)).astype(np.float32)
    v = r.standard_normal((T, n_h, dv)).astype(np.float32)
    beta = np.zeros((T, n_h), np.float32)
    g = (-r.uniform(0.05, 0.5, (T, dk))).astype(np.float32)
    S0 = r.standard_normal((dk, dv))
    o, S = one_token_seq(runner, q, k, v, beta, g, S0)
    G = np.cumsum(g.astype(np.float64), axis=0)
    np.testing.assert_allclose(S, np.exp(G[-1])[:, None] * S0, rtol=1e-12, atol=1e-14)
    for t in range(T):
        qh = q[t] / np.sqrt(np.sum(q[t].astype(np.float64) ** 2) + 1e-6) / np.sqrt(dk)
        np.testing.assert_allclose(o[t], (np.exp(G[t])[:, None] * S0).T @ qh, rtol=1e-10,
                                   atol=1e-13)


def pin_orthonormal_substeps(runner):
    """One token whose n_h substep keys are orthonormal, every gate 1, no decay: each write
    stores its association exactly and leaves the others alone, so afterwards S^T k_j = v_j
    for every j, S x = S_0 x for x orthogonal to all keys, and o = S^T (s q^)."""
    r = rng(63)
    n_h, dk, dv = 3, 16, 5
    k = exact_orthonormal_keys(r, n_h, dk)[None]
    v = r.standard_normal((1, n_h, dv)).astype(np.float32)
    q = r.standard_normal((1, dk)).astype(np.float32)
    beta = np.ones((1, n_h), np.float32)
    g = np.zeros(1, np.float32)
    S0 = r.standard_normal((dk, dv))
    o, S = one_token_seq(runner, q, k, v, beta, g, S0, l2norm=False)    # the keys are unit
    for j in range(n_h):
        np.testing.assert_allclose(S.T @ k[0, j].astype(np.float64), v[0, j], rtol=0, atol=1e-12)
    Kf = k[0].astype(np.float64)
    x = r.standard_normal(dk)
    x -= Kf.T @ (Kf @ x)
    np.testing.assert_allclose(S.T @ x, S0.T @ x, rtol=0, atol=1e-12)
    qh = q[0].astype(np.float64) / np.sqrt(dk)
    np.testing.assert_allclose(o[0], S.T @ qh, rtol=0, atol=1e-12)


def pin_last_write_read(runner):
    """Two substeps writing the same unit key with gate 1: the second overwrites the first,
    and the query reads after it, so o = v_2 for q = k (scale 1)."""
    r = rng(64)
    dk, dv = 8, 4
    kk = np.zeros(dk, np.float32)
    kk[[1, 3, 4, 6]] = [0.5, -0.5, 0.5, 0.5]
    k = np.stack([kk, kk])[None]
    v = r.standard_normal((1, 2, dv)).astype(np.float32)
    beta = np.ones((1, 2), np.float32)
    g = (-r.uniform(0.1, 0.5, 1)).astype(np.float32)
    S0 = r.standard_normal((dk, dv))
    o, S = one_token_seq(runner, kk[None], k, v, beta, g, S0, scale=1.0, l2norm=False)
    np.testing.assert_allclose(S.T @ kk.astype(np.float64), v[0, 1], rtol=0, atol=1e-12)
    np.testing.assert_allclose(o[0], v[0, 1], rtol=0, atol=1e-12)


def pin_one_substep_is_gated_deltanet(runner):
    """n_h = 1 is the plain gated delta rule (the recurrence the other oracle pins fix)."""
    r = rng(65)
    T, HK, HV, dk, dv = 7, 1, 2, 8, 6
    q = r.standard_normal((T, HK, dk)).astype(np.float32)
    k = r.standard_normal((T, HK, dk)).astype(np.float32)
    v = r.standard_normal((T, HV, dv)).astype(np.float32)
    beta = r.uniform(0.1, 0.9, (T, HV)).astype(np.float32)
    g = (-r.uniform(0.01, 0.6, (T, HV))).astype(np.float32)
    pool = r.standard_normal((1, HV, dk, dv))
    o, P = runner(offsets=[0, T], slot_idx=[0], q=q, k=k[:, None], v=v[:, None],
                  beta=beta[:, None], g=g, per_channel=False, pool=pool)
    o2, P2 = oracle.run_arrays(offsets=[0, T], slot_idx=[0], q=q, k=k, v=v, beta=beta, g=g,
                               per_channel=False, pool=pool, nthreads=1)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(P, P2, rtol=0, atol=1e-13)


GDP_PINS = [pin_virtual_sequence, pin_decay_once_per_token, pin_orthonormal_substeps,
            pin_last_write_read, pin_one_substep_is_gated_deltanet]


@pytest.mark.parametrize("pin", GDP_PINS, ids=[p.__name__ for p in GDP_PINS])
def test_gdp_pin(pin):
    pin(gdp_runner(0))


@pytest.mark.parametrize("mutant", [6, 7])
def test_gdp_mutants_are_caught(mutant):
    """The substep loop's planted mistakes (the forget step repeated at every substep; the
    read taken after the first substep) each fail at least one pin."""
    runner = gdp_runner(mutant)
    failed = []
    for pin in GDP_PINS:
        try:
            pin(runner)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} passed every pin"
