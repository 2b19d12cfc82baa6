"""Pins for the fp64 oracle: what the pages and the mathematics fix, not the oracle itself.

Each pin is a function `pin_*(runner)` that raises AssertionError on a mismatch.
`runner` is the oracle's C recurrence (optionally a planted-mistake build), so the
same pins also prove that they catch plausible mistakes (`test_mutants_are_caught`).

Sources of each fact:
  "You Could Have Come Up With Kimi Delta Attention" (KDA page): sec. 2.1 (beta=1 recall,
    orthogonal directions untouched), 2.2 (gradient step), 2.3/3/4.1 (erase-write form),
    4 (per-channel forget; GDN is the equal-channel case), 6 (chunkwise closed form).
  "From Attention to Learned Memory" (blog): sec. 1-2 (causal parallel form with a cached
    prefix state S0; chunk C=1 / C=L extremes).
  "Linear attention visualized": DeltaNet worked example (Alice/Bob, golden fixture);
    "every valid C provides exact results" (chunkwise algorithm).
  Modular "gated_delta" module: GQA key head = value head // ratio, ragged offsets,
    slot-indexed pool with untouched slots.
"""
import functools
import json
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def runner_for(mutant=0):
    return functools.partial(oracle.run_arrays, mutant=mutant, nthreads=2)


def one_seq(runner, q, k, v, beta, g, S0, **kw):
    """Run one sequence / one head through the C oracle; returns (o [T,dv], S [dk,dv])."""
    T, dk = q.shape
    dv = v.shape[1]
    per_channel = g.ndim == 2
    o, pool = runner(offsets=[0, T], slot_idx=[0], q=q[:, None, :], k=k[:, None, :],
                     v=v[:, None, :], beta=beta[:, None],
                     g=(g[:, None, :] if per_channel else g[:, None]), per_channel=per_channel,
                     pool=S0[None, None], **kw)
    return o[:, 0, :], pool[0, 0]


def states_after_each(runner, q, k, v, beta, g, S0, **kw):
    """S_t for t = 0..T by running prefixes (S_0 = S0)."""
    out = [np.array(S0, np.float64)]
    for t in range(1, q.shape[0] + 1):
        _, S = one_seq(runner, q[:t], k[:t], v[:t], beta[:t], g[:t], S0, **kw)
        out.append(S)
    return out


def exact_unit_keys(r, T, dk):
    """Unit keys exactly representable in fp32: four entries of +-1/2, rest zero."""
    k = np.zeros((T, dk), np.float32)
    for t in range(T):
        idx = r.choice(dk, 4, replace=False)
        k[t, idx] = r.choice([-0.5, 0.5], 4)
    return k


def small_inputs(seed, T=9, dk=8, dv=6, per_channel=True):
    r = rng(seed)
    q = r.standard_normal((T, dk)).astype(np.float32)
    k = r.standard_normal((T, dk)).astype(np.float32)
    v = r.standard_normal((T, dv)).astype(np.float32)
    beta = r.uniform(0.1, 0.9, T).astype(np.float32)
    g = (-r.uniform(0.01, 0.6, (T, dk) if per_channel else T)).astype(np.float32)
    S0 = r.standard_normal((dk, dv)) * 0.3
    return q, k, v, beta, g, S0


# ------------------------------------------------------------------------------------ pins

def pin_beta_one_recall(runner):
    """KDA page sec. 2.1: with beta=1 and a unit key the write is read back exactly,
    S_t k_t = v_t, with or without decay (the prediction uses the decayed state)."""
    r = rng(11)
    T, dk, dv = 10, 8, 5
    q, _, v, _, g, S0 = small_inputs(12, T, dk, dv)
    k = exact_unit_keys(r, T, dk)
    beta = np.ones(T, np.float32)
    states = states_after_each(runner, q, k, v, beta, g, S0, scale=1.0, l2norm=False)
    for t in range(1, T + 1):
        got = k[t - 1].astype(np.float64) @ states[t]     # stored orientation: k^T S = (S_math k)^T
        np.testing.assert_allclose(got, v[t - 1], rtol=0, atol=1e-12)


def pin_orthogonal_directions_untouched(runner):
    """KDA page sec. 2.1: for x orthogonal to k_t, (S_t - S~_t) x = 0, S~_t the decayed state."""
    T, dk, dv = 8, 8, 5
    q, k, v, beta, g, S0 = small_inputs(13, T, dk, dv)
    states = states_after_each(runner, q, k, v, beta, g, S0, scale=1.0, l2norm=True)
    kn = k / np.sqrt(np.sum(k.astype(np.float64) ** 2, axis=1, keepdims=True) + oracle.L2_EPS)
    r = rng(14)
    for t in range(1, T + 1):
        Stil = np.exp(g[t - 1].astype(np.float64))[:, None] * states[t - 1]
        x = r.standard_normal(dk)
        x -= (x @ kn[t - 1]) / (kn[t - 1] @ kn[t - 1]) * kn[t - 1]
        np.testing.assert_allclose(x @ (states[t] - Stil), 0.0, atol=1e-12)
        # and the change along k_t is the full correction e_t (not zero)
        assert np.max(np.abs(kn[t - 1] @ (states[t] - Stil))) > 1e-3


def pin_erase_write_form(runner):
    """KDA page sec. 4.1: S_t = S_{t-1} D_t (I - beta k k^T) + beta v k^T (DPLR transition),
    checked in the stored orientation S^T = (I - beta k k^T) D_t S^T_{t-1} + beta k v^T."""
    T, dk, dv = 7, 8, 6
    q, k, v, beta, g, S0 = small_inputs(15, T, dk, dv)
    states = states_after_each(runner, q, k, v, beta, g, S0, scale=1.0, l2norm=True)
    kn = k / np.sqrt(np.sum(k.astype(np.float64) ** 2, axis=1, keepdims=True) + oracle.L2_EPS)
    for t in range(1, T + 1):
        kk, b = kn[t - 1], float(beta[t - 1])
        D = np.diag(np.exp(g[t - 1].astype(np.float64)))
        expect = (np.eye(dk) - b * np.outer(kk, kk)) @ D @ states[t - 1] + b * np.outer(kk, v[t - 1])
        np.testing.assert_allclose(states[t], expect, rtol=0, atol=1e-12)


def pin_gradient_step(runner):
    """KDA page sec. 2.2: S_t = S~_t - beta grad_S 1/2 ||S k - v||^2 at S~_t, the gradient
    taken numerically here (central differences), not from the closed form."""
    T, dk, dv = 4, 5, 3
    q, k, v, beta, g, S0 = small_inputs(16, T, dk, dv)
    states = states_after_each(runner, q, k, v, beta, g, S0, scale=1.0, l2norm=True)
    kn = k / np.sqrt(np.sum(k.astype(np.float64) ** 2, axis=1, keepdims=True) + oracle.L2_EPS)
    h = 1e-6
    for t in range(1, T + 1):
        Stil = np.exp(g[t - 1].astype(np.float64))[:, None] * states[t - 1]   # stored [dk, dv]
        loss = lambda S: 0.5 * np.sum((kn[t - 1] @ S - v[t - 1]) ** 2)
        grad = np.zeros_like(Stil)
        for c in range(dk):
            for j in range(dv):
                P, M = Stil.copy(), Stil.copy()
                P[c, j] += h; M[c, j] -= h
                grad[c, j] = (loss(P) - loss(M)) / (2 * h)
        np.testing.assert_allclose(states[t], Stil - float(beta[t - 1]) * grad, atol=1e-7)


def pin_linear_attention_bruteforce(runner):
    """Blog sec. 1-2: without decay and without the delta term the read equals the causal
    parallel form s (Q K^T masked) V plus the cached-prefix term s Q S0."""
    T, dk, dv = 11, 8, 6
    q, k, v, _, _, S0 = small_inputs(17, T, dk, dv)
    beta = np.ones(T, np.float32)
    g = np.zeros(T, np.float32)
    o, S = one_seq(runner, q, k, v, beta, g, S0, scale=0.0, l2norm=True, delta_rule=False)
    ref = oracle.causal_linear_attention(q, k, v, S0, scale=0.0, l2norm=True)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    kn = k / np.sqrt(np.sum(k.astype(np.float64) ** 2, axis=1, keepdims=True) + oracle.L2_EPS)
    np.testing.assert_allclose(S, S0 + kn.T @ v, atol=1e-12)


def pin_gated_linear_attention_parallel(runner):
    """"Linear attention visualized", RetNet, Mamba-2 and GLA sections: without the delta term
    the decayed recurrence equals its parallel form.  A write at position j reaches the
    query at t >= j through the decay of the tokens after it, so its score is
    q^_t . (k^_j * exp(G_t - G_j)) with G the inclusive cumulative log-decay (the diagonal
    is undecayed), it carries beta_j v_j (Mamba-2's write step), and the incoming state
    enters as (q^_t * exp(G_t)) S0.  The final state is Diag(exp(G_T)) S0 plus every write
    decayed to the end.  Scalar gate (Mamba-2) and per-channel gate (GLA)."""
    T, dk, dv = 10, 8, 5
    for per_channel in (False, True):
        q, k, v, beta, g, S0 = small_inputs(19 + per_channel, T, dk, dv, per_channel=per_channel)
        o, S = one_seq(runner, q, k, v, beta, g, S0, scale=0.0, l2norm=True, delta_rule=False)
        qn = q / np.sqrt(np.sum(q.astype(np.float64) ** 2, axis=1, keepdims=True) + oracle.L2_EPS)
        qn = qn / np.sqrt(dk)
        kn = k / np.sqrt(np.sum(k.astype(np.float64) ** 2, axis=1, keepdims=True) + oracle.L2_EPS)
        G = np.cumsum(g.astype(np.float64), axis=0)
        if not per_channel:
            G = np.repeat(G[:, None], dk, axis=1)
        # scores[t, j] = sum_c q^_t[c] k^_j[c] exp(G_t[c] - G_j[c]), causal (j <= t)
        scores = np.einsum("tc,jc,tjc->tj", qn, kn, np.exp(G[:, None, :] - G[None, :, :]))
        scores *= np.tril(np.ones((T, T)))
        bv = beta.astype(np.float64)[:, None] * v.astype(np.float64)
        ref = scores @ bv + (qn * np.exp(G)) @ S0
        np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
        S_ref = np.exp(G[-1])[:, None] * S0 + (kn * np.exp(G[-1] - G)).T @ bv
        np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-12)


def pin_beta_zero_pure_decay(runner):
    """Closed form: beta = 0 leaves only the forget gate, S_T = Diag(exp(sum g)) S0 and
    o_t = s q_t^T S_t (KDA page sec. 4, forget then read)."""
    T, dk, dv = 12, 8, 5
    q, k, v, _, g, S0 = small_inputs(18, T, dk, dv)
    beta = np.zeros(T, np.float32)
    o, S = one_seq(runner, q, k, v, beta, g, S0, scale=0.0, l2norm=True)
    G = np.cumsum(g.astype(np.float64), axis=0)
    np.testing.assert_allclose(S, np.exp(G[-1])[:, None] * S0, rtol=1e-13, atol=1e-15)
    qn = q / np.sqrt(np.sum(q.astype(np.float64) ** 2, axis=1, keepdims=True) + oracle.L2_EPS)
    for t in range(T):
        np.testing.assert_allclose(o[t], (qn[t] / np.sqrt(dk)) @ (np.exp(G[t])[:, None] * S0),
                                   rtol=1e-12, atol=1e-14)


def pin_orthonormal_keys(runner):
    """Closed form: no decay, beta = 1, mutually orthonormal keys -> every association is
    stored exactly, S_T k_i = v_i for all i, and S_T = (I - sum k k^T) S0 + sum k v^T."""
    dk, dv, T = 8, 5, 6
    r = rng(19)
    Qm, _ = np.linalg.qr(r.standard_normal((dk, dk)))
    # exactly representable orthonormal keys: signed, permuted standard basis vectors
    perm = r.permutation(dk)[:T]
    k = np.zeros((T, dk), np.float32)
    for t, c in enumerate(perm):
        k[t, c] = 1.0 if r.uniform() < 0.5 else -1.0
    v = r.standard_normal((T, dv)).astype(np.float32)
    q = r.standard_normal((T, dk)).astype(np.float32)
    S0 = r.standard_normal((dk, dv))
    o, S = one_seq(runner, q, k, v, np.ones(T, np.float32), np.zeros(T, np.float32), S0,
                   scale=1.0, l2norm=False)
    kd = k.astype(np.float64)
    for i in range(T):
        np.testing.assert_allclose(kd[i] @ S, v[i], atol=1e-13)
    np.testing.assert_allclose(S, (np.eye(dk) - kd.T @ kd) @ S0 + kd.T @ v, atol=1e-13)


def pin_equal_channels_is_scalar_gate(runner):
    """"Linear attention visualized", KDA: with a_t = a_t 1 KDA reduces exactly to GDN."""
    T, dk, dv = 10, 8, 6
    q, k, v, beta, g, S0 = small_inputs(20, T, dk, dv, per_channel=False)
    o1, S1 = one_seq(runner, q, k, v, beta, g, S0)
    o2, S2 = one_seq(runner, q, k, v, beta, np.repeat(g[:, None], dk, axis=1), S0)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(S1, S2)


def pin_alice_bob(runner):
    """"Linear attention visualized", DeltaNet worked example (golden fixture)."""
    with open(os.path.join(HERE, "golden", "alice_bob.json")) as f:
        gold = json.load(f)
    k = np.array([t["key"] for t in gold["tokens"]], np.float32)
    v = np.array([t["value"] for t in gold["tokens"]], np.float32)
    q = np.array([t["query"] for t in gold["tokens"]], np.float32)
    for case in gold["cases"]:
        T = len(k)
        o, S = one_seq(runner, q, k, v, np.full(T, case["beta"], np.float32),
                       np.zeros(T, np.float32), np.zeros((2, 3)), scale=1.0, l2norm=False)
        np.testing.assert_allclose(o, case["reads"], atol=1e-15)
        np.testing.assert_allclose(S, case["final_state_rows_are_key_channels"], atol=1e-15)


def pin_gqa_ragged_pool(runner):
    """Modular gated_delta: key head = value head // (HV/HK); each sequence of the ragged
    batch uses its own slot; slots not named in slot_idx are untouched; packing order
    does not change any sequence's result."""
    r = rng(21)
    HK, HV, dk, dv = 2, 4, 8, 6
    lens = [5, 0, 9, 3]
    T = sum(lens)
    offs = np.concatenate([[0], np.cumsum(lens)])
    q = r.standard_normal((T, HK, dk)).astype(np.float32)
    k = r.standard_normal((T, HK, dk)).astype(np.float32)
    v = r.standard_normal((T, HV, dv)).astype(np.float32)
    beta = r.uniform(0.1, 0.9, (T, HV)).astype(np.float32)
    g = (-r.uniform(0.01, 0.5, (T, HV, dk))).astype(np.float32)
    pool = r.standard_normal((6, HV, dk, dv))
    slots = np.array([4, 0, 2, 5])
    o, P = runner(offsets=offs, slot_idx=slots, q=q, k=k, v=v, beta=beta, g=g, per_channel=True,
                  pool=pool)
    np.testing.assert_array_equal(P[[1, 3]], pool[[1, 3]])          # untouched slots
    np.testing.assert_array_equal(P[0], pool[0])                      # empty sequence
    for b in range(4):
        for h in range(HV):
            sl = slice(offs[b], offs[b + 1])
            ob, Sb = one_seq(runner, q[sl, h // 2], k[sl, h // 2], v[sl, h], beta[sl, h],
                             g[sl, h], pool[slots[b], h])
            np.testing.assert_allclose(o[sl, h], ob, rtol=0, atol=1e-13)
            np.testing.assert_allclose(P[slots[b], h], Sb, rtol=0, atol=1e-13)


PINS = [pin_beta_one_recall, pin_orthogonal_directions_untouched, pin_erase_write_form,
        pin_gradient_step, pin_linear_attention_bruteforce, pin_gated_linear_attention_parallel,
        pin_beta_zero_pure_decay,
        pin_orthonormal_keys, pin_equal_channels_is_scalar_gate, pin_alice_bob,
        pin_gqa_ragged_pool]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(runner_for(0))


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5])
def test_mutants_are_caught(mutant):
    """Each planted mistake in the oracle (wrong decay sign, wrong prediction sign, dropped
    beta, query used as write key, transposed state read) fails at least one pin."""
    runner = runner_for(mutant)
    failed = []
    for pin in PINS:
        try:
            pin(runner)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} passed every pin"


# ------------------------------------------------------------- the other oracle functions

@pytest.mark.parametrize("chunk", [1, 2, 3, 4, 8, 16, 37])
@pytest.mark.parametrize("per_channel", [False, True])
def test_chunk_form_equals_recurrence(chunk, per_channel):
    """KDA page sec. 6 ("must produce the same state and outputs as the token recurrence")
    and "every valid C provides exact results": the dense chunk closed form matches the
    recurrence for every chunk size, including C=1 and C=T, with a ragged last chunk."""
    T, dk, dv = 37, 8, 6
    q, k, v, beta, g, S0 = small_inputs(30 + chunk, T, dk, dv, per_channel=per_channel)
    o_ref, S_ref = one_seq(runner_for(0), q, k, v, beta, g, S0)
    o, S = oracle.chunk_form(q, k, v, beta, g, S0, chunk=chunk)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-12)


def test_numpy_recurrence_matches_c():
    """The numpy transcription and the C recurrence agree (catches indexing slips)."""
    q, k, v, beta, g, S0 = small_inputs(40, 23, 16, 12)
    o1, S1 = oracle.recurrence_py(q, k, v, beta, g, S0)
    o2, S2 = one_seq(runner_for(0), q, k, v, beta, g, S0)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(S1, S2, rtol=0, atol=1e-13)


def test_l2_norm_makes_input_scale_irrelevant():
    """Modular gated_delta (keys and queries are L2-normalised before use): positive
    rescaling of a q or k row changes nothing beyond the epsilon of the norm."""
    q, k, v, beta, g, S0 = small_inputs(41, 15, 8, 6)
    s = rng(42).uniform(0.5, 4.0, (15, 1)).astype(np.float32)
    o1, S1 = one_seq(runner_for(0), q, k, v, beta, g, S0)
    o2, S2 = one_seq(runner_for(0), q * s, k * s, v, beta, g, S0)
    np.testing.assert_allclose(o1, o2, atol=1e-5)
    np.testing.assert_allclose(S1, S2, atol=1e-5)


def test_decode_steps_equal_prefill():
    """KDA page sec. 6.6: recurrent and chunked modes are two schedules of one recurrence;
    n single-token steps from a state equal one prefill of the n tokens from that state."""
    import workloads
    dp = workloads.make_decode_problem("t", num_seqs=3, steps=5, num_k_heads=2, num_v_heads=4,
                                       d=8, qkv_dtype="bf16", state_dtype="f32",
                                       decay_kind="per_channel", zero_state=False, seed=7)
    o_dec, pool_dec = oracle.run_decode(dp, nthreads=2)
    B, S = dp.num_seqs, dp.steps
    # token-major ragged layout: sequence b's tokens are steps 0..S-1
    tq = lambda a: np.ascontiguousarray(np.swapaxes(a, 0, 1).reshape((B * S,) + a.shape[2:]))
    o_pre, pool_pre = oracle.run_arrays(
        offsets=np.arange(B + 1) * S, slot_idx=dp.slot_idx,
        q=tq(workloads.as_f32(dp.q, dp.qkv_dtype)), k=tq(workloads.as_f32(dp.k, dp.qkv_dtype)),
        v=tq(workloads.as_f32(dp.v, dp.qkv_dtype)), beta=tq(dp.beta), g=tq(dp.g),
        per_channel=True, pool=workloads.as_f32(dp.pool, dp.state_dtype), scale=0.0, nthreads=2)
    np.testing.assert_allclose(pool_dec, pool_pre, rtol=0, atol=1e-14)
    np.testing.assert_allclose(np.swapaxes(o_dec, 0, 1).reshape(B * S, 4, 8), o_pre, atol=1e-14)


def test_round_to_bf16_matches_bit_level_rounding():
    """The oracle's bf16 rounding equals round-to-nearest-even on the bit pattern (for
    values exactly representable in fp32, including exact ties)."""
    import workloads
    r = rng(50)
    x = (r.standard_normal(10000) * np.exp(r.uniform(-8, 8, 10000))).astype(np.float32)
    ties = np.array([1.00390625, 1.01171875, -3.0078125, 0.0], np.float32)  # 1+2^-8, 1+3*2^-8
    x = np.concatenate([x, ties])
    ref = workloads.bf16_bits_to_f32(workloads.f32_to_bf16_bits(x)).astype(np.float64)
    np.testing.assert_array_equal(oracle.round_to_bf16(x.astype(np.float64)), ref)
    assert oracle.round_to_bf16(np.array([1.00390625]))[0] == 1.0          # tie to even
    assert oracle.round_to_bf16(np.array([1.01171875]))[0] == 1.015625     # tie to even (up)
