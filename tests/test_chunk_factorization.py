"""The factorisation of the chunk form that the tensor-core prefill computes, written out in fp64
numpy and checked against the oracle's token-by-token recurrence.

Per chunk, in the state's stored orientation (S is d_k x d_v, rows = key channels), with G_i the
cumulative log-decay from the chunk start through token i:

  K~_i = k^_i exp(G_i),  Q~_i = s q^_i exp(G_i),  K_end_i = k^_i exp(G_last - G_i),  gam = exp(G_last)
  A_kk[i, j] = beta_i <k^_i, k^_j exp(G_i - G_j)>  (j < i),   T = (I + A_kk)^-1,   TB = T diag(beta)
  A_qk[i, j] = s <q^_i, k^_j exp(G_i - G_j)>        (j <= i)
  Kb = K_end^T TB,   A1o = A_qk TB
  E' = V - K~ S,   S' = diag(gam) S + Kb E',   O = Q~ S + A1o E'

("You Could Have Come Up With Kimi Delta Attention", sec. 6.2-6.5: the corrections there are
E = TB (V - K~ S), so W = TB K~ and U = TB V need never be formed.)  The additive write drops
the prediction: A_kk = 0 and K~ S = 0.

The compact single-kernel form folds both products into one left operand instead:
  [E; O] = [TB | -W; A_qk TB | Q~ - A_qk W] [V; S],   W = TB K~,   S' = diag(gam) S + K_end^T E.
"""
import numpy as np
import pytest

import oracle


def factorised(q, k, v, beta, g, S0, *, chunk, delta_rule=True, slip=None):
    T, dk = q.shape
    scale = 1.0 / np.sqrt(dk)
    qn = q / np.sqrt(np.sum(q * q, axis=1, keepdims=True) + 1e-6)
    kn = k / np.sqrt(np.sum(k * k, axis=1, keepdims=True) + 1e-6)
    gg = g if g.ndim == 2 else np.repeat(g[:, None], dk, axis=1)
    S = S0.copy()
    o = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, chunk):
        sl = slice(c0, min(c0 + chunk, T))
        kc, qc, vc, bc = kn[sl], qn[sl], v[sl], beta[sl]
        n = kc.shape[0]
        G = np.cumsum(gg[sl], axis=0)                      # [n, dk]
        Kt = kc * np.exp(G) if delta_rule else np.zeros_like(kc)
        Qt = scale * qc * np.exp(G)
        Kend = kc * np.exp(G[-1] - G)
        gam = np.exp(G[-1])
        Akk = np.zeros((n, n))
        Aqk = np.zeros((n, n))
        for i in range(n):
            for j in range(i + 1):
                dec = np.exp(G[i] - G[j])
                Aqk[i, j] = scale * np.dot(qc[i], kc[j] * dec)
                if j < i and delta_rule:
                    Akk[i, j] = bc[i] * np.dot(kc[i], kc[j] * dec)
        TB = np.linalg.solve(np.eye(n) + Akk, np.diag(bc))
        Kb = Kend.T @ TB                                   # [dk, n]
        A1o = Aqk @ TB                                     # [n, n]
        if slip == "transposed_A1o":
            A1o = A1o.T
        Ep = vc - Kt @ S                                   # [n, dv]
        o[sl] = Qt @ S + A1o @ (vc if slip == "raw_v_in_output" else Ep)
        S = (S if slip == "no_state_decay" else gam[:, None] * S) + Kb @ Ep
    return o, S


def folded(q, k, v, beta, g, S0, *, chunk, delta_rule=True):
    """The compact kernel's single product per chunk, same definitions as above."""
    T, dk = q.shape
    scale = 1.0 / np.sqrt(dk)
    qn = q / np.sqrt(np.sum(q * q, axis=1, keepdims=True) + 1e-6)
    kn = k / np.sqrt(np.sum(k * k, axis=1, keepdims=True) + 1e-6)
    gg = g if g.ndim == 2 else np.repeat(g[:, None], dk, axis=1)
    S = S0.copy()
    o = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, chunk):
        sl = slice(c0, min(c0 + chunk, T))
        kc, qc, vc, bc = kn[sl], qn[sl], v[sl], beta[sl]
        n = kc.shape[0]
        G = np.cumsum(gg[sl], axis=0)
        Kt = kc * np.exp(G) if delta_rule else np.zeros_like(kc)
        Qt = scale * qc * np.exp(G)
        Kend = kc * np.exp(G[-1] - G)
        dec = np.exp(G[:, None, :] - G[None, :, :])        # [i, j, channel]
        Akk = np.tril(bc[:, None] * np.einsum("ic,jc,ijc->ij", kc, kc, dec), -1)
        Aqk = np.tril(scale * np.einsum("ic,jc,ijc->ij", qc, kc, dec))
        if not delta_rule:
            Akk[:] = 0.0
        TB = np.linalg.solve(np.eye(n) + Akk, np.diag(bc))
        W = TB @ Kt
        left = np.block([[TB, -W], [Aqk @ TB, Qt - Aqk @ W]])          # [2n, n + dk]
        EO = left @ np.vstack([vc, S])
        E, O = EO[:n], EO[n:]
        o[sl] = O
        S = np.exp(G[-1])[:, None] * S + Kend.T @ E
    return o, S


def inputs(seed, T, dk, dv, per_channel):
    r = np.random.Generator(np.random.PCG64(seed))
    q = r.standard_normal((T, dk))
    k = r.standard_normal((T, dk))
    v = r.standard_normal((T, dv))
    beta = r.uniform(0.1, 1.0, T)
    g = -r.uniform(0.0, 0.2, (T, dk) if per_channel else T)
    S0 = r.standard_normal((dk, dv)) * 0.3
    return q, k, v, beta, g, S0


@pytest.mark.parametrize("per_channel", [False, True])
@pytest.mark.parametrize("delta_rule", [True, False])
@pytest.mark.parametrize("T,chunk", [(150, 64), (64, 64), (5, 16), (33, 16)])
def test_factorisation_equals_the_recurrence(per_channel, delta_rule, T, chunk):
    q, k, v, beta, g, S0 = inputs(T * 7 + chunk + 2 * per_channel + delta_rule, T, 16, 8,
                                  per_channel)
    o, S = factorised(q, k, v, beta, g, S0, chunk=chunk, delta_rule=delta_rule)
    o_ref, S_ref = oracle.recurrence_py(q, k, v, beta, g, S0, delta_rule=delta_rule)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-11 * max(1.0, np.abs(o_ref).max()))
    np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-11 * max(1.0, np.abs(S_ref).max()))


@pytest.mark.parametrize("per_channel", [False, True])
@pytest.mark.parametrize("delta_rule", [True, False])
def test_folded_form_equals_the_recurrence(per_channel, delta_rule):
    q, k, v, beta, g, S0 = inputs(11 + 2 * per_channel + delta_rule, 150, 16, 8, per_channel)
    o, S = folded(q, k, v, beta, g, S0, chunk=64, delta_rule=delta_rule)
    o_ref, S_ref = oracle.recurrence_py(q, k, v, beta, g, S0, delta_rule=delta_rule)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-11 * max(1.0, np.abs(o_ref).max()))
    np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-11 * max(1.0, np.abs(S_ref).max()))


@pytest.mark.parametrize("slip", ["no_state_decay", "raw_v_in_output", "transposed_A1o"])
def test_a_one_term_slip_is_caught(slip):
    """Each slip planted in the factorisation (the state's decay left out of the update, V in
    place of E' in the output, A1o transposed) fails the comparison above."""
    q, k, v, beta, g, S0 = inputs(3, 70, 16, 8, False)
    o_ref, S_ref = oracle.recurrence_py(q, k, v, beta, g, S0)
    o, S = factorised(q, k, v, beta, g, S0, chunk=64, slip=slip)
    assert max(np.abs(o - o_ref).max(), np.abs(S - S_ref).max()) > 1e-3


def subblock_matrices(q, k, beta, G, *, tau=12.0, row_scale=256.0):
    """A_kk, A_qk of one chunk as the per-channel tensor-core front kernel forms them: the
    chunk's tokens in sub-blocks of 16, row i of sub-block I scaled by exp(G_i - G_ref(I))
    (G_ref(I) = G at the last token before I, 0 for I = 0) and by 2^8; a key j of an earlier
    sub-block J by exp(G_ref(I) - G_end(J)) exp(G_end(J) - G_j) / 2^8 (both factors <= 1 for a
    non-increasing G); a key of the row's own sub-block by exp(G_ref(J) - G_end(J))
    exp(G_end(J) - G_j) / 2^8, except in the channels whose decay from G_ref(J) exceeds tau
    inside the sub-block, whose pairs are summed directly with exp(G_i - G_j)."""
    n, dk = k.shape
    scale = 1.0 / np.sqrt(dk)
    qn = scale * q / np.sqrt(np.sum(q * q, axis=1, keepdims=True) + 1e-6)
    kn = k / np.sqrt(np.sum(k * k, axis=1, keepdims=True) + 1e-6)
    nb = (n + 15) // 16
    blk = np.arange(n) // 16
    ref = np.zeros((nb, dk))
    end = np.zeros((nb, dk))
    for I in range(nb):
        if I > 0:
            ref[I] = G[16 * I - 1]
        end[I] = G[min(16 * I + 15, n - 1)]
    slow = np.array([ref[J] - G[16 * J:16 * J + 16].min(axis=0) > tau for J in range(nb)])
    eps = np.exp(end[blk] - G)                              # exp(G_end(J) - G_j) <= 1
    ke = kn * eps / row_scale
    A = np.zeros((2, n, n))
    for w, x in enumerate((kn, qn)):
        R = x * np.exp(G - ref[blk]) * row_scale            # exp(G_i - G_ref(I)) <= 1
        for i in range(n):
            I = blk[i]
            for j in range(i + 1):
                J = blk[j]
                if J < I:
                    A[w, i, j] = np.dot(R[i], ke[j] * np.exp(ref[I] - end[J]))
                else:
                    col = np.where(slow[J], 0.0, ke[j] * np.exp(ref[J] - end[J]))
                    exact = np.where(slow[J], x[i] * kn[j] * np.exp(G[i] - G[j]), 0.0)
                    A[w, i, j] = np.dot(R[i], col) + exact.sum()
    return beta[:, None] * np.tril(A[0], -1), np.tril(A[1])


@pytest.mark.parametrize("factor", [1.0, 4.0, 10.0, 33.0])
@pytest.mark.parametrize("n", [64, 50, 17])
def test_subblock_factorization_of_the_intra_chunk_matrices(factor, n):
    """The per-channel front kernel's sub-block form of A_kk and A_qk equals the pairwise
    definition (KDA page, sec. 6.3: exp(G_i - G_j) per pair and channel) in fp64, at decays
    from the kda_prefill workload's to 33x it, where most channels take the exact pairs."""
    r = np.random.default_rng(int(factor * 10) + n)
    q, k = r.standard_normal((n, 128)), r.standard_normal((n, 128))
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal(n)))
    G = np.cumsum(-np.exp(r.normal(-2.0, 0.5, (n, 128))) * factor, axis=0)
    Akk, Aqk = subblock_matrices(q, k, beta, G)
    qn = q / np.sqrt(np.sum(q * q, axis=1, keepdims=True) + 1e-6) / np.sqrt(128)
    kn = k / np.sqrt(np.sum(k * k, axis=1, keepdims=True) + 1e-6)
    ref_kk, ref_qk = np.zeros((n, n)), np.zeros((n, n))
    for i in range(n):
        for j in range(i + 1):
            dec = np.exp(G[i] - G[j])
            ref_qk[i, j] = np.dot(qn[i], kn[j] * dec)
            if j < i:
                ref_kk[i, j] = beta[i] * np.dot(kn[i], kn[j] * dec)
    assert np.allclose(Akk, ref_kk, rtol=1e-12, atol=1e-14)
    assert np.allclose(Aqk, ref_qk, rtol=1e-12, atol=1e-14)
    if factor >= 10.0:                                    # the exact pairs are exercised
        refs = [np.zeros(128)] + [G[16 * J - 1] for J in range(1, (n + 15) // 16)]
        assert any(np.any(ref - G[16 * J:16 * J + 16].min(axis=0) > 12.0)
                   for J, ref in enumerate(refs))
