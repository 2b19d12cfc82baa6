"""Pins for the front-end oracle (`oracle/conv.py`): the causal short convolution, SiLU and the
gate activations, checked against closed forms, a library convolution and an invariant.
"""
import numpy as np

from oracle import conv as oc


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def one_seq(x, w, bias=None, state=None):
    T, cd = x.shape
    cs = None if state is None else state[None]
    y, _, _, ns = oc.conv_gates(x=x, weight=w, bias=bias, a=np.zeros((T, 1)), b=np.zeros((T, 1)),
                                A_log=None, dt_bias=None, offsets=[0, T], slot_idx=[0],
                                conv_state=cs, num_v_heads=1, per_channel=False)
    return y, (None if ns is None else ns[0])


def test_identity_tap_is_silu():
    """Only the last tap set: each output is SiLU of the same token's input."""
    r = rng(1)
    x = r.standard_normal((9, 5))
    w = np.zeros((5, 4))
    w[:, 3] = 1.0
    y, _ = one_seq(x, w)
    np.testing.assert_allclose(y, x / (1 + np.exp(-x)), rtol=0, atol=1e-15)


def test_first_tap_reads_the_conv_state():
    """Only the first tap set: output t is SiLU of the input W - 1 tokens earlier, which for
    the first W - 1 tokens is the slot's cached input (oldest first)."""
    r = rng(2)
    W = 4
    x = r.standard_normal((7, 3))
    state = r.standard_normal((3, W - 1))
    w = np.zeros((3, W))
    w[:, 0] = 1.0
    y, ns = one_seq(x, w, state=state)
    prev = np.concatenate([state.T, x], axis=0)        # position t - 3 at row t
    np.testing.assert_allclose(y, prev[:7] / (1 + np.exp(-prev[:7])), rtol=0, atol=1e-15)
    np.testing.assert_array_equal(ns, x[-(W - 1):].T)


def test_matches_library_convolution():
    """Per channel the pre-activation equals numpy's full convolution with the reversed taps
    (a causal correlation), zero left context, plus the bias."""
    r = rng(3)
    x = r.standard_normal((20, 4))
    w = r.standard_normal((4, 3))
    bias = r.standard_normal(4)
    y, _ = one_seq(x, w, bias=bias)
    for c in range(4):
        z = np.convolve(x[:, c], w[c, ::-1])[:20] + bias[c]
        np.testing.assert_allclose(y[:, c], z / (1 + np.exp(-z)), rtol=1e-13, atol=1e-14)


def test_split_sequence_equals_whole():
    """Running a sequence in two calls, the conv state carrying the boundary, gives the
    outputs and the final state of one call; a piece shorter than W - 1 is handled too."""
    r = rng(4)
    W = 4
    x = r.standard_normal((11, 6))
    w = r.standard_normal((6, W))
    s0 = r.standard_normal((6, W - 1))
    y, ns = one_seq(x, w, state=s0)
    for cut in (1, 2, 5):
        y1, s1 = one_seq(x[:cut], w, state=s0)
        y2, s2 = one_seq(x[cut:], w, state=s1)
        np.testing.assert_allclose(np.concatenate([y1, y2]), y, rtol=0, atol=1e-14)
        np.testing.assert_allclose(s2, ns, rtol=0, atol=0)


def test_gates():
    """beta = sigmoid(b); log-decay -softplus(a) = log sigmoid(-a) (so the decay is
    sigmoid(-a), in (0, 1)); with a log-rate and a step bias, -exp(A_log) softplus(a + b_dt);
    per-channel biases broadcast per (head, channel)."""
    r = rng(5)
    T, HV, d = 6, 3, 4
    a = r.standard_normal((T, HV)) * 3
    b = r.standard_normal((T, HV)) * 3
    _, g, beta, _ = oc.conv_gates(x=np.zeros((T, 1)), weight=np.ones((1, 1)), bias=None, a=a, b=b,
                                  A_log=None, dt_bias=None, offsets=[0, T], slot_idx=[0],
                                  conv_state=None, num_v_heads=HV, per_channel=False)
    np.testing.assert_allclose(beta, 1 / (1 + np.exp(-b)), rtol=1e-15)
    np.testing.assert_allclose(g, np.log(1 / (1 + np.exp(a))), rtol=1e-12, atol=1e-15)
    A_log = r.standard_normal(HV)
    dtb = r.standard_normal(HV)
    _, g2, _, _ = oc.conv_gates(x=np.zeros((T, 1)), weight=np.ones((1, 1)), bias=None, a=a, b=b,
                                A_log=A_log, dt_bias=dtb, offsets=[0, T], slot_idx=[0],
                                conv_state=None, num_v_heads=HV, per_channel=False)
    np.testing.assert_allclose(g2, -np.exp(A_log) * np.log1p(np.exp(a + dtb)), rtol=1e-12)
    ap = r.standard_normal((T, HV, d))
    dtp = r.standard_normal(HV * d)
    _, g3, _, _ = oc.conv_gates(x=np.zeros((T, 1)), weight=np.ones((1, 1)), bias=None, a=ap, b=b,
                                A_log=A_log, dt_bias=dtp, offsets=[0, T], slot_idx=[0],
                                conv_state=None, num_v_heads=HV, per_channel=True)
    np.testing.assert_allclose(
        g3, -np.exp(A_log)[None, :, None] * np.log1p(np.exp(ap + dtp.reshape(HV, d))), rtol=1e-12)


def test_ragged_batch_and_slots():
    """Each sequence of a ragged batch starts from its own slot; an empty sequence leaves its
    slot unchanged; slots no sequence names are untouched."""
    r = rng(6)
    W, cd = 3, 4
    lens = [5, 0, 1, 6]
    offs = np.concatenate([[0], np.cumsum(lens)])
    T = int(offs[-1])
    x = r.standard_normal((T, cd))
    w = r.standard_normal((cd, W))
    pool = r.standard_normal((6, cd, W - 1))
    slots = [4, 0, 2, 5]
    y, _, _, ns = oc.conv_gates(x=x, weight=w, bias=None, a=np.zeros((T, 1)), b=np.zeros((T, 1)),
                                A_log=None, dt_bias=None, offsets=offs, slot_idx=slots,
                                conv_state=pool, num_v_heads=1, per_channel=False)
    for s, slot in enumerate(slots):
        ys, st = one_seq(x[offs[s]:offs[s + 1]], w, state=pool[slot])
        np.testing.assert_allclose(y[offs[s]:offs[s + 1]], ys, rtol=0, atol=0)
        np.testing.assert_array_equal(ns[slot], st)
    np.testing.assert_array_equal(ns[0], pool[0])          # the empty sequence's slot
    np.testing.assert_array_equal(ns[[1, 3]], pool[[1, 3]])
    # a one-token sequence shifts its state by one
    np.testing.assert_array_equal(ns[2], np.concatenate([pool[2][:, 1:], x[5:6].T], axis=1))
