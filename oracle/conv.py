"""fp64 reference of the front end that feeds the recurrence ("Pass 1").

TEST INFRASTRUCTURE ONLY, like the rest of `oracle/`: it shares no code with the CUDA library.

The Modular "gated_delta" module names the step before its recurrence: a short convolution
over the packed projection whose channels are [Q | K | V] (key_dim, key_dim, value_dim wide),
plus a per-token decay with the softplus applied and a beta with the sigmoid applied.  "From
Attention to Learned Memory", sec. 1, applies SiLU to the features; the linear-attention page's
Mamba-2 section builds the decay from a log-rate A_log and a step softplus(x + b_dt), so that
log a = -exp(A_log) softplus(x + b_dt).  The plainest reading of "short convolution", taken
here: depthwise and causal, each channel's output at token t is sum_i w[c, i] x[t - W + 1 + i]
(+ bias), the W - 1 inputs before a sequence's first token coming from its slot of a conv-state
pool (zeros for a fresh sequence), followed by SiLU(z) = z sigmoid(z).  The pool slot then
holds the sequence's last W - 1 inputs (older ones first).
"""
from __future__ import annotations

import numpy as np


def silu(z):
    z = np.asarray(z, np.float64)
    return z / (1.0 + np.exp(-z))


def softplus(z):
    z = np.asarray(z, np.float64)
    return np.logaddexp(0.0, z)


def conv_gates(*, x, weight, bias, a, b, A_log, dt_bias, offsets, slot_idx, conv_state,
               num_v_heads: int, per_channel: bool):
    """x [T, conv_dim]; weight [conv_dim, W]; bias [conv_dim] or None; a [T, HV] or
    [T, HV, d]; b [T, HV]; A_log [HV] or None; dt_bias [HV] / [HV * d] or None;
    offsets [B + 1]; slot_idx [B]; conv_state [num_slots, conv_dim, W - 1] or None.

    Returns (y [T, conv_dim], log_decay (shape of a), beta [T, HV], new conv_state), fp64.
    """
    x = np.asarray(x, np.float64)
    w = np.asarray(weight, np.float64)
    T, cd = x.shape
    W = w.shape[1]
    offsets = np.asarray(offsets, np.int64)
    y = np.zeros((T, cd))
    state = None if conv_state is None else np.array(conv_state, np.float64, copy=True)
    new_state = None if state is None else state.copy()
    for s in range(offsets.shape[0] - 1):
        bos, eos = int(offsets[s]), int(offsets[s + 1])
        ctx = np.zeros((W - 1, cd)) if state is None else state[int(slot_idx[s])].T   # [W-1, cd]
        xs = np.concatenate([ctx, x[bos:eos]], axis=0)   # position bos - W + 1 + j at row j
        for t in range(eos - bos):
            z = np.sum(w.T * xs[t:t + W], axis=0)        # taps i = 0..W-1 on x[t-W+1+i]
            if bias is not None:
                z = z + np.asarray(bias, np.float64)
            y[bos + t] = silu(z)
        if new_state is not None and W > 1:
            new_state[int(slot_idx[s])] = xs[-(W - 1):].T
    a = np.asarray(a, np.float64)
    HV = num_v_heads
    z = a.copy()
    if dt_bias is not None:
        z = z + np.asarray(dt_bias, np.float64).reshape((HV, -1) if per_channel else (HV,))
    rate = np.ones(HV) if A_log is None else np.exp(np.asarray(A_log, np.float64))
    g = -(rate[:, None] if per_channel else rate) * softplus(z)
    beta = 1.0 / (1.0 + np.exp(-np.asarray(b, np.float64)))
    return y, g, beta, new_state
