"""Speculative-decode verification window and the fold of accepted records, through the C ABI.

The verify call runs `window` draft tokens per sequence from the slot's state without
writing the state back; the fold then applies the first `accepted[b]` records.  The
oracle for both is the fp64 recurrence: verify's outputs are the recurrence's outputs
over the window, and the folded state is the recurrence's state after the accepted
prefix of the window (each sequence's own prefix length).
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_deltanet_gb300 as kda
import oracle
import workloads
from workloads import torch_io

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-3, "f32": 1e-4}
DEV = "cuda:0"


def rel_err(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(x)), "non-finite output"
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(x - ref)) / (den if den > 0 else 1.0))


def rel_err_bf16_storage(x, ref):
    """As rel_err, after discounting half a bf16 ulp of the reference (the storage rounding)."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-300))) - 8)
    den = np.max(np.abs(ref))
    return float(np.max(np.maximum(np.abs(x - ref) - half_ulp, 0.0)) / (den if den > 0 else 1.0))


def window_problem(num_seqs, window, d, qkv, state, decay, seed, hk=2, hv=4):
    return workloads.make_problem("verify", num_seqs=num_seqs, lengths=[window] * num_seqs,
                                  num_k_heads=hk, num_v_heads=hv, d=d, qkv_dtype=qkv,
                                  state_dtype=state, decay_kind=decay, chunk=64,
                                  zero_state=False, num_slots=num_seqs + 3, seed=seed)


def run_verify(p, window):
    t = torch_io.prefill_inputs(p, DEV)
    o, ring = kda.verify_window(t["q"], t["k"], t["v"], t["beta"], t["log_decay"], t["slot_idx"],
                                t["state_pool"], window=window, scale=p.scale)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    return t, o, ring


def oracle_prefix(p, window, accepted):
    """The oracle over the first accepted[b] tokens of each sequence's window."""
    rows = np.concatenate([np.arange(b * window, b * window + a) for b, a in enumerate(accepted)]
                          + [np.zeros(0, np.int64)]).astype(np.int64)
    offsets = np.zeros(len(accepted) + 1, np.int64)
    offsets[1:] = np.cumsum(accepted)
    f = lambda x: workloads.as_f32(x, p.qkv_dtype)[rows]
    return oracle.run_arrays(offsets=offsets, slot_idx=p.slot_idx, q=f(p.q), k=f(p.k), v=f(p.v),
                             beta=p.beta[rows], g=p.g[rows],
                             per_channel=(p.decay_kind == "per_channel"),
                             pool=workloads.as_f32(p.pool, p.state_dtype), scale=p.scale)


CASES = [(128, "bf16", "f32", "per_channel"), (128, "bf16", "bf16", "per_channel"),
         (128, "bf16", "f32", "scalar"), (128, "bf16", "bf16", "scalar"),
         (128, "f32", "f32", "per_channel"), (16, "f32", "f32", "scalar"),
         (16, "bf16", "bf16", "per_channel")]


@pytest.mark.parametrize("d,qkv,state,decay", CASES)
@pytest.mark.parametrize("window", [1, 7, 64])
def test_verify_outputs_match_oracle_and_leave_the_pool_untouched(d, qkv, state, decay, window):
    p = window_problem(5, window, d, qkv, state, decay, seed=300 + window + d)
    before = torch_io.prefill_inputs(p, DEV)["state_pool"]
    t, o, ring = run_verify(p, window)
    o_ref, _ = oracle.run(p)
    assert rel_err(o.double().cpu().numpy(), o_ref) <= TOL[qkv]
    assert torch.equal(t["state_pool"], before)
    assert ring.shape == (5, window, 4, 3 * d if decay == "per_channel" else 2 * d + 4)


@pytest.mark.parametrize("d,qkv,state,decay", CASES)
def test_fold_of_accepted_prefix_matches_oracle(d, qkv, state, decay):
    window = 12
    accepted = np.array([0, 12, 5, 1, 11, 7], np.int64)
    p = window_problem(len(accepted), window, d, qkv, state, decay, seed=400 + d)
    t, _, ring = run_verify(p, window)
    pool = t["state_pool"]
    before = pool.clone()
    acc = torch.tensor(accepted, dtype=torch.int32, device=DEV)
    kda.fold_accepted(ring, acc, t["slot_idx"], pool, window=window, num_k_heads=p.num_k_heads,
                      per_channel=(decay == "per_channel"))
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    _, pool_ref = oracle_prefix(p, window, accepted)
    got = torch_io.pool_to_f64(pool)
    slots = np.asarray(p.slot_idx, np.int64)
    err = rel_err_bf16_storage if state == "bf16" else rel_err
    assert err(got[slots], pool_ref[slots]) <= TOL[qkv]
    # accepted = 0 leaves the slot bit-identical; slots no sequence names are untouched
    assert torch.equal(pool[int(slots[0])], before[int(slots[0])])
    untouched = sorted(set(range(p.num_slots)) - set(slots.tolist()))
    assert torch.equal(pool[untouched], before[untouched])


def test_ring_records_hold_normalised_key_correction_and_decay():
    """Record contents at t = 0, from the pages' definitions: k^ = k/|k|, alpha = exp(g),
    e = beta (v - (S0 Diag(alpha))^T k^) with S0 the slot's state."""
    p = window_problem(3, 4, 128, "bf16", "f32", "per_channel", seed=77)
    _, _, ring = run_verify(p, 4)
    ring = ring.double().cpu().numpy()
    k = workloads.as_f32(p.k, "bf16").astype(np.float64)
    v = workloads.as_f32(p.v, "bf16").astype(np.float64)
    pool = workloads.as_f32(p.pool, "f32").astype(np.float64)
    D, HV = 128, 4
    for b in range(3):
        row = b * 4
        for h in range(HV):
            kh = k[row, h // 2]
            khat = kh / np.sqrt(kh @ kh + 1e-6)
            alpha = np.exp(p.g[row, h].astype(np.float64))
            S0 = pool[p.slot_idx[b], h]                     # [d_k, d_v]
            e = p.beta[row, h] * (v[row, h] - (alpha[:, None] * S0).T @ khat)
            rec = ring[b, 0, h]
            assert np.max(np.abs(rec[:D] - khat)) <= 1e-5
            assert rel_err(rec[D:2 * D], e) <= 1e-4
            assert rel_err(rec[2 * D:], alpha) <= 1e-6


def test_fold_of_whole_window_equals_prefill():
    """Folding every record equals running the window through the prefill."""
    p = window_problem(4, 40, 128, "bf16", "f32", "scalar", seed=91)
    t, o, ring = run_verify(p, 40)
    pool_fold = t["state_pool"]
    acc = torch.full((4,), 40, dtype=torch.int32, device=DEV)
    kda.fold_accepted(ring, acc, t["slot_idx"], pool_fold, window=40, per_channel=False)
    t2 = torch_io.prefill_inputs(p, DEV)
    o_pf = kda.prefill(**t2, chunk=64, scale=p.scale)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    assert rel_err(o.double().cpu().numpy(), o_pf.double().cpu().numpy()) <= TOL["bf16"]
    slots = t["slot_idx"].long()
    assert rel_err(pool_fold[slots].double().cpu().numpy(),
                   t2["state_pool"][slots].double().cpu().numpy()) <= TOL["bf16"]


def test_fold_rejects_more_accepted_than_the_window():
    """accepted[b] > window sets the device error and leaves that sequence's slot alone;
    the other sequences are folded."""
    p = window_problem(3, 6, 128, "bf16", "f32", "per_channel", seed=55)
    t, _, ring = run_verify(p, 6)
    pool = t["state_pool"]
    before = pool.clone()
    acc = torch.tensor([3, 7, 6], dtype=torch.int32, device=DEV)
    kda.fold_accepted(ring, acc, t["slot_idx"], pool, window=6)
    assert kda.get_device_error() == 6
    s = [int(x) for x in p.slot_idx]
    assert torch.equal(pool[s[1]], before[s[1]])
    assert not torch.equal(pool[s[0]], before[s[0]])
    bad = torch.tensor([0, 99, 1], dtype=torch.int32, device=DEV)
    kda.verify_window(t["q"], t["k"], t["v"], t["beta"], t["log_decay"], bad, pool, window=6)
    assert kda.get_device_error() == 2
    assert kda.get_device_error() == 0


@pytest.mark.parametrize("qkv", ["bf16", "f32"])
def test_verify_with_log_decay_only_4_byte_aligned(qkv):
    """Per-channel log-decay rows are staged in 16-byte pieces when the array is 16-byte aligned
    and in 4-byte pieces otherwise (the entry point asks for 4 bytes): both give the same o and
    ring."""
    window = 9
    p = window_problem(6, window, 128, qkv, "f32", "per_channel", seed=515)
    t = torch_io.prefill_inputs(p, DEV)
    g = t["log_decay"]
    buf = torch.empty(g.numel() + 1, dtype=g.dtype, device=DEV)
    g_off = buf[1:].view(g.shape)
    g_off.copy_(g)
    assert g_off.data_ptr() % 16 == 4
    outs = []
    for lg in (g, g_off):
        o, ring = kda.verify_window(t["q"], t["k"], t["v"], t["beta"], lg, t["slot_idx"], t["state_pool"],
                                    window=window, scale=p.scale)
        torch.cuda.synchronize()
        assert kda.get_device_error() == 0
        outs.append((o, ring))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    o_ref, _ = oracle.run(p)
    assert rel_err(outs[1][0].double().cpu().numpy(), o_ref) <= TOL[qkv]
