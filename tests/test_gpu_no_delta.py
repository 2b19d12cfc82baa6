"""The additive write (KDA_FLAG_NO_DELTA, `delta_rule=False`) through the C ABI against the fp64
oracle's recurrence with the correction's prediction left out (e_t = beta_t v_t).

Cases: Gated Linear Attention (per-channel gate), Mamba-2 (scalar gate, beta the write step),
RetNet (one constant decay) and plain causal linear attention (no decay, beta = 1)
("Linear attention visualized", those sections; "From Attention to Learned Memory", sec. 1-2),
on every prefill path (two tensor-core kernels, the single tensor-core kernel, CUDA cores),
the decode step, and the verify window with the fold of its accepted prefix.

Tolerance as the other parity tests: rel = max|x - ref| / max|ref| per tensor, <= 2e-3 for
bf16 q/k/v and <= 1e-4 for fp32; a bf16 pool is compared after discounting half a bf16 ulp.
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
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-300))) - 8)
    den = np.max(np.abs(ref))
    return float(np.max(np.maximum(np.abs(x - ref) - half_ulp, 0.0)) / (den if den > 0 else 1.0))


def problem(name, lengths, HK, HV, d, qkv, state, decay, chunk, gate="random", seed=0):
    """A seeded ragged problem; gate 'random' keeps the generated gate and beta, 'retnet' sets
    one constant log-decay, 'none' sets log-decay 0 and beta 1 (plain linear attention)."""
    p = workloads.make_problem(name, num_seqs=len(lengths), lengths=lengths, num_k_heads=HK,
                               num_v_heads=HV, d=d, qkv_dtype=qkv, state_dtype=state,
                               decay_kind=decay, chunk=chunk, zero_state=False,
                               num_slots=len(lengths) + 3, seed=seed)
    if gate == "retnet":
        p.g[...] = np.float32(np.log(0.97))
    elif gate == "none":
        p.g[...] = 0.0
        p.beta[...] = 1.0
    return p


def check(p, **kw):
    t = torch_io.prefill_inputs(p, DEV)
    o = kda.prefill(**t, chunk=p.chunk, scale=p.scale, delta_rule=False, **kw)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    o = o.double().cpu().numpy()
    pool = torch_io.pool_to_f64(t["state_pool"])
    o_ref, pool_ref = oracle.run(p, delta_rule=False)
    touched = np.asarray(p.slot_idx, np.int64)
    tol = TOL[p.qkv_dtype]
    eo = rel_err(o, o_ref)
    es = (rel_err_bf16_storage if p.state_dtype == "bf16" else rel_err)(pool[touched],
                                                                        pool_ref[touched])
    assert eo <= tol and es <= tol, f"{p.name}: o err {eo:.3e}, state err {es:.3e} (tol {tol})"
    untouched = np.setdiff1d(np.arange(p.num_slots), touched)
    np.testing.assert_array_equal(pool[untouched],
                                  torch_io.pool_to_f64(torch_io.tensor(p.pool, p.state_dtype))[untouched])
    # the additive write really differs from the delta rule on these inputs
    o_delta, _ = oracle.run(p)
    assert rel_err(o_ref, o_delta) > 10 * tol


CASES = [
    # name, lengths, HK, HV, d, qkv, state, decay, chunk, gate, path
    ("gla-tc", [300, 1, 63, 65, 128], 2, 4, 128, "bf16", "f32", "per_channel", 64, "random", {}),
    ("mamba2-tc", [257, 31, 64], 4, 4, 128, "bf16", "f32", "scalar", 64, "random", {}),
    ("retnet-tc-bf16pool", [200, 90], 1, 2, 128, "bf16", "bf16", "scalar", 64, "retnet", {}),
    ("linear-attn-tc", [150, 64, 7], 2, 2, 128, "bf16", "f32", "scalar", 64, "none", {}),
    ("gla-compact", [300, 1, 65], 2, 4, 128, "bf16", "f32", "per_channel", 64, "random",
     {"compact": True}),
    ("mamba2-compact", [129, 40], 2, 2, 128, "bf16", "bf16", "scalar", 64, "random",
     {"compact": True}),
    ("gla-cuda-cores", [130, 17], 2, 4, 128, "bf16", "f32", "per_channel", 64, "random",
     {"cuda_cores": True}),
    ("gla-f32-d16-c16", [1, 15, 16, 17, 100], 1, 2, 16, "f32", "f32", "per_channel", 16, "random",
     {}),
    ("linear-attn-f32-d16-c32", [33, 70], 2, 2, 16, "f32", "f32", "scalar", 32, "none", {}),
    ("gla-f32-d128-c32", [81, 47], 2, 4, 128, "f32", "bf16", "per_channel", 32, "random", {}),
]


@pytest.mark.parametrize("cfg", CASES, ids=[c[0] for c in CASES])
def test_additive_write_prefill(cfg):
    name, lengths, HK, HV, d, qkv, state, decay, chunk, gate, kw = cfg
    check(problem(name, lengths, HK, HV, d, qkv, state, decay, chunk, gate,
                  seed=sum(map(ord, name))), **kw)


def test_additive_write_full_prefill_workload():
    """The gdn_prefill shapes (4 x 4096 tokens, 16 heads, d=128, scalar gate) as Mamba-2:
    every output and final state."""
    check(workloads.workload("gdn_prefill"))


@pytest.mark.parametrize("decay,state", [("per_channel", "f32"), ("scalar", "bf16")])
def test_additive_write_decode(decay, state):
    dp = workloads.make_decode_problem("dec", num_seqs=5, steps=7, num_k_heads=2, num_v_heads=4,
                                       d=128, qkv_dtype="bf16", state_dtype=state,
                                       decay_kind=decay, zero_state=False, seed=23, num_slots=9)
    t = torch_io.decode_inputs(dp, DEV)
    outs = [kda.decode_step(t["q"][s], t["k"][s], t["v"][s], t["beta"][s], t["log_decay"][s],
                            t["slot_idx"], t["state_pool"], delta_rule=False)
            for s in range(dp.steps)]
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    o = torch.stack(outs).double().cpu().numpy()
    o_ref, pool_ref = oracle.run_decode(dp, delta_rule=False)
    pool = torch_io.pool_to_f64(t["state_pool"])
    touched = dp.slot_idx.astype(np.int64)
    assert rel_err(o, o_ref) <= TOL["bf16"]
    if state == "bf16":
        # both sides round to bf16 after every step, from values within the tolerance of each
        # other: the two roundings can land on adjacent bf16 values, one ulp apart
        ref = pool_ref[touched]
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-300))) - 7)
        es = float(np.max(np.maximum(np.abs(pool[touched] - ref) - ulp, 0.0)) / np.max(np.abs(ref)))
    else:
        es = rel_err(pool[touched], pool_ref[touched])
    assert es <= TOL["bf16"], es


def test_additive_write_verify_and_fold():
    """The verify window's outputs are the additive recurrence's outputs over the window, its
    records hold e = beta v, and folding an accepted prefix gives the state after it."""
    window, accepted = 9, np.array([0, 9, 4, 1], np.int64)
    p = problem("verify", [window] * len(accepted), 2, 4, 128, "bf16", "f32", "per_channel", 64,
                seed=611)
    t = torch_io.prefill_inputs(p, DEV)
    o, ring = kda.verify_window(t["q"], t["k"], t["v"], t["beta"], t["log_decay"], t["slot_idx"],
                                t["state_pool"], window=window, scale=p.scale, delta_rule=False)
    torch.cuda.synchronize()
    o_ref, _ = oracle.run(p, delta_rule=False)
    assert rel_err(o.double().cpu().numpy(), o_ref) <= TOL["bf16"]
    v = workloads.as_f32(p.v, "bf16").astype(np.float64)
    e = p.beta.astype(np.float64)[:, :, None] * v                     # [B*window, HV, D]
    rec = ring.double().cpu().numpy().reshape(len(accepted) * window, 4, -1)[:, :, 128:256]
    assert rel_err(rec, e) <= 1e-6
    acc = torch.tensor(accepted, dtype=torch.int32, device=DEV)
    kda.fold_accepted(ring, acc, t["slot_idx"], t["state_pool"], window=window,
                      num_k_heads=p.num_k_heads, per_channel=True)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    rows = np.concatenate([np.arange(b * window, b * window + a)
                           for b, a in enumerate(accepted)]).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(accepted)]).astype(np.int64)
    f = lambda x: workloads.as_f32(x, "bf16")[rows]
    _, pool_ref = oracle.run_arrays(offsets=offsets, slot_idx=p.slot_idx, q=f(p.q), k=f(p.k),
                                    v=f(p.v), beta=p.beta[rows], g=p.g[rows], per_channel=True,
                                    pool=workloads.as_f32(p.pool, "f32"), scale=p.scale,
                                    delta_rule=False)
    slots = np.asarray(p.slot_idx, np.int64)
    got = torch_io.pool_to_f64(t["state_pool"])
    assert rel_err(got[slots], pool_ref[slots]) <= TOL["bf16"]
