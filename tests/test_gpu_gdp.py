"""Gated DeltaProduct on the GPU (kda_gdp_prefill_fwd / kda_gdp_decode_step through the C ABI)
against the fp64 oracle's direct n_h-substep recurrence.

Tolerance as the other parity tests: rel = max|x - ref| / max|ref| per tensor, <= 2e-3 for bf16
q/k/v, <= 1e-4 for fp32; a bf16 pool is compared after discounting half a bf16 ulp.
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


def gpu_gdp(p, **kw):
    t = torch_io.prefill_inputs(p, DEV)
    o = kda.gdp_prefill(t["q"], t["k"], t["v"], t["beta"], t["log_decay"], t["input_row_offsets"],
                        t["slot_idx"], t["state_pool"], chunk=p.chunk, scale=p.scale, **kw)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    return o.double().cpu().numpy(), torch_io.pool_to_f64(t["state_pool"])


def check(p, **kw):
    o, pool = gpu_gdp(p, **kw)
    o_ref, pool_ref = oracle.run_gdp(p)
    tol = TOL[p.qkv_dtype]
    touched = np.asarray(p.slot_idx, np.int64)
    eo = rel_err(o, o_ref)
    es = (rel_err_bf16_storage if p.state_dtype == "bf16" else rel_err)(pool[touched],
                                                                        pool_ref[touched])
    assert eo <= tol and es <= tol, f"{p.name}: o err {eo:.3e}, state err {es:.3e} (tol {tol})"
    untouched = np.setdiff1d(np.arange(p.num_slots), touched)
    np.testing.assert_array_equal(pool[untouched],
                                  torch_io.pool_to_f64(torch_io.tensor(p.pool, p.state_dtype))[untouched])


SMALL = [
    # name, lengths, n_h, HK, HV, d, qkv, state, decay, chunk
    ("f32-d16-n2-scalar", [1, 17, 40], 2, 1, 2, 16, "f32", "f32", "scalar", 16),
    ("f32-d16-n3-kda-gqa", [5, 0, 33], 3, 2, 4, 16, "f32", "f32", "per_channel", 32),
    ("bf16-d128-n2-gdn", [100, 1, 64, 37], 2, 2, 2, 128, "bf16", "f32", "scalar", 64),
    ("bf16-d128-n3-kda", [70, 129], 3, 1, 2, 128, "bf16", "bf16", "per_channel", 64),
    ("bf16-d128-n1-kda", [90, 3], 1, 2, 4, 128, "bf16", "f32", "per_channel", 64),
    ("bf16-d128-n4-gdn-c16", [50], 4, 2, 2, 128, "bf16", "f32", "scalar", 16),
]


@pytest.mark.parametrize("cfg", SMALL, ids=[c[0] for c in SMALL])
def test_gdp_small(cfg):
    name, lengths, n_h, HK, HV, d, qkv, state, decay, chunk = cfg
    p = workloads.make_gdp_problem(name, num_seqs=len(lengths), lengths=lengths, n_h=n_h,
                                   num_k_heads=HK, num_v_heads=HV, d=d, qkv_dtype=qkv,
                                   state_dtype=state, decay_kind=decay, chunk=chunk,
                                   zero_state=False, num_slots=len(lengths) + 2,
                                   seed=sum(map(ord, name)))
    check(p)


def test_gdp_prefill_workload():
    """Every output and final state of gdp_prefill (4 x 4096 tokens, 2 substeps, 16 heads)."""
    check(workloads.workload("gdp_prefill"))


def test_gdp_one_substep_is_the_prefill():
    """n_h = 1 runs the plain prefill on the same inputs: identical results."""
    p = workloads.make_gdp_problem("n1", num_seqs=2, lengths=[130, 64], n_h=1, num_k_heads=2,
                                   num_v_heads=2, d=128, qkv_dtype="bf16", state_dtype="f32",
                                   decay_kind="per_channel", chunk=64, zero_state=False, seed=5)
    o1, pool1 = gpu_gdp(p)
    t = torch_io.prefill_inputs(p, DEV)
    o2 = kda.prefill(t["q"], t["k"][:, 0], t["v"][:, 0], t["beta"][:, 0], t["log_decay"],
                     t["input_row_offsets"], t["slot_idx"], t["state_pool"], chunk=64)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(o1, o2.double().cpu().numpy())
    np.testing.assert_array_equal(pool1, torch_io.pool_to_f64(t["state_pool"]))


@pytest.mark.parametrize("decay,state", [("scalar", "f32"), ("per_channel", "bf16")])
def test_gdp_decode_steps(decay, state):
    """Consecutive decode steps, one token of n_h transitions per sequence each, equal the
    oracle over the sequences those tokens form."""
    B, steps, n_h = 6, 5, 3
    p = workloads.make_gdp_problem("dec", num_seqs=B, lengths=[steps] * B, n_h=n_h,
                                   num_k_heads=2, num_v_heads=4, d=128, qkv_dtype="bf16",
                                   state_dtype=state, decay_kind=decay, chunk=64,
                                   zero_state=False, num_slots=B + 2, seed=17)
    t = torch_io.prefill_inputs(p, DEV)
    pool = t["state_pool"]
    outs = []
    for s in range(steps):
        rows = torch.arange(B, device=DEV) * steps + s
        outs.append(kda.gdp_decode_step(t["q"][rows].contiguous(), t["k"][rows].contiguous(),
                                        t["v"][rows].contiguous(), t["beta"][rows].contiguous(),
                                        t["log_decay"][rows].contiguous(), t["slot_idx"], pool))
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    o = torch.stack(outs, 1).reshape(B * steps, 4, 128).double().cpu().numpy()
    # the oracle step by step; a bf16 pool is stored in bf16 between calls (the pool dtype is
    # the storage dtype), so its fp64 state is rounded to bf16 after each step
    qf, kf, vf = (oracle._widen(x, "bf16") for x in (p.q, p.k, p.v))
    pool_ref = oracle._widen(p.pool, state).astype(np.float64)
    o_ref = np.zeros_like(o)
    for s in range(steps):
        rows = np.arange(B) * steps + s
        o_s, pool_ref = oracle.run_gdp_arrays(
            offsets=np.arange(B + 1), slot_idx=p.slot_idx, q=qf[rows], k=kf[rows], v=vf[rows],
            beta=p.beta[rows], g=p.g[rows], per_channel=(decay == "per_channel"), pool=pool_ref)
        if state == "bf16":
            pool_ref = oracle.round_to_bf16(pool_ref)
        o_ref[rows] = o_s
    touched = np.asarray(p.slot_idx, np.int64)
    eo = rel_err(o, o_ref)
    x, ref = torch_io.pool_to_f64(pool)[touched], pool_ref[touched]
    if state == "bf16":
        # both sides round to bf16 after every step, from values that differ within the
        # tolerance: the two roundings can land on adjacent bf16 values, one ulp apart
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-300))) - 7)
        es = float(np.max(np.maximum(np.abs(x - ref) - ulp, 0.0)) / np.max(np.abs(ref)))
    else:
        es = rel_err(x, ref)
    assert eo <= 2e-3 and es <= 2e-3, (eo, es)
