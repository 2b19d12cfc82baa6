"""The front end before the recurrence (kda_conv_gates_fwd through the C ABI) against the fp64
oracle of `oracle/conv.py`, and the front end feeding the prefill against the two oracles in
sequence.

Tolerances: y in bf16 is compared after discounting half a bf16 ulp of the reference (its
storage rounding) against the 2e-3 bound, y in fp32 against 1e-4; the gates against 1e-5
(fp32 transcendental functions); the conv state holds copies of inputs and is compared exactly.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_deltanet_gb300 as kda
import oracle
from oracle import conv as oc

pytestmark = pytest.mark.gpu
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


def to_dev(arr, dtype):
    t = torch.from_numpy(np.ascontiguousarray(arr, np.float32))
    return t.to(DEV).to(torch.bfloat16 if dtype == "bf16" else torch.float32)


def exact(arr, dtype):
    """The values a tensor of `dtype` holds (bf16: round to nearest even), as fp64."""
    t = torch.from_numpy(np.ascontiguousarray(arr, np.float32))
    if dtype == "bf16":
        t = t.to(torch.bfloat16).to(torch.float32)
    return t.numpy().astype(np.float64)


def inputs(seed, lens, HK, HV, d, dtype, W, per_channel, num_slots):
    r = np.random.Generator(np.random.PCG64(seed))
    T = int(sum(lens))
    CD = (2 * HK + HV) * d
    return dict(
        x=exact(r.standard_normal((T, CD)), dtype),
        w=(r.standard_normal((CD, W)) * 0.5).astype(np.float32),
        bias=(r.standard_normal(CD) * 0.1).astype(np.float32),
        a=r.standard_normal((T, HV, d) if per_channel else (T, HV)).astype(np.float32),
        b=r.standard_normal((T, HV)).astype(np.float32),
        A_log=(r.standard_normal(HV) * 0.5).astype(np.float32),
        dt_bias=(r.standard_normal(HV * d if per_channel else HV) * 0.5).astype(np.float32),
        state=exact(r.standard_normal((num_slots, CD, W - 1)), dtype),
        offsets=np.concatenate([[0], np.cumsum(lens)]).astype(np.uint32),
        slots=r.permutation(num_slots)[:len(lens)].astype(np.uint32),
    )


def run_gpu(x, HK, HV, d, dtype, offsets=True):
    t = {k: to_dev(x[k], dtype if k in ("x", "state") else "f32")
         for k in ("x", "w", "bias", "a", "b", "A_log", "dt_bias", "state")}
    off = torch.from_numpy(x["offsets"].astype(np.int32)).to(DEV) if offsets else None
    slots = torch.from_numpy(x["slots"].astype(np.int32)).to(DEV)
    y, g, beta = kda.conv_gates(t["x"], t["w"], t["a"], t["b"], num_k_heads=HK, num_v_heads=HV,
                                d=d, conv_bias=t["bias"], A_log=t["A_log"], dt_bias=t["dt_bias"],
                                input_row_offsets=off, slot_idx=slots, conv_state=t["state"])
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    return y, g, beta, t["state"]


def run_oracle(x, HV, per_channel, offsets=None):
    return oc.conv_gates(x=x["x"], weight=x["w"], bias=x["bias"], a=x["a"], b=x["b"],
                         A_log=x["A_log"], dt_bias=x["dt_bias"],
                         offsets=x["offsets"] if offsets is None else offsets,
                         slot_idx=x["slots"], conv_state=x["state"], num_v_heads=HV,
                         per_channel=per_channel)


CASES = [
    # name, lens, HK, HV, d, dtype, W, per_channel
    ("bf16-w4-kda", [70, 0, 1, 3, 130], 2, 4, 128, "bf16", 4, True),
    ("bf16-w2-gdn", [65, 64, 2], 1, 2, 128, "bf16", 2, False),
    ("f32-w4-d16", [9, 0, 40, 1], 2, 2, 16, "f32", 4, True),
    ("f32-w3-d16", [5, 77], 1, 1, 16, "f32", 3, False),
    ("bf16-w1", [33, 31], 1, 1, 128, "bf16", 1, False),
]


@pytest.mark.parametrize("cfg", CASES, ids=[c[0] for c in CASES])
def test_conv_gates_match_oracle(cfg):
    name, lens, HK, HV, d, dtype, W, pc = cfg
    x = inputs(sum(map(ord, name)), lens, HK, HV, d, dtype, W, pc, len(lens) + 2)
    if W > 1:                                   # with a conv-state pool
        y, g, beta, state = run_gpu(x, HK, HV, d, dtype)
    else:                                       # one tap: no state to carry
        x["state"] = None
        y, g, beta, state = run_gpu_nostate(x, HK, HV, d, dtype)
    y_ref, g_ref, beta_ref, state_ref = run_oracle(x, HV, pc)
    yy = y.double().cpu().numpy()
    ey = rel_err_bf16_storage(yy, y_ref) if dtype == "bf16" else rel_err(yy, y_ref)
    assert ey <= (2e-3 if dtype == "bf16" else 1e-4), ey
    assert rel_err(g.double().cpu().numpy(), g_ref) <= 1e-5
    assert rel_err(beta.double().cpu().numpy(), beta_ref) <= 1e-5
    if W > 1:
        np.testing.assert_array_equal(state.double().cpu().numpy(), state_ref)


def run_gpu_nostate(x, HK, HV, d, dtype):
    t = {k: to_dev(x[k], dtype if k == "x" else "f32")
         for k in ("x", "w", "bias", "a", "b", "A_log", "dt_bias")}
    off = torch.from_numpy(x["offsets"].astype(np.int32)).to(DEV)
    y, g, beta = kda.conv_gates(t["x"], t["w"], t["a"], t["b"], num_k_heads=HK, num_v_heads=HV,
                                d=d, conv_bias=t["bias"], A_log=t["A_log"], dt_bias=t["dt_bias"],
                                input_row_offsets=off)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    return y, g, beta, None


def test_decode_form_steps_equal_the_prefill_form():
    """One token per sequence per call (no offsets), the conv state carried between calls,
    equals one call over the sequences those tokens form."""
    B, steps, HK, HV, d, W = 5, 6, 1, 2, 128, 4
    x = inputs(91, [steps] * B, HK, HV, d, "bf16", W, True, B + 2)
    _, _, _, state_ref = run_oracle(x, HV, True)
    y_ref, _, _, _ = run_oracle(x, HV, True)
    t = {k: to_dev(x[k], "bf16" if k in ("x", "state") else "f32")
         for k in ("x", "w", "bias", "a", "b", "A_log", "dt_bias", "state")}
    slots = torch.from_numpy(x["slots"].astype(np.int32)).to(DEV)
    ys = []
    for s in range(steps):
        rows = torch.arange(B, device=DEV) * steps + s
        y, _, _ = kda.conv_gates(t["x"][rows].contiguous(), t["w"], t["a"][rows].contiguous(),
                                 t["b"][rows].contiguous(), num_k_heads=HK, num_v_heads=HV, d=d,
                                 conv_bias=t["bias"], A_log=t["A_log"], dt_bias=t["dt_bias"],
                                 slot_idx=slots, conv_state=t["state"])
        ys.append(y)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    y = torch.stack(ys, 1).reshape(B * steps, -1).double().cpu().numpy()
    assert rel_err_bf16_storage(y, y_ref) <= 2e-3
    np.testing.assert_array_equal(t["state"].double().cpu().numpy(), state_ref)


@pytest.mark.parametrize("per_channel", [False, True])
def test_front_end_feeds_the_prefill(per_channel):
    """y's column blocks are q, k, v of the prefill (row stride conv_dim), with the gates as
    beta and log-decay: the outputs and final states match the prefill oracle run on the
    front-end oracle's outputs."""
    lens, HK, HV, d, W = [150, 0, 64, 7], 2, 4, 128, 4
    x = inputs(17 + per_channel, lens, HK, HV, d, "bf16", W, per_channel, len(lens) + 2)
    # a slow decay rate (log-decay about -0.03 per token), the regime of the tensor-core path
    x["A_log"][:] = np.float32(np.log(0.05))
    y, g, beta, _ = run_gpu(x, HK, HV, d, "bf16")
    T, kd = y.shape[0], HK * d
    q = y[:, :kd].view(T, HK, d)
    k = y[:, kd:2 * kd].view(T, HK, d)
    v = y[:, 2 * kd:].view(T, HV, d)
    r = np.random.Generator(np.random.PCG64(5))
    pool0 = (r.standard_normal((len(lens) + 2, HV, d, d)) * 0.02).astype(np.float32)
    pool = torch.from_numpy(pool0).to(DEV)
    off = torch.from_numpy(x["offsets"].astype(np.int32)).to(DEV)
    slots = torch.from_numpy(x["slots"].astype(np.int32)).to(DEV)
    o = kda.prefill(q, k, v, beta, g, off, slots, pool, chunk=64)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    y_ref, g_ref, beta_ref, _ = run_oracle(x, HV, per_channel)
    yb = exact(y_ref, "bf16")                            # the front end's bf16 output
    o_ref, pool_ref = oracle.run_arrays(
        offsets=x["offsets"].astype(np.int64), slot_idx=x["slots"].astype(np.int64),
        q=yb[:, :kd].reshape(T, HK, d), k=yb[:, kd:2 * kd].reshape(T, HK, d),
        v=yb[:, 2 * kd:].reshape(T, HV, d), beta=beta_ref.astype(np.float32),
        g=g_ref.astype(np.float32), per_channel=per_channel, pool=pool0.astype(np.float64))
    assert rel_err(o.double().cpu().numpy(), o_ref) <= 2e-3
    touched = x["slots"].astype(np.int64)
    assert rel_err(pool.double().cpu().numpy()[touched], pool_ref[touched]) <= 2e-3
