"""Host-side pieces of bench.py that feed its JSON line, checked on CPU: the algorithmic byte
and tensor-core FLOP models against hand counts for the gdn_prefill shapes, and the reference
arm's line (the oracle timed on the host, on the kda_prefill headline workload) against the
contract's keys."""
import json
import os
import subprocess
import sys
from types import SimpleNamespace

import numpy as np

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def shapes(lengths, hk, hv, decay_kind, state_dtype="f32"):
    """The shape fields the models read, without drawing the workload's tensors."""
    lengths = np.asarray(lengths, np.int64)
    return SimpleNamespace(lengths=lengths, total_tokens=int(lengths.sum()), num_k_heads=hk,
                           num_v_heads=hv, d_k=128, d_v=128, qkv_dtype="bf16",
                           state_dtype=state_dtype, decay_kind=decay_kind)


GDN_PREFILL = shapes([4096] * 4, 16, 16, "scalar")        # the gdn_prefill workload's sizes
KDA_PREFILL = shapes([16384] * 2, 32, 32, "per_channel")   # the kda_prefill workload's sizes


def test_prefill_algorithmic_bytes_gdn_prefill():
    """4 x 4096 tokens, 16 key and value heads, d = 128, bf16 q/k/v, fp32 beta, scalar
    log-decay, fp32 o and an fp32 state read and written once per live sequence."""
    b = bench.prefill_algorithmic_bytes(GDN_PREFILL)
    T, H, d = 16384, 16, 128
    assert b["q"] == b["k"] == b["v"] == T * H * d * 2 == 67108864
    assert b["beta"] == b["g"] == T * H * 4
    assert b["o"] == T * H * d * 4
    assert b["state"] == 2 * 4 * H * d * d * 4
    assert sum(b.values()) == 346030080


def test_prefill_algorithmic_bytes_per_channel_decay():
    b = bench.prefill_algorithmic_bytes(KDA_PREFILL)
    assert b["g"] == 32768 * 32 * 128 * 4


def test_tensor_core_flops_gdn_prefill():
    """Per (chunk, value head): the A-GEMM [K; Q] K^T (M 128, N 64, K 128) and two M 128 N 64
    K 64 products in the front; per chunk, value head and 64-column value tile in the chain
    one M 128 N 64 K 128 product and two M 128 N 64 K 64 products."""
    f = bench.tc_executed_flops(GDN_PREFILL)
    units = 4 * (4096 // 64) * 16

    def mma(m, n, k):
        return 2 * m * n * k

    front = mma(128, 64, 128) + 2 * mma(128, 64, 64)
    chain = 2 * (mma(128, 64, 128) + 2 * mma(128, 64, 64))
    assert f["tc_front"] == front * units == 17179869184
    assert f["tc_chain"] == chain * units == 34359738368
    g = bench.tc_executed_flops(KDA_PREFILL)
    kda_units = 2 * (16384 // 64) * 32
    assert g["tc_front"] == (3 * mma(128, 64, 128) + 2 * mma(128, 64, 64)) * kda_units


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` times the oracle on the host and prints one JSON line with
    the metric, its unit, the CPU-baseline block and an end-to-end block that moves no bytes."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == "prefill tokens/s" and line["unit"] == "tokens/s"
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["steps"] == 1 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["config"]["workload"] == "kda_prefill"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
