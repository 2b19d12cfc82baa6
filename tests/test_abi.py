"""The C ABI without a GPU: the library loads, exports every function include/kda.h declares,
and rejects bad arguments on the host (before anything touches CUDA)."""
import ctypes
import os
import re

import pytest
import torch

from gated_delta_rule_deltanet_gb300 import _lib, build as kbuild
from gated_delta_rule_deltanet_gb300.kda import make_params

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return _lib.load()


def declared_functions():
    with open(os.path.join(ROOT, "include", "kda.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_params_struct_layout_matches_header():
    # kda_params_t: 6 x int32, int64, 4 x int32, float, int32, uint32, (pad), 3 x int64
    assert ctypes.sizeof(_lib.KdaParams) == 88
    assert _lib.KdaParams.total_tokens.offset == 24
    assert _lib.KdaParams.q_row_stride.offset == 64


def test_version_and_strings(lib):
    assert lib.kda_abi_version() == 1
    for s in range(6):
        assert lib.kda_status_string(s)
    assert lib.kda_status_string(0) == b"ok"


def good(**kw):
    base = dict(num_seqs=2, num_k_heads=4, num_v_heads=8, d=128, num_slots=4, total_tokens=100,
                chunk=64)
    base.update(kw)
    return make_params(**base)


def ws_status(lib, p):
    n = ctypes.c_size_t(0)
    return lib.kda_prefill_workspace_size(ctypes.byref(p), ctypes.byref(n)), n.value


def test_workspace_size_positive_and_monotone(lib):
    s, a = ws_status(lib, good())
    assert s == _lib.KDA_OK and a > 0
    s, b = ws_status(lib, good(total_tokens=10_000))
    assert s == _lib.KDA_OK and b > a
    s, c = ws_status(lib, good(num_seqs=0, total_tokens=0))
    assert s == _lib.KDA_OK


@pytest.mark.parametrize("kw,status", [
    (dict(num_k_heads=3), _lib.KDA_ERR_INVALID_ARG),        # HV % HK != 0
    (dict(num_k_heads=0), _lib.KDA_ERR_INVALID_ARG),
    (dict(num_slots=0), _lib.KDA_ERR_INVALID_ARG),
    (dict(num_seqs=-1), _lib.KDA_ERR_INVALID_ARG),
    (dict(total_tokens=-5), _lib.KDA_ERR_INVALID_ARG),
    (dict(total_tokens=1 << 31), _lib.KDA_ERR_INVALID_ARG),
    (dict(d=64), _lib.KDA_ERR_UNSUPPORTED),                 # head size not built
    (dict(chunk=48), _lib.KDA_ERR_UNSUPPORTED),             # chunk not in {16, 32, 64}
    (dict(chunk=128), _lib.KDA_ERR_UNSUPPORTED),
    (dict(q_row_stride=100), _lib.KDA_ERR_INVALID_ARG),     # narrower than a row
    (dict(q_row_stride=4 * 128 + 1), _lib.KDA_ERR_INVALID_ARG),  # rows not 16-byte aligned
])
def test_bad_params_rejected_on_host(lib, kw, status):
    assert ws_status(lib, good(**kw))[0] == status


def test_bad_enums_rejected(lib):
    p = good()
    p.qkv_dtype = 7
    assert ws_status(lib, p)[0] == _lib.KDA_ERR_INVALID_ARG
    p = good()
    p.decay_kind = 3
    assert ws_status(lib, p)[0] == _lib.KDA_ERR_INVALID_ARG
    p = good()
    p.flags = 0x80
    assert ws_status(lib, p)[0] == _lib.KDA_ERR_INVALID_ARG
    p = good()
    p.d_v = 16
    assert ws_status(lib, p)[0] == _lib.KDA_ERR_UNSUPPORTED


def test_null_and_misaligned_pointers_rejected_before_launch(lib):
    """These return before any CUDA call, so they run without a GPU."""
    p = good()
    P = ctypes.c_void_p
    a = P(1 << 20)                     # never dereferenced: validation fails first
    assert lib.kda_prefill_fwd(None, a, a, a, a, a, a, a, a, a, a, 1 << 30, None) == \
        _lib.KDA_ERR_INVALID_ARG
    assert lib.kda_prefill_fwd(ctypes.byref(p), a, a, a, a, a, None, a, a, a, a, 1 << 30,
                               None) == _lib.KDA_ERR_INVALID_ARG
    mis = P((1 << 20) + 8)
    assert lib.kda_prefill_fwd(ctypes.byref(p), mis, a, a, a, a, a, a, a, a, a, 1 << 30,
                               None) == _lib.KDA_ERR_INVALID_ARG
    # per-channel log-decay 16-byte aligned, scalar 4-byte (the latter then fails on the
    # missing workspace)
    g4 = P((1 << 20) + 4)
    pc = good(per_channel=True)
    assert lib.kda_prefill_fwd(ctypes.byref(pc), a, a, a, a, g4, a, a, a, a, None, 1 << 30,
                               None) == _lib.KDA_ERR_INVALID_ARG
    sc = good(per_channel=False)
    assert lib.kda_prefill_fwd(ctypes.byref(sc), a, a, a, a, g4, a, a, a, a, None, 1 << 30,
                               None) == _lib.KDA_ERR_WORKSPACE
    # workspace missing / too small / misaligned
    assert lib.kda_prefill_fwd(ctypes.byref(p), a, a, a, a, a, a, a, a, a, None, 1 << 30,
                               None) == _lib.KDA_ERR_WORKSPACE
    assert lib.kda_prefill_fwd(ctypes.byref(p), a, a, a, a, a, a, a, a, a, a, 16, None) == \
        _lib.KDA_ERR_WORKSPACE
    assert lib.kda_prefill_fwd(ctypes.byref(p), a, a, a, a, a, a, a, a, a, P((1 << 20) + 16),
                               1 << 30, None) == _lib.KDA_ERR_WORKSPACE
    # decode
    assert lib.kda_decode_step(ctypes.byref(p), a, a, a, a, None, a, a, a, None) == \
        _lib.KDA_ERR_INVALID_ARG
    assert lib.kda_decode_step(ctypes.byref(p), a, a, mis, a, a, a, a, a, None) == \
        _lib.KDA_ERR_INVALID_ARG
    assert lib.kda_get_device_error(None, None) == _lib.KDA_ERR_INVALID_ARG


def test_empty_batch_is_a_no_op(lib):
    """num_seqs = 0 returns OK without touching CUDA (nothing to do)."""
    p = good(num_seqs=0, total_tokens=0)
    assert lib.kda_prefill_fwd(ctypes.byref(p), None, None, None, None, None, None, None, None,
                               None, None, 0, None) == _lib.KDA_OK
    assert lib.kda_decode_step(ctypes.byref(p), None, None, None, None, None, None, None, None,
                               None) == _lib.KDA_OK


def test_path_query(lib):
    from gated_delta_rule_deltanet_gb300 import kda as K
    import torch
    assert K.uses_tensor_cores(good())                               # bf16, d=128, chunk 64
    assert not K.uses_tensor_cores(good(cuda_cores=True))
    assert not K.uses_tensor_cores(good(chunk=32))
    assert not K.uses_tensor_cores(good(qkv_dtype=torch.float32))
    assert not K.uses_tensor_cores(good(d=16))
    assert lib.kda_prefill_uses_tensor_cores(None) == -1


def test_ring_record_length(lib):
    """Records are [k^ | e | alpha]; scalar decay pads its one alpha to 4 floats so every
    record starts on a 16-byte boundary."""
    pc = make_params(num_seqs=1, num_k_heads=1, num_v_heads=1, d=128, num_slots=1)
    sc = make_params(num_seqs=1, num_k_heads=1, num_v_heads=1, d=128, num_slots=1,
                         per_channel=False)
    assert lib.kda_ring_record_elems(ctypes.byref(pc)) == 3 * 128
    assert lib.kda_ring_record_elems(ctypes.byref(sc)) == 2 * 128 + 4
    assert lib.kda_ring_record_elems(ctypes.byref(good(d=64))) == -1
    assert lib.kda_ring_record_elems(None) == -1


def test_verify_and_fold_reject_bad_arguments_before_launch(lib):
    p = good()
    a = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 4)
    args = [a] * 6
    for w in (0, 65, -1):
        assert lib.kda_verify_window(ctypes.byref(p), *args, w, a, a, a, None) == \
            _lib.KDA_ERR_INVALID_ARG
        assert lib.kda_fold_accepted(ctypes.byref(p), a, w, a, a, a, None) == \
            _lib.KDA_ERR_INVALID_ARG
    assert lib.kda_verify_window(ctypes.byref(p), *args, 4, a, a, None, None) == \
        _lib.KDA_ERR_INVALID_ARG                                   # no ring
    assert lib.kda_verify_window(ctypes.byref(p), *args, 4, a, a, odd, None) == \
        _lib.KDA_ERR_INVALID_ARG                                   # ring not 16-byte aligned
    assert lib.kda_fold_accepted(ctypes.byref(p), odd, 4, a, a, a, None) == \
        _lib.KDA_ERR_INVALID_ARG
    assert lib.kda_fold_accepted(ctypes.byref(p), a, 4, None, a, a, None) == \
        _lib.KDA_ERR_INVALID_ARG                                   # no accepted counts
    assert lib.kda_verify_window(ctypes.byref(good(d=64)), *args, 4, a, a, a, None) == \
        _lib.KDA_ERR_UNSUPPORTED
    empty = good(num_seqs=0)
    assert lib.kda_verify_window(ctypes.byref(empty), *([None] * 6), 4, None, None, None,
                                 None) == _lib.KDA_OK
    assert lib.kda_fold_accepted(ctypes.byref(empty), None, 4, None, None, None, None) == \
        _lib.KDA_OK


def test_compact_flag_shrinks_the_tensor_core_workspace(lib):
    """The two-kernel tensor-core form stores 57,856 bytes of chain operands per chunk
    and value head; the single-kernel form needs only the chunk table."""
    p = good(total_tokens=4096, num_seqs=2)
    c = good(total_tokens=4096, num_seqs=2, compact=True)
    assert lib.kda_prefill_uses_tensor_cores(ctypes.byref(c)) == 1
    full, small = ws_status(lib, p)[1], ws_status(lib, c)[1]
    assert full - small >= (4096 // 64) * 8 * 57856
    assert small < 64 * 1024
    q = good()
    q.flags |= 16                                           # an unknown flag
    assert ws_status(lib, q)[0] == _lib.KDA_ERR_INVALID_ARG
    nd = good(total_tokens=4096, num_seqs=2, delta_rule=False)  # additive write: same paths
    assert ws_status(lib, nd) == ws_status(lib, p)
    assert lib.kda_prefill_uses_tensor_cores(ctypes.byref(nd)) == 1


def gdp_ws(lib, p, n_h, decode=0):
    n = ctypes.c_size_t(0)
    st = lib.kda_gdp_workspace_size(ctypes.byref(p) if p is not None else None, n_h, decode,
                                    ctypes.byref(n))
    return st, int(n.value)


def test_gdp_rejects_bad_arguments_before_launch(lib):
    """Gated DeltaProduct: substep count, virtual length, pointers and workspace are checked
    on the host; the workspace covers the virtual sequence plus the prefill's own."""
    p = good(total_tokens=1024, num_seqs=2)
    for n_h in (0, -1, 65):
        assert gdp_ws(lib, p, n_h)[0] == _lib.KDA_ERR_INVALID_ARG
    st1, w1 = gdp_ws(lib, p, 1)
    st3, w3 = gdp_ws(lib, p, 3)
    assert st1 == st3 == _lib.KDA_OK and w3 > w1 > 0
    n = ctypes.c_size_t(0)
    assert lib.kda_prefill_workspace_size(ctypes.byref(p), ctypes.byref(n)) == _lib.KDA_OK
    assert w1 >= int(n.value) + 1024 * 8 * 128 * 4                   # virtual o at least
    big = good(total_tokens=(1 << 30), num_seqs=1)
    assert gdp_ws(lib, big, 2)[0] == _lib.KDA_ERR_UNSUPPORTED        # T * n_h >= 2^31
    assert gdp_ws(lib, good(total_tokens=1024, num_seqs=2, delta_rule=False), 2)[0] == \
        _lib.KDA_ERR_UNSUPPORTED                                     # defined on the delta rule
    dec = good(num_seqs=4, total_tokens=0, chunk=0)
    assert gdp_ws(lib, dec, 2, decode=1)[0] == _lib.KDA_OK           # decode: chunk 0 -> 64
    assert gdp_ws(lib, dec, 2, decode=0)[0] != _lib.KDA_OK
    a = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 8)
    args = [a] * 9
    assert lib.kda_gdp_prefill_fwd(ctypes.byref(p), 0, *args, a, 1 << 40, None) == \
        _lib.KDA_ERR_INVALID_ARG
    assert lib.kda_gdp_prefill_fwd(ctypes.byref(p), 2, a, a, a, a, a, None, a, a, a, a,
                                   1 << 40, None) == _lib.KDA_ERR_INVALID_ARG   # no offsets
    assert lib.kda_gdp_prefill_fwd(ctypes.byref(p), 2, a, mis, a, a, a, a, a, a, a, a,
                                   1 << 40, None) == _lib.KDA_ERR_INVALID_ARG   # misaligned k
    assert lib.kda_gdp_prefill_fwd(ctypes.byref(p), 2, *args, a, 16, None) == \
        _lib.KDA_ERR_WORKSPACE
    assert lib.kda_gdp_decode_step(ctypes.byref(dec), 2, a, a, a, a, a, None, a, a, a, 1 << 40,
                                   None) == _lib.KDA_ERR_INVALID_ARG            # no slots
    empty = good(num_seqs=0, total_tokens=0)
    assert lib.kda_gdp_prefill_fwd(ctypes.byref(empty), 2, *([None] * 10), 0, None) == _lib.KDA_OK


def test_backward_rejects_bad_arguments_before_launch(lib):
    """kda_prefill_bwd validates on the host like the forward: missing arrays, misalignment and
    a short workspace are refused before anything is launched; the workspace covers the
    recorded per-chunk states and their gradients."""
    p = good(total_tokens=1024, num_seqs=2)
    n = ctypes.c_size_t(0)
    assert lib.kda_prefill_bwd_workspace_size(ctypes.byref(p), ctypes.byref(n)) == _lib.KDA_OK
    chunks = 1024 // 64 + 2
    assert n.value >= 2 * chunks * 8 * 128 * 128 * 4                 # states and gradients
    assert lib.kda_prefill_bwd_workspace_size(ctypes.byref(good(chunk=48)),
                                              ctypes.byref(n)) == _lib.KDA_ERR_UNSUPPORTED
    # every call below must fail validation: none may reach a launch
    a = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 2)
    args = [a] * 17     # q k v beta g offsets slots pool d_o d_state dq dk dv dbeta dg d_state0 ws
    none_do = list(args)
    none_do[8] = None                                                 # d_o
    assert lib.kda_prefill_bwd(ctypes.byref(p), *none_do, 1 << 40, None) == \
        _lib.KDA_ERR_INVALID_ARG
    bad = list(args)
    bad[10] = mis                                                     # dq misaligned
    assert lib.kda_prefill_bwd(ctypes.byref(p), *bad, 1 << 40, None) == _lib.KDA_ERR_INVALID_ARG
    assert lib.kda_prefill_bwd(ctypes.byref(p), *args, 16, None) == _lib.KDA_ERR_WORKSPACE
    empty = good(num_seqs=0, total_tokens=0)
    assert lib.kda_prefill_bwd(ctypes.byref(empty), *([None] * 17), 0, None) == _lib.KDA_OK


def test_conv_front_end_rejects_bad_arguments_before_launch(lib):
    """kda_conv_gates_fwd checks widths, missing arrays, alignment and row strides on the host
    (every call below fails before any launch)."""
    p = good(total_tokens=64, num_seqs=2)
    a = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 4)
    args = [a] * 13          # x w bias a b A_log dt_bias offsets slots state y log_decay beta
    for width in (0, 5, -1):
        assert lib.kda_conv_gates_fwd(ctypes.byref(p), width, *args, None) == \
            _lib.KDA_ERR_UNSUPPORTED
    missing = list(args)
    missing[0] = None                                            # x
    assert lib.kda_conv_gates_fwd(ctypes.byref(p), 4, *missing, None) == _lib.KDA_ERR_INVALID_ARG
    nos = list(args)
    nos[8] = None                                                # state without slots
    assert lib.kda_conv_gates_fwd(ctypes.byref(p), 4, *nos, None) == _lib.KDA_ERR_INVALID_ARG
    bad = list(args)
    bad[10] = mis                                                # y misaligned
    assert lib.kda_conv_gates_fwd(ctypes.byref(p), 4, *bad, None) == _lib.KDA_ERR_INVALID_ARG
    strided = good(total_tokens=64, num_seqs=2, q_row_stride=1024)
    assert lib.kda_conv_gates_fwd(ctypes.byref(strided), 4, *args, None) == \
        _lib.KDA_ERR_INVALID_ARG
    empty = good(total_tokens=0, num_seqs=0)
    assert lib.kda_conv_gates_fwd(ctypes.byref(empty), 4, *([None] * 13), None) == _lib.KDA_OK


def test_backward_compact_workspace_is_bounded(lib):
    """KDA_FLAG_COMPACT bounds the backward's workspace on the tensor-core configuration:
    windows of chunk positions (512 (chunk, value head) slots) plus one checkpointed state per
    window and sequence.  On the kda_prefill shapes (2 x 16384 tokens, 32 heads, d = 128) it
    stays under 0.5 GiB, against several GB for the default form."""
    def size(**kw):
        n = ctypes.c_size_t(0)
        p = make_params(num_seqs=2, num_k_heads=32, num_v_heads=32, d=128, num_slots=2,
                            total_tokens=32768, **kw)
        assert lib.kda_prefill_bwd_workspace_size(ctypes.byref(p), ctypes.byref(n)) == _lib.KDA_OK
        return n.value
    default, compact = size(), size(compact=True)
    assert compact <= 512 * 2 ** 20 < 4 * 2 ** 30 < default
    # the bound does not grow with the sequence length, apart from the checkpoints (64 KB per
    # window of 8 chunks and head)
    n = ctypes.c_size_t(0)
    p4 = make_params(num_seqs=2, num_k_heads=32, num_v_heads=32, d=128, num_slots=2,
                         total_tokens=4 * 32768, compact=True)
    assert lib.kda_prefill_bwd_workspace_size(ctypes.byref(p4), ctypes.byref(n)) == _lib.KDA_OK
    assert n.value - compact <= 3 * 32768 // 64 // 8 * 32 * 128 * 128 * 4 + 2 ** 20
    # fp32 inputs run on CUDA cores, where the flag does not apply
    f32 = make_params(num_seqs=2, num_k_heads=32, num_v_heads=32, d=128, num_slots=2,
                          total_tokens=32768, qkv_dtype=torch.float32, compact=True)
    assert lib.kda_prefill_bwd_workspace_size(ctypes.byref(f32), ctypes.byref(n)) == _lib.KDA_OK
    assert n.value > 4 * 2 ** 30
