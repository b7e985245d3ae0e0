"""The C ABI on the host: the library loads, exports every declared entry
point, and rejects malformed arguments with the documented status before any
device work (these tests never launch a kernel and need no GPU)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ccv():
    from causal_depthwise_conv1d_gb300 import build
    build.build()
    import causal_depthwise_conv1d_gb300 as ccv
    ccv.load_library()
    return ccv


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(ccv_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(ccv):
    from causal_depthwise_conv1d_gb300 import binding
    names = declared_functions()
    assert {"ccv_fwd", "ccv_last_error", "ccv_last_kernel", "ccv_version"} <= set(names)
    lib = ctypes.CDLL(binding.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    nm = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True, text=True)
    if nm.returncode == 0:
        exported = set(re.findall(r"\bT (ccv_\w+)", nm.stdout))
        assert set(names) <= exported


def test_version(ccv):
    assert ccv.ccv_version() == (1, 0)


FAKE = 0x10000  # never dereferenced: validation rejects before any device work


def call(ccv, **kw):
    args = dict(x=FAKE, x_strides=(64, 16, 1), out=FAKE * 2, out_strides=(64, 16, 1), weight=FAKE * 3,
                weight_strides=(4, 1), bias=0, bias_stride=1, seq_idx=0, seq_idx_strides=None,
                initial_states=0, initial_states_strides=None, final_states_out=0,
                final_states_strides=None, B=2, C=4, L=16, K=4, dtype=0, activation=1, stream=0)
    args.update(kw)
    try:
        ccv.ccv_fwd_ptr(**args)
    except ccv.CcvError as e:
        return e.status, str(e)
    return 0, ""


@pytest.mark.parametrize("kw,status,needle", [
    (dict(K=1), 2, "K must be 2, 3 or 4"),
    (dict(K=5), 2, "K must be 2, 3 or 4"),
    (dict(K=0), 1, "K must be >= 1"),
    (dict(B=-1), 1, ">= 0"),
    (dict(L=-3), 1, ">= 0"),
    (dict(dtype=7), 1, "unknown dtype"),
    (dict(activation=3), 1, "unknown activation"),
    (dict(x=0), 1, "x is required"),
    (dict(out=0), 1, "out is required"),
    (dict(weight=0), 1, "weight is required"),
    (dict(x_strides=None), 1, "x is required"),
    (dict(out=FAKE), 1, "alias"),
    (dict(out=FAKE + 4), 1, "overlaps"),
    (dict(out_strides=(64, 0, 1)), 1, "zero stride"),
    (dict(seq_idx=FAKE * 5, seq_idx_strides=(16, 1), initial_states=FAKE * 6,
          initial_states_strides=(12, 3, 1)), 2, "seq_idx together with initial_states"),
    (dict(seq_idx=FAKE * 5), 1, "seq_idx_strides is required"),
    (dict(initial_states=FAKE * 6), 1, "initial_states_strides is required"),
    (dict(final_states_out=FAKE * 7), 1, "final_states_strides is required"),
    (dict(final_states_out=FAKE * 7, final_states_strides=(12, 0, 1)), 1, "zero stride"),
    (dict(final_states_out=FAKE, final_states_strides=(12, 3, 1)), 1, "must not alias"),
    (dict(x=FAKE + 2), 1, "aligned"),
    (dict(dtype=1, out=FAKE * 2 + 1), 1, "aligned"),
    (dict(seq_idx=FAKE * 5 + 2, seq_idx_strides=(16, 1)), 1, "aligned"),
    (dict(x_strides=(1 << 62, 16, 1)), 1, "overflows"),
    (dict(B=1 << 40, C=1 << 20, L=1 << 10), 1, "too large"),
])
def test_validation_errors(ccv, kw, status, needle):
    st, msg = call(ccv, **kw)
    assert st == status, msg
    assert needle in msg
    assert needle in ccv.ccv_last_error()


def test_zero_sized_problems_are_noops(ccv):
    assert call(ccv, B=0)[0] == 0
    assert call(ccv, C=0)[0] == 0
    assert ccv.ccv_last_kernel() == "none"


def call_update(ccv, **kw):
    from causal_depthwise_conv1d_gb300 import binding
    import ctypes
    args = dict(x=FAKE, xs=(16, 4, 1), out=FAKE * 2, os=(16, 4, 1), state=FAKE * 4, ss=(12, 3, 1),
                w=FAKE * 3, ws=(4, 1), bias=0, bs=1, B=2, C=4, S=1, K=4, dtype=0, act=1)
    args.update(kw)
    lib = ccv.load_library()
    a = binding._arr
    rc = lib.ccv_update(args["x"] or None, a(args["xs"]) if args["xs"] else None, args["out"] or None,
                        a(args["os"]) if args["os"] else None, args["state"] or None,
                        a(args["ss"]) if args["ss"] else None, args["w"] or None, a(args["ws"]), args["bias"] or None,
                        args["bs"], args["B"], args["C"], args["S"], args["K"], args["dtype"], args["act"], None)
    return rc, ccv.ccv_last_error()


@pytest.mark.parametrize("kw,status,needle", [
    (dict(K=5), 2, "K must be 2, 3 or 4"),
    (dict(state=0), 1, "conv_state is required"),
    (dict(out=FAKE * 4), 1, "must not alias"),
    (dict(x=FAKE * 4), 1, "must not alias"),
    (dict(ss=(12, 0, 1)), 1, "zero stride"),
    (dict(S=-1), 1, ">= 0"),
    (dict(dtype=9), 1, "unknown dtype"),
])
def test_update_validation_errors(ccv, kw, status, needle):
    rc, msg = call_update(ccv, **kw)
    assert rc == status, msg
    assert needle in msg


def test_update_zero_rows_is_noop(ccv):
    assert call_update(ccv, B=0)[0] == 0


def ws_size(ccv, xs=(64, 16, 1), gs=None, dxs=None, B=2, C=4, L=16, K=4, dtype=0):
    return ccv.ccv_bwd_workspace_size(xs, gs or xs, dxs or xs, B, C, L, K, dtype)


def test_bwd_workspace_size(ccv):
    # unit time stride: rows cut into 1024-step partitions, ~2^15 pieces
    c2 = (8 * 5120 * 2048, 2048, 1)
    assert ws_size(ccv, c2, B=8, C=5120, L=2048) == 8 * 1 * 5 * 5120 * 4
    c5 = (16 * 4194304, 4194304, 1)
    assert ws_size(ccv, c5, B=1, C=16, L=4194304, K=3) == 1 * 2048 * 4 * 16 * 4
    # channel-last: 16-step partitions, at most 2432 pieces of 128 channels
    c4 = (16384 * 4096, 1, 4096)
    n = 2432 // 32
    chunk = -(-(-(-16384 // n)) // 16) * 16
    assert ws_size(ccv, c4, B=1, C=4096, L=16384) == (-(-16384 // chunk)) * 5 * 4096 * 4
    # nothing to reduce
    assert ws_size(ccv, B=0) == 0 and ws_size(ccv, L=0) == 0 and ws_size(ccv, C=0) == 0
    from causal_depthwise_conv1d_gb300 import binding
    with pytest.raises(ccv.CcvError):
        ws_size(ccv, K=5)
    del binding


def call_bwd(ccv, **kw):
    args = dict(x=FAKE, x_strides=(64, 16, 1), weight=FAKE * 3, weight_strides=(4, 1), bias=0, bias_stride=1,
                seq_idx=0, seq_idx_strides=None, initial_states=0, initial_states_strides=None,
                dout=FAKE * 8, dout_strides=(64, 16, 1), dfinal_states=0, dfinal_states_strides=None,
                dx=FAKE * 9, dx_strides=(64, 16, 1), dweight=FAKE * 10, dweight_strides=(4, 1), dbias=0,
                dbias_stride=1, dinitial_states=0, dinitial_states_strides=None, workspace=FAKE * 16,
                workspace_bytes=1 << 20, B=2, C=4, L=16, K=4, dtype=0, activation=1, stream=0)
    args.update(kw)
    try:
        ccv.ccv_bwd_ptr(**args)
    except ccv.CcvError as e:
        return e.status, str(e)
    return 0, ""


@pytest.mark.parametrize("kw,status,needle", [
    (dict(K=5), 2, "K must be 2, 3 or 4"),
    (dict(dtype=4), 1, "unknown dtype"),
    (dict(activation=2), 1, "unknown activation"),
    (dict(seq_idx=FAKE * 5, seq_idx_strides=(16, 1), initial_states=FAKE * 6,
          initial_states_strides=(12, 3, 1)), 2, "seq_idx together with initial_states"),
    (dict(dinitial_states=FAKE * 11, dinitial_states_strides=(12, 3, 1)), 1, "requires initial_states"),
    (dict(dx=0), 1, "dx is required"),
    (dict(dout=0), 1, "dout is required"),
    (dict(weight=0), 1, "weight is required"),
    (dict(dx=FAKE * 8), 1, "must not alias"),
    (dict(dx=FAKE * 8 + 8), 1, "must not alias"),
    (dict(dweight=FAKE * 3), 1, "must not alias"),
    (dict(dx_strides=(64, 0, 1)), 1, "zero stride"),
    (dict(dweight_strides=(0, 1)), 1, "zero stride"),
    (dict(workspace_bytes=16), 1, "workspace too small"),
    (dict(workspace=0), 1, "workspace too small"),
    (dict(workspace=FAKE * 16 + 4), 1, "16-byte aligned"),
    (dict(dx=FAKE * 9 + 2), 1, "aligned"),
    (dict(x_strides=(1 << 62, 16, 1)), 1, "overflows"),
    (dict(dfinal_states=FAKE * 12), 1, "dfinal_states_strides is required"),
])
def test_bwd_validation_errors(ccv, kw, status, needle):
    st, msg = call_bwd(ccv, **kw)
    assert st == status, msg
    assert needle in msg


def test_bwd_workspace_not_needed_without_parameter_gradients(ccv):
    # validation passes with no workspace when neither dweight nor dbias is
    # wanted; the call then fails only at the device step (no GPU here) or
    # succeeds on a GPU machine -- either way not with a workspace error
    st, msg = call_bwd(ccv, dweight=0, workspace=0, workspace_bytes=0, x=0, dout=0, dx=0, L=0)
    assert "workspace" not in msg


def test_mixed_entry_points_validate_the_weight_dtype(ccv):
    from causal_depthwise_conv1d_gb300 import binding
    a = dict(x=FAKE, x_strides=(64, 16, 1), out=FAKE * 2, out_strides=(64, 16, 1), weight=FAKE * 3,
             weight_strides=(4, 1), bias=0, bias_stride=1, seq_idx=0, seq_idx_strides=None, initial_states=0,
             initial_states_strides=None, final_states_out=0, final_states_strides=None, B=2, C=4, L=16, K=4,
             dtype=binding.CCV_F16, activation=1, stream=0)
    with pytest.raises(ccv.CcvError, match="unknown weight dtype"):
        ccv.ccv_fwd_ptr(**a, weight_dtype=5)
    # FP32 weights must be 4-byte aligned even when x is 16-bit
    with pytest.raises(ccv.CcvError, match="aligned"):
        ccv.ccv_fwd_ptr(**dict(a, weight=FAKE * 3 + 2), weight_dtype=binding.CCV_F32)
    args = dict(x=FAKE, x_strides=(64, 16, 1), weight=FAKE * 3 + 2, weight_strides=(4, 1), bias=0, bias_stride=1,
                seq_idx=0, seq_idx_strides=None, initial_states=0, initial_states_strides=None,
                dout=FAKE * 8, dout_strides=(64, 16, 1), dfinal_states=0, dfinal_states_strides=None,
                dx=FAKE * 9, dx_strides=(64, 16, 1), dweight=FAKE * 10, dweight_strides=(4, 1), dbias=0,
                dbias_stride=1, dinitial_states=0, dinitial_states_strides=None, workspace=FAKE * 16,
                workspace_bytes=1 << 20, B=2, C=4, L=16, K=4, dtype=binding.CCV_BF16, activation=1, stream=0)
    with pytest.raises(ccv.CcvError, match="aligned"):
        ccv.ccv_bwd_ptr(**args, weight_dtype=binding.CCV_F32)


def test_bounded_wait_hook_arguments(ccv):
    """Host-side only: a negative stage is rejected; a set-then-cleared
    setting leaves nothing pending (no launch happens here)."""
    with pytest.raises(ccv.CcvError) as e:
        ccv.ccv_test_bounded_wait(1000, -1)
    assert e.value.status == 1
    ccv.ccv_test_bounded_wait(1000, 0)
    ccv.ccv_test_bounded_wait(0, 0)


def test_noalloc_rejects_problems_beyond_its_scratch_on_the_host(ccv):
    """ccv_bwd_noalloc checks the partials' size against its fixed scratch
    before any device call (the pointers below are never dereferenced)."""
    from causal_depthwise_conv1d_gb300 import binding
    lib = binding.load_library()
    arr = binding._arr
    B, C, L, K = 128, 8192, 4096, 4
    xs = (C * L, L, 1)
    need = ccv.ccv_bwd_workspace_size(xs, xs, xs, B, C, L, K, binding.CCV_BF16)
    assert need > 16 << 20
    fake = 0x1000
    rc = lib.ccv_bwd_noalloc(fake, arr(xs), fake, arr((K, 1)), None, 0, None, None, None, None,
                             fake, arr(xs), None, None, fake, arr(xs), fake, arr((K, 1)), None, 0, None, None,
                             B, C, L, K, binding.CCV_BF16, 1, None)
    assert rc == 1  # CCV_ERR_INVALID_ARG
    msg = lib.ccv_last_error().decode()
    assert "scratch" in msg and str(need) in msg
