"""The C-ABI library loads, exports every entry point include/q.h declares,
and rejects bad arguments on the host before any CUDA call (no GPU needed:
every call below fails validation, so nothing is launched)."""
import ctypes
import os
import re

import pytest

import nvfp4_quantization_current_gb300 as Q
from nvfp4_quantization_current_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q.h")


@pytest.fixture(scope="module")
def L():
    B.build()
    return Q.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*((?:q|dq)_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["q_amax", "q_current_scaling", "q_delayed_scaling", "q_delayed_scale_update", "q_mxfp8",
              "q_mxfp8_requant_col", "q_blockwise", "q_blockwise_mx", "q_nvfp4", "q_nvfp4_rht_amax",
              "q_nvfp4_rht_colT", "q_nvfp4_rht_amax2", "q_nvfp4_recipe",
              "dq_current_scaling", "dq_mxfp8", "dq_blockwise",
              "dq_nvfp4", "q_last_error", "q_abi_version", "q_selftest_inject_launch_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), n
        assert n in Q.SIGNATURES, n
    assert L.q_abi_version() == 4


A = ctypes.c_void_p(0x10000)        # an aligned non-NULL address that is never dereferenced
MIS = ctypes.c_void_p(0x10008)      # 8-byte aligned only


def status_of(L, fn, *args):
    st = getattr(L, fn)(*args)
    return st, L.q_last_error().decode()


def test_current_scaling_validation(L):
    st, msg = status_of(L, "q_current_scaling", None, Q.Q_BF16, 4, 16, Q.Q_E4M3, A, None, A, 0, A, None, None)
    assert st == Q.Q_ERR_ARG and "x is NULL" in msg
    st, _ = status_of(L, "q_current_scaling", A, 7, 4, 16, Q.Q_E4M3, A, None, A, 0, A, None, None)
    assert st == Q.Q_ERR_DTYPE
    st, _ = status_of(L, "q_current_scaling", A, Q.Q_BF16, 4, 16, 9, A, None, A, 0, A, None, None)
    assert st == Q.Q_ERR_ARG
    st, _ = status_of(L, "q_current_scaling", A, Q.Q_BF16, 4, 16, Q.Q_E4M3, None, None, A, 0, A, None, None)
    assert st == Q.Q_ERR_ARG                       # nothing requested
    st, _ = status_of(L, "q_current_scaling", MIS, Q.Q_BF16, 4, 16, Q.Q_E4M3, A, None, A, 0, A, None, None)
    assert st == Q.Q_ERR_ALIGN
    st, _ = status_of(L, "q_current_scaling", A, Q.Q_BF16, 24, 16, Q.Q_E4M3, None, A, A, 0, A, None, None)
    assert st == Q.Q_ERR_SHAPE                     # colT needs M % 16
    st, _ = status_of(L, "q_current_scaling", A, Q.Q_BF16, -1, 16, Q.Q_E4M3, A, None, A, 0, A, None, None)
    assert st == Q.Q_ERR_SHAPE
    st, msg = status_of(L, "q_current_scaling", A, Q.Q_BF16, 1 << 40, 1 << 30, Q.Q_E4M3, A, None, A, 0, A, None, None)
    assert st == Q.Q_ERR_SHAPE and "too large" in msg
    st, _ = status_of(L, "q_current_scaling", A, Q.Q_BF16, 4, 16, Q.Q_E4M3, A, None, None, 0, A, None, None)
    assert st == Q.Q_ERR_ARG                       # amax required
    st, _ = status_of(L, "q_current_scaling", A, Q.Q_BF16, 4, 16, Q.Q_E4M3, A, None, A, 5, A, None, None)
    assert st == Q.Q_ERR_ARG                       # bad amax mode


def test_delayed_scaling_validation(L):
    st, _ = status_of(L, "q_delayed_scaling", A, Q.Q_BF16, 4, 16, Q.Q_E4M3, A, None, None, A, A, None, None)
    assert st == Q.Q_ERR_ARG                       # ds required
    st, _ = status_of(L, "q_delayed_scaling", A, Q.Q_BF16, 4, 16, Q.Q_E4M3, A, None, A, None, A, None, None)
    assert st == Q.Q_ERR_ARG                       # amax_out required
    st, _ = status_of(L, "q_delayed_scaling", A, Q.Q_BF16, 24, 16, Q.Q_E4M3, None, A, A, A, A, None, None)
    assert st == Q.Q_ERR_SHAPE                     # colT needs M % 16
    st, _ = status_of(L, "q_delayed_scaling", A, Q.Q_BF16, 4, 16, Q.Q_E4M3, None, None, A, A, A, None, None)
    assert st == Q.Q_ERR_ARG                       # nothing requested
    st, msg = status_of(L, "q_delayed_scale_update", A, 0, 0, Q.Q_HIST_MAX, Q.Q_E4M3, A, None)
    assert st == Q.Q_ERR_SHAPE and ">= 1" in msg
    st, _ = status_of(L, "q_delayed_scale_update", A, 16, 16, Q.Q_HIST_MAX, Q.Q_E4M3, A, None)
    assert st == Q.Q_ERR_ARG                       # pos outside the window
    st, _ = status_of(L, "q_delayed_scale_update", A, 16, 3, 7, Q.Q_E4M3, A, None)
    assert st == Q.Q_ERR_ARG                       # bad algo
    st, _ = status_of(L, "q_delayed_scale_update", A, 16, 3, Q.Q_HIST_MAX, Q.Q_E4M3, None, None)
    assert st == Q.Q_ERR_ARG                       # ds required


def test_rht_validation(L):
    args = lambda M, K, mask, rnd, qc, sbc, amax, mode, sg: (A, Q.Q_BF16, M, K, mask, rnd, 0, 0, qc, sbc, amax, mode, sg,
                                                           None, None)
    st, _ = status_of(L, "q_nvfp4_rht_colT", *args(24, 32, 0x1234, Q.Q_RN, A, A, A, 0, A))
    assert st == Q.Q_ERR_SHAPE                     # M % 16
    st, _ = status_of(L, "q_nvfp4_rht_colT", *args(32, 24, 0x1234, Q.Q_RN, A, A, A, 0, A))
    assert st == Q.Q_ERR_SHAPE                     # K % 16
    st, msg = status_of(L, "q_nvfp4_rht_colT", *args(32, 32, 0x10000, Q.Q_RN, A, A, A, 0, A))
    assert st == Q.Q_ERR_ARG and "bit 15" in msg
    st, _ = status_of(L, "q_nvfp4_rht_colT", *args(32, 32, 0x1234, 2, A, A, A, 0, A))
    assert st == Q.Q_ERR_ARG                       # bad rounding
    st, _ = status_of(L, "q_nvfp4_rht_colT", *args(32, 32, 0x1234, Q.Q_RN, None, A, A, 0, A))
    assert st == Q.Q_ERR_ARG                       # q_colT required
    st, _ = status_of(L, "q_nvfp4_rht_colT", *args(32, 32, 0x1234, Q.Q_RN, A, A, A, 0, None))
    assert st == Q.Q_ERR_ARG                       # s_global required
    st, _ = status_of(L, "q_nvfp4_rht_amax", A, Q.Q_BF16, 32, 24, 0x1, A, None, None)
    assert st == Q.Q_ERR_SHAPE
    st, _ = status_of(L, "q_nvfp4_rht_amax", A, Q.Q_BF16, 32, 32, 0x1, None, None, None)
    assert st == Q.Q_ERR_ARG


def test_selftest_validation(L):
    st, _ = status_of(L, "q_selftest_wait_timeout", None, 1000, None)
    assert st == Q.Q_ERR_ARG
    st, msg = status_of(L, "q_selftest_wait_timeout", A, 0, None)
    assert st == Q.Q_ERR_ARG and "wait_ns" in msg
    st, _ = status_of(L, "q_selftest_wait_timeout", A, 2_000_000_000, None)
    assert st == Q.Q_ERR_ARG


def test_requant_validation(L):
    st, _ = status_of(L, "q_mxfp8_requant_col", A, A, 48, 64, Q.Q_E4M3, A, A, None, None)
    assert st == Q.Q_ERR_SHAPE                     # M % 32
    st, _ = status_of(L, "q_mxfp8_requant_col", A, A, 64, 48, Q.Q_E4M3, A, A, None, None)
    assert st == Q.Q_ERR_SHAPE                     # K % 32
    st, _ = status_of(L, "q_mxfp8_requant_col", MIS, A, 64, 64, Q.Q_E4M3, A, A, None, None)
    assert st == Q.Q_ERR_ALIGN
    st, _ = status_of(L, "q_mxfp8_requant_col", A, A, 64, 64, 4, A, A, None, None)
    assert st == Q.Q_ERR_ARG


def test_block_recipes_validation(L):
    st, _ = status_of(L, "q_mxfp8", A, Q.Q_BF16, 64, 48, Q.Q_E4M3, A, A, None, None, None, None)
    assert st == Q.Q_ERR_SHAPE                     # K % 32
    st, _ = status_of(L, "q_mxfp8", A, Q.Q_BF16, 48, 64, Q.Q_E4M3, None, None, A, A, None, None)
    assert st == Q.Q_ERR_SHAPE                     # M % 32 with the columnwise output
    st, _ = status_of(L, "q_mxfp8", A, Q.Q_BF16, 64, 64, Q.Q_E4M3, A, None, None, None, None, None)
    assert st == Q.Q_ERR_ARG                       # missing scale buffer
    st, _ = status_of(L, "q_blockwise", A, Q.Q_BF16, 128, 192, Q.Q_T1x128, A, A, None, None, None, None)
    assert st == Q.Q_ERR_SHAPE
    st, _ = status_of(L, "q_blockwise", A, Q.Q_BF16, 192, 128, Q.Q_T128x128, A, A, None, None, None, None)
    assert st == Q.Q_ERR_SHAPE
    st, _ = status_of(L, "q_blockwise", A, Q.Q_BF16, 128, 128, 3, A, A, None, None, None, None)
    assert st == Q.Q_ERR_ARG
    st, _ = status_of(L, "q_nvfp4", A, Q.Q_BF16, 16, 24, Q.Q_B1x16, Q.Q_RN, 0, 0, A, A, None, None, A, 0, A, None, None)
    assert st == Q.Q_ERR_SHAPE
    st, _ = status_of(L, "q_nvfp4", A, Q.Q_BF16, 16, 32, Q.Q_B1x16, 2, 0, 0, A, A, None, None, A, 0, A, None, None)
    assert st == Q.Q_ERR_ARG
    st, _ = status_of(L, "q_nvfp4", A, Q.Q_BF16, 16, 32, Q.Q_B1x16, Q.Q_RN, 0, 0, A, A, None, None, A, 0, None, None, None)
    assert st == Q.Q_ERR_ARG                       # s_global required


def test_blockwise_mx_validation(L):
    st, _ = status_of(L, "q_blockwise_mx", A, Q.Q_BF16, 128, 192, Q.Q_T1x128, A, A, None, None, None, None)
    assert st == Q.Q_ERR_SHAPE                     # K % 128
    st, _ = status_of(L, "q_blockwise_mx", A, Q.Q_BF16, 192, 128, Q.Q_T128x128, A, A, None, None, None, None)
    assert st == Q.Q_ERR_SHAPE                     # M % 128 for 2D tiles
    st, _ = status_of(L, "q_blockwise_mx", A, Q.Q_BF16, 64, 128, Q.Q_T1x128, None, None, A, A, None, None)
    assert st == Q.Q_ERR_SHAPE                     # M % 128 with the transposed copy
    st, _ = status_of(L, "q_blockwise_mx", A, Q.Q_BF16, 128, 128, 3, A, A, None, None, None, None)
    assert st == Q.Q_ERR_ARG
    st, msg = status_of(L, "q_blockwise_mx", A, Q.Q_BF16, 128, 128, Q.Q_T1x128, A, ctypes.c_void_p(0x10002),
                        None, None, None, None)
    assert st == Q.Q_ERR_ALIGN and "e8m0_row" in msg
    st, msg = status_of(L, "q_blockwise_mx", A, Q.Q_BF16, 128, 128, Q.Q_T1x128, None, None, A,
                        ctypes.c_void_p(0x10002), None, None)
    assert st == Q.Q_ERR_ALIGN and "e8m0_colT" in msg
    st, _ = status_of(L, "q_blockwise_mx", A, Q.Q_BF16, 128, 128, Q.Q_T1x128, None, None, None, None, None, None)
    assert st == Q.Q_ERR_ARG                       # neither direction
    st, _ = status_of(L, "q_blockwise_mx", A, Q.Q_BF16, 0, 128, Q.Q_T1x128, None, None, None, None, None, None)
    assert st == Q.Q_OK                            # empty: nothing to do


def test_nvfp4_recipe_validation(L):
    U64 = ctypes.c_uint64
    args = lambda M, K, mask=0x1234, rnd=Q.Q_RN, amax_row=A, mode=Q.Q_AMAX_COMPUTE: (
        A, Q.Q_BF16, M, K, mask, rnd, U64(0), U64(0), A, A, amax_row, A, A, A, A, A, mode, None, None)
    st, _ = status_of(L, "q_nvfp4_recipe", *args(32, 24))
    assert st == Q.Q_ERR_SHAPE                     # K % 16
    st, _ = status_of(L, "q_nvfp4_recipe", *args(24, 32))
    assert st == Q.Q_ERR_SHAPE                     # M % 16
    st, _ = status_of(L, "q_nvfp4_recipe", *args(32, 32, mask=0x10000))
    assert st == Q.Q_ERR_ARG
    st, _ = status_of(L, "q_nvfp4_recipe", *args(32, 32, rnd=2))
    assert st == Q.Q_ERR_ARG
    st, msg = status_of(L, "q_nvfp4_recipe", *args(32, 32, amax_row=None))
    assert st == Q.Q_ERR_ARG and "amax_row" in msg
    st, msg = status_of(L, "q_nvfp4_recipe", *args(32, 32, mode=7))
    assert st == Q.Q_ERR_ARG and "amax_mode" in msg
    st, msg = status_of(L, "q_nvfp4_rht_amax2", A, Q.Q_BF16, 32, 32, 0x1234, A, ctypes.c_void_p(0x10002), None, None)
    assert st == Q.Q_ERR_ALIGN and "amax_x" in msg
    st, _ = status_of(L, "q_nvfp4_rht_amax2", A, Q.Q_BF16, 32, 40, 0x1234, A, A, None, None)
    assert st == Q.Q_ERR_SHAPE


def test_dequant_validation(L):
    st, _ = status_of(L, "dq_current_scaling", A, A, 4, 4, Q.Q_E4M3, 5, A, None)
    assert st == Q.Q_ERR_DTYPE
    st, _ = status_of(L, "dq_mxfp8", A, A, 4, 48, Q.Q_E4M3, Q.Q_ROW, Q.Q_F32, A, None)
    assert st == Q.Q_ERR_SHAPE
    st, _ = status_of(L, "dq_mxfp8", A, MIS, 32, 48, Q.Q_E4M3, Q.Q_COL, Q.Q_F32, A, None)
    assert st == Q.Q_ERR_ALIGN
    st, _ = status_of(L, "dq_blockwise", A, A, 4, 100, Q.Q_T1x128, Q.Q_F32, A, None)
    assert st == Q.Q_ERR_SHAPE
    st, _ = status_of(L, "dq_nvfp4", A, A, A, 4, 24, Q.Q_B1x16, Q.Q_F32, A, None)
    assert st == Q.Q_ERR_SHAPE
    st, _ = status_of(L, "dq_nvfp4", A, A, A, 8, 32, Q.Q_B16x16, Q.Q_F32, A, None)
    assert st == Q.Q_ERR_SHAPE
    st, _ = status_of(L, "dq_nvfp4", A, A, None, 16, 32, Q.Q_B1x16, Q.Q_F32, A, None)
    assert st == Q.Q_ERR_ARG


def test_binding_refuses_cpu_tensors():
    import torch
    with pytest.raises(ValueError, match="CUDA"):
        Q.q_current_scaling(torch.zeros(4, 16))


def test_nvfp4_columnwise_scale_buffers_need_16_byte_alignment(L):
    """sb_colT is written in 8-byte pieces by every NVFP4 entry point that
    produces it, so a 1-byte-aligned pointer is refused on the host."""
    U64 = ctypes.c_uint64
    odd = ctypes.c_void_p(0x10001)
    st, msg = status_of(L, "q_nvfp4_recipe", A, Q.Q_BF16, 32, 32, 0x1234, Q.Q_RN, U64(0), U64(0), A, A, A, A,
                        A, odd, A, A, Q.Q_AMAX_COMPUTE, None, None)
    assert st == Q.Q_ERR_ALIGN and "sb_colT" in msg
    st, msg = status_of(L, "q_nvfp4", A, Q.Q_BF16, 16, 32, Q.Q_B1x16, Q.Q_RN, 0, 0, None, None, A, odd, A, 0, A,
                        None, None)
    assert st == Q.Q_ERR_ALIGN and "sb_colT" in msg
    st, msg = status_of(L, "q_nvfp4_rht_colT", A, Q.Q_BF16, 32, 32, 0x1, Q.Q_RN, 0, 0, A, odd, A, 0, A, None, None)
    assert st == Q.Q_ERR_ALIGN and "sb_colT" in msg


def _valid_calls():
    """One argument list per launching entry point that passes every host
    check (A is aligned and never dereferenced: the injected failure stops
    the call before anything is enqueued)."""
    U64 = ctypes.c_uint64
    return {
        "q_amax": (A, Q.Q_BF16, 64, A, None, None),
        "q_current_scaling": (A, Q.Q_BF16, 16, 16, Q.Q_E4M3, A, A, A, Q.Q_AMAX_COMPUTE, A, None, None),
        "q_delayed_scaling": (A, Q.Q_BF16, 16, 16, Q.Q_E4M3, A, A, A, A, A, None, None),
        "q_delayed_scale_update": (A, 16, 3, Q.Q_HIST_MAX, Q.Q_E4M3, A, None),
        "q_mxfp8": (A, Q.Q_BF16, 32, 32, Q.Q_E4M3, A, A, A, A, None, None),
        "q_mxfp8_requant_col": (A, A, 32, 32, Q.Q_E4M3, A, A, None, None),
        "q_blockwise": (A, Q.Q_BF16, 128, 128, Q.Q_T1x128, A, A, A, A, None, None),
        "q_blockwise_mx": (A, Q.Q_BF16, 128, 128, Q.Q_T1x128, A, A, A, A, None, None),
        "q_nvfp4": (A, Q.Q_BF16, 16, 32, Q.Q_B1x16, Q.Q_SR, 1, 0, A, A, A, A, A, Q.Q_AMAX_COMPUTE, A, None, None),
        "q_nvfp4_rht_amax": (A, Q.Q_BF16, 16, 16, 0x1, A, None, None),
        "q_nvfp4_rht_amax2": (A, Q.Q_BF16, 16, 16, 0x1, A, A, None, None),
        "q_nvfp4_rht_colT": (A, Q.Q_BF16, 16, 16, 0x1, Q.Q_RN, 0, 0, A, A, A, Q.Q_AMAX_COMPUTE, A, None, None),
        "q_nvfp4_recipe": (A, Q.Q_BF16, 16, 16, 0x1, Q.Q_RN, U64(0), U64(0), A, A, A, A, A, A, A, A,
                           Q.Q_AMAX_COMPUTE, None, None),
        "q_selftest_wait_timeout": (A, 1000, None),
        "dq_current_scaling": (A, A, 4, 4, Q.Q_E4M3, Q.Q_F32, A, None),
        "dq_mxfp8": (A, A, 4, 32, Q.Q_E4M3, Q.Q_ROW, Q.Q_F32, A, None),
        "dq_blockwise": (A, A, 4, 128, Q.Q_T1x128, Q.Q_F32, A, None),
        "dq_nvfp4": (A, A, A, 4, 32, Q.Q_B1x16, Q.Q_F32, A, None),
    }


def test_injected_launch_failure_returns_q_err_cuda(L):
    """A CUDA launch failure reaches the caller as Q_ERR_CUDA with a message
    naming the entry point and the CUDA error, from every entry point that
    launches (failures injected on the host: no GPU, nothing enqueued)."""
    calls = _valid_calls()
    declared = set(declared_functions())
    launching = declared - {"q_last_error", "q_abi_version", "q_selftest_inject_launch_error"}
    assert launching == set(calls)
    try:
        for name, args in calls.items():
            assert L.q_selftest_inject_launch_error(1) == Q.Q_OK
            st, msg = status_of(L, name, *args)
            assert st == Q.Q_ERR_CUDA, (name, st, msg)
            assert name in msg and "cudaErrorLaunchFailure" in msg, (name, msg)
        # n failures are consumed one launch at a time
        assert L.q_selftest_inject_launch_error(2) == Q.Q_OK
        for _ in range(2):
            st, _ = status_of(L, "q_amax", *calls["q_amax"])
            assert st == Q.Q_ERR_CUDA
        # the binding raises QuantError carrying the status
        assert L.q_selftest_inject_launch_error(1) == Q.Q_OK
        with pytest.raises(Q.QuantError) as ei:
            Q._call("dq_nvfp4", *calls["dq_nvfp4"])
        assert ei.value.status == Q.Q_ERR_CUDA
        st, msg = status_of(L, "q_selftest_inject_launch_error", -1)
        assert st == Q.Q_ERR_ARG and "negative" in msg
    finally:
        L.q_selftest_inject_launch_error(0)
