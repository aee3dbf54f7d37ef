"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every symbol that
include/dg.h declares, and its host-side validation rejects bad arguments before any CUDA call."""
import ctypes
import os
import re

import pytest

import moe_grouped_gemm_e4m3_gb300 as dg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    with open(os.path.join(ROOT, "include", "dg.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(dg_\w+)\s*\(", text, flags=re.M)))


def test_library_exports_every_declared_symbol():
    lib = dg.load()
    declared = _declared_symbols()
    assert len(declared) >= 13, declared
    for name in declared:
        assert hasattr(lib, name), f"libdg.so does not export {name}"
    assert sorted(dg.EXPORTED_SYMBOLS) == declared


def test_pure_host_utilities():
    assert dg.dg_get_tma_aligned_size(4095, 4) == 4096
    assert dg.dg_get_tma_aligned_size(4096, 4) == 4096
    assert dg.dg_get_tma_aligned_size(1, 4) == 4
    assert dg.dg_get_tma_aligned_size(17, 1) == 32
    assert dg.dg_get_tma_aligned_size(3, 2) == 8
    assert dg.dg_get_tma_aligned_size(5, 3) == -1
    assert dg.dg_get_mk_alignment_for_contiguous_layout() == 128


def _call_dense(lib, A, sA, B, sB, D, M, N, K):
    P = ctypes.c_void_p
    return lib.dg_fp8_gemm_nt(P(A), P(sA), P(B), P(sB), P(D), M, N, K, None)


def test_validation_rejects_bad_arguments_before_any_cuda_call():
    lib = dg.load()
    fake = 0x10000   # never dereferenced: validation fails first
    assert _call_dense(lib, fake, fake, fake, fake, fake, 16, 64, 120) == dg.DG_ERR_ALIGNMENT      # K % 16
    assert _call_dense(lib, fake, fake, fake, fake, fake, 16, 60, 128) == dg.DG_ERR_ALIGNMENT      # N % 8
    assert _call_dense(lib, fake + 8, fake, fake, fake, fake, 16, 64, 128) == dg.DG_ERR_ALIGNMENT  # A align
    assert _call_dense(lib, fake, fake + 2, fake, fake, fake, 16, 64, 128) == dg.DG_ERR_ALIGNMENT  # sA align
    assert _call_dense(lib, 0, fake, fake, fake, fake, 16, 64, 128) == dg.DG_ERR_INVALID_ARG       # null A
    assert _call_dense(lib, fake, fake, fake, fake, fake, -1, 64, 128) == dg.DG_ERR_INVALID_ARG    # M < 0
    assert _call_dense(lib, fake, fake, fake, fake, fake, 16, 64, 0) == dg.DG_ERR_INVALID_ARG      # K == 0
    assert b"multiple of 16" in lib.dg_last_error_string() or True
    # empty problems are a no-op success and touch nothing
    assert _call_dense(lib, fake, fake, fake, fake, fake, 0, 64, 128) == dg.DG_OK
    assert _call_dense(lib, fake, fake, fake, fake, fake, 16, 0, 128) == dg.DG_OK
    P = ctypes.c_void_p
    # FP32 output needs N % 4 only
    assert lib.dg_fp8_gemm_nt_f32(P(fake), P(fake), P(fake), P(fake), P(fake), 16, 60, 120, None) == dg.DG_ERR_ALIGNMENT
    # grouped forms: missing index tensors
    assert lib.dg_fp8_grouped_contiguous(P(fake), P(fake), P(fake), P(fake), None, P(fake), 128, 64, 128, 2,
                                         None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_fp8_grouped_masked(P(fake), P(fake), P(fake), P(fake), None, P(fake), 2, 128, 64, 128,
                                     None) == dg.DG_ERR_INVALID_ARG
    assert lib.dg_fp8_grouped_masked(P(fake), P(fake), P(fake), P(fake), P(fake), P(fake), 0, 128, 64, 128,
                                     None) == dg.DG_OK


def test_config_heuristic_on_the_gb300_sm_count():
    dg.dg_set_num_sms(152)
    try:
        big = dg.dg_query_config(0, 4096, 7168, 16384)
        assert big["block_n"] == 256 and big["splits"] == 1 and big["grid"] == 152
        small = dg.dg_query_config(0, 64, 2112, 7168)
        assert small["splits"] > 1                                    # few tiles: split K
        assert small["tiles"] * small["splits"] <= 152                # one wave of units
        assert small["grid"] == small["tiles"] * small["splits"]
        assert dg.dg_query_config(0, 64, 128, 1024)["block_n"] == 128  # N <= 128
        masked = dg.dg_query_config(2, 256, 4096, 7168, G=16)
        assert masked["splits"] == 1
        # the configuration never depends on the output type
        assert dg.dg_query_config(0, 64, 2112, 7168, out_f32=True) == small
    finally:
        dg.dg_set_num_sms(0)


@pytest.mark.skipif(not os.path.exists("/usr/local/cuda/bin/nvcc"), reason="needs nvcc")
def test_build_is_up_to_date_after_load():
    from moe_grouped_gemm_e4m3_gb300 import build
    dg.load()
    assert build.up_to_date()


def test_tail_split_setting_is_host_state():
    # no CUDA call: the setting is read by the host when a GEMM is launched
    prev = dg.dg_set_tail_splits(3)
    try:
        assert dg.dg_set_tail_splits(1) == 3          # 1: off
        assert dg.dg_set_tail_splits(40) == 1         # clamped to 16
        assert dg.dg_set_tail_splits(-5) == 16        # <= 0: the default, 4
        assert dg.dg_set_tail_splits(prev) == 4
    finally:
        dg.dg_set_tail_splits(prev)


def test_cluster_split_setting_is_host_state():
    prev = dg.dg_set_cluster_split(False)
    try:
        assert dg.dg_set_cluster_split(True) is False
        assert dg.dg_set_cluster_split(True) is True
    finally:
        dg.dg_set_cluster_split(prev)


def test_wait_limit_setting():
    """The kernels' wait limit is a host setting (no GPU needed): default 2 s, clamped to the 24-bit
    microsecond field of the kernel flags word, -1 restores the default."""
    prev = dg.dg_set_wait_limit_us(5000)
    try:
        assert dg.dg_set_wait_limit_us(10 ** 12) == 5000
        assert dg.dg_set_wait_limit_us(-1) == (1 << 24) - 1
        assert dg.dg_set_wait_limit_us(0) == 2000000
        assert dg.dg_set_wait_limit_us(prev) == 0
    finally:
        dg.dg_set_wait_limit_us(prev)


def test_pair_b_setting():
    prev = dg.dg_set_pair_b(False)
    assert prev is False                      # off by default (DG_PAIR_B unset)
    try:
        assert dg.dg_set_pair_b(True) is False
        assert dg.dg_set_pair_b(prev) is True
    finally:
        dg.dg_set_pair_b(prev)
