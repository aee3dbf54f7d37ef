"""The allocation-free dense entry point, dg_fp8_gemm_nt_noalloc, through the C ABI.

It exists for callers that cannot let libdg call cudaMalloc (a framework whose caching allocator
owns the device memory, a serving loop that must not block on cudaMalloc's synchronisation). Its
split-K scratch is a fixed array inside the library that every call reuses, so this test makes two
calls in a row and checks both against the allocating entry point, dg_fp8_gemm_nt, within the
tolerance of the parity tests (and, since both run the same kernel with the same configuration,
bit for bit). The file name sorts last so that a run stopping at the first failure has already run
every other test; it passes alone in a fresh process too.
"""
import numpy as np
import pytest
import torch

import dg_inputs
from _dg_testlib import COS_TOL, MAX_REL_TOL, bf16_sentinel, bits16, dev, metrics

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    import moe_grouped_gemm_e4m3_gb300 as m
    m.load()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return m


# few tiles (split-K through the fixed scratch) and one shape that needs no scratch
@pytest.mark.parametrize("M,N,K", [(64, 2112, 7168), (128, 4096, 7168), (100, 1000, 2048), (4096, 2112, 1024)])
def test_noalloc_matches_allocating_entry_point_twice(dg, M, N, K):
    a = dg_inputs.make_a(M, K, seed=M + K)
    b = dg_inputs.make_b(1, N, K, seed=N + K)
    A, sA, B, sB = dev(a.A), dev(a.sA), dev(b.B[0]), dev(b.sB[0])
    ref = bf16_sentinel((M, N))
    dg.dg_fp8_gemm_nt(A, sA, B, sB, ref)
    outs = []
    for _ in range(2):                       # the scratch array keeps the previous call's contents
        D = bf16_sentinel((M, N))
        dg.dg_fp8_gemm_nt_noalloc(A, sA, B, sB, D)
        outs.append(D)
    torch.cuda.synchronize()
    assert dg.dg_get_device_status() == 0
    r = ref.float().cpu().numpy()
    for D in outs:
        assert not torch.any(bits16(D) == -1), "output not fully written"
        m = metrics(D.float().cpu().numpy(), r)
        assert m["finite"] and m["max_rel"] <= MAX_REL_TOL and m["one_minus_cos"] <= COS_TOL, m
        assert torch.equal(bits16(D), bits16(ref))


def test_noalloc_rejects_bad_arguments(dg):
    a = dg_inputs.make_a(16, 128, seed=1)
    b = dg_inputs.make_b(1, 64, 128, seed=1)
    D = bf16_sentinel((16, 60))
    with pytest.raises(dg.DGError) as e:
        dg.dg_fp8_gemm_nt_noalloc(dev(a.A), dev(a.sA), dev(b.B[0][:60].copy()), dev(b.sB[0]), D)
    assert e.value.status == dg.DG_ERR_ALIGNMENT
