"""tcgen05 building blocks on the GPU: one tile product through the same shared-memory
layouts (128-byte swizzle, K-major), descriptors, tensor-memory stores/loads and
mbarrier completion as the tensor-core forward, against a plain fp32 matmul."""
import pytest
import torch

import exact_flow_recurrence_gb300 as efla

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("a_mn,b_mn,a_tm", [(False, False, False), (True, False, False),
                                            (False, True, False), (True, True, False),
                                            (False, False, True), (False, True, True)])
@pytest.mark.parametrize("N,K", [(64, 64), (64, 128), (128, 64), (128, 128), (192, 64), (256, 128)])
def test_tile_product(N, K, a_mn, b_mn, a_tm):
    g = torch.Generator(device="cuda").manual_seed(N * 1000 + K)
    A = torch.randn((128, K), generator=g, device="cuda").half()
    B = torch.randn((N, K), generator=g, device="cuda").half()
    C = torch.randn((128, N), generator=g, device="cuda")
    D = efla.efla_tc_selftest(A, B, C, a_mn_major=a_mn, b_mn_major=b_mn, a_in_tmem=a_tm)
    efla.efla_get_status()
    ref = C + A.float() @ B.float().T
    err = (D - ref).abs().max().item()
    assert err < 1e-3 * ref.abs().max().item(), err


@pytest.mark.parametrize("a_mn,b_mn,a_tm", [(False, False, False), (True, True, False), (False, True, True)])
def test_structured_operands_locate_rows_and_columns(a_mn, b_mn, a_tm):
    """A = identity, B with distinct entries: D[r][n] must be exactly B[n][r]."""
    K, N = 128, 128
    A = torch.zeros((128, K), device="cuda")
    A[torch.arange(128), torch.arange(128) % K] = 1.0
    B = (torch.arange(N * K, device="cuda").reshape(N, K) % 251).float() / 8.0
    D = efla.efla_tc_selftest(A.half(), B.half(), torch.zeros((128, N), device="cuda"),
                              a_mn_major=a_mn, b_mn_major=b_mn, a_in_tmem=a_tm)
    efla.efla_get_status()
    assert torch.equal(D, (A @ B.T))


@pytest.mark.parametrize("b_mn,a_tm", [(True, True), (False, True), (True, False)])
def test_wide_n_blocks_in_order(b_mn, a_tm):
    """N = 192 (three 64-wide B blocks): D[r][n] must be exactly B[n][r] for A = identity."""
    K, N = 64, 192
    A = torch.zeros((128, K), device="cuda")
    A[torch.arange(128), torch.arange(128) % K] = 1.0
    B = (torch.arange(N * K, device="cuda").reshape(N, K) % 241).float() / 4.0
    D = efla.efla_tc_selftest(A.half(), B.half(), torch.zeros((128, N), device="cuda"),
                              a_mn_major=False, b_mn_major=b_mn, a_in_tmem=a_tm)
    efla.efla_get_status()
    assert torch.equal(D, (A @ B.T))
