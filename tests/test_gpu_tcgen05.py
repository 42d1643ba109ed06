"""The tcgen05 building blocks of the attention kernel on one 128x128x128 tile:
TMA boxes with 128-byte swizzle, K-major and MN-major shared-memory
descriptors, and a TMEM-resident A operand, against a float64 product."""
import numpy as np
import pytest
import torch

import block_sparse_attention_token_gb300 as sp

pytestmark = [pytest.mark.gpu, pytest.mark.timeout(300)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _tiles(seed):
    g = torch.Generator().manual_seed(seed)
    a = torch.randn(128, 128, generator=g).bfloat16()
    b = torch.randn(128, 128, generator=g).bfloat16()
    return a, b


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_umma_tile(mode):
    a, b = _tiles(mode + 1)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = sp.diag_umma_tile(a.cuda(), b.cuda(), mode, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    A, Bm = a.double().numpy(), b.double().numpy()
    ref = A @ Bm.T if mode == 0 else A @ Bm
    got = d.cpu().double().numpy()
    err = np.abs(got - ref).max()
    if err > 1e-3 and mode > 0:
        # report whether the other assignment of leading/stride offsets would have matched
        alt = sp.diag_umma_tile(a.cuda(), b.cuda(), mode, lbo=1024, sbo=16384).cpu().double().numpy()
        print(f"mode {mode}: max err {err:.3g}; with lbo/sbo swapped {np.abs(alt - ref).max():.3g}")
    assert err < 1e-3, f"mode {mode}: max err {err:.3g}"


def test_bounded_wait_times_out_and_the_context_stays_usable():
    """A wait that nothing completes gives up after its limit, reports
    SPARSP_ERR_TIMEOUT through the status word, and the kernel returns: the
    next launches on the same context run normally."""
    import time
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    sp.diag_wait_timeout(50_000_000, st)          # 50 ms
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert st.item() == sp.TIMEOUT
    assert 0.04 < elapsed < 5.0
    # the context still works: a tile product matches its reference
    g = torch.Generator(device="cpu").manual_seed(3)
    a = torch.randn(128, 128, generator=g).bfloat16().cuda()
    b = torch.randn(128, 128, generator=g).bfloat16().cuda()
    d = sp.diag_umma_tile(a, b, 0)
    torch.cuda.synchronize()
    ref = a.float() @ b.float().t()
    assert torch.allclose(d, ref, rtol=1e-3, atol=1e-2)
