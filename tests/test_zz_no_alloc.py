"""sparsp_select_noalloc: the selection entry point for callers that cannot
allocate device memory at call time (for example an inference-engine plug-in
whose enqueue step must not allocate, or a service that reserves all of its
device memory at start-up). Its scratch is a fixed array inside the library
instead of a caller workspace. Called through the C ABI, it must give exactly
what sparsp_select gives, on two calls in a row with different inputs (the
shared array keeps the previous call's contents, which must not leak), and
the same CSR as the oracle's selection on the same scores."""
import ctypes

import numpy as np
import pytest
import torch

import block_sparse_attention_token_gb300 as sp
import synth
from oracle import sparsp_oracle as orc
from tests.gpu_helpers import compare_csr

pytestmark = [pytest.mark.gpu, pytest.mark.timeout(300)]


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return sp.lib()


def _select_with_workspace(lib, shape, scores, p, k, stream):
    rows = shape.rows
    rp = torch.empty(rows + 1, dtype=torch.int32, device="cuda")
    ci = torch.full((rows * shape.nb,), -1, dtype=torch.int32, device="cuda")
    ws = torch.empty(lib.sparsp_select_workspace_size(ctypes.byref(shape)), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.sparsp_select(ctypes.byref(shape), scores.data_ptr(), ctypes.c_float(p), k, rp.data_ptr(),
                           ci.data_ptr(), ws.data_ptr(), ws.numel(), st.data_ptr(), stream)
    assert rc == sp.OK
    return rp, ci, st


def _select_no_alloc(lib, shape, scores, p, k, stream):
    rows = shape.rows
    rp = torch.empty(rows + 1, dtype=torch.int32, device="cuda")
    ci = torch.full((rows * shape.nb,), -1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.sparsp_select_noalloc(ctypes.byref(shape), scores.data_ptr(), ctypes.c_float(p), k, rp.data_ptr(),
                                   ci.data_ptr(), st.data_ptr(), stream)
    assert rc == sp.OK, sp.status_string(rc)
    return rp, ci, st


@pytest.mark.parametrize("dims,p,k", [
    # Wan-14B layer shape: 40 heads x 240 blocks = 9,600 rows
    ((1, 40, 20, 32, 48, 128, 2, 8, 8), 0.95, 8),
    # training shape: 24 heads x 512 blocks = 12,288 rows, Top-k only
    ((1, 24, 16, 64, 64, 128, 2, 8, 8), 0.0, 52),
])
def test_no_alloc_select_matches_workspace_select_twice(lib, dims, p, k):
    shape = sp.make_shape(*dims, "bf16")
    stream = torch.cuda.current_stream().cuda_stream
    for call, seed in enumerate((101, 202)):
        S = torch.from_numpy(synth.random_scores(seed + dims[1], shape.rows, shape.nb, scale=2.0 + call)).cuda()
        rp_ref, ci_ref, st_ref = _select_with_workspace(lib, shape, S, p, k, stream)
        rp, ci, st = _select_no_alloc(lib, shape, S, p, k, stream)
        torch.cuda.synchronize()
        assert st.item() == 0 and st_ref.item() == 0
        assert torch.equal(rp, rp_ref), f"call {call}: row_ptr differs"
        nnz = int(rp[-1].item())
        assert torch.equal(ci[:nnz], ci_ref[:nnz]), f"call {call}: col_idx differs"
        assert nnz > 0
        compare_csr(rp.cpu().numpy(), ci.cpu().numpy(), orc.select(S.cpu().numpy(), p, k))


def test_no_alloc_select_larger_call_then_smaller_and_a_nan_row(lib):
    """A large call fills more rows of the shared array than a smaller call
    that follows it; the smaller call must not see the larger one's rows. A
    row holding NaN is written empty (threshold 0, count 0) and reported, and
    the rows after it are unaffected. Each call is compared bit for bit with
    sparsp_select on its own workspace, and the finite rows with the oracle."""
    stream = torch.cuda.current_stream().cuda_stream
    calls = [
        ((1, 24, 16, 64, 64, 128, 2, 8, 8), 0.9, 4, 7, None),     # 12,288 rows
        ((1, 3, 4, 16, 24, 128, 2, 8, 8), 0.8, 2, 8, None),       # 36 rows
        ((1, 5, 6, 8, 24, 128, 2, 4, 8), 0.7, 3, 9, (17, 3)),      # 90 rows, NaN in row 17
    ]
    for call, (dims, p, k, seed, nan_at) in enumerate(calls):
        shape = sp.make_shape(*dims, "bf16")
        S_np = synth.random_scores(seed, shape.rows, shape.nb, scale=3.0)
        if nan_at is not None:
            S_np[nan_at] = np.nan
        S = torch.from_numpy(S_np).cuda()
        rp_ref, ci_ref, st_ref = _select_with_workspace(lib, shape, S, p, k, stream)
        rp, ci, st = _select_no_alloc(lib, shape, S, p, k, stream)
        torch.cuda.synchronize()
        want = sp.DATA if nan_at is not None else 0
        assert st.item() == want and st_ref.item() == want, (call, st.item(), st_ref.item())
        assert torch.equal(rp, rp_ref), f"call {call}: row_ptr differs"
        nnz = int(rp[-1].item())
        assert torch.equal(ci[:nnz], ci_ref[:nnz]), f"call {call}: col_idx differs"
        rp_h, ci_h = rp.cpu().numpy(), ci.cpu().numpy()
        good = np.arange(shape.rows)
        if nan_at is not None:
            r = nan_at[0]
            assert rp_h[r + 1] == rp_h[r], "the NaN row must be empty"
            good = np.delete(good, r)
        # the finite rows against the oracle (bit for bit, up to rows whose Top-p
        # crossing lies within float32 rounding of p)
        counts = np.diff(rp_h)[good]
        rp_sub = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        ci_sub = np.concatenate([ci_h[rp_h[r]:rp_h[r + 1]] for r in good]).astype(np.int32)
        compare_csr(rp_sub, ci_sub, orc.select(S_np[good], p, k))


def test_no_alloc_select_rejects_too_many_rows(lib):
    # 65 heads x 1024 blocks = 66,560 rows > 65,536
    shape = sp.make_shape(1, 65, 16, 64, 128, 128, 2, 8, 8, "bf16")
    assert shape.rows > 65536
    fake = 1 << 20
    rc = lib.sparsp_select_noalloc(ctypes.byref(shape), fake, ctypes.c_float(0.9), 1, fake, fake, None, None)
    assert rc == sp.WORKSPACE
