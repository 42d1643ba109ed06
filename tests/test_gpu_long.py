"""Long sequences: 2,048 and 4,096 blocks per head (up to 524,288 tokens in
128-token blocks, the sequence lengths of "Dynamic Sparsity in Large-Scale
Video DiT Training", summary), and 1,024-block heads for the d = 64 and the
64-token-block (paired) tcgen05 kernels, forward and backward. The steps run
in the pipeline's launch configuration; cheap outputs are compared in full
with the oracle, attention values and gradients on sampled blocks the oracle
computes one by one."""
import numpy as np
import pytest
import torch

import block_sparse_attention_token_gb300 as sp
import synth
from oracle import sparsp_oracle as orc
from tests.gpu_helpers import OracleChain, compare_csr, compare_values, dev, host, i32, status_word

pytestmark = [pytest.mark.gpu, pytest.mark.slow, pytest.mark.timeout(1800)]

W = synth.Workload
LONG = {
    # 64-token blocks, d = 64: 2,048 blocks of 2x4x8 tokens (131,072 tokens), Top-p
    "long2k-d64": W("long-131k-d64-bf16", 1, 2, 64, 32, 64, 64, 2, 4, 8, "bf16", "mean", 0.9, 8, 8, 8,
                    False, False, 41),
    # 128-token blocks, d = 128: 2,048 blocks (262,144 tokens), Top-k 10%
    "long2k-d128": W("long-262k-bf16", 1, 2, 128, 64, 64, 64, 2, 8, 8, "bf16", "mean", 0.0, 205, 8, 8,
                     False, True, 42),
    # 4,096 blocks (524,288 tokens), one head, Top-k 10%
    "long4k": W("long-524k-bf16", 1, 1, 128, 128, 64, 64, 2, 8, 8, "bf16", "mean", 0.0, 410, 8, 8,
                False, False, 43),
    # 128-token blocks, d = 64: 1,024 blocks (131,072 tokens), Top-k 10%, with a backward
    "long1k-d64": W("long-131k-bt128-d64-bf16", 1, 2, 64, 32, 64, 64, 2, 8, 8, "bf16", "mean", 0.0, 103, 8, 8,
                    False, True, 44),
    # 64-token blocks (pairs), d = 128: 1,024 blocks of 1x8x8 (65,536 tokens), Top-k 10%, with a backward
    "long1k-bt64": W("long-65k-bt64-bf16", 1, 2, 128, 16, 64, 64, 1, 8, 8, "bf16", "mean", 0.0, 103, 8, 8,
                     False, True, 45),
}


class Run:
    def __init__(self, name):
        self.wl = synth.WORKLOADS.get(name) or LONG[name]
        self.data = synth.make(self.wl)
        self.shape = sp.shape_of(self.wl)
        self.ch = OracleChain(self.wl, self.data)
        wl = self.wl
        self.pipe = sp.Pipeline(self.shape, wl.estimator, wl.top_p, wl.k_floor, wl.P, backward=wl.backward)
        self.q, self.k, self.v = (dev(self.data[x], wl) for x in ("q", "k", "v"))
        self.pipe.forward(self.q, self.k, self.v)
        torch.cuda.synchronize()


@pytest.fixture(scope="module", params=list(LONG))
def run(request):
    import __graft_entry__
    __graft_entry__.build()
    r = Run(request.param)
    yield r
    del r
    torch.cuda.empty_cache()


def test_long_reorder_scores_and_status(run):
    assert run.shape.nb in (1024, 2048, 4096)
    assert run.pipe.status.item() == 0
    assert np.array_equal(host(run.pipe.qb), run.ch.qb)
    S = run.ch.S64
    np.testing.assert_allclose(host(run.pipe.scores).astype(np.float64), S, rtol=2e-5, atol=2e-5 * np.abs(S).max())


def test_long_selection_bitexact(run):
    """The CTA-per-row selection (rows longer than 1,024 blocks) against the
    oracle on the same float32 scores, bit for bit."""
    wl, ch = run.wl, run.ch
    assert int((ch.sel.margin < 1e-12).sum()) == 0
    st = status_word()
    rp, ci = sp.select(run.shape, torch.from_numpy(ch.S32).cuda(), wl.top_p, wl.k_floor, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert compare_csr(host(rp), host(ci), ch.sel) == 0
    counts = np.diff(ch.sel.row_ptr)
    print(f"{wl.name}: nb {run.shape.nb}, row lengths {counts.min()}..{counts.max()}, nnz {int(ch.sel.row_ptr[-1])}")


def test_long_demand_and_schedule_bitexact(run):
    wl, ch, g = run.wl, run.ch, run.ch.g
    ref = orc.kv_demand(ch.sel.row_ptr, ch.sel.col_idx, g.B, g.H, g.nb, wl.P, g.Bt, g.d, wl.elem_bytes)
    st = status_word()
    out = sp.kv_demand(run.shape, wl.P, i32(ch.sel.row_ptr), i32(ch.sel.col_idx), status=st)
    items = sp.lpt_schedule(run.shape, i32(ch.sel.row_ptr))
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(host(out.bitmap).view(np.uint32).ravel(), ref.bitmap.ravel())
    assert np.array_equal(host(out.dem_ptr), ref.dem_ptr)
    assert np.array_equal(host(out.dem_idx)[:int(ref.dem_ptr[-1])], ref.dem_idx)
    assert host(out.bytes).astype(np.uint64).tolist() == ref.bytes.tolist()
    assert np.array_equal(host(items), orc.lpt_order(ch.sel.row_ptr, g.B, g.H, g.nb))


def test_long_attention_forward_sampled(run):
    wl, ch, g = run.wl, run.ch, run.ch.g
    st = status_word()
    rp, ci = i32(ch.sel.row_ptr), i32(ch.sel.col_idx)
    o, lse = sp.attn_fwd(run.shape, run.pipe.qb, run.pipe.kb, run.pipe.vb, rp, ci, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    on, ln = host(o), host(lse)
    assert np.isfinite(on).all() and np.isfinite(ln).all()
    counts = np.diff(ch.sel.row_ptr)
    rng = np.random.default_rng(3)
    mags = np.abs(on.reshape(g.B * g.H * g.nb, -1)).max(axis=1)
    pick = {int(np.argmax(counts)), int(np.argmin(counts)), len(counts) - 1, int(np.argmax(mags))}
    pick |= set(int(x) for x in rng.choice(len(counts), size=4, replace=False))
    rows = sorted((r // (g.H * g.nb), (r // g.nb) % g.H, r % g.nb) for r in pick)
    O, L = orc.attn_fwd(ch.qb, ch.kb, ch.vb, ch.sel.row_ptr, ch.sel.col_idx, g.Bt, ch.scale, rows=rows)
    for (b, h, i) in rows:
        sl = slice(i * g.Bt, (i + 1) * g.Bt)
        compare_values(on[b, h, sl], O[b, h, sl], wl, f"O {(b, h, i)}")
        compare_values(ln[b, h, sl], L[b, h, sl], wl, f"LSE {(b, h, i)}")


def test_long_attention_backward_sampled(run):
    """Gradients with the CSR transpose of 2,048-block heads: dQ of sampled
    rows, dK and dV of the two key blocks of lowest fan-in and one at the
    lower quartile."""
    wl, ch, g = run.wl, run.ch, run.ch.g
    if not wl.backward:
        pytest.skip("forward-only workload")
    dob = orc.reorder(run.data["do"], g)
    st = status_word()
    rp, ci = i32(ch.sel.row_ptr), i32(ch.sel.col_idx)
    o, lse = sp.attn_fwd(run.shape, run.pipe.qb, run.pipe.kb, run.pipe.vb, rp, ci, status=st)
    dq, dk, dv = sp.attn_bwd(run.shape, run.pipe.qb, run.pipe.kb, run.pipe.vb, o, lse, dev(dob, wl), rp, ci,
                             status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    cp, _ = orc.csc_of(ch.sel.row_ptr, ch.sel.col_idx, g.B, g.H, g.nb)
    fan_in = np.diff(cp)
    order = [int(c) for c in np.argsort(fan_in, kind="stable") if fan_in[c] > 0]
    cols = [order[0], order[1], order[len(order) // 4]]
    to_bhj = lambda c: (c // (g.H * g.nb), (c // g.nb) % g.H, c % g.nb)
    kblocks = [to_bhj(c) for c in cols]
    qblocks = [to_bhj(r) for r in (0, g.nb // 3, g.B * g.H * g.nb - 1)]
    dQ, dK, dV = orc.attn_bwd(ch.qb, ch.kb, ch.vb, dob, ch.sel.row_ptr, ch.sel.col_idx, g.Bt, ch.scale,
                              q_blocks=qblocks, k_blocks=kblocks)
    dqn, dkn, dvn = host(dq), host(dk), host(dv)
    for (b, h, i) in qblocks:
        sl = slice(i * g.Bt, (i + 1) * g.Bt)
        compare_values(dqn[b, h, sl], dQ[b, h, sl], wl, f"dQ {(b, h, i)}")
    for (b, h, j) in kblocks:
        sl = slice(j * g.Bt, (j + 1) * g.Bt)
        compare_values(dkn[b, h, sl], dK[b, h, sl], wl, f"dK {(b, h, j)}")
        compare_values(dvn[b, h, sl], dV[b, h, sl], wl, f"dV {(b, h, j)}")
