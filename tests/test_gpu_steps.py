"""GPU parity of every step against the oracle, element by element, on
workloads the oracle finishes in seconds (several tiles, ragged item counts,
both tile sizes, both head dimensions, fp32 and bf16), plus edge cases."""
import dataclasses
import math
import os

import numpy as np
import pytest
import torch

import block_sparse_attention_token_gb300 as sp
import synth
from oracle import sparsp_oracle as orc
from tests.gpu_helpers import (OracleChain, compare_augmented, compare_csr, compare_values, dev, host, i32,
                               jaccard_rows, status_word, workload)

pytestmark = [pytest.mark.gpu, pytest.mark.timeout(900)]

W = synth.Workload
SMALL = {
    "tiny": synth.WORKLOADS["tiny"],
    "medium": synth.WORKLOADS["medium"],
    # 2 batches x 3 heads, Bt = 128, d = 128: 72 items (fewer than the SMs)
    "r128": W("ragged-1.5k-bf16", 2, 3, 128, 4, 16, 24, 2, 8, 8, "bf16", "mean", 0.9, 2, 3, 2, False, True, 31),
    # Bt = 64 with d = 128 and an odd tile lattice (3 x 2 x 3)
    "r64": W("ragged-1.2k-bf16", 1, 5, 128, 6, 8, 24, 2, 4, 8, "bf16", "mean", 0.8, 3, 5, 3, False, True, 32),
    # Bt = 128 with d = 64
    "r128d64": W("ragged-2k-d64-bf16", 1, 4, 64, 4, 16, 32, 2, 8, 8, "bf16", "mean", 0.85, 2, 4, 2, False, True, 33),
    # fp32, Bt = 128, d = 128
    "f32big": W("f32-1k-d128", 1, 3, 128, 4, 8, 32, 2, 8, 8, "f32", "mean", 0.9, 1, 2, 1, False, False, 34),
    # 640 items: more than one wave of persistent CTAs with a ragged tail; low-rank scores
    "wave": W("wave-4k-lowrank-bf16", 1, 20, 128, 4, 32, 32, 2, 8, 8, "bf16", "lowrank", 0.0, 6, 4, 4, False, True, 35),
    # Bt = 64, d = 64 with an odd number of blocks (3 x 1 x 3 = 9): the last query
    # block of every head has no partner in the paired tcgen05 forward
    "r64odd": W("ragged-odd-576-bf16", 2, 3, 64, 6, 4, 24, 2, 4, 8, "bf16", "mean", 0.6, 2, 3, 2, False, True, 36),
}
BWD = ["medium", "r128", "r64", "r128d64", "wave", "r64odd"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _setup(name):
    wl = SMALL[name]
    _, data = workload(wl)
    return wl, data, sp.shape_of(wl)


@pytest.mark.parametrize("name", list(SMALL))
def test_reorder_bitexact(name):
    wl, data, shape = _setup(name)
    g = orc.grid_of(wl)
    q = dev(data["q"], wl)
    qb = sp.reorder(shape, q)
    ref = orc.reorder(data["q"], g)
    assert np.array_equal(host(qb), ref)
    back = sp.reorder(shape, qb, inverse=True)
    assert torch.equal(back, q)


@pytest.mark.parametrize("name", list(SMALL))
def test_block_scores(name):
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    qb, kb = dev(ch.qb, wl), dev(ch.kb, wl)
    if wl.estimator == "lowrank":
        wq, wk = (torch.from_numpy(data[x]).cuda() for x in ("wq", "wk"))
        S = sp.block_scores(shape, qb, kb, sp.EST_LOWRANK, wq, wk, 16)
    else:
        S = sp.block_scores(shape, qb, kb)
    torch.cuda.synchronize()
    got = host(S).astype(np.float64)
    scale = np.abs(ch.S64).max()
    np.testing.assert_allclose(got, ch.S64, rtol=2e-5, atol=2e-5 * scale)


@pytest.mark.parametrize("name", list(SMALL))
def test_reorder_pool_fused(name):
    """Fused tile reorder + pooling: the reorder is bit-exact, the means and the
    scores computed from them match the oracle."""
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    qb, qm = sp.reorder_pool(shape, dev(data["q"], wl))
    kb, km = sp.reorder_pool(shape, dev(data["k"], wl))
    assert np.array_equal(host(qb), ch.qb) and np.array_equal(host(kb), ch.kb)
    np.testing.assert_allclose(host(qm), orc.pool_means(ch.qb, ch.g.Bt), rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(host(km), orc.pool_means(ch.kb, ch.g.Bt), rtol=1e-5, atol=1e-6)
    if wl.estimator == "lowrank":
        wq, wk = (torch.from_numpy(data[x]).cuda() for x in ("wq", "wk"))
        S = sp.block_scores_pooled(shape, qm, km, sp.EST_LOWRANK, wq, wk, 16)
    else:
        S = sp.block_scores_pooled(shape, qm, km)
    torch.cuda.synchronize()
    np.testing.assert_allclose(host(S).astype(np.float64), ch.S64, rtol=2e-5, atol=2e-5 * np.abs(ch.S64).max())


@pytest.mark.parametrize("name", list(SMALL))
def test_select_bitexact_on_oracle_scores(name):
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    st = status_word()
    rp, ci = sp.select(shape, torch.from_numpy(ch.S32).cuda(), wl.top_p, wl.k_floor, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert int((ch.sel.margin < 1e-12).sum()) == 0
    assert compare_csr(host(rp), host(ci), ch.sel) == 0


@pytest.mark.parametrize("p,k", [(0.0, 0), (0.0, 3), (1.0, 0), (0.5, 999), (0.3, 1), (0.999, 2)])
def test_select_extremes(p, k):
    shape = sp.make_shape(1, 3, 4, 8, 32, 64, 4, 4, 4, "bf16")      # nb = 1*2*8 = 16
    S = synth.random_scores(41, 3 * 16, 16, scale=3.0)
    S[5, 3] = S[5, 7]          # exact ties
    S[9, :] = 0.0              # a flat row
    ref = orc.select(S, p, k)
    rp, ci = sp.select(shape, torch.from_numpy(S).cuda(), p, k)
    compare_csr(host(rp), host(ci), ref)


def test_select_rows_at_the_topp_crossing():
    """Rows built so that the Top-p decision turns on the last bit of e_j.
    Row r = [s0_r, 0, ..., 0] (nb = 16) has e = fl32(exp(-s0_r)) for the 15
    zeros and 1 for s0_r, so the prefix masses 1 + (k-1)e and Z = 1 + 15e are
    exact in float64; at p = 0.5 the count is 7 exactly when e <= 1/3. The
    values s0_r step through consecutive float32 numbers around ln 3, so e
    crosses 1/3 among them: a float32 exponential that is off by an ulp from
    the correctly rounded value would pick the wrong count on some row."""
    H = 16
    shape = sp.make_shape(1, H, 4, 8, 32, 64, 4, 4, 4, "bf16")      # nb = 16, 256 rows
    s0 = np.float32(math.log(3.0))
    for _ in range(shape.rows // 2):
        s0 = np.nextafter(s0, np.float32(0.0))
    S = np.zeros((shape.rows, 16), dtype=np.float32)
    for r in range(shape.rows):
        S[r, r % 16] = s0
        s0 = np.nextafter(s0, np.float32(10.0))
    ref = orc.select(S, 0.5, 1)
    counts = np.diff(ref.row_ptr)
    assert set(counts.tolist()) == {7, 8}, "the rows must straddle the crossing"
    st = status_word()
    rp, ci = sp.select(shape, torch.from_numpy(S).cuda(), 0.5, 1, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert compare_csr(host(rp), host(ci), ref) == 0
    assert np.array_equal(host(rp), ref.row_ptr)


def test_select_nan_row_is_empty_and_reported():
    shape = sp.make_shape(1, 1, 4, 8, 32, 64, 4, 4, 4, "bf16")
    S = synth.random_scores(42, 16, 16)
    S[4, 2] = np.nan
    S[11, 0] = np.inf
    st = status_word()
    rp, ci = sp.select(shape, torch.from_numpy(S).cuda(), 0.9, 2, status=st)
    rp = host(rp)
    assert st.item() == sp.DATA
    assert rp[5] - rp[4] == 0 and rp[12] - rp[11] == 0
    good = np.delete(np.arange(16), [4, 11])
    ref = orc.select(S[good], 0.9, 2)
    assert np.array_equal(np.diff(rp)[good], np.diff(ref.row_ptr))


def test_kv_gather_rejects_bad_lists():
    """Lists handed to sparsp_kv_gather by the caller: an index outside
    [0, nb) or a total beyond B*H*P*nb is reported (SPARSP_ERR_DATA) and never
    used as an address; the valid slots are still copied."""
    wl, data, shape = _setup("r128")
    ch = OracleChain(wl, data)
    g = ch.g
    k, v = dev(ch.kb, wl), dev(ch.vb, wl)
    good = sp.kv_demand(shape, wl.P, i32(ch.sel.row_ptr), i32(ch.sel.col_idx))
    torch.cuda.synchronize()
    total = int(good.dem_ptr[-1].item())
    dem_idx = good.dem_idx.clone()
    dem_idx[1] = g.nb + 7                      # out of range
    dem_idx[2] = -1
    out = dataclasses.replace(good, kg=torch.zeros((total, g.Bt, g.d), dtype=k.dtype, device="cuda"),
                              vg=torch.zeros((total, g.Bt, g.d), dtype=k.dtype, device="cuda"), dem_idx=dem_idx)
    st = status_word()
    sp.kv_gather(shape, wl.P, out, k, v, status=st)
    torch.cuda.synchronize()
    assert st.item() == sp.DATA
    j0 = int(dem_idx[0].item())
    assert torch.equal(out.kg[0], k[0, 0, j0 * g.Bt:(j0 + 1) * g.Bt])   # slot 0: partition 0 of head 0
    assert (out.kg[1] == 0).all() and (out.kg[2] == 0).all()
    bad_ptr = good.dem_ptr.clone()
    bad_ptr[-1] = shape.B * shape.H * wl.P * g.nb + 1
    st2 = status_word()
    sp.kv_gather(shape, wl.P, dataclasses.replace(out, dem_ptr=bad_ptr, dem_idx=good.dem_idx), k, v, status=st2)
    torch.cuda.synchronize()
    assert st2.item() == sp.DATA


@pytest.mark.parametrize("name", list(SMALL))
def test_kv_demand_bitexact(name):
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    g = ch.g
    ref = orc.kv_demand(ch.sel.row_ptr, ch.sel.col_idx, g.B, g.H, g.nb, wl.P, g.Bt, g.d, wl.elem_bytes,
                        ch.kb, ch.vb)
    st = status_word()
    out = sp.kv_demand(shape, wl.P, i32(ch.sel.row_ptr), i32(ch.sel.col_idx), dev(ch.kb, wl), dev(ch.vb, wl),
                       status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(host(out.bitmap).view(np.uint32).ravel(), ref.bitmap.ravel())
    assert np.array_equal(host(out.dem_ptr), ref.dem_ptr)
    total = int(ref.dem_ptr[-1])
    assert np.array_equal(host(out.dem_idx)[:total], ref.dem_idx)
    assert np.array_equal(host(out.kg)[:total], ref.kg)
    assert np.array_equal(host(out.vg)[:total], ref.vg)
    assert host(out.bytes).astype(np.uint64).tolist() == ref.bytes.tolist()


def test_kv_demand_capacity_shortfall():
    wl, data, shape = _setup("r64")
    ch = OracleChain(wl, data)
    g = ch.g
    ref = orc.kv_demand(ch.sel.row_ptr, ch.sel.col_idx, g.B, g.H, g.nb, wl.P, g.Bt, g.d, 2, ch.kb, ch.vb)
    cap = int(ref.dem_ptr[-1]) // 2
    st = status_word()
    out = sp.kv_demand(shape, wl.P, i32(ch.sel.row_ptr), i32(ch.sel.col_idx), dev(ch.kb, wl), dev(ch.vb, wl),
                       gather_cap=cap, status=st)
    torch.cuda.synchronize()
    assert st.item() == sp.CAPACITY
    assert np.array_equal(host(out.kg)[:cap], ref.kg[:cap])
    assert np.array_equal(host(out.dem_idx)[:int(ref.dem_ptr[-1])], ref.dem_idx)
    # sets only (no gather), one partition and one partition per block
    for P in (1, g.nb):
        r2 = orc.kv_demand(ch.sel.row_ptr, ch.sel.col_idx, g.B, g.H, g.nb, P, g.Bt, g.d, 2)
        o2 = sp.kv_demand(shape, P, i32(ch.sel.row_ptr), i32(ch.sel.col_idx))
        assert np.array_equal(host(o2.dem_ptr), r2.dem_ptr)
        assert np.array_equal(host(o2.dem_idx)[:int(r2.dem_ptr[-1])], r2.dem_idx)
        assert host(o2.bytes).astype(np.uint64).tolist() == r2.bytes.tolist()


@pytest.mark.parametrize("name", ["r64", "medium", "wave"])
def test_kv_gather_alone(name):
    """The lists from kv_demand without buffers, then kv_gather on another
    stream: the gathered tiles equal the oracle's; a short capacity is
    reported and the slots below it are still right."""
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    g = ch.g
    ref = orc.kv_demand(ch.sel.row_ptr, ch.sel.col_idx, g.B, g.H, g.nb, wl.P, g.Bt, g.d, wl.elem_bytes,
                        ch.kb, ch.vb)
    total = int(ref.dem_ptr[-1])
    kb, vb = dev(ch.kb, wl), dev(ch.vb, wl)
    st = status_word()
    lists = sp.kv_demand(shape, wl.P, i32(ch.sel.row_ptr), i32(ch.sel.col_idx), status=st)
    assert lists.kg is None
    kg = torch.empty((total + 3, g.Bt, g.d), dtype=kb.dtype, device="cuda")
    out = sp.DemandOut(lists.bitmap, lists.dem_ptr, lists.dem_idx, kg, torch.empty_like(kg), lists.bytes)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        sp.kv_gather(shape, wl.P, out, kb, vb, status=st, stream=side)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(host(out.kg)[:total], ref.kg)
    assert np.array_equal(host(out.vg)[:total], ref.vg)
    cap = total // 3
    out.kg.zero_()
    st2 = status_word()
    sp.kv_gather(shape, wl.P, out, kb, vb, gather_cap=cap, status=st2)
    torch.cuda.synchronize()
    assert st2.item() == sp.CAPACITY
    assert np.array_equal(host(out.kg)[:cap], ref.kg[:cap])


@pytest.mark.parametrize("name", list(SMALL))
def test_placement_and_placed_demand_bitexact(name):
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    g = ch.g
    own_ref = orc.placement(ch.sel.row_ptr, ch.sel.col_idx, g.B, g.H, g.nb, wl.P)
    st = status_word()
    owner = sp.placement(shape, wl.P, i32(ch.sel.row_ptr), i32(ch.sel.col_idx), status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(host(owner), own_ref)
    ref = orc.kv_demand(ch.sel.row_ptr, ch.sel.col_idx, g.B, g.H, g.nb, wl.P, g.Bt, g.d, wl.elem_bytes,
                        ch.kb, ch.vb, owner=own_ref)
    out = sp.kv_demand(shape, wl.P, i32(ch.sel.row_ptr), i32(ch.sel.col_idx), dev(ch.kb, wl), dev(ch.vb, wl),
                       status=st, owner=owner)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(host(out.bitmap).view(np.uint32).ravel(), ref.bitmap.ravel())
    assert np.array_equal(host(out.dem_ptr), ref.dem_ptr)
    total = int(ref.dem_ptr[-1])
    assert np.array_equal(host(out.dem_idx)[:total], ref.dem_idx)
    assert np.array_equal(host(out.kg)[:total], ref.kg)
    assert np.array_equal(host(out.vg)[:total], ref.vg)
    assert host(out.bytes).astype(np.uint64).tolist() == ref.bytes.tolist()


@pytest.mark.parametrize("P", [31, 32, 33, 100, 128])
def test_placement_partition_counts(P):
    """Both ways of picking the partition (a warp for up to 32 partitions,
    the whole CTA above) against the oracle, bit for bit."""
    wl, data, shape = _setup("medium")
    ch = OracleChain(wl, data)
    g = ch.g
    assert P <= g.nb
    own_ref = orc.placement(ch.sel.row_ptr, ch.sel.col_idx, g.B, g.H, g.nb, P)
    st = status_word()
    owner = sp.placement(shape, P, i32(ch.sel.row_ptr), i32(ch.sel.col_idx), status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(host(owner), own_ref)


def test_placement_hand_example_and_extremes():
    import json
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "placement_hand.json")))
    # 6 tiles of 4x4x4 tokens in one head
    shape = sp.make_shape(1, 1, 24, 4, 4, 64, 4, 4, 4, "bf16")
    assert shape.nb == gold["nb"]
    rows = gold["rows"]
    rp = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    ci = np.array([j for r in rows for j in r], dtype=np.int32)
    owner = sp.placement(shape, gold["P"], i32(rp), i32(ci))
    dem = sp.kv_demand(shape, gold["P"], i32(rp), i32(ci), owner=owner)
    torch.cuda.synchronize()
    assert host(owner)[0].tolist() == gold["owner"]
    tile2 = shape.Bt * shape.d * 2 * 2
    assert int(host(dem.bytes)[2]) == gold["remote_blocks_placed"] * tile2
    # one partition, and one partition per block, on a selected workload
    wl, data, shape = _setup("r64")
    ch = OracleChain(wl, data)
    g = ch.g
    for P in (1, g.nb):
        own_ref = orc.placement(ch.sel.row_ptr, ch.sel.col_idx, g.B, g.H, g.nb, P)
        owner = sp.placement(shape, P, i32(ch.sel.row_ptr), i32(ch.sel.col_idx))
        assert np.array_equal(host(owner), own_ref)
        r2 = orc.kv_demand(ch.sel.row_ptr, ch.sel.col_idx, g.B, g.H, g.nb, P, g.Bt, g.d, 2, owner=own_ref)
        o2 = sp.kv_demand(shape, P, i32(ch.sel.row_ptr), i32(ch.sel.col_idx), owner=owner)
        assert np.array_equal(host(o2.dem_ptr), r2.dem_ptr)
        assert np.array_equal(host(o2.dem_idx)[:int(r2.dem_ptr[-1])], r2.dem_idx)
        assert host(o2.bytes).astype(np.uint64).tolist() == r2.bytes.tolist()


def test_placed_demand_rejects_bad_owner():
    wl, data, shape = _setup("r64")
    ch = OracleChain(wl, data)
    g = ch.g
    own = orc.placement(ch.sel.row_ptr, ch.sel.col_idx, g.B, g.H, g.nb, wl.P)
    bad = own.copy()
    bad[0, 3] = wl.P          # block 3 belongs to no partition
    st = status_word()
    out = sp.kv_demand(shape, wl.P, i32(ch.sel.row_ptr), i32(ch.sel.col_idx), status=st,
                       owner=torch.from_numpy(bad).cuda())
    torch.cuda.synchronize()
    assert st.item() == sp.DATA
    # the other blocks are still served: the sets equal the oracle's with block 3 in no partition
    members = [[i for i in range(g.nb) if bad[0, i] == r] for r in range(wl.P)]
    ptr = host(out.dem_ptr)
    idx = host(out.dem_idx)
    for h in range(g.H):
        for r in range(wl.P):
            part = h * wl.P + r
            want = sorted({int(j) for i in members[r]
                           for j in ch.sel.col_idx[ch.sel.row_ptr[h * g.nb + i]:ch.sel.row_ptr[h * g.nb + i + 1]]})
            assert idx[ptr[part]:ptr[part + 1]].tolist() == want


def _csr_np(rows):
    rp = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    return rp, np.array([j for r in rows for j in r], dtype=np.int32)


@pytest.mark.parametrize("name", list(SMALL))
def test_balance_heads_bitexact(name):
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    g = ch.g
    costs = orc.head_costs(ch.sel.row_ptr, g.B, g.H, g.nb)
    for M in sorted({0, 1, wl.P, g.H * wl.P}):
        hr, mv = orc.balance_heads(costs, wl.P, M)
        out = sp.balance_heads(shape, wl.P, i32(ch.sel.row_ptr), M)
        torch.cuda.synchronize()
        assert np.array_equal(host(out.head_rank), hr), M
        assert host(out.migrations)[:g.B].tolist() == mv.tolist()
        hr0, _ = orc.balance_heads(costs, wl.P, 0)
        loads = host(out.loads)
        for b in range(g.B):
            assert loads[b, 0].tolist() == orc.rank_loads(costs[b], hr0[b], wl.P).tolist()
            assert loads[b, 1].tolist() == orc.rank_loads(costs[b], hr[b], wl.P).tolist()


def test_balance_hand_example():
    import json
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "balance_hand.json")))
    # 6 heads of 6 tiles (4x4x4 tokens); head h holds costs[h] pairs spread over its rows
    shape = sp.make_shape(1, 6, 24, 4, 4, 64, 4, 4, 4, "bf16")
    rows = []
    for c in gold["costs"]:
        for i in range(6):
            n = min(6, max(0, c - 6 * i))
            rows.append(list(range(n)))
    rp, _ = _csr_np(rows)
    out = sp.balance_heads(shape, gold["P"], i32(rp), 10)
    one = sp.balance_heads(shape, gold["P"], i32(rp), 1)
    torch.cuda.synchronize()
    assert host(out.head_rank)[0].tolist() == gold["head_rank"]
    assert int(host(out.migrations)[0]) == gold["migrations"]
    assert host(out.loads)[0, 0].tolist() == gold["contiguous_loads"]
    assert host(out.loads)[0, 1].tolist() == gold["loads"]
    assert host(one.head_rank)[0].tolist() == gold["head_rank_one_move"]


def test_augment_hand_example():
    import json
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "augment_hand.json")))
    # 3 tiles of 4x4x4 tokens, 2 heads
    shape = sp.make_shape(1, 2, 12, 4, 4, 64, 4, 4, 4, "bf16")
    assert shape.nb == gold["nb"]
    rp, ci = _csr_np(gold["rows"])
    S = torch.tensor(gold["scores"], dtype=torch.float32).cuda()
    st = status_word()
    rp2, ci2, added = sp.augment(shape, gold["P"], S, i32(rp), i32(ci), i32([gold["head_rank"]]), status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    rp2, ci2 = host(rp2), host(ci2)
    rows = [ci2[rp2[r]:rp2[r + 1]].tolist() for r in range(len(gold["rows"]))]
    assert rows == gold["augmented_rows"]
    assert host(added)[0].tolist() == gold["added"]


@pytest.mark.parametrize("name", list(SMALL))
def test_augment_matches_oracle(name):
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    g = ch.g
    hr, _ = orc.balance_heads(orc.head_costs(ch.sel.row_ptr, g.B, g.H, g.nb), wl.P, wl.P)
    ref = orc.augment(ch.S32.reshape(-1, g.nb), ch.sel.row_ptr, ch.sel.col_idx, g.B, g.H, g.nb, hr, wl.P)
    st = status_word()
    rp2, ci2, added = sp.augment(shape, wl.P, torch.from_numpy(ch.S32).cuda(), i32(ch.sel.row_ptr),
                                 i32(ch.sel.col_idx), i32(hr), status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert host(added).tolist() == ref.added.tolist()
    V = orc.block_values(ch.S32.reshape(-1, g.nb))
    n = compare_augmented(host(rp2), host(ci2), ref, ch.sel.row_ptr, ch.sel.col_idx, V, hr, g.B, g.H, g.nb, wl.P)
    print(f"{wl.name}: added {ref.added.tolist()}, rows differing from the oracle {n}")


def test_augment_edges():
    wl, data, shape = _setup("r64")
    ch = OracleChain(wl, data)
    g = ch.g
    S = torch.from_numpy(ch.S32).cuda()
    rp, ci = i32(ch.sel.row_ptr), i32(ch.sel.col_idx)
    # one rank: it is the critical one, nothing is added
    rp2, ci2, added = sp.augment(shape, 1, S, rp, ci, i32(np.zeros((g.B, g.H))))
    torch.cuda.synchronize()
    assert host(added).sum() == 0
    assert np.array_equal(host(rp2), ch.sel.row_ptr)
    assert np.array_equal(host(ci2)[:int(ch.sel.row_ptr[-1])], ch.sel.col_idx)
    # one head per rank and an empty selection: every rank is filled up to the critical head
    hr = np.arange(g.H, dtype=np.int32)[None, :].repeat(g.B, 0)
    ref = orc.augment(ch.S32.reshape(-1, g.nb), ch.sel.row_ptr, ch.sel.col_idx, g.B, g.H, g.nb, hr, g.H)
    rp2, ci2, added = sp.augment(shape, g.H, S, rp, ci, i32(hr))
    torch.cuda.synchronize()
    assert host(added).tolist() == ref.added.tolist()
    V = orc.block_values(ch.S32.reshape(-1, g.nb))
    compare_augmented(host(rp2), host(ci2), ref, ch.sel.row_ptr, ch.sel.col_idx, V, hr, g.B, g.H, g.nb, g.H)
    # a head on no rank: reported, its rows are copied unchanged
    bad = hr.copy()
    bad[0, 1] = g.H
    st = status_word()
    rp2, ci2, _ = sp.augment(shape, g.H, S, rp, ci, i32(bad), status=st)
    torch.cuda.synchronize()
    assert st.item() == sp.DATA
    rp2, ci2 = host(rp2), host(ci2)
    for i in range(g.nb):
        r = g.nb + i
        assert ci2[rp2[r]:rp2[r + 1]].tolist() == ch.sel.col_idx[ch.sel.row_ptr[r]:ch.sel.row_ptr[r + 1]].tolist()
    # a CSR capacity that is too small
    st = status_word()
    sp.augment(shape, g.H, S, rp, ci, i32(hr), col_idx_out=torch.empty(int(ch.sel.row_ptr[-1]), dtype=torch.int32,
                                                                        device="cuda"), status=st)
    torch.cuda.synchronize()
    assert st.item() == sp.CAPACITY


@pytest.mark.parametrize("name,pattern,P", [("r64", "mod4", 2), ("medium", "top16", 3)])
def test_augment_ties_across_rows(name, pattern, P):
    """Scores that repeat across rows and heads make whole groups of equal
    candidate values, so a rank's cut falls inside a group and the ties are
    shared out in (head, row, block) order (over a hundred rows for the
    top-of-16 pattern): the CSR must equal the oracle's."""
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    g = ch.g
    rows = g.B * g.H * g.nb
    j = np.arange(g.nb)
    level = j % 4 if pattern == "mod4" else (j % 16 == 0)
    S = np.tile(level.astype(np.float32), (rows, 1))
    costs = orc.head_costs(ch.sel.row_ptr, g.B, g.H, g.nb)
    hr, _ = orc.balance_heads(costs, P, 0)
    ref = orc.augment(S, ch.sel.row_ptr, ch.sel.col_idx, g.B, g.H, g.nb, hr, P)
    V = orc.block_values(S)
    split = 0
    for b in range(g.B):
        for r in range(P):
            rows_r = [(b * g.H + h) * g.nb + i for h in range(g.H) if hr[b, h] == r for i in range(g.nb)]
            cand = np.ones((len(rows_r), g.nb), bool)
            for k, row in enumerate(rows_r):
                cand[k, ch.sel.col_idx[ch.sel.row_ptr[row]:ch.sel.row_ptr[row + 1]]] = False
            vals = V[rows_r][cand]
            n_gt = int((vals > ref.cut[b, r]).sum())
            n_eq = int((vals == ref.cut[b, r]).sum())
            split += n_gt < int(ref.added[b, r]) < n_gt + n_eq
    assert split > 0, "no rank's cut falls inside a group of equal values"
    st = status_word()
    rp2, ci2, added = sp.augment(shape, P, torch.from_numpy(S).cuda(), i32(ch.sel.row_ptr), i32(ch.sel.col_idx),
                                 i32(hr), status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert host(added).tolist() == ref.added.tolist()
    rp2, ci2 = host(rp2), host(ci2)
    assert np.array_equal(rp2, ref.row_ptr)
    assert np.array_equal(ci2[:rp2[-1]], ref.col_idx)


@pytest.mark.parametrize("name,rank", [("tiny", 16), ("medium", 16), ("r128", 16), ("wave", 16), ("tiny", 1),
                                       ("medium", 5), ("r128", 64)])
def test_predictor_fit_matches_oracle(name, rank):
    wl, data, shape = _setup(name)
    g = orc.grid_of(wl)
    qb, kb = (orc.reorder(data[x], g) for x in ("q", "k"))
    qm = orc.pool_means(qb, g.Bt).astype(np.float32)
    km = orc.pool_means(kb, g.Bt).astype(np.float32)
    rng = np.random.default_rng(40)
    wq = (rng.standard_normal((g.H, g.d, rank)) / np.sqrt(g.d)).astype(np.float32)
    wk = (rng.standard_normal((g.H, g.d, rank)) / np.sqrt(g.d)).astype(np.float32)
    loss_ref, gq_ref, gk_ref = orc.predictor_loss_grad(qm, km, wq, wk)
    Wq, Wk = torch.from_numpy(wq).cuda(), torch.from_numpy(wk).cuda()
    Qm, Km = torch.from_numpy(qm).cuda(), torch.from_numpy(km).cuda()
    loss, gq, gk = sp.predictor_fit(shape, Qm, Km, Wq, Wk, lr=0.0)
    torch.cuda.synchronize()
    assert torch.equal(Wq, torch.from_numpy(wq).cuda()) and torch.equal(Wk, torch.from_numpy(wk).cuda())
    np.testing.assert_allclose(host(loss), loss_ref, rtol=1e-4)
    for got, ref in ((host(gq), gq_ref), (host(gk), gk_ref)):
        assert np.abs(got - ref).max() <= 1e-4 * np.abs(ref).max()
    # the step, and bitwise reproducibility
    lr = 0.05
    loss2, gq2, gk2 = sp.predictor_fit(shape, Qm, Km, Wq, Wk, lr=lr)
    torch.cuda.synchronize()
    assert torch.equal(loss2, loss) and torch.equal(gq2, gq) and torch.equal(gk2, gk)
    wq_ref, wk_ref, _ = orc.predictor_step(qm, km, wq, wk, lr)
    for got, ref, gr in ((host(Wq), wq_ref, gq_ref), (host(Wk), wk_ref, gk_ref)):
        assert np.abs(got - ref).max() <= lr * 1e-4 * np.abs(gr).max() + 1e-6 * np.abs(ref).max()
    if rank != 16:
        return
    # a few steps lower every head's loss
    for _ in range(5):
        sp.predictor_fit(shape, Qm, Km, Wq, Wk, lr=lr)
    loss3, _, _ = sp.predictor_fit(shape, Qm, Km, Wq, Wk, lr=0.0)
    torch.cuda.synchronize()
    assert (host(loss3) < host(loss)).all()


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("flat", [False, True])
def test_lpt_schedule_bitexact(name, flat):
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    g = ch.g
    items = sp.lpt_schedule(shape, i32(ch.sel.row_ptr), sp.SCHED_FLAT if flat else 0)
    ref = orc.lpt_order(ch.sel.row_ptr, g.B, g.H, g.nb, grouped=not flat)
    assert np.array_equal(host(items), ref)


@pytest.mark.parametrize("name", list(SMALL))
def test_csr_transpose_bitexact(name):
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    g = ch.g
    cp, ri = sp.csr_transpose(shape, i32(ch.sel.row_ptr), i32(ch.sel.col_idx))
    rcp, rri = orc.csc_of(ch.sel.row_ptr, ch.sel.col_idx, g.B, g.H, g.nb)
    assert np.array_equal(host(cp), rcp)
    assert np.array_equal(host(ri)[:len(rri)], rri)


def _attn_fwd_check(name, flags):
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    st = status_word()
    o, lse = sp.attn_fwd(shape, dev(ch.qb, wl), dev(ch.kb, wl), dev(ch.vb, wl), i32(ch.sel.row_ptr),
                         i32(ch.sel.col_idx), flags=flags, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    O, L = orc.attn_fwd(ch.qb, ch.kb, ch.vb, ch.sel.row_ptr, ch.sel.col_idx, ch.g.Bt, ch.scale)
    compare_values(host(o), O, wl, "O")
    compare_values(host(lse), L, wl, "LSE")
    return o, lse


@pytest.mark.parametrize("name", list(SMALL))
def test_attn_fwd(name):
    _attn_fwd_check(name, 0)


@pytest.mark.parametrize("name", ["medium", "r128", "wave"])
def test_attn_fwd_schedules_and_kernels_agree_bitwise(name):
    o1, l1 = _attn_fwd_check(name, 0)
    o2, l2 = _attn_fwd_check(name, sp.SCHED_FLAT)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o3, l3 = _attn_fwd_check(name, sp.KERNEL_PORTABLE)
    o4, l4 = _attn_fwd_check(name, sp.KERNEL_PORTABLE | sp.SCHED_FLAT)
    assert torch.equal(o3, o4) and torch.equal(l3, l4)
    o5, l5 = _attn_fwd_check(name, 0)
    assert torch.equal(o1, o5) and torch.equal(l1, l5)


@pytest.mark.parametrize("name", ["wave", "r128", "medium", "r64", "tiny"])
def test_attn_grid_size_does_not_change_results(name):
    """The persistent kernels pull work items from one counter, so the grid
    only changes which CTA runs an item, never how: forward (O, LSE) and
    backward (dQ, dK, dV) with 1, 7 and the full grid of CTAs are bitwise
    equal, and the full-grid run matches the oracle."""
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    q, k, v = dev(ch.qb, wl), dev(ch.kb, wl), dev(ch.vb, wl)
    rp, ci = i32(ch.sel.row_ptr), i32(ch.sel.col_idx)
    bwd = wl.dtype == "bf16"
    if bwd:
        do = synth.round_bf16(np.random.default_rng(wl.seed + 200).standard_normal(data["q"].shape,
                                                                                   dtype=np.float32))
        dob = dev(orc.reorder(do, ch.g), wl)
    runs = []
    for cap in (0, 1, 7):
        flags = sp.GRID_CAP(cap) if cap else 0
        st = status_word()
        o, lse = sp.attn_fwd(shape, q, k, v, rp, ci, flags=flags, status=st)
        grads = sp.attn_bwd(shape, q, k, v, o, lse, dob, rp, ci, flags=flags, status=st) if bwd else ()
        torch.cuda.synchronize()
        assert st.item() == 0, (cap, sp.status_string(st.item()))
        runs.append((o, lse, *grads))
    O, L = orc.attn_fwd(ch.qb, ch.kb, ch.vb, ch.sel.row_ptr, ch.sel.col_idx, ch.g.Bt, ch.scale)
    compare_values(host(runs[0][0]), O, wl, "O")
    compare_values(host(runs[0][1]), L, wl, "LSE")
    for cap, run in zip((1, 7), runs[1:]):
        for a, b, what in zip(runs[0], run, ("O", "LSE", "dQ", "dK", "dV")):
            assert torch.equal(a, b), f"{what} differs with a grid of {cap}"


@pytest.mark.parametrize("name", ["medium", "r128", "r64", "r128d64", "wave"])
def test_attn_fwd_raster_output(name):
    """O written straight into raster order equals the inverse reorder of the
    block-ordered O, bit for bit, and LSE is unchanged; the kernels without
    raster stores refuse the flag."""
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    q, k, v = dev(ch.qb, wl), dev(ch.kb, wl), dev(ch.vb, wl)
    rp, ci = i32(ch.sel.row_ptr), i32(ch.sel.col_idx)
    st = status_word()
    ob, lb = sp.attn_fwd(shape, q, k, v, rp, ci, status=st)
    o_r, lr = sp.attn_fwd(shape, q, k, v, rp, ci, flags=sp.OUT_RASTER, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert o_r.shape == (shape.B, shape.N, shape.H, shape.d)
    assert torch.equal(o_r, sp.reorder(shape, ob, inverse=True))
    assert torch.equal(lr, lb)
    with pytest.raises(sp.SparspError):
        sp.attn_fwd(shape, q, k, v, rp, ci, flags=sp.OUT_RASTER | sp.KERNEL_PORTABLE)


@pytest.mark.parametrize("overlap", [True, False])
@pytest.mark.parametrize("name", ["medium", "r128", "r64odd"])
def test_pipeline_raster_inputs(name, overlap):
    """A forward-only step that reads the raster inputs itself (no reorder
    pass) gives the block-ordered step's O, LSE, CSR and gathered tiles, bit
    for bit, also through HostPipeline from pinned host memory."""
    wl, data, shape = _setup(name)
    args = [dev(data[x], wl) for x in ("q", "k", "v")]
    plain = sp.Pipeline(shape, wl.estimator, wl.top_p, wl.k_floor, wl.P, overlap_demand=overlap)
    direct = sp.Pipeline(shape, wl.estimator, wl.top_p, wl.k_floor, wl.P, overlap_demand=overlap,
                         raster_inputs=True)
    o1, l1 = [t.clone() for t in plain.forward(*args)]
    o2, l2 = [t.clone() for t in direct.forward(*args)]
    torch.cuda.synchronize()
    assert plain.status.item() == 0 and direct.status.item() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(plain.row_ptr, direct.row_ptr)
    total = int(plain.demand.dem_ptr[-1].item())
    assert torch.equal(plain.demand.kg[:total], direct.demand.kg[:total])
    assert torch.equal(plain.demand.vg[:total], direct.demand.vg[:total])
    hp = sp.HostPipeline(direct)
    hin = [t.cpu().pin_memory() for t in args]
    ho = torch.empty(o1.shape, dtype=o1.dtype).pin_memory()
    for _ in range(3):
        hp.step(*hin, ho)
    hp.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(ho.cuda(), o1)


@pytest.mark.parametrize("name", ["tiny", "medium", "r128", "r64odd"])
def test_raster_pooling_and_gather(name):
    """Tile means from a pooling read of raster input (no reordered copy)
    equal those of the fused reorder, and the demand gather from raster K, V
    equals the gather from the block-ordered tensors, bit for bit."""
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    x = dev(data["q"], wl)
    _, m1 = sp.reorder_pool(shape, x)
    m2 = sp.pool_means(shape, x)
    rp, ci = i32(ch.sel.row_ptr), i32(ch.sel.col_idx)
    st = status_word()
    blocked = sp.kv_demand(shape, wl.P, rp, ci, dev(ch.kb, wl), dev(ch.vb, wl), status=st)
    raster = dataclasses.replace(blocked, kg=torch.full_like(blocked.kg, 3), vg=torch.full_like(blocked.vg, 3))
    sp.kv_gather(shape, wl.P, raster, dev(data["k"], wl), dev(data["v"], wl), status=st, raster=True)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(m1, m2)
    total = int(blocked.dem_ptr[-1].item())
    assert total > 0
    assert torch.equal(blocked.kg[:total], raster.kg[:total]) and torch.equal(blocked.vg[:total], raster.vg[:total])


@pytest.mark.parametrize("out_raster", [False, True])
@pytest.mark.parametrize("name", ["medium", "r128", "r64", "r128d64", "wave", "r64odd"])
def test_attn_fwd_raster_input(name, out_raster):
    """With IN_RASTER the kernel reads Q, K, V in raster order [B, N, H, d]
    (each block one 5-D TMA box) and gives bit for bit what it gives on the
    block-ordered tensors; the portable kernels refuse the flag."""
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    rp, ci = i32(ch.sel.row_ptr), i32(ch.sel.col_idx)
    qb, kb, vb = dev(ch.qb, wl), dev(ch.kb, wl), dev(ch.vb, wl)
    qr, kr, vr = (dev(data[x], wl) for x in ("q", "k", "v"))
    extra = sp.OUT_RASTER if out_raster else 0
    st = status_word()
    o1, l1 = sp.attn_fwd(shape, qb, kb, vb, rp, ci, flags=extra, status=st)
    o2, l2 = sp.attn_fwd(shape, qr, kr, vr, rp, ci, flags=extra | sp.IN_RASTER, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    with pytest.raises(sp.SparspError):
        sp.attn_fwd(shape, qr, kr, vr, rp, ci, flags=sp.IN_RASTER | sp.KERNEL_PORTABLE)


@pytest.mark.parametrize("portable", [False, True])
@pytest.mark.parametrize("name", ["r128", "tiny", "r64", "medium", "r64odd", "r128d64"])
def test_attn_fwd_empty_and_bad_rows(name, portable):
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    g = ch.g
    rp = ch.sel.row_ptr.astype(np.int64)
    counts = np.diff(rp)
    counts[1] = 0                                   # an empty row
    counts[-1] = 0
    rows = [np.asarray(ch.sel.col_idx[rp[r]:rp[r + 1]]) if counts[r] else np.zeros(0, np.int64)
            for r in range(len(counts))]
    rows[2] = rows[2].copy()
    rows[2][0] = g.nb + 5                           # out of range -> the row is skipped
    ci = np.concatenate(rows).astype(np.int32)
    rp2 = np.concatenate([[0], np.cumsum([len(x) for x in rows])]).astype(np.int32)
    st = status_word()
    sentinel = 7.0
    o = torch.full((g.B, g.H, g.N, g.d), sentinel, dtype=shape.torch_dtype, device="cuda")
    lse = torch.full((g.B, g.H, g.N), sentinel, device="cuda")
    sp.attn_fwd(shape, dev(ch.qb, wl), dev(ch.kb, wl), dev(ch.vb, wl), i32(rp2), i32(ci), o=o, lse=lse,
                flags=sp.KERNEL_PORTABLE if portable else 0, status=st)
    torch.cuda.synchronize()
    assert st.item() == sp.DATA
    O, L = host(o), host(lse)
    Bt = g.Bt
    assert (O[0, 0, Bt:2 * Bt] == 0).all() and np.isneginf(L[0, 0, Bt:2 * Bt]).all()
    assert (O[0, 0, 2 * Bt:3 * Bt] == sentinel).all() and (L[0, 0, 2 * Bt:3 * Bt] == sentinel).all()
    ok = [r for r in range(len(counts)) if r not in (1, 2, len(counts) - 1)]
    rows_ok = [(r // (g.H * g.nb), (r // g.nb) % g.H, r % g.nb) for r in ok[:6]]
    Oref, Lref = orc.attn_fwd(ch.qb, ch.kb, ch.vb, rp2, ci, Bt, ch.scale, rows=rows_ok)
    for (b, h, i) in rows_ok:
        sl = slice(i * Bt, (i + 1) * Bt)
        compare_values(O[b, h, sl], Oref[b, h, sl], wl, "O")


@pytest.mark.parametrize("name,seed", [("r64odd", 0), ("r64", 1), ("medium", 2)])
def test_attn_fwd_pairs_with_unrelated_rows(name, seed):
    """64-token blocks run as pairs of neighbouring query blocks over the union
    of their two rows. Random rows of random lengths (some empty, some with
    every block, most sharing few blocks with their neighbour) exercise every
    mask: O and LSE match the oracle, empty rows give O = 0 and LSE = -inf."""
    wl, data, shape = _setup(name)
    g = orc.grid_of(wl)
    rng = np.random.default_rng(500 + seed)
    rows = []
    for r in range(g.B * g.H * g.nb):
        kind = rng.integers(0, 6)
        n = 0 if kind == 0 else (g.nb if kind == 1 else int(rng.integers(1, g.nb + 1)))
        rows.append(np.sort(rng.choice(g.nb, size=n, replace=False)))
    rp = np.concatenate([[0], np.cumsum([len(x) for x in rows])]).astype(np.int32)
    ci = np.concatenate(rows).astype(np.int32)
    qb, kb, vb = (orc.reorder(data[x], g) for x in ("q", "k", "v"))
    st = status_word()
    o, lse = sp.attn_fwd(shape, dev(qb, wl), dev(kb, wl), dev(vb, wl), i32(rp), i32(ci), status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    O, L = orc.attn_fwd(qb, kb, vb, rp, ci, g.Bt, 1.0 / math.sqrt(g.d))
    on, ln = host(o), host(lse)
    empty = [r for r in range(len(rows)) if len(rows[r]) == 0]
    assert empty, "the seed must give some empty rows"
    for r in empty:
        b, h, i = r // (g.H * g.nb), (r // g.nb) % g.H, r % g.nb
        sl = slice(i * g.Bt, (i + 1) * g.Bt)
        assert (on[b, h, sl] == 0).all() and np.isneginf(ln[b, h, sl]).all()
        O[b, h, sl] = 0.0
        L[b, h, sl] = 0.0
        ln[b, h, sl] = 0.0
    compare_values(on, O, wl, "O")
    compare_values(ln, L, wl, "LSE")


def test_attn_fwd_pair_rejects_a_repeated_index():
    """A row listing a key block twice is reported (SPARSP_ERR_DATA) by the
    paired 64-token kernel and skipped; its partner row is still computed."""
    wl, data, shape = _setup("r64odd")
    ch = OracleChain(wl, data)
    g = ch.g
    rows = [ch.sel.col_idx[ch.sel.row_ptr[r]:ch.sel.row_ptr[r + 1]].copy() for r in range(g.B * g.H * g.nb)]
    rows[2] = np.concatenate([rows[2], rows[2][:1]])            # row 2 repeats its first block
    rp = np.concatenate([[0], np.cumsum([len(x) for x in rows])]).astype(np.int32)
    ci = np.concatenate(rows).astype(np.int32)
    st = status_word()
    o = torch.full((g.B, g.H, g.N, g.d), 7.0, dtype=shape.torch_dtype, device="cuda")
    lse = torch.full((g.B, g.H, g.N), 7.0, device="cuda")
    sp.attn_fwd(shape, dev(ch.qb, wl), dev(ch.kb, wl), dev(ch.vb, wl), i32(rp), i32(ci), o=o, lse=lse, status=st)
    torch.cuda.synchronize()
    assert st.item() == sp.DATA
    on = host(o)
    assert (on[0, 0, 2 * g.Bt:3 * g.Bt] == 7.0).all()
    O, _ = orc.attn_fwd(ch.qb, ch.kb, ch.vb, ch.sel.row_ptr, ch.sel.col_idx, g.Bt, ch.scale, rows=[(0, 0, 3)])
    compare_values(on[0, 0, 3 * g.Bt:4 * g.Bt], O[0, 0, 3 * g.Bt:4 * g.Bt], wl, "O of the partner row")


def test_attn_bwd_pair_rejects_a_repeated_index():
    """The dQ kernel with 64-token blocks (pairs) reports a CSR row that lists a
    key block twice (SPARSP_ERR_DATA), leaves that row block's dQ unwritten and
    still computes its partner's."""
    wl, data, shape = _setup("r64odd")
    ch = OracleChain(wl, data)
    g = ch.g
    q, k, v = dev(ch.qb, wl), dev(ch.kb, wl), dev(ch.vb, wl)
    rp, ci = i32(ch.sel.row_ptr), i32(ch.sel.col_idx)
    o, lse = sp.attn_fwd(shape, q, k, v, rp, ci)
    rows = [ch.sel.col_idx[ch.sel.row_ptr[r]:ch.sel.row_ptr[r + 1]].copy() for r in range(g.B * g.H * g.nb)]
    rows[2] = np.concatenate([rows[2], rows[2][:1]])            # row 2 repeats its first block
    rp2 = np.concatenate([[0], np.cumsum([len(x) for x in rows])]).astype(np.int32)
    ci2 = np.concatenate(rows).astype(np.int32)
    dob = orc.reorder(synth.round_bf16(np.random.default_rng(wl.seed + 9).standard_normal(
        data["q"].shape, dtype=np.float32)), g)
    st = status_word()
    dq = torch.full_like(q, 7.0)
    sp.attn_bwd(shape, q, k, v, o, lse, dev(dob, wl), i32(rp2), i32(ci2), dq=dq, status=st)
    torch.cuda.synchronize()
    assert st.item() == sp.DATA
    dqn = host(dq)
    assert (dqn[0, 0, 2 * g.Bt:3 * g.Bt] == 7.0).all()
    dQ, _, _ = orc.attn_bwd(ch.qb, ch.kb, ch.vb, dob, ch.sel.row_ptr, ch.sel.col_idx, g.Bt, ch.scale,
                            q_blocks={(0, 0, 3)}, k_blocks=set())
    compare_values(dqn[0, 0, 3 * g.Bt:4 * g.Bt], dQ[0, 0, 3 * g.Bt:4 * g.Bt], wl, "dQ of the partner row")


@pytest.mark.parametrize("name", BWD)
def test_attn_bwd(name):
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    do = data.get("do")
    if do is None:      # forward-only workload: a seeded upstream gradient
        do = synth.round_bf16(np.random.default_rng(wl.seed + 100).standard_normal(data["q"].shape,
                                                                                   dtype=np.float32))
    dob = orc.reorder(do, ch.g)
    st = status_word()
    q, k, v = dev(ch.qb, wl), dev(ch.kb, wl), dev(ch.vb, wl)
    rp, ci = i32(ch.sel.row_ptr), i32(ch.sel.col_idx)
    o, lse = sp.attn_fwd(shape, q, k, v, rp, ci, status=st)
    dq, dk, dv = sp.attn_bwd(shape, q, k, v, o, lse, dev(dob, wl), rp, ci, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    dQ, dK, dV = orc.attn_bwd(ch.qb, ch.kb, ch.vb, dob, ch.sel.row_ptr, ch.sel.col_idx, ch.g.Bt, ch.scale)
    compare_values(host(dq), dQ, wl, "dQ")
    compare_values(host(dk), dK, wl, "dK")
    compare_values(host(dv), dV, wl, "dV")
    # deterministic: a second run is bitwise identical
    dq2, dk2, dv2 = sp.attn_bwd(shape, q, k, v, o, lse, dev(dob, wl), rp, ci, flags=sp.SCHED_FLAT)
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)
    # dK and dV by two kernels instead of one: the same gradients against the oracle
    st3 = status_word()
    dq3, dk3, dv3 = sp.attn_bwd(shape, q, k, v, o, lse, dev(dob, wl), rp, ci, flags=sp.BWD_SPLIT_KV, status=st3)
    torch.cuda.synchronize()
    assert st3.item() == 0
    assert torch.equal(dq, dq3)
    compare_values(host(dk3), dK, wl, "dK (two kernels)")
    compare_values(host(dv3), dV, wl, "dV (two kernels)")


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("name", ["r128", "wave", "r64", "r128d64", "medium", "r64odd"])
def test_attn_bwd_raster_output(name, split):
    """With OUT_RASTER the backward reads the raster O the forward wrote and
    writes dQ, dK, dV straight into raster order: bit for bit the inverse
    reorder of the block-ordered gradients. The portable kernels refuse the
    flag before enqueuing anything."""
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    dob = orc.reorder(synth.round_bf16(np.random.default_rng(wl.seed + 101).standard_normal(
        data["q"].shape, dtype=np.float32)), ch.g)
    q, k, v, do = dev(ch.qb, wl), dev(ch.kb, wl), dev(ch.vb, wl), dev(dob, wl)
    rp, ci = i32(ch.sel.row_ptr), i32(ch.sel.col_idx)
    st = status_word()
    extra = sp.BWD_SPLIT_KV if split else 0
    o, lse = sp.attn_fwd(shape, q, k, v, rp, ci, status=st)
    o_r, lse_r = sp.attn_fwd(shape, q, k, v, rp, ci, flags=sp.OUT_RASTER, status=st)
    grads = sp.attn_bwd(shape, q, k, v, o, lse, do, rp, ci, flags=extra, status=st)
    raster = sp.attn_bwd(shape, q, k, v, o_r, lse_r, do, rp, ci, flags=sp.OUT_RASTER | extra, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    for a, b, what in zip(grads, raster, ("dQ", "dK", "dV")):
        assert torch.equal(sp.reorder(shape, a, inverse=True), b), f"{what} in raster order differs"
    with pytest.raises(sp.SparspError):
        sp.attn_bwd(shape, q, k, v, o_r, lse_r, do, rp, ci, flags=sp.OUT_RASTER | sp.KERNEL_PORTABLE)


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("name", ["tiny", "medium", "r128", "wave"])
def test_pipeline_end_to_end(name, fused):
    """The whole chain on the GPU (its own scores and selection) against the
    oracle's own chain: selection agreement is reported, outputs are compared
    on every row whose block set agrees."""
    wl, data, shape = _setup(name)
    ch = OracleChain(wl, data)
    g = ch.g
    pipe = sp.Pipeline(shape, wl.estimator, wl.top_p, wl.k_floor, wl.P, backward=wl.backward,
                       fused_estimation=fused)
    args = [dev(data[x], wl) for x in ("q", "k", "v")]
    kw = {}
    if wl.estimator == "lowrank":
        kw = dict(wq=torch.from_numpy(data["wq"]).cuda(), wk=torch.from_numpy(data["wk"]).cuda())
    o, lse = pipe.forward(*args, **kw)
    torch.cuda.synchronize()
    assert pipe.status.item() == 0
    rp, ci = host(pipe.row_ptr), host(pipe.col_idx)
    jac = jaccard_rows(rp, ci, ch.sel.row_ptr, ch.sel.col_idx)
    print(f"{wl.name}: block-set agreement (mean row Jaccard) {jac:.6f}")
    assert jac > 0.99
    same = [r for r in range(len(rp) - 1)
            if np.array_equal(ci[rp[r]:rp[r + 1]], ch.sel.col_idx[ch.sel.row_ptr[r]:ch.sel.row_ptr[r + 1]])]
    O, _ = orc.attn_fwd(ch.qb, ch.kb, ch.vb, ch.sel.row_ptr, ch.sel.col_idx, g.Bt, ch.scale)
    ob = orc.reorder(host(o), g)
    for r in same:
        b, h, i = r // (g.H * g.nb), (r // g.nb) % g.H, r % g.nb
        sl = slice(i * g.Bt, (i + 1) * g.Bt)
        compare_values(ob[b, h, sl], O[b, h, sl], wl, f"O row {r}")


@pytest.mark.parametrize("name", ["medium", "r128", "wave"])
def test_pipeline_overlapped_demand_equals_serial(name):
    """KV demand beside attention on its own stream gives the same O, LSE,
    bitmap, lists, gathered tiles and byte counts as the serial order, over
    several back-to-back steps (the side streams' buffers are reused)."""
    wl, data, shape = _setup(name)
    args = [dev(data[x], wl) for x in ("q", "k", "v")]
    kw = {}
    if wl.estimator == "lowrank":
        kw = dict(wq=torch.from_numpy(data["wq"]).cuda(), wk=torch.from_numpy(data["wk"]).cuda())
    serial = sp.Pipeline(shape, wl.estimator, wl.top_p, wl.k_floor, wl.P, overlap_demand=False)
    over = sp.Pipeline(shape, wl.estimator, wl.top_p, wl.k_floor, wl.P, overlap_demand=True)
    o1, l1 = serial.forward(*args, **kw)
    for _ in range(3):
        o2, l2 = over.forward(*args, **kw)
    torch.cuda.synchronize()
    assert serial.status.item() == 0 and over.status.item() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    d1, d2 = serial.demand, over.demand
    assert torch.equal(d1.bitmap, d2.bitmap) and torch.equal(d1.dem_ptr, d2.dem_ptr)
    assert torch.equal(d1.bytes, d2.bytes)
    total = int(d1.dem_ptr[-1].item())
    assert torch.equal(d1.dem_idx[:total], d2.dem_idx[:total])
    assert torch.equal(d1.kg[:total], d2.kg[:total]) and torch.equal(d1.vg[:total], d2.vg[:total])


@pytest.mark.parametrize("name", ["tiny", "medium", "r128", "wave"])
def test_pipeline_graph_replay(name):
    """A captured step (Pipeline.capture, one CUDA graph) replays bit for bit
    what the eager step computes, and follows new inputs written in place into
    the bound buffers; with a backward workload the graph holds the backward
    too."""
    wl, data, shape = _setup(name)
    args = [dev(data[x], wl) for x in ("q", "k", "v")]
    kw = {}
    if wl.estimator == "lowrank":
        kw = dict(wq=torch.from_numpy(data["wq"]).cuda(), wk=torch.from_numpy(data["wk"]).cuda())
    do = dev(synth.round_bf16(np.random.default_rng(wl.seed + 7).standard_normal(data["q"].shape,
                                                                              dtype=np.float32)), wl)
    eager = sp.Pipeline(shape, wl.estimator, wl.top_p, wl.k_floor, wl.P, backward=wl.backward)
    graphed = sp.Pipeline(shape, wl.estimator, wl.top_p, wl.k_floor, wl.P, backward=wl.backward)
    step = graphed.capture(*args, **kw, dout=do if wl.backward else None)

    def run_eager():
        out = eager.forward(*args, **kw)
        return [t.clone() for t in (out + eager.backward(do) if wl.backward else out)]

    for _ in range(2):
        want = run_eager()
        got = [t.clone() for t in step.replay()]
        torch.cuda.synchronize()
        assert eager.status.item() == 0 and graphed.status.item() == 0
        assert len(got) == len(want)
        for a, b in zip(got, want):
            assert torch.equal(a, b)
        # new inputs, written in place into the buffers the graph is bound to
        for t in args:
            t.mul_(-1.5)


@pytest.mark.parametrize("name", ["medium", "r128"])
def test_pipeline_with_placement(name):
    """Placement inside the pipeline: owner and demand equal the oracle's on
    the GPU's own CSR, and attention output is unchanged (placement only moves
    KV demand, never the attended sets)."""
    wl, data, shape = _setup(name)
    args = [dev(data[x], wl) for x in ("q", "k", "v")]
    plain = sp.Pipeline(shape, wl.estimator, wl.top_p, wl.k_floor, wl.P)
    placed = sp.Pipeline(shape, wl.estimator, wl.top_p, wl.k_floor, wl.P, placement=True)
    o1, _ = plain.forward(*args)
    o2, _ = placed.forward(*args)
    torch.cuda.synchronize()
    assert placed.status.item() == 0
    assert torch.equal(o1, o2)
    g = orc.grid_of(wl)
    rp, ci = host(placed.row_ptr), host(placed.col_idx)
    own_ref = orc.placement(rp, ci, g.B, g.H, g.nb, wl.P)
    assert np.array_equal(host(placed.owner), own_ref)
    ref = orc.kv_demand(rp, ci, g.B, g.H, g.nb, wl.P, g.Bt, g.d, wl.elem_bytes, owner=own_ref)
    assert host(placed.demand.bytes).astype(np.uint64).tolist() == ref.bytes.tolist()
    assert placed.kernels_per_forward() == plain.kernels_per_forward() + 2


@pytest.mark.parametrize("name", ["medium", "wave"])
def test_pipeline_with_balance_and_augment(name):
    """Balancing + augmentation inside the pipeline: attention runs on the
    augmented CSR, whose outputs match the oracle's attention on that CSR, and
    the backward uses the same CSR."""
    wl, data, shape = _setup(name)
    g = orc.grid_of(wl)
    args = [dev(data[x], wl) for x in ("q", "k", "v")]
    kw = {}
    if wl.estimator == "lowrank":
        kw = dict(wq=torch.from_numpy(data["wq"]).cuda(), wk=torch.from_numpy(data["wk"]).cuda())
    pipe = sp.Pipeline(shape, wl.estimator, wl.top_p, wl.k_floor, wl.P, migrations=wl.P, augment=True,
                       backward=True)
    o, lse = pipe.forward(*args, **kw)
    torch.cuda.synchronize()
    assert pipe.status.item() == 0
    rp, ci = (host(t) for t in pipe.csr)
    rp0 = host(pipe.row_ptr)
    costs = orc.head_costs(rp0, g.B, g.H, g.nb)
    hr, _ = orc.balance_heads(costs, wl.P, wl.P)
    assert np.array_equal(host(pipe.balance.head_rank), hr)
    assert int(rp[-1]) == int(rp0[-1]) + int(host(pipe.added).sum())
    assert pipe.kernels_per_forward() == sp.Pipeline(shape, wl.estimator, wl.top_p, wl.k_floor, wl.P,
                                                      backward=True).kernels_per_forward() + 15
    qb, kb, vb = (orc.reorder(data[x], g) for x in ("q", "k", "v"))
    O, _ = orc.attn_fwd(qb, kb, vb, rp, ci, g.Bt, 1.0 / math.sqrt(g.d))
    compare_values(orc.reorder(host(o), g), O, wl, "O on the augmented CSR")
    dout = torch.randn_like(args[0])
    pipe.backward(dout)
    torch.cuda.synchronize()
    assert pipe.status.item() == 0


def test_pipeline_with_predictor_fitting():
    """A fitting step inside the pipeline: selection uses the weights before
    the step, the weights afterwards equal a standalone step from the same
    start, and the reported loss is the oracle's."""
    wl, data, shape = _setup("wave")
    g = orc.grid_of(wl)
    args = [dev(data[x], wl) for x in ("q", "k", "v")]
    wq0, wk0 = (torch.from_numpy(data[x]).cuda() for x in ("wq", "wk"))
    plain = sp.Pipeline(shape, wl.estimator, wl.top_p, wl.k_floor, wl.P)
    o1, _ = plain.forward(*args, wq=wq0, wk=wk0)
    wq, wk = wq0.clone(), wk0.clone()
    fit = sp.Pipeline(shape, wl.estimator, wl.top_p, wl.k_floor, wl.P, predictor_lr=0.01)
    o2, _ = fit.forward(*args, wq=wq, wk=wk)
    torch.cuda.synchronize()
    assert fit.status.item() == 0
    assert torch.equal(o1, o2)
    wq2, wk2 = wq0.clone(), wk0.clone()
    sp.predictor_fit(shape, fit.qmeans, fit.kmeans, wq2, wk2, lr=0.01)
    torch.cuda.synchronize()
    assert torch.equal(wq, wq2) and torch.equal(wk, wk2) and not torch.equal(wq, wq0)
    qb, kb = (orc.reorder(data[x], g) for x in ("q", "k"))
    loss_ref, _, _ = orc.predictor_loss_grad(orc.pool_means(qb, g.Bt), orc.pool_means(kb, g.Bt),
                                             data["wq"], data["wk"])
    np.testing.assert_allclose(host(fit.predictor_loss), loss_ref, rtol=1e-4)
    assert fit.kernels_per_forward() == plain.kernels_per_forward() + 7


def test_host_pipeline_overlapped_steps_match_device_pipeline():
    """Pinned-host streaming (copies overlapped with neighbouring steps) gives,
    step for step, exactly what the device pipeline gives."""
    wl = SMALL["r128"]
    _, data = workload(wl)
    shape = sp.shape_of(wl)
    pipe = sp.Pipeline(shape, wl.estimator, wl.top_p, wl.k_floor, wl.P)
    hp = sp.HostPipeline(pipe)
    steps = []
    for n in range(4):
        scale = 1.0 + 0.25 * n
        hq, hk, hv = (torch.from_numpy(synth.round_bf16(data[x] * np.float32(scale))).bfloat16().pin_memory()
                      for x in "qkv")
        steps.append((hq, hk, hv, torch.empty_like(hq).pin_memory()))
    for hq, hk, hv, ho in steps:
        hp.step(hq, hk, hv, ho)
    hp.synchronize()
    torch.cuda.synchronize()
    for hq, hk, hv, ho in steps:
        o, _ = pipe.forward(hq.cuda(), hk.cuda(), hv.cuda())
        torch.cuda.synchronize()
        assert torch.equal(ho, o.cpu())
    assert pipe.status.item() == 0


def test_host_pipeline_training_steps_match_device_pipeline():
    """Overlapped forward + backward steps from pinned host memory give, step
    for step, exactly the device pipeline's O, dQ, dK and dV."""
    wl = SMALL["r128"]
    _, data = workload(wl)
    shape = sp.shape_of(wl)
    pipe = sp.Pipeline(shape, wl.estimator, wl.top_p, wl.k_floor, wl.P, backward=True)
    hp = sp.HostPipeline(pipe)
    rng = np.random.default_rng(50)
    steps = []
    for n in range(3):
        scale = np.float32(1.0 + 0.25 * n)
        hq, hk, hv = (torch.from_numpy(synth.round_bf16(data[x] * scale)).bfloat16().pin_memory() for x in "qkv")
        hdo = torch.from_numpy(synth.round_bf16(rng.standard_normal(data["q"].shape).astype(np.float32))
                               ).bfloat16().pin_memory()
        outs = tuple(torch.empty_like(hq).pin_memory() for _ in range(4))
        steps.append(((hq, hk, hv, hdo), outs))
    for ins, outs in steps:
        hp.train_step(*ins, *outs)
    hp.synchronize()
    torch.cuda.synchronize()
    for (hq, hk, hv, hdo), (ho, hdq, hdk, hdv) in steps:
        o, _ = pipe.forward(hq.cuda(), hk.cuda(), hv.cuda())
        o = o.clone()
        dq, dk, dv = pipe.backward(hdo.cuda())
        torch.cuda.synchronize()
        assert torch.equal(ho, o.cpu())
        for h, d in ((hdq, dq), (hdk, dk), (hdv, dv)):
            assert torch.equal(h, d.cpu())
    assert pipe.status.item() == 0
