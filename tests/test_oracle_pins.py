"""Pins that tie the CPU oracle to the pages and to mathematics, not to itself.

Each test checks an oracle function against a hand-worked example, a closed
form, a brute-force enumeration, an invariant, or a library routine that the
oracle does not call (PyTorch's scaled_dot_product_attention and autograd).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import synth
from oracle import sparsp_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _tiny():
    wl = synth.WORKLOADS["tiny"]
    data = synth.make(wl)
    g = orc.grid_of(wl)
    qb, kb, vb = (orc.reorder(data[x], g) for x in ("q", "k", "v"))
    return wl, g, data, qb, kb, vb


# ----------------------------------------------------------------- reorder

def test_reorder_hand_example():
    gold = _load("reorder_hand.json")
    g = orc.Grid(1, 1, **{k: gold["grid"][k] for k in ("T", "Y", "X")}, d=1,
                 **{k: gold["grid"][k] for k in ("ta", "tb", "tc")})
    assert orc.blocked_position(g).tolist() == gold["blocked_position"]


def test_reorder_is_bijection_and_inverse():
    wl, g, data, qb, _, _ = _tiny()
    pos = orc.blocked_position(g)
    assert sorted(pos.tolist()) == list(range(g.N))
    back = orc.reorder_inverse(qb, g)
    assert np.array_equal(back, data["q"])


def test_reorder_tokens_lie_in_their_tile():
    # brute force over every token: its (t, y, x) is inside the box of the tile
    # whose rows it lands in, and each tile's rows hold exactly Bt tokens
    g = orc.Grid(1, 1, 4, 8, 12, 1, 2, 4, 3)
    pos = orc.blocked_position(g)
    nY, nX = g.Y // g.tb, g.X // g.tc
    seen = {}
    for n in range(g.N):
        t, y, x = n // (g.Y * g.X), (n // g.X) % g.Y, n % g.X
        j = int(pos[n]) // g.Bt
        bt, by, bx = j // (nY * nX), (j // nX) % nY, j % nX
        assert bt * g.ta <= t < (bt + 1) * g.ta
        assert by * g.tb <= y < (by + 1) * g.tb
        assert bx * g.tc <= x < (bx + 1) * g.tc
        seen[j] = seen.get(j, 0) + 1
    assert set(seen.values()) == {g.Bt} and len(seen) == g.nb


def test_reorder_rejects_indivisible_grid():
    with pytest.raises(ValueError):
        orc.blocked_position(orc.Grid(1, 1, 3, 4, 4, 1, 2, 2, 2))


# ----------------------------------------------------------------- scores

def test_mean_scores_equal_token_pair_average():
    wl, g, data, qb, kb, _ = _tiny()
    S = orc.scores_mean(qb, kb, g.Bt)
    S_tok = orc.scores_mean_tokenpairs(qb, kb, g.Bt)
    assert S.shape == (1, 2, 16, 16)
    np.testing.assert_allclose(S, S_tok, rtol=1e-10, atol=1e-12)


def test_mean_scores_hand_values():
    # two blocks of two tokens, d = 2: block means are (1, 1), (0, 2) for Q
    # and (2, 0), (1, -1) for K
    qb = np.array([[[[1, 0], [1, 2], [0, 1], [0, 3]]]], dtype=np.float64)
    kb = np.array([[[[3, 0], [1, 0], [1, -2], [1, 0]]]], dtype=np.float64)
    S = orc.scores_mean(qb, kb, 2)
    assert S[0, 0].tolist() == [[2.0, 0.0], [0.0, -2.0]]


def test_lowrank_tokenlevel_equals_pooled_and_reduces_to_mean():
    wl, g, data, qb, kb, _ = _tiny()
    rng = np.random.default_rng(11)
    wq = rng.normal(size=(g.H, g.d, 16)) / 8
    wk = rng.normal(size=(g.H, g.d, 16)) / 8
    S_pool = orc.scores_lowrank(qb, kb, wq, wk, g.Bt)
    S_tok = orc.scores_lowrank_tokenlevel(qb, kb, wq, wk, g.Bt)
    np.testing.assert_allclose(S_pool, S_tok, rtol=1e-9, atol=1e-12)
    some = [(0, 1, 3, 5), (0, 0, 15, 0)]
    np.testing.assert_allclose(orc.scores_lowrank_tokenlevel(qb, kb, wq, wk, g.Bt, pairs=some),
                               [S_tok[p] for p in some], rtol=1e-12)
    eye = np.broadcast_to(np.eye(g.d), (g.H, g.d, g.d))
    np.testing.assert_allclose(orc.scores_lowrank(qb, kb, eye, eye, g.Bt),
                               orc.scores_mean_tokenpairs(qb, kb, g.Bt), rtol=1e-10, atol=1e-12)


# ----------------------------------------------------------------- select

def test_softmax_rows_sum_to_one_and_two_point_closed_form():
    rng = np.random.default_rng(3)
    for _ in range(20):
        s = rng.normal(size=37) * 5
        assert abs(orc.row_softmax(s).sum() - 1.0) < 1e-12
    delta = 0.731
    pi = orc.row_softmax([delta, 0.0])
    assert abs(pi[0] - 1.0 / (1.0 + math.exp(-delta))) < 1e-15


def test_select_hand_examples():
    for case in _load("select_hand.json")["cases"]:
        S = np.array([case["scores"]], dtype=np.float32)
        sel = orc.select(S, case["p"], case["k"])
        assert sel.col_idx.tolist() == case["selected"], case["why"]
        assert sel.row_ptr.tolist() == [0, len(case["selected"])]


def test_select_topp_minimal_by_subset_brute_force():
    # nb = 16: enumerate all 2^16 subsets; the smallest subset whose softmax
    # mass reaches p has the size the oracle picks, and the oracle's set is a
    # subset of that size with the largest mass
    S = synth.random_scores(5, 6, 16, scale=2.0)
    masks = np.array(list(itertools.product([0, 1], repeat=16)), dtype=bool)
    sizes = masks.sum(axis=1)
    for p in (0.3, 0.6, 0.9):
        sel = orc.select(S, p, 1)
        for r in range(S.shape[0]):
            pi = orc.row_softmax(S[r].astype(np.float64))
            mass = masks.astype(np.float64) @ pi
            reach = mass >= float(np.float32(p)) - 1e-12
            best = sizes[reach].min()
            got = sel.col_idx[sel.row_ptr[r]:sel.row_ptr[r + 1]]
            assert len(got) == best
            assert abs(pi[got].sum() - mass[(sizes == best)].max()) < 1e-12
            assert list(got) == sorted(got)


def test_select_p_extremes_and_floor():
    S = synth.random_scores(9, 50, 24)
    dense = orc.select(S, 1.0, 0)
    assert dense.col_idx.tolist() == list(range(24)) * 50
    for k in (0, 1, 5, 30):
        s0 = orc.select(S, 0.0, k)
        counts = np.diff(s0.row_ptr)
        assert (counts == min(max(k, 1), 24)).all()
        # the kept blocks are the top-scoring ones
        for r in range(50):
            got = s0.col_idx[s0.row_ptr[r]:s0.row_ptr[r + 1]]
            thr = np.sort(S[r])[::-1][counts[r] - 1]
            assert (S[r][got] >= thr).all()
    for k in (2, 7, 24, 99):
        sel = orc.select(S, 0.5, k)
        assert (np.diff(sel.row_ptr) >= min(k, 24)).all()


def test_select_tie_break_by_index():
    S = np.array([[1.0, 2.0, 2.0, 2.0, 1.0, 2.0]], dtype=np.float32)
    assert orc.select(S, 0.0, 2).col_idx.tolist() == [1, 2]
    assert orc.select(S, 0.0, 5).col_idx.tolist() == [0, 1, 2, 3, 5]
    # -0.0 and +0.0 are the same score
    S = np.array([[-0.0, 0.0, -1.0]], dtype=np.float32)
    assert orc.select(S, 0.0, 1).col_idx.tolist() == [0]


def test_select_rejects_nonfinite():
    with pytest.raises(ValueError):
        orc.select(np.array([[0.0, np.nan]], dtype=np.float32), 0.5, 1)


# ----------------------------------------------------------------- demand

def test_demand_hand_example():
    gold = _load("demand_hand.json")
    dem = orc.kv_demand(np.array(gold["row_ptr"]), np.array(gold["col_idx"]), gold["B"], gold["H"],
                        gold["nb"], gold["P"], gold["Bt"], gold["d"], gold["elem_bytes"])
    assert dem.bitmap.ravel().tolist() == gold["bitmap"]
    assert dem.dem_ptr.tolist() == gold["dem_ptr"]
    assert dem.dem_idx.tolist() == gold["dem_idx"]
    b = gold["bytes"]
    assert dem.bytes.tolist() == [b["demanded"], b["all"], b["remote_demanded"], b["remote_all"]]


def test_demand_brute_force_and_bounds():
    wl, g, data, qb, kb, vb = _tiny()
    S = orc.scores_mean(qb, kb, g.Bt).astype(np.float32).reshape(-1, g.nb)
    sel = orc.select(S, wl.top_p, wl.k_floor)
    dem = orc.kv_demand(sel.row_ptr, sel.col_idx, g.B, g.H, g.nb, wl.P, g.Bt, g.d, 4, kb, vb)
    # brute force: a block is demanded by partition r iff some row of r has it
    M = orc.token_mask(sel.row_ptr, sel.col_idx, g.B, g.H, g.nb, g.Bt)[:, :, ::g.Bt, ::g.Bt]
    slot = 0
    for h in range(g.H):
        for r, (lo, hi) in enumerate(orc.partition_bounds(g.nb, wl.P)):
            want = np.nonzero(M[0, h, lo:hi].any(axis=0))[0]
            got = dem.dem_idx[dem.dem_ptr[h * wl.P + r]:dem.dem_ptr[h * wl.P + r + 1]]
            assert got.tolist() == want.tolist()
            for j in want:
                assert (dem.bitmap[0, h, r, j // 32] >> (j % 32)) & 1
                assert np.array_equal(dem.kg[slot], kb[0, h, j * g.Bt:(j + 1) * g.Bt])
                assert np.array_equal(dem.vg[slot], vb[0, h, j * g.Bt:(j + 1) * g.Bt])
                slot += 1
    assert slot == len(dem.dem_idx) <= wl.P * g.nb * g.B * g.H
    demanded, all_b, rdem, rall = (int(x) for x in dem.bytes)
    assert demanded <= all_b and rdem <= rall and rall * wl.P == all_b * (wl.P - 1)


# ----------------------------------------------------------------- attention forward

def test_attention_closed_form_two_keys():
    # one query block of one token, two key blocks of one token, d = 2
    qb = np.array([[[[1.0, 0.0], [0.0, 0.0]]]])
    kb = np.array([[[[1.0, 0.0], [0.0, 1.0]]]])
    vb = np.array([[[[2.0, 0.0], [0.0, 4.0]]]])
    rp = np.array([0, 2, 3])
    ci = np.array([0, 1, 1])
    O, L = orc.attn_fwd(qb, kb, vb, rp, ci, 1, scale=1.0)
    p0 = math.e / (math.e + 1.0)
    np.testing.assert_allclose(O[0, 0, 0], [2 * p0, 4 * (1 - p0)], rtol=1e-14)
    assert abs(L[0, 0, 0] - math.log(math.e + 1.0)) < 1e-14
    # the second query block sees only key 1: O = v1, LSE = 0 for a zero query
    np.testing.assert_allclose(O[0, 0, 1], [0.0, 4.0])
    assert L[0, 0, 1] == 0.0


def test_attention_equals_masked_dense_brute_force():
    wl, g, data, qb, kb, vb = _tiny()
    S = orc.scores_mean(qb, kb, g.Bt).astype(np.float32).reshape(-1, g.nb)
    sel = orc.select(S, wl.top_p, wl.k_floor)
    scale = 1 / math.sqrt(g.d)
    O, L = orc.attn_fwd(qb, kb, vb, sel.row_ptr, sel.col_idx, g.Bt, scale)
    M = orc.token_mask(sel.row_ptr, sel.col_idx, g.B, g.H, g.nb, g.Bt)
    Od, Ld = orc.attn_dense_masked(qb, kb, vb, M, scale)
    np.testing.assert_allclose(O, Od, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(L, Ld, rtol=1e-12)
    # exp(LSE) is the masked row sum of exp(scores)
    s = scale * np.einsum("bhqd,bhkd->bhqk", qb.astype(np.float64), kb.astype(np.float64))
    np.testing.assert_allclose(np.exp(L), np.where(M, np.exp(s), 0).sum(-1), rtol=1e-12)
    # same thing through PyTorch's attention with a boolean mask
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qb.astype(np.float64)), torch.from_numpy(kb.astype(np.float64)),
        torch.from_numpy(vb.astype(np.float64)), attn_mask=torch.from_numpy(M), scale=scale)
    np.testing.assert_allclose(O, ref.numpy(), rtol=1e-10, atol=1e-12)


def test_attention_all_blocks_is_dense_attention_and_equivariant():
    wl, g, data, qb, kb, vb = _tiny()
    S = orc.scores_mean(qb, kb, g.Bt).astype(np.float32).reshape(-1, g.nb)
    sel = orc.select(S, 1.0, 0)                       # p = 1: every block
    O, L = orc.attn_fwd(qb, kb, vb, sel.row_ptr, sel.col_idx, g.Bt)
    # dense attention on the raster layout, through PyTorch, then reordered:
    # the block organisation only permutes tokens
    q, k, v = (torch.from_numpy(np.transpose(data[x], (0, 2, 1, 3)).astype(np.float64)) for x in "qkv")
    dense = torch.nn.functional.scaled_dot_product_attention(q, k, v).numpy()   # [B,H,N,d] raster
    dense_raster = np.transpose(dense, (0, 2, 1, 3))
    np.testing.assert_allclose(orc.reorder(dense_raster, g), O, rtol=1e-10, atol=1e-12)


def test_attention_constant_values_and_empty_row():
    wl, g, data, qb, kb, vb = _tiny()
    S = orc.scores_mean(qb, kb, g.Bt).astype(np.float32).reshape(-1, g.nb)
    sel = orc.select(S, wl.top_p, wl.k_floor)
    const = np.broadcast_to(np.arange(g.d, dtype=np.float64), vb.shape)
    O, _ = orc.attn_fwd(qb, kb, const, sel.row_ptr, sel.col_idx, g.Bt)
    np.testing.assert_allclose(O, const, rtol=1e-13)
    rp = np.array([0, 0, 1]); ci = np.array([1])
    O, L = orc.attn_fwd(qb[:, :1, :2 * g.Bt], kb[:, :1, :2 * g.Bt], vb[:, :1, :2 * g.Bt], rp, ci, g.Bt)
    assert (O[0, 0, :g.Bt] == 0).all() and np.isneginf(L[0, 0, :g.Bt]).all()


# ----------------------------------------------------------------- attention backward

def _micro_case():
    wl, data = synth.micro()
    g = orc.grid_of(wl)
    qb, kb, vb, dob = (orc.reorder(data[x], g).astype(np.float64) for x in ("q", "k", "v", "do"))
    S = orc.scores_mean(qb, kb, g.Bt).astype(np.float32).reshape(-1, g.nb)
    sel = orc.select(S, 0.7, 1)
    return g, qb, kb, vb, dob, sel


def test_backward_matches_central_differences_everywhere():
    g, qb, kb, vb, dob, sel = _micro_case()
    assert 0 < len(sel.col_idx) < g.B * g.H * g.nb * g.nb       # genuinely sparse
    scale = 1 / math.sqrt(g.d)

    def loss(q, k, v):
        O, _ = orc.attn_fwd(q, k, v, sel.row_ptr, sel.col_idx, g.Bt, scale)
        return float((dob * O).sum())

    dQ, dK, dV = orc.attn_bwd(qb, kb, vb, dob, sel.row_ptr, sel.col_idx, g.Bt, scale)
    h = 1e-6
    for name, X, G in (("q", qb, dQ), ("k", kb, dK), ("v", vb, dV)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            xp = X.copy(); xp[idx] += h
            xm = X.copy(); xm[idx] -= h
            args = {"q": qb, "k": kb, "v": vb}
            args[name] = xp
            fp = loss(args["q"], args["k"], args["v"])
            args[name] = xm
            fm = loss(args["q"], args["k"], args["v"])
            num[idx] = (fp - fm) / (2 * h)
        np.testing.assert_allclose(G, num, rtol=1e-6, atol=1e-8, err_msg=name)


def test_backward_matches_autograd_of_masked_dense_and_sampling():
    wl, g, data, qb, kb, vb = _tiny()
    rng = np.random.default_rng(21)
    dob = rng.standard_normal(qb.shape)
    S = orc.scores_mean(qb, kb, g.Bt).astype(np.float32).reshape(-1, g.nb)
    sel = orc.select(S, wl.top_p, wl.k_floor)
    scale = 1 / math.sqrt(g.d)
    dQ, dK, dV = orc.attn_bwd(qb, kb, vb, dob, sel.row_ptr, sel.col_idx, g.Bt, scale)
    M = torch.from_numpy(orc.token_mask(sel.row_ptr, sel.col_idx, g.B, g.H, g.nb, g.Bt))
    q, k, v = (torch.tensor(x.astype(np.float64), requires_grad=True) for x in (qb, kb, vb))
    s = scale * q @ k.transpose(-1, -2)
    s = s.masked_fill(~M, float("-inf"))
    O = torch.softmax(s, dim=-1) @ v
    (O * torch.from_numpy(dob)).sum().backward()
    np.testing.assert_allclose(dQ, q.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dK, k.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dV, v.grad.numpy(), rtol=1e-9, atol=1e-11)
    # restricting to a few blocks gives the same entries
    qs = [(0, 1, 3), (0, 0, 15)]
    ks = [(0, 0, 2), (0, 1, 9)]
    sQ, sK, sV = orc.attn_bwd(qb, kb, vb, dob, sel.row_ptr, sel.col_idx, g.Bt, scale, q_blocks=qs, k_blocks=ks)
    for (b, h, i) in qs:
        sl = slice(i * g.Bt, (i + 1) * g.Bt)
        np.testing.assert_allclose(sQ[b, h, sl], dQ[b, h, sl], rtol=1e-12, atol=1e-14)
    for (b, h, j) in ks:
        sl = slice(j * g.Bt, (j + 1) * g.Bt)
        np.testing.assert_allclose(sK[b, h, sl], dK[b, h, sl], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(sV[b, h, sl], dV[b, h, sl], rtol=1e-12, atol=1e-14)


# ----------------------------------------------------------------- schedule, CSC

def test_lpt_order_properties():
    rng = np.random.default_rng(4)
    B, H, nb = 2, 3, 10
    counts = rng.integers(1, nb + 1, size=B * H * nb)
    rp = np.concatenate([[0], np.cumsum(counts)])
    for grouped in (True, False):
        order = orc.lpt_order(rp, B, H, nb, grouped)
        assert sorted(order.tolist()) == list(range(B * H * nb))
        c = counts[order]
        if not grouped:
            assert (np.diff(c) <= 0).all()
            # equal costs stay in item order
            for a, b2 in zip(order[:-1], order[1:]):
                if counts[a] == counts[b2]:
                    assert a < b2
        else:
            heads = order // nb
            # each head is one contiguous run, heads by total cost descending
            runs = [heads[0]] + [y for x, y in zip(heads[:-1], heads[1:]) if x != y]
            assert len(runs) == B * H
            tot = [counts[h * nb:(h + 1) * nb].sum() for h in runs]
            assert all(x >= y for x, y in zip(tot[:-1], tot[1:]))
            for h in range(B * H):
                assert (np.diff(counts[order[heads == h]]) <= 0).all()


def test_csc_is_transpose():
    wl, g, data, qb, kb, vb = _tiny()
    S = orc.scores_mean(qb, kb, g.Bt).astype(np.float32).reshape(-1, g.nb)
    sel = orc.select(S, wl.top_p, wl.k_floor)
    cp, ri = orc.csc_of(sel.row_ptr, sel.col_idx, g.B, g.H, g.nb)
    M = orc.token_mask(sel.row_ptr, sel.col_idx, g.B, g.H, g.nb, g.Bt)[:, :, ::g.Bt, ::g.Bt]
    for h in range(g.H):
        for j in range(g.nb):
            c = h * g.nb + j
            assert ri[cp[c]:cp[c + 1]].tolist() == np.nonzero(M[0, h, :, j])[0].tolist()


# ----------------------------------------------------------------- placement

def _csr(rows):
    rp = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int64)
    return rp, np.concatenate([np.asarray(r, dtype=np.int64) for r in rows])


def test_placement_hand_example():
    gold = _load("placement_hand.json")
    rp, ci = _csr(gold["rows"])
    owner = orc.placement(rp, ci, gold["B"], gold["H"], gold["nb"], gold["P"])
    assert owner[0].tolist() == gold["owner"]
    dem = orc.kv_demand(rp, ci, 1, 1, gold["nb"], gold["P"], 1, 1, 1, owner=owner)
    assert int(dem.bytes[2]) == gold["remote_blocks_placed"] * 2      # tile bytes 1*1*1, K and V


def test_placement_separates_independent_groups():
    # two groups of blocks that only select each other: an optimal placement
    # puts each group on one partition and ships nothing
    nb, groups = 8, [[0, 1, 4, 5], [2, 3, 6, 7]]
    rows = [sorted(next(g for g in groups if i in g)) for i in range(nb)]
    rp, ci = _csr(rows * 2)                         # two heads with the same pattern
    owner = orc.placement(rp, ci, 1, 2, nb, 2)
    for g in groups:
        assert len({int(owner[0, i]) for i in g}) == 1
    placed = orc.kv_demand(rp, ci, 1, 2, nb, 2, 1, 1, 1, owner=owner)
    contiguous = orc.kv_demand(rp, ci, 1, 2, nb, 2, 1, 1, 1)
    assert int(placed.bytes[2]) == 0 < int(contiguous.bytes[2])
    assert int(placed.bytes[3]) == int(contiguous.bytes[3])


def test_placement_is_a_balanced_assignment_and_contiguous_owner_is_the_default():
    wl, g, data, qb, kb, vb = _tiny()
    S = orc.scores_mean(qb, kb, g.Bt).astype(np.float32).reshape(-1, g.nb)
    sel = orc.select(S, wl.top_p, wl.k_floor)
    for P in (1, 2, 3, 16):
        owner = orc.placement(sel.row_ptr, sel.col_idx, g.B, g.H, g.nb, P)
        counts = np.bincount(owner[0], minlength=P)
        assert counts.tolist() == [hi - lo for (lo, hi) in orc.partition_bounds(g.nb, P)]
    contiguous = np.zeros((1, g.nb), np.int32)
    for r, (lo, hi) in enumerate(orc.partition_bounds(g.nb, 4)):
        contiguous[0, lo:hi] = r
    a = orc.kv_demand(sel.row_ptr, sel.col_idx, g.B, g.H, g.nb, 4, g.Bt, g.d, 4, kb, vb)
    b = orc.kv_demand(sel.row_ptr, sel.col_idx, g.B, g.H, g.nb, 4, g.Bt, g.d, 4, kb, vb, owner=contiguous)
    assert np.array_equal(a.bitmap, b.bitmap) and np.array_equal(a.dem_idx, b.dem_idx)
    assert a.bytes.tolist() == b.bytes.tolist() and np.array_equal(a.kg, b.kg)


# ------------------------------------------- load balancing and augmentation

def test_balance_hand_example():
    gold = _load("balance_hand.json")
    costs = np.array([gold["costs"]], dtype=np.int64)
    P = gold["P"]
    hr0, mv0 = orc.balance_heads(costs, P, 0)
    assert orc.rank_loads(costs[0], hr0[0], P).tolist() == gold["contiguous_loads"] and mv0[0] == 0
    hr, mv = orc.balance_heads(costs, P, 10)
    assert hr[0].tolist() == gold["head_rank"] and int(mv[0]) == gold["migrations"]
    assert orc.rank_loads(costs[0], hr[0], P).tolist() == gold["loads"]
    hr1, _ = orc.balance_heads(costs, P, 1)
    assert hr1[0].tolist() == gold["head_rank_one_move"]
    assert orc.imbalance(gold["contiguous_loads"]) == gold["imbalance_before"]
    assert orc.imbalance(gold["loads"]) == gold["imbalance_after"]


def test_balance_invariants_and_stopping_rule():
    rng = np.random.default_rng(7)
    for trial in range(40):
        H = int(rng.integers(2, 13))
        P = int(rng.integers(1, H + 1))
        costs = rng.integers(0, 50, size=(2, H)) ** 2         # heavy-tailed head costs
        hr0, _ = orc.balance_heads(costs, P, 0)
        hr, mv = orc.balance_heads(costs, P, H * P * 4)
        for b in range(2):
            before = orc.rank_loads(costs[b], hr0[b], P)
            after = orc.rank_loads(costs[b], hr[b], P)
            assert after.sum() == costs[b].sum()               # work is conserved
            assert after.max() <= before.max()                 # never worse than the contiguous split
            assert set(hr[b].tolist()) <= set(range(P))
            # stopped because no head of the critical rank improves the pair
            c, t = int(np.argmax(after)), int(np.argmin(after))
            for h in range(H):
                if hr[b, h] == c:
                    assert max(after[c] - costs[b, h], after[t] + costs[b, h]) >= after[c]
    # equal costs and H divisible by P: already balanced, nothing moves
    hr, mv = orc.balance_heads(np.full((1, 12), 5), 4, 100)
    assert mv[0] == 0 and orc.imbalance(orc.rank_loads(np.full(12, 5), hr[0], 4)) == 1.0


def test_block_values_are_the_row_softmax():
    from scipy.special import softmax
    rng = np.random.default_rng(8)
    S = (rng.standard_normal((20, 37)) * 3).astype(np.float32)
    V = orc.block_values(S)
    ref = softmax(S.astype(np.float64), axis=1)
    np.testing.assert_allclose(V, ref, rtol=2e-6, atol=0)
    assert np.abs(V.astype(np.float64).sum(axis=1) - 1).max() < 1e-5


def test_augment_hand_example():
    gold = _load("augment_hand.json")
    rp, ci = _csr(gold["rows"])
    S = np.array(gold["scores"], dtype=np.float32)
    aug = orc.augment(S, rp, ci, gold["B"], gold["H"], gold["nb"], np.array([gold["head_rank"]]), gold["P"])
    rows = [aug.col_idx[aug.row_ptr[r]:aug.row_ptr[r + 1]].tolist() for r in range(len(gold["rows"]))]
    assert rows == gold["augmented_rows"]
    assert aug.added[0].tolist() == gold["added"] and aug.loads[0].tolist() == gold["loads"]
    np.testing.assert_allclose(aug.cut[0], gold["cut"], rtol=1e-6)
    np.testing.assert_allclose(aug.next_value[0], gold["next_value"], rtol=1e-6)


def test_augment_fills_slack_with_the_best_blocks():
    from scipy.special import softmax
    wl, g, data, qb, kb, vb = _tiny()
    S = orc.scores_mean(qb, kb, g.Bt).astype(np.float32).reshape(-1, g.nb)
    # a lopsided selection: head 0 keeps 3 blocks per row, head 1 one block
    rows = []
    for h in range(g.H):
        for i in range(g.nb):
            order = np.argsort(-S[h * g.nb + i], kind="stable")
            rows.append(sorted(order[:3 if h == 0 else 1].tolist()))
    rp, ci = _csr(rows)
    hr, _ = orc.balance_heads(orc.head_costs(rp, 1, g.H, g.nb), 2, 0)
    aug = orc.augment(S, rp, ci, 1, g.H, g.nb, hr, 2)
    V = softmax(S.astype(np.float64), axis=1)
    top = 3 * g.nb
    assert aug.loads[0].tolist() == [top, top] and aug.added[0].tolist() == [0, 2 * g.nb]
    added, left = [], []
    for i in range(g.nb):
        r = g.nb + i
        new = set(aug.col_idx[aug.row_ptr[r]:aug.row_ptr[r + 1]].tolist())
        assert set(rows[r]) <= new                              # nothing is dropped
        added += [V[r, j] for j in new - set(rows[r])]
        left += [V[r, j] for j in range(g.nb) if j not in new]
        assert sorted(new) == list(aug.col_idx[aug.row_ptr[r]:aug.row_ptr[r + 1]])
    assert min(added) >= max(left) * (1 - 1e-6)                 # the best candidates were taken
    for r in range(g.nb):                                        # the critical head is untouched
        assert aug.col_idx[aug.row_ptr[r]:aug.row_ptr[r + 1]].tolist() == rows[r]


def test_augment_without_slack_changes_nothing():
    rows = [[0, 1], [1], [0], [0, 1]]          # two heads of 2 blocks, 3 pairs each
    rp, ci = _csr(rows)
    S = np.zeros((4, 2), dtype=np.float32)
    aug = orc.augment(S, rp, ci, 1, 2, 2, np.array([[0, 1]]), 2)
    assert aug.added.sum() == 0
    assert aug.row_ptr.tolist() == rp.tolist() and aug.col_idx.tolist() == ci.tolist()


# --------------------------------------------------------- predictor fitting

def test_predictor_hand_example():
    gold = _load("predictor_hand.json")
    qm = np.full((1, 1, 1, 1), gold["qm"])
    km = np.full((1, 1, 1, 1), gold["km"])
    wq = np.full((1, 1, 1), gold["wq"])
    wk = np.full((1, 1, 1), gold["wk"])
    loss, gwq, gwk = orc.predictor_loss_grad(qm, km, wq, wk)
    assert loss[0] == gold["loss"] and gwq.item() == gold["gwq"] and gwk.item() == gold["gwk"]
    wq2, wk2, _ = orc.predictor_step(qm, km, wq, wk, gold["lr"])
    assert abs(wq2.item() - gold["wq_next"]) < 1e-12 and abs(wk2.item() - gold["wk_next"]) < 1e-12


def test_predictor_gradient_matches_central_differences():
    rng = np.random.default_rng(11)
    B, H, nb, d, r = 2, 2, 5, 6, 3
    qm, km = rng.standard_normal((2, B, H, nb, d))
    wq, wk = rng.standard_normal((2, H, d, r)) * 0.5
    _, gwq, gwk = orc.predictor_loss_grad(qm, km, wq, wk)
    eps = 1e-6
    for W, G, which in ((wq, gwq, 0), (wk, gwk, 1)):
        for idx in np.ndindex(W.shape):
            Wp, Wm = W.copy(), W.copy()
            Wp[idx] += eps
            Wm[idx] -= eps
            args_p = (qm, km, Wp, wk) if which == 0 else (qm, km, wq, Wp)
            args_m = (qm, km, Wm, wk) if which == 0 else (qm, km, wq, Wm)
            num = (orc.predictor_loss_grad(*args_p)[0] - orc.predictor_loss_grad(*args_m)[0]) / (2 * eps)
            h = idx[0]
            assert abs(num[h] - G[idx]) <= 1e-6 * max(1.0, abs(G[idx])), (which, idx, num[h], G[idx])
            other = [x for x in range(H) if x != h]
            assert np.all(np.abs(num[other]) < 1e-9)            # a head's weights touch only its loss


def test_predictor_exact_fit_has_zero_loss():
    # r = d with Wk = Wq^{-T}: (q Wq)(k Wk)^T = q k^T exactly, so loss and gradients vanish
    rng = np.random.default_rng(12)
    B, H, nb, d = 2, 3, 4, 5
    qm, km = rng.standard_normal((2, B, H, nb, d))
    wq = rng.standard_normal((H, d, d)) + 3 * np.eye(d)
    wk = np.stack([np.linalg.inv(w).T for w in wq])
    loss, gwq, gwk = orc.predictor_loss_grad(qm, km, wq, wk)
    assert np.abs(loss).max() < 1e-18 and np.abs(gwq).max() < 1e-9 and np.abs(gwk).max() < 1e-9


def test_predictor_steps_descend():
    rng = np.random.default_rng(13)
    B, H, nb, d, r = 1, 2, 8, 16, 4
    qm, km = rng.standard_normal((2, B, H, nb, d)) * 0.5
    wq, wk = rng.standard_normal((2, H, d, r)) * 0.3
    losses = []
    for _ in range(20):
        wq, wk, loss = orc.predictor_step(qm, km, wq, wk, 0.01)
        losses.append(loss)
    losses = np.array(losses)
    assert np.all(np.diff(losses, axis=0) < 0)                   # every step lowers every head's loss
    assert np.all(losses[-1] < 0.9 * losses[0])
