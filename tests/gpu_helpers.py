"""Shared pieces of the GPU parity tests: workload caching, device transfer,
oracle chains and the comparison rules.

Expected values always come from the oracle run on the generator's inputs
(never from the CUDA path). The two paths meet only at the inputs.
"""
from __future__ import annotations

import functools
import math

import numpy as np
import torch

import block_sparse_attention_token_gb300 as sp
import synth
from oracle import sparsp_oracle as orc

BF16_MAX_ABS, BF16_MEAN_ABS = 1e-2, 1e-3
F32_TOL = 1e-4


@functools.lru_cache(maxsize=8)
def workload(name: str):
    wl = synth.WORKLOADS[name] if isinstance(name, str) and name in synth.WORKLOADS else name
    return wl, synth.make(wl)


def dev(x: np.ndarray, wl) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return t.bfloat16() if wl.dtype == "bf16" else t.float()


def i32(x) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(np.asarray(x, dtype=np.int32))).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy() if t.dtype in (torch.bfloat16, torch.float16) else t.cpu().numpy()


def status_word() -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device="cuda")


class OracleChain:
    """The oracle's own forward chain on a workload's inputs (blocked tensors,
    fp32-rounded scores, CSR)."""

    def __init__(self, wl, data, blocked: bool = True):
        self.wl, self.g = wl, orc.grid_of(wl)
        g = self.g
        self.qb, self.kb, self.vb = (orc.reorder(data[x], g) for x in ("q", "k", "v"))
        if wl.estimator == "lowrank":
            S = orc.scores_lowrank(self.qb, self.kb, data["wq"], data["wk"], g.Bt)
        else:
            S = orc.scores_mean(self.qb, self.kb, g.Bt)
        self.S64 = S
        self.S32 = S.astype(np.float32)
        self.sel = orc.select(self.S32.reshape(-1, g.nb), wl.top_p, wl.k_floor)
        self.scale = 1.0 / math.sqrt(g.d)


def compare_values(got: np.ndarray, ref: np.ndarray, wl, what: str):
    """Attention values: bf16 max-abs 1e-2 and mean-abs 1e-3; fp32 max-abs 1e-4."""
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got.astype(np.float64) - ref)
    if wl.dtype == "bf16":
        assert err.max() <= BF16_MAX_ABS, f"{what}: max-abs {err.max():.3e}"
        assert err.mean() <= BF16_MEAN_ABS, f"{what}: mean-abs {err.mean():.3e}"
    else:
        assert err.max() <= F32_TOL, f"{what}: max-abs {err.max():.3e}"
    return float(err.max()), float(err.mean())


def bf16_floor(ref: np.ndarray) -> tuple[float, float]:
    """Max and mean absolute error of the oracle's own values rounded to bf16:
    the error a bf16 output cannot avoid."""
    r32 = np.ascontiguousarray(ref, dtype=np.float32)
    err = np.abs(synth.round_bf16(r32.copy()).astype(np.float64) - ref)
    return float(err.max()), float(err.mean())


def compare_csr(row_ptr: np.ndarray, col_idx: np.ndarray, sel: orc.Selection) -> int:
    """Bit-exact CSR, except rows the oracle flags as within its ambiguity band
    of the Top-p threshold (1e-12 of the row's mass: float64 summation order),
    where any count in the admissible range (and the corresponding prefix of
    the score order) is accepted. Returns the number of such rows whose count
    differed from the oracle's first choice."""
    R = len(sel.row_ptr) - 1
    assert row_ptr.shape == (R + 1,)
    if np.array_equal(row_ptr, sel.row_ptr) and np.array_equal(col_idx[:row_ptr[-1]], sel.col_idx):
        return 0
    n_alt = 0
    for r in range(R):
        got = col_idx[row_ptr[r]:row_ptr[r + 1]]
        want = sel.col_idx[sel.row_ptr[r]:sel.row_ptr[r + 1]]
        if np.array_equal(got, want):
            continue
        m = len(got)
        assert sel.m_lo[r] <= m <= sel.m_hi[r], f"row {r}: count {m} vs oracle {len(want)} (margin {sel.margin[r]:.2e})"
        assert np.array_equal(got, np.sort(sel.order[r][:m])), f"row {r}: wrong block set"
        n_alt += 1
    return n_alt


def jaccard_rows(rp_a, ci_a, rp_b, ci_b) -> float:
    """Mean per-row Jaccard similarity of two CSRs' block sets."""
    R = len(rp_a) - 1
    tot = 0.0
    for r in range(R):
        a = set(ci_a[rp_a[r]:rp_a[r + 1]].tolist())
        b = set(ci_b[rp_b[r]:rp_b[r + 1]].tolist())
        u = len(a | b)
        tot += 1.0 if u == 0 else len(a & b) / u
    return tot / R


def compare_augmented(rp, ci, ref: orc.Augmented, rp0, ci0, V, head_rank, B, H, nb, P, rel=1e-6) -> int:
    """The GPU's augmented CSR against the oracle's. Per rank, the number of
    added blocks is exact; every row keeps its selected blocks; every added
    block is worth at least the oracle's cut and every candidate left out at
    most the cut (both within `rel`, the float32 rounding of the values).
    Where no candidate value lies strictly inside that band around a cut, the
    whole CSR must equal the oracle's bit for bit. Returns the number of rows
    that differ from the oracle."""
    R = B * H * nb
    assert rp.shape == (R + 1,)
    diff_rows = 0
    band_empty = True
    for b in range(B):
        for r in range(P):
            cut = float(ref.cut[b, r])
            n_add = 0
            for h in range(H):
                if int(head_rank[b, h]) != r:
                    continue
                for i in range(nb):
                    row = (b * H + h) * nb + i
                    old = set(int(j) for j in ci0[rp0[row]:rp0[row + 1]])
                    new_list = [int(j) for j in ci[rp[row]:rp[row + 1]]]
                    assert new_list == sorted(set(new_list)), f"row {row} not ascending/unique"
                    new = set(new_list)
                    assert old <= new, f"row {row} lost selected blocks"
                    ref_new = set(int(j) for j in ref.col_idx[ref.row_ptr[row]:ref.row_ptr[row + 1]])
                    diff_rows += new != ref_new
                    for j in new - old:
                        assert V[row, j] >= cut * (1 - rel), (row, j, V[row, j], cut)
                    for j in range(nb):
                        if j not in new:
                            assert j in old or V[row, j] <= cut * (1 + rel) or ref.added[b, r] == 0, \
                                (row, j, V[row, j], cut)
                        if j not in old and V[row, j] != cut and abs(V[row, j] - cut) <= cut * rel:
                            band_empty = False
                    n_add += len(new - old)
            assert n_add == int(ref.added[b, r]), (b, r, n_add, int(ref.added[b, r]))
    if band_empty:
        assert np.array_equal(rp, ref.row_ptr) and np.array_equal(ci[:rp[-1]], ref.col_idx)
    return diff_rows
