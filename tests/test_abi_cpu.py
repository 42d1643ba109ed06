"""libsparsp loads, exports every symbol its header declares, and rejects bad
arguments on the host before touching CUDA (no GPU needed: every call here
fails validation, so nothing is launched)."""
import ctypes
import os
import re
import subprocess

import pytest

import block_sparse_attention_token_gb300 as sp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    from block_sparse_attention_token_gb300 import build
    build.build()
    return sp.lib()


def declared_symbols():
    text = "".join(open(h).read() for h in HEADERS)
    return sorted(set(re.findall(r"SPARSP_API\s+[\w\s\*]+?\b(sparsp_\w+)\s*\(", text)))


def test_header_declares_the_six_calls():
    names = declared_symbols()
    for call in ("sparsp_reorder", "sparsp_block_scores", "sparsp_select", "sparsp_kv_demand",
                 "sparsp_attn_fwd", "sparsp_attn_bwd"):
        assert call in names


def test_every_declared_symbol_is_exported(lib):
    exported = subprocess.run(["nm", "-D", "--defined-only", sp.LIB_PATH], capture_output=True,
                              text=True, check=True).stdout
    names = set(re.findall(r"\s(sparsp_\w+)$", exported, flags=re.M))
    missing = [n for n in declared_symbols() if n not in names]
    assert not missing, missing
    # the binding wires every declared call
    assert set(declared_symbols()) <= set(sp._SIG)
    # nothing else leaks out of the library
    assert all(n.startswith("sparsp_") for n in names)


def test_version_and_status_strings(lib):
    assert lib.sparsp_version() == 1
    assert sp.status_string(0) == "SPARSP_OK"
    assert sp.status_string(7) == "SPARSP_ERR_DATA"
    assert sp.status_string(99) == "SPARSP_ERR_UNKNOWN"


GOOD = dict(B=1, H=2, T=4, Y=16, X=16, d=64, ta=4, tb=4, tc=4, dtype=sp.BF16)
FAKE = 1 << 20          # an aligned, never-dereferenced address


def shape(**kw):
    args = dict(GOOD)
    args.update(kw)
    return sp.make_shape(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(T=5), sp.SHAPE),              # grid not divisible by tile
    (dict(B=0), sp.SHAPE),
    (dict(d=96), sp.UNSUPPORTED),
    (dict(ta=2), sp.UNSUPPORTED),       # Bt = 32
    (dict(dtype=7), sp.UNSUPPORTED),
    (dict(T=128, Y=64, X=64), sp.UNSUPPORTED),  # nb = 8192 > 4096
    (dict(H=128, T=64, Y=64, X=64), sp.UNSUPPORTED),   # B*H*nb^2 = 128 * 4096^2 >= 2^31
])
def test_shape_validation(lib, kw, code):
    s = shape(**kw)
    assert lib.sparsp_reorder(ctypes.byref(s), FAKE, FAKE * 2, 0, None) == code


def test_null_and_misaligned_pointers(lib):
    s = shape()
    assert lib.sparsp_reorder(None, FAKE, FAKE * 2, 0, None) == sp.INVALID_ARG
    assert lib.sparsp_reorder(ctypes.byref(s), None, FAKE, 0, None) == sp.INVALID_ARG
    assert lib.sparsp_reorder(ctypes.byref(s), FAKE + 8, FAKE * 2, 0, None) == sp.ALIGN
    # overlapping in/out
    assert lib.sparsp_reorder(ctypes.byref(s), FAKE, FAKE + 4096, 0, None) == sp.INVALID_ARG


def test_workspace_sizes(lib):
    s = shape()
    rows = s.B * s.H * s.nb
    assert lib.sparsp_select_workspace_size(ctypes.byref(s)) == rows * 8
    assert lib.sparsp_block_scores_workspace_size(ctypes.byref(s), sp.EST_MEAN, 16) == 2 * rows * s.d * 4
    assert lib.sparsp_block_scores_workspace_size(ctypes.byref(s), sp.EST_LOWRANK, 16) == 2 * rows * 16 * 4
    assert lib.sparsp_lpt_workspace_size(ctypes.byref(s)) == s.B * s.H * (2 * s.nb + 1) * 4
    fwd = lib.sparsp_attn_workspace_size(ctypes.byref(s), 0)
    bwd = lib.sparsp_attn_workspace_size(ctypes.byref(s), 1)
    assert fwd >= rows * 4 + 16 and bwd > fwd + s.B * s.H * s.N * 4
    bad = shape(T=5)
    assert lib.sparsp_attn_workspace_size(ctypes.byref(bad), 0) == 0


def test_call_validation_codes(lib):
    s = shape()
    S = ctypes.byref(s)
    f = ctypes.c_float
    # select: NaN p, negative floor, small workspace
    assert lib.sparsp_select(S, FAKE, f(float("nan")), 1, FAKE, FAKE, FAKE, 1 << 30, None, None) == sp.INVALID_ARG
    assert lib.sparsp_select(S, FAKE, f(0.9), -1, FAKE, FAKE, FAKE, 1 << 30, None, None) == sp.INVALID_ARG
    assert lib.sparsp_select(S, FAKE, f(0.9), 1, FAKE, FAKE, FAKE, 8, None, None) == sp.WORKSPACE
    # scores: bad estimator, low-rank without weights, rank out of range, small workspace
    assert lib.sparsp_block_scores(S, 5, FAKE, FAKE, None, None, 16, FAKE, FAKE, 1 << 30, None) == sp.INVALID_ARG
    assert lib.sparsp_block_scores(S, sp.EST_LOWRANK, FAKE, FAKE, None, FAKE, 16, FAKE, FAKE, 1 << 30,
                                   None) == sp.INVALID_ARG
    assert lib.sparsp_block_scores(S, sp.EST_LOWRANK, FAKE, FAKE, FAKE, FAKE, 65, FAKE, FAKE, 1 << 30,
                                   None) == sp.UNSUPPORTED
    assert lib.sparsp_block_scores(S, sp.EST_MEAN, FAKE, FAKE, None, None, 16, FAKE, FAKE, 4, None) == sp.WORKSPACE
    # demand: P out of range, kg without vg, negative capacity
    args = (FAKE, FAKE, None, FAKE, FAKE, FAKE)
    assert lib.sparsp_kv_demand(S, 0, *args, None, None, None, None, 0, FAKE, None, None) == sp.SHAPE
    assert lib.sparsp_kv_demand(S, s.nb + 1, *args, None, None, None, None, 0, FAKE, None, None) == sp.SHAPE
    assert lib.sparsp_kv_demand(S, 2, *args, FAKE, FAKE, FAKE, None, 4, FAKE, None, None) == sp.INVALID_ARG
    assert lib.sparsp_kv_demand(S, 2, *args, FAKE, FAKE, FAKE, FAKE, -1, FAKE, None, None) == sp.INVALID_ARG
    assert lib.sparsp_kv_demand(S, 2, FAKE, FAKE, FAKE + 4, FAKE, FAKE, FAKE, None, None, None, None, 0, FAKE,
                                None, None) == sp.ALIGN
    # gather alone: P out of range, a missing buffer, negative capacity, misaligned list
    g = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)
    assert lib.sparsp_kv_gather(S, 0, *g, 4, None, None) == sp.SHAPE
    assert lib.sparsp_kv_gather(S, s.nb + 1, *g, 4, None, None) == sp.SHAPE
    assert lib.sparsp_kv_gather(S, 2, FAKE, FAKE, FAKE, FAKE, FAKE, None, 4, None, None) == sp.INVALID_ARG
    assert lib.sparsp_kv_gather(S, 2, None, FAKE, FAKE, FAKE, FAKE, FAKE, 4, None, None) == sp.INVALID_ARG
    assert lib.sparsp_kv_gather(S, 2, *g, -1, None, None) == sp.INVALID_ARG
    assert lib.sparsp_kv_gather(S, 2, FAKE, FAKE + 4, FAKE, FAKE, FAKE, FAKE, 4, None, None) == sp.ALIGN
    # the same checks for the gather from raster K and V
    assert lib.sparsp_kv_gather_raster(S, 0, *g, 4, None, None) == sp.SHAPE
    assert lib.sparsp_kv_gather_raster(S, 2, FAKE, FAKE, FAKE, FAKE, FAKE, None, 4, None, None) == sp.INVALID_ARG
    assert lib.sparsp_kv_gather_raster(S, 2, *g, -1, None, None) == sp.INVALID_ARG
    assert lib.sparsp_kv_gather_raster(S, 2, FAKE, FAKE, FAKE + 4, FAKE, FAKE, FAKE, 4, None, None) == sp.ALIGN
    # pooling: the reordered copy is optional, the means are not; a copy over its input is refused
    assert lib.sparsp_reorder_pool(S, FAKE, FAKE, None, None) == sp.INVALID_ARG
    assert lib.sparsp_reorder_pool(S, FAKE, FAKE, FAKE, None) == sp.INVALID_ARG
    # placement: P out of range, missing owner, small workspace
    need = lib.sparsp_placement_workspace_size(S)
    assert need == s.B * s.nb * s.nb * 4
    assert lib.sparsp_placement(S, 0, FAKE, FAKE, FAKE, FAKE, need, None, None) == sp.SHAPE
    assert lib.sparsp_placement(S, s.nb + 1, FAKE, FAKE, FAKE, FAKE, need, None, None) == sp.SHAPE
    assert lib.sparsp_placement(S, 2, FAKE, FAKE, None, FAKE, need, None, None) == sp.INVALID_ARG
    assert lib.sparsp_placement(S, 2, FAKE, FAKE, FAKE, FAKE, need - 1, None, None) == sp.WORKSPACE
    # balancing: P out of range, negative migrations, too many heads
    assert lib.sparsp_balance_heads(S, 0, 1, FAKE, FAKE, FAKE, None, None) == sp.SHAPE
    assert lib.sparsp_balance_heads(S, s.H + 1, 1, FAKE, FAKE, FAKE, None, None) == sp.SHAPE
    assert lib.sparsp_balance_heads(S, 1, -1, FAKE, FAKE, FAKE, None, None) == sp.INVALID_ARG
    big = ctypes.byref(shape(H=4096))
    assert lib.sparsp_balance_heads(big, 2, 1, FAKE, FAKE, FAKE, None, None) == sp.UNSUPPORTED
    # augmentation: small workspace, negative capacity, missing head ranks
    need = lib.sparsp_augment_workspace_size(S, 2)
    assert need >= s.B * s.H * s.nb * s.nb * 4
    assert lib.sparsp_augment(S, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, None, FAKE, need - 1, None,
                              None) == sp.WORKSPACE
    assert lib.sparsp_augment(S, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, -1, None, FAKE, need, None,
                              None) == sp.INVALID_ARG
    assert lib.sparsp_augment(S, 2, FAKE, FAKE, FAKE, None, FAKE, FAKE, 16, None, FAKE, need, None,
                              None) == sp.INVALID_ARG
    # predictor fitting: rank out of range, NaN step, small workspace
    needp = lib.sparsp_predictor_workspace_size(S, 16)
    assert needp > 0 and lib.sparsp_predictor_workspace_size(S, 65) == 0
    assert lib.sparsp_predictor_fit(S, 65, FAKE, FAKE, FAKE, FAKE, f(0.0), None, None, None, FAKE, needp,
                                    None) == sp.UNSUPPORTED
    assert lib.sparsp_predictor_fit(S, 16, FAKE, FAKE, FAKE, FAKE, f(float("nan")), None, None, None, FAKE,
                                    needp, None) == sp.INVALID_ARG
    assert lib.sparsp_predictor_fit(S, 16, FAKE, FAKE, FAKE, FAKE, f(0.1), None, None, None, FAKE, needp - 1,
                                    None) == sp.WORKSPACE
    # bounded-wait diagnostic: limit out of range, missing status word
    assert lib.sparsp_diag_wait_timeout(10, FAKE, None) == sp.INVALID_ARG
    assert lib.sparsp_diag_wait_timeout(10_000_000_000, FAKE, None) == sp.INVALID_ARG
    assert lib.sparsp_diag_wait_timeout(50_000_000, None, None) == sp.INVALID_ARG
    # tile diagnostic: the status word is required
    assert lib.sparsp_diag_umma_tile(FAKE, FAKE, FAKE, 0, 16, 1024, None, None) == sp.INVALID_ARG
    # attention: NaN scale, small workspace, misaligned optional pointer, fp32 backward
    p7 = (FAKE,) * 5
    assert lib.sparsp_attn_fwd(S, *p7, f(float("nan")), FAKE, FAKE, FAKE, 1 << 30, 0, None, None,
                               None) == sp.INVALID_ARG
    assert lib.sparsp_attn_fwd(S, *p7, f(0.0), FAKE, FAKE, FAKE, 8, 0, None, None, None) == sp.WORKSPACE
    assert lib.sparsp_attn_fwd(S, *p7, f(0.0), FAKE, FAKE, FAKE, 1 << 30, 0, FAKE + 4, None,
                               None) == sp.ALIGN
    s32 = shape(dtype=sp.F32)
    # option bits outside the defined ones are refused by every call that takes options
    assert lib.sparsp_attn_fwd(S, *p7, f(0.0), FAKE, FAKE, FAKE, 1 << 30, 1 << 9, None, None,
                               None) == sp.INVALID_ARG
    assert lib.sparsp_attn_bwd(S, *((FAKE,) * 8), f(0.0), FAKE, FAKE, FAKE, FAKE, 1 << 30, 1 << 9, None, None,
                               None) == sp.INVALID_ARG
    assert lib.sparsp_lpt_schedule(S, FAKE, 1 << 9, FAKE, FAKE, 1 << 30, None) == sp.INVALID_ARG
    assert lib.sparsp_attn_fwd(S, *p7, f(0.0), FAKE, FAKE, FAKE, 1 << 30, 1 << 28, None, None,
                               None) == sp.INVALID_ARG     # above the grid-cap field
    # the grid-cap field itself is accepted (the call then fails on the next check: the workspace)
    assert lib.sparsp_attn_fwd(S, *p7, f(0.0), FAKE, FAKE, FAKE, 8, sp.GRID_CAP(7), None, None,
                               None) == sp.WORKSPACE
    assert lib.sparsp_attn_bwd(S, *((FAKE,) * 8), f(0.0), FAKE, FAKE, FAKE, FAKE, 8, sp.GRID_CAP(4095), None,
                               None, None) == sp.WORKSPACE
    assert sp.GRID_CAP(7) == 7 << 16
    with pytest.raises(ValueError):
        sp.GRID_CAP(0)
    # raster O is written by the tcgen05 kernel only: fp32, or the portable kernel, is refused
    assert lib.sparsp_attn_fwd(ctypes.byref(s32), *p7, f(0.0), FAKE, FAKE, FAKE, 1 << 30, sp.OUT_RASTER, None,
                               None, None) == sp.UNSUPPORTED
    assert lib.sparsp_attn_fwd(S, *p7, f(0.0), FAKE, FAKE, FAKE, 1 << 30, sp.OUT_RASTER | sp.KERNEL_PORTABLE,
                               None, None, None) == sp.UNSUPPORTED
    assert lib.sparsp_attn_bwd(ctypes.byref(s32), *((FAKE,) * 8), f(0.0), FAKE, FAKE, FAKE, FAKE, 1 << 30, 0,
                               None, None, None) == sp.UNSUPPORTED
    # raster inputs: the tcgen05 forward only (no GPU here, so not even that); never the backward
    assert lib.sparsp_attn_fwd(S, *p7, f(0.0), FAKE, FAKE, FAKE, 1 << 30, sp.IN_RASTER | sp.KERNEL_PORTABLE,
                               None, None, None) == sp.UNSUPPORTED
    assert lib.sparsp_attn_bwd(S, *((FAKE,) * 8), f(0.0), FAKE, FAKE, FAKE, FAKE, 1 << 30, sp.IN_RASTER, None,
                               None, None) == sp.UNSUPPORTED
    assert lib.sparsp_attn_bwd(S, *((FAKE,) * 8), f(0.0), FAKE, FAKE, FAKE, FAKE, 8, 0, None, None,
                               None) == sp.WORKSPACE
    assert lib.sparsp_lpt_schedule(S, FAKE, sp.SCHED_FLAT, FAKE, FAKE, 4, None) == sp.WORKSPACE
    assert lib.sparsp_csr_transpose(S, FAKE, None, FAKE, FAKE, None, None) == sp.INVALID_ARG


def test_no_alloc_select_host_checks(lib):
    f = ctypes.c_float
    big = shape(B=1, H=65, T=16, Y=64, X=128, d=128, ta=2, tb=8, tc=8)    # 66,560 rows
    assert lib.sparsp_select_noalloc(ctypes.byref(big), FAKE, f(0.9), 1, FAKE, FAKE, None, None) == sp.WORKSPACE
    s = shape()
    assert lib.sparsp_select_noalloc(ctypes.byref(s), None, f(0.9), 1, FAKE, FAKE, None, None) == sp.INVALID_ARG
    assert lib.sparsp_select_noalloc(ctypes.byref(s), FAKE, f(0.9), -1, FAKE, FAKE, None, None) == sp.INVALID_ARG


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(sp, "_lib", None)
    monkeypatch.setattr(sp, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        sp.lib()


def test_block_limits(lib):
    """nb up to 4,096 is accepted by the hot-path calls (their workspace sizes
    are non-zero); placement and augmentation stop at 1,024 blocks."""
    big = shape(T=64, Y=64, X=64)                       # 4x4x4 tiles: nb = 16*16*16 = 4096
    assert big.nb == 4096
    b = ctypes.byref(big)
    assert lib.sparsp_select_workspace_size(b) == big.rows * 8
    assert lib.sparsp_attn_workspace_size(b, 1) > 0
    assert lib.sparsp_lpt_workspace_size(b) > 0
    assert lib.sparsp_placement_workspace_size(b) == 0
    assert lib.sparsp_augment_workspace_size(b, 2) == 0
    assert lib.sparsp_placement(b, 2, FAKE, FAKE, FAKE, FAKE, 1 << 40, None, None) == sp.UNSUPPORTED
    assert lib.sparsp_augment(b, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, None, FAKE, 1 << 40, None,
                              None) == sp.UNSUPPORTED
    at_limit = shape(T=32, Y=64, X=64)                  # nb = 2048: placement still refused above 1024
    assert lib.sparsp_placement_workspace_size(ctypes.byref(at_limit)) == 0
    small = shape(T=16, Y=64, X=64)                     # nb = 1024
    assert lib.sparsp_placement_workspace_size(ctypes.byref(small)) > 0
