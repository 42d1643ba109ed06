"""Python binding of libsparsp (ctypes): dynamic per-head block-sparse attention
for 3D video-DiT token sequences on one GB300.

Argument marshalling only: every step runs in the library's CUDA kernels.
PyTorch supplies device memory and the current CUDA stream. There is no CPU
fallback: if the library cannot be loaded, every call raises.

Calls mirror the C ABI in include/sparsp.h (same names, without the prefix).
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# SPARSP_DEBUG=1 in the environment selects the debug build (build(debug=True)),
# whose kernels also bounds-check the addresses they derive themselves
DEBUG = os.environ.get("SPARSP_DEBUG") == "1"
LIB_PATH = os.path.join(_PKG, "libsparsp_debug.so" if DEBUG else "libsparsp.so")

OK, INVALID_ARG, UNSUPPORTED, SHAPE, ALIGN, WORKSPACE, CAPACITY, DATA, CUDA, TIMEOUT = range(10)
F32, BF16 = 0, 1
EST_MEAN, EST_LOWRANK = 0, 1
SCHED_FLAT = 1
KERNEL_PORTABLE = 2
BWD_SPLIT_KV = 4
OUT_RASTER = 8
IN_RASTER = 16
GRID_CAP_SHIFT = 16


def GRID_CAP(n: int) -> int:
    """Option bits that cap the attention kernels' persistent grid at n CTAs (1..4095)."""
    if not 1 <= n <= 4095:
        raise ValueError("grid cap must be in [1, 4095]")
    return n << GRID_CAP_SHIFT
PROF_SLOTS = 1024


class SparspError(RuntimeError):
    def __init__(self, call: str, status: int):
        self.status = status
        super().__init__(f"{call} failed: {status_string(status)} ({status})")


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "H", "T", "Y", "X", "d", "ta", "tb", "tc", "dtype")]

    @property
    def N(self):
        return self.T * self.Y * self.X

    @property
    def Bt(self):
        return self.ta * self.tb * self.tc

    @property
    def nb(self):
        return self.N // self.Bt

    @property
    def rows(self):
        return self.B * self.H * self.nb

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == F32 else torch.bfloat16


def make_shape(B, H, T, Y, X, d, ta, tb, tc, dtype) -> Shape:
    if isinstance(dtype, str):
        dtype = F32 if dtype in ("f32", "float32") else BF16
    return Shape(B, H, T, Y, X, d, ta, tb, tc, dtype)


def shape_of(wl) -> Shape:
    """Shape of a workload description with fields B, H, T, Y, X, d, ta, tb, tc, dtype."""
    return make_shape(wl.B, wl.H, wl.T, wl.Y, wl.X, wl.d, wl.ta, wl.tb, wl.tc, wl.dtype)


_lib = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_SIG = {
    "sparsp_status_string": (ctypes.c_char_p, [_I32]),
    "sparsp_version": (_I32, []),
    "sparsp_device_sm_count": (_I32, []),
    "sparsp_reorder": (_I32, [_P, _P, _P, _I32, _P]),
    "sparsp_block_scores_workspace_size": (ctypes.c_size_t, [_P, _I32, _I32]),
    "sparsp_block_scores": (_I32, [_P, _I32, _P, _P, _P, _P, _I32, _P, _P, ctypes.c_size_t, _P]),
    "sparsp_reorder_pool": (_I32, [_P, _P, _P, _P, _P]),
    "sparsp_block_scores_pooled_workspace_size": (ctypes.c_size_t, [_P, _I32, _I32]),
    "sparsp_block_scores_pooled": (_I32, [_P, _I32, _P, _P, _P, _P, _I32, _P, _P, ctypes.c_size_t, _P]),
    "sparsp_select_workspace_size": (ctypes.c_size_t, [_P]),
    "sparsp_select": (_I32, [_P, _P, ctypes.c_float, _I32, _P, _P, _P, ctypes.c_size_t, _P, _P]),
    "sparsp_select_noalloc": (_I32, [_P, _P, ctypes.c_float, _I32, _P, _P, _P, _P]),
    "sparsp_kv_demand": (_I32, [_P, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int64, _P, _P,
                                _P]),
    "sparsp_kv_gather": (_I32, [_P, _I32, _P, _P, _P, _P, _P, _P, ctypes.c_int64, _P, _P]),
    "sparsp_kv_gather_raster": (_I32, [_P, _I32, _P, _P, _P, _P, _P, _P, ctypes.c_int64, _P, _P]),
    "sparsp_placement_workspace_size": (ctypes.c_size_t, [_P]),
    "sparsp_placement": (_I32, [_P, _I32, _P, _P, _P, _P, ctypes.c_size_t, _P, _P]),
    "sparsp_balance_heads": (_I32, [_P, _I32, _I32, _P, _P, _P, _P, _P]),
    "sparsp_augment_workspace_size": (ctypes.c_size_t, [_P, _I32]),
    "sparsp_augment": (_I32, [_P, _I32, _P, _P, _P, _P, _P, _P, ctypes.c_int64, _P, _P, ctypes.c_size_t, _P, _P]),
    "sparsp_predictor_workspace_size": (ctypes.c_size_t, [_P, _I32]),
    "sparsp_predictor_fit": (_I32, [_P, _I32, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "sparsp_lpt_workspace_size": (ctypes.c_size_t, [_P]),
    "sparsp_lpt_schedule": (_I32, [_P, _P, ctypes.c_uint32, _P, _P, ctypes.c_size_t, _P]),
    "sparsp_attn_workspace_size": (ctypes.c_size_t, [_P, _I32]),
    "sparsp_attn_fwd": (_I32, [_P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P, ctypes.c_size_t,
                               ctypes.c_uint32, _P, _P, _P]),
    "sparsp_attn_bwd": (_I32, [_P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P, _P,
                               ctypes.c_size_t, ctypes.c_uint32, _P, _P, _P]),
    "sparsp_csr_transpose": (_I32, [_P, _P, _P, _P, _P, _P, _P]),
    "sparsp_diag_umma_tile": (_I32, [_P, _P, _P, _I32, _I32, _I32, _P, _P]),
    "sparsp_diag_wait_timeout": (_I32, [ctypes.c_uint64, _P, _P]),
}


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{os.path.basename(LIB_PATH)} is not built ({LIB_PATH}); run "
                               f"block_sparse_attention_token_gb300.build.build(debug={DEBUG})")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIG.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib = h
    return _lib


def status_string(st: int) -> str:
    return lib().sparsp_status_string(int(st)).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(name, st):
    if st != OK:
        raise SparspError(name, st)


def _sref(shape: Shape):
    return ctypes.byref(shape)


def _empty(n_bytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(n_bytes), 16), dtype=torch.uint8, device=device)


# ----------------------------------------------------------------- step 1

def reorder(shape: Shape, x: torch.Tensor, out: torch.Tensor | None = None, inverse: bool = False,
            stream=None) -> torch.Tensor:
    """Raster [B,N,H,d] -> blocked [B,H,N,d] (or back with inverse=True)."""
    if out is None:
        dims = (shape.B, shape.N, shape.H, shape.d) if inverse else (shape.B, shape.H, shape.N, shape.d)
        out = torch.empty(dims, dtype=x.dtype, device=x.device)
    _check("sparsp_reorder", lib().sparsp_reorder(_sref(shape), _ptr(x), _ptr(out), int(inverse), _stream(stream)))
    return out


# ----------------------------------------------------------------- step 2

def block_scores_workspace_size(shape, estimator=EST_MEAN, rank=16) -> int:
    return lib().sparsp_block_scores_workspace_size(_sref(shape), estimator, rank)


def block_scores(shape: Shape, q, k, estimator=EST_MEAN, wq=None, wk=None, rank=16, out=None, ws=None,
                 stream=None) -> torch.Tensor:
    if out is None:
        out = torch.empty((shape.B, shape.H, shape.nb, shape.nb), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = _empty(block_scores_workspace_size(shape, estimator, rank), q.device)
    _check("sparsp_block_scores", lib().sparsp_block_scores(
        _sref(shape), estimator, _ptr(q), _ptr(k), _ptr(wq), _ptr(wk), rank, _ptr(out), _ptr(ws),
        ws.numel(), _stream(stream)))
    return out


def reorder_pool(shape: Shape, x: torch.Tensor, out: torch.Tensor | None = None,
                 means: torch.Tensor | None = None, stream=None):
    """Raster -> blocked, plus the fp32 tile means [B, H, nb, d] from the same pass."""
    if out is None:
        out = torch.empty((shape.B, shape.H, shape.N, shape.d), dtype=x.dtype, device=x.device)
    if means is None:
        means = torch.empty((shape.B, shape.H, shape.nb, shape.d), dtype=torch.float32, device=x.device)
    _check("sparsp_reorder_pool", lib().sparsp_reorder_pool(_sref(shape), _ptr(x), _ptr(out), _ptr(means),
                                                            _stream(stream)))
    return out, means


def pool_means(shape: Shape, x: torch.Tensor, means: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The fp32 tile means [B, H, nb, d] of raster x alone (no reordered copy)."""
    if means is None:
        means = torch.empty((shape.B, shape.H, shape.nb, shape.d), dtype=torch.float32, device=x.device)
    _check("sparsp_reorder_pool", lib().sparsp_reorder_pool(_sref(shape), _ptr(x), None, _ptr(means),
                                                            _stream(stream)))
    return means


def block_scores_pooled(shape: Shape, qmeans, kmeans, estimator=EST_MEAN, wq=None, wk=None, rank=16, out=None,
                        ws=None, stream=None) -> torch.Tensor:
    if out is None:
        out = torch.empty((shape.B, shape.H, shape.nb, shape.nb), dtype=torch.float32, device=qmeans.device)
    if ws is None:
        n = lib().sparsp_block_scores_pooled_workspace_size(_sref(shape), estimator, rank)
        ws = _empty(n, qmeans.device)
    _check("sparsp_block_scores_pooled", lib().sparsp_block_scores_pooled(
        _sref(shape), estimator, _ptr(qmeans), _ptr(kmeans), _ptr(wq), _ptr(wk), rank, _ptr(out), _ptr(ws),
        ws.numel(), _stream(stream)))
    return out


# ----------------------------------------------------------------- step 3

def select_workspace_size(shape) -> int:
    return lib().sparsp_select_workspace_size(_sref(shape))


def select(shape: Shape, scores, top_p: float, k_floor: int, row_ptr=None, col_idx=None, ws=None,
           status=None, stream=None):
    """Returns (row_ptr, col_idx); col_idx has capacity B*H*nb*nb, nnz = row_ptr[-1]."""
    dev = scores.device
    if row_ptr is None:
        row_ptr = torch.empty(shape.rows + 1, dtype=torch.int32, device=dev)
    if col_idx is None:
        col_idx = torch.empty(shape.rows * shape.nb, dtype=torch.int32, device=dev)
    if ws is None:
        ws = _empty(select_workspace_size(shape), dev)
    _check("sparsp_select", lib().sparsp_select(
        _sref(shape), _ptr(scores), float(top_p), int(k_floor), _ptr(row_ptr), _ptr(col_idx), _ptr(ws),
        ws.numel(), _ptr(status), _stream(stream)))
    return row_ptr, col_idx


# ----------------------------------------------------------------- step 4

@dataclass
class DemandOut:
    bitmap: torch.Tensor
    dem_ptr: torch.Tensor
    dem_idx: torch.Tensor
    kg: torch.Tensor | None
    vg: torch.Tensor | None
    bytes: torch.Tensor


def kv_demand(shape: Shape, P: int, row_ptr, col_idx, k=None, v=None, gather_cap: int | None = None,
              out: DemandOut | None = None, status=None, stream=None, owner=None) -> DemandOut:
    """KV demand of P partitions: contiguous query-block ranges, or the block
    owner map `owner` [B, nb] int32 (e.g. from `placement`)."""
    dev = row_ptr.device
    if out is None:
        W = (shape.nb + 31) // 32
        parts = shape.B * shape.H * P
        kg = vg = None
        if k is not None:
            cap = parts * shape.nb if gather_cap is None else gather_cap
            kg = torch.empty((max(cap, 1), shape.Bt, shape.d), dtype=k.dtype, device=dev)
            vg = torch.empty_like(kg)
        out = DemandOut(torch.empty((shape.B, shape.H, P, W), dtype=torch.int32, device=dev),
                        torch.empty(parts + 1, dtype=torch.int32, device=dev),
                        torch.empty(parts * shape.nb, dtype=torch.int32, device=dev), kg, vg,
                        torch.empty(4, dtype=torch.int64, device=dev))
    cap = 0 if out.kg is None else (out.kg.shape[0] if gather_cap is None else gather_cap)
    _check("sparsp_kv_demand", lib().sparsp_kv_demand(
        _sref(shape), int(P), _ptr(row_ptr), _ptr(col_idx), _ptr(owner), _ptr(out.bitmap), _ptr(out.dem_ptr),
        _ptr(out.dem_idx), _ptr(k), _ptr(v), _ptr(out.kg), _ptr(out.vg), int(cap), _ptr(out.bytes),
        _ptr(status), _stream(stream)))
    return out


def kv_gather(shape: Shape, P: int, dem: DemandOut, k, v, gather_cap: int | None = None, status=None,
              stream=None, raster: bool = False) -> DemandOut:
    """The gather of kv_demand alone, into dem.kg / dem.vg, from the lists
    (dem.dem_ptr, dem.dem_idx) of an earlier kv_demand call; it can run on a
    second stream beside attention. raster: k and v in raster order [B, N, H, d]."""
    if dem.kg is None or dem.vg is None:
        raise ValueError("kv_gather needs DemandOut with kg and vg buffers")
    cap = dem.kg.shape[0] if gather_cap is None else gather_cap
    name = "sparsp_kv_gather_raster" if raster else "sparsp_kv_gather"
    _check(name, getattr(lib(), name)(
        _sref(shape), int(P), _ptr(dem.dem_ptr), _ptr(dem.dem_idx), _ptr(k), _ptr(v), _ptr(dem.kg), _ptr(dem.vg),
        int(cap), _ptr(status), _stream(stream)))
    return dem


def placement_workspace_size(shape: Shape) -> int:
    return lib().sparsp_placement_workspace_size(_sref(shape))


def placement(shape: Shape, P: int, row_ptr, col_idx, owner=None, ws=None, status=None,
              stream=None) -> torch.Tensor:
    """Block -> partition assignment [B, nb] int32 from the co-selection
    affinity of the CSR (dependency-aware placement)."""
    dev = row_ptr.device
    if owner is None:
        owner = torch.empty((shape.B, shape.nb), dtype=torch.int32, device=dev)
    if ws is None:
        ws = _empty(placement_workspace_size(shape), dev)
    _check("sparsp_placement", lib().sparsp_placement(
        _sref(shape), int(P), _ptr(row_ptr), _ptr(col_idx), _ptr(owner), _ptr(ws), ws.numel(),
        _ptr(status), _stream(stream)))
    return owner


@dataclass
class Balance:
    head_rank: torch.Tensor     # int32 [B, H]
    loads: torch.Tensor         # int64 [B, 2, P]: before, after
    migrations: torch.Tensor    # int32 [B]


def balance_heads(shape: Shape, P: int, row_ptr, max_migrations: int, out: Balance | None = None,
                  stream=None) -> Balance:
    """Heads of each batch element on P virtual ranks: contiguous split, then
    greedy migrations of heavy heads off the critical rank."""
    dev = row_ptr.device
    if out is None:
        out = Balance(torch.empty((shape.B, shape.H), dtype=torch.int32, device=dev),
                      torch.empty((shape.B, 2, P), dtype=torch.int64, device=dev),
                      torch.empty(max(shape.B, 4), dtype=torch.int32, device=dev))
    _check("sparsp_balance_heads", lib().sparsp_balance_heads(
        _sref(shape), int(P), int(max_migrations), _ptr(row_ptr), _ptr(out.head_rank), _ptr(out.loads),
        _ptr(out.migrations), _stream(stream)))
    return out


def augment_workspace_size(shape: Shape, P: int) -> int:
    return lib().sparsp_augment_workspace_size(_sref(shape), int(P))


def augment(shape: Shape, P: int, scores, row_ptr, col_idx, head_rank, row_ptr_out=None, col_idx_out=None,
            added=None, ws=None, status=None, stream=None):
    """Slack-aware augmentation of the CSR: each rank's slack up to the critical
    load is filled with its heads' best unselected blocks. Returns
    (row_ptr_out, col_idx_out, added [B, P])."""
    dev = row_ptr.device
    if row_ptr_out is None:
        row_ptr_out = torch.empty(shape.rows + 1, dtype=torch.int32, device=dev)
    if col_idx_out is None:
        col_idx_out = torch.empty(shape.rows * shape.nb, dtype=torch.int32, device=dev)
    if added is None:
        added = torch.empty((shape.B, P), dtype=torch.int64, device=dev)
    if ws is None:
        ws = _empty(augment_workspace_size(shape, P), dev)
    _check("sparsp_augment", lib().sparsp_augment(
        _sref(shape), int(P), _ptr(scores), _ptr(row_ptr), _ptr(col_idx), _ptr(head_rank), _ptr(row_ptr_out),
        _ptr(col_idx_out), int(col_idx_out.numel()), _ptr(added), _ptr(ws), ws.numel(), _ptr(status),
        _stream(stream)))
    return row_ptr_out, col_idx_out, added


def predictor_fit(shape: Shape, qmeans, kmeans, wq, wk, lr: float = 0.0, rank: int | None = None,
                  loss=None, gwq=None, gwk=None, ws=None, stream=None):
    """Loss and gradients of the low-rank predictor against the real block
    scores (mean squared error per head), and the step W -= lr * grad in place
    when lr != 0. Returns (loss [H], gwq, gwk) at the weights before the step."""
    dev = qmeans.device
    rank = wq.shape[-1] if rank is None else rank
    if loss is None:
        loss = torch.empty(shape.H, dtype=torch.float32, device=dev)
    if gwq is None:
        gwq = torch.empty_like(wq)
    if gwk is None:
        gwk = torch.empty_like(wk)
    if ws is None:
        ws = _empty(lib().sparsp_predictor_workspace_size(_sref(shape), int(rank)), dev)
    _check("sparsp_predictor_fit", lib().sparsp_predictor_fit(
        _sref(shape), int(rank), _ptr(qmeans), _ptr(kmeans), _ptr(wq), _ptr(wk), float(lr), _ptr(loss),
        _ptr(gwq), _ptr(gwk), _ptr(ws), ws.numel(), _stream(stream)))
    return loss, gwq, gwk


# ----------------------------------------------------------------- step 5

def lpt_schedule(shape: Shape, row_ptr, flags=0, items=None, stream=None) -> torch.Tensor:
    dev = row_ptr.device
    if items is None:
        items = torch.empty(shape.rows, dtype=torch.int32, device=dev)
    ws = _empty(lib().sparsp_lpt_workspace_size(_sref(shape)), dev)
    _check("sparsp_lpt_schedule", lib().sparsp_lpt_schedule(
        _sref(shape), _ptr(row_ptr), int(flags), _ptr(items), _ptr(ws), ws.numel(), _stream(stream)))
    return items


def csr_transpose(shape: Shape, row_ptr, col_idx, nnz_cap=None, status=None, stream=None):
    dev = row_ptr.device
    col_ptr = torch.empty(shape.rows + 1, dtype=torch.int32, device=dev)
    cap = col_idx.numel() if nnz_cap is None else nnz_cap
    row_idx = torch.empty(max(cap, 4), dtype=torch.int32, device=dev)
    _check("sparsp_csr_transpose", lib().sparsp_csr_transpose(
        _sref(shape), _ptr(row_ptr), _ptr(col_idx), _ptr(col_ptr), _ptr(row_idx), _ptr(status),
        _stream(stream)))
    return col_ptr, row_idx


def attn_workspace_size(shape: Shape, backward: bool = False) -> int:
    return lib().sparsp_attn_workspace_size(_sref(shape), int(backward))


def attn_fwd(shape: Shape, q, k, v, row_ptr, col_idx, scale: float = 0.0, o=None, lse=None, ws=None,
             flags: int = 0, prof=None, status=None, stream=None):
    """Returns (O blocked [B,H,N,d], or raster [B,N,H,d] with OUT_RASTER; LSE [B,H,N] fp32)."""
    dev = q.device
    if o is None:
        o = torch.empty((shape.B, shape.N, shape.H, shape.d) if flags & OUT_RASTER else
                        (shape.B, shape.H, shape.N, shape.d), dtype=q.dtype, device=dev)
    if lse is None:
        lse = torch.empty((shape.B, shape.H, shape.N), dtype=torch.float32, device=dev)
    if ws is None:
        ws = _empty(attn_workspace_size(shape, False), dev)
    _check("sparsp_attn_fwd", lib().sparsp_attn_fwd(
        _sref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(row_ptr), _ptr(col_idx), float(scale), _ptr(o),
        _ptr(lse), _ptr(ws), ws.numel(), int(flags), _ptr(prof), _ptr(status), _stream(stream)))
    return o, lse


def attn_bwd(shape: Shape, q, k, v, o, lse, dout, row_ptr, col_idx, scale: float = 0.0, dq=None, dk=None,
             dv=None, ws=None, flags: int = 0, prof=None, status=None, stream=None):
    """Returns (dQ, dK, dV), blocked [B,H,N,d] bf16; raster [B,N,H,d] with OUT_RASTER
    in flags (o is then the raster O of attn_fwd with OUT_RASTER)."""
    dev = q.device
    dims = (shape.B, shape.N, shape.H, shape.d) if flags & OUT_RASTER else tuple(q.shape)
    dq = torch.empty(dims, dtype=q.dtype, device=dev) if dq is None else dq
    dk = torch.empty(dims, dtype=k.dtype, device=dev) if dk is None else dk
    dv = torch.empty(dims, dtype=v.dtype, device=dev) if dv is None else dv
    if ws is None:
        ws = _empty(attn_workspace_size(shape, True), dev)
    _check("sparsp_attn_bwd", lib().sparsp_attn_bwd(
        _sref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(row_ptr),
        _ptr(col_idx), float(scale), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(), int(flags),
        _ptr(prof), _ptr(status), _stream(stream)))
    return dq, dk, dv


def diag_umma_tile(a: torch.Tensor, b: torch.Tensor, mode: int, lbo: int = 16384, sbo: int = 1024,
                   status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """One 128x128x128 bf16 tcgen05 tile product (layout diagnostic, include/sparsp_diag.h).
    status: device int32 word that receives SPARSP_ERR_TIMEOUT if a bounded wait
    expires (a fresh zeroed one is used when None; check it after synchronising)."""
    d = torch.empty((128, 128), dtype=torch.float32, device=a.device)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=a.device)
    _check("sparsp_diag_umma_tile", lib().sparsp_diag_umma_tile(_ptr(a), _ptr(b), _ptr(d), int(mode), int(lbo),
                                                                int(sbo), _ptr(status), _stream(stream)))
    return d


def diag_wait_timeout(limit_ns: int, status: torch.Tensor, stream=None) -> None:
    """Runs the tensor-core kernels' bounded wait on a barrier nothing completes
    (include/sparsp_diag.h); *status receives SPARSP_ERR_TIMEOUT after limit_ns."""
    _check("sparsp_diag_wait_timeout", lib().sparsp_diag_wait_timeout(int(limit_ns), _ptr(status), _stream(stream)))


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


from .pipeline import GraphedStep, Pipeline  # noqa: E402,F401
from .streaming import HostPipeline  # noqa: E402,F401
