"""CPU oracle for dynamic per-head block-sparse attention over video tokens.

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module. It shares no code with the CUDA path
(no kernels, headers, helpers or constants) and never imports it.

Plain NumPy, float64 accumulation, written step by step from the pages:

* Step 1, video-aware block organisation: "mlsift.com tag listing" (sequence
  parallelism), Top-p video sparse-attention entry, abstract.
* Step 2, block scores: mean-pooled Q.K per block, or the per-head rank-16
  low-rank predictor of "Dynamic Sparsity in Large-Scale Video DiT Training",
  "How DSV works / The idea".
* Step 3, selection: Top-p routing with a Top-k safety floor (the same
  mlsift.com entry), compacted per head into a CSR of key-block indices.
* Step 4, KV demand of P contiguous query partitions: the one-GPU analogue of
  Demand-Directed KV Routing in "SparSP: Exploiting Communication Sparsity for
  Sequence-Parallel Video DiTs", abstract.
* Step 5, block-sparse attention forward and backward over the CSR:
  "Dynamic Sparsity in Large-Scale Video DiT Training", "How DSV works"
  (sparse attention only on the critical pairs, never materialising the full
  score matrix), and the FlashAttention comparison of the mlsift.com entry.
* The longest-first work order: the straggler problem of the mlsift.com entry
  and the lopsided per-head work of "How DSV works" (third paragraph).
* Dependency-aware placement of blocks on the P partitions: SparSP, abstract.
* Virtual-rank load balancing (head migration) and slack-aware sparse
  augmentation: the mlsift.com entry, abstract.
* Predictor fitting: "How DSV works / The idea" (the loss is read as the mean
  squared error of the predicted block scores; the pages do not define it).

Parity pins for every function live in tests/test_oracle_*.py. Every
function here has at least one pin that does not re-run its own formula.

Conventions
-----------
Raster layout [B, N, H, d], N = T*Y*X, x fastest. Tile (a, b, c), Bt = a*b*c,
tiles numbered with the x tile fastest; inside a tile, tokens are numbered
with x fastest. Block-ordered layout [B, H, N, d]: row j*Bt + o is token o of
tile j.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


# ---------------------------------------------------------------------------
# Step 1: video-aware block organisation
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Grid:
    B: int
    H: int
    T: int
    Y: int
    X: int
    d: int
    ta: int
    tb: int
    tc: int

    @property
    def N(self):
        return self.T * self.Y * self.X

    @property
    def Bt(self):
        return self.ta * self.tb * self.tc

    @property
    def nb(self):
        return self.N // self.Bt


def grid_of(wl) -> Grid:
    return Grid(wl.B, wl.H, wl.T, wl.Y, wl.X, wl.d, wl.ta, wl.tb, wl.tc)


def blocked_position(g: Grid) -> np.ndarray:
    """For each raster token n, its row in the block-ordered layout.

    Token (t, y, x) lies in tile (t//a, y//b, x//c), numbered x-tile fastest,
    at in-tile offset ((t%a)*b + y%b)*c + x%c.
    """
    if g.T % g.ta or g.Y % g.tb or g.X % g.tc:
        raise ValueError("grid not divisible by tile")
    nY, nX = g.Y // g.tb, g.X // g.tc
    n = np.arange(g.N, dtype=np.int64)
    t, rem = np.divmod(n, g.Y * g.X)
    y, x = np.divmod(rem, g.X)
    tile = ((t // g.ta) * nY + (y // g.tb)) * nX + (x // g.tc)
    off = ((t % g.ta) * g.tb + (y % g.tb)) * g.tc + (x % g.tc)
    return tile * g.Bt + off


def reorder(x_raster: np.ndarray, g: Grid) -> np.ndarray:
    """[B, N, H, d] raster -> [B, H, N, d] block-ordered."""
    pos = blocked_position(g)
    out = np.empty((g.B, g.H, g.N, x_raster.shape[-1]), dtype=x_raster.dtype)
    xt = np.transpose(x_raster, (0, 2, 1, 3))          # [B, H, N, d] in raster token order
    out[:, :, pos, :] = xt
    return out


def reorder_inverse(x_blocked: np.ndarray, g: Grid) -> np.ndarray:
    """[B, H, N, d] block-ordered -> [B, N, H, d] raster."""
    pos = blocked_position(g)
    xt = x_blocked[:, :, pos, :]                        # raster token order
    return np.ascontiguousarray(np.transpose(xt, (0, 2, 1, 3)))


# ---------------------------------------------------------------------------
# Step 2: block scores
# ---------------------------------------------------------------------------

def pool_means(xb: np.ndarray, Bt: int) -> np.ndarray:
    """Per-block mean of a block-ordered [B, H, N, d] tensor -> [B, H, nb, d] (float64)."""
    B, H, N, d = xb.shape
    return xb.astype(np.float64).reshape(B, H, N // Bt, Bt, d).mean(axis=3)


def scores_mean(qb: np.ndarray, kb: np.ndarray, Bt: int) -> np.ndarray:
    """Mean-pooled estimator: S[b,h,i,j] = mean(Q over block i) . mean(K over block j).

    No 1/sqrt(d) factor: the estimator is the plain pooled dot product.
    """
    qm = pool_means(qb, Bt)
    km = pool_means(kb, Bt)
    return np.einsum("bhid,bhjd->bhij", qm, km)


def scores_mean_tokenpairs(qb: np.ndarray, kb: np.ndarray, Bt: int) -> np.ndarray:
    """The same estimator as the mean of q.k over all Bt*Bt token pairs of each block pair.

    Brute force over the full token-level Q K^T; small inputs only.
    """
    B, H, N, d = qb.shape
    nb = N // Bt
    full = np.einsum("bhnd,bhmd->bhnm", qb.astype(np.float64), kb.astype(np.float64))
    return full.reshape(B, H, nb, Bt, nb, Bt).mean(axis=(3, 5))


def scores_lowrank(qb: np.ndarray, kb: np.ndarray, wq: np.ndarray, wk: np.ndarray, Bt: int) -> np.ndarray:
    """Low-rank predictor pooled to blocks, computed as pool-then-project.

    Per head h the predictor scores token pairs by (q Wq[h]) . (k Wk[h]) with
    Wq, Wk of shape [d, r] ("Dynamic Sparsity in Large-Scale Video DiT
    Training", "How DSV works": two small per-head matrices of inner dimension
    sixteen). The block score is that product averaged over the block pair;
    because it is bilinear this equals (mean q Wq) . (mean k Wk), which is
    what this function evaluates. scores_lowrank_tokenlevel evaluates the
    definition itself.
    """
    qm = pool_means(qb, Bt)                     # [B, H, nb, d]
    km = pool_means(kb, Bt)
    qp = np.einsum("bhid,hdr->bhir", qm, wq.astype(np.float64))
    kp = np.einsum("bhjd,hdr->bhjr", km, wk.astype(np.float64))
    return np.einsum("bhir,bhjr->bhij", qp, kp)


def scores_lowrank_tokenlevel(qb, kb, wq, wk, Bt, pairs=None):
    """Definition of the pooled low-rank score, evaluated at token level.

    pairs: optional list of (b, h, i, j); returns an array of those entries.
    Without pairs, the full [B, H, nb, nb] tensor (small inputs only).
    """
    B, H, N, d = qb.shape
    nb = N // Bt
    if pairs is None:
        out = np.zeros((B, H, nb, nb))
        for b in range(B):
            for h in range(H):
                a = qb[b, h].astype(np.float64) @ wq[h].astype(np.float64)     # [N, r]
                c = kb[b, h].astype(np.float64) @ wk[h].astype(np.float64)
                full = a @ c.T                                                  # [N, N]
                out[b, h] = full.reshape(nb, Bt, nb, Bt).mean(axis=(1, 3))
        return out
    vals = []
    for (b, h, i, j) in pairs:
        a = qb[b, h, i * Bt:(i + 1) * Bt].astype(np.float64) @ wq[h].astype(np.float64)
        c = kb[b, h, j * Bt:(j + 1) * Bt].astype(np.float64) @ wk[h].astype(np.float64)
        vals.append((a @ c.T).mean())
    return np.array(vals)


# ---------------------------------------------------------------------------
# Step 3: Top-p selection with a Top-k floor, compacted to CSR
# ---------------------------------------------------------------------------

def row_softmax(s: np.ndarray) -> np.ndarray:
    """Softmax of one score row, in float64."""
    s = np.asarray(s, dtype=np.float64)
    e = np.exp(s - s.max())
    return e / e.sum()


def _exp_f32(row: np.ndarray) -> np.ndarray:
    """e_j = exp(S_j - max S) of one float32 score row, correctly rounded to
    float32: the difference is taken in float32, its exponential in float64,
    and that is rounded once to float32."""
    diff = (row - row.max()).astype(np.float32)
    return np.exp(diff.astype(np.float64)).astype(np.float32)


@dataclass
class Selection:
    row_ptr: np.ndarray        # int32 [R+1]
    col_idx: np.ndarray        # int32 [nnz]
    order: list                # per row: int64 array, blocks by (score desc, index asc)
    m_lo: np.ndarray           # per row: smallest admissible count (== m_hi unless near-threshold)
    m_hi: np.ndarray
    margin: np.ndarray         # per row: distance of the Top-p crossing from p (relative mass)


def select(S: np.ndarray, top_p: float, k_floor: int, ambiguity: float = 1e-12) -> Selection:
    """Top-p routing with a Top-k safety floor, per query-block row.

    S: float32 [R, nb] (R = B*H*nb rows, row r = (b*H + h)*nb + i).
    For each row:
      1. softmax over the row: e_j = exp(S_j - max S), pi_j = e_j / sum e;
      2. order the blocks by (S_j descending, j ascending);
      3. m_p = smallest m whose leading prefix holds mass >= p
         (m_p = 0 when p <= 0, m_p = nb when p >= 1);
      4. m = min(nb, max(m_p, k_floor, 1))  (the safety floor; never empty);
      5. keep the first m blocks of that order, stored in ascending index order.
    e_j is the float32 rounding of exp(S_j - max S) (the exponent argument
    itself a float32 difference), and Z and the prefix masses are float64 sums
    of those values: the precision the device takes this decision in. Both
    sides then hold identical e_j, and their prefix sums differ only by the
    order of float64 additions (about 1e-13 of Z for nb <= 4096). Rows whose
    crossing lies within `ambiguity` (relative mass) of p admit the
    neighbouring count too; m_lo..m_hi records that.
    """
    S = np.asarray(S)
    if S.dtype != np.float32:
        raise TypeError("scores must be float32")
    if np.isnan(S).any() or np.isinf(S).any():
        raise ValueError("non-finite score")
    R, nb = S.shape
    p = float(np.float32(top_p))
    counts = np.zeros(R, dtype=np.int64)
    cols = []
    orders = []
    m_lo = np.zeros(R, dtype=np.int64)
    m_hi = np.zeros(R, dtype=np.int64)
    margin = np.full(R, np.inf)
    floor = max(int(k_floor), 1)
    for r in range(R):
        row = S[r] + np.float32(0.0)                       # -0.0 == +0.0
        order = np.argsort(-row.astype(np.float64), kind="stable")
        orders.append(order)
        e = _exp_f32(row).astype(np.float64)
        Z = e.sum()
        if p <= 0.0:
            m_p = 0
            cands = [0]
        elif p >= 1.0:
            m_p = nb
            cands = [nb]
        else:
            C = np.cumsum(e[order])
            target = p * Z
            m_p = min(nb, int(np.count_nonzero(C < target)) + 1)
            cands = [m_p]
            # distance of the two prefix sums that bracket the crossing
            lo_gap = abs(C[m_p - 2] - target) / Z if m_p >= 2 else np.inf
            hi_gap = abs(C[m_p - 1] - target) / Z
            margin[r] = min(lo_gap, hi_gap)
            if lo_gap < ambiguity:
                cands.append(m_p - 1)
            if hi_gap < ambiguity and m_p < nb:
                cands.append(m_p + 1)
        ms = [min(nb, max(c, floor)) for c in cands]
        m = min(nb, max(m_p, floor))
        m_lo[r], m_hi[r] = min(ms), max(ms)
        counts[r] = m
        cols.append(np.sort(order[:m]))
    row_ptr = np.zeros(R + 1, dtype=np.int64)
    row_ptr[1:] = np.cumsum(counts)
    col_idx = np.concatenate(cols) if cols else np.zeros(0, np.int64)
    return Selection(row_ptr.astype(np.int32), col_idx.astype(np.int32), orders, m_lo, m_hi, margin)


# ---------------------------------------------------------------------------
# Step 4: KV demand of P contiguous query partitions
# ---------------------------------------------------------------------------

def partition_bounds(nb: int, P: int) -> list[tuple[int, int]]:
    """Partition r owns query blocks [floor(r*nb/P), floor((r+1)*nb/P))."""
    return [((r * nb) // P, ((r + 1) * nb) // P) for r in range(P)]


@dataclass
class Demand:
    bitmap: np.ndarray     # uint32 [B, H, P, ceil(nb/32)]
    dem_ptr: np.ndarray    # int32 [B*H*P + 1]
    dem_idx: np.ndarray    # int32 [total]
    kg: np.ndarray | None  # [total, Bt, d]
    vg: np.ndarray | None
    bytes: np.ndarray      # uint64 [4]: demanded, all, remote_demanded, remote_all


def kv_demand(row_ptr, col_idx, B, H, nb, P, Bt, d, elem_bytes, kb=None, vb=None, owner=None) -> Demand:
    """The key/value blocks each query partition needs, as the one-GPU analogue
    of routing KV blocks only to the ranks that request them ("SparSP", abstract).

    Demand of partition r = union of the CSR rows of its query blocks.
    Byte counts (K and V both counted):
      demanded        = sum |demand| * Bt*d*elem * 2
      all             = B*H*P*nb * Bt*d*elem * 2   (every partition receives all KV)
      remote_demanded = demanded blocks outside the partition's own range
      remote_all      = all blocks outside the partition's own range
    owner: optional [B, nb] partition of every block (see placement); default:
    the contiguous split partition_bounds.
    """
    W = (nb + 31) // 32
    bitmap = np.zeros((B, H, P, W), dtype=np.uint32)
    sets = []
    tile = Bt * d * elem_bytes * 2
    demanded = remote_dem = remote_all = 0
    bounds = partition_bounds(nb, P)
    for b in range(B):
        if owner is None:
            members = [list(range(lo, hi)) for (lo, hi) in bounds]
        else:
            members = [[i for i in range(nb) if int(owner[b][i]) == r] for r in range(P)]
        for h in range(H):
            for r in range(P):
                own = set(members[r])
                want = set()
                for i in members[r]:
                    row = (b * H + h) * nb + i
                    want.update(int(j) for j in col_idx[row_ptr[row]:row_ptr[row + 1]])
                ordered = sorted(want)
                sets.append(ordered)
                for j in ordered:
                    bitmap[b, h, r, j // 32] |= np.uint32(1 << (j % 32))
                demanded += len(ordered) * tile
                remote_dem += sum(1 for j in ordered if j not in own) * tile
                remote_all += (nb - len(own)) * tile
    dem_ptr = np.zeros(len(sets) + 1, dtype=np.int64)
    dem_ptr[1:] = np.cumsum([len(s) for s in sets])
    dem_idx = np.array([j for s in sets for j in s], dtype=np.int32)
    kg = vg = None
    if kb is not None:
        kg = np.zeros((len(dem_idx), Bt, kb.shape[-1]), dtype=kb.dtype)
        vg = np.zeros_like(kg)
        slot = 0
        for s_i, s in enumerate(sets):
            bh = s_i // P
            b, h = divmod(bh, H)
            for j in s:
                kg[slot] = kb[b, h, j * Bt:(j + 1) * Bt]
                vg[slot] = vb[b, h, j * Bt:(j + 1) * Bt]
                slot += 1
    all_bytes = B * H * P * nb * tile
    byts = np.array([demanded, all_bytes, remote_dem, remote_all], dtype=np.uint64)
    return Demand(bitmap, dem_ptr.astype(np.int32), dem_idx, kg, vg, byts)


def affinity(row_ptr, col_idx, H, nb, b):
    """Co-selection counts of batch element b: W[i][j] = number of heads in which
    query block i selected key block j, plus the same with i and j swapped
    (i != j; the diagonal is 0)."""
    W = np.zeros((nb, nb), dtype=np.int64)
    for h in range(H):
        for i in range(nb):
            r = (b * H + h) * nb + i
            for j in col_idx[row_ptr[r]:row_ptr[r + 1]]:
                j = int(j)
                if j != i:
                    W[i, j] += 1
                    W[j, i] += 1
    return W


def placement(row_ptr, col_idx, B, H, nb, P) -> np.ndarray:
    """Dependency-aware placement of blocks on P partitions ("SparSP:
    Exploiting Communication Sparsity for Sequence-Parallel Video DiTs",
    abstract: sequence blocks distributed according to the sparse attention
    pattern), one assignment per batch element shared by all heads, with the
    partition sizes of the contiguous split.

    Deterministic greedy on the co-selection affinity W:
      blocks in order of total affinity sum_j W[i][j] descending (ties: lower i);
      each goes to the partition with spare capacity whose already-placed
      blocks have the largest affinity to it (ties: more spare capacity, then
      lower partition index).
    Returns owner [B, nb] int32.
    """
    caps0 = [hi - lo for (lo, hi) in partition_bounds(nb, P)]
    owner = np.full((B, nb), -1, dtype=np.int32)
    for b in range(B):
        W = affinity(row_ptr, col_idx, H, nb, b)
        total = W.sum(axis=1)
        order = sorted(range(nb), key=lambda i: (-int(total[i]), i))
        caps = list(caps0)
        for i in order:
            best = None
            for r in range(P):
                if caps[r] == 0:
                    continue
                score = int(sum(W[i, j] for j in range(nb) if owner[b, j] == r))
                key = (score, caps[r], -r)
                if best is None or key > best[0]:
                    best = (key, r)
            r = best[1]
            owner[b, i] = r
            caps[r] -= 1
    return owner


# ---------------------------------------------------------------------------
# Step 5: block-sparse attention over the CSR
# ---------------------------------------------------------------------------

def _row_of(b, h, i, H, nb):
    return (b * H + h) * nb + i


def _selected_kv(xb, b, h, cols, Bt):
    if len(cols) == 0:
        return np.zeros((0, xb.shape[-1]))
    return np.concatenate([xb[b, h, j * Bt:(j + 1) * Bt].astype(np.float64) for j in cols], axis=0)


def attn_fwd_row(qb, kb, vb, row_ptr, col_idx, Bt, scale, b, h, i):
    """O and LSE of query block i of head (b, h): softmax attention over the
    key tokens of the selected blocks only. Empty row: O = 0, LSE = -inf."""
    H, N = qb.shape[1], qb.shape[2]
    nb = N // Bt
    r = _row_of(b, h, i, H, nb)
    cols = col_idx[row_ptr[r]:row_ptr[r + 1]]
    q = qb[b, h, i * Bt:(i + 1) * Bt].astype(np.float64)
    if len(cols) == 0:
        return np.zeros_like(q), np.full(Bt, -np.inf)
    ks = _selected_kv(kb, b, h, cols, Bt)
    vs = _selected_kv(vb, b, h, cols, Bt)
    s = scale * (q @ ks.T)
    mx = s.max(axis=1, keepdims=True)
    lse = (mx + np.log(np.exp(s - mx).sum(axis=1, keepdims=True)))[:, 0]
    p = np.exp(s - lse[:, None])
    return p @ vs, lse


def attn_fwd(qb, kb, vb, row_ptr, col_idx, Bt, scale=None, rows=None):
    """Block-sparse attention forward. rows: optional list of (b, h, i).

    Returns (O [B,H,N,d] float64, LSE [B,H,N] float64); rows not requested stay NaN.
    """
    B, H, N, d = qb.shape
    nb = N // Bt
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    O = np.full((B, H, N, d), np.nan)
    L = np.full((B, H, N), np.nan)
    todo = rows if rows is not None else [(b, h, i) for b in range(B) for h in range(H) for i in range(nb)]
    for (b, h, i) in todo:
        o, l = attn_fwd_row(qb, kb, vb, row_ptr, col_idx, Bt, scale, b, h, i)
        O[b, h, i * Bt:(i + 1) * Bt] = o
        L[b, h, i * Bt:(i + 1) * Bt] = l
    return O, L


def token_mask(row_ptr, col_idx, B, H, nb, Bt):
    """Token-level mask M[b,h,q,k] = [block(k) is selected by block(q)] (small inputs)."""
    N = nb * Bt
    M = np.zeros((B, H, N, N), dtype=bool)
    for b in range(B):
        for h in range(H):
            for i in range(nb):
                r = _row_of(b, h, i, H, nb)
                for j in col_idx[row_ptr[r]:row_ptr[r + 1]]:
                    M[b, h, i * Bt:(i + 1) * Bt, j * Bt:(j + 1) * Bt] = True
    return M


def attn_dense_masked(qb, kb, vb, M, scale):
    """Dense softmax attention over all N tokens with an explicit boolean mask (brute force)."""
    s = scale * np.einsum("bhqd,bhkd->bhqk", qb.astype(np.float64), kb.astype(np.float64))
    s = np.where(M, s, -np.inf)
    mx = s.max(axis=-1, keepdims=True)
    w = np.where(M, np.exp(s - mx), 0.0)
    z = w.sum(axis=-1, keepdims=True)
    O = np.einsum("bhqk,bhkd->bhqd", w / z, vb.astype(np.float64))
    return O, (mx + np.log(z))[..., 0]


def attn_bwd(qb, kb, vb, dob, row_ptr, col_idx, Bt, scale=None, q_blocks=None, k_blocks=None):
    """Gradients of L = sum(dO * O) w.r.t. Q, K, V with the selection held fixed.

    For each selected (query block i, key block j) pair, with O and LSE from
    the forward above and D = rowsum(dO * O):
      P  = exp(scale * Q_i K_j^T - LSE_i)
      dV_j += P^T dO_i
      dP = dO_i V_j^T
      dS = P * (dP - D_i)
      dQ_i += scale * dS K_j
      dK_j += scale * dS^T Q_i
    q_blocks / k_blocks: optional sets of (b, h, block) whose dQ / (dK, dV)
    are wanted; other entries stay NaN. Only the rows needed are processed.
    Returns (dQ, dK, dV) as float64 [B, H, N, d].
    """
    B, H, N, d = qb.shape
    nb = N // Bt
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    want_q = None if q_blocks is None else set(q_blocks)
    want_k = None if k_blocks is None else set(k_blocks)
    dQ = np.full((B, H, N, d), np.nan)
    dK = np.full((B, H, N, d), np.nan)
    dV = np.full((B, H, N, d), np.nan)
    if want_k is None:
        dK[:] = 0.0
        dV[:] = 0.0
    else:
        for (b, h, j) in want_k:
            dK[b, h, j * Bt:(j + 1) * Bt] = 0.0
            dV[b, h, j * Bt:(j + 1) * Bt] = 0.0
    for b in range(B):
        for h in range(H):
            for i in range(nb):
                r = _row_of(b, h, i, H, nb)
                cols = [int(j) for j in col_idx[row_ptr[r]:row_ptr[r + 1]]]
                need_q = want_q is None or (b, h, i) in want_q
                need_k = want_k is None or any((b, h, j) in want_k for j in cols)
                if not (need_q or need_k):
                    continue
                q = qb[b, h, i * Bt:(i + 1) * Bt].astype(np.float64)
                do = dob[b, h, i * Bt:(i + 1) * Bt].astype(np.float64)
                if len(cols) == 0:
                    if need_q:
                        dQ[b, h, i * Bt:(i + 1) * Bt] = 0.0
                    continue
                o, lse = attn_fwd_row(qb, kb, vb, row_ptr, col_idx, Bt, scale, b, h, i)
                D = (do * o).sum(axis=1)
                dq = np.zeros((Bt, d))
                for j in cols:
                    k = kb[b, h, j * Bt:(j + 1) * Bt].astype(np.float64)
                    v = vb[b, h, j * Bt:(j + 1) * Bt].astype(np.float64)
                    P = np.exp(scale * (q @ k.T) - lse[:, None])
                    dP = do @ v.T
                    dS = P * (dP - D[:, None])
                    dq += scale * (dS @ k)
                    if want_k is None or (b, h, j) in want_k:
                        dV[b, h, j * Bt:(j + 1) * Bt] += P.T @ do
                        dK[b, h, j * Bt:(j + 1) * Bt] += scale * (dS.T @ q)
                if need_q:
                    dQ[b, h, i * Bt:(i + 1) * Bt] = dq
    return dQ, dK, dV


# ---------------------------------------------------------------------------
# Step 5c: longest-first work order
# ---------------------------------------------------------------------------

def lpt_order(row_ptr, B, H, nb, grouped=True) -> np.ndarray:
    """Work items (b, h, i), encoded (b*H + h)*nb + i, longest first.

    The cost of item (b, h, i) is its CSR row length (the number of selected
    key blocks, proportional to its attention work).
    grouped=True: heads ordered by total cost descending (ties: head index
      ascending); inside a head, rows by cost descending (ties: i ascending).
      Each head's query blocks stay together, so its K/V stays cache-resident.
    grouped=False: all items by cost descending, ties by (head, i) ascending.
    """
    rp = np.asarray(row_ptr, dtype=np.int64)
    cost = rp[1:] - rp[:-1]
    items = list(range(B * H * nb))
    if not grouped:
        return np.array(sorted(items, key=lambda it: (-cost[it], it)), dtype=np.int32)
    head_cost = [int(cost[bh * nb:(bh + 1) * nb].sum()) for bh in range(B * H)]
    heads = sorted(range(B * H), key=lambda bh: (-head_cost[bh], bh))
    out = []
    for bh in heads:
        out.extend(sorted(range(bh * nb, (bh + 1) * nb), key=lambda it: (-cost[it], it)))
    return np.array(out, dtype=np.int32)


def csc_of(row_ptr, col_idx, B, H, nb):
    """Transpose of the per-head CSR: for each key block, the query blocks
    that selected it, ascending. Returns (col_ptr [B*H*nb+1], row_idx [nnz])."""
    lists = [[] for _ in range(B * H * nb)]
    for bh in range(B * H):
        for i in range(nb):
            r = bh * nb + i
            for j in col_idx[row_ptr[r]:row_ptr[r + 1]]:
                lists[bh * nb + int(j)].append(i)
    col_ptr = np.zeros(B * H * nb + 1, dtype=np.int64)
    col_ptr[1:] = np.cumsum([len(x) for x in lists])
    row_idx = np.array([i for x in lists for i in x], dtype=np.int32)
    return col_ptr.astype(np.int32), row_idx


# ---------------------------------------------------------------------------
# Virtual-rank load balancing and slack-aware augmentation
# ---------------------------------------------------------------------------

def head_costs(row_ptr, B, H, nb) -> np.ndarray:
    """Attention work of every head: the number of selected block pairs of its
    rows (each pair costs the same 4*Bt^2*d flops). Returns int64 [B, H]."""
    rp = np.asarray(row_ptr, dtype=np.int64)
    return np.array([[int(rp[(b * H + h + 1) * nb] - rp[(b * H + h) * nb]) for h in range(H)]
                     for b in range(B)], dtype=np.int64)


def rank_loads(costs_b, head_rank_b, P) -> np.ndarray:
    """Sum of the head costs held by each of the P ranks (one batch element)."""
    loads = np.zeros(P, dtype=np.int64)
    for h, c in enumerate(costs_b):
        loads[int(head_rank_b[h])] += int(c)
    return loads


def imbalance(loads) -> float:
    """Critical (maximum) rank load over the mean rank load; 1.0 when idle."""
    loads = np.asarray(loads, dtype=np.int64)
    total = int(loads.sum())
    return 1.0 if total == 0 else float(loads.max()) * len(loads) / total


def balance_heads(costs, P, max_migrations):
    """Runtime Load Balancing over P virtual ranks (the mlsift.com tag listing,
    Top-p video sparse-attention entry, abstract: a few heavy heads migrate to
    shorten the critical path), one batch element at a time.

    Start: the contiguous head split, rank r holding heads
    [floor(r*H/P), floor((r+1)*H/P)). Then, at most max_migrations times:
      c = the most loaded rank, t = the least loaded (ties: lower rank);
      among the heads on c pick the one whose move to t gives the smallest
      max(L_c - cost, L_t + cost) (ties: lower head index);
      move it only if that value is below L_c, else stop.
    Every move lowers the sum of squared loads, so the loop ends.
    Returns (head_rank [B, H] int32, migrations [B] int64).
    """
    costs = np.asarray(costs, dtype=np.int64)
    B, H = costs.shape
    head_rank = np.zeros((B, H), dtype=np.int32)
    moves = np.zeros(B, dtype=np.int64)
    for b in range(B):
        for r, (lo, hi) in enumerate(partition_bounds(H, P)):
            head_rank[b, lo:hi] = r
        loads = rank_loads(costs[b], head_rank[b], P)
        for _ in range(int(max_migrations)):
            c = int(np.argmax(loads))
            t = int(np.argmin(loads))
            best = None
            for h in range(H):
                if head_rank[b, h] != c:
                    continue
                x = int(costs[b, h])
                new_max = max(int(loads[c]) - x, int(loads[t]) + x)
                if best is None or new_max < best[0]:
                    best = (new_max, h)
            if best is None or best[0] >= loads[c]:
                break
            h = best[1]
            head_rank[b, h] = t
            loads[c] -= costs[b, h]
            loads[t] += costs[b, h]
            moves[b] += 1
    return head_rank, moves


def block_values(S) -> np.ndarray:
    """The value of every block of a row: its softmax mass, taken as selection
    takes it (e_j = exp(S_j - max) correctly rounded to float32, Z = sum e in
    float64), rounded to float32: v_j = fl32(e_j / Z). S: float32 [R, nb]."""
    S = np.asarray(S)
    if S.dtype != np.float32:
        raise TypeError("scores must be float32")
    out = np.zeros(S.shape, dtype=np.float32)
    for r in range(S.shape[0]):
        row = S[r] + np.float32(0.0)
        e = _exp_f32(row).astype(np.float64)
        out[r] = (e / e.sum()).astype(np.float32)
    return out


@dataclass
class Augmented:
    row_ptr: np.ndarray        # int32 [R+1], the augmented CSR
    col_idx: np.ndarray        # int32 [nnz'], ascending per row
    added: np.ndarray          # int64 [B, P], blocks added per rank
    loads: np.ndarray          # int64 [B, P], rank loads after augmentation
    cut: np.ndarray            # float32 [B, P], value of the last block added (0 if none)
    next_value: np.ndarray     # float32 [B, P], best value left out (0 if none)


def augment(S, row_ptr, col_idx, B, H, nb, head_rank, P) -> Augmented:
    """Slack-Aware Sparse Augmentation (the mlsift.com tag listing, Top-p video
    sparse-attention entry, abstract: slack left on non-critical ranks is
    filled with additional high-value blocks).

    With the heads placed on ranks (head_rank [B, H]) and loads L_r in block
    pairs, the critical load is L* = max_r L_r; rank r has slack L* - L_r.
    Its candidates are the unselected blocks (h, i, j) of the rows of its
    heads, valued by block_values; it takes the min(slack, #candidates) best,
    ordered by (value descending, row (b*H + h)*nb + i ascending, j ascending).
    The critical path (L*) is unchanged. Returns the augmented CSR (rows stay
    ascending) with per-rank counts.
    """
    V = block_values(S)
    rp = np.asarray(row_ptr, dtype=np.int64)
    costs = head_costs(rp, B, H, nb)
    rows = [set(int(j) for j in col_idx[rp[r]:rp[r + 1]]) for r in range(B * H * nb)]
    added = np.zeros((B, P), dtype=np.int64)
    loads_out = np.zeros((B, P), dtype=np.int64)
    cut = np.zeros((B, P), dtype=np.float32)
    nxt = np.zeros((B, P), dtype=np.float32)
    for b in range(B):
        loads = rank_loads(costs[b], head_rank[b], P)
        top = int(loads.max())
        for r in range(P):
            cands = []
            for h in range(H):
                if int(head_rank[b, h]) != r:
                    continue
                for i in range(nb):
                    row = (b * H + h) * nb + i
                    for j in range(nb):
                        if j not in rows[row]:
                            cands.append((-float(V[row, j]), row, j))
            cands.sort()
            take = min(top - int(loads[r]), len(cands))
            for (_, row, j) in cands[:take]:
                rows[row].add(j)
            added[b, r] = take
            loads_out[b, r] = int(loads[r]) + take
            if take > 0:
                cut[b, r] = -cands[take - 1][0]
            if take < len(cands):
                nxt[b, r] = -cands[take][0]
    counts = [len(x) for x in rows]
    new_ptr = np.zeros(len(rows) + 1, dtype=np.int64)
    new_ptr[1:] = np.cumsum(counts)
    new_idx = np.array([j for x in rows for j in sorted(x)], dtype=np.int32)
    return Augmented(new_ptr.astype(np.int32), new_idx, added, loads_out, cut, nxt)


# ---------------------------------------------------------------------------
# Predictor fitting
# ---------------------------------------------------------------------------

def predictor_loss_grad(qm, km, wq, wk):
    """Loss and gradients for fitting the per-head low-rank predictor
    ("Dynamic Sparsity in Large-Scale Video DiT Training", "How DSV works / The
    idea": two small per-head matrices whose product approximates the real
    query-key scores, trained beside the main graph with a magnitude-preserving
    loss that the pages do not define).

    Read as the mean squared error between the predictor's block scores and the
    real block scores of the same pooled means, per head over the batch and all
    block pairs (the squared error keeps the scores' magnitudes, not only their
    order):
        E[b,h,i,j] = (qm[b,h,i] Wq[h]) . (km[b,h,j] Wk[h]) - qm[b,h,i] . km[b,h,j]
        L[h] = sum_{b,i,j} E^2 / (B nb^2)
    qm, km: [B, H, nb, d]; wq, wk: [H, d, r]. Returns (L [H], dL/dWq [H, d, r],
    dL/dWk [H, d, r]) in float64. The gradients are the chain rule of L:
        dL/dWq[h] = 2/(B nb^2) sum_b qm[b,h]^T (E[b,h] (km[b,h] Wk[h]))
        dL/dWk[h] = 2/(B nb^2) sum_b km[b,h]^T (E[b,h]^T (qm[b,h] Wq[h]))
    """
    qm = np.asarray(qm, dtype=np.float64)
    km = np.asarray(km, dtype=np.float64)
    wq = np.asarray(wq, dtype=np.float64)
    wk = np.asarray(wk, dtype=np.float64)
    B, H, nb, d = qm.shape
    A = np.einsum("bhid,hdr->bhir", qm, wq)
    Bk = np.einsum("bhjd,hdr->bhjr", km, wk)
    E = np.einsum("bhir,bhjr->bhij", A, Bk) - np.einsum("bhid,bhjd->bhij", qm, km)
    n = B * nb * nb
    loss = (E ** 2).sum(axis=(0, 2, 3)) / n
    GA = np.einsum("bhij,bhjr->bhir", E, Bk)
    GB = np.einsum("bhij,bhir->bhjr", E, A)
    gwq = 2.0 / n * np.einsum("bhid,bhir->hdr", qm, GA)
    gwk = 2.0 / n * np.einsum("bhjd,bhjr->hdr", km, GB)
    return loss, gwq, gwk


def predictor_step(qm, km, wq, wk, lr):
    """One plain gradient step on predictor_loss_grad's loss (the predictor is
    updated as the forward pass runs): W <- W - lr dL/dW for both matrices,
    with the gradients taken at the current weights. Returns (wq', wk', L)."""
    loss, gwq, gwk = predictor_loss_grad(qm, km, wq, wk)
    return np.asarray(wq, np.float64) - lr * gwq, np.asarray(wk, np.float64) - lr * gwk, loss
