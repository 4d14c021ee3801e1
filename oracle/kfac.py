"""The K-FAC preconditioning step in float64, written from the SPD-KFAC paper.

Source: "Accelerating Distributed K-FAC with Smart Parallelism of Computing and
Communication Tasks" (SPD-KFAC).  Its display equations were lost in the text
we have; the surviving prose fixes the following, and each function cites it:

  §II-B (KFAC): the Fisher block of layer l is approximated by the Kronecker
      product of two symmetric factors built from the layer input a_{l-1} and
      the output gradient g_l (Eq. (3)); A_{l-1} and G_l are computed by the
      equations the paper calls Eq. (7) and Eq. (8).  The Kronecker inverse
      identity turns the update into G^-1 grad A^-1, and Tikhonov damping adds
      gamma*I to each factor before inverting (the damped update rule).
  §II-C (D-KFAC): each worker p has local factors A^p, G^p that are
      aggregated over the P workers before inverting.
  §III-B (load-balancing placement): the damped inverses (A + lambda*I)^-1,
      (G + lambda*I)^-1 of the aggregated factors.
  §IV (implementation): the inverse is computed through a Cholesky
      decomposition; the inverse of a symmetric factor is symmetric, so only
      its upper triangle (d(d+1)/2 elements) needs to travel.

Readings where the pages are silent:
  * factor normalisation is the mean over the rows a worker holds
    (A^p = a_p^T a_p / rows_p); conv layers use per-sample spatially summed
    output gradients for G (G^p = gs_p^T gs_p / samples_p);
  * aggregation over workers is the mean of the P local factors;
  * the running average starts from the first aggregated factor
    (R_1 = F_1) and then R_t = decay*R_{t-1} + (1-decay)*F_t;
  * damping is applied to a copy: the running factor stays undamped.
"""
from __future__ import annotations

import math

import numpy as np


# ---------------------------------------------------------------- factors
def factor(x: np.ndarray, scale: float) -> np.ndarray:
    """Kronecker factor scale * x^T x of one worker's rows.

    §II-B, Eq. (7)/(8): A = E[a a^T] over the samples, G = E[g g^T]; with the
    samples as the rows of ``x`` this is x^T x / rows (``scale = 1/rows``).
    """
    x = np.asarray(x, dtype=np.float64)
    return scale * (x.T @ x)


def shard_factors(x: np.ndarray, P: int, scale: float | None = None):
    """Local factors of P workers holding equal contiguous row blocks of ``x``.

    §II-C: worker p computes A^p (or G^p) from its own locally sampled rows.
    ``scale`` defaults to 1/rows_p.
    """
    rows = x.shape[0]
    if rows % P:
        raise ValueError("rows must split into P equal shards")
    rp = rows // P
    s = 1.0 / rp if scale is None else scale
    return [factor(x[p * rp:(p + 1) * rp], s) for p in range(P)]


def aggregate(shards) -> np.ndarray:
    """§II-C: the workers' local factors are aggregated before inverting.

    Reading: the aggregate is the mean over the P workers (an all-reduce sum
    followed by 1/P), which keeps the full-batch normalisation.
    """
    acc = np.zeros_like(np.asarray(shards[0], dtype=np.float64))
    for s in shards:
        acc = acc + np.asarray(s, dtype=np.float64)
    return acc / len(shards)


def update_running(F: np.ndarray, R_prev: np.ndarray | None, decay: float,
                   first_step: bool) -> np.ndarray:
    """Running average of the aggregated factor across K-FAC steps.

    The pages name no averaging rule; the reading is R_1 = F_1 and
    R_t = decay * R_{t-1} + (1 - decay) * F_t, ``decay`` weighting the old value.
    """
    F = np.asarray(F, dtype=np.float64)
    if first_step:
        return F.copy()
    return decay * np.asarray(R_prev, dtype=np.float64) + (1.0 - decay) * F


def damp(R: np.ndarray, gamma: float) -> np.ndarray:
    """§II-B damped update rule: Tikhonov damping R + gamma*I (on a copy)."""
    D = np.array(R, dtype=np.float64, copy=True)
    D[np.diag_indices_from(D)] += gamma
    return D


# ---------------------------------------------------------------- inverse
def cholesky_lower(D: np.ndarray):
    """Cholesky factor D = L L^T, column by column (Cholesky-Crout order).

    §IV: the inverse is computed through a Cholesky decomposition.  Returns
    ``(L, info)``; ``info = j`` (1-based) when the j-th pivot is not positive
    (the leading minor of order j is not positive definite), else 0.
    """
    D = np.asarray(D, dtype=np.float64)
    n = D.shape[0]
    L = np.zeros((n, n), dtype=np.float64)
    for j in range(n):
        s = D[j, j] - L[j, :j] @ L[j, :j]
        if not (s > 0.0) or not math.isfinite(s):
            return L, j + 1
        ljj = math.sqrt(s)
        L[j, j] = ljj
        if j + 1 < n:
            L[j + 1:, j] = (D[j + 1:, j] - L[j + 1:, :j] @ L[j, :j]) / ljj
    return L, 0


def lower_tri_inverse(L: np.ndarray) -> np.ndarray:
    """W = L^-1 for lower-triangular L by forward substitution on I, row by row:
    row i of L W = I gives W[i, :i+1] = (e_i - L[i, :i] W[:i, :i+1]) / L[i, i]."""
    L = np.asarray(L, dtype=np.float64)
    n = L.shape[0]
    W = np.zeros((n, n), dtype=np.float64)
    for i in range(n):
        rhs = np.zeros(i + 1)
        rhs[i] = 1.0
        if i:
            rhs = rhs - L[i, :i] @ W[:i, :i + 1]
        W[i, :i + 1] = rhs / L[i, i]
    return W


def spd_inverse(D: np.ndarray):
    """Inverse of an SPD matrix through its Cholesky factor (§IV):
    D = L L^T  =>  D^-1 = L^-T L^-1 = W^T W with W = L^-1.

    The product is formed for the upper triangle and mirrored, so the result
    is exactly symmetric (§III-B: the inverse of a symmetric factor is
    symmetric).  Returns ``(X, info)``; X is None when info != 0.
    """
    L, info = cholesky_lower(D)
    if info:
        return None, info
    W = lower_tri_inverse(L)
    X = W.T @ W
    iu = np.triu_indices_from(X, 1)
    X[(iu[1], iu[0])] = X[iu]
    return X, 0


def damped_inverse(D: np.ndarray, gamma_extra: float = 0.0):
    """(D + gamma_extra*I)^-1 of an already damped factor (§III-B)."""
    Dd = damp(D, gamma_extra) if gamma_extra else np.asarray(D, dtype=np.float64)
    return spd_inverse(Dd)


# ---------------------------------------------------------------- precondition
def precondition(XG: np.ndarray, grad: np.ndarray, XA: np.ndarray) -> np.ndarray:
    """§II-B damped update rule: (G + gamma I)^-1 grad (A + gamma I)^-1.

    ``grad`` is d_out x d_in (rows follow G, columns follow A), so with
    column-major vec, vec(XG grad XA) = (XA (x) XG) vec(grad) for symmetric XA.
    """
    return (np.asarray(XG, np.float64) @ np.asarray(grad, np.float64)) @ np.asarray(XA, np.float64)


def kron_precondition_bruteforce(A, G, grad, gamma: float) -> np.ndarray:
    """Brute force of the same update: materialise the damped Kronecker block
    (A + gamma I) (x) (G + gamma I) (§II-B, Eq. (3) with per-factor damping)
    and solve it against vec(grad) (column-major vec).  Only for tiny layers."""
    A = np.asarray(A, np.float64)
    G = np.asarray(G, np.float64)
    grad = np.asarray(grad, np.float64)
    K = np.kron(damp(A, gamma), damp(G, gamma))
    v = np.linalg.solve(K, grad.reshape(-1, order="F"))
    return v.reshape(grad.shape, order="F")


def weight_step(W: np.ndarray, V: np.ndarray, lr: float) -> np.ndarray:
    """§II-B damped update rule, the step itself: the weights move against the
    preconditioned gradient, W - lr * V."""
    return np.asarray(W, np.float64) - float(lr) * np.asarray(V, np.float64)


# ---------------------------------------------------------------- conv helper
def spatial_sum(g: np.ndarray, batch: int, hw: int) -> np.ndarray:
    """Per-sample sum of a conv layer's output gradients over its H*W
    positions: gs[b, c] = sum_{s < hw} g[b*hw + s, c].  (Reading: the pages do
    not describe conv factors; this is the form the G factor is built from.)"""
    g = np.asarray(g, np.float64)
    return g.reshape(batch, hw, g.shape[1]).sum(axis=1)


def im2col3x3(x: np.ndarray, bias: bool = True) -> np.ndarray:
    """Patch rows of a 3 x 3, stride 1, zero-padding 1 convolution over an NHWC
    activation x[b, h, w, c] (the conv layer's input a of the Kronecker factor
    A; reading: the pages do not describe conv factors).  Row (b, h, w), in
    that order; column (dh * 3 + dw) * C + c holds x[b, h + dh - 1, w + dw - 1, c]
    (0 outside the image); with `bias` a last column of ones."""
    x = np.asarray(x, np.float64)
    B, H, W, C = x.shape
    xp = np.zeros((B, H + 2, W + 2, C))
    xp[:, 1:H + 1, 1:W + 1, :] = x
    cols = [xp[:, dh:dh + H, dw:dw + W, :].reshape(B * H * W, C) for dh in range(3) for dw in range(3)]
    if bias:
        cols.append(np.ones((B * H * W, 1)))
    return np.concatenate(cols, axis=1)


# ---------------------------------------------------------------- index maps
def upper_tiles(d: int, tile: int = 128):
    """Upper-triangle tiles (i, j), i <= j, of a d x d symmetric matrix cut into
    tile x tile blocks, row-major over i (§III-A: only upper triangles count)."""
    T = -(-d // tile)
    return [(i, j) for i in range(T) for j in range(i, T)]


def factor_tile_units(d: int, bm: int = 128, bn: int = 256):
    """Work units that cover the upper-triangle tiles of a d x d factor, in
    pairs of row blocks (the tensor-core SYRK runs a CTA pair per pair):
    pair s = row blocks (2s, 2s+1) takes the columns [s*bn, d) in chunks of at
    most bn (bn = 2*bm); each chunk gives the units (2s, j0, w) and
    (2s+1, j0, w).  A unit stores only its columns >= i*bm of an existing row
    block i (see ``stored_part``)."""
    assert bn == 2 * bm
    n0 = -(-d // bn)
    units = []
    for s in range(n0):
        for v in range(n0 - s):
            j0 = bn * (s + v)
            w = min(bn, d - j0)
            units.append((2 * s, j0, w))
            units.append((2 * s + 1, j0, w))
    return units


def stored_part(unit, d: int, bm: int = 128):
    """(rows, cols) ranges of a unit that land in the factor (possibly empty)."""
    i, j0, w = unit
    r0, r1 = i * bm, min(i * bm + bm, d)
    c0, c1 = max(j0, i * bm), j0 + w
    return (r0, max(r0, r1)), (c0, max(c0, c1))


def packed_index(i: int, j: int, d: int) -> int:
    """0-based position of (i, j), i <= j, in the row-major packed upper
    triangle of d(d+1)/2 elements (§IV: only the upper triangle incl. the
    diagonal is sent)."""
    if not 0 <= i <= j < d:
        raise ValueError("need 0 <= i <= j < d")
    return i * d - i * (i - 1) // 2 + (j - i)


def pack_upper(M: np.ndarray) -> np.ndarray:
    """The d(d+1)/2 upper-triangle elements of a symmetric d x d matrix, row
    by row: row r contributes M[r, r:] (§III-A: a symmetric factor is
    communicated as its upper triangle; §IV: so is the symmetric inverse)."""
    M = np.asarray(M)
    d = M.shape[0]
    return np.concatenate([M[r, r:] for r in range(d)])


def unpack_upper(p: np.ndarray, d: int, mirror: bool = True) -> np.ndarray:
    """The matrix whose upper triangle ``p`` packs (``pack_upper``'s layout);
    with ``mirror`` the strict lower triangle is filled from it, else it is
    left NaN."""
    p = np.asarray(p)
    if p.shape[0] != d * (d + 1) // 2:
        raise ValueError("packed length is not d(d+1)/2")
    M = np.full((d, d), np.nan, dtype=p.dtype)
    start = 0
    for r in range(d):
        M[r, r:] = p[start:start + d - r]
        start += d - r
    if mirror:
        il = np.tril_indices(d, -1)
        M[il] = M.T[il]
    return M


# ---------------------------------------------------------------- one step
def kfac_step(layer_data, P: int, gamma: float, decay: float, first_step: bool,
              running=None, conv=None):
    """One K-FAC step over a list of layers.

    ``layer_data[l]`` holds ``a`` (rows x d_in), ``g`` (rows x d_out) and
    ``grad`` (d_out x d_in).  ``conv[l]`` is None for a linear layer or
    (batch, hw) for a conv layer.  ``running[l]`` is the (R_A, R_G) pair of the
    previous step.  Returns a dict per layer with the aggregated factors, the
    running and damped factors, the inverses and the preconditioned gradient.
    """
    out = []
    for l, data in enumerate(layer_data):
        a, g = data["a"], data["g"]
        cv = None if conv is None else conv[l]
        SA = shard_factors(a, P)
        if cv is None:
            SG = shard_factors(g, P)
        else:
            batch, hw = cv
            SG = shard_factors(spatial_sum(g, batch, hw), P)
        FA, FG = aggregate(SA), aggregate(SG)
        prev = (None, None) if running is None else running[l]
        RA = update_running(FA, prev[0], decay, first_step)
        RG = update_running(FG, prev[1], decay, first_step)
        DA, DG = damp(RA, gamma), damp(RG, gamma)
        XA, ia = spd_inverse(DA)
        XG, ig = spd_inverse(DG)
        V = None if (ia or ig) else precondition(XG, data["grad"], XA)
        out.append(dict(SA=SA, SG=SG, FA=FA, FG=FG, RA=RA, RG=RG, DA=DA, DG=DG,
                        XA=XA, XG=XG, info=(ia, ig), V=V))
    return out
