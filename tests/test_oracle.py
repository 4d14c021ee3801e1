"""Pins of the fp64 oracle against what the SPD-KFAC page and plain mathematics
fix: brute force on tiny inputs, closed forms, invariants, library special
cases and the page's printed ResNet-50 factor sizes.  Each pin is chosen so a
plausible slip (a dropped term, a wrong index, a transposed operand, a wrong
normalisation) fails it.  CPU only."""
import math
import os

import numpy as np
import pytest
import scipy.linalg

import oracle
import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def rnd(*shape, seed=0):
    return np.random.default_rng(seed).standard_normal(shape)


# ------------------------------------------------------------------ factors
def test_factor_matches_triple_loop():
    x = np.array([[1, 2, -1, 0], [3, 0, 2, 1], [-2, 1, 1, 4]], dtype=np.float64)
    S = oracle.factor(x, 1.0 / 3)
    rows, d = x.shape
    for i in range(d):
        for j in range(d):
            acc = 0.0
            for k in range(rows):
                acc += x[k, i] * x[k, j]
            assert S[i, j] == pytest.approx(acc / 3, rel=0, abs=1e-15)
    # an x x^T slip (rows x rows) or a missing scale cannot pass
    assert S.shape == (d, d)


def test_factor_symmetric_psd():
    x = rnd(37, 21)
    S = oracle.factor(x, 1 / 37)
    assert np.array_equal(S, S.T)
    assert np.linalg.eigvalsh(S).min() >= -1e-12 * np.abs(S).max()


@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_shard_mean_equals_full_batch(P):
    # D-KFAC aggregation: the mean of P equal-shard factors is the full-batch factor
    x = rnd(64, 17, seed=P)
    full = oracle.factor(x, 1 / 64)
    agg = oracle.aggregate(oracle.shard_factors(x, P))
    assert np.abs(agg - full).max() <= 1e-14 * np.abs(full).max()
    with pytest.raises(ValueError):
        oracle.shard_factors(x[:63], 2)


def test_shard_factor_uses_its_own_rows():
    x = np.zeros((4, 2))
    x[0] = [1, 0]
    x[3] = [0, 2]
    s0, s1 = oracle.shard_factors(x, 2)
    assert np.array_equal(s0, np.array([[0.5, 0], [0, 0]]))
    assert np.array_equal(s1, np.array([[0, 0], [0, 2.0]]))


# ------------------------------------------------------------------ running average + damping
def test_running_average_closed_form():
    xi = 0.95
    Fs = [np.array([[float(t * t + 1)]]) for t in range(1, 11)]
    R = None
    for t, F in enumerate(Fs, start=1):
        R = oracle.update_running(F, R, xi, first_step=(t == 1))
        # solution of the recurrence: xi^(t-1) F_1 + (1-xi) sum_{s=2..t} xi^(t-s) F_s
        closed = xi ** (t - 1) * Fs[0][0, 0] + (1 - xi) * sum(
            xi ** (t - s) * Fs[s - 1][0, 0] for s in range(2, t + 1))
        assert R[0, 0] == pytest.approx(closed, rel=1e-14)


def test_running_average_fixed_point_and_first_step():
    F = rnd(5, 5)
    F = F + F.T
    R = oracle.update_running(F, None, 0.9, True)
    assert np.array_equal(R, F) and R is not F
    for _ in range(5):
        R = oracle.update_running(F, R, 0.9, False)
    assert np.abs(R - F).max() <= 1e-14 * np.abs(F).max()
    # decay weights the OLD value
    R2 = oracle.update_running(np.zeros((5, 5)), F, 0.9, False)
    assert np.abs(R2 - 0.9 * F).max() <= 1e-15 * np.abs(F).max()


def test_running_average_checkpoint_resume():
    Fs = [rnd(6, 6, seed=s) for s in range(10)]
    R = None
    for t, F in enumerate(Fs):
        R = oracle.update_running(F, R, 0.95, t == 0)
    Rh = None
    for t, F in enumerate(Fs[:5]):
        Rh = oracle.update_running(F, Rh, 0.95, t == 0)
    saved = Rh.copy()
    for F in Fs[5:]:
        saved = oracle.update_running(F, saved, 0.95, False)
    assert np.array_equal(saved, R)


def test_damp_adds_gamma_to_diagonal_only_on_a_copy():
    R = rnd(4, 4)
    R0 = R.copy()
    D = oracle.damp(R, 0.25)
    assert np.array_equal(R, R0)
    assert np.array_equal(D - np.diag(np.diag(D)), R - np.diag(np.diag(R)))
    assert np.allclose(np.diag(D) - np.diag(R), 0.25, rtol=0, atol=1e-15)


# ------------------------------------------------------------------ Cholesky / inverse
def spd(n, seed=0, gamma=1e-2):
    x = rnd(n + 3, n, seed=seed)
    return x.T @ x / (n + 3) + gamma * np.eye(n)


def test_cholesky_2x2_closed_form():
    a, b, c = 4.0, 2.0, 5.0
    L, info = oracle.cholesky_lower(np.array([[a, b], [b, c]]))
    assert info == 0
    assert np.allclose(L, [[2.0, 0.0], [1.0, 2.0]], rtol=0, atol=1e-15)


@pytest.mark.parametrize("n", [1, 7, 64, 129])
def test_cholesky_reconstructs_and_matches_lapack(n):
    D = spd(n, seed=n)
    L, info = oracle.cholesky_lower(D)
    assert info == 0
    assert np.array_equal(np.triu(L, 1), np.zeros_like(L))
    assert (np.diag(L) > 0).all()
    assert np.abs(L @ L.T - D).max() <= 1e-13 * np.abs(D).max()
    assert np.abs(L - np.linalg.cholesky(D)).max() <= 1e-12 * np.abs(L).max()


def test_cholesky_reports_first_bad_pivot():
    assert oracle.cholesky_lower(np.diag([1.0, -1.0]))[1] == 2
    # leading 2x2 minor is singular: [[1,1],[1,1]]
    D = np.array([[1.0, 1.0, 0], [1.0, 1.0, 0], [0, 0, 1.0]])
    assert oracle.cholesky_lower(D)[1] == 2
    D = spd(5)
    D[3, 3] = np.nan
    assert oracle.cholesky_lower(D)[1] == 4
    assert oracle.spd_inverse(np.diag([2.0, 0.0, 1.0]))[1] == 2


def test_lower_tri_inverse_closed_form():
    # L = I - (subdiagonal ones)  =>  L^-1 = lower-triangular matrix of ones
    n = 9
    L = np.eye(n) - np.eye(n, k=-1)
    W = oracle.lower_tri_inverse(L)
    assert np.array_equal(W, np.tril(np.ones((n, n))))
    L = np.tril(rnd(30, 30)) + 6 * np.eye(30)
    W = oracle.lower_tri_inverse(L)
    ref = scipy.linalg.solve_triangular(L, np.eye(30), lower=True)
    assert np.abs(W - ref).max() <= 1e-13 * np.abs(ref).max()


def test_spd_inverse_sherman_morrison():
    # D = gamma I + c 1 1^T  =>  D^-1 = (I - c/(gamma + n c) 1 1^T)/gamma
    n, gamma, c = 50, 1e-3, 0.3
    D = gamma * np.eye(n) + c * np.ones((n, n))
    X, info = oracle.spd_inverse(D)
    ref = (np.eye(n) - c / (gamma + n * c) * np.ones((n, n))) / gamma
    assert info == 0
    assert np.abs(X - ref).max() <= 1e-9 * np.abs(ref).max()


def test_spd_inverse_hilbert_exact():
    n = 6
    H = scipy.linalg.hilbert(n)
    X, info = oracle.spd_inverse(H)
    ref = scipy.linalg.invhilbert(n, exact=True).astype(np.float64)
    assert info == 0
    assert np.abs(X - ref).max() <= 1e-6 * np.abs(ref).max()


@pytest.mark.parametrize("n", [3, 65, 200])
def test_spd_inverse_identity_symmetry_and_numpy(n):
    D = spd(n, seed=3 * n)
    X, info = oracle.spd_inverse(D)
    assert info == 0
    assert np.array_equal(X, X.T)
    assert np.linalg.norm(X @ D - np.eye(n)) / math.sqrt(n) <= 1e-11
    ref = np.linalg.inv(D)
    assert np.abs(X - ref).max() <= 1e-10 * np.abs(ref).max()


def test_damped_inverse_adds_gamma():
    D = spd(10)
    X, _ = oracle.damped_inverse(D, 0.5)
    assert np.abs(X - np.linalg.inv(D + 0.5 * np.eye(10))).max() < 1e-12


# ------------------------------------------------------------------ preconditioning
@pytest.mark.parametrize("d_in,d_out", [(4, 3), (6, 5), (65, 32)])
def test_precondition_equals_bruteforce_kronecker(d_in, d_out):
    gamma = 0.03
    a = rnd(40, d_in, seed=d_in)
    g = rnd(40, d_out, seed=d_out) * 0.1
    A, G = oracle.factor(a, 1 / 40), oracle.factor(g, 1 / 40)
    grad = g.T @ a / 40
    XA, _ = oracle.spd_inverse(oracle.damp(A, gamma))
    XG, _ = oracle.spd_inverse(oracle.damp(G, gamma))
    V = oracle.precondition(XG, grad, XA)
    Vb = oracle.kron_precondition_bruteforce(A, G, grad, gamma)
    assert np.abs(V - Vb).max() <= 1e-10 * np.abs(Vb).max()
    # damping the Kronecker product as a whole is a different operator
    K = np.kron(A, G) + gamma * np.eye(d_in * d_out)
    Vw = np.linalg.solve(K, grad.reshape(-1, order="F")).reshape(grad.shape, order="F")
    assert np.abs(Vw - Vb).max() > 1e-3 * np.abs(Vb).max()
    # the transposed layer (d_in x d_out gradient) is preconditioned by the swapped factors
    assert np.abs(XA @ grad.T @ XG - V.T).max() < 1e-9 * np.abs(V).max()


def test_weight_step_values_and_quadratic_minimiser():
    # the step itself, by hand
    W = np.array([[1.0, -2.0], [0.5, 4.0]])
    V = np.array([[0.25, 1.0], [-2.0, 0.0]])
    assert np.array_equal(oracle.weight_step(W, V, 0.5), np.array([[0.875, -2.5], [1.5, 4.0]]))
    # f(W) = 1/2 <W, G W A> - <B, W> has curvature exactly A (x) G and gradient
    # G W A - B: one damped K-FAC step with lr = 1 from any W lands on the
    # minimiser G^-1 B A^-1 as gamma -> 0
    A, G = spd(5, seed=11), spd(4, seed=12)
    B = rnd(4, 5, seed=13)
    W0 = rnd(4, 5, seed=14)
    grad = G @ W0 @ A - B
    XA, _ = oracle.spd_inverse(oracle.damp(A, 1e-12))
    XG, _ = oracle.spd_inverse(oracle.damp(G, 1e-12))
    W1 = oracle.weight_step(W0, oracle.precondition(XG, grad, XA), 1.0)
    assert np.abs(G @ W1 @ A - B).max() <= 1e-8 * np.abs(B).max()
    # with damping the step is shorter along every direction: f decreases, not to the minimum
    XA, _ = oracle.spd_inverse(oracle.damp(A, 0.5))
    XG, _ = oracle.spd_inverse(oracle.damp(G, 0.5))
    W2 = oracle.weight_step(W0, oracle.precondition(XG, grad, XA), 1.0)
    f = lambda W: 0.5 * np.sum(W * (G @ W @ A)) - np.sum(B * W)
    assert f(W1) < f(W2) < f(W0)


def test_precondition_self_adjoint_and_linear():
    # adjoint test <P(U), V> = <U, P(V)> for the symmetric map P(V) = XG V XA
    XG, _ = oracle.spd_inverse(spd(7, seed=1))
    XA, _ = oracle.spd_inverse(spd(9, seed=2))
    U, V = rnd(7, 9, seed=3), rnd(7, 9, seed=4)
    lhs = np.sum(oracle.precondition(XG, U, XA) * V)
    rhs = np.sum(U * oracle.precondition(XG, V, XA))
    assert lhs == pytest.approx(rhs, rel=1e-12)
    comb = oracle.precondition(XG, 2.0 * U - 3.0 * V, XA)
    sep = 2.0 * oracle.precondition(XG, U, XA) - 3.0 * oracle.precondition(XG, V, XA)
    assert np.abs(comb - sep).max() <= 1e-12 * np.abs(sep).max()


# ------------------------------------------------------------------ conv helper
def test_spatial_sum_loops():
    B, hw, C = 3, 4, 5
    g = rnd(B * hw, C)
    gs = oracle.spatial_sum(g, B, hw)
    for b in range(B):
        for c in range(C):
            assert gs[b, c] == pytest.approx(sum(g[b * hw + s, c] for s in range(hw)), abs=1e-14)


# ------------------------------------------------------------------ index maps
@pytest.mark.parametrize("d", [1, 10, 127, 128, 129, 256, 385, 1025])
def test_factor_tile_units_cover_upper_tiles_once(d):
    bm, bn = 128, 256
    units = oracle.factor_tile_units(d, bm, bn)
    seen = np.zeros((d, d), dtype=np.int32)
    for u in units:
        i, j0, w = u
        assert 1 <= w <= bn and j0 % bn == 0 and j0 + w <= d
        # what a unit computes but drops: at most its first bm columns (the
        # lower tile of the pair's second row block), or all of a stand-in
        (r0, r1), (c0, c1) = oracle.stored_part(u, d, bm)
        assert c0 - j0 in (0, bm) or r0 >= d
        seen[r0:r1, c0:c1] += 1
    r = np.arange(d)[:, None]
    c = np.arange(d)[None, :]
    want = (c >= (r // bm) * bm).astype(np.int32)
    assert np.array_equal(seen, want)
    # units come in pairs of row blocks (2s, 2s+1) sharing their columns,
    # ordered by pair, then column
    assert all(units[2 * k][0] + 1 == units[2 * k + 1][0] and units[2 * k][0] % 2 == 0
               and units[2 * k][1:] == units[2 * k + 1][1:] for k in range(len(units) // 2))
    assert units[0::2] == sorted(units[0::2])


def test_im2col3x3_by_loops_and_as_convolution():
    rng = np.random.default_rng(31)
    B, H, W, C, Co = 2, 4, 5, 3, 2
    x = rng.standard_normal((B, H, W, C))
    P = oracle.im2col3x3(x)
    assert P.shape == (B * H * W, 9 * C + 1)
    # entry by entry against nested loops over the padded image
    for b in range(B):
        for h in range(H):
            for w in range(W):
                r = (b * H + h) * W + w
                for dh in range(3):
                    for dw in range(3):
                        for c in range(C):
                            hh, ww = h + dh - 1, w + dw - 1
                            v = x[b, hh, ww, c] if 0 <= hh < H and 0 <= ww < W else 0.0
                            assert P[r, (dh * 3 + dw) * C + c] == v
                assert P[r, -1] == 1.0
    # patches times the flattened kernel is the convolution (cross-correlation)
    K = rng.standard_normal((Co, 3, 3, C))
    bias = rng.standard_normal(Co)
    out = P @ np.concatenate([K.reshape(Co, 9 * C), bias[:, None]], axis=1).T
    for b in range(B):
        for h in range(H):
            for w in range(W):
                for o in range(Co):
                    acc = bias[o]
                    for dh in range(3):
                        for dw in range(3):
                            hh, ww = h + dh - 1, w + dw - 1
                            if 0 <= hh < H and 0 <= ww < W:
                                acc += K[o, dh, dw] @ x[b, hh, ww]
                    assert abs(out[(b * H + h) * W + w, o] - acc) <= 1e-12
    # an interior position sees all nine taps, a corner four
    assert np.count_nonzero(P[(0 * H + 1) * W + 1, :-1]) == 9 * C
    assert np.count_nonzero(P[0, :-1]) == 4 * C


@pytest.mark.parametrize("d", [1, 5, 128, 300])
def test_upper_tiles_count(d):
    T = -(-d // 128)
    t = oracle.upper_tiles(d)
    assert len(t) == T * (T + 1) // 2
    assert t == [(i, j) for i in range(T) for j in range(T) if i <= j]


def test_packed_index_enumeration():
    for d in (1, 2, 7, 33):
        k = 0
        for i in range(d):
            for j in range(i, d):
                assert oracle.packed_index(i, j, d) == k
                k += 1
        assert k == d * (d + 1) // 2
    with pytest.raises(ValueError):
        oracle.packed_index(2, 1, 4)


def test_pack_upper_follows_the_enumerated_index_and_round_trips():
    rng = np.random.default_rng(3)
    for d in (1, 2, 5, 33):
        M = rng.standard_normal((d, d))
        M = M + M.T
        p = oracle.pack_upper(M)
        assert p.shape == (d * (d + 1) // 2,)
        for i in range(d):
            for j in range(i, d):
                assert p[oracle.packed_index(i, j, d)] == M[i, j]
        assert np.array_equal(oracle.unpack_upper(p, d), M)
        U = oracle.unpack_upper(p, d, mirror=False)
        assert np.array_equal(np.triu(U), np.triu(M)) and np.isnan(U[np.tril_indices(d, -1)]).all()
    # the packed form holds exactly the upper triangle: an asymmetric matrix
    # packs its upper part only, so unpacking gives the symmetrised upper part
    A = np.arange(16.0).reshape(4, 4)
    assert list(oracle.pack_upper(A)) == [0, 1, 2, 3, 5, 6, 7, 10, 11, 15]
    assert np.array_equal(oracle.unpack_upper(oracle.pack_upper(A), 4), np.triu(A) + np.triu(A, 1).T)
    with pytest.raises(ValueError):
        oracle.unpack_upper(np.zeros(5), 3)


# ------------------------------------------------------------------ page pin: ResNet-50 sizes
def _resnet50_layers():
    """(kernel, C_in, C_out) of the 53 convolutions of ResNet-50, then the fc."""
    layers = [(7, 3, 64)]
    c_in = 64
    for planes, blocks in ((64, 3), (128, 4), (256, 6), (512, 3)):
        for b in range(blocks):
            layers += [(1, c_in, planes), (3, planes, planes), (1, planes, 4 * planes)]
            if b == 0:
                layers.append((1, c_in, 4 * planes))
            c_in = 4 * planes
    return layers


def _golden(name):
    vals = {}
    with open(os.path.join(HERE, "golden", name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    return vals


def test_resnet50_factor_sizes_match_page():
    gold = _golden("resnet50_factor_counts.txt")
    convs = _resnet50_layers()
    assert len(convs) == 53
    tri = lambda d: d * (d + 1) // 2
    # conv factors: A dim = k*k*C_in (no bias column), G dim = C_out; fc 2048 -> 1000
    dA = [k * k * ci for k, ci, co in convs] + [2048]
    dG = [co for k, ci, co in convs] + [1000]
    params = sum(k * k * ci * co + 2 * co for k, ci, co in convs) + 2048 * 1000 + 1000
    trunc = lambda v: math.floor(v / 1e5) / 10
    assert trunc(params) == gold["params_millions"]
    assert trunc(sum(map(tri, dA))) == gold["factor_A_upper_elements_millions"]
    assert trunc(sum(map(tri, dG))) == gold["factor_G_upper_elements_millions"]
    assert min(map(tri, dA + dG)) == gold["min_factor_upper_elements"]
    assert max(map(tri, dA + dG)) == gold["max_factor_upper_elements"]
    # the resnet_conv workload uses exactly these 3x3 conv shapes (+1 bias column)
    cfg = synth.config("resnet_conv")
    threes = sorted({(ci, co) for k, ci, co in convs if k == 3})
    assert [(l.d_in - 1) // 9 for l in cfg.layers] == [c for c, _ in threes]


# ------------------------------------------------------------------ whole step on a tiny layer
def test_kfac_step_single_linear_matches_bruteforce():
    cfg = synth.config("single_linear")
    data = synth.layer_inputs(cfg, 0, 0)
    (res,) = oracle.kfac_step([data], cfg.P, cfg.gamma, 0.0, True)
    a = data["a"].astype(np.float64)
    g = data["g"].astype(np.float64)
    A = a.T @ a / cfg.batch
    G = g.T @ g / cfg.batch
    Vb = oracle.kron_precondition_bruteforce(A, G, data["grad"], cfg.gamma)
    assert np.abs(res["V"] - Vb).max() <= 1e-9 * np.abs(Vb).max()
    assert res["info"] == (0, 0)


def test_inputs_are_seeded_and_bf16_exact():
    cfg = synth.config("mlp")
    d1 = synth.layer_inputs(cfg, 2, 1)
    d2 = synth.layer_inputs(cfg, 2, 1)
    assert np.array_equal(d1["a"], d2["a"]) and np.array_equal(d1["g"], d2["g"])
    assert np.array_equal(synth.round_bf16(d1["a"]), d1["a"])
    assert (d1["a"][:, -1] == 1).all() and (d1["a"][:, :-1] >= 0).all()
    d3 = synth.layer_inputs(cfg, 3, 1)
    assert not np.array_equal(d1["g"], d3["g"])
