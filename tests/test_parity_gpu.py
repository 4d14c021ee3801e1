"""GPU parity: every stage of the CUDA path against the fp64 oracle on the same
seeded inputs, through the C ABI.

Tolerances (stated by the step's specification): factors <= 1e-5 relative
Frobenius; running average / damping <= 1e-6 (a few fp32 roundings of a
closed form); inverses ||X D - I||_F / sqrt(n) <= 1e-3 and <= 1e-3 relative to
the oracle's inverse of the same fp32 damped factor; preconditioned gradient
<= 2e-3 relative Frobenius, oracle fed the GPU's inverses and gradient.
Sentinels (NaN) in lower tiles and padding catch stray reads and writes."""
import numpy as np
import pytest
import torch

import oracle
import synth
from infra_fac_factors_gb300 import capi
from infra_fac_factors_gb300.step import KFACStep, LayerSpec

from gpu_util import (ensure_built, pad, rel_fro, residual, stream, to_dev, upper_from_full,
                      upper_tile_mask)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    ensure_built()
    torch.cuda.init()


def sync():
    torch.cuda.synchronize()
    assert capi.kfac_device_status(clear=True) == capi.KFAC_OK


# ------------------------------------------------------------------ a1/a2: factors
def run_factors(x, P, dtype, mirror=0, ld_extra=0):
    rows, d = x.shape
    ldx = pad(d, 8 if dtype == capi.KFAC_BF16 else 4)
    xt = to_dev(x, dtype, ldx)
    ldo = pad(d, 4) + ld_extra
    out = torch.full((P, d, ldo), float("nan"), dtype=torch.float32, device="cuda")
    rp = rows // P
    capi.kfac_factors([capi.kfac_factor_args(xt.data_ptr(), rows, d, ldx, out.data_ptr(), ldo, d * ldo, 1.0 / rp)],
                      dtype, P, mirror, stream())
    sync()
    return out.cpu().numpy()


@pytest.mark.parametrize("d,rows_p,P", [
    (10, 64, 1), (65, 100, 2), (128, 64, 1), (129, 37, 3), (256, 1, 2), (300, 200, 2),
    (513, 64, 4), (700, 300, 1), (1025, 128, 2),
])
def test_factors_bf16_tensor_cores(d, rows_p, P):
    rng = np.random.default_rng(d * 1000 + rows_p)
    x = synth.round_bf16(rng.standard_normal((rows_p * P, d)).astype(np.float32))
    res = run_factors(x, P, capi.KFAC_BF16, ld_extra=4)
    m = upper_tile_mask(d)
    for p in range(P):
        ref = oracle.factor(x[p * rows_p:(p + 1) * rows_p], 1.0 / rows_p)
        got = res[p][:, :d]
        assert rel_fro(got, ref, m) <= 1e-5, (p, rel_fro(got, ref, m))
        assert np.isnan(got[~m]).all(), "lower tiles must stay untouched"
        assert np.isnan(res[p][:, d:]).all(), "padding must stay untouched"


def test_factors_bf16_mirror_gives_full_symmetric():
    rng = np.random.default_rng(7)
    d, rp, P = 300, 96, 2
    x = synth.round_bf16(rng.standard_normal((rp * P, d)).astype(np.float32))
    res = run_factors(x, P, capi.KFAC_BF16, mirror=1)
    for p in range(P):
        got = res[p][:, :d]
        ref = oracle.factor(x[p * rp:(p + 1) * rp], 1.0 / rp)
        assert not np.isnan(got).any()
        assert rel_fro(got, ref) <= 1e-5
        assert np.abs(got - got.T).max() <= 1e-6 * np.abs(got).max()


def test_factors_bf16_single_worker_row_tail_and_structure():
    # rows not a multiple of the 64-row stage and ReLU-like non-negative data (large mean)
    rng = np.random.default_rng(11)
    d, rows = 577, 196
    x = synth.round_bf16(np.maximum(rng.standard_normal((rows * 2, d)), 0).astype(np.float32))
    x[:, -1] = 1.0
    res = run_factors(x, 2, capi.KFAC_BF16)
    m = upper_tile_mask(d)
    for p in range(2):
        ref = oracle.factor(x[p * rows:(p + 1) * rows], 1.0 / rows)
        assert rel_fro(res[p][:, :d], ref, m) <= 1e-5


@pytest.mark.parametrize("d,rows_p,P", [(65, 128, 1), (32, 128, 1), (200, 4, 8), (130, 33, 2)])
def test_factors_fp32_cuda_cores(d, rows_p, P):
    rng = np.random.default_rng(d + rows_p)
    x = rng.standard_normal((rows_p * P, d)).astype(np.float32)
    res = run_factors(x, P, capi.KFAC_FP32)
    m = upper_tile_mask(d)
    for p in range(P):
        ref = oracle.factor(x[p * rows_p:(p + 1) * rows_p], 1.0 / rows_p)
        assert rel_fro(res[p][:, :d], ref, m) <= 1e-5
        assert np.isnan(res[p][:, :d][~m]).all()


def test_spatial_sum():
    rng = np.random.default_rng(3)
    B, hw, C = 6, 49, 130
    g = synth.round_bf16((rng.standard_normal((B * hw, C)) * 1e-3).astype(np.float32))
    ldg = pad(C, 8)
    gt = to_dev(g, capi.KFAC_BF16, ldg)
    ldgs = pad(C, 4)
    gs = torch.full((B, ldgs), float("nan"), device="cuda")
    capi.kfac_spatial_sum(gt.data_ptr(), capi.KFAC_BF16, B, hw, C, ldg, gs.data_ptr(), ldgs, stream())
    sync()
    ref = oracle.spatial_sum(g, B, hw)
    got = gs.cpu().numpy()[:, :C]
    assert rel_fro(got, ref) <= 1e-6


# ------------------------------------------------------------------ a3: reduce + running average + damping
@pytest.mark.parametrize("d,P", [(10, 4), (129, 8), (300, 3), (1025, 2)])
def test_update_running_three_steps(d, P):
    rng = np.random.default_rng(d * 10 + P)
    ld = pad(d, 4) + 4
    stride = d * ld
    m = upper_tile_mask(d)
    shards = torch.full((P, d, ld), float("nan"), device="cuda")
    running = torch.full((d, ld), float("nan"), device="cuda")
    damped = torch.full((d, ld), float("nan"), device="cuda")
    decay, gamma = 0.95, 1e-3
    R = None
    for t in range(3):
        S = [rng.standard_normal((d, d)).astype(np.float32) for _ in range(P)]
        host = np.full((P, d, ld), np.nan, dtype=np.float32)
        for p in range(P):
            host[p, :, :d][m] = S[p][m]
        shards.copy_(torch.from_numpy(host))
        args = [capi.kfac_running_args(shards.data_ptr(), stride, running.data_ptr(), damped.data_ptr(), d, ld)]
        capi.kfac_update_running(args, P, decay, gamma, t == 0, stream())
        sync()
        F = oracle.aggregate([s.astype(np.float64) for s in S])
        R = oracle.update_running(F, R, decay, t == 0)
        Dref = oracle.damp(R, gamma)
        got_R = running.cpu().numpy()
        got_D = damped.cpu().numpy()
        assert rel_fro(got_R[:, :d], R, m) <= 1e-6
        assert rel_fro(got_D[:, :d], Dref, m) <= 1e-6
        assert np.isnan(got_R[:, :d][~m]).all() and np.isnan(got_D[:, :d][~m]).all()
        assert np.isnan(got_D[:, d:]).all()
        R = got_R[:, :d].astype(np.float64)  # continue from the GPU's state (stage-wise)
        R[~m] = 0.0


# ------------------------------------------------------------------ a4: damped inverse
def spd_case(d, rng, gamma=1e-2, rows=None, relu=False):
    rows = rows or d + 16
    x = rng.standard_normal((rows, d))
    if relu:
        x = np.maximum(x, 0)
    return (x.T @ x / rows + gamma * np.eye(d)).astype(np.float32)


def run_inverse(Ds, refine, gamma_extra=0.0):
    bufs, outs, args = [], [], []
    for D in Ds:
        d = D.shape[0]
        ld = pad(d, 4) + 4
        host = np.full((d, ld), np.nan, dtype=np.float32)
        iu = np.triu_indices(d)
        host[iu] = D[iu]
        b = torch.from_numpy(host).cuda()
        o = torch.full((d, ld), float("nan"), device="cuda")
        bufs.append(b)
        outs.append(o)
        args.append(capi.kfac_inverse_args(b.data_ptr(), o.data_ptr(), d, ld, ld))
    n = len(Ds)
    info = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    route = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    wsb = capi.kfac_damped_inverse_workspace(args, refine)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    capi.kfac_damped_inverse(args, gamma_extra, refine, info.data_ptr(), route.data_ptr(), ws.data_ptr(), wsb,
                             stream())
    sync()
    return [o.cpu().numpy()[:, :D.shape[0]] for o, D in zip(outs, Ds)], info.cpu().numpy(), route.cpu().numpy()


SIZES = [1, 5, 64, 127, 128, 129, 300, 385]


@pytest.mark.parametrize("refine", [capi.KFAC_REFINE_NONE, capi.KFAC_REFINE_AUTO, capi.KFAC_REFINE_ALWAYS])
def test_damped_inverse_batched_variable_sizes(refine):
    rng = np.random.default_rng(100 + refine)
    Ds = [spd_case(d, rng) for d in SIZES]
    Xs, info, route = run_inverse(Ds, refine)
    assert (info == 0).all()
    if refine == capi.KFAC_REFINE_AUTO:
        assert set(route.tolist()) <= {0, 1, 2}, route
    else:
        assert (route == (1 if refine == capi.KFAC_REFINE_ALWAYS else 0)).all(), route
    for D, X in zip(Ds, Xs):
        ref, i = oracle.spd_inverse(D.astype(np.float64))
        assert i == 0
        assert np.array_equal(X, X.T), "inverse must be exactly symmetric"
        assert rel_fro(X, ref) <= 1e-3
        assert residual(X, D) <= 1e-3
        if refine == capi.KFAC_REFINE_ALWAYS:
            assert rel_fro(X, ref) <= 1e-6


def test_damped_inverse_gamma_extra():
    rng = np.random.default_rng(5)
    D = spd_case(200, rng)
    (X,), info, _ = run_inverse([D], capi.KFAC_REFINE_NONE, gamma_extra=0.5)
    ref, _ = oracle.damped_inverse(D.astype(np.float64), 0.5)
    assert info[0] == 0 and rel_fro(X, ref) <= 1e-5


def test_damped_inverse_auto_sends_ill_conditioned_away_from_the_fp32_pass():
    rng = np.random.default_rng(9)
    # rank-deficient ReLU factor (rows < d) with tiny damping: kappa ~ 1e6; AUTO
    # does not keep its fp32 result: the tensor-core Newton step (route 3) or,
    # failing that, the fp64 pass (route 1) gives it
    D_bad = spd_case(640, rng, gamma=1e-4, rows=200, relu=True)
    D_ok = spd_case(200, rng)
    Xs, info, route = run_inverse([D_bad, D_ok], capi.KFAC_REFINE_AUTO)
    assert list(info) == [0, 0]
    assert route[0] in (1, 3) and route[1] == 0, route
    for D, X in zip((D_bad, D_ok), Xs):
        ref, _ = oracle.spd_inverse(D.astype(np.float64))
        assert rel_fro(X, ref) <= 1e-3
        assert residual(X, D) <= 1e-3
        assert np.array_equal(X, X.T)


def conv_like_factor(d, rows, gamma, rng):
    """A damped factor shaped like a conv layer's A: ReLU patches with a ones
    column, rows < d (rank-deficient), so kappa ~ max eigenvalue / gamma."""
    a = np.maximum(rng.standard_normal((rows, d)), 0.0)
    a[:, -1] = 1.0
    a = synth.round_bf16(a.astype(np.float32)).astype(np.float64)
    return (a.T @ a / rows + gamma * np.eye(d)).astype(np.float32)


@pytest.mark.parametrize("d,rows", [(385, 200), (1153, 784), (2305, 1024)])
def test_damped_inverse_newton_step_on_tensor_cores(d, rows):
    # kappa ~ 1e5 .. 1e6: the fp32 pass alone misses the AUTO bar; one Newton
    # step with the residual formed exactly (error-free slices on tensor cores)
    # lands at the fp32 storage floor of the inverse
    rng = np.random.default_rng(d)
    D = conv_like_factor(d, rows, 1e-3, rng)
    (X,), info, route = run_inverse([D], capi.KFAC_REFINE_AUTO)
    (X32,), _, _ = run_inverse([D], capi.KFAC_REFINE_NONE)
    Dd = D.astype(np.float64)
    ref, _ = oracle.spd_inverse(Dd)
    assert info[0] == 0
    r32, r = residual(X32, Dd), residual(X, Dd)
    assert route[0] == 3, (route, r32)  # settled on tensor cores, not by the fp64 pass
    assert np.array_equal(X, X.T)
    assert r <= 1e-3 and rel_fro(X, ref) <= 1e-3, (r, rel_fro(X, ref))
    # the step gains what fp32 storage allows: the residual drops below the
    # fp32 pass's and the error against the oracle far below it
    assert r <= 5e-4 and r < r32, (r, r32)
    assert rel_fro(X, ref) <= 0.1 * rel_fro(X32, ref), (rel_fro(X, ref), rel_fro(X32, ref))


def test_newton_step_matrices_among_well_conditioned_ones():
    # candidates and the rest in one batch: only the candidates change
    rng = np.random.default_rng(77)
    Ds = [spd_case(300, rng), conv_like_factor(577, 300, 1e-3, rng), spd_case(129, rng),
          conv_like_factor(1025, 600, 1e-3, rng)]
    Xs, info, route = run_inverse(Ds, capi.KFAC_REFINE_AUTO)
    Xn, _, _ = run_inverse(Ds, capi.KFAC_REFINE_NONE)
    assert (info == 0).all()
    for D, X, X24, r in zip(Ds, Xs, Xn, route):
        ref, _ = oracle.spd_inverse(D.astype(np.float64))
        assert rel_fro(X, ref) <= 1e-3 and residual(X, D) <= 1e-3, (D.shape, r)
        if r == 0:
            assert np.array_equal(X, X24)
    assert route[0] == 0 and route[2] == 0 and route[1] == 3 and route[3] == 3, route


def gershgorin_ratio(D):
    D = np.asarray(D, np.float64)
    off = np.abs(D).sum(1) - np.abs(np.diag(D))
    lo, hi = (np.diag(D) - off).min(), (np.diag(D) + off).max()
    return hi / lo if lo > 0 else np.inf


def test_damped_inverse_auto_takes_16bit_operands_when_gershgorin_allows():
    # AUTO runs the fp32 pass with two-slice (16-bit) operands for a matrix whose
    # Gershgorin discs bound its condition number by 16, and with three slices
    # otherwise; the residual probe still checks both
    rng = np.random.default_rng(31)
    cases = []
    for d in (1, 130, 640, 1025):  # G-like: gamma I plus a tiny factor (kappa ~ 1)
        g = rng.standard_normal((256, d)) * 1e-4
        cases.append(((g.T @ g / 256) + 1e-3 * np.eye(d)).astype(np.float32))
    for scale, d in ((0.6, 300), (0.88, 300), (0.95, 300)):  # diagonally dominant: bounds ~4, ~15.7, ~39
        M = rng.standard_normal((d, d))
        M = (M + M.T) / 2
        np.fill_diagonal(M, 0.0)
        M *= scale / np.abs(M).sum(1).max()
        cases.append((np.eye(d) + M).astype(np.float32))
    cases.append(spd_case(257, rng))  # Wishart with rows ~ d: no Gershgorin bound
    want = [2 if gershgorin_ratio(D) <= 16 else 0 for D in cases]
    assert want == [2, 2, 2, 2, 2, 2, 0, 0]
    Xs, info, route = run_inverse(cases, capi.KFAC_REFINE_AUTO)
    assert (info == 0).all()
    assert list(route) == want, route
    Xn, _, route_n = run_inverse(cases, capi.KFAC_REFINE_NONE)
    assert (route_n == 0).all()  # NONE keeps 24-bit operands for every matrix
    for D, X, X24, r in zip(cases, Xs, Xn, route):
        ref, _ = oracle.spd_inverse(D.astype(np.float64))
        assert np.array_equal(X, X.T)
        if r == 2:
            assert rel_fro(X, ref) <= 1e-4 and residual(X, D) <= 1e-4, (D.shape, rel_fro(X, ref), residual(X, D))
        else:
            assert np.array_equal(X, X24)  # the 24-bit route is the NONE pass, bit for bit
            assert rel_fro(X, ref) <= 1e-3 and residual(X, D) <= 1e-3


def test_auto_refinement_graph_matches_direct_launches():
    # AUTO runs its Newton step and its fp64 pass from a cached CUDA graph whose
    # IF nodes skip them when nothing is flagged; while the launch profile
    # records, the same passes are launched one by one.  Both give the same
    # bits, with nothing flagged, with a matrix the Newton step settles, and
    # with one that goes on to the fp64 pass (a negative pivot fails there too).
    rng = np.random.default_rng(77)
    bad = spd_case(300, rng)
    bad[200, 200] = -1.0
    newton = conv_like_factor(385, 200, 1e-3, rng)
    ok = spd_case(200, rng)
    for batch in ([ok], [bad, newton, ok]):
        capi.kfac_profile(1)
        try:
            Xp, infop, routep = run_inverse(batch, capi.KFAC_REFINE_AUTO)
        finally:
            capi.kfac_profile(0)
        Xg, infog, routeg = run_inverse(batch, capi.KFAC_REFINE_AUTO)
        Xg2, infog2, routeg2 = run_inverse(batch, capi.KFAC_REFINE_AUTO)  # the graph again, built once
        assert list(infop) == list(infog) == list(infog2)
        assert list(routep) == list(routeg) == list(routeg2)
        for a, b, c, i in zip(Xp, Xg, Xg2, infop):
            if i == 0:
                assert np.array_equal(a, b) and np.array_equal(b, c)
    assert list(routep) == [1, 3, 0] and infop[0] > 0 and infop[1] == 0 and infop[2] == 0, (routep, infop)


def test_damped_inverse_reports_first_bad_pivot():
    rng = np.random.default_rng(4)
    D = spd_case(300, rng)
    D[200, 200] = -1.0
    D2 = spd_case(20, rng)
    for refine in (capi.KFAC_REFINE_NONE, capi.KFAC_REFINE_AUTO, capi.KFAC_REFINE_ALWAYS):
        Xs, info, route = run_inverse([D, D2], refine)
        _, want = oracle.cholesky_lower(D.astype(np.float64))
        assert want > 0
        assert info[0] == want, (refine, info)
        assert info[1] == 0
        ref, _ = oracle.spd_inverse(D2.astype(np.float64))
        assert rel_fro(Xs[1], ref) <= 1e-3
    # a NaN in the factor is a failed pivot too
    D3 = spd_case(150, rng)
    D3[140, 140] = np.nan
    _, info, _ = run_inverse([D3], capi.KFAC_REFINE_NONE)
    assert info[0] == 141


# ------------------------------------------------------------------ a5: precondition
def run_precondition(XG, grad, XA, precision=capi.KFAC_PRECOND_FP32, with_route=False, weight=None, lr=0.0):
    """out (and with `weight`: the stepped weights) of one layer's call."""
    d_out, d_in = grad.shape
    ldg, lda, ldw, ldo = pad(d_out, 4), pad(d_in, 4) + 4, pad(d_in, 4), pad(d_in, 4) + 8
    tg = to_dev(XG, capi.KFAC_FP32, ldg)
    ta = to_dev(XA, capi.KFAC_FP32, lda)
    tw = to_dev(grad, capi.KFAC_FP32, ldw)
    out = torch.full((d_out, ldo), float("nan"), device="cuda")
    ldW = pad(d_in, 4) + 12
    tW = to_dev(weight, capi.KFAC_FP32, ldW) if weight is not None else None
    args = [capi.kfac_precond_args(tg.data_ptr(), ldg, tw.data_ptr(), ldw, ta.data_ptr(), lda, out.data_ptr(), ldo,
                                   d_out, d_in, tW.data_ptr() if tW is not None else None, ldW, lr)]
    wsb = capi.kfac_precondition_workspace(args)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    route = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    capi.kfac_precondition(args, precision, route.data_ptr(), ws.data_ptr(), wsb, stream())
    sync()
    got = out.cpu().numpy()
    assert np.isnan(got[:, d_in:]).all()  # padding of out untouched
    if weight is not None:
        Wn = tW.cpu().numpy()
        assert (Wn[:, d_in:] == 0).all()  # padding untouched
        return got, int(route.item()), Wn[:, :d_in]
    if with_route:
        return got, int(route.item())
    return got


def test_precondition_identity_is_exact():
    # every partial sum is exactly representable: the three bf16 slices must reassemble grad bit for bit
    rng = np.random.default_rng(21)
    d_out, d_in = 200, 300
    grad = rng.standard_normal((d_out, d_in)).astype(np.float32)
    got = run_precondition(np.eye(d_out, dtype=np.float32), grad, np.eye(d_in, dtype=np.float32))
    assert np.array_equal(got[:, :d_in], grad)


def test_precondition_diagonal_uses_all_24_bits():
    # single-term sums: the result is the fp32 product up to the dropped slice terms (< 2^-23)
    rng = np.random.default_rng(22)
    d_out, d_in = 130, 257
    grad = rng.standard_normal((d_out, d_in)).astype(np.float32)
    s = (rng.random(d_in) + 0.5).astype(np.float32)
    got = run_precondition(np.eye(d_out, dtype=np.float32), grad, np.diag(s))
    ref = grad.astype(np.float64) * s.astype(np.float64)[None, :]
    assert np.abs(got[:, :d_in] - ref).max() <= 3e-7 * np.abs(ref).max()


@pytest.mark.parametrize("precision", [capi.KFAC_PRECOND_FP32, capi.KFAC_PRECOND_AUTO])
@pytest.mark.parametrize("d_out,d_in", [(3, 4), (32, 65), (129, 300), (10, 1025), (300, 129)])
def test_precondition(d_out, d_in, precision):
    rng = np.random.default_rng(d_out * 7 + d_in)
    XG, _ = oracle.spd_inverse(spd_case(d_out, rng).astype(np.float64))
    XA, _ = oracle.spd_inverse(spd_case(d_in, rng).astype(np.float64))
    XG, XA = XG.astype(np.float32), XA.astype(np.float32)
    grad = (rng.standard_normal((d_out, d_in)) * 1e-2).astype(np.float32)
    got, route = run_precondition(XG, grad, XA, precision, with_route=True)
    ref = oracle.precondition(XG, grad, XA)
    err = rel_fro(got[:, :d_in], ref)
    assert err <= 2e-3
    if precision == capi.KFAC_PRECOND_FP32:
        assert route == 6
    else:
        assert route in (3, 6)
        if route == 3:  # kept only when the 16-bit result passed the check
            assert err <= 1e-3


def amplifying_layer(rows, d_in, d_out, gamma, rng):
    """A layer whose gradient lies in the row space of a rank-deficient input
    (rows < d_in): the damped inverse has gain 1/gamma off that space, the
    cancellation that 16-bit operands cannot carry."""
    a = rng.standard_normal((rows, d_in))
    g = rng.standard_normal((rows, d_out)) * 1e-3
    XA, _ = oracle.spd_inverse(a.T @ a / rows + gamma * np.eye(d_in))
    XG, _ = oracle.spd_inverse(g.T @ g / rows + gamma * np.eye(d_out))
    grad = g.T @ a / rows
    return XG.astype(np.float32), grad.astype(np.float32), XA.astype(np.float32)


def test_precondition_auto_recomputes_amplifying_layer():
    # 16-bit operands give ~1e-2 here (the MLP's first steps); the check must
    # catch it and the six-MMA pass must meet the bar
    rng = np.random.default_rng(23)
    XG, grad, XA = amplifying_layer(64, 300, 200, 1e-3, rng)
    ref = oracle.precondition(XG, grad, XA)
    got, route = run_precondition(XG, grad, XA, capi.KFAC_PRECOND_AUTO, with_route=True)
    assert route == 6
    assert rel_fro(got[:, :300], ref) <= 2e-3
    exact, _ = run_precondition(XG, grad, XA, capi.KFAC_PRECOND_FP32, with_route=True)
    assert np.array_equal(got[:, :300], exact[:, :300])  # the recomputation is the FP32 path's result


@pytest.mark.parametrize("precision", [capi.KFAC_PRECOND_FP32, capi.KFAC_PRECOND_AUTO])
@pytest.mark.parametrize("rows", [64, 4096])
def test_precondition_fused_weight_step(precision, rows):
    # rows = 64: the amplifying layer (AUTO recomputes it: the step comes from the
    # recomputed tiles); rows = 4096: kept at 16 bits (the step comes from the
    # stored out in the last launch)
    rng = np.random.default_rng(25 + rows)
    XG, grad, XA = amplifying_layer(rows, 300, 200, 1e-3, rng)
    W = rng.standard_normal(grad.shape).astype(np.float32)
    lr = np.float32(0.05)
    got, route, Wn = run_precondition(XG, grad, XA, precision, weight=W, lr=float(lr))
    V = got[:, :300]
    if precision == capi.KFAC_PRECOND_AUTO:
        assert route == (6 if rows == 64 else 3)
    # one fused multiply-add per element from the call's own out
    exact = (W.astype(np.float64) - np.float64(lr) * V.astype(np.float64)).astype(np.float32)
    assert (np.abs(Wn - exact) <= np.spacing(np.abs(exact))).all()
    # against the oracle: the step's error is lr times out's error, plus W's rounding
    Vref = oracle.precondition(XG, grad, XA)
    ref = oracle.weight_step(W, Vref, float(lr))
    bound = 2e-3 * float(lr) * np.linalg.norm(Vref) + 2.0 ** -23 * np.linalg.norm(W)
    assert np.linalg.norm(Wn - ref) <= bound


def test_precondition_auto_keeps_benign_layer():
    # full-rank input (rows >> d_in): no amplification, 16-bit operands suffice
    rng = np.random.default_rng(24)
    XG, grad, XA = amplifying_layer(4096, 300, 200, 1e-3, rng)
    ref = oracle.precondition(XG, grad, XA)
    got, route = run_precondition(XG, grad, XA, capi.KFAC_PRECOND_AUTO, with_route=True)
    assert route == 3
    assert rel_fro(got[:, :300], ref) <= 4e-4


# ------------------------------------------------------------------ whole configurations, stage-wise
def layer_specs(cfg):
    return [LayerSpec(l.d_in, l.d_out, cfg.rows(l), cfg.batch, l.hw) for l in cfg.layers]


def snapshot(step, li):
    A, G = step.fa[li], step.fg[li]
    f = lambda t: t.cpu().numpy()
    return dict(SA=f(A.shards)[:, :, :A.d], SG=f(G.shards)[:, :, :G.d], RA=f(A.running)[:, :A.d],
                RG=f(G.running)[:, :G.d], DA=f(A.damped)[:, :A.d], DG=f(G.damped)[:, :G.d],
                XA=f(A.inv)[:, :A.d], XG=f(G.inv)[:, :G.d])


def check_config(key, steps, check_layers=None, inv_steps=None):
    cfg = synth.config(key)
    specs = layer_specs(cfg)
    step = KFACStep(specs, cfg.P, cfg.gamma, cfg.decay or 0.0, cfg.in_dtype, refine=capi.KFAC_REFINE_AUTO)
    check_layers = range(len(specs)) if check_layers is None else check_layers
    prevR = {}
    report = []
    for t in range(steps):
        data = [synth.layer_inputs(cfg, t, li) for li in range(len(specs))]
        for li, dd in enumerate(data):
            step.set_layer_inputs(li, torch.from_numpy(dd["a"]), torch.from_numpy(dd["g"]),
                                  torch.from_numpy(dd["grad"]))
        s = step.stream_handle()
        step.factors(s)
        sync()
        shards = {li: snapshot(step, li) for li in check_layers}
        step.update_running(t == 0, s)
        step.inverse(s)
        step.precondition(s)
        sync()
        info = step.info.cpu().numpy()
        assert (info == 0).all(), info
        last = t in (inv_steps if inv_steps is not None else (steps - 1,))
        for li in check_layers:
            L = specs[li]
            snap = snapshot(step, li)
            a = data[li]["a"]
            g = data[li]["g"]
            gsrc = oracle.spatial_sum(g, L.batch, L.hw) if L.hw > 1 else g
            for name, x, S in (("A", a, shards[li]["SA"]), ("G", gsrc, shards[li]["SG"])):
                d = S.shape[1]
                m = upper_tile_mask(d)
                for p, ref in enumerate(oracle.shard_factors(x, cfg.P)):
                    e = rel_fro(S[p], ref, m)
                    assert e <= 1e-5, (key, t, li, name, p, e)
            for name in ("A", "G"):
                S = shards[li]["S" + name].astype(np.float64)
                d = S.shape[1]
                m = upper_tile_mask(d)
                F = oracle.aggregate(list(S))
                R = oracle.update_running(F, prevR.get((li, name)), cfg.decay or 0.0, t == 0)
                Dm = oracle.damp(R, cfg.gamma)
                assert rel_fro(snap["R" + name], R, m) <= 1e-6
                assert rel_fro(snap["D" + name], Dm, m) <= 1e-6
                Rg = snap["R" + name].astype(np.float64)
                Rg[~m] = 0
                prevR[(li, name)] = Rg
                if last:
                    Dg = snap["D" + name].astype(np.float64)
                    Dsym = np.triu(Dg) + np.triu(Dg, 1).T
                    X = snap["X" + name]
                    ref, i = oracle.spd_inverse(Dsym)
                    assert i == 0
                    err, res = rel_fro(X, ref), residual(X, Dsym)
                    report.append((li, name, d, err, res))
                    assert err <= 1e-3 and res <= 1e-3, (key, li, name, err, res)
            if last:
                V = step.out[li].cpu().numpy()[:, :L.d_in]
                ref = oracle.precondition(snap["XG"], data[li]["grad"], snap["XA"])
                assert rel_fro(V, ref) <= 2e-3, (key, li, rel_fro(V, ref))
    return step, report


def test_config_single_linear_with_bruteforce_end_to_end():
    step, _ = check_config("single_linear", 1)
    cfg = synth.config("single_linear")
    dd = synth.layer_inputs(cfg, 0, 0)
    (res,) = oracle.kfac_step([dd], cfg.P, cfg.gamma, 0.0, True)
    V = step.out[0].cpu().numpy()[:, :65]
    assert rel_fro(V, res["V"]) <= 2e-3


def test_config_mlp_ten_steps():
    # every step: the first steps see rank-deficient factors (256 samples, 785/1025 inputs)
    check_config("mlp", 10, inv_steps=range(10))


def test_config_resnet_conv_one_step():
    check_config("resnet_conv", 1)


def test_config_bert_layer_twenty_steps():
    # the workload's 20 running-average steps: every step's worker factors,
    # running and damped factors against the oracle; inverses and
    # preconditioned gradients on the first and the last step
    check_config("bert_layer", 20, inv_steps=(0, 19))


def test_step_applies_the_weight_step_after_routing():
    # two layers of 256 rows: a 785-wide input (rank-deficient: AUTO recomputes
    # it with 24-bit operands) and a 65-wide one (kept at 16 bits); from zero
    # weights one step must leave weight = -lr * out exactly in both
    rng = np.random.default_rng(26)
    specs = [LayerSpec(785, 64, 256, 256, 1), LayerSpec(65, 64, 256, 256, 1)]
    step = KFACStep(specs, 4, 1e-3, 0.95, "bf16", refine=capi.KFAC_REFINE_AUTO, weight_lr=0.25)
    for li, L in enumerate(specs):
        a = synth.round_bf16(np.maximum(rng.standard_normal((256, L.d_in)), 0.0)).astype(np.float32)
        a[:, -1] = 1.0
        g = synth.round_bf16(rng.standard_normal((256, L.d_out)) * 1e-3).astype(np.float32)
        grad = (g.astype(np.float64).T @ a.astype(np.float64) / 256).astype(np.float32)
        step.set_layer_inputs(li, torch.from_numpy(a), torch.from_numpy(g), torch.from_numpy(grad))
    step.step(first_step=True)
    sync()
    assert step.pc_route.cpu().numpy().tolist() == [6, 3]  # both paths of the last launch
    for li, L in enumerate(specs):
        V = step.out[li].cpu().numpy()[:, :L.d_in]
        W = step.weight[li].cpu().numpy()
        assert np.array_equal(W[:, :L.d_in], (np.float32(-0.25) * V).astype(np.float32))
        assert (W[:, L.d_in:] == 0).all()


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    # a wait that nothing ends (an mbarrier no one arrives on) must give up after
    # its limit (here 2e8 cycles, ~0.1 s), record KFAC_ERR_TIMEOUT and return
    assert capi.kfac_device_status(clear=True) in (capi.KFAC_OK, capi.KFAC_ERR_TIMEOUT)
    capi.kfac_wait_selftest(200_000_000, stream())
    torch.cuda.synchronize()  # the kernel returned on its own
    assert capi.kfac_device_status(clear=True) == capi.KFAC_ERR_TIMEOUT
    assert capi.kfac_device_status() == capi.KFAC_OK
    # the library still computes on the same context
    rng = np.random.default_rng(27)
    XG, _ = oracle.spd_inverse(spd_case(40, rng).astype(np.float64))
    XA, _ = oracle.spd_inverse(spd_case(70, rng).astype(np.float64))
    grad = rng.standard_normal((40, 70)).astype(np.float32)
    got = run_precondition(XG.astype(np.float32), grad, XA.astype(np.float32))
    assert rel_fro(got[:, :70], oracle.precondition(XG, grad, XA)) <= 2e-3
    assert capi.kfac_device_status() == capi.KFAC_OK
