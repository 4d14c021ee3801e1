"""Parity at the benchmark's full size (24-layer BERT-large stack: 96 linear
layers, 192 factors up to 4097 x 4097, 4096 rows in P = 8 worker shards), in
the launch configuration bench.py times.  The oracle computes sampled outputs
one by one; the rest is checked through properties that hold at any size."""
import numpy as np
import pytest
import torch

import oracle
import synth
from infra_fac_factors_gb300 import capi
from infra_fac_factors_gb300.step import KFACStep, LayerSpec

from gpu_util import ensure_built, rel_fro, residual, upper_tile_mask

pytestmark = pytest.mark.gpu

CFG = synth.config("bert_large")
# one layer of each kind, spread over the stack
LAYERS = [0, 5, 46, 95]


@pytest.fixture(scope="module")
def run():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    ensure_built()
    specs = [LayerSpec(l.d_in, l.d_out, CFG.rows(l), CFG.batch, l.hw) for l in CFG.layers]
    st = KFACStep(specs, CFG.P, CFG.gamma, CFG.decay, CFG.in_dtype, refine=capi.KFAC_REFINE_AUTO)
    inputs = {}
    for li in range(len(specs)):
        dd = synth.device_layer_inputs(CFG, 0, li)
        st.set_layer_inputs(li, dd["a"], dd["g"], dd["grad"])
        if li in LAYERS:
            inputs[li] = {k: v.float().cpu().numpy() for k, v in dd.items()}
        del dd
    s = st.stream_handle()
    st.factors(s)
    torch.cuda.synchronize()
    shards = {li: (st.fa[li].shards.cpu().numpy(), st.fg[li].shards.cpu().numpy()) for li in LAYERS}
    st.update_running(True, s)
    st.inverse(s)
    st.precondition(s)
    torch.cuda.synchronize()
    first = {li: {n: getattr(F, n).cpu().numpy() for n in ("running", "damped", "inv")}
             for li in LAYERS for F in (st.fa[li],)}
    assert capi.kfac_device_status(clear=True) == capi.KFAC_OK
    return dict(step=st, specs=specs, inputs=inputs, shards=shards, first=first)


def test_all_inverses_succeeded_in_fp32(run):
    st = run["step"]
    assert (st.info.cpu().numpy() == 0).all()
    # the BERT-large factors are well conditioned: AUTO keeps all of them in the
    # fp32 pass; the G factors (gamma I plus a factor about 1e-5 of it) have
    # Gershgorin bounds near 1 and take 16-bit operands, the A factors 24-bit
    route = st.route.cpu().numpy()
    facs = st.factor_list()
    for i, r in enumerate(route):
        F = facs[st.inv_order[i]]
        is_g = st.inv_order[i] >= len(st.layers)
        assert r == (2 if is_g else 0), (i, F.d, r)


def test_sampled_factor_entries(run):
    rng = np.random.default_rng(0)
    P = CFG.P
    for li in LAYERS:
        x_a, x_g = run["inputs"][li]["a"], run["inputs"][li]["g"]
        for x, S in ((x_a, run["shards"][li][0]), (x_g, run["shards"][li][1])):
            rows, d = x.shape
            rp = rows // P
            for _ in range(48):
                p = int(rng.integers(P))
                r = int(rng.integers(d))
                c = int(rng.integers((r // 128) * 128, d))
                xs = x[p * rp:(p + 1) * rp].astype(np.float64)
                ref = xs[:, r] @ xs[:, c] / rp
                norm = np.sqrt((xs[:, r] @ xs[:, r]) * (xs[:, c] @ xs[:, c])) / rp
                assert abs(S[p, r, c] - ref) <= 1e-5 * norm, (li, p, r, c, S[p, r, c], ref)


def test_whole_shard_factor_per_layer_kind(run):
    # one whole worker factor of each layer kind (a different worker each),
    # every upper-tile element against the oracle
    P = CFG.P
    for k, li in enumerate(LAYERS):
        for x, S in ((run["inputs"][li]["a"], run["shards"][li][0]), (run["inputs"][li]["g"], run["shards"][li][1])):
            rows, d = x.shape
            rp = rows // P
            p = (3 * k + 1) % P
            ref = oracle.factor(x[p * rp:(p + 1) * rp], 1.0 / rp)
            m = upper_tile_mask(d)
            assert rel_fro(S[p][:, :d], ref, m) <= 1e-5, (li, p, d)


def test_running_average_and_damping_properties(run):
    for li in LAYERS:
        S = run["shards"][li][0]
        F = run["first"][li]
        d = S.shape[1]
        m = upper_tile_mask(d)
        R = F["running"][:, :d]
        D = F["damped"][:, :d]
        mean = oracle.aggregate([s.astype(np.float64) for s in S[:, :, :d]])
        assert rel_fro(R, mean, m) <= 1e-6
        # damped = running + gamma on the diagonal, bit for bit in fp32
        off = m & ~np.eye(d, dtype=bool)
        assert np.array_equal(D[off], R[off])
        assert np.array_equal(np.diag(D), (np.diag(R) + np.float32(CFG.gamma)).astype(np.float32))


@pytest.mark.parametrize("li", LAYERS)
def test_inverse_residual_and_symmetry(run, li):
    st = run["step"]
    for F in (st.fa[li], st.fg[li]):
        Dg = F.damped.cpu().numpy()[:, :F.d].astype(np.float64)
        D = np.triu(Dg) + np.triu(Dg, 1).T
        X = F.inv.cpu().numpy()[:, :F.d]
        assert np.array_equal(X, X.T)
        assert residual(X, D) <= 1e-3, (li, F.d, residual(X, D))


def test_inverse_matches_oracle_on_largest_factor(run):
    st = run["step"]
    F = st.fa[95]  # FFN-out input factor, 4097 x 4097, rank-deficient + damping
    Dg = F.damped.cpu().numpy()[:, :F.d].astype(np.float64)
    D = np.triu(Dg) + np.triu(Dg, 1).T
    ref, info = oracle.spd_inverse(D)
    assert info == 0
    assert rel_fro(F.inv.cpu().numpy()[:, :F.d], ref) <= 1e-3


def test_sampled_preconditioned_rows(run):
    st = run["step"]
    rng = np.random.default_rng(1)
    for li in LAYERS:
        L = run["specs"][li]
        XG = st.fg[li].inv.cpu().numpy()[:, :L.d_out].astype(np.float64)
        XA = st.fa[li].inv.cpu().numpy()[:, :L.d_in].astype(np.float64)
        grad = st.grad[li].cpu().numpy()[:, :L.d_in].astype(np.float64)
        V = st.out[li].cpu().numpy()[:, :L.d_in]
        rows = rng.choice(L.d_out, size=8, replace=False)
        ref = (XG[rows] @ grad) @ XA
        assert rel_fro(V[rows], ref) <= 2e-3, (li, rel_fro(V[rows], ref))


def test_preconditioned_ffn_out_layer_whole(run):
    # the layer with the largest cancellation (rank-deficient 4097-wide input):
    # the whole 1024 x 4097 result against the oracle, and the products used
    st = run["step"]
    li = 95
    L = run["specs"][li]
    XG = st.fg[li].inv.cpu().numpy()[:, :L.d_out]
    XA = st.fa[li].inv.cpu().numpy()[:, :L.d_in]
    grad = st.grad[li].cpu().numpy()[:, :L.d_in]
    V = st.out[li].cpu().numpy()[:, :L.d_in]
    assert rel_fro(V, oracle.precondition(XG, grad, XA)) <= 2e-3
    route = st.pc_route.cpu().numpy()
    assert set(route.tolist()) <= {3, 6}
