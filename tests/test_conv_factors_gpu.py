"""GPU parity of the implicit-im2col conv factors (kfac_conv_factors) against
the fp64 oracle: oracle.factor of oracle.im2col3x3 of each worker's images.

Tolerance: factors <= 1e-5 relative Frobenius (bf16 products are exact in
fp32; the error is fp32 accumulation).  NaN sentinels in the lower tiles and
the padding catch stray writes."""
import numpy as np
import pytest
import torch

import oracle
import synth
from infra_fac_factors_gb300 import capi

from gpu_util import ensure_built, pad, rel_fro, stream, upper_tile_mask

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


def conv_args(x_dev, shape, out, ldo, P):
    B, H, W, C = shape
    d = 9 * C + 1
    rows_p = B // P * H * W
    return capi.kfac_conv_factor_args(x_dev.data_ptr(), B, H, W, C, out.data_ptr(), ldo, d * ldo, 1.0 / rows_p)


def run_conv(x, P, mirror=0, ld_extra=4):
    B, H, W, C = x.shape
    d = 9 * C + 1
    ldo = pad(d, 4) + ld_extra
    xt = torch.from_numpy(np.ascontiguousarray(x)).cuda().to(torch.bfloat16)
    out = torch.full((P, d, ldo), float("nan"), dtype=torch.float32, device="cuda")
    capi.kfac_conv_factors([conv_args(xt, x.shape, out, ldo, P)], P, mirror, stream())
    sync()
    return out.cpu().numpy()


def oracle_shard(x, P, p):
    B = x.shape[0]
    X = oracle.im2col3x3(x[p * B // P:(p + 1) * B // P])
    return oracle.factor(X, 1.0 / X.shape[0])


def check_upper(res, x, P, shards=None):
    B, H, W, C = x.shape
    d = 9 * C + 1
    m = upper_tile_mask(d)
    for p in (range(P) if shards is None else shards):
        ref = oracle_shard(x, P, p)
        got = res[p][:, :d]
        err = rel_fro(got, ref, m)
        assert err <= 1e-5, (p, err)
        assert np.isnan(got[~m]).all(), "lower tiles must stay untouched"
        assert np.isnan(res[p][:, d:]).all(), "padding must stay untouched"


@pytest.mark.parametrize("shape,P", [
    ((4, 5, 7, 64), 2),      # 70 patch rows per worker: one full 64-row stage and a ragged one
    ((2, 3, 3, 128), 1),     # every position touches the zero padding
    ((3, 1, 1, 64), 3),      # 1 x 1 images: only the centre tap and the bias are non-zero
    ((2, 2, 65, 64), 2),     # one-row-high images, a width past two 64-row stages
    ((8, 24, 24, 64), 2),    # 2304 rows per worker: three 1024-row accumulation chunks
    ((2, 6, 5, 192), 2),     # d = 1729: fourteen 128-row blocks, three 64-channel boxes per tap
    ((4, 33, 1, 64), 2),     # one-pixel-wide images: a 64-row block spans two images
])
def test_conv_factors_match_oracle(shape, P):
    x = synth.conv_activations(shape, ("test", *shape, P))
    check_upper(run_conv(x, P), x, P)


def test_conv_factors_mirror_gives_full_symmetric():
    shape, P = (2, 6, 5, 64), 2
    x = synth.conv_activations(shape, ("mirror",))
    res = run_conv(x, P, mirror=1, ld_extra=0)
    d = 9 * shape[3] + 1
    for p in range(P):
        got = res[p][:, :d]
        assert not np.isnan(got).any()
        assert rel_fro(got, oracle_shard(x, P, p)) <= 1e-5
        assert np.abs(got - got.T).max() <= 1e-6 * np.abs(got).max()


def test_conv_factors_signed_inputs_and_bias_column():
    # signed activations (no ReLU): cancellation in the sums; the bias row of
    # each factor is the patch mean and its corner is exactly 1
    shape, P = (4, 4, 4, 64), 4
    x = synth.conv_activations(shape, ("signed",), dist="normal")
    res = run_conv(x, P)
    check_upper(res, x, P)
    d = 9 * shape[3] + 1
    for p in range(P):
        assert res[p][d - 1, d - 1] == 1.0


def test_conv_factors_several_layers_in_one_call():
    P = 4
    shapes = [(4, 7, 7, 64), (8, 3, 5, 128), (4, 2, 2, 256)]
    xs, outs, args, lds = [], [], [], []
    for k, sh in enumerate(shapes):
        x = synth.conv_activations(sh, ("multi", k))
        d = 9 * sh[3] + 1
        ldo = pad(d, 4)
        xt = torch.from_numpy(np.ascontiguousarray(x)).cuda().to(torch.bfloat16)
        out = torch.full((P, d, ldo), float("nan"), dtype=torch.float32, device="cuda")
        xs.append((x, xt))
        outs.append(out)
        args.append(conv_args(xt, sh, out, ldo, P))
    capi.kfac_conv_factors(args, P, 0, stream())
    sync()
    for (x, _), out in zip(xs, outs):
        check_upper(out.cpu().numpy(), x, P)


@pytest.mark.parametrize("layer_index", [0, 1, 2, 3])
def test_conv_factors_resnet_full_size_sampled_workers(layer_index):
    # the ResNet-50 3 x 3 conv shapes at batch 32 in 8 workers; the first and
    # last workers' factors are compared whole with the oracle
    cfg = synth.config("resnet_conv")
    layer = cfg.layers[layer_index]
    shape = synth.conv_shape(cfg, layer)
    P = cfg.P
    x = synth.conv_activations(shape, (cfg.key, 0, layer_index))
    res = run_conv(x, P, ld_extra=0)
    check_upper(res, x, P, shards=(0, P - 1))


def run_step_and_check(specs, images, P, gamma, decay, steps, g_sigma, seed):
    """Run KFACStep for `steps` steps on `specs` (conv layers given by their
    NHWC activations of shape images[li], linear layers by a) and check every
    stage: worker factors against the oracle on the patch matrices
    (oracle.im2col3x3) of the same activations, each later stage against the
    oracle fed the GPU's previous stage, as in the config tests."""
    from infra_fac_factors_gb300.step import KFACStep
    from gpu_util import residual

    step = KFACStep(specs, P, gamma, decay, "bf16", refine=capi.KFAC_REFINE_AUTO, n_groups=2)
    prevR = {}
    for t in range(steps):
        data = []
        for li, L in enumerate(specs):
            rng = np.random.default_rng((seed, t, li))
            g = synth.round_bf16((rng.standard_normal((L.rows, L.d_out)) * g_sigma).astype(np.float32))
            if L.image is not None:
                x = synth.conv_activations(images[li], (seed, t, li))
                a, src = oracle.im2col3x3(x), torch.from_numpy(x)
                gsrc = oracle.spatial_sum(g, L.batch, L.hw)
            else:
                a = synth.round_bf16(rng.standard_normal((L.rows, L.d_in)).astype(np.float32))
                a[:, -1] = 1.0
                src, gsrc = torch.from_numpy(a), g
            grad = (g.astype(np.float64).T @ a.astype(np.float64) / L.batch).astype(np.float32)
            data.append((a, gsrc, grad))
            step.set_layer_inputs(li, src, torch.from_numpy(g), torch.from_numpy(grad))
        step.step(first_step=(t == 0))
        sync()
        assert (step.info.cpu().numpy() == 0).all()
        for li, L in enumerate(specs):
            a, gsrc, grad = data[li]
            X = {}
            for name, F, src in (("A", step.fa[li], a), ("G", step.fg[li], gsrc)):
                d = F.d
                m = upper_tile_mask(d)
                S = F.shards.cpu().numpy()[:, :, :d].astype(np.float64)
                for p, ref in enumerate(oracle.shard_factors(src, P)):
                    assert rel_fro(S[p], ref, m) <= 1e-5, (t, li, name, p, rel_fro(S[p], ref, m))
                R = oracle.update_running(oracle.aggregate(list(S)), prevR.get((li, name)), decay, t == 0)
                del S
                Rg = F.running.cpu().numpy()[:, :d].astype(np.float64)
                assert rel_fro(Rg, R, m) <= 1e-6
                Rg[~m] = 0
                prevR[(li, name)] = Rg
                Dg = F.damped.cpu().numpy()[:, :d].astype(np.float64)
                assert rel_fro(Dg, oracle.damp(R, gamma), m) <= 1e-6
                Dsym = np.triu(Dg) + np.triu(Dg, 1).T
                X[name] = F.inv.cpu().numpy()[:, :d]
                Xref, info = oracle.spd_inverse(Dsym)
                assert info == 0
                err, res = rel_fro(X[name], Xref), residual(X[name], Dsym)
                assert err <= 1e-3 and res <= 1e-3, (t, li, name, err, res)
            V = step.out[li].cpu().numpy()[:, :L.d_in]
            assert rel_fro(V, oracle.precondition(X["G"], grad, X["A"])) <= 2e-3, (t, li)


def test_step_with_conv_layers_given_by_their_images():
    # two 3 x 3 conv layers given as NHWC activations and one linear layer, two steps
    from infra_fac_factors_gb300.step import LayerSpec

    P, batch = 4, 8
    images = [(batch, 6, 6, 64), (batch, 3, 5, 128), None]
    d_outs = [64, 96]
    specs = [LayerSpec(9 * C + 1, d_out, B * H * W, B, H * W, image=(H, W))
             for (B, H, W, C), d_out in zip(images[:2], d_outs)]
    specs.append(LayerSpec(129, 80, 64, 64))
    run_step_and_check(specs, images, P, 1e-3, 0.9, 2, 1e-2, seed=1)


def test_step_resnet_conv_workload_from_images():
    # the ResNet-50 3 x 3 conv workload at full size (batch 32, P = 8) with its
    # factor A formed from NHWC activations, one step, every stage checked
    from infra_fac_factors_gb300.step import LayerSpec

    cfg = synth.config("resnet_conv")
    images, specs = [], []
    for layer in cfg.layers:
        B, H, W, C = synth.conv_shape(cfg, layer)
        images.append((B, H, W, C))
        specs.append(LayerSpec(layer.d_in, layer.d_out, cfg.rows(layer), cfg.batch, layer.hw, image=(H, W)))
    run_step_and_check(specs, images, cfg.P, cfg.gamma, 0.0, 1, cfg.g_sigma, seed=2)


def test_conv_factors_more_problems_than_one_launch_holds():
    # 13 layers x 8 workers = 104 (layer, worker) problems: two launches
    P = 8
    shapes = [(8, 2 + k % 3, 3 + k % 2, 64 * (1 + k % 2)) for k in range(13)]
    xs, outs, args = [], [], []
    for k, sh in enumerate(shapes):
        x = synth.conv_activations(sh, ("many", k))
        d = 9 * sh[3] + 1
        ldo = pad(d, 4)
        xt = torch.from_numpy(np.ascontiguousarray(x)).cuda().to(torch.bfloat16)
        out = torch.full((P, d, ldo), float("nan"), dtype=torch.float32, device="cuda")
        xs.append((x, xt))
        outs.append(out)
        args.append(conv_args(xt, sh, out, ldo, P))
    capi.kfac_conv_factors(args, P, 0, stream())
    sync()
    for (x, _), out in zip(xs, outs):
        check_upper(out.cpu().numpy(), x, P)
