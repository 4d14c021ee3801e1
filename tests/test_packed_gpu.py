"""Packed upper triangles (kfac_pack_upper / kfac_unpack_upper) against the
oracle's packed layout, bit for bit, and a checkpoint of the running factors
in packed form: ten steps equal five steps, a packed save and restore of the
running factors into a fresh step, and five more steps, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import synth
from infra_fac_factors_gb300 import capi
from infra_fac_factors_gb300.step import KFACStep, LayerSpec

from gpu_util import ensure_built, pad, stream

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _nan_matrix(d, ld, rng):
    """d x ld fp32: symmetric values on the upper triangle, NaN below it and in
    the padding columns (elements the packing must never read)."""
    M = np.full((d, ld), np.nan, dtype=np.float32)
    S = rng.standard_normal((d, d)).astype(np.float32)
    iu = np.triu_indices(d)
    M[iu] = S[iu]
    return M


def _fused(sizes, rng, ld_extra=4):
    mats, hosts, args = [], [], []
    total = sum(d * (d + 1) // 2 for d in sizes)
    packed = torch.full((total + 1,), float("nan"), dtype=torch.float32, device="cuda")  # +1: a guard
    off = 0
    offs = []
    for d in sizes:
        ld = pad(d, 4) + ld_extra
        M = _nan_matrix(d, ld, rng)
        t = torch.from_numpy(M).cuda()
        mats.append(t)
        hosts.append(M)
        args.append(capi.kfac_pack_args(t.data_ptr(), d, ld, packed.data_ptr() + 4 * off))
        offs.append(off)
        off += d * (d + 1) // 2
    return mats, hosts, args, packed, offs, total


SIZES = [1, 2, 3, 31, 127, 128, 129, 577, 1025, 4097]


def test_pack_is_bit_exact_in_one_launch():
    rng = np.random.default_rng(1)
    mats, hosts, args, packed, offs, total = _fused(SIZES, rng)
    torch.cuda.synchronize()
    n0 = capi.kfac_launch_count()
    capi.kfac_pack_upper(args, stream())
    torch.cuda.synchronize()
    assert capi.kfac_launch_count() - n0 == 1  # every matrix in one fused launch
    got = packed.cpu().numpy()
    assert np.isnan(got[total])  # nothing written past the last packed row
    for d, M, off in zip(SIZES, hosts, offs):
        want = oracle.pack_upper(M[:, :d])
        assert np.array_equal(got[off:off + want.size], want), d
        # the packed index table of the oracle, bit for bit, on sampled entries
        for i, j in ((0, 0), (0, d - 1), (d - 1, d - 1), (d // 2, d // 2), (d // 3, (2 * d) // 3)):
            assert got[off + oracle.packed_index(i, j, d)] == M[i, j]


@pytest.mark.parametrize("mirror", [False, True])
def test_unpack_is_bit_exact_and_touches_nothing_else(mirror):
    rng = np.random.default_rng(2)
    mats, hosts, args, packed, offs, total = _fused(SIZES, rng)
    capi.kfac_pack_upper(args, stream())
    for t in mats:
        t.fill_(float("nan"))
    capi.kfac_unpack_upper(args, mirror, stream())
    torch.cuda.synchronize()
    for d, M, t in zip(SIZES, hosts, mats):
        got = t.cpu().numpy()
        want = oracle.unpack_upper(oracle.pack_upper(M[:, :d]), d, mirror=mirror)
        assert np.array_equal(got[:, :d], want, equal_nan=True), d
        assert np.isnan(got[:, d:]).all()  # padding columns untouched


def test_more_matrices_than_one_launch_holds():
    rng = np.random.default_rng(3)
    sizes = [int(v) for v in rng.integers(1, 70, size=300)]
    mats, hosts, args, packed, offs, total = _fused(sizes, rng, ld_extra=0)
    capi.kfac_pack_upper(args, stream())
    torch.cuda.synchronize()
    got = packed.cpu().numpy()
    want = np.concatenate([oracle.pack_upper(M[:, :d]) for d, M in zip(sizes, hosts)])
    assert np.array_equal(got[:total], want)


# ------------------------------------------------------------------ checkpoint / resume
def _specs(cfg):
    return [LayerSpec(l.d_in, l.d_out, cfg.rows(l), cfg.batch, l.hw) for l in cfg.layers]


def _feed(step, cfg, t):
    for li in range(len(cfg.layers)):
        dd = synth.layer_inputs(cfg, t, li)
        step.set_layer_inputs(li, torch.from_numpy(dd["a"]), torch.from_numpy(dd["g"]),
                              torch.from_numpy(dd["grad"]))


def _state(step):
    out = []
    for F in step.factor_list():
        d = F.d
        iu = np.triu_indices(d)
        out.append((F.running.cpu().numpy()[:, :d][iu], F.damped.cpu().numpy()[:, :d][iu],
                    F.inv.cpu().numpy()[:, :d]))
    return out, [o.cpu().numpy() for o in step.out], step.route.cpu().numpy(), step.pc_route.cpu().numpy()


def test_checkpoint_resume_through_packed_running_factors_is_bit_identical():
    cfg = synth.config("mlp")  # rank-deficient early factors: AUTO routes some to fp64
    steps, cut = 10, 5
    mk = lambda: KFACStep(_specs(cfg), cfg.P, cfg.gamma, cfg.decay, cfg.in_dtype, refine=capi.KFAC_REFINE_AUTO)
    whole = mk()
    for t in range(steps):
        _feed(whole, cfg, t)
        whole.step(first_step=(t == 0))
    torch.cuda.synchronize()
    ref = _state(whole)
    del whole

    first = mk()
    for t in range(cut):
        _feed(first, cfg, t)
        first.step(first_step=(t == 0))
    facs = first.factor_list()
    total = sum(F.d * (F.d + 1) // 2 for F in facs)
    buf = torch.empty(total, dtype=torch.float32, device="cuda")
    args, off = [], 0
    for F in facs:
        args.append(capi.kfac_pack_args(F.running.data_ptr(), F.d, F.ld, buf.data_ptr() + 4 * off))
        off += F.d * (F.d + 1) // 2
    capi.kfac_pack_upper(args, stream())
    saved = buf.cpu().numpy().copy()  # the checkpoint: half the bytes of the square factors
    assert saved.nbytes == 4 * total
    del first, buf

    resumed = mk()
    buf = torch.from_numpy(saved).cuda()
    args, off = [], 0
    for F in resumed.factor_list():
        args.append(capi.kfac_pack_args(F.running.data_ptr(), F.d, F.ld, buf.data_ptr() + 4 * off))
        off += F.d * (F.d + 1) // 2
    capi.kfac_unpack_upper(args, True, stream())
    for t in range(cut, steps):
        _feed(resumed, cfg, t)
        resumed.step(first_step=False)
    torch.cuda.synchronize()
    got = _state(resumed)
    assert capi.kfac_device_status(clear=True) == capi.KFAC_OK
    for (r0, d0, x0), (r1, d1, x1) in zip(ref[0], got[0]):
        assert np.array_equal(r0, r1) and np.array_equal(d0, d1) and np.array_equal(x0, x1)
    for v0, v1 in zip(ref[1], got[1]):
        assert np.array_equal(v0, v1)
    assert np.array_equal(ref[2], got[2]) and np.array_equal(ref[3], got[3])
