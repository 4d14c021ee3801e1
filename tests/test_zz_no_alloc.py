"""kfac_precondition_static: preconditioning for callers that cannot allocate
device memory (their memory belongs to another allocator, or their hot path
must not allocate), through the C ABI.  Its result must match
kfac_precondition, which takes a caller-provided workspace, on two calls in a
row; its scratch is the library's fixed array, shared by all calls.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process."""
import numpy as np
import pytest
import torch

from infra_fac_factors_gb300 import capi

from gpu_util import ensure_built, pad, rel_fro, stream, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    ensure_built()


def spd_inverse_f32(d, rng):
    x = rng.standard_normal((d + 16, d))
    return np.linalg.inv(x.T @ x / (d + 16) + 1e-2 * np.eye(d)).astype(np.float32)


def make_layers(seed, shapes):
    """Device buffers and argument structs of several layers (d_out, d_in)."""
    rng = np.random.default_rng(seed)
    keep, args = [], []
    for d_out, d_in in shapes:
        XG, XA = spd_inverse_f32(d_out, rng), spd_inverse_f32(d_in, rng)
        grad = (rng.standard_normal((d_out, d_in)) * 1e-2).astype(np.float32)
        ldg, lda, ldw, ldo = pad(d_out, 4), pad(d_in, 4), pad(d_in, 4) + 4, pad(d_in, 4)
        tg, ta, tw = to_dev(XG, capi.KFAC_FP32, ldg), to_dev(XA, capi.KFAC_FP32, lda), to_dev(grad, capi.KFAC_FP32, ldw)
        o1 = torch.full((d_out, ldo), float("nan"), device="cuda")
        o2 = torch.full((d_out, ldo), float("nan"), device="cuda")
        keep += [tg, ta, tw, o1, o2]
        a1 = capi.kfac_precond_args(tg.data_ptr(), ldg, tw.data_ptr(), ldw, ta.data_ptr(), lda, o1.data_ptr(), ldo,
                                    d_out, d_in)
        a2 = capi.kfac_precond_args(tg.data_ptr(), ldg, tw.data_ptr(), ldw, ta.data_ptr(), lda, o2.data_ptr(), ldo,
                                    d_out, d_in)
        args.append((a1, a2, o1, o2, d_in))
    return keep, args


def test_static_scratch_matches_workspace_version_twice():
    assert capi.kfac_precondition_static_capacity() == 64 << 20
    for call, (seed, shapes) in enumerate(((1, [(300, 513), (65, 129)]), (2, [(129, 300), (512, 1025)]))):
        keep, layers = make_layers(seed, shapes)
        ws_args = [a1 for a1, _, _, _, _ in layers]
        st_args = [a2 for _, a2, _, _, _ in layers]
        wsb = capi.kfac_precondition_workspace(ws_args)
        assert 0 < wsb <= capi.kfac_precondition_static_capacity()
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        precision = capi.KFAC_PRECOND_AUTO if call == 0 else capi.KFAC_PRECOND_FP32
        capi.kfac_precondition(ws_args, precision, 0, ws.data_ptr(), wsb, stream())
        capi.kfac_precondition_static(st_args, precision, 0, stream())
        torch.cuda.synchronize()
        assert capi.kfac_device_status(clear=True) == capi.KFAC_OK
        for _, _, o1, o2, d_in in layers:
            ref = o1.cpu().numpy()[:, :d_in]
            got = o2.cpu().numpy()[:, :d_in]
            assert not np.isnan(got).any(), call
            assert rel_fro(got, ref) <= 2e-3, (call, rel_fro(got, ref))


def test_static_scratch_rejects_oversized_layers():
    # a 4096 x 4097 layer needs about 300 MB of scratch: refused before any launch
    big = capi.kfac_precond_args(1 << 20, 4096, 2 << 20, 4100, 3 << 20, 4100, 4 << 20, 4100, 4096, 4097)
    assert capi.kfac_precondition_workspace([big]) > capi.kfac_precondition_static_capacity()
    assert capi.kfac_precondition_static([big], capi.KFAC_PRECOND_AUTO, 0, check=False) == capi.KFAC_ERR_WORKSPACE
    bad = capi.kfac_precond_args(1 << 20, 4, 2 << 20, 8, 3 << 20, 8, 2 << 20, 8, 4, 8)  # out aliases grad
    assert capi.kfac_precondition_static([bad], capi.KFAC_PRECOND_AUTO, 0, check=False) == capi.KFAC_ERR_INVALID_ARG
