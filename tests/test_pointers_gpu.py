"""Every data pointer must be device memory of the current GPU: host memory
(pinned or pageable) is refused with KFAC_ERR_INVALID_ARG before any launch.
The tensor-core kernels encode their operands into TMA tensor maps, some of
them loaded with cluster multicast, which must cover this GPU's memory only."""
import numpy as np
import pytest
import torch

from infra_fac_factors_gb300 import capi
from gpu_util import ensure_built, stream

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _host_buffers(nbytes):
    pinned = torch.zeros(nbytes // 4, dtype=torch.float32).pin_memory()
    pageable = np.zeros(nbytes // 4, dtype=np.float32)
    return pinned, pageable


def test_host_pointers_are_refused_before_any_launch():
    d, ld, rows, P = 64, 64, 256, 2
    x = torch.zeros((rows, ld), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((P, d, ld), dtype=torch.float32, device="cuda")
    pinned, pageable = _host_buffers(P * d * ld * 4)
    hosts = (pinned.data_ptr(), pageable.ctypes.data)
    s = stream()
    torch.cuda.synchronize()
    n0 = capi.kfac_launch_count()
    for hp in hosts:
        bad_out = capi.kfac_factor_args(x.data_ptr(), rows, d, ld, hp, ld, d * ld, 1.0 / (rows // P))
        bad_in = capi.kfac_factor_args(hp, rows, d, ld, out.data_ptr(), ld, d * ld, 1.0 / (rows // P))
        for a in (bad_out, bad_in):
            assert capi.kfac_factors([a], capi.KFAC_BF16, P, 0, s, check=False) == capi.KFAC_ERR_INVALID_ARG
        run = capi.kfac_running_args(hp, d * ld, out[0].data_ptr(), out[1].data_ptr(), d, ld)
        assert capi.kfac_update_running([run], 1, 0.5, 0.1, True, s, check=False) == capi.KFAC_ERR_INVALID_ARG
        inv = [capi.kfac_inverse_args(out[0].data_ptr(), hp, d, ld, ld)]
        wsb = capi.kfac_damped_inverse_workspace(inv, capi.KFAC_REFINE_AUTO)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        info = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert capi.kfac_damped_inverse(inv, 0.0, 1, info.data_ptr(), 0, ws.data_ptr(), wsb, s,
                                        check=False) == capi.KFAC_ERR_INVALID_ARG
        pc = [capi.kfac_precond_args(out[0].data_ptr(), ld, hp, ld, out[1].data_ptr(), ld,
                                     x.data_ptr(), ld, d, d)]
        pcb = capi.kfac_precondition_workspace(pc)
        pws = torch.empty(pcb, dtype=torch.uint8, device="cuda")
        assert capi.kfac_precondition(pc, capi.KFAC_PRECOND_AUTO, 0, pws.data_ptr(), pcb, s,
                                      check=False) == capi.KFAC_ERR_INVALID_ARG
        assert capi.kfac_precondition_static(pc, capi.KFAC_PRECOND_AUTO, 0, s,
                                             check=False) == capi.KFAC_ERR_INVALID_ARG
    # a host workspace is refused too
    good = [capi.kfac_inverse_args(out[0].data_ptr(), out[1].data_ptr(), d, ld, ld)]
    wsb = capi.kfac_damped_inverse_workspace(good, capi.KFAC_REFINE_AUTO)
    hws = torch.empty(wsb, dtype=torch.uint8).pin_memory()
    info = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert capi.kfac_damped_inverse(good, 0.0, 1, info.data_ptr(), 0, hws.data_ptr(), wsb, s,
                                    check=False) == capi.KFAC_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert capi.kfac_launch_count() == n0  # nothing was launched
    # and the library still works on device memory afterwards, with no error left behind
    ok = capi.kfac_factor_args(x.data_ptr(), rows, d, ld, out.data_ptr(), ld, d * ld, 1.0 / (rows // P))
    assert capi.kfac_factors([ok], capi.KFAC_BF16, P, 0, s, check=False) == capi.KFAC_OK
    torch.cuda.synchronize()
    assert capi.kfac_device_status(clear=True) == capi.KFAC_OK
