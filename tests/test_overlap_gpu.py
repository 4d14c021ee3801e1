"""KFACStep.step overlaps the factor pass of one layer group with the
running-average pass of the previous group on a second stream.  Each
kernel's result for a factor does not depend on how the layers are grouped,
so the overlapped step must reproduce the stage-by-stage sequence bit for
bit."""
import numpy as np
import pytest
import torch

import synth
from infra_fac_factors_gb300 import capi
from infra_fac_factors_gb300.step import KFACStep, LayerSpec

from gpu_util import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    ensure_built()


def run(key, steps, overlapped, n_groups):
    cfg = synth.config(key)
    specs = [LayerSpec(l.d_in, l.d_out, cfg.rows(l), cfg.batch, l.hw) for l in cfg.layers]
    st = KFACStep(specs, cfg.P, cfg.gamma, cfg.decay or 0.0, cfg.in_dtype, refine=capi.KFAC_REFINE_AUTO,
                  n_groups=n_groups)
    stream = torch.cuda.current_stream()
    for t in range(steps):
        for li in range(len(specs)):
            dd = synth.layer_inputs(cfg, t, li)
            st.set_layer_inputs(li, torch.from_numpy(dd["a"]), torch.from_numpy(dd["g"]),
                                torch.from_numpy(dd["grad"]))
        if overlapped:
            st.step(t == 0, stream)
        else:
            s = stream.cuda_stream
            st.factors(s)
            st.update_running(t == 0, s)
            st.inverse(s)
            st.precondition(s)
    torch.cuda.synchronize()
    assert capi.kfac_device_status(clear=True) == capi.KFAC_OK
    return ([o.cpu().numpy() for o in st.out], [F.inv.cpu().numpy() for F in st.factor_list()],
            [F.running.cpu().numpy() for F in st.factor_list()])


@pytest.mark.parametrize("key,steps,n_groups", [("mlp", 3, 2), ("mlp", 2, 4), ("resnet_conv", 1, 3), ("bert_layer", 2, 4)])
def test_overlapped_step_equals_stage_sequence(key, steps, n_groups):
    seq = run(key, steps, False, n_groups)
    ovl = run(key, steps, True, n_groups)
    for a_list, b_list in zip(seq, ovl):
        for a, b in zip(a_list, b_list):
            assert np.array_equal(a, b)


def test_kernel_profile_counts_the_step_work():
    # one steady-state step of one encoder layer with per-launch events on:
    # the recorded work of the factor and running-average launches is the
    # step's algorithmic work, and every kind of the default path appears
    cfg = synth.config("bert_layer")
    specs = [LayerSpec(l.d_in, l.d_out, cfg.rows(l), cfg.batch, l.hw) for l in cfg.layers]
    st = KFACStep(specs, cfg.P, cfg.gamma, cfg.decay, cfg.in_dtype, refine=capi.KFAC_REFINE_AUTO, n_groups=2)
    for li in range(len(specs)):
        dd = synth.device_layer_inputs(cfg, 0, li)
        st.set_layer_inputs(li, dd["a"], dd["g"], dd["grad"])
    st.step(first_step=True)
    torch.cuda.synchronize()
    capi.kfac_profile(True)
    st.step(first_step=False)
    capi.kfac_profile(False)
    torch.cuda.synchronize()
    prof = {k: capi.kfac_profile_read(k) for k in capi.KERNEL_KINDS}
    work = st.algorithmic_work()
    assert abs(prof["syrk"]["work"] - work["factor_flops"]) <= 1e-9 * work["factor_flops"]
    assert abs(prof["running"]["work"] - work["update_bytes"]) <= 1e-9 * work["update_bytes"]
    for k in ("syrk", "running", "inv_panel", "inv_update", "inv_lauum", "gemm16", "gemm24"):
        assert prof[k]["launches"] > 0 and prof[k]["ms"] > 0, (k, prof[k])
    # the 16-bit GEMMs carry the layer's 2 M N K products; the 24-bit re-run picks its layers on the device
    assert abs(prof["gemm16"]["work"] - work["precond_flops"]) <= 1e-9 * work["precond_flops"]
    assert prof["gemm24"]["work"] == 0.0
    for k in ("inv_diag", "inv_prep", "inv_aux"):  # the inverse's CUDA-core launches, timed without work
        assert prof[k]["launches"] > 0 and prof[k]["work"] == 0.0, (k, prof[k])
    # the timeline lists the same launches on one time axis
    tl = capi.kfac_profile_timeline()
    assert len(tl) == sum(p["launches"] for p in prof.values())
    assert tl[0]["start_ms"] == 0.0 and all(0.0 <= e["start_ms"] <= e["end_ms"] for e in tl)
    for k in capi.KERNEL_KINDS:
        got = sum(e["end_ms"] - e["start_ms"] for e in tl if e["kind"] == k)
        assert abs(got - prof[k]["ms"]) <= 1e-3 * max(prof[k]["ms"], 1.0), k
