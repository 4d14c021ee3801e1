"""The C-ABI library without a GPU: it loads, exports every symbol kfac.h
declares, its struct layouts agree with a C compiler's, its tile map equals
the oracle's enumeration bit for bit, and invalid arguments are rejected on
the host before any launch."""
import ctypes as C
import os
import re
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from infra_fac_factors_gb300 import build, capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kfac.h")


@pytest.fixture(scope="module", autouse=True)
def built_library():
    build.build()
    return capi.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kfac_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_function():
    names = declared_functions()
    assert len(names) == 22
    out = subprocess.run(["nm", "-D", "--defined-only", capi.library_path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (kfac_[a-z_0-9]+)$", out, flags=re.M))
    for n in names:
        assert n in exported, n
        assert hasattr(capi.lib(), n)
    assert set(names) == set(capi.exported_symbols)


def test_struct_layouts_match_c_compiler():
    src = r"""
#include <stdio.h>
#include <stddef.h>
#include "kfac.h"
#define S(t) printf(#t " %zu\n", sizeof(t));
#define O(t, f) printf(#t "." #f " %zu\n", offsetof(t, f));
int main(void) {
  S(kfac_factor_args) O(kfac_factor_args, out) O(kfac_factor_args, scale)
  S(kfac_running_args) O(kfac_running_args, damped) O(kfac_running_args, ld)
  S(kfac_inverse_args) O(kfac_inverse_args, ld_out)
  S(kfac_precond_args) O(kfac_precond_args, out) O(kfac_precond_args, d_in)
  S(kfac_conv_factor_args) O(kfac_conv_factor_args, C) O(kfac_conv_factor_args, out)
  O(kfac_conv_factor_args, scale)
  S(kfac_pack_args) O(kfac_pack_args, ld) O(kfac_pack_args, packed)
  return 0;
}
"""
    with tempfile.TemporaryDirectory() as td:
        c = os.path.join(td, "l.c")
        exe = os.path.join(td, "l")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-I", os.path.dirname(HEADER), c, "-o", exe], check=True)
        lines = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    got = dict(l.split() for l in lines if l)
    for name, st in (("kfac_factor_args", capi.kfac_factor_args), ("kfac_running_args", capi.kfac_running_args),
                     ("kfac_inverse_args", capi.kfac_inverse_args), ("kfac_precond_args", capi.kfac_precond_args),
                     ("kfac_conv_factor_args", capi.kfac_conv_factor_args),
                     ("kfac_pack_args", capi.kfac_pack_args)):
        assert int(got[name]) == C.sizeof(st), name
        for key, val in got.items():
            if key.startswith(name + "."):
                field = key.split(".")[1]
                assert getattr(st, field).offset == int(val), key


@pytest.mark.parametrize("d", [1, 2, 10, 64, 127, 128, 129, 255, 256, 257, 385, 577, 1025, 1153, 2305, 3072,
                               4096, 4097, 4609])
def test_factor_tile_map_bit_exact(d):
    assert capi.kfac_factor_tile_map(d) == oracle.factor_tile_units(d, 128, 256)


def test_status_strings_and_version():
    assert capi.kfac_status_string(0) == "KFAC_OK"
    assert capi.kfac_status_string(5) == "KFAC_ERR_TIMEOUT"
    assert capi.kfac_status_string(99) == "KFAC_ERR_UNKNOWN"
    assert capi.kfac_version() >= 100


# Fake (never dereferenced) device addresses: validation rejects before any CUDA call.
A16 = 1 << 20


def fa(**kw):
    base = dict(x=A16, rows=64, d=10, ld_x=16, out=A16 * 2, ld_out=16, stride_out=160, scale=1 / 32)
    base.update(kw)
    return capi.kfac_factor_args(**base)


@pytest.mark.parametrize("kw,dtype,P", [
    (dict(x=None), capi.KFAC_BF16, 2),
    (dict(x=A16 + 2), capi.KFAC_BF16, 2),          # misaligned base
    (dict(rows=63), capi.KFAC_BF16, 2),            # rows % P
    (dict(d=0), capi.KFAC_BF16, 2),
    (dict(ld_x=12), capi.KFAC_BF16, 2),            # bf16 ld not a multiple of 8
    (dict(ld_x=8), capi.KFAC_BF16, 2),             # ld < d
    (dict(ld_out=18), capi.KFAC_BF16, 2),          # fp32 ld not a multiple of 4
    (dict(stride_out=100), capi.KFAC_BF16, 2),     # shards overlap
    (dict(scale=float("nan")), capi.KFAC_BF16, 2),
    (dict(), 7, 2),                                # dtype
    (dict(), capi.KFAC_BF16, 0),                   # P
])
def test_factors_rejects_invalid(kw, dtype, P):
    assert capi.kfac_factors([fa(**kw)], dtype, P, check=False) == capi.KFAC_ERR_INVALID_ARG


def ra(**kw):
    base = dict(shards=A16, stride_shard=16 * 16, running=A16 * 2, damped=A16 * 3, d=16, ld=16)
    base.update(kw)
    return capi.kfac_running_args(**base)


@pytest.mark.parametrize("kw,decay,gamma,P", [
    (dict(), 1.0, 1e-3, 2), (dict(), -0.1, 1e-3, 2), (dict(), 0.9, -1e-3, 2),
    (dict(), 0.9, float("inf"), 2), (dict(damped=A16 * 2), 0.9, 1e-3, 2),
    (dict(ld=14), 0.9, 1e-3, 2), (dict(stride_shard=16), 0.9, 1e-3, 2), (dict(shards=None), 0.9, 1e-3, 2),
    (dict(), 0.9, 1e-3, 0),
])
def test_update_running_rejects_invalid(kw, decay, gamma, P):
    assert capi.kfac_update_running([ra(**kw)], P, decay, gamma, False, check=False) == capi.KFAC_ERR_INVALID_ARG


def ia(**kw):
    base = dict(damped=A16, inv=A16 * 2, d=8, ld_in=8, ld_out=8)
    base.update(kw)
    return capi.kfac_inverse_args(**base)


def test_inverse_rejects_invalid():
    ok = [ia()]
    ws = capi.kfac_damped_inverse_workspace(ok, capi.KFAC_REFINE_AUTO)
    assert ws > 0
    assert capi.kfac_damped_inverse_workspace(ok, capi.KFAC_REFINE_NONE) <= ws
    for bad in (ia(d=0), ia(ld_in=6), ia(inv=A16), ia(ld_out=7), ia(damped=None)):
        assert capi.kfac_damped_inverse_workspace([bad], 1) == 0
        assert capi.kfac_damped_inverse([bad], 0.0, 1, A16, 0, A16 * 4, ws, check=False) == capi.KFAC_ERR_INVALID_ARG
    assert capi.kfac_damped_inverse(ok, 0.0, 3, A16, 0, A16 * 4, ws, check=False) == capi.KFAC_ERR_INVALID_ARG
    assert capi.kfac_damped_inverse(ok, -1.0, 1, A16, 0, A16 * 4, ws, check=False) == capi.KFAC_ERR_INVALID_ARG
    assert capi.kfac_damped_inverse(ok, 0.0, 1, 0, 0, A16 * 4, ws, check=False) == capi.KFAC_ERR_INVALID_ARG
    assert capi.kfac_damped_inverse(ok, 0.0, 1, A16, 0, A16 * 4, ws - 1, check=False) == capi.KFAC_ERR_WORKSPACE
    assert capi.kfac_damped_inverse(ok, 0.0, 1, A16, 0, A16 * 4 + 16, ws, check=False) == capi.KFAC_ERR_WORKSPACE
    assert capi.kfac_damped_inverse(ok, 0.0, 1, A16, 0, 0, ws, check=False) == capi.KFAC_ERR_WORKSPACE


def pa(**kw):
    base = dict(inv_g=A16, ld_g=8, grad=A16 * 2, ld_grad=12, inv_a=A16 * 3, ld_a=12, out=A16 * 4, ld_out=12,
                d_out=8, d_in=12)
    base.update(kw)
    return capi.kfac_precond_args(**base)


def test_precondition_rejects_invalid():
    ws = capi.kfac_precondition_workspace([pa()])
    # four operands as three bf16 slices: grad 8x16, inv_a 12x16, inv_g 8x8, tmp^T 12x8, each 256-B aligned;
    # then the probe vectors (12 + 8 rows of 8 fp32), the 2 x 8 x 8 fp64 bilinear sums and the flag
    assert ws == (768 + 1280 + 512 + 768) + 768 + 1024 + 256
    assert capi.kfac_precondition_workspace([pa(weight=A16 * 6, ld_weight=12, lr=0.1)]) == ws
    for bad in (pa(d_in=0), pa(ld_g=4), pa(ld_grad=10), pa(out=A16 * 2), pa(inv_a=A16 + 4),
                # the weight step: aliasing out, misaligned, too short a row, ld not a multiple of 4
                pa(weight=A16 * 4, ld_weight=12), pa(weight=A16 * 6 + 4, ld_weight=12),
                pa(weight=A16 * 6, ld_weight=8), pa(weight=A16 * 6, ld_weight=14)):
        assert capi.kfac_precondition_workspace([bad]) == 0
        assert capi.kfac_precondition([bad], 0, 0, A16 * 5, ws, check=False) == capi.KFAC_ERR_INVALID_ARG
    assert capi.kfac_precondition([pa()], 0, 0, A16 * 5, ws - 4, check=False) == capi.KFAC_ERR_WORKSPACE
    # precision outside the enum, and a route array that is not 4-byte aligned
    assert capi.kfac_precondition([pa()], 2, 0, A16 * 5, ws, check=False) == capi.KFAC_ERR_INVALID_ARG
    assert capi.kfac_precondition([pa()], capi.KFAC_PRECOND_AUTO, A16 + 2, A16 * 5, ws,
                                  check=False) == capi.KFAC_ERR_INVALID_ARG


def ca(**kw):
    base = dict(x=A16, B=4, H=5, W=7, C=64, out=A16 * 2, ld_out=580, stride_out=577 * 580, scale=1.0)
    base.update(kw)
    return capi.kfac_conv_factor_args(**base)


@pytest.mark.parametrize("kw,P", [
    (dict(x=None), 2),
    (dict(x=A16 + 2), 2),                # misaligned activations
    (dict(out=A16 + 4), 2),              # misaligned output
    (dict(C=96), 2),                     # C % 64
    (dict(C=0), 2),
    (dict(C=7296), 2),                   # d = 9 C + 1 above the limit
    (dict(B=3), 2),                      # B % P
    (dict(H=0), 2),
    (dict(W=-1), 2),
    (dict(B=2, H=1 << 16, W=1 << 15), 2),  # B H W above 2^31 - 1
    (dict(ld_out=576), 2),               # ld_out < d
    (dict(ld_out=578), 2),               # fp32 ld not a multiple of 4
    (dict(stride_out=100), 2),           # shards overlap
    (dict(scale=float("inf")), 2),
    (dict(), 0),                         # P
])
def test_conv_factors_rejects_invalid(kw, P):
    assert capi.kfac_conv_factors([ca(**kw)], P, check=False) == capi.KFAC_ERR_INVALID_ARG


def test_spatial_sum_rejects_invalid():
    f = capi.kfac_spatial_sum
    assert f(0, 0, 2, 4, 8, 8, A16, 8, check=False) == capi.KFAC_ERR_INVALID_ARG
    assert f(A16, 0, 2, 4, 8, 4, A16, 8, check=False) == capi.KFAC_ERR_INVALID_ARG
    assert f(A16, 0, 0, 4, 8, 8, A16, 8, check=False) == capi.KFAC_ERR_INVALID_ARG
    assert f(A16, 1, 2, 4, 8, 8, A16, 6, check=False) == capi.KFAC_ERR_INVALID_ARG


def test_pack_unpack_reject_invalid():
    pk = lambda **kw: capi.kfac_pack_args(**{**dict(mat=A16, d=10, ld=12, packed=A16 * 64), **kw})
    for bad in (pk(mat=0), pk(packed=0), pk(mat=A16 + 4), pk(packed=A16 * 64 + 2), pk(d=0), pk(d=65537),
                pk(ld=9), pk(ld=14), pk(packed=A16 + 40),  # packed overlapping mat
                pk(packed=A16 - 16)):                        # mat overlapping packed's tail
        assert capi.kfac_pack_upper([bad], check=False) == capi.KFAC_ERR_INVALID_ARG
        assert capi.kfac_unpack_upper([bad], True, check=False) == capi.KFAC_ERR_INVALID_ARG
    assert capi.kfac_pack_upper([], check=False) == capi.KFAC_OK
    assert capi.kfac_unpack_upper([], check=False) == capi.KFAC_OK


def test_wait_selftest_rejects_limits_outside_the_kernels_range():
    assert capi.kfac_wait_selftest(10, check=False) == capi.KFAC_ERR_INVALID_ARG
    assert capi.kfac_wait_selftest(5_000_000_000, check=False) == capi.KFAC_ERR_INVALID_ARG


def test_empty_calls_are_no_ops():
    assert capi.kfac_factors([], capi.KFAC_BF16, 1, check=False) == capi.KFAC_OK
    assert capi.kfac_conv_factors([], 1, check=False) == capi.KFAC_OK
    assert capi.kfac_update_running([], 1, 0.5, 0.0, True, check=False) == capi.KFAC_OK
    assert capi.kfac_precondition([], 0, 0, 0, 0, check=False) == capi.KFAC_OK


def test_constant_time_tile_map_equals_enumeration():
    # the kernels decode work units with factor_unit_fast; it must agree with the
    # enumerated map (factor_unit, pinned to the oracle above) unit for unit
    src = r"""
#include <cstdio>
#include "tilemap.cuh"
using namespace kfac;
int main() {
  long long bad = 0, n = 0;
  const int big[] = {16384, 32768, 65536};
  for (int q = 0; q < 3000 + 3; ++q) {
    const int d = q < 3000 ? q + 1 + (q / 1000) * 2000 : big[q - 3000];
    const long long nu = factor_units(d);
    for (long long t = 0; t < nu; ++t, ++n) {
      int i1, w1, i2, j2, w2; int64_t j1;
      factor_unit(d, t, i1, j1, w1);
      factor_unit_fast(d, (int)t, i2, j2, w2);
      bad += (i1 != i2 || j1 != j2 || w1 != w2);
    }
  }
  printf("%lld %lld\n", n, bad);
  return 0;
}
"""
    csrc = os.path.join(ROOT, "infra_fac_factors_gb300", "csrc")
    with tempfile.TemporaryDirectory() as td:
        c = os.path.join(td, "t.cpp")
        exe = os.path.join(td, "t")
        open(c, "w").write(src)
        subprocess.run(["g++", "-O2", "-std=c++17", "-D__host__=", "-D__device__=", "-I", csrc, c, "-o", exe],
                       check=True)
        n, bad = map(int, subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split())
    # every unit of every size decoded: sum over the sizes of 2 * n0 (n0 + 1) / 2, n0 = ceil(d / 256)
    sizes = [q + 1 + (q // 1000) * 2000 for q in range(3000)] + [16384, 32768, 65536]
    assert n == sum((-(-d // 256)) * (-(-d // 256) + 1) for d in sizes) and bad == 0


def test_profile_api_without_launches():
    capi.kfac_profile(True)
    for kind in capi.KERNEL_KINDS:
        assert capi.kfac_profile_read(kind) == {"launches": 0, "ms": 0.0, "work": 0.0}
    assert capi.kfac_profile_count() == 0 and capi.kfac_profile_timeline() == []
    capi.kfac_profile(False)
    with pytest.raises(capi.KFACError):
        capi.kfac_profile_read(len(capi.KERNEL_KINDS))
    with pytest.raises(capi.KFACError):
        capi.kfac_profile_launch(0)


def _run_host_program(src):
    csrc = os.path.join(ROOT, "infra_fac_factors_gb300", "csrc")
    with tempfile.TemporaryDirectory() as td:
        c = os.path.join(td, "t.cpp")
        exe = os.path.join(td, "t")
        open(c, "w").write(src)
        subprocess.run(["g++", "-O2", "-std=c++17", "-D__host__=", "-D__device__=", "-I", csrc, c, "-o", exe],
                       check=True)
        return subprocess.run([exe], capture_output=True, text=True, check=True).stdout


def test_conv_kblock_positions_equal_division():
    # the conv factor kernel steps each k-block's first output position by 64
    # with carries; it must equal (n, h, w) = divmod of the row index, for every
    # image size up to 70 x 70 and a few wide / tall ones, over 40 k-blocks past
    # a worker's last image
    src = r"""
#include <cstdio>
#include "conv_geom.cuh"
using namespace kfac;
int main() {
  long long bad = 0, n_checked = 0;
  auto check = [&](int H, int W) {
    const ConvGeom g = make_conv_geom(64, H, W, 64);
    int n = 0, h = 0, w = 0;
    const long long hw = (long long)H * W;
    const long long blocks = (3 * hw + 63) / 64 + 40;
    for (long long kb = 0; kb < blocks; ++kb, ++n_checked) {
      const long long lp = kb * 64;
      bad += (n != lp / hw || h != (lp % hw) / W || w != lp % W);
      conv_step(g, n, h, w);
    }
  };
  for (int H = 1; H <= 70; ++H)
    for (int W = 1; W <= 70; ++W) check(H, W);
  const int odd[][2] = {{1, 1000}, {1000, 1}, {3, 4097}, {224, 224}, {2, 63}, {2, 65}};
  for (auto& s : odd) check(s[0], s[1]);
  printf("%lld %lld\n", n_checked, bad);
  return 0;
}
"""
    n, bad = map(int, _run_host_program(src).split())
    assert n > 100000 and bad == 0


@pytest.mark.parametrize("C", [64, 128, 192, 512])
def test_conv_box_sources_follow_the_oracle_patch_columns(C):
    # box q of the patch matrix: the (tap, first channel) the kernel loads for
    # it, checked column by column against oracle.im2col3x3 on an image whose
    # every pixel value encodes its (h, w, c)
    src = r"""
#include <cstdio>
#include "conv_geom.cuh"
using namespace kfac;
int main() {
  const int C = %d;
  const ConvGeom g = make_conv_geom(C, 1, 1, 64);
  for (int q = 0; q < 9 * C / 64 + 3; ++q) {
    const ConvBox b = conv_box_source(g, q);
    printf("%%d %%d %%d %%d %%d\n", q, b.kind, b.dh, b.dw, b.c0);
  }
  return 0;
}
""" % C
    boxes = [tuple(map(int, l.split())) for l in _run_host_program(src).strip().splitlines()]
    H = W = 3
    x = np.zeros((1, H, W, C))
    for h in range(H):
        for w in range(W):
            x[0, h, w, :] = 1 + (h * W + w) * C + np.arange(C)  # distinct, non-zero
    X = oracle.im2col3x3(x)[H * W // 2]  # the centre position sees all nine taps inside the image
    d = 9 * C + 1
    for q, kind, dh, dw, c0 in boxes:
        for j in range(64):
            col = 64 * q + j
            if kind == 0:
                assert col < 9 * C
                want = x[0, 1 + dh - 1, 1 + dw - 1, c0 + j]
                assert X[col] == want, (q, j)
            elif kind == 1:
                assert 64 * q == 9 * C and (X[col] == 1.0 if j == 0 else col >= d)
            else:
                assert 64 * q > 9 * C


def test_residual_probes_algebra_and_spread():
    # The inverse's four probes v_p(i) = s(i) H4[p][c(i)] (probes.cuh): the
    # mean over p of v_p(i) v_p(j) is s(i) s(j) when the hashed classes agree,
    # else zero; classes and signs are balanced.  For a rank-one residual
    # u u^T, the estimate's square over the truth is mean_p (u.v_p)^2 / |u|^2;
    # with u on every 4th index (a periodic pattern that would put all of u in
    # one class if the class were i mod 4: chi-square with one degree of
    # freedom, an estimate below half the truth 38 % of the time) it must
    # behave like four independent probes (chi2_4 / 4 < 1/4: 9.0 %).  The
    # Newton step's sixteen independent probes: chi2_16 / 16 < 1/4: 0.11 %.
    # The preconditioning check's right probes (gemm_tc.h), u on every 8th
    # index: chi2_8 / 8 < 1/4: 1.9 % (i mod 8 classes would give 38 %).
    src = r"""
#include <cuda_runtime.h>
#include <cstdio>
#include <random>
#include "probes.cuh"
#include "gemm_tc.h"
using namespace kfac;
static float zright(long long i, int k) {  // right probe k of the preconditioning check, by its definition
  const unsigned hh = probe_hash((unsigned)(i >> 3));
  const int e = (int)(i & 7);
  const float sg = ((hh >> e) & 1u) ? -1.f : 1.f;
  return sg * hadamard8(k, e ^ probe_class_offset(hh, 0));
}
int main() {
  long long bad = 0;
  for (long long i = 0; i < 2048; ++i)
    for (long long j = 0; j < 2048; j += 7) {
      float a = 0.f;
      for (int p = 0; p < 4; ++p) a += probe4(i, p) * probe4(j, p);
      const float want = probe_class(i) == probe_class(j) ? 4.f * probe_base_sign(i) * probe_base_sign(j) : 0.f;
      bad += a != want;
      for (int p = 0; p < 4; ++p) bad += probe4(i, p) * probe4(i, p) != 1.f;
    }
  long long cls[4] = {0, 0, 0, 0}, pos = 0;
  for (long long i = 0; i < 1000000; ++i) {
    ++cls[probe_class(i)];
    pos += probe_base_sign(i) > 0.f;
  }
  std::mt19937_64 rng(12345);
  std::normal_distribution<double> n01;
  const int d = 1024, trials = 20000;
  long long u4 = 0, u16 = 0, u8 = 0;
  std::vector<double> u(d);
  for (int t = 0; t < trials; ++t) {
    double n2 = 0.0;
    for (int i = 0; i < d; ++i) {
      u[i] = (i % 4 == 0) ? n01(rng) : 0.0;
      n2 += u[i] * u[i];
    }
    double e4 = 0.0, e16 = 0.0;
    for (int p = 0; p < 4; ++p) {
      double s = 0.0;
      for (int i = 0; i < d; i += 4) s += u[i] * probe4(i, p);
      e4 += s * s;
    }
    for (int p = 0; p < 16; ++p) {
      double s = 0.0;
      for (int i = 0; i < d; i += 4) s += u[i] * probe16(i, p);
      e16 += s * s;
    }
    u4 += e4 / 4.0 / n2 < 0.25;
    u16 += e16 / 16.0 / n2 < 0.25;
    double m2 = 0.0, e8 = 0.0;
    for (int i = 0; i < d; i += 8) m2 += u[i] * u[i];
    for (int k = 0; k < 8; ++k) {
      double s = 0.0;
      for (int i = 0; i < d; i += 8) s += u[i] * zright(i, k);
      e8 += s * s;
    }
    u8 += e8 / 8.0 / m2 < 0.25;
  }
  printf("%lld %lld %lld %lld %lld %lld %lld %lld %lld\n", bad, cls[0], cls[1], cls[2], cls[3], pos, u4, u16, u8);
  return 0;
}
"""
    csrc = os.path.join(ROOT, "infra_fac_factors_gb300", "csrc")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    with tempfile.TemporaryDirectory() as td:
        c = os.path.join(td, "t.cpp")
        exe = os.path.join(td, "t")
        open(c, "w").write(src)
        subprocess.run(["g++", "-O2", "-std=c++17", "-I", csrc, "-I", cuda_inc, c, "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()
    bad, c0, c1, c2, c3, pos, u4, u16, u8 = map(int, out)
    assert bad == 0
    assert all(abs(cnt - 250000) < 2500 for cnt in (c0, c1, c2, c3)) and abs(pos - 500000) < 2500
    trials = 20000
    assert 0.075 < u4 / trials < 0.106, u4        # chi2_4 / 4 < 1/4: 0.0902
    assert u16 / trials < 0.004, u16              # chi2_16 / 16 < 1/4: 0.0011
    assert u8 / trials < 0.035, u8                # chi2_8 / 8 < 1/4: 0.019
