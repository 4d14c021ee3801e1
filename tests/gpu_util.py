"""Helpers shared by the GPU parity tests (no K-FAC arithmetic here)."""
import numpy as np
import torch

from infra_fac_factors_gb300 import build, capi

_built = False


def ensure_built():
    global _built
    if not _built:
        build.build()
        capi.lib()
        _built = True


def pad(v, m):
    return (v + m - 1) // m * m


def stream():
    return torch.cuda.current_stream().cuda_stream


def upper_tile_mask(d):
    r = np.arange(d)[:, None]
    c = np.arange(d)[None, :]
    return c >= (r // 128) * 128


def rel_fro(got, ref, mask=None):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if mask is not None:
        got, ref = got[mask], ref[mask]
    den = np.linalg.norm(ref)
    return np.linalg.norm(got - ref) / (den if den > 0 else 1.0)


def residual(X, D):
    X = np.asarray(X, np.float64)
    D = np.asarray(D, np.float64)
    n = D.shape[0]
    return np.linalg.norm(X @ D - np.eye(n)) / np.sqrt(n)


def to_dev(x_f32, dtype, ld):
    """Host float32 array (values exact in `dtype`) -> padded device tensor."""
    rows, d = x_f32.shape
    tdt = torch.bfloat16 if dtype == capi.KFAC_BF16 else torch.float32
    t = torch.zeros((rows, ld), dtype=tdt, device="cuda")
    t[:, :d] = torch.from_numpy(np.ascontiguousarray(x_f32)).to("cuda").to(tdt)
    return t


def upper_from_full(S, d, ld):
    """fp32 device buffer d x ld holding `S` (float64 host) on the upper tiles
    and NaN elsewhere (lower tiles and padding must never be read)."""
    buf = np.full((d, ld), np.nan, dtype=np.float32)
    m = upper_tile_mask(d)
    buf[:, :d][m] = S[m]
    return torch.from_numpy(buf).cuda()
