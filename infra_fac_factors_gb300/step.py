"""One K-FAC preconditioning step over a list of layers, through the C ABI.

``KFACStep`` owns the device buffers of every layer (PyTorch allocates them;
nothing else of PyTorch is used) and issues, per step, the library calls of
the step in order (SPD-KFAC §II-B/§II-C):

  1. kfac_spatial_sum       (conv layers: per-sample sum of g over H*W)
  2. kfac_factors           per-worker factors A^p, G^p of all layers
     kfac_conv_factors      (conv layers given by their NHWC activations: A
                            from the implicit im2col of a 3 x 3 convolution)
  3. kfac_update_running    mean over workers, running average, damping
  4. kfac_damped_inverse    (A + gamma I)^-1, (G + gamma I)^-1 of all factors
  5. kfac_precondition      (G + gamma I)^-1 grad (A + gamma I)^-1 of all layers

``step`` can overlap 2 and 3 (``n_groups`` > 1): the layers are cut into
groups of about equal factor work, and the running-average pass of group i
(memory-bound, on a second stream) runs while the tensor-core factor pass of
group i + 1 runs on the caller's stream.  The default is one group, i.e. the
two passes in sequence: on the BERT-large workload the overlap measured
slower (56.0 ms per step with eight groups, 55.0 ms with one), both passes
contending for HBM (the factor pass writes the worker factors that the
running-average pass reads).

Buffers are row-major with leading dimensions padded to 16-byte multiples
(bf16 inputs) or 128-byte multiples (fp32 factor matrices).
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Tuple

import torch

from . import capi


def _pad(v: int, m: int) -> int:
    return (v + m - 1) // m * m


@dataclasses.dataclass
class LayerSpec:
    d_in: int            # factor A dimension (incl. bias column)
    d_out: int           # factor G dimension
    rows: int            # rows of a and g per step
    batch: int           # samples per step (conv: rows = batch * hw)
    hw: int = 1          # spatial positions (1 for linear layers)
    # (H, W) for a 3 x 3 conv layer (stride 1, padding 1) whose input is given
    # as NHWC activations (batch x H x W x C, C = (d_in - 1) / 9, bf16); its A
    # factor then comes from kfac_conv_factors instead of a patch matrix
    image: Optional[Tuple[int, int]] = None


def layer_groups(layers: Sequence[LayerSpec], n_groups: int):
    """Cut the layers into at most `n_groups` contiguous, non-empty groups of
    about equal factor work (rows * d^2 summed over both factors); returns
    [(first, end)] covering every layer once, in order."""
    work = [L.rows * L.d_in ** 2 + (L.batch if L.hw > 1 else L.rows) * L.d_out ** 2 for L in layers]
    total = float(sum(work)) or 1.0
    n = max(1, min(n_groups, len(layers)))
    bounds, acc, cut = [0], 0.0, 1
    for li, w in enumerate(work):
        acc += w
        if cut < n and acc >= total * cut / n and li + 1 < len(layers):
            bounds.append(li + 1)
            cut += 1
    bounds.append(len(layers))
    return list(zip(bounds[:-1], bounds[1:]))


class FactorBufs:
    def __init__(self, d: int, P: int, device):
        self.d = d
        self.ld = _pad(d, 32)
        self.P = P
        self.stride = d * self.ld
        self.shards = torch.zeros((P, d, self.ld), dtype=torch.float32, device=device)
        self.running = torch.zeros((d, self.ld), dtype=torch.float32, device=device)
        self.damped = torch.zeros((d, self.ld), dtype=torch.float32, device=device)
        self.inv = torch.zeros((d, self.ld), dtype=torch.float32, device=device)


class KFACStep:
    def __init__(self, layers: Sequence[LayerSpec], P: int, gamma: float, decay: float, in_dtype: str,
                 refine: int = capi.KFAC_REFINE_AUTO, device="cuda", n_groups: int = 1,
                 precond_precision: int = capi.KFAC_PRECOND_AUTO, inverse_order: str = "size",
                 weight_lr: Optional[float] = None):
        self.layers = list(layers)
        self.P = P
        self.gamma = float(gamma)
        self.decay = float(decay)
        self.in_dtype = in_dtype
        self.refine = refine
        self.precond_precision = precond_precision
        if inverse_order not in ("size", "call"):
            raise ValueError("inverse_order is 'size' or 'call'")
        self.inverse_order = inverse_order
        # with weight_lr, the preconditioning call also steps weight[l] -= lr * out[l]
        self.weight_lr = weight_lr
        self.device = torch.device(device)
        tdt = torch.bfloat16 if in_dtype == "bf16" else torch.float32
        self.kdt = capi.KFAC_BF16 if in_dtype == "bf16" else capi.KFAC_FP32
        vec = 8 if in_dtype == "bf16" else 4
        dev = self.device
        self.a, self.g, self.gs, self.grad, self.out, self.weight = [], [], [], [], [], []
        self.fa: List[FactorBufs] = []
        self.fg: List[FactorBufs] = []
        for L in self.layers:
            if L.rows % P:
                raise ValueError("rows must split into P equal shards")
            if L.image is not None:
                H, W = L.image
                C = (L.d_in - 1) // 9
                if in_dtype != "bf16" or 9 * C + 1 != L.d_in or C % 64 or H * W != L.hw or L.rows != L.batch * L.hw:
                    raise ValueError("a layer given by its image needs bf16, d_in = 9 C + 1 with C % 64 == 0 "
                                     "and rows = batch * H * W")
                self.a.append(torch.zeros((L.batch, H, W, C), dtype=tdt, device=dev))
            else:
                self.a.append(torch.zeros((L.rows, _pad(L.d_in, vec)), dtype=tdt, device=dev))
            self.g.append(torch.zeros((L.rows, _pad(L.d_out, vec)), dtype=tdt, device=dev))
            if L.hw > 1:
                if L.batch % P:
                    raise ValueError("conv layers need batch % P == 0")
                self.gs.append(torch.zeros((L.batch, _pad(L.d_out, 4)), dtype=torch.float32, device=dev))
            else:
                self.gs.append(None)
            self.grad.append(torch.zeros((L.d_out, _pad(L.d_in, 32)), dtype=torch.float32, device=dev))
            self.out.append(torch.zeros((L.d_out, _pad(L.d_in, 32)), dtype=torch.float32, device=dev))
            if weight_lr is not None:
                self.weight.append(torch.zeros((L.d_out, _pad(L.d_in, 32)), dtype=torch.float32, device=dev))
            self.fa.append(FactorBufs(L.d_in, P, dev))
            self.fg.append(FactorBufs(L.d_out, P, dev))
        nf = 2 * len(self.layers)
        self.info = torch.zeros(nf, dtype=torch.int32, device=dev)
        self.route = torch.zeros(nf, dtype=torch.int32, device=dev)
        # MMAs per multiply-add each layer's preconditioned gradient came from (3 or 6)
        self.pc_route = torch.zeros(len(self.layers), dtype=torch.int32, device=dev)
        self._build_args()
        self._build_groups(n_groups)
        self._side = torch.cuda.Stream(device=dev)
        self._ev_fac = [torch.cuda.Event() for _ in self._groups]
        self._ev_side = torch.cuda.Event()
        self.inv_ws_bytes = capi.kfac_damped_inverse_workspace(self._inv_args, refine)
        self.pc_ws_bytes = capi.kfac_precondition_workspace(self._pc_args)
        if self.inv_ws_bytes == 0 or self.pc_ws_bytes == 0:
            raise ValueError("workspace query rejected the arguments")
        self.inv_ws = torch.empty(self.inv_ws_bytes, dtype=torch.uint8, device=dev)
        self.pc_ws = torch.empty(self.pc_ws_bytes, dtype=torch.uint8, device=dev)

    # ------------------------------------------------------------------ argument arrays
    def factor_list(self):
        """All factors in call order: A of every layer, then G of every layer."""
        return self.fa + self.fg

    def _build_args(self):
        P = self.P
        fa_main, fa_fp32 = [], []   # factors from a (dtype of a), factors from fp32 spatial sums
        self._fac_conv = {}         # layer -> A factor from NHWC activations
        self._main_index = {}       # ("A" | "G", layer) -> index in fa_main
        for li, L in enumerate(self.layers):
            A = self.fa[li]
            if L.image is not None:
                B, H, W, C = self.a[li].shape
                self._fac_conv[li] = capi.kfac_conv_factor_args(self.a[li].data_ptr(), B, H, W, C,
                                                                A.shards.data_ptr(), A.ld, A.stride,
                                                                1.0 / (L.rows // P))
                continue
            self._main_index[("A", li)] = len(fa_main)
            fa_main.append(capi.kfac_factor_args(self.a[li].data_ptr(), L.rows, L.d_in, self.a[li].shape[1],
                                                 A.shards.data_ptr(), A.ld, A.stride, 1.0 / (L.rows // P)))
        for li, L in enumerate(self.layers):
            G = self.fg[li]
            if L.hw > 1:
                gs = self.gs[li]
                fa_fp32.append(capi.kfac_factor_args(gs.data_ptr(), L.batch, L.d_out, gs.shape[1],
                                                     G.shards.data_ptr(), G.ld, G.stride, 1.0 / (L.batch // P)))
            else:
                self._main_index[("G", li)] = len(fa_main)
                fa_main.append(capi.kfac_factor_args(self.g[li].data_ptr(), L.rows, L.d_out, self.g[li].shape[1],
                                                     G.shards.data_ptr(), G.ld, G.stride, 1.0 / (L.rows // P)))
        self._fac_main = fa_main
        self._fac_fp32 = fa_fp32
        self._run_args = [capi.kfac_running_args(F.shards.data_ptr(), F.stride, F.running.data_ptr(),
                                                 F.damped.data_ptr(), F.d, F.ld) for F in self.factor_list()]
        # Inverse batch order: largest factors first ("size", the longest-job-first
        # rule the pages' inverse placement uses), so that the persistent grids of
        # every sweep launch start on the longest jobs; or the factor_list order.
        # info[] and route[] follow the batch order; inv_order[i] is the
        # factor_list index of batch entry i.
        facs = self.factor_list()
        order = list(range(len(facs)))
        if self.inverse_order == "size":
            order.sort(key=lambda i: -facs[i].d)
        self.inv_order = order
        self._inv_args = [capi.kfac_inverse_args(facs[i].damped.data_ptr(), facs[i].inv.data_ptr(), facs[i].d,
                                                 facs[i].ld, facs[i].ld) for i in order]
        self._pc_args = []
        for li, L in enumerate(self.layers):
            A, G = self.fa[li], self.fg[li]
            W = self.weight[li] if self.weight_lr is not None else None
            self._pc_args.append(capi.kfac_precond_args(
                G.inv.data_ptr(), G.ld, self.grad[li].data_ptr(), self.grad[li].shape[1],
                A.inv.data_ptr(), A.ld, self.out[li].data_ptr(), self.out[li].shape[1], L.d_out, L.d_in,
                W.data_ptr() if W is not None else None, W.shape[1] if W is not None else 0,
                float(self.weight_lr or 0.0)))

    def _build_groups(self, n_groups: int):
        """The argument arrays of each layer group (see layer_groups)."""
        nl = len(self.layers)
        self._groups = []
        for b, e in layer_groups(self.layers, n_groups):
            lis = range(b, e)
            main = [self._fac_main[self._main_index[(side, li)]] for side in ("A", "G") for li in lis
                    if (side, li) in self._main_index]
            fp32 = [self._fac_fp32[self._n_conv_before(li)] for li in lis if self.layers[li].hw > 1]
            conv = [self._fac_conv[li] for li in lis if li in self._fac_conv]
            run = [self._run_args[li] for li in lis] + [self._run_args[nl + li] for li in lis]
            self._groups.append((list(lis), main, fp32, conv, run))

    def _n_conv_before(self, li: int) -> int:
        return sum(1 for L in self.layers[:li] if L.hw > 1)

    # ------------------------------------------------------------------ inputs
    def set_layer_inputs(self, li: int, a: torch.Tensor, g: torch.Tensor, grad: torch.Tensor,
                         non_blocking: bool = False):
        """Copy one layer's inputs (any device) into the padded device buffers;
        `a` is the NHWC activation tensor for a layer given by its image."""
        L = self.layers[li]
        if L.image is not None:
            self.a[li].copy_(a, non_blocking=non_blocking)
        else:
            self.a[li][:, :L.d_in].copy_(a, non_blocking=non_blocking)
        self.g[li][:, :L.d_out].copy_(g, non_blocking=non_blocking)
        self.grad[li][:, :L.d_in].copy_(grad, non_blocking=non_blocking)

    # ------------------------------------------------------------------ the step
    def stream_handle(self, stream: Optional[torch.cuda.Stream] = None) -> int:
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        return s.cuda_stream

    def factors(self, stream: int):
        P = self.P
        for li, L in enumerate(self.layers):
            if L.hw > 1:
                gs = self.gs[li]
                capi.kfac_spatial_sum(self.g[li].data_ptr(), self.kdt, L.batch, L.hw, L.d_out,
                                      self.g[li].shape[1], gs.data_ptr(), gs.shape[1], stream)
        if self._fac_main:
            capi.kfac_factors(self._fac_main, self.kdt, P, 0, stream)
        if self._fac_conv:
            capi.kfac_conv_factors(list(self._fac_conv.values()), P, 0, stream)
        if self._fac_fp32:
            capi.kfac_factors(self._fac_fp32, capi.KFAC_FP32, P, 0, stream)

    def update_running(self, first_step: bool, stream: int):
        decay = 0.0 if first_step else self.decay
        capi.kfac_update_running(self._run_args, self.P, decay, self.gamma, first_step, stream)

    def inverse(self, stream: int):
        capi.kfac_damped_inverse(self._inv_args, 0.0, self.refine, self.info.data_ptr(), self.route.data_ptr(),
                                 self.inv_ws.data_ptr(), self.inv_ws_bytes, stream)

    def precondition(self, stream: int):
        capi.kfac_precondition(self._pc_args, self.precond_precision, self.pc_route.data_ptr(),
                               self.pc_ws.data_ptr(), self.pc_ws_bytes, stream)

    def factors_and_running(self, first_step: bool, stream: Optional[torch.cuda.Stream] = None):
        """Stages 2 and 3, the running-average pass of each layer group on a
        second stream behind the factor pass of the next group; returns when
        both are ordered before later work on `stream`."""
        main = stream if stream is not None else torch.cuda.current_stream(self.device)
        ms, ss = main.cuda_stream, self._side.cuda_stream
        decay = 0.0 if first_step else self.decay
        self._side.wait_stream(main)  # the side stream's earlier work must not overtake the inputs
        for (lis, fmain, ffp32, fconv, run), ev in zip(self._groups, self._ev_fac):
            for li in lis:
                L = self.layers[li]
                if L.hw > 1:
                    gs = self.gs[li]
                    capi.kfac_spatial_sum(self.g[li].data_ptr(), self.kdt, L.batch, L.hw, L.d_out,
                                          self.g[li].shape[1], gs.data_ptr(), gs.shape[1], ms)
            if fmain:
                capi.kfac_factors(fmain, self.kdt, self.P, 0, ms)
            if fconv:
                capi.kfac_conv_factors(fconv, self.P, 0, ms)
            if ffp32:
                capi.kfac_factors(ffp32, capi.KFAC_FP32, self.P, 0, ms)
            ev.record(main)
            self._side.wait_event(ev)
            capi.kfac_update_running(run, self.P, decay, self.gamma, first_step, ss)
        self._ev_side.record(self._side)
        main.wait_event(self._ev_side)

    def step(self, first_step: bool, stream: Optional[torch.cuda.Stream] = None, marks=None):
        """One whole step on `stream`; `marks` (optional, four CUDA events) are
        recorded at its start and after stages 2+3, 4 and 5."""
        main = stream if stream is not None else torch.cuda.current_stream(self.device)
        s = main.cuda_stream
        if marks is not None:
            marks[0].record(main)
        self.factors_and_running(first_step, main)
        if marks is not None:
            marks[1].record(main)
        self.inverse(s)
        if marks is not None:
            marks[2].record(main)
        self.precondition(s)
        if marks is not None:
            marks[3].record(main)

    # ------------------------------------------------------------------ counts
    def algorithmic_work(self):
        """Per-step algorithmic work of each stage (upper-triangle convention).

        factor flops: 2 * rows * d(d+1)/2 per factor; update bytes: (P + 1 reads
        + 2 writes) * 4 * d(d+1)/2 per factor (P + 2 accesses on a first step);
        inverse flops: d^3 per factor; precondition flops: 2 d_out d_in (d_out + d_in).
        """
        fac = upd = inv = pc = 0
        for li, L in enumerate(self.layers):
            rows_g = L.batch if L.hw > 1 else L.rows
            for d, rows in ((L.d_in, L.rows), (L.d_out, rows_g)):
                tri = d * (d + 1) // 2
                fac += 2 * rows * tri
                upd += (self.P + 3) * 4 * tri
                inv += d ** 3
            pc += 2 * L.d_out * L.d_in * (L.d_out + L.d_in)
        return dict(factor_flops=fac, update_bytes=upd, inverse_flops=inv, precond_flops=pc)
