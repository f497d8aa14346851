"""One backward recalibration of an MoE layer's FC2 through the C ABI.

``Recalibration`` owns the device buffers of one layer shape (allocated once
with torch, which is used here only for device memory and streams) and
enqueues the six library calls of the path on one stream, with no host
synchronisation in between:

    lrm_route_stats -> lrm_score -> lrm_select -> lrm_compact
                    -> lrm_grouped_dgrad -> lrm_grouped_wgrad

(LRMoE Alg. 1; the input-gradient product runs before the
weight-gradient product, the order TopoEP sec. 3.3 schedules them in).
"""

from __future__ import annotations

import dataclasses
from fractions import Fraction

import torch

from . import lrm as L


def capacity(T: int, E: int, k: int, cf: Fraction) -> int:
    """C = floor(CF * T k / E), as the library computes it (lrm_capacity)."""
    return L.lrm_capacity(L.dims_of(T, E, k, 8, 8), cf)


def max_retained_rows(T: int, E: int, k: int, cf: Fraction, rho: Fraction) -> int:
    """Upper bound of sum_e ceil(rho * min(n_e, C)) over any routing, as the
    library computes it (lrm_max_rows)."""
    return L.lrm_max_rows(L.dims_of(T, E, k, 8, 8), cf, rho)


@dataclasses.dataclass
class Fc1Buffers:
    """Device buffers of the FC1 side (allocated on first use)."""

    ones: torch.Tensor  # [N] fp32: unit gate weights for compacting the FC1 inputs
    xc: torch.Tensor  # [rows, h] bf16: compacted expert inputs
    abc: torch.Tensor  # [rows, 2I] bf16: compacted saved FC1 outputs
    dh1: torch.Tensor  # [rows, 2I] bf16: FC1 output gradient
    dxc: torch.Tensor  # [rows, h] bf16: FC1 input gradient per retained row
    dW1: torch.Tensor  # [E, 2I, h] fp32
    dx: torch.Tensor  # [T, h] bf16: input gradient of every token
    ws: torch.Tensor  # pair -> row map of lrm_combine_rows


@dataclasses.dataclass
class Buffers:
    counts: torch.Tensor
    offsets: torch.Tensor
    bucket: torch.Tensor
    P: torch.Tensor
    f: torch.Tensor
    quota: torch.Tensor
    summary: torch.Tensor
    ws_route: torch.Tensor
    ws_select: torch.Tensor
    score: torch.Tensor
    sel_offsets: torch.Tensor
    sel_ids: torch.Tensor
    delta_c: torch.Tensor
    phi_c: torch.Tensor
    alpha_c: torch.Tensor
    dphi_c: torch.Tensor
    dW: torch.Tensor


class Recalibration:
    """Device buffers plus the library calls of one recalibration step."""

    def __init__(self, T, E, k, h, I, cf=Fraction(5, 4), rho=Fraction(3, 4), device=0, max_rows=None):
        self.T, self.E, self.k, self.h, self.I = int(T), int(E), int(k), int(h), int(I)
        self.N = self.T * self.k
        self.cf = Fraction(cf)
        self.rho = Fraction(rho)
        self.device = torch.device("cuda", device) if isinstance(device, int) else torch.device(device)
        self.dims = L.dims_of(T, E, k, h, I)
        self.ctx = L.lrm_create(self.device.index or 0)
        self.C = L.lrm_capacity(self.dims, self.cf)
        self.max_rows = L.lrm_max_rows(self.dims, self.cf, self.rho) if max_rows is None else int(max_rows)
        dev = self.device
        ws_bytes = L.lrm_workspace_size(self.ctx, L.LRM_OP_ROUTE_STATS, self.dims)
        ws_sel = L.lrm_workspace_size(self.ctx, L.LRM_OP_SELECT, self.dims)
        i32 = dict(dtype=torch.int32, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        bf = dict(dtype=torch.bfloat16, device=dev)
        R = max(1, self.max_rows)
        self.buf = Buffers(
            counts=torch.empty(E, **i32),
            offsets=torch.empty(E + 1, **i32),
            bucket=torch.empty(max(1, self.N), **i32),
            P=torch.empty(E, **f32),
            f=torch.empty(E, **f32),
            quota=torch.empty(E, **i32),
            summary=torch.zeros(L.SUMMARY_BYTES, dtype=torch.uint8, device=dev),
            ws_route=torch.empty(max(256, ws_bytes), dtype=torch.uint8, device=dev),
            ws_select=torch.empty(max(256, ws_sel), dtype=torch.uint8, device=dev),
            score=torch.empty(max(1, self.N), **f32),
            sel_offsets=torch.empty(E + 1, **i32),
            sel_ids=torch.empty(R, **i32),
            delta_c=torch.empty(R, h, **bf),
            phi_c=torch.empty(R, I, **bf),
            alpha_c=torch.empty(R, **f32),
            dphi_c=torch.empty(R, I, **bf),
            dW=torch.empty(E, h, I, **f32),
        )
        self.ws_bytes = self.buf.ws_route.numel()

    def close(self):
        if getattr(self, "ctx", None):
            L.lrm_destroy(self.ctx)
            self.ctx = None

    def __del__(self):  # pragma: no cover - best effort
        try:
            self.close()
        except Exception:
            pass

    # -- the steps -----------------------------------------------------------

    def route_stats(self, logits, expert_idx, stream=None, quota_override=None):
        b = self.buf
        L.lrm_route_stats(self.ctx, logits, expert_idx, self.dims, self.cf, self.rho, b.counts, b.offsets,
                          b.bucket, b.P, b.f, b.quota, b.summary, b.ws_route, self.ws_bytes, stream)
        if quota_override is not None:
            b.quota.copy_(quota_override)

    def score(self, g, phi, alpha, stream=None, metric: int = L.METRIC_LRM, seed: int = 0):
        """Step 2.  `metric` selects the LRM (default) or one of the ablation's
        alternatives (gradient L2, gradient L1, seeded random)."""
        if metric == L.METRIC_LRM:
            L.lrm_score(self.ctx, g, phi, alpha, self.dims, self.buf.score, stream)
        else:
            L.lrm_score_metric(self.ctx, metric, g, phi, alpha, self.dims, seed, self.buf.score, stream)

    def select(self, stream=None, score=None):
        b = self.buf
        L.lrm_select(self.ctx, b.score if score is None else score, b.offsets, b.bucket, b.quota, self.dims,
                     self.max_rows, b.sel_offsets, b.sel_ids, b.ws_select, b.ws_select.numel(), stream)

    def compact(self, g, phi, alpha, stream=None):
        b = self.buf
        L.lrm_compact(self.ctx, g, phi, alpha, b.sel_offsets, b.sel_ids, self.dims, self.max_rows, b.delta_c,
                      b.phi_c, b.alpha_c, stream)

    def dgrad(self, W, stream=None):
        b = self.buf
        L.lrm_grouped_dgrad(self.ctx, b.delta_c, W, b.sel_offsets, self.dims, self.max_rows, b.dphi_c, stream)

    def dgrad_scatter(self, W, dphi_rows, stream=None, zero_dropped: bool = True):
        """Step 5a with the inverse mapping: the input gradient of every
        retained pair goes to its row of `dphi_rows` ([N, I] bf16, the layout
        of phi); with `zero_dropped` the rows of the other pairs become zeros."""
        b = self.buf
        L.lrm_grouped_dgrad_scatter(self.ctx, b.delta_c, W, b.sel_offsets, b.sel_ids, self.dims, self.max_rows,
                                    dphi_rows, stream)
        if zero_dropped:
            if getattr(self, "_ws_zero", None) is None:
                nbytes = L.lrm_workspace_size(self.ctx, L.LRM_OP_ZERO_DROPPED, self.dims)
                self._ws_zero = torch.empty(max(nbytes, 4), dtype=torch.uint8, device=self.buf.dW.device)
            L.lrm_zero_dropped_rows(self.ctx, b.sel_offsets, b.sel_ids, self.dims, self.max_rows, dphi_rows,
                                    self._ws_zero, self._ws_zero.numel(), stream)

    def fc1_backward(self, x, ab, W1, stream=None):
        """The FC1 side of the expert backward on the retained pairs (SwiGLU
        read), after the FC2 steps: the compacted FC1 inputs, dh1 from the FC2
        input gradient, the FC1 input gradient of every retained row, the FC1
        weight gradient and the input gradient of every token.  x [T, h] and
        ab [N, 2I] bf16 (expert inputs, saved [a | b]), W1 [E, 2I, h] bf16.
        Results: self.fc1.dW1 [E, 2I, h] fp32 and self.fc1.dx [T, h] bf16."""
        f = self._fc1_buffers()
        b = self.buf
        T, E, k, h, I = self.dims.T, self.dims.E, self.dims.k, self.dims.h, self.dims.I
        d_in = L.Dims(T, E, k, h, 2 * I)  # compact: token rows of width h, pair rows of width 2I
        d_fc1 = L.Dims(T, E, k, 2 * I, h)  # the FC2 kernels with K = 2I and output width h
        L.lrm_compact(self.ctx, x, ab, f.ones, b.sel_offsets, b.sel_ids, d_in, self.max_rows, f.xc, f.abc, None,
                      stream)
        L.lrm_swiglu_backward(self.ctx, b.dphi_c, f.abc, b.sel_offsets, self.dims, self.max_rows, f.dh1, stream)
        L.lrm_grouped_dgrad(self.ctx, f.dh1, W1, b.sel_offsets, d_fc1, self.max_rows, f.dxc, stream)
        L.lrm_grouped_wgrad(self.ctx, f.dh1, f.xc, b.sel_offsets, d_fc1, self.max_rows, 0, f.dW1, stream)
        L.lrm_combine_rows(self.ctx, f.dxc, b.sel_offsets, b.sel_ids, self.dims, self.max_rows, h, f.dx, f.ws,
                           f.ws.numel(), stream)

    def _fc1_buffers(self):
        if getattr(self, "fc1", None) is None:
            T, E, k, h, I = self.dims.T, self.dims.E, self.dims.k, self.dims.h, self.dims.I
            dev = self.buf.dW.device
            bf = dict(dtype=torch.bfloat16, device=dev)
            rows = max(self.max_rows, 1)
            ws = L.lrm_workspace_size(self.ctx, L.LRM_OP_COMBINE, self.dims)
            self.fc1 = Fc1Buffers(
                ones=torch.ones(T * k, dtype=torch.float32, device=dev),
                xc=torch.empty(rows, h, **bf), abc=torch.empty(rows, 2 * I, **bf),
                dh1=torch.empty(rows, 2 * I, **bf), dxc=torch.empty(rows, h, **bf),
                dW1=torch.empty(E, 2 * I, h, dtype=torch.float32, device=dev), dx=torch.empty(T, h, **bf),
                ws=torch.empty(max(ws, 4), dtype=torch.uint8, device=dev))
        return self.fc1

    def wgrad(self, stream=None, accumulate=0):
        b = self.buf
        L.lrm_grouped_wgrad(self.ctx, b.delta_c, b.phi_c, b.sel_offsets, self.dims, self.max_rows, accumulate,
                            b.dW, stream)

    def wgrad_bf16(self, stream=None, accumulate=0):
        """Step 5b with the weight gradient stored as bf16 in ``self.dW_bf16``
        ([E, h, I], allocated on first use)."""
        b = self.buf
        if getattr(self, "dW_bf16", None) is None:
            self.dW_bf16 = torch.zeros(self.E, self.h, self.I, dtype=torch.bfloat16, device=b.dW.device)
        L.lrm_grouped_wgrad_bf16(self.ctx, b.delta_c, b.phi_c, b.sel_offsets, self.dims, self.max_rows, accumulate,
                                 self.dW_bf16, stream)

    def backward_steps(self, g, phi, alpha, W, stream=None, metric: int = L.METRIC_LRM, seed: int = 0,
                       dw_bf16: bool = False):
        """score -> select -> compact -> dgrad -> wgrad (quotas already set);
        with `dw_bf16` the weight gradient goes to ``self.dW_bf16``."""
        self.score(g, phi, alpha, stream, metric=metric, seed=seed)
        self.select(stream)
        self.compact(g, phi, alpha, stream)
        self.dgrad(W, stream)
        if dw_bf16:
            self.wgrad_bf16(stream)
        else:
            self.wgrad(stream)

    def run(self, logits, expert_idx, g, phi, alpha, W, stream=None, dw_bf16: bool = False, side_stream=None):
        """The whole path, enqueued on one stream.  Route statistics and score
        read disjoint inputs, so with `side_stream` (a torch stream; `stream`
        must then be a torch stream or None) route statistics run on it beside
        score, and select waits for both."""
        if side_stream is None:
            self.route_stats(logits, expert_idx, stream)
            self.backward_steps(g, phi, alpha, W, stream, dw_bf16=dw_bf16)
            return
        main = torch.cuda.current_stream(self.device) if stream is None else stream
        if not isinstance(main, torch.cuda.Stream) or not isinstance(side_stream, torch.cuda.Stream):
            raise TypeError("run(side_stream=...) needs torch streams for both branches")
        fork = torch.cuda.Event()
        fork.record(main)
        side_stream.wait_event(fork)
        self.route_stats(logits, expert_idx, side_stream)
        self.score(g, phi, alpha, main)
        join = torch.cuda.Event()
        join.record(side_stream)
        main.wait_event(join)
        self.select(main)
        self.compact(g, phi, alpha, main)
        self.dgrad(W, main)
        if dw_bf16:
            self.wgrad_bf16(main)
        else:
            self.wgrad(main)

    def summary(self) -> dict:
        raw = bytes(self.buf.summary.cpu().numpy().tobytes())
        s = L.RouteSummary.from_buffer_copy(raw)
        return {name: getattr(s, name) for name, _ in L.RouteSummary._fields_}

    def device_status(self, stream=None) -> int:
        return L.lrm_get_device_status(self.ctx, stream)


class StepGraph:
    """The whole step (route stats through the weight gradient) captured once
    as a CUDA graph over fixed device buffers: one launch per step instead of
    one call per kernel, so the host issues nothing per kernel.  Route
    statistics form a branch of their own beside score (they read disjoint
    inputs), joined before select.  The graph reads the tensors it was
    captured with; a caller feeds a new batch by writing into them
    (``copy_``) before ``replay``.  The first, eager run does each kernel's
    one-time set-up (function attributes, occupancy), which must not happen
    inside a capture."""

    def __init__(self, rec: "Recalibration", logits, expert_idx, g, phi, alpha, W, dw_bf16: bool = False):
        self.rec = rec
        self.inputs = dict(logits=logits, expert_idx=expert_idx, g=g, phi=phi, alpha=alpha, W=W)
        dev = rec.device
        side = torch.cuda.Stream(dev)
        branch = torch.cuda.Stream(dev)  # the route statistics branch
        side.wait_stream(torch.cuda.current_stream(dev))
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            rec.run(logits, expert_idx, g, phi, alpha, W, stream=side, dw_bf16=dw_bf16, side_stream=branch)
            side.synchronize()
            with torch.cuda.graph(self.graph, stream=side):
                rec.run(logits, expert_idx, g, phi, alpha, W, stream=side, dw_bf16=dw_bf16, side_stream=branch)
        torch.cuda.current_stream(dev).wait_stream(side)

    def replay(self) -> None:
        """Enqueue one step on the current stream."""
        self.graph.replay()


def to_device_inputs(inp, device="cuda"):
    """Copy a workloads.Inputs record to device tensors (bf16 bits viewed as bf16)."""
    import numpy as np

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    return dict(
        logits=torch.from_numpy(inp.logits).to(device),
        expert_idx=torch.from_numpy(inp.expert_idx).to(device),
        alpha=torch.from_numpy(inp.alpha).to(device),
        g=bf(inp.g),
        phi=bf(inp.phi),
        W=bf(inp.W),
    )


INPUT_NAMES = ("logits", "expert_idx", "g", "phi", "alpha", "W")
OUTPUT_NAMES = ("dW", "dphi_c", "sel_offsets", "sel_ids", "summary")


class HostPipeline:
    """The path over a sequence of host-resident layer batches, with the
    host->device copies of one batch and the device->host copies of the one
    before it running on their own streams while a third computes.

    Two slots (each a ``Recalibration`` with its own device inputs and
    outputs) alternate; events order every reuse: a slot's inputs are not
    overwritten before its last compute has read them, and its outputs are
    not recomputed before they were copied out.  Of the compacted input
    gradient only the retained rows go back: a batch's small outputs (the
    selection offsets first) are copied right after its compute, and its
    ``dphi_c`` rows are copied, exactly ``sel_offsets[E]`` of them, when the
    next batch is submitted (or at ``synchronize``), once that count is on
    the host.  ``submit`` otherwise only enqueues; the caller keeps each host
    buffer untouched until ``synchronize`` (or until two later submits have
    returned).  Host buffers should be pinned for the copies to run
    asynchronously.
    """

    SMALL = ("sel_offsets", "summary", "sel_ids")

    def __init__(self, T, E, k, h, I, cf=Fraction(5, 4), rho=Fraction(3, 4), device=0):
        self.recs = [Recalibration(T, E, k, h, I, cf, rho, device=device) for _ in range(2)]
        dev = self.recs[0].device
        self.device = dev
        self.E = int(E)
        N = int(T) * int(k)
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.dev_in = [dict(logits=torch.empty(T, E, dtype=torch.float32, device=dev),
                            expert_idx=torch.empty(T, k, dtype=torch.int32, device=dev),
                            g=torch.empty(T, h, **bf), phi=torch.empty(N, I, **bf),
                            alpha=torch.empty(N, dtype=torch.float32, device=dev), W=torch.empty(E, h, I, **bf))
                       for _ in range(2)]
        self.s_in, self.s_comp, self.s_out = (torch.cuda.Stream(dev) for _ in range(3))
        self.ev_in, self.ev_comp, self.ev_out, self.ev_small = (
            [torch.cuda.Event() for _ in range(2)] for _ in range(4))
        self.submitted = 0
        self.pending = None  # (slot, host_out) whose dphi_c rows are still to be copied
        self.d2h_bytes = 0  # device -> host bytes enqueued so far

    def _flush(self) -> None:
        if self.pending is None:
            return
        s, host_out = self.pending
        self.pending = None
        self.ev_small[s].synchronize()  # the batch's selection offsets are on the host
        rows = int(host_out["sel_offsets"][self.E])
        rows = max(0, min(rows, host_out["dphi_c"].shape[0]))
        with torch.cuda.stream(self.s_out):
            if rows:
                host_out["dphi_c"][:rows].copy_(self.recs[s].buf.dphi_c[:rows], non_blocking=True)
        self.d2h_bytes += rows * host_out["dphi_c"].stride(0) * host_out["dphi_c"].element_size()
        self.ev_out[s].record(self.s_out)

    def submit(self, host_in: dict, host_out: dict) -> int:
        """Enqueue one batch: copy `host_in` (the six inputs, by name) in, run
        the path, copy the results into `host_out` (dW, the retained rows of
        dphi_c, sel_offsets, sel_ids, summary).  Returns the slot used."""
        s = self.submitted % 2
        rec, din = self.recs[s], self.dev_in[s]
        reuse = self.submitted >= 2
        if reuse:
            self.s_in.wait_event(self.ev_comp[s])
        with torch.cuda.stream(self.s_in):
            for name in INPUT_NAMES:
                din[name].copy_(host_in[name], non_blocking=True)
        self.ev_in[s].record(self.s_in)
        self.s_comp.wait_event(self.ev_in[s])
        if reuse:
            self.s_comp.wait_event(self.ev_out[s])
        rec.run(din["logits"], din["expert_idx"], din["g"], din["phi"], din["alpha"], din["W"], stream=self.s_comp)
        self.ev_comp[s].record(self.s_comp)
        # the previous batch's retained rows go out first, then this batch's outputs
        self._flush()
        self.s_out.wait_event(self.ev_comp[s])
        b = rec.buf
        with torch.cuda.stream(self.s_out):
            for name in self.SMALL:
                host_out[name].copy_(getattr(b, name), non_blocking=True)
            self.ev_small[s].record(self.s_out)
            host_out["dW"].copy_(b.dW, non_blocking=True)
        self.d2h_bytes += sum(host_out[n].numel() * host_out[n].element_size() for n in self.SMALL + ("dW",))
        self.pending = (s, host_out)
        self.submitted += 1
        return s

    def host_outputs(self, pin: bool = True) -> dict:
        """A set of host buffers shaped for ``submit``'s results."""
        b = self.recs[0].buf
        out = {name: torch.empty_like(getattr(b, name), device="cpu") for name in OUTPUT_NAMES}
        return {k2: v.pin_memory() for k2, v in out.items()} if pin else out

    def synchronize(self) -> None:
        self._flush()
        for st in (self.s_in, self.s_comp, self.s_out):
            st.synchronize()

    def device_status(self) -> int:
        flags = 0
        for rec in self.recs:
            flags |= rec.device_status(self.s_comp)
        self.s_comp.synchronize()
        return flags

    def close(self) -> None:
        for rec in self.recs:
            rec.close()
