"""Device buffers and call sequence of one step of the CTR path.

``CtrPath`` owns the device memory of one workload (tables, index buffers,
dedup outputs, interaction tensors, workspaces) through torch, and runs the
step as a sequence of libctr calls on one CUDA stream:

    dedup -> pooled gather (into the interaction input X) -> dot interaction
          -> interaction backward -> per-unique-row gradient reduce + SGD update

Which steps a workload runs follows its configuration (forward-only
workloads stop after the interaction; the TensorNet-style workload pools from
the batch-sized unique-row matrix).  No arithmetic of the method happens here.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np
import torch

from . import ctr
from .workload import Config

TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}
_MODES = {"cross": ctr.INTERACT_CROSS, "with_self": ctr.INTERACT_WITH_SELF, "full": ctr.INTERACT_FULL_GRAM}


class CtrPath:
    def __init__(self, cfg: Config, n_ids: int, device="cuda", fill: bool = True, table_chunk_rows: int = 1 << 24,
                 keep_sorted_pos: bool = False, fm: bool = False, optimizer: str = "sgd", eps: float = 1e-8,
                 betas=(0.9, 0.999), stochastic_rounding: bool = False, sr_seed: int = 0x5EED):
        self.cfg = cfg
        self.dev = torch.device(device)
        self.n_ids = int(n_ids)
        F, B, d, n = cfg.num_fields, cfg.batch, cfg.d, cfg.n_vectors
        tdt = TORCH_DT[cfg.dtype]
        self.table = torch.empty((cfg.total_rows, d), dtype=tdt, device=self.dev)
        if fill:
            self.fill_table(table_chunk_rows)
        cap = max(self.n_ids, 1)
        i64, i32 = torch.int64, torch.int32
        self.ids = torch.empty(cap, dtype=i64, device=self.dev)
        self.offsets = torch.empty(F * B + 1, dtype=i64, device=self.dev)
        self.unique_rows = torch.empty(cap, dtype=i64, device=self.dev)
        self.n_unique = torch.zeros(1, dtype=i64, device=self.dev)
        self.inverse = torch.empty(cap, dtype=i32, device=self.dev)
        # the stable sort permutation is an optional output: without it the dedup's
        # sort carries bags instead of positions and skips a gather
        self.sorted_pos = torch.empty(cap, dtype=i32, device=self.dev) if keep_sorted_pos else None
        self.sorted_bag = torch.empty(cap, dtype=i32, device=self.dev)
        self.run_offsets = torch.empty(cap + 1, dtype=i32, device=self.dev)
        self.unique_offsets = torch.empty(cfg.num_tables + 1, dtype=i64, device=self.dev)
        self.U = torch.empty((cap, d), dtype=tdt, device=self.dev) if cfg.dedup_gather else None
        # interaction input: slot 0 = dense, slots 1..F = pooled
        self.X = torch.zeros((B, n, d), dtype=tdt, device=self.dev)
        self.out = torch.empty((B, cfg.out_width), dtype=tdt, device=self.dev) if cfg.interaction else None
        self.pooled = None if cfg.interaction else torch.empty((B, F, d), dtype=tdt, device=self.dev)
        self.dout = torch.empty((B, cfg.out_width), dtype=torch.float32, device=self.dev) \
            if cfg.backward == "full" else None
        self.dX = torch.empty((B, n, d), dtype=torch.float32, device=self.dev) if cfg.backward == "full" else None
        self.grad_pooled = torch.empty((B, F, d), dtype=torch.float32, device=self.dev) \
            if cfg.backward == "pooled_grad" else None
        self.grad_unique = None
        # FM second-order term of every bag, written by the gather when requested
        self.fm = torch.empty(F * B, dtype=torch.float32, device=self.dev) if fm else None
        # optimizer state of the row update (zero-initialised, indexed by global row)
        self.optimizer = optimizer
        self.opt_kind = {"sgd": ctr.OPT_SGD, "adagrad": ctr.OPT_ADAGRAD, "rowwise_adagrad": ctr.OPT_ROWWISE_ADAGRAD,
                         "adam": ctr.OPT_ADAM}[optimizer]
        self.eps, self.betas, self.opt_step = eps, betas, 0
        # bf16 tables: stochastic rounding of the updated rows, a fresh seed per update
        self.stochastic_rounding = bool(stochastic_rounding) and cfg.dtype == "bf16"
        self.sr_seed, self.updates = int(sr_seed), 0
        self.last_sr_seed = None  # the seed of the latest update's rounding
        R = cfg.total_rows
        self.state0 = None if optimizer == "sgd" else torch.zeros(
            (R,) if optimizer == "rowwise_adagrad" else (R, d), dtype=torch.float32, device=self.dev)
        self.state1 = torch.zeros((R, d), dtype=torch.float32, device=self.dev) if optimizer == "adam" else None
        total_rows = cfg.total_rows
        self.ws_dedup = ctr.workspace(ctr.ctr_dedup_workspace_size(cap, F, B, total_rows), self.dev)
        self.ws_bag = ctr.workspace(ctr.ctr_embedding_bag_workspace_size(), self.dev)
        self.ws_int = ctr.workspace(ctr.ctr_interaction_workspace_size(), self.dev)
        self.ws_bwd = ctr.workspace(ctr.ctr_bwd_update_workspace_size(cap, d), self.dev)
        self.b2t = np.asarray(cfg.field_to_table, dtype=np.int32)
        self.row_base = cfg.row_base
        self._side = None          # side stream of the overlapped dedup and long runs (created on first use)
        # when set (DeviceBatches), every step first copies these dense vectors into slot 0 of X
        self.dense_src = None
        # the long-run and short-run phases of the backward are persistent grids that each
        # fill the GPU, so overlapping them was measured slower: off by default
        self.overlap_backward = False

    # -- inputs -----------------------------------------------------------
    def fill_table(self, chunk_rows: int = 1 << 24) -> None:
        cfg = self.cfg
        flat = self.table.view(-1)
        for r0 in range(0, cfg.total_rows, chunk_rows):
            r1 = min(cfg.total_rows, r0 + chunk_rows)
            ctr.ctr_fill_table(flat[r0 * cfg.d:r1 * cfg.d], cfg.d, r0, cfg.fill_kind, cfg.fill_seed, cfg.fill_scale)

    def upload(self, w: Dict[str, np.ndarray], non_blocking: bool = False) -> None:
        """Copy a workload's host arrays into the device buffers."""
        n = w["ids"].size
        assert n == self.n_ids, (n, self.n_ids)
        if n:
            self.ids[:n].copy_(torch.from_numpy(w["ids"]), non_blocking=non_blocking)
        self.offsets.copy_(torch.from_numpy(w["offsets"]), non_blocking=non_blocking)
        dense = w["dense"]
        dt = torch.from_numpy(dense.view(np.int16)).view(torch.bfloat16) if self.cfg.dtype == "bf16" \
            else torch.from_numpy(dense)
        self.X[:, 0, :].copy_(dt, non_blocking=non_blocking)
        if self.grad_pooled is not None and "grad_pooled" in w:
            self.grad_pooled.copy_(torch.from_numpy(w["grad_pooled"]), non_blocking=non_blocking)
        if self.dout is not None and "dout" in w:
            self.dout.copy_(torch.from_numpy(w["dout"]), non_blocking=non_blocking)

    def reset_status(self) -> None:
        for ws in (self.ws_dedup, self.ws_bag, self.ws_int, self.ws_bwd):
            ctr.ctr_status_reset(ws)

    def check_status(self) -> Dict[str, int]:
        return {k: ctr.ctr_check_status(ws) for k, ws in
                (("dedup", self.ws_dedup), ("bag", self.ws_bag), ("interaction", self.ws_int), ("bwd", self.ws_bwd))}

    # -- steps ------------------------------------------------------------
    def dedup(self, phases: int = ctr.DEDUP_ALL) -> None:
        cfg = self.cfg
        ctr.ctr_dedup_phases(self.ids, self.offsets, cfg.num_fields, cfg.batch, self.b2t, self.row_base,
                             self.unique_rows, self.n_unique, self.inverse, self.sorted_pos, self.sorted_bag,
                             self.run_offsets, self.unique_offsets, phases, self.ws_dedup, n_ids=self.n_ids)

    def forward(self) -> None:
        cfg = self.cfg
        F, B, d, n = cfg.num_fields, cfg.batch, cfg.d, cfg.n_vectors
        pool = ctr.POOL_MEAN if cfg.pool == "mean" else ctr.POOL_SUM
        if self.pooled is not None:
            out, sb, sf = self.pooled, F * d, d
        else:
            out, sb, sf = self.X[:, 1:, :], n * d, d
        if cfg.dedup_gather:
            ctr.ctr_gather_rows(self.table, d, self.unique_rows, self.n_unique, self.U, self.ws_bag)
            ctr.ctr_embedding_bag_fwd(self.U, d, self.inverse, self.offsets, F, B, None, None, pool, out, sb, sf,
                                      self.ws_bag, n_indices=self.n_ids, fm_out=self.fm)
        else:
            ctr.ctr_embedding_bag_fwd(self.table, d, self.ids, self.offsets, F, B, self.b2t, self.row_base, pool,
                                      out, sb, sf, self.ws_bag, n_indices=self.n_ids, fm_out=self.fm)

    def interaction(self) -> None:
        cfg = self.cfg
        ctr.ctr_dot_interaction_mode(self.X, cfg.n_vectors, cfg.d, _MODES[cfg.interaction_mode], self.out, self.ws_int)

    def interaction_bwd(self) -> None:
        cfg = self.cfg
        ctr.ctr_dot_interaction_bwd_mode(self.dout, self.X, cfg.n_vectors, cfg.d, _MODES[cfg.interaction_mode], self.dX,
                                         self.ws_int)

    def bwd_update(self, grad_unique_out: Optional[torch.Tensor] = None, overlap: bool = False) -> None:
        """Per-unique-row gradient reduce + row update.

        With overlap, the long runs' pieces are summed on a side stream while
        the short runs are reduced and updated on the current one (the two
        phases touch disjoint rows), and the long runs are finished after both.
        """
        cfg = self.cfg
        F, B, d, n = cfg.num_fields, cfg.batch, cfg.d, cfg.n_vectors
        pool = ctr.POOL_MEAN if cfg.pool == "mean" else ctr.POOL_SUM
        if self.dX is not None:
            G, sb, sf = self.dX[:, 1:, :], n * d, d
        else:
            G, sb, sf = self.grad_pooled, F * d, d
        args = (G, sb, sf, self.offsets, F, B, pool, self.unique_rows, self.n_unique, self.run_offsets, self.sorted_bag,
                max(self.n_ids, 1), cfg.lr, self.table, d, grad_unique_out)
        self.updates += 1
        if self.opt_kind != ctr.OPT_SGD or self.stochastic_rounding:
            if self.opt_kind != ctr.OPT_SGD:
                self.opt_step += 1
            self.last_sr_seed = (self.sr_seed * 0x9E3779B97F4A7C15 + self.updates) & ((1 << 64) - 1)
            opt = ctr.optimizer(self.opt_kind, eps=self.eps, beta1=self.betas[0], beta2=self.betas[1],
                                step=max(self.opt_step, 1), state0=self.state0, state1=self.state1,
                                stochastic_rounding=self.stochastic_rounding, sr_seed=self.last_sr_seed)
            ctr.ctr_embedding_bag_bwd_update_opt(*args, ctr.BWD_ALL, opt, self.ws_bwd)
            return
        if not overlap:
            ctr.ctr_embedding_bag_bwd_update(*args, self.ws_bwd)
            return
        main = torch.cuda.current_stream(self.dev)
        side = self._side_stream()
        self._ev_bwd.record(main)
        side.wait_event(self._ev_bwd)
        with torch.cuda.stream(side):
            ctr.ctr_embedding_bag_bwd_update_phases(*args, ctr.BWD_LONG_RUNS, self.ws_bwd)
        self._ev_long.record(side)
        ctr.ctr_embedding_bag_bwd_update_phases(*args, ctr.BWD_SHORT_RUNS, self.ws_bwd)
        main.wait_event(self._ev_long)
        ctr.ctr_embedding_bag_bwd_update_phases(*args, ctr.BWD_FINISH, self.ws_bwd)

    def _side_stream(self) -> torch.cuda.Stream:
        if self._side is None:
            self._side = torch.cuda.Stream(self.dev)
            self._ev_start = torch.cuda.Event()
            self._ev_dedup = torch.cuda.Event()
            self._ev_bwd = torch.cuda.Event()
            self._ev_long = torch.cuda.Event()
        return self._side

    def step(self) -> None:
        """One pass of the workload's hot path, on the current stream.

        When the forward pools straight from the tables, only the backward needs
        the dedup: it then runs on a side stream, concurrently with the gather and
        the interaction (its kernels are mostly latency-bound, theirs bandwidth-
        bound), and the backward waits for it.  The side stream first waits for
        everything queued before the step, and the step's end (on the current
        stream) comes after the dedup, so the step orders like a sequential one.
        (Running the radix passes after the interaction backward instead, with
        only the dedup's first part beside the gather, was slower.)
        """
        cfg = self.cfg
        needs_dedup = cfg.backward != "none" or cfg.dedup_gather
        overlap = needs_dedup and not cfg.dedup_gather and cfg.backward != "none"
        if self.dense_src is not None:
            self.X[:, 0, :].copy_(self.dense_src, non_blocking=True)
        if overlap:
            main = torch.cuda.current_stream(self.dev)
            side = self._side_stream()
            self._ev_start.record(main)
            side.wait_event(self._ev_start)
            with torch.cuda.stream(side):
                self.dedup()
            self._ev_dedup.record(side)
        elif needs_dedup:
            self.dedup()
        self.forward()
        if cfg.interaction:
            self.interaction()
        if cfg.backward == "full":
            self.interaction_bwd()
        if overlap:
            torch.cuda.current_stream(self.dev).wait_event(self._ev_dedup)
        if cfg.backward != "none":
            self.bwd_update(overlap=self.overlap_backward)

    def capture(self) -> "StepGraph":
        """One step captured as a CUDA graph (the same kernels, streams and buffers), replayed
        with `.replay()` on the current stream: one launch per step instead of one per kernel.

        A graph fixes the host-side values of the step it captured: the ID count, and Adam's
        step number and the stochastic-rounding seed, which change every step, so those two
        are refused here (SGD and both Adagrads are step-independent)."""
        if self.opt_kind == ctr.OPT_ADAM or self.stochastic_rounding:
            raise ValueError("a captured step would repeat Adam's step number or the rounding seed")
        g = torch.cuda.CUDAGraph()
        n0 = ctr.ctr_launch_count()
        with torch.cuda.graph(g):
            self.step()
        return StepGraph(g, ctr.ctr_launch_count() - n0, self.n_ids)


class StepGraph:
    """A captured CtrPath step: `replay()` runs it on the current stream; `launches` is the
    number of library kernels it holds, `n_ids` the ID count it was captured for."""

    def __init__(self, graph, launches: int, n_ids: int):
        self.graph, self.launches, self.n_ids = graph, int(launches), int(n_ids)

    def replay(self) -> None:
        self.graph.replay()


class DeviceBatches:
    """Several batches of one workload held on the device at once, each in its own input
    buffers (IDs, offsets, upstream gradient, dense vectors).  `bind(k)` points the path
    at batch k mod the count; the path's steps then read that batch, starting with a copy
    of its dense vectors into slot 0 of X (inside a captured step too).  The batches must
    share the ID count (a captured step fixes it)."""

    def __init__(self, path: CtrPath, batches):
        self.path = path
        cfg = path.cfg
        self.names = ["ids", "offsets"] + [k for k in ("dout", "grad_pooled") if getattr(path, k) is not None]
        self.sets = []
        for j, w in enumerate(batches):
            if w["ids"].size != path.n_ids:
                raise ValueError(f"batch {j} has {w['ids'].size} IDs; the path holds {path.n_ids}")
            bufs = {k: (getattr(path, k) if j == 0 else torch.empty_like(getattr(path, k))) for k in self.names}
            n = w["ids"].size
            if n:
                bufs["ids"][:n].copy_(torch.from_numpy(w["ids"]))
            bufs["offsets"].copy_(torch.from_numpy(w["offsets"]))
            for k in ("dout", "grad_pooled"):
                if k in bufs:
                    bufs[k].copy_(torch.from_numpy(w[k]))
            dense = w["dense"]
            dt = torch.from_numpy(dense.view(np.int16)).view(torch.bfloat16) if cfg.dtype == "bf16" \
                else torch.from_numpy(dense)
            bufs["dense"] = dt.to(path.dev)
            self.sets.append(bufs)

    def __len__(self):
        return len(self.sets)

    def bind(self, k: int) -> None:
        bufs = self.sets[k % len(self.sets)]
        for name in self.names:
            setattr(self.path, name, bufs[name])
        self.path.dense_src = bufs["dense"]


class HostPipeline:
    """Runs CtrPath steps over batches held in pinned host memory, with the copies overlapped.

    `depth` device buffer sets hold the per-batch inputs (IDs, offsets, dense
    vectors, upstream gradient) and the step's output.  While step k runs on
    the compute stream, the inputs of step k + depth - 1 are copied in on one
    copy stream and the output of step k-1 is copied out on another, so the
    host<->device transfers hide behind the kernels; a copy may take up to
    depth - 1 steps (host-to-device copies on the GB300 machine occasionally stall
    for tens of milliseconds).  Every batch's inputs and every step's output
    still cross the host boundary, in full, once per step.

    A batch is a dict with pinned CPU tensors "ids" (int64), "offsets" (int64,
    [F*B+1]), "dense" ([B, d], the table dtype), and "dout" ([B, width] fp32) or
    "grad_pooled" ([B, F, d] fp32) when the workload has a backward.  Outputs are
    pinned CPU tensors shaped like the step's result (the interaction output, or
    the pooled vectors for workloads without one).
    """

    def __init__(self, path: CtrPath, graphs: bool = False, depth: int = 4):
        if depth < 2:
            raise ValueError("the pipeline needs at least two buffer sets")
        self.path = path
        self.depth = D = int(depth)
        cfg = path.cfg
        path.dense_src = None  # the pipeline copies each batch's dense vectors itself
        self.result_name = "out" if path.out is not None else "pooled"
        names = ["ids", "offsets"] + [k for k in ("dout", "grad_pooled") if getattr(path, k) is not None]
        self.sets = []
        for s in range(D):
            bufs = {k: (getattr(path, k) if s == 0 else torch.empty_like(getattr(path, k))) for k in names}
            bufs["dense"] = torch.empty((cfg.batch, cfg.d), dtype=path.X.dtype, device=path.dev)
            res = getattr(path, self.result_name)
            bufs["result"] = res if s == 0 else torch.empty_like(res)
            self.sets.append(bufs)
        self.names = names
        self.compute = torch.cuda.current_stream(path.dev)
        self.h2d = torch.cuda.Stream(path.dev)
        self.d2h = torch.cuda.Stream(path.dev)
        self.ev_in = [torch.cuda.Event() for _ in range(D)]
        self.ev_done = [torch.cuda.Event() for _ in range(D)]
        self.ev_out = [torch.cuda.Event() for _ in range(D)]
        for s in range(D):   # create the events in a completed state
            self.ev_done[s].record(self.compute)
            self.ev_out[s].record(self.compute)
        # with graphs: one captured step per buffer set (batches must keep the ID count)
        self.graphs = None
        if graphs:
            self.graphs = []
            for s in range(D):
                self._bind(s)
                self.graphs.append(path.capture())
            self._bind(0)

    def _bind(self, s):
        bufs = self.sets[s]
        for name in self.names:
            setattr(self.path, name, bufs[name])
        setattr(self.path, self.result_name, bufs["result"])

    def _copy_in(self, batch, s):
        bufs = self.sets[s]
        with torch.cuda.stream(self.h2d):
            self.h2d.wait_event(self.ev_done[s])            # the step that last read set s has finished
            n = batch["ids"].numel()
            bufs["ids"][:n].copy_(batch["ids"], non_blocking=True)
            bufs["offsets"].copy_(batch["offsets"], non_blocking=True)
            bufs["dense"].copy_(batch["dense"], non_blocking=True)
            for k in ("dout", "grad_pooled"):
                if k in bufs:
                    bufs[k].copy_(batch[k], non_blocking=True)
            self.ev_in[s].record(self.h2d)

    def run(self, batches, outputs, start_event=None) -> None:
        """Step over `batches`, writing step k's result into `outputs[k]` (both pinned host memory).

        The call returns once everything is queued; the compute stream waits for
        the last output copy, so an event recorded on it afterwards (or a
        synchronize) covers the whole run.  `start_event`, if given, is recorded
        on the compute stream before the first copy.
        """
        path = self.path
        K = len(batches)
        if K == 0:
            return
        if start_event is not None:
            start_event.record(self.compute)
        D = self.depth
        self.h2d.wait_stream(self.compute)
        for j in range(min(D - 1, K)):
            self._copy_in(batches[j], j)
        for k in range(K):
            s = k % D
            bufs = self.sets[s]
            n = batches[k]["ids"].numel()
            if n > path.ids.numel():
                raise ValueError(f"batch {k} has {n} IDs, more than the path's capacity {path.ids.numel()}")
            self.compute.wait_event(self.ev_in[s])
            self.compute.wait_event(self.ev_out[s])         # the previous output in this set has been copied out
            path.X[:, 0, :].copy_(bufs["dense"], non_blocking=True)
            if self.graphs is not None:
                if n != self.graphs[s].n_ids:
                    raise ValueError(f"batch {k} has {n} IDs; the captured steps were for {self.graphs[s].n_ids}")
                self.graphs[s].replay()
            else:
                path.n_ids = n
                self._bind(s)
                path.step()
            self.ev_done[s].record(self.compute)
            if k + D - 1 < K:
                self._copy_in(batches[k + D - 1], (k + D - 1) % D)
            with torch.cuda.stream(self.d2h):
                self.d2h.wait_event(self.ev_done[s])
                outputs[k].copy_(bufs["result"], non_blocking=True)
                self.ev_out[s].record(self.d2h)
        for s in range(D):
            self.compute.wait_event(self.ev_out[s])
