"""One MoE layer step over the seven C-ABI calls, with preallocated buffers.

route -> stats update -> predict (next layer) -> replicate -> dispatch ->
grouped expert FFN -> combine, all enqueued on the current CUDA stream with
no host synchronisation.  This is orchestration only; every step is a libmoe
kernel.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import (MOE_OP_DISPATCH, MOE_OP_EXPERT_FFN, MOE_OP_EXPERT_FFN_COMBINE, MOE_OP_LAYER_FRONT, MoEStats,
               moe_combine, moe_dispatch, moe_expert_ffn, moe_expert_ffn_combine, moe_expert_ffn_gather, moe_ffn_backward, moe_ffn_backward_workspace_bytes,
               moe_ffn_launches, moe_layer_front, moe_predict, moe_replicate, moe_replicate_predicted,
               moe_replicate_weights, moe_expert_ffn_slots, moe_route, moe_route_backward, moe_stats_update,
               workspace_bytes)

__all__ = ["MoELayerStep", "MoESaved", "ChunkedLayerStep", "HostPipeline", "capture_slot_graphs"]


def _front_launches(T: int, E: int, k: int, layer: int) -> int:
    """Kernels moe_layer_front launches on this device: one cooperative launch
    (routing, a grid-wide barrier, then the dispatch) when all its blocks fit,
    else route/count, then the statistics block beside the plan, scatter and
    copy of every tile."""
    from . import moe_layer_front_launches
    return moe_layer_front_launches(T, E, k, layer > 0)


class MoESaved:
    """What the backward of one layer keeps from its forward: the routing
    (idx, w), the dispatch (group offsets, the replica groups' experts or
    None, perm, inv_perm) and the FFN output y in dispatched order."""

    __slots__ = ("idx", "w", "go", "ge", "perm", "inv", "y")

    def __init__(self, idx, w, go, ge, perm, inv, y):
        self.idx, self.w, self.go, self.ge, self.perm, self.inv, self.y = idx, w, go, ge, perm, inv, y


class MoELayerStep:
    """Buffers for layers of one shape (T, E, k, H, F, act); call `run` per layer.

    replicate=True feeds the replica table of the layer's own histogram into
    dispatch and the FFN (hot experts split into replica groups; the output is
    unchanged); it needs stats, whose update writes that histogram.  stats
    (MoEStats) is shared by all layers of a model.
    fused=True (needs stats) runs route, statistics, prediction, replicas and
    dispatch as moe_layer_front (two launches); fused=False makes the five
    separate calls.  gather=True leaves the token rows in place: dispatch
    writes only the permutation and the FFN's first GEMM reads the rows of x
    through it (moe_expert_ffn_gather); gather=False copies the rows into
    dispatch order first.  replicate_from="prediction" takes layer j's replica
    table from the prediction made at layer j-1 (its p_next) instead of layer
    j's own histogram -- replicas decided before routing -- with `budget`
    bounding the total copies (-1 = none); layer 0 uses its histogram, and
    every layer must run with predict=True (layer j reads what layer j-1
    predicted).
    physical_replicas=True copies each replica's weights into its own slot
    (moe_replicate_weights) and runs the FFN over the slots; `weights` must
    then be the buffers of replica_buffers().  The output is the same in
    every combination.  fuse_combine=True runs the combine in the second
    GEMM's epilogue (moe_expert_ffn_combine; Y is not stored, so the output
    differs by about one bf16 rounding and save=True is not available)."""

    def __init__(self, T: int, E: int, k: int, H: int, F: int, act: str, stats: Optional[MoEStats] = None,
                 replicate: bool = True, thresh=(6, 5), max_copies: int = -1, renorm: bool = True,
                 small_group_threshold: int = 64, fused: bool = True, gather: bool = False,
                 replicate_from: str = "histogram", budget: int = -1, physical_replicas: bool = False,
                 fuse_combine: bool = False, device="cuda"):
        self.T, self.E, self.k, self.H, self.F, self.act = T, E, k, H, F, act
        self.A = T * k
        self.stats = stats
        self.replicate = replicate
        self.thresh, self.max_copies, self.renorm = thresh, max_copies, renorm
        self.small = small_group_threshold
        self.fused = fused and stats is not None
        if replicate_from not in ("histogram", "prediction"):
            raise ValueError("replicate_from must be 'histogram' or 'prediction'")
        if replicate and stats is None:
            raise ValueError("replication reads the layer's histogram, which the statistics update writes: "
                             "pass stats, or replicate=False")
        if replicate_from == "prediction" and (stats is None or not replicate):
            raise ValueError("replicate_from='prediction' needs stats (the prediction) and replicate=True")
        self.replicate_from = replicate_from
        self.budget = budget
        self.physical = physical_replicas and replicate
        if budget >= 0 and not self.fused:
            raise ValueError("a copies budget needs the fused front (fused=True with stats)")
        self.gather = gather
        self.fuse_combine = fuse_combine
        if fuse_combine and (gather or self.physical):
            raise ValueError("fuse_combine works with rows copied into dispatch order and aliased replicas")
        d = torch.device(device)
        i32, f32, bf = torch.int32, torch.float32, torch.bfloat16
        A = self.A
        self.idx = [torch.empty((T, k), dtype=i32, device=d) for _ in range(2)]  # ping-pong: prev layer kept
        self.w = torch.empty((T, k), dtype=f32, device=d)
        self.hist = torch.empty(E, dtype=i32, device=d)
        self.p_seq = torch.empty(E, dtype=f32, device=d)
        self.cond = torch.empty((E, E), dtype=f32, device=d)
        self.pn = [torch.empty(E, dtype=f32, device=d) for _ in range(2)]  # ping-pong with idx
        self.p_next = self.pn[0]
        self.copies = torch.empty(E, dtype=i32, device=d)
        self.pred_load = torch.empty(E, dtype=i32, device=d)
        self.gslot = torch.empty(2 * E, dtype=i32, device=d)
        self.rep_base = torch.empty(E + 1, dtype=i32, device=d)
        self.group_expert = torch.empty(2 * E, dtype=i32, device=d)
        self.go = torch.empty(2 * E + 1, dtype=i32, device=d)
        self.perm = torch.empty(A, dtype=i32, device=d)
        self.inv = torch.empty(A, dtype=i32, device=d)
        self.xp = None if gather else torch.empty((A, H), dtype=bf, device=d)
        self.y = torch.empty((A, H), dtype=bf, device=d)
        self.ws_dispatch = torch.empty(max(workspace_bytes(MOE_OP_DISPATCH, T, k, E),
                                           workspace_bytes(MOE_OP_LAYER_FRONT, T, k, E), 16),
                                       dtype=torch.uint8, device=d)
        op = MOE_OP_EXPERT_FFN_COMBINE if fuse_combine else MOE_OP_EXPERT_FFN
        self.ws_ffn = torch.empty(max(workspace_bytes(op, T, k, E, H, F), 1024), dtype=torch.uint8, device=d)
        self.ws_bwd = None   # allocated by the first backward
        self.saved = None    # the last run(save=True)
        self._save = False
        self._cur = 0

    def run(self, it: int, layer: int, logits, x, weights, out, events=None, predict: bool = True,
            save: bool = False):
        """Enqueue one layer.  weights = (w1, w3 or None, w2).  `events`, if
        given, is a dict stage -> (start, end) torch.cuda.Event recorded
        around each stage on the current stream.  save=True copies what the
        layer's backward needs into a MoESaved (self.saved), since the step's
        buffers are reused by the next layer."""
        self._save = save
        def mark(stage, i):
            if events is not None and stage in events:
                events[stage][i].record()

        prev = self.idx[self._cur ^ 1] if layer > 0 else None
        idx = self.idx[self._cur]
        self.p_next = self.pn[self._cur]
        # the prediction for this layer, made at the layer before (when there was one)
        share = self.pn[self._cur ^ 1] if (self.replicate_from == "prediction" and layer > 0 and predict) else None
        if self.fused:
            last = layer == self.stats.L - 1
            mark("front", 0)
            out_front = {"idx": idx, "w": self.w, "hist": self.hist, "p_seq": self.p_seq,
                         "cond": None if last else self.cond, "p_next": None if last else self.p_next,
                         "copies": self.copies, "rep_base": self.rep_base, "group_expert": self.group_expert,
                         "group_offsets": self.go, "perm": self.perm, "inv_perm": self.inv, "xp": self.xp}
            moe_layer_front(logits, None if self.gather else x, self.stats, it, layer, self.k, idx_prev=prev,
                            renorm=self.renorm, predict=predict, replicate=self.replicate, thresh=self.thresh,
                            max_copies=self.max_copies, rep_share=share, budget=self.budget, out=out_front,
                            workspace=self.ws_dispatch)
            mark("front", 1)
            rb, ge = (self.rep_base, self.group_expert) if self.replicate else (None, None)
            return self._expert_and_combine(x, weights, rb, ge, out, mark)
        mark("route", 0)
        moe_route(logits, self.k, self.renorm, idx=idx, w=self.w)
        mark("route", 1)
        if self.stats is not None:
            mark("stats", 0)
            moe_stats_update(self.stats, it, layer, idx, prev, hist_out=self.hist)
            mark("stats", 1)
            if predict and layer < self.stats.L - 1:
                mark("predict", 0)
                moe_predict(self.stats, layer, out=(self.p_seq, self.cond, self.p_next))
                mark("predict", 1)
        rb = ge = None
        if self.replicate:
            mark("replicate", 0)
            if share is not None:
                moe_replicate_predicted(share, self.A, self.thresh, self.max_copies, self.budget,
                                        out=(self.pred_load, self.copies, self.rep_base, self.group_expert))
            else:
                moe_replicate(self.hist, self.A, self.thresh, self.max_copies,
                              out=(self.copies, self.rep_base, self.group_expert))
            mark("replicate", 1)
            rb, ge = self.rep_base, self.group_expert
        mark("dispatch", 0)
        moe_dispatch(None if self.gather else x, idx, self.E, rb, out=(self.go, self.perm, self.inv, self.xp),
                     workspace=self.ws_dispatch)
        mark("dispatch", 1)
        return self._expert_and_combine(x, weights, rb, ge, out, mark)

    @staticmethod
    def replica_buffers(weights):
        """(w1, w3, w2) [E, ...] -> buffers of 2E-1 slots with the experts in
        slots 0..E-1, for physical_replicas=True."""
        out = []
        for w in weights:
            if w is None:
                out.append(None)
                continue
            E = w.shape[0]
            b = torch.empty((2 * E - 1,) + tuple(w.shape[1:]), dtype=w.dtype, device=w.device)
            b[:E].copy_(w)
            out.append(b)
        return tuple(out)

    def _expert_and_combine(self, x, weights, rb, ge, out, mark):
        w1, w3, w2 = weights
        mark("ffn", 0)
        if self.physical:
            if w1.shape[0] != 2 * self.E - 1:
                raise ValueError("physical_replicas needs the 2E-1 slot buffers of replica_buffers()")
            moe_replicate_weights(self.rep_base, w1, group_slot=self.gslot)
            moe_replicate_weights(self.rep_base, w2, group_slot=self.gslot)
            if w3 is not None:
                moe_replicate_weights(self.rep_base, w3, group_slot=self.gslot)
            moe_expert_ffn_slots(self.xp, self.go, self.gslot, w1, w3, w2, self.act, self.small, y=self.y,
                                 workspace=self.ws_ffn)
        elif self.fuse_combine:
            if self._save:
                raise ValueError("save=True needs Y, which fuse_combine does not store")
            moe_expert_ffn_combine(self.xp, self.go, ge, rb, self.perm, self.w, w1, w3, w2, self.act, self.small,
                                   out=out, workspace=self.ws_ffn)
            mark("ffn", 1)
            mark("combine", 0)  # the combine ran inside the FFN
            mark("combine", 1)
            self._cur ^= 1
            return out
        elif self.gather:
            moe_expert_ffn_gather(x, self.perm, self.k, self.go, ge, rb, w1, w3, w2, self.act, self.small, y=self.y,
                                  workspace=self.ws_ffn)
        else:
            moe_expert_ffn(self.xp, self.go, ge, rb, w1, w3, w2, self.act, self.small, y=self.y,
                           workspace=self.ws_ffn)
        mark("ffn", 1)
        mark("combine", 0)
        moe_combine(self.y, self.inv, self.w, out=out)
        mark("combine", 1)
        if self._save:
            self.saved = MoESaved(self.idx[self._cur].clone(), self.w.clone(), self.go.clone(),
                                  None if ge is None else ge.clone(), self.perm.clone(), self.inv.clone(),
                                  self.y.clone())
        self._cur ^= 1
        return out

    def backward(self, saved: MoESaved, logits, x, weights, dout, grads=None, dlogits=None, accumulate: bool = False,
                 wgrad_bf16: bool = False):
        """Backward of one layer run with save=True: dout = dL/d(out) [T, H]
        bf16.  Returns (dx [T, H] bf16, dlogits [T, E] f32, (dW1, dW3 or None,
        dW2) f32).  Every row of an expert adds into that expert's gradient,
        whichever replica group served it.  weights = the experts' (w1, w3,
        w2) [E, ...] (with physical replicas, their first E slots).  `grads`
        may give (dx, dw, dW1, dW3, dW2) buffers to write into; with
        accumulate=True the weight gradients are added to what grads hold
        (gradient accumulation over micro-batches); wgrad_bf16=True returns
        them rounded once to bf16."""
        w1, w3, w2 = (None if w is None else w[:self.E] for w in weights)
        if self.ws_bwd is None:
            n = moe_ffn_backward_workspace_bytes(self.T, self.k, self.E, self.H, self.F)
            self.ws_bwd = torch.empty(n, dtype=torch.uint8, device=dout.device)
        dx, dw, dw1, dw3, dw2 = moe_ffn_backward(x, dout, saved.w, saved.y, saved.perm, saved.inv, saved.go, saved.ge,
                                                 w1, w3, w2, self.act, workspace=self.ws_bwd, out=grads,
                                                 accumulate=accumulate, wgrad_bf16=wgrad_bf16)
        dl = moe_route_backward(logits, saved.idx, dw, self.renorm, out=dlogits)
        return dx, dl, (dw1, dw3, dw2)

    def launches(self, layer: int, L: int, predict: bool = True) -> int:
        front = _front_launches(self.T, self.E, self.k, layer)
        if self.physical:   # slot map + copy kernel per weight matrix, FFN over 2E-1 slots
            ffn = (moe_ffn_launches(self.A, 2 * self.E - 1, self.H, self.F, self.act, self.small, False)
                   + 2 * (3 if self.act == "swiglu" else 2))
        else:
            ffn = moe_ffn_launches(self.A, self.E, self.H, self.F, self.act, self.small, self.gather)
        if self.fuse_combine:  # the two-launch kernels (the fused one stores Y), the finalize pass, no combine
            ffn = moe_ffn_launches(self.A, self.E, self.H, self.F, self.act, self.small, True) + 1
            return (front if self.fused else 1 + 4 + (1 if self.stats is not None else 0)
                    + (1 if self.stats is not None and predict and layer < L - 1 else 0)
                    + (1 if self.replicate else 0)) + ffn
        if self.fused:
            return front + ffn + 1
        n = 1 + (3 if self.gather else 4) + ffn + 1
        if self.stats is not None:
            n += 1
            if predict and layer < L - 1:
                n += 1
        if self.replicate:
            n += 1
        return n


class ChunkedLayerStep:
    """EPS-MoE's single-GPU expert pipeline (EPS-MoE review, pipeline of
    dispatch, expert computation and combine over PN chunks of the tokens).

    The front (route, statistics, prediction, replica table) runs once for
    the whole layer, so the window statistics are those of the unchunked
    layer; then each of `chunks` token chunks is dispatched, run through the
    expert FFN and combined on one of two streams, so that a chunk's
    dispatch can overlap the previous chunk's FFN where the GPU has room.
    The output equals MoELayerStep's bit for bit (each row's FFN and each
    token's combine are the same arithmetic; replica groups alias their
    expert's weights)."""

    def __init__(self, T: int, E: int, k: int, H: int, F: int, act: str, stats: MoEStats, chunks: int = 2,
                 replicate: bool = True, thresh=(6, 5), max_copies: int = -1, renorm: bool = True,
                 small_group_threshold: int = 64, device="cuda"):
        if chunks < 1 or T % chunks:
            raise ValueError("chunks must divide T")
        self.T, self.E, self.k, self.H, self.F, self.act = T, E, k, H, F, act
        self.stats, self.chunks = stats, chunks
        self.replicate, self.thresh, self.max_copies, self.renorm = replicate, thresh, max_copies, renorm
        self.small = small_group_threshold
        d = torch.device(device)
        i32, f32, bf = torch.int32, torch.float32, torch.bfloat16
        A = T * k
        Tc = T // chunks
        Ac = Tc * k
        self.Tc = Tc
        self.idx = [torch.empty((T, k), dtype=i32, device=d) for _ in range(2)]
        self.w = torch.empty((T, k), dtype=f32, device=d)
        self.hist = torch.empty(E, dtype=i32, device=d)
        self.p_seq = torch.empty(E, dtype=f32, device=d)
        self.cond = torch.empty((E, E), dtype=f32, device=d)
        self.p_next = torch.empty(E, dtype=f32, device=d)
        self.copies = torch.empty(E, dtype=i32, device=d)
        self.rep_base = torch.empty(E + 1, dtype=i32, device=d)
        self.group_expert = torch.empty(2 * E, dtype=i32, device=d)
        self.go_full = torch.empty(2 * E + 1, dtype=i32, device=d)
        self.perm_full = torch.empty(A, dtype=i32, device=d)
        self.inv_full = torch.empty(A, dtype=i32, device=d)
        self.ws_front = torch.empty(max(workspace_bytes(MOE_OP_LAYER_FRONT, T, k, E), 16), dtype=torch.uint8,
                                    device=d)
        # per stream: chunk buffers
        self.streams = [torch.cuda.Stream(device=d) for _ in range(2)]
        self.buf = []
        for _ in range(2):
            self.buf.append({
                "go": torch.empty(2 * E + 1, dtype=i32, device=d),
                "perm": torch.empty(Ac, dtype=i32, device=d),
                "inv": torch.empty(Ac, dtype=i32, device=d),
                "xp": torch.empty((Ac, H), dtype=bf, device=d),
                "y": torch.empty((Ac, H), dtype=bf, device=d),
                "ws_d": torch.empty(max(workspace_bytes(MOE_OP_DISPATCH, Tc, k, E), 16), dtype=torch.uint8, device=d),
                "ws_f": torch.empty(max(workspace_bytes(MOE_OP_EXPERT_FFN, Tc, k, E, H, F), 1024),
                                    dtype=torch.uint8, device=d),
                "free": torch.cuda.Event(),
            })
        self.front_done = torch.cuda.Event()
        self._fresh = [True, True]
        self._cur = 0

    def run(self, it: int, layer: int, logits, x, weights, out, events=None, predict: bool = True):
        main = torch.cuda.current_stream()
        prev = self.idx[self._cur ^ 1] if layer > 0 else None
        idx = self.idx[self._cur]
        last = layer == self.stats.L - 1
        fo = {"idx": idx, "w": self.w, "hist": self.hist, "p_seq": self.p_seq,
              "cond": None if last else self.cond, "p_next": None if last else self.p_next,
              "copies": self.copies, "rep_base": self.rep_base, "group_expert": self.group_expert,
              "group_offsets": self.go_full, "perm": self.perm_full, "inv_perm": self.inv_full, "xp": None}
        moe_layer_front(logits, None, self.stats, it, layer, self.k, idx_prev=prev, renorm=self.renorm,
                        predict=predict, replicate=self.replicate, thresh=self.thresh, max_copies=self.max_copies,
                        out=fo, workspace=self.ws_front)
        self.front_done.record(main)
        if events is not None and "ffn" in events:   # the chunked part: dispatch, FFN and combine of all chunks
            events["ffn"][0].record(main)
        rb, ge = (self.rep_base, self.group_expert) if self.replicate else (None, None)
        w1, w3, w2 = weights
        Tc = self.Tc
        # the previous run's chunks were joined into the main stream before the
        # front, so a buffer only waits for an earlier chunk of this run
        self._fresh = [True, True]
        for c in range(self.chunks):
            j = c & 1
            s, b = self.streams[j], self.buf[j]
            s.wait_event(self.front_done)
            if not self._fresh[j]:
                s.wait_event(b["free"])
            with torch.cuda.stream(s):
                rows = slice(c * Tc, (c + 1) * Tc)
                moe_dispatch(x[rows], idx[rows], self.E, rb, out=(b["go"], b["perm"], b["inv"], b["xp"]),
                             workspace=b["ws_d"])
                moe_expert_ffn(b["xp"], b["go"], ge, rb, w1, w3, w2, self.act, self.small, y=b["y"],
                               workspace=b["ws_f"])
                moe_combine(b["y"], b["inv"], self.w[rows], out=out[rows])
                b["free"].record(s)
            self._fresh[j] = False
        for j in range(2):
            if not self._fresh[j]:
                main.wait_event(self.buf[j]["free"])
        if events is not None and "ffn" in events:
            events["ffn"][1].record(main)
        self._cur ^= 1
        return out

    def launches(self, layer: int, L: int, predict: bool = True) -> int:
        ffn = moe_ffn_launches(self.Tc * self.k, self.E, self.H, self.F, self.act, self.small, False)
        return _front_launches(self.T, self.E, self.k, layer) + self.chunks * (4 + ffn + 1)


class HostPipeline:
    """Run layers whose inputs and outputs live in (pinned) host memory.

    Three streams overlap the work: the copy of layer j+1's logits and X to
    the device, the seven calls of layer j, and the copy of layer j-1's output
    back to the host.  Device staging buffers are double-buffered; events order
    each buffer's reuse.  Host tensors should be pinned for the copies to run
    asynchronously."""

    def __init__(self, step: MoELayerStep, device="cuda"):
        self.step = step
        d = torch.device(device)
        T, E, H = step.T, step.E, step.H
        self.d_logits = [torch.empty((T, E), dtype=torch.float32, device=d) for _ in range(2)]
        self.d_x = [torch.empty((T, H), dtype=torch.bfloat16, device=d) for _ in range(2)]
        self.d_out = [torch.empty((T, H), dtype=torch.bfloat16, device=d) for _ in range(2)]
        self.h2d = torch.cuda.Stream(device=d)
        self.d2h = torch.cuda.Stream(device=d)
        self.in_ready = [torch.cuda.Event() for _ in range(2)]
        self.in_free = [torch.cuda.Event() for _ in range(2)]
        self.out_ready = [torch.cuda.Event() for _ in range(2)]
        self.out_free = [torch.cuda.Event() for _ in range(2)]
        self._fresh = [True, True]

    def run(self, it: int, h_logits, h_x, weights, h_out, layers=None):
        """h_logits[j] [T,E] f32, h_x[j] [T,H] bf16, h_out[j] [T,H] bf16 host
        tensors; weights[j] = (w1, w3, w2) on the device.  Enqueues every layer
        and returns; synchronise the current stream (or the device) before
        reading h_out."""
        comp = torch.cuda.current_stream()
        L = len(h_x) if layers is None else layers
        for j in range(L):
            b = j & 1
            with torch.cuda.stream(self.h2d):
                if not self._fresh[b]:
                    self.h2d.wait_event(self.in_free[b])
                self.d_logits[b].copy_(h_logits[j], non_blocking=True)
                self.d_x[b].copy_(h_x[j], non_blocking=True)
                self.in_ready[b].record(self.h2d)
            comp.wait_event(self.in_ready[b])
            if not self._fresh[b]:
                comp.wait_event(self.out_free[b])
            self.step.run(it, j, self.d_logits[b], self.d_x[b], weights[j], self.d_out[b])
            self.in_free[b].record(comp)
            self.out_ready[b].record(comp)
            with torch.cuda.stream(self.d2h):
                self.d2h.wait_event(self.out_ready[b])
                h_out[j].copy_(self.d_out[b], non_blocking=True)
                self.out_free[b].record(self.d2h)
            self._fresh[b] = False
        # the caller's stream covers the last copies back
        comp.wait_stream(self.d2h)


def capture_slot_graphs(run_iteration, slots: int, make_events=None):
    """One CUDA graph per window slot of a multi-layer iteration.

    The statistics update uses the iteration only modulo the window s, so a
    graph captured for slot q replays every iteration i with i mod s = q
    exactly.  `run_iteration(q, events)` enqueues one whole iteration (every
    layer) for slot q on the current stream; `make_events()`, if given,
    returns the per-layer stage events recorded inside that graph (external
    events, readable after a replay).  Returns (graphs, events), one entry per
    slot; replay graph i mod s for iteration i."""
    graphs, evs = [], []
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        for q in range(slots):
            g = torch.cuda.CUDAGraph()
            ev = None if make_events is None else make_events()
            with torch.cuda.graph(g, stream=cap):
                run_iteration(q, ev)
            graphs.append(g)
            evs.append(ev)
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    return graphs, evs
