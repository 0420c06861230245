"""One decode step over every layer, as the engine's executor runs it.

Step = metadata bind once (cache.py page, bullets 25-28), then for each layer
the KV append (cache.py page, bullet 40), split-KV decode attention and the
partial merge (workspace.py page, bullets 1 and 14).  Inputs live in static
buffers owned by the runner so a whole step can be captured once into a CUDA
graph and replayed at fixed addresses (workspace.py page, bullets 6-7; one
graph per batch size, executor.py page, bullets 4-5, 7-8).
"""
from __future__ import annotations

import torch

from . import _abi
from .workspace import Workspace


class BindTracker:
    """Host record of the last bind (the engine's _BindState; cache.py page,
    bullets 1-4): picks STEADY when the same tasks each grew by one token."""

    def __init__(self):
        self.ids = None
        self.lens = None

    def mode(self, ids, lens):
        steady = _abi.pkv_is_steady_increment(self.ids, self.lens, list(ids), list(lens))
        self.ids, self.lens = list(ids), list(lens)
        return _abi.PKV_BIND_STEADY if steady else _abi.PKV_BIND_REBUILD


class DecodeRunner:
    """Drives libpkv for one batch size on one stream."""

    def __init__(self, ws: Workspace, batch: int, *, num_splits: int = 1, flags: int = 0,
                 scale: float | None = None, stream: torch.cuda.Stream | None = None,
                 fused: bool = True, plan: bool = False, out_per_layer: bool = False):
        self.ws = ws
        self.batch = batch
        sh = ws.shape
        self.num_splits = num_splits
        self.flags = flags
        self.scale = scale if scale is not None else sh["head_dim"] ** -0.5
        self.stream = stream
        NL, B = sh["n_layers"], batch
        dev = ws.device
        self.q_in = torch.zeros((NL, B, sh["n_q_heads"], sh["head_dim"]), dtype=torch.bfloat16,
                                device=dev)
        self.k_in = torch.zeros((NL, B, sh["n_kv_heads"], sh["head_dim"]), dtype=torch.bfloat16,
                                device=dev)
        self.v_in = torch.zeros_like(self.k_in)
        # out_per_layer: every layer writes its own output rows (layer l's into
        # outs[l], through a copy of the workspace struct whose `out` points
        # there), so a step leaves all its layers' results behind instead of
        # the last one's in ws.out.  bf16, or fp32 with PKV_FLAG_OUT_F32.
        self.outs = None
        self.views = None
        if out_per_layer:
            odt = torch.float32 if flags & _abi.PKV_FLAG_OUT_F32 else torch.bfloat16
            self.outs = torch.zeros((NL, B, sh["n_q_heads"], sh["head_dim"]), dtype=odt,
                                    device=dev)
            self.views = []
            for l in range(NL):
                v = _abi.PkvWorkspace.from_buffer_copy(ws.struct)
                v.out = self.outs[l].data_ptr()
                self.views.append(v)
        self.graph = None
        self.fused = fused
        flat = sh["index_mode"] == _abi.PKV_IDX_FLAT
        # kernels one step launches: bind (+ flat index build), then per layer
        # one fused kernel, or append + attention (+ merge when split)
        split = num_splits > 1
        mma = (not (flags & _abi.PKV_FLAG_FORCE_SIMT) and sh["head_dim"] in (64, 128)
               and sh["n_q_heads"] // sh["n_kv_heads"] in (1, 2, 4, 8, 16))
        # plan=True: the fused layers take the step's split plan, made once after
        # the bind (pkv_plan_step).  Off by default: with the layers pipelined by
        # programmatic dependent launch the plan saves no time, and a one-layer
        # step pays for the extra launch.
        self.use_plan = plan and fused and mma and ws.work_plan is not None
        per_layer = 1 if fused and mma else 2 + int(split)
        self.launches_per_step = (1 + int(flat) + int(self.use_plan and 0 < batch <= 256) +
                                  NL * per_layer)

    def _wsl(self, l):
        return self.views[l] if self.views is not None else self.ws

    # --- pieces -------------------------------------------------------------
    def bind(self, mode=_abi.PKV_BIND_STEADY):
        _abi.pkv_bind_step(self.ws, self.batch, mode, 0, 0, None, None, self._s())
        if self.use_plan:
            _abi.pkv_plan_step(self.ws, self.batch, self.num_splits, self.flags, self._s())

    def layer(self, l, events=None):
        """Layer l: one fused launch (append + attention + merge), or the
        three separate kernels when built with fused=False."""
        s = self._s()
        if self.fused:
            if events is not None:
                events[0].record(s)
            # Layers after the first read metadata the step's bind wrote two or
            # more launches earlier, so they may start before layer l-1 ends.
            early = _abi.PKV_FLAG_PLAN_EARLY if (l > 0 and events is None) else 0
            use = _abi.PKV_FLAG_USE_PLAN if self.use_plan else 0
            _abi.pkv_decode_layer(self._wsl(l), self.batch, l, self.q_in[l], self.k_in[l],
                                  self.v_in[l], self.scale, self.num_splits,
                                  self.flags | early | use, s)
            if events is not None:
                events[1].record(s)
            return
        _abi.pkv_bind_step(self.ws, self.batch, _abi.PKV_BIND_APPEND_ONLY, l, 1, self.k_in[l],
                           self.v_in[l], s)
        if events is not None:
            events[0].record(s)
        _abi.pkv_decode_attn(self._wsl(l), self.batch, l, self.q_in[l], self.scale,
                             self.num_splits, self.flags, s)
        if events is not None:
            events[1].record(s)
        if self.num_splits > 1:
            _abi.pkv_merge_partials(self._wsl(l), self.batch, self.num_splits, self.flags, s)

    def step(self, mode=_abi.PKV_BIND_STEADY, layer_events=None):
        """Bind, then every layer.  ``layer_events[l]`` = (start, end) CUDA
        events recorded around that layer's attention kernel."""
        self.bind(mode)
        for l in range(self.ws.shape["n_layers"]):
            self.layer(l, None if layer_events is None else layer_events[l])

    # --- CUDA graph -----------------------------------------------------------
    def capture(self, mode=_abi.PKV_BIND_STEADY, layer_events=None):
        """Capture one whole step (bind + all layers) into a CUDA graph.

        ``layer_events[l]`` (events made with ``external=True``) become event
        record nodes around layer l's attention kernel."""
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=self.ws.device)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                self.step(mode, layer_events)
        torch.cuda.current_stream().wait_stream(side)
        self.graph = g
        return g

    def replay(self):
        self.graph.replay()

    def _s(self):
        if self.stream is not None:
            return self.stream
        return torch.cuda.current_stream()
