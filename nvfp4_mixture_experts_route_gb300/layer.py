"""The routed NVFP4 expert block as one object over the C ABI.

``NvFp4MoE`` holds one layer's prepared weights and scalars on the device and
runs the hot path on the current stream: routing metadata, the expert body
(input quantization, GEMM1 + SwiGLU + requant, GEMM2) and the post-expert
finalize, as one call (moe_nvfp4_moe_block) or as the routed body then the
finalize. It only allocates (once, then reuses) and passes
pointers; the work is the library's.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B


class NvFp4MoE:
    def __init__(self, raw: dict, a1_gscale: float, a2_gscale: float, gamma_bits, eps: float = 1e-6,
                 tile_m: int = 32, weight_before_norm: bool = True, device="cuda", fused_norm: bool | None = None):
        """``raw``: numpy or torch uint8 w13 [E,2I,H/2], w13_sf [E,2I,H/16],
        w2 [E,H,I/2], w2_sf [E,H,I/16]; fp32 g1_alphas, g1_scale_c, g2_alphas
        [E]. ``gamma_bits``: bf16 bit patterns [H] (uint16) or a bf16 tensor.
        ``fused_norm``: True: the whole block through moe_nvfp4_moe_block
        (GEMM2's epilogue also writes the rows' sums of squares; the finalize
        runs from them); False: moe_nvfp4_experts_routed, then
        moe_post_expert_finalize; None (the default): the first for route
        tiles of at most 64 rows (decode batches), the second otherwise (at
        prefill the sums of squares cost GEMM2 more than they save in the
        finalize)."""
        dev = torch.device(device)
        t = {k: torch.as_tensor(raw[k]).to(dev) for k in ("w13", "w13_sf", "w2", "w2_sf")}
        self.E, twoI, half_h = t["w13"].shape
        self.I, self.H = twoI // 2, 2 * half_h
        self.prepared = B.prepare_weights(t["w13"], t["w13_sf"], t["w2"], t["w2_sf"])
        del t
        f32 = dict(dtype=torch.float32, device=dev)
        self.g1_alphas = torch.as_tensor(raw["g1_alphas"]).to(**f32).contiguous()
        self.g1_scale_c = torch.as_tensor(raw["g1_scale_c"]).to(**f32).contiguous()
        self.g2_alphas = torch.as_tensor(raw["g2_alphas"]).to(**f32).contiguous()
        self.a1_gscale = torch.tensor([a1_gscale], **f32)
        self.a2_gscale = torch.tensor([a2_gscale], **f32)
        if isinstance(gamma_bits, torch.Tensor) and gamma_bits.dtype == torch.bfloat16:
            g = gamma_bits
        else:
            g = torch.from_numpy(np.asarray(gamma_bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
        self.gamma = g.to(dev).contiguous()
        self.eps = float(eps)
        self.tile_m = tile_m
        self.weight_before_norm = weight_before_norm
        self.fused_norm = fused_norm
        self.device = dev
        self.weights = B.weights_struct(self.prepared, self.g1_alphas, self.g1_scale_c, self.g2_alphas)
        self._buffers: dict = {}

    def buffers(self, T: int, K: int) -> dict:
        """Per-(T, K) metadata, workspace and output buffers, made once."""
        key = (T, K)
        if key not in self._buffers:
            P, _ = B.route_sizes(T, K, self.E, self.tile_m)
            self._buffers[key] = {
                "route": B.alloc_route(T, K, self.E, self.tile_m, self.device),
                "ws": B.alloc_workspace(T, K, self.E, self.H, self.I, self.tile_m, self.device),
                "rows": torch.empty((max(P, 1), self.H), dtype=torch.bfloat16, device=self.device),
                "row_sumsq": torch.empty((max(P, 1), self.H // 32), dtype=torch.float32, device=self.device),
                "out": torch.empty((T, self.H), dtype=torch.bfloat16, device=self.device),
                "status": torch.zeros(1, dtype=torch.int32, device=self.device),
            }
        return self._buffers[key]

    def forward(self, x, topk_ids, topk_weights, out=None, status=None):
        """x bf16 [T, H], topk_ids int32 [T, K], topk_weights fp32 [T, K] ->
        bf16 [T, H]. Returns (out, buffers) ; buffers hold the metadata and the
        GEMM2 rows of this call."""
        T, K = topk_ids.shape
        b = self.buffers(T, K)
        st = b["status"] if status is None else status
        o = b["out"] if out is None else out
        fused = self.fused_norm
        if fused is None:
            fused = B.experts_kernels(self.tile_m) == 2
        if fused:
            B.moe_block(self.weights, topk_ids, topk_weights, b["route"], x=x, a1_gscale=self.a1_gscale,
                        a2_gscale=self.a2_gscale, gamma=self.gamma, eps=self.eps,
                        weight_before_norm=self.weight_before_norm, H=self.H, I=self.I, E=self.E,
                        gemm2_rows=b["rows"], row_sumsq=b["row_sumsq"], out=o, ws=b["ws"], status=st)
            return o, b
        # routing and the expert body in one call (for few routes the routing
        # runs inside the input quantizer)
        B.nvfp4_experts_routed(self.weights, topk_ids, b["route"], x=x, a1_gscale=self.a1_gscale,
                               a2_gscale=self.a2_gscale, H=self.H, I=self.I, E=self.E, gemm2_rows=b["rows"],
                               ws=b["ws"], status=st)
        B.post_expert_finalize(b["rows"], b["route"].expanded_to_permuted, topk_weights, self.gamma, self.eps,
                               self.weight_before_norm, out=o, status=st)
        return o, b

    # -- CUDA-graph serving path -------------------------------------------
    def graph_buffers(self, T: int, K: int) -> dict:
        """Static input and output tensors of the graphed step for (T, K):
        ``x`` bf16 [T, H], ``topk_ids`` int32 [T, K], ``topk_weights`` fp32
        [T, K] (fill them, e.g. straight from pinned host memory), and
        ``out`` bf16 [T, H] (read it after ``replay``)."""
        key = ("graph", T, K)
        if key not in self._buffers:
            dev = self.device
            # x, topk_ids and topk_weights share one allocation (``inputs``,
            # bytes) so that a caller can fill all three with one copy, e.g.
            # from a pinned host buffer laid out by ``input_layout``.
            offs, nbytes = self.input_layout(T, K)
            flat = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
            self._buffers[key] = {
                "inputs": flat,
                "x": flat[offs["x"]:offs["x"] + T * self.H * 2].view(torch.bfloat16).view(T, self.H),
                "topk_ids": flat[offs["topk_ids"]:offs["topk_ids"] + T * K * 4].view(torch.int32).view(T, K),
                "topk_weights": flat[offs["topk_weights"]:offs["topk_weights"] + T * K * 4]
                .view(torch.float32).view(T, K),
                "out": torch.empty((T, self.H), dtype=torch.bfloat16, device=dev),
                "graph": None,
            }
            self._buffers[key]["topk_ids"].fill_(-1)
        return self._buffers[key]

    def host_buffers(self, T: int, K: int) -> dict:
        """Pinned host staging of the step for (T, K): ``host_inputs`` (bytes
        laid out by ``input_layout``: x, topk_ids, topk_weights) and
        ``host_out`` bf16 [T, H]. ``replay_host`` copies the one in and the
        other out inside its graph."""
        key = ("host", T, K)
        if key not in self._buffers:
            _, nbytes = self.input_layout(T, K)
            self._buffers[key] = {
                "host_inputs": torch.zeros(nbytes, dtype=torch.uint8).pin_memory(),
                "host_out": torch.empty((T, self.H), dtype=torch.bfloat16).pin_memory(),
                "graph": None,
            }
        return self._buffers[key]

    def zero_copy(self, T: int, K: int) -> bool:
        """Whether ``replay_host(T, K)`` runs zero-copy: at decode sizes (route
        tiles of at most 64 rows) its kernels read the step's inputs straight
        from ``host_inputs`` and the finalize writes ``host_out`` directly,
        where the device maps that page-locked memory at its own address;
        otherwise two copies run around the step."""
        h = self.host_buffers(T, K)
        decode = B.experts_kernels(self.tile_m) == 2
        fused = self.fused_norm if self.fused_norm is not None else decode
        return bool(fused and decode and
                    B.device_reads_host(h["host_inputs"]) and B.device_reads_host(h["host_out"]))

    def replay_host(self, T: int, K: int) -> torch.Tensor:
        """One CUDA graph replay of a serving step from pinned host memory:
        the step's inputs come from ``host_buffers(T, K)["host_inputs"]``
        and its output lands in ``host_out``, all on the current stream.
        Zero-copy at decode sizes (``zero_copy``: the kernels read and write
        the pinned buffers over the host link themselves), else a copy in,
        the step, and a copy out. Returns ``host_out``; read it after the
        stream is synchronised."""
        h = self.host_buffers(T, K)
        if self.zero_copy(T, K):
            offs, _ = self.input_layout(T, K)
            hi = h["host_inputs"]
            x = hi[offs["x"]:offs["x"] + T * self.H * 2].view(torch.bfloat16).view(T, self.H)
            ids = hi[offs["topk_ids"]:offs["topk_ids"] + T * K * 4].view(torch.int32).view(T, K)
            tw = hi[offs["topk_weights"]:offs["topk_weights"] + T * K * 4].view(torch.float32).view(T, K)

            def step():
                self.forward(x, ids, tw, out=h["host_out"])
        else:
            g = self.graph_buffers(T, K)

            def step():
                g["inputs"].copy_(h["host_inputs"], non_blocking=True)
                self.forward(g["x"], g["topk_ids"], g["topk_weights"], out=g["out"])
                h["host_out"].copy_(g["out"], non_blocking=True)

        if h["graph"] is None:
            step()  # warm-up, outside capture
            torch.cuda.current_stream(self.device).synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                step()
            h["graph"] = graph
        h["graph"].replay()
        return h["host_out"]

    def input_layout(self, T: int, K: int) -> tuple[dict, int]:
        """Byte offsets of x, topk_ids and topk_weights inside ``inputs`` (each
        16-byte aligned) and its size."""
        up = lambda n: (n + 15) // 16 * 16  # noqa: E731
        o_ids = up(T * self.H * 2)
        o_w = o_ids + up(T * K * 4)
        return {"x": 0, "topk_ids": o_ids, "topk_weights": o_w}, o_w + up(T * K * 4)

    def replay(self, T: int, K: int) -> torch.Tensor:
        """Run the step on ``graph_buffers(T, K)`` as one CUDA graph replay
        (captured on first use: routing, expert body and finalize, with the
        weights current at capture time). Returns the static ``out``."""
        g = self.graph_buffers(T, K)
        if g["graph"] is None:
            self.forward(g["x"], g["topk_ids"], g["topk_weights"], out=g["out"])  # warm-up, outside capture
            torch.cuda.current_stream(self.device).synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                self.forward(g["x"], g["topk_ids"], g["topk_weights"], out=g["out"])
            g["graph"] = graph
        g["graph"].replay()
        return g["out"]

    # -- pipelined serving from pinned host memory --------------------------
    def host_pipeline(self, T: int, K: int, depth: int = 2) -> dict:
        """Slots of the pipelined serving call for (T, K): ``depth`` sets of
        pinned ``host_inputs`` (bytes laid out by ``input_layout``) and
        ``host_out`` bf16 [T, H], each with its own device buffers and step
        graph, and three streams (copy in, step, copy out)."""
        key = ("pipe", T, K, depth)
        if key not in self._buffers:
            offs, nbytes = self.input_layout(T, K)
            dev = self.device
            slots = []
            for _ in range(depth):
                flat = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
                s = {
                    "host_inputs": torch.zeros(nbytes, dtype=torch.uint8).pin_memory(),
                    "host_out": torch.empty((T, self.H), dtype=torch.bfloat16).pin_memory(),
                    "inputs": flat,
                    "x": flat[offs["x"]:offs["x"] + T * self.H * 2].view(torch.bfloat16).view(T, self.H),
                    "topk_ids": flat[offs["topk_ids"]:offs["topk_ids"] + T * K * 4].view(torch.int32).view(T, K),
                    "topk_weights": flat[offs["topk_weights"]:offs["topk_weights"] + T * K * 4]
                    .view(torch.float32).view(T, K),
                    "out": torch.empty((T, self.H), dtype=torch.bfloat16, device=dev),
                    "graph": None,
                    "used": False,
                    "in_ready": torch.cuda.Event(),
                    "computed": torch.cuda.Event(),
                    "out_ready": torch.cuda.Event(),
                }
                s["topk_ids"].fill_(-1)
                slots.append(s)
            self._buffers[key] = {"slots": slots, "copy_in": torch.cuda.Stream(dev),
                                  "step": torch.cuda.Stream(dev), "copy_out": torch.cuda.Stream(dev)}
        return self._buffers[key]

    def pipeline_begin(self, T: int, K: int, depth: int = 2) -> None:
        """Order the pipeline's streams after the work already on the current
        stream (call once before a run of ``submit_host``)."""
        p = self.host_pipeline(T, K, depth)
        ev = torch.cuda.Event()
        ev.record(torch.cuda.current_stream(self.device))
        for st in (p["copy_in"], p["step"], p["copy_out"]):
            st.wait_event(ev)

    def submit_host(self, T: int, K: int, slot: int, depth: int = 2) -> torch.cuda.Event:
        """Enqueue one serving step on slot ``slot`` of ``host_pipeline``: the
        copy of its ``host_inputs`` to the device, the step (one graph replay:
        routing, expert body, finalize), and the copy of its output to
        ``host_out``, each on its own stream, ordered by events. Consecutive
        steps on alternating slots overlap one step's copies with the
        neighbouring steps' kernels. Returns the event after which ``host_out``
        of this slot holds the result. Fill ``host_inputs`` before the call,
        and wait for the slot's previous event before refilling it or reading
        its ``host_out``. The steps share the layer's workspace for (T, K)
        with ``forward``, ``replay`` and ``replay_host``: between
        ``pipeline_begin`` and ``pipeline_join`` make no other call of this
        layer for the same shape."""
        p = self.host_pipeline(T, K, depth)
        s = p["slots"][slot]
        cin, stp, cout = p["copy_in"], p["step"], p["copy_out"]
        if s["used"]:
            cin.wait_event(s["computed"])  # the slot's device inputs were read by its last step
        with torch.cuda.stream(cin):
            s["inputs"].copy_(s["host_inputs"], non_blocking=True)
            s["in_ready"].record(cin)
        stp.wait_event(s["in_ready"])
        if s["used"]:
            stp.wait_event(s["out_ready"])  # the slot's device output was copied out
        with torch.cuda.stream(stp):
            if s["graph"] is None:
                self.forward(s["x"], s["topk_ids"], s["topk_weights"], out=s["out"])  # warm-up, outside capture
                stp.synchronize()
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph):
                    self.forward(s["x"], s["topk_ids"], s["topk_weights"], out=s["out"])
                s["graph"] = graph
            s["graph"].replay()
            s["computed"].record(stp)
        cout.wait_event(s["computed"])
        with torch.cuda.stream(cout):
            s["host_out"].copy_(s["out"], non_blocking=True)
            s["out_ready"].record(cout)
        s["used"] = True
        return s["out_ready"]

    def pipeline_join(self, T: int, K: int, depth: int = 2) -> None:
        """Make the current stream wait for every step submitted so far."""
        p = self.host_pipeline(T, K, depth)
        cur = torch.cuda.current_stream(self.device)
        for s in p["slots"]:
            if s["used"]:
                cur.wait_event(s["out_ready"])
