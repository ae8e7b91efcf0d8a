"""The MXFP4 latent-MoE layer as a Python object over the C-ABI.

Holds the expert weights on the device (canonical packed E2M1 codes, scales
prepacked once into the library's TILED layout) and calls moe_forward. Only
allocation and argument marshalling happen here.
"""
import torch

from . import abi


class MoeLayer:
    """Routed experts of one latent-MoE layer.

    w13 u8 [E][2I][d/2] (gate rows, then up rows), w13_s u8 [E][2I][d/32],
    w2 u8 [E][d][I/2], w2_s u8 [E][d][I/32], all CUDA tensors in the canonical
    layout; the layer keeps its own prepacked copies (BOXED codes, TILED
    scales), so the canonical tensors may be freed afterwards.
    """

    def __init__(self, w13, w13_s, w2, w2_s, k, kernel=abi.GEMM_AUTO, stream=None):
        E, two_i, half_d = w13.shape
        self.E, self.I, self.d, self.k, self.kernel = E, two_i // 2, half_d * 2, k, kernel
        dev = w13.device
        # one-time weight preparation: codes into the BOXED layout, scales TILED
        self.w13 = torch.empty_like(w13)
        self.w2 = torch.empty_like(w2)
        abi.moe_prepack_weights(w13.contiguous(), E * two_i, self.d, self.w13, stream)
        abi.moe_prepack_weights(w2.contiguous(), E * self.d, self.I, self.w2, stream)
        self.w13_sf = torch.empty(abi.moe_tiled_scale_bytes(E * two_i, self.d), dtype=torch.uint8,
                                  device=dev)
        self.w2_sf = torch.empty(abi.moe_tiled_scale_bytes(E * self.d, self.I), dtype=torch.uint8,
                                 device=dev)
        abi.moe_prepack_scales(w13_s.contiguous(), E * two_i, self.d, self.w13_sf, stream)
        abi.moe_prepack_scales(w2_s.contiguous(), E * self.d, self.I, self.w2_sf, stream)

    def weight_bytes_per_expert(self):
        return 3 * self.d * self.I // 2 + 3 * self.d * self.I // 32

    def kernel_for(self, T):
        """The grouped-GEMM kernel family a call with T tokens uses."""
        return self.kernel or abi.moe_default_kernel(T, self.E, self.k)

    def workspace(self, T):
        n = abi.moe_workspace_size(T, self.d, self.E, self.k, self.I)
        return torch.empty(n, dtype=torch.uint8, device=self.w13.device)

    def forward(self, x, logits, ws=None, y=None, topk_ids=None, topk_w=None, stream=None,
                a4w4=False):
        """y = the layer on x. a4w4: MXFP4 stage-1 activations (moe_forward_a4w4;
        the kernel family then applies to stage 2)."""
        T = x.shape[0]
        if ws is None:
            ws = self.workspace(T)
        if y is None:
            y = torch.empty(T, self.d, dtype=torch.bfloat16, device=x.device)
        fn = abi.moe_forward_a4w4 if a4w4 else abi.moe_forward
        fn(T, self.d, self.E, self.k, self.I, self.kernel_for(T), x, logits, self.w13, self.w13_sf,
           self.w2, self.w2_sf, y, ws, topk_ids, topk_w, stream)
        return y

    def capture(self, x, logits, ws=None, y=None, topk_ids=None, topk_w=None, a4w4=False):
        """Records one forward on the given (static) buffers as a CUDA graph.

        The layer's entry points are stream-ordered and neither allocate nor
        synchronise, so the whole step (status reset, routing, grouping,
        quantisation, both GEMMs, combine) becomes one graph launch. Refill x
        and logits in place and call the returned graph's replay(); y (and the
        routing outputs, if given) hold the result. One eager call runs first
        so one-time host set-up happens outside the capture."""
        T = x.shape[0]
        if ws is None:
            ws = self.workspace(T)
        if y is None:
            y = torch.empty(T, self.d, dtype=torch.bfloat16, device=x.device)
        self.forward(x, logits, ws=ws, y=y, topk_ids=topk_ids, topk_w=topk_w, a4w4=a4w4)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.forward(x, logits, ws=ws, y=y, topk_ids=topk_ids, topk_w=topk_w, a4w4=a4w4)
        return g, y, ws


class MoeBlock:
    """The composed latent-MoE block (moe_block_forward): latent down
    projection and router on the hidden state, the routed experts in the
    latent, the two shared experts beside them on a second stream, and one
    output GEMM that adds the latent up projection of the routed output to the
    shared experts' down projection.

    BF16 weights (CUDA tensors): w_down [d][hidden], w_router [E][hidden],
    w_shared13 [2*shared_I][hidden] (both shared experts' gate rows, then
    their up rows), w_out [hidden][d + shared_I] (latent up columns, then the
    shared experts' down columns). Routed weights as MoeLayer.
    """

    def __init__(self, w_down, w_router, w_shared13, w_out, w13, w13_s, w2, w2_s, k,
                 kernel=abi.GEMM_AUTO):
        self.layer = MoeLayer(w13, w13_s, w2, w2_s, k, kernel=kernel)
        self.w_down, self.w_router = w_down.contiguous(), w_router.contiguous()
        self.w_shared13, self.w_out = w_shared13.contiguous(), w_out.contiguous()
        self.hidden = w_down.shape[1]
        self.shared_I = w_shared13.shape[0] // 2

    def dims(self, T):
        L = self.layer
        return (T, self.hidden, L.d, L.E, L.k, L.I, self.shared_I)

    def workspace(self, T):
        n = abi.moe_block_workspace_size(*self.dims(T))
        return torch.empty(n, dtype=torch.uint8, device=self.w_down.device)

    def forward(self, h, ws=None, out=None, stream=None, shared_stream=None):
        """out = the block on hidden states h bf16 [T][hidden]. shared_stream:
        the stream the shared experts run on (None: everything on `stream`)."""
        T = h.shape[0]
        if ws is None:
            ws = self.workspace(T)
        if out is None:
            out = torch.empty(T, self.hidden, dtype=torch.bfloat16, device=h.device)
        L = self.layer
        abi.moe_block_forward(*self.dims(T), L.kernel_for(T), h, self.w_down, self.w_router,
                              self.w_shared13, self.w_out, L.w13, L.w13_sf, L.w2, L.w2_sf, out,
                              ws, stream=stream, shared_stream=shared_stream)
        return out


class HostPipeline:
    """Runs the layer on batches held in (pinned) host memory with the copies
    off the compute stream.

    Batch i's inputs go host -> device on a copy stream while batch i-1
    computes; its output goes device -> host on a second copy stream while
    batch i+1 computes. `depth` sets of device buffers rotate; a set is
    refilled only after the forward that read it has finished, and its y only
    after the copy that drained it. submit() enqueues and returns at once;
    y_h holds batch i's result once synchronize() (or the event submit
    returns) has completed. All batches have T tokens.
    """

    def __init__(self, layer, T, depth=2, a4w4=False, device=None):
        dev = device or layer.w13.device
        self.layer, self.T, self.a4w4 = layer, T, a4w4
        self.compute = torch.cuda.current_stream(dev)
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        self.ws = layer.workspace(T)
        self.sets = []
        for _ in range(depth):
            self.sets.append({
                "x": torch.empty(T, layer.d, dtype=torch.bfloat16, device=dev),
                "logits": torch.empty(T, layer.E, dtype=torch.float32, device=dev),
                "y": torch.empty(T, layer.d, dtype=torch.bfloat16, device=dev),
                "in_ready": torch.cuda.Event(), "inputs_free": None, "y_free": None,
            })
        self.n = 0

    def submit(self, x_h, logits_h, y_h):
        """Enqueues one batch: x_h bf16 [T][d], logits_h fp32 [T][E] in,
        y_h bf16 [T][d] out (host tensors, pinned for asynchronous copies).
        Returns an event that completes when y_h holds the result."""
        T, d, E = self.T, self.layer.d, self.layer.E
        if (tuple(x_h.shape) != (T, d) or x_h.dtype != torch.bfloat16
                or tuple(logits_h.shape) != (T, E) or logits_h.dtype != torch.float32
                or tuple(y_h.shape) != (T, d) or y_h.dtype != torch.bfloat16):
            raise ValueError("HostPipeline.submit: expected x bf16 [%d][%d], logits fp32 "
                             "[%d][%d], y bf16 [%d][%d]" % (T, d, T, E, T, d))
        b = self.sets[self.n % len(self.sets)]
        self.n += 1
        with torch.cuda.stream(self.h2d):
            if b["inputs_free"] is not None:
                self.h2d.wait_event(b["inputs_free"])
            b["x"].copy_(x_h, non_blocking=True)
            b["logits"].copy_(logits_h, non_blocking=True)
            b["in_ready"].record(self.h2d)
        self.compute.wait_event(b["in_ready"])
        if b["y_free"] is not None:
            self.compute.wait_event(b["y_free"])
        self.layer.forward(b["x"], b["logits"], ws=self.ws, y=b["y"], stream=self.compute,
                           a4w4=self.a4w4)
        done = torch.cuda.Event()
        done.record(self.compute)
        b["inputs_free"] = done
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(done)
            y_h.copy_(b["y"], non_blocking=True)
            out = torch.cuda.Event()
            out.record(self.d2h)
        b["y_free"] = out
        return out

    def synchronize(self):
        self.h2d.synchronize()
        self.compute.synchronize()
        self.d2h.synchronize()
