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
