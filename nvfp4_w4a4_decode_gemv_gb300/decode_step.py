"""One synthetic Qwen3-shaped decode step through the C ABI.

Per layer (the four NVFP4 projections of a Qwen3 decoder layer, ReSET project
page "Core contribution"; reading note §6.1 setup):

    xq   = NVFP4(BF16(RMSNorm(h)))         nvfp4_rms_norm_quantize    (one launch)
    qkv  = xq . Wqkv^T                     nvfp4_gemv_smallm_packed   FP32 [M, 10240]
    xo   = NVFP4(BF16(qkv[:, :8192]))      nvfp4_quantize_f32         (the query part; no attention)
    o    = xo . Wo^T                                                  FP32 [M, 5120]
    xg   = NVFP4(BF16(RMSNorm(o)))         nvfp4_rms_norm_quantize
    gu   = xg . Wgate_up^T                                            FP32 [M, 51200]
    xd   = NVFP4(BF16(SiLU(gate) * up))    nvfp4_silu_mul_quantize
    h    = xd . Wdown^T                                               FP32 [M, 5120] -> next layer

then logits = BF16(RMSNorm(h)) . Wlm^T (nvfp4_bf16_gemv_tc) and the ReSET sampler
(reset_sample).  Weights are random (N(0, 0.02) in BF16, quantized and packed
once); the step is issued on one stream and can be captured as one CUDA graph.
Every computation runs in the library's kernels; this module only orders the
calls and owns the buffers.
"""
import torch

from . import api, synth
from ._lib import ResetParams


class DecodeStep:
    def __init__(self, M: int, layers: int, shapes=synth.QWEN3_32B, vocab: int = synth.LM_HEAD_VOCAB,
                 seed: int = 0, eps: float = 1e-6, reset: ResetParams | None = None, keep_rowmajor: bool = False,
                 device="cuda", share_weights: "DecodeStep | None" = None):
        (_, hidden, n_qkv), (_, k_o, _), (_, _, n_gu), (_, k_d, _) = shapes
        self.M, self.layers, self.hidden, self.vocab, self.eps = M, layers, hidden, vocab, eps
        self.n_qkv, self.k_o, self.n_gu, self.k_d = n_qkv, k_o, n_gu, k_d
        dev = torch.device(device)
        self.device = dev
        self.weights = []          # per layer: {name: NVFP4PackedWeight}
        self.rowmajor = []         # per layer (keep_rowmajor): {name: NVFP4Tensor}
        if share_weights is not None:  # another step's weights and lm_head (steps of other M on one model)
            assert share_weights.layers == layers and share_weights.hidden == hidden
            self.weights, self.rowmajor = share_weights.weights, share_weights.rowmajor
        for layer in range(0 if share_weights is not None else layers):
            packed, rm = {}, {}
            for i, (name, K, N) in enumerate(shapes):
                g = torch.Generator(device=dev)
                g.manual_seed(seed * 100003 + layer * 16 + i)
                wb = (torch.randn((N, K), generator=g, device=dev) * synth.W_STD).to(torch.bfloat16)
                wq = api.nvfp4_quantize_act(wb)
                del wb
                packed[name] = api.nvfp4_pack_weights(wq)
                if keep_rowmajor:
                    rm[name] = wq
            self.weights.append(packed)
            self.rowmajor.append(rm)
        if share_weights is not None:
            self.lm_head = share_weights.lm_head
        else:
            g = torch.Generator(device=dev)
            g.manual_seed(seed * 100003 + 99991)
            self.lm_head = (torch.randn((vocab, hidden), generator=g, device=dev) * synth.W_STD).to(torch.bfloat16)
        # activations and intermediates (reused by every layer)
        f32 = dict(dtype=torch.float32, device=dev)
        self.h_in = torch.zeros((M, hidden), **f32)          # the step's input hidden state
        self.h = torch.empty((M, hidden), **f32)
        self.r = torch.empty((M, hidden), dtype=torch.bfloat16, device=dev)
        self.xq = api.NVFP4Tensor.empty(M, hidden, dev)
        self.y_qkv = torch.empty((M, n_qkv), **f32)
        self.xq_o = api.NVFP4Tensor.empty(M, k_o, dev)
        self.y_o = torch.empty((M, hidden), **f32)
        self.xq_gu = api.NVFP4Tensor.empty(M, hidden, dev)
        self.y_gu = torch.empty((M, n_gu), **f32)
        self.xq_d = api.NVFP4Tensor.empty(M, k_d, dev)
        self.logits = torch.empty((M, vocab), **f32)
        need = max(api.nvfp4_gemv_workspace_bytes(M, N, K) for _, K, N in shapes)
        self.ws = torch.zeros(need, dtype=torch.uint8, device=dev)
        rp = reset or ResetParams(0.6, 0.3, 1.0, 8)
        self.sampler = api.ResetSampler(M, vocab, rp.tau0, rp.t_low, rp.t_high, rp.w, device=dev)
        self.sampler.params = rp                     # threshold policy and top-p as given
        self.step_start = torch.zeros(M, dtype=torch.uint8, device=dev)
        self.u = torch.zeros(M, dtype=torch.float32, device=dev)
        self.graph = None

    # ---- the chain ------------------------------------------------------------
    def _layer(self, layer: int, h_in: torch.Tensor, stream, trace):
        w = self.weights[layer]
        api.nvfp4_rms_norm_quantize(h_in, eps=self.eps, out=self.xq, r_out=self.r_out(trace), stream=stream)
        api.nvfp4_gemv_smallm_packed(self.xq, w["qkv"], y=self.y_qkv, workspace=self.ws, stream=stream)
        api.nvfp4_quantize_f32(self.y_qkv, K=self.k_o, out=self.xq_o, stream=stream)
        api.nvfp4_gemv_smallm_packed(self.xq_o, w["o"], y=self.y_o, workspace=self.ws, stream=stream)
        if trace is not None:
            nv = lambda t: (t.codes.clone(), t.scales.clone(), t.global_scale.clone())
            trace.append({"h_in": h_in.clone(), "r": self.r.clone(), "xq": nv(self.xq), "y_qkv": self.y_qkv.clone(),
                          "xq_o": nv(self.xq_o), "y_o": self.y_o.clone()})
        api.nvfp4_rms_norm_quantize(self.y_o, eps=self.eps, out=self.xq_gu, r_out=self.r_out(trace), stream=stream)
        api.nvfp4_gemv_smallm_packed(self.xq_gu, w["gate_up"], y=self.y_gu, workspace=self.ws, stream=stream)
        api.nvfp4_silu_mul_quantize(self.y_gu, out=self.xq_d, stream=stream)
        api.nvfp4_gemv_smallm_packed(self.xq_d, w["down"], y=self.h, workspace=self.ws, stream=stream)
        if trace is not None:
            trace[-1].update({"r2": self.r.clone(), "xq_gu": nv(self.xq_gu), "y_gu": self.y_gu.clone(),
                              "xq_d": (self.xq_d.codes.clone(), self.xq_d.scales.clone(),
                                       self.xq_d.global_scale.clone()),
                              "h_out": self.h.clone()})

    def r_out(self, trace):
        """Where the fused normalize+quantize launches put their BF16 rows: only
        traced runs keep them (the projections read the NVFP4 codes)."""
        return self.r if trace is not None else None

    def run(self, stream=None, trace=None):
        """Issue one decode step on `stream` (the current stream by default):
        h_in, step_start, u -> sampler.token / .H / .T.  With a list `trace`,
        the intermediates of every layer are appended to it (eager runs only)."""
        h_in = self.h_in
        for layer in range(self.layers):
            self._layer(layer, h_in, stream, trace)
            h_in = self.h
        api.nvfp4_rms_norm_bf16(h_in, eps=self.eps, out=self.r, stream=stream)   # the last layer's output
        api.nvfp4_bf16_gemv_tc(self.r, self.lm_head, y=self.logits, workspace=self.ws, stream=stream)
        if trace is not None:
            trace.append({"h_final": h_in.clone(), "r_final": self.r.clone(), "logits": self.logits.clone()})
        return self.sampler(self.logits, self.step_start, self.u, stream=stream)

    def capture(self):
        """Capture one step as a CUDA graph (run eagerly once first so that
        every kernel's attributes are set outside the capture)."""
        stream = torch.cuda.Stream(device=self.device)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(self.graph, stream=stream):
                self.run()
        return self.graph
