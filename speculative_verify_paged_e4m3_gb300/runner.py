"""Sixteen layers of one workload resident on the GPU, run back to back and under CUDA-graph
replay, as the pages time them ("[Perf] Reduce DFlash2 attention cost and screen exact QK reuse",
Test Plan: sixteen distinct layer KV allocations, alternating graph replay trials).

Every layer owns its Q, K/V page pools, block table, scales, output and LSE; the layers share one
plan and one workspace (they run in order on one stream). Marshalling only: the computation is the
library's kernels.
"""
from __future__ import annotations

import torch

from . import binding as B
from . import workload as W


def algorithmic_bytes(w: W.Workload, plan) -> dict:
    """Bytes one layer's kernels must move at minimum (for the roofline), per launch.

    partial kernel: K and V codes of the N logical tokens, the used block-table entries, Q, and
    the split state it writes; combine: the split state it reads, out and lse.
    """
    D, G = w.head_dim, w.num_q_heads // w.num_kv_heads
    R = w.q_len * G
    kv = w.kv_bytes_per_layer()
    bt = sum(-(-n // w.page_size) for n in w.context) * 4
    q = w.batch * w.q_len * w.num_q_heads * D * 2
    _, _, act = B.dflash_verify_attn_split_slots(plan, w.context)
    active = sum(act)
    state = active * R * (D + 2) * 4
    out = w.batch * w.q_len * w.num_q_heads * (D * 2 + 4)
    return dict(partial=kv + bt + q + state, combine=state + out, kv=kv, bt=bt, q=q,
                state=state, out=out, active_splits=active)


class LayerStack:
    def __init__(self, w: W.Workload, device="cuda", num_splits=0, kernel=B.DFLASH_KERNEL_AUTO,
                 layers=None, flags=0):
        self.w = w
        self.device = torch.device(device)
        n_layers = w.layers if layers is None else layers
        self.layers = [W.make_layer(w, l, device=self.device) for l in range(n_layers)]
        self.att = B.VerifyAttention(w.batch, w.q_len, w.num_q_heads, w.num_kv_heads,
                                     w.head_dim, w.page_size, w.max_pages_per_seq, w.num_pages,
                                     w.max_ctx, device=self.device.index or 0,
                                     num_splits=num_splits, kernel=kernel, flags=flags)
        shape = (w.batch, w.q_len, w.num_q_heads, w.head_dim)
        self.outs = [torch.empty(shape, dtype=torch.float16, device=self.device)
                     for _ in self.layers]
        self.lses = [torch.empty(shape[:3], dtype=torch.float32, device=self.device)
                     for _ in self.layers]
        self.graph = None

    @property
    def plan(self):
        return self.att.plan

    def launch(self, stream=None, plan=None):
        """16 x (partial attention + combine), enqueued on the stream (with another plan of the
        same shapes, e.g. other launch flags, when given)."""
        plan = self.plan if plan is None else plan
        for lay, out, lse in zip(self.layers, self.outs, self.lses):
            B.dflash_verify_attn_forward(plan, lay["q"], lay["k_pool"], lay["v_pool"],
                                         lay["block_table"], lay["context_lens"], lay["k_scale"],
                                         lay["v_scale"], self.att.workspace, out, lse, stream)

    def launch_partial(self, stream=None):
        """Only the partial-attention kernels of the 16 layers."""
        for lay in self.layers:
            B.dflash_verify_attn_run(self.plan, lay["q"], lay["k_pool"], lay["v_pool"],
                                     lay["block_table"], lay["context_lens"], lay["k_scale"],
                                     lay["v_scale"], self.att.workspace, stream)

    def launch_combine(self, stream=None):
        """Only the combine kernels of the 16 layers (re-reading the workspace state)."""
        for lay, out, lse in zip(self.layers, self.outs, self.lses):
            B.dflash_verify_attn_combine(self.plan, self.att.workspace, lay["context_lens"], out,
                                         lse, stream)

    def _capture(self, fn):
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream(self.device).wait_stream(s)
        torch.cuda.synchronize(self.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize(self.device)
        return g

    def capture(self):
        """Capture one 16-layer step into a CUDA graph (warm-up launch first)."""
        self.graph = self._capture(self.launch)
        return self.graph

    def capture_kernel_graphs(self):
        """Graphs of the 16 partial kernels alone and of the 16 combine kernels alone, so that
        each kernel's device time can be taken from CUDA events without host launch gaps."""
        return self._capture(self.launch_partial), self._capture(self.launch_combine)

    def replay(self):
        self.graph.replay()
