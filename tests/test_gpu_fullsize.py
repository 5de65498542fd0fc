"""Full-size workloads in the launch configuration the benchmark times (16 layers, each with its
own KV allocation, launched as programmatic dependents, captured in one CUDA graph and replayed),
checked against the oracle on sampled layers (the first and the last: every row of those layers,
element by element)."""
import gc

import pytest
import torch

from gpu_helpers import compare, oracle_forward, to_np
from speculative_verify_paged_e4m3_gb300 import workload as W

pytestmark = pytest.mark.gpu

CASES = [W.config1(), W.config2(), W.config3(), W.config5(), W.config6(4, 65536)] + [
    W.config4(q, n) for n in W.TAIL_CONTEXTS for q in W.TAIL_QLENS] + [
    W.config4(16, 262144), W.config4(10, 65536)]  # more rows than one CTA holds: row blocks


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_verify_paged_e4m3_gb300 import build
    build.build()


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_full_size_graph_replay_sampled_layers(w):
    from speculative_verify_paged_e4m3_gb300 import binding as B
    from speculative_verify_paged_e4m3_gb300.runner import LayerStack
    stack = LayerStack(w, device="cuda", flags=B.DFLASH_PROBLEM_PDL)
    try:
        stack.capture()
        stack.replay()
        torch.cuda.synchronize()
        status = stack.att.workspace_views()[0].item()
        assert status == 0, f"device status flags {status:#x}"
        for layer in (0, w.layers - 1):
            inp = {k: v.cpu() for k, v in stack.layers[layer].items()}
            ref_out, ref_lse = oracle_forward(inp)
            compare(to_np(stack.outs[layer]), to_np(stack.lses[layer]), ref_out, ref_lse,
                    what=f"{w.name} layer {layer}")
    finally:
        del stack
        gc.collect()
        torch.cuda.empty_cache()
