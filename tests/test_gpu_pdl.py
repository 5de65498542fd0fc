"""Programmatic dependent launch (DFLASH_PROBLEM_PDL): the kernels start while the kernel before
them drains, and must still see everything that kernel writes.

* Layers back to back on one stream and one shared workspace (the partial kernel of layer l + 1
  overlaps the combine of layer l, which still reads the workspace the partial kernel writes):
  the same bits as without the flag, launched eagerly and replayed from a CUDA graph.
* The kernel just before the forward writes Q (an elementwise kernel over a large buffer whose
  last elements are Q; Q starts as NaN): the output must be the oracle's for the new Q.
* The kernel just before the forward is the drafted tokens' KV write (their slots start as NaN
  codes): the attention must see the written codes.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import compare, oracle_forward, to_device, to_np
from speculative_verify_paged_e4m3_gb300 import workload as W

pytestmark = pytest.mark.gpu

D = 256


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_verify_paged_e4m3_gb300 import build
    build.build()


def stack_outputs(stack):
    torch.cuda.synchronize()
    return [to_np(o).copy() for o in stack.outs], [to_np(x).copy() for x in stack.lses]


@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("context", [3000, 70000])
def test_layers_back_to_back_same_bits_as_without(kernel, context):
    from speculative_verify_paged_e4m3_gb300 import binding as B
    from speculative_verify_paged_e4m3_gb300.runner import LayerStack
    w = W.Workload(f"pdl{context}", layers=4, context=(context,), seed_base=81000 + context)
    plain = LayerStack(w, device="cuda", kernel=kernel)
    pdl = LayerStack(w, device="cuda", kernel=kernel, flags=B.DFLASH_PROBLEM_PDL)
    plain.launch()
    want_out, want_lse = stack_outputs(plain)
    for o in pdl.outs:
        o.fill_(float("nan"))
    pdl.launch()
    got_out, got_lse = stack_outputs(pdl)
    for a, b in zip(got_out + got_lse, want_out + want_lse):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    pdl.capture()
    for o in pdl.outs:
        o.fill_(float("nan"))
    pdl.replay()
    pdl.replay()
    got_out, got_lse = stack_outputs(pdl)
    for a, b in zip(got_out + got_lse, want_out + want_lse):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    # and against the oracle, layer by layer (on the stack's own inputs, drawn on the device)
    for l in (0, 3):
        ref_out, ref_lse = oracle_forward({k: v.cpu() for k, v in pdl.layers[l].items()})
        compare(got_out[l], got_lse[l], ref_out, ref_lse, what=f"layer {l}")


@pytest.mark.parametrize("kernel", [1, 2])
def test_q_written_by_the_preceding_kernel_is_seen(kernel):
    from speculative_verify_paged_e4m3_gb300 import binding as B
    w = W.Workload("pdl_q", layers=1, context=(5000,), seed_base=82000)
    inp = W.make_layer(w, 0, device="cpu")
    dev = to_device(inp)
    q_src = dev["q"].clone()
    n_q = q_src.numel()
    big = 32 << 20  # elements: the writing kernel runs for a while, Q is its last stretch
    src = torch.zeros(big + n_q, dtype=torch.float16, device="cuda")
    src[big:] = q_src.reshape(-1)
    dst = torch.full_like(src, float("nan"))
    q_dev = dst[big:].view(q_src.shape)
    att = B.VerifyAttention(1, 8, 6, 1, D, 16, w.max_pages_per_seq, dev["k_pool"].shape[0],
                            w.max_ctx, kernel=kernel, flags=B.DFLASH_PROBLEM_PDL)
    for _ in range(2):
        dst.fill_(float("nan"))
        torch.add(src, 0, out=dst)  # an elementwise kernel, launched just before the forward
        out, lse = att(q_dev, dev["k_pool"], dev["v_pool"], dev["block_table"],
                       dev["context_lens"], dev["k_scale"], dev["v_scale"])
        torch.cuda.synchronize()
        ref_out, ref_lse = oracle_forward(inp)
        compare(to_np(out), to_np(lse), ref_out, ref_lse, what="Q from the preceding kernel")


@pytest.mark.parametrize("kernel", [1, 2])
def test_drafted_kv_written_by_the_preceding_kernel_is_seen(kernel):
    from speculative_verify_paged_e4m3_gb300 import binding as B
    q_len, P = 8, 16
    for n in (5000, 4097, 300):
        w = W.Workload(f"pdl_kv{n}", layers=1, context=(n,), seed_base=83000 + n)
        inp = W.make_layer(w, 0, device="cpu")
        rng = np.random.default_rng(n)
        k_new = torch.from_numpy(
            (rng.standard_normal((1, q_len, 1, D)) * 0.8).astype(np.float16))
        v_new = torch.from_numpy(
            (rng.standard_normal((1, q_len, 1, D)) * 0.8).astype(np.float16))
        dev = to_device(inp)
        # the drafted tokens' slots hold NaN codes until the KV write replaces them
        bt = inp["block_table"].numpy()[0]
        for pos in range(n - q_len, n):
            page = int(bt[pos // P])
            dev["k_pool"][page, pos % P] = 0x7F
            dev["v_pool"][page, pos % P] = 0x7F
        att = B.VerifyAttention(1, q_len, 6, 1, D, P, w.max_pages_per_seq,
                                dev["k_pool"].shape[0], w.max_ctx, kernel=kernel,
                                flags=B.DFLASH_PROBLEM_PDL)
        att.kv_write(k_new.cuda(), v_new.cuda(), dev["block_table"], dev["context_lens"],
                     dev["k_scale"], dev["v_scale"], dev["k_pool"], dev["v_pool"])
        out, lse = att(dev["q"], dev["k_pool"], dev["v_pool"], dev["block_table"],
                       dev["context_lens"], dev["k_scale"], dev["v_scale"])
        torch.cuda.synchronize()
        written = {k: v.cpu() for k, v in dev.items()}
        assert not np.any((to_np(written["k_pool"])[bt[(n - 1) // P], (n - 1) % P] & 0x7F)
                          == 0x7F), "the KV write did not land"
        ref_out, ref_lse = oracle_forward(written)
        compare(to_np(out), to_np(lse), ref_out, ref_lse, what=f"drafted KV, n={n}")
