"""Failure detection on the GPU without a fault.

Every mbarrier wait of the GEMM kernels is bounded (clock64 budget) and
watches an abort flag in the workspace status words.  The debug hook
MOE_MXQ_DEBUG_INJECT_WAIT=1 makes each CTA's MMA warp first wait on a barrier
that nothing completes.  That wait must give up on its own (~10 ms), record
MOE_ERR_TIMEOUT with its site, raise the abort flag so that the producer and
epilogue warps of every CTA leave their loops (after draining their own
copies and MMAs), and leave the context usable: the next call in the same
process matches the oracle.
"""
import time

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

WAIT_SITE_INJECTED = 7


def _tiny(tile_n=0, wl=None, schedule=0):
    import workloads as W
    from moe_expert_layer_counting_gb300.layer import MoELayer, QuantizedExperts
    wl = wl or W.WORKLOADS["tiny"]
    x, logits = W.tokens(wl)
    l1, l2 = W.all_expert_weights(wl, "cpu")
    qe = QuantizedExperts.from_bf16(l1.cuda(), l2.cuda())
    return wl, x, logits, l1, l2, MoELayer(qe, wl.k, wl.T, tile_n=tile_n, schedule=schedule)


def _oracle_y(wl, x, logits, l1, l2):
    from oracle import moe as O

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    w1q, w1s = O.quantize_weight(bits(l1))
    w2q, w2s = O.quantize_weight(bits(l2))
    return O.forward(bits(x), logits.numpy(), w1q, w1s, w2q, w2s, wl.k)["y"]


@pytest.mark.parametrize("case", ["tile16", "tile32", "pairs", "pair_layer"])
def test_injected_wait_times_out_then_recovers(monkeypatch, case):
    """tile16: GEMM1 + GEMM2 + combine in one launch (CTAs also wait on one
    another's arrival counters); tile32: separate GEMM launches; pairs: the
    GEMMs on CTA pairs as separate launches (the leader's MMA issuers take the
    injected wait, the other CTA of each pair must give up through the abort
    flag); pair_layer: a larger problem whose GEMM1 + GEMM2 + combine run in
    one launch on CTA pairs under the expert-wave schedule (GEMM2 items also
    wait on arrival counters)."""
    from helpers import lib
    lib()
    import workloads as W
    from moe_expert_layer_counting_gb300 import binding as B
    from oracle import formats as F

    if case == "pair_layer":
        wl = W.Workload("pair_layer", T=700, H=512, I=256, E=6, k=2, sigma=0.02, seed=21)
        wl, x, logits, l1, l2, layer = _tiny(0, wl, schedule=2)
    else:
        wl, x, logits, l1, l2, layer = _tiny({"tile16": 16, "tile32": 32, "pairs": 224}[case])
    xd, ld = x.cuda(), logits.cuda()
    layer(xd, ld)                                  # warm-up (module load, tensor maps)
    torch.cuda.synchronize()
    assert layer.device_status() == B.MOE_OK

    monkeypatch.setenv("MOE_MXQ_DEBUG_INJECT_WAIT", "1")
    t0 = time.perf_counter()
    layer(xd, ld)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    words = layer.workspace[:20].view(torch.int32).cpu().tolist()
    assert layer.device_status() == B.MOE_ERR_TIMEOUT, words
    assert words[1] == 1, f"abort flag not raised: {words}"
    assert words[2] == WAIT_SITE_INJECTED, f"timeout recorded at site {words[2]}: {words}"
    assert elapsed < 5.0, f"the failing call took {elapsed:.2f} s"

    monkeypatch.delenv("MOE_MXQ_DEBUG_INJECT_WAIT")
    y = layer(xd, ld)
    torch.cuda.synchronize()
    assert layer.device_status() == B.MOE_OK
    ref = _oracle_y(wl, x, logits, l1, l2)
    g = F.bf16_bits_to_f64(y.cpu().view(torch.int16).numpy().view(np.uint16))
    r = F.bf16_bits_to_f64(ref)
    fro = np.linalg.norm(g - r) / np.linalg.norm(r)
    assert fro <= 5e-3 and np.max(np.abs(g - r)) <= 1e-2 * np.max(np.abs(r))
