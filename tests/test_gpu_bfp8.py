"""Block-FP8 variant on the GPU against the float64 oracle (oracle/bfp8.py).

Casts are bit-exact (codes and float32 scales).  The layer is compared in
full: routing indices and the permute bit-exact, the requantised h within one
E4M3 step (at most 0.1 % of codes may move by one step; scales within 1e-4
relative -- the two sides' h differ by float32 accumulation), y within the
layer's tolerance (relative Frobenius error <= 5e-3, max error <= 1e-2 of
max |y|).  Shapes cover the MonoMoe kernel design's fixed shape (8 tokens,
E = 256, H = 2048, I = 512, top-8), several token tiles per expert, one
token, k = 1, a 7168-wide hidden size, ragged counts, E not a multiple
of 32, E = 300 (the chain of separate launches), and more GEMM1 items than
CTAs on both launch paths."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import bfp8 as OB
from oracle import formats as F
from oracle import moe as O
from tests import helpers as Hp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return Hp.lib()


def _rows_with_wide_range(rows, K, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, K, generator=g)
    mag = torch.exp2(torch.randint(-30, 31, (rows, K // 128, 1), generator=g).float())
    x = (x.view(rows, K // 128, 128) * mag).view(rows, K)
    x[0, :128] = 0.0
    x[1, 128:256] = -0.0
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("rows,K,seed", [(37, 1152, 1), (8, 2048, 2), (1, 128, 3)])
def test_quantize_act_bit_exact(B, rows, K, seed):
    x = _rows_with_wide_range(max(rows, 2), K, seed)[:rows].contiguous()
    q = torch.empty(rows, K, dtype=torch.uint8, device="cuda")
    s = torch.empty(rows, K // 128, dtype=torch.float32, device="cuda")
    B.bfp8_quantize_act(x.cuda(), q, s)
    torch.cuda.synchronize()
    q_r, s_r = OB.quantize_act(Hp.bits16(x))
    assert np.array_equal(q.cpu().numpy(), q_r)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_r.view(np.uint32))


def test_quantize_act_tiny_and_huge_groups_bit_exact(B):
    """Groups whose float32 scale is subnormal (BF16 values down to 2^-133, scale
    = amax / 448 below 2^-126) and groups near the BF16 maximum: the divides are
    IEEE round-to-nearest with subnormals on both sides, codes saturate at 448."""
    g = torch.Generator().manual_seed(9)
    x = torch.randn(6, 1024, generator=g)
    exps = torch.tensor([-133, -131, -128, -126, -120, 120, 124, 125], dtype=torch.float32)
    x = (x.view(6, 8, 128) * torch.exp2(exps)[None, :, None]).view(6, 1024)
    xb = x.to(torch.bfloat16)
    q = torch.empty(6, 1024, dtype=torch.uint8, device="cuda")
    s = torch.empty(6, 8, dtype=torch.float32, device="cuda")
    B.bfp8_quantize_act(xb.cuda(), q, s)
    torch.cuda.synchronize()
    q_r, s_r = OB.quantize_act(Hp.bits16(xb))
    assert np.any((s_r > 0) & (s_r < np.float32(2.0 ** -126)))      # subnormal scales occur
    assert np.array_equal(q.cpu().numpy(), q_r)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_r.view(np.uint32))


def test_quantize_weight_bit_exact(B):
    g = torch.Generator().manual_seed(4)
    w = torch.randn(3, 256, 384, generator=g) * 0.02
    w *= torch.exp2(torch.randint(-8, 9, (3, 2, 1, 3, 1), generator=g).float()).expand(3, 2, 128, 3, 128) \
        .reshape(3, 256, 384)
    w[1, 128:, 256:] = 0.0                          # an all-zero block
    wb = w.to(torch.bfloat16)
    q = torch.empty(3, 256, 384, dtype=torch.uint8, device="cuda")
    s = torch.empty(3, 2, 3, dtype=torch.float32, device="cuda")
    q_r, s_r = OB.quantize_weight(Hp.bits16(wb))
    for layout in (B.BFP8_LAYOUT_CANONICAL, B.BFP8_LAYOUT_TILED):
        q.zero_(); s.zero_()
        B.bfp8_quantize_weight(wb.cuda(), q, s, layout=layout)
        torch.cuda.synchronize()
        got = q.cpu().numpy()
        if layout == B.BFP8_LAYOUT_TILED:
            got = tiled_to_canonical(got, 3, 256, 384)
        assert np.array_equal(got, q_r), layout
        assert np.array_equal(s.cpu().numpy().view(np.uint32), s_r.view(np.uint32)), layout
    assert s_r[1, 1, 2] == 0.0


def tiled_to_canonical(codes: np.ndarray, G: int, N: int, K: int) -> np.ndarray:
    """Tile-contiguous codes [G][N/128][K/128][128][128] -> row-major [G][N][K]."""
    t = codes.reshape(G, N // 128, K // 128, 128, 128)
    return t.transpose(0, 1, 3, 2, 4).reshape(G, N, K)


class BSetup:
    """A workload's tokens and block-FP8 experts on the GPU, and the oracle's
    quantised view of the experts its routing touches."""

    def __init__(self, B, wl, scoring="softmax", renorm=True, layout=None):
        self.wl, self.B = wl, B
        self.layout = B.BFP8_LAYOUT_TILED if layout is None else layout
        E, H, I = wl.E, wl.H, wl.I
        self.x, self.logits = W.tokens(wl)
        self.idx_ref, self.w_ref = O.route_topk(self.logits.numpy(), wl.k, scoring, renorm)
        touched = set(np.nonzero(O.permute(self.idx_ref, E)[0])[0].tolist())
        self.w1q = torch.empty(E, 2 * I, H, dtype=torch.uint8, device="cuda")
        self.w1s = torch.empty(E, 2 * I // 128, H // 128, dtype=torch.float32, device="cuda")
        self.w2q = torch.empty(E, H, I, dtype=torch.uint8, device="cuda")
        self.w2s = torch.empty(E, H // 128, I // 128, dtype=torch.float32, device="cuda")
        self.w1q_ref = np.zeros((E, 2 * I, H), np.uint8)
        self.w1s_ref = np.zeros((E, 2 * I // 128, H // 128), np.float32)
        self.w2q_ref = np.zeros((E, H, I), np.uint8)
        self.w2s_ref = np.zeros((E, H // 128, I // 128), np.float32)
        self.touched = sorted(touched)
        for e in range(E):
            l1, l2 = W.expert_weights(wl, e, "cuda")
            B.bfp8_quantize_weight(l1[None].contiguous(), self.w1q[e:e + 1], self.w1s[e:e + 1], layout=self.layout)
            B.bfp8_quantize_weight(l2[None].contiguous(), self.w2q[e:e + 1], self.w2s[e:e + 1], layout=self.layout)
            if e in touched:
                q1, s1 = OB.quantize_weight(Hp.bits16(l1.cpu())[None])
                q2, s2 = OB.quantize_weight(Hp.bits16(l2.cpu())[None])
                self.w1q_ref[e], self.w1s_ref[e], self.w2q_ref[e], self.w2s_ref[e] = q1[0], s1[0], q2[0], s2[0]
        torch.cuda.synchronize()

    def check_weights_bit_exact(self, experts):
        H, I = self.wl.H, self.wl.I
        for e in experts:
            q1, q2 = self.w1q[e].cpu().numpy(), self.w2q[e].cpu().numpy()
            if self.layout == self.B.BFP8_LAYOUT_TILED:
                q1 = tiled_to_canonical(q1, 1, 2 * I, H)[0]
                q2 = tiled_to_canonical(q2, 1, H, I)[0]
            assert np.array_equal(q1, self.w1q_ref[e]), e
            assert np.array_equal(q2, self.w2q_ref[e]), e
            assert np.array_equal(self.w1s[e].cpu().numpy().view(np.uint32), self.w1s_ref[e].view(np.uint32)), e
            assert np.array_equal(self.w2s[e].cpu().numpy().view(np.uint32), self.w2s_ref[e].view(np.uint32)), e

    def run(self, route_mode=0):
        B, wl = self.B, self.wl
        T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
        P = T * k
        dev = "cuda"
        y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(B.moe_bfp8_workspace_size(T, H, I, E, k), dtype=torch.uint8, device=dev)
        out = dict(idx=torch.empty(T, k, dtype=torch.int32, device=dev),
                   w=torch.empty(T, k, dtype=torch.float32, device=dev),
                   counts=torch.empty(E, dtype=torch.int32, device=dev),
                   offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                   perm=torch.empty(max(P, 1), dtype=torch.int32, device=dev),
                   hq=torch.empty(max(P, 1), I, dtype=torch.uint8, device=dev),
                   hs=torch.empty(max(P, 1), I // 128, dtype=torch.float32, device=dev))
        B.moe_forward_bfp8(self.x.cuda(), self.logits.cuda(), self.w1q, self.w1s, self.w2q, self.w2s, k, y, ws,
                           topk_idx_out=out["idx"], topk_w_out=out["w"], counts_out=out["counts"],
                           offsets_out=out["offsets"], perm_out=out["perm"], hq_out=out["hq"],
                           hs_out=out["hs"], route_mode=route_mode, weight_layout=self.layout)
        torch.cuda.synchronize()
        assert B.moe_get_device_status(ws) == 0
        res = {n: t.cpu().numpy() for n, t in out.items()}
        res["y"] = Hp.bits16(y.cpu())
        return res


def check_bfp8_h(hq_g, hs_g, hq_r, hs_r, max_code_frac=1e-3, scale_rtol=1e-4):
    """Requantised h: float32 scales within ``scale_rtol``; dequantised values
    within one E4M3 step (at the coarser of the two values' binades, times the
    larger scale); codes that differ at all on at most 0.1 % of elements."""
    assert np.all(np.isfinite(hs_g))
    assert np.all(np.abs(hs_g.astype(np.float64) - hs_r) <= scale_rtol * np.abs(hs_r)), "h scales differ"
    vg = OB.dequant_rows(hq_g, hs_g)
    vr = OB.dequant_rows(hq_r, hs_r)
    smax = np.repeat(np.maximum(hs_g, hs_r).astype(np.float64), 128, axis=1)
    mag = np.maximum(np.abs(vg), np.abs(vr)) / np.where(smax > 0, smax, 1.0)
    step = np.where(mag < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(mag, 2.0 ** -6))) - 3))
    assert np.all(np.abs(vg - vr) <= step * smax * (1 + 1e-3)), "an h value differs by more than one E4M3 step"
    frac = np.count_nonzero(hq_g != hq_r) / max(hq_r.size, 1)
    assert frac <= max_code_frac, f"{frac:.2e} of h codes differ"
    return frac


SHAPES = {
    "monomoe_shape": W.Workload("monomoe_shape", T=8, H=2048, I=512, E=256, k=8, sigma=0.02, seed=1),
    "tiny": W.Workload("bfp8_tiny", T=64, H=256, I=128, E=8, k=2, sigma=0.02, seed=0),
    "one_token": W.Workload("bfp8_one", T=1, H=256, I=128, E=5, k=3, sigma=0.05, seed=21),
    "ragged": W.Workload("bfp8_ragged", T=100, H=384, I=256, E=37, k=4, sigma=0.03, seed=22),
    "wide_H": W.Workload("bfp8_wide", T=3, H=7168, I=256, E=9, k=2, sigma=0.01, seed=23),
    "k1": W.Workload("bfp8_k1", T=40, H=512, I=256, E=10, k=1, sigma=0.03, seed=24),
    # E > 256: routing, permute and cast as separate launches, then the separate GEMMs
    "wide_E": W.Workload("bfp8_wideE", T=5, H=256, I=128, E=300, k=4, sigma=0.05, seed=25),
    # E = 1, k = 1: every pair on one expert, three token tiles (the last ragged)
    "one_expert": W.Workload("bfp8_one_expert", T=40, H=256, I=128, E=1, k=1, sigma=0.05, seed=28),
    # more GEMM1 items than CTAs (several items per CTA), single launch / chain
    "many_items_single": W.Workload("bfp8_many1", T=64, H=256, I=2048, E=64, k=8, sigma=0.02, seed=26),
    "many_items_chain": W.Workload("bfp8_many2", T=100, H=256, I=2048, E=64, k=8, sigma=0.02, seed=27),
}


@pytest.mark.parametrize("name,layout", [(n, 1) for n in SHAPES] + [("monomoe_shape", 0), ("ragged", 0)])
def test_forward_bfp8(B, name, layout):
    """layout 1: tile-contiguous weight codes; 0: row-major."""
    wl = SHAPES[name]
    st = BSetup(B, wl, layout=layout)
    st.check_weights_bit_exact(st.touched[:4])
    g = st.run()
    ref = OB.forward(Hp.bits16(st.x), st.logits.numpy(), st.w1q_ref, st.w1s_ref, st.w2q_ref, st.w2s_ref, wl.k)
    assert np.array_equal(g["idx"], ref["topk_idx"])
    assert np.all(np.abs(g["w"] - ref["topk_w"]) <= 8 * np.spacing(np.abs(ref["topk_w"]).astype(np.float32)))
    assert np.array_equal(g["counts"], ref["counts"]) and np.array_equal(g["offsets"], ref["offsets"])
    P = wl.T * wl.k
    assert np.array_equal(g["perm"][:P], ref["perm"])
    perm = ref["perm"]
    check_bfp8_h(g["hq"][:P], g["hs"][:P], ref["hq"][perm], ref["hs"][perm])
    Hp.assert_bf16_close(g["y"], ref["y"], what=name)
    if wl.k == 1:
        assert np.all(g["w"] == 1.0)


@pytest.mark.parametrize("scoring,renorm,mode", [("sigmoid", False, 1 | 4), ("softmax", False, 4), ("raw", False, 2 | 4)])
def test_forward_bfp8_routing_modes(B, scoring, renorm, mode):
    wl = SHAPES["tiny"]
    st = BSetup(B, wl, scoring, renorm)
    g = st.run(route_mode=mode)
    ref = OB.forward(Hp.bits16(st.x), st.logits.numpy(), st.w1q_ref, st.w1s_ref, st.w2q_ref, st.w2s_ref, wl.k,
                     scoring=scoring, renormalize=renorm)
    assert np.array_equal(g["idx"], ref["topk_idx"])
    Hp.assert_bf16_close(g["y"], ref["y"], what=f"{scoring}/{renorm}")


def test_forward_bfp8_zero_input_and_empty_batch(B):
    wl = SHAPES["tiny"]
    st = BSetup(B, wl)
    st.x = torch.zeros_like(st.x)
    g = st.run()
    assert np.all(g["y"] == 0) and np.all(g["hq"] == 0) and np.all(g["hs"] == 0)
    # T = 0: a no-op that still clears the optional count outputs
    E = wl.E
    ws = torch.empty(B.moe_bfp8_workspace_size(0, wl.H, wl.I, E, wl.k), dtype=torch.uint8, device="cuda")
    counts = torch.full((E,), 7, dtype=torch.int32, device="cuda")
    x0 = torch.empty(0, wl.H, dtype=torch.bfloat16, device="cuda")
    l0 = torch.empty(0, E, dtype=torch.float32, device="cuda")
    y0 = torch.empty(0, wl.H, dtype=torch.bfloat16, device="cuda")
    B.moe_forward_bfp8(x0, l0, st.w1q, st.w1s, st.w2q, st.w2s, wl.k, y0, ws, counts_out=counts)
    torch.cuda.synchronize()
    assert int(counts.abs().sum()) == 0


def test_forward_bfp8_repeatable_and_graph_capturable(B):
    """Two eager calls and a CUDA-graph replay give identical bits."""
    wl = SHAPES["monomoe_shape"]
    st = BSetup(B, wl)
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    x, logits = st.x.cuda(), st.logits.cuda()
    ws = torch.empty(B.moe_bfp8_workspace_size(T, H, I, E, k), dtype=torch.uint8, device="cuda")
    ys = [torch.empty(T, H, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    for y in ys[:2]:
        B.moe_forward_bfp8(x, logits, st.w1q, st.w1s, st.w2q, st.w2s, k, y, ws)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            B.moe_forward_bfp8(x, logits, st.w1q, st.w1s, st.w2q, st.w2s, k, ys[2], ws, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(ys[0].view(torch.int16), ys[1].view(torch.int16))
    assert torch.equal(ys[0].view(torch.int16), ys[2].view(torch.int16))


def test_forward_bfp8_gemm_phase_reruns(B):
    """phases = GEMM1 (or GEMM2) re-runs one GEMM on the state a whole-layer call
    left: h comes back bit-identical and y is not touched."""
    wl = SHAPES["ragged"]
    st = BSetup(B, wl)
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    P = T * k
    x, logits = st.x.cuda(), st.logits.cuda()
    ws = torch.empty(B.moe_bfp8_workspace_size(T, H, I, E, k), dtype=torch.uint8, device="cuda")
    y = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    hq = torch.empty(P, I, dtype=torch.uint8, device="cuda")
    hs = torch.empty(P, I // 128, dtype=torch.float32, device="cuda")
    kw = dict(hq_out=hq, hs_out=hs)
    B.moe_forward_bfp8(x, logits, st.w1q, st.w1s, st.w2q, st.w2s, k, y, ws, **kw)
    torch.cuda.synchronize()
    hq0, hs0, y0 = hq.clone(), hs.clone(), y.clone()
    hq.zero_(); hs.zero_(); y.fill_(1.0)
    B.moe_forward_bfp8(x, logits, st.w1q, st.w1s, st.w2q, st.w2s, k, y, ws, phases=B.PHASE_GEMM1, **kw)
    B.moe_forward_bfp8(x, logits, st.w1q, st.w1s, st.w2q, st.w2s, k, y, ws, phases=B.PHASE_GEMM2, **kw)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == 0
    assert torch.equal(hq, hq0) and torch.equal(hs.view(torch.int32), hs0.view(torch.int32))
    assert bool((y == 1.0).all())
    assert not torch.equal(y.view(torch.int16), y0.view(torch.int16))


@pytest.mark.parametrize("name", ["monomoe_shape", "ragged"])
def test_forward_bfp8_injected_wait_times_out_then_recovers(B, monkeypatch, name):
    """MOE_MXQ_DEBUG_INJECT_WAIT=1: each CTA's MMA warp first waits on a barrier
    nothing completes; the wait gives up (~10 ms), records MOE_ERR_TIMEOUT at
    site 7, raises the abort flag, every other wait of the launch (stages,
    TMEM slots, arrival counters of the single launch) gives up, and the next
    call in the same process is correct.  monomoe_shape: front + single
    launch; ragged: the chain of separate launches."""
    import time
    wl = SHAPES[name]
    st = BSetup(B, wl)
    T, H, I, E, k = wl.T, wl.H, wl.I, wl.E, wl.k
    x, logits = st.x.cuda(), st.logits.cuda()
    ws = torch.empty(B.moe_bfp8_workspace_size(T, H, I, E, k), dtype=torch.uint8, device="cuda")
    y = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    B.moe_forward_bfp8(x, logits, st.w1q, st.w1s, st.w2q, st.w2s, k, y, ws)
    torch.cuda.synchronize()
    monkeypatch.setenv("MOE_MXQ_DEBUG_INJECT_WAIT", "1")
    t0 = time.perf_counter()
    B.moe_forward_bfp8(x, logits, st.w1q, st.w1s, st.w2q, st.w2s, k, y, ws)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    words = ws[:20].view(torch.int32).cpu().tolist()
    assert B.moe_get_device_status(ws) == B.MOE_ERR_TIMEOUT, words
    assert words[1] == 1 and words[2] == 7, words
    assert elapsed < 5.0, f"the failing call took {elapsed:.2f} s"
    monkeypatch.delenv("MOE_MXQ_DEBUG_INJECT_WAIT")
    g = st.run()
    ref = OB.forward(Hp.bits16(st.x), st.logits.numpy(), st.w1q_ref, st.w1s_ref, st.w2q_ref, st.w2s_ref, k)
    Hp.assert_bf16_close(g["y"], ref["y"], what=name)


def test_bfp8_layer_container_fewer_tokens_than_capacity(B):
    """layer.MoELayerBfp8 sized for 64 tokens, called with 37: the workspace is
    sliced to the call's size and the result matches the oracle on those tokens."""
    from moe_expert_layer_counting_gb300.layer import Bfp8Experts, MoELayerBfp8
    wl = W.WORKLOADS["tiny"]
    x, logits = W.tokens(wl)
    l1, l2 = W.all_expert_weights(wl, "cpu")
    layer = MoELayerBfp8(Bfp8Experts.from_bf16(l1.cuda(), l2.cuda()), wl.k, max_tokens=64)
    n = 37
    y = layer(x[:n].contiguous().cuda(), logits[:n].contiguous().cuda())
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    q1, s1 = OB.quantize_weight(Hp.bits16(l1))
    q2, s2 = OB.quantize_weight(Hp.bits16(l2))
    ref = OB.forward(Hp.bits16(x[:n]), logits[:n].numpy(), q1, s1, q2, s2, wl.k)
    Hp.assert_bf16_close(Hp.bits16(y.cpu()), ref["y"], what="MoELayerBfp8")
