"""moe_forward across shapes that take each dispatch path, compared in full
with the oracle.

moe_forward picks one of three front ends from the problem size: the fused
small-problem kernel (T <= 64, E <= 256, T*k*H <= 4M), routing + permute + a
pool-order cast (P*H <= 16M), or routing + permute + a token-order cast that
writes each token's codes to its k pool rows (larger), and the token tile from the mean pairs per routed expert; 224-token
tiles run on CTA pairs where the weight tiles pair up.  The
shapes below are small enough for the float64 oracle, with ragged counts,
E not a multiple of 32, a single token, k = 1, and a few thousand pairs."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe as O
from tests import helpers as Hp
from tests.test_gpu_expert import Setup, _forward

pytestmark = pytest.mark.gpu

# name: (T, H, I, E, k) -- expected path and tile in the comment
SHAPES = {
    "one_token": (1, 256, 128, 5, 3),            # front kernel, 16-token tiles
    "odd_E": (37, 384, 128, 77, 5),             # front kernel, E not a multiple of 32
    "E256_k8": (64, 256, 128, 256, 8),          # front kernel at its largest T and E
    "k1": (40, 512, 256, 10, 1),                # front kernel, k = 1 (weight 1)
    "pool_cast": (100, 256, 128, 24, 4),        # T > 64: routing + permute + pool cast
    "wide_H_front": (3, 7168, 128, 9, 2),       # front kernel, 224 column groups
    "large_path": (2048, 1024, 128, 64, 8),     # P*H > 16M: token-order cast, 224-token tiles
    "token_cast_odd_H": (2000, 1152, 128, 40, 8),   # token-order cast, H/8 = 144: a half-warp last step; H/128 odd: one-CTA 224 tiles
    "one_expert": (40, 256, 128, 1, 1),         # front kernel, E = 1, k = 1: three token tiles of one expert
    # 224-token tiles on CTA pairs (weight tiles pair up: 2I/128 and H/128 even)
    "pair_ragged": (700, 512, 256, 6, 2),       # ~233 pairs per expert: one or two tiles, ragged last tile
    "pair_two_sf_groups": (600, 256, 256, 8, 2),  # ~150 pairs: MMA N = 160, token scales in two 128-row groups
    "pair_fallback": (300, 384, 128, 4, 2),     # H/128 = 3 odd: the one-CTA 224-token kernel instead
}


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return Hp.lib()


@pytest.mark.parametrize("name,schedule", [(n, 0) for n in SHAPES] +
                         [(n, 2) for n in ("large_path", "pair_ragged", "pair_two_sf_groups", "pair_fallback")])
def test_forward_shape(B, name, schedule):
    """schedule 2: the expert-wave single launch where the shape runs on CTA
    pairs (the one-CTA fallback ignores it)."""
    T, H, I, E, k = SHAPES[name]
    wl = W.Workload(name, T=T, H=H, I=I, E=E, k=k, sigma=0.02, seed=11 + len(name))
    st = Setup(B, wl, weight_device="cuda")
    y_g, _ = _forward(B, st, schedule=schedule)
    ref = O.forward(Hp.bits16(st.x), st.logits.numpy(), st.w1q_ref, st.w1s_ref, st.w2q_ref, st.w2s_ref, k)
    Hp.assert_bf16_close(y_g, ref["y"], what=name)
    if k == 1:
        assert np.all(st.w_ref == 1.0)


@pytest.mark.parametrize("name,scoring,renorm", [("tiny", "sigmoid", True), ("small_decode", "sigmoid", False),
                                                 ("small_decode", "softmax", False), ("tiny", "raw", False)])
def test_forward_routing_modes(B, name, scoring, renorm):
    """The whole layer with each routing mode (small-problem kernel), in full
    against the oracle with the same mode."""
    wl = W.WORKLOADS[name]
    st = Setup(B, wl)
    st.idx_ref, st.w_ref = O.route_topk(st.logits.numpy(), wl.k, scoring, renorm)
    code = {"softmax": B.ROUTE_SOFTMAX, "sigmoid": B.ROUTE_SIGMOID, "raw": B.ROUTE_RAW}[scoring]
    mode = code | (0 if renorm else B.ROUTE_NO_RENORM)
    y = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device="cuda")
    ws = torch.empty(B.moe_workspace_size(wl.T, wl.H, wl.I, wl.E, wl.k), dtype=torch.uint8, device="cuda")
    B.moe_forward(st.x.cuda(), st.logits.cuda(), st.qe.w1q, st.qe.w1s, st.qe.w2q, st.qe.w2s, wl.k, y, ws,
                  topk_idx_out=idx, route_mode=mode)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == 0
    assert np.array_equal(idx.cpu().numpy(), st.idx_ref)
    ref = O.forward(Hp.bits16(st.x), st.logits.numpy(), st.w1q_ref, st.w1s_ref, st.w2q_ref, st.w2s_ref, wl.k,
                    scoring=scoring, renormalize=renorm)
    Hp.assert_bf16_close(Hp.bits16(y), ref["y"], what=f"{name} {scoring} renorm={renorm}")


@pytest.mark.parametrize("name", ["tiny", "small_decode"])
def test_dropped_pairs_end_to_end(B, name):
    """Pairs marked dropped (index < 0, as the MegaMoE dispatch skips them)
    through the separate entry points: permute (not counted, inv_perm -1),
    the expert GEMMs (never see them) and the combine (skips them); y in full
    against the oracle on the same indices."""
    wl = W.WORKLOADS[name]
    st = Setup(B, wl)
    rng = np.random.default_rng(wl.seed + 99)
    idx = st.idx_ref.copy()
    idx[rng.random(idx.shape) < 0.25] = -1
    w = st.w_ref
    dev = "cuda"
    T, k, E, H, I = wl.T, wl.k, wl.E, wl.H, wl.I
    idx_d, w_d = torch.from_numpy(idx).to(dev), torch.from_numpy(w).to(dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.full((T * k,), -7, dtype=torch.int32, device=dev)
    inv = torch.empty(T * k, dtype=torch.int32, device=dev)
    pws = torch.empty(B.moe_permute_workspace_size(T, E, k), dtype=torch.uint8, device=dev)
    B.moe_permute(idx_d, E, counts, offsets, perm, inv, pws)
    c_ref, o_ref, p_ref, i_ref = O.permute(idx, E)
    torch.cuda.synchronize()
    assert np.array_equal(counts.cpu().numpy(), c_ref) and np.array_equal(offsets.cpu().numpy(), o_ref)
    n = int(o_ref[-1])
    assert np.array_equal(perm.cpu().numpy()[:n], p_ref[:n]) and np.array_equal(inv.cpu().numpy(), i_ref)
    xq, xs = torch.from_numpy(st.xq_ref).to(dev), torch.from_numpy(st.xs_ref).to(dev)
    y_pairs = torch.zeros(k, T, H, dtype=torch.bfloat16, device=dev)
    ews = torch.empty(B.moe_expert_workspace_size(T, H, I, E, k), dtype=torch.uint8, device=dev)
    B.moe_expert_forward(xq, xs, st.qe.w1q, st.qe.w1s, st.qe.w2q, st.qe.w2s, idx_d, w_d, counts, offsets, perm,
                         y_pairs, ews)
    y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    B.moe_combine(y_pairs, idx_d, y)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ews) == 0
    yp_ref = O.expert_forward(st.xq_ref, st.xs_ref, st.w1q_ref, st.w1s_ref, st.w2q_ref, st.w2s_ref, idx, w, E)
    Hp.assert_bf16_close(Hp.bits16(y), O.combine(yp_ref, idx), what=f"{name} with dropped pairs")


@pytest.mark.parametrize("tile_n", [16, 32, 64, 224])
def test_forward_tiny_tile_sizes(B, tile_n):
    """The small-problem path with every launch structure: 16-token tiles run
    GEMM1 + GEMM2 + combine in one launch, larger tiles as separate launches."""
    wl = W.WORKLOADS["tiny"]
    st = Setup(B, wl)
    y_g, _ = _forward(B, st, tile_n=tile_n)
    ref = O.forward(Hp.bits16(st.x), st.logits.numpy(), st.w1q_ref, st.w1s_ref, st.w2q_ref, st.w2s_ref, wl.k)
    Hp.assert_bf16_close(y_g, ref["y"], what=f"tiny tile_n={tile_n}")
