"""GPU parity of the grouped expert GEMMs (moe_expert_forward) and of the
fused layer (moe_forward) against the oracle.

Small workloads (Tiny, small-expert decode) are compared in full; the large
ones at full size on a seeded sample of tokens (moe_forward's output rows
against the oracle's layer on those tokens), on every pair of a sample of
experts (hottest, coldest, random), and on properties that hold at any size
(routing, counts, offsets and perm bit-exact; y equal to the oracle's combine
of the GPU's own per-pair rows)."""
import numpy as np
import pytest
import torch

import workloads as W
from moe_expert_layer_counting_gb300.layer import QuantizedExperts
from oracle import formats as F
from oracle import moe as O
from tests import helpers as Hp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return Hp.lib()


# ---------------------------------------------------------------- setup

class Setup:
    """One workload on the GPU plus the oracle's view of the experts it needs."""

    def __init__(self, B, wl, oracle_experts="touched", weight_device=None, pool=None):
        self.wl = wl
        self.B = B
        wdev = weight_device or ("cpu" if wl.E * 3 * wl.H * wl.I <= 2 ** 22 else "cuda")
        self.x, self.logits = W.tokens(wl)
        self.idx_ref, self.w_ref = O.route_topk(self.logits.numpy(), wl.k)
        self.counts_ref, self.offsets_ref, self.perm_ref, self.inv_ref = O.permute(self.idx_ref, wl.E)
        self.qe = QuantizedExperts(wl.E, wl.H, wl.I)
        touched = np.nonzero(self.counts_ref)[0]
        if oracle_experts == "touched":
            want = set(touched.tolist())
        else:
            want = set(oracle_experts)
        E, I, H = wl.E, wl.I, wl.H
        self.w1q_ref = np.zeros((E, 2 * I, H // 2), np.uint8)
        self.w1s_ref = np.zeros((E, 2 * I, H // 32), np.uint8)
        self.w2q_ref = np.zeros((E, H, I // 2), np.uint8)
        self.w2s_ref = np.zeros((E, H, I // 32), np.uint8)
        self.oracle_experts = sorted(want)
        pending = {}
        for e in range(E):
            l1, l2 = W.expert_weights(wl, e, wdev)
            self.qe.set_expert(e, l1.cuda(), l2.cuda())
            if e in want:
                b1, b2 = Hp.bits16(l1)[None], Hp.bits16(l2)[None]
                if pool is None:
                    self._store(e, O.quantize_weight(b1), O.quantize_weight(b2))
                else:
                    pending[e] = (pool.submit(O.quantize_weight, b1), pool.submit(O.quantize_weight, b2))
        for e, (f1, f2) in pending.items():
            self._store(e, f1.result(), f2.result())
        torch.cuda.synchronize()
        self.xq_ref, self.xs_ref = O.quantize_act(Hp.bits16(self.x))

    def _store(self, e, l1_q, l2_q):
        self.w1q_ref[e], self.w1s_ref[e] = l1_q[0][0], l1_q[1][0]
        self.w2q_ref[e], self.w2s_ref[e] = l2_q[0][0], l2_q[1][0]

    def oracle_weights(self):
        """Expert id -> the oracle's (w1q, w1s, w2q, w2s) for the oracle's experts."""
        return {e: (self.w1q_ref[e], self.w1s_ref[e], self.w2q_ref[e], self.w2s_ref[e])
                for e in self.oracle_experts}

    def check_weights_bitexact(self):
        """GPU-quantised weights (MMA layouts) against the oracle, for the oracle's experts."""
        wl = self.wl
        E, I, H = wl.E, wl.I, wl.H
        for e in self.oracle_experts:
            s1 = 2 * I * H // 32
            s2 = H * I // 32
            q1, c1 = Hp.mma_to_canonical(Hp.to_np_u8(self.qe.w1q[e])[None],
                                         Hp.to_np_u8(self.qe.w1s[e * s1:(e + 1) * s1]), 1, 2 * I, H, True)
            q2, c2 = Hp.mma_to_canonical(Hp.to_np_u8(self.qe.w2q[e])[None],
                                         Hp.to_np_u8(self.qe.w2s[e * s2:(e + 1) * s2]), 1, H, I, False)
            assert np.array_equal(q1[0], self.w1q_ref[e]) and np.array_equal(c1[0], self.w1s_ref[e]), e
            assert np.array_equal(q2[0], self.w2q_ref[e]) and np.array_equal(c2[0], self.w2s_ref[e]), e

    def oracle_pairs(self):
        """Oracle y_pairs / hq / hs for the pairs of the oracle's experts."""
        return O.expert_forward(self.xq_ref, self.xs_ref, self.w1q_ref, self.w1s_ref, self.w2q_ref,
                                self.w2s_ref, self.idx_ref, self.w_ref, self.wl.E,
                                experts=self.oracle_experts, return_h=True)

    def run_expert_forward(self, tile_n=0, w_dev=None):
        """moe_expert_forward on the oracle's routing/permute and activations
        (top-k weights: the oracle's, or ``w_dev`` when given)."""
        B, wl = self.B, self.wl
        P = wl.T * wl.k
        dev = "cuda"
        xq = torch.from_numpy(self.xq_ref).to(dev)
        xs = torch.from_numpy(self.xs_ref).to(dev)
        idx = torch.from_numpy(self.idx_ref).to(dev)
        w = torch.from_numpy(self.w_ref).to(dev) if w_dev is None else w_dev
        counts = torch.from_numpy(self.counts_ref).to(dev)
        offsets = torch.from_numpy(self.offsets_ref).to(dev)
        perm = torch.from_numpy(self.perm_ref).to(dev)
        y_pairs = torch.zeros(wl.k, wl.T, wl.H, dtype=torch.bfloat16, device=dev)
        hq = torch.zeros(P, wl.I, dtype=torch.uint8, device=dev)
        hs = torch.zeros(P, wl.I // 32, dtype=torch.uint8, device=dev)
        ws = torch.empty(B.moe_expert_workspace_size(wl.T, wl.H, wl.I, wl.E, wl.k), dtype=torch.uint8, device=dev)
        B.moe_expert_forward(xq, xs, self.qe.w1q, self.qe.w1s, self.qe.w2q, self.qe.w2s, idx, w, counts, offsets,
                             perm, y_pairs, ws, hq=hq, hs=hs, tile_n=tile_n)
        torch.cuda.synchronize()
        assert B.moe_get_device_status(ws) == 0
        return Hp.bits16(y_pairs), Hp.to_np_u8(hq), Hp.to_np_u8(hs)


def _compare_pairs(st, y_pairs_g, hq_g, hs_g, y_ref, hq_ref, hs_ref, what):
    """Compare, for the pairs of the oracle's experts, the requantised h (pool
    order on the GPU, pair order in the oracle) and the per-pair BF16 rows."""
    wl = st.wl
    sel = np.isin(st.idx_ref.reshape(-1), st.oracle_experts)
    pairs = np.nonzero(sel)[0]
    pos = st.inv_ref[pairs]
    Hp.check_requantised_h(hq_g[pos], hs_g[pos], hq_ref[pairs], hs_ref[pairs])
    t, j = pairs // wl.k, pairs % wl.k
    Hp.assert_bf16_close(y_pairs_g[j, t], y_ref[j, t], what=what)


@pytest.mark.parametrize("tile_n", [16, 32, 64, 128, 224])
def test_expert_forward_tiny_every_tile(B, tile_n):
    st = Setup(B, W.WORKLOADS["tiny"])
    st.check_weights_bitexact()
    y_ref, hq_ref, hs_ref = st.oracle_pairs()
    y_g, hq_g, hs_g = st.run_expert_forward(tile_n)
    _compare_pairs(st, y_g, hq_g, hs_g, y_ref, hq_ref, hs_ref, f"tiny tile_n={tile_n}")


def test_expert_forward_small_decode(B):
    st = Setup(B, W.WORKLOADS["small_decode"])
    st.check_weights_bitexact()
    y_ref, hq_ref, hs_ref = st.oracle_pairs()
    for tile_n in (0, 32):
        y_g, hq_g, hs_g = st.run_expert_forward(tile_n)
        _compare_pairs(st, y_g, hq_g, hs_g, y_ref, hq_ref, hs_ref, f"small_decode tile_n={tile_n}")


def _forward(B, st, tile_n=0, schedule=0):
    wl = st.wl
    dev = "cuda"
    y = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device=dev)
    w = torch.empty(wl.T, wl.k, dtype=torch.float32, device=dev)
    counts = torch.empty(wl.E, dtype=torch.int32, device=dev)
    offsets = torch.empty(wl.E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(wl.T * wl.k, dtype=torch.int32, device=dev)
    ws = torch.empty(B.moe_workspace_size(wl.T, wl.H, wl.I, wl.E, wl.k), dtype=torch.uint8, device=dev)
    B.moe_forward(st.x.cuda(), st.logits.cuda(), st.qe.w1q, st.qe.w1s, st.qe.w2q, st.qe.w2s, wl.k, y, ws,
                  topk_idx_out=idx, topk_w_out=w, counts_out=counts, offsets_out=offsets, perm_out=perm,
                  tile_n=tile_n, schedule=schedule)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == 0
    assert np.array_equal(idx.cpu().numpy(), st.idx_ref)
    assert np.array_equal(counts.cpu().numpy(), st.counts_ref)
    assert np.array_equal(offsets.cpu().numpy(), st.offsets_ref)
    assert np.array_equal(perm.cpu().numpy(), st.perm_ref)
    wg = w.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(wg - st.w_ref) <= 8 * np.spacing(st.w_ref.astype(np.float32)))
    return Hp.bits16(y), w


@pytest.mark.parametrize("wl_name", ["tiny", "small_decode"])
def test_forward_full(B, wl_name):
    st = Setup(B, W.WORKLOADS[wl_name])
    y_g, _ = _forward(B, st)
    ref = O.forward(Hp.bits16(st.x), st.logits.numpy(), st.w1q_ref, st.w1s_ref, st.w2q_ref, st.w2s_ref,
                    st.wl.k)
    Hp.assert_bf16_close(y_g, ref["y"], what=wl_name)


def _sample_experts(counts, n_random=2, seed=0):
    nz = np.nonzero(counts)[0]
    order = nz[np.argsort(counts[nz], kind="stable")]
    pick = list(order[-2:]) + list(order[:2])
    rng = np.random.default_rng(seed)
    pick += list(rng.choice(nz, size=min(n_random, nz.size), replace=False))
    return sorted(set(int(e) for e in pick))


@pytest.fixture(scope="module")
def pool():
    with Hp.oracle_pool() as p:
        yield p


@pytest.mark.parametrize("wl_name,schedule", [("large_decode", 0), ("prefill", 0), ("skewed_prefill", 0),
                                              ("skewed_prefill", 2)])
def test_large_workloads_sampled(B, pool, wl_name, schedule):
    """The large workloads through moe_forward at full size.

    * routing, counts, offsets and perm: bit-exact on every token (in _forward);
    * y of a seeded sample of tokens (the first and last tokens of the two
      hottest and the two coldest non-empty experts, the last tokens of
      expert 0, random ones) against the oracle's layer run on those tokens
      with its own cast, routing and weights (schedule 2: the prefill
      workloads' GEMMs and combine as one expert-wave launch);
    * per-pair rows and h of a sample of experts (moe_expert_forward);
    * y of every token against the oracle's combine of the GPU's own
      per-pair rows (computed with the layer's routing weights)."""
    wl = W.WORKLOADS[wl_name]
    x, logits = W.tokens(wl)
    idx_ref, _ = O.route_topk(logits.numpy(), wl.k)
    counts_ref = O.permute(idx_ref, wl.E)[0]
    experts = _sample_experts(counts_ref, seed=wl.seed)
    toks = Hp.sample_tokens(idx_ref, counts_ref, n_random=4, seed=wl.seed)
    need = sorted(set(experts) | set(int(e) for e in idx_ref[toks].reshape(-1)))
    st = Setup(B, wl, oracle_experts=need, weight_device="cuda", pool=pool)
    st.check_weights_bitexact()
    y_fwd, w_dev = _forward(B, st, schedule=schedule)
    # sampled tokens: moe_forward's rows against the oracle's layer
    ref = Hp.oracle_forward_tokens(pool, Hp.bits16(x)[toks], logits.numpy()[toks], st.oracle_weights(), wl.k)
    assert np.array_equal(ref["topk_idx"], st.idx_ref[toks])
    Hp.assert_bf16_close(y_fwd[toks], ref["y"], what=f"{wl_name} tokens {toks.tolist()}")
    # per-pair rows of the sampled experts against the oracle
    st.oracle_experts = experts
    y_ref, hq_ref, hs_ref = st.oracle_pairs()
    y_g, hq_g, hs_g = st.run_expert_forward()
    _compare_pairs(st, y_g, hq_g, hs_g, y_ref, hq_ref, hs_ref, f"{wl_name} sampled experts {experts}")
    # every token: the fused output is the combine of the per-pair rows computed
    # with the same (GPU) routing weights; the oracle sums in float64, the GPU
    # in FP32 (the BF16 results agree except at rare rounding ties)
    y_same, _, _ = st.run_expert_forward(w_dev=w_dev)
    want = O.combine(y_same, st.idx_ref)
    gv, rv = F.bf16_bits_to_f64(y_fwd), F.bf16_bits_to_f64(want)
    assert np.all(np.abs(gv - rv) <= np.abs(rv) * 2.0 ** -7 + 1e-38)
    assert np.mean(y_fwd != want) <= 1e-3


@pytest.mark.parametrize("wl_name,tile_n", [("tiny", 16), ("tiny", 128), ("tiny", 224), ("small_decode", 0)])
def test_gemm2_on_oracle_h(B, wl_name, tile_n):
    """GEMM2 alone, fed with the oracle's own requantised h (pool order): the
    only difference left is FP32 accumulation before the BF16 cast, so the
    per-pair rows agree to one BF16 ulp, and almost all bit for bit."""
    st = Setup(B, W.WORKLOADS[wl_name])
    wl = st.wl
    y_ref, hq_ref, hs_ref = st.oracle_pairs()
    dev = "cuda"
    perm = st.perm_ref
    hq = torch.from_numpy(np.ascontiguousarray(hq_ref[perm])).to(dev)
    hs = torch.from_numpy(np.ascontiguousarray(hs_ref[perm])).to(dev)
    y_pairs = torch.zeros(wl.k, wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(B.moe_expert_workspace_size(wl.T, wl.H, wl.I, wl.E, wl.k), dtype=torch.uint8, device=dev)
    t = lambda a: torch.from_numpy(a).to(dev)  # noqa: E731
    B.moe_expert_forward(t(st.xq_ref), t(st.xs_ref), st.qe.w1q, st.qe.w1s, st.qe.w2q, st.qe.w2s, t(st.idx_ref),
                         t(st.w_ref), t(st.counts_ref), t(st.offsets_ref), t(perm), y_pairs, ws, hq=hq, hs=hs,
                         tile_n=tile_n, phases=B.PHASE_H_SCALES | B.PHASE_GEMM2)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == 0
    pairs = np.nonzero(st.idx_ref.reshape(-1) >= 0)[0]
    tt, jj = pairs // wl.k, pairs % wl.k
    g = F.bf16_bits_to_f64(Hp.bits16(y_pairs)[jj, tt])
    r = F.bf16_bits_to_f64(y_ref[jj, tt])
    assert np.all(np.abs(g - r) <= np.abs(r) * 2.0 ** -7 + 1e-30)
    assert np.mean(g != r) <= 1e-2
