"""GPU parity of the element-wise and integer kernels against the oracle:
activation and weight casts (bit-exact), routing (indices bit-exact, weights
within a few float32 ulp), counting-sort permute (bit-exact) and combine."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import formats as F
from oracle import moe as O
from tests import helpers as Hp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return Hp.lib()


def _special_rows(K):
    """Rows that hit the edges: zeros, -0, subnormal BF16, huge, ties, one-hot."""
    rows = [np.zeros(K, np.float32), -np.zeros(K, np.float32)]
    r = np.zeros(K, np.float32); r[3] = 1e-40; r[40] = -2e-39; rows.append(r)
    r = np.full(K, 3.0e38, np.float32); r[1::2] *= -1; rows.append(r)
    r = np.zeros(K, np.float32); r[::7] = 448.0; r[1::7] = 3 * 2.0 ** -10 * 1.0; rows.append(r)
    r = np.linspace(-3, 3, K).astype(np.float32); rows.append(r)
    r = np.zeros(K, np.float32); r[5] = -1.0; rows.append(r)
    return torch.from_numpy(np.stack(rows)).to(torch.bfloat16)


@pytest.mark.parametrize("wl_name", ["tiny", "small_decode", "large_decode"])
def test_quantize_act_bitexact(B, wl_name):
    wl = W.WORKLOADS[wl_name]
    x, _ = W.tokens(wl)
    x = torch.cat([x, _special_rows(wl.H)])
    xd = x.cuda()
    q = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    s = torch.empty(x.shape[0], x.shape[1] // 32, dtype=torch.uint8, device="cuda")
    B.mxq_quantize_act(xd, q, s)
    torch.cuda.synchronize()
    q_ref, s_ref = O.quantize_act(Hp.bits16(x))
    assert np.array_equal(Hp.to_np_u8(s), s_ref)
    assert np.array_equal(Hp.to_np_u8(q), q_ref)


def test_quantize_act_ragged_rows(B):
    x = torch.randn(37, 96).to(torch.bfloat16)     # K = 3 groups, 37 rows (tail of a block)
    q = torch.empty(37, 96, dtype=torch.uint8, device="cuda")
    s = torch.empty(37, 3, dtype=torch.uint8, device="cuda")
    B.mxq_quantize_act(x.cuda(), q, s)
    q_ref, s_ref = O.quantize_act(Hp.bits16(x))
    assert np.array_equal(Hp.to_np_u8(q), q_ref) and np.array_equal(Hp.to_np_u8(s), s_ref)


def test_quantize_weight_canonical_bitexact(B):
    g = torch.Generator().manual_seed(3)
    w = (torch.randn(3, 256, 384, generator=g) * 0.02)
    w[0, 0, :32] = 0.0
    w[0, 1, :32] = -0.0
    w[0, 2, :64] = torch.linspace(-6, 6, 64)
    w[1, 3, :] = 3.0e38
    w[2, 4, 7] = 1e-40
    w = w.to(torch.bfloat16)
    q = torch.empty(3, 256, 192, dtype=torch.uint8, device="cuda")
    s = torch.empty(3, 256, 12, dtype=torch.uint8, device="cuda")
    B.mxq_quantize_weight(w.cuda(), B.LAYOUT_CANONICAL, q, s)
    q_ref, s_ref = O.quantize_weight(Hp.bits16(w))
    assert np.array_equal(Hp.to_np_u8(s), s_ref)
    assert np.array_equal(Hp.to_np_u8(q), q_ref)


@pytest.mark.parametrize("layout", [1, 2])
def test_quantize_weight_mma_layout(B, layout):
    G, N, K = 2, 256, 512
    w = (torch.randn(G, N, K, generator=torch.Generator().manual_seed(layout)) * 0.05).to(torch.bfloat16)
    q = torch.empty(G, N, K // 2, dtype=torch.uint8, device="cuda")
    s = torch.empty(G * N * K // 32, dtype=torch.uint8, device="cuda")
    B.mxq_quantize_weight(w.cuda(), layout, q, s)
    q_ref, s_ref = O.quantize_weight(Hp.bits16(w))
    qm, sm = Hp.canonical_to_mma(q_ref, s_ref, interleave=(layout == 1))
    assert np.array_equal(Hp.to_np_u8(q), qm)
    assert np.array_equal(Hp.to_np_u8(s), sm)
    q2, s2 = Hp.mma_to_canonical(Hp.to_np_u8(q), Hp.to_np_u8(s), G, N, K, layout == 1)
    assert np.array_equal(q2, q_ref) and np.array_equal(s2, s_ref)


def _route_cases():
    out = []
    for name in W.WORKLOADS:
        wl = W.WORKLOADS[name]
        _, logits = W.tokens(wl)
        out.append((name, logits[:512], wl.k))
    g = np.random.default_rng(1)
    pool = np.array([-1.0, -0.0, 0.0, 0.5, 0.5, 2.0], np.float32)
    out.append(("ties", torch.from_numpy(pool[g.integers(0, 6, (300, 64))]), 6))
    out.append(("wide_E", torch.randn(50, 1024, generator=torch.Generator().manual_seed(2)), 32))
    out.append(("k1", torch.randn(40, 10, generator=torch.Generator().manual_seed(3)), 1))
    # E just above one and eight warp widths (register key arrays of 8 and 32 per lane)
    out.append(("E33", torch.randn(70, 33, generator=torch.Generator().manual_seed(4)), 32))
    out.append(("E257", torch.randn(70, 257, generator=torch.Generator().manual_seed(5)), 8))
    ties = torch.from_numpy(pool[g.integers(0, 6, (64, 300))])
    out.append(("ties_E300", ties, 32))
    return out


@pytest.mark.parametrize("case", _route_cases(), ids=lambda c: c[0])
def test_route_topk(B, case):
    _, logits, k = case
    T, E = logits.shape
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    B.moe_route_topk(logits.contiguous().cuda(), k, idx, w)
    idx_ref, w_ref = O.route_topk(logits.numpy(), k)
    assert np.array_equal(idx.cpu().numpy(), idx_ref)
    wg = w.cpu().numpy().astype(np.float64)
    # expf (<= 2 ulp), one rounded subtraction, the sum and the division:
    # bounded well inside 8 float32 ulp of the reference weight
    ulp = np.spacing(np.abs(w_ref).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(wg - w_ref) <= 8 * ulp + 1e-30)
    if k == 1:
        assert np.all(wg == 1.0)


def _permute_cases():
    cases = []
    for name in W.WORKLOADS:
        wl = W.WORKLOADS[name]
        _, logits = W.tokens(wl)
        idx, _ = O.route_topk(logits.numpy(), wl.k)
        cases.append((name, idx, wl.E))
    rng = np.random.default_rng(5)
    idx = np.stack([rng.choice(1024, 8, replace=False) for _ in range(3000)]).astype(np.int32)
    cases.append(("E1024", idx, 1024))
    idx = np.stack([rng.choice(16, 4, replace=False) for _ in range(700)]).astype(np.int32)
    idx[rng.random(idx.shape) < 0.2] = -1                      # dropped pairs
    cases.append(("dropped", idx, 16))
    cases.append(("one_pair", np.array([[3]], np.int32), 5))
    cases.append(("all_one_expert", np.zeros((5000, 1), np.int32), 7))
    return cases


@pytest.mark.parametrize("case", _permute_cases(), ids=lambda c: c[0])
def test_permute_bitexact(B, case):
    _, idx, E = case
    T, k = idx.shape
    P = T * k
    ws = torch.empty(B.moe_permute_workspace_size(T, E, k), dtype=torch.uint8, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.full((P,), -7, dtype=torch.int32, device="cuda")
    inv = torch.empty(P, dtype=torch.int32, device="cuda")
    B.moe_permute(torch.from_numpy(idx).cuda(), E, counts, offsets, perm, inv, ws)
    c_ref, o_ref, p_ref, i_ref = O.permute(idx, E)
    assert np.array_equal(counts.cpu().numpy(), c_ref)
    assert np.array_equal(offsets.cpu().numpy(), o_ref)
    n = int(o_ref[-1])
    assert np.array_equal(perm.cpu().numpy()[:n], p_ref)
    assert np.all(perm.cpu().numpy()[n:] == -7)              # entries past offsets[E] untouched
    assert np.array_equal(inv.cpu().numpy(), i_ref)
    assert B.moe_get_device_status(ws) == 0


def test_permute_reports_out_of_range_index(B):
    idx = torch.tensor([[0, 1], [2, 9]], dtype=torch.int32, device="cuda")     # 9 >= E
    E = 4
    ws = torch.empty(B.moe_permute_workspace_size(2, E, 2), dtype=torch.uint8, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(4, dtype=torch.int32, device="cuda")
    inv = torch.empty(4, dtype=torch.int32, device="cuda")
    B.moe_permute(idx, E, counts, offsets, perm, inv, ws)
    assert B.moe_get_device_status(ws) == B.MOE_ERR_DEVICE_INDEX
    assert counts.cpu().tolist() == [1, 1, 1, 0] and inv.cpu().tolist()[3] == -1
    # the next call resets the status word
    B.moe_permute(idx.clamp(max=3), E, counts, offsets, perm, inv, ws)
    assert B.moe_get_device_status(ws) == 0


def test_permute_empty(B):
    E = 8
    ws = torch.empty(max(B.moe_permute_workspace_size(0, E, 2), 256), dtype=torch.uint8, device="cuda")
    counts = torch.full((E,), 5, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), 5, dtype=torch.int32, device="cuda")
    dummy = torch.empty(1, dtype=torch.int32, device="cuda")
    B.moe_permute(torch.empty(0, 2, dtype=torch.int32, device="cuda"), E, counts, offsets, dummy, dummy, ws)
    assert counts.cpu().tolist() == [0] * E and offsets.cpu().tolist() == [0] * (E + 1)


@pytest.mark.parametrize("T,k,H", [(64, 2, 256), (8, 8, 2048), (129, 3, 128)])
def test_combine(B, T, k, H):
    g = torch.Generator().manual_seed(T + k)
    yp = (torch.randn(k, T, H, generator=g) * 0.1).to(torch.bfloat16)
    idx = torch.randint(0, 16, (T, k), generator=g, dtype=torch.int32)
    idx[torch.rand(T, k, generator=g) < 0.15] = -1
    y = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    B.moe_combine(yp.cuda(), idx.cuda(), y)
    y_ref = O.combine(Hp.bits16(yp), idx.numpy())
    got = Hp.bits16(y)
    # FP32 slot sum vs float64: the BF16 results agree except at rare rounding ties
    gv, rv = F.bf16_bits_to_f64(got), F.bf16_bits_to_f64(y_ref)
    ulp = np.abs(rv) * 2.0 ** -7 + 1e-38
    assert np.all(np.abs(gv - rv) <= ulp)
    assert np.mean(got != y_ref) <= 1e-3


# ---------------------------------------------------------------- routing variants
_MODES = {"softmax_full": ("softmax", False), "sigmoid": ("sigmoid", True),
          "sigmoid_raw_scores": ("sigmoid", False), "raw": ("raw", False)}


def _mode_code(B, scoring, renorm):
    code = {"softmax": B.ROUTE_SOFTMAX, "sigmoid": B.ROUTE_SIGMOID, "raw": B.ROUTE_RAW}[scoring]
    return code | (0 if renorm else B.ROUTE_NO_RENORM)


@pytest.mark.parametrize("mode", list(_MODES))
@pytest.mark.parametrize("case", _route_cases(), ids=lambda c: c[0])
def test_route_topk_modes(B, case, mode):
    """Selection bit-exact in every mode.  Weights: raw bit-exact; sigmoid
    without renormalisation: expf (<= 2 ulp) scaled by e/(1+e) <= 1, one add
    and one divide: <= 4 ulp; sigmoid renormalised: plus a k-term sum and a
    divide: <= 8 + k ulp; softmax over all E: expf of a rounded difference
    (<= 2 ulp + |d| * 2^-24 with |d| < 32 here), an E-term sum
    (<= (E/32 + 5) * 2^-24 relative), a divide: <= 40 + E/32 ulp."""
    _, logits, k = case
    scoring, renorm = _MODES[mode]
    T, E = logits.shape
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    B.moe_route_topk(logits.contiguous().cuda(), k, idx, w, mode=_mode_code(B, scoring, renorm))
    idx_ref, w_ref = O.route_topk(logits.numpy(), k, scoring, renorm)
    assert np.array_equal(idx.cpu().numpy(), idx_ref)
    wg = w.cpu().numpy()
    if scoring == "raw":
        assert np.array_equal(wg.view(np.uint32), w_ref.view(np.uint32))
        return
    bound = {"sigmoid": (8 + k) if renorm else 4, "softmax": 40 + E / 32}[scoring]
    ulp = np.spacing(np.abs(w_ref).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(wg.astype(np.float64) - w_ref) <= bound * ulp + 1e-30)
