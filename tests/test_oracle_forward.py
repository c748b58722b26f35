"""Pins for the oracle's whole-layer arithmetic (CPU only)."""
import math

import numpy as np
import torch

import workloads as W
from oracle import formats as F
from oracle import moe as O


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _small_layer(T, H, I, E, k, seed, sigma=0.05):
    g = torch.Generator().manual_seed(seed)
    x = _bits(torch.randn(T, H, generator=g))
    logits = torch.randn(T, E, generator=g).numpy()
    l1 = _bits(torch.randn(E, 2 * I, H, generator=g) * sigma)
    l2 = _bits(torch.randn(E, H, I, generator=g) * sigma)
    w1q, w1s = O.quantize_weight(l1)
    w2q, w2s = O.quantize_weight(l2)
    return x, logits, w1q, w1s, w2q, w2s


def test_single_expert_equals_dense_swiglu_mlp():
    """E = 1, k = 1 (weight 1): the layer is a dense SwiGLU MLP on quantised operands."""
    T, H, I = 24, 64, 96
    x, logits, w1q, w1s, w2q, w2s = _small_layer(T, H, I, 1, 1, seed=1)
    out = O.forward(x, logits, w1q, w1s, w2q, w2s, k=1)
    assert np.all(out["topk_w"] == 1.0) and np.all(out["topk_idx"] == 0)

    # dense MLP written without routing, permute or the oracle's GEMM helpers
    xf = F.bf16_bits_to_f64(x)
    xq, xs = O.quantize_act(x)
    xd = F.decode_e4m3(xq) * np.repeat(2.0 ** (xs.astype(np.int64) - 127), 32, axis=1)
    w1 = F.decode_e2m1(F.unpack_e2m1(w1q[0])) * np.repeat(2.0 ** (w1s[0].astype(np.int64) - 127), 32, axis=1)
    w2 = F.decode_e2m1(F.unpack_e2m1(w2q[0])) * np.repeat(2.0 ** (w2s[0].astype(np.int64) - 127), 32, axis=1)
    assert np.max(np.abs(xd - xf)) <= np.max(np.abs(xf)) / 8      # sanity of the FP8 cast
    y = np.zeros((T, H))
    for t in range(T):
        gate = w1[:I] @ xd[t]
        up = w1[I:] @ xd[t]
        h = np.array([g / (1.0 + math.exp(-g)) * u for g, u in zip(gate, up)])
        hq, hs = O.quantize_groups_e4m3(h[None, :])
        hd = F.decode_e4m3(hq[0]) * np.repeat(2.0 ** (hs[0].astype(np.int64) - 127), 32)
        y[t] = w2 @ hd
    want = F.f64_to_bf16_bits(y)
    assert np.array_equal(out["y"], want)
    assert np.array_equal(out["y_pairs"][0], want)


def test_zero_input_gives_zero_output():
    T, H, I, E, k = 8, 64, 64, 4, 2
    _, logits, w1q, w1s, w2q, w2s = _small_layer(T, H, I, E, k, seed=2)
    x = np.zeros((T, H), dtype=np.uint16)
    out = O.forward(x, logits, w1q, w1s, w2q, w2s, k=k)
    assert np.all(out["y"] == 0) and np.all(out["hq"] == 0) and np.all(out["hs"] == 0)


def test_relabelling_experts_leaves_output_unchanged():
    T, H, I, E, k = 16, 64, 64, 6, 3
    x, logits, w1q, w1s, w2q, w2s = _small_layer(T, H, I, E, k, seed=3)
    out = O.forward(x, logits, w1q, w1s, w2q, w2s, k=k)
    sigma = np.array([4, 0, 5, 2, 1, 3])        # new expert j is old expert sigma[j]
    out2 = O.forward(x, logits[:, sigma], w1q[sigma], w1s[sigma], w2q[sigma], w2s[sigma], k=k)
    # slots keep the same order (distinct logits), so every per-pair row matches
    assert np.array_equal(out["y"], out2["y"])
    assert np.array_equal(out["y_pairs"], out2["y_pairs"])


def test_one_hot_layer_is_predictable():
    """One-hot token and weights: every value follows by hand.

    x[t] = 1 at column a; gate row f of W1 has 1.0 at column a, up row f has
    2.0 there; W2 row n has v at column f.  acc_gate = 1, acc_up = 2, so
    h_f = 2 silu(1) = 1.46212 and FP8 holds it as 384 * 2^-8 = 1.5 (scale
    2^-8).  Then y[n] = 1.5 v exactly.
    """
    T, H, I, E, k = 1, 64, 32, 1, 1
    a, f, n, v = 37, 5, 50, 0.75
    x = np.zeros((T, H), np.float32); x[0, a] = 1.0
    l1 = np.zeros((E, 2 * I, H), np.float32); l1[0, f, a] = 1.0; l1[0, I + f, a] = 2.0
    l2 = np.zeros((E, H, I), np.float32); l2[0, n, f] = v
    w1q, w1s = O.quantize_weight(_bits(torch.from_numpy(l1)))
    w2q, w2s = O.quantize_weight(_bits(torch.from_numpy(l2)))
    out = O.forward(_bits(torch.from_numpy(x)), np.zeros((T, E), np.float32),
                    w1q, w1s, w2q, w2s, k=k)
    h = out["hq"][0]
    assert h[f] == 0x7C and np.count_nonzero(h) == 1
    assert out["hs"][0, 0] == 127 - 8
    y = F.bf16_bits_to_f64(out["y"][0])
    want = np.zeros(H); want[n] = 1.5 * v
    assert np.array_equal(y, want)


def _scalar_loop_layer(x_bits, logits, w1q, w1s, w2q, w2s, k, tokens):
    """Second implementation in plain Python scalars, for a few tokens of Tiny."""
    E, twoI, H2 = w1q.shape
    H = H2 * 2
    I = twoI // 2

    def e4m3_val(c):
        mag = c & 0x7F
        ex, m = mag >> 3, mag & 7
        v = m * 2.0 ** -9 if ex == 0 else (1 + m / 8) * 2.0 ** (ex - 7)
        return -v if c & 0x80 else v

    def e2m1_val(c):
        return [0, .5, 1, 1.5, 2, 3, 4, 6][c & 7] * (-1 if c & 8 else 1)

    def w_val(q, s, e, r, c):
        byte = int(q[e, r, c // 2])
        code = byte & 0xF if c % 2 == 0 else byte >> 4
        return e2m1_val(code) * 2.0 ** (int(s[e, r, c // 32]) - 127)

    def quant32(vals):
        amax = max(abs(v) for v in vals)
        e = -127
        if amax > 0:
            e = -200
            while 448.0 * 2.0 ** e < amax:
                e += 1
        e = max(e, -127)
        out = []
        for v in vals:
            q = v * 2.0 ** -e
            best = min(range(127), key=lambda c: (abs(abs(q) - e4m3_val(c)), c % 2))
            out.append(e4m3_val(best) * (-1 if q < 0 else 1) * 2.0 ** e)
        return out

    res = {}
    for t in tokens:
        xs_row = [float(v) for v in F.bf16_bits_to_f64(x_bits[t])]
        xq_row = []
        for g in range(H // 32):
            xq_row += quant32(xs_row[32 * g:32 * g + 32])
        lg = [float(v) for v in logits[t]]
        sel = sorted(range(E), key=lambda e: (-lg[e], e))[:k]
        ex = [math.exp(lg[e] - lg[sel[0]]) for e in sel]
        wts = [float(np.float32(v / sum(ex))) for v in ex]
        total = [0.0] * H
        for j, e in enumerate(sel):
            acc = [sum(xq_row[c] * w_val(w1q, w1s, e, r, c) for c in range(H)) for r in range(2 * I)]
            h = [acc[i] / (1 + math.exp(-acc[i])) * acc[I + i] * wts[j] for i in range(I)]
            hd = []
            for g in range(I // 32):
                hd += quant32(h[32 * g:32 * g + 32])
            y = [sum(hd[i] * w_val(w2q, w2s, e, n, i) for i in range(I)) for n in range(H)]
            yb = F.bf16_bits_to_f64(F.f64_to_bf16_bits(np.array(y)))
            total = [a + b for a, b in zip(total, yb)]
        res[t] = F.f64_to_bf16_bits(np.array(total))
    return res


def test_tiny_against_scalar_loop_implementation():
    wl = W.WORKLOADS["tiny"]
    x, logits = W.tokens(wl)
    l1, l2 = W.all_expert_weights(wl, "cpu")
    xb = _bits(x)
    w1q, w1s = O.quantize_weight(_bits(l1))
    w2q, w2s = O.quantize_weight(_bits(l2))
    out = O.forward(xb, logits.numpy(), w1q, w1s, w2q, w2s, k=wl.k)
    toks = [0, 17, 63]
    ref = _scalar_loop_layer(xb, logits.numpy(), w1q, w1s, w2q, w2s, wl.k, toks)
    for t in toks:
        assert np.array_equal(out["y"][t], ref[t]), t


def test_pooled_sampled_tokens_equal_the_oracle_forward():
    """The large-workload parity test runs the oracle on a sample of tokens
    with its per-expert work spread over a process pool; that orchestration
    gives exactly oracle.moe.forward's rows for those tokens (Tiny, every
    token of a sample that includes both ends of each expert)."""
    from tests import helpers as Hp
    T, H, I, E, k = 40, 64, 64, 6, 2
    x, logits, w1q, w1s, w2q, w2s = _small_layer(T, H, I, E, k, seed=11)
    full = O.forward(x, logits, w1q, w1s, w2q, w2s, k)
    toks = Hp.sample_tokens(full["topk_idx"], full["counts"], n_random=3, seed=5)
    assert 0 < toks.size < T
    weights = {e: (w1q[e], w1s[e], w2q[e], w2s[e]) for e in range(E)}
    with Hp.oracle_pool(workers=2) as pool:
        got = Hp.oracle_forward_tokens(pool, x[toks], logits[toks], weights, k, chunk=2)
    assert np.array_equal(got["topk_idx"], full["topk_idx"][toks])
    assert np.array_equal(got["y_pairs"], full["y_pairs"][:, toks])
    assert np.array_equal(got["y"], full["y"][toks])
