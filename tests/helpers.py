"""Shared helpers of the test-suite: building/loading the library, moving
workloads to the GPU, the host-side restatement of the MMA weight layouts,
and the comparison rules used by the parity tests."""
from __future__ import annotations

import functools
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import formats as F  # noqa: E402


@functools.lru_cache(maxsize=None)
def lib():
    """Builds (if stale) and imports the binding."""
    import __graft_entry__
    __graft_entry__.build()
    from moe_expert_layer_counting_gb300 import binding
    return binding


def bits16(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def to_np_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().numpy().view(np.uint8)


# ---------------------------------------------------------------- MMA weight layouts (host restatement)

def l1_row_source(N: int) -> np.ndarray:
    """Input row held by stored row r of the gate/up interleave (groups of 8)."""
    half = N // 2
    r = np.arange(N)
    b, c = r // 16, r % 16
    return np.where(c < 8, 8 * b + c, half + 8 * b + c - 8)


def canonical_to_mma(q: np.ndarray, s: np.ndarray, interleave: bool):
    """Canonical (codes [G,N,K/2], scales [G,N,K/32]) -> MMA layout (codes, flat chunk scales)."""
    G, N, K2 = q.shape
    K = 2 * K2
    if interleave:
        src = l1_row_source(N)
        q = q[:, src]
        s = s[:, src]
    NT, KB = N // 128, K // 128
    sc = s.reshape(G, NT, 128, KB, 4)                 # [g, nt, rr, kb, kk]
    chunk = np.zeros((G, NT, KB, 512), dtype=np.uint8)
    rr = np.arange(128)
    pos = (rr % 32) * 16 + (rr // 32) * 4             # [rr]
    for kk in range(4):
        chunk[:, :, :, pos + kk] = sc[:, :, :, :, kk].transpose(0, 1, 3, 2)
    qt = q.reshape(G, NT, 128, KB, 64).transpose(0, 1, 3, 2, 4)        # [g, nt, kb, row, 64 B]
    return np.ascontiguousarray(qt).reshape(G, N, K2), chunk.reshape(-1)


def mma_to_canonical(q: np.ndarray, chunk: np.ndarray, G: int, N: int, K: int, interleave: bool):
    NT, KB = N // 128, K // 128
    q = np.ascontiguousarray(q.reshape(G, NT, KB, 128, 64).transpose(0, 1, 3, 2, 4)).reshape(G, N, K // 2)
    c = chunk.reshape(G, NT, KB, 512)
    rr = np.arange(128)
    pos = (rr % 32) * 16 + (rr // 32) * 4
    s = np.zeros((G, NT, 128, KB, 4), dtype=np.uint8)
    for kk in range(4):
        s[:, :, :, :, kk] = c[:, :, :, pos + kk].transpose(0, 1, 3, 2)
    s = s.reshape(G, N, K // 32)
    if interleave:
        src = l1_row_source(N)
        inv = np.empty_like(src)
        inv[src] = np.arange(N)
        q = q[:, inv]
        s = s[:, inv]
    return q, s


# ---------------------------------------------------------------- comparison rules

def assert_bf16_close(got_bits: np.ndarray, ref_bits: np.ndarray, rel_fro=5e-3, max_abs_frac=1e-2, what=""):
    """The layer's output tolerance: relative Frobenius error <= 5e-3 and
    max |error| <= 1e-2 * max |y_ref| (values compared as float64)."""
    g = F.bf16_bits_to_f64(got_bits)
    r = F.bf16_bits_to_f64(ref_bits)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = g - r
    nr = np.linalg.norm(r)
    fro = np.linalg.norm(err) / max(nr, 1e-300)
    mx = np.max(np.abs(err)) if err.size else 0.0
    ref_max = np.max(np.abs(r)) if r.size else 0.0
    assert fro <= rel_fro, f"{what}: relative Frobenius error {fro:.3e} > {rel_fro}"
    assert mx <= max_abs_frac * ref_max + 1e-30, f"{what}: max abs error {mx:.3e} > {max_abs_frac} * {ref_max:.3e}"
    return fro, mx


def e4m3_code_rank(codes: np.ndarray) -> np.ndarray:
    """Signed position of an E4M3 code on the number line (adjacent codes differ by 1)."""
    c = codes.astype(np.int64)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def check_requantised_h(hq_g, hs_g, hq_r, hs_r, amax_ref=None, max_code_frac=1e-3):
    """FP8 intermediates: codes may differ by one step on at most 0.1% of the
    elements; a scale byte may differ by one only where the two sides' group
    amax straddles a power-of-two boundary (then the codes of that group are
    compared on dequantised values, within one code step of the coarser
    scale).  Returns (fraction of differing codes, number of scale mismatches)."""
    hq_g = hq_g.astype(np.uint8); hq_r = hq_r.astype(np.uint8)
    rows, I = hq_r.shape
    sg = hs_g.astype(np.int64); sr = hs_r.astype(np.int64)
    smis = sg != sr
    assert np.all(np.abs(sg - sr) <= 1), "scale bytes differ by more than one"
    same_scale = np.repeat(~smis, 32, axis=1)
    d = np.abs(e4m3_code_rank(hq_g) - e4m3_code_rank(hq_r))
    assert np.all(d[same_scale] <= 1), "an FP8 code differs by more than one step"
    n_code = int(np.count_nonzero(d[same_scale]))
    if smis.any():
        vg = F.decode_e4m3(hq_g) * np.repeat(F.scale_value(hs_g), 32, axis=1)
        vr = F.decode_e4m3(hq_r) * np.repeat(F.scale_value(hs_r), 32, axis=1)
        # widest gap between neighbouring E4M3 values is 32 (256..448) times the scale
        step = np.repeat(F.scale_value(np.maximum(hs_g, hs_r).astype(np.uint8)), 32, axis=1) * 32.0
        bad = np.abs(vg - vr)[~same_scale] > step[~same_scale]
        assert not bad.any(), "a rescaled group differs by more than one code step"
        n_code += int(np.count_nonzero((vg != vr)[~same_scale]))
    frac = n_code / max(hq_r.size, 1)
    assert frac <= max_code_frac, f"{frac:.2e} of FP8 codes differ (> {max_code_frac})"
    assert smis.sum() <= max(1, int(1e-3 * smis.size)), f"{int(smis.sum())} scale bytes differ"
    return frac, int(smis.sum())


# ---------------------------------------------------------------- the oracle on many large experts

def oracle_pool(workers=None):
    """Process pool for running the oracle on many large experts at once.

    Started with the spawn method, so it is safe to create after CUDA was
    initialised in this process (a forked child of a CUDA process can hang)."""
    import concurrent.futures as cf
    import multiprocessing as mp
    n = workers or max(1, min(16, len(os.sched_getaffinity(0))))
    return cf.ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"))


def sample_tokens(idx: np.ndarray, counts: np.ndarray, n_random: int, seed: int) -> np.ndarray:
    """Tokens of a large workload whose output rows are compared with the oracle.

    For each of the two hottest and the two coldest non-empty experts: its
    first and last token (an expert's last token sits in its ragged last token
    tile), all of its tokens when it has at most three; the last two tokens
    of expert 0 (the hottest expert of the skewed workload); then
    ``n_random`` further tokens drawn with ``seed``."""
    T = idx.shape[0]
    nz = np.nonzero(counts)[0]
    order = nz[np.argsort(counts[nz], kind="stable")]
    pick = set()
    for e in list(order[:2]) + list(order[-2:]):
        toks = np.nonzero((idx == e).any(axis=1))[0]
        pick.update(int(t) for t in (toks if toks.size <= 3 else (toks[0], toks[-1])))
    t0 = np.nonzero((idx == 0).any(axis=1))[0]
    pick.update(int(t) for t in t0[-2:])
    rng = np.random.default_rng(seed)
    rest = np.setdiff1d(np.arange(T), np.array(sorted(pick), dtype=np.int64))
    pick.update(int(t) for t in rng.choice(rest, size=min(n_random, rest.size), replace=False))
    return np.array(sorted(pick), dtype=np.int64)


def oracle_forward_tokens(pool, x_bits, logits, weights, k, chunk=2):
    """The oracle's layer on a few tokens, its per-expert work spread over ``pool``.

    Same steps as ``oracle.moe.forward``: the oracle's activation cast and
    routing of these tokens, then ``oracle.moe.expert_forward`` per group of
    ``chunk`` experts (the expert ids renumbered inside each group, the
    other experts' pairs marked dropped), each pair's row taken from the group
    that holds its expert, and ``oracle.moe.combine``.  ``weights`` maps an
    expert id to its oracle-quantised (w1q, w1s, w2q, w2s); it must hold
    every expert the tokens route to."""
    from oracle import moe as O
    xq, xs = O.quantize_act(x_bits)
    idx, w = O.route_topk(logits, k)
    experts = sorted(set(int(e) for e in idx.reshape(-1)))
    missing = [e for e in experts if e not in weights]
    assert not missing, f"oracle weights missing for experts {missing}"
    jobs = []
    for c in range(0, len(experts), chunk):
        sub = experts[c:c + chunk]
        local = np.full(idx.shape, -1, np.int32)
        for i, e in enumerate(sub):
            local[idx == e] = i
        ws = [np.stack([weights[e][j] for e in sub]) for j in range(4)]
        jobs.append((local, pool.submit(O.expert_forward, xq, xs, *ws, local, w, len(sub))))
    y_pairs = np.zeros((k, idx.shape[0], xq.shape[1]), np.uint16)
    for local, fut in jobs:
        yp = fut.result()
        mine = (local >= 0).T                                  # [k, T]
        y_pairs[mine] = yp[mine]
    return {"topk_idx": idx, "topk_w": w, "y_pairs": y_pairs, "y": O.combine(y_pairs, idx)}
