"""moe_permute_noalloc: the permute for callers that cannot allocate device
memory (its scratch is the library's own device array).  Checked through the
C ABI against the oracle's permute and against moe_permute (the entry point
with a caller workspace) on the same inputs, on two calls in a row, so that
contents left in the shared array by one call cannot change the next call's
result; with the device status written to a caller buffer and to the
library's own array.

This file is collected last on purpose (pytest collects test files in name
order): a failure here comes after every other test has run."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe as O
from tests import helpers as Hp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return Hp.lib()


def _cases():
    out = []
    for name in ("tiny", "small_decode", "prefill", "skewed_prefill"):
        wl = W.WORKLOADS[name]
        _, logits = W.tokens(wl)
        idx, _ = O.route_topk(logits.numpy(), wl.k)
        out.append((name, idx, wl.E))
    rng = np.random.default_rng(9)
    idx = np.stack([rng.choice(1024, 8, replace=False) for _ in range(4000)]).astype(np.int32)   # 32000 pairs
    out.append(("E1024", idx, 1024))
    idx = np.stack([rng.choice(16, 4, replace=False) for _ in range(900)]).astype(np.int32)
    idx[rng.random(idx.shape) < 0.2] = -1
    out.append(("dropped", idx, 16))
    return out


def _outputs(E, P):
    dev = "cuda"
    return (torch.full((E,), -3, dtype=torch.int32, device=dev),
            torch.full((E + 1,), -3, dtype=torch.int32, device=dev),
            torch.full((P,), -3, dtype=torch.int32, device=dev),
            torch.full((P,), -3, dtype=torch.int32, device=dev))


@pytest.mark.parametrize("status_out", ["caller", "library"])
@pytest.mark.parametrize("case", _cases(), ids=lambda c: c[0])
def test_noalloc_permute_matches_oracle_and_workspace_permute(B, case, status_out):
    """Two calls in a row, each bit-exact against the oracle's permute and
    equal to moe_permute's outputs.  status_out = "caller": the device status
    goes to a caller buffer; "library": to the library's own array (no
    device_status argument), read back through the outputs only."""
    _, idx_np, E = case
    T, k = idx_np.shape
    P = T * k
    c_ref, o_ref, p_ref, i_ref = O.permute(idx_np, E)
    n = int(o_ref[-1])
    idx = torch.from_numpy(idx_np).cuda()
    ws = torch.empty(B.moe_permute_workspace_size(T, E, k), dtype=torch.uint8, device="cuda")
    ref = _outputs(E, P)
    B.moe_permute(idx, E, *ref, ws)
    for call in range(2):
        got = _outputs(E, P)
        st = torch.full((1,), 99, dtype=torch.int32, device="cuda") if status_out == "caller" else None
        B.moe_permute_noalloc(idx, E, *got, device_status=st)
        torch.cuda.synchronize()
        counts, offsets, perm, inv = (t.cpu().numpy() for t in got)
        assert np.array_equal(counts, c_ref), f"call {call}"
        assert np.array_equal(offsets, o_ref), f"call {call}"
        assert np.array_equal(perm[:n], p_ref), f"call {call}"
        assert np.all(perm[n:] == -3), f"call {call}: entries past offsets[E] written"
        assert np.array_equal(inv, i_ref), f"call {call}"
        for g, r in zip(got, ref):
            assert torch.equal(g, r), f"call {call}"
        if st is not None:
            assert int(st.item()) == 0


def test_noalloc_permute_reports_bad_index(B):
    idx = torch.tensor([[0, 1], [2, 9]], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _outputs(4, 4)
    B.moe_permute_noalloc(idx, 4, *out, device_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == B.MOE_ERR_DEVICE_INDEX
    assert out[0].cpu().tolist() == [1, 1, 1, 0]


def test_noalloc_permute_rejects_problems_beyond_its_array(B):
    T, E, k = 8192, 1024, 8          # 64 blocks x 1024 experts x 4 B of histogram > 64 KiB
    assert B.moe_permute_workspace_size(T, E, k) - 256 > 65536
    idx = torch.zeros(T, k, dtype=torch.int32, device="cuda")
    out = _outputs(E, T * k)
    rc = B.moe_permute_noalloc(idx, E, *out, check=False)
    assert rc == B.MOE_ERR_UNSUPPORTED_SHAPE
    torch.cuda.synchronize()
    assert torch.all(out[0] == -3)                 # nothing was enqueued
