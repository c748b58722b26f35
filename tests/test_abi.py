"""CPU checks of the C ABI: the library loads, exports every declared entry
point, its argument structs have the C layout, and host-side validation
rejects bad arguments before anything is enqueued (no GPU needed: every case
here returns before the first CUDA call)."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

from tests import helpers as Hp

HEADER = os.path.join(Hp.ROOT, "include", "moe_mxq.h")
HEADERS = [os.path.join(Hp.ROOT, "include", h) for h in sorted(os.listdir(os.path.join(Hp.ROOT, "include")))
           if h.endswith(".h")]


def _declared():
    text = "".join(open(h).read() for h in HEADERS)
    return sorted(set(re.findall(r"MOE_API\s+(?:const\s+char\s*\*|int|size_t)\s*(\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    B = Hp.lib()
    names = _declared()
    assert len(names) >= 19 and "moe_forward_bfp8" in names
    for n in names:
        assert hasattr(B.lib, n), n
    assert set(names) == set(B.EXPORTED)


def test_struct_layout_matches_c(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    src = tmp_path / "sz.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "moe_mxq.h"\n'
        'int main(void){printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(moe_expert_args), sizeof(moe_forward_args),'
        ' offsetof(moe_expert_args, tile_n), offsetof(moe_expert_args, workspace_bytes),'
        ' offsetof(moe_forward_args, tile_n), offsetof(moe_forward_args, workspace_bytes)); return 0;}\n')
    exe = tmp_path / "sz"
    subprocess.run([cc, "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    B = Hp.lib()
    want = [ctypes.sizeof(B.MoeExpertArgs), ctypes.sizeof(B.MoeForwardArgs),
            B.MoeExpertArgs.tile_n.offset, B.MoeExpertArgs.workspace_bytes.offset,
            B.MoeForwardArgs.tile_n.offset, B.MoeForwardArgs.workspace_bytes.offset]
    assert got == want


def test_host_validation_rejects_bad_arguments():
    B = Hp.lib()
    L = B.lib
    s0 = ctypes.c_void_p(0)
    p = ctypes.c_void_p(0x1000)         # never dereferenced: validation fails first
    assert L.mxq_quantize_act(p, -1, 64, p, p, s0) == B.MOE_ERR_INVALID_ARG
    assert L.mxq_quantize_act(p, 4, 48, p, p, s0) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.mxq_quantize_act(None, 4, 64, p, p, s0) == B.MOE_ERR_INVALID_ARG
    assert L.mxq_quantize_act(ctypes.c_void_p(0x1001), 4, 64, p, p, s0) == B.MOE_ERR_MISALIGNED
    assert L.mxq_quantize_act(p, 0, 64, p, p, s0) == B.MOE_OK            # empty: no-op
    assert L.mxq_quantize_weight(p, 1, 128, 128, 9, p, p, s0) == B.MOE_ERR_INVALID_ARG
    assert L.mxq_quantize_weight(p, 1, 100, 128, 1, p, p, s0) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_route_topk(p, 4, 8, 9, p, p, s0) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_route_topk(p, 4, 2048, 2, p, p, s0) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_route_topk(p, 0, 8, 2, p, p, s0) == B.MOE_OK
    for bad_mode in (3, 7, 8, -1):
        assert L.moe_route_topk_ex(p, 4, 8, 2, bad_mode, p, p, s0) == B.MOE_ERR_INVALID_ARG
    for mode in (B.ROUTE_SIGMOID, B.ROUTE_RAW, B.ROUTE_SOFTMAX | B.ROUTE_NO_RENORM, B.ROUTE_RAW | B.ROUTE_NO_RENORM):
        assert L.moe_route_topk_ex(p, 0, 8, 2, mode, p, p, s0) == B.MOE_OK
    ws_small = 16
    assert L.moe_permute(p, 4, 8, 2, p, p, p, p, p, ws_small, s0) == B.MOE_ERR_WORKSPACE_TOO_SMALL
    assert L.moe_permute(p, 4, 8, 2, p, p, p, p, ctypes.c_void_p(0x1010), 1 << 20, s0) == B.MOE_ERR_MISALIGNED
    assert L.moe_combine(p, p, 4, 33, 64, p, s0) == B.MOE_ERR_UNSUPPORTED_SHAPE
    a = B.MoeExpertArgs()
    a.struct_size = 3
    assert L.moe_expert_forward(ctypes.byref(a), s0) == B.MOE_ERR_INVALID_ARG
    a.struct_size = ctypes.sizeof(a)
    a.T, a.H, a.I, a.E, a.k = 8, 200, 128, 4, 2
    assert L.moe_expert_forward(ctypes.byref(a), s0) == B.MOE_ERR_UNSUPPORTED_SHAPE
    a.H, a.tile_n = 256, 48
    assert L.moe_expert_forward(ctypes.byref(a), s0) == B.MOE_ERR_INVALID_ARG
    f = B.MoeForwardArgs()
    f.struct_size = ctypes.sizeof(f)
    f.T, f.H, f.I, f.E, f.k = 8, 256, 128, 4, 2
    f.workspace, f.workspace_bytes = 0x1000, 100
    assert L.moe_forward(ctypes.byref(f), s0) == B.MOE_ERR_WORKSPACE_TOO_SMALL
    for bad_phases in (32, 1, 8):                     # unknown bit; TOKEN_SCALES / H_SCALES are not forward phases
        f.phases = bad_phases
        assert L.moe_forward(ctypes.byref(f), s0) == B.MOE_ERR_INVALID_ARG
    f.phases = 0
    for bad_schedule in (-1, 3):
        f.schedule = bad_schedule
        assert L.moe_forward(ctypes.byref(f), s0) == B.MOE_ERR_INVALID_ARG
    f.schedule = B.SCHEDULE_EXPERT_WAVES
    f.workspace = 0x1080                              # not 256-byte aligned
    assert L.moe_forward(ctypes.byref(f), s0) == B.MOE_ERR_MISALIGNED
    assert B.moe_status_string(B.MOE_ERR_TIMEOUT).startswith("a device-side wait")


def test_workspace_sizes_grow_with_the_problem():
    B = Hp.lib()
    small = B.moe_workspace_size(8, 2048, 512, 256, 8)
    big = B.moe_workspace_size(4096, 7168, 2048, 256, 8)
    assert 0 < small < big
    # prefill: y_pairs (P*H*2 = 470 MB) dominates
    assert big >= 4096 * 8 * 7168 * 2
    assert B.moe_expert_workspace_size(64, 256, 128, 8, 2) > 0
    assert B.moe_permute_workspace_size(8192, 256, 8) >= 256 + 32 * 256 * 4


def test_bfp8_struct_layout_matches_c(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    src = tmp_path / "sz.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "moe_bfp8.h"\n'
        'int main(void){printf("%zu %zu %zu %zu %zu\\n", sizeof(moe_bfp8_args), offsetof(moe_bfp8_args, route_mode),'
        ' offsetof(moe_bfp8_args, x), offsetof(moe_bfp8_args, hs_out), offsetof(moe_bfp8_args, phases));'
        ' return 0;}\n')
    exe = tmp_path / "sz"
    subprocess.run([cc, "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    B = Hp.lib()
    A = B.MoeBfp8Args
    assert got == [ctypes.sizeof(A), A.route_mode.offset, A.x.offset, A.hs_out.offset, A.phases.offset]


def test_bfp8_host_validation_rejects_bad_arguments():
    B = Hp.lib()
    L = B.lib
    s0 = ctypes.c_void_p(0)
    p = ctypes.c_void_p(0x1000)
    assert L.bfp8_quantize_act(p, -1, 128, p, p, s0) == B.MOE_ERR_INVALID_ARG
    assert L.bfp8_quantize_act(p, 4, 96, p, p, s0) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.bfp8_quantize_act(None, 4, 128, p, p, s0) == B.MOE_ERR_INVALID_ARG
    assert L.bfp8_quantize_act(p, 4, 128, p, ctypes.c_void_p(0x1002), s0) == B.MOE_ERR_MISALIGNED
    assert L.bfp8_quantize_act(p, 4, 128, ctypes.c_void_p(0x1004), p, s0) == B.MOE_ERR_MISALIGNED
    assert L.bfp8_quantize_act(p, 0, 128, p, p, s0) == B.MOE_OK
    assert L.bfp8_quantize_weight(p, 1, 64, 128, 0, p, p, s0) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.bfp8_quantize_weight(p, -1, 128, 128, 0, p, p, s0) == B.MOE_ERR_INVALID_ARG
    assert L.bfp8_quantize_weight(p, 1, 128, 128, 2, p, p, s0) == B.MOE_ERR_INVALID_ARG
    assert L.bfp8_quantize_weight(p, 0, 128, 128, 1, p, p, s0) == B.MOE_OK
    assert L.moe_bfp8_workspace_size(-1, 128, 128, 4, 2) == 0
    assert L.moe_bfp8_workspace_size(8, 2048, 512, 256, 8) > 8 * 8 * 2048 * 4
    a = B.MoeBfp8Args()
    a.struct_size = 7
    assert L.moe_forward_bfp8(ctypes.byref(a), s0) == B.MOE_ERR_INVALID_ARG
    a.struct_size = ctypes.sizeof(a)
    a.T, a.H, a.I, a.E, a.k = 8, 192, 128, 4, 2
    assert L.moe_forward_bfp8(ctypes.byref(a), s0) == B.MOE_ERR_UNSUPPORTED_SHAPE      # H % 128
    a.H, a.k = 256, 5
    assert L.moe_forward_bfp8(ctypes.byref(a), s0) == B.MOE_ERR_UNSUPPORTED_SHAPE      # k > E
    a.k, a.route_mode = 2, 3
    assert L.moe_forward_bfp8(ctypes.byref(a), s0) == B.MOE_ERR_INVALID_ARG            # bad routing mode
    a.route_mode, a.phases = 0, 1
    assert L.moe_forward_bfp8(ctypes.byref(a), s0) == B.MOE_ERR_INVALID_ARG            # bad phase mask
    a.phases, a.weight_layout = 0, 5
    assert L.moe_forward_bfp8(ctypes.byref(a), s0) == B.MOE_ERR_INVALID_ARG            # bad weight layout
    a.weight_layout = 1
    assert L.moe_forward_bfp8(ctypes.byref(a), s0) == B.MOE_ERR_INVALID_ARG            # no workspace
    a.workspace = ctypes.c_void_p(0x1080)
    assert L.moe_forward_bfp8(ctypes.byref(a), s0) == B.MOE_ERR_MISALIGNED
    a.workspace, a.workspace_bytes = ctypes.c_void_p(0x10000), 64
    assert L.moe_forward_bfp8(ctypes.byref(a), s0) == B.MOE_ERR_WORKSPACE_TOO_SMALL
    a.workspace_bytes = L.moe_bfp8_workspace_size(8, 256, 128, 4, 2)
    assert L.moe_forward_bfp8(ctypes.byref(a), s0) == B.MOE_ERR_INVALID_ARG            # null tensors
    a.x = a.logits = a.y = a.w1q = a.w1s = a.w2q = a.w2s = p
    a.y = ctypes.c_void_p(0x1008)
    assert L.moe_forward_bfp8(ctypes.byref(a), s0) == B.MOE_ERR_MISALIGNED
