"""ctypes binding of libmoe_mxq.so -- argument marshalling only.

Every function has the name of the C entry point it calls (include/moe_mxq.h,
include/moe_bfp8.h)
and takes torch tensors for the device buffers; all work runs in the
library's CUDA kernels on the given (default: current) stream.  PyTorch is
used for device memory and streams only.  A non-zero status raises MoeError.
There is no CPU fallback: importing this module without the built library
raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

# MOE_MXQ_LIB may point at another build of the same library (e.g. one built
# with -DMOE_MXQ_WAIT_STATS for wait-time accounting).
_LIB_PATH = os.environ.get("MOE_MXQ_LIB") or os.path.join(os.path.dirname(os.path.abspath(__file__)),
                                                          "libmoe_mxq.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"{_LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
        "or `python moe_expert_layer_counting_gb300/build.py`")

lib = ctypes.CDLL(_LIB_PATH)

_i64, _i32, _sz, _p = ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t, ctypes.c_void_p

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED_SHAPE = 2
MOE_ERR_MISALIGNED = 3
MOE_ERR_WORKSPACE_TOO_SMALL = 4
MOE_ERR_CUDA = 5
MOE_ERR_TIMEOUT = 6
MOE_ERR_DEVICE_INDEX = 7

LAYOUT_CANONICAL, LAYOUT_MMA_L1, LAYOUT_MMA_L2 = 0, 1, 2
PHASE_TOKEN_SCALES, PHASE_GEMM1, PHASE_GEMM2, PHASE_H_SCALES, PHASE_RESET = 1, 2, 4, 8, 16
SCHEDULE_DEFAULT, SCHEDULE_SEPARATE, SCHEDULE_EXPERT_WAVES = 0, 1, 2
ROUTE_SOFTMAX, ROUTE_SIGMOID, ROUTE_RAW, ROUTE_NO_RENORM = 0, 1, 2, 4
BFP8_LAYOUT_CANONICAL, BFP8_LAYOUT_TILED = 0, 1

EXPORTED = ["mxq_quantize_act", "mxq_quantize_weight", "moe_route_topk", "moe_route_topk_ex",
            "moe_permute_workspace_size",
            "moe_permute", "moe_permute_noalloc", "moe_expert_workspace_size", "moe_expert_forward", "moe_combine",
            "moe_workspace_size", "moe_forward", "moe_get_device_status", "moe_status_string", "moe_version",
            "bfp8_quantize_act", "bfp8_quantize_weight", "moe_bfp8_workspace_size", "moe_forward_bfp8"]


class MoeExpertArgs(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32),
                ("T", _i64), ("H", _i64), ("I", _i64),
                ("E", _i32), ("k", _i32),
                ("xq", _p), ("xs", _p),
                ("w1q", _p), ("w1s", _p), ("w2q", _p), ("w2s", _p),
                ("topk_idx", _p), ("topk_w", _p),
                ("counts", _p), ("offsets", _p), ("perm", _p),
                ("y_pairs", _p), ("hq", _p), ("hs", _p),
                ("tile_n", _i32), ("phases", _i32),
                ("workspace", _p), ("workspace_bytes", _sz)]


class MoeForwardArgs(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32),
                ("T", _i64), ("H", _i64), ("I", _i64),
                ("E", _i32), ("k", _i32),
                ("x", _p), ("logits", _p),
                ("w1q", _p), ("w1s", _p), ("w2q", _p), ("w2s", _p),
                ("y", _p),
                ("topk_idx_out", _p), ("topk_w_out", _p),
                ("counts_out", _p), ("offsets_out", _p), ("perm_out", _p),
                ("tile_n", _i32),
                ("workspace", _p), ("workspace_bytes", _sz),
                ("route_mode", _i32), ("phases", _i32), ("schedule", _i32)]


class MoeBfp8Args(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32),
                ("T", _i64), ("H", _i64), ("I", _i64),
                ("E", _i32), ("k", _i32), ("route_mode", _i32),
                ("x", _p), ("logits", _p), ("w1q", _p), ("w1s", _p), ("w2q", _p), ("w2s", _p), ("y", _p),
                ("topk_idx_out", _p), ("topk_w_out", _p), ("counts_out", _p), ("offsets_out", _p),
                ("perm_out", _p), ("hq_out", _p), ("hs_out", _p),
                ("workspace", _p), ("workspace_bytes", _sz), ("weight_layout", _i32), ("phases", _i32)]


lib.mxq_quantize_act.argtypes = [_p, _i64, _i64, _p, _p, _p]
lib.mxq_quantize_weight.argtypes = [_p, _i64, _i64, _i64, ctypes.c_int, _p, _p, _p]
lib.moe_route_topk.argtypes = [_p, _i64, _i32, _i32, _p, _p, _p]
lib.moe_route_topk_ex.argtypes = [_p, _i64, _i32, _i32, _i32, _p, _p, _p]
lib.moe_permute_workspace_size.argtypes = [_i64, _i32, _i32]
lib.moe_permute_workspace_size.restype = _sz
lib.moe_permute.argtypes = [_p, _i64, _i32, _i32, _p, _p, _p, _p, _p, _sz, _p]
lib.moe_permute_noalloc.argtypes = [_p, _i64, _i32, _i32, _p, _p, _p, _p, _p, _p]
lib.moe_expert_workspace_size.argtypes = [_i64, _i64, _i64, _i32, _i32]
lib.moe_expert_workspace_size.restype = _sz
lib.moe_expert_forward.argtypes = [ctypes.POINTER(MoeExpertArgs), _p]
lib.moe_combine.argtypes = [_p, _p, _i64, _i32, _i64, _p, _p]
lib.moe_workspace_size.argtypes = [_i64, _i64, _i64, _i32, _i32]
lib.moe_workspace_size.restype = _sz
lib.moe_forward.argtypes = [ctypes.POINTER(MoeForwardArgs), _p]
lib.bfp8_quantize_act.argtypes = [_p, _i64, _i64, _p, _p, _p]
lib.bfp8_quantize_weight.argtypes = [_p, _i64, _i64, _i64, ctypes.c_int, _p, _p, _p]
lib.moe_bfp8_workspace_size.argtypes = [_i64, _i64, _i64, _i32, _i32]
lib.moe_bfp8_workspace_size.restype = _sz
lib.moe_forward_bfp8.argtypes = [ctypes.POINTER(MoeBfp8Args), _p]
lib.moe_get_device_status.argtypes = [_p, _p, ctypes.POINTER(ctypes.c_int)]
lib.moe_status_string.argtypes = [ctypes.c_int]
lib.moe_status_string.restype = ctypes.c_char_p
lib.moe_version.restype = ctypes.c_char_p
for _name in ("mxq_quantize_act", "mxq_quantize_weight", "moe_route_topk", "moe_route_topk_ex", "moe_permute",
              "moe_permute_noalloc",
              "moe_expert_forward",
              "moe_combine", "moe_forward", "moe_get_device_status", "bfp8_quantize_act", "bfp8_quantize_weight",
              "moe_forward_bfp8"):
    getattr(lib, _name).restype = ctypes.c_int


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {moe_status_string(code)} (status {code})")
        self.code = code


def moe_status_string(code: int) -> str:
    return lib.moe_status_string(int(code)).decode()


def moe_version() -> str:
    return lib.moe_version().decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where)


def mxq_quantize_act(x: torch.Tensor, q: torch.Tensor, s: torch.Tensor, stream=None, check=True) -> int:
    """x bf16 [rows, K] -> q uint8 [rows, K] (E4M3), s uint8 [rows, K/32] (UE8M0)."""
    rows, K = x.shape
    rc = lib.mxq_quantize_act(_ptr(x), rows, K, _ptr(q), _ptr(s), _stream(stream))
    if check:
        _check(rc, "mxq_quantize_act")
    return rc


def mxq_quantize_weight(w: torch.Tensor, layout: int, q: torch.Tensor, s: torch.Tensor, stream=None,
                        check=True) -> int:
    """w bf16 [G, N, K] -> q uint8 [G, N, K/2] (packed E2M1), s uint8 (G*N*K/32 bytes)."""
    G, N, K = w.shape
    rc = lib.mxq_quantize_weight(_ptr(w), G, N, K, layout, _ptr(q), _ptr(s), _stream(stream))
    if check:
        _check(rc, "mxq_quantize_weight")
    return rc


def moe_route_topk(logits: torch.Tensor, k: int, topk_idx: torch.Tensor, topk_w: torch.Tensor, stream=None,
                   check=True, mode: int = ROUTE_SOFTMAX) -> int:
    T, E = logits.shape
    if mode == ROUTE_SOFTMAX:
        rc = lib.moe_route_topk(_ptr(logits), T, E, k, _ptr(topk_idx), _ptr(topk_w), _stream(stream))
    else:
        rc = lib.moe_route_topk_ex(_ptr(logits), T, E, k, mode, _ptr(topk_idx), _ptr(topk_w), _stream(stream))
    if check:
        _check(rc, "moe_route_topk")
    return rc


def moe_permute_workspace_size(T: int, E: int, k: int) -> int:
    return int(lib.moe_permute_workspace_size(T, E, k))


def moe_permute(topk_idx: torch.Tensor, E: int, counts, offsets, perm, inv_perm, workspace: torch.Tensor,
                stream=None, check=True) -> int:
    T, k = topk_idx.shape
    rc = lib.moe_permute(_ptr(topk_idx), T, E, k, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv_perm),
                         _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    if check:
        _check(rc, "moe_permute")
    return rc


def moe_permute_noalloc(topk_idx: torch.Tensor, E: int, counts, offsets, perm, inv_perm, device_status=None,
                        stream=None, check=True) -> int:
    """moe_permute without a workspace: the scratch is the library's own
    device array (see include/moe_mxq.h for the size limit and sharing rules)."""
    T, k = topk_idx.shape
    rc = lib.moe_permute_noalloc(_ptr(topk_idx), T, E, k, _ptr(counts), _ptr(offsets), _ptr(perm),
                                 _ptr(inv_perm), _ptr(device_status), _stream(stream))
    if check:
        _check(rc, "moe_permute_noalloc")
    return rc


def moe_expert_workspace_size(T: int, H: int, I: int, E: int, k: int) -> int:
    return int(lib.moe_expert_workspace_size(T, H, I, E, k))


def moe_expert_forward(xq, xs, w1q, w1s, w2q, w2s, topk_idx, topk_w, counts, offsets, perm, y_pairs,
                       workspace, hq=None, hs=None, tile_n: int = 0, phases: int = 0, stream=None,
                       check=True) -> int:
    T, H = xq.shape
    E = w1q.shape[0]
    I = w2q.shape[2] * 2
    k = topk_idx.shape[1]
    a = MoeExpertArgs(ctypes.sizeof(MoeExpertArgs), T, H, I, E, k,
                      _ptr(xq), _ptr(xs), _ptr(w1q), _ptr(w1s), _ptr(w2q), _ptr(w2s),
                      _ptr(topk_idx), _ptr(topk_w), _ptr(counts), _ptr(offsets), _ptr(perm),
                      _ptr(y_pairs), _ptr(hq), _ptr(hs), tile_n, phases,
                      _ptr(workspace), workspace.numel() * workspace.element_size())
    rc = lib.moe_expert_forward(ctypes.byref(a), _stream(stream))
    if check:
        _check(rc, "moe_expert_forward")
    return rc


def moe_combine(y_pairs: torch.Tensor, topk_idx: torch.Tensor, y: torch.Tensor, stream=None, check=True) -> int:
    k, T, H = y_pairs.shape
    rc = lib.moe_combine(_ptr(y_pairs), _ptr(topk_idx), T, k, H, _ptr(y), _stream(stream))
    if check:
        _check(rc, "moe_combine")
    return rc


def moe_workspace_size(T: int, H: int, I: int, E: int, k: int) -> int:
    return int(lib.moe_workspace_size(T, H, I, E, k))


def moe_forward(x, logits, w1q, w1s, w2q, w2s, k: int, y, workspace, topk_idx_out=None, topk_w_out=None,
                counts_out=None, offsets_out=None, perm_out=None, tile_n: int = 0, stream=None, check=True,
                route_mode: int = ROUTE_SOFTMAX, phases: int = 0, schedule: int = 0) -> int:
    T, H = x.shape
    E = logits.shape[1]
    I = w2q.shape[2] * 2
    a = MoeForwardArgs(ctypes.sizeof(MoeForwardArgs), T, H, I, E, k,
                       _ptr(x), _ptr(logits), _ptr(w1q), _ptr(w1s), _ptr(w2q), _ptr(w2s), _ptr(y),
                       _ptr(topk_idx_out), _ptr(topk_w_out), _ptr(counts_out), _ptr(offsets_out),
                       _ptr(perm_out), tile_n, _ptr(workspace), workspace.numel() * workspace.element_size(),
                       route_mode, phases, schedule)
    rc = lib.moe_forward(ctypes.byref(a), _stream(stream))
    if check:
        _check(rc, "moe_forward")
    return rc


def moe_get_device_status(workspace: torch.Tensor, stream=None) -> int:
    out = ctypes.c_int(0)
    _check(lib.moe_get_device_status(_ptr(workspace), _stream(stream), ctypes.byref(out)),
           "moe_get_device_status")
    return int(out.value)


# ---------------------------------------------------------------- block-FP8 variant (include/moe_bfp8.h)

def bfp8_quantize_act(x: torch.Tensor, q: torch.Tensor, s: torch.Tensor, stream=None, check=True) -> int:
    """x bf16 [rows, K] -> q uint8 [rows, K] (E4M3), s float32 [rows, K/128]."""
    rows, K = x.shape
    rc = lib.bfp8_quantize_act(_ptr(x), rows, K, _ptr(q), _ptr(s), _stream(stream))
    if check:
        _check(rc, "bfp8_quantize_act")
    return rc


def bfp8_quantize_weight(w: torch.Tensor, q: torch.Tensor, s: torch.Tensor, layout: int = BFP8_LAYOUT_TILED,
                         stream=None, check=True) -> int:
    """w bf16 [G, N, K] -> q uint8 (E4M3, G*N*K codes in ``layout``), s float32 [G, N/128, K/128]."""
    G, N, K = w.shape
    rc = lib.bfp8_quantize_weight(_ptr(w), G, N, K, layout, _ptr(q), _ptr(s), _stream(stream))
    if check:
        _check(rc, "bfp8_quantize_weight")
    return rc


def moe_bfp8_workspace_size(T: int, H: int, I: int, E: int, k: int) -> int:
    return int(lib.moe_bfp8_workspace_size(T, H, I, E, k))


def moe_forward_bfp8(x, logits, w1q, w1s, w2q, w2s, k: int, y, workspace, topk_idx_out=None, topk_w_out=None,
                     counts_out=None, offsets_out=None, perm_out=None, hq_out=None, hs_out=None,
                     route_mode: int = ROUTE_SOFTMAX, phases: int = 0, weight_layout: int = BFP8_LAYOUT_TILED,
                     stream=None, check=True) -> int:
    T, H = x.shape
    E = logits.shape[1]
    I = w2s.shape[2] * 128
    a = MoeBfp8Args(ctypes.sizeof(MoeBfp8Args), T, H, I, E, k, route_mode,
                    _ptr(x), _ptr(logits), _ptr(w1q), _ptr(w1s), _ptr(w2q), _ptr(w2s), _ptr(y),
                    _ptr(topk_idx_out), _ptr(topk_w_out), _ptr(counts_out), _ptr(offsets_out), _ptr(perm_out),
                    _ptr(hq_out), _ptr(hs_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                    weight_layout, phases)
    rc = lib.moe_forward_bfp8(ctypes.byref(a), _stream(stream))
    if check:
        _check(rc, "moe_forward_bfp8")
    return rc
