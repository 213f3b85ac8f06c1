"""Python binding of libnvfp4moe (ctypes).

Argument marshalling only: every function checks tensor dtypes, shapes and
devices, allocates output tensors with torch when the caller passes none,
and calls the C entry point of the same name on the current CUDA stream.
All arithmetic of the layer runs in the library's CUDA kernels; there is no
CPU or PyTorch fallback, and importing this module fails loudly when the
shared library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libnvfp4moe.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libnvfp4moe.so is not built at {LIB_PATH}; build it with `python -c 'import __graft_entry__ as g; "
        f"g.build()'` (nvcc, sm_103a). There is no fallback implementation.")

_lib = ctypes.CDLL(LIB_PATH)

# ---- constants (mirror include/nvfp4moe.h) ---------------------------------
OK = 0
ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_SMEM, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE_DATA = range(1, 8)
SCORE = {"softmax": 0, "sigmoid": 1}
QUANT_COMPUTE_GLOBAL = 1
QUANT_SCALES_BLOCKED = 2
EPI_BF16, EPI_SWIGLU_NVFP4, EPI_SWIGLU_F32, EPI_SWIGLU_MXFP4, EPI_FINALIZE_F32 = 0, 1, 2, 3, 4
TILE_TOKEN_MAJOR = -1  # grouped GEMM tile_n: 128 tokens as M, two weight tiles as one N = 256 operand
TILE_TOKEN_MAJOR_PAIR = -2  # the same on a pair of SMs: 256 tokens as M (cta_group::2 MMAs)
W_ROWMAJOR, W_TILED = 0, 1  # grouped GEMM weight layouts

_i, _i64, _sz, _p, _f = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float
_SIGS = {
    "nvfp4moe_version": (_i, []),
    "nvfp4moe_status_string": (ctypes.c_char_p, [_i]),
    "nvfp4moe_last_error_detail": (ctypes.c_char_p, []),
    "nvfp4moe_device_check": (_i, [_i]),
    "nvfp4moe_sync_status": (_i, [_p]),
    "nvfp4moe_set_wait_limit_us": (_i, [ctypes.c_uint32]),
    "nvfp4moe_wait_limit_us": (ctypes.c_uint32, []),
    "nvfp4moe_wait_selftest": (_i, [ctypes.c_uint32, ctypes.c_uint32, _p]),
    "nvfp4moe_blocked_scales_bytes": (_sz, [_i64, _i64]),
    "nvfp4moe_mxfp4_blocked_scales_bytes": (_sz, [_i64, _i64]),
    "moe_quantize_mxfp4": (_i, [_p, _i64, _i64, _i, _p, _p, _p]),
    "moe_permute_mxfp4": (_i, [_p, _i, _i, _i, _p, _p, _i, _p, _p, _p, _p, _p, _p, _p, _p, _sz, _p]),
    "moe_prepare_mxfp4": (_i, [_p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p,
                               _p, _sz, _p]),
    "moe_grouped_gemm_mxfp4": (_i, [_p, _p, _p, _p, _i, _i64, _i64, _p, _p, _i, _i, _i, _p, _p, _i, _i, _p, _sz, _p]),
    "moe_grouped_gemm_mxfp4_range": (_i, [_p, _p, _p, _p, _i, _i64, _i64, _p, _p, _i, _i, _i, _p, _p, _i, _i,
                                          ctypes.c_int32, ctypes.c_int32, _p, _sz, _p]),
    "nvfp4moe_tiled_weights_bytes": (_sz, [_i64, _i]),
    "nvfp4moe_tile_weights": (_i, [_p, _i64, _i, _p, _p]),
    "moe_route_topk": (_i, [_p, _p, _i, _i, _i, _i, _i, _p, _p, _p]),
    "moe_route_batch_aware_workspace_size": (_sz, [_i]),
    "moe_route_batch_aware": (_i, [_p, _p, _i, _i, _i, _i, _i, _i, _p, _p, _p, _sz, _p]),
    "moe_quantize_nvfp4_workspace_size": (_sz, [_i64, _i64, _i]),
    "moe_quantize_nvfp4": (_i, [_p, _i64, _i64, _p, _i, _p, _p, _p, _sz, _p]),
    "moe_scales_to_blocked": (_i, [_p, _i64, _i64, _p, _p]),
    "moe_permute_rows_capacity": (_i64, [_i, _i, _i]),
    "moe_permute_workspace_size": (_sz, [_i, _i, _i]),
    "moe_permute": (_i, [_p, _i, _i, _i, _p, _p, _i, _p, _p, _p, _p, _p, _p, _p, _p, _sz, _p]),
    "moe_permute_no_alloc": (_i, [_p, _i, _i, _i, _p, _p, _i, _p, _p, _p, _p, _p, _p, _p, _p]),
    "moe_prepare_workspace_size": (_sz, [_i, _i, _i]),
    "moe_prepare": (_i, [_p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p,
                         _p, _sz, _p]),
    "moe_grouped_gemm_nvfp4_workspace_size": (_sz, [_i, _i, _i, _i]),
    "nvfp4moe_gemm_tile_choice": (_i, [_i, _i, _i64, _i]),
    "moe_grouped_gemm_nvfp4": (_i, [_p, _p, _p, _p, _p, _i, _i64, _i64, _p, _p, _p, _i, _i, _i, _p, _p, _p, _i,
                                    _i, _p, _sz, _p]),
    "moe_grouped_gemm_nvfp4_range": (_i, [_p, _p, _p, _p, _p, _i, _i64, _i64, _p, _p, _p, _i, _i, _i, _p, _p, _p,
                                          _i, _i, ctypes.c_int32, ctypes.c_int32, _p, _sz, _p]),
    "moe_finalize": (_i, [_p, _p, _p, _i, _i, _i, _i64, _p, _p]),
    "moe_grouped_gemm_nvfp4_finalize": (_i, [_p, _p, _p, _p, _p, _i, _i64, _i64, _p, _p, _p, _i, _i, _p, _p, _i, _i,
                                             _p, _i, _i, ctypes.c_int32, ctypes.c_int32, _p, _sz, _p]),
    "moe_finalize_f32": (_i, [_p, _i, _i, _p, _p]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class Nvfp4MoeError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = _lib.nvfp4moe_status_string(status).decode()
        detail = _lib.nvfp4moe_last_error_detail().decode()
        super().__init__(f"{where}: status {status} ({msg}): {detail}")


def _check(status, where):
    if status != OK:
        raise Nvfp4MoeError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need(t, dtype, shape=None, name="tensor"):
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def _empty(shape, dtype, device):
    return torch.empty(shape, dtype=dtype, device=device)


# ---- library / device --------------------------------------------------------
def version():
    return _lib.nvfp4moe_version()


def device_check(device=None):
    dev = torch.cuda.current_device() if device is None else int(device)
    _check(_lib.nvfp4moe_device_check(dev), "nvfp4moe_device_check")


def sync_status():
    """Synchronise the current stream and raise on sticky device flags."""
    _check(_lib.nvfp4moe_sync_status(_stream()), "nvfp4moe_sync_status")


def set_wait_limit_us(us):
    """Limit of every bounded device wait, in microseconds (0: the default, 2 s)."""
    _check(_lib.nvfp4moe_set_wait_limit_us(int(us)), "nvfp4moe_set_wait_limit_us")


def wait_limit_us():
    return int(_lib.nvfp4moe_wait_limit_us())


def wait_selftest(expected_arrivals, arrivals):
    """Enqueue the bounded-wait self-test (see the header); a phase that can
    never complete shows up as ERR_TIMEOUT at the next sync_status()."""
    _check(_lib.nvfp4moe_wait_selftest(int(expected_arrivals), int(arrivals), _stream()), "nvfp4moe_wait_selftest")


def blocked_scales_bytes(rows, cols, fmt="nvfp4"):
    if fmt == "mxfp4":
        return int(_lib.nvfp4moe_mxfp4_blocked_scales_bytes(rows, cols))
    return int(_lib.nvfp4moe_blocked_scales_bytes(rows, cols))


# ---- a1 ------------------------------------------------------------------------
def moe_route_topk(logits, k, score_fn="sigmoid", renormalize=True, bias=None, topk_idx=None, topk_w=None):
    T, E = logits.shape
    _need(logits, torch.float32, name="logits")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    if topk_idx is None:
        topk_idx = _empty((T, k), torch.int32, logits.device)
    if topk_w is None:
        topk_w = _empty((T, k), torch.float32, logits.device)
    _need(topk_idx, torch.int32, (T, k), "topk_idx")
    _need(topk_w, torch.float32, (T, k), "topk_w")
    _check(_lib.moe_route_topk(_ptr(logits), _ptr(bias), T, E, k, SCORE[score_fn], int(bool(renormalize)),
                               _ptr(topk_idx), _ptr(topk_w), _stream()), "moe_route_topk")
    return topk_idx, topk_w


def moe_route_batch_aware(logits, k, k_primary, score_fn="sigmoid", renormalize=True, bias=None, topk_idx=None,
                          topk_w=None, workspace=None):
    """Batch-aware routing: each token's top-k_primary experts form the
    batch's active set; each token then takes its best k experts, members of
    the set first.  k_primary == k is moe_route_topk."""
    T, E = logits.shape
    _need(logits, torch.float32, name="logits")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    dev = logits.device
    topk_idx = _empty((T, k), torch.int32, dev) if topk_idx is None else topk_idx
    topk_w = _empty((T, k), torch.float32, dev) if topk_w is None else topk_w
    _need(topk_idx, torch.int32, (T, k), "topk_idx")
    _need(topk_w, torch.float32, (T, k), "topk_w")
    if workspace is None:
        workspace = _empty((int(_lib.moe_route_batch_aware_workspace_size(E)),), torch.uint8, dev)
    _check(_lib.moe_route_batch_aware(_ptr(logits), _ptr(bias), T, E, k, int(k_primary), SCORE[score_fn],
                                      int(bool(renormalize)), _ptr(topk_idx), _ptr(topk_w), _ptr(workspace),
                                      workspace.numel(), _stream()), "moe_route_batch_aware")
    return topk_idx, topk_w


# ---- a2 ------------------------------------------------------------------------
def moe_quantize_nvfp4(x, global_scale=None, compute_global=None, blocked=False, packed=None, scales=None,
                       workspace=None):
    """Returns (packed [rows, cols/2] u8, scales u8, global_scale f32 [1])."""
    _need(x, torch.bfloat16, name="x")
    rows, cols = x.shape
    dev = x.device
    if compute_global is None:
        compute_global = global_scale is None
    if global_scale is None:
        global_scale = _empty((1,), torch.float32, dev)
    _need(global_scale, torch.float32, (1,), "global_scale")
    flags = (QUANT_COMPUTE_GLOBAL if compute_global else 0) | (QUANT_SCALES_BLOCKED if blocked else 0)
    if packed is None:
        packed = _empty((rows, cols // 2), torch.uint8, dev)
    if scales is None:
        scales = _empty((blocked_scales_bytes(rows, cols),) if blocked else (rows, cols // 16), torch.uint8, dev)
    _need(packed, torch.uint8, name="packed")
    _need(scales, torch.uint8, name="scales")
    ws_bytes = int(_lib.moe_quantize_nvfp4_workspace_size(rows, cols, flags))
    if ws_bytes and workspace is None:
        workspace = _empty((ws_bytes,), torch.uint8, dev)
    _check(_lib.moe_quantize_nvfp4(_ptr(x), rows, cols, _ptr(global_scale), flags, _ptr(packed), _ptr(scales),
                                   _ptr(workspace) if ws_bytes else None,
                                   workspace.numel() if (ws_bytes and workspace is not None) else 0, _stream()),
           "moe_quantize_nvfp4")
    return packed, scales, global_scale


def moe_scales_to_blocked(scales, cols, out=None):
    _need(scales, torch.uint8, name="scales")
    rows = scales.shape[0]
    if out is None:
        out = _empty((blocked_scales_bytes(rows, cols),), torch.uint8, scales.device)
    _check(_lib.moe_scales_to_blocked(_ptr(scales), rows, cols, _ptr(out), _stream()), "moe_scales_to_blocked")
    return out


def quantize_expert_weights(w):
    """bf16 [E, N, K] -> (packed [E, N, K/2], blocked scales [E, bytes], per-expert scales [E]).

    One moe_quantize_nvfp4 call per expert matrix, each computing its own
    per-tensor scale."""
    _need(w, torch.bfloat16, name="w")
    E, N, K = w.shape
    dev = w.device
    packed = _empty((E, N, K // 2), torch.uint8, dev)
    scales = _empty((E, blocked_scales_bytes(N, K)), torch.uint8, dev)
    gscale = _empty((E,), torch.float32, dev)
    ws = _empty((64,), torch.uint8, dev)
    for e in range(E):
        moe_quantize_nvfp4(w[e], global_scale=gscale[e:e + 1], compute_global=True, blocked=True,
                           packed=packed[e], scales=scales[e], workspace=ws)
    return packed, scales, gscale


# ---- MXFP4 variant of a2 ---------------------------------------------------------
def moe_quantize_mxfp4(x, blocked=False, packed=None, scales=None):
    """MXFP4: returns (packed [rows, cols/2] u8, scales u8 row-major [rows, cols/32] or blocked)."""
    _need(x, torch.bfloat16, name="x")
    rows, cols = x.shape
    dev = x.device
    if packed is None:
        packed = _empty((rows, cols // 2), torch.uint8, dev)
    if scales is None:
        scales = _empty((blocked_scales_bytes(rows, cols, "mxfp4"),) if blocked else (rows, cols // 32),
                        torch.uint8, dev)
    _need(packed, torch.uint8, name="packed")
    _need(scales, torch.uint8, name="scales")
    _check(_lib.moe_quantize_mxfp4(_ptr(x), rows, cols, QUANT_SCALES_BLOCKED if blocked else 0, _ptr(packed),
                                   _ptr(scales), _stream()), "moe_quantize_mxfp4")
    return packed, scales


def quantize_expert_weights_mx(w):
    """bf16 [E, N, K] -> MXFP4 (packed [E, N, K/2], blocked scales [E, bytes])."""
    _need(w, torch.bfloat16, name="w")
    E, N, K = w.shape
    packed = _empty((E, N, K // 2), torch.uint8, w.device)
    scales = _empty((E, blocked_scales_bytes(N, K, "mxfp4")), torch.uint8, w.device)
    for e in range(E):
        moe_quantize_mxfp4(w[e], blocked=True, packed=packed[e], scales=scales[e])
    return packed, scales


@dataclass
class TiledWeights:
    """Packed expert weights [E, N, K/2] in the tiled layout (nvfp4moe_tile_weights):
    each 128-row x 128-byte box the grouped GEMM loads is contiguous."""
    data: torch.Tensor  # uint8, nvfp4moe_tiled_weights_bytes(E * N, K) bytes
    E: int
    N: int
    K: int


def tile_expert_weights(packed):
    """Packed [E, N, K/2] (NVFP4 or MXFP4 codes) -> TiledWeights."""
    _need(packed, torch.uint8, name="packed")
    E, N, Kh = packed.shape
    K = 2 * Kh
    n = int(_lib.nvfp4moe_tiled_weights_bytes(E * N, K))
    if n == 0:
        raise ValueError(f"cannot tile [{E}, {N}, {Kh}] (E*N % 128, K % 64)")
    out = _empty((n,), torch.uint8, packed.device)
    _check(_lib.nvfp4moe_tile_weights(_ptr(packed), E * N, K, _ptr(out), _stream()), "nvfp4moe_tile_weights")
    return TiledWeights(out, E, N, K)


def _weights_args(w_packed):
    """(E, N, K, pointer, layout) of row-major packed weights or TiledWeights."""
    if isinstance(w_packed, TiledWeights):
        return w_packed.E, w_packed.N, w_packed.K, _ptr(w_packed.data), W_TILED
    _need(w_packed, torch.uint8, name="w_packed")
    E, N, Kh = w_packed.shape
    return E, N, 2 * Kh, _ptr(w_packed), W_ROWMAJOR


# ---- a3 ------------------------------------------------------------------------
def moe_permute_rows_capacity(T, E, k):
    return int(_lib.moe_permute_rows_capacity(T, E, k))


@dataclass
class Permutation:
    counts: torch.Tensor
    offsets: torch.Tensor
    row_offsets: torch.Tensor
    perm_to_flat: torch.Tensor
    flat_to_perm: torch.Tensor
    a_packed: torch.Tensor
    a_scales: torch.Tensor
    rows_capacity: int


def alloc_permutation(T, E, k, H, device, fmt="nvfp4"):
    cap = moe_permute_rows_capacity(T, E, k)
    return Permutation(
        counts=_empty((E,), torch.int32, device), offsets=_empty((E + 1,), torch.int32, device),
        row_offsets=_empty((E + 1,), torch.int32, device), perm_to_flat=_empty((cap,), torch.int32, device),
        flat_to_perm=_empty((T * k,), torch.int32, device), a_packed=_empty((cap, H // 2), torch.uint8, device),
        a_scales=_empty((blocked_scales_bytes(cap, H, fmt),), torch.uint8, device), rows_capacity=cap)


def moe_permute_workspace_size(T, E, k):
    return int(_lib.moe_permute_workspace_size(T, E, k))


def moe_permute(topk_idx, E, xq, xs, out: Permutation = None, workspace=None):
    _need(topk_idx, torch.int32, name="topk_idx")
    T, k = topk_idx.shape
    H = xq.shape[1] * 2
    _need(xq, torch.uint8, (T, H // 2), "xq")
    _need(xs, torch.uint8, (T, H // 16), "xs")
    dev = topk_idx.device
    if out is None:
        out = alloc_permutation(T, E, k, H, dev)
    ws_bytes = moe_permute_workspace_size(T, E, k)
    if workspace is None:
        workspace = _empty((ws_bytes,), torch.uint8, dev)
    _check(_lib.moe_permute(_ptr(topk_idx), T, E, k, _ptr(xq), _ptr(xs), H, _ptr(out.counts), _ptr(out.offsets),
                            _ptr(out.row_offsets), _ptr(out.perm_to_flat), _ptr(out.flat_to_perm),
                            _ptr(out.a_packed), _ptr(out.a_scales), _ptr(workspace), workspace.numel(), _stream()),
           "moe_permute")
    return out


def moe_permute_mxfp4(topk_idx, E, xq, xs, out: Permutation = None, workspace=None):
    """moe_permute for MXFP4 rows (xs row-major [T, H/32]; a_scales blocked MXFP4)."""
    _need(topk_idx, torch.int32, name="topk_idx")
    T, k = topk_idx.shape
    H = xq.shape[1] * 2
    _need(xq, torch.uint8, (T, H // 2), "xq")
    _need(xs, torch.uint8, (T, H // 32), "xs")
    dev = topk_idx.device
    if out is None:
        out = alloc_permutation(T, E, k, H, dev, "mxfp4")
    ws_bytes = moe_permute_workspace_size(T, E, k)
    if workspace is None:
        workspace = _empty((ws_bytes,), torch.uint8, dev)
    _check(_lib.moe_permute_mxfp4(_ptr(topk_idx), T, E, k, _ptr(xq), _ptr(xs), H, _ptr(out.counts),
                                  _ptr(out.offsets), _ptr(out.row_offsets), _ptr(out.perm_to_flat),
                                  _ptr(out.flat_to_perm), _ptr(out.a_packed), _ptr(out.a_scales), _ptr(workspace),
                                  workspace.numel(), _stream()), "moe_permute_mxfp4")
    return out


def moe_permute_no_alloc(topk_idx, E, xq, xs, out: Permutation = None):
    """moe_permute on the library's own scratch (no workspace argument).

    For callers that cannot allocate device memory at call time; the C call
    allocates nothing (pass `out` to make the whole call allocation-free)."""
    _need(topk_idx, torch.int32, name="topk_idx")
    T, k = topk_idx.shape
    H = xq.shape[1] * 2
    _need(xq, torch.uint8, (T, H // 2), "xq")
    _need(xs, torch.uint8, (T, H // 16), "xs")
    if out is None:
        out = alloc_permutation(T, E, k, H, topk_idx.device)
    _check(_lib.moe_permute_no_alloc(_ptr(topk_idx), T, E, k, _ptr(xq), _ptr(xs), H, _ptr(out.counts),
                                     _ptr(out.offsets), _ptr(out.row_offsets), _ptr(out.perm_to_flat),
                                     _ptr(out.flat_to_perm), _ptr(out.a_packed), _ptr(out.a_scales), _stream()),
           "moe_permute_no_alloc")
    return out


# ---- a1 + a2 + a3 in one launch ------------------------------------------------------
def moe_prepare_workspace_size(T, E, k):
    return int(_lib.moe_prepare_workspace_size(T, E, k))


def alloc_prepare_workspace(T, E, k, device):
    """Zero-filled workspace for moe_prepare (its barrier words must start at 0)."""
    return torch.zeros((moe_prepare_workspace_size(T, E, k),), dtype=torch.uint8, device=device)


def moe_prepare(logits, x, k, score_fn="sigmoid", renormalize=True, bias=None, topk_idx=None, topk_w=None,
                x_gscale=None, xq=None, xs=None, out: Permutation = None, workspace=None, k_primary=None):
    """Route, quantise and permute in one launch.

    Returns (topk_idx, topk_w, x_gscale, xq, xs, Permutation), each equal bit
    for bit to moe_route_topk (moe_route_batch_aware when k_primary < k) +
    moe_quantize_nvfp4 + moe_permute."""
    k_primary = k if k_primary is None else int(k_primary)
    _need(logits, torch.float32, name="logits")
    _need(x, torch.bfloat16, name="x")
    T, E = logits.shape
    H = x.shape[1]
    if x.shape[0] != T:
        raise ValueError(f"x has {x.shape[0]} rows, logits {T}")
    dev = x.device
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    topk_idx = _empty((T, k), torch.int32, dev) if topk_idx is None else topk_idx
    topk_w = _empty((T, k), torch.float32, dev) if topk_w is None else topk_w
    x_gscale = _empty((1,), torch.float32, dev) if x_gscale is None else x_gscale
    xq = _empty((T, H // 2), torch.uint8, dev) if xq is None else xq
    xs = _empty((T, H // 16), torch.uint8, dev) if xs is None else xs
    _need(topk_idx, torch.int32, (T, k), "topk_idx")
    _need(topk_w, torch.float32, (T, k), "topk_w")
    _need(x_gscale, torch.float32, (1,), "x_gscale")
    _need(xq, torch.uint8, (T, H // 2), "xq")
    _need(xs, torch.uint8, (T, H // 16), "xs")
    if out is None:
        out = alloc_permutation(T, E, k, H, dev)
    if workspace is None:
        workspace = alloc_prepare_workspace(T, E, k, dev)
    _need(workspace, torch.uint8, name="workspace")
    _check(_lib.moe_prepare(_ptr(logits), _ptr(bias), _ptr(x), T, E, k, k_primary, H, SCORE[score_fn],
                            int(bool(renormalize)),
                            _ptr(topk_idx), _ptr(topk_w), _ptr(x_gscale), _ptr(xq), _ptr(xs), _ptr(out.counts),
                            _ptr(out.offsets), _ptr(out.row_offsets), _ptr(out.perm_to_flat),
                            _ptr(out.flat_to_perm), _ptr(out.a_packed), _ptr(out.a_scales), _ptr(workspace),
                            workspace.numel(), _stream()),
           "moe_prepare")
    return topk_idx, topk_w, x_gscale, xq, xs, out


def moe_prepare_mxfp4(logits, x, k, score_fn="sigmoid", renormalize=True, bias=None, topk_idx=None, topk_w=None,
                      xq=None, xs=None, out: Permutation = None, workspace=None, k_primary=None):
    """moe_prepare for MXFP4: returns (topk_idx, topk_w, xq, xs [T, H/32], Permutation)."""
    k_primary = k if k_primary is None else int(k_primary)
    _need(logits, torch.float32, name="logits")
    _need(x, torch.bfloat16, name="x")
    T, E = logits.shape
    H = x.shape[1]
    dev = x.device
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    topk_idx = _empty((T, k), torch.int32, dev) if topk_idx is None else topk_idx
    topk_w = _empty((T, k), torch.float32, dev) if topk_w is None else topk_w
    xq = _empty((T, H // 2), torch.uint8, dev) if xq is None else xq
    xs = _empty((T, H // 32), torch.uint8, dev) if xs is None else xs
    _need(topk_idx, torch.int32, (T, k), "topk_idx")
    _need(topk_w, torch.float32, (T, k), "topk_w")
    _need(xq, torch.uint8, (T, H // 2), "xq")
    _need(xs, torch.uint8, (T, H // 32), "xs")
    if out is None:
        out = alloc_permutation(T, E, k, H, dev, "mxfp4")
    if workspace is None:
        workspace = alloc_prepare_workspace(T, E, k, dev)
    _need(workspace, torch.uint8, name="workspace")
    _check(_lib.moe_prepare_mxfp4(_ptr(logits), _ptr(bias), _ptr(x), T, E, k, k_primary, H, SCORE[score_fn],
                                  int(bool(renormalize)), _ptr(topk_idx), _ptr(topk_w), _ptr(xq), _ptr(xs),
                                  _ptr(out.counts), _ptr(out.offsets), _ptr(out.row_offsets), _ptr(out.perm_to_flat),
                                  _ptr(out.flat_to_perm), _ptr(out.a_packed), _ptr(out.a_scales), _ptr(workspace),
                                  workspace.numel(), _stream()),
           "moe_prepare_mxfp4")
    return topk_idx, topk_w, xq, xs, out


# ---- a4/a5 ---------------------------------------------------------------------
def gemm_tile_choice(E, N, m_total, tile_n=0):
    """The tile orientation a grouped GEMM call runs (see the header)."""
    return int(_lib.nvfp4moe_gemm_tile_choice(int(E), int(N), int(m_total), int(tile_n)))



def alloc_gemm_workspace(device):
    """Zero-filled tile-scheduler workspace for the grouped GEMMs (dynamic schedule)."""
    return torch.zeros((int(_lib.moe_grouped_gemm_nvfp4_workspace_size(1, 128, 64, EPI_BF16)),), dtype=torch.uint8,
                       device=device)


def _ws_args(workspace):
    if workspace is None:
        return None, 0
    _need(workspace, torch.uint8, name="workspace")
    return _ptr(workspace), workspace.numel()


ALL_ROWS = (1, 2 ** 31 - 1)


def moe_grouped_gemm_nvfp4(a_packed, a_scales, a_gscale, counts, row_offsets, w_packed, w_scales, w_gscale,
                           epilogue=EPI_BF16, c_gscale=None, m_total=None, tile_n=0, out=None, out_scales=None,
                           workspace=None, rows=ALL_ROWS):
    """Returns c_out (and c_scales for EPI_SWIGLU_NVFP4).  workspace: a zeroed
    alloc_gemm_workspace() for the dynamic tile schedule, None for static.
    w_packed: row-major [E, N, K/2] or TiledWeights.  m_total: the routed
    rows (T*k), not the padded capacity; it picks the tile orientation.
    rows = (min_rows, max_rows): only experts with that many rows
    (moe_grouped_gemm_nvfp4_range); the default covers every expert."""
    if m_total is None:
        raise ValueError("m_total (the routed rows, T*k) is required: it chooses the tile orientation")
    E, N, K, w_ptr, w_layout = _weights_args(w_packed)
    cap = a_packed.shape[0]
    dev = a_packed.device
    _need(a_packed, torch.uint8, (cap, K // 2), "a_packed")
    _need(a_scales, torch.uint8, name="a_scales")
    _need(a_gscale, torch.float32, (1,), "a_gscale")
    _need(counts, torch.int32, (E,), "counts")
    _need(row_offsets, torch.int32, (E + 1,), "row_offsets")
    _need(w_scales, torch.uint8, name="w_scales")
    _need(w_gscale, torch.float32, (E,), "w_gscale")
    if a_scales.numel() < blocked_scales_bytes(cap, K) or w_scales.numel() < E * blocked_scales_bytes(N, K):
        raise ValueError("scale buffers smaller than the blocked layout needs")
    if epilogue == EPI_BF16:
        if out is None:
            out = _empty((cap, N), torch.bfloat16, dev)
        _need(out, torch.bfloat16, (cap, N), "out")
    elif epilogue == EPI_SWIGLU_NVFP4:
        I = N // 2
        if out is None:
            out = _empty((cap, I // 2), torch.uint8, dev)
        if out_scales is None:
            out_scales = _empty((blocked_scales_bytes(cap, I),), torch.uint8, dev)
        _need(out, torch.uint8, (cap, I // 2), "out")
        _need(out_scales, torch.uint8, name="out_scales")
        _need(c_gscale, torch.float32, (1,), "c_gscale")
    elif epilogue == EPI_SWIGLU_F32:
        if out is None:
            out = _empty((cap, N // 2), torch.float32, dev)
        _need(out, torch.float32, (cap, N // 2), "out")
    else:
        raise ValueError(f"epilogue {epilogue}")
    ws_p, ws_n = _ws_args(workspace)
    args = (_ptr(a_packed), _ptr(a_scales), _ptr(a_gscale), _ptr(counts), _ptr(row_offsets), E, cap, int(m_total),
            w_ptr, _ptr(w_scales), _ptr(w_gscale), N, K, epilogue, _ptr(c_gscale), _ptr(out), _ptr(out_scales),
            int(tile_n), w_layout)
    if tuple(rows) == ALL_ROWS:
        _check(_lib.moe_grouped_gemm_nvfp4(*args, ws_p, ws_n, _stream()), "moe_grouped_gemm_nvfp4")
    else:
        _check(_lib.moe_grouped_gemm_nvfp4_range(*args, int(rows[0]), int(rows[1]), ws_p, ws_n, _stream()),
               "moe_grouped_gemm_nvfp4_range")
    return (out, out_scales) if epilogue == EPI_SWIGLU_NVFP4 else out


def moe_grouped_gemm_mxfp4(a_packed, a_scales, counts, row_offsets, w_packed, w_scales, epilogue=EPI_BF16,
                           m_total=None, tile_n=0, out=None, out_scales=None, workspace=None, rows=ALL_ROWS):
    """MXFP4 grouped GEMM.  Returns c_out (and c_scales for EPI_SWIGLU_MXFP4).
    w_packed: row-major [E, N, K/2] or TiledWeights."""
    if m_total is None:
        raise ValueError("m_total (the routed rows, T*k) is required: it chooses the tile orientation")
    E, N, K, w_ptr, w_layout = _weights_args(w_packed)
    cap = a_packed.shape[0]
    dev = a_packed.device
    _need(a_packed, torch.uint8, (cap, K // 2), "a_packed")
    _need(a_scales, torch.uint8, name="a_scales")
    _need(counts, torch.int32, (E,), "counts")
    _need(row_offsets, torch.int32, (E + 1,), "row_offsets")
    _need(w_scales, torch.uint8, name="w_scales")
    if a_scales.numel() < blocked_scales_bytes(cap, K, "mxfp4") or \
            w_scales.numel() < E * blocked_scales_bytes(N, K, "mxfp4"):
        raise ValueError("scale buffers smaller than the MXFP4 blocked layout needs")
    if epilogue == EPI_BF16:
        out = _empty((cap, N), torch.bfloat16, dev) if out is None else out
        _need(out, torch.bfloat16, (cap, N), "out")
    elif epilogue == EPI_SWIGLU_MXFP4:
        I = N // 2
        out = _empty((cap, I // 2), torch.uint8, dev) if out is None else out
        out_scales = _empty((blocked_scales_bytes(cap, I, "mxfp4"),), torch.uint8, dev) if out_scales is None \
            else out_scales
        _need(out, torch.uint8, (cap, I // 2), "out")
        _need(out_scales, torch.uint8, name="out_scales")
    elif epilogue == EPI_SWIGLU_F32:
        out = _empty((cap, N // 2), torch.float32, dev) if out is None else out
        _need(out, torch.float32, (cap, N // 2), "out")
    else:
        raise ValueError(f"epilogue {epilogue}")
    ws_p, ws_n = _ws_args(workspace)
    args = (_ptr(a_packed), _ptr(a_scales), _ptr(counts), _ptr(row_offsets), E, cap, int(m_total), w_ptr,
            _ptr(w_scales), N, K, epilogue, _ptr(out), _ptr(out_scales), int(tile_n), w_layout)
    if tuple(rows) == ALL_ROWS:
        _check(_lib.moe_grouped_gemm_mxfp4(*args, ws_p, ws_n, _stream()), "moe_grouped_gemm_mxfp4")
    else:
        _check(_lib.moe_grouped_gemm_mxfp4_range(*args, int(rows[0]), int(rows[1]), ws_p, ws_n, _stream()),
               "moe_grouped_gemm_mxfp4_range")
    return (out, out_scales) if epilogue == EPI_SWIGLU_MXFP4 else out


def moe_grouped_gemm_nvfp4_finalize(a_packed, a_scales, a_gscale, counts, row_offsets, w_packed, w_scales, w_gscale,
                                    perm_to_flat, topk_w, out_f32, m_total=None, tile_n=0, workspace=None,
                                    rows=ALL_ROWS):
    """Down projection with the finalize fused into its epilogue: adds
    topk_w[f] * bf16(Y[r]) into out_f32[f // k] (float32 atomics, so the
    order of a token's k additions is not fixed).  out_f32 [T, N] must be
    zero (moe_finalize_f32 leaves it so).  Returns out_f32."""
    if m_total is None:
        raise ValueError("m_total (the routed rows, T*k) is required: it chooses the tile orientation")
    E, N, K, w_ptr, w_layout = _weights_args(w_packed)
    cap = a_packed.shape[0]
    T, k = topk_w.shape
    _need(a_packed, torch.uint8, (cap, K // 2), "a_packed")
    _need(a_scales, torch.uint8, name="a_scales")
    _need(a_gscale, torch.float32, (1,), "a_gscale")
    _need(counts, torch.int32, (E,), "counts")
    _need(row_offsets, torch.int32, (E + 1,), "row_offsets")
    _need(w_scales, torch.uint8, name="w_scales")
    _need(w_gscale, torch.float32, (E,), "w_gscale")
    _need(perm_to_flat, torch.int32, (cap,), "perm_to_flat")
    _need(topk_w, torch.float32, name="topk_w")
    _need(out_f32, torch.float32, (T, N), "out_f32")
    ws_p, ws_n = _ws_args(workspace)
    _check(_lib.moe_grouped_gemm_nvfp4_finalize(_ptr(a_packed), _ptr(a_scales), _ptr(a_gscale), _ptr(counts),
                                                _ptr(row_offsets), E, cap, int(m_total), w_ptr, _ptr(w_scales),
                                                _ptr(w_gscale), N, K, _ptr(perm_to_flat), _ptr(topk_w), T, k,
                                                _ptr(out_f32), int(tile_n), w_layout, int(rows[0]), int(rows[1]),
                                                ws_p, ws_n, _stream()),
           "moe_grouped_gemm_nvfp4_finalize")
    return out_f32


def moe_finalize_f32(acc_f32, out=None):
    """out = bf16(acc_f32), and acc_f32 zeroed for the next fused finalize."""
    _need(acc_f32, torch.float32, name="acc_f32")
    T, H = acc_f32.shape
    if out is None:
        out = _empty((T, H), torch.bfloat16, acc_f32.device)
    _need(out, torch.bfloat16, (T, H), "out")
    _check(_lib.moe_finalize_f32(_ptr(acc_f32), T, H, _ptr(out), _stream()), "moe_finalize_f32")
    return out


# ---- a6 ------------------------------------------------------------------------
def moe_finalize(y, flat_to_perm, topk_w, out=None):
    _need(y, torch.bfloat16, name="y")
    T, k = topk_w.shape
    cap, H = y.shape
    _need(flat_to_perm, torch.int32, (T * k,), "flat_to_perm")
    _need(topk_w, torch.float32, name="topk_w")
    if out is None:
        out = _empty((T, H), torch.bfloat16, y.device)
    _need(out, torch.bfloat16, (T, H), "out")
    _check(_lib.moe_finalize(_ptr(y), _ptr(flat_to_perm), _ptr(topk_w), T, k, H, cap, _ptr(out), _stream()),
           "moe_finalize")
    return out


# ---- the whole layer -------------------------------------------------------------
class MoELayer:
    """Quantised expert weights plus every buffer of one layer shape.

    forward() enqueues the layer on the current stream.  Buffers are
    allocated for one batch size T (at construction when T is given, else at
    the first call, and again when T changes); otherwise forward() allocates
    nothing, and the tensor it returns is overwritten by the next call
    unless the caller passes `out`.  With fused_prepare (the default):
    moe_prepare (route + quantise + permute; moe_prepare_mxfp4 for
    fmt="mxfp4"), the gate/up GEMM with SwiGLU and requantisation, the down
    GEMM and finalize -- otherwise the six separate calls.

    Each grouped GEMM runs a launch plan: a list of (tile_n, (min_rows,
    max_rows)) launches that together cover every expert.  With autotune
    (the default when tile_n is (0, 0)) the first forward() of a batch size
    times the candidate plans (autotune()) on that batch and keeps the
    fastest for the batch size: it synchronises the stream, so make that
    first call outside stream capture.  Otherwise each GEMM is one launch
    with the given tile_n."""

    def __init__(self, w_gu, w_d, k, score_fn="sigmoid", renormalize=True, h_scale=2.0 ** -4, bias=None,
                 T=None, tile_n=(0, 0), fused_prepare=True, k_primary=None, fmt="nvfp4", dynamic_schedule=True,
                 tiled_weights=True, autotune=True, fused_finalize=False):
        if fmt not in ("nvfp4", "mxfp4"):
            raise ValueError(f"fmt {fmt}")
        self.fmt = fmt
        # one zeroed tile-scheduler workspace for both GEMMs (they run in sequence)
        self.g_ws = alloc_gemm_workspace(w_gu.device) if dynamic_schedule else None
        self.fused_prepare = bool(fused_prepare)
        # batch-aware routing when k_primary < k (moe_route_batch_aware)
        self.k_primary = k if k_primary is None else int(k_primary)
        self.E, two_i, self.H = w_gu.shape
        self.I = two_i // 2
        self.k, self.score_fn, self.renormalize = k, score_fn, renormalize
        self.device = w_gu.device
        self.bias = bias
        self.tile_n = tuple(tile_n)
        # Finalize fused into the down GEMM (NVFP4): float32 atomics into a
        # zeroed [T, H] accumulator, then one conversion kernel; the order of a
        # token's k additions is not fixed, so the output is not
        # bit-reproducible.  Off by default.
        if fused_finalize and fmt != "nvfp4":
            raise ValueError("the fused finalize is built for NVFP4 layers")
        self.fused_finalize = bool(fused_finalize)
        self.autotune_enabled = bool(autotune) and self.tile_n == (0, 0)
        self.plans = {}          # batch size -> (gate/up plan, down plan), from autotune()
        if fmt == "mxfp4":
            self.w_gu_packed, self.w_gu_scales = quantize_expert_weights_mx(w_gu)
            self.w_d_packed, self.w_d_scales = quantize_expert_weights_mx(w_d)
            self.w_gu_gscale = self.w_d_gscale = None
        else:
            self.w_gu_packed, self.w_gu_scales, self.w_gu_gscale = quantize_expert_weights(w_gu)
            self.w_d_packed, self.w_d_scales, self.w_d_gscale = quantize_expert_weights(w_d)
        # Tiled weights: each GEMM weight box is one contiguous 16 KB block, which
        # streams faster from HBM (the row-major copies are freed).
        if tiled_weights:
            self.w_gu_packed = tile_expert_weights(self.w_gu_packed)
            self.w_d_packed = tile_expert_weights(self.w_d_packed)
        self.h_scale = torch.full((1,), h_scale, dtype=torch.float32, device=self.device)
        self.T = None
        if T is not None:
            self._alloc(T)

    def _alloc(self, T):
        dev, E, k, H, I = self.device, self.E, self.k, self.H, self.I
        self.T = T
        self.topk_idx = _empty((T, k), torch.int32, dev)
        self.topk_w = _empty((T, k), torch.float32, dev)
        self.x_gscale = _empty((1,), torch.float32, dev)
        self.xq = _empty((T, H // 2), torch.uint8, dev)
        self.xs = _empty((T, H // (32 if self.fmt == "mxfp4" else 16)), torch.uint8, dev)
        self.q_ws = _empty((max(1, int(_lib.moe_quantize_nvfp4_workspace_size(T, H, QUANT_COMPUTE_GLOBAL))),),
                           torch.uint8, dev)
        self.r_ws = _empty((int(_lib.moe_route_batch_aware_workspace_size(E)),), torch.uint8, dev)
        self.perm = alloc_permutation(T, E, k, H, dev, self.fmt)
        self.p_ws = _empty((moe_permute_workspace_size(T, E, k),), torch.uint8, dev)
        self.prep_ws = alloc_prepare_workspace(T, E, k, dev)
        cap = self.perm.rows_capacity
        self.hq = _empty((cap, I // 2), torch.uint8, dev)
        self.hs = _empty((blocked_scales_bytes(cap, I, self.fmt),), torch.uint8, dev)
        self.y = None if self.fused_finalize else _empty((cap, H), torch.bfloat16, dev)
        self.acc = torch.zeros((T, H), dtype=torch.float32, device=dev) if self.fused_finalize else None
        self.out = _empty((T, H), torch.bfloat16, dev)

    # ---- the steps of forward() (bench.py times them one by one) ----
    def prepare(self, x, logits):
        """a1-a3: routing, quantisation of x and the permutation."""
        p = self.perm
        if self.fmt == "mxfp4":
            if self.fused_prepare:
                moe_prepare_mxfp4(logits, x, self.k, self.score_fn, self.renormalize, self.bias, self.topk_idx,
                                  self.topk_w, self.xq, self.xs, out=p, workspace=self.prep_ws, k_primary=self.k_primary)
            else:
                self._route(logits)
                moe_quantize_mxfp4(x, packed=self.xq, scales=self.xs)
                moe_permute_mxfp4(self.topk_idx, self.E, self.xq, self.xs, out=p, workspace=self.p_ws)
            return
        if self.fused_prepare:
            moe_prepare(logits, x, self.k, self.score_fn, self.renormalize, self.bias, self.topk_idx, self.topk_w,
                        self.x_gscale, self.xq, self.xs, out=p, workspace=self.prep_ws, k_primary=self.k_primary)
        else:
            self._route(logits)
            moe_quantize_nvfp4(x, global_scale=self.x_gscale, compute_global=True, packed=self.xq,
                               scales=self.xs, workspace=self.q_ws)
            moe_permute(self.topk_idx, self.E, self.xq, self.xs, out=p, workspace=self.p_ws)

    def plan(self, T=None):
        """(gate/up plan, down plan) of batch size T: lists of (tile_n, (min_rows, max_rows))."""
        T = self.T if T is None else T
        if T in self.plans:
            return self.plans[T]
        return [(self.tile_n[0], ALL_ROWS)], [(self.tile_n[1], ALL_ROWS)]

    def _gemm(self, which, tile_n, rows):
        p, m_total = self.perm, self.T * self.k
        if which == "gate_up":
            if self.fmt == "mxfp4":
                moe_grouped_gemm_mxfp4(p.a_packed, p.a_scales, p.counts, p.row_offsets, self.w_gu_packed,
                                       self.w_gu_scales, EPI_SWIGLU_MXFP4, m_total=m_total, tile_n=tile_n,
                                       out=self.hq, out_scales=self.hs, workspace=self.g_ws, rows=rows)
            else:
                moe_grouped_gemm_nvfp4(p.a_packed, p.a_scales, self.x_gscale, p.counts, p.row_offsets,
                                       self.w_gu_packed, self.w_gu_scales, self.w_gu_gscale, EPI_SWIGLU_NVFP4,
                                       c_gscale=self.h_scale, m_total=m_total, tile_n=tile_n, out=self.hq,
                                       out_scales=self.hs, workspace=self.g_ws, rows=rows)
        elif self.fused_finalize:
            moe_grouped_gemm_nvfp4_finalize(self.hq, self.hs, self.h_scale, p.counts, p.row_offsets, self.w_d_packed,
                                            self.w_d_scales, self.w_d_gscale, p.perm_to_flat, self.topk_w, self.acc,
                                            m_total=m_total, tile_n=tile_n, workspace=self.g_ws, rows=rows)
        elif self.fmt == "mxfp4":
            moe_grouped_gemm_mxfp4(self.hq, self.hs, p.counts, p.row_offsets, self.w_d_packed, self.w_d_scales,
                                   EPI_BF16, m_total=m_total, tile_n=tile_n, out=self.y, workspace=self.g_ws,
                                   rows=rows)
        else:
            moe_grouped_gemm_nvfp4(self.hq, self.hs, self.h_scale, p.counts, p.row_offsets, self.w_d_packed,
                                   self.w_d_scales, self.w_d_gscale, EPI_BF16, m_total=m_total, tile_n=tile_n,
                                   out=self.y, workspace=self.g_ws, rows=rows)

    def gemm_gate_up(self, plan=None):
        """a4: gate/up GEMM with the fused SwiGLU + requantisation, by launch plan."""
        for tile_n, rows in (self.plan()[0] if plan is None else plan):
            self._gemm("gate_up", tile_n, rows)

    def gemm_down(self, plan=None):
        """a5: down GEMM to bf16, by launch plan."""
        for tile_n, rows in (self.plan()[1] if plan is None else plan):
            self._gemm("down", tile_n, rows)

    def finalize(self, out=None):
        """a6: the router-weighted sum back to token order (fused finalize:
        the conversion of the float32 accumulator, which it zeroes)."""
        if self.fused_finalize:
            return moe_finalize_f32(self.acc, out=self.out if out is None else out)
        return moe_finalize(self.y, self.perm.flat_to_perm, self.topk_w, out=self.out if out is None else out)

    def forward(self, x, logits, out=None):
        T = x.shape[0]
        if self.T != T:
            self._alloc(T)
        if self.autotune_enabled and T not in self.plans:
            self.autotune(x, logits)
        self.prepare(x, logits)
        self.gemm_gate_up()
        self.gemm_down()
        return self.finalize(out)

    __call__ = forward

    def capture(self, x, logits, stream=None):
        """Captures one forward() on the tensors x and logits into a CUDA
        graph and returns it; graph.replay() then runs the whole layer (every
        kernel launch of prepare, both GEMM plans and finalize) with no host
        work per step, reading x and logits where they are and writing
        self.out.  Copy each step's inputs into x and logits before replaying.
        The launch plans for x's batch size are chosen first (autotune, which
        synchronises); nothing in forward() synchronises or allocates, so the
        capture holds exactly the eager launches."""
        T = x.shape[0]
        if self.T != T:
            self._alloc(T)
        if self.autotune_enabled and T not in self.plans:
            self.autotune(x, logits)
        side = torch.cuda.Stream(device=self.device) if stream is None else stream
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            self.forward(x, logits)      # one eager step on the capture stream first
            side.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                self.forward(x, logits)
        torch.cuda.current_stream(self.device).wait_stream(side)
        return graph

    # ---- tile autotuner ----
    def candidate_plans(self, which, T=None):
        """Launch plans the autotuner times for one GEMM at batch size T: one
        launch per orientation (the automatic choice, weight rows as M,
        token-major, token-major on CTA pairs), and splits that run experts
        with at least h rows token-major (single SM or pairs) and the rest
        with weight rows as M."""
        T = self.T if T is None else T
        N = 2 * self.I if which == "gate_up" else self.H
        plans = [[(0, ALL_ROWS)], [(128, ALL_ROWS)]]
        if N % 256 == 0:
            plans += [[(TILE_TOKEN_MAJOR, ALL_ROWS)], [(TILE_TOKEN_MAJOR_PAIR, ALL_ROWS)]]
            for h in (32, 128, 512):
                if T * self.k >= h:
                    for tm in (TILE_TOKEN_MAJOR, TILE_TOKEN_MAJOR_PAIR):
                        plans.append([(tm, (h, ALL_ROWS[1])), (128, (1, h))])
        return plans

    def autotune(self, x, logits, reps=5):
        """Times every candidate plan of both GEMMs on this batch (CUDA events,
        median of `reps` launches after one warm-up) and keeps the fastest for
        x's batch size; returns {"gate_up": (plan, ms), "down": (plan, ms)}.
        Every plan computes the same outputs (up to float32 summation order);
        only the launch configuration differs.  Synchronises the stream."""
        T = x.shape[0]
        if self.T != T:
            self._alloc(T)
        self.prepare(x, logits)
        chosen, report = [], {}
        for which, run in (("gate_up", self.gemm_gate_up), ("down", self.gemm_down)):
            best = None
            for plan in self.candidate_plans(which, T):
                times = []
                for i in range(reps + 1):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    run(plan)
                    e1.record()
                    e1.synchronize()
                    if i:
                        times.append(e0.elapsed_time(e1))
                ms = sorted(times)[len(times) // 2]
                if best is None or ms < best[1]:
                    best = (plan, ms)
            if which == "gate_up":
                run(best[0])             # the down GEMM's input, from the chosen plan
            chosen.append(best[0])
            report[which] = best
        if self.fused_finalize:
            self.acc.zero_()         # the timed down GEMMs added into the accumulator
        sync_status()
        self.plans[T] = tuple(chosen)
        return report

    def _route(self, logits):
        if self.k_primary < self.k:
            moe_route_batch_aware(logits, self.k, self.k_primary, self.score_fn, self.renormalize, self.bias,
                                  self.topk_idx, self.topk_w, workspace=self.r_ws)
        else:
            moe_route_topk(logits, self.k, self.score_fn, self.renormalize, self.bias, self.topk_idx, self.topk_w)

    # kernels launched by one forward(): fused prepare 1 (else route 1-2, quantise 1-2, permute 3),
    # one per launch of each GEMM plan, finalize 1
    @property
    def launches_per_forward(self):
        gu, down = self.plan()
        if self.fused_prepare:
            head = 1
        else:
            route = 2 if self.k_primary < self.k else 1
            quantise = 1 if self.fmt == "mxfp4" else 2
            head = route + quantise + 3
        return head + len(gu) + len(down) + 1
