"""Python binding of libfp8blk (block-scaled FP8 linear algebra on GB300).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libfp8blk.so`` behind its C ABI (``include/fp8blk.h``). PyTorch
allocates device memory and supplies the current stream. There is no CPU or
PyTorch fallback: if the library is missing every call raises.

Names follow the DeepSeek-V3 inference kernels ("Administrator & Developer
Guide", 8.5 The Triton kernels): act_quant, weight_dequant, fp8_gemm, plus
the FP8 linear layer of 6.3 and the block weight quantisation of the README's
weight_scale_inv section.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

__all__ = [
    "SCALE_FP32", "SCALE_UE8M0", "SCALE_PROMOTE", "BLOCK", "lib", "lib_path", "header_functions", "Fp8BlkError",
    "act_quant", "weight_quant", "weight_dequant", "fp8_gemm", "linear", "linear_host",
    "gemm_workspace_bytes", "linear_workspace_bytes", "linear_host_workspace_bytes", "linear_kernels",
    "last_device_error",
    "swiglu_gemm", "ffn", "moe_permute", "moe_workspace_bytes", "moe_grouped_gemm", "moe_gate", "moe_route",
]

SCALE_FP32 = 0
SCALE_UE8M0 = 1
SCALE_PROMOTE = 0x10   # | SCALE_UE8M0: GEMMs keep the per-block promotion
BLOCK = 128

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
HEADER = os.path.join(_ROOT, "include", "fp8blk.h")
_LIB_PATH = os.path.join(_PKG, "libfp8blk.so")
_lib = None
_lib_lock = threading.Lock()


class Fp8BlkError(RuntimeError):
    pass


def lib_path() -> str:
    return _LIB_PATH


def header_functions() -> list[str]:
    """Names of the functions the public header declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"FP8BLK_API\s+[\w\s\*]*?\b(fp8blk_\w+)\s*\(", text)))


def lib():
    """The loaded libfp8blk (ctypes). Raises if it has not been built."""
    global _lib
    with _lib_lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise Fp8BlkError(f"{_LIB_PATH} is missing: build it with __graft_entry__.build() "
                                  "or python fp8_block_scaled_quant_gb300/_build.py")
            L = ctypes.CDLL(_LIB_PATH)
            vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
            L.fp8blk_status_string.argtypes = [i32]
            L.fp8blk_status_string.restype = ctypes.c_char_p
            L.fp8blk_version.argtypes = []
            L.fp8blk_version.restype = i32
            L.fp8blk_act_quant.argtypes = [vp, i64, i64, vp, vp, i32, vp]
            L.fp8blk_weight_quant.argtypes = [vp, i64, i64, vp, vp, i32, vp]
            L.fp8blk_weight_dequant.argtypes = [vp, vp, i64, i64, vp, vp]
            L.fp8blk_gemm_workspace_bytes.argtypes = [i64, i64, i64]
            L.fp8blk_gemm_workspace_bytes.restype = sz
            L.fp8blk_gemm.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, vp, sz, vp]
            L.fp8blk_linear_workspace_bytes.argtypes = [i64, i64, i64]
            L.fp8blk_linear_workspace_bytes.restype = sz
            L.fp8blk_linear.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, vp, sz, vp]
            L.fp8blk_linear_host_workspace_bytes.argtypes = [i64, i64, i64]
            L.fp8blk_linear_host_workspace_bytes.restype = sz
            L.fp8blk_linear_host.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, vp, sz, vp]
            L.fp8blk_linear_kernels.argtypes = [i64, i64, i64, ctypes.POINTER(i32)]
            L.fp8blk_last_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint)]
            for name in header_functions():
                if getattr(L, name).restype is ctypes.c_int:
                    getattr(L, name).restype = i32
            _lib = L
    return _lib


def _check(status: int, what: str):
    if status != 0:
        msg = lib().fp8blk_status_string(status).decode()
        raise Fp8BlkError(f"{what}: {msg} (status {status})")


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t: torch.Tensor, dtype, name: str, ndim: int = 2):
    if not t.is_cuda:
        raise Fp8BlkError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise Fp8BlkError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise Fp8BlkError(f"{name}: Input tensors must have {ndim} dimensions")
    if not t.is_contiguous():
        raise Fp8BlkError(f"{name}: Input tensor must be contiguous")


# ---- workspaces: zero-filled device buffers cached per (device, stream) ------

_ws_cache: dict = {}


def workspace(nbytes: int, device: torch.device, key: str = "gemm") -> torch.Tensor:
    """A zero-initialised uint8 device buffer of at least nbytes, reused by
    every call on the same device, stream and key. The GEMM leaves its
    counters at zero, so the buffer never needs clearing again."""
    stream = torch.cuda.current_stream(device).cuda_stream
    k = (device.index, stream, key)
    buf = _ws_cache.get(k)
    if buf is None or buf.numel() < nbytes:
        buf = torch.zeros(max(nbytes, 256) + 256, dtype=torch.uint8, device=device)
        _ws_cache[k] = buf
    off = (-buf.data_ptr()) % 256
    return buf[off:off + max(nbytes, 1)]


# ---- operations --------------------------------------------------------------

def act_quant(x: torch.Tensor, scale_fmt: int = SCALE_FP32, q: torch.Tensor | None = None,
              s: torch.Tensor | None = None):
    """x bf16 [M, K] -> (q float8_e4m3fn [M, K], s float32 [M, K/128])."""
    _need(x, torch.bfloat16, "x")
    M, K = x.shape
    if K % BLOCK:
        raise Fp8BlkError(f"Last dimension size must be divisible by block_size (block_size={BLOCK})")
    if q is None:
        q = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=x.device)
    if s is None:
        s = torch.empty((M, K // BLOCK), dtype=torch.float32, device=x.device)
    _check(lib().fp8blk_act_quant(_ptr(x), M, K, _ptr(q), _ptr(s), scale_fmt, _stream(x.device)), "act_quant")
    return q, s


def weight_quant(w: torch.Tensor, scale_fmt: int = SCALE_FP32):
    """w float32 [N, K] -> (q float8_e4m3fn [N, K], s float32 [ceil(N/128), ceil(K/128)])."""
    _need(w, torch.float32, "w")
    N, K = w.shape
    q = torch.empty((N, K), dtype=torch.float8_e4m3fn, device=w.device)
    s = torch.empty(((N + BLOCK - 1) // BLOCK, (K + BLOCK - 1) // BLOCK), dtype=torch.float32, device=w.device)
    _check(lib().fp8blk_weight_quant(_ptr(w), N, K, _ptr(q), _ptr(s), scale_fmt, _stream(w.device)),
           "weight_quant")
    return q, s


def weight_dequant(q: torch.Tensor, s: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """q float8_e4m3fn [N, K], s float32 [ceil(N/128), ceil(K/128)] -> bf16 [N, K]."""
    _need(q, torch.float8_e4m3fn, "q")
    _need(s, torch.float32, "s")
    N, K = q.shape
    if tuple(s.shape) != ((N + BLOCK - 1) // BLOCK, (K + BLOCK - 1) // BLOCK):
        raise Fp8BlkError("scale must have shape (ceil(N/128), ceil(K/128))")
    if out is None:
        out = torch.empty((N, K), dtype=torch.bfloat16, device=q.device)
    _check(lib().fp8blk_weight_dequant(_ptr(q), _ptr(s), N, K, _ptr(out), _stream(q.device)), "weight_dequant")
    return out


def gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().fp8blk_gemm_workspace_bytes(M, N, K))


def linear_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().fp8blk_linear_workspace_bytes(M, N, K))


def linear_host_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().fp8blk_linear_host_workspace_bytes(M, N, K))


def linear_kernels(M: int, N: int, K: int) -> int:
    """Kernels one linear() call of this shape launches on the current device:
    1 when act_quant runs inside the GEMM kernel, 2 when it is a kernel of its
    own, 0 for an empty problem."""
    n = ctypes.c_int(0)
    _check(lib().fp8blk_linear_kernels(M, N, K, ctypes.byref(n)), "linear_kernels")
    return n.value


def fp8_gemm(a: torch.Tensor, a_s: torch.Tensor, w: torch.Tensor, w_s: torch.Tensor,
             scale_fmt: int = SCALE_FP32, out: torch.Tensor | None = None,
             ws: torch.Tensor | None = None) -> torch.Tensor:
    """a e4m3 [M, K], a_s fp32 [M, K/128], w e4m3 [N, K], w_s fp32 [ceil(N/128), K/128] -> bf16 [M, N]."""
    _need(a, torch.float8_e4m3fn, "a")
    _need(w, torch.float8_e4m3fn, "w")
    _need(a_s, torch.float32, "a_s")
    _need(w_s, torch.float32, "w_s")
    M, K = a.shape
    N = w.shape[0]
    if w.shape[1] != K:
        raise Fp8BlkError("a and w must share K")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    nbytes = gemm_workspace_bytes(M, N, K)
    if ws is None:
        ws = workspace(nbytes, a.device)
    _check(lib().fp8blk_gemm(_ptr(a), _ptr(a_s), _ptr(w), _ptr(w_s), _ptr(out), M, N, K, scale_fmt, _ptr(ws),
                             ws.numel(), _stream(a.device)), "fp8_gemm")
    return out


def linear(x: torch.Tensor, w: torch.Tensor, w_s: torch.Tensor, scale_fmt: int = SCALE_FP32,
           out: torch.Tensor | None = None, ws: torch.Tensor | None = None) -> torch.Tensor:
    """FP8 linear layer: fp8_gemm(act_quant(x), w). x bf16 [M, K] -> bf16 [M, N]."""
    _need(x, torch.bfloat16, "x")
    _need(w, torch.float8_e4m3fn, "w")
    _need(w_s, torch.float32, "w_s")
    M, K = x.shape
    N = w.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = workspace(linear_workspace_bytes(M, N, K), x.device, "linear")
    _check(lib().fp8blk_linear(_ptr(x), _ptr(w), _ptr(w_s), _ptr(out), M, N, K, scale_fmt, _ptr(ws), ws.numel(),
                               _stream(x.device)), "linear")
    return out


def linear_host(x_host: torch.Tensor, w: torch.Tensor, w_s: torch.Tensor, y_host: torch.Tensor,
                scale_fmt: int = SCALE_FP32, ws: torch.Tensor | None = None) -> torch.Tensor:
    """The FP8 linear layer on host bf16 buffers, enqueued on the current stream of
    w's device: pinned buffers are read and written in place by the kernels,
    pageable ones are copied in and out. y_host is valid after that stream is
    synchronised."""
    if x_host.is_cuda or y_host.is_cuda:
        raise Fp8BlkError("x_host and y_host must be host tensors")
    if x_host.dtype != torch.bfloat16 or y_host.dtype != torch.bfloat16:
        raise Fp8BlkError("x_host and y_host must be bf16")
    if not (x_host.is_contiguous() and y_host.is_contiguous()):
        raise Fp8BlkError("Input tensor must be contiguous")
    _need(w, torch.float8_e4m3fn, "w")
    M, K = x_host.shape
    N = w.shape[0]
    if tuple(y_host.shape) != (M, N):
        raise Fp8BlkError("y_host must be [M, N]")
    if ws is None:
        ws = workspace(linear_host_workspace_bytes(M, N, K), w.device, "linear_host")
    _check(lib().fp8blk_linear_host(_ptr(x_host), _ptr(w), _ptr(w_s), _ptr(y_host), M, N, K, scale_fmt, _ptr(ws),
                                    ws.numel(), _stream(w.device)), "linear_host")
    return y_host


def last_device_error(device: torch.device | None = None) -> int:
    """Synchronises the current stream and returns (and clears) the device
    error bits: 0 when no kernel gave up waiting."""
    device = device or torch.device("cuda", torch.cuda.current_device())
    bits = ctypes.c_uint(0)
    st = lib().fp8blk_last_device_error(_stream(device), ctypes.byref(bits))
    if st not in (0, 6):
        _check(st, "last_device_error")
    return int(bits.value)


# ---- SwiGLU FFN and routed experts -------------------------------------------

def _set_types(name, argtypes, restype=ctypes.c_int):
    f = getattr(lib(), name)
    f.argtypes = argtypes
    f.restype = restype
    return f


def swiglu_gemm(x: torch.Tensor, x_s: torch.Tensor, w1: torch.Tensor, w1_s: torch.Tensor, w3: torch.Tensor,
                w3_s: torch.Tensor, scale_fmt: int = SCALE_FP32, ws: torch.Tensor | None = None):
    """act_quant(bf16(silu(bf16(x w1^T))) * bf16(x w3^T)) -> (u float8_e4m3fn [M, inter], u_s float32 [M, inter/128])."""
    for t, n, dt in ((x, "x", torch.float8_e4m3fn), (w1, "w1", torch.float8_e4m3fn), (w3, "w3", torch.float8_e4m3fn),
                     (x_s, "x_s", torch.float32), (w1_s, "w1_s", torch.float32), (w3_s, "w3_s", torch.float32)):
        _need(t, dt, n)
    M, dim = x.shape
    inter = w1.shape[0]
    u = torch.empty((M, inter), dtype=torch.float8_e4m3fn, device=x.device)
    us = torch.empty((M, inter // BLOCK), dtype=torch.float32, device=x.device)
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    nb = _set_types("fp8blk_swiglu_workspace_bytes", [i64, i64, i64], sz)(M, inter, dim)
    if ws is None:
        ws = workspace(nb, x.device, "swiglu")
    f = _set_types("fp8blk_swiglu_gemm", [vp] * 8 + [i64, i64, i64, i32, vp, sz, vp])
    _check(f(_ptr(x), _ptr(x_s), _ptr(w1), _ptr(w1_s), _ptr(w3), _ptr(w3_s), _ptr(u), _ptr(us), M, inter, dim,
             scale_fmt, _ptr(ws), ws.numel(), _stream(x.device)), "swiglu_gemm")
    return u, us


def ffn_workspace_bytes(M: int, dim: int, inter: int) -> int:
    i64 = ctypes.c_int64
    return int(_set_types("fp8blk_ffn_workspace_bytes", [i64, i64, i64], ctypes.c_size_t)(M, dim, inter))


def ffn(x: torch.Tensor, w1, w1_s, w3, w3_s, w2, w2_s, scale_fmt: int = SCALE_FP32,
        out: torch.Tensor | None = None, ws: torch.Tensor | None = None) -> torch.Tensor:
    """Dense SwiGLU FFN with FP8 Linears: x bf16 [M, dim] -> bf16 [M, dim]."""
    _need(x, torch.bfloat16, "x")
    M, dim = x.shape
    inter = w1.shape[0]
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    nb = ffn_workspace_bytes(M, dim, inter)
    if ws is None:
        ws = workspace(nb, x.device, "ffn")
    if out is None:
        out = torch.empty((M, dim), dtype=torch.bfloat16, device=x.device)
    f = _set_types("fp8blk_ffn", [vp] * 8 + [i64, i64, i64, i32, vp, sz, vp])
    _check(f(_ptr(x), _ptr(w1), _ptr(w1_s), _ptr(w3), _ptr(w3_s), _ptr(w2), _ptr(w2_s), _ptr(out), M, dim, inter,
             scale_fmt, _ptr(ws), ws.numel(), _stream(x.device)), "ffn")
    return out


def moe_permute(topk_idx: torch.Tensor, E: int):
    """topk_idx int32 [T, topk] -> (counts int32 [E], offsets int32 [E+1], perm int32 [T*topk]);
    perm past offsets[E] is unspecified."""
    _need(topk_idx, torch.int32, "topk_idx")
    T, k = topk_idx.shape
    dev = topk_idx.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    nbytes = int(_set_types("fp8blk_moe_permute_workspace_bytes", [i64] * 3, sz)(T, k, E))
    ws = workspace(nbytes, dev, "moe_permute")
    f = _set_types("fp8blk_moe_permute", [vp, i64, i64, i64, vp, vp, vp, vp, sz, vp])
    _check(f(_ptr(topk_idx), T, k, E, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(ws), ws.numel(), _stream(dev)),
           "moe_permute")
    return counts, offsets, perm[: T * k]


def mla_absorb(inp: torch.Tensor, wkv_b: torch.Tensor, wkv_b_s: torch.Tensor, mode: str,
               out: torch.Tensor | None = None, dn: int = 128, dv: int = 128) -> torch.Tensor:
    """MLA absorb projections with the FP8 wkv_b (e4m3 [H*(dn+dv), C] + block scales).
    mode "qk": q_nope bf16 [T, H, dn] -> bf16 [T, H, C]; mode "v": x bf16 [T, H, C] -> bf16 [T, H, dv]."""
    _need(inp, torch.bfloat16, "inp", ndim=3)
    _need(wkv_b, torch.float8_e4m3fn, "wkv_b")
    _need(wkv_b_s, torch.float32, "wkv_b_s")
    T, H = inp.shape[0], inp.shape[1]
    C = wkv_b.shape[1]
    if out is None:
        out = torch.empty((T, H, C if mode == "qk" else dv), dtype=torch.bfloat16, device=inp.device)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    name = "fp8blk_mla_absorb_qk" if mode == "qk" else "fp8blk_mla_absorb_v"
    f = _set_types(name, [vp] * 4 + [i64] * 5 + [vp])
    _check(f(_ptr(inp), _ptr(wkv_b), _ptr(wkv_b_s), _ptr(out), T, H, dn, dv, C, _stream(inp.device)), name)
    return out


SCORE_SOFTMAX, SCORE_SIGMOID = 0, 1


def moe_gate(logits: torch.Tensor, bias: torch.Tensor | None = None, n_groups: int = 1, topk_groups: int = 1,
             topk: int = 8, score_func: int = SCORE_SIGMOID, route_scale: float = 1.0, normalize: bool = True,
             idx: torch.Tensor | None = None, w: torch.Tensor | None = None):
    """Gate logits fp32 [T, E] (+ bias fp32 [E]) -> (topk_idx int32 [T, topk],
    topk_w fp32 [T, topk]): scores, group-limited top-k, weights."""
    _need(logits, torch.float32, "logits")
    if bias is not None:
        _need(bias, torch.float32, "bias", ndim=1)
    T, E = logits.shape
    dev = logits.device
    if idx is None:
        idx = torch.empty((T, topk), dtype=torch.int32, device=dev)
    if w is None:
        w = torch.empty((T, topk), dtype=torch.float32, device=dev)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    f = _set_types("fp8blk_moe_gate", [vp, vp, i64, i64, i64, i64, i64, i32, ctypes.c_float, i32, vp, vp, vp])
    _check(f(_ptr(logits), _ptr(bias), T, E, n_groups, topk_groups, topk, score_func, float(route_scale),
             int(bool(normalize)), _ptr(idx), _ptr(w), _stream(dev)), "moe_gate")
    return idx, w


def moe_route(logits: torch.Tensor, bias: torch.Tensor | None = None, n_groups: int = 1, topk_groups: int = 1,
              topk: int = 8, score_func: int = SCORE_SIGMOID, route_scale: float = 1.0, normalize: bool = True,
              out=None):
    """Gate and routing permutation in one call: logits fp32 [T, E] (+ bias)
    -> (topk_idx int32 [T, topk], topk_w fp32 [T, topk], counts int32 [E],
    offsets int32 [E+1], perm int32 [T*topk]). `out` may pass those five
    tensors to be written in place."""
    _need(logits, torch.float32, "logits")
    if bias is not None:
        _need(bias, torch.float32, "bias", ndim=1)
    T, E = logits.shape
    dev = logits.device
    if out is None:
        out = (torch.empty((T, topk), dtype=torch.int32, device=dev),
               torch.empty((T, topk), dtype=torch.float32, device=dev),
               torch.empty(E, dtype=torch.int32, device=dev), torch.empty(E + 1, dtype=torch.int32, device=dev),
               torch.empty(max(T * topk, 1), dtype=torch.int32, device=dev))
    idx, w, counts, offsets, perm = out
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    nbytes = int(_set_types("fp8blk_moe_route_workspace_bytes", [i64] * 3, sz)(T, topk, E))
    ws = workspace(nbytes, dev, "moe_route")
    f = _set_types("fp8blk_moe_route", [vp, vp, i64, i64, i64, i64, i64, i32, ctypes.c_float, i32] + [vp] * 6 +
                   [sz, vp])
    _check(f(_ptr(logits), _ptr(bias), T, E, n_groups, topk_groups, topk, score_func, float(route_scale),
             int(bool(normalize)), _ptr(idx), _ptr(w), _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(ws), ws.numel(),
             _stream(dev)), "moe_route")
    return idx, w, counts, offsets, perm[: T * topk]


def moe_workspace_bytes(T: int, topk: int, E: int, dim: int, inter: int, n_shared: int = 0) -> int:
    i64 = ctypes.c_int64
    return int(_set_types("fp8blk_moe_workspace_bytes", [i64] * 6, ctypes.c_size_t)(T, topk, E, dim, inter, n_shared))


def moe_grouped_gemm(x: torch.Tensor, x_s: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor,
                     w1, w1_s, w3, w3_s, w2, w2_s, E: int, scale_fmt: int = SCALE_FP32,
                     out: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                     n_shared: int = 0) -> torch.Tensor:
    """Routed-expert SwiGLU FFN over stacked block-FP8 experts.
    x e4m3 [T, dim] (+ x_s), topk_idx int32 / topk_w fp32 [T, topk] (ids < E),
    w1/w3 e4m3 [(E+n_shared)*inter, dim], w2 e4m3 [(E+n_shared)*dim, inter] (+ block scales)
    -> bf16 [T, dim]; the last n_shared experts are shared (every token, weight 1, added as y + z)."""
    _need(x, torch.float8_e4m3fn, "x")
    _need(topk_idx, torch.int32, "topk_idx")
    _need(topk_w, torch.float32, "topk_w")
    T, dim = x.shape
    k = topk_idx.shape[1]
    inter = w2.shape[1]
    if ws is None:
        ws = workspace(moe_workspace_bytes(T, k, E, dim, inter, n_shared), x.device, "moe")
    if out is None:
        out = torch.empty((T, dim), dtype=torch.bfloat16, device=x.device)
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    f = _set_types("fp8blk_moe_grouped_gemm", [vp] * 11 + [i64] * 6 + [i32, vp, sz, vp])
    _check(f(_ptr(x), _ptr(x_s), _ptr(topk_idx), _ptr(topk_w), _ptr(w1), _ptr(w1_s), _ptr(w3), _ptr(w3_s),
             _ptr(w2), _ptr(w2_s), _ptr(out), T, k, E, dim, inter, n_shared, scale_fmt, _ptr(ws), ws.numel(),
             _stream(x.device)), "moe_grouped_gemm")
    return out
