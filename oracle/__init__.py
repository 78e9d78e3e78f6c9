"""CPU oracle for the block-scaled FP8 linear-algebra path.

TEST INFRASTRUCTURE ONLY. The functions here define what the CUDA library
must compute; they are plain, slow and single-threaded. Only the tests, the
smoke check (``__graft_entry__.smoke``) and the benchmark's CPU-baseline leg
may import this package. The library (``fp8_block_scaled_quant_gb300``)
never imports it and shares no code with it.

The arithmetic lives in ``fp8blk_oracle.c`` (plain C, fp64 where the pages
leave the precision free); this module only compiles it with gcc and calls it
through ctypes on numpy arrays. Each function cites the page passage it
follows in the C source.

Parity pins: every function is pinned by ``tests/test_oracle_*.py`` against
closed forms, invariants, a library routine (torch's CPU float8_e4m3fn and
bf16 casts, numpy fp64 matmul) or brute force on tiny inputs. No function is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8blk_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BLOCK = 128


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc into oracle/liboracle.so. IEEE semantics:
    no fast-math, no FMA contraction."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-frounding-math", _SRC, "-o", tmp, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_decode.restype = ctypes.c_double
            L.orc_e4m3_encode.argtypes = [ctypes.c_float]
            L.orc_e4m3_encode.restype = ctypes.c_uint8
            L.orc_bf16_encode.argtypes = [ctypes.c_double]
            L.orc_bf16_encode.restype = ctypes.c_uint16
            L.orc_bf16_decode.argtypes = [ctypes.c_uint16]
            L.orc_bf16_decode.restype = ctypes.c_double
            L.orc_block_scale.argtypes = [ctypes.c_float, i32]
            L.orc_block_scale.restype = ctypes.c_float
            L.orc_act_quant.argtypes = [vp, i64, i64, i32, vp, vp]
            L.orc_weight_quant.argtypes = [vp, i64, i64, i32, vp, vp]
            L.orc_weight_dequant.argtypes = [vp, vp, i64, i64, vp]
            L.orc_gemm.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp]
            L.orc_gemm_points.argtypes = [vp, vp, vp, vp, i64, vp, vp, i64, vp]
            L.orc_swiglu.argtypes = [vp, vp, i64, vp]
            L.orc_moe_permute.argtypes = [vp, i64, i64, i64, vp, vp, vp]
            L.orc_moe_permute.restype = i32
            L.orc_expert_ffn.argtypes = [vp] * 8 + [i64, i64, i32, vp]
            L.orc_expert_ffn.restype = i32
            L.orc_expert_ffn_u.argtypes = [vp] * 8 + [i64, i64, i32, vp, vp, vp]
            L.orc_expert_ffn_u.restype = i32
            L.orc_moe_token.argtypes = [vp, vp, vp, vp, i64, i64] + [vp] * 6 + [i64, i64, i32, i64, i64, vp]
            L.orc_moe_token.restype = i32
            L.orc_mla_absorb.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i32, vp]
            L.orc_moe_gate.argtypes = [vp, vp, i64, i64, i64, i64, i64, i32, ctypes.c_float, i32, vp, vp]
            L.orc_moe_gate.restype = i32
            L.orc_e4m3_encode_array.argtypes = [vp, i64, vp]
            L.orc_bf16_encode_array.argtypes = [vp, i64, vp]
            _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- scalar helpers -------------------------------------------------------

def e4m3_encode(v: float) -> int:
    return int(lib().orc_e4m3_encode(float(v)))


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    """e4m3 codes of float32 values (one oracle encode per element)."""
    v = _c(v, np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_decode(code: int) -> float:
    return float(lib().orc_e4m3_decode(int(code)))


def e4m3_decode_array(codes: np.ndarray) -> np.ndarray:
    """fp64 values of an array of e4m3 codes (one oracle call per code)."""
    table = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def bf16_encode(v: float) -> int:
    return int(lib().orc_bf16_encode(float(v)))


def block_scale(amax: float, ue8m0: bool) -> float:
    return float(lib().orc_block_scale(float(amax), int(bool(ue8m0))))


# ---- A1 act_quant ---------------------------------------------------------

def act_quant(x_bf16_bits: np.ndarray, ue8m0: bool = False):
    """x: uint16 bf16 bits [M, K], K % 128 == 0 -> (q uint8 [M, K], s float32 [M, K/128])."""
    x = _c(x_bf16_bits, np.uint16)
    M, K = x.shape
    if K % BLOCK:
        raise ValueError("Last dimension size must be divisible by block_size (128)")
    q = np.empty((M, K), np.uint8)
    s = np.empty((M, K // BLOCK), np.float32)
    lib().orc_act_quant(_ptr(x), M, K, int(bool(ue8m0)), _ptr(q), _ptr(s))
    return q, s


# ---- weight quantisation (synthetic inputs) ------------------------------

def weight_quant(w: np.ndarray, ue8m0: bool = False):
    """w: float32 [N, K] -> (q uint8 [N, K], s float32 [ceil(N/128), ceil(K/128)])."""
    w = _c(w, np.float32)
    N, K = w.shape
    q = np.empty((N, K), np.uint8)
    s = np.empty(((N + BLOCK - 1) // BLOCK, (K + BLOCK - 1) // BLOCK), np.float32)
    lib().orc_weight_quant(_ptr(w), N, K, int(bool(ue8m0)), _ptr(q), _ptr(s))
    return q, s


# ---- A3 weight_dequant ----------------------------------------------------

def weight_dequant(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """q uint8 [N, K], s float32 [ceil(N/128), ceil(K/128)] -> bf16 bits [N, K]."""
    q = _c(q, np.uint8)
    s = _c(s, np.float32)
    N, K = q.shape
    if s.shape != ((N + BLOCK - 1) // BLOCK, (K + BLOCK - 1) // BLOCK):
        raise ValueError("scale shape must be (ceil(N/128), ceil(K/128))")
    out = np.empty((N, K), np.uint16)
    lib().orc_weight_dequant(_ptr(q), _ptr(s), N, K, _ptr(out))
    return out


# ---- A2 fp8_gemm ------------------------------------------------------------

def gemm(qa, a_s, qw, w_s) -> np.ndarray:
    """fp64 reference of the block-scaled product, [M, N]."""
    qa, qw = _c(qa, np.uint8), _c(qw, np.uint8)
    a_s, w_s = _c(a_s, np.float32), _c(w_s, np.float32)
    M, K = qa.shape
    N = qw.shape[0]
    assert qw.shape[1] == K and K % BLOCK == 0
    assert a_s.shape == (M, K // BLOCK) and w_s.shape == ((N + BLOCK - 1) // BLOCK, K // BLOCK)
    out = np.empty((M, N), np.float64)
    lib().orc_gemm(_ptr(qa), _ptr(a_s), _ptr(qw), _ptr(w_s), M, N, K, _ptr(out))
    return out


def gemm_points(qa, a_s, qw, w_s, ms, ns) -> np.ndarray:
    """fp64 reference at the listed (ms[i], ns[i]) output elements."""
    qa, qw = _c(qa, np.uint8), _c(qw, np.uint8)
    a_s, w_s = _c(a_s, np.float32), _c(w_s, np.float32)
    ms, ns = _c(ms, np.int64), _c(ns, np.int64)
    K = qa.shape[1]
    out = np.empty(ms.shape[0], np.float64)
    lib().orc_gemm_points(_ptr(qa), _ptr(a_s), _ptr(qw), _ptr(w_s), K, _ptr(ms), _ptr(ns),
                          ms.shape[0], _ptr(out))
    return out


def bf16_round(ref: np.ndarray) -> np.ndarray:
    """bf16 bits of fp64 values, one rounding each (no double rounding)."""
    v = _c(ref, np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().orc_bf16_encode_array(_ptr(v), v.size, _ptr(out))
    return out


# ---- A4 SwiGLU ----------------------------------------------------------------

def swiglu(h1_bits, h3_bits) -> np.ndarray:
    h1, h3 = _c(h1_bits, np.uint16), _c(h3_bits, np.uint16)
    u = np.empty_like(h1)
    lib().orc_swiglu(_ptr(h1), _ptr(h3), h1.size, _ptr(u))
    return u


def ffn_rows(xq, xs, w1q, w1s, w3q, w3s, w2q, w2s, rows, ue8m0=False, return_u=False):
    """Dense SwiGLU FFN chain for the listed rows of an already-quantised x:
    h = bf16(w1 x), bf16(w3 x) -> swiglu -> act_quant -> fp64 product with w2.
    Returns fp64 [len(rows), dim_out]; with return_u also the quantised
    intermediate (uq uint8 [len(rows), inter], us float32 [len(rows), inter/128])."""
    xq, xs = _c(xq, np.uint8), _c(xs, np.float32)
    w1q, w3q, w2q = _c(w1q, np.uint8), _c(w3q, np.uint8), _c(w2q, np.uint8)
    w1s, w3s, w2s = _c(w1s, np.float32), _c(w3s, np.float32), _c(w2s, np.float32)
    dim = xq.shape[1]
    inter = w1q.shape[0]
    dout = w2q.shape[0]
    assert w2q.shape[1] == inter
    rows = list(rows)
    out = np.empty((len(rows), dout), np.float64)
    uq = np.empty((len(rows), inter), np.uint8)
    us = np.empty((len(rows), inter // BLOCK), np.float32)
    L = lib()
    for i, r in enumerate(rows):
        o = np.empty(dout, np.float64)
        xr = np.ascontiguousarray(xq[r])
        sr = np.ascontiguousarray(xs[r])
        if dout != dim:
            raise ValueError("the FFN maps dim -> dim")
        ur = np.empty(inter, np.uint8)
        sr_u = np.empty(inter // BLOCK, np.float32)
        rc = L.orc_expert_ffn_u(_ptr(xr), _ptr(sr), _ptr(w1q), _ptr(w1s), _ptr(w3q), _ptr(w3s),
                                _ptr(w2q), _ptr(w2s), dim, inter, int(bool(ue8m0)), _ptr(o), _ptr(ur), _ptr(sr_u))
        if rc:
            raise MemoryError("oracle expert FFN failed")
        out[i] = o
        uq[i] = ur
        us[i] = sr_u
    return (out, uq, us) if return_u else out


# ---- A5 MoE permutation --------------------------------------------------------

def moe_permute(idx: np.ndarray, E: int):
    """idx int32 [T, topk] -> (counts int32 [E], offsets int32 [E+1], perm int32 [T*topk])."""
    idx = _c(idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    rc = lib().orc_moe_permute(_ptr(idx), T, k, E, _ptr(counts), _ptr(offsets), _ptr(perm))
    if rc:
        raise ValueError("expert index out of range")
    return counts, offsets, perm


# ---- A6/A7 MoE output -----------------------------------------------------------

def moe_tokens(xq, xs, idx, wts, w1q, w1s, w3q, w3s, w2q, w2s, tokens, ue8m0=False, n_shared=0):
    """MoE output rows (bf16 bits [len(tokens), dim]) for the listed tokens.
    Stacked expert weights: w1q/w3q [(E+n_shared)*inter, dim], w2q [(E+n_shared)*dim, inter];
    the last n_shared experts are shared: every token uses them with weight 1."""
    xq, xs = _c(xq, np.uint8), _c(xs, np.float32)
    idx, wts = _c(idx, np.int32), _c(wts, np.float32)
    w1q, w3q, w2q = _c(w1q, np.uint8), _c(w3q, np.uint8), _c(w2q, np.uint8)
    w1s, w3s, w2s = _c(w1s, np.float32), _c(w3s, np.float32), _c(w2s, np.float32)
    T, dim = xq.shape
    topk = idx.shape[1]
    inter = w2q.shape[1]
    E = w2q.shape[0] // dim - n_shared
    y = np.empty((len(tokens), dim), np.uint16)
    L = lib()
    for i, t in enumerate(tokens):
        row = np.empty(dim, np.uint16)
        rc = L.orc_moe_token(_ptr(xq), _ptr(xs), _ptr(idx), _ptr(wts), int(t), topk,
                             _ptr(w1q), _ptr(w1s), _ptr(w3q), _ptr(w3s), _ptr(w2q), _ptr(w2s),
                             dim, inter, int(bool(ue8m0)), E, n_shared, _ptr(row))
        if rc:
            raise MemoryError("oracle MoE token failed")
        y[i] = row
    return y


# ---- MoE gate (scores, group-limited top-k, weights) -----------------------------

def moe_gate(logits, bias, n_groups: int, topk_groups: int, topk: int, sigmoid: bool,
             route_scale: float = 1.0, normalize: bool = True):
    """logits fp32 [T, E] (+ bias fp32 [E] or None) -> (indices int32 [T, topk]
    in descending selection-key order, weights fp32 [T, topk])."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    b = None if bias is None else _c(bias, np.float32)
    idx = np.empty((T, topk), np.int32)
    w = np.empty((T, topk), np.float32)
    rc = lib().orc_moe_gate(_ptr(logits), None if b is None else _ptr(b), T, E, n_groups, topk_groups, topk,
                            int(bool(sigmoid)), float(route_scale), int(bool(normalize)), _ptr(idx), _ptr(w))
    if rc:
        raise ValueError("gate shape outside the rules")
    return idx, w


# ---- MLA absorb projections ------------------------------------------------------

def mla_absorb(inp_bits, wq, ws, H: int, dn: int, dv: int, mode: str):
    """mode "qk": q_nope bf16 bits [T, H, dn] -> bf16 bits [T, H, C];
    mode "v": x bf16 bits [T, H, C] -> bf16 bits [T, H, dv]. wq e4m3 codes
    [H*(dn+dv), C] with block scales ws [H*(dn+dv)/128, C/128]."""
    inp = _c(inp_bits, np.uint16)
    wq, ws = _c(wq, np.uint8), _c(ws, np.float32)
    C = wq.shape[1]
    T = inp.shape[0]
    out = np.empty((T, H, C if mode == "qk" else dv), np.uint16)
    lib().orc_mla_absorb(_ptr(inp), _ptr(wq), _ptr(ws), T, H, dn, dv, C, 0 if mode == "qk" else 1, _ptr(out))
    return out
