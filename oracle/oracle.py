"""ctypes wrapper around the scalar C oracle (``smoe_oracle.c``).

TEST INFRASTRUCTURE ONLY: used by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``.  Arrays are numpy; bf16 data travels as
``uint16`` bit patterns and fp16 scales as ``uint16`` bit patterns.

Each wrapper names the page and section it follows; the C file holds the
arithmetic and the readings (G1-G5) where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

__all__ = [
    "build_oracle", "lib", "quantize", "pack", "unpack", "dequantize", "encode", "decode",
    "grid", "f16_to_f32", "f32_to_f16", "stream_bytes", "scales_bytes", "blob_bytes",
    "make_blob", "router_logits", "route", "expert_ffn", "moe_apply", "moe_apply_threads",
    "moe_forward",
    "GROUP", "NCAND",
]

GROUP = 64
NCAND = 64

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "smoe_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build_oracle(force: bool = False) -> str:
    """Compile the oracle with contraction and fast-math off (plain gcc)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread",
            "-o", tmp, _SRC, "-lm",
        ])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            # SMOE_ORACLE_SO lets the mutation test load a deliberately broken
            # copy of the oracle and check that the pins reject it.
            L = ctypes.CDLL(os.environ.get("SMOE_ORACLE_SO") or build_oracle())
            P, I64, I32, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
            L.oracle_quantize.argtypes = [P, I64, I64, ctypes.c_int, P, P, P, P, P]
            L.oracle_quantize.restype = ctypes.c_int
            L.oracle_pack.argtypes = [P, I64, ctypes.c_int, P]
            L.oracle_unpack.argtypes = [P, I64, ctypes.c_int, P]
            L.oracle_dequantize.argtypes = [P, P, I64, I64, ctypes.c_int, P]
            L.oracle_dequantize.restype = ctypes.c_int
            L.oracle_stream_bytes.argtypes = [I64, I64, ctypes.c_int]
            L.oracle_stream_bytes.restype = I64
            L.oracle_scales_bytes.argtypes = [I64, I64, ctypes.c_int]
            L.oracle_scales_bytes.restype = I64
            L.oracle_blob_bytes.argtypes = [I64, I64, ctypes.c_int]
            L.oracle_blob_bytes.restype = I64
            L.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.oracle_f16_to_f32.restype = F
            L.oracle_f32_to_f16.argtypes = [F]
            L.oracle_f32_to_f16.restype = ctypes.c_uint16
            L.oracle_grid.argtypes = [P]
            L.oracle_encode.argtypes = [F, F, ctypes.c_int]
            L.oracle_encode.restype = ctypes.c_uint8
            L.oracle_decode.argtypes = [ctypes.c_uint8, F, ctypes.c_int]
            L.oracle_decode.restype = F
            L.oracle_router_logits.argtypes = [P, P, I64, I32, I32, P]
            L.oracle_route.argtypes = [P, I64, I32, I32, I32, P, P, P]
            L.oracle_route.restype = ctypes.c_int
            L.oracle_expert_ffn.argtypes = [P, I32, I32, ctypes.c_int, P, P, P]
            L.oracle_expert_ffn.restype = ctypes.c_int
            L.oracle_moe_apply.argtypes = [I32, I32, I32, I32, ctypes.c_int, P, P, I32, P, P,
                                           I64, P, P, P]
            L.oracle_moe_apply.restype = ctypes.c_int
            L.oracle_moe_forward.argtypes = [I32, I32, I32, I32, I32, ctypes.c_int, P, P, P, P,
                                             I32, P, P, I64, P, P, P, P]
            L.oracle_moe_forward.restype = ctypes.c_int
            L.oracle_route_ex.argtypes = [P, I64, I32, I32, I32, P, I32, F, P, P]
            L.oracle_route_ex.restype = ctypes.c_int
            L.oracle_moe_forward_ex.argtypes = [I32, I32, I32, I32, I32, ctypes.c_int, P, P, P,
                                                I32, F, P, P, P, I32, P, P, I64, P, P, P, P]
            L.oracle_moe_apply_mixed.argtypes = [I32, I32, I32, I32, ctypes.c_int, P, P, P, I32,
                                                 P, P, I64, P, P, P]
            L.oracle_moe_apply_mixed.restype = ctypes.c_int
            L.oracle_route_ex2.argtypes = [P, I64, I32, I32, I32, P, I32, F, P, P, P]
            L.oracle_route_ex2.restype = ctypes.c_int
            L.oracle_moe_forward_ex.restype = ctypes.c_int
            L.oracle_moe_apply_threads.argtypes = [I32, I32, I32, I32, ctypes.c_int, P, P, P, I32,
                                                   P, P, I64, P, P, P, ctypes.c_int]
            L.oracle_moe_apply_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- scalars

def f16_to_f32(h: int) -> float:
    return float(lib().oracle_f16_to_f32(int(h)))


def f32_to_f16(f: float) -> int:
    return int(lib().oracle_f32_to_f16(float(np.float32(f))))


def grid() -> np.ndarray:
    """linspace(0.1, 1.0, 64) as fp32 ("SMOE Quantisation", L2-MSE Scale Optimiser)."""
    t = np.zeros(NCAND, np.float32)
    lib().oracle_grid(_p(t))
    return t


def encode(w: float, s: float, bits: int) -> int:
    return int(lib().oracle_encode(float(np.float32(w)), float(np.float32(s)), bits))


def decode(c: int, s: float, bits: int) -> float:
    return float(np.float32(lib().oracle_decode(int(c), float(np.float32(s)), bits)))


# ---------------------------------------------------------------- sizes

def stream_bytes(rows: int, cols: int, bits: int) -> int:
    return int(lib().oracle_stream_bytes(rows, cols, bits))


def scales_bytes(rows: int, cols: int, group: int = GROUP) -> int:
    return int(lib().oracle_scales_bytes(rows, cols, group))


def blob_bytes(d: int, f: int, bits: int) -> int:
    return int(lib().oracle_blob_bytes(d, f, bits))


# ---------------------------------------------------------------- quantiser

def quantize(w_bf16: np.ndarray, bits: int, with_mse: bool = False):
    """Grid-search quantise a bf16 [rows, cols] tensor ("SMOE Quantisation").

    Returns a dict with ``codes_lsb`` (uint8 stream), ``scales_f16`` (uint16),
    ``scale_f32`` (float32 per group), ``j_best`` (int32 per group, -1 for an
    all-zero group) and, with ``with_mse``, ``mse`` float64 [groups, 64].
    """
    w = _c(w_bf16, np.uint16)
    rows, cols = w.shape
    n = rows * cols
    ng = n // GROUP
    codes = np.zeros(stream_bytes(rows, cols, bits), np.uint8)
    sc16 = np.zeros(ng, np.uint16)
    sc32 = np.zeros(ng, np.float32)
    jb = np.zeros(ng, np.int32)
    mse = np.zeros((ng, NCAND), np.float64) if with_mse else None
    rc = lib().oracle_quantize(_p(w), rows, cols, bits, _p(codes), _p(sc16), _p(sc32), _p(jb),
                               _p(mse))
    if rc:
        raise ValueError(f"oracle_quantize rejected rows={rows} cols={cols} bits={bits}")
    out = {"codes_lsb": codes, "scales_f16": sc16, "scale_f32": sc32, "j_best": jb}
    if with_mse:
        out["mse"] = mse
    return out


def pack(codes: np.ndarray, bits: int) -> np.ndarray:
    c = _c(codes, np.uint8).ravel()
    out = np.zeros((c.size * bits + 7) // 8, np.uint8)
    lib().oracle_pack(_p(c), c.size, bits, _p(out))
    return out


def unpack(packed: np.ndarray, n: int, bits: int) -> np.ndarray:
    p = _c(packed, np.uint8).ravel()
    out = np.zeros(n, np.uint8)
    lib().oracle_unpack(_p(p), n, bits, _p(out))
    return out


def dequantize(codes_lsb, scales_f16, rows: int, cols: int, bits: int) -> np.ndarray:
    c = _c(codes_lsb, np.uint8)
    s = _c(scales_f16, np.uint16)
    out = np.zeros((rows, cols), np.float32)
    if lib().oracle_dequantize(_p(c), _p(s), rows, cols, bits, _p(out)):
        raise ValueError("oracle_dequantize rejected its arguments")
    return out


def make_blob(gate_q: dict, up_q: dict, down_q: dict) -> np.ndarray:
    """Concatenate quantised sub-tensors in the ".smoe Binary Format" Expert
    Blob order: [gate codes][gate scales][up codes][up scales][down codes]
    [down scales] (no padding)."""
    parts = []
    for q in (gate_q, up_q, down_q):
        parts.append(np.asarray(q["codes_lsb"], np.uint8))
        parts.append(np.asarray(q["scales_f16"], np.uint16).view(np.uint8))
    return np.ascontiguousarray(np.concatenate(parts))


# ---------------------------------------------------------------- router

def router_logits(wr_bf16: np.ndarray, x: np.ndarray) -> np.ndarray:
    wr = _c(wr_bf16, np.uint16)
    xx = _c(x, np.float32)
    E, d = wr.shape
    T = xx.shape[0]
    out = np.zeros((T, E), np.float32)
    lib().oracle_router_logits(_p(wr), _p(xx), T, E, d, _p(out))
    return out


def route(logits: np.ndarray, k: int, norm: bool, bias: np.ndarray | None = None,
          router_sigmoid: bool = False, routed_scaling_factor: float = 1.0,
          mask: np.ndarray | None = None):
    """Top-k routing ("CMF v2 -- Format Specification", 2.2 MoE): softmax or
    per-expert sigmoid scores, selection-only bias, renormalisation, then
    the routed scaling factor; an optional routing mask (§5: uint8
    bitfield, LSB-first) limits selection and softmax to the routable
    experts."""
    lg = _c(logits, np.float32)
    T, E = lg.shape
    b = None if bias is None else _c(bias, np.float32)
    m = None if mask is None else _c(mask, np.uint8)
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    if lib().oracle_route_ex2(_p(lg), T, E, k, int(bool(norm)), _p(b), int(bool(router_sigmoid)),
                              ctypes.c_float(routed_scaling_factor), _p(m), _p(ids), _p(w)):
        raise ValueError("oracle_route rejected its arguments")
    return ids, w


# ---------------------------------------------------------------- experts

def expert_ffn(blob: np.ndarray, d: int, f: int, bits: int, x: np.ndarray):
    """One expert's SwiGLU FFN on one token; returns (out [d], h [f])."""
    b = _c(blob, np.uint8)
    xx = _c(x, np.float32)
    out = np.zeros(d, np.float32)
    h = np.zeros(f, np.float32)
    if lib().oracle_expert_ffn(_p(b), d, f, bits, _p(xx), _p(out), _p(h)):
        raise ValueError("oracle_expert_ffn rejected its arguments")
    return out, h


def _blob_table(blobs, E):
    arr = (ctypes.c_void_p * E)()
    keep = []
    for e in range(E):
        b = blobs.get(e) if isinstance(blobs, dict) else blobs[e]
        if b is None:
            arr[e] = None
        else:
            b = _c(b, np.uint8)
            keep.append(b)
            arr[e] = b.ctypes.data
    return arr, keep


def moe_apply(d, f, E, k, bits, blobs, x, ids, weights, shared_blob=None, fs=0,
              shared_gate=None, expert_bits=None):
    """Apply a given routing to T tokens (rank-order combine, shared expert);
    expert_bits: each routed expert's own depth (shared expert at bits)."""
    xx = _c(x, np.float32)
    T = xx.shape[0]
    table, keep = _blob_table(blobs, E)
    sb = None if shared_blob is None else _c(shared_blob, np.uint8)
    sg = None if shared_gate is None else _c(shared_gate, np.uint16)
    ii = _c(ids, np.int32)
    ww = _c(weights, np.float32)
    y = np.zeros((T, d), np.float32)
    eb_ = None if expert_bits is None else _c(expert_bits, np.int32)
    rc = lib().oracle_moe_apply_mixed(d, f, E, k, bits, _p(eb_), ctypes.cast(table, ctypes.c_void_p),
                                      _p(sb), fs, _p(sg), _p(xx), T, _p(ii), _p(ww), _p(y))
    if rc:
        raise ValueError(f"oracle_moe_apply failed ({rc})")
    del keep
    return y


def moe_apply_threads(d, f, E, k, bits, blobs, x, ids, weights, nthreads, shared_blob=None,
                      fs=0, shared_gate=None, expert_bits=None):
    """moe_apply with the (token, slot) expert FFNs spread over nthreads
    threads; the same bits as moe_apply (the combine stays serial)."""
    xx = _c(x, np.float32)
    T = xx.shape[0]
    table, keep = _blob_table(blobs, E)
    sb = None if shared_blob is None else _c(shared_blob, np.uint8)
    sg = None if shared_gate is None else _c(shared_gate, np.uint16)
    ii = _c(ids, np.int32)
    ww = _c(weights, np.float32)
    y = np.zeros((T, d), np.float32)
    eb_ = None if expert_bits is None else _c(expert_bits, np.int32)
    rc = lib().oracle_moe_apply_threads(d, f, E, k, bits, _p(eb_),
                                        ctypes.cast(table, ctypes.c_void_p), _p(sb), fs, _p(sg),
                                        _p(xx), T, _p(ii), _p(ww), _p(y), int(nthreads))
    if rc:
        raise ValueError(f"oracle_moe_apply_threads failed ({rc})")
    del keep
    return y


def moe_forward(d, f, E, k, norm, bits, router_w, blobs, x, expert_bias=None,
                shared_blob=None, fs=0, shared_gate=None, router_sigmoid=False,
                routed_scaling_factor=1.0, mask=None, expert_bits=None):
    """Full MoE layer forward; returns (y, ids, weights, logits)."""
    xx = _c(x, np.float32)
    T = xx.shape[0]
    wr = _c(router_w, np.uint16)
    table, keep = _blob_table(blobs, E)
    eb = None if expert_bias is None else _c(expert_bias, np.float32)
    sb = None if shared_blob is None else _c(shared_blob, np.uint8)
    sg = None if shared_gate is None else _c(shared_gate, np.uint16)
    y = np.zeros((T, d), np.float32)
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    lg = np.zeros((T, E), np.float32)
    mk = None if mask is None else _c(mask, np.uint8)
    ebits = None if expert_bits is None else _c(expert_bits, np.int32)
    rc = lib().oracle_moe_forward_ex(d, f, E, k, int(bool(norm)), bits, _p(ebits), _p(wr), _p(eb),
                                     int(bool(router_sigmoid)), ctypes.c_float(routed_scaling_factor),
                                     _p(mk), ctypes.cast(table, ctypes.c_void_p), _p(sb), fs, _p(sg),
                                     _p(xx), T, _p(y), _p(ids), _p(w), _p(lg))
    if rc:
        raise ValueError(f"oracle_moe_forward failed ({rc})")
    del keep
    return y, ids, w, lg
