"""Thin ctypes binding of libsmoe.so (the C ABI in include/smoe.h).

Argument marshalling only: every step of the method runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors (PyTorch provides device memory
and streams); the binding passes ``data_ptr()`` and the current stream.  If
the library is missing the binding raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsmoe.so")
SYNTH_PATH = os.path.join(_HERE, "_build", "libsmoe_synth.so")

SMOE_OK = 0
STATUS_NAMES = {0: "SMOE_OK", -1: "SMOE_ERR_INVALID_ARG", -2: "SMOE_ERR_UNSUPPORTED",
                -3: "SMOE_ERR_WORKSPACE", -4: "SMOE_ERR_CUDA", -5: "SMOE_ERR_DEVICE_FAULT",
                -6: "SMOE_ERR_TIMEOUT"}
SMOE_F32, SMOE_BF16 = 0, 1

# Bytes of the built-in workspace of smoe_moe_forward_noalloc
# (SMOE_NOALLOC_SCRATCH_BYTES in include/smoe.h).
NOALLOC_SCRATCH_BYTES = 32 << 20

EXPORTED = [
    "smoe_status_string", "smoe_stream_bytes", "smoe_scales_bytes", "smoe_expert_tiles_bytes",
    "smoe_repacked_bytes", "smoe_quantize", "smoe_repack", "smoe_unpack",
    "smoe_route_from_logits", "smoe_moe_workspace_bytes", "smoe_moe_workspace_init",
    "smoe_moe_forward", "smoe_moe_forward_stage", "smoe_get_device_status",
    "smoe_moe_forward_noalloc", "smoe_moe_forward_path", "smoe_moe_path",
    "smoe_vault_parse", "smoe_vault_find_expert", "smoe_vault_repack_layer",
    "smoe_route_from_logits_ex", "smoe_moe_forward_ex",
    "smoe_repacked_bytes_mixed", "smoe_repack_mixed", "smoe_unpack_mixed",
    "smoe_moe_workspace_bytes_mixed", "smoe_moe_forward_mixed", "smoe_moe_forward_stage_mixed",
    "smoe_debug_set_waits", "smoe_moe_path_dtype",
]

# Execution paths (SMOE_PATH_* in include/smoe.h).
PATH_AUTO, PATH_STREAM, PATH_GROUPED = 0, 1, 2


class RouterOpts(ctypes.Structure):
    """smoe_router_opts (include/smoe.h)."""
    _fields_ = [("router_sigmoid", ctypes.c_int32), ("routed_scaling_factor", ctypes.c_float),
                ("expert_mask", ctypes.c_void_p)]


class VaultInfo(ctypes.Structure):
    """smoe_vault_info (include/smoe.h)."""
    _fields_ = [("version", ctypes.c_uint32), ("num_moe_layers", ctypes.c_uint32),
                ("max_experts_per_layer", ctypes.c_uint32), ("total_experts", ctypes.c_uint32),
                ("table_offset", ctypes.c_uint64), ("data_offset", ctypes.c_uint64),
                ("group_size", ctypes.c_uint32), ("bits", ctypes.c_uint32),
                ("d_model", ctypes.c_uint32), ("vocab_size", ctypes.c_uint32),
                ("ffn_dim", ctypes.c_uint32), ("reserved_ext", ctypes.c_uint32),
                ("has_arch", ctypes.c_int32), ("arch_flags", ctypes.c_uint32),
                ("rope_theta", ctypes.c_float), ("num_heads", ctypes.c_uint32),
                ("num_kv_heads", ctypes.c_uint32), ("head_dim", ctypes.c_uint32),
                ("moe_top_k", ctypes.c_uint32), ("moe_ffn_dim", ctypes.c_uint32),
                ("dense_ffn_dim", ctypes.c_uint32), ("shared_expert_ffn_dim", ctypes.c_uint32),
                ("activation", ctypes.c_uint32), ("num_hidden_layers", ctypes.c_uint32),
                ("rms_norm_eps", ctypes.c_float), ("model_type", ctypes.c_char * 25)]


class VaultTensor(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_uint32), ("cols", ctypes.c_uint32),
                ("packed_offset", ctypes.c_uint64), ("packed_size", ctypes.c_uint64),
                ("scales_offset", ctypes.c_uint64), ("scales_size", ctypes.c_uint64)]


class VaultExpert(ctypes.Structure):
    """smoe_vault_expert (include/smoe.h)."""
    _fields_ = [("layer_id", ctypes.c_uint32), ("expert_id", ctypes.c_uint32),
                ("byte_offset", ctypes.c_uint64), ("raw_size", ctypes.c_uint64),
                ("padded_size", ctypes.c_uint64), ("num_groups", ctypes.c_uint64),
                ("tensor", VaultTensor * 3)]


class SmoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")
        self.status = status


class LayerDesc(ctypes.Structure):
    """Mirror of smoe_layer_desc."""
    _fields_ = [
        ("d_model", ctypes.c_int32), ("ffn_dim", ctypes.c_int32),
        ("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
        ("norm_topk_prob", ctypes.c_int32), ("bits", ctypes.c_int32),
        ("group_size", ctypes.c_int32),
        ("router_w", ctypes.c_void_p), ("expert_bias", ctypes.c_void_p),
        ("expert_tiles", ctypes.c_void_p), ("shared_tiles", ctypes.c_void_p),
        ("shared_ffn_dim", ctypes.c_int32), ("shared_gate_w", ctypes.c_void_p),
    ]


_lib = None
_synth = None


def load(path: str | None = None):
    """Load libsmoe.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libsmoe.so not built ({p}); run __graft_entry__.build()")
    L = ctypes.CDLL(p)
    P, I64, I32, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int
    S = ctypes.c_size_t
    L.smoe_status_string.argtypes = [I]
    L.smoe_status_string.restype = ctypes.c_char_p
    L.smoe_stream_bytes.argtypes = [I64, I64, I]
    L.smoe_stream_bytes.restype = S
    L.smoe_scales_bytes.argtypes = [I64, I64, I]
    L.smoe_scales_bytes.restype = S
    L.smoe_expert_tiles_bytes.argtypes = [I32, I32, I, I]
    L.smoe_expert_tiles_bytes.restype = S
    L.smoe_repacked_bytes.argtypes = [I32, I32, I32, I, I]
    L.smoe_repacked_bytes.restype = S
    L.smoe_quantize.argtypes = [P, I64, I64, I, I, P, P, P]
    L.smoe_quantize.restype = I
    L.smoe_repack.argtypes = [P, P, I32, I32, I32, I, I, P, S, P]
    L.smoe_repack.restype = I
    L.smoe_unpack.argtypes = [P, I32, I32, I32, I, I, P, P, P]
    L.smoe_unpack.restype = I
    L.smoe_route_from_logits.argtypes = [P, I64, I32, I32, I, P, P, P, P]
    L.smoe_route_from_logits.restype = I
    L.smoe_moe_workspace_bytes.argtypes = [ctypes.POINTER(LayerDesc), I64]
    L.smoe_moe_workspace_bytes.restype = S
    L.smoe_moe_workspace_init.argtypes = [P, S, P]
    L.smoe_moe_workspace_init.restype = I
    L.smoe_moe_forward.argtypes = [ctypes.POINTER(LayerDesc), P, I, I64, P, P, S, P, P, P]
    L.smoe_moe_forward.restype = I
    L.smoe_moe_forward_stage.argtypes = [ctypes.POINTER(LayerDesc), P, I, I64, P, P, S, P, P,
                                          I, P]
    L.smoe_moe_forward_stage.restype = I
    L.smoe_moe_forward_noalloc.argtypes = [ctypes.POINTER(LayerDesc), P, I, I64, P, P, P, P]
    L.smoe_moe_forward_noalloc.restype = I
    L.smoe_moe_forward_path.argtypes = [ctypes.POINTER(LayerDesc), P, I, I64, P, P, S, P, P, I,
                                         P]
    L.smoe_moe_forward_path.restype = I
    L.smoe_moe_path.argtypes = [ctypes.POINTER(LayerDesc), I64]
    L.smoe_moe_path.restype = I
    L.smoe_moe_path_dtype.argtypes = [ctypes.POINTER(LayerDesc), I64, I]
    L.smoe_moe_path_dtype.restype = I
    RP = ctypes.POINTER(RouterOpts)
    L.smoe_route_from_logits_ex.argtypes = [P, I64, I32, I32, I, P, RP, P, P, P]
    L.smoe_route_from_logits_ex.restype = I
    L.smoe_moe_forward_ex.argtypes = [ctypes.POINTER(LayerDesc), RP, P, I, I64, P, P, S, P, P, I,
                                      P]
    L.smoe_moe_forward_ex.restype = I
    VP = ctypes.POINTER(VaultInfo)
    L.smoe_vault_parse.argtypes = [P, S, ctypes.c_uint64, VP]
    L.smoe_vault_parse.restype = I
    L.smoe_vault_find_expert.argtypes = [P, S, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                         ctypes.POINTER(VaultExpert)]
    L.smoe_vault_find_expert.restype = I
    L.smoe_vault_repack_layer.argtypes = [P, S, P, ctypes.c_uint64, ctypes.c_uint32,
                                          ctypes.c_uint32, P, S, P]
    L.smoe_vault_repack_layer.restype = I
    U8P = ctypes.POINTER(ctypes.c_uint8)
    L.smoe_repacked_bytes_mixed.argtypes = [I32, I32, I32, U8P, I]
    L.smoe_repacked_bytes_mixed.restype = S
    L.smoe_repack_mixed.argtypes = [P, P, I32, I32, I32, U8P, I, P, S, P]
    L.smoe_repack_mixed.restype = I
    L.smoe_unpack_mixed.argtypes = [P, I32, I32, I32, U8P, I, P, P, P]
    L.smoe_unpack_mixed.restype = I
    L.smoe_moe_workspace_bytes_mixed.argtypes = [ctypes.POINTER(LayerDesc), I64]
    L.smoe_moe_workspace_bytes_mixed.restype = S
    L.smoe_moe_forward_mixed.argtypes = [ctypes.POINTER(LayerDesc), U8P, RP, P, I, I64, P, P, S,
                                         P, P, I, P]
    L.smoe_moe_forward_mixed.restype = I
    L.smoe_moe_forward_stage_mixed.argtypes = [ctypes.POINTER(LayerDesc), U8P, P, I, I64, P, P,
                                               S, P, P, I, P]
    L.smoe_moe_forward_stage_mixed.restype = I
    L.smoe_get_device_status.argtypes = [P]
    L.smoe_get_device_status.restype = I
    L.smoe_debug_set_waits.argtypes = [ctypes.c_longlong, I]
    L.smoe_debug_set_waits.restype = None
    _lib = L
    return L


def load_synth():
    global _synth
    if _synth is None:
        if not os.path.exists(SYNTH_PATH):
            raise RuntimeError(f"libsmoe_synth.so not built ({SYNTH_PATH})")
        S = ctypes.CDLL(SYNTH_PATH)
        S.smoe_synth_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_uint64, ctypes.c_float, ctypes.c_float,
                                      ctypes.c_uint64, ctypes.c_uint64, ctypes.c_void_p]
        S.smoe_synth_bf16.restype = ctypes.c_int
        _synth = S
    return _synth


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, what: str):
    if rc != SMOE_OK:
        raise SmoeError(rc, what)


# ------------------------------------------------------------------ sizes

def stream_bytes(rows, cols, bits):
    return int(load().smoe_stream_bytes(rows, cols, bits))


def scales_bytes(rows, cols, group_size=64):
    return int(load().smoe_scales_bytes(rows, cols, group_size))


def expert_tiles_bytes(d, f, bits, group_size=64):
    return int(load().smoe_expert_tiles_bytes(d, f, bits, group_size))


def repacked_bytes(d, f, n_experts, bits, group_size=64):
    return int(load().smoe_repacked_bytes(d, f, n_experts, bits, group_size))


def _bits_array(expert_bits):
    """Per-expert depths as a host uint8 array (kept alive by the caller)."""
    vals = [int(b) for b in expert_bits]
    return (ctypes.c_uint8 * max(len(vals), 1))(*vals)


def repacked_bytes_mixed(d, f, expert_bits, group_size=64):
    eb = _bits_array(expert_bits)
    return int(load().smoe_repacked_bytes_mixed(d, f, len(expert_bits), eb, group_size))


# ------------------------------------------------------------------ quantise

def quantize(w_bf16: torch.Tensor, bits: int, codes=None, scales=None, stream=None):
    """smoe_quantize on a bf16 [rows, cols] CUDA tensor; returns (codes, scales)."""
    rows, cols = w_bf16.shape
    if codes is None:
        codes = torch.empty(stream_bytes(rows, cols, bits), dtype=torch.uint8, device=w_bf16.device)
    if scales is None:
        scales = torch.empty(rows * cols // 64, dtype=torch.int16, device=w_bf16.device)
    _check(load().smoe_quantize(_ptr(w_bf16), rows, cols, bits, 64, _ptr(codes), _ptr(scales),
                                _stream(stream)), "smoe_quantize")
    return codes, scales


def _ptr_array(ts):
    arr = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = t.data_ptr()
    return arr


def repack(codes: list, scales: list, d: int, f: int, n_experts: int, bits: int, out=None,
           stream=None):
    """smoe_repack: codes/scales are lists of 3*E CUDA tensors (gate, up, down per expert)."""
    nbytes = repacked_bytes(d, f, n_experts, bits)
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=codes[0].device)
    _check(load().smoe_repack(_ptr_array(codes), _ptr_array(scales), d, f, n_experts, bits, 64,
                              _ptr(out), out.numel() * out.element_size(), _stream(stream)),
           "smoe_repack")
    return out


def repack_mixed(codes: list, scales: list, d: int, f: int, expert_bits, out=None, stream=None):
    """smoe_repack_mixed: expert e's streams at depth expert_bits[e]."""
    n = len(expert_bits)
    eb = _bits_array(expert_bits)
    nbytes = repacked_bytes_mixed(d, f, expert_bits)
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=codes[0].device)
    _check(load().smoe_repack_mixed(_ptr_array(codes), _ptr_array(scales), d, f, n, eb, 64,
                                    _ptr(out), out.numel() * out.element_size(), _stream(stream)),
           "smoe_repack_mixed")
    return out


def unpack_mixed(tiles, d: int, f: int, expert_bits, stream=None):
    """smoe_unpack_mixed: returns (codes list, scales list) of 3*E tensors."""
    dev = tiles.device
    codes, scales = [], []
    for b in expert_bits:
        for kind in range(3):
            R, K = (f, d) if kind < 2 else (d, f)
            codes.append(torch.empty(stream_bytes(R, K, int(b)), dtype=torch.uint8, device=dev))
            scales.append(torch.empty(R * K // 64, dtype=torch.int16, device=dev))
    eb = _bits_array(expert_bits)
    _check(load().smoe_unpack_mixed(_ptr(tiles), d, f, len(expert_bits), eb, 64,
                                    _ptr_array(codes), _ptr_array(scales), _stream(stream)),
           "smoe_unpack_mixed")
    return codes, scales


def unpack(tiles, d: int, f: int, n_experts: int, bits: int, stream=None):
    """smoe_unpack: returns (codes list, scales list) of 3*E tensors."""
    dev = tiles.device
    codes, scales = [], []
    for _ in range(n_experts):
        for kind in range(3):
            R, K = (f, d) if kind < 2 else (d, f)
            codes.append(torch.empty(stream_bytes(R, K, bits), dtype=torch.uint8, device=dev))
            scales.append(torch.empty(R * K // 64, dtype=torch.int16, device=dev))
    _check(load().smoe_unpack(_ptr(tiles), d, f, n_experts, bits, 64, _ptr_array(codes),
                              _ptr_array(scales), _stream(stream)), "smoe_unpack")
    return codes, scales


# ------------------------------------------------------------------ route

def _opts(router_sigmoid, routed_scaling_factor, expert_mask=None):
    """smoe_router_opts, or None for the defaults.  expert_mask: a host
    uint8 bitfield (numpy array or bytes), LSB-first, bit e = expert e
    routable; the returned options keep it alive."""
    if not router_sigmoid and routed_scaling_factor == 1.0 and expert_mask is None:
        return None
    o = RouterOpts(int(bool(router_sigmoid)), float(routed_scaling_factor), None)
    if expert_mask is not None:
        buf = ctypes.create_string_buffer(bytes(bytearray(expert_mask)), len(bytes(bytearray(expert_mask))))
        o._mask_buf = buf
        o.expert_mask = ctypes.cast(buf, ctypes.c_void_p)
    return o


def route_from_logits(logits: torch.Tensor, k: int, norm: bool, bias=None, stream=None,
                      router_sigmoid=False, routed_scaling_factor=1.0, expert_mask=None):
    """smoe_route_from_logits (smoe_route_from_logits_ex with router options)."""
    T, E = logits.shape
    ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    o = _opts(router_sigmoid, routed_scaling_factor, expert_mask)
    if o is None:
        _check(load().smoe_route_from_logits(_ptr(logits), T, E, k, int(bool(norm)), _ptr(bias),
                                             _ptr(ids), _ptr(w), _stream(stream)),
               "smoe_route_from_logits")
    else:
        _check(load().smoe_route_from_logits_ex(_ptr(logits), T, E, k, int(bool(norm)),
                                                _ptr(bias), ctypes.byref(o), _ptr(ids), _ptr(w),
                                                _stream(stream)), "smoe_route_from_logits_ex")
    return ids, w


# ------------------------------------------------------------------ forward

class MoELayer:
    """Holds one layer's device tensors and its smoe_layer_desc."""

    def __init__(self, d, f, E, k, norm, bits, router_w, expert_tiles, expert_bias=None,
                 shared_tiles=None, shared_f=0, shared_gate_w=None, expert_bits=None):
        """expert_bits: per-expert depths of a bank written by repack_mixed
        (then `bits` is the shared expert's depth); None = all at `bits`."""
        self.d, self.f, self.E, self.k, self.norm, self.bits = d, f, E, k, bool(norm), bits
        self.expert_bits = None if expert_bits is None else [int(b) for b in expert_bits]
        self._ebits = None if expert_bits is None else _bits_array(expert_bits)
        self.router_w, self.expert_tiles, self.expert_bias = router_w, expert_tiles, expert_bias
        self.shared_tiles, self.shared_f, self.shared_gate_w = shared_tiles, shared_f, shared_gate_w
        self.desc = LayerDesc(
            d, f, E, k, int(bool(norm)), bits, 64,
            router_w.data_ptr(), None if expert_bias is None else expert_bias.data_ptr(),
            expert_tiles.data_ptr(), None if shared_tiles is None else shared_tiles.data_ptr(),
            shared_f, None if shared_gate_w is None else shared_gate_w.data_ptr())

    def workspace_bytes(self, T: int) -> int:
        if self.expert_bits is not None:
            n = int(load().smoe_moe_workspace_bytes_mixed(ctypes.byref(self.desc), T))
        else:
            n = int(load().smoe_moe_workspace_bytes(ctypes.byref(self.desc), T))
        if n == 0 and T >= 0:
            raise SmoeError(-1, "smoe_moe_workspace_bytes")
        return n


def workspace(layer: MoELayer, T: int, device=None, stream=None):
    """Allocate and zero a workspace for `layer` at T tokens."""
    n = layer.workspace_bytes(T)
    ws = torch.empty(n + 256, dtype=torch.uint8, device=device or layer.router_w.device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + n]
    _check(load().smoe_moe_workspace_init(_ptr(ws), n, _stream(stream)), "workspace_init")
    return ws


def forward(layer: MoELayer, x: torch.Tensor, ws: torch.Tensor, y=None, ids=None, w=None,
            stream=None, path=None, router_sigmoid=False, routed_scaling_factor=1.0,
            expert_mask=None):
    """smoe_moe_forward (smoe_moe_forward_path when `path` is given,
    smoe_moe_forward_ex with router options); x is [T, d] fp32 or bf16;
    returns y fp32 [T, d]."""
    T = x.shape[0]
    if y is None:
        y = torch.empty((T, layer.d), dtype=torch.float32, device=x.device)
    dt = SMOE_BF16 if x.dtype == torch.bfloat16 else SMOE_F32
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("x must be fp32 or bf16")
    o = _opts(router_sigmoid, routed_scaling_factor, expert_mask)
    if layer.expert_bits is not None:
        _check(load().smoe_moe_forward_mixed(ctypes.byref(layer.desc), layer._ebits,
                                             None if o is None else ctypes.byref(o), _ptr(x), dt,
                                             T, _ptr(y), _ptr(ws), ws.numel(), _ptr(ids),
                                             _ptr(w), PATH_AUTO if path is None else int(path),
                                             _stream(stream)), "smoe_moe_forward_mixed")
    elif o is not None:
        _check(load().smoe_moe_forward_ex(ctypes.byref(layer.desc), ctypes.byref(o), _ptr(x), dt,
                                          T, _ptr(y), _ptr(ws), ws.numel(), _ptr(ids), _ptr(w),
                                          PATH_AUTO if path is None else int(path),
                                          _stream(stream)), "smoe_moe_forward_ex")
    elif path is None:
        _check(load().smoe_moe_forward(ctypes.byref(layer.desc), _ptr(x), dt, T, _ptr(y), _ptr(ws),
                                       ws.numel(), _ptr(ids), _ptr(w), _stream(stream)),
               "smoe_moe_forward")
    else:
        _check(load().smoe_moe_forward_path(ctypes.byref(layer.desc), _ptr(x), dt, T, _ptr(y),
                                            _ptr(ws), ws.numel(), _ptr(ids), _ptr(w), int(path),
                                            _stream(stream)), "smoe_moe_forward_path")
    return y


def path_for(layer: MoELayer, T: int, x_dtype=None) -> int:
    """smoe_moe_path_dtype: the execution path smoe_moe_forward (and, for a
    layer with per-expert depths, smoe_moe_forward_mixed) takes at T tokens
    of x_dtype (a torch dtype; default bf16 -- fp32 tokens always stream)."""
    dt = SMOE_F32 if x_dtype == torch.float32 else SMOE_BF16
    return int(load().smoe_moe_path_dtype(ctypes.byref(layer.desc), T, dt))


def forward_noalloc(layer: MoELayer, x: torch.Tensor, y=None, ids=None, w=None, stream=None):
    """smoe_moe_forward_noalloc: the forward with the library's built-in
    workspace (no workspace argument; calls on one device must not overlap)."""
    if layer.expert_bits is not None:
        raise ValueError("smoe_moe_forward_noalloc takes layers of one depth only")
    T = x.shape[0]
    if y is None:
        y = torch.empty((T, layer.d), dtype=torch.float32, device=x.device)
    dt = SMOE_BF16 if x.dtype == torch.bfloat16 else SMOE_F32
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("x must be fp32 or bf16")
    _check(load().smoe_moe_forward_noalloc(ctypes.byref(layer.desc), _ptr(x), dt, T, _ptr(y),
                                           _ptr(ids), _ptr(w), _stream(stream)),
           "smoe_moe_forward_noalloc")
    return y


def forward_stage(layer: MoELayer, stage: int, x: torch.Tensor, ws: torch.Tensor, y: torch.Tensor,
                  ids=None, w=None, stream=None):
    """smoe_moe_forward_stage (smoe_moe_forward_stage_mixed for a layer with
    per-expert depths): one of the forward's three launch stages."""
    dt = SMOE_BF16 if x.dtype == torch.bfloat16 else SMOE_F32
    if layer.expert_bits is not None:
        _check(load().smoe_moe_forward_stage_mixed(ctypes.byref(layer.desc), layer._ebits, _ptr(x),
                                                   dt, x.shape[0], _ptr(y), _ptr(ws), ws.numel(),
                                                   _ptr(ids), _ptr(w), stage, _stream(stream)),
               f"smoe_moe_forward_stage_mixed({stage})")
        return y
    _check(load().smoe_moe_forward_stage(ctypes.byref(layer.desc), _ptr(x), dt, x.shape[0],
                                         _ptr(y), _ptr(ws), ws.numel(), _ptr(ids), _ptr(w), stage,
                                         _stream(stream)), f"smoe_moe_forward_stage({stage})")
    return y


def vault_parse(meta: bytes, file_bytes: int) -> "VaultInfo":
    """smoe_vault_parse on a host byte string (the file's metadata region)."""
    info = VaultInfo()
    buf = ctypes.create_string_buffer(bytes(meta), len(meta))
    _check(load().smoe_vault_parse(buf, len(meta), file_bytes, ctypes.byref(info)),
           "smoe_vault_parse")
    return info


def vault_find_expert(meta: bytes, file_bytes: int, layer: int, expert: int) -> "VaultExpert":
    out = VaultExpert()
    buf = ctypes.create_string_buffer(bytes(meta), len(meta))
    _check(load().smoe_vault_find_expert(buf, len(meta), file_bytes, layer, expert,
                                         ctypes.byref(out)), "smoe_vault_find_expert")
    return out


def vault_repack_layer(meta: bytes, vault_dev: torch.Tensor, layer: int, num_experts: int,
                       d: int, f: int, bits: int, stream=None) -> torch.Tensor:
    """smoe_vault_repack_layer: the layer's tile bank from a device copy of
    the vault (uint8 tensor holding the whole file)."""
    n = load().smoe_repacked_bytes(d, f, num_experts, bits, 64)
    tiles = torch.empty(n, dtype=torch.uint8, device=vault_dev.device)
    buf = ctypes.create_string_buffer(bytes(meta), len(meta))
    _check(load().smoe_vault_repack_layer(buf, len(meta), _ptr(vault_dev), vault_dev.numel(), layer,
                                          num_experts, _ptr(tiles), n, _stream(stream)),
           "smoe_vault_repack_layer")
    return tiles


def device_status(stream=None) -> int:
    return int(load().smoe_get_device_status(_stream(stream)))


def debug_set_waits(poll_cycles: int = 0, stall_routing: bool = False):
    """Testing only (smoe_debug_set_waits): short bounded waits in the layer
    kernel and, with stall_routing, a routing step that waits for logits no
    CTA writes; debug_set_waits() restores the defaults."""
    load().smoe_debug_set_waits(int(poll_cycles), 1 if stall_routing else 0)


def synth_bf16(out: torch.Tensor, key: int, sigma: float, p_out=0.0, out_mult=10.0, p_zero=0.0,
               start=0, stream=None):
    """Fill a CUDA uint16/bf16 tensor with the seeded generator's bf16 bits."""
    import numpy as np
    t_out = min(int(round(p_out * 4294967296.0)), 1 << 32)
    t_zero = min(int(round(p_zero * 4294967296.0)), 1 << 32)
    rc = load_synth().smoe_synth_bf16(_ptr(out), out.numel(), start, key,
                                      float(np.float32(sigma)), float(np.float32(sigma * out_mult)),
                                      t_out, t_zero, _stream(stream))
    if rc != 0:
        raise RuntimeError(f"smoe_synth_bf16 failed ({rc})")
    return out
