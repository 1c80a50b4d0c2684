"""Seeded synthetic inputs shared by the tests, the oracle checks and the bench.

This module holds none of the method's arithmetic: it only draws numbers.
Every tensor comes from one counter-based generator, so any expert of any
layer can be regenerated on the host by itself, bit for bit, and the device
twin in ``csrc/synth.cu`` (used by the benchmark to fill ~100 GB of weights)
produces the same bits.

Generator (counter-based SplitMix64, Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; finaliser constants of Stafford's
"Mix13" variant as in Vigna's public splitmix64.c):

    mix64(z) = let z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
                   z = (z ^ (z >> 27)) * 0x94D049BB133111EB
               in  z ^ (z >> 31)
    word(key, i) = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)    (mod 2^64)

Element ``i`` of a stream with key ``key`` uses words 4i .. 4i+3:
  * words 4i..4i+2 give twelve 16-bit uniforms u_0..u_11 (low half first);
    C = 2 * sum(u) - 12 * 65535 is an integer with mean 0 and standard
    deviation ~2^17, so z = C * 2^-17 is an Irwin-Hall(12) approximation of
    N(0, 1) that is exact in fp32;
  * word 4i+3: low 32 bits < p_out * 2^32 marks an outlier, high 32 bits
    < p_zero * 2^32 marks an exact zero.
The value is fl32(z * s) with s = fl32(sigma) or fl32(sigma * outlier_mult),
then zeroed if marked, then rounded to bf16 (nearest, ties to even).

Stream keys: key(seed, a, b, c) = mix64(mix64(mix64(mix64(seed + G) ^ a) ^ b) ^ c)
with G the golden gamma above; (a, b, c) name the tensor, e.g.
(layer, expert, role) with role 0/1/2 = gate/up/down, 3 = router,
4 = activations, 5 = shared-expert gate vector, 6 = expert bias.
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
M1 = np.uint64(0xBF58476D1CE4E5B9)
M2 = np.uint64(0x94D049BB133111EB)
MASK64 = (1 << 64) - 1

ROLE_GATE, ROLE_UP, ROLE_DOWN, ROLE_ROUTER, ROLE_X, ROLE_SHARED_GATE, ROLE_BIAS = range(7)
SHARED_EXPERT = 0xFFFF  # expert index used for the shared expert's streams


def _mix64_int(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, a: int = 0, b: int = 0, c: int = 0) -> int:
    k = _mix64_int(seed + 0x9E3779B97F4A7C15)
    k = _mix64_int(k ^ (a & MASK64))
    k = _mix64_int(k ^ (b & MASK64))
    return _mix64_int(k ^ (c & MASK64))


def _mix64(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * M1
        z = (z ^ (z >> np.uint64(27))) * M2
    return z ^ (z >> np.uint64(31))


def words(key: int, start: int, count: int) -> np.ndarray:
    """SplitMix64 outputs word(key, start) .. word(key, start + count - 1)."""
    i = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + i * GAMMA
    return _mix64(z)


def _thresh(p: float) -> int:
    return min(int(round(p * 4294967296.0)), 0xFFFFFFFF + 1)


def _f32_to_bf16_rne(v: np.ndarray) -> np.ndarray:
    u = v.astype(np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def values_f32(key: int, n: int, sigma: float, p_out: float = 0.0, out_mult: float = 10.0,
               p_zero: float = 0.0, start: int = 0, chunk: int = 1 << 22) -> np.ndarray:
    """fp32 values of elements start .. start+n-1 of a stream (before bf16)."""
    s_norm = np.float32(sigma)
    s_out = np.float32(sigma * out_mult)
    t_out = np.uint64(_thresh(p_out))
    t_zero = np.uint64(_thresh(p_zero))
    out = np.empty(n, np.float32)
    for c0 in range(0, n, chunk):
        m = min(chunk, n - c0)
        w = words(key, 4 * (start + c0), 4 * m).reshape(m, 4)
        acc = np.zeros(m, np.int64)
        for q in range(3):
            x = w[:, q]
            for h in range(4):
                acc += ((x >> np.uint64(16 * h)) & np.uint64(0xFFFF)).astype(np.int64)
        C = 2 * acc - 12 * 65535
        z = C.astype(np.float32) * np.float32(2.0 ** -17)
        fl = w[:, 3]
        is_out = (fl & np.uint64(0xFFFFFFFF)) < t_out
        is_zero = (fl >> np.uint64(32)) < t_zero
        s = np.where(is_out, s_out, s_norm).astype(np.float32)
        v = (z * s).astype(np.float32)
        v[is_zero] = np.float32(0.0)
        out[c0:c0 + m] = v
    return out


def values_bf16_numpy(key: int, n: int, sigma: float, p_out: float = 0.0,
                      out_mult: float = 10.0, p_zero: float = 0.0, start: int = 0) -> np.ndarray:
    """bf16 bit patterns (uint16) of a stream: the definition, in numpy."""
    return _f32_to_bf16_rne(values_f32(key, n, sigma, p_out, out_mult, p_zero, start))


# The same stream computed by csrc/synth_host.c (plain C, built here with gcc
# on first use): identical bits, about a hundred times faster, so that whole
# full-size experts can be regenerated on the host.
_HOST_SO = None


def _host_lib():
    global _HOST_SO
    if _HOST_SO is None:
        import ctypes
        import os
        import subprocess
        here = os.path.dirname(os.path.abspath(__file__))
        src = os.path.join(here, "csrc", "synth_host.c")
        out_dir = os.path.join(here, "_build")
        so = os.path.join(out_dir, "libsynth_host.so")
        os.makedirs(out_dir, exist_ok=True)
        if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
            tmp = so + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                                   "-shared", "-o", tmp, src])
            os.replace(tmp, so)
        lib = ctypes.CDLL(so)
        lib.synth_values_bf16.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_float,
                                          ctypes.c_float, ctypes.c_uint64, ctypes.c_uint64,
                                          ctypes.c_int64, ctypes.c_void_p]
        lib.synth_values_bf16.restype = ctypes.c_int
        _HOST_SO = lib
    return _HOST_SO


def values_bf16(key: int, n: int, sigma: float, p_out: float = 0.0, out_mult: float = 10.0,
                p_zero: float = 0.0, start: int = 0) -> np.ndarray:
    """bf16 bit patterns (uint16) of a stream (the C twin of
    values_bf16_numpy; tests/test_synth.py checks the two agree)."""
    out = np.empty(n, np.uint16)
    if n:
        _host_lib().synth_values_bf16(key & MASK64, n, float(np.float32(sigma)),
                                      float(np.float32(sigma * out_mult)), _thresh(p_out),
                                      _thresh(p_zero), start, out.ctypes.data)
    return out


# ------------------------------------------------------------------ workloads

class Workload:
    """A synthetic MoE layer workload shaped like one of the pages' models."""

    def __init__(self, name, d, f, E, k, norm, bits_list, T_list, layers, seed,
                 x_dtype="bf16", p_out=0.01, p_zero=0.0, router_p_out=None,
                 router_p_zero=None, shared_f=0, shared_gate=False, zipf_s=None, zipf_tau=None):
        self.name, self.d, self.f, self.E, self.k, self.norm = name, d, f, E, k, norm
        self.bits_list, self.T_list, self.layers, self.seed = bits_list, T_list, layers, seed
        self.x_dtype, self.p_out, self.p_zero = x_dtype, p_out, p_zero
        self.router_p_out = p_out if router_p_out is None else router_p_out
        self.router_p_zero = p_zero if router_p_zero is None else router_p_zero
        self.shared_f, self.shared_gate, self.zipf_s = shared_f, shared_gate, zipf_s
        self.zipf_tau = zipf_tau

    sigma = 0.02

    def expert_weight(self, layer, expert, role):
        """bf16 [rows, cols] of gate (0) / up (1) / down (2) in HF [out, in]."""
        f = self.shared_f if expert == SHARED_EXPERT else self.f
        rows, cols = (f, self.d) if role in (ROLE_GATE, ROLE_UP) else (self.d, f)
        key = stream_key(self.seed, layer, expert, role)
        return values_bf16(key, rows * cols, self.sigma, self.p_out, 10.0,
                           self.p_zero).reshape(rows, cols)

    def router_weight(self, layer):
        key = stream_key(self.seed, layer, 0, ROLE_ROUTER)
        return values_bf16(key, self.E * self.d, self.sigma, self.router_p_out, 10.0,
                           self.router_p_zero).reshape(self.E, self.d)

    def shared_gate_weight(self, layer):
        key = stream_key(self.seed, layer, SHARED_EXPERT, ROLE_SHARED_GATE)
        return values_bf16(key, self.d, self.sigma).reshape(self.d)

    # ---------------------------------------------------------- Zipf routing
    # Workload construction for the batched Qwen-like config: expert
    # popularity p_e proportional to rank^-s over a seeded permutation, turned
    # into the selection-only expert_bias tau * ln p_e; tau is calibrated so
    # that the share of tokens whose top-k contains the most popular expert
    # matches p_1 within 10 %.  The same bias array is an input to both the
    # GPU path and the oracle.

    def zipf_ranks(self):
        """rank[e] in 1..E (1 = most popular), a seeded permutation."""
        key = stream_key(self.seed, 0, 0, ROLE_BIAS)
        order = np.argsort(words(key, 0, self.E), kind="stable")
        rank = np.empty(self.E, dtype=np.int64)
        rank[order] = np.arange(1, self.E + 1)
        return rank

    def zipf_p(self):
        r = self.zipf_ranks().astype(np.float64) ** (-self.zipf_s)
        return r / r.sum()

    def zipf_bias(self, tau=None):
        """fp32 [E] selection-only bias tau * ln p_e."""
        tau = self.zipf_tau if tau is None else tau
        return (tau * np.log(self.zipf_p())).astype(np.float32)

    def zipf_logits(self, layer, n_tokens):
        x, _ = self.activations(layer, n_tokens)
        r = bf16_to_f32(self.router_weight(layer)).astype(np.float64)
        return x.astype(np.float64) @ r.T

    def zipf_share(self, layer, tau, n_tokens, logits=None):
        """Share of the first n_tokens tokens whose top-k (by logit plus bias,
        numpy argpartition) contains the most popular expert."""
        lg = self.zipf_logits(layer, n_tokens) if logits is None else logits
        key = lg + self.zipf_bias(tau).astype(np.float64)
        top = np.argpartition(-key, self.k - 1, axis=1)[:, :self.k]
        hot = int(np.argmin(self.zipf_ranks()))
        return float(np.mean(np.any(top == hot, axis=1)))

    def calibrate_zipf_tau(self, layer=0, n_tokens=4096, iters=30):
        """Bisection on tau in [0, 8] for share(tau) = p_1 (within 10 %)."""
        target = float(self.zipf_p().max())
        lg = self.zipf_logits(layer, n_tokens)
        lo, hi = 0.0, 8.0
        for _ in range(iters):
            mid = 0.5 * (lo + hi)
            sh = self.zipf_share(layer, mid, n_tokens, lg)
            if abs(sh - target) <= 0.1 * target:
                return mid, sh, target
            if sh < target:
                lo = mid
            else:
                hi = mid
        return mid, sh, target

    def mixed_bits(self, q4_share=0.25):
        """Per-expert depths of a mixed layer: the round(q4_share * E) most
        popular experts (zipf_ranks) at Q4, the others at Q2 -- more bits
        where the router sends more tokens."""
        n4 = int(round(q4_share * self.E))
        return [4 if int(r) <= n4 else 2 for r in self.zipf_ranks()]

    def activations(self, layer, T, start_token=0):
        """x [T, d]: fp32 values (bf16-rounded when x_dtype == 'bf16').

        Returns (x_f32, x_bits) where x_bits is the uint16 bf16 pattern for
        bf16 workloads and None for fp32 ones."""
        key = stream_key(self.seed, layer, 0, ROLE_X)
        if self.x_dtype == "bf16":
            # the bf16 rounding of the fp32 stream, i.e. values_bf16 (C twin)
            bits = values_bf16(key, T * self.d, 1.0, start=start_token * self.d).reshape(T, self.d)
            return bf16_to_f32(bits), bits
        v = values_f32(key, T * self.d, 1.0, start=start_token * self.d).reshape(T, self.d)
        return v, None


WORKLOADS = {
    "tiny": Workload("tiny MoE layer d256 f128 E8 k2 renorm Q4", 256, 128, 8, 2, True, [4], [4],
                     1, 0, x_dtype="f32", p_out=0.01, p_zero=0.20),
    "deepseek16b": Workload("DeepSeek-MoE-16B-like layer d2048 f1408 E64 k6", 2048, 1408, 64, 6,
                            False, [4, 2], [1], 27, 1),
    "qwen235b": Workload("Qwen3-235B-like decode d4096 f1536 E128 k8 renorm Q4", 4096, 1536, 128,
                         8, True, [4], [1], 94, 2),
    "qwen235b_batched": Workload("Qwen3-235B-like layer batched (Zipf 1.1)", 4096, 1536, 128, 8,
                                 True, [4], [1, 8, 64, 512, 4096], 1, 3, zipf_s=1.1,
                                 # calibrate_zipf_tau(layer 0, 4096 tokens): share 0.2424 vs p_1 0.2257
                                 zipf_tau=0.375),
    # the largest layer the kernels take (d, f, shared f and k at their limits)
    "edge_max": Workload("maximum-size layer d4096 f2048 E16 k16 + shared 2048", 4096, 2048, 16,
                         16, True, [4, 2], [1, 9], 1, 5, shared_f=2048, shared_gate=True),
    "a3b35b": Workload("35B-A3B-like fine-grained layer d2048 f512 E256 k8 + shared", 2048, 512,
                       256, 8, True, [4, 2], [1, 256], 40, 4, shared_f=512, shared_gate=True),
}
