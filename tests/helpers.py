"""Shared helpers for the GPU parity tests: build a layer on the device from
seeded host weights, quantised either by the oracle (then copied up) or by
the GPU, and evaluate the oracle on the same inputs."""
from __future__ import annotations

import numpy as np

import oracle as O
from bit_expert_weight_gb300 import synth as Y

ROLES = (Y.ROLE_GATE, Y.ROLE_UP, Y.ROLE_DOWN)


def to_dev_bf16(bits_u16, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits_u16).view(np.int16)).to(dev).view(
        torch.bfloat16)


def to_dev(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


class HostLayer:
    """Seeded weights of one layer, quantised by the oracle."""

    def __init__(self, wl: Y.Workload, layer: int, bits: int, experts=None, expert_bits=None):
        """expert_bits: per-expert depths (a mixed layer; `bits` is then the
        shared expert's depth)."""
        self.wl, self.layer, self.bits = wl, layer, bits
        self.d, self.f, self.E, self.k = wl.d, wl.f, wl.E, wl.k
        self.router = wl.router_weight(layer)
        self.experts = list(range(wl.E)) if experts is None else list(experts)
        self.expert_bits = None if expert_bits is None else [int(b) for b in expert_bits]
        self.q = {}      # expert -> [q_gate, q_up, q_down] (oracle quantised)
        self.blob = {}
        for e in self.experts:
            be = bits if expert_bits is None else self.expert_bits[e]
            qs = [O.quantize(wl.expert_weight(layer, e, r), be) for r in ROLES]
            self.q[e] = qs
            self.blob[e] = O.make_blob(*qs)
        self.shared_blob = None
        self.shared_gate = None
        if wl.shared_f:
            qs = [O.quantize(wl.expert_weight(layer, Y.SHARED_EXPERT, r), bits) for r in ROLES]
            self.q["shared"] = qs
            self.shared_blob = O.make_blob(*qs)
            if wl.shared_gate:
                self.shared_gate = wl.shared_gate_weight(layer)

    def device_layer(self, dev, expert_bias=None):
        """Upload oracle-quantised streams, repack them on the GPU, return a MoELayer."""
        import bit_expert_weight_gb300.smoe as S
        codes, scales = [], []
        for e in range(self.E):
            for q in self.q[e]:
                codes.append(to_dev(q["codes_lsb"], dev))
                scales.append(to_dev(q["scales_f16"].view(np.int16), dev))
        if self.expert_bits is None:
            tiles = S.repack(codes, scales, self.d, self.f, self.E, self.bits)
        else:
            tiles = S.repack_mixed(codes, scales, self.d, self.f, self.expert_bits)
        sh_tiles, sh_gate = None, None
        if self.shared_blob is not None:
            sc = [to_dev(q["codes_lsb"], dev) for q in self.q["shared"]]
            ss = [to_dev(q["scales_f16"].view(np.int16), dev) for q in self.q["shared"]]
            sh_tiles = S.repack(sc, ss, self.d, self.wl.shared_f, 1, self.bits)
            if self.shared_gate is not None:
                sh_gate = to_dev_bf16(self.shared_gate, dev)
        bias_t = None if expert_bias is None else to_dev(expert_bias.astype(np.float32), dev)
        lay = S.MoELayer(self.d, self.f, self.E, self.k, self.wl.norm, self.bits,
                         to_dev_bf16(self.router, dev), tiles, expert_bias=bias_t,
                         shared_tiles=sh_tiles, shared_f=self.wl.shared_f, shared_gate_w=sh_gate,
                         expert_bits=self.expert_bits)
        lay._keep = (codes, scales)
        return lay

    def oracle_forward(self, x, expert_bias=None, **router):
        return O.moe_forward(self.d, self.f, self.E, self.k, self.wl.norm, self.bits,
                             self.router, self.blob, x, expert_bias=expert_bias,
                             shared_blob=self.shared_blob, fs=self.wl.shared_f,
                             shared_gate=self.shared_gate, expert_bits=self.expert_bits, **router)

    def oracle_apply(self, x, ids, w):
        return O.moe_apply(self.d, self.f, self.E, self.k, self.bits, self.blob, x, ids, w,
                           shared_blob=self.shared_blob, fs=self.wl.shared_f,
                           shared_gate=self.shared_gate, expert_bits=self.expert_bits)


def near_tie_tokens(logits, k, bias=None, rel=1e-5):
    """Tokens whose k-th and (k+1)-th selection keys are within rel*max|l|."""
    key = logits if bias is None else (logits + bias[None, :]).astype(np.float32)
    out = []
    for t in range(key.shape[0]):
        s = np.sort(key[t])[::-1]
        if k < s.size and abs(s[k - 1] - s[k]) < rel * max(np.abs(logits[t]).max(), 1e-30):
            out.append(t)
    return out


def check_forward(y, ids_gpu, w_gpu, hl: HostLayer, x, expert_bias=None, tol=1e-3):
    """Compare a GPU forward with the oracle: ids bit-exact except on near-tie
    tokens (which are then recomputed by the oracle with the GPU's routing),
    weights within 1e-5, y within tol * ||y_ref||_inf."""
    y_ref, ids_ref, w_ref, lg = hl.oracle_forward(x, expert_bias)
    ties = set(near_tie_tokens(lg, hl.k, expert_bias))
    mism = [t for t in range(x.shape[0]) if not np.array_equal(ids_gpu[t], ids_ref[t])]
    assert set(mism) <= ties, f"routing differs on non-tie tokens {sorted(set(mism) - ties)}"
    if mism:
        y_ref = y_ref.copy()
        y_ref[mism] = hl.oracle_apply(x[mism], ids_gpu[mism], w_gpu[mism])
        w_ref = w_ref.copy()
        w_ref[mism] = w_gpu[mism]
    assert np.allclose(w_gpu, w_ref, rtol=1e-5, atol=1e-6)
    err = float(np.abs(y - y_ref).max())
    bound = tol * float(np.abs(y_ref).max())
    assert err <= bound, f"max abs err {err:.3e} > {bound:.3e}"
    return err, bound, len(mism)
