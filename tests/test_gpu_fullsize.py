"""GPU parity at the full layer geometries of the benchmark workloads, in the
launch configuration bench.py times (one layer per forward call).

The oracle cannot run a whole full-size layer in seconds, so each test
samples a few tokens: the oracle routes them from fixed host logits and
quantises only the experts they select; every other expert is generated and
quantised on the device (it does not affect the sampled tokens).  The GPU
forward runs over all T tokens; the sampled rows of y, their expert ids
(bit-exact except near ties) and weights are compared with the oracle.
"""
import multiprocessing as mp
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O  # noqa: E402
from bit_expert_weight_gb300 import synth as Y  # noqa: E402

from helpers import near_tie_tokens, to_dev, to_dev_bf16  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ROLES = (Y.ROLE_GATE, Y.ROLE_UP, Y.ROLE_DOWN)


def _oracle_expert(args):
    """Pool worker: host weights of one expert, quantised by the oracle."""
    wl_name, layer, e, bits = args
    wl = Y.WORKLOADS[wl_name]
    qs = [O.quantize(wl.expert_weight(layer, e, r), bits) for r in ROLES]
    return e, [(q["codes_lsb"], q["scales_f16"]) for q in qs]


@pytest.fixture(scope="module")
def pool():
    # spawn: the workers never inherit a CUDA context
    p = mp.get_context("spawn").Pool(max(1, min(16, os.cpu_count() or 1)))
    yield p
    p.close()
    p.join()


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_expert_weight_gb300 import build
    build.build()
    import bit_expert_weight_gb300.smoe as S
    S.load()
    return S


class FullLayer:
    """One full-geometry layer: oracle-quantised experts for the sampled
    tokens' selections, device-quantised experts elsewhere."""

    def __init__(self, S, pool, wl_name, layer, bits, sample, bias=None, expert_bits=None):
        """expert_bits: per-expert depths (a mixed layer; `bits` is then the
        shared expert's depth)."""
        wl = Y.WORKLOADS[wl_name]
        self.wl, self.layer, self.bits, self.sample, self.bias = wl, layer, bits, list(sample), bias
        self.expert_bits = None if expert_bits is None else [int(b) for b in expert_bits]
        bits_of = (lambda e: bits) if expert_bits is None else (lambda e: self.expert_bits[e])
        self.router = wl.router_weight(layer)
        xs = np.stack([wl.activations(layer, 1, start_token=t)[0][0] for t in self.sample])
        self.x_sample = xs
        lg = O.router_logits(self.router, xs)
        ids, _ = O.route(lg, wl.k, wl.norm, bias)
        self.logits = lg
        chosen = sorted(set(int(e) for e in np.asarray(ids).ravel()))
        jobs = [(wl_name, layer, e, bits_of(e)) for e in chosen]
        if wl.shared_f:
            jobs.append((wl_name, layer, Y.SHARED_EXPERT, bits))
        got = dict(pool.map(_oracle_expert, jobs))
        self.blob = {e: O.make_blob(*[{"codes_lsb": c, "scales_f16": s} for c, s in got[e]])
                     for e in chosen}
        self.shared_blob = None
        if wl.shared_f:
            self.shared_blob = O.make_blob(*[{"codes_lsb": c, "scales_f16": s}
                                             for c, s in got[Y.SHARED_EXPERT]])
        # device bank
        codes, scales = [], []
        for e in range(wl.E):
            for r_i, r in enumerate(ROLES):
                if e in got:
                    c, s = got[e][r_i]
                    codes.append(to_dev(c, DEV))
                    scales.append(to_dev(s.view(np.int16), DEV))
                else:
                    c, s = self._device_quantised(S, e, r, bits_of(e))
                    codes.append(c)
                    scales.append(s)
        if expert_bits is None:
            tiles = S.repack(codes, scales, wl.d, wl.f, wl.E, bits)
        else:
            tiles = S.repack_mixed(codes, scales, wl.d, wl.f, self.expert_bits)
        sh_tiles, sh_gate = None, None
        if wl.shared_f:
            sc = [to_dev(c, DEV) for c, _ in got[Y.SHARED_EXPERT]]
            ss = [to_dev(s.view(np.int16), DEV) for _, s in got[Y.SHARED_EXPERT]]
            sh_tiles = S.repack(sc, ss, wl.d, wl.shared_f, 1, bits)
            if wl.shared_gate:
                self.shared_gate = wl.shared_gate_weight(layer)
                sh_gate = to_dev_bf16(self.shared_gate, DEV)
        if not wl.shared_gate:
            self.shared_gate = None
        bias_t = None if bias is None else to_dev(bias.astype(np.float32), DEV)
        self.lay = S.MoELayer(wl.d, wl.f, wl.E, wl.k, wl.norm, bits, to_dev_bf16(self.router, DEV),
                              tiles, expert_bias=bias_t, shared_tiles=sh_tiles, shared_f=wl.shared_f,
                              shared_gate_w=sh_gate, expert_bits=self.expert_bits)
        del codes, scales

    def _device_quantised(self, S, e, role, bits):
        wl = self.wl
        rows, cols = (wl.f, wl.d) if role in (Y.ROLE_GATE, Y.ROLE_UP) else (wl.d, wl.f)
        w = torch.empty(rows * cols, dtype=torch.int16, device=DEV)
        S.synth_bf16(w, Y.stream_key(wl.seed, self.layer, e, role), wl.sigma, p_out=wl.p_out,
                     p_zero=wl.p_zero)
        return S.quantize(w.view(torch.bfloat16).view(rows, cols), bits)

    def device_x(self, S, T):
        """x [T, d] bf16 on the device: the generator's device twin."""
        wl = self.wl
        x = torch.empty(T * wl.d, dtype=torch.int16, device=DEV)
        S.synth_bf16(x, Y.stream_key(wl.seed, self.layer, 0, Y.ROLE_X), 1.0)
        return x.view(torch.bfloat16).view(T, wl.d)

    def check(self, S, T, tol=None, path=None, x_f32=False):
        """tol defaults to the bar of the path the forward takes: 1e-3 on the
        streaming path (fp32 accumulation), 2e-2 on the grouped tensor-core
        path (bf16 operands).  path forces a path (smoe_moe_forward_path).
        Sampled tokens at or past T are skipped.  x_f32: the tokens as fp32
        values of the seeded stream (not rounded to bf16)."""
        wl = self.wl
        xdt = torch.float32 if x_f32 else torch.bfloat16
        grouped = (path == S.PATH_GROUPED or
                   (path in (None, S.PATH_AUTO) and S.path_for(self.lay, T, xdt) == S.PATH_GROUPED))
        if tol is None:
            tol = 2e-2 if grouped else 1e-3
        sample = [t for t in self.sample if t < T]
        assert sample
        if x_f32:
            key = Y.stream_key(wl.seed, self.layer, 0, Y.ROLE_X)
            xh = Y.values_f32(key, T * wl.d, 1.0).reshape(T, wl.d)
            xt = torch.from_numpy(xh).to(DEV)
            x_sample = xh[sample]
        else:
            xt = self.device_x(S, T)
            x_sample = self.x_sample[[self.sample.index(t) for t in sample]]
        ws = S.workspace(self.lay, T)
        ids = torch.empty((T, wl.k), dtype=torch.int32, device=DEV)
        w = torch.empty((T, wl.k), dtype=torch.float32, device=DEV)
        y = S.forward(self.lay, xt, ws, ids=ids, w=w, path=path)
        torch.cuda.synchronize()
        assert S.device_status() == 0
        # the device x rows are the host generator's rows, bit for bit
        xs = xt[sample].float().cpu().numpy()
        assert np.array_equal(xs, x_sample)
        yg = y[sample].cpu().numpy()
        idg = ids[sample].cpu().numpy()
        wg = w[sample].cpu().numpy()
        y_ref, ids_ref, w_ref, lg = O.moe_forward(wl.d, wl.f, wl.E, wl.k, wl.norm, self.bits,
                                                  self.router, self.blob, x_sample,
                                                  expert_bias=self.bias,
                                                  shared_blob=self.shared_blob, fs=wl.shared_f,
                                                  shared_gate=self.shared_gate,
                                                  expert_bits=self.expert_bits)
        ties = set(near_tie_tokens(lg, wl.k, self.bias))
        mism = [i for i in range(len(sample)) if not np.array_equal(idg[i], ids_ref[i])]
        assert set(mism) <= ties, f"routing differs on non-tie sampled tokens {mism}"
        ok = [i for i in range(len(sample)) if i not in mism]
        assert np.allclose(wg[ok], w_ref[ok], rtol=1e-5, atol=1e-6)
        err = float(np.abs(yg[ok] - y_ref[ok]).max()) if ok else 0.0
        bound = tol * float(np.abs(y_ref[ok]).max()) if ok else 1.0
        assert err <= bound, f"T={T}: max abs err {err:.3e} > {bound:.3e}"
        return err, bound


@pytest.mark.parametrize("bits", [4, 2])
def test_deepseek16b_layer_full_size(S, pool, bits):
    fl = FullLayer(S, pool, "deepseek16b", 0, bits, sample=[0])
    fl.check(S, 1)


@pytest.mark.parametrize("layer", [0, 31, 62, 93])
def test_qwen235b_decode_layer_full_size(S, pool, layer):
    """The 94-layer Qwen3-235B-like decode stack, spot-checked on four
    evenly spaced layers (each its own seeded weights and token)."""
    fl = FullLayer(S, pool, "qwen235b", layer, 4, sample=[0])
    fl.check(S, 1)


@pytest.mark.parametrize("bits", [4, 2])
def test_a3b35b_layer_full_size(S, pool, bits):
    """Shared expert with a sigmoid gate; T = 1 and T = 256 (sampled)."""
    fl = FullLayer(S, pool, "a3b35b", 0, bits, sample=[0, 3, 255])
    fl.check(S, 256)
    fl1 = FullLayer(S, pool, "a3b35b", 1, bits, sample=[0])
    fl1.check(S, 1)


@pytest.mark.parametrize("bits", [4, 2])
def test_a3b35b_grouped_path_full_size(S, pool, bits):
    """The 256-token batch forced onto the grouped path: 256 experts (two
    128-expert tiles of router logits), the gated shared expert as a
    segment of all 256 tokens, Q4 and Q2."""
    fl = FullLayer(S, pool, "a3b35b", 2, bits, sample=[0, 100, 255])
    fl.check(S, 256, path=S.PATH_GROUPED)


def segment_picks(wl, layer, T, bias):
    """Tokens whose grouped-path rows lie where the first tokens' rows never
    do.  The sort is stable in token order, so the rank of a token among the
    tokens that chose expert e is its row in e's segment: the hot expert's
    rank-128 and rank-200 tokens (the second m-tile, at 4,096 tokens the
    second accumulator of a paired item), its last token (the ragged last
    m-tile), the last token of a segment of 33..64 rows (a 64-row activation
    box) and of one of 1..32 rows (a 32-row box), and token T - 1.  Picked
    from a host routing of all T tokens (fp64 logits plus the bias, top-k
    with ties to the lower index); the oracle still routes the picked tokens
    itself.  Returns (tokens, {what: token})."""
    x, _ = wl.activations(layer, T)
    r = Y.bf16_to_f32(wl.router_weight(layer)).astype(np.float64)
    key = x.astype(np.float64) @ r.T
    if bias is not None:
        key = key + bias.astype(np.float64)
    top = np.argsort(-key, axis=1, kind="stable")[:, :wl.k]
    counts = np.bincount(top.ravel(), minlength=wl.E)
    hot = int(np.argmax(counts))
    rows_hot = np.nonzero((top == hot).any(axis=1))[0]
    what = {"last token": T - 1, "hot last row": int(rows_hot[-1])}
    if len(rows_hot) > 128:
        what["hot row 128"] = int(rows_hot[128])
    if len(rows_hot) > 200:
        what["hot row 200"] = int(rows_hot[200])
    for name, lo, hi in (("64-row box", 33, 64), ("32-row box", 1, 32)):
        cand = [e for e in range(wl.E) if lo <= counts[e] <= hi]
        if cand:
            what[name] = int(np.nonzero((top == cand[0]).any(axis=1))[0][-1])
    return sorted(set(what.values())), what


def test_segment_picks_reach_the_second_m_tile():
    """At 4,096 tokens (256 routed rows per expert on average: paired
    m-tiles) the hot expert's segment spans several m-tiles, so the picks
    include a second-m-tile row and a ragged last m-tile."""
    wl = Y.WORKLOADS["qwen235b_batched"]
    toks, what = segment_picks(wl, 0, 4096, wl.zipf_bias())
    assert "hot row 128" in what and "hot row 200" in what
    assert what["last token"] == 4095 and all(0 <= t < 4096 for t in toks)


def test_qwen235b_batched_zipf_full_size(S, pool):
    """Zipf(1.1)-skewed selection bias; T = 8 and 64 with tokens 0 and 5,
    T = 512 and 4096 with tokens picked to reach the second m-tile of a
    paired item, the ragged last m-tile, the 64- and 32-row activation boxes
    and the last token (segment_picks)."""
    wl = Y.WORKLOADS["qwen235b_batched"]
    bias = wl.zipf_bias()
    fl = FullLayer(S, pool, "qwen235b_batched", 0, 4, sample=[0, 5], bias=bias)
    for T in (8, 64):
        fl.check(S, T)
    for T in (512, 4096):
        toks, _ = segment_picks(wl, 0, T, bias)
        fl = FullLayer(S, pool, "qwen235b_batched", 0, 4, sample=toks, bias=bias)
        fl.check(S, T)


def test_qwen235b_batched_mixed_depth_full_size(S, pool):
    """Mixed depths at the batched geometry: the 32 most popular experts
    (Zipf rank) at Q4, the other 96 at Q2, with the Zipf selection bias;
    T = 8 and 64 with tokens 0 and 5, T = 512 and 4096 (the benchmark's
    batch) with the segment_picks tokens."""
    wl = Y.WORKLOADS["qwen235b_batched"]
    bias = wl.zipf_bias()
    eb = wl.mixed_bits(0.25)
    fl = FullLayer(S, pool, "qwen235b_batched", 0, 4, sample=[0, 5], bias=bias, expert_bits=eb)
    for T in (64, 8):
        fl.check(S, T)
    for T in (512, 4096):
        toks, _ = segment_picks(wl, 0, T, bias)
        fl = FullLayer(S, pool, "qwen235b_batched", 0, 4, sample=toks, bias=bias, expert_bits=eb)
        fl.check(S, T)


def test_a3b35b_mixed_depth_full_size(S, pool):
    """256 experts at alternating depths and the gated shared expert at Q2."""
    fl = FullLayer(S, pool, "a3b35b", 3, 2, sample=[0, 200],
                   expert_bits=[4 if e % 2 == 0 else 2 for e in range(256)])
    fl.check(S, 256)


@pytest.mark.parametrize("bits", [4, 2])
def test_maximum_size_layer(S, pool, bits):
    """The largest layer the kernels take: d 4096 (two gate/up chunks per
    strip), f and shared f 2048 (a down strip fills one ring stage), k = E =
    16 with a gated shared expert; bf16 and fp32 tokens (hi + lo split); one
    token (fused routing and combine), 9 tokens (separate stages), 16 tokens
    on the grouped path."""
    fl = FullLayer(S, pool, "edge_max", 0, bits, sample=[0, 8])
    fl.check(S, 1)
    fl.check(S, 1, x_f32=True)
    fl.check(S, 9)
    fl.check(S, 9, x_f32=True)
    fl.check(S, 16, path=S.PATH_GROUPED)
