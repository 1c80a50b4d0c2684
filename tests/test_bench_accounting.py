"""bench.py's algorithmic bytes, flops and launch counts (the numerators of
the roofline it reports), checked on the CPU against sizes the pages print
and against counts written out by hand."""
import os
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from bit_expert_weight_gb300 import synth as Y  # noqa: E402


class FakeModel:
    """The fields of bench.DeviceModel the accounting reads."""

    def __init__(self, wl, bits, ids, T, x_dtype=torch.bfloat16, grouped=False):
        self.wl, self.bits, self.T, self.grouped = wl, bits, T, grouped
        self.expert_bits, self.shared_bits = bench.depths(wl, bits)
        self.ids = [torch.tensor(np.asarray(i, dtype=np.int32)) for i in ids]
        self.x = [torch.zeros((T, wl.d), dtype=x_dtype) for _ in ids]


def test_expert_bytes_match_the_pages_blob_sizes():
    # ".smoe Binary Format": a Qwen3-235B expert (d 4096, f 1536) is
    # 10,027,008 B at Q4 and 5,308,416 B at Q2 (codes + fp16 scales)
    wl = Y.WORKLOADS["qwen235b"]
    assert bench.expert_bytes(wl, wl.f, 4, 3) == 10_027_008
    assert bench.expert_bytes(wl, wl.f, 2, 3) == 5_308_416


def test_decode_layer_bytes():
    ds = Y.WORKLOADS["deepseek16b"]  # 6 selected experts of 4,595,712 B + router + x/y
    m = FakeModel(ds, 4, [[[0, 1, 2, 3, 4, 5]]], 1)
    assert bench.layer_algorithmic_bytes(m) == 6 * 4_595_712 + 64 * 2048 * 2 + 2048 * (2 + 4)
    qw = Y.WORKLOADS["qwen235b"]
    m = FakeModel(qw, 4, [[list(range(8))]], 1)
    assert bench.layer_algorithmic_bytes(m) == 8 * 10_027_008 + 128 * 4096 * 2 + 4096 * 6
    # the same expert chosen twice is read once
    m = FakeModel(ds, 4, [[[0, 1, 2, 3, 4, 5], [5, 4, 3, 2, 1, 0]]], 2)
    assert bench.layer_algorithmic_bytes(m) == 6 * 4_595_712 + 64 * 2048 * 2 + 2 * 2048 * 6


def test_mixed_depth_bytes_follow_each_experts_depth():
    qw = Y.WORKLOADS["qwen235b_batched"]
    m = FakeModel(qw, "mixed", [[list(range(8))]], 1)
    eb = m.expert_bits
    assert eb.count(4) == 32 and eb.count(2) == 96
    want = sum(10_027_008 if eb[e] == 4 else 5_308_416 for e in range(8))
    assert bench.layer_algorithmic_bytes(m) == want + 128 * 4096 * 2 + 4096 * 6


def test_gateup_flops_and_bytes():
    qw = Y.WORKLOADS["qwen235b_batched"]
    T = 4096
    ids = np.arange(T * 8, dtype=np.int32).reshape(T, 8) % 128
    m = FakeModel(qw, 4, [ids], T, grouped=True)
    assert bench.gateup_flops(m) == 4.0 * T * 8 * 4096 * 1536 == 824_633_720_832.0
    # every expert's gate and up (2/3 of its blob), token rows in, bf16 h out
    assert bench.gateup_bytes(m) == 128 * (2 * 10_027_008 // 3) + T * 4096 * 2 + T * 8 * 1536 * 2


def test_launches_per_layer():
    ds = Y.WORKLOADS["deepseek16b"]
    assert bench.launches_per_layer(FakeModel(ds, 4, [[[0] * 6]], 1)) == 1       # fused
    assert bench.launches_per_layer(FakeModel(ds, 4, [[[0] * 6] * 9], 9)) == 3   # router, layer, combine
    # grouped, bf16 tokens: logits GEMM, routing, sort, gather, 2 GEMMs, combine
    assert bench.launches_per_layer(FakeModel(ds, 4, [[[0] * 6]], 64, grouped=True)) == 7
    assert bench.launches_per_layer(
        FakeModel(ds, 4, [[[0] * 6]], 64, x_dtype=torch.float32, grouped=True)) == 6
    # two depths: one gate/up and one down GEMM per depth
    assert bench.launches_per_layer(FakeModel(ds, "mixed", [[[0] * 6]], 64, grouped=True)) == 9


def test_parity_and_routing_summaries():
    y_ref = np.array([[1.0, -2.0], [0.5, 4.0]])
    p = bench.parity_summary(y_ref + np.array([[0.0, 0.002], [0.0, 0.0]]), y_ref, 1e-3)
    assert p["max_abs_err"] == pytest.approx(0.002) and p["ref_max_abs"] == 4.0
    assert p["rel"] == pytest.approx(5e-4) and p["ok"]
    assert not bench.parity_summary(y_ref + 0.01, y_ref, 1e-3)["ok"]
    wl = Y.WORKLOADS["tiny"]
    E = wl.E
    bits = [4] * E
    bits[3] = 2
    r = bench.routing_summary([np.array([[0, 1], [1, 3]]), np.array([[1, 2], [3, 3]])], wl, bits, 4)
    assert r["histogram"] == [1, 3, 1, 3] + [0] * (E - 4)
    assert r["distinct_experts_per_layer"] == 3.0
    assert r["max_expert_share"] == 3 / 8
    # streamed weights: experts {0, 1, 3} and {1, 2, 3}, expert 3 at Q2, plus
    # the shared expert in each layer
    q4 = 3 * (wl.f * wl.d // 2 + wl.f * wl.d // 32)
    q2 = 3 * (wl.f * wl.d // 4 + wl.f * wl.d // 32)
    sh = 3 * (wl.shared_f * wl.d // 2 + wl.shared_f * wl.d // 32) if wl.shared_f else 0
    assert r["weight_MB_per_step"] * 1e6 == pytest.approx(4 * q4 + 2 * q2 + 2 * sh)


def test_oracle_leg_returns_time_and_output():
    """The CPU baseline leg times the oracle and keeps its output for the
    parity field (tiny workload, 2 tokens): one thread and several threads
    give the same output."""
    wl = Y.WORKLOADS["tiny"]
    preps = bench.prepare_oracle(wl, 4, [0], 2)
    sec, y = bench.time_oracle(wl, 4, preps[0])
    assert sec > 0 and y.shape == (2, wl.d) and np.isfinite(y).all()
    sec4, y4 = bench.time_oracle(wl, 4, preps[0], nthreads=4)
    assert sec4 > 0 and np.array_equal(y, y4)
    mean_s, passes, ys = bench.time_oracle_layers(wl, 4, preps, 2, 0.0)
    assert mean_s > 0 and passes == 1 and np.array_equal(ys[0], y)


def test_check_layers_are_the_spot_check_layers():
    """Qwen3-235B-like stack: the oracle spot-checks layers 0, 31, 62 and 93
    of 94; short stacks are checked whole."""
    assert bench.check_layers(94) == [0, 31, 62, 93]
    assert bench.check_layers(27) == [0, 9, 17, 26]
    assert bench.check_layers(2) == [0, 1]


def test_both_arms_print_the_same_config():
    """The reference arm's config dict is computed from the workload alone,
    like the GPU arm's (resident bytes of the 94-layer Q4 stack: 128 x 94 x
    10,027,008 B)."""
    wl = Y.WORKLOADS["qwen235b"]
    c = bench.config_dict(wl, 94, 1, 4, 1, True)
    assert c == bench.config_dict(wl, 94, 1, 4, 1, True)
    assert c["resident_GB"] == round(128 * 94 * 10_027_008 / 1e9, 3)
    assert c["layers"] == 94 and c["tokens_per_step"] == 1 and c["bits"] == 4


def test_kernel_code_ignores_comments_and_layout():
    """The traffic table is keyed on the kernel's code: a comment or layout
    edit keeps the key, a code edit changes it."""
    a = "int f(int x) {\n    return x + 1; // one\n}\n/* block\n comment */\n"
    b = "int f(int x)\n{\n  return x + 1;\n}\n"
    c = "int f(int x) { return x + 2; }"
    assert bench.kernel_code(a) == bench.kernel_code(b)
    assert bench.kernel_code(a) != bench.kernel_code(c)
