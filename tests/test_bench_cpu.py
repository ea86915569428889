"""The benchmark's work accounting, on the CPU: a call's algorithmic bytes and flops match
the formulas written out by hand, a batched call reads its shared x once, and the decode
step is the sum of its calls."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_linear_bytes_and_flops_by_hand():
    out, inp, r, M = 6912, 1152, 16, 4
    # W0, U, V, s, x, y in bf16
    by_hand = 2 * (out * inp + out * r + inp * r + out + M * inp + M * out)
    assert bench.linear_bytes(out, inp, r, M) == by_hand
    # the shared-block product, the down and up projections, and the scale
    assert bench.linear_flops(out, inp, r, M) == 2 * M * out * inp + 2 * M * inp * r + 2 * M * r * out + M * out


def test_batched_calls_read_x_once():
    r, M = 16, 16
    gate, up = bench.FAMS["gate_proj"], bench.FAMS["up_proj"]
    two_calls = bench.linear_bytes(*gate, r, M) + bench.linear_bytes(*up, r, M)
    assert bench.gate_up_bytes(r, M) == two_calls - 2 * M * gate[1]
    q, k, v = (bench.FAMS[f] for f in ("q_proj", "k_proj", "v_proj"))
    three_calls = sum(bench.linear_bytes(*s, r, M) for s in (q, k, v))
    assert bench.qkv_bytes([q, k, v], r, M) == three_calls - 2 * 2 * M * q[1]


def test_step_is_the_sum_of_its_calls():
    per_pass = {M: sum(bench.call_bytes(kind, M) for kind in ("qkv", "o_proj", "gate_up", "down_proj"))
                for M in bench.DECODE_MS}
    assert bench.step_bytes() == bench.LAYERS * sum(per_pass.values())
    # the separate-call step reads the MLP input once more per layer and pass
    extra = bench.LAYERS * sum(2 * M * bench.FAMS["gate_proj"][1] for M in bench.DECODE_MS)
    assert bench.step_bytes(fuse_gateup=False) - bench.step_bytes() == extra


def test_sweep_grid_covers_both_paths():
    assert len(bench.SWEEP_SHAPES) * len(bench.SWEEP_RANKS) * len(bench.SWEEP_MS) == 50
    # below and above the decode kernel's token limit, and ranks from none to 256
    assert min(bench.SWEEP_MS) <= 32 < max(bench.SWEEP_MS)
    assert 0 in bench.SWEEP_RANKS and max(bench.SWEEP_RANKS) == 256
    # each point's W0 copies together exceed the 126 MB L2 of the part
    for out, inp in bench.SWEEP_SHAPES.values():
        assert bench.SWEEP_COPIES * out * inp * 2 > 126 * 2**20


def test_roofline_time_takes_the_larger_bound():
    hbm, pk = 6801.3e9, 1970.5e12
    for (out, inp), r, M in (((6912, 1152), 16, 1), ((6912, 1152), 64, 4096)):
        B, F = bench.linear_bytes(out, inp, r, M), bench.linear_flops(out, inp, r, M)
        t_star = max(B / hbm, F / pk)
        assert t_star == (B / hbm if M == 1 else F / pk)
    assert np.isclose(pk / hbm, 289.7, rtol=1e-3)   # the ridge, in flops per byte


def test_committed_traffic_capture_matches_the_sources():
    """The DRAM traffic the bench reports comes from profiles/dram_traffic.json only while the
    kernel sources hash to the value recorded with it; the committed capture must describe the
    committed sources and cover every decode call type of the step, each reading its operands
    once (traffic within a few percent of the algorithmic bytes)."""
    import json
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        rec = json.load(f)
    assert rec["source_hash"] == bench.kernel_source_hash()
    for M in bench.DECODE_MS:
        for kind in ("qkv", "o_proj", "gate_up", "down_proj"):
            ent = rec["launches"][f"decode:{kind}:M{M}"]
            assert ent["algorithmic_bytes"] == bench.call_bytes(kind, M)
            assert 0.95 < ent["dram_bytes"] / ent["algorithmic_bytes"] < 1.05, (kind, M)
            traffic, src = bench.captured_traffic(f"decode:{kind}:M{M}")
            assert traffic == ent["dram_bytes"] and src.startswith("ncu capture")


def test_mlp_and_decomposition_accounting_by_hand():
    r, M = 16, 4
    (go, gi), (uo, ui), (do, di) = (bench.FAMS[f] for f in ("gate_proj", "up_proj", "down_proj"))
    weights = sum(2 * (o * i + r * (o + i) + o) for o, i in ((go, gi), (uo, ui), (do, di)))
    assert bench.mlp_bytes(M) == weights + 2 * M * gi + 2 * M * do
    # the fused MLP moves what the step's gate/up and down calls move, less the intermediates
    assert bench.mlp_bytes(M) == (bench.gate_up_bytes(r, M) + bench.linear_bytes(do, di, r, M)
                                  - 2 * M * (go + uo) - 2 * M * di)
    m, n, k = 1152, 1024, 24
    assert bench.rsvd_flops(m, n, k, 0) == 2 * (2 * m * n * k) + 2 * (4 * m * k * k) + 2 * m * k * k
    assert bench.rsvd_flops(m, n, k, 1) - bench.rsvd_flops(m, n, k, 0) == 2 * (2 * m * n * k + 4 * m * k * k)
