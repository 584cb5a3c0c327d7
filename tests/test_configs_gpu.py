"""The five workloads at their full sizes, checked against the float64 oracle
on sampled (layer, sequence, KV head) units, each run two ways:

* "two_calls": every layer makes the two calls of the decode notes' order,
  gqa_kv_append then gqa_decode_attn, on one stream;
* "bench_step": exactly what bench.py times: one gqa_decode_step per layer
  (append fused into the attention) with GQA_STEP_EARLY_STREAM, every layer
  back to back on one stream, over the layers the bench rotates through
  (a single-layer workload whose layers fit in L2 runs as many seeded
  replicas as the bench does), so the launch grids, the whole-unit work
  split and the overlap of consecutive launches are the timed ones.

A unit's inputs (its query heads, its cache rows below L_i - 1, its new K/V
row) are copied to the host BEFORE the step runs, so no oracle input passes
through the CUDA path; the oracle then performs the append and the attention
itself and is compared with the GPU's output rows of that unit."""
import numpy as np
import pytest
import torch

import oracle
from gqa_kv_cache_append_gb300.inputs import bench_layers, make_layer, seq_lens_for, workload
from tests.util import assert_close, to_np

pytestmark = pytest.mark.gpu

MODES = ["two_calls", "bench_step"]


def _b():
    from gqa_kv_cache_append_gb300 import binding
    return binding


def _snapshot(x, cfg, i, j):
    L = int(x["lens"][i])
    r = cfg.r
    return dict(
        q=to_np(x["q"][i:i + 1, j * r:(j + 1) * r])[0],
        k=to_np(x["k_cache"][i:i + 1, j:j + 1, :L])[0],
        v=to_np(x["v_cache"][i:i + 1, j:j + 1, :L])[0],
        kn=to_np(x["k_new"][i:i + 1, j:j + 1])[0],
        vn=to_np(x["v_new"][i:i + 1, j:j + 1])[0],
        L=L, tag=to_np(x["q"][:1, :1])[1])


def run_workload(cfg, sample_layers, sample_units, mode):
    """Allocate every layer on the device, snapshot the sampled units, run
    the full step in `mode`, compare.  Returns the max error seen.  Sampled
    layer -1 is the last layer of the run."""
    B = _b()
    torch.cuda.empty_cache()
    if mode == "bench_step":
        l2 = torch.cuda.get_device_properties(0).L2_cache_size
        cfg = workload(cfg.name, g=cfg.g, layers=bench_layers(cfg, seq_lens_for(cfg), l2))
    layers = [make_layer(cfg, l, "cuda") for l in range(cfg.layers)]
    snaps = {}
    for l in sorted({l % cfg.layers for l in sample_layers}):
        for (i, j) in sample_units(layers[l]):
            snaps[(l, i, j)] = _snapshot(layers[l], cfg, i, j)
    outs = [torch.empty((cfg.b, cfg.h, cfg.d), dtype=cfg.torch_dtype, device="cuda")
            for _ in range(cfg.layers)]
    stream = torch.cuda.current_stream()
    for l, x in enumerate(layers):
        if mode == "two_calls":
            B.decode_step(x["q"], x["k_cache"], x["v_cache"], x["k_new"], x["v_new"],
                          x["seq_lens"], cfg.g, cfg.scale, outs[l], stream=stream)
        else:
            B.gqa_decode_step(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                              x["seq_lens"], cfg.b, cfg.h, cfg.g, cfg.d, cfg.dv, cfg.scale,
                              outs[l], flags=B.GQA_STEP_EARLY_STREAM, stream=stream)
    assert B.gqa_device_status(stream) == 0
    worst = 0.0
    for (l, i, j), s in snaps.items():
        ref, _, _ = oracle.decode_step(s["q"], s["k"], s["v"], s["kn"], s["vn"], [s["L"]], 1,
                                       cfg.scale, dtype=s["tag"])
        r = cfg.r
        got = oracle.widen(to_np(outs[l][i:i + 1, j * r:(j + 1) * r])[0], s["tag"])
        worst = max(worst, assert_close(got, ref, s["tag"],
                                        f"{cfg.name} {mode} l{l} i{i} j{j}"))
        # the appended rows landed where the oracle put them
        assert torch.equal(layers[l]["k_cache"][i, j, s["L"] - 1], layers[l]["k_new"][i, j])
        assert torch.equal(layers[l]["v_cache"][i, j, s["L"] - 1], layers[l]["v_new"][i, j])
    del layers, outs
    torch.cuda.empty_cache()
    return worst


@pytest.mark.parametrize("mode", MODES)
def test_mqa_f32_full(mode):
    cfg = workload("mqa_f32_b1_h8_d64_m256")
    run_workload(cfg, [0, -1], lambda x: [(0, 0)], mode)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("g", [32, 8, 4, 1])
def test_gqa_sweep_full(g, mode):
    cfg = workload("gqa_sweep_b16_h32_d128_m4096", g=g)
    units = lambda x: [(i, j) for i in (0, 9, 15) for j in sorted({0, g // 2, g - 1})]
    run_workload(cfg, [0, -1], units, mode)


@pytest.mark.parametrize("mode", MODES)
def test_llama3_70b_full(mode):
    cfg = workload("llama3_70b_b32_m8192")
    units = lambda x: [(i, j) for i in (0, 17, 31) for j in range(cfg.g)]
    run_workload(cfg, [0, 41, 79], units, mode)


@pytest.mark.parametrize("mode", MODES)
def test_qwen25_7b_ragged_full(mode):
    cfg = workload("qwen25_7b_b64_ragged")

    def units(x):
        lens = x["lens"]
        pick = sorted({int(np.argmax(lens)), int(np.argmin(lens)), 0, 63, 30})
        return [(i, j) for i in pick for j in range(cfg.g)]
    run_workload(cfg, [0, 13, 27], units, mode)


@pytest.mark.parametrize("mode", MODES)
def test_long_mqa_peaked_full(mode):
    cfg = workload("long_mqa_b8_m131072")
    run_workload(cfg, [0, -1], lambda x: [(i, 0) for i in range(cfg.b)], mode)
