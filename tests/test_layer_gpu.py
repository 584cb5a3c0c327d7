"""The projections around the step and the whole incremental layer through
the C ABI, against the float64 oracle on the same bf16 inputs.

Projections (q / k_new / v_new = x . P, y = o . P_o) are compared with the
unrounded float64 products (bf16 bound 2e-2 + 1e-2 |ref|); the layer's y
against the oracle layer, which rounds q, the new rows and o to bf16 at the
points the CUDA path stores them.  Cases: batches 1..128 (32, 64 and 128
MMA columns, partial ones), widths 128..8192 (tiles held whole and tiles cut
between CTAs), MHA / GQA / MQA heads, determinism of the cut-tile sums, and
the Llama-3-70B-shaped layer at full size."""
import math

import numpy as np
import pytest
import torch

import oracle
from gqa_kv_cache_append_gb300.inputs import DecodeConfig, make_layer, make_layer_weights
from tests.util import assert_close, bits, to_np

pytestmark = pytest.mark.gpu


def _b():
    from gqa_kv_cache_append_gb300 import binding
    return binding


def cfg_of(b, h, g, D, cap=256, seed=0, layers=1):
    return DecodeConfig(f"layer_b{b}_h{h}_g{g}_D{D}", layers, b, h, g, 128, cap, "bf16",
                        1.0 / math.sqrt(128), 700 + seed, d_model=D)


def np_bf16(t):
    return to_np(t)[0]


@pytest.mark.parametrize("b,h,g,D", [
    (1, 8, 8, 128),      # one chunk per tile: every tile whole
    (7, 8, 2, 1024),
    (32, 64, 8, 2048),   # Llama heads, tiles cut between CTAs
    (33, 28, 4, 3584),   # 64 MMA columns, Qwen width
    (100, 32, 1, 512),   # 128 MMA columns, MQA
    (128, 4, 4, 8192),   # the full 128 columns, few long tiles
])
def test_project_qkv(b, h, g, D):
    B = _b()
    cfg = cfg_of(b, h, g, D, seed=b)
    w = make_layer_weights(cfg, 0, "cpu")
    d = {k: v.cuda() for k, v in w.items()}
    q = torch.full((b, h, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    kn = torch.full((b, g, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    vn = torch.full((b, g, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    B.gqa_project_qkv(d["x"], d["P_q"], d["P_k"], d["P_v"], q, kn, vn, b, D, h, g, 128, 128)
    assert B.gqa_device_status() == 0
    rq, rk, rv = oracle.project_qkv(np_bf16(w["x"]), np_bf16(w["P_q"]), np_bf16(w["P_k"]),
                                    np_bf16(w["P_v"]), "bf16")
    for got, ref, name in ((q, rq, "q"), (kn, rk, "k_new"), (vn, rv, "v_new")):
        assert_close(oracle.widen(np_bf16(got), "bf16"), ref, "bf16", name)


@pytest.mark.parametrize("b,h,D", [(1, 8, 128), (32, 64, 8192), (64, 28, 3584), (128, 16, 256)])
def test_project_out(b, h, D):
    B = _b()
    cfg = cfg_of(b, h, h, D, seed=h)
    w = make_layer_weights(cfg, 0, "cpu")
    gen = torch.Generator().manual_seed(11 + b)
    o = torch.randn((b, h, 128), generator=gen).to(torch.bfloat16)
    y = torch.full((b, D), 7.0, dtype=torch.bfloat16, device="cuda")
    B.gqa_project_out(o.cuda(), w["P_o"].cuda(), y, b, D, h, 128)
    assert B.gqa_device_status() == 0
    ref = oracle.project_out(np_bf16(o), np_bf16(w["P_o"]), "bf16")
    assert_close(oracle.widen(np_bf16(y), "bf16"), ref, "bf16", "y")


def test_cut_tiles_are_summed_deterministically():
    B = _b()
    b, h, g, D = 32, 64, 8, 8192
    cfg = cfg_of(b, h, g, D, seed=3)
    w = {k: v.cuda() for k, v in make_layer_weights(cfg, 0, "cpu").items()}
    outs = []
    for _ in range(3):
        q = torch.empty((b, h, 128), dtype=torch.bfloat16, device="cuda")
        kn = torch.empty((b, g, 128), dtype=torch.bfloat16, device="cuda")
        vn = torch.empty((b, g, 128), dtype=torch.bfloat16, device="cuda")
        B.gqa_project_qkv(w["x"], w["P_q"], w["P_k"], w["P_v"], q, kn, vn, b, D, h, g, 128, 128)
        y = torch.empty((b, D), dtype=torch.bfloat16, device="cuda")
        B.gqa_project_out(q, w["P_o"], y, b, D, h, 128)
        outs.append((bits(q), bits(kn), bits(vn), bits(y)))
    for o in outs[1:]:
        for a, c in zip(outs[0], o):
            assert np.array_equal(a, c)


def run_layer(cfg, lens, flags=0):
    B = _b()
    lens = np.asarray(lens, dtype=np.int32)
    x = make_layer(cfg, 0, "cpu", lens=lens)
    w = make_layer_weights(cfg, 0, "cpu")
    dc = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    dw = {k: v.cuda() for k, v in w.items()}
    y = torch.full((cfg.b, cfg.D), 7.0, dtype=torch.bfloat16, device="cuda")
    B.gqa_decode_layer(dw["x"], dw["P_q"], dw["P_k"], dw["P_v"], dw["P_o"], dc["k_cache"],
                       dc["v_cache"], dc["seq_lens"], cfg.b, cfg.D, cfg.h, cfg.g, 128, 128,
                       cfg.scale, y, flags=flags)
    assert B.gqa_device_status() == 0
    ry, kc, vc, _, _ = oracle.decode_layer(
        np_bf16(w["x"]), np_bf16(w["P_q"]), np_bf16(w["P_k"]), np_bf16(w["P_v"]),
        np_bf16(w["P_o"]), np_bf16(x["k_cache"]), np_bf16(x["v_cache"]), lens, cfg.g,
        cfg.scale, dtype="bf16")
    assert_close(oracle.widen(np_bf16(y), "bf16"), ry, "bf16", cfg.name)
    # every cache row but the appended one is untouched; the appended rows
    # are, bit for bit, the new rows gqa_project_qkv gives for the same x
    # (the append is a copy), and those are within the bf16 bound of the
    # float64 projections
    q = torch.empty((cfg.b, cfg.h, 128), dtype=torch.bfloat16, device="cuda")
    kn = torch.empty((cfg.b, cfg.g, 128), dtype=torch.bfloat16, device="cuda")
    vn = torch.empty((cfg.b, cfg.g, 128), dtype=torch.bfloat16, device="cuda")
    B.gqa_project_qkv(dw["x"], dw["P_q"], dw["P_k"], dw["P_v"], q, kn, vn, cfg.b, cfg.D, cfg.h,
                      cfg.g, 128, 128)
    _, rk, rv = oracle.project_qkv(np_bf16(w["x"]), np_bf16(w["P_q"]), np_bf16(w["P_k"]),
                                   np_bf16(w["P_v"]), "bf16")
    assert_close(oracle.widen(np_bf16(kn), "bf16"), rk, "bf16", "k_new")
    assert_close(oracle.widen(np_bf16(vn), "bf16"), rv, "bf16", "v_new")
    gk, gv = np_bf16(dc["k_cache"]), np_bf16(dc["v_cache"])
    kn_b, vn_b = np_bf16(kn), np_bf16(vn)
    for i in range(cfg.b):
        L = int(lens[i])
        keep = np.ones(cfg.cap, dtype=bool)
        keep[L - 1] = False
        assert np.array_equal(gk[i][:, keep], kc[i][:, keep])
        assert np.array_equal(gv[i][:, keep], vc[i][:, keep])
        assert np.array_equal(gk[i, :, L - 1], kn_b[i])
        assert np.array_equal(gv[i, :, L - 1], vn_b[i])


@pytest.mark.parametrize("b,h,g,D,cap,lens", [
    (3, 8, 2, 512, 300, [1, 129, 300]),
    (32, 64, 8, 1024, 200, None),
    (5, 32, 1, 4096, 1000, [1000, 3, 517, 128, 129]),
])
def test_decode_layer(b, h, g, D, cap, lens):
    cfg = cfg_of(b, h, g, D, cap=cap, seed=h + g)
    if lens is None:
        lens = np.random.default_rng(5).integers(1, cap + 1, size=b)
    run_layer(cfg, lens)


def test_decode_layer_early_flag_same_bits():
    B = _b()
    cfg = cfg_of(4, 16, 4, 1024, cap=400, seed=21)
    lens = np.array([400, 200, 1, 129], dtype=np.int32)
    x = make_layer(cfg, 0, "cpu", lens=lens)
    w = {k: v.cuda() for k, v in make_layer_weights(cfg, 0, "cpu").items()}
    ys = []
    for flags in (0, B.GQA_STEP_EARLY_STREAM):
        dc = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
        y = torch.empty((cfg.b, cfg.D), dtype=torch.bfloat16, device="cuda")
        B.gqa_decode_layer(w["x"], w["P_q"], w["P_k"], w["P_v"], w["P_o"], dc["k_cache"],
                           dc["v_cache"], dc["seq_lens"], cfg.b, cfg.D, cfg.h, cfg.g, 128, 128,
                           cfg.scale, y, flags=flags)
        ys.append((bits(y), bits(dc["k_cache"])))
    assert np.array_equal(ys[0][0], ys[1][0]) and np.array_equal(ys[0][1], ys[1][1])


def test_llama_layer_full_size():
    """One Llama-3-70B-shaped layer at full size: b=32, D=8192, h=64, g=8,
    L=8192 (the KV of the layer is 1 GiB, the weights 0.3 GB)."""
    cfg = cfg_of(32, 64, 8, 8192, cap=8192, seed=99)
    run_layer(cfg, np.full(32, 8192))
