"""Decode attention through the C ABI against the float64 oracle on the same
inputs (fp32: max-abs 1e-5; bf16 with fp32 accumulation: 2e-2 + 1e-2 |ref|).

Cases span several tiles and a ragged tail: lengths of 1, tile - 1, tile,
tile + 1, ragged batches, units split across many CTAs and units held by one,
MHA (g = h), MQA (g = 1), r = 7 (not a power of two), NaN in the padding rows,
a peaked softmax, and the error paths (device status word, bounded wait)."""
import math

import numpy as np
import pytest
import torch

import oracle
from gqa_kv_cache_append_gb300.inputs import DecodeConfig, make_layer
from tests.util import assert_close, bits, to_np

pytestmark = pytest.mark.gpu


def _b():
    from gqa_kv_cache_append_gb300 import binding
    return binding


def run_step(cfg: DecodeConfig, lens, pad_fill=None, layer=0, check=True, fused=False, flags=0):
    """Append + attend on the GPU (two calls, or one fused gqa_decode_step
    with `flags`), oracle on the same host inputs; returns the max error."""
    B = _b()
    x = make_layer(cfg, layer, "cpu", lens=np.asarray(lens, dtype=np.int32), pad_fill=pad_fill)
    d = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    out = torch.full((cfg.b, cfg.h, cfg.d), 3.0, dtype=cfg.torch_dtype, device="cuda")
    B.decode_step(d["q"], d["k_cache"], d["v_cache"], d["k_new"], d["v_new"], d["seq_lens"],
                  cfg.g, cfg.scale, out, fused=fused, flags=flags)
    assert B.gqa_device_status() == 0
    tag = to_np(x["q"])[1]
    args = [to_np(x[k])[0] for k in ("q", "k_cache", "v_cache", "k_new", "v_new")]
    if pad_fill is not None:
        # the oracle reads no row >= L_i either; hand it finite padding so the
        # comparison does not depend on that
        args[1] = np.where(np.isfinite(oracle.widen(args[1], tag)), args[1], 0).astype(args[1].dtype)
        args[2] = np.where(np.isfinite(oracle.widen(args[2], tag)), args[2], 0).astype(args[2].dtype)
    ref, kc, vc = oracle.decode_step(*args, np.asarray(lens), cfg.g, cfg.scale, dtype=tag)
    got = oracle.widen(to_np(out)[0], tag)
    if pad_fill is None:
        assert to_np(d["k_cache"])[0].tobytes() == kc.tobytes()
        assert to_np(d["v_cache"])[0].tobytes() == vc.tobytes()
    return assert_close(got, ref, tag, cfg.name) if check else (got, ref)


def cfg_of(dtype, b, h, g, d, cap, seed=0, kind="plain"):
    return DecodeConfig(f"{dtype}_b{b}_h{h}_g{g}_d{d}_c{cap}", 1, b, h, g, d, cap, dtype,
                        1.0 / math.sqrt(d), 100 + seed, kind=kind)


# ---- CUDA-core kernel: fp32 (tile 128 at d=64, 64 at d=128); 16-bit data on
# request (tile 128 at d=64)
@pytest.mark.parametrize("b,h,g,d,cap,lens", [
    (1, 8, 1, 64, 256, [256]),                  # the fp32 MQA workload shape
    (2, 8, 2, 64, 200, [1, 200]),
    (3, 6, 3, 64, 130, [63, 64, 65]),
    (2, 16, 1, 64, 300, [129, 300]),            # r = 16
    (2, 12, 4, 128, 100, [31, 33]),             # fp32 d=128, one partial tile
    (4, 5, 5, 128, 97, [97, 1, 50, 32]),        # MHA
])
def test_simt_fp32(b, h, g, d, cap, lens):
    run_step(cfg_of("f32", b, h, g, d, cap, seed=b + h), lens)


# fp32 with d_k = d_v = 128 and at most 8 query rows per KV head: the launch
# with eight compute warps (two chunks of a K row per lane, 16 lanes a row)
@pytest.mark.parametrize("b,h,g,cap,lens", [
    (3, 16, 2, 640, [640, 63, 129]),         # r = 8, tile edges (tile 64)
    (2, 4, 4, 200, [200, 1]),                # r = 1
    (1, 8, 1, 12000, [11999]),               # one unit over many CTAs: combine kernel
    (24, 16, 4, 700, None),                  # units split across CTAs, merged in the kernel
    (4, 64, 8, 4096, [4096, 3000, 17, 2049]),  # Llama-shaped heads, ragged
])
def test_simt_fp32_eight_warps(b, h, g, cap, lens):
    if lens is None:
        lens = np.random.default_rng(b + cap).integers(1, cap + 1, b).astype(np.int32)
    run_step(cfg_of("f32", b, h, g, 128, cap, seed=b * 3 + g), lens)
    run_step(cfg_of("f32", b, h, g, 128, cap, seed=b * 3 + g), lens, fused=True)


def test_simt_fp32_eight_warps_nan_padding():
    lens = [1, 63, 64, 65, 300]
    run_step(cfg_of("f32", 5, 16, 2, 128, 320, seed=6), lens, pad_fill=float("nan"))


@pytest.mark.parametrize("b,h,g,cap,lens", [
    (2, 8, 1, 300, [300, 127]), (3, 4, 4, 260, [128, 129, 1]), (2, 14, 2, 513, [513, 200]),
])
@pytest.mark.parametrize("cuda_cores", [False, True])
def test_bf16_d64(b, h, g, cap, lens, cuda_cores):
    """Head dim 64: the tensor-core kernel, and the CUDA-core kernel on
    request (GQA_STEP_CUDA_CORES, fused step)."""
    from gqa_kv_cache_append_gb300 import binding as B
    flags = B.GQA_STEP_CUDA_CORES if cuda_cores else 0
    run_step(cfg_of("bf16", b, h, g, 64, cap, seed=cap), lens, fused=cuda_cores, flags=flags)


# ---- tensor-core kernel: bf16 d=128, tile 128, r padded to 16 or 32
@pytest.mark.parametrize("b,h,g,cap,lens", [
    (1, 8, 1, 1, [1]),
    (1, 8, 8, 127, [127]),                      # MHA, one partial tile
    (2, 16, 2, 128, [128, 1]),
    (2, 16, 2, 129, [129, 2]),
    (1, 32, 1, 1000, [1000]),                   # MQA, r = 32
    (2, 28, 4, 700, [700, 385]),                # r = 7
    (3, 64, 8, 300, [300, 256, 255]),           # r = 8
    (2, 48, 2, 257, [257, 129]),                # r = 24 -> 32 columns
    (4, 17, 1, 200, [200, 199, 131, 5]),        # r = 17
])
def test_tc_bf16(b, h, g, cap, lens):
    run_step(cfg_of("bf16", b, h, g, 128, cap, seed=b * cap), lens)


# ---- fused append + attention (one launch): same cache bits, same bound
@pytest.mark.parametrize("dtype,b,h,g,d,cap,lens", [
    ("bf16", 3, 64, 8, 128, 300, [300, 256, 128]),      # new row at a tile's last row
    ("bf16", 2, 28, 4, 128, 700, [700, 1]),
    ("bf16", 1, 32, 1, 128, 5000, [4097]),              # split unit, new row alone in its tile
    ("bf16", 4, 16, 16, 128, 129, [129, 127, 64, 2]),
    ("f32", 2, 8, 1, 64, 256, [256, 65]),
    ("f32", 3, 12, 4, 128, 100, [32, 33, 1]),
    ("bf16", 2, 8, 1, 64, 300, [300, 128]),
])
def test_fused_step(dtype, b, h, g, d, cap, lens):
    run_step(cfg_of(dtype, b, h, g, d, cap, seed=7 * b + cap), lens, fused=True)


def test_fused_step_matches_two_calls_bitwise():
    B = _b()
    cfg = cfg_of("bf16", 6, 64, 8, 128, 3000, seed=31)
    lens = np.array([3000, 1, 128, 2049, 777, 2560], dtype=np.int32)
    x = make_layer(cfg, 0, "cuda", lens=lens)
    outs, caches = [], []
    for fused in (False, True):
        kc, vc = x["k_cache"].clone(), x["v_cache"].clone()
        out = torch.empty((cfg.b, cfg.h, cfg.d), dtype=torch.bfloat16, device="cuda")
        B.decode_step(x["q"], kc, vc, x["k_new"], x["v_new"], x["seq_lens"], cfg.g, cfg.scale,
                      out, fused=fused)
        outs.append(out)
        caches.append((kc, vc))
    assert B.gqa_device_status() == 0
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(caches[0][0], caches[1][0]) and torch.equal(caches[0][1], caches[1][1])


@pytest.mark.parametrize("dtype,b,h,g,d,cap,lens", [
    ("bf16", 8, 64, 8, 128, 2000, None),          # units split in-kernel
    ("bf16", 2, 32, 1, 128, 9000, [9000, 4500]),  # few long units: combine kernel
    ("f32", 8, 64, 8, 128, 2000, None),           # the CUDA-core kernel
    ("f32", 1, 8, 1, 64, 256, [256]),             # the fp32 MQA step's shape
    ("f32", 2, 16, 1, 128, 9000, [9000, 4500]),   # CUDA-core kernel + combine kernel
])
def test_early_stream_matches_ordered_calls(dtype, b, h, g, d, cap, lens):
    """Six layers back to back with GQA_STEP_EARLY_STREAM give the same
    outputs and caches, bit for bit, as the default ordered calls (on the
    tensor-core and the CUDA-core kernel)."""
    B = _b()
    cfg = cfg_of(dtype, b, h, g, d, cap, seed=b + g)
    lens = np.asarray(lens if lens is not None else [cap - 37 * i for i in range(b)], np.int32)
    layers = [make_layer(cfg, l, "cuda", lens=lens) for l in range(6)]
    results = []
    for flags in (0, B.GQA_STEP_EARLY_STREAM):
        kcs = [x["k_cache"].clone() for x in layers]
        vcs = [x["v_cache"].clone() for x in layers]
        outs = [torch.empty((b, h, d), dtype=cfg.torch_dtype, device="cuda") for _ in layers]
        torch.cuda.synchronize()
        for rep in range(3):
            for l, x in enumerate(layers):
                B.gqa_decode_step(x["q"], x["k_new"], x["v_new"], kcs[l], vcs[l], x["seq_lens"],
                                  b, h, g, d, d, cfg.scale, outs[l], flags=flags)
        torch.cuda.synchronize()
        results.append((outs, kcs, vcs))
    assert B.gqa_device_status() == 0
    for l in range(len(layers)):
        assert torch.equal(results[0][0][l], results[1][0][l])
        assert torch.equal(results[0][1][l], results[1][1][l])
        assert torch.equal(results[0][2][l], results[1][2][l])
    # and the ordered result is right
    x = layers[0]
    args = [to_np(x[k])[0] for k in ("q", "k_cache", "v_cache", "k_new", "v_new")]
    tag = to_np(x["q"])[1]
    ref, _, _ = oracle.decode_step(*args, lens, g, cfg.scale, dtype=tag)
    assert_close(oracle.widen(to_np(results[1][0][0])[0], tag), ref, tag)


@pytest.mark.parametrize("b,h,g,cap", [(4, 64, 8, 1500), (2, 32, 1, 6000)])
def test_graph_capture_replay(b, h, g, cap):
    """Several layers' steps captured in a CUDA graph and replayed give the
    same outputs, bit for bit, as the same calls made eagerly (the append is
    idempotent for fixed lengths)."""
    B = _b()
    cfg = cfg_of("bf16", b, h, g, 128, cap, seed=h + g)
    lens = np.asarray([cap - 71 * i for i in range(b)], np.int32)
    layers = [make_layer(cfg, l, "cuda", lens=lens) for l in range(4)]
    s = torch.cuda.Stream()
    eager = [torch.empty((b, h, 128), dtype=torch.bfloat16, device="cuda") for _ in layers]
    replayed = [torch.full_like(o, 9.0) for o in eager]

    def step(outs):
        for x, o in zip(layers, outs):
            B.gqa_decode_step(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                              x["seq_lens"], b, h, g, 128, 128, cfg.scale, o,
                              flags=B.GQA_STEP_EARLY_STREAM, stream=s)
    with torch.cuda.stream(s):
        step(eager)            # grows the workspace of stream s before the capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            step(replayed)
        for _ in range(3):
            graph.replay()
    torch.cuda.synchronize()
    assert B.gqa_device_status(s) == 0
    for e, r_ in zip(eager, replayed):
        assert torch.equal(e, r_)


def test_fused_step_bad_length_appends_nothing():
    B = _b()
    cfg = cfg_of("bf16", 3, 16, 2, 128, 300, seed=8)
    x = make_layer(cfg, 0, "cuda", lens=np.array([300, 300, 300], dtype=np.int32))
    before_k = x["k_cache"].clone()
    lens = torch.tensor([300, 0, 301], dtype=torch.int32, device="cuda")
    out = torch.full((cfg.b, cfg.h, cfg.d), 5.0, dtype=torch.bfloat16, device="cuda")
    B.gqa_decode_step(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], lens, cfg.b,
                      cfg.h, cfg.g, 128, 128, cfg.scale, out)
    assert B.gqa_device_status() == B.GQA_DEV_BAD_SEQ_LEN
    assert torch.equal(x["k_cache"][1:], before_k[1:])
    assert torch.all(out[1:] == 5.0)
    assert torch.equal(x["k_cache"][0, :, 299], x["k_new"][0])


def test_tc_many_splits_long_sequence():
    # one unit of 40 tiles spread over many CTAs: exercises the combine
    run_step(cfg_of("bf16", 1, 8, 1, 128, 5000, seed=3), [5000])


@pytest.mark.parametrize("dtype,d,cap,lens", [
    ("bf16", 128, 20000, [5000]),          # 40 tiles over 152 CTAs: most ranges empty
    ("bf16", 128, 9000, [300, 1, 4000]),
    ("f32", 64, 12000, [1000, 3]),         # CUDA-core kernel, same situation
])
def test_fewer_tiles_than_ctas(dtype, d, cap, lens):
    h, g = (8, 1) if dtype == "bf16" else (4, 2)
    run_step(cfg_of(dtype, len(lens), h, g, d, cap, seed=cap % 97), lens)


def test_tc_ragged_batch_with_nan_padding():
    lens = [1, 127, 128, 129, 1000, 2049, 3, 700]
    run_step(cfg_of("bf16", 8, 28, 4, 128, 2100, seed=9), lens, pad_fill=float("nan"))


def test_simt_ragged_batch_with_nan_padding():
    lens = [1, 63, 64, 65, 300]
    run_step(cfg_of("f32", 5, 8, 2, 64, 320, seed=4), lens, pad_fill=float("nan"))


def test_tc_peaked_softmax():
    cfg = DecodeConfig("peaked", 1, 4, 32, 1, 128, 3000, "bf16", 1 / math.sqrt(128), 77,
                       kind="boost")
    run_step(cfg, [3000, 2999, 1500, 64])


def test_results_are_deterministic():
    B = _b()
    cfg = cfg_of("bf16", 4, 32, 4, 128, 2000, seed=1)
    x = make_layer(cfg, 0, "cuda")
    outs = []
    for _ in range(2):
        out = torch.empty((cfg.b, cfg.h, cfg.d), dtype=torch.bfloat16, device="cuda")
        B.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], cfg.b, cfg.h,
                          cfg.g, 128, 128, cfg.scale, out)
        outs.append(out)
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("dtype,h,g,d", [("bf16", 64, 8, 128), ("bf16", 32, 1, 128),
                                         ("f32", 8, 2, 64)])
def test_in_kernel_merge_is_deterministic(dtype, h, g, d):
    """Units split across CTAs and merged by the last CTA to finish (few
    pieces per unit): the pieces are merged in CTA order whichever CTA
    merges, so repeated runs give the same bits."""
    B = _b()
    b = 96 if g == 1 else 24
    cfg = cfg_of(dtype, b, h, g, d, 700, seed=3)
    x = make_layer(cfg, 0, "cuda", lens=np.random.default_rng(8).integers(1, 701, b).astype(np.int32))
    outs = []
    for _ in range(3):
        out = torch.empty((cfg.b, cfg.h, cfg.d), dtype=cfg.torch_dtype, device="cuda")
        B.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], cfg.b, cfg.h,
                          cfg.g, d, d, cfg.scale, out)
        outs.append(bits(out))
    assert B.gqa_device_status() == 0
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


@pytest.mark.parametrize("b,h,g,cap", [(1, 8, 1, 20000), (8, 32, 1, 8192), (5, 16, 2, 6000)])
def test_combine_kernel_is_deterministic(b, h, g, cap, monkeypatch):
    """Units over many CTAs merged by the combine kernel (up to ~150 pieces a
    unit, ragged lengths; GQA_CLUSTER=0 keeps the tensor-core kernel off its
    cluster launch): fixed merge order, the same bits every run."""
    B = _b()
    monkeypatch.setenv("GQA_CLUSTER", "0")
    assert B.gqa_decode_plan(b, 1, h, g, 128, 128, cap, "bf16")["kernels"] == 2
    cfg = cfg_of("bf16", b, h, g, 128, cap, seed=b + h)
    lens = np.random.default_rng(b).integers(cap // 2, cap + 1, b).astype(np.int32)
    x = make_layer(cfg, 0, "cuda", lens=lens)
    outs = []
    for _ in range(3):
        out = torch.empty((cfg.b, cfg.h, cfg.d), dtype=cfg.torch_dtype, device="cuda")
        B.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], cfg.b, cfg.h,
                          cfg.g, 128, 128, cfg.scale, out)
        outs.append(bits(out))
    assert B.gqa_device_status() == 0
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_bad_length_is_reported_and_other_rows_are_right():
    B = _b()
    cfg = cfg_of("bf16", 3, 16, 2, 128, 300, seed=2)
    x = make_layer(cfg, 0, "cpu", lens=np.array([300, 300, 300], dtype=np.int32))
    d = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    lens = torch.tensor([300, 301, 0], dtype=torch.int32, device="cuda")
    sentinel = torch.full((cfg.b, cfg.h, cfg.d), 5.0, dtype=torch.bfloat16, device="cuda")
    B.gqa_decode_attn(d["q"], d["k_cache"], d["v_cache"], lens, cfg.b, cfg.h, cfg.g, 128, 128,
                      cfg.scale, sentinel)
    assert B.gqa_device_status() == B.GQA_DEV_BAD_SEQ_LEN
    assert torch.all(sentinel[1:] == 5.0)
    args = [to_np(x[k])[0] for k in ("q", "k_cache", "v_cache")]
    ref = oracle.grouped_decode_attention(args[0][:1], args[1][:1], args[2][:1], [300], cfg.g,
                                          cfg.scale, dtype="bf16")
    assert_close(oracle.widen(to_np(sentinel[:1])[0], "bf16"), ref, "bf16")


def test_bounded_wait_reports_timeout():
    B = _b()
    assert B.gqa_device_status() == 0
    B.gqa_selftest_wait_timeout(1 << 20)
    assert B.gqa_device_status() == B.GQA_DEV_WAIT_TIMEOUT
    assert B.gqa_device_status() == 0


def test_error_codes_reach_python():
    B = _b()
    q = torch.zeros((1, 6, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 4, 8, 128), dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(B.GqaError) as e:
        B.gqa_decode_attn(q, k, k, lens, 1, 6, 4, 128, 128, 1.0, out)
    assert e.value.code == B.GQA_ERR_SHAPE
    with pytest.raises(B.GqaError) as e:
        B.gqa_decode_attn(q.double(), k.double(), k.double(), lens, 1, 6, 2, 128, 128, 1.0,
                          out.double())
    assert e.value.code == B.GQA_ERR_DTYPE
    raw = torch.zeros(1 * 6 * 128 + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.GqaError) as e:
        B.gqa_decode_attn(raw[1:], k, k, lens, 1, 6, 2, 128, 128, 1.0, out)
    assert e.value.code == B.GQA_ERR_ALIGN
