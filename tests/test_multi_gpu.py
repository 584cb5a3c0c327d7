"""n new tokens per sequence in one step (the batched form with the causal
mask) through the C ABI against the float64 oracle on the same inputs.

Cases: lengths equal to n (the first new token at position 0), new rows
straddling a tile boundary, n * r = 16 and 32 query rows per KV head, r = 1
with n = 20 and 32 (more new rows than the kernel carries in registers),
r = 7, units split across CTAs where a CTA's share holds positions that some
of the new tokens must not see (empty partials, merged in the decode kernel
and in the combine kernel), NaN padding, n = 1 against the one-token calls,
fused against two calls, and a length below n."""
import math

import numpy as np
import pytest
import torch

import oracle
from gqa_kv_cache_append_gb300.inputs import DecodeConfig, make_layer, make_layer_multi
from tests.util import assert_close, bits, to_np

pytestmark = pytest.mark.gpu


def _b():
    from gqa_kv_cache_append_gb300 import binding
    return binding


def cfg_of(dtype, b, h, g, d, cap, seed=0):
    return DecodeConfig(f"{dtype}_b{b}_h{h}_g{g}_d{d}_c{cap}", 1, b, h, g, d, cap, dtype,
                        1.0 / math.sqrt(d), 300 + seed)


def gpu_step(cfg, n, x, fused=True, flags=0):
    """Run the step on copies of x on the GPU; returns (out, k_cache, v_cache)."""
    B = _b()
    d = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    out = torch.full((cfg.b, n, cfg.h, cfg.d), 3.0, dtype=cfg.torch_dtype, device="cuda")
    if fused:
        B.gqa_decode_step_multi(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                                d["seq_lens"], cfg.b, n, cfg.h, cfg.g, cfg.d, cfg.d, cfg.scale,
                                out, flags=flags)
    else:
        B.gqa_kv_append_multi(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                              d["seq_lens"], cfg.b, n, cfg.g, cfg.d, cfg.d)
        B.gqa_decode_attn_multi(d["q"], d["k_cache"], d["v_cache"], d["seq_lens"], cfg.b, n,
                                cfg.h, cfg.g, cfg.d, cfg.d, cfg.scale, out)
    return out, d["k_cache"], d["v_cache"]


def run_multi(cfg, n, lens, fused=True, pad_fill=None):
    lens = np.asarray(lens, dtype=np.int32)
    x = make_layer_multi(cfg, n, 0, "cpu", lens=lens, pad_fill=pad_fill)
    out, kc_d, vc_d = gpu_step(cfg, n, x, fused=fused)
    assert _b().gqa_device_status() == 0
    tag = to_np(x["q"])[1]
    args = [to_np(x[k])[0] for k in ("q", "k_cache", "v_cache", "k_new", "v_new")]
    if pad_fill is not None:
        for a in (1, 2):
            args[a] = np.where(np.isfinite(oracle.widen(args[a], tag)), args[a],
                               0).astype(args[a].dtype)
    ref, kc, vc = oracle.decode_step_multi(*args, lens, cfg.g, cfg.scale, dtype=tag)
    if pad_fill is None:
        assert to_np(kc_d)[0].tobytes() == kc.tobytes()
        assert to_np(vc_d)[0].tobytes() == vc.tobytes()
    got = oracle.widen(to_np(out)[0], tag)
    return assert_close(got, ref, tag, f"{cfg.name}_n{n}")


# ---- tensor-core kernel (bf16, d = 128): n * r query rows on the MMA N axis
@pytest.mark.parametrize("b,n,h,g,cap,lens", [
    (3, 4, 16, 2, 300, [4, 130, 300]),         # L = n; rows 126..129 straddle tiles
    (2, 2, 64, 8, 1000, [1000, 515]),          # Llama-shaped heads, 16 rows
    (2, 4, 64, 8, 700, [700, 257]),            # 32 rows: two softmax warpgroups
    (2, 32, 4, 4, 200, [200, 33]),             # r = 1, n = 32
    (1, 20, 8, 8, 300, [140]),                 # r = 1, new rows 120..139 straddle
    (2, 4, 28, 4, 2000, [129, 2000]),          # r = 7
])
def test_tc_multi(b, n, h, g, cap, lens):
    run_multi(cfg_of("bf16", b, h, g, 128, cap, seed=b * n), n, lens)


@pytest.mark.parametrize("fused", [True, False])
def test_tc_multi_split_units_with_unseen_tiles(fused):
    # 96 units of 3 tiles over 152 CTAs (merged in the decode kernel): a CTA
    # holding only a unit's last tile (rows 256, 257 = tokens 2, 3) has
    # nothing for tokens 0 and 1
    run_multi(cfg_of("bf16", 96, 8, 1, 128, 384, seed=7), 4, [258] * 96, fused=fused)


def test_tc_multi_combine_kernel_with_unseen_tiles():
    # one unit of 100 tiles over 128 CTAs: the combine kernel merges, and the
    # last tile's CTA (rows 12672, 12673 = tokens 2, 3) is empty for tokens 0, 1
    run_multi(cfg_of("bf16", 1, 8, 1, 128, 16384, seed=8), 4, [99 * 128 + 2])


def test_tc_multi_nan_padding():
    run_multi(cfg_of("bf16", 2, 16, 4, 128, 400, seed=9), 3, [131, 250],
              pad_fill=float("nan"))


# ---- CUDA-core kernel: fp32 (tile 128 at d = 64, 64 at d = 128); bf16 d = 64
# (tensor-core kernel)
@pytest.mark.parametrize("dtype,b,n,h,g,d,cap,lens", [
    ("f32", 3, 4, 8, 4, 64, 200, [4, 130, 200]),   # rows 126..129 straddle tiles
    ("f32", 2, 2, 16, 4, 128, 300, [300, 65]),     # 8 rows, d = 128: eight compute warps
    ("f32", 2, 4, 4, 2, 128, 200, [66, 130]),      # 8 rows; rows 62..65 straddle tiles
    ("f32", 2, 3, 5, 1, 128, 100, [3, 34]),        # 15 rows: the 16-row launch
    ("f32", 1, 8, 2, 1, 64, 12800, [99 * 128 + 2]),  # combine kernel, unseen tile
    ("f32", 96, 4, 2, 1, 64, 192, [130] * 96),     # in-kernel merge, unseen tiles
    ("bf16", 2, 4, 4, 2, 64, 300, [129, 300]),     # 8 rows
])
def test_simt_multi(dtype, b, n, h, g, d, cap, lens):
    run_multi(cfg_of(dtype, b, h, g, d, cap, seed=n + h), n, lens)


@pytest.mark.parametrize("dtype,d,h,g", [("bf16", 128, 64, 8), ("f32", 64, 8, 1)])
def test_fused_equals_two_calls_bitwise(dtype, d, h, g):
    cfg = cfg_of(dtype, 3, h, g, d, 600, seed=11)
    lens = np.array([600, 131, 3], dtype=np.int32)
    n = 3 if dtype == "bf16" else 2
    x = make_layer_multi(cfg, n, 0, "cpu", lens=lens)
    o1, k1, v1 = gpu_step(cfg, n, x, fused=True)
    o2, k2, v2 = gpu_step(cfg, n, x, fused=False)
    assert np.array_equal(bits(o1), bits(o2))
    assert np.array_equal(bits(k1), bits(k2)) and np.array_equal(bits(v1), bits(v2))


@pytest.mark.parametrize("dtype,d,h,g", [("bf16", 128, 64, 8), ("f32", 64, 8, 2)])
def test_one_token_equals_the_single_token_calls(dtype, d, h, g):
    B = _b()
    cfg = cfg_of(dtype, 2, h, g, d, 300, seed=12)
    lens = np.array([300, 129], dtype=np.int32)
    x = make_layer(cfg, 0, "cpu", lens=lens)
    xm = dict(x)
    xm["q"] = x["q"][:, None].contiguous()
    xm["k_new"] = x["k_new"][:, None].contiguous()
    xm["v_new"] = x["v_new"][:, None].contiguous()
    o1, k1, v1 = gpu_step(cfg, 1, xm, fused=True)
    d_ = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    o2 = torch.empty((cfg.b, cfg.h, cfg.d), dtype=cfg.torch_dtype, device="cuda")
    B.gqa_decode_step(d_["q"], d_["k_new"], d_["v_new"], d_["k_cache"], d_["v_cache"],
                      d_["seq_lens"], cfg.b, cfg.h, cfg.g, d, d, cfg.scale, o2)
    assert np.array_equal(bits(o1[:, 0]), bits(o2))
    assert np.array_equal(bits(k1), bits(d_["k_cache"]))
    assert np.array_equal(bits(v1), bits(d_["v_cache"]))


def test_early_stream_multi_layer_bitwise():
    """Two layers' fused steps back to back with GQA_STEP_EARLY_STREAM give
    the bits of the ordered launches."""
    B = _b()
    cfg = cfg_of("bf16", 4, 32, 8, 128, 1024, seed=13)
    lens = np.array([1024, 700, 129, 4], dtype=np.int32)
    n = 4
    layers = [make_layer_multi(cfg, n, l, "cpu", lens=lens) for l in range(2)]
    outs = []
    for flags in (0, B.GQA_STEP_EARLY_STREAM):
        res = []
        ds = [{k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)} for x in layers]
        for dl in ds:
            o = torch.empty((cfg.b, n, cfg.h, cfg.d), dtype=cfg.torch_dtype, device="cuda")
            B.gqa_decode_step_multi(dl["q"], dl["k_new"], dl["v_new"], dl["k_cache"],
                                    dl["v_cache"], dl["seq_lens"], cfg.b, n, cfg.h, cfg.g,
                                    cfg.d, cfg.d, cfg.scale, o, flags=flags)
            res.append((o, dl["k_cache"], dl["v_cache"]))
        torch.cuda.synchronize()
        outs.append(res)
    for (o1, k1, v1), (o2, k2, v2) in zip(*outs):
        assert np.array_equal(bits(o1), bits(o2))
        assert np.array_equal(bits(k1), bits(k2)) and np.array_equal(bits(v1), bits(v2))


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_length_below_n_is_reported_and_skipped(dtype, d):
    B = _b()
    cfg = cfg_of(dtype, 2, 8, 2, d, 200, seed=14)
    n = 4
    lens = np.array([200, 3], dtype=np.int32)       # 3 < n: bad
    x = make_layer_multi(cfg, n, 0, "cpu", lens=lens)
    kc0 = bits(x["k_cache"]).copy()
    out, kc, vc = gpu_step(cfg, n, x, fused=True)
    assert B.gqa_device_status() & B.GQA_DEV_BAD_SEQ_LEN
    # the bad sequence: no output written, no cache row touched
    assert torch.all(out[1].float().cpu() == 3.0)
    assert np.array_equal(bits(kc)[1], kc0[1])
    # the good one is still right
    tag = to_np(x["q"])[1]
    args = [to_np(x[k])[0][:1] for k in ("q", "k_cache", "v_cache", "k_new", "v_new")]
    ref, _, _ = oracle.decode_step_multi(*args, lens[:1], cfg.g, cfg.scale, dtype=tag)
    assert_close(oracle.widen(to_np(out)[0][:1], tag), ref, tag, "good sequence")
