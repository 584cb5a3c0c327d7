"""The paged KV cache (block table over a block pool) through the C ABI,
against the float64 oracle on the same pool and table.

The pools are the contiguous test caches scattered over a seeded random
permutation of blocks (unused blocks filled with NaN, so a read outside the
table would show).  Cases: block sizes 16..256 on the tensor-core kernel
(several blocks per tile, and several tiles per block) and with fp32 and
head dim 64, ragged lengths at block and tile edges, units split
across CTAs (merged in the decode kernel and in the combine kernel), the
fused step against the two calls and against the contiguous cache (same
bits), a bad table entry, and steps with n new tokens (the causal n-token
step through the table)."""
import math

import numpy as np
import pytest
import torch

import oracle
from gqa_kv_cache_append_gb300.inputs import DecodeConfig, make_layer, to_paged
from tests.util import assert_close, bits, to_np

pytestmark = pytest.mark.gpu


def _b():
    from gqa_kv_cache_append_gb300 import binding
    return binding


def cfg_of(dtype, b, h, g, d, cap, seed=0):
    return DecodeConfig(f"paged_{dtype}_b{b}_h{h}_g{g}_d{d}_c{cap}", 1, b, h, g, d, cap, dtype,
                        1.0 / math.sqrt(d), 800 + seed)


def paged_inputs(cfg, lens, bs, fill=float("nan")):
    lens = np.asarray(lens, dtype=np.int32)
    x = make_layer(cfg, 0, "cpu", lens=lens)
    kp, vp, table = to_paged(x["k_cache"], x["v_cache"], bs, seed=cfg.seed + bs, fill=fill)
    return x, kp, vp, table, lens


def run_paged(cfg, lens, bs, fused=True):
    B = _b()
    x, kp, vp, table, lens = paged_inputs(cfg, lens, bs)
    d = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    kp_d, vp_d, t_d = kp.cuda(), vp.cuda(), table.cuda()
    out = torch.full((cfg.b, cfg.h, cfg.d), 3.0, dtype=cfg.torch_dtype, device="cuda")
    if fused:
        B.gqa_decode_step_paged(d["q"], d["k_new"], d["v_new"], kp_d, vp_d, t_d, d["seq_lens"],
                                cfg.b, cfg.h, cfg.g, cfg.d, cfg.d, cfg.scale, out)
    else:
        B.gqa_kv_append_paged(d["k_new"], d["v_new"], kp_d, vp_d, t_d, d["seq_lens"], cfg.b,
                              cfg.g, cfg.d, cfg.d)
        B.gqa_decode_attn_paged(d["q"], kp_d, vp_d, t_d, d["seq_lens"], cfg.b, cfg.h, cfg.g,
                                cfg.d, cfg.d, cfg.scale, out)
    assert B.gqa_device_status() == 0
    tag = to_np(x["q"])[1]
    ref, kp2, vp2 = oracle.decode_step_paged(
        to_np(x["q"])[0], to_np(kp)[0], to_np(vp)[0], to_np(x["k_new"])[0], to_np(x["v_new"])[0],
        table.numpy(), lens, cfg.g, cfg.scale, bs, dtype=tag)
    assert to_np(kp_d)[0].tobytes() == kp2.tobytes()
    assert to_np(vp_d)[0].tobytes() == vp2.tobytes()
    assert_close(oracle.widen(to_np(out)[0], tag), ref, tag, f"{cfg.name}_bs{bs}")
    return out


# ---- tensor-core kernel (bf16, d = 128, tile 128)
@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
def test_tc_paged_block_sizes(bs):
    cfg = cfg_of("bf16", 4, 16, 2, 128, 512, seed=bs)
    run_paged(cfg, [1, bs - 1 if bs > 1 else 1, 257, 512], bs)


@pytest.mark.parametrize("b,h,g,cap,lens,bs", [
    (2, 64, 8, 1024, [1024, 129], 16),           # Llama heads
    (3, 32, 1, 2048, [2048, 1, 1500], 64),       # r = 32, two softmax warpgroups
    (1, 8, 1, 16384, [99 * 128 + 2], 128),       # one unit over many CTAs: combine kernel
    (96, 8, 1, 384, [258] * 96, 32),             # split units merged in the decode kernel
])
def test_tc_paged_shapes(b, h, g, cap, lens, bs):
    run_paged(cfg_of("bf16", b, h, g, 128, cap, seed=b + bs), lens, bs)


def test_tc_paged_two_calls():
    run_paged(cfg_of("bf16", 3, 16, 4, 128, 640, seed=5), [640, 300, 17], 64, fused=False)


# ---- CUDA-core kernel: fp32 (tile 128 at d = 64, 64 at d = 128); bf16 d = 64 on
# the tensor-core kernel
@pytest.mark.parametrize("dtype,d,bs", [("f32", 64, 16), ("f32", 64, 64), ("f32", 64, 256),
                                        ("f32", 128, 16), ("bf16", 64, 32), ("bf16", 64, 128)])
def test_simt_paged(dtype, d, bs):
    cfg = cfg_of(dtype, 3, 8, 2, d, 512, seed=bs + d)
    run_paged(cfg, [1, 300, 512], bs)


def test_simt_paged_split_units():
    cfg = cfg_of("f32", 1, 8, 1, 64, 8192, seed=9)
    run_paged(cfg, [99 * 64 + 2], 16)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_paged_equals_contiguous_bitwise(dtype, d):
    """Same tiles in the same order: the paged and the contiguous step give
    the same bits."""
    B = _b()
    cfg = cfg_of(dtype, 3, 16, 2, d, 1024, seed=31)
    x, kp, vp, table, lens = paged_inputs(cfg, [1024, 500, 129], 64)
    d_ = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    o1 = torch.empty((cfg.b, cfg.h, cfg.d), dtype=cfg.torch_dtype, device="cuda")
    B.gqa_decode_step(d_["q"], d_["k_new"], d_["v_new"], d_["k_cache"], d_["v_cache"],
                      d_["seq_lens"], cfg.b, cfg.h, cfg.g, cfg.d, cfg.d, cfg.scale, o1)
    o2 = torch.empty_like(o1)
    B.gqa_decode_step_paged(d_["q"], d_["k_new"], d_["v_new"], kp.cuda(), vp.cuda(),
                            table.cuda(), d_["seq_lens"], cfg.b, cfg.h, cfg.g, cfg.d, cfg.d,
                            cfg.scale, o2)
    assert np.array_equal(bits(o1), bits(o2))


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_bad_block_entry_is_reported(dtype, d):
    """A table entry outside the pool: status bit, nothing written through
    it, no access outside the pools; the other sequences are right."""
    B = _b()
    cfg = cfg_of(dtype, 2, 8, 2, d, 256, seed=41)
    x, kp, vp, table, lens = paged_inputs(cfg, [256, 200], 64, fill=0.0)
    bad = table.clone()
    bad[1, 3] = 10 ** 6                        # the block holding row 199 of sequence 1
    d_ = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    kp_d, vp_d = kp.cuda(), vp.cuda()
    out = torch.full((cfg.b, cfg.h, cfg.d), 3.0, dtype=cfg.torch_dtype, device="cuda")
    B.gqa_decode_step_paged(d_["q"], d_["k_new"], d_["v_new"], kp_d, vp_d, bad.cuda(),
                            d_["seq_lens"], cfg.b, cfg.h, cfg.g, cfg.d, cfg.d, cfg.scale, out)
    assert B.gqa_device_status() & B.GQA_DEV_BAD_BLOCK
    tag = to_np(x["q"])[1]
    ref, kp2, _ = oracle.decode_step_paged(
        to_np(x["q"])[0][:1], to_np(kp)[0], to_np(vp)[0], to_np(x["k_new"])[0][:1],
        to_np(x["v_new"])[0][:1], table.numpy()[:1], lens[:1], cfg.g, cfg.scale, 64, dtype=tag)
    assert_close(oracle.widen(to_np(out)[0][:1], tag), ref, tag, "good sequence")
    # sequence 0's append landed; sequence 1's (through the bad entry) did not
    got = to_np(kp_d)[0]
    assert got.tobytes() == kp2.tobytes()


@pytest.mark.parametrize("dtype,d,b,n,h,g,cap,lens,bs", [
    ("bf16", 128, 3, 4, 16, 2, 512, [4, 130, 512], 16),       # new rows straddle blocks/tiles
    ("bf16", 128, 2, 4, 64, 8, 1024, [1024, 257], 64),        # 32 query rows per KV head
    ("bf16", 128, 1, 4, 8, 1, 16384, [99 * 128 + 2], 128),    # combine kernel, unseen tiles
    ("f32", 64, 3, 3, 8, 2, 256, [3, 65, 256], 16),           # CUDA-core kernel
])
@pytest.mark.parametrize("fused", [True, False])
def test_paged_multi_token(dtype, d, b, n, h, g, cap, lens, bs, fused):
    from gqa_kv_cache_append_gb300.inputs import make_layer_multi
    B = _b()
    cfg = cfg_of(dtype, b, h, g, d, cap, seed=n + bs)
    lens = np.asarray(lens, dtype=np.int32)
    x = make_layer_multi(cfg, n, 0, "cpu", lens=lens)
    kp, vp, table = to_paged(x["k_cache"], x["v_cache"], bs, seed=cfg.seed, fill=float("nan"))
    dd = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    kp_d, vp_d, t_d = kp.cuda(), vp.cuda(), table.cuda()
    out = torch.full((b, n, h, d), 3.0, dtype=cfg.torch_dtype, device="cuda")
    if fused:
        B.gqa_decode_step_paged(dd["q"], dd["k_new"], dd["v_new"], kp_d, vp_d, t_d,
                                dd["seq_lens"], b, h, g, d, d, cfg.scale, out, n=n)
    else:
        B.gqa_kv_append_paged(dd["k_new"], dd["v_new"], kp_d, vp_d, t_d, dd["seq_lens"], b, g, d,
                              d, n=n)
        B.gqa_decode_attn_paged(dd["q"], kp_d, vp_d, t_d, dd["seq_lens"], b, h, g, d, d,
                                cfg.scale, out, n=n)
    assert B.gqa_device_status() == 0
    tag = to_np(x["q"])[1]
    ref, kp2, vp2 = oracle.decode_step_paged_multi(
        to_np(x["q"])[0], to_np(kp)[0], to_np(vp)[0], to_np(x["k_new"])[0], to_np(x["v_new"])[0],
        table.numpy(), lens, g, cfg.scale, bs, dtype=tag)
    assert to_np(kp_d)[0].tobytes() == kp2.tobytes()
    assert to_np(vp_d)[0].tobytes() == vp2.tobytes()
    assert_close(oracle.widen(to_np(out)[0], tag), ref, tag, f"paged n={n} bs={bs}")
