"""Head dims 64 and 128 on the tensor-core kernel, d_k and d_v independently
(the pages' einsums take separate k and v widths), and head dims above 128
(192 and 256, up to 16 query rows per KV head), through the C ABI against
the float64 oracle on the same 16-bit inputs.

Cases: bf16 and fp16; (d_k, d_v) = (64, 64), (64, 128), (128, 64); 1, 8,
16 and 32 query rows per KV head (one and two softmax warpgroups); ragged
lengths at tile edges; units held whole and split across CTAs (merged in the
decode kernel and in the combine kernel); the fused step and the two calls
(appended rows bit-exact); n new tokens with the causal mask; the paged
cache; the allocation-free call; and the CUDA-core kernel on request
(GQA_STEP_CUDA_CORES) on the same inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.util import assert_close, bits, to_np

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "f16": torch.float16}


def _b():
    from gqa_kv_cache_append_gb300 import binding
    return binding


def _case(dtype, b, n, h, g, dk, dv, cap, lens, seed):
    """Seeded N(0,1) inputs with K and V widths of their own (the workload
    generators use one head dim).  n = 0: the one-token layouts."""
    gen = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(s, generator=gen).to(DT[dtype])
    nn = max(n, 1)
    tok = () if n == 0 else (n,)
    return dict(q=r(b, *tok, h, dk), k_cache=r(b, g, cap, dk), v_cache=r(b, g, cap, dv),
                k_new=r(b, *tok, g, dk), v_new=r(b, *tok, g, dv),
                seq_lens=torch.tensor(lens, dtype=torch.int32)), nn


def _np(x, k):
    return to_np(x[k])[0]


def run_one(dtype, b, h, g, dk, dv, cap, lens, fused=True, flags=0, seed=0):
    B = _b()
    x, _ = _case(dtype, b, 0, h, g, dk, dv, cap, lens, seed)
    d = {k: v.cuda() for k, v in x.items()}
    out = torch.full((b, h, dv), 3.0, dtype=DT[dtype], device="cuda")
    scale = 1 / math.sqrt(dk)
    if fused:
        B.gqa_decode_step(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                          d["seq_lens"], b, h, g, dk, dv, scale, out, flags=flags)
    else:
        B.gqa_kv_append(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["seq_lens"], b, g,
                        dk, dv)
        B.gqa_decode_attn(d["q"], d["k_cache"], d["v_cache"], d["seq_lens"], b, h, g, dk, dv,
                          scale, out)
    assert B.gqa_device_status() == 0
    ref, kc, vc = oracle.decode_step(*(_np(x, k) for k in ("q", "k_cache", "v_cache", "k_new",
                                                             "v_new")),
                                     np.asarray(lens), g, scale, dtype=dtype)
    assert to_np(d["k_cache"])[0].tobytes() == kc.tobytes()
    assert to_np(d["v_cache"])[0].tobytes() == vc.tobytes()
    assert_close(oracle.widen(to_np(out)[0], dtype), ref, dtype,
                 f"{dtype} dk{dk} dv{dv} b{b} h{h} g{g}")
    return out


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64)])
@pytest.mark.parametrize("b,h,g,cap,lens", [
    (3, 8, 1, 400, [400, 129, 1]),            # r = 8
    (2, 32, 1, 300, [300, 128]),              # r = 32: two softmax warpgroups
    (4, 16, 16, 256, [1, 127, 128, 256]),     # r = 1 (MHA)
    (2, 32, 2, 520, [520, 3]),                # r = 16
    (1, 8, 1, 16384, [99 * 128 + 2]),         # one unit over many CTAs: combine kernel
    (96, 8, 2, 384, [258] * 96),              # split units merged in the decode kernel
])
def test_tc_head_dims(dtype, dk, dv, b, h, g, cap, lens):
    from gqa_kv_cache_append_gb300 import binding as B
    assert B.gqa_decode_plan(b, 1, h, g, dk, dv, cap, dtype)["tensor_core"]
    run_one(dtype, b, h, g, dk, dv, cap, lens, seed=dk + 3 * dv + b + h)


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64)])
def test_tc_head_dims_two_calls(dk, dv):
    run_one("bf16", 3, 16, 2, dk, dv, 640, [640, 300, 17], fused=False, seed=dk + dv)


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 64)])
def test_tc_head_dims_nan_padding(dk, dv):
    """Rows past L_i hold NaN: they must not reach the result (masked
    logits, zeroed V rows)."""
    B = _b()
    b, h, g, cap, lens = 2, 16, 2, 300, [131, 250]
    x, _ = _case("bf16", b, 0, h, g, dk, dv, cap, lens, seed=17)
    for t in (x["k_cache"], x["v_cache"]):
        for i, L in enumerate(lens):
            t[i, :, L:] = float("nan")
    d = {k: v.cuda() for k, v in x.items()}
    out = torch.empty((b, h, dv), dtype=torch.bfloat16, device="cuda")
    B.gqa_decode_attn(d["q"], d["k_cache"], d["v_cache"], d["seq_lens"], b, h, g, dk, dv, 0.1,
                      out)
    assert B.gqa_device_status() == 0
    # the oracle gets finite padding: the comparison must not depend on it
    kc, vc = (torch.nan_to_num(x[k], nan=0.0) for k in ("k_cache", "v_cache"))
    ref = oracle.grouped_decode_attention(_np(x, "q"), to_np(kc)[0], to_np(vc)[0],
                                          np.asarray(lens), g, 0.1, dtype="bf16")
    assert_close(oracle.widen(to_np(out)[0], "bf16"), ref, "bf16", "nan padding")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64)])
@pytest.mark.parametrize("fused", [True, False])
def test_tc_head_dims_multi_token(dtype, dk, dv, fused):
    """4 new tokens, 8 heads per KV head: 32 query rows, causal mask; the new
    rows straddle a tile edge for one sequence."""
    B = _b()
    b, n, h, g, cap, lens = 3, 4, 16, 2, 512, [4, 130, 512]
    x, _ = _case(dtype, b, n, h, g, dk, dv, cap, lens, seed=dk + dv + n)
    d = {k: v.cuda() for k, v in x.items()}
    out = torch.full((b, n, h, dv), 3.0, dtype=DT[dtype], device="cuda")
    scale = 1 / math.sqrt(dk)
    if fused:
        B.gqa_decode_step_multi(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                                d["seq_lens"], b, n, h, g, dk, dv, scale, out)
    else:
        B.gqa_kv_append_multi(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                              d["seq_lens"], b, n, g, dk, dv)
        B.gqa_decode_attn_multi(d["q"], d["k_cache"], d["v_cache"], d["seq_lens"], b, n, h, g,
                                dk, dv, scale, out)
    assert B.gqa_device_status() == 0
    ref, kc, vc = oracle.decode_step_multi(*(_np(x, k) for k in ("q", "k_cache", "v_cache",
                                                                   "k_new", "v_new")),
                                           np.asarray(lens), g, scale, dtype=dtype)
    assert to_np(d["k_cache"])[0].tobytes() == kc.tobytes()
    assert to_np(d["v_cache"])[0].tobytes() == vc.tobytes()
    assert_close(oracle.widen(to_np(out)[0], dtype), ref, dtype, f"n={n} dk{dk} dv{dv}")


@pytest.mark.parametrize("dk,dv,bs,n", [(64, 64, 16, 1), (64, 128, 128, 1), (128, 64, 64, 1),
                                        (64, 64, 32, 3), (128, 64, 256, 3),
                                        # head dims above 128
                                        (256, 256, 16, 1), (192, 128, 64, 1), (128, 256, 256, 3),
                                        (256, 128, 32, 3), (192, 192, 16, 1), (192, 128, 16, 3)])
def test_tc_head_dims_paged(dk, dv, bs, n):
    from gqa_kv_cache_append_gb300.inputs import to_paged
    B = _b()
    b, h, g, cap, lens = 3, 8, 2, 512, [max(1, n), 300, 512]
    x, _ = _case("bf16", b, n if n > 1 else 0, h, g, dk, dv, cap, lens, seed=bs + dk)
    kp, _, table = to_paged(x["k_cache"], x["k_cache"], bs, seed=7, fill=float("nan"))
    _, vp, _ = to_paged(x["v_cache"], x["v_cache"], bs, seed=7, fill=float("nan"))
    d = {k: v.cuda() for k, v in x.items()}
    kp_d, vp_d = kp.cuda(), vp.cuda()
    out = torch.full(tuple(x["q"].shape[:-1]) + (dv,), 3.0, dtype=torch.bfloat16, device="cuda")
    B.gqa_decode_step_paged(d["q"], d["k_new"], d["v_new"], kp_d, vp_d, table.cuda(),
                            d["seq_lens"], b, h, g, dk, dv, 0.1, out, n=n)
    assert B.gqa_device_status() == 0
    args = (_np(x, "q"), to_np(kp)[0], to_np(vp)[0], _np(x, "k_new"), _np(x, "v_new"),
            table.numpy(), np.asarray(lens), g, 0.1, bs)
    if n == 1:
        ref, kp2, vp2 = oracle.decode_step_paged(*args, dtype="bf16")
    else:
        ref, kp2, vp2 = oracle.decode_step_paged_multi(*args, dtype="bf16")
    assert to_np(kp_d)[0].tobytes() == kp2.tobytes()
    assert to_np(vp_d)[0].tobytes() == vp2.tobytes()
    assert_close(oracle.widen(to_np(out)[0], "bf16"), ref, "bf16", f"paged dk{dk} dv{dv} n{n}")


def test_tc_head_dim_64_paged_equals_contiguous_bitwise():
    """Same tiles in the same order: the same bits through the table."""
    from gqa_kv_cache_append_gb300.inputs import to_paged
    B = _b()
    b, h, g, dk, dv, cap, lens = 3, 16, 2, 64, 64, 1024, [1024, 500, 129]
    x, _ = _case("bf16", b, 0, h, g, dk, dv, cap, lens, seed=31)
    d = {k: v.cuda() for k, v in x.items()}
    kp, vp, table = to_paged(x["k_cache"], x["v_cache"], 64, seed=3)
    o1 = torch.empty((b, h, dv), dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty_like(o1)
    B.gqa_decode_attn(d["q"], d["k_cache"], d["v_cache"], d["seq_lens"], b, h, g, dk, dv, 0.1,
                      o1)
    B.gqa_decode_attn_paged(d["q"], kp.cuda(), vp.cuda(), table.cuda(), d["seq_lens"], b, h, g,
                            dk, dv, 0.1, o2)
    assert B.gqa_device_status() == 0
    assert np.array_equal(bits(o1), bits(o2))


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 64)])
def test_tc_head_dims_noalloc(dk, dv):
    B = _b()
    b, h, g, cap, lens = 4, 16, 2, 2048, [2048, 1, 700, 1500]
    x, _ = _case("bf16", b, 0, h, g, dk, dv, cap, lens, seed=dk + 1)
    d = {k: v.cuda() for k, v in x.items()}
    out = torch.empty((b, h, dv), dtype=torch.bfloat16, device="cuda")
    B.gqa_decode_attn_noalloc(d["q"], d["k_cache"], d["v_cache"], d["seq_lens"], b, h, g, dk, dv,
                              0.1, out)
    assert B.gqa_device_status() == 0
    ref = oracle.grouped_decode_attention(_np(x, "q"), _np(x, "k_cache"), _np(x, "v_cache"),
                                          np.asarray(lens), g, 0.1, dtype="bf16")
    assert_close(oracle.widen(to_np(out)[0], "bf16"), ref, "bf16", "noalloc")


@pytest.mark.parametrize("dtype,dk,dv,h,g", [("bf16", 64, 64, 8, 1), ("bf16", 128, 128, 64, 8),
                                             ("f16", 128, 64, 16, 2), ("bf16", 64, 128, 4, 4)])
def test_cuda_core_kernel_on_request(dtype, dk, dv, h, g):
    """GQA_STEP_CUDA_CORES runs the CUDA-core kernel on shapes the tensor-core
    kernel takes: both within the dtype's bound of the oracle."""
    B = _b()
    assert not B.gqa_decode_plan(3, 1, h, g, dk, dv, 700, dtype,
                                 flags=B.GQA_STEP_CUDA_CORES)["tensor_core"]
    for flags in (B.GQA_STEP_CUDA_CORES, 0):
        run_one(dtype, 3, h, g, dk, dv, 700, [700, 65, 1], flags=flags, seed=h + dk)


def test_cuda_core_multi_token_on_request():
    """The n-token step on the CUDA-core kernel with 16-bit data (8 query
    rows per KV head: 2 tokens x 4 heads), d_k != d_v."""
    B = _b()
    b, n, h, g, dk, dv, cap, lens = 3, 2, 8, 2, 64, 128, 300, [2, 129, 300]
    x, _ = _case("bf16", b, n, h, g, dk, dv, cap, lens, seed=77)
    d = {k: v.cuda() for k, v in x.items()}
    out = torch.full((b, n, h, dv), 3.0, dtype=torch.bfloat16, device="cuda")
    B.gqa_decode_step_multi(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                            d["seq_lens"], b, n, h, g, dk, dv, 0.125, out,
                            flags=B.GQA_STEP_CUDA_CORES)
    assert B.gqa_device_status() == 0
    ref, kc, vc = oracle.decode_step_multi(*(_np(x, k) for k in ("q", "k_cache", "v_cache",
                                                                   "k_new", "v_new")),
                                           np.asarray(lens), g, 0.125, dtype="bf16")
    assert to_np(d["k_cache"])[0].tobytes() == kc.tobytes()
    assert to_np(d["v_cache"])[0].tobytes() == vc.tobytes()
    assert_close(oracle.widen(to_np(out)[0], "bf16"), ref, "bf16", "CUDA cores, n = 2")


# ---- 64-wide heads (d_k = d_v = 64) take tiles of 256 positions: lengths,
# new rows and paged blocks at the 128- and 256-position edges
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("b,h,g,cap,lens", [
    (6, 8, 1, 600, [1, 127, 128, 129, 255, 256]),
    (5, 32, 2, 1100, [257, 383, 384, 385, 1100]),   # r = 16
    (2, 32, 1, 800, [511, 513]),                     # r = 32: two softmax warpgroups
    (1, 8, 1, 40000, [40000 - 77]),                  # one unit over many CTAs
    (128, 8, 1, 1024, [1024] * 128),                 # one whole unit per CTA
    (256, 8, 1, 512, [512] * 256),                   # two whole units per CTA
])
def test_wide_tiles(dtype, b, h, g, cap, lens):
    from gqa_kv_cache_append_gb300 import binding as B
    assert B.gqa_decode_plan(b, 1, h, g, 64, 64, cap, dtype)["tile"] == 256
    run_one(dtype, b, h, g, 64, 64, cap, lens, seed=b + 5 * h + cap)


@pytest.mark.parametrize("fused", [True, False])
def test_wide_tiles_multi_token(fused):
    """4 new tokens x 8 heads: the new rows straddle the two halves of a tile
    (L = 130) and two tiles (L = 258)."""
    B = _b()
    b, n, h, g, dk, dv, cap, lens = 4, 4, 16, 2, 64, 64, 600, [258, 130, 4, 600]
    x, _ = _case("bf16", b, n, h, g, dk, dv, cap, lens, seed=91)
    d = {k: v.cuda() for k, v in x.items()}
    out = torch.full((b, n, h, dv), 3.0, dtype=torch.bfloat16, device="cuda")
    if fused:
        B.gqa_decode_step_multi(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                                d["seq_lens"], b, n, h, g, dk, dv, 0.125, out)
    else:
        B.gqa_kv_append_multi(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                              d["seq_lens"], b, n, g, dk, dv)
        B.gqa_decode_attn_multi(d["q"], d["k_cache"], d["v_cache"], d["seq_lens"], b, n, h, g,
                                dk, dv, 0.125, out)
    assert B.gqa_device_status() == 0
    ref, kc, vc = oracle.decode_step_multi(*(_np(x, k) for k in ("q", "k_cache", "v_cache",
                                                                   "k_new", "v_new")),
                                           np.asarray(lens), g, 0.125, dtype="bf16")
    assert to_np(d["k_cache"])[0].tobytes() == kc.tobytes()
    assert to_np(d["v_cache"])[0].tobytes() == vc.tobytes()
    assert_close(oracle.widen(to_np(out)[0], "bf16"), ref, "bf16", "wide tiles, n = 4")


@pytest.mark.parametrize("bs,n", [(16, 1), (64, 3), (128, 1), (256, 1), (512, 3)])
def test_wide_tiles_paged(bs, n):
    """Blocks shorter than a 128-row box (one box each), as long as a box
    (two blocks a tile) and longer than a tile (both boxes from one block)."""
    from gqa_kv_cache_append_gb300.inputs import to_paged
    B = _b()
    b, h, g, dk, dv, cap, lens = 3, 8, 2, 64, 64, 1024, [max(1, n), 385, 1024]
    x, _ = _case("bf16", b, n if n > 1 else 0, h, g, dk, dv, cap, lens, seed=bs + n)
    kp, _, table = to_paged(x["k_cache"], x["k_cache"], bs, seed=9, fill=float("nan"))
    _, vp, _ = to_paged(x["v_cache"], x["v_cache"], bs, seed=9, fill=float("nan"))
    d = {k: v.cuda() for k, v in x.items()}
    kp_d, vp_d = kp.cuda(), vp.cuda()
    out = torch.full(tuple(x["q"].shape[:-1]) + (dv,), 3.0, dtype=torch.bfloat16, device="cuda")
    B.gqa_decode_step_paged(d["q"], d["k_new"], d["v_new"], kp_d, vp_d, table.cuda(),
                            d["seq_lens"], b, h, g, dk, dv, 0.1, out, n=n)
    assert B.gqa_device_status() == 0
    args = (_np(x, "q"), to_np(kp)[0], to_np(vp)[0], _np(x, "k_new"), _np(x, "v_new"),
            table.numpy(), np.asarray(lens), g, 0.1, bs)
    if n == 1:
        ref, kp2, vp2 = oracle.decode_step_paged(*args, dtype="bf16")
    else:
        ref, kp2, vp2 = oracle.decode_step_paged_multi(*args, dtype="bf16")
    assert to_np(kp_d)[0].tobytes() == kp2.tobytes()
    assert to_np(vp_d)[0].tobytes() == vp2.tobytes()
    assert_close(oracle.widen(to_np(out)[0], "bf16"), ref, "bf16", f"wide paged bs{bs} n{n}")


# ---- head dims above 128 (d_k, d_v in {128, 192, 256}, not both 128): the
# tensor-core kernel's variant with separate K and V chunks in the ring and
# two O products for d_v > 128; up to 16 query rows per KV head ----
DEEP_DIMS = [(256, 256), (192, 128), (128, 256), (256, 128), (192, 192)]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("dk,dv", DEEP_DIMS)
@pytest.mark.parametrize("b,h,g,cap,lens", [
    (3, 8, 1, 400, [400, 129, 1]),            # r = 8
    (4, 16, 16, 256, [1, 127, 128, 256]),     # r = 1 (MHA)
    (2, 32, 2, 520, [520, 3]),                # r = 16
    (1, 8, 1, 16384, [99 * 128 + 2]),         # one unit over many CTAs
    (96, 8, 2, 384, [258] * 96),              # split units merged in the decode kernel
    (16, 32, 4, 1024, [1024] * 16),           # every unit in two pieces: clusters of two
])
def test_tc_deep_head_dims(dtype, dk, dv, b, h, g, cap, lens):
    from gqa_kv_cache_append_gb300 import binding as B
    p = B.gqa_decode_plan(b, 1, h, g, dk, dv, cap, dtype)
    assert p["tensor_core"] and p["tile"] == 128
    run_one(dtype, b, h, g, dk, dv, cap, lens, seed=dk + 3 * dv + b + h)


@pytest.mark.parametrize("dk,dv", DEEP_DIMS)
def test_tc_deep_head_dims_two_calls(dk, dv):
    run_one("bf16", 3, 16, 2, dk, dv, 640, [640, 300, 17], fused=False, seed=dk + dv)


@pytest.mark.parametrize("dk,dv", [(256, 256), (192, 128)])
def test_tc_deep_head_dims_nan_padding(dk, dv):
    """Rows past L_i hold NaN: masked logits and zeroed V rows keep them out
    (with d_v = 128 the second half of a V slot is never read)."""
    B = _b()
    b, h, g, cap, lens = 2, 16, 2, 300, [131, 250]
    x, _ = _case("bf16", b, 0, h, g, dk, dv, cap, lens, seed=19)
    for t in (x["k_cache"], x["v_cache"]):
        for i, L in enumerate(lens):
            t[i, :, L:] = float("nan")
    d = {k: v.cuda() for k, v in x.items()}
    out = torch.empty((b, h, dv), dtype=torch.bfloat16, device="cuda")
    B.gqa_decode_attn(d["q"], d["k_cache"], d["v_cache"], d["seq_lens"], b, h, g, dk, dv, 0.1,
                      out)
    assert B.gqa_device_status() == 0
    kc, vc = (torch.nan_to_num(x[k], nan=0.0) for k in ("k_cache", "v_cache"))
    ref = oracle.grouped_decode_attention(_np(x, "q"), to_np(kc)[0], to_np(vc)[0],
                                          np.asarray(lens), g, 0.1, dtype="bf16")
    assert_close(oracle.widen(to_np(out)[0], "bf16"), ref, "bf16", "deep nan padding")


@pytest.mark.parametrize("dk,dv", [(256, 256), (192, 128), (128, 256)])
@pytest.mark.parametrize("n,h,g", [(2, 16, 2), (4, 8, 2), (16, 4, 4)])
def test_tc_deep_head_dims_multi_token(dk, dv, n, h, g):
    """n new tokens, n * h / g = 16 (or 4) query rows per KV head, causal
    mask; new rows straddle a tile edge for one sequence."""
    B = _b()
    b, cap = 3, 512
    lens = [n, 130, 512]
    x, _ = _case("bf16", b, n, h, g, dk, dv, cap, lens, seed=dk + dv + n)
    d = {k: v.cuda() for k, v in x.items()}
    out = torch.full((b, n, h, dv), 3.0, dtype=torch.bfloat16, device="cuda")
    scale = 1 / math.sqrt(dk)
    B.gqa_decode_step_multi(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                            d["seq_lens"], b, n, h, g, dk, dv, scale, out)
    assert B.gqa_device_status() == 0
    ref, kc, vc = oracle.decode_step_multi(*(_np(x, k) for k in ("q", "k_cache", "v_cache",
                                                                   "k_new", "v_new")),
                                           np.asarray(lens), g, scale, dtype="bf16")
    assert to_np(d["k_cache"])[0].tobytes() == kc.tobytes()
    assert to_np(d["v_cache"])[0].tobytes() == vc.tobytes()
    assert_close(oracle.widen(to_np(out)[0], "bf16"), ref, "bf16", f"deep n={n} dk{dk} dv{dv}")


def test_tc_deep_head_dims_deterministic_and_noalloc():
    """The same bits on every run, and through the allocation-free call."""
    B = _b()
    b, h, g, dk, dv, cap, lens = 4, 16, 2, 256, 256, 3000, [3000, 1, 1500, 2999]
    x, _ = _case("bf16", b, 0, h, g, dk, dv, cap, lens, seed=5)
    d = {k: v.cuda() for k, v in x.items()}
    outs = []
    for call in ("attn", "attn", "noalloc"):
        out = torch.empty((b, h, dv), dtype=torch.bfloat16, device="cuda")
        fn = B.gqa_decode_attn if call == "attn" else B.gqa_decode_attn_noalloc
        fn(d["q"], d["k_cache"], d["v_cache"], d["seq_lens"], b, h, g, dk, dv, 0.1, out)
        outs.append(out)
    assert B.gqa_device_status() == 0
    assert np.array_equal(bits(outs[0]), bits(outs[1]))
    assert np.array_equal(bits(outs[0]), bits(outs[2]))
    ref = oracle.grouped_decode_attention(_np(x, "q"), _np(x, "k_cache"), _np(x, "v_cache"),
                                          np.asarray(lens), g, 0.1, dtype="bf16")
    assert_close(oracle.widen(to_np(outs[0])[0], "bf16"), ref, "bf16", "deep determinism")


@pytest.mark.parametrize("dk,dv", [(256, 256), (192, 128), (128, 256), (128, 128), (64, 64)])
@pytest.mark.parametrize("flags", [0, 1])
def test_tc_long_segments(monkeypatch, dk, dv, flags):
    """Two CTAs for four units of 32 tiles: every CTA streams whole units,
    so its ring slots cycle through many fills (with wide heads a slot holds
    K and V chunks by turns).  flags = 1: the early-streaming step."""
    monkeypatch.setenv("GQA_CTAS", "2")
    B = _b()
    b, h, g, cap = 2, 16, 2, 4096
    lens = [4096, 4096 - 77]
    x, _ = _case("bf16", b, 0, h, g, dk, dv, cap, lens, seed=dk * 7 + dv + flags)
    d = {k: v.cuda() for k, v in x.items()}
    assert B.gqa_decode_plan(b, 1, h, g, dk, dv, cap, "bf16")["ctas"] == 2
    out = torch.empty((b, h, dv), dtype=torch.bfloat16, device="cuda")
    scale = 1 / math.sqrt(dk)
    B.gqa_decode_step(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                      d["seq_lens"], b, h, g, dk, dv, scale, out,
                      flags=B.GQA_STEP_EARLY_STREAM if flags else 0)
    assert B.gqa_device_status() == 0
    ref, kc, vc = oracle.decode_step(*(_np(x, k) for k in ("q", "k_cache", "v_cache", "k_new",
                                                             "v_new")),
                                     np.asarray(lens), g, scale, dtype="bf16")
    assert to_np(d["k_cache"])[0].tobytes() == kc.tobytes()
    assert to_np(d["v_cache"])[0].tobytes() == vc.tobytes()
    assert_close(oracle.widen(to_np(out)[0], "bf16"), ref, "bf16", f"long segments {dk}/{dv}")


@pytest.mark.parametrize("dk,dv", [(256, 256), (192, 128), (128, 128)])
@pytest.mark.parametrize("flags", [0, 1])
def test_tc_long_segments_paged(monkeypatch, dk, dv, flags):
    """The long-segment case through a shuffled table of 16-row blocks."""
    from gqa_kv_cache_append_gb300.inputs import to_paged
    monkeypatch.setenv("GQA_CTAS", "2")
    B = _b()
    b, h, g, cap, bs = 2, 16, 2, 4096, 16
    lens = [4096, 4096 - 77]
    x, _ = _case("bf16", b, 0, h, g, dk, dv, cap, lens, seed=dk + dv + 11 * flags)
    kp, _, table = to_paged(x["k_cache"], x["k_cache"], bs, seed=5, fill=float("nan"))
    _, vp, _ = to_paged(x["v_cache"], x["v_cache"], bs, seed=5, fill=float("nan"))
    d = {k: v.cuda() for k, v in x.items()}
    kp_d, vp_d = kp.cuda(), vp.cuda()
    out = torch.empty((b, h, dv), dtype=torch.bfloat16, device="cuda")
    scale = 1 / math.sqrt(dk)
    B.gqa_decode_step_paged(d["q"], d["k_new"], d["v_new"], kp_d, vp_d, table.cuda(),
                            d["seq_lens"], b, h, g, dk, dv, scale, out,
                            flags=B.GQA_STEP_EARLY_STREAM if flags else 0)
    assert B.gqa_device_status() == 0
    ref, kp2, vp2 = oracle.decode_step_paged(_np(x, "q"), to_np(kp)[0], to_np(vp)[0],
                                             _np(x, "k_new"), _np(x, "v_new"), table.numpy(),
                                             np.asarray(lens), g, scale, bs, dtype="bf16")
    assert to_np(kp_d)[0].tobytes() == kp2.tobytes()
    assert to_np(vp_d)[0].tobytes() == vp2.tobytes()
    assert_close(oracle.widen(to_np(out)[0], "bf16"), ref, "bf16", f"paged long {dk}/{dv}")
