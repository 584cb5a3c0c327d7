"""K and V head dims that differ (d_k != d_v; the pages' P_k [h, d, k] and
P_v [h, d, v] let them), through the C ABI against the float64 oracle:
contiguous and paged caches, fused and two-call steps, units held whole and
split across CTAs (merged in the decode kernel and in the combine kernel),
fp32 (CUDA-core kernel) and bf16 (tensor-core kernel)."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.util import assert_close, to_np

pytestmark = pytest.mark.gpu


def _b():
    from gqa_kv_cache_append_gb300 import binding
    return binding


def _case(dtype, b, h, g, dk, dv, cap, lens, seed):
    """Seeded N(0,1) inputs with different K and V widths (drawn here: the
    workload generators use one head dim)."""
    gen = torch.Generator().manual_seed(seed)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    r = lambda *s: torch.randn(s, generator=gen).to(dt)
    return dict(q=r(b, h, dk), k_cache=r(b, g, cap, dk), v_cache=r(b, g, cap, dv),
                k_new=r(b, g, dk), v_new=r(b, g, dv),
                seq_lens=torch.tensor(lens, dtype=torch.int32)), dt


@pytest.mark.parametrize("dtype,b,h,g,dk,dv,cap,lens", [
    ("f32", 3, 8, 2, 64, 128, 300, [1, 65, 300]),
    ("f32", 2, 16, 1, 128, 64, 200, [200, 33]),          # r = 16
    ("bf16", 3, 8, 1, 64, 128, 400, [400, 129, 1]),
    ("bf16", 2, 4, 4, 128, 64, 260, [128, 259]),
    ("f32", 1, 4, 1, 64, 128, 8192, [99 * 32 + 2]),      # one unit over many CTAs: combine
    ("f32", 96, 2, 1, 128, 64, 160, [70] * 96),          # split units merged in the kernel
])
@pytest.mark.parametrize("fused", [True, False])
def test_dk_ne_dv(dtype, b, h, g, dk, dv, cap, lens, fused):
    B = _b()
    x, dt = _case(dtype, b, h, g, dk, dv, cap, lens, seed=dk * 7 + dv + b)
    d = {k: v.cuda() for k, v in x.items()}
    out = torch.full((b, h, dv), 3.0, dtype=dt, device="cuda")
    if fused:
        B.gqa_decode_step(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                          d["seq_lens"], b, h, g, dk, dv, 1 / math.sqrt(dk), out)
    else:
        B.gqa_kv_append(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["seq_lens"], b, g,
                        dk, dv)
        B.gqa_decode_attn(d["q"], d["k_cache"], d["v_cache"], d["seq_lens"], b, h, g, dk, dv,
                          1 / math.sqrt(dk), out)
    assert B.gqa_device_status() == 0
    tag = to_np(x["q"])[1]
    ref, kc, vc = oracle.decode_step(*(to_np(x[k])[0] for k in ("q", "k_cache", "v_cache",
                                                                 "k_new", "v_new")),
                                     np.asarray(lens), g, 1 / math.sqrt(dk), dtype=tag)
    assert to_np(d["k_cache"])[0].tobytes() == kc.tobytes()
    assert to_np(d["v_cache"])[0].tobytes() == vc.tobytes()
    assert_close(oracle.widen(to_np(out)[0], tag), ref, tag, f"dk{dk}_dv{dv}")


@pytest.mark.parametrize("dtype,dk,dv,bs", [("f32", 64, 128, 16), ("bf16", 128, 64, 64)])
def test_dk_ne_dv_paged(dtype, dk, dv, bs):
    from gqa_kv_cache_append_gb300.inputs import to_paged
    B = _b()
    b, h, g, cap, lens = 3, 8, 2, 256, [256, 100, 1]
    x, dt = _case(dtype, b, h, g, dk, dv, cap, lens, seed=5)
    kp, _, table = to_paged(x["k_cache"], x["k_cache"], bs, seed=7, fill=float("nan"))
    _, vp, _ = to_paged(x["v_cache"], x["v_cache"], bs, seed=7, fill=float("nan"))
    d = {k: v.cuda() for k, v in x.items()}
    kp_d, vp_d = kp.cuda(), vp.cuda()
    out = torch.full((b, h, dv), 3.0, dtype=dt, device="cuda")
    B.gqa_decode_step_paged(d["q"], d["k_new"], d["v_new"], kp_d, vp_d, table.cuda(),
                            d["seq_lens"], b, h, g, dk, dv, 0.1, out)
    assert B.gqa_device_status() == 0
    tag = to_np(x["q"])[1]
    ref, kp2, vp2 = oracle.decode_step_paged(
        to_np(x["q"])[0], to_np(kp)[0], to_np(vp)[0], to_np(x["k_new"])[0], to_np(x["v_new"])[0],
        table.numpy(), np.asarray(lens), g, 0.1, bs, dtype=tag)
    assert to_np(kp_d)[0].tobytes() == kp2.tobytes()
    assert to_np(vp_d)[0].tobytes() == vp2.tobytes()
    assert_close(oracle.widen(to_np(out)[0], tag), ref, tag, "paged dk != dv")
