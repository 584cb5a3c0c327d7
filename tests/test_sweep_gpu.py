"""A seeded sweep of random decode shapes through the C ABI against the
float64 oracle: sequences, query and KV heads (r = 1..32), ragged lengths
(including 1 and tile edges), one or n new tokens, head dims 64 / 128 for
K and V independently, bf16 / fp16 / fp32, contiguous or paged caches,
fused step or the two calls; and a second sweep over the head dims above
128 (128 / 192 / 256 for K and V, not both 128; bf16 / fp16, at most 16
query rows per KV head).  Each case draws its own shape from a fixed
generator, so the set is the same every run; the appended rows are
compared bit for bit, the outputs within the dtype's bound."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.util import assert_close, to_np

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
N_CASES = 40
N_WIDE = 24


def _shape(case, wide=False):
    rng = np.random.default_rng((9500 if wide else 9000) + case)
    dtype = (["bf16", "f16"][case % 2]) if wide else ["bf16", "f16", "f32"][case % 3]
    g = int(rng.choice([1, 2, 4, 8]))
    n = int(rng.choice([1, 1, 1, 2, 4]))
    rmax = (16 if (dtype == "f32" or wide) else 32) // n
    r = int(rng.choice([x for x in (1, 2, 4, 7, 8, 16, 32) if x <= rmax]))
    b = int(rng.integers(1, 9))
    if wide:
        dk, dv = 128, 128
        while dk == 128 and dv == 128:
            dk = int(rng.choice([128, 192, 256]))
            dv = int(rng.choice([128, 192, 256]))
    else:
        dk = int(rng.choice([64, 128]))
        dv = int(rng.choice([64, 128]))
    cap = int(rng.choice([128, 256, 640, 1500, 4096]))
    lens = rng.integers(n, cap + 1, size=b)
    edge = [n, 127, 128, 129, cap]
    for i in range(b):
        if rng.random() < 0.3:
            lens[i] = max(n, min(cap, int(rng.choice(edge))))
    paged = int(rng.choice([0, 0, 16, 64, 256])) if cap % 256 == 0 else 0
    fused = bool(rng.random() < 0.7)
    return dict(dtype=dtype, b=b, n=n, h=g * r, g=g, dk=dk, dv=dv, cap=cap,
                lens=lens.astype(np.int32), paged=paged, fused=fused, seed=case)


@pytest.mark.parametrize("case", range(N_CASES))
def test_random_shape(case):
    _run(_shape(case))


@pytest.mark.parametrize("case", range(N_WIDE))
def test_random_wide_shape(case):
    _run(_shape(case, wide=True))


def _run(s):
    from gqa_kv_cache_append_gb300 import binding as B
    from gqa_kv_cache_append_gb300.inputs import to_paged
    case = s["seed"]
    dt, b, n, h, g, dk, dv, cap = (s[k] for k in ("dtype", "b", "n", "h", "g", "dk", "dv", "cap"))
    gen = torch.Generator().manual_seed(77 + case)
    rnd = lambda *sh: torch.randn(sh, generator=gen).to(DT[dt])
    tok = (n,) if n > 1 else ()
    x = dict(q=rnd(b, *tok, h, dk), k_cache=rnd(b, g, cap, dk), v_cache=rnd(b, g, cap, dv),
             k_new=rnd(b, *tok, g, dk), v_new=rnd(b, *tok, g, dv))
    lens = s["lens"]
    scale = 1.0 / math.sqrt(dk)
    d = {k: v.cuda() for k, v in x.items()}
    d["seq_lens"] = torch.from_numpy(lens.copy()).cuda()
    out = torch.full((b, *tok, h, dv), 3.0, dtype=DT[dt], device="cuda")
    args = [to_np(x[k])[0] for k in ("q", "k_cache", "v_cache", "k_new", "v_new")]
    if s["paged"]:
        bs = s["paged"]
        kp, _, table = to_paged(x["k_cache"], x["k_cache"], bs, seed=case, fill=float("nan"))
        _, vp, _ = to_paged(x["v_cache"], x["v_cache"], bs, seed=case, fill=float("nan"))
        kp_d, vp_d, t_d = kp.cuda(), vp.cuda(), table.cuda()
        if s["fused"]:
            B.gqa_decode_step_paged(d["q"], d["k_new"], d["v_new"], kp_d, vp_d, t_d,
                                    d["seq_lens"], b, h, g, dk, dv, scale, out, n=n)
        else:
            B.gqa_kv_append_paged(d["k_new"], d["v_new"], kp_d, vp_d, t_d, d["seq_lens"], b, g,
                                  dk, dv, n=n)
            B.gqa_decode_attn_paged(d["q"], kp_d, vp_d, t_d, d["seq_lens"], b, h, g, dk, dv,
                                    scale, out, n=n)
        pargs = (args[0], to_np(kp)[0], to_np(vp)[0], args[3], args[4], table.numpy(), lens, g,
                 scale, bs)
        if n == 1:
            ref, kc, vc = oracle.decode_step_paged(*pargs, dtype=dt)
        else:
            ref, kc, vc = oracle.decode_step_paged_multi(*pargs, dtype=dt)
        got_k, got_v = to_np(kp_d)[0], to_np(vp_d)[0]
    else:
        if n == 1:
            if s["fused"]:
                B.gqa_decode_step(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                                  d["seq_lens"], b, h, g, dk, dv, scale, out)
            else:
                B.gqa_kv_append(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                                d["seq_lens"], b, g, dk, dv)
                B.gqa_decode_attn(d["q"], d["k_cache"], d["v_cache"], d["seq_lens"], b, h, g,
                                  dk, dv, scale, out)
            ref, kc, vc = oracle.decode_step(*args, lens, g, scale, dtype=dt)
        else:
            if s["fused"]:
                B.gqa_decode_step_multi(d["q"], d["k_new"], d["v_new"], d["k_cache"],
                                        d["v_cache"], d["seq_lens"], b, n, h, g, dk, dv, scale,
                                        out)
            else:
                B.gqa_kv_append_multi(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                                      d["seq_lens"], b, n, g, dk, dv)
                B.gqa_decode_attn_multi(d["q"], d["k_cache"], d["v_cache"], d["seq_lens"], b, n,
                                        h, g, dk, dv, scale, out)
            ref, kc, vc = oracle.decode_step_multi(*args, lens, g, scale, dtype=dt)
        got_k, got_v = to_np(d["k_cache"])[0], to_np(d["v_cache"])[0]
    assert B.gqa_device_status() == 0, s
    assert got_k.tobytes() == kc.tobytes(), s
    assert got_v.tobytes() == vc.tobytes(), s
    assert_close(oracle.widen(to_np(out)[0], dt), ref, dt, str(s))
