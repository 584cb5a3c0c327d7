"""gqa_decode_attn_noalloc: the decode for callers that cannot allocate
device memory (engines that gave all free HBM to their own KV pool, loops
that must not take cudaMalloc's device-wide synchronisation).  Its split
partials live in the library's fixed device array.

Checked through the C ABI against gqa_decode_attn on the same inputs, on
consecutive calls of different shapes (the array keeps the previous call's
contents, which must not matter), plus the size limit.  This file is named
to be collected last."""
import math

import numpy as np
import pytest
import torch

import oracle
from gqa_kv_cache_append_gb300.inputs import DecodeConfig, make_layer
from tests.util import assert_close, to_np

pytestmark = pytest.mark.gpu


def _b():
    from gqa_kv_cache_append_gb300 import binding
    return binding


def _both(cfg, lens):
    """Run the allocating and the allocation-free entry points on the same
    appended cache; return both outputs as float64."""
    B = _b()
    x = make_layer(cfg, 0, "cuda", lens=np.asarray(lens, dtype=np.int32))
    B.gqa_kv_append(x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], x["seq_lens"],
                    cfg.b, cfg.g, cfg.d, cfg.d)
    ref = torch.empty((cfg.b, cfg.h, cfg.d), dtype=cfg.torch_dtype, device="cuda")
    got = torch.full_like(ref, 7.0)
    B.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], cfg.b, cfg.h, cfg.g,
                      cfg.d, cfg.d, cfg.scale, ref)
    B.gqa_decode_attn_noalloc(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], cfg.b, cfg.h,
                              cfg.g, cfg.d, cfg.d, cfg.scale, got)
    assert B.gqa_device_status() == 0
    tag = to_np(ref)[1]
    return oracle.widen(to_np(got)[0], tag), oracle.widen(to_np(ref)[0], tag), tag


def _cfg(dtype, b, h, g, d, cap, seed):
    return DecodeConfig(f"noalloc_{dtype}_b{b}_h{h}_g{g}", 1, b, h, g, d, cap, dtype,
                        1.0 / math.sqrt(d), seed)


def test_matches_the_allocating_entry_point_on_consecutive_calls():
    # first call: Llama-3-70B head layout, units split across CTAs
    got, ref, tag = _both(_cfg("bf16", 8, 64, 8, 128, 3000, 11), [3000, 2999, 1, 128, 129,
                                                                    2048, 700, 1500])
    assert_close(got, ref, tag, "noalloc call 1")
    # second call, right after: another shape (MQA, r = 32, long rows) that
    # reuses the same array with a different slot layout
    got, ref, tag = _both(_cfg("bf16", 2, 32, 1, 128, 20000, 12), [20000, 777])
    assert_close(got, ref, tag, "noalloc call 2")
    # and the CUDA-core kernel (fp32)
    got, ref, tag = _both(_cfg("f32", 3, 8, 2, 64, 500, 13), [500, 64, 65])
    assert_close(got, ref, tag, "noalloc call 3")


def test_calls_beyond_the_scratch_limit_are_rejected():
    B = _b()
    b, h, g, d, cap = 4096, 64, 8, 128, 1       # needs ~136 MB of partial slots
    q = torch.zeros((b, h, d), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((b, g, cap, d), dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(b, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 3.0)
    with pytest.raises(B.GqaError) as e:
        B.gqa_decode_attn_noalloc(q, kc, kc, lens, b, h, g, d, d, 1.0, out)
    assert e.value.code == B.GQA_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert bool(torch.all(out == 3.0))
