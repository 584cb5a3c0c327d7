"""gqa_decode_attn_noalloc: the decode for callers that cannot allocate
device memory (engines that gave all free HBM to their own KV pool, loops
that must not take cudaMalloc's device-wide synchronisation).  Its split
partials live in the library's fixed device array.

Checked through the C ABI on consecutive calls of different shapes (the
array keeps the previous call's contents, which must not matter): bit for
bit against gqa_decode_attn on the same inputs (the same kernel, grid and
slot layout), and against the float64 oracle on inputs copied to the host
before the calls.  Also: the exact size limit (the largest accepted call
and one unit more), and that a call allocates no device memory.  This file
is named to be collected last."""
import math

import numpy as np
import pytest
import torch

import oracle
from gqa_kv_cache_append_gb300.inputs import DecodeConfig, make_layer
from tests.util import assert_close, bits, to_np

pytestmark = pytest.mark.gpu

# bytes of the array that hold the partials (the first 256 KiB of the 4 MiB
# hold the arrival counters)
PARTIAL_BYTES = (4 << 20) - (256 << 10)


def _b():
    from gqa_kv_cache_append_gb300 import binding
    return binding


def _both(cfg, lens):
    """Append, then run the allocating and the allocation-free entry points on
    the same cache.  Returns (noalloc out, gqa_decode_attn out, oracle out as
    float64, dtype tag); the oracle's inputs are host copies taken before any
    call."""
    B = _b()
    x = make_layer(cfg, 0, "cuda", lens=np.asarray(lens, dtype=np.int32))
    host = {k: to_np(x[k]) for k in ("q", "k_cache", "v_cache", "k_new", "v_new")}
    tag = host["q"][1]
    B.gqa_kv_append(x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], x["seq_lens"],
                    cfg.b, cfg.g, cfg.d, cfg.d)
    ref = torch.empty((cfg.b, cfg.h, cfg.d), dtype=cfg.torch_dtype, device="cuda")
    got = torch.full_like(ref, 7.0)
    B.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], cfg.b, cfg.h, cfg.g,
                      cfg.d, cfg.d, cfg.scale, ref)
    B.gqa_decode_attn_noalloc(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], cfg.b, cfg.h,
                              cfg.g, cfg.d, cfg.d, cfg.scale, got)
    assert B.gqa_device_status() == 0
    want, _, _ = oracle.decode_step(host["q"][0], host["k_cache"][0], host["v_cache"][0],
                                    host["k_new"][0], host["v_new"][0], np.asarray(lens),
                                    cfg.g, cfg.scale, dtype=tag)
    return got, ref, want, tag


def _check(cfg, lens, what):
    got, ref, want, tag = _both(cfg, lens)
    assert np.array_equal(bits(got), bits(ref)), f"{what}: differs from gqa_decode_attn"
    assert_close(oracle.widen(to_np(got)[0], tag), want, tag, what)


def _cfg(dtype, b, h, g, d, cap, seed):
    return DecodeConfig(f"noalloc_{dtype}_b{b}_h{h}_g{g}", 1, b, h, g, d, cap, dtype,
                        1.0 / math.sqrt(d), seed)


def test_matches_the_allocating_entry_point_on_consecutive_calls():
    # first call: Llama-3-70B head layout, units split across CTAs
    _check(_cfg("bf16", 8, 64, 8, 128, 3000, 11), [3000, 2999, 1, 128, 129, 2048, 700, 1500],
           "noalloc call 1")
    # second call, right after: another shape (MQA, r = 32, long rows) that
    # reuses the same array with a different slot layout
    _check(_cfg("bf16", 2, 32, 1, 128, 20000, 12), [20000, 777], "noalloc call 2")
    # and the CUDA-core kernel (fp32)
    _check(_cfg("f32", 3, 8, 2, 64, 500, 13), [500, 64, 65], "noalloc call 3")


def _largest_batch(h, g, d, cap):
    """The largest b whose partials fit: (b*g + C) * (h/g) * (d + 2) * 4 bytes,
    C the CTAs the call's plan launches."""
    B = _b()
    slot = (h // g) * (d + 2) * 4
    b = 1
    while True:
        nxt = b + 1
        c = B.gqa_decode_plan(nxt, 1, h, g, d, d, cap, "bf16")["ctas"]
        if (nxt * g + c) * slot > PARTIAL_BYTES:
            return b
        b = nxt


def test_largest_accepted_call_and_one_unit_more():
    B = _b()
    h, g, d, cap = 64, 8, 128, 256
    b = _largest_batch(h, g, d, cap)
    # the largest accepted batch runs and matches (ragged, short lengths)
    lens = (np.arange(b) * 37) % cap + 1
    _check(_cfg("bf16", b, h, g, d, cap, 14), lens, f"noalloc at the limit (b={b})")
    # one sequence more is refused before any launch, `out` untouched
    b1 = b + 1
    q = torch.zeros((b1, h, d), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((b1, g, cap, d), dtype=torch.bfloat16, device="cuda")
    seq = torch.ones(b1, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 3.0)
    torch.cuda.synchronize()
    with pytest.raises(B.GqaError) as e:
        B.gqa_decode_attn_noalloc(q, kc, kc, seq, b1, h, g, d, d, 1.0, out)
    assert e.value.code == B.GQA_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert bool(torch.all(out == 3.0))


def test_far_beyond_the_scratch_limit_is_rejected():
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


def test_a_call_on_a_fresh_stream_allocates_no_device_memory():
    B = _b()
    cfg = _cfg("bf16", 4, 32, 4, 128, 4096, 15)
    x = make_layer(cfg, 0, "cuda")
    out = torch.empty((cfg.b, cfg.h, cfg.d), dtype=torch.bfloat16, device="cuda")
    args = (x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], cfg.b, cfg.h, cfg.g, cfg.d,
            cfg.d, cfg.scale, out)
    # load the kernels once (module loading may reserve memory)
    B.gqa_decode_attn_noalloc(*args)
    torch.cuda.synchronize()
    fresh = torch.cuda.Stream()
    first = out.clone()
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    B.gqa_decode_attn_noalloc(*args, stream=fresh)
    fresh.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    assert np.array_equal(bits(out), bits(first))
    assert B.gqa_device_status(fresh) == 0
