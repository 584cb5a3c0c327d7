"""KV append through the C ABI: bit-exact against the oracle, touching only
row L_i - 1 (past rows never change: decode notes "한 번 한 계산은 다시 하지
않기", why only K and V are stored), the prefill/decode trace of the same
page, canary rows past cap, and bad lengths reported on the status word."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from tests.util import bits

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _b():
    from gqa_kv_cache_append_gb300 import binding
    return binding


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("b,g,d,cap", [(1, 1, 64, 256), (3, 2, 128, 17), (16, 8, 128, 4096),
                                       (5, 3, 64, 9)])
def test_append_bit_exact(dtype, b, g, d, cap):
    B = _b()
    gen = torch.Generator().manual_seed(b * 7 + g)
    dev = "cuda"
    # raw random bit patterns (NaN/inf included) must be copied exactly
    kc = torch.randint(-2 ** 15, 2 ** 15, (b, g, cap + 1, d), generator=gen, dtype=torch.int32)
    if dtype == torch.bfloat16:
        kc = kc.to(torch.int16).view(torch.bfloat16)
    else:
        kc = (kc * 65537).view(torch.float32)
    vc = kc.flip(0).clone()
    kn = torch.randn((b, g, d), generator=gen).to(dtype)
    vn = torch.randn((b, g, d), generator=gen).to(dtype)
    lens = torch.randint(1, cap + 1, (b,), generator=gen, dtype=torch.int32)
    lens[0] = cap
    k_dev, v_dev = kc.to(dev), vc.to(dev)
    # pass a view with `cap` rows inside a [.., cap+1, ..] allocation per unit is
    # not contiguous; use a flat buffer with one canary row after the cache
    flat_k = torch.empty(b * g * cap * d + d, dtype=dtype, device=dev)
    flat_v = torch.empty_like(flat_k)
    flat_k[:b * g * cap * d] = k_dev[:, :, :cap].reshape(-1)
    flat_v[:b * g * cap * d] = v_dev[:, :, :cap].reshape(-1)
    canary = torch.full((d,), 12345.0 if dtype == torch.float32 else 7.0, dtype=dtype)
    flat_k[-d:] = canary.to(dev)
    flat_v[-d:] = canary.to(dev)
    B.gqa_kv_append(kn.to(dev), vn.to(dev), flat_k, flat_v, lens.to(dev), b, g, d, d, cap=cap)
    assert B.gqa_device_status() == 0
    want_k, want_v = oracle.kv_append(bits(kc[:, :, :cap]), bits(vc[:, :, :cap]), bits(kn),
                                      bits(vn), lens.numpy())
    got_k = bits(flat_k[:b * g * cap * d].view(b, g, cap, d))
    got_v = bits(flat_v[:b * g * cap * d].view(b, g, cap, d))
    assert np.array_equal(got_k, want_k)
    assert np.array_equal(got_v, want_v)
    assert np.array_equal(bits(flat_k[-d:]), bits(canary))
    assert np.array_equal(bits(flat_v[-d:]), bits(canary))


def test_decode_trace_replay():
    """Prefill 16, then decode steps to 17, 18, 19 cached tokens: each step
    appends one row and attends over the grown cache; compared with the
    oracle's step on the same inputs."""
    B = _b()
    trace = json.load(open(os.path.join(GOLDEN, "decode_trace.json")))["steps"]
    b, h, g, d, cap = 2, 8, 2, 128, 19
    gen = torch.Generator().manual_seed(5)
    kc = torch.randn((b, g, cap, d), generator=gen).to(torch.bfloat16)
    vc = torch.randn((b, g, cap, d), generator=gen).to(torch.bfloat16)
    k_dev, v_dev = kc.cuda(), vc.cuda()
    host_k, host_v = bits(kc), bits(vc)
    for step in trace[1:]:
        L = step["cache_tokens_after"]
        q = torch.randn((b, h, d), generator=gen).to(torch.bfloat16)
        kn = torch.randn((b, g, d), generator=gen).to(torch.bfloat16)
        vn = torch.randn((b, g, d), generator=gen).to(torch.bfloat16)
        lens = torch.full((b,), L, dtype=torch.int32)
        out = torch.empty((b, h, d), dtype=torch.bfloat16, device="cuda")
        B.decode_step(q.cuda(), k_dev, v_dev, kn.cuda(), vn.cuda(), lens.cuda(), g, 0.1, out)
        o_ref, host_k, host_v = oracle.decode_step(bits(q), host_k, host_v, bits(kn), bits(vn),
                                                   lens.numpy(), g, 0.1, dtype="bf16")
        assert np.array_equal(bits(k_dev), host_k)
        assert np.array_equal(bits(v_dev), host_v)
        got = oracle.widen(bits(out), "bf16")
        assert np.all(np.abs(got - o_ref) <= 2e-2 + 1e-2 * np.abs(o_ref))
    assert B.gqa_device_status() == 0


@pytest.mark.parametrize("bad", [0, -3, 18])
def test_bad_length_sets_status_and_writes_nothing(bad):
    B = _b()
    b, g, d, cap = 3, 2, 64, 17
    kc = torch.randn((b, g, cap, d)).cuda()
    vc = torch.randn((b, g, cap, d)).cuda()
    before_k, before_v = kc.clone(), vc.clone()
    kn = torch.randn((b, g, d)).cuda()
    vn = torch.randn((b, g, d)).cuda()
    lens = torch.tensor([5, bad, 17], dtype=torch.int32).cuda()
    assert B.gqa_device_status() == 0
    B.gqa_kv_append(kn, vn, kc, vc, lens, b, g, d, d)
    assert B.gqa_device_status() == B.GQA_DEV_BAD_SEQ_LEN
    assert torch.equal(kc[1], before_k[1]) and torch.equal(vc[1], before_v[1])
    assert torch.equal(kc[0, :, 4], kn[0]) and torch.equal(kc[2, :, 16], kn[2])
    assert B.gqa_device_status() == 0  # read-and-clear
