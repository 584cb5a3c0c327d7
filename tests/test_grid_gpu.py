"""How the decode kernel hands out work, through the C ABI against the
float64 oracle on the same inputs.

When every sequence has the same number of tiles, the tensor-core kernel may
give each CTA whole (sequence, KV head) units instead of an even share of
all tiles: one unit per CTA when that still uses at least 70 % of the CTAs,
two with 128-wide heads, never on a paged cache.  The cases below size the
batch from the device's SM count so that each regime is reached: one and
two whole units per CTA, the same batches just outside the rule (too few
units, three per CTA, a ragged batch, 64-wide heads, d_v != d_k, a paged
cache), lengths that differ inside one tile (still equal in tiles), one and
n new tokens, bf16 and fp16.  Every output is compared with the oracle and
the appended rows bit for bit."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.util import assert_close, to_np

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "f16": torch.float16}


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _b():
    from gqa_kv_cache_append_gb300 import binding
    return binding


def _units(regime, nsm, g):
    """A unit count (a multiple of g) in the given regime for nsm CTAs."""
    lo1 = -(-7 * nsm // 10)                         # fewest units for one per CTA
    want = {"one": nsm - 8,                         # lo1 <= u < nsm
            "two": 2 * nsm - 16,                    # 2 lo1 <= u < 2 nsm, even
            "three": 3 * nsm - 24,                  # more than two per CTA
            "few": (6 * nsm) // 10}[regime]         # under 70 %, over half
    u = (want // (2 * g)) * 2 * g
    if regime == "one":
        assert lo1 <= u < nsm
    if regime == "two":
        assert 2 * lo1 <= u < 2 * nsm and (u // 2) * 2 == u
    return u


def _run(dtype, b, n, h, g, dk, dv, cap, lens, paged=0, seed=0):
    B = _b()
    from gqa_kv_cache_append_gb300.inputs import to_paged
    gen = torch.Generator().manual_seed(500 + seed)
    rnd = lambda *s: torch.randn(s, generator=gen).to(DT[dtype])
    tok = (n,) if n > 1 else ()
    x = dict(q=rnd(b, *tok, h, dk), k_cache=rnd(b, g, cap, dk), v_cache=rnd(b, g, cap, dv),
             k_new=rnd(b, *tok, g, dk), v_new=rnd(b, *tok, g, dv))
    lens = np.asarray(lens, dtype=np.int32)
    scale = 1.0 / math.sqrt(dk)
    d = {k: v.cuda() for k, v in x.items()}
    d_lens = torch.from_numpy(lens.copy()).cuda()
    out = torch.full((b, *tok, h, dv), 3.0, dtype=DT[dtype], device="cuda")
    args = [to_np(x[k])[0] for k in ("q", "k_cache", "v_cache", "k_new", "v_new")]
    if paged:
        kp, _, table = to_paged(x["k_cache"], x["k_cache"], paged, seed=seed, fill=float("nan"))
        _, vp, _ = to_paged(x["v_cache"], x["v_cache"], paged, seed=seed, fill=float("nan"))
        kp_d, vp_d, t_d = kp.cuda(), vp.cuda(), table.cuda()
        B.gqa_decode_step_paged(d["q"], d["k_new"], d["v_new"], kp_d, vp_d, t_d, d_lens, b, h,
                                g, dk, dv, scale, out, n=n)
        pargs = (args[0], to_np(kp)[0], to_np(vp)[0], args[3], args[4], table.numpy(), lens, g,
                 scale, paged)
        step = oracle.decode_step_paged if n == 1 else oracle.decode_step_paged_multi
        ref, kc, vc = step(*pargs, dtype=dtype)
        got_k, got_v = to_np(kp_d)[0], to_np(vp_d)[0]
    else:
        if n == 1:
            B.gqa_decode_step(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d_lens,
                              b, h, g, dk, dv, scale, out)
            ref, kc, vc = oracle.decode_step(*args, lens, g, scale, dtype=dtype)
        else:
            B.gqa_decode_step_multi(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                                    d_lens, b, n, h, g, dk, dv, scale, out)
            ref, kc, vc = oracle.decode_step_multi(*args, lens, g, scale, dtype=dtype)
        got_k, got_v = to_np(d["k_cache"])[0], to_np(d["v_cache"])[0]
    assert B.gqa_device_status() == 0
    assert got_k.tobytes() == kc.tobytes()
    assert got_v.tobytes() == vc.tobytes()
    return assert_close(oracle.widen(to_np(out)[0], dtype), ref, dtype,
                        f"{dtype} b{b} n{n} h{h} g{g} {dk}/{dv} paged{paged}")


# (regime, dtype, n, h, g, dk, dv, cap, paged)
CASES = [
    ("one", "bf16", 1, 64, 8, 128, 128, 260, 0),    # one whole unit per CTA
    ("two", "bf16", 1, 32, 8, 128, 128, 300, 0),    # two per CTA (128-wide heads)
    ("one", "bf16", 1, 64, 8, 64, 64, 260, 0),      # 64-wide heads: one per CTA
    ("two", "bf16", 1, 32, 8, 64, 64, 300, 0),      # 64-wide heads: even split
    ("two", "bf16", 1, 32, 8, 128, 64, 300, 0),     # d_v != d_k: even split
    ("three", "bf16", 1, 32, 8, 128, 128, 260, 0),  # three per CTA: even split
    ("few", "bf16", 1, 64, 8, 128, 128, 260, 0),    # under 70 % of the CTAs
    ("two", "bf16", 1, 32, 8, 128, 128, 256, 16),   # paged: the rule is off
    ("one", "bf16", 2, 64, 8, 128, 128, 260, 0),    # 2 new tokens, 16 rows
    ("two", "bf16", 4, 32, 8, 128, 128, 300, 0),    # 4 new tokens, 16 rows
    ("one", "bf16", 4, 32, 4, 128, 128, 384, 0),    # r = 8, 32 rows
    ("one", "f16", 1, 64, 8, 128, 128, 260, 0),
    ("two", "f16", 1, 16, 4, 128, 128, 200, 0),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_equal_tiles(case):
    regime, dtype, n, h, g, dk, dv, cap, paged = CASES[case]
    b = _units(regime, _sms(), g) // g
    _run(dtype, b, n, h, g, dk, dv, cap, [cap] * b, paged=paged, seed=case)


@pytest.mark.parametrize("regime", ["one", "two"])
def test_lengths_differ_inside_one_tile(regime):
    """Lengths 257..384 all take three 128-position tiles: the batch still
    counts as equal, and each unit's own length bounds its positions."""
    g, h = 8, 32 if regime == "two" else 64
    b = _units(regime, _sms(), g) // g
    lens = np.random.default_rng(11).integers(257, 385, b)
    lens[0], lens[-1] = 257, 384
    _run("bf16", b, 1, h, g, 128, 128, 384, lens, seed=40)


@pytest.mark.parametrize("regime", ["one", "two"])
def test_one_sequence_a_tile_longer(regime):
    """One sequence a tile longer than the rest: the batch is ragged in
    tiles, so the even split over all CTAs applies."""
    g, h = 8, 32 if regime == "two" else 64
    b = _units(regime, _sms(), g) // g
    lens = [256] * b
    lens[b // 2] = 300
    _run("bf16", b, 1, h, g, 128, 128, 300, lens, seed=41)


def test_single_position_units():
    """L = 1 everywhere (the first token of every sequence), one whole unit
    per CTA: each CTA's only tile holds one valid row."""
    g = 8
    b = _units("one", _sms(), g) // g
    _run("bf16", b, 1, 64, g, 128, 128, 128, [1] * b, seed=42)
