"""The seeded input recipes (CPU): the generators both the CUDA path and the
oracle take their inputs from must build what the workloads describe.

- Mean-pooled KV heads (GQA lesson, conversion of an MHA checkpoint): the
  cache at g KV heads is the average of each contiguous group of h/g heads
  of the same MHA draw, so the entries' variance falls to g/h.
- Peaked softmax (long-context MQA): round(1 %) of the positions of every
  sequence get every query head's logit raised by the boost (8), the new
  row included when its position is drawn; nothing else changes.
- Ragged lengths: uniform in [512, 32768], reproducible from the seed.
- Determinism: the same seed gives the same bits; another layer another
  draw."""
import dataclasses

import numpy as np
import pytest
import torch

from gqa_kv_cache_append_gb300.inputs import DecodeConfig, make_layer, seq_lens_for, workload


def _cfg(**kw):
    base = DecodeConfig("t", 1, 2, 8, 8, 16, 64, "f32", 0.25, 9, kind="meanpool")
    return dataclasses.replace(base, **kw)


def test_meanpool_averages_contiguous_groups_of_one_mha_draw():
    mha = make_layer(_cfg(g=8))                      # g = h: the MHA draw itself
    for g in (4, 2, 1):
        x = make_layer(_cfg(g=g))
        r = 8 // g
        for key in ("k_cache", "v_cache"):
            full = mha[key].double().numpy()         # [b, h, cap, d]
            want = full.reshape(2, g, r, *full.shape[2:]).mean(axis=2)
            got = x[key].double().numpy()
            assert np.max(np.abs(got - want)) < 1e-6, (g, key)
            if g > 1:
                # an interleaved grouping (head a -> KV head a mod g) differs
                inter = full.reshape(2, r, g, *full.shape[2:]).mean(axis=1)
                assert np.max(np.abs(got - inter)) > 0.1
        for key in ("k_new", "v_new"):
            full = mha[key].double().numpy()
            want = full.reshape(2, g, r, -1).mean(axis=2)
            assert np.max(np.abs(x[key].double().numpy() - want)) < 1e-6
        # the queries are not pooled
        assert torch.equal(x["q"], mha["q"])


def test_meanpool_variance_is_g_over_h():
    for g in (8, 2):
        x = make_layer(_cfg(g=g, b=4, cap=2048))
        var = float(x["k_cache"].double().var())
        assert abs(var - g / 8) < 0.05 * g / 8 + 0.01, (g, var)


def _boost_cfg(kind):
    return DecodeConfig("t", 1, 2, 4, 1, 16, 1000, "f32", 0.25, 5, kind=kind)


def test_boost_raises_every_head_logit_at_one_percent_of_positions():
    lens = np.array([1000, 700], dtype=np.int32)
    boosted = make_layer(_boost_cfg("boost"), lens=lens)
    plain = make_layer(_boost_cfg("plain"), lens=lens)   # the same draws (fp32)
    assert torch.equal(boosted["q"], plain["q"])
    assert torch.equal(boosted["v_cache"], plain["v_cache"])
    for i, L in enumerate(lens):
        q = boosted["q"][i].double().numpy()              # [h, d]
        # the cache after the append: row L - 1 holds k_new
        kb = boosted["k_cache"][i, 0].double().numpy().copy()
        kp = plain["k_cache"][i, 0].double().numpy().copy()
        kb[L - 1] = boosted["k_new"][i, 0].double().numpy()
        kp[L - 1] = plain["k_new"][i, 0].double().numpy()
        dlogit = 0.25 * (kb[:L] - kp[:L]) @ q.T           # [L, h]
        hit = np.any(np.abs(dlogit) > 1e-3, axis=1)
        assert int(hit.sum()) == round(0.01 * L)
        assert np.allclose(dlogit[hit], 8.0, atol=1e-3)
        assert np.all(np.abs(dlogit[~hit]) <= 1e-6)
        # rows past L_i are not touched
        assert np.array_equal(boosted["k_cache"][i, 0, L:].numpy(),
                              plain["k_cache"][i, 0, L:].numpy())


def test_boost_includes_the_new_row_when_drawn():
    # over several layers (different draws) the appended position is
    # boosted at least once: 20 of 100 positions per draw
    cfg = DecodeConfig("t", 1, 1, 4, 1, 16, 100, "f32", 0.25, 5, kind="boost",
                       boost_frac=0.2)
    plain = dataclasses.replace(cfg, kind="plain")
    seen = 0
    for layer in range(30):
        b = make_layer(cfg, layer)
        p = make_layer(plain, layer)
        seen += int(not torch.equal(b["k_new"], p["k_new"]))
    assert seen > 0


def test_ragged_lengths_are_uniform_in_range_and_seeded():
    cfg = workload("qwen25_7b_b64_ragged")
    lens = seq_lens_for(cfg)
    assert lens.dtype == np.int32 and lens.shape == (64,)
    assert lens.min() >= 512 and lens.max() <= 32768
    assert np.array_equal(lens, seq_lens_for(cfg))
    big = seq_lens_for(dataclasses.replace(cfg, b=20000))
    assert abs(big.mean() - (512 + 32768) / 2) < 0.02 * 32768
    assert big.min() < 600 and big.max() > 32700


@pytest.mark.parametrize("name", ["mqa_f32_b1_h8_d64_m256", "gqa_sweep_b16_h32_d128_m4096"])
def test_same_seed_same_bits_other_layer_other_draw(name):
    cfg = dataclasses.replace(workload(name), b=1, cap=256)
    a, b, c = make_layer(cfg, 0), make_layer(cfg, 0), make_layer(cfg, 1)
    for key in ("q", "k_cache", "v_cache", "k_new", "v_new"):
        assert torch.equal(a[key], b[key])
        assert not torch.equal(a[key], c[key])
