"""Pins of the oracle's layer around the step (CPU, no GPU): the projections
of x into q and the new K/V rows, the output projection, and the storage
rounding between them.

Each pin checks the oracle against something other than itself:
  * the literal MultiheadSelfAttentionIncremental of the MQA review §2.4
    (einsum by einsum, with the concat of the new row) at g = h;
  * the literal MultiquerySelfAttentionIncremental of §3 (P_k [d, k],
    P_v [d, v]) at g = 1;
  * grouped KV heads = MHA whose K/V projections and caches repeat each KV
    head r = h / g times;
  * plain Python loops on tiny sizes;
  * the bf16 rounding against torch's float32 -> bfloat16 conversion, and
    against the definition of round-to-nearest-even on float64 values.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import oracle as orc


TOL = 1e-10


def _softmax(x, axis=-1):
    e = np.exp(x - x.max(axis=axis, keepdims=True))
    return e / e.sum(axis=axis, keepdims=True)


def _mha_layer_literal(x, prev_K, prev_V, P_q, P_k, P_v, P_o, scale):
    # MQA review §2.4, step by step
    q = np.einsum("bd,hdk->bhk", x, P_q)
    new_K = np.concatenate([prev_K, np.einsum("bd,hdk->bhk", x, P_k)[:, :, None]], axis=2)
    new_V = np.concatenate([prev_V, np.einsum("bd,hdv->bhv", x, P_v)[:, :, None]], axis=2)
    logits = scale * np.einsum("bhk,bhmk->bhm", q, new_K)
    weights = _softmax(logits)
    o = np.einsum("bhm,bhmv->bhv", weights, new_V)
    y = np.einsum("bhv,hdv->bd", o, P_o)
    return y, new_K, new_V


def _mqa_layer_literal(x, prev_K, prev_V, P_q, P_k, P_v, P_o, scale):
    # MQA review §3, step by step (no KV-head axis)
    q = np.einsum("bd,hdk->bhk", x, P_q)
    new_K = np.concatenate([prev_K, np.einsum("bd,dk->bk", x, P_k)[:, None]], axis=1)
    new_V = np.concatenate([prev_V, np.einsum("bd,dv->bv", x, P_v)[:, None]], axis=1)
    logits = scale * np.einsum("bhk,bmk->bhm", q, new_K)
    weights = _softmax(logits)
    o = np.einsum("bhm,bmv->bhv", weights, new_V)
    y = np.einsum("bhv,hdv->bd", o, P_o)
    return y, new_K, new_V


def _case(rng, b, D, h, g, dk, dv, cap):
    return dict(
        x=rng.standard_normal((b, D)),
        P_q=rng.standard_normal((h, D, dk)) / np.sqrt(D),
        P_k=rng.standard_normal((g, D, dk)) / np.sqrt(D),
        P_v=rng.standard_normal((g, D, dv)) / np.sqrt(D),
        P_o=rng.standard_normal((h, D, dv)) / np.sqrt(h * dv),
        kc=rng.standard_normal((b, g, cap, dk)),
        vc=rng.standard_normal((b, g, cap, dv)),
    )


@pytest.mark.parametrize("b,D,h,dk,dv,L", [(2, 12, 3, 4, 5, 6), (3, 16, 4, 8, 8, 1)])
def test_layer_at_g_equals_h_is_the_literal_mha_layer(b, D, h, dk, dv, L):
    rng = np.random.default_rng(1000 + D)
    c = _case(rng, b, D, h, h, dk, dv, L + 2)
    lens = np.full(b, L)
    y, kc, vc, _, _ = oracle.decode_layer(c["x"], c["P_q"], c["P_k"], c["P_v"], c["P_o"],
                                          c["kc"], c["vc"], lens, h, 0.4)
    y2, K2, V2 = _mha_layer_literal(c["x"], c["kc"][:, :, :L - 1], c["vc"][:, :, :L - 1],
                                    c["P_q"], c["P_k"], c["P_v"], c["P_o"], 0.4)
    assert np.max(np.abs(y - y2)) < TOL
    assert np.max(np.abs(kc[:, :, :L] - K2)) < TOL
    assert np.max(np.abs(vc[:, :, :L] - V2)) < TOL


@pytest.mark.parametrize("b,D,h,dk,dv,L", [(2, 10, 4, 3, 6, 5), (1, 8, 8, 4, 4, 9)])
def test_layer_at_g_equals_1_is_the_literal_mqa_layer(b, D, h, dk, dv, L):
    rng = np.random.default_rng(2000 + D)
    c = _case(rng, b, D, h, 1, dk, dv, L)
    lens = np.full(b, L)
    y, kc, vc, _, _ = oracle.decode_layer(c["x"], c["P_q"], c["P_k"], c["P_v"], c["P_o"],
                                          c["kc"], c["vc"], lens, 1, 0.7)
    y2, K2, V2 = _mqa_layer_literal(c["x"], c["kc"][:, 0, :L - 1], c["vc"][:, 0, :L - 1],
                                    c["P_q"], c["P_k"][0], c["P_v"][0], c["P_o"], 0.7)
    assert np.max(np.abs(y - y2)) < TOL
    assert np.max(np.abs(kc[:, 0, :L] - K2)) < TOL
    assert np.max(np.abs(vc[:, 0, :L] - V2)) < TOL


@pytest.mark.parametrize("h,g", [(6, 2), (8, 4), (4, 1)])
def test_grouped_layer_is_mha_on_repeated_kv_heads(h, g):
    rng = np.random.default_rng(3000 + h * g)
    b, D, dk, dv, cap = 3, 14, 5, 4, 7
    c = _case(rng, b, D, h, g, dk, dv, cap)
    lens = np.array([1, 7, 4])
    r = h // g
    y, kc, vc, _, _ = oracle.decode_layer(c["x"], c["P_q"], c["P_k"], c["P_v"], c["P_o"],
                                          c["kc"], c["vc"], lens, g, 0.3)
    rep = lambda a: np.repeat(a, r, axis=0 if a.ndim == 3 else 1)
    y2, kc2, _, _, _ = oracle.decode_layer(c["x"], c["P_q"], rep(c["P_k"]), rep(c["P_v"]),
                                           c["P_o"], rep(c["kc"]), rep(c["vc"]), lens, h, 0.3)
    assert np.max(np.abs(y - y2)) < TOL
    assert np.max(np.abs(rep(kc) - kc2)) < TOL


def test_layer_bruteforce_loops():
    rng = np.random.default_rng(44)
    b, D, h, g, dk, dv, cap = 2, 5, 4, 2, 3, 2, 4
    c = _case(rng, b, D, h, g, dk, dv, cap)
    lens = np.array([2, 4])
    scale = 0.9
    y, kc, vc, _, _ = oracle.decode_layer(c["x"], c["P_q"], c["P_k"], c["P_v"], c["P_o"],
                                          c["kc"], c["vc"], lens, g, scale)
    r = h // g
    for i in range(b):
        x = c["x"][i]
        q = [[sum(x[d] * c["P_q"][a, d, k] for d in range(D)) for k in range(dk)]
             for a in range(h)]
        kn = [[sum(x[d] * c["P_k"][j, d, k] for d in range(D)) for k in range(dk)]
              for j in range(g)]
        vn = [[sum(x[d] * c["P_v"][j, d, v] for d in range(D)) for v in range(dv)]
              for j in range(g)]
        L = int(lens[i])
        o = []
        for a in range(h):
            j = a // r
            K = [list(c["kc"][i, j, p]) for p in range(L - 1)] + [kn[j]]
            V = [list(c["vc"][i, j, p]) for p in range(L - 1)] + [vn[j]]
            s = [scale * sum(q[a][k] * K[p][k] for k in range(dk)) for p in range(L)]
            m = max(s)
            e = [np.exp(t - m) for t in s]
            z = sum(e)
            o.append([sum(e[p] / z * V[p][v] for p in range(L)) for v in range(dv)])
        for d in range(D):
            want = sum(o[a][v] * c["P_o"][a, d, v] for a in range(h) for v in range(dv))
            assert abs(want - y[i, d]) < TOL
        for j in range(g):
            assert np.max(np.abs(np.array(kn[j]) - kc[i, j, L - 1])) < TOL


def test_bf16_rounding_matches_torch_on_float32_values():
    rng = np.random.default_rng(5)
    f = rng.standard_normal(20000).astype(np.float32) * np.float32(3.0)
    # exact ties: low 16 bits 0x8000, with even and odd bf16 mantissas
    ties = (rng.integers(0x3000, 0x4F00, 400).astype(np.uint32) << 16) | 0x8000
    f = np.concatenate([f, ties.view(np.float32), -ties.view(np.float32),
                        np.array([0.0, 1.0, -2.5, 65504.0], dtype=np.float32)])
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.to_storage(f.astype(np.float64), "bf16")
    assert np.array_equal(got, want)


def test_bf16_rounding_is_nearest_even_on_float64_values():
    rng = np.random.default_rng(6)
    a = rng.standard_normal(5000) * 10.0 ** rng.integers(-20, 20, 5000)
    bits = oracle.to_storage(a, "bf16")
    got = orc.bf16_bits_to_f64(bits)
    up = orc.bf16_bits_to_f64((bits.astype(np.int32) + 1).astype(np.uint16))
    dn = orc.bf16_bits_to_f64((bits.astype(np.int32) - 1).astype(np.uint16))
    err = np.abs(a - got)
    assert np.all(err <= np.abs(a - up)) and np.all(err <= np.abs(a - dn))
    tie = (err == np.abs(a - up)) | (err == np.abs(a - dn))
    assert np.all((bits[tie] & 1) == 0)


def test_storage_rounding_points_of_the_layer():
    """In bf16 storage, q and the new rows are the rounded float64
    projections, and y is the output projection of the rounded o."""
    rng = np.random.default_rng(7)
    b, D, h, g, dk, dv, cap = 2, 32, 4, 2, 8, 8, 6
    c = _case(rng, b, D, h, g, dk, dv, cap)
    enc = {k: oracle.to_storage(v, "bf16") for k, v in c.items()}
    lens = np.array([6, 3])
    y, kc, vc, q_s, o_s = oracle.decode_layer(enc["x"], enc["P_q"], enc["P_k"], enc["P_v"],
                                              enc["P_o"], enc["kc"], enc["vc"], lens, g, 0.5,
                                              dtype="bf16")
    q, kn, vn = oracle.project_qkv(enc["x"], enc["P_q"], enc["P_k"], enc["P_v"], "bf16")
    assert np.array_equal(q_s, oracle.to_storage(q, "bf16"))
    for i in range(b):
        assert np.array_equal(kc[i, :, lens[i] - 1], oracle.to_storage(kn[i], "bf16"))
        assert np.array_equal(vc[i, :, lens[i] - 1], oracle.to_storage(vn[i], "bf16"))
    assert np.max(np.abs(y - oracle.project_out(o_s, enc["P_o"], "bf16"))) == 0.0
    # and the bf16 layer stays close to the float64 layer on the same inputs
    wide = {k: orc.bf16_bits_to_f64(v) for k, v in enc.items()}
    y64, _, _, _, _ = oracle.decode_layer(wide["x"], wide["P_q"], wide["P_k"], wide["P_v"],
                                          wide["P_o"], wide["kc"], wide["vc"], lens, g, 0.5)
    assert np.max(np.abs(y - y64)) < 2e-2


def test_pins_catch_swapped_k_and_v_projections(monkeypatch):
    real = orc.project_qkv

    def swapped(x, P_q, P_k, P_v, dtype="f64"):
        q, k, v = real(x, P_q, P_v, P_k, dtype)
        return q, k, v
    monkeypatch.setattr(orc, "project_qkv", swapped)
    with pytest.raises(AssertionError):
        test_layer_at_g_equals_h_is_the_literal_mha_layer(2, 12, 3, 4, 4, 6)


def test_pins_catch_an_output_projection_over_the_wrong_axis(monkeypatch):
    monkeypatch.setattr(orc, "project_out",
                        lambda o, P_o, dtype="f64": np.einsum(
                            "bhv,hdv->bd", orc.widen(o, dtype)[:, ::-1], orc.widen(P_o, dtype)))
    with pytest.raises(AssertionError):
        test_layer_bruteforce_loops()


def test_f16_rounding_matches_torch_and_nearest_even():
    rng = np.random.default_rng(8)
    f = (rng.standard_normal(20000) * 10.0 ** rng.integers(-3, 4, 20000)).astype(np.float32)
    want = torch.from_numpy(f.copy()).to(torch.float16).numpy()
    got = oracle.to_storage(f.astype(np.float64), "f16")
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))
    # float64 values between float16 neighbours: nearest, ties to even
    a = rng.standard_normal(5000) * 3.0
    h = oracle.to_storage(a, "f16")
    bits = h.view(np.uint16).astype(np.int32)
    up = (bits + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    dn = (bits - 1).astype(np.uint16).view(np.float16).astype(np.float64)
    err = np.abs(a - h.astype(np.float64))
    assert np.all(err <= np.abs(a - up)) and np.all(err <= np.abs(a - dn))
    assert np.array_equal(oracle.widen(h, "f16"), h.astype(np.float64))
