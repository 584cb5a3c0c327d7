"""Pins for the float64 oracle against what the pages and the mathematics fix.

The pages print no attention output values, so the oracle's attention is
pinned by independent formulations and closed forms:
  * brute-force per-head loops of single-query dot-product attention
    ([논문 리뷰] Fast Transformer Decoding (velog), §2.1);
  * g = h against the multi-head incremental einsums (§2.4), g = 1 against
    the multi-query einsums (§3);
  * GQA against MHA run on KV heads repeated h/g times (GQA lesson
    "クエリヘッドはそのまま、キー・バリューヘッドだけ減らす", the lab section);
  * the incremental result against the last row of the batched causal form
    (§2.3), replayed over the decode trace of the decode notes
    "한 번 한 계산은 다시 하지 않기" (쉽게 보기 table);
  * closed forms (one row, zero query, equal keys, one dominant logit);
  * the counts the pages print (tests/golden/kv_counts.json).
The mutation tests at the end plant plausible mistakes in the oracle and check
that these pins catch them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TOL = 1e-12


def _rand_case(rng, b, h, g, cap, dk, dv, lens=None):
    q = rng.standard_normal((b, h, dk))
    k = rng.standard_normal((b, g, cap, dk))
    v = rng.standard_normal((b, g, cap, dv))
    if lens is None:
        lens = rng.integers(1, cap + 1, size=b)
    return q, k, v, np.asarray(lens, dtype=np.int64)


# --------------------------------------------------------------------------
# independent formulations, written here from the pages
# --------------------------------------------------------------------------
def _dot_product_attention_loops(q, K, V):
    """§2.1: logits = q.K_m, weights = softmax(logits), y = sum_m w_m V_m,
    in plain Python loops with math.exp."""
    m = len(K)
    logits = [sum(q[c] * K[p][c] for c in range(len(q))) for p in range(m)]
    top = max(logits)
    ex = [math.exp(s - top) for s in logits]
    tot = sum(ex)
    return [sum(ex[p] / tot * V[p][c] for p in range(m))
            for c in range(len(V[0]))]


def _softmax(x, axis=-1):
    e = np.exp(x - x.max(axis=axis, keepdims=True))
    return e / e.sum(axis=axis, keepdims=True)


def _mha_incremental(q, K, V, scale):
    """§2.4 with equal lengths: "bhk,bhmk->bhm", softmax, "bhm,bhmv->bhv"."""
    logits = np.einsum("bhk,bhmk->bhm", q, K) * scale
    return np.einsum("bhm,bhmv->bhv", _softmax(logits), V)


def _mqa_incremental(q, K, V, scale):
    """§3: "bhk,bmk->bhm", softmax, "bhm,bmv->bhv"."""
    logits = np.einsum("bhk,bmk->bhm", q, K) * scale
    return np.einsum("bhm,bmv->bhv", _softmax(logits), V)


def _batched_causal(Q, K, V, scale):
    """§2.3 with self-attention over n positions and an additive causal mask:
    "bhnk,bhmk->bhnm" + mask, softmax, "bhnm,bhmv->bhnv"."""
    n = Q.shape[2]
    mask = np.where(np.arange(n)[None, :] <= np.arange(n)[:, None], 0.0, -np.inf)
    logits = np.einsum("bhnk,bhmk->bhnm", Q, K) * scale + mask
    return np.einsum("bhnm,bhmv->bhnv", _softmax(logits), V)


# --------------------------------------------------------------------------
# widening
# --------------------------------------------------------------------------
def test_bf16_widening_closed_forms():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x8000, 0x7F80, 0x0001,
                     0x4049, 0x7F7F], dtype=np.uint16)
    want = [1.0, -2.0, 1.0 + 2.0 ** -7, 0.0, -0.0, math.inf, 2.0 ** -133,
            3.140625, (2 - 2 ** -7) * 2.0 ** 127]
    got = oracle.bf16_bits_to_f64(bits)
    assert list(got) == want
    assert math.copysign(1.0, got[4]) == -1.0


def test_f32_widening_is_exact():
    x = np.array([0.1, -3.3, 1e-30, 7.0], dtype=np.float32)
    assert np.array_equal(oracle.widen(x, "f32"), x.astype(np.float64))
    # every float32 is a bf16 pattern plus low bits: the top half widens to
    # the value of the truncated float32
    hi = (x.view(np.uint32) >> 16).astype(np.uint16)
    trunc = (x.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
    assert np.array_equal(oracle.widen(hi, "bf16"), trunc.astype(np.float64))


# --------------------------------------------------------------------------
# append
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_append_writes_exactly_one_row(dtype):
    rng = np.random.default_rng(0)
    b, g, cap, d = 3, 2, 9, 5
    if dtype is np.uint16:
        kc = rng.integers(0, 2 ** 16, size=(b, g, cap, d)).astype(np.uint16)
        vc = rng.integers(0, 2 ** 16, size=(b, g, cap, d)).astype(np.uint16)
        kn = rng.integers(0, 2 ** 16, size=(b, g, d)).astype(np.uint16)
        vn = rng.integers(0, 2 ** 16, size=(b, g, d)).astype(np.uint16)
    else:
        kc = rng.standard_normal((b, g, cap, d)).astype(np.float32)
        vc = rng.standard_normal((b, g, cap, d)).astype(np.float32)
        kn = rng.standard_normal((b, g, d)).astype(np.float32)
        vn = rng.standard_normal((b, g, d)).astype(np.float32)
    lens = np.array([1, 9, 4])
    k2, v2 = oracle.kv_append(kc, vc, kn, vn, lens)
    for i in range(b):
        for j in range(g):
            for p in range(cap):
                if p == lens[i] - 1:
                    assert k2[i, j, p].tobytes() == kn[i, j].tobytes()
                    assert v2[i, j, p].tobytes() == vn[i, j].tobytes()
                else:
                    assert k2[i, j, p].tobytes() == kc[i, j, p].tobytes()
                    assert v2[i, j, p].tobytes() == vc[i, j, p].tobytes()
    # inputs untouched
    assert not np.shares_memory(k2, kc)


def test_append_rejects_lengths_outside_cap():
    kc = np.zeros((1, 1, 4, 2))
    kn = np.zeros((1, 1, 2))
    for bad in (0, 5, -1):
        with pytest.raises(ValueError):
            oracle.kv_append(kc, kc, kn, kn, [bad])


def test_decode_trace_of_the_notes():
    """Prefill 16 positions, then three decode steps: the cache holds 16, 17,
    18, 19 tokens, past rows never change, and every step's output equals the
    matching row of the batched causal form."""
    trace = json.load(open(os.path.join(GOLDEN, "decode_trace.json")))["steps"]
    rng = np.random.default_rng(1)
    b, h, g, d, cap = 2, 4, 2, 6, 19
    n_total = trace[-1]["cache_tokens_after"]
    Kall = rng.standard_normal((b, g, n_total, d))
    Vall = rng.standard_normal((b, g, n_total, d))
    Qall = rng.standard_normal((b, h, n_total, d))
    scale = 0.4
    kc = np.full((b, g, cap, d), np.nan)
    vc = np.full((b, g, cap, d), np.nan)
    p0, p1 = trace[0]["positions"]
    kc[:, :, p0:p1 + 1] = Kall[:, :, p0:p1 + 1]
    vc[:, :, p0:p1 + 1] = Vall[:, :, p0:p1 + 1]
    filled = trace[0]["cache_tokens_after"]
    r = h // g
    causal = _batched_causal(Qall, np.repeat(Kall, r, axis=1),
                             np.repeat(Vall, r, axis=1), scale)
    for step in trace[1:]:
        pos = step["positions"][0]
        L = step["cache_tokens_after"]
        assert L == filled + 1 and pos == L - 1
        before_k = kc.copy()
        o, kc, vc = oracle.decode_step(Qall[:, :, pos], kc, vc, Kall[:, :, pos],
                                       Vall[:, :, pos], [L] * b, g, scale)
        assert np.array_equal(kc[:, :, :L - 1], before_k[:, :, :L - 1])
        assert np.isnan(kc[:, :, L:]).all()
        assert np.max(np.abs(o - causal[:, :, pos])) < TOL
        filled = L
    assert filled == n_total


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------
@pytest.mark.parametrize("b,h,g,cap,dk,dv", [
    (1, 1, 1, 1, 1, 1), (2, 6, 3, 7, 5, 4), (2, 4, 1, 6, 3, 3),
    (1, 6, 6, 5, 2, 5), (2, 6, 2, 7, 4, 2)])
def test_bruteforce_loops(b, h, g, cap, dk, dv):
    rng = np.random.default_rng(b * 100 + h * 10 + g)
    q, k, v, lens = _rand_case(rng, b, h, g, cap, dk, dv)
    scale = 0.7
    o = oracle.grouped_decode_attention(q, k, v, lens, g, scale)
    r = h // g
    for i in range(b):
        for a in range(h):
            j = a // r
            L = int(lens[i])
            want = _dot_product_attention_loops(
                [scale * x for x in q[i, a]], k[i, j, :L].tolist(),
                v[i, j, :L].tolist())
            assert np.max(np.abs(np.array(want) - o[i, a])) < TOL


def test_g_equals_h_is_mha():
    rng = np.random.default_rng(2)
    b, h, m, d = 2, 5, 11, 7
    q, k, v, _ = _rand_case(rng, b, h, h, m, d, d, lens=[m] * b)
    o = oracle.grouped_decode_attention(q, k, v, [m] * b, h, 0.3)
    assert np.max(np.abs(o - _mha_incremental(q, k, v, 0.3))) < TOL


def test_g_equals_1_is_mqa():
    rng = np.random.default_rng(3)
    b, h, m, d = 3, 6, 9, 4
    q, k, v, _ = _rand_case(rng, b, h, 1, m, d, d, lens=[m] * b)
    o = oracle.grouped_decode_attention(q, k, v, [m] * b, 1, 0.5)
    assert np.max(np.abs(o - _mqa_incremental(q, k[:, 0], v[:, 0], 0.5))) < TOL


@pytest.mark.parametrize("h,g", [(8, 2), (12, 3), (32, 8), (6, 1), (4, 4)])
def test_gqa_is_mha_on_repeated_heads(h, g):
    rng = np.random.default_rng(h * g)
    b, m, d = 2, 10, 8
    q, k, v, _ = _rand_case(rng, b, h, g, m, d, d, lens=[m] * b)
    o = oracle.grouped_decode_attention(q, k, v, [m] * b, g, 0.25)
    r = h // g
    want = _mha_incremental(q, np.repeat(k, r, axis=1), np.repeat(v, r, axis=1),
                            0.25)
    assert np.max(np.abs(o - want)) < TOL


def test_ragged_lengths_ignore_padding():
    rng = np.random.default_rng(4)
    b, h, g, cap, d = 3, 4, 2, 12, 5
    q, k, v, _ = _rand_case(rng, b, h, g, cap, d, d)
    lens = np.array([1, 7, 12])
    base = oracle.grouped_decode_attention(q, k, v, lens, g, 1.0)
    k2, v2 = k.copy(), v.copy()
    for i, L in enumerate(lens):
        k2[i, :, L:] = np.nan
        v2[i, :, L:] = 1e300
    assert np.array_equal(oracle.grouped_decode_attention(q, k2, v2, lens, g,
                                                          1.0), base)


def test_weights_sum_to_one_and_are_positive():
    rng = np.random.default_rng(5)
    q, k, _, lens = _rand_case(rng, 3, 8, 2, 20, 6, 6)
    for w in oracle.attention_weights(q, k, lens, 2, 3.0):
        assert np.all(w > 0)
        assert np.max(np.abs(w.sum(axis=-1) - 1.0)) < TOL


def test_single_row_returns_v_new_exactly():
    rng = np.random.default_rng(6)
    b, h, g, cap, d = 2, 4, 2, 5, 3
    q, k, v, _ = _rand_case(rng, b, h, g, cap, d, d)
    kn = rng.standard_normal((b, g, d))
    vn = rng.standard_normal((b, g, d))
    o, _, _ = oracle.decode_step(q, k, v, kn, vn, [1, 1], g, 0.9)
    r = h // g
    for a in range(h):
        assert np.array_equal(o[:, a], vn[:, a // r])


def test_zero_query_and_equal_keys_give_the_mean_of_v():
    rng = np.random.default_rng(7)
    b, h, g, cap, d = 2, 6, 3, 9, 4
    q, k, v, lens = _rand_case(rng, b, h, g, cap, d, d, lens=[9, 4])
    r = h // g
    o = oracle.grouped_decode_attention(np.zeros_like(q), k, v, lens, g, 1.0)
    for i in range(b):
        for a in range(h):
            mean = v[i, a // r, :lens[i]].mean(axis=0)
            assert np.max(np.abs(o[i, a] - mean)) < TOL
    k_eq = np.broadcast_to(k[:, :, :1], k.shape).copy()
    o2 = oracle.grouped_decode_attention(q, k_eq, v, lens, g, 1.0)
    assert np.max(np.abs(o2 - o)) < TOL


def test_dominant_logit_selects_its_row():
    rng = np.random.default_rng(8)
    b, h, g, cap, d = 1, 4, 1, 16, 8
    q, k, v, _ = _rand_case(rng, b, h, g, cap, d, d, lens=[cap])
    # least-norm u with q_a . u = 1 for every head; a row along u gets a
    # logit 1000 above the others for every head
    Q = q[0]
    u = Q.T @ np.linalg.solve(Q @ Q.T, np.ones(h))
    k[0, 0] *= 1e-3
    k[0, 0, 11] = 1000.0 * u
    o = oracle.grouped_decode_attention(q, k, v, [cap], g, 1.0)
    for a in range(h):
        assert np.max(np.abs(o[0, a] - v[0, 0, 11])) < TOL


def test_scale_multiplies_the_logits():
    rng = np.random.default_rng(9)
    q, k, v, lens = _rand_case(rng, 2, 4, 2, 8, 5, 5)
    a = oracle.grouped_decode_attention(q * 3.0, k, v, lens, 2, 0.5)
    bb = oracle.grouped_decode_attention(q, k, v, lens, 2, 1.5)
    assert np.max(np.abs(a - bb)) < TOL


def test_bf16_inputs_match_their_widened_values():
    rng = np.random.default_rng(10)
    q, k, v, lens = _rand_case(rng, 2, 4, 2, 8, 8, 8)
    to_bits = lambda x: (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    qb, kb, vb = to_bits(q), to_bits(k), to_bits(v)
    o = oracle.grouped_decode_attention(qb, kb, vb, lens, 2, 0.5, dtype="bf16")
    want = oracle.grouped_decode_attention(
        oracle.bf16_bits_to_f64(qb), oracle.bf16_bits_to_f64(kb),
        oracle.bf16_bits_to_f64(vb), lens, 2, 0.5)
    assert np.array_equal(o, want)


def test_divisibility_rule():
    q = np.zeros((1, 6, 2))
    k = np.zeros((1, 4, 3, 2))
    with pytest.raises(ValueError):
        oracle.grouped_decode_attention(q, k, k, [3], 4, 1.0)


# --------------------------------------------------------------------------
# counts printed by the pages
# --------------------------------------------------------------------------
def test_kv_cache_counts_against_the_pages():
    gold = json.load(open(os.path.join(GOLDEN, "kv_counts.json")))
    t = gold["llama3_70b_bytes_per_token"]
    x = t["inputs"]
    assert oracle.kv_cache_bytes_per_token(x["layers"], x["kv_heads"],
                                           x["head_dim"], x["bytes_per_elt"]) == t["value"]
    assert t["value"] == 320 * 1024
    t = gold["llama3_70b_bytes_8192_tokens"]
    x = t["inputs"]
    n = oracle.kv_cache_bytes(x["layers"], x["kv_heads"], x["tokens"],
                              x["head_dim"], x["bytes_per_elt"])
    assert n == t["value"] and n == t["gib"] * 2 ** 30
    t = gold["llama3_70b_mha_counterfactual_8192_tokens"]
    x = t["inputs"]
    n = oracle.kv_cache_bytes(x["layers"], x["kv_heads"], x["tokens"],
                              x["head_dim"], x["bytes_per_elt"])
    assert n == t["gib"] * 2 ** 30
    assert n == 8 * gold["llama3_70b_bytes_8192_tokens"]["value"]


@pytest.mark.parametrize("h", [8, 32, 64])
def test_mqa_cache_is_one_hth_of_mha(h):
    assert oracle.kv_cache_elements(3, h, 100, 64) == h * oracle.kv_cache_elements(3, 1, 100, 64)


def test_element_count_formula_against_arrays():
    layers, g, length, d = 3, 4, 17, 8
    arrays = [np.zeros((g, length, d)) for _ in range(2 * layers)]
    assert sum(a.size for a in arrays) == oracle.kv_cache_elements(layers, g, length, d)


def test_multiplications_do_not_depend_on_g():
    h, n, d, dm = 32, 4096, 128, 4096
    rows = [oracle.attention_multiplications(h, g, n, d, dm) for g in (32, 8, 4, 1)]
    assert len({r["scores"] for r in rows}) == 1
    assert len({r["weighted_sum"] for r in rows}) == 1
    assert rows[0]["scores"] == h * n * n * d
    assert [r["k_proj"] for r in rows] == [n * dm * g * d for g in (32, 8, 4, 1)]
    # the score count equals the multiplications of a brute-force count
    hh, nn, dd = 3, 4, 5
    cnt = sum(1 for _ in range(hh) for _ in range(nn) for _ in range(nn) for _ in range(dd))
    assert oracle.attention_multiplications(hh, 1, nn, dd, 7)["scores"] == cnt


# --------------------------------------------------------------------------
# planted mistakes: each must be caught by a pin above
# --------------------------------------------------------------------------
def _pins_pass():
    try:
        test_bruteforce_loops(2, 6, 2, 7, 4, 2)
        test_gqa_is_mha_on_repeated_heads(8, 2)
        test_g_equals_h_is_mha()
        test_g_equals_1_is_mqa()
        test_decode_trace_of_the_notes()
        test_single_row_returns_v_new_exactly()
        test_ragged_lengths_ignore_padding()
    except (AssertionError, ValueError, IndexError):
        return False
    return True


def test_pins_pass_on_the_oracle():
    assert _pins_pass()


def test_pins_catch_interleaved_grouping(monkeypatch):
    def wrong(q64, g):          # query head a -> KV head a % g
        b, h, dk = q64.shape
        return q64.reshape(b, h // g, g, dk).transpose(0, 2, 1, 3)
    monkeypatch.setattr(orc, "_group_view", wrong)
    assert not _pins_pass()


def test_pins_catch_a_dropped_scale(monkeypatch):
    real = orc.attention_weights
    monkeypatch.setattr(orc, "attention_weights",
                        lambda q, k, l, g, s: real(q, k, l, g, 1.0))
    assert not _pins_pass()


def test_pins_catch_an_off_by_one_length(monkeypatch):
    real = orc._check_lens
    monkeypatch.setattr(orc, "_check_lens",
                        lambda lens, b, cap: np.maximum(real(lens, b, cap) - 1, 1))
    assert not _pins_pass()


def test_pins_catch_a_transposed_value_operand(monkeypatch):
    real = orc.widen

    def wrong(x, dtype):
        a = real(x, dtype)
        if a.ndim == 4 and a.shape[-1] == a.shape[-2]:
            return a.swapaxes(-1, -2).copy()
        return a
    monkeypatch.setattr(orc, "widen", wrong)
    # square [cap, d] blocks make the transposition shape-preserving
    rng = np.random.default_rng(11)
    q, k, v, _ = _rand_case(rng, 1, 4, 2, 6, 6, 6, lens=[6])
    o = orc.grouped_decode_attention(q, k, v, [6], 2, 1.0)
    want = _mha_incremental(q, np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1), 1.0)
    assert np.max(np.abs(o - want)) > 1e-3


def test_pins_catch_appending_at_the_wrong_row(monkeypatch):
    def wrong(k_cache, v_cache, k_new, v_new, seq_lens):
        kc = np.array(k_cache, copy=True)
        vc = np.array(v_cache, copy=True)
        for i, L in enumerate(np.asarray(seq_lens).reshape(-1)):
            kc[i, :, min(int(L), kc.shape[2] - 1)] = k_new[i]
            vc[i, :, min(int(L), kc.shape[2] - 1)] = v_new[i]
        return kc, vc
    monkeypatch.setattr(orc, "kv_append", wrong)
    assert not _pins_pass()


# --------------------------------------------------------------------------
# n new tokens per step (causal): the batched masked form of §2.3
# --------------------------------------------------------------------------
@pytest.mark.parametrize("b,h,g,n,cap", [(2, 4, 2, 3, 9), (1, 6, 1, 4, 4), (2, 8, 8, 2, 11),
                                         (3, 6, 3, 1, 7)])
def test_multi_token_step_is_the_batched_causal_rows(b, h, g, n, cap):
    """Appending n tokens and attending causally equals the last n rows of
    the §2.3 batched form over the whole sequence with its causal mask."""
    rng = np.random.default_rng(100 + n * h)
    lens = rng.integers(n, cap + 1, size=b)
    r = h // g
    scale = 0.35
    kc = rng.standard_normal((b, g, cap, 5))
    vc = rng.standard_normal((b, g, cap, 4))
    kn = rng.standard_normal((b, n, g, 5))
    vn = rng.standard_normal((b, n, g, 4))
    q = rng.standard_normal((b, n, h, 5))
    o, k2, v2 = oracle.decode_step_multi(q, kc, vc, kn, vn, lens, g, scale)
    for i in range(b):
        L = int(lens[i])
        # the full sequence as the batched form sees it: old rows then new
        K = k2[i:i + 1, :, :L]
        V = v2[i:i + 1, :, :L]
        Q = np.zeros((1, h, L, 5))
        Q[0, :, L - n:] = q[i].transpose(1, 0, 2)
        full = _batched_causal(Q, np.repeat(K, r, axis=1), np.repeat(V, r, axis=1), scale)
        for s_ in range(n):
            assert np.max(np.abs(o[i, s_] - full[0, :, L - n + s_])) < TOL
        # the appended rows and nothing else changed
        for j in range(g):
            for p in range(cap):
                if L - n <= p < L:
                    assert np.array_equal(k2[i, j, p], kn[i, p - (L - n), j])
                else:
                    assert np.array_equal(k2[i, j, p], kc[i, j, p])


def test_multi_token_step_with_one_token_is_the_single_step():
    rng = np.random.default_rng(55)
    b, h, g, cap = 3, 8, 2, 10
    lens = np.array([1, 10, 6])
    kc = rng.standard_normal((b, g, cap, 6))
    vc = rng.standard_normal((b, g, cap, 6))
    kn = rng.standard_normal((b, 1, g, 6))
    vn = rng.standard_normal((b, 1, g, 6))
    q = rng.standard_normal((b, 1, h, 6))
    o1, k1, v1 = oracle.decode_step_multi(q, kc, vc, kn, vn, lens, g, 0.5)
    o2, k2, v2 = oracle.decode_step(q[:, 0], kc, vc, kn[:, 0], vn[:, 0], lens, g, 0.5)
    assert np.max(np.abs(o1[:, 0] - o2)) < TOL
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2)


def test_multi_token_bruteforce_loops():
    rng = np.random.default_rng(66)
    b, h, g, n, cap = 2, 4, 2, 3, 8
    lens = np.array([3, 8])
    q = rng.standard_normal((b, n, h, 3))
    k = rng.standard_normal((b, g, cap, 3))
    v = rng.standard_normal((b, g, cap, 2))
    o = oracle.grouped_decode_attention_multi(q, k, v, lens, g, 0.8)
    r = h // g
    for i in range(b):
        L = int(lens[i])
        for s_ in range(n):
            P = L - n + s_
            for a in range(h):
                j = a // r
                want = _dot_product_attention_loops(
                    [0.8 * x for x in q[i, s_, a]], k[i, j, :P + 1].tolist(),
                    v[i, j, :P + 1].tolist())
                assert np.max(np.abs(np.array(want) - o[i, s_, a])) < TOL


def test_multi_token_rejects_lengths_below_n():
    kc = np.zeros((1, 1, 5, 2))
    kn = np.zeros((1, 3, 1, 2))
    with pytest.raises(ValueError):
        oracle.kv_append_multi(kc, kc, kn, kn, [2])


# --------------------------------------------------------------------------
# paged KV cache: the block table is a relabelling of the contiguous cache
# --------------------------------------------------------------------------
def _paged_case(rng, b, g, d, bs, max_blocks, lens, spare=3):
    """A contiguous cache and the same data scattered over a shuffled pool."""
    nb = b * max_blocks + spare
    perm = rng.permutation(nb)
    table = perm[: b * max_blocks].reshape(b, max_blocks)
    kc = rng.standard_normal((b, g, max_blocks * bs, d))
    vc = rng.standard_normal((b, g, max_blocks * bs, d))
    kp = rng.standard_normal((nb, g, bs, d))        # unrelated data everywhere else
    vp = rng.standard_normal((nb, g, bs, d))
    for i in range(b):
        for m in range(max_blocks):
            kp[table[i, m]] = kc[i, :, m * bs:(m + 1) * bs]
            vp[table[i, m]] = vc[i, :, m * bs:(m + 1) * bs]
    return table, kc, vc, kp, vp


@pytest.mark.parametrize("bs,max_blocks,lens", [(4, 3, [1, 12, 5]), (2, 5, [10, 2, 7]),
                                                (8, 1, [8, 3, 1])])
def test_paged_step_equals_the_contiguous_step(bs, max_blocks, lens):
    rng = np.random.default_rng(900 + bs)
    b, h, g, d = 3, 4, 2, 5
    table, kc, vc, kp, vp = _paged_case(rng, b, g, d, bs, max_blocks, lens)
    q = rng.standard_normal((b, h, d))
    kn = rng.standard_normal((b, g, d))
    vn = rng.standard_normal((b, g, d))
    o1, kp2, vp2 = oracle.decode_step_paged(q, kp, vp, kn, vn, table, lens, g, 0.6, bs)
    o2, kc2, vc2 = oracle.decode_step(q, kc, vc, kn, vn, lens, g, 0.6)
    assert np.max(np.abs(o1 - o2)) < TOL
    # exactly one row changed per (i, j): the block and row the table names
    changed = np.argwhere(np.any(kp2 != kp, axis=-1))
    want = {(table[i, (L - 1) // bs], j, (L - 1) % bs) for i, L in enumerate(lens)
            for j in range(g)}
    assert {tuple(c) for c in changed} == want
    for i, L in enumerate(lens):
        blk, r = table[i, (L - 1) // bs], (L - 1) % bs
        assert np.array_equal(kp2[blk, :, r], kn[i]) and np.array_equal(vp2[blk, :, r], vn[i])
    assert np.array_equal(oracle.gather_paged(kp2, table, lens, bs)[:, :, :max(lens)],
                          np.where(np.arange(max(lens))[None, None, :, None] <
                                   np.array(lens)[:, None, None, None], kc2[:, :, :max(lens)], 0))


def test_paged_rows_bruteforce():
    table = np.array([[5, 2, 7], [0, 1, 3]])
    rows = oracle.paged_rows(table, 7, 0, 3)
    assert rows.tolist() == [[5, 0], [5, 1], [5, 2], [2, 0], [2, 1], [2, 2], [7, 0]]
    assert oracle.paged_rows(table, 1, 1, 3).tolist() == [[0, 0]]


def test_paged_rejects_bad_tables():
    kp = np.zeros((4, 1, 2, 3))
    with pytest.raises(ValueError):
        oracle.gather_paged(kp, np.array([[0, 9]]), [3], 2)      # block 9 outside the pool
    with pytest.raises(ValueError):
        oracle.gather_paged(kp, np.array([[0, 1]]), [5], 2)      # length beyond the table


@pytest.mark.parametrize("bs,n", [(4, 3), (2, 5), (8, 1)])
def test_paged_multi_step_equals_the_contiguous_multi_step(bs, n):
    rng = np.random.default_rng(950 + bs * n)
    b, h, g, d, max_blocks = 3, 4, 2, 5, 4
    lens = [n, bs * max_blocks, n + bs]
    table, kc, vc, kp, vp = _paged_case(rng, b, g, d, bs, max_blocks, lens)
    q = rng.standard_normal((b, n, h, d))
    kn = rng.standard_normal((b, n, g, d))
    vn = rng.standard_normal((b, n, g, d))
    o1, kp2, _ = oracle.decode_step_paged_multi(q, kp, vp, kn, vn, table, lens, g, 0.6, bs)
    o2, kc2, _ = oracle.decode_step_multi(q, kc, vc, kn, vn, lens, g, 0.6)
    assert np.max(np.abs(o1 - o2)) < TOL
    got = oracle.gather_paged(kp2, table, lens, bs)
    for i, L in enumerate(lens):
        assert np.array_equal(got[i, :, :L], kc2[i, :, :L])
