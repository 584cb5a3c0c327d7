"""Plain float64 CPU oracle for the grouped-KV incremental decode step.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code
with the CUDA path (no kernels, headers, helpers or constants) and imports
nothing from it; the two meet only through the seeded input generators.

What it computes is the plain definition, written out in float64 from inputs
that are widened exactly (fp32 -> f64 and bf16 -> f64 are both exact):

  1. append   K[i, j, L_i-1, :] = k_new[i, j, :],  V likewise
  2. logits   s[i, a, p] = scale * sum_c q[i, a, c] * K[i, a // r, p, c],  p < L_i
  3. softmax  w = exp(s - max_p s) / sum_p exp(s - max_p s)
  4. output   o[i, a, :] = sum_p w[i, a, p] * V[i, a // r, p, :]

with h query heads, g KV heads, r = h / g and L_i = seq_lens[i] the attended
length *after* the append.  No blocking, fusion or reordering beyond what the
definition states; numpy's einsum / matmul serve as the contraction steps.

Sources (page title, then section):
  [MQA review]  "[논문 리뷰] Fast Transformer Decoding: One Write-Head is All
                You Need" (velog): §2.1 Dot-Product Attention,
                §2.4 Multi-head Attention (Incremental), §3 Multi Query
                Attention.
  [GQA lesson]  "クエリヘッドはそのまま、キー・バリューヘッドだけ減らす"
                (ttlab, r-tf2-gqa): the g-knob table, the "what shrinks and
                what does not" counts, the grouping rule of the lab section.
  [Decode notes] "한 번 한 계산은 다시 하지 않기" (albangk, 05-faster-
                repetition): the per-layer decode pseudo code, "why only K and
                V are stored", and the per-token memory arithmetic.

Readings where the pages are silent or open:
  * scale: the pages' einsums carry no 1/sqrt(d); the caller passes ``scale``
    (scale = 1 reproduces the pages literally).
  * seq_lens[i] is the length after the append; rows >= L_i are padding.
  * query head a reads KV head a // r (contiguous groups, [GQA lesson] lab).
  * no mask in the incremental form: every cached row p < L_i is visible.
  * L_i outside [1, cap] is invalid; this oracle raises ValueError.

Parity of the attention values is pinned indirectly (the pages print no
attention outputs): see tests/test_oracle_pins.py.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_bits_to_f64",
    "widen",
    "kv_append",
    "grouped_decode_attention",
    "attention_weights",
    "decode_step",
    "kv_cache_elements",
    "kv_cache_bytes_per_token",
    "kv_cache_bytes",
    "attention_multiplications",
    "kv_append_multi",
    "grouped_decode_attention_multi",
    "decode_step_multi",
    "to_storage",
    "project_qkv",
    "project_out",
    "decode_layer",
    "paged_rows",
    "gather_paged",
    "kv_append_paged",
    "decode_step_paged",
    "kv_append_paged_multi",
    "decode_step_paged_multi",
]


# ---------------------------------------------------------------------------
# exact widening
# ---------------------------------------------------------------------------
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 values, given as their raw 16-bit patterns, to float64.

    A bfloat16 is the top half of an IEEE float32, so shifting the pattern
    into the high 16 bits of a 32-bit word gives the float32 with the same
    value; float32 -> float64 is exact.
    """
    b = np.asarray(bits)
    if b.dtype not in (np.uint16, np.int16):
        raise TypeError("bf16 input must be given as uint16/int16 bit patterns")
    w = b.astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return w.view(np.float32).astype(np.float64)


def widen(x, dtype: str) -> np.ndarray:
    """Return ``x`` as float64.  ``dtype`` is 'f32' (x holds float32 values),
    'f16' (float16 values) or 'bf16' (x holds uint16 bit patterns); every
    widening is exact."""
    if dtype == "bf16":
        return bf16_bits_to_f64(x)
    if dtype == "f16":
        a = np.asarray(x)
        if a.dtype != np.float16:
            raise TypeError("f16 input must be a float16 array")
        return a.astype(np.float64)
    if dtype == "f32":
        a = np.asarray(x)
        if a.dtype != np.float32:
            raise TypeError("f32 input must be a float32 array")
        return a.astype(np.float64)
    if dtype == "f64":
        return np.asarray(x, dtype=np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def _check_lens(seq_lens, b: int, cap: int) -> np.ndarray:
    lens = np.asarray(seq_lens, dtype=np.int64).reshape(-1)
    if lens.shape[0] != b:
        raise ValueError("seq_lens must hold one length per sequence")
    if np.any(lens < 1) or np.any(lens > cap):
        raise ValueError("every seq_len must lie in [1, cap]")
    return lens


# ---------------------------------------------------------------------------
# step 1: append ([MQA review] §2.4 / §3: concat on the position axis;
#         [Decode notes] pseudo code: kCache.push / vCache.push)
# ---------------------------------------------------------------------------
def kv_append(k_cache, v_cache, k_new, v_new, seq_lens):
    """Write the new token's K/V rows into the caches.

    k_cache [b, g, cap, d_k], v_cache [b, g, cap, d_v], k_new [b, g, d_k],
    v_new [b, g, d_v]; any numpy dtype (the copy is exact, bit for bit).
    Returns new arrays; row L_i-1 of every (i, j) is replaced and every other
    row is left as it was (past K/V never change under the causal mask,
    [Decode notes] "why only K and V are stored").
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    b, g, cap, _ = kc.shape
    lens = _check_lens(seq_lens, b, cap)
    for i in range(b):
        row = int(lens[i]) - 1
        for j in range(g):
            kc[i, j, row, :] = k_new[i, j, :]
            vc[i, j, row, :] = v_new[i, j, :]
    return kc, vc


# ---------------------------------------------------------------------------
# steps 2-4: logits, softmax, weighted sum over the grouped cache
# ---------------------------------------------------------------------------
def _group_view(q64: np.ndarray, g: int) -> np.ndarray:
    """[b, h, d_k] -> [b, g, r, d_k]: query head a = j * r + t belongs to KV
    head j (contiguous blocks of r = h / g heads, [GQA lesson] lab section;
    h must be divisible by g, [GQA lesson] g-knob table)."""
    b, h, dk = q64.shape
    if g < 1 or h % g != 0:
        raise ValueError("h must be divisible by g")
    return q64.reshape(b, g, h // g, dk)


def attention_weights(q64, k64, seq_lens, g: int, scale: float):
    """Softmax weights per sequence: list over i of arrays [g, r, L_i].

    q64 [b, h, d_k], k64 [b, g, cap, d_k], both float64, the cache already
    holding the appended row.  Logits follow "bhk,bhmk->bhm" ([MQA review]
    §2.4) with the KV head axis reduced to g, and "bhk,bmk->bhm" (§3) at g=1;
    softmax is tf.softmax over the position axis, written with the max
    subtracted (the same value in exact arithmetic).
    """
    b, g_, cap, _ = k64.shape
    if g_ != g:
        raise ValueError("k cache KV-head count differs from g")
    lens = _check_lens(seq_lens, b, cap)
    qg = _group_view(q64, g)
    out = []
    for i in range(b):
        L = int(lens[i])
        s = scale * np.einsum("jtc,jpc->jtp", qg[i], k64[i, :, :L, :])
        s = s - s.max(axis=-1, keepdims=True)
        e = np.exp(s)
        out.append(e / e.sum(axis=-1, keepdims=True))
    return out


def grouped_decode_attention(q, k_cache, v_cache, seq_lens, g: int,
                             scale: float, dtype: str = "f64") -> np.ndarray:
    """o [b, h, d_v] in float64 for the cache as given (append already done).

    q [b, h, d_k], k_cache [b, g, cap, d_k], v_cache [b, g, cap, d_v] in the
    encoding named by ``dtype`` (see ``widen``).  The weighted sum follows
    "bhm,bhmv->bhv" ([MQA review] §2.4) / "bhm,bmv->bhv" (§3).
    """
    q64 = widen(q, dtype)
    k64 = widen(k_cache, dtype)
    v64 = widen(v_cache, dtype)
    b, h, _ = q64.shape
    dv = v64.shape[-1]
    if v64.shape[:3] != k64.shape[:3]:
        raise ValueError("k and v caches disagree in [b, g, cap]")
    w = attention_weights(q64, k64, seq_lens, g, scale)
    lens = np.asarray(seq_lens, dtype=np.int64).reshape(-1)
    o = np.empty((b, g, h // g, dv), dtype=np.float64)
    for i in range(b):
        L = int(lens[i])
        o[i] = np.einsum("jtp,jpv->jtv", w[i], v64[i, :, :L, :])
    return o.reshape(b, h, dv)


def decode_step(q, k_cache, v_cache, k_new, v_new, seq_lens, g: int,
                scale: float, dtype: str = "f64"):
    """One decode step of one layer in the order of the [Decode notes] pseudo
    code: push the new K and V rows, then attend over the grown cache.

    Returns (o [b, h, d_v] float64, k_cache', v_cache') where the caches are
    new arrays in the input encoding.
    """
    kc, vc = kv_append(k_cache, v_cache, k_new, v_new, seq_lens)
    o = grouped_decode_attention(q, kc, vc, seq_lens, g, scale, dtype)
    return o, kc, vc


# ---------------------------------------------------------------------------
# n new tokens per step ([MQA review] §2.3: n queries per sequence in one
# step with an additive mask [b, h, n, m]; causal self-attention: the query
# at position P attends positions <= P)
# ---------------------------------------------------------------------------
def kv_append_multi(k_cache, v_cache, k_new, v_new, seq_lens):
    """Write n new K/V rows per (sequence, KV head): k_new [b, n, g, d_k],
    v_new [b, n, g, d_v]; row L_i - n + s of the cache receives token s.
    Bit-exact copies; every other row is left as it was."""
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    b, g, cap, _ = kc.shape
    n = np.asarray(k_new).shape[1]
    lens = _check_lens(seq_lens, b, cap)
    if np.any(lens < n):
        raise ValueError("every seq_len must be at least the number of new tokens")
    for i in range(b):
        for s_ in range(n):
            row = int(lens[i]) - n + s_
            for j in range(g):
                kc[i, j, row, :] = k_new[i, s_, j, :]
                vc[i, j, row, :] = v_new[i, s_, j, :]
    return kc, vc


def grouped_decode_attention_multi(q, k_cache, v_cache, seq_lens, g: int,
                                   scale: float, dtype: str = "f64") -> np.ndarray:
    """o [b, n, h, d_v] for n queries per sequence at positions
    L_i - n + s (s = 0..n-1), each attending the cached positions p <= its
    own (the additive causal mask of [MQA review] §2.3: 0 where p <= P,
    -inf elsewhere), heads grouped as in grouped_decode_attention."""
    q64 = widen(q, dtype)
    k64 = widen(k_cache, dtype)
    v64 = widen(v_cache, dtype)
    b, n, h, dk = q64.shape
    dv = v64.shape[-1]
    cap = k64.shape[2]
    lens = _check_lens(seq_lens, b, cap)
    if np.any(lens < n):
        raise ValueError("every seq_len must be at least the number of queries")
    r = h // g
    o = np.empty((b, n, h, dv), dtype=np.float64)
    for i in range(b):
        L = int(lens[i])
        qg = q64[i].reshape(n, g, r, dk)                       # [n, g, r, dk]
        s = scale * np.einsum("sjtc,jpc->sjtp", qg, k64[i, :, :L, :])
        pos = np.arange(L)[None, :]
        own = (L - n + np.arange(n))[:, None]
        mask = np.where(pos <= own, 0.0, -np.inf)              # [n, L]
        s = s + mask[:, None, None, :]
        s = s - s.max(axis=-1, keepdims=True)
        e = np.exp(s)
        w = e / e.sum(axis=-1, keepdims=True)
        o[i] = np.einsum("sjtp,jpv->sjtv", w, v64[i, :, :L, :]).reshape(n, h, dv)
    return o


def decode_step_multi(q, k_cache, v_cache, k_new, v_new, seq_lens, g: int,
                      scale: float, dtype: str = "f64"):
    """Append the n new rows, then attend causally (one step, n tokens)."""
    kc, vc = kv_append_multi(k_cache, v_cache, k_new, v_new, seq_lens)
    o = grouped_decode_attention_multi(q, kc, vc, seq_lens, g, scale, dtype)
    return o, kc, vc


# ---------------------------------------------------------------------------
# the layer around the step ([MQA review] §2.4 MultiheadSelfAttentionIncremental
# and §3 MultiquerySelfAttentionIncremental): projections of x into q and the
# new K/V rows, the step, and the output projection
# ---------------------------------------------------------------------------
def to_storage(a64, dtype: str):
    """Round float64 values to the storage encoding named by ``dtype``:
    'bf16' -> uint16 bit patterns of the round-to-nearest-even bfloat16,
    'f32' -> float32 and 'f16' -> float16 (numpy's conversions round to
    nearest even), 'f64' -> unchanged.  The bf16 rounding keeps 8 significant bits of the float64
    value directly (no intermediate float32); it is exact for magnitudes in
    the normal bfloat16 range [2^-126, 2^128) and for 0."""
    a = np.asarray(a64, dtype=np.float64)
    if dtype == "f64":
        return a.copy()
    if dtype == "f32":
        return a.astype(np.float32)
    if dtype == "f16":
        return a.astype(np.float16)
    if dtype != "bf16":
        raise ValueError(f"unknown dtype {dtype!r}")
    m, e = np.frexp(a)                       # a = m * 2^e, 0.5 <= |m| < 1
    r = np.round(np.ldexp(m, 8))             # 8 significant bits, ties to even
    v = np.ldexp(r, e - 8).astype(np.float32)   # exact: 8 bits fit a float32
    return (v.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def project_qkv(x, P_q, P_k, P_v, dtype: str = "f64"):
    """q = "bd,hdk->bhk"(x, P_q), k_new = "bd,gdk->bgk"(x, P_k), v_new =
    "bd,gdv->bgv"(x, P_v) in float64 ([MQA review] §2.4, with the KV-head
    axis of P_k / P_v reduced to g as §3 reduces it to one: P_q [h, D, d_k],
    P_k [g, D, d_k], P_v [g, D, d_v], x [b, D] in the ``dtype`` encoding)."""
    x64 = widen(x, dtype)
    q = np.einsum("bd,hdk->bhk", x64, widen(P_q, dtype))
    kn = np.einsum("bd,gdk->bgk", x64, widen(P_k, dtype))
    vn = np.einsum("bd,gdv->bgv", x64, widen(P_v, dtype))
    return q, kn, vn


def project_out(o, P_o, dtype: str = "f64"):
    """y = "bhv,hdv->bd"(o, P_o) in float64 ([MQA review] §2.4 / §3):
    o [b, h, d_v], P_o [h, D, d_v]."""
    return np.einsum("bhv,hdv->bd", widen(o, dtype), widen(P_o, dtype))


def decode_layer(x, P_q, P_k, P_v, P_o, k_cache, v_cache, seq_lens, g: int,
                 scale: float, dtype: str = "f64"):
    """One incremental layer: project x, append the new K/V rows, attend,
    project the output ([MQA review] §2.4 / §3, grouped KV heads).

    The tensors the layer stores (q, the new K/V rows, o) are held in the
    storage encoding ``dtype``: each is computed in float64 and rounded once
    to it (``to_storage``) before the next step reads it; y is returned in
    float64.  Returns (y [b, D], k_cache', v_cache', q, o) with the caches,
    q and o in the storage encoding.
    """
    q, kn, vn = project_qkv(x, P_q, P_k, P_v, dtype)
    q_s, kn_s, vn_s = (to_storage(t, dtype) for t in (q, kn, vn))
    o, kc, vc = decode_step(q_s, k_cache, v_cache, kn_s, vn_s, seq_lens, g, scale, dtype)
    o_s = to_storage(o, dtype)
    y = project_out(o_s, P_o, dtype)
    return y, kc, vc, q_s, o_s


# ---------------------------------------------------------------------------
# paged KV cache ([Decode notes] memory section: serving engines keep the KV
# cache in GPU memory, the vLLM PagedAttention paper it cites; the block
# table is that paper's mapping): the cache of every layer is a pool of
# fixed-size blocks, pool [num_blocks, g, B, d]; logical position p of
# sequence i lives in row p mod B of block block_table[i, p div B].
# ---------------------------------------------------------------------------
def paged_rows(block_table, seq_len_i: int, i: int, block_size: int) -> np.ndarray:
    """Physical (block, row-in-block) of the positions 0 .. L_i - 1 of
    sequence i, as an int array [L_i, 2]."""
    p = np.arange(int(seq_len_i))
    blocks = np.asarray(block_table)[i, p // block_size]
    return np.stack([blocks, p % block_size], axis=1)


def _check_paged(pool, block_table, seq_lens, block_size):
    nb, g, bs, _ = np.asarray(pool).shape
    if bs != block_size:
        raise ValueError("pool rows per block differ from block_size")
    bt = np.asarray(block_table)
    b, max_blocks = bt.shape
    lens = _check_lens(seq_lens, b, max_blocks * block_size)
    for i in range(b):
        used = bt[i, : (int(lens[i]) + block_size - 1) // block_size]
        if np.any(used < 0) or np.any(used >= nb):
            raise ValueError("block table entry outside the pool")
    return lens


def gather_paged(pool, block_table, seq_lens, block_size: int):
    """The contiguous cache [b, g, max_blocks * B, d] that the pool and the
    table describe; rows at or beyond L_i are zero."""
    pool = np.asarray(pool)
    lens = _check_paged(pool, block_table, seq_lens, block_size)
    b, max_blocks = np.asarray(block_table).shape
    nb, g, bs, d = pool.shape
    out = np.zeros((b, g, max_blocks * block_size, d), dtype=pool.dtype)
    for i in range(b):
        rows = paged_rows(block_table, lens[i], i, block_size)
        for p, (blk, r) in enumerate(rows):
            out[i, :, p, :] = pool[blk, :, r, :]
    return out


def kv_append_paged(k_pool, v_pool, k_new, v_new, block_table, seq_lens, block_size: int):
    """Write the new token's rows at position L_i - 1 of every (i, j): row
    (L_i - 1) mod B of block block_table[i, (L_i - 1) div B].  Bit-exact;
    every other pool row is left as it was."""
    kp = np.array(k_pool, copy=True)
    vp = np.array(v_pool, copy=True)
    lens = _check_paged(kp, block_table, seq_lens, block_size)
    bt = np.asarray(block_table)
    for i in range(bt.shape[0]):
        p = int(lens[i]) - 1
        blk, r = bt[i, p // block_size], p % block_size
        for j in range(kp.shape[1]):
            kp[blk, j, r, :] = k_new[i, j, :]
            vp[blk, j, r, :] = v_new[i, j, :]
    return kp, vp


def kv_append_paged_multi(k_pool, v_pool, k_new, v_new, block_table, seq_lens,
                          block_size: int):
    """n new rows per (sequence, KV head): token s goes to position
    L_i - n + s, i.e. row (L_i - n + s) mod B of block
    block_table[i, (L_i - n + s) div B]; k_new / v_new [b, n, g, d]."""
    kp = np.array(k_pool, copy=True)
    vp = np.array(v_pool, copy=True)
    lens = _check_paged(kp, block_table, seq_lens, block_size)
    bt = np.asarray(block_table)
    n = np.asarray(k_new).shape[1]
    if np.any(lens < n):
        raise ValueError("every seq_len must be at least the number of new tokens")
    for i in range(bt.shape[0]):
        for s_ in range(n):
            p = int(lens[i]) - n + s_
            blk, r = bt[i, p // block_size], p % block_size
            for j in range(kp.shape[1]):
                kp[blk, j, r, :] = k_new[i, s_, j, :]
                vp[blk, j, r, :] = v_new[i, s_, j, :]
    return kp, vp


def decode_step_paged_multi(q, k_pool, v_pool, k_new, v_new, block_table, seq_lens, g: int,
                            scale: float, block_size: int, dtype: str = "f64"):
    """The n-token causal step (decode_step_multi) on a paged cache."""
    kp, vp = kv_append_paged_multi(k_pool, v_pool, k_new, v_new, block_table, seq_lens,
                                   block_size)
    kc = gather_paged(kp, block_table, seq_lens, block_size)
    vc = gather_paged(vp, block_table, seq_lens, block_size)
    o = grouped_decode_attention_multi(q, kc, vc, seq_lens, g, scale, dtype)
    return o, kp, vp


def decode_step_paged(q, k_pool, v_pool, k_new, v_new, block_table, seq_lens, g: int,
                      scale: float, block_size: int, dtype: str = "f64"):
    """One decode step on a paged cache: append, then attend over the
    positions the table maps (the same arithmetic as decode_step on the
    gathered cache).  Returns (o, k_pool', v_pool')."""
    kp, vp = kv_append_paged(k_pool, v_pool, k_new, v_new, block_table, seq_lens, block_size)
    kc = gather_paged(kp, block_table, seq_lens, block_size)
    vc = gather_paged(vp, block_table, seq_lens, block_size)
    o = grouped_decode_attention(q, kc, vc, seq_lens, g, scale, dtype)
    return o, kp, vp


# ---------------------------------------------------------------------------
# counts ([GQA lesson] "what shrinks" section; [Decode notes] memory section;
#         [MQA review] §3 shape change)
# ---------------------------------------------------------------------------
def kv_cache_elements(layers: int, kv_heads: int, length: int,
                      head_dim: int) -> int:
    """Reals held in the KV cache: 2 (K and V) x layers x KV heads x length x
    head dim.  The query-head count does not appear ([GQA lesson])."""
    return 2 * layers * kv_heads * length * head_dim


def kv_cache_bytes_per_token(layers: int, kv_heads: int, head_dim: int,
                             bytes_per_elt: int = 2) -> int:
    """Bytes one token leaves in the cache: 2 x layers x KV heads x head dim x
    element bytes ([Decode notes] memory section, 2 bytes for fp16/bf16)."""
    return kv_cache_elements(layers, kv_heads, 1, head_dim) * bytes_per_elt


def kv_cache_bytes(layers: int, kv_heads: int, tokens: int, head_dim: int,
                   bytes_per_elt: int = 2) -> int:
    """Cache bytes of one request holding ``tokens`` positions."""
    return kv_cache_elements(layers, kv_heads, tokens, head_dim) * bytes_per_elt


def attention_multiplications(h: int, g: int, n: int, d: int,
                              d_model: int) -> dict:
    """Multiplications of one pass of one layer over n positions, by term,
    as counted in [GQA lesson] "what shrinks": the score and weighted-sum
    terms are h*n*n*d each and carry no g; the K and V projections are
    n*d_model*(g*d) each."""
    if h % g != 0:
        raise ValueError("h must be divisible by g")
    return {
        "scores": h * n * n * d,
        "weighted_sum": h * n * n * d,
        "k_proj": n * d_model * (g * d),
        "v_proj": n * d_model * (g * d),
    }
