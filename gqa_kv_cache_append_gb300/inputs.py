"""Seeded synthetic decode-step inputs shaped like the pages' workloads.

This module only draws and lays out data; it holds none of the decode
arithmetic (no logits, softmax or weighted sums).  The tests feed the same
tensors to the CUDA path and to the float64 oracle, and the bench times the
CUDA path on them.

Recipe (per layer l of a workload with seed s):
  * a torch.Generator on the target device, seeded with s * 1000 + l, draws
    in this order: the K cache, the V cache, q, k_new, v_new, each N(0, 1)
    in float32 and then rounded to the storage dtype (bf16 or fp16 round-to-
    nearest-even, or kept as fp32);
  * 'meanpool' workloads first draw an h-head (MHA) K/V cache, k_new and
    v_new, then average every contiguous block of h/g heads in float32 before
    the rounding (the MHA -> GQA conversion by group mean, from the GQA
    lesson "クエリヘッドはそのまま、キー・バリューヘッドだけ減らす", section
    on merging groups); g = h leaves the MHA data untouched;
  * 'boost' workloads pick round(0.01 * L_i) positions per sequence without
    replacement (torch.randperm on a CPU generator seeded s * 1000 + l + 7)
    and add (boost / scale) * u to their K rows before rounding, where u is
    the least-norm solution of Q_i u = 1 for the sequence's bf16-rounded
    query block Q_i [h, d]; every head's logit at those rows then rises by
    about ``boost`` (exactly, before the bf16 rounding of K);
  * ragged workloads take lengths numpy.random.default_rng(s).integers(lo,
    hi, size=b, endpoint=True); the others use L_i = cap for every sequence.
Rows at or beyond L_i are padding; ``pad_fill`` can fill them with NaN (or a
large value) to check that nothing reads them into the result.

Steps with n new tokens per sequence (make_layer_multi, 'plain' workloads
only) draw in the same order from a generator seeded s * 1000 + l + 100000 * n:
the K cache, the V cache, q [b, n, h, d], k_new [b, n, g, d], v_new
[b, n, g, d].

The projections of a whole layer (make_layer_weights) come from a generator
seeded s * 1000 + l + 500000: P_q [h, D, d], P_k [g, D, d], P_v [g, D, d],
each N(0, 1/D); P_o [h, D, d], N(0, 1/(h d)); then x [b, D], N(0, 1); all
rounded to the storage dtype.  D is the model width of the workload (the
pages' d), so q, the new rows and y stay of order one.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

__all__ = ["DecodeConfig", "WORKLOADS", "workload", "seq_lens_for",
           "make_layer", "make_layer_multi", "make_layer_weights", "to_paged", "layer_bytes",
           "layer_flops", "projection_bytes", "bench_layers"]


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    name: str
    layers: int
    b: int
    h: int
    g: int
    d: int
    cap: int
    dtype: str                 # 'bf16', 'f16' or 'f32'
    scale: float
    seed: int
    kind: str = "plain"        # 'plain' | 'meanpool' | 'boost'
    ragged: Optional[tuple] = None   # (lo, hi) inclusive, or None = full
    boost: float = 8.0
    boost_frac: float = 0.01
    d_model: int = 0           # model width D; 0 means h * d
    d_v: int = 0               # head dim of V and out; 0 means d (d is d_k)

    @property
    def r(self) -> int:
        return self.h // self.g

    @property
    def dv(self) -> int:
        return self.d_v if self.d_v else self.d

    @property
    def D(self) -> int:
        return self.d_model if self.d_model else self.h * self.d

    @property
    def elt(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def torch_dtype(self):
        return {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[self.dtype]


_S128 = 1.0 / math.sqrt(128.0)

# The five workloads, with the sizes the pages' models give.
WORKLOADS = {
    # single-layer MQA step in fp32 (255 cached rows + 1 appended)
    "mqa_f32_b1_h8_d64_m256": DecodeConfig(
        "mqa_f32_b1_h8_d64_m256", 1, 1, 8, 1, 64, 256, "f32", 1.0 / 8.0, 1),
    # g-knob sweep, mean-pooled from one MHA cache (g set per run)
    "gqa_sweep_b16_h32_d128_m4096": DecodeConfig(
        "gqa_sweep_b16_h32_d128_m4096", 1, 16, 32, 8, 128, 4096, "bf16",
        _S128, 2, kind="meanpool"),
    # Llama-3-70B-shaped step: 80 layers, 64 query / 8 KV heads, width 8192
    "llama3_70b_b32_m8192": DecodeConfig(
        "llama3_70b_b32_m8192", 80, 32, 64, 8, 128, 8192, "bf16", _S128, 3,
        d_model=8192),
    # Qwen2.5-7B-shaped ragged batch: 28 layers, 28 query / 4 KV heads,
    # width 3584
    "qwen25_7b_b64_ragged": DecodeConfig(
        "qwen25_7b_b64_ragged", 28, 64, 28, 4, 128, 32768, "bf16", _S128, 4,
        ragged=(512, 32768), d_model=3584),
    # long-context MQA with a peaked softmax
    "long_mqa_b8_m131072": DecodeConfig(
        "long_mqa_b8_m131072", 1, 8, 32, 1, 128, 131072, "bf16", _S128, 5,
        kind="boost"),
}


def workload(name: str, **overrides) -> DecodeConfig:
    """The named workload, optionally with fields replaced (e.g. g for the
    sweep, or smaller b / cap / layers for quick parity runs)."""
    return dataclasses.replace(WORKLOADS[name], **overrides)


def seq_lens_for(cfg: DecodeConfig) -> np.ndarray:
    """Post-append lengths L_i (int32 [b])."""
    if cfg.ragged is None:
        return np.full(cfg.b, cfg.cap, dtype=np.int32)
    lo, hi = cfg.ragged
    lens = np.random.default_rng(cfg.seed).integers(lo, hi, size=cfg.b,
                                                    endpoint=True)
    return np.minimum(lens, cfg.cap).astype(np.int32)


def layer_bytes(cfg: DecodeConfig, lens: np.ndarray, n: int = 1) -> int:
    """Algorithmic bytes of one decode-attention call: the K and V rows below
    L_i of every KV head, plus q and out of the n new tokens (padding and
    split partials are not counted)."""
    kv = int(np.sum(lens, dtype=np.int64)) * cfg.g * (cfg.d + cfg.dv) * cfg.elt
    return kv + cfg.b * n * cfg.h * (cfg.d + cfg.dv) * cfg.elt


def bench_layers(cfg: DecodeConfig, lens: np.ndarray, l2_bytes: int, n: int = 1,
                 extra_per_layer: int = 0) -> int:
    """Layers a timed step rotates through: the workload's own, or, when all
    of them together fit four times over in an L2 of ``l2_bytes``, enough
    independent replicas of the layer (same shapes, the next layer seeds)
    that one step streams at least 4 x L2, so every step reads its K/V from
    HBM.  ``extra_per_layer``: bytes a layer reads besides the attention
    call's (e.g. projection weights)."""
    per_layer = layer_bytes(cfg, lens, n) + extra_per_layer
    if cfg.layers * per_layer >= 4 * l2_bytes:
        return cfg.layers
    return -(-4 * l2_bytes // per_layer)


def layer_flops(cfg: DecodeConfig, lens: np.ndarray, n: int = 1) -> int:
    """Multiply-add flops of one decode-attention call (2 per product, for
    q.K over d_k and for w.V over d_v); with n new tokens the causal mask
    leaves token s the positions below L_i - n + s + 1."""
    lens = np.asarray(lens, dtype=np.int64)
    seen = int(np.sum(lens)) * n - cfg.b * (n * (n - 1) // 2)
    return 2 * cfg.h * (cfg.d + cfg.dv) * seen


def _randn(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def _pool(x: torch.Tensor, g: int) -> torch.Tensor:
    """Average contiguous blocks of h/g heads on dim 1 (float32)."""
    b, h = x.shape[:2]
    if g == h:
        return x
    return x.reshape(b, g, h // g, *x.shape[2:]).mean(dim=2)


def make_layer(cfg: DecodeConfig, layer: int = 0, device="cpu",
               lens: Optional[np.ndarray] = None, pad_fill=None) -> dict:
    """Inputs of one layer: q [b,h,d], k_cache [b,g,cap,d], v_cache
    [b,g,cap,d_v], k_new [b,g,d], v_new [b,g,d_v] in the storage dtype,
    seq_lens int32 [b] on ``device``, plus the host copy ``lens``."""
    if cfg.h % cfg.g != 0:
        raise ValueError("h must be divisible by g")
    device = torch.device(device)
    if lens is None:
        lens = seq_lens_for(cfg)
    lens = np.asarray(lens, dtype=np.int32)
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed * 1000 + layer)
    b, h, g, d, cap = cfg.b, cfg.h, cfg.g, cfg.d, cfg.cap
    dv = cfg.dv
    dt = cfg.torch_dtype

    if cfg.kind == "meanpool":
        if dv != d:
            raise ValueError("the mean-pooled workload has one head dim")
        k_cache = _pool(_randn((b, h, cap, d), gen, device), g).to(dt)
        v_cache = _pool(_randn((b, h, cap, d), gen, device), g).to(dt)
        q = _randn((b, h, d), gen, device).to(dt)
        k_new = _pool(_randn((b, h, d), gen, device), g).to(dt)
        v_new = _pool(_randn((b, h, d), gen, device), g).to(dt)
    elif cfg.kind in ("plain", "boost"):
        if cfg.kind == "plain" and dt != torch.float32:
            # draw and round block by block to bound the float32 temporary
            k_cache = torch.empty((b, g, cap, d), dtype=dt, device=device)
            v_cache = torch.empty((b, g, cap, dv), dtype=dt, device=device)
            for dst in (k_cache, v_cache):
                for i in range(b):
                    dst[i].copy_(_randn((g, cap, dst.shape[-1]), gen, device))
        else:
            k_cache = _randn((b, g, cap, d), gen, device)
            v_cache = _randn((b, g, cap, dv), gen, device)
        q = _randn((b, h, d), gen, device).to(dt)
        k_new = _randn((b, g, d), gen, device)
        v_new = _randn((b, g, dv), gen, device).to(dt)
        if cfg.kind == "boost":
            if g != 1:
                raise ValueError("the boosted workload is MQA (g = 1)")
            k_cache, k_new = _boost(cfg, layer, q, k_cache, k_new, lens)
        k_cache = k_cache.to(dt)
        v_cache = v_cache.to(dt)
        k_new = k_new.to(dt)
    else:
        raise ValueError(f"unknown workload kind {cfg.kind!r}")

    if pad_fill is not None:
        for i in range(b):
            L = int(lens[i])
            if L < cap:
                k_cache[i, :, L:, :] = pad_fill
                v_cache[i, :, L:, :] = pad_fill

    return {
        "q": q.contiguous(), "k_cache": k_cache.contiguous(),
        "v_cache": v_cache.contiguous(), "k_new": k_new.contiguous(),
        "v_new": v_new.contiguous(),
        "seq_lens": torch.from_numpy(lens.copy()).to(device),
        "lens": lens,
    }


def make_layer_multi(cfg: DecodeConfig, n: int, layer: int = 0, device="cpu",
                     lens: Optional[np.ndarray] = None, pad_fill=None) -> dict:
    """Inputs of one layer's step with n new tokens per sequence: q
    [b, n, h, d], k_cache [b, g, cap, d], v_cache [b, g, cap, d_v], k_new
    [b, n, g, d], v_new [b, n, g, d_v] in the storage dtype, seq_lens int32
    [b] (post-append, >= n) on ``device``, plus the host copy ``lens``.
    'plain' workloads only."""
    if cfg.kind != "plain":
        raise ValueError("multi-token inputs are drawn for plain workloads only")
    if cfg.h % cfg.g != 0 or n < 1:
        raise ValueError("h must be divisible by g and n >= 1")
    device = torch.device(device)
    if lens is None:
        lens = seq_lens_for(cfg)
    lens = np.asarray(lens, dtype=np.int32)
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed * 1000 + layer + 100000 * n)
    b, h, g, d, cap = cfg.b, cfg.h, cfg.g, cfg.d, cfg.cap
    dv = cfg.dv
    dt = cfg.torch_dtype
    k_cache = torch.empty((b, g, cap, d), dtype=dt, device=device)
    v_cache = torch.empty((b, g, cap, dv), dtype=dt, device=device)
    for dst in (k_cache, v_cache):
        for i in range(b):
            dst[i].copy_(_randn((g, cap, dst.shape[-1]), gen, device))
    q = _randn((b, n, h, d), gen, device).to(dt)
    k_new = _randn((b, n, g, d), gen, device).to(dt)
    v_new = _randn((b, n, g, dv), gen, device).to(dt)
    if pad_fill is not None:
        for i in range(b):
            L = int(lens[i])
            if L < cap:
                k_cache[i, :, L:, :] = pad_fill
                v_cache[i, :, L:, :] = pad_fill
    return {
        "q": q.contiguous(), "k_cache": k_cache, "v_cache": v_cache,
        "k_new": k_new.contiguous(), "v_new": v_new.contiguous(),
        "seq_lens": torch.from_numpy(lens.copy()).to(device),
        "lens": lens,
    }


def make_layer_weights(cfg: DecodeConfig, layer: int = 0, device="cpu") -> dict:
    """Projection weights of one layer in the pages' layouts and the layer
    input: P_q [h, D, d], P_k [g, D, d], P_v [g, D, d], P_o [h, D, d],
    x [b, D], in the storage dtype on ``device``."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed * 1000 + layer + 500000)
    b, h, g, d, D = cfg.b, cfg.h, cfg.g, cfg.d, cfg.D
    dt = cfg.torch_dtype
    out = {}
    for name, shape, std in (("P_q", (h, D, d), D ** -0.5), ("P_k", (g, D, d), D ** -0.5),
                             ("P_v", (g, D, d), D ** -0.5), ("P_o", (h, D, d), (h * d) ** -0.5)):
        w = torch.empty(shape, dtype=dt, device=device)
        for a in range(shape[0]):
            w[a].copy_(_randn(shape[1:], gen, device) * std)
        out[name] = w
    out["x"] = _randn((b, D), gen, device).to(dt)
    return out


def to_paged(k_cache: torch.Tensor, v_cache: torch.Tensor, block_size: int, seed: int,
             spare: int = 3, fill=None):
    """Lay a contiguous cache [b, g, cap, d] (V: [b, g, cap, d_v]) out as a
    paged one: pools [num_blocks, g, block_size, d] with num_blocks =
    b * cap / block_size + spare, and a block table [b, cap / block_size]
    int32 that maps the blocks
    of every sequence to a seeded random permutation of the pool
    (torch.randperm on a CPU generator seeded ``seed``).  Unused blocks hold
    ``fill`` (default zeros).  A pure relabelling: no arithmetic."""
    b, g, cap, _ = k_cache.shape
    if cap % block_size:
        raise ValueError("cap must be a multiple of block_size")
    mb = cap // block_size
    nb = b * mb + spare
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    perm = torch.randperm(nb, generator=gen)
    table = perm[: b * mb].reshape(b, mb).to(torch.int32)
    pools = []
    for cache in (k_cache, v_cache):
        d = cache.shape[-1]
        pool = torch.zeros((nb, g, block_size, d), dtype=cache.dtype, device=cache.device)
        if fill is not None:
            pool.fill_(fill)
        blocks = cache.reshape(b, g, mb, block_size, d).permute(0, 2, 1, 3, 4)
        pool[table.reshape(-1).long().to(cache.device)] = blocks.reshape(b * mb, g, block_size, d)
        pools.append(pool)
    return pools[0], pools[1], table.to(k_cache.device)


def projection_bytes(cfg: DecodeConfig) -> int:
    """Algorithmic bytes of the projections of one layer: the weights P_q,
    P_k, P_v, P_o once, x and y, and q / k_new / v_new / o written and read."""
    w = (2 * cfg.h + 2 * cfg.g) * cfg.D * cfg.d * cfg.elt
    act = 2 * cfg.b * cfg.D * cfg.elt
    inter = 2 * cfg.b * (2 * cfg.h + 2 * cfg.g) * cfg.d * cfg.elt
    return w + act + inter


def _boost(cfg, layer, q, k_cache, k_new, lens):
    """Raise every head's logit by about cfg.boost at 1 % of the positions."""
    cpu_gen = torch.Generator(device="cpu")
    cpu_gen.manual_seed(cfg.seed * 1000 + layer + 7)
    qd = q.float().cpu().double().numpy()          # bf16-rounded query
    for i in range(cfg.b):
        L = int(lens[i])
        n = int(round(cfg.boost_frac * L))
        if n == 0:
            continue
        pos = torch.randperm(L, generator=cpu_gen)[:n]
        Q = qd[i]                                   # [h, d]
        u = Q.T @ np.linalg.solve(Q @ Q.T, np.ones(Q.shape[0]))
        du = torch.from_numpy((cfg.boost / cfg.scale) * u).float()
        du = du.to(k_cache.device)
        rows = pos[pos < L - 1].to(k_cache.device)
        k_cache[i, 0, rows, :] += du
        if bool((pos == L - 1).any()):
            k_new[i, 0, :] += du
    return k_cache, k_new
