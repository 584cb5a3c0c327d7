"""Split units merged across thread-block clusters (tensor-core kernel).

When a call cuts every (sequence, KV head) unit into exactly two pieces,
the tensor-core kernel is launched in clusters of two; when it would cut
every unit into three or more pieces, in clusters of C CTAs, k clusters per
unit.  Either way the kernel merges the pieces itself: over distributed shared memory when
every unit has the same number of tiles (then, with k > 1, the k cluster
results through the split workspace), through the split workspace when the
lengths are ragged.  GQA_CLUSTER=0 takes the combine kernel instead; a size
from 2 to 16 forces that cluster size.

Every case is checked against the float64 oracle on the same host inputs,
under the automatic plan, forced sizes (one and several clusters per unit)
and the combine kernel, with bit-identical results on a second run."""
import numpy as np
import pytest
import torch

from tests.test_decode_gpu import cfg_of, run_step
from tests.test_multi_gpu import cfg_of as cfg_multi, run_multi
from tests.test_paged_gpu import cfg_of as cfg_paged, run_paged
from tests.util import bits

pytestmark = pytest.mark.gpu

MODES = ["auto", "0", "2", "4", "9", "16"]


def _b():
    from gqa_kv_cache_append_gb300 import binding
    return binding


@pytest.fixture
def cluster_mode(request, monkeypatch):
    mode = request.param
    if mode == "auto":
        monkeypatch.delenv("GQA_CLUSTER", raising=False)
    else:
        monkeypatch.setenv("GQA_CLUSTER", mode)
    return mode


def _plan(b, n, h, g, d, cap, dtype="bf16"):
    return _b().gqa_decode_plan(b, n, h, g, d, d, cap, dtype)


@pytest.mark.parametrize("cluster_mode", MODES, indirect=True)
@pytest.mark.parametrize("b,h,g,d,cap,lens", [
    (8, 32, 1, 128, 4096, [4096] * 8),            # long-context MQA shape, equal lengths
    (1, 8, 1, 128, 16384, [16384]),               # one unit over every SM: k > 1
    (1, 32, 1, 128, 12800, [12800 - 5]),          # ragged tail of the last tile
    (2, 64, 8, 64, 2048, [2048, 2048]),           # 16 units, r = 8, d = 64
    (4, 28, 4, 128, 3000, [3000, 1, 2999, 1500]),  # ragged, r = 7, a 1-row sequence
    (3, 16, 2, 128, 2000, [129, 2000, 640]),      # ragged
    (2, 16, 16, 128, 900, [900, 900]),            # MHA, 7-8 tiles a unit: empty CTAs
])
def test_cluster_merge(cluster_mode, b, h, g, d, cap, lens):
    cfg = cfg_of("bf16", b, h, g, d, cap, seed=b * 7 + h)
    p = _plan(b, 1, h, g, d, cap)
    if cluster_mode == "0":
        assert p["cluster"] == 0
    elif cluster_mode != "auto" and p["ctas"] > 2 * b * g:
        assert p["cluster"] == int(cluster_mode) or p["cluster"] == 0
    run_step(cfg, lens)
    run_step(cfg, lens, fused=True)


@pytest.mark.parametrize("cluster_mode", ["auto", "0"], indirect=True)
@pytest.mark.parametrize("b,h,g,d,cap,lens", [
    (16, 32, 4, 128, 4096, [4096] * 16),          # 64 units of 32 tiles: pairs
    (16, 32, 4, 128, 4096, [4096, 3000, 4096, 17, 2500, 4096, 4096, 1,
                            4000, 4096, 129, 4096, 128, 4096, 4096, 3333]),  # ragged
    (38, 8, 2, 128, 1000, [1000] * 38),           # 76 units: every SM of 152
    (16, 64, 4, 64, 4096, [4096] * 16),           # 64-wide heads: 256-position tiles
])
def test_cluster_pairs(cluster_mode, b, h, g, d, cap, lens):
    cfg = cfg_of("bf16", b, h, g, d, cap, seed=b * 5 + g)
    p = _plan(b, 1, h, g, d, cap)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if cluster_mode == "auto" and sms // (b * g) == 2:  # two CTAs per unit
        assert (p["cluster"], p["ctas"], p["kernels"]) == (2, 2 * b * g, 1)
    if cluster_mode == "0":
        assert p["cluster"] == 0
    run_step(cfg, lens)
    run_step(cfg, lens, fused=True)


def test_auto_plan_chooses_clusters_for_short_split_calls():
    # 16 units of 32 tiles: a cluster launch (no combine kernel)
    p = _plan(16, 1, 32, 1, 128, 4096)
    assert p["cluster"] >= 2 and p["kernels"] == 1 and p["ctas"] % (16 * p["cluster"]) == 0
    p = _plan(16, 1, 32, 1, 128, 4096, "f16")
    assert p["cluster"] >= 2 and p["kernels"] == 1
    # 8 units of 1024 tiles: every CTA streams, the combine kernel merges
    p = _plan(8, 1, 32, 1, 128, 131072)
    assert p["cluster"] == 0 and p["kernels"] == 2
    # the CUDA-core kernel keeps the combine kernel
    p = _plan(1, 1, 8, 1, 64, 20000, "f32")
    assert p["cluster"] == 0 and p["kernels"] == 2


@pytest.mark.parametrize("cluster_mode", ["auto", "2", "16"], indirect=True)
@pytest.mark.parametrize("lens", [[6000] * 4, [6000, 100, 5000, 3]])
def test_cluster_merge_is_deterministic(cluster_mode, lens):
    B = _b()
    from gqa_kv_cache_append_gb300.inputs import make_layer
    cfg = cfg_of("bf16", 4, 32, 1, 128, 6000, seed=31)
    x = make_layer(cfg, 0, "cuda", lens=np.asarray(lens, dtype=np.int32))
    outs = []
    for _ in range(3):
        out = torch.empty((cfg.b, cfg.h, cfg.d), dtype=torch.bfloat16, device="cuda")
        B.gqa_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["seq_lens"], cfg.b, cfg.h,
                          cfg.g, 128, 128, cfg.scale, out)
        outs.append(bits(out))
    assert B.gqa_device_status() == 0
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


@pytest.mark.parametrize("cluster_mode", ["auto", "4"], indirect=True)
@pytest.mark.parametrize("b,n,h,g,cap,lens", [
    (2, 4, 32, 4, 6000, [6000, 6000]),     # 8 units, 32 query rows, equal lengths
    (1, 2, 16, 1, 9000, [8999]),           # one unit, new rows straddle a tile
    (2, 4, 16, 2, 5000, [5000, 130]),      # ragged
])
def test_cluster_merge_multi_token(cluster_mode, b, n, h, g, cap, lens):
    run_multi(cfg_multi("bf16", b, h, g, 128, cap, seed=n + cap), n, lens)


@pytest.mark.parametrize("cluster_mode", ["auto", "8"], indirect=True)
@pytest.mark.parametrize("bs", [16, 256])
@pytest.mark.parametrize("lens", [[8192, 8192], [8192, 3001]])
def test_cluster_merge_paged(cluster_mode, bs, lens):
    run_paged(cfg_paged("bf16", 2, 32, 1, 128, 8192, seed=bs), lens, bs)
