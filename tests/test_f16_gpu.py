"""fp16 storage (IEEE half, the other 2-byte format the pages name beside
bf16) through the C ABI against the float64 oracle: the tensor-core kernel
(one and n tokens, split units merged in the kernel and in the combine
kernel), head dim 64 and d_k != d_v, the paged cache,
and the append (bit copies).  Bound: 1e-2 + 5e-3 |ref| (fp32 accumulation,
fp16 inputs and softmax weights)."""
import numpy as np
import pytest

from tests.test_decode_gpu import cfg_of, run_step
from tests.test_multi_gpu import cfg_of as multi_cfg, run_multi
from tests.test_paged_gpu import cfg_of as paged_cfg, run_paged

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("b,h,g,d,cap,lens", [
    (2, 64, 8, 128, 1000, [1000, 129]),        # Llama heads, tensor cores
    (3, 32, 1, 128, 2048, [2048, 1, 700]),     # r = 32
    (1, 8, 1, 128, 16384, [99 * 128 + 2]),     # one unit over many CTAs: combine kernel
    (96, 8, 1, 128, 384, [258] * 96),          # split units merged in the decode kernel
    (3, 8, 2, 64, 300, [1, 65, 300]),          # head dim 64
])
@pytest.mark.parametrize("fused", [True, False])
def test_f16_step(b, h, g, d, cap, lens, fused):
    run_step(cfg_of("f16", b, h, g, d, cap, seed=b + h), lens, fused=fused)


def test_f16_multi_token():
    run_multi(multi_cfg("f16", 2, 64, 8, 128, 700, seed=3), 4, [700, 257])


@pytest.mark.parametrize("bs", [16, 128])
def test_f16_paged(bs):
    run_paged(paged_cfg("f16", 3, 16, 2, 128, 512, seed=bs), [1, 300, 512], bs)


def test_f16_nan_padding():
    run_step(cfg_of("f16", 2, 16, 4, 128, 300, seed=9), [131, 250], pad_fill=float("nan"))
