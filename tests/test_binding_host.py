"""The Python binding's argument marshalling (CPU): tensors that the
kernels could not read or write whole are refused before the library is
called — host tensors, strided views, tensors smaller than the shapes
passed, lengths or block tables that are not int32."""
import pytest
import torch


def _b():
    from gqa_kv_cache_append_gb300 import build
    build.build()
    from gqa_kv_cache_append_gb300 import binding
    return binding


def _args(b=2, h=8, g=2, d=128, cap=64, dt=torch.bfloat16):
    return dict(q=torch.zeros((b, h, d), dtype=dt), k=torch.zeros((b, g, cap, d), dtype=dt),
                v=torch.zeros((b, g, cap, d), dtype=dt), kn=torch.zeros((b, g, d), dtype=dt),
                vn=torch.zeros((b, g, d), dtype=dt), lens=torch.ones(b, dtype=torch.int32),
                out=torch.zeros((b, h, d), dtype=dt))


def _attn(B, a, b=2, h=8, g=2, d=128):
    # stream 0 given: no CUDA runtime call is needed to marshal the arguments
    B.gqa_decode_attn(a["q"], a["k"], a["v"], a["lens"], b, h, g, d, d, 0.1, a["out"], stream=0)


def test_host_tensors_are_refused():
    B = _b()
    with pytest.raises(ValueError, match="CUDA tensor"):
        _attn(B, _args())


def test_strided_views_are_refused():
    B = _b()
    a = _args()
    a["q"] = torch.zeros((2, 128, 8), dtype=torch.bfloat16).transpose(1, 2)
    with pytest.raises(ValueError, match="q: must be contiguous"):
        _attn(B, a)


@pytest.mark.parametrize("key,shape", [("q", (2, 8, 64)), ("k", (2, 2, 32, 128)),
                                       ("v", (1, 2, 64, 128)), ("out", (2, 4, 128)),
                                       ("lens", (1,))])
def test_tensors_smaller_than_the_shapes_are_refused(key, shape):
    B = _b()
    a = _args()
    a[key] = torch.zeros(shape, dtype=a[key].dtype)
    with pytest.raises(ValueError, match="bytes, the shapes passed need"):
        # cap is given, so a short cache is caught by its size
        B.gqa_decode_attn(a["q"], a["k"], a["v"], a["lens"], 2, 8, 2, 128, 128, 0.1, a["out"],
                          cap=64)


def test_lengths_must_be_int32():
    B = _b()
    a = _args()
    a["lens"] = torch.ones(2, dtype=torch.int64)
    with pytest.raises(ValueError, match="seq_lens: must be int32"):
        _attn(B, a)


def test_step_multi_paged_and_layer_check_their_tensors():
    B = _b()
    a = _args()
    with pytest.raises(ValueError, match="k_new: holds"):
        B.gqa_decode_step(a["q"], a["kn"][:1], a["vn"], a["k"], a["v"], a["lens"], 2, 8, 2, 128,
                          128, 0.1, a["out"])
    with pytest.raises(ValueError, match="q: holds"):
        B.gqa_decode_attn_multi(a["q"], a["k"], a["v"], a["lens"], 2, 3, 8, 2, 128, 128, 0.1,
                                a["out"])
    pool = torch.zeros((8, 2, 16, 128), dtype=torch.bfloat16)
    table = torch.zeros((2, 4), dtype=torch.int64)
    with pytest.raises(ValueError, match="block_table: must be int32"):
        B.gqa_decode_attn_paged(a["q"], pool, pool, table, a["lens"], 2, 8, 2, 128, 128, 0.1,
                                a["out"])
    with pytest.raises(ValueError, match="v_pool: holds"):
        B.gqa_decode_attn_paged(a["q"], pool, pool[:4], table.int(), a["lens"], 2, 8, 2, 128,
                                128, 0.1, a["out"])
    x = torch.zeros((2, 1024), dtype=torch.bfloat16)
    w = torch.zeros((8, 1024, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="w_k: holds"):
        B.gqa_project_qkv(x, w, w[:1], w[:2], a["q"], a["kn"], a["vn"], 2, 1024, 8, 2, 128, 128)
    with pytest.raises(ValueError, match="CUDA tensor"):
        B.gqa_project_out(a["q"], w, x, 2, 1024, 8, 128, stream=0)
