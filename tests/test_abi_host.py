"""C-ABI checks that need no GPU: the library loads, exports every function
include/gqa.h declares, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa.h")


def _lib():
    from gqa_kv_cache_append_gb300 import build
    build.build()
    from gqa_kv_cache_append_gb300 import binding
    return binding


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gqa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("gqa_kv_append", "gqa_decode_attn", "gqa_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol():
    b = _lib()
    out = subprocess.run(["nm", "-D", "--defined-only", b.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(\S+)$", out, flags=re.M))
    for n in declared_functions():
        assert n in exported, n
        assert n in b.SIGNATURES, n
        getattr(b.lib, n)


def test_status_strings_and_version():
    b = _lib()
    assert b.status_string(0) == "GQA_OK"
    assert b.status_string(-2) == "GQA_ERR_SHAPE"
    assert b.gqa_version() >= 100


A = 0x10000  # a 16-byte aligned address that is never dereferenced


def _attn(lib_, **kw):
    args = dict(q=A, k=A, v=A, lens=A, b=2, h=8, g=2, dk=128, dv=128, scale=0.1,
                out=A, cap=64, dtype=1)
    args.update(kw)
    return lib_.lib.gqa_decode_attn(args["q"], args["k"], args["v"], args["lens"], args["b"],
                                 args["h"], args["g"], args["dk"], args["dv"],
                                 args["scale"], args["out"], args["cap"], args["dtype"],
                                 None)


def _app(lib_, **kw):
    args = dict(kn=A, vn=A, k=A, v=A, lens=A, b=2, g=2, dk=128, dv=128, cap=64, dtype=1)
    args.update(kw)
    return lib_.lib.gqa_kv_append(args["kn"], args["vn"], args["k"], args["v"], args["lens"],
                               args["b"], args["g"], args["dk"], args["dv"], args["cap"],
                               args["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), -1), (dict(out=0), -1), (dict(lens=0), -1),
    (dict(dtype=3), -3), (dict(dtype=-1), -3),
    (dict(h=6, g=4), -2), (dict(b=0), -2), (dict(g=0), -2), (dict(cap=0), -2),
    (dict(dk=0), -2), (dict(b=40000, g=8, h=8, cap=8000), -2),
    (dict(q=A + 8), -4), (dict(k=A + 2), -4), (dict(out=A + 4), -4), (dict(lens=A + 2), -4),
    (dict(dk=128, dv=32), -5), (dict(dk=96, dv=96), -5), (dict(h=64, g=1), -5),
    (dict(dk=128, dv=64, h=66, g=2), -5),       # 33 query rows per KV head
    (dict(dtype=0, h=34, g=1), -5), (dict(dtype=0, dk=64, dv=128, h=17, g=1), -5),
    # head dims above 128: 16-bit data, at most 16 query rows per KV head
    (dict(dk=256, dv=256, h=34, g=2), -5), (dict(dtype=0, dk=256, dv=256), -5),
    (dict(dk=192, dv=64), -5), (dict(dk=64, dv=256), -5), (dict(dk=320, dv=128), -5),
])
def test_decode_attn_host_checks(kw, code):
    assert _attn(_lib(), **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(kn=0), -1), (dict(lens=0), -1), (dict(dtype=7), -3),
    (dict(b=0), -2), (dict(cap=0), -2), (dict(dv=0), -2),
    (dict(dk=4, dtype=1), -5), (dict(k=A + 4), -4),
])
def test_kv_append_host_checks(kw, code):
    assert _app(_lib(), **kw) == code


def test_decode_step_host_checks():
    b = _lib()
    f = b.lib.gqa_decode_step
    args = [A, A, A, A, A, A, 2, 8, 2, 128, 128, 0.1, A, 64, 1, 0, None]
    assert f(*args[:1], 0, *args[2:]) == -1          # k_new null
    assert f(*args[:2], 0, *args[3:]) == -1          # v_new null
    assert f(*args[:1], A + 8, *args[2:]) == -4      # k_new misaligned
    bad = list(args)
    bad[7] = 6
    bad[8] = 4
    assert f(*bad) == -2                             # h % g
    bad = list(args)
    bad[15] = 6
    assert f(*bad) == -5                             # unknown flag bits


def test_null_status_pointer():
    b = _lib()
    assert b.lib.gqa_device_status(None, None) == -1


def test_valid_arguments_without_a_gpu_report_a_cuda_error():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    b = _lib()
    assert _attn(b) in (-6, -7)
    assert _app(b) in (-6, -7)


def _attn_multi(lib_, **kw):
    args = dict(q=A, k=A, v=A, lens=A, b=2, n=3, h=8, g=2, dk=128, dv=128, scale=0.1,
                out=A, cap=64, dtype=1)
    args.update(kw)
    return lib_.lib.gqa_decode_attn_multi(
        args["q"], args["k"], args["v"], args["lens"], args["b"], args["n"], args["h"],
        args["g"], args["dk"], args["dv"], args["scale"], args["out"], args["cap"],
        args["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), -1), (dict(n=0), -2), (dict(n=-1), -2), (dict(n=65, cap=64), -2),
    (dict(h=6, g=4), -2), (dict(q=A + 8), -4),
    (dict(n=9, h=8, g=2), -5),                  # 9 * 4 query rows > 32
    (dict(n=3, dtype=0, h=12, g=2), -5),        # fp32: 18 rows > 16
    (dict(n=3, dtype=1, dk=64, dv=128, h=22, g=2), -5),  # bf16: 33 rows > 32
    (dict(dtype=3), -3),
])
def test_decode_attn_multi_host_checks(kw, code):
    assert _attn_multi(_lib(), **kw) == code


def test_multi_step_and_append_host_checks():
    b = _lib()
    f = b.lib.gqa_decode_step_multi
    args = [A, A, A, A, A, A, 2, 3, 8, 2, 128, 128, 0.1, A, 64, 1, 0, None]
    assert f(*args[:1], 0, *args[2:]) == -1          # k_new null
    bad = list(args)
    bad[7] = 0
    assert f(*bad) == -2                             # n < 1
    bad = list(args)
    bad[16] = 4
    assert f(*bad) == -5                             # unknown flag bits
    bad[16] = 2                                      # CUDA-core kernel: 12 rows > 8 in bf16
    assert f(*bad) == -5
    app = b.lib.gqa_kv_append_multi
    aargs = [A, A, A, A, A, 2, 3, 2, 128, 128, 64, 1, None]
    bad = list(aargs)
    bad[6] = 0
    assert app(*bad) == -2                           # n < 1
    bad = list(aargs)
    bad[6] = 65
    assert app(*bad) == -2                           # n > cap
    bad = list(aargs)
    bad[0] = 0
    assert app(*bad) == -1


def test_projection_and_layer_host_checks():
    b = _lib()
    pq = b.lib.gqa_project_qkv
    # x, wq, wk, wv, q, kn, vn, b, D, h, g, dk, dv, dtype, flags, stream
    args = [A, A, A, A, A, A, A, 4, 256, 8, 2, 128, 128, 1, 0, None]

    def call(f, base, **idx):
        a = list(base)
        for k, v in idx.items():
            a[int(k[1:])] = v
        return f(*a)
    assert call(pq, args, i0=0) == -1                 # x null
    assert call(pq, args, i13=0) == -5                # fp32: no projection kernel
    assert call(pq, args, i13=5) == -3
    assert call(pq, args, i8=200) == -5               # D not a multiple of 128
    assert call(pq, args, i7=129) == -5               # b > 128
    assert call(pq, args, i7=0) == -2
    assert call(pq, args, i11=64, i12=64) == -5       # head dim 64
    assert call(pq, args, i9=6, i10=4) == -2          # h % g
    assert call(pq, args, i4=A + 2) == -4
    assert call(pq, args, i14=4) == -5                # unknown flag
    po = b.lib.gqa_project_out
    oargs = [A, A, A, 4, 256, 8, 128, 1, 0, None]
    assert call(po, oargs, i1=0) == -1
    assert call(po, oargs, i6=64) == -5
    assert call(po, oargs, i2=A + 8) == -4
    dl = b.lib.gqa_decode_layer
    largs = [A, A, A, A, A, A, A, A, 4, 256, 8, 2, 128, 128, 0.1, A, 64, 1, 0, None]
    assert call(dl, largs, i4=0) == -1                # w_o null
    assert call(dl, largs, i5=0) == -1                # k_cache null
    assert call(dl, largs, i16=0) == -2               # cap
    assert call(dl, largs, i7=A + 2) == -4            # seq_lens misaligned
    assert call(dl, largs, i17=0) == -5


def test_paged_host_checks():
    b = _lib()
    f = b.lib.gqa_decode_attn_paged
    # q, kp, vp, table, lens, b, n, h, g, dk, dv, scale, out, bs, max_blocks, num_blocks, dtype,
    # stream
    args = [A, A, A, A, A, 2, 1, 8, 2, 128, 128, 0.1, A, 64, 4, 16, 1, None]

    def call(fn, base, **idx):
        a = list(base)
        for k, v in idx.items():
            a[int(k[1:])] = v
        return fn(*a)
    assert call(f, args, i3=0) == -1                  # table null
    assert call(f, args, i3=A + 2) == -4              # table misaligned
    assert call(f, args, i13=24) == -5                # block size not a power of two
    assert call(f, args, i13=8) == -5                 # below 16
    assert call(f, args, i14=0) == -2
    assert call(f, args, i15=0) == -2
    assert call(f, args, i16=4) == -3
    assert call(f, args, i6=0) == -2                  # n < 1
    assert call(f, args, i6=9) == -5                  # 9 tokens x 4 heads > 32 rows
    assert call(f, args, i7=64, i9=256, i10=256) == -5  # head dims above 128: 16 rows at most
    st = b.lib.gqa_decode_step_paged
    sargs = [A, A, A, A, A, A, A, 2, 1, 8, 2, 128, 128, 0.1, A, 64, 4, 16, 1, 0, None]
    assert call(st, sargs, i1=0) == -1
    assert call(st, sargs, i19=4) == -5               # unknown flag
    ap = b.lib.gqa_kv_append_paged
    aargs = [A, A, A, A, A, A, 2, 1, 2, 128, 128, 64, 4, 16, 1, None]
    assert call(ap, aargs, i4=0) == -1
    assert call(ap, aargs, i11=48) == -5
    assert call(ap, aargs, i7=0) == -2


def test_decode_plan_query():
    """gqa_decode_plan on the host (SM count given): persistent grid of at
    most one CTA per SM and at most one per tile (with fewer (sequence, KV
    head) units than SMs, a whole number of CTAs per unit).  Where that cuts
    every unit into exactly two pieces, the tensor-core kernel is launched in
    clusters of two.  Where it cuts every unit into three or more pieces
    (more CTAs than twice the units),
    the CUDA-core kernel adds the combine kernel, and the tensor-core kernel
    is launched in clusters of C CTAs, k per unit (the most CTAs over the
    sizes 2..16, then the fewest clusters per unit; the host-only plan lets
    every SM take part in clusters of any size) when k <= 2 and the
    streaming time its fewer CTAs give up, capacity at 7.4 TB/s, is below
    2 us; else the combine kernel merges.  The workspace holds the
    partials ((b*g + C) * rows * (d_v + 2) floats) and the arrival counters
    (2*b*g, or b*g*C in a cluster launch)."""
    b = _lib()
    p = b.gqa_decode_plan(32, 1, 64, 8, 128, 128, 8192, "bf16", num_sms=152)
    assert p["tensor_core"] and p["tile"] == 128 and p["ctas"] == 152 and p["kernels"] == 1
    assert p["cluster"] == 0
    # 64-wide heads: tiles of 256 positions (fp32: the CUDA-core kernel's 128)
    assert b.gqa_decode_plan(32, 1, 64, 8, 64, 64, 8192, "bf16", num_sms=152)["tile"] == 256
    assert b.gqa_decode_plan(32, 1, 64, 8, 64, 64, 8192, "f16", num_sms=152)["tile"] == 256
    assert b.gqa_decode_plan(32, 1, 64, 8, 64, 128, 8192, "bf16", num_sms=152)["tile"] == 128
    # head dims above 128 (up to 16 query rows): the tensor-core kernel, 128 positions
    for dk, dv in [(256, 256), (192, 128), (128, 256), (256, 128), (192, 192)]:
        p2 = b.gqa_decode_plan(32, 1, 64, 8, dk, dv, 8192, "bf16", num_sms=152)
        assert p2["tensor_core"] and p2["tile"] == 128
        assert p2["workspace_bytes"] == (32 * 8 + 152) * 8 * (dv + 2) * 4 + 2 * 32 * 8 * 4
    assert p["workspace_bytes"] == (32 * 8 + 152) * 8 * 130 * 4 + 2 * 32 * 8 * 4
    # long-context MQA: 8 units of 1024 tiles; the best cluster plan (two
    # clusters of 9 per unit, 144 CTAs) would give up ~3.8 us of streaming:
    # 152 CTAs and the combine kernel
    p = b.gqa_decode_plan(8, 1, 32, 1, 128, 128, 131072, "bf16", num_sms=152)
    assert (p["ctas"], p["cluster"], p["kernels"]) == (152, 0, 2)
    # the g = 1 point of the sweep: 16 units of 32 tiles, clusters of 9
    p = b.gqa_decode_plan(16, 1, 32, 1, 128, 128, 4096, "bf16", num_sms=152)
    assert (p["ctas"], p["cluster"], p["kernels"]) == (144, 9, 1)
    p = b.gqa_decode_plan(32, 4, 64, 8, 128, 128, 8192, "f16", num_sms=152)
    assert p["tensor_core"] and p["kernels"] == 1
    for (bb, n, h, g, dk, dv, cap, dt) in [(1, 1, 8, 1, 64, 64, 256, "f32"),
                                           (3, 1, 8, 2, 128, 64, 1000, "bf16"),
                                           (5, 1, 8, 2, 128, 128, 20000, "bf16"),
                                           (16, 1, 32, 8, 128, 128, 4096, "bf16"),
                                           (12, 1, 32, 8, 128, 128, 4096, "bf16"),
                                           (16, 1, 32, 1, 128, 128, 4096, "bf16"),
                                           (64, 1, 28, 4, 128, 128, 32768, "bf16"),
                                           (1, 1, 32, 1, 128, 128, 131072, "f16"),
                                           (8, 1, 32, 1, 64, 64, 131072, "bf16"),
                                           (16, 1, 32, 1, 64, 64, 2048, "bf16"),
                                           (16, 1, 32, 4, 128, 128, 4096, "bf16"),
                                           (38, 1, 8, 2, 128, 128, 1000, "bf16"),
                                           (38, 1, 8, 2, 128, 128, 1000, "f32"),
                                           (1, 1, 8, 8, 128, 128, 1, "bf16")]:
        p = b.gqa_decode_plan(bb, n, h, g, dk, dv, cap, dt, num_sms=152)
        unit_tiles = -(-cap // p["tile"])
        tiles = bb * g * unit_tiles
        units = bb * g
        # fewer units than SMs, at most half as many: a whole number of CTAs
        # per unit
        aligned = min(units * (152 // units) if 2 * units <= 152 else 152, tiles)
        rows = n * h // g
        assert p["tensor_core"] == (dt != "f32")
        clustered = False
        if aligned > 2 * units and p["tensor_core"]:
            pieces = min(aligned // units, unit_tiles)
            best = max((units * c * min(pieces // c, (152 // c) // units), c)
                       for c in range(2, 17) if c <= pieces)
            k = best[0] // (units * best[1])
            stream = units * unit_tiles * p["tile"] * (dk + dv) * 2 / 7.4e12
            clustered = best[0] > 0 and k <= 2 and stream * (1 - best[0] / aligned) < 2e-6
        if aligned == 2 * units and p["tensor_core"]:
            assert (p["ctas"], p["cluster"], p["kernels"]) == (aligned, 2, 1)
            counters = units * 2
        elif clustered:
            assert p["ctas"] == best[0] and p["cluster"] == best[1] and p["kernels"] == 1
            assert p["ctas"] % (units * p["cluster"]) == 0
            counters = units * p["cluster"]
        else:
            assert 1 <= p["ctas"] == aligned and p["cluster"] == 0
            assert p["kernels"] == (2 if p["ctas"] > 2 * bb * g else 1)
            counters = 2 * units
        assert p["workspace_bytes"] == ((bb * g + p["ctas"]) * rows * (dv + 2) * 4
                                        + max(counters, 2 * units) * 4)
    # the CUDA-core kernel on request: bf16 up to 8 query rows per KV head
    p = b.gqa_decode_plan(32, 1, 64, 8, 128, 128, 8192, "bf16", num_sms=152,
                          flags=b.GQA_STEP_CUDA_CORES)
    assert not p["tensor_core"] and p["tile"] == 64
    plan = b.lib.gqa_decode_plan
    assert plan(2, 1, 8, 3, 128, 128, 64, 1, 0, 152, None, None, None, None, None, None) == -2
    assert plan(2, 1, 8, 2, 128, 128, 64, 7, 0, 152, None, None, None, None, None, None) == -3
    assert plan(2, 1, 8, 2, 96, 96, 64, 1, 0, 152, None, None, None, None, None, None) == -5
    assert plan(2, 1, 8, 2, 128, 128, 64, 1, 0, -1, None, None, None, None, None, None) == -2
    assert plan(2, 1, 32, 2, 128, 128, 64, 1, 2, 152, None, None, None, None, None, None) == -5
    assert plan(2, 1, 8, 2, 128, 128, 64, 1, 4, 152, None, None, None, None, None, None) == -5
