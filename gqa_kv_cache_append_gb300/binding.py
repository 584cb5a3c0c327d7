"""Thin ctypes binding of libgqa.so (include/gqa.h), same names as the C ABI.

Argument marshalling only: tensors become device pointers, torch dtypes
become GQA_F32 / GQA_BF16, and the current torch CUDA stream is passed when
no stream is given.  Every step of the computation runs in the library's
CUDA kernels; there is no fallback.  Loading fails loudly when the library
has not been built (``python -m gqa_kv_cache_append_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB

GQA_F32 = 0
GQA_BF16 = 1
GQA_F16 = 2

GQA_OK = 0
GQA_ERR_NULL = -1
GQA_ERR_SHAPE = -2
GQA_ERR_DTYPE = -3
GQA_ERR_ALIGN = -4
GQA_ERR_UNSUPPORTED = -5
GQA_ERR_CUDA = -6
GQA_ERR_DEVICE = -7
GQA_ERR_SCRATCH_LIMIT = -8

GQA_STEP_EARLY_STREAM = 1
GQA_STEP_CUDA_CORES = 2

GQA_DEV_BAD_SEQ_LEN = 1
GQA_DEV_WAIT_TIMEOUT = 2
GQA_DEV_INTERNAL = 4
GQA_DEV_BAD_BLOCK = 8

# every function the header declares, with its C signature
_VP, _I, _F, _LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong
SIGNATURES = {
    "gqa_kv_append": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _VP]),
    "gqa_decode_attn": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, _VP, _I, _I, _VP]),
    "gqa_decode_attn_noalloc": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, _VP, _I, _I,
                                     _VP]),
    "gqa_decode_step": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, _VP, _I,
                             _I, _I, _VP]),
    "gqa_kv_append_multi": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I, _VP]),
    "gqa_decode_attn_multi": (_I, [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _VP, _I, _I,
                                   _VP]),
    "gqa_decode_step_multi": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F,
                                   _VP, _I, _I, _I, _VP]),
    "gqa_project_qkv": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I,
                             _I, _VP]),
    "gqa_project_out": (_I, [_VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _VP]),
    "gqa_decode_layer": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I,
                              _F, _VP, _I, _I, _I, _VP]),
    "gqa_kv_append_paged": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I, _I,
                                 _I, _VP]),
    "gqa_decode_attn_paged": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _VP, _I,
                                   _I, _I, _I, _VP]),
    "gqa_decode_step_paged": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I,
                                   _F, _VP, _I, _I, _I, _I, _I, _VP]),
    "gqa_decode_plan": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(_I),
                             ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I),
                             ctypes.POINTER(_LL), ctypes.POINTER(_I)]),
    "gqa_device_status": (_I, [_VP, ctypes.POINTER(ctypes.c_uint32)]),
    "gqa_selftest_wait_timeout": (_I, [_LL, _VP]),
    "gqa_status_string": (ctypes.c_char_p, [_I]),
    "gqa_version": (_I, []),
}


class GqaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code} ({status_string(code)})")
        self.code = code


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB):
        raise ImportError(
            f"{LIB} is missing: build it with `python -m gqa_kv_cache_append_gb300.build` "
            "(or __graft_entry__.build()); there is no fallback implementation")
    lib = ctypes.CDLL(LIB)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def status_string(code: int) -> str:
    return lib.gqa_status_string(int(code)).decode()


def _ptr(x, name: str = "tensor", nbytes: int = 0, index: bool = False) -> int:
    """Device address of a tensor argument (raw integers pass through
    unchecked).  The kernels read and write whole extents through it, so a
    host tensor, a strided view, a tensor smaller than the shapes passed
    (nbytes) or, for lengths and block tables (index), another type than
    int32 is refused here, before anything is launched."""
    if isinstance(x, torch.Tensor):
        if not x.is_contiguous():
            raise ValueError(f"{name}: must be contiguous")
        if index and x.dtype != torch.int32:
            raise ValueError(f"{name}: must be int32, got {x.dtype}")
        have = x.numel() * x.element_size()
        if have < nbytes:
            raise ValueError(f"{name}: holds {have} bytes, the shapes passed need {nbytes}")
        if not x.is_cuda:
            # reported by _call once every argument has been checked
            return _HostTensor(name, x.device)
        return x.data_ptr()
    return int(x) if x is not None else 0


class _HostTensor:
    """Stands for a tensor argument that is not on a CUDA device."""

    def __init__(self, name, device):
        self.name, self.device = name, device


def _call(fn_name: str, fn, *args) -> None:
    """Call a library entry point once no argument is a host tensor; raise
    GqaError on a non-zero return code."""
    for a in args:
        if isinstance(a, _HostTensor):
            raise ValueError(f"{a.name}: a CUDA tensor is required, got one on {a.device}")
    _check(fn_name, fn(*args))


def _elt(code: int) -> int:
    """Bytes per element of a dtype code (0 for an unknown code, which the
    library rejects)."""
    return {GQA_F32: 4, GQA_BF16: 2, GQA_F16: 2}.get(code, 0)


def _n(*dims) -> int:
    """Product of the dims, 0 when one is not positive (the library then
    reports the shape error)."""
    out = 1
    for d in dims:
        d = int(d)
        if d <= 0:
            return 0
        out *= d
    return out


def _dtype(x, dtype) -> int:
    if dtype is not None:
        return int(dtype)
    if isinstance(x, torch.Tensor):
        if x.dtype == torch.bfloat16:
            return GQA_BF16
        if x.dtype == torch.float32:
            return GQA_F32
        if x.dtype == torch.float16:
            return GQA_F16
        return -99  # the library rejects it with GQA_ERR_DTYPE
    raise ValueError("dtype must be given when passing raw pointers")


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(fn: str, code: int) -> None:
    if code != GQA_OK:
        raise GqaError(fn, code)


def gqa_kv_append(k_new, v_new, k_cache, v_cache, seq_lens, b, g, d_k, d_v,
                  cap=None, dtype=None, stream=None) -> None:
    """Write row seq_lens[i] - 1 of every (i, j) of the caches (in place)."""
    if cap is None:
        cap = k_cache.shape[2]
    dt = _dtype(k_cache, dtype)
    e = _elt(dt)
    _call("gqa_kv_append", lib.gqa_kv_append,
        _ptr(k_new, "k_new", _n(b, g, d_k) * e), _ptr(v_new, "v_new", _n(b, g, d_v) * e),
        _ptr(k_cache, "k_cache", _n(b, g, cap, d_k) * e),
        _ptr(v_cache, "v_cache", _n(b, g, cap, d_v) * e),
        _ptr(seq_lens, "seq_lens", _n(b) * 4, index=True),
        int(b), int(g), int(d_k), int(d_v), int(cap), dt, _stream(stream))


def gqa_decode_attn(q, k_cache, v_cache, seq_lens, b, h, g, d_k, d_v, scale,
                    out, cap=None, dtype=None, stream=None) -> None:
    """out[i, a, :] = softmax_p(scale * q[i, a] . K[i, a // (h/g), p]) V[...]."""
    if cap is None:
        cap = k_cache.shape[2]
    dt = _dtype(q, dtype)
    e = _elt(dt)
    _call("gqa_decode_attn", lib.gqa_decode_attn,
        _ptr(q, "q", _n(b, h, d_k) * e), _ptr(k_cache, "k_cache", _n(b, g, cap, d_k) * e),
        _ptr(v_cache, "v_cache", _n(b, g, cap, d_v) * e),
        _ptr(seq_lens, "seq_lens", _n(b) * 4, index=True), int(b), int(h),
        int(g), int(d_k), int(d_v), float(scale), _ptr(out, "out", _n(b, h, d_v) * e), int(cap),
        dt, _stream(stream))


def gqa_decode_step(q, k_new, v_new, k_cache, v_cache, seq_lens, b, h, g, d_k, d_v,
                    scale, out, cap=None, dtype=None, flags=0, stream=None) -> None:
    """Append k_new / v_new at row seq_lens[i] - 1 and attend, in one launch.
    flags=GQA_STEP_EARLY_STREAM: see include/gqa.h (the kernels still running
    ahead on the stream must not write seq_lens or this call's older rows)."""
    if cap is None:
        cap = k_cache.shape[2]
    dt = _dtype(q, dtype)
    e = _elt(dt)
    _call("gqa_decode_step", lib.gqa_decode_step,
        _ptr(q, "q", _n(b, h, d_k) * e), _ptr(k_new, "k_new", _n(b, g, d_k) * e),
        _ptr(v_new, "v_new", _n(b, g, d_v) * e), _ptr(k_cache, "k_cache", _n(b, g, cap, d_k) * e),
        _ptr(v_cache, "v_cache", _n(b, g, cap, d_v) * e),
        _ptr(seq_lens, "seq_lens", _n(b) * 4, index=True),
        int(b), int(h), int(g), int(d_k), int(d_v), float(scale),
        _ptr(out, "out", _n(b, h, d_v) * e), int(cap), dt, int(flags), _stream(stream))


def gqa_decode_attn_noalloc(q, k_cache, v_cache, seq_lens, b, h, g, d_k, d_v, scale,
                            out, cap=None, dtype=None, stream=None) -> None:
    """gqa_decode_attn for callers that cannot allocate device memory: the
    split partials live in the library's fixed 4 MiB device array instead of
    a cudaMalloc'd workspace.  Calls share that array, so calls that overlap
    on the GPU race; make the first call on a device before any stream
    capture (it looks up the array's device address)."""
    if cap is None:
        cap = k_cache.shape[2]
    dt = _dtype(q, dtype)
    e = _elt(dt)
    _call("gqa_decode_attn_noalloc", lib.gqa_decode_attn_noalloc,
        _ptr(q, "q", _n(b, h, d_k) * e), _ptr(k_cache, "k_cache", _n(b, g, cap, d_k) * e),
        _ptr(v_cache, "v_cache", _n(b, g, cap, d_v) * e),
        _ptr(seq_lens, "seq_lens", _n(b) * 4, index=True), int(b), int(h),
        int(g), int(d_k), int(d_v), float(scale), _ptr(out, "out", _n(b, h, d_v) * e), int(cap),
        dt, _stream(stream))


def gqa_kv_append_multi(k_new, v_new, k_cache, v_cache, seq_lens, b, n, g, d_k, d_v,
                        cap=None, dtype=None, stream=None) -> None:
    """Write rows seq_lens[i] - n .. seq_lens[i] - 1 of every (i, j) of the
    caches from k_new / v_new [b, n, g, d] (in place)."""
    if cap is None:
        cap = k_cache.shape[2]
    dt = _dtype(k_cache, dtype)
    e = _elt(dt)
    _call("gqa_kv_append_multi", lib.gqa_kv_append_multi,
        _ptr(k_new, "k_new", _n(b, n, g, d_k) * e), _ptr(v_new, "v_new", _n(b, n, g, d_v) * e),
        _ptr(k_cache, "k_cache", _n(b, g, cap, d_k) * e),
        _ptr(v_cache, "v_cache", _n(b, g, cap, d_v) * e),
        _ptr(seq_lens, "seq_lens", _n(b) * 4, index=True),
        int(b), int(n), int(g), int(d_k), int(d_v), int(cap), dt, _stream(stream))


def gqa_decode_attn_multi(q, k_cache, v_cache, seq_lens, b, n, h, g, d_k, d_v, scale,
                          out, cap=None, dtype=None, stream=None) -> None:
    """n queries per sequence (q, out [b, n, h, d]) with the causal mask:
    token s sees positions p <= seq_lens[i] - n + s."""
    if cap is None:
        cap = k_cache.shape[2]
    dt = _dtype(q, dtype)
    e = _elt(dt)
    _call("gqa_decode_attn_multi", lib.gqa_decode_attn_multi,
        _ptr(q, "q", _n(b, n, h, d_k) * e), _ptr(k_cache, "k_cache", _n(b, g, cap, d_k) * e),
        _ptr(v_cache, "v_cache", _n(b, g, cap, d_v) * e),
        _ptr(seq_lens, "seq_lens", _n(b) * 4, index=True), int(b), int(n), int(h),
        int(g), int(d_k), int(d_v), float(scale), _ptr(out, "out", _n(b, n, h, d_v) * e),
        int(cap), dt, _stream(stream))


def gqa_decode_step_multi(q, k_new, v_new, k_cache, v_cache, seq_lens, b, n, h, g, d_k,
                          d_v, scale, out, cap=None, dtype=None, flags=0,
                          stream=None) -> None:
    """Append the n new rows and attend causally, in one launch."""
    if cap is None:
        cap = k_cache.shape[2]
    dt = _dtype(q, dtype)
    e = _elt(dt)
    _call("gqa_decode_step_multi", lib.gqa_decode_step_multi,
        _ptr(q, "q", _n(b, n, h, d_k) * e), _ptr(k_new, "k_new", _n(b, n, g, d_k) * e),
        _ptr(v_new, "v_new", _n(b, n, g, d_v) * e),
        _ptr(k_cache, "k_cache", _n(b, g, cap, d_k) * e),
        _ptr(v_cache, "v_cache", _n(b, g, cap, d_v) * e),
        _ptr(seq_lens, "seq_lens", _n(b) * 4, index=True),
        int(b), int(n), int(h), int(g), int(d_k), int(d_v), float(scale),
        _ptr(out, "out", _n(b, n, h, d_v) * e), int(cap), dt, int(flags), _stream(stream))


def gqa_project_qkv(x, w_q, w_k, w_v, q, k_new, v_new, b, d_model, h, g, d_k, d_v,
                    dtype=None, flags=0, stream=None) -> None:
    """q / k_new / v_new = x . P_q / P_k / P_v ("bd,hdk->bhk" and its KV forms)."""
    dt = _dtype(x, dtype)
    e, D = _elt(dt), d_model
    _call("gqa_project_qkv", lib.gqa_project_qkv,
        _ptr(x, "x", _n(b, D) * e), _ptr(w_q, "w_q", _n(h, D, d_k) * e),
        _ptr(w_k, "w_k", _n(g, D, d_k) * e), _ptr(w_v, "w_v", _n(g, D, d_v) * e),
        _ptr(q, "q", _n(b, h, d_k) * e), _ptr(k_new, "k_new", _n(b, g, d_k) * e),
        _ptr(v_new, "v_new", _n(b, g, d_v) * e),
        int(b), int(d_model), int(h), int(g), int(d_k), int(d_v), dt, int(flags),
        _stream(stream))


def gqa_project_out(o, w_o, y, b, d_model, h, d_v, dtype=None, flags=0, stream=None) -> None:
    """y = "bhv,hdv->bd"(o, P_o)."""
    dt = _dtype(o, dtype)
    e, D = _elt(dt), d_model
    _call("gqa_project_out", lib.gqa_project_out,
        _ptr(o, "o", _n(b, h, d_v) * e), _ptr(w_o, "w_o", _n(h, D, d_v) * e),
        _ptr(y, "y", _n(b, D) * e), int(b), int(d_model), int(h), int(d_v), dt, int(flags),
        _stream(stream))


def gqa_decode_layer(x, w_q, w_k, w_v, w_o, k_cache, v_cache, seq_lens, b, d_model, h, g,
                     d_k, d_v, scale, y, cap=None, dtype=None, flags=0, stream=None) -> None:
    """The incremental layer: project x, append, attend, project the output."""
    if cap is None:
        cap = k_cache.shape[2]
    dt = _dtype(x, dtype)
    e, D = _elt(dt), d_model
    _call("gqa_decode_layer", lib.gqa_decode_layer,
        _ptr(x, "x", _n(b, D) * e), _ptr(w_q, "w_q", _n(h, D, d_k) * e),
        _ptr(w_k, "w_k", _n(g, D, d_k) * e), _ptr(w_v, "w_v", _n(g, D, d_v) * e),
        _ptr(w_o, "w_o", _n(h, D, d_v) * e), _ptr(k_cache, "k_cache", _n(b, g, cap, d_k) * e),
        _ptr(v_cache, "v_cache", _n(b, g, cap, d_v) * e),
        _ptr(seq_lens, "seq_lens", _n(b) * 4, index=True), int(b), int(d_model), int(h),
        int(g), int(d_k), int(d_v), float(scale), _ptr(y, "y", _n(b, D) * e), int(cap), dt,
        int(flags), _stream(stream))


def _paged_ptrs(k_pool, v_pool, block_table, b, g, d_k, d_v, e):
    """Checked pool and table pointers, and (block_size, max_blocks,
    num_blocks) read from the pool [num_blocks, g, block_size, d_k] and the
    table [b, max_blocks]."""
    nb, _, bs, _ = k_pool.shape
    mb = block_table.shape[1]
    return (_ptr(k_pool, "k_pool", _n(nb, g, bs, d_k) * e),
            _ptr(v_pool, "v_pool", _n(nb, g, bs, d_v) * e),
            _ptr(block_table, "block_table", _n(b, mb) * 4, index=True), int(bs), int(mb), int(nb))


def gqa_kv_append_paged(k_new, v_new, k_pool, v_pool, block_table, seq_lens, b, g, d_k, d_v,
                        n=1, dtype=None, stream=None) -> None:
    """Append n new rows per sequence into a paged cache (pools
    [num_blocks, g, block_size, d], block_table [b, max_blocks])."""
    dt = _dtype(k_pool, dtype)
    e = _elt(dt)
    kp, vp, tp, bs, mb, nb = _paged_ptrs(k_pool, v_pool, block_table, b, g, d_k, d_v, e)
    _call("gqa_kv_append_paged", lib.gqa_kv_append_paged,
        _ptr(k_new, "k_new", _n(b, n, g, d_k) * e), _ptr(v_new, "v_new", _n(b, n, g, d_v) * e),
        kp, vp, tp, _ptr(seq_lens, "seq_lens", _n(b) * 4, index=True),
        int(b), int(n), int(g), int(d_k), int(d_v), bs, mb, nb, dt, _stream(stream))


def gqa_decode_attn_paged(q, k_pool, v_pool, block_table, seq_lens, b, h, g, d_k, d_v, scale,
                          out, n=1, dtype=None, stream=None) -> None:
    """gqa_decode_attn (n = 1) or gqa_decode_attn_multi over a paged cache."""
    dt = _dtype(q, dtype)
    e = _elt(dt)
    kp, vp, tp, bs, mb, nb = _paged_ptrs(k_pool, v_pool, block_table, b, g, d_k, d_v, e)
    _call("gqa_decode_attn_paged", lib.gqa_decode_attn_paged,
        _ptr(q, "q", _n(b, n, h, d_k) * e), kp, vp, tp,
        _ptr(seq_lens, "seq_lens", _n(b) * 4, index=True), int(b), int(n),
        int(h), int(g), int(d_k), int(d_v), float(scale), _ptr(out, "out", _n(b, n, h, d_v) * e),
        bs, mb, nb, dt, _stream(stream))


def gqa_decode_step_paged(q, k_new, v_new, k_pool, v_pool, block_table, seq_lens, b, h, g, d_k,
                          d_v, scale, out, n=1, dtype=None, flags=0, stream=None) -> None:
    """Append and attend over a paged cache in one launch (n new tokens)."""
    dt = _dtype(q, dtype)
    e = _elt(dt)
    kp, vp, tp, bs, mb, nb = _paged_ptrs(k_pool, v_pool, block_table, b, g, d_k, d_v, e)
    _call("gqa_decode_step_paged", lib.gqa_decode_step_paged,
        _ptr(q, "q", _n(b, n, h, d_k) * e), _ptr(k_new, "k_new", _n(b, n, g, d_k) * e),
        _ptr(v_new, "v_new", _n(b, n, g, d_v) * e), kp, vp, tp,
        _ptr(seq_lens, "seq_lens", _n(b) * 4, index=True), int(b), int(n), int(h), int(g),
        int(d_k), int(d_v), float(scale), _ptr(out, "out", _n(b, n, h, d_v) * e), bs, mb, nb,
        dt, int(flags), _stream(stream))


_DTYPES = {"f32": GQA_F32, "bf16": GQA_BF16, "f16": GQA_F16}


def gqa_decode_plan(b, n, h, g, d_k, d_v, cap, dtype, num_sms=0, flags=0) -> dict:
    """How a decode call with these shapes runs (host only when num_sms > 0):
    kernels per call, decode CTAs, positions per tile, tensor-core kernel or
    not, split workspace bytes, CTAs per cluster (0: no clusters).  dtype:
    GQA_* code or "f32"/"bf16"/"f16"; flags: as for gqa_decode_step."""
    dt = _DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    k, c, t, tc, cl = (ctypes.c_int(0) for _ in range(5))
    ws = ctypes.c_longlong(0)
    _check("gqa_decode_plan", lib.gqa_decode_plan(
        int(b), int(n), int(h), int(g), int(d_k), int(d_v), int(cap), dt, int(flags),
        int(num_sms),
        ctypes.byref(k), ctypes.byref(c), ctypes.byref(t), ctypes.byref(tc), ctypes.byref(ws),
        ctypes.byref(cl)))
    return {"kernels": k.value, "ctas": c.value, "tile": t.value, "tensor_core": bool(tc.value),
            "workspace_bytes": ws.value, "cluster": cl.value}


def gqa_device_status(stream=None) -> int:
    """Read and clear the device status word (synchronizes the stream)."""
    bits = ctypes.c_uint32(0)
    _check("gqa_device_status", lib.gqa_device_status(_stream(stream), ctypes.byref(bits)))
    return int(bits.value)


def gqa_selftest_wait_timeout(budget_cycles: int, stream=None) -> None:
    _check("gqa_selftest_wait_timeout",
           lib.gqa_selftest_wait_timeout(int(budget_cycles), _stream(stream)))


def gqa_version() -> int:
    return int(lib.gqa_version())


def decode_step(q, k_cache, v_cache, k_new, v_new, seq_lens, g, scale, out,
                stream=None, fused=False, flags=0) -> None:
    """One layer's decode step in the order of the decode notes: push the new
    K/V rows, then attend.  fused=False makes the two C-ABI calls
    (gqa_kv_append, gqa_decode_attn); fused=True makes one gqa_decode_step."""
    b, h, d = q.shape
    if fused:
        gqa_decode_step(q, k_new, v_new, k_cache, v_cache, seq_lens, b, h, g, d,
                        v_cache.shape[-1], scale, out, flags=flags, stream=stream)
        return
    gqa_kv_append(k_new, v_new, k_cache, v_cache, seq_lens, b, g, d, v_new.shape[-1],
                  stream=stream)
    gqa_decode_attn(q, k_cache, v_cache, seq_lens, b, h, g, d, v_cache.shape[-1],
                    scale, out, stream=stream)
