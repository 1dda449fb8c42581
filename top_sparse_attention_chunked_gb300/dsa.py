"""Python binding of libdsa (argument marshalling only).

Every function here has the name of the C entry point it calls and does no
arithmetic of its own: it checks that the tensors it is handed are contiguous
CUDA tensors of the dtype and shape the problem implies, passes their device
pointers and PyTorch's current stream to the C ABI, and raises DsaError on a
non-zero status. There is no fallback: if libdsa.so is missing the first call
raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")

# mirrors include/dsa.h
DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_WORKSPACE = 0, 1, 2, 3
DSA_ERR_MISALIGNED, DSA_ERR_CUDA, DSA_ERR_TIMEOUT, DSA_ERR_NO_DEVICE = 4, 5, 6, 7
DSA_BF16, DSA_FP16, DSA_INT8, DSA_FP32 = 0, 1, 2, 3
DSA_OP_INDEX_SCORES, DSA_OP_TOPK, DSA_OP_DECODE, DSA_OP_PREFILL = 0, 1, 2, 3
DSA_MAX_BATCH = 64
DSA_KERNEL_INDEXER, DSA_KERNEL_TOPK_HIST, DSA_KERNEL_TOPK_SELECT = 0, 1, 2
DSA_KERNEL_TOPK_ROW, DSA_KERNEL_ATTENTION, DSA_KERNEL_APPEND = 3, 4, 5

EXPORTED = ["dsa_workspace_size", "dsa_index_scores", "dsa_topk",
            "dsa_sparse_attn_decode", "dsa_sparse_attn_prefill",
            "dsa_read_device_status", "dsa_last_error_string", "dsa_status_string",
            "dsa_version", "dsa_timing_select", "dsa_timing_read", "dsa_topk_noalloc",
            "dsa_last_launches", "dsa_cache_append", "dsa_index_scores_paged",
            "dsa_sparse_attn_decode_paged", "dsa_sparse_attn_prefill_paged",
            "dsa_cache_append_paged", "dsa_rmsnorm_rotary", "dsa_rope_append",
            "dsa_sparse_attn_decode_aux", "dsa_set_wait_budget"]

_DT = {"bf16": DSA_BF16, "fp16": DSA_FP16, "int8": DSA_INT8, "fp32": DSA_FP32}
_TORCH_DT = {DSA_BF16: torch.bfloat16, DSA_FP16: torch.float16, DSA_INT8: torch.int8,
             DSA_FP32: torch.float32}


class DsaKvPages(ctypes.Structure):
    """dsa_kv_pages: a paged kI / K / V pool and its device block table."""
    _fields_ = [
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("blocks_per_seq", ctypes.c_int32),
        ("block_table", ctypes.c_void_p),
    ]


class DsaRopeProblem(ctypes.Structure):
    """dsa_rope_problem (RMSNorm + rotary embedding)."""
    _fields_ = [
        ("tokens", ctypes.c_int64),
        ("heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("rotary_dim", ctypes.c_int32),
        ("max_pos", ctypes.c_int32),
        ("eps", ctypes.c_float),
        ("x_dtype", ctypes.c_int32),
        ("cos_dtype", ctypes.c_int32),
        ("y_dtype", ctypes.c_int32),
    ]


class DsaRopeParams(ctypes.Structure):
    """dsa_rope_params (the rope half of dsa_rope_append)."""
    _fields_ = [
        ("eps", ctypes.c_float),
        ("max_pos", ctypes.c_int32),
        ("cos_dtype", ctypes.c_int32),
        ("rotary_dim", ctypes.c_int32),
        ("rotary_dim_index", ctypes.c_int32),
        ("cos", ctypes.c_void_p),
        ("sin", ctypes.c_void_p),
        ("cos_index", ctypes.c_void_p),
        ("sin_index", ctypes.c_void_p),
        ("gamma_q", ctypes.c_void_p),
        ("gamma_k", ctypes.c_void_p),
        ("gamma_qI", ctypes.c_void_p),
        ("gamma_kI", ctypes.c_void_p),
    ]


class DsaProblem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("q_len", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("idx_heads", ctypes.c_int32),
        ("idx_dim", ctypes.c_int32),
        ("cache_capacity", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("total_len", ctypes.c_int32 * DSA_MAX_BATCH),
        ("softmax_scale", ctypes.c_float),
        ("q_dtype", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("out_dtype", ctypes.c_int32),
        ("attn_split_keys", ctypes.c_int32),
        ("kv_strides", ctypes.c_int64 * 3),
    ]


class DsaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} (status {status})")
        self.status = status


_lib = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libdsa.so (built in-tree by build_lib.build()); raise if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    # DSA_LIBRARY names another build of the library (e.g. libdsa_debug.so)
    p = path or os.environ.get("DSA_LIBRARY") or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libdsa.so not found at {p}: build it with "
                           "top_sparse_attention_chunked_gb300.build_lib.build()")
    lib = ctypes.CDLL(p)
    vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    P = ctypes.POINTER(DsaProblem)
    PG = ctypes.POINTER(DsaKvPages)
    sig = {
        "dsa_workspace_size": (sz, [P, i32]),
        "dsa_index_scores": (i32, [P, vp, vp, vp, vp, vp, sz, vp]),
        "dsa_topk": (i32, [P, vp, vp, vp, sz, vp]),
        "dsa_sparse_attn_decode": (i32, [P] + [vp] * 11 + [sz, vp]),
        "dsa_sparse_attn_prefill": (i32, [P] + [vp] * 11 + [sz, vp]),
        "dsa_sparse_attn_decode_aux": (i32, [P] + [vp] * 13 + [sz, vp]),
        "dsa_set_wait_budget": (i32, [ctypes.c_longlong]),
        "dsa_read_device_status": (i32, [vp, sz, vp, ctypes.POINTER(ctypes.c_uint32)]),
        "dsa_last_error_string": (ctypes.c_char_p, []),
        "dsa_status_string": (ctypes.c_char_p, [i32]),
        "dsa_version": (i32, []),
        "dsa_last_launches": (i32, [ctypes.c_char_p, ctypes.c_size_t]),
        "dsa_timing_select": (i32, [i32]),
        "dsa_timing_read": (i32, [ctypes.POINTER(ctypes.c_float)]),
        "dsa_topk_noalloc": (i32, [P, vp, vp, vp]),
        "dsa_cache_append": (i32, [P] + [vp] * 9),
        "dsa_index_scores_paged": (i32, [P, PG, vp, vp, vp, vp, vp, sz, vp]),
        "dsa_sparse_attn_decode_paged": (i32, [P, PG] + [vp] * 11 + [sz, vp]),
        "dsa_sparse_attn_prefill_paged": (i32, [P, PG] + [vp] * 11 + [sz, vp]),
        "dsa_cache_append_paged": (i32, [P, PG] + [vp] * 9),
        "dsa_rmsnorm_rotary": (i32, [ctypes.POINTER(DsaRopeProblem)] + [vp] * 7),
        "dsa_rope_append": (i32, [P, ctypes.POINTER(DsaRopeParams)] + [vp] * 11),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _check(status: int):
    if status != DSA_OK:
        lib = load_library()
        raise DsaError(status, lib.dsa_last_error_string().decode())


def make_problem(batch: int, q_len: int, total_len: Sequence[int] | int, top_k: int,
                 num_q_heads: int = 24, num_kv_heads: int = 2, cache_capacity: Optional[int] = None,
                 q_dtype="bf16", kv_dtype="bf16", out_dtype=None, softmax_scale: float = 0.0,
                 head_dim: int = 128, idx_heads: int = 16, idx_dim: int = 64,
                 attn_split_keys: int = 0, kv_strides: Optional[Sequence[int]] = None) -> DsaProblem:
    """Fill a DsaProblem; dtypes by name ('bf16', 'fp16', 'int8', 'fp32');
    kv_strides: the K / V caches' (batch, token, head) strides in elements
    (None: the default token-major layout)."""
    if isinstance(total_len, int):
        total_len = [total_len] * max(1, min(batch, DSA_MAX_BATCH))
    p = DsaProblem()
    p.batch, p.q_len = batch, q_len
    p.num_q_heads, p.num_kv_heads, p.head_dim = num_q_heads, num_kv_heads, head_dim
    p.idx_heads, p.idx_dim = idx_heads, idx_dim
    p.cache_capacity = cache_capacity if cache_capacity is not None else max(total_len)
    p.top_k = top_k
    for b, t in enumerate(list(total_len)[:DSA_MAX_BATCH]):
        p.total_len[b] = int(t)
    p.softmax_scale = softmax_scale
    p.q_dtype = _DT[q_dtype]
    p.kv_dtype = _DT[kv_dtype]
    p.out_dtype = _DT[out_dtype if out_dtype is not None else q_dtype]
    p.attn_split_keys = attn_split_keys
    if kv_strides is not None:
        for i, v in enumerate(kv_strides):
            p.kv_strides[i] = int(v)
    return p


def problem_for(wl, **overrides) -> DsaProblem:
    """DsaProblem of a dsa_inputs.Workload."""
    kw = dict(batch=wl.batch, q_len=wl.q_len, total_len=wl.total_len, top_k=wl.top_k,
              num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
              cache_capacity=wl.cap, q_dtype=wl.q_dtype, kv_dtype=wl.kv_dtype,
              head_dim=wl.head_dim, idx_heads=wl.idx_heads, idx_dim=wl.idx_dim)
    kw.update(overrides)
    return make_problem(**kw)


def _ptr(t: Optional[torch.Tensor], name: str, dtype=None, shape=None):
    """The device address of a checked tensor (an int; ctypes passes it as a
    void pointer). The checks are ordered and written for a low per-call cost:
    the step calls run once per layer and token."""
    if t is None:
        return None
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and t.shape != shape:
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int:
    """The CUDA stream to enqueue on: the given one, else the current stream
    of the current device (read without building a stream object)."""
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def dsa_workspace_size(p: DsaProblem, op: int) -> int:
    lib = load_library()
    n = lib.dsa_workspace_size(ctypes.byref(p), op)
    if n == 0:
        raise DsaError(DSA_ERR_INVALID_ARG, lib.dsa_last_error_string().decode())
    return n


def alloc_workspace(p: DsaProblem, op: int, device="cuda") -> torch.Tensor:
    """Caller-owned workspace (torch allocations are 256-byte aligned)."""
    return torch.empty(dsa_workspace_size(p, op), dtype=torch.uint8, device=device)


def _ws(ws: torch.Tensor):
    return _ptr(ws, "workspace", torch.uint8), ws.numel()


def make_pages(block_table: torch.Tensor, block_size: int, num_blocks: int) -> DsaKvPages:
    """A dsa_kv_pages for a device int32 block table [B, blocks_per_seq]
    (the table tensor is kept alive by the returned object)."""
    _ptr(block_table, "block_table", torch.int32)
    if block_table.dim() != 2:
        raise ValueError("block_table must be [B, blocks_per_seq]")
    pg = DsaKvPages(block_size, num_blocks, block_table.shape[1], block_table.data_ptr())
    pg._table = block_table
    return pg


def _kv_ptr(p: DsaProblem, t, name, dtype, shape):
    """A K / V cache pointer: the default layout is checked by shape; with
    kv_strides the tensor only has to be contiguous and hold the last row."""
    st = p.kv_strides
    if not (st[0] or st[1] or st[2]):
        return _ptr(t, name, dtype, shape)
    ptr = _ptr(t, name, dtype)
    last = (p.batch - 1) * st[0] + (p.cache_capacity - 1) * st[1] + (p.num_kv_heads - 1) * st[2] + 128
    if t.numel() < last:
        raise ValueError(f"{name} holds {t.numel()} elements, the strides reach {last}")
    return ptr


def _cache_shapes(p: DsaProblem, pages: Optional[DsaKvPages]):
    """Leading dims of the kI / K / V / scale arrays: [B, cap] or the pool."""
    if pages is None:
        return (p.batch, p.cache_capacity)
    return (pages.num_blocks * pages.block_size,)


def dsa_index_scores(p: DsaProblem, qI, w, kI, scores, workspace, stream=None, pages=None):
    B, S, cap = p.batch, p.q_len, p.cache_capacity
    lib = load_library()
    wp, wn = _ws(workspace)
    lead = _cache_shapes(p, pages)
    args = [ctypes.byref(p), _ptr(qI, "qI", torch.bfloat16, (B, S, 16, 64)),
            _ptr(w, "w", torch.float32, (B, S, 16)), _ptr(kI, "kI", torch.bfloat16, lead + (64,)),
            _ptr(scores, "scores", torch.float32, (B, S, cap)), wp, wn, _stream(stream)]
    if pages is None:
        _check(lib.dsa_index_scores(*args))
    else:
        _check(lib.dsa_index_scores_paged(args[0], ctypes.byref(pages), *args[1:]))


def dsa_topk(p: DsaProblem, scores, idx, workspace, stream=None):
    B, S, cap = p.batch, p.q_len, p.cache_capacity
    lib = load_library()
    wp, wn = _ws(workspace)
    _check(lib.dsa_topk(ctypes.byref(p), _ptr(scores, "scores", torch.float32, (B, S, cap)),
                        _ptr(idx, "idx", torch.int32, (B, S, p.top_k)), wp, wn, _stream(stream)))


def dsa_topk_noalloc(p: DsaProblem, scores, idx, stream=None):
    """dsa_topk without a workspace, for callers that cannot allocate device
    memory (the library keeps the scratch in a static device array; at most
    8 query rows of at most 131,072 visible keys). Every call shares that one
    array: calls that could overlap on the GPU (other streams or threads)
    must be serialised by the caller."""
    B, S, cap = p.batch, p.q_len, p.cache_capacity
    lib = load_library()
    _check(lib.dsa_topk_noalloc(ctypes.byref(p),
                                _ptr(scores, "scores", torch.float32, (B, S, cap)),
                                _ptr(idx, "idx", torch.int32, (B, S, p.top_k)), _stream(stream)))


def dsa_cache_append(p: DsaProblem, kI_new, k_new, v_new, kI, k, v, k_scale=None,
                     v_scale=None, stream=None, pages=None):
    """Write the q_len new tokens of every sequence into cache rows
    total_len[b]-q_len .. total_len[b]-1 (INT8 caches: quantised on write);
    with `pages` (make_pages) the caches are paged pools."""
    B, S, Hkv = p.batch, p.q_len, p.num_kv_heads
    lib = load_library()
    qdt, kvdt = _TORCH_DT[p.q_dtype], _TORCH_DT[p.kv_dtype]
    lead = _cache_shapes(p, pages)
    args = [_ptr(kI_new, "kI_new", torch.bfloat16, (B, S, 64)),
            _ptr(k_new, "k_new", qdt, (B, S, Hkv, 128)), _ptr(v_new, "v_new", qdt, (B, S, Hkv, 128)),
            _ptr(kI, "kI", torch.bfloat16, lead + (64,)), _ptr(k, "k", kvdt, lead + (Hkv, 128)),
            _ptr(v, "v", kvdt, lead + (Hkv, 128)),
            _ptr(k_scale, "k_scale", torch.float32, lead + (Hkv,)),
            _ptr(v_scale, "v_scale", torch.float32, lead + (Hkv,)), _stream(stream)]
    if pages is None:
        _check(lib.dsa_cache_append(ctypes.byref(p), *args))
    else:
        _check(lib.dsa_cache_append_paged(ctypes.byref(p), ctypes.byref(pages), *args))


def dsa_rmsnorm_rotary(x, gamma, y, eps=1e-6, cos_cache=None, sin_cache=None, positions=None,
                       rotary_dim=None, stream=None):
    """RMSNorm + rotary embedding of x [N, H, D] (BF16/FP16) into y (BF16/FP16,
    may be x); gamma [D] fp32; cos / sin caches [max_pos, rotary_dim / 2] in
    fp32 or bf16 with positions [N] int32 (omit all three for RMSNorm only)."""
    lib = load_library()
    if x.dim() != 3:
        raise ValueError("x must be [tokens, heads, head_dim]")
    N, H, D = x.shape
    r = 0 if cos_cache is None else (rotary_dim if rotary_dim is not None else 2 * cos_cache.shape[1])
    inv = {v: k for k, v in _TORCH_DT.items()}
    rp = DsaRopeProblem(N, H, D, r, 0 if cos_cache is None else cos_cache.shape[0], eps,
                        inv[x.dtype], inv[cos_cache.dtype] if cos_cache is not None else DSA_FP32,
                        inv[y.dtype])
    if cos_cache is not None and tuple(cos_cache.shape) != (cos_cache.shape[0], r // 2):
        raise ValueError("cos_cache must be [max_pos, rotary_dim / 2]")
    _check(lib.dsa_rmsnorm_rotary(
        ctypes.byref(rp), _ptr(x, "x", None, (N, H, D)), _ptr(gamma, "gamma", torch.float32, (D,)),
        _ptr(cos_cache, "cos_cache"), _ptr(sin_cache, "sin_cache", cos_cache.dtype if cos_cache is not None else None,
                                         tuple(cos_cache.shape) if cos_cache is not None else None),
        _ptr(positions, "positions", torch.int32, (N,)), _ptr(y, "y", None, (N, H, D)),
        _stream(stream)))


def dsa_rope_append(p: DsaProblem, q, qI, k_new, kI_new, v_new, kI, k, v, k_scale, v_scale,
                    gamma_q, gamma_k, gamma_qI, gamma_kI, eps=1e-6, cos=None, sin=None,
                    cos_index=None, sin_index=None, stream=None):
    """RMSNorm + RoPE of q, qI (in place), k_new, kI_new and the cache append
    of kI, k, v in one launch (positions total_len[b] - q_len + s)."""
    B, S, Hq, Hkv, cap = p.batch, p.q_len, p.num_q_heads, p.num_kv_heads, p.cache_capacity
    lib = load_library()
    qdt, kvdt = _TORCH_DT[p.q_dtype], _TORCH_DT[p.kv_dtype]
    caches = [c for c in (cos, cos_index) if c is not None]
    cdt = {torch.float32: DSA_FP32, torch.bfloat16: DSA_BF16}[caches[0].dtype] if caches else DSA_FP32
    rp = DsaRopeParams(eps, caches[0].shape[0] if caches else 0, cdt,
                       0 if cos is None else 2 * cos.shape[1],
                       0 if cos_index is None else 2 * cos_index.shape[1],
                       None if cos is None else cos.data_ptr(), None if sin is None else sin.data_ptr(),
                       None if cos_index is None else cos_index.data_ptr(),
                       None if sin_index is None else sin_index.data_ptr(),
                       _ptr(gamma_q, "gamma_q", torch.float32, (128,)),
                       _ptr(gamma_k, "gamma_k", torch.float32, (128,)),
                       _ptr(gamma_qI, "gamma_qI", torch.float32, (64,)),
                       _ptr(gamma_kI, "gamma_kI", torch.float32, (64,)))
    for t, n in ((cos, "cos"), (sin, "sin"), (cos_index, "cos_index"), (sin_index, "sin_index")):
        _ptr(t, n)
    _check(lib.dsa_rope_append(
        ctypes.byref(p), ctypes.byref(rp), _ptr(q, "q", qdt, (B, S, Hq, 128)),
        _ptr(qI, "qI", torch.bfloat16, (B, S, 16, 64)), _ptr(k_new, "k_new", qdt, (B, S, Hkv, 128)),
        _ptr(kI_new, "kI_new", torch.bfloat16, (B, S, 64)), _ptr(v_new, "v_new", qdt, (B, S, Hkv, 128)),
        _ptr(kI, "kI", torch.bfloat16, (B, cap, 64)), _ptr(k, "k", kvdt, (B, cap, Hkv, 128)),
        _ptr(v, "v", kvdt, (B, cap, Hkv, 128)), _ptr(k_scale, "k_scale", torch.float32, (B, cap, Hkv)),
        _ptr(v_scale, "v_scale", torch.float32, (B, cap, Hkv)), _stream(stream)))


def _attn(fn_name, p, q, qI, w, kI, k, v, k_scale, v_scale, idx_out, out, workspace, stream,
          pages=None):
    B, S, Hq, Hkv = p.batch, p.q_len, p.num_q_heads, p.num_kv_heads
    lib = load_library()
    wp, wn = _ws(workspace)
    kvdt = _TORCH_DT[p.kv_dtype]
    lead = _cache_shapes(p, pages)
    args = [
        _ptr(q, "q", _TORCH_DT[p.q_dtype], (B, S, Hq, 128)),
        _ptr(qI, "qI", torch.bfloat16, (B, S, 16, 64)),
        _ptr(w, "w", torch.float32, (B, S, 16)),
        _ptr(kI, "kI", torch.bfloat16, lead + (64,)),
        _kv_ptr(p, k, "k", kvdt, lead + (Hkv, 128)),
        _kv_ptr(p, v, "v", kvdt, lead + (Hkv, 128)),
        _ptr(k_scale, "k_scale", torch.float32, lead + (Hkv,)),
        _ptr(v_scale, "v_scale", torch.float32, lead + (Hkv,)),
        _ptr(idx_out, "idx_out", torch.int32, (B, S, p.top_k)),
        _ptr(out, "out", _TORCH_DT[p.out_dtype], (B, S, Hq, 128)),
        wp, wn, _stream(stream),
    ]
    if pages is None:
        _check(getattr(lib, fn_name)(ctypes.byref(p), *args))
    else:
        _check(getattr(lib, fn_name + "_paged")(ctypes.byref(p), ctypes.byref(pages), *args))


def dsa_sparse_attn_decode(p, q, qI, w, kI, k, v, k_scale, v_scale, idx_out, out, workspace,
                           stream=None, pages=None):
    _attn("dsa_sparse_attn_decode", p, q, qI, w, kI, k, v, k_scale, v_scale, idx_out, out,
          workspace, stream, pages)


def dsa_sparse_attn_decode_aux(p, q, qI, w, kI, k, v, k_scale, v_scale, k_aux, v_aux, idx_out,
                               out, workspace, stream=None):
    """dsa_sparse_attn_decode with the new tokens' own K / V rows k_aux, v_aux
    [B, S, Hkv, 128] in the query dtype (read at their values for selected
    keys at or after each sequence's first new token)."""
    B, S, Hq, Hkv = p.batch, p.q_len, p.num_q_heads, p.num_kv_heads
    lib = load_library()
    wp, wn = _ws(workspace)
    kvdt = _TORCH_DT[p.kv_dtype]
    qdt = _TORCH_DT[p.q_dtype]
    lead = _cache_shapes(p, None)
    _check(lib.dsa_sparse_attn_decode_aux(
        ctypes.byref(p),
        _ptr(q, "q", qdt, (B, S, Hq, 128)),
        _ptr(qI, "qI", torch.bfloat16, (B, S, 16, 64)),
        _ptr(w, "w", torch.float32, (B, S, 16)),
        _ptr(kI, "kI", torch.bfloat16, lead + (64,)),
        _kv_ptr(p, k, "k", kvdt, lead + (Hkv, 128)),
        _kv_ptr(p, v, "v", kvdt, lead + (Hkv, 128)),
        _ptr(k_scale, "k_scale", torch.float32, lead + (Hkv,)),
        _ptr(v_scale, "v_scale", torch.float32, lead + (Hkv,)),
        _ptr(k_aux, "k_aux", qdt, (B, S, Hkv, 128)),
        _ptr(v_aux, "v_aux", qdt, (B, S, Hkv, 128)),
        _ptr(idx_out, "idx_out", torch.int32, (B, S, p.top_k)),
        _ptr(out, "out", _TORCH_DT[p.out_dtype], (B, S, Hq, 128)),
        wp, wn, _stream(stream)))


def dsa_sparse_attn_prefill(p, q, qI, w, kI, k, v, k_scale, v_scale, idx_out, out, workspace,
                            stream=None, pages=None):
    _attn("dsa_sparse_attn_prefill", p, q, qI, w, kI, k, v, k_scale, v_scale, idx_out, out,
          workspace, stream, pages)


def dsa_read_device_status(workspace, stream=None) -> int:
    lib = load_library()
    wp, wn = _ws(workspace)
    st = ctypes.c_uint32(0)
    _check(lib.dsa_read_device_status(wp, wn, _stream(stream), ctypes.byref(st)))
    return st.value


def dsa_set_wait_budget(cycles: int):
    """Budget of the indexer's pipeline waits for this thread's later calls
    (SM cycles; negative: the default)."""
    _check(load_library().dsa_set_wait_budget(int(cycles)))


def dsa_timing_select(kind: int):
    _check(load_library().dsa_timing_select(kind))


def dsa_timing_read() -> float:
    ms = ctypes.c_float(0.0)
    _check(load_library().dsa_timing_read(ctypes.byref(ms)))
    return ms.value


def dsa_last_launches() -> list:
    """Names of the kernels the last library call on this thread enqueued."""
    buf = ctypes.create_string_buffer(1024)
    n = load_library().dsa_last_launches(buf, len(buf))
    names = [x for x in buf.value.decode().split(",") if x]
    return names if len(names) == n else names + ["?"] * (n - len(names))


def dsa_version() -> int:
    return load_library().dsa_version()
