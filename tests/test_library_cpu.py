"""Host-side checks of libdsa that need no GPU: the shared library builds for
sm_103a, loads, exports every function include/dsa.h declares, sizes
workspaces, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


@pytest.fixture(scope="module")
def lib():
    from top_sparse_attention_chunked_gb300 import build_lib, dsa
    build_lib.build()
    return dsa.load_library()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z_]+)\s*\(", text)))


def test_header_functions_are_exported(lib):
    names = header_functions()
    assert "dsa_sparse_attn_decode" in names and len(names) >= 10
    for n in names:
        assert hasattr(lib, n), f"{n} declared in dsa.h but not exported"


def test_binding_names_match_header():
    from top_sparse_attention_chunked_gb300 import dsa
    assert sorted(dsa.EXPORTED) == header_functions()


def test_problem_struct_matches_header():
    from top_sparse_attention_chunked_gb300.dsa import DsaProblem
    # 9 ints, 64 lengths, 1 float, 4 ints, then 3 int64 strides (8-aligned: no padding)
    assert DsaProblem.kv_strides.offset == 4 * (9 + 64 + 1 + 4)
    assert ctypes.sizeof(DsaProblem) == 4 * (9 + 64 + 1 + 4) + 8 * 3


def _prob(**kw):
    from top_sparse_attention_chunked_gb300.dsa import make_problem
    base = dict(batch=1, q_len=1, total_len=131072, top_k=2048, num_q_heads=24,
                num_kv_heads=2, kv_dtype="fp16")
    base.update(kw)
    return make_problem(**base)


def test_workspace_sizes(lib):
    from top_sparse_attention_chunked_gb300.dsa import (DSA_OP_DECODE, DSA_OP_PREFILL,
                                                        DSA_OP_TOPK, dsa_workspace_size)
    n = dsa_workspace_size(_prob(), DSA_OP_DECODE)
    # scores (512 KiB) + candidates (1 MiB) + bitmap + idx + histograms
    assert 1_500_000 < n < 4_000_000
    pre = _prob(q_len=8192, total_len=40960, kv_dtype="bf16")
    m = dsa_workspace_size(pre, DSA_OP_PREFILL)
    assert m >= 8192 * 40960 * 4            # the materialised scores
    assert dsa_workspace_size(_prob(q_len=8, total_len=262144), DSA_OP_TOPK) > 8 * 262144 * 8


@pytest.mark.parametrize("kw,frag", [
    (dict(batch=0), "batch"),
    (dict(batch=65), "batch"),
    (dict(top_k=0), "top_k"),
    (dict(top_k=200000), "top_k"),
    (dict(total_len=[131073], cache_capacity=131072), "total_len"),
    (dict(q_len=2, total_len=1, cache_capacity=16, top_k=1), "total_len"),
    (dict(num_q_heads=25), "multiple"),
    (dict(head_dim=64), "head_dim"),
    (dict(idx_heads=8), "index heads"),
    (dict(q_dtype="fp16", kv_dtype="bf16"), "FP16 query"),
    (dict(q_len=17, total_len=4096), "decode takes"),
    (dict(attn_split_keys=24), "attn_split_keys"),
])
def test_invalid_problems_rejected_on_host(lib, kw, frag):
    from top_sparse_attention_chunked_gb300.dsa import DSA_OP_DECODE
    p = _prob(**kw)
    assert lib.dsa_workspace_size(ctypes.byref(p), DSA_OP_DECODE) == 0
    assert frag in lib.dsa_last_error_string().decode()


def _call_decode(lib, p, ws_bytes, ptrs=None, ws=0x10000):
    a = ptrs or {}
    vals = [a.get(n, 0x1000) for n in ("q", "qI", "w", "kI", "k", "v")]
    return lib.dsa_sparse_attn_decode(ctypes.byref(p), *[ctypes.c_void_p(v) for v in vals],
                                      ctypes.c_void_p(a.get("ks")), ctypes.c_void_p(a.get("vs")),
                                      None, ctypes.c_void_p(a.get("out", 0x2000)),
                                      ctypes.c_void_p(ws), ws_bytes, None)


def test_bad_pointers_rejected_before_cuda(lib):
    from top_sparse_attention_chunked_gb300.dsa import (DSA_ERR_INVALID_ARG, DSA_ERR_MISALIGNED,
                                                        DSA_ERR_WORKSPACE, DSA_OP_DECODE)
    p = _prob()
    need = lib.dsa_workspace_size(ctypes.byref(p), DSA_OP_DECODE)
    assert _call_decode(lib, p, need, {"q": 0}) == DSA_ERR_INVALID_ARG
    assert _call_decode(lib, p, need, {"kI": 0x1008}) == DSA_ERR_MISALIGNED
    assert _call_decode(lib, p, need - 1) == DSA_ERR_WORKSPACE
    assert _call_decode(lib, p, need, ws=0x10010) == DSA_ERR_WORKSPACE
    # scales only with an INT8 cache
    assert _call_decode(lib, p, need, {"ks": 0x3000, "vs": 0x3000}) == DSA_ERR_INVALID_ARG
    p8 = _prob(kv_dtype="int8")
    need8 = lib.dsa_workspace_size(ctypes.byref(p8), DSA_OP_DECODE)
    assert _call_decode(lib, p8, need8) == DSA_ERR_INVALID_ARG


def test_valid_call_without_gpu_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from top_sparse_attention_chunked_gb300.dsa import DSA_ERR_NO_DEVICE, DSA_OP_DECODE
    p = _prob()
    need = lib.dsa_workspace_size(ctypes.byref(p), DSA_OP_DECODE)
    assert _call_decode(lib, p, need) == DSA_ERR_NO_DEVICE


def test_status_strings(lib):
    assert lib.dsa_status_string(0) == b"DSA_OK"
    assert lib.dsa_status_string(6) == b"DSA_ERR_TIMEOUT"
    assert lib.dsa_version() >= 100


def _call_append(lib, p, ptrs=None):
    a = {"kI_new": 0x1000, "k_new": 0x10000, "v_new": 0x20000, "kI": 0x100000,
         "k": 0x1000000, "v": 0x2000000}
    a.update(ptrs or {})
    vals = [a[n] for n in ("kI_new", "k_new", "v_new", "kI", "k", "v")]
    return lib.dsa_cache_append(ctypes.byref(p), *[ctypes.c_void_p(v) for v in vals],
                                ctypes.c_void_p(a.get("ks")), ctypes.c_void_p(a.get("vs")), None)


def test_cache_append_rejects_bad_arguments_before_cuda(lib):
    from top_sparse_attention_chunked_gb300.dsa import (DSA_ERR_INVALID_ARG, DSA_ERR_MISALIGNED,
                                                        DSA_ERR_UNSUPPORTED)
    p = _prob(q_len=4, total_len=64, cache_capacity=64, top_k=8)   # 2 KV heads, FP16 cache
    assert _call_append(lib, p, {"k_new": 0}) == DSA_ERR_INVALID_ARG
    assert _call_append(lib, p, {"v": 0x2000008}) == DSA_ERR_MISALIGNED
    assert _call_append(lib, p, {"ks": 0x3000000, "vs": 0x3001000}) == DSA_ERR_INVALID_ARG
    # new K rows (4 x 2 x 256 B = 2 KiB from 0x10000) overlapping the V cache
    assert _call_append(lib, p, {"v": 0x10400}) == DSA_ERR_INVALID_ARG
    assert "overlaps" in lib.dsa_last_error_string().decode()
    # adjacent but disjoint is fine up to the device check
    p8 = _prob(q_len=4, total_len=64, cache_capacity=64, top_k=8, kv_dtype="int8")
    assert _call_append(lib, p8) == DSA_ERR_INVALID_ARG                 # scales missing
    assert _call_append(lib, p8, {"ks": 0x3000000, "vs": 0x3000002}) == DSA_ERR_MISALIGNED
    assert _call_append(lib, _prob(q_len=65, total_len=64, cache_capacity=64, top_k=8)) \
        == DSA_ERR_INVALID_ARG                                          # q_len > total_len
    assert _call_append(lib, _prob(q_len=4, total_len=64, cache_capacity=64, top_k=8,
                                   q_dtype="fp16", kv_dtype="bf16")) == DSA_ERR_UNSUPPORTED


def test_cache_append_without_gpu_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from top_sparse_attention_chunked_gb300.dsa import DSA_ERR_NO_DEVICE
    p = _prob(q_len=4, total_len=64, cache_capacity=64, top_k=8)
    assert _call_append(lib, p, {"v_new": 0x10800}) == DSA_ERR_NO_DEVICE


def _pages(bs=256, nb=1037, per_seq=1024, table=0x40000):
    from top_sparse_attention_chunked_gb300.dsa import DsaKvPages
    return DsaKvPages(bs, nb, per_seq, table)


def _call_decode_paged(lib, p, pg, ws_bytes, ws=0x10000):
    vals = [0x1000] * 6
    return lib.dsa_sparse_attn_decode_paged(ctypes.byref(p), ctypes.byref(pg) if pg else None,
                                            *[ctypes.c_void_p(v) for v in vals], None, None, None,
                                            ctypes.c_void_p(0x2000), ctypes.c_void_p(ws),
                                            ws_bytes, None)


@pytest.mark.parametrize("pg_kw,status,frag", [
    (dict(bs=100, per_seq=1311), 2, "power of two"),
    (dict(bs=64, per_seq=2048), 2, "power of two"),
    (dict(nb=0), 1, "num_blocks"),
    (dict(per_seq=1000), 1, "blocks_per_seq * block_size"),
    (dict(table=0), 1, "block_table is NULL"),
    (dict(table=0x40002), 4, "4-byte aligned"),
    (dict(nb=1 << 22), 2, "below 2^31"),
])
def test_paged_descriptor_rejected_on_host(lib, pg_kw, status, frag):
    from top_sparse_attention_chunked_gb300.dsa import DSA_OP_DECODE
    p = _prob(q_len=8, total_len=262144, kv_dtype="int8")
    need = lib.dsa_workspace_size(ctypes.byref(p), DSA_OP_DECODE)
    assert _call_decode_paged(lib, p, _pages(**pg_kw), need) == status
    assert frag in lib.dsa_last_error_string().decode()


def test_paged_calls_need_a_descriptor(lib):
    from top_sparse_attention_chunked_gb300.dsa import DSA_ERR_INVALID_ARG, DSA_OP_DECODE
    p = _prob(q_len=8, total_len=262144, kv_dtype="int8")
    need = lib.dsa_workspace_size(ctypes.byref(p), DSA_OP_DECODE)
    assert _call_decode_paged(lib, p, None, need) == DSA_ERR_INVALID_ARG
    assert lib.dsa_cache_append_paged(ctypes.byref(p), None, *([None] * 9)) == DSA_ERR_INVALID_ARG
    assert lib.dsa_index_scores_paged(ctypes.byref(p), None, None, None, None, None, None, 0,
                                      None) == DSA_ERR_INVALID_ARG


def test_paged_valid_call_without_gpu_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from top_sparse_attention_chunked_gb300.dsa import DSA_ERR_NO_DEVICE, DSA_OP_DECODE
    p = _prob(q_len=8, total_len=262144, kv_dtype="int8")
    need = lib.dsa_workspace_size(ctypes.byref(p), DSA_OP_DECODE)
    vals = [0x1000] * 6
    rc = lib.dsa_sparse_attn_decode_paged(ctypes.byref(p), ctypes.byref(_pages()),
                                          *[ctypes.c_void_p(v) for v in vals],
                                          ctypes.c_void_p(0x3000), ctypes.c_void_p(0x3000), None,
                                          ctypes.c_void_p(0x2000), ctypes.c_void_p(0x10000), need,
                                          None)
    assert rc == DSA_ERR_NO_DEVICE


def _rope(**kw):
    from top_sparse_attention_chunked_gb300.dsa import DsaRopeProblem
    base = dict(tokens=16, heads=4, head_dim=128, rotary_dim=128, max_pos=64, eps=1e-6,
                x_dtype=0, cos_dtype=3, y_dtype=0)
    base.update(kw)
    return DsaRopeProblem(**base)


def _call_rope(lib, rp, x=0x10000, y=0x20000):
    vp = ctypes.c_void_p
    return lib.dsa_rmsnorm_rotary(ctypes.byref(rp) if rp is not None else None, vp(x), vp(0x3000),
                                  vp(0x4000), vp(0x5000), vp(0x6000), vp(y), None)


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), 2), (dict(rotary_dim=7), 1), (dict(rotary_dim=130), 1),
    (dict(eps=-1.0), 1), (dict(heads=0), 1), (dict(tokens=-1), 1), (dict(max_pos=0), 1),
    (dict(x_dtype=2), 2), (dict(cos_dtype=1), 2),
])
def test_rmsnorm_rotary_rejects_bad_problems(lib, kw, status):
    assert _call_rope(lib, _rope(**kw)) == status


def test_rmsnorm_rotary_pointer_rules(lib):
    from top_sparse_attention_chunked_gb300.dsa import (DSA_ERR_INVALID_ARG, DSA_ERR_MISALIGNED)
    assert _call_rope(lib, None) == DSA_ERR_INVALID_ARG
    assert _call_rope(lib, _rope(), x=0x10008) == DSA_ERR_MISALIGNED
    # 16 x 4 x 128 bf16 = 16 KiB: y starting inside x overlaps it
    assert _call_rope(lib, _rope(), y=0x10000 + 0x2000) == DSA_ERR_INVALID_ARG
    assert "overlaps" in lib.dsa_last_error_string().decode()


def test_rmsnorm_rotary_in_place_and_empty_pass_host_checks(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from top_sparse_attention_chunked_gb300.dsa import DSA_ERR_NO_DEVICE
    assert _call_rope(lib, _rope(), y=0x10000) == DSA_ERR_NO_DEVICE      # in place is allowed
    assert _call_rope(lib, _rope(tokens=0)) == DSA_ERR_NO_DEVICE


def _rope_params(**kw):
    from top_sparse_attention_chunked_gb300.dsa import DsaRopeParams
    base = dict(eps=1e-6, max_pos=64, cos_dtype=3, rotary_dim=128, rotary_dim_index=64,
                cos=0x7000, sin=0x7100, cos_index=0x7200, sin_index=0x7300, gamma_q=0x7400,
                gamma_k=0x7500, gamma_qI=0x7600, gamma_kI=0x7700)
    base.update(kw)
    return DsaRopeParams(**base)


def _call_rope_append(lib, p, rp, ks=None, vs=None):
    vp = ctypes.c_void_p
    ptrs = [0x100000, 0x200000, 0x300000, 0x400000, 0x500000, 0x1000000, 0x2000000, 0x3000000]
    return lib.dsa_rope_append(ctypes.byref(p), ctypes.byref(rp) if rp is not None else None,
                               *[vp(x) for x in ptrs], vp(ks), vp(vs), None)


@pytest.mark.parametrize("kw", [dict(rotary_dim=130), dict(rotary_dim_index=66), dict(rotary_dim=3),
                                dict(gamma_k=0), dict(cos=0), dict(sin_index=0), dict(eps=-1.0),
                                dict(max_pos=0)])
def test_rope_append_rejects_bad_parameters(lib, kw):
    from top_sparse_attention_chunked_gb300.dsa import DSA_ERR_INVALID_ARG
    p = _prob(q_len=4, total_len=64, cache_capacity=64, top_k=8)
    assert _call_rope_append(lib, p, _rope_params(**kw)) == DSA_ERR_INVALID_ARG


def test_rope_append_host_rules(lib):
    import torch
    from top_sparse_attention_chunked_gb300.dsa import DSA_ERR_INVALID_ARG, DSA_ERR_NO_DEVICE
    p = _prob(q_len=4, total_len=64, cache_capacity=64, top_k=8)
    assert _call_rope_append(lib, p, None) == DSA_ERR_INVALID_ARG
    assert _call_rope_append(lib, p, _rope_params(), ks=0x4000000) == DSA_ERR_INVALID_ARG  # FP16 cache
    p8 = _prob(q_len=4, total_len=64, cache_capacity=64, top_k=8, kv_dtype="int8")
    assert _call_rope_append(lib, p8, _rope_params()) == DSA_ERR_INVALID_ARG              # scales missing
    if not torch.cuda.is_available():
        assert _call_rope_append(lib, p, _rope_params()) == DSA_ERR_NO_DEVICE
