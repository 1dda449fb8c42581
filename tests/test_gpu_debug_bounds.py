"""The debug build of the library (-DDSA_DEBUG_BOUNDS: every row an
index-driven gather computes is checked against the extent of the array it
reads; a row outside it sets a bit of the workspace status word and the access
is skipped, never a trap). On representative calls -- decode on BF16 / FP16 /
INT8 caches, with auxiliary K/V, on a BNSH-strided cache, on a paged pool, and
prefill -- the debug build reports nothing and gives the release build's
results bit for bit (the checks do not touch the arithmetic)."""
import numpy as np
import pytest
import torch

from dsa_inputs import make_inputs, small_workload
from tests._helpers import to_device
from tests.test_gpu_paged import paged_vs_dense

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from top_sparse_attention_chunked_gb300 import build_lib, dsa as D
    build_lib.build()
    rel = D.load_library()
    dbg = D.load_library(build_lib.build(debug=True))
    D._lib = rel
    return D, rel, dbg


def _with(D, lib, fn):
    keep = D._lib
    D._lib = lib
    try:
        return fn()
    finally:
        D._lib = keep


def _call(D, wl, cpu, prefill=False, bnsh=False, aux=None):
    dev = to_device(cpu)
    strides = (wl.num_kv_heads * wl.cap * 128, 128, wl.cap * 128) if bnsh else None
    p = D.problem_for(wl, total_len=[int(t) for t in cpu["total_len"]], kv_strides=strides)
    ws = D.alloc_workspace(p, D.DSA_OP_PREFILL if prefill else D.DSA_OP_DECODE)
    ws.fill_(0xA5)
    out = torch.empty(wl.batch, wl.q_len, wl.num_q_heads, 128, dtype=D._TORCH_DT[p.out_dtype],
                      device="cuda")
    idx = torch.empty(wl.batch, wl.q_len, wl.top_k, dtype=torch.int32, device="cuda")
    k, v = dev["k"], dev["v"]
    if bnsh:
        k = k.permute(0, 2, 1, 3).contiguous()
        v = v.permute(0, 2, 1, 3).contiguous()
    args = (p, dev["q"], dev["qI"], dev["w"], dev["kI"], k, v, dev["k_scale"], dev["v_scale"])
    if aux is not None:
        D.dsa_sparse_attn_decode_aux(*args, aux[0].cuda(), aux[1].cuda(), idx, out, ws)
    elif prefill:
        D.dsa_sparse_attn_prefill(*args, idx, out, ws)
    else:
        D.dsa_sparse_attn_decode(*args, idx, out, ws)
    torch.cuda.synchronize()
    assert D.dsa_read_device_status(ws) == 0, "a bounds check or a wait reported a fault"
    return idx.cpu().numpy(), out.float().cpu().numpy()


CASES = {
    "decode_bf16": dict(kv="bf16", q_len=4),
    "decode_fp16": dict(kv="fp16", q_len=1),
    "decode_int8": dict(kv="int8", q_len=8),
    "decode_aux": dict(kv="fp16", q_len=4, aux=True),
    "decode_bnsh": dict(kv="bf16", q_len=2, bnsh=True),
    "prefill_bf16": dict(kv="bf16", q_len=48, prefill=True),
    "prefill_int8": dict(kv="int8", q_len=40, prefill=True),
}


@pytest.mark.parametrize("name", list(CASES))
def test_debug_build_reports_nothing_and_matches_release(libs, name):
    D, rel, dbg = libs
    c = CASES[name]
    wl = small_workload(batch=2, q_len=c["q_len"], total_len=2500, num_q_heads=24,
                        num_kv_heads=2, top_k=300, kv_dtype=c["kv"], seed=900 + len(name))
    cpu = make_inputs(wl)
    aux = None
    if c.get("aux"):
        g = torch.Generator().manual_seed(3)
        qdt = torch.bfloat16 if wl.q_dtype == "bf16" else torch.float16
        aux = tuple(torch.randn(wl.batch, wl.q_len, wl.num_kv_heads, 128, generator=g).to(qdt)
                    for _ in range(2))
    kw = dict(prefill=c.get("prefill", False), bnsh=c.get("bnsh", False), aux=aux)
    i0, o0 = _with(D, rel, lambda: _call(D, wl, cpu, **kw))
    i1, o1 = _with(D, dbg, lambda: _call(D, wl, cpu, **kw))
    assert (i0 == i1).all()
    assert np.array_equal(o0, o1)


@pytest.mark.parametrize("prefill", [False, True])
def test_debug_build_paged(libs, prefill):
    """A paged pool (shuffled blocks, unmapped blocks -1, the rest of the pool
    NaN): the debug build gives the dense call's results, status 0."""
    D, rel, dbg = libs
    wl = small_workload(batch=2, q_len=200 if prefill else 3, total_len=1400, num_q_heads=8,
                        num_kv_heads=2, top_k=256, kv_dtype="bf16", capacity=1536, seed=64)
    _with(D, dbg, lambda: paged_vs_dense(D, wl, 256, 4, prefill, seed=5))
