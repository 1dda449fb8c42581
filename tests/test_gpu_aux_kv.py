"""GPU parity of dsa_sparse_attn_decode_aux (floating auxiliary K/V, reading
R14 of PR #33997): the new tokens' own K / V rows, given in the query's
floating type beside an FP16 (or INT8 / BF16) cache, are attended at their own
values. Checked against oracle.sparse_attention_aux on the GPU's own
selection (relative L2 2e-3, INT8 cache 5e-3), with auxiliary values beyond
FP16's range whose cache copies are +-inf."""
import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
from dsa_inputs import make_inputs, small_workload
from tests._helpers import TOL_16BIT, TOL_INT8, check_selection, f64_inputs, rel_l2, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from top_sparse_attention_chunked_gb300 import build_lib, dsa as D
    build_lib.build()
    D.load_library()
    return D


def aux_inputs(wl, big=True, seed=7):
    """The workload's inputs plus k_aux / v_aux: the new tokens' K / V in the
    query dtype. With `big`, a seeded tenth of their elements is scaled to
    +-(70,000 .. 131,072) (exact in BF16, beyond FP16), and the cache copies
    of the new rows are the cache-type conversions (+-inf there). The new
    tokens' index keys get +3 so most query rows select them."""
    cpu = make_inputs(wl)
    S, B = wl.q_len, wl.batch
    T = cpu["total_len"].numpy()
    g = torch.Generator().manual_seed(seed)
    qdt = torch.bfloat16 if wl.q_dtype == "bf16" else torch.float16
    ka = torch.randn(B, S, wl.num_kv_heads, 128, generator=g).to(qdt)
    va = torch.randn(B, S, wl.num_kv_heads, 128, generator=g).to(qdt)
    if big:
        for t in (ka, va):
            m = torch.rand(t.shape, generator=g) < 0.1
            mag = 70000.0 + torch.rand(t.shape, generator=g) * 61072.0
            sign = torch.where(torch.rand(t.shape, generator=g) < 0.5, -1.0, 1.0)
            t[m] = (sign * mag)[m].to(qdt)
    for b in range(B):
        past = int(T[b]) - S
        cpu["kI"][b, past:past + S] = (cpu["kI"][b, past:past + S].float() + 3.0).to(torch.bfloat16)
        if wl.kv_dtype != "int8":
            cdt = torch.bfloat16 if wl.kv_dtype == "bf16" else torch.float16
            cpu["k"][b, past:past + S] = ka[b].float().to(cdt)
            cpu["v"][b, past:past + S] = va[b].float().to(cdt)
    return cpu, ka, va


def run_aux(D, wl, cpu, ka, va):
    dev = to_device(cpu)
    p = D.problem_for(wl, total_len=[int(t) for t in cpu["total_len"]])
    ws = D.alloc_workspace(p, D.DSA_OP_DECODE)
    ws.fill_(0xA5)
    out = torch.empty(wl.batch, wl.q_len, wl.num_q_heads, 128, dtype=D._TORCH_DT[p.out_dtype],
                      device="cuda")
    idx = torch.empty(wl.batch, wl.q_len, wl.top_k, dtype=torch.int32, device="cuda")
    D.dsa_sparse_attn_decode_aux(p, dev["q"], dev["qI"], dev["w"], dev["kI"], dev["k"], dev["v"],
                                 dev["k_scale"], dev["v_scale"], ka.cuda(), va.cuda(), idx, out, ws)
    torch.cuda.synchronize()
    assert D.dsa_read_device_status(ws) == 0
    return idx.cpu().numpy(), out.float().cpu().numpy().astype(np.float64)


def check_aux(wl, cpu, ka, va, idx, out, rows=None):
    f = f64_inputs(cpu)
    B, S = wl.batch, wl.q_len
    todo = rows if rows is not None else [(b, s) for b in range(B) for s in range(S)]
    picked_new = 0
    for b, s in todo:
        n = O.visible_len(int(f["total_len"][b]), S, s)
        ref = O.index_scores_row(f["qI"][b, s], f["w"][b, s], f["kI"][b], n)
        check_selection(ref, idx[b, s], wl.top_k)
        picked_new += int((idx[b, s] >= int(f["total_len"][b]) - S).sum())
    assert picked_new > 0, "no query row selected a new token: the case tests nothing"
    att = O.sparse_attention_aux(f["q"], f["k"], f["v"], idx, wl.num_kv_heads,
                                 ka.double().numpy(), va.double().numpy(), f["total_len"],
                                 f["k_scale"], f["v_scale"], rows=todo)
    sel = np.array([[b, s] for b, s in todo])
    got, ref = out[sel[:, 0], sel[:, 1]], att[sel[:, 0], sel[:, 1]]
    assert np.isfinite(got).all(), "non-finite output: an auxiliary value was converted"
    tol = TOL_INT8 if wl.kv_dtype == "int8" else TOL_16BIT
    err = rel_l2(got, ref)
    assert err <= tol, f"relative L2 {err:.3e} > {tol}"
    return err


@pytest.mark.parametrize("kv_dtype,q_len,batch", [("fp16", 1, 1), ("fp16", 4, 2), ("fp16", 16, 1),
                                                  ("int8", 8, 2), ("bf16", 3, 3)])
def test_aux_beyond_fp16_range(dsa, kv_dtype, q_len, batch):
    wl = small_workload(batch=batch, q_len=q_len, total_len=3000, num_q_heads=24, num_kv_heads=2,
                        top_k=512, kv_dtype=kv_dtype, seed=300 + q_len)
    cpu, ka, va = aux_inputs(wl)
    idx, out = run_aux(dsa, wl, cpu, ka, va)
    check_aux(wl, cpu, ka, va, idx, out)


def test_aux_ragged_lengths_and_small_group(dsa):
    wl = small_workload(batch=3, q_len=5, total_len=2000, num_q_heads=8, num_kv_heads=2,
                        top_k=256, kv_dtype="fp16", seed=77)
    cpu, ka, va = aux_inputs(wl)
    cpu["total_len"] = torch.tensor([2000, 700, 37], dtype=torch.int32)
    cpu2, ka, va = cpu, ka, va
    # the new tokens of the shorter sequences sit at their own positions
    for b, T in enumerate([700, 37]):
        b += 1
        cpu2["kI"][b, T - 5:T] = (cpu2["kI"][b, T - 5:T].float() + 3.0).to(torch.bfloat16)
        cpu2["k"][b, T - 5:T] = ka[b].float().to(torch.float16)
        cpu2["v"][b, T - 5:T] = va[b].float().to(torch.float16)
    idx, out = run_aux(dsa, wl, cpu2, ka, va)
    check_aux(wl, cpu2, ka, va, idx, out)


def test_aux_equal_to_cache_matches_plain_decode(dsa):
    """Auxiliary rows equal to the cache's new rows (in range): the output is
    the plain decode's, within the tolerance."""
    wl = small_workload(batch=2, q_len=8, total_len=4096, num_q_heads=24, num_kv_heads=2,
                        top_k=512, kv_dtype="bf16", seed=91)
    cpu, ka, va = aux_inputs(wl, big=False)
    idx, out = run_aux(dsa, wl, cpu, ka, va)
    check_aux(wl, cpu, ka, va, idx, out)
    dev = to_device(cpu)
    p = dsa.problem_for(wl)
    ws = dsa.alloc_workspace(p, dsa.DSA_OP_DECODE)
    out2 = torch.empty_like(torch.from_numpy(out)).to(dsa._TORCH_DT[p.out_dtype]).cuda()
    idx2 = torch.empty(wl.batch, wl.q_len, wl.top_k, dtype=torch.int32, device="cuda")
    dsa.dsa_sparse_attn_decode(p, dev["q"], dev["qI"], dev["w"], dev["kI"], dev["k"], dev["v"],
                               None, None, idx2, out2, ws)
    torch.cuda.synchronize()
    assert (idx2.cpu().numpy() == idx).all()
    assert rel_l2(out2.float().cpu().numpy().astype(np.float64), out) <= TOL_16BIT


def test_aux_grouped_decode_32k_sampled(dsa):
    """The grouped-decode shape at full size (4 x 8 query tokens on a 32,768
    context, 24 / 2 heads, FP16 cache, BF16 auxiliary rows beyond FP16)."""
    wl = small_workload(batch=4, q_len=8, total_len=32768, num_q_heads=24, num_kv_heads=2,
                        top_k=2048, kv_dtype="fp16", seed=1002)
    cpu, ka, va = aux_inputs(wl)
    idx, out = run_aux(dsa, wl, cpu, ka, va)
    check_aux(wl, cpu, ka, va, idx, out, rows=[(0, 0), (1, 7), (2, 3), (3, 5)])


def test_aux_arguments_are_checked(dsa):
    wl = small_workload(batch=1, q_len=2, total_len=500, num_q_heads=8, num_kv_heads=2,
                        top_k=64, kv_dtype="fp16", seed=5)
    cpu, ka, va = aux_inputs(wl)
    dev = to_device(cpu)
    p = dsa.problem_for(wl)
    ws = dsa.alloc_workspace(p, dsa.DSA_OP_DECODE)
    out = torch.empty(1, 2, 8, 128, dtype=torch.bfloat16, device="cuda")
    lib = dsa.load_library()
    import ctypes
    rc = lib.dsa_sparse_attn_decode_aux(ctypes.byref(p), ctypes.c_void_p(dev["q"].data_ptr()),
                                        ctypes.c_void_p(dev["qI"].data_ptr()),
                                        ctypes.c_void_p(dev["w"].data_ptr()),
                                        ctypes.c_void_p(dev["kI"].data_ptr()),
                                        ctypes.c_void_p(dev["k"].data_ptr()),
                                        ctypes.c_void_p(dev["v"].data_ptr()), None, None,
                                        None, None, None, ctypes.c_void_p(out.data_ptr()),
                                        ctypes.c_void_p(ws.data_ptr()), ws.numel(), None)
    assert rc == dsa.DSA_ERR_INVALID_ARG
