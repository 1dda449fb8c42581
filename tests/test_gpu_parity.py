"""GPU parity: libdsa (through its C ABI) against the float64 oracle on seeded
inputs. Bars: top-k bit-exact on a given fp32 score tensor; indexer scores
within the fp32 accumulation error bound; full-pipeline selections equal up
to keys within 1e-5 (relative) of the k-th score; outputs within 2e-3
relative L2 (BF16/FP16 cache) or 5e-3 (INT8 cache) of the oracle run on the
GPU's own selection."""
import math

import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
from dsa_inputs import WORKLOADS, Workload, make_inputs, small_workload
from tests._helpers import (TOL_16BIT, TOL_INT8, check_index_row, check_selection, f64_inputs,
                            rel_l2, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from top_sparse_attention_chunked_gb300 import build_lib, dsa as D
    build_lib.build()
    D.load_library()
    return D


# ---------------------------------------------------------------- helpers
def run_step(D, wl: Workload, cpu=None, prefill=False, **prob_kw):
    cpu = cpu if cpu is not None else make_inputs(wl)
    dev = to_device(cpu)
    p = D.problem_for(wl, **prob_kw)
    op = D.DSA_OP_PREFILL if prefill else D.DSA_OP_DECODE
    ws = D.alloc_workspace(p, op)
    ws.fill_(0xA5)   # never assume a clean workspace
    out = torch.empty(wl.batch, wl.q_len, wl.num_q_heads, 128,
                      dtype=D._TORCH_DT[p.out_dtype], device="cuda")
    idx = torch.empty(wl.batch, wl.q_len, wl.top_k, dtype=torch.int32, device="cuda")
    fn = D.dsa_sparse_attn_prefill if prefill else D.dsa_sparse_attn_decode
    fn(p, dev["q"], dev["qI"], dev["w"], dev["kI"], dev["k"], dev["v"], dev["k_scale"],
       dev["v_scale"], idx, out, ws)
    torch.cuda.synchronize()
    assert D.dsa_read_device_status(ws) == 0
    return cpu, idx.cpu().numpy(), out.float().cpu().numpy().astype(np.float64)


def check_step(wl, cpu, idx, out, rows=None, softmax_scale=0.0):
    f = f64_inputs(cpu)
    B, S = wl.batch, wl.q_len
    todo = rows if rows is not None else [(b, s) for b in range(B) for s in range(S)]
    ndiff = 0
    for b, s in todo:
        n = O.visible_len(int(f["total_len"][b]), S, s)
        ref = O.index_scores_row(f["qI"][b, s], f["w"][b, s], f["kI"][b], n)
        ndiff += check_selection(ref, idx[b, s], wl.top_k)
    att = O.sparse_attention(f["q"], f["k"], f["v"], idx, wl.num_kv_heads, f["k_scale"],
                             f["v_scale"], softmax_scale, rows=todo)
    got = np.stack([out[b, s] for b, s in todo])
    ref = np.stack([att[b, s] for b, s in todo])
    err = rel_l2(got, ref)
    tol = TOL_INT8 if wl.kv_dtype == "int8" else TOL_16BIT
    assert err <= tol, f"relative L2 {err:.3e} > {tol}"
    return err, ndiff


# ---------------------------------------------------------------- indexer
@pytest.mark.parametrize("B,S,T,cap", [
    (1, 1, 4096, 4096), (2, 3, [1000, 700], 1024), (2, 8, [2048 + 77, 300], 2200),
    (1, 16, 5000, 5003), (1, 37, 3001, 3001), (3, 5, [130, 9, 257], 300),
])
def test_index_scores_parity(dsa, B, S, T, cap):
    wl = small_workload(batch=B, q_len=S, total_len=max(T) if isinstance(T, list) else T,
                        capacity=cap, top_k=8, seed=21 + S)
    cpu = make_inputs(wl)
    if isinstance(T, list):
        cpu["total_len"] = torch.tensor(T, dtype=torch.int32)
    p = dsa.problem_for(wl, total_len=(T if isinstance(T, list) else [T] * B))
    dev = to_device(cpu)
    scores = torch.full((B, S, cap), -7.25, dtype=torch.float32, device="cuda")
    ws = dsa.alloc_workspace(p, dsa.DSA_OP_INDEX_SCORES)
    dsa.dsa_index_scores(p, dev["qI"], dev["w"], dev["kI"], scores, ws)
    got = scores.cpu().numpy()
    f = f64_inputs(cpu)
    for b in range(B):
        for s in range(S):
            n = O.visible_len(int(f["total_len"][b]), S, s)
            check_index_row(got[b, s], f["qI"][b, s], f["w"][b, s], f["kI"][b], n)
            assert (got[b, s, n:] == -7.25).all(), "wrote past the visible length"


def test_index_scores_split_query_bit_exact(dsa):
    """Blocks of 16 queries split their queries between the two epilogue
    groups, hold the head weights in registers and take half of the heads'
    ReLU as x + |x| against halved weights; a block of one query reads the
    weights from shared memory and uses max(x, 0). For finite dot products
    the two give the same real products, summed in the same order, so every
    visible score must match bit for bit: each of 16 queries is scored alone,
    on a cache cut to the keys it sees inside the block."""
    S, T, cap = 16, 3001, 3001
    wl = small_workload(batch=1, q_len=S, total_len=T, capacity=cap, top_k=8, seed=77)
    cpu = make_inputs(wl)
    dev = to_device(cpu)
    p = dsa.problem_for(wl, total_len=[T])
    blk = torch.full((1, S, cap), -7.25, dtype=torch.float32, device="cuda")
    dsa.dsa_index_scores(p, dev["qI"], dev["w"], dev["kI"], blk, dsa.alloc_workspace(p, dsa.DSA_OP_INDEX_SCORES))
    wl1 = small_workload(batch=1, q_len=1, total_len=T, capacity=cap, top_k=8, seed=77)
    for s in range(S):
        n = O.visible_len(T, S, s)
        p1 = dsa.problem_for(wl1, total_len=[n])
        one = torch.full((1, 1, cap), -7.25, dtype=torch.float32, device="cuda")
        dsa.dsa_index_scores(p1, dev["qI"][:, s:s + 1].contiguous(), dev["w"][:, s:s + 1].contiguous(),
                             dev["kI"], one, dsa.alloc_workspace(p1, dsa.DSA_OP_INDEX_SCORES))
        a, b = blk[0, s, :n].cpu(), one[0, 0, :n].cpu()
        assert torch.equal(a, b), f"query {s}: {int((a != b).sum())} of {n} scores differ"


def test_index_scores_full_128k(dsa):
    wl = WORKLOADS["decode_128k"]
    cpu = make_inputs(wl)
    dev = to_device(cpu)
    p = dsa.problem_for(wl)
    scores = torch.empty(1, 1, wl.cap, dtype=torch.float32, device="cuda")
    ws = dsa.alloc_workspace(p, dsa.DSA_OP_INDEX_SCORES)
    dsa.dsa_index_scores(p, dev["qI"], dev["w"], dev["kI"], scores, ws)
    f = f64_inputs(cpu)
    check_index_row(scores.cpu().numpy()[0, 0], f["qI"][0, 0], f["w"][0, 0], f["kI"][0], wl.total_len)


# ---------------------------------------------------------------- top-k (bit-exact)
def _topk_case(dsa, B, S, T, cap, k, kind, seed):
    g = torch.Generator().manual_seed(seed)
    if kind == "ties":
        sc = torch.randint(-3, 4, (B, S, cap), generator=g).float()
    elif kind == "zeros":
        sc = torch.zeros(B, S, cap)
        sc[..., ::3] = -0.0
    elif kind == "inf":
        sc = torch.randn(B, S, cap, generator=g)
        sc[sc < -1.0] = float("-inf")
    else:
        sc = torch.randn(B, S, cap, generator=g) * 10
    Ts = T if isinstance(T, list) else [T] * B
    p = dsa.make_problem(batch=B, q_len=S, total_len=Ts, top_k=k, cache_capacity=cap)
    ws = dsa.alloc_workspace(p, dsa.DSA_OP_TOPK)
    ws.fill_(0x5A)
    idx = torch.full((B, S, k), -99, dtype=torch.int32, device="cuda")
    dsa.dsa_topk(p, sc.cuda(), idx, ws)
    got = idx.cpu().numpy()
    v = sc.numpy().astype(np.float64)
    for b in range(B):
        for s in range(S):
            n = O.visible_len(Ts[b], S, s)
            ref = O.topk_select_row(v[b, s, :n], k)
            assert np.array_equal(got[b, s], ref), (b, s, n, k)


@pytest.mark.parametrize("kind", ["ties", "cont", "zeros", "inf"])
@pytest.mark.parametrize("B,S,T,cap,k", [
    (2, 3, [5000, 3000], 5000, 100), (1, 1, 4096, 4096, 512), (2, 2, [2049, 2], 4100, 2048),
    (1, 4, 70, 80, 64), (1, 1, 1, 1, 1), (1, 2, 9000, 9000, 8999),
    (1, 1, 600000, 600000, 2048),   # longer than the cluster select: global merge path
    (2, 1, [300000, 262145], 300000, 2048),   # 24 keys a thread, clusters of 13 CTAs (one row ragged)
    (1, 2, 40000, 40000, 3000),     # tie-heavy rows with > 8,192 threshold-bin candidates
])
def test_topk_bitexact_chunked(dsa, kind, B, S, T, cap, k):
    _topk_case(dsa, B, S, T, cap, k, kind, seed=hash((kind, B, S, k)) & 0xFFFF)


@pytest.mark.parametrize("kind", ["ties", "cont", "zeros"])
@pytest.mark.parametrize("S,T,k", [(400, 3000, 256), (320, 700, 700), (512, 2048, 1)])
def test_topk_bitexact_rows(dsa, kind, S, T, k):
    # many rows -> the whole-row shared-memory select
    _topk_case(dsa, 1, S, T, T, k, kind, seed=S + k)


@pytest.mark.parametrize("name", ["decode_128k", "decode_256k_int8"])
def test_topk_bitexact_full_size(dsa, name):
    wl = WORKLOADS[name]
    cpu = make_inputs(wl)
    f = f64_inputs(cpu)
    sc = O.index_scores(f["qI"], f["w"], f["kI"], f["total_len"]).astype(np.float32)
    sc = np.nan_to_num(sc, nan=0.0)
    p = dsa.problem_for(wl)
    ws = dsa.alloc_workspace(p, dsa.DSA_OP_TOPK)
    idx = torch.empty(wl.batch, wl.q_len, wl.top_k, dtype=torch.int32, device="cuda")
    dsa.dsa_topk(p, torch.from_numpy(sc).cuda(), idx, ws)
    got = idx.cpu().numpy()
    for s in range(wl.q_len):
        n = O.visible_len(wl.total_len, wl.q_len, s)
        assert np.array_equal(got[0, s], O.topk_select_row(sc[0, s, :n].astype(np.float64), wl.top_k))


# ---------------------------------------------------------------- whole step
@pytest.mark.parametrize("name", ["decode_4k", "grouped_decode_32k", "decode_128k",
                                  "decode_256k_int8"])
def test_decode_parity_workloads(dsa, name):
    wl = WORKLOADS[name]
    cpu, idx, out = run_step(dsa, wl)
    err, ndiff = check_step(wl, cpu, idx, out)
    print(f"{name}: rel L2 {err:.2e}, selection differences {ndiff}")


@pytest.mark.parametrize("kv", ["bf16", "fp16", "int8"])
@pytest.mark.parametrize("B,S,T,cap,Hq,Hkv,k", [
    (2, 3, 1000, 1024, 8, 2, 64), (1, 8, 5000, 5000, 24, 2, 2048), (2, 1, 300, 4096, 4, 4, 512),
    (1, 16, 2100, 2100, 32, 1, 100),
])
def test_decode_parity_small(dsa, kv, B, S, T, cap, Hq, Hkv, k):
    wl = small_workload(batch=B, q_len=S, total_len=T, capacity=cap, num_q_heads=Hq,
                        num_kv_heads=Hkv, top_k=k, kv_dtype=kv, seed=B * 100 + S)
    cpu, idx, out = run_step(dsa, wl)
    check_step(wl, cpu, idx, out)


@pytest.mark.parametrize("qd,kv", [("fp16", "fp16"), ("fp16", "int8")])
def test_decode_fp16_query(dsa, qd, kv):
    wl = small_workload(batch=1, q_len=2, total_len=3000, top_k=256, q_dtype=qd, kv_dtype=kv,
                        seed=77)
    cpu, idx, out = run_step(dsa, wl)
    check_step(wl, cpu, idx, out)


@pytest.mark.parametrize("split", [16, 48, 256])
def test_decode_split_counts_agree(dsa, split):
    wl = small_workload(batch=1, q_len=4, total_len=6000, top_k=1000, num_q_heads=24,
                        num_kv_heads=2, kv_dtype="fp16", seed=5)
    cpu, idx, out = run_step(dsa, wl, attn_split_keys=split)
    check_step(wl, cpu, idx, out)


def test_decode_fp32_output_and_ragged_lengths(dsa):
    wl = small_workload(batch=3, q_len=2, total_len=4000, capacity=4096, top_k=300, seed=9)
    cpu = make_inputs(wl)
    cpu["total_len"] = torch.tensor([4000, 17, 2500], dtype=torch.int32)
    _, idx, out = run_step(dsa, wl, cpu=cpu, total_len=[4000, 17, 2500], out_dtype="fp32")
    err, _ = check_step(wl, cpu, idx, out)
    assert err < 2e-4   # no output rounding: only the attention arithmetic


@pytest.mark.parametrize("kv", ["bf16", "fp16", "int8"])
@pytest.mark.parametrize("B,S,T,cap,Hq,Hkv,k", [
    (2, 40, 300, 320, 24, 2, 64), (1, 130, 2500, 2500, 24, 2, 2048), (1, 33, 33, 33, 8, 2, 8),
    (2, 17, 1000, 1100, 32, 1, 200), (1, 50, 4000, 4000, 4, 4, 3000),
])
def test_prefill_parity_small(dsa, kv, B, S, T, cap, Hq, Hkv, k):
    wl = small_workload(batch=B, q_len=S, total_len=T, capacity=cap, num_q_heads=Hq,
                        num_kv_heads=Hkv, top_k=k, kv_dtype=kv, seed=S + Hq)
    cpu, idx, out = run_step(dsa, wl, prefill=True)
    check_step(wl, cpu, idx, out)


def test_prefill_fp16_query_fp16_cache(dsa):
    wl = small_workload(batch=1, q_len=64, total_len=900, top_k=300, q_dtype="fp16",
                        kv_dtype="fp16", seed=41)
    cpu, idx, out = run_step(dsa, wl, prefill=True)
    check_step(wl, cpu, idx, out)


@pytest.mark.parametrize("qd", ["bf16", "fp16"])
def test_prefill_int8_ragged(dsa, qd):
    """INT8 prefill with a BF16 or FP16 query, ragged lengths and more
    selected keys than one 128-key tile."""
    wl = small_workload(batch=2, q_len=70, total_len=3000, capacity=3100, num_q_heads=24,
                        num_kv_heads=2, top_k=600, q_dtype=qd, kv_dtype="int8", seed=47)
    cpu = make_inputs(wl)
    cpu["total_len"] = torch.tensor([3000, 2200], dtype=torch.int32)
    cpu, idx, out = run_step(dsa, wl, cpu=cpu, prefill=True, total_len=[3000, 2200])
    check_step(wl, cpu, idx, out)


def test_prefill_int8_8k_on_32k_sampled(dsa):
    """The prefill workload's shape with an INT8 cache, on 8 sampled rows."""
    base = WORKLOADS["prefill_8k_on_32k"]
    wl = Workload("prefill_int8", base.batch, base.q_len, base.total_len, base.num_q_heads,
                  base.num_kv_heads, base.top_k, base.q_dtype, "int8", seed=base.seed)
    cpu, idx, out = run_step(dsa, wl, prefill=True)
    rng = np.random.default_rng(1)
    rows = sorted({0, wl.q_len - 1, *rng.integers(0, wl.q_len, 6).tolist()})
    check_step(wl, cpu, idx, out, rows=[(0, s) for s in rows])


def test_prefill_and_decode_agree(dsa):
    """The same 8 query tokens through the decode path and the prefill path."""
    wl = small_workload(batch=2, q_len=8, total_len=6000, num_q_heads=24, num_kv_heads=2,
                        top_k=2048, kv_dtype="bf16", seed=43)
    cpu = make_inputs(wl)
    _, idx_d, out_d = run_step(dsa, wl, cpu=cpu, out_dtype="fp32")
    _, idx_p, out_p = run_step(dsa, wl, cpu=cpu, prefill=True, out_dtype="fp32")
    check_step(wl, cpu, idx_d, out_d)
    check_step(wl, cpu, idx_p, out_p)
    if np.array_equal(idx_d, idx_p):
        assert rel_l2(out_p, out_d) < 1e-5


def test_prefill_parity_8k_on_32k_sampled(dsa):
    wl = WORKLOADS["prefill_8k_on_32k"]
    cpu, idx, out = run_step(dsa, wl, prefill=True)
    rng = np.random.default_rng(0)
    rows = sorted({0, wl.q_len - 1, *rng.integers(0, wl.q_len, 14).tolist()})
    check_step(wl, cpu, idx, out, rows=[(0, s) for s in rows])


# ---------------------------------------------------------------- degenerate cases
def test_single_key_cache(dsa):
    wl = small_workload(batch=1, q_len=1, total_len=1, capacity=1, top_k=1, seed=3)
    cpu, idx, out = run_step(dsa, wl)
    assert idx[0, 0, 0] == 0
    check_step(wl, cpu, idx, out)


def test_topk_larger_than_context(dsa):
    wl = small_workload(batch=2, q_len=3, total_len=50, capacity=4096, top_k=4000, seed=4)
    cpu, idx, out = run_step(dsa, wl)
    for s in range(3):
        n = 50 - 3 + s + 1
        assert idx[0, s, :n].tolist() == list(range(n)) and (idx[0, s, n:] == -1).all()
    check_step(wl, cpu, idx, out)


def test_decode_all_equal_scores_long_row(dsa):
    """kI = 0 over 50,000 keys: every score ties, the threshold bin holds all
    keys (more than the cluster select gathers), the lowest indices win."""
    wl = small_workload(batch=1, q_len=1, total_len=50000, top_k=2048, seed=16)
    cpu = make_inputs(wl)
    cpu["kI"].zero_()
    _, idx, out = run_step(dsa, wl, cpu=cpu)
    assert idx[0, 0].tolist() == list(range(2048))
    check_step(wl, cpu, idx, out)


def test_all_equal_scores_take_the_lowest_indices(dsa):
    wl = small_workload(batch=1, q_len=2, total_len=9000, top_k=700, seed=6)
    cpu = make_inputs(wl)
    cpu["kI"].zero_()
    _, idx, out = run_step(dsa, wl, cpu=cpu)
    assert idx[0, 0].tolist() == list(range(700))
    check_step(wl, cpu, idx, out)


def test_uniform_query_averages_selected_values(dsa):
    wl = small_workload(batch=1, q_len=1, total_len=3000, top_k=333, kv_dtype="fp16", seed=8)
    cpu = make_inputs(wl)
    cpu["q"].zero_()
    _, idx, out = run_step(dsa, wl, cpu=cpu, out_dtype="fp32")
    sel = idx[0, 0][idx[0, 0] >= 0]
    v = cpu["v"].double().numpy()[0, sel]
    for h in range(8):
        np.testing.assert_allclose(out[0, 0, h], v[:, h // 4].mean(axis=0), rtol=1e-4, atol=1e-5)


@pytest.mark.parametrize("spacing", [0, 14, 15, 16, 40, 100])
@pytest.mark.parametrize("split", [0, 16, 32, 2048])
def test_int8_large_value_scale_worked_example(dsa, spacing, split):
    """PR #33847's case: logits 0 and 88, value codes 1 and 0, value scale
    2^120; expected 2^120 e^-88 / (1 + e^-88). Keys with logit -1000 pad the
    gap so the two candidates land in one tile, different tiles, different
    warps, or different split blocks."""
    m = 2 + spacing
    wl = Workload("worked", 1, 1, m, 1, 1, m, "bf16", "int8", seed=1)
    cpu = make_inputs(wl)
    q = torch.zeros(1, 1, 1, 128)
    q[0, 0, 0, 0] = 88.0
    cpu["q"] = q.to(torch.bfloat16)
    k = torch.zeros(1, m, 1, 128, dtype=torch.int8)
    k[0, m - 1, 0, 0] = 1
    k[0, 1:m - 1, 0, 0] = -1
    ks = torch.ones(1, m, 1)
    ks[0, 1:m - 1, 0] = 1000.0 / 88.0
    v = torch.zeros(1, m, 1, 128, dtype=torch.int8)
    v[0, 0, 0, :] = 1
    cpu.update(k=k, v=v, k_scale=ks, v_scale=torch.full((1, m, 1), 2.0 ** 120))
    _, idx, out = run_step(dsa, wl, cpu=cpu, softmax_scale=1.0, out_dtype="fp32",
                           attn_split_keys=split)
    expect = 2.0 ** 120 * math.exp(-88) / (1 + math.exp(-88))
    np.testing.assert_allclose(out[0, 0, 0], expect, rtol=2e-5)


@pytest.mark.parametrize("spacing", [0, 126, 127, 300])
def test_int8_large_value_scale_worked_example_prefill(dsa, spacing):
    """PR #33847's case through the prefill call: the two candidates in one
    128-key stretch or far apart."""
    m = 2 + spacing
    wl = Workload("worked_pf", 1, 1, m, 1, 1, m, "bf16", "int8", seed=1)
    cpu = make_inputs(wl)
    q = torch.zeros(1, 1, 1, 128)
    q[0, 0, 0, 0] = 88.0
    cpu["q"] = q.to(torch.bfloat16)
    k = torch.zeros(1, m, 1, 128, dtype=torch.int8)
    k[0, m - 1, 0, 0] = 1
    k[0, 1:m - 1, 0, 0] = -1
    ks = torch.ones(1, m, 1)
    ks[0, 1:m - 1, 0] = 1000.0 / 88.0
    v = torch.zeros(1, m, 1, 128, dtype=torch.int8)
    v[0, 0, 0, :] = 1
    cpu.update(k=k, v=v, k_scale=ks, v_scale=torch.full((1, m, 1), 2.0 ** 120))
    _, idx, out = run_step(dsa, wl, cpu=cpu, prefill=True, softmax_scale=1.0, out_dtype="fp32")
    expect = 2.0 ** 120 * math.exp(-88) / (1 + math.exp(-88))
    np.testing.assert_allclose(out[0, 0, 0], expect, rtol=2e-5)


def test_workspace_reuse_across_shapes(dsa):
    big = WORKLOADS["decode_4k"]
    small = small_workload(batch=1, q_len=1, total_len=300, capacity=4096, num_q_heads=8,
                           num_kv_heads=2, top_k=512, seed=12)
    pb, ps = dsa.problem_for(big), dsa.problem_for(small)
    ws = dsa.alloc_workspace(pb, dsa.DSA_OP_DECODE)
    assert ws.numel() >= dsa.dsa_workspace_size(ps, dsa.DSA_OP_DECODE)
    outs = []
    for wl, p in ((big, pb), (small, ps), (big, pb)):
        cpu = make_inputs(wl)
        dev = to_device(cpu)
        out = torch.empty(1, 1, wl.num_q_heads, 128, dtype=torch.bfloat16, device="cuda")
        dsa.dsa_sparse_attn_decode(p, dev["q"], dev["qI"], dev["w"], dev["kI"], dev["k"],
                                   dev["v"], None, None, None, out, ws)
        outs.append(out.float().cpu())
    assert torch.equal(outs[0], outs[2])


# ---------------------------------------------------------------- single-token decode
@pytest.mark.parametrize("kv", ["bf16", "fp16", "int8"])
def test_single_token_ragged_batch(dsa, kv):
    wl = small_workload(batch=3, q_len=1, total_len=40000, capacity=40000, num_q_heads=24,
                        num_kv_heads=2, top_k=2048, kv_dtype=kv, seed=31)
    cpu = make_inputs(wl)
    lens = [40000, 17, 25000]
    cpu["total_len"] = torch.tensor(lens, dtype=torch.int32)
    _, idx, out = run_step(dsa, wl, cpu=cpu, total_len=lens, out_dtype="fp32")
    assert (idx[1, 0, :17] == np.arange(17)).all() and (idx[1, 0, 17:] == -1).all()
    check_step(wl, cpu, idx, out)


def test_single_token_topk_above_context(dsa):
    wl = small_workload(batch=2, q_len=1, total_len=50, capacity=4096, top_k=4000, seed=41)
    cpu, idx, out = run_step(dsa, wl)
    for b in range(2):
        assert idx[b, 0, :50].tolist() == list(range(50)) and (idx[b, 0, 50:] == -1).all()
    check_step(wl, cpu, idx, out)
