"""GPU parity of the paged-cache entry points: every paged call must give the
dense call's results bit for bit when the dense caches are scattered over a
shuffled pool of blocks. Blocks that hold no visible token are marked -1 in
the table and the rest of the pool is filled with NaN (16-bit) or NaN scales
(INT8), so a read of any row outside the mapped blocks would show up in the
output or in the device status word."""
import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
from dsa_inputs import make_append_inputs, make_inputs, small_workload, to_f64
from tests._helpers import TOL_16BIT, TOL_INT8, f64_inputs, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from top_sparse_attention_chunked_gb300 import build_lib, dsa as D
    build_lib.build()
    D.load_library()
    return D


def _poison(t: torch.Tensor):
    if t.dtype in (torch.bfloat16, torch.float16, torch.float32):
        t.fill_(float("nan"))
    else:
        t.fill_(127)


def scatter_to_pool(dense: dict, lens, block_size: int, spare: int, seed: int, share=None):
    """Pools and a block table holding the dense caches' first total_len[b]
    rows of every sequence in shuffled blocks; `spare` extra unused blocks.
    share=(b_from, b_to, nblk): sequence b_to maps its first nblk blocks to
    b_from's (a shared prefix; the dense caches must agree there)."""
    kI = dense["kI"]
    B, cap = kI.shape[0], kI.shape[1]
    per_seq = cap // block_size
    used = [(-(-int(t) // block_size)) for t in lens]
    nblocks = sum(used) + spare
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(nblocks, generator=g).tolist()
    table = torch.full((B, per_seq), -1, dtype=torch.int32)
    k = 0
    for b in range(B):
        for j in range(used[b]):
            table[b, j] = perm[k]
            k += 1
    if share is not None:
        bf, bt, n = share
        table[bt, :n] = table[bf, :n]
    pools = {}
    for name in ("kI", "k", "v", "k_scale", "v_scale"):
        d = dense.get(name)
        if d is None:
            pools[name] = None
            continue
        pool = torch.empty((nblocks * block_size,) + tuple(d.shape[2:]), dtype=d.dtype)
        _poison(pool)
        for b in range(B):
            for j in range(used[b]):
                blk = int(table[b, j])
                pool[blk * block_size:(blk + 1) * block_size] = d[b, j * block_size:(j + 1) * block_size]
        pools[name] = pool.contiguous()
    return pools, table, nblocks


def _dev(x):
    return x.cuda() if isinstance(x, torch.Tensor) else x


def run_attn(D, p, dev, kv, prefill, pages=None, ws=None):
    op = D.DSA_OP_PREFILL if prefill else D.DSA_OP_DECODE
    ws = ws if ws is not None else D.alloc_workspace(p, op)
    out = torch.empty(p.batch, p.q_len, p.num_q_heads, 128, dtype=D._TORCH_DT[p.out_dtype],
                      device="cuda")
    idx = torch.empty(p.batch, p.q_len, p.top_k, dtype=torch.int32, device="cuda")
    fn = D.dsa_sparse_attn_prefill if prefill else D.dsa_sparse_attn_decode
    fn(p, dev["q"], dev["qI"], dev["w"], kv["kI"], kv["k"], kv["v"], kv["k_scale"], kv["v_scale"],
       idx, out, ws, pages=pages)
    torch.cuda.synchronize()
    return idx, out, ws


def _same(a: torch.Tensor, b: torch.Tensor):
    if a.dtype in (torch.bfloat16, torch.float16):
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    if a.dtype == torch.float32:
        return torch.equal(a.view(torch.int32), b.view(torch.int32))
    return torch.equal(a, b)


def paged_vs_dense(D, wl, block_size, spare, prefill, seed, share=None, mutate=None):
    cpu = make_inputs(wl)
    lens = [wl.total_len] * wl.batch
    if mutate:
        mutate(cpu)
    pools, table, nblocks = scatter_to_pool(cpu, lens, block_size, spare, seed, share)
    dev = {k: _dev(v) for k, v in cpu.items()}
    p = D.problem_for(wl)
    dense = {k: dev[k] for k in ("kI", "k", "v", "k_scale", "v_scale")}
    idx_d, out_d, ws = run_attn(D, p, dev, dense, prefill)
    assert D.dsa_read_device_status(ws) == 0
    table_d = table.cuda()
    pages = D.make_pages(table_d, block_size, nblocks)
    pk = {k: _dev(v) for k, v in pools.items()}
    ws.fill_(0xA5)
    idx_p, out_p, _ = run_attn(D, p, dev, pk, prefill, pages=pages, ws=ws)
    assert D.dsa_read_device_status(ws) == 0
    assert torch.equal(idx_p, idx_d)
    assert _same(out_p, out_d)
    return cpu, idx_d, out_d, pools, table, nblocks


@pytest.mark.parametrize("kv", ["bf16", "fp16", "int8"])
def test_paged_decode_matches_dense(dsa, kv):
    wl = small_workload(batch=3, q_len=2, total_len=1400, num_q_heads=8, num_kv_heads=2,
                        top_k=256, kv_dtype=kv, capacity=1536, seed=61)
    paged_vs_dense(dsa, wl, 256, 5, False, seed=1)


@pytest.mark.parametrize("kv", ["bf16", "fp16", "int8"])
def test_paged_prefill_matches_dense(dsa, kv):
    wl = small_workload(batch=2, q_len=300, total_len=1200, num_q_heads=8, num_kv_heads=2,
                        top_k=300, kv_dtype=kv, capacity=1280, seed=62)
    paged_vs_dense(dsa, wl, 128, 3, True, seed=2)


def test_paged_decode_against_oracle(dsa):
    """The paged decode checked directly against the oracle on the gathered
    caches (the selection within the tie band, the output within 2e-3)."""
    wl = small_workload(batch=2, q_len=3, total_len=2000, num_q_heads=8, num_kv_heads=2,
                        top_k=200, kv_dtype="bf16", capacity=2048, seed=63)
    cpu, idx_d, out_d, pools, table, nblocks = paged_vs_dense(dsa, wl, 512, 2, False, seed=3)
    lens = [wl.total_len] * wl.batch
    view = {n: O.gather_pages(to_f64(pools[n]), table.numpy(), 512, lens)
            for n in ("kI", "k", "v")}
    f = f64_inputs(cpu)
    idx = idx_d.cpu().numpy()
    att = O.sparse_attention(f["q"], view["k"], view["v"], idx, wl.num_kv_heads, None, None, 0.0)
    for b in range(wl.batch):
        for s in range(wl.q_len):
            n = O.visible_len(wl.total_len, wl.q_len, s)
            ref = O.index_scores_row(f["qI"][b, s], f["w"][b, s], view["kI"][b], n)
            kth = np.sort(ref)[::-1][min(wl.top_k, n) - 1]
            sel = set(idx[b, s][idx[b, s] >= 0].tolist())
            want = set(np.argsort(-ref, kind="stable")[:min(wl.top_k, n)].tolist())
            for t in sel ^ want:
                assert abs(ref[t] - kth) <= 1e-5 * abs(kth)
    assert rel_l2(out_d.float().cpu().numpy().astype(np.float64), att) <= TOL_16BIT


def test_paged_shared_prefix(dsa):
    """Two sequences whose first three blocks are the same physical blocks
    (a common prefix): the paged decode equals the dense decode on caches
    that hold the prefix twice."""
    wl = small_workload(batch=2, q_len=1, total_len=1000, num_q_heads=8, num_kv_heads=2,
                        top_k=128, kv_dtype="fp16", capacity=1024, seed=64)

    def copy_prefix(cpu):
        for n in ("kI", "k", "v"):
            cpu[n][1, :384] = cpu[n][0, :384]
    paged_vs_dense(dsa, wl, 128, 1, False, seed=4, share=(0, 1, 3), mutate=copy_prefix)


def test_paged_index_scores_matches_dense(dsa):
    D = dsa
    wl = small_workload(batch=2, q_len=5, total_len=900, num_q_heads=8, num_kv_heads=2,
                        top_k=8, capacity=1024, seed=65)
    cpu = make_inputs(wl)
    pools, table, nblocks = scatter_to_pool(cpu, [900, 900], 128, 2, seed=5)
    p = D.problem_for(wl)
    ws = D.alloc_workspace(p, D.DSA_OP_INDEX_SCORES)
    sd = torch.zeros(2, 5, 1024, dtype=torch.float32, device="cuda")
    sp = torch.zeros_like(sd)
    D.dsa_index_scores(p, _dev(cpu["qI"]), _dev(cpu["w"]), _dev(cpu["kI"]), sd, ws)
    pages = D.make_pages(table.cuda(), 128, nblocks)
    D.dsa_index_scores(p, _dev(cpu["qI"]), _dev(cpu["w"]), _dev(pools["kI"]), sp, ws, pages=pages)
    torch.cuda.synchronize()
    assert D.dsa_read_device_status(ws) == 0
    assert _same(sp, sd)


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_paged_append_matches_dense(dsa, kv):
    """Append into a paged pool: the gathered caches equal the dense append's
    bit for bit and every pool row outside the written ones keeps its bytes."""
    D = dsa
    B, S, H, cap, T, bs = 2, 70, 2, 512, [300, 512], 128
    cpu = make_append_inputs(B, S, H, cap, T, "bf16", kv, seed=66)
    pools, table, nblocks = scatter_to_pool(cpu, T, bs, 2, seed=6)
    p = D.make_problem(batch=B, q_len=S, total_len=T, top_k=1, num_q_heads=H, num_kv_heads=H,
                       cache_capacity=cap, q_dtype="bf16", kv_dtype=kv)
    dev = {k: _dev(v) for k, v in cpu.items()}
    D.dsa_cache_append(p, dev["kI_new"], dev["k_new"], dev["v_new"], dev["kI"], dev["k"], dev["v"],
                       dev["k_scale"], dev["v_scale"])
    pk = {k: _dev(v) for k, v in pools.items()}
    before = {k: v.clone() for k, v in pk.items() if v is not None}
    pages = D.make_pages(table.cuda(), bs, nblocks)
    D.dsa_cache_append(p, dev["kI_new"], dev["k_new"], dev["v_new"], pk["kI"], pk["k"], pk["v"],
                       pk["k_scale"], pk["v_scale"], pages=pages)
    torch.cuda.synchronize()
    written = torch.zeros(nblocks * bs, dtype=torch.bool)
    for b in range(B):
        for s in range(S):
            t = T[b] - S + s
            row = int(table[b, t // bs]) * bs + t % bs
            written[row] = True
            for n in ("kI", "k", "v", "k_scale", "v_scale"):
                if pk[n] is None:
                    continue
                assert _same(pk[n][row], dev[n][b, t]), (n, b, s)
    keep = (~written).cuda()
    for n, v in before.items():
        a, c = pk[n][keep], v[keep]
        if a.dtype.is_floating_point:
            a = a.view(torch.int16 if a.element_size() == 2 else torch.int32)
            c = c.view(torch.int16 if c.element_size() == 2 else torch.int32)
        assert torch.equal(a, c), n


def test_paged_decode_256k_int8_pool_of_1037_blocks(dsa):
    """The pages' 256K layout: block_size 256 and a pool of 1,037 blocks, of
    which 1,024 hold the 262,144-token INT8 cache, against the dense decode."""
    from dsa_inputs import WORKLOADS
    wl = WORKLOADS["decode_256k_int8"]
    paged_vs_dense(dsa, wl, 256, 13, False, seed=7)


def test_bad_block_entry_is_reported(dsa):
    """A table entry outside the pool for a block that holds visible keys is
    read as block 0 (no memory outside the pool is touched) and reported by
    dsa_read_device_status; the next correct call succeeds."""
    D = dsa
    wl = small_workload(batch=1, q_len=1, total_len=1024, num_q_heads=8, num_kv_heads=2,
                        top_k=1024, kv_dtype="bf16", capacity=1024, seed=67)
    cpu = make_inputs(wl)
    pools, table, nblocks = scatter_to_pool(cpu, [1024], 256, 0, seed=8)
    bad = table.clone()
    bad[0, 2] = nblocks + 5
    dev = {k: _dev(v) for k, v in cpu.items()}
    pk = {k: _dev(v) for k, v in pools.items()}
    p = D.problem_for(wl)
    _, _, ws = run_attn(D, p, dev, pk, False, pages=D.make_pages(bad.cuda(), 256, nblocks))
    with pytest.raises(D.DsaError) as e:
        D.dsa_read_device_status(ws)
    assert e.value.status == D.DSA_ERR_INVALID_ARG
    _, _, ws = run_attn(D, p, dev, pk, False, pages=D.make_pages(table.cuda(), 256, nblocks), ws=ws)
    assert D.dsa_read_device_status(ws) == 0
