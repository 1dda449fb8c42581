"""dsa_topk_noalloc: the workspace-free top-k, for callers that cannot
allocate device memory (operator plugins handed only their tensors, engines
whose memory is fixed at start-up, latency paths that cannot take
cudaMalloc's device synchronisation). Its scratch is a static device array in
the library. Checked through the C ABI against dsa_topk, bit for bit (the
top-k tolerance), on two calls in a row that share that scratch. This file
is collected last so a stop-at-first-failure run has done everything else."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def D():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from top_sparse_attention_chunked_gb300 import build_lib, dsa
    build_lib.build()
    dsa.load_library()
    return dsa


def _scores(shape, kind, seed):
    g = torch.Generator().manual_seed(seed)
    if kind == "ties":
        return torch.randint(-2, 3, shape, generator=g).float()
    return torch.randn(shape, generator=g) * 5


def test_noalloc_topk_matches_workspace_topk_twice(D):
    cases = [  # (batch, q_len, total_len, cap, top_k, kind)
        (1, 1, 131072, 131072, 2048, "cont"),
        (2, 4, [9000, 5000], 9100, 700, "ties"),
    ]
    for i, (B, S, T, cap, k, kind) in enumerate(cases):
        Ts = T if isinstance(T, list) else [T] * B
        p = D.make_problem(batch=B, q_len=S, total_len=Ts, top_k=k, cache_capacity=cap)
        sc = _scores((B, S, cap), kind, 100 + i).cuda()
        ref = torch.full((B, S, k), -7, dtype=torch.int32, device="cuda")
        ws = D.alloc_workspace(p, D.DSA_OP_TOPK)
        D.dsa_topk(p, sc, ref, ws)
        got = torch.full((B, S, k), -9, dtype=torch.int32, device="cuda")
        D.dsa_topk_noalloc(p, sc, got)
        torch.cuda.synchronize()
        assert torch.equal(got.cpu(), ref.cpu()), f"call {i}: differs from dsa_topk"


def test_noalloc_topk_capacity_above_its_scratch_length(D):
    """A cache capacity beyond the scratch's row length is fine while the
    visible length stays within it (the kernels index only visible keys);
    one row also against the oracle's selection directly."""
    import oracle.dsa_oracle as O
    B, S, cap, T, k = 1, 2, 200000, 131072, 2048
    p = D.make_problem(batch=B, q_len=S, total_len=[T], top_k=k, cache_capacity=cap)
    sc = _scores((B, S, cap), "cont", 501).cuda()
    sc[:, :, T:] = float("nan")   # never read
    ref = torch.full((B, S, k), -7, dtype=torch.int32, device="cuda")
    ws = D.alloc_workspace(p, D.DSA_OP_TOPK)
    D.dsa_topk(p, sc, ref, ws)
    for _ in range(2):
        got = torch.full((B, S, k), -9, dtype=torch.int32, device="cuda")
        D.dsa_topk_noalloc(p, sc, got)
        torch.cuda.synchronize()
        assert torch.equal(got.cpu(), ref.cpu())
    row = sc[0, 1, :T].double().cpu().numpy()
    assert (got[0, 1].cpu().numpy() == O.topk_select_row(row, k)).all()


def test_noalloc_topk_rejects_sizes_beyond_its_scratch(D):
    sc = torch.zeros(1, 9, 64, device="cuda")
    idx = torch.zeros(1, 9, 8, dtype=torch.int32, device="cuda")
    p = D.make_problem(batch=1, q_len=9, total_len=64, top_k=8)
    with pytest.raises(D.DsaError) as e:
        D.dsa_topk_noalloc(p, sc, idx)
    assert e.value.status == D.DSA_ERR_UNSUPPORTED
    p = D.make_problem(batch=1, q_len=1, total_len=131073, top_k=8)
    sc = torch.zeros(1, 1, 131073, device="cuda")
    idx = torch.zeros(1, 1, 8, dtype=torch.int32, device="cuda")
    with pytest.raises(D.DsaError) as e:
        D.dsa_topk_noalloc(p, sc, idx)
    assert e.value.status == D.DSA_ERR_UNSUPPORTED
