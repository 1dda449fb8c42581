"""The decode call's selection (the indexer's histograms feeding the cluster
or chunked top-k) must equal the oracle's top-k of the very scores the
indexer computes -- dsa_index_scores on the same inputs gives them bit for
bit -- index for index, -1 padding included. Covers one and many query rows,
ragged lengths, top_k above the context, ties at the threshold, every score
equal (the threshold bin holds the whole row), negative scores, scores of
large magnitude, and the full-size decode shapes."""
import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
from dsa_inputs import WORKLOADS, make_inputs, small_workload
from tests._helpers import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from top_sparse_attention_chunked_gb300 import build_lib, dsa as D
    build_lib.build()
    D.load_library()
    return D


def decode_vs_oracle(D, wl, cpu, total_len=None):
    dev = to_device(cpu)
    lens = total_len if total_len is not None else [int(t) for t in cpu["total_len"]]
    p = D.problem_for(wl, total_len=lens)
    ws = D.alloc_workspace(p, D.DSA_OP_DECODE)
    ws.fill_(0xA5)
    out = torch.empty(wl.batch, wl.q_len, wl.num_q_heads, 128, dtype=D._TORCH_DT[p.out_dtype],
                      device="cuda")
    idx = torch.empty(wl.batch, wl.q_len, wl.top_k, dtype=torch.int32, device="cuda")
    D.dsa_sparse_attn_decode(p, dev["q"], dev["qI"], dev["w"], dev["kI"], dev["k"], dev["v"],
                             dev["k_scale"], dev["v_scale"], idx, out, ws)
    torch.cuda.synchronize()
    assert D.dsa_read_device_status(ws) == 0
    ws2 = D.alloc_workspace(p, D.DSA_OP_INDEX_SCORES)
    sc = torch.zeros(wl.batch, wl.q_len, wl.cap, dtype=torch.float32, device="cuda")
    D.dsa_index_scores(p, dev["qI"], dev["w"], dev["kI"], sc, ws2)
    torch.cuda.synchronize()
    sc = sc.cpu().numpy()
    got = idx.cpu().numpy()
    for b in range(wl.batch):
        for s in range(wl.q_len):
            n = O.visible_len(lens[b], wl.q_len, s)
            ref = O.topk_select_row(sc[b, s, :n].astype(np.float64), wl.top_k)
            assert np.array_equal(got[b, s], ref), f"row ({b}, {s}) differs"
    return got


@pytest.mark.parametrize("B,S,T,k", [(1, 1, 4096, 512), (2, 3, 5000, 700), (3, 8, 20000, 2048),
                                     (1, 16, 9000, 1000), (4, 5, 33000, 2048), (1, 2, 300, 400),
                                     (2, 1, 129, 1), (1, 4, 128, 128)])
def test_decode_select_bitexact(dsa, B, S, T, k):
    wl = small_workload(batch=B, q_len=S, total_len=T, num_q_heads=8, num_kv_heads=2, top_k=k,
                        capacity=max(T, k), seed=1100 + B * 31 + S)
    decode_vs_oracle(dsa, wl, make_inputs(wl))


def test_decode_select_ragged_lengths(dsa):
    wl = small_workload(batch=4, q_len=3, total_len=12000, num_q_heads=8, num_kv_heads=2,
                        top_k=1500, seed=1201)
    decode_vs_oracle(dsa, wl, make_inputs(wl), total_len=[12000, 3, 700, 9001])


def test_decode_select_ties_at_threshold(dsa):
    """Blocks of identical index keys: many exactly equal scores straddle the
    k-th largest, so the lower indices must win inside the tie."""
    wl = small_workload(batch=1, q_len=2, total_len=16000, top_k=1000, seed=1202)
    cpu = make_inputs(wl)
    kI = cpu["kI"]
    g = torch.Generator().manual_seed(5)
    proto = kI[0, torch.randint(0, 16000, (40,), generator=g)]
    kI[0] = proto[torch.randint(0, 40, (16000,), generator=g)]
    decode_vs_oracle(dsa, wl, cpu)


def test_decode_select_all_equal_overflow(dsa):
    """Every score 0: the whole row is one histogram bin, more candidates than
    the cluster select gathers; the lowest indices win."""
    wl = small_workload(batch=1, q_len=1, total_len=50000, top_k=2048, seed=1203)
    cpu = make_inputs(wl)
    cpu["kI"].zero_()
    got = decode_vs_oracle(dsa, wl, cpu)
    assert got[0, 0].tolist() == list(range(2048))


def test_decode_select_negative_scores(dsa):
    """Negative head weights: every score is <= 0."""
    wl = small_workload(batch=2, q_len=2, total_len=7000, top_k=900, seed=1204)
    cpu = make_inputs(wl)
    cpu["w"].neg_()
    decode_vs_oracle(dsa, wl, cpu)


def test_decode_select_large_scores(dsa):
    """Index queries scaled by 2^12: scores far above 2^16."""
    wl = small_workload(batch=1, q_len=3, total_len=9000, top_k=700, seed=1205)
    cpu = make_inputs(wl)
    cpu["qI"] = (cpu["qI"].float() * 4096.0).to(torch.bfloat16)
    decode_vs_oracle(dsa, wl, cpu)


@pytest.mark.parametrize("name", ["decode_4k", "grouped_decode_32k", "decode_128k",
                                  "decode_256k_int8"])
def test_decode_select_full_size(dsa, name):
    wl = WORKLOADS[name]
    decode_vs_oracle(dsa, wl, make_inputs(wl))


@pytest.mark.parametrize("S,zero", [(8, False), (8, True), (16, False)])
def test_decode_select_wide_slices(dsa, S, zero):
    """Rows of up to 200,000 keys. Eight rows: clusters of 16 CTAs would not
    all be resident at once, so the select takes 24 keys a thread in clusters
    of 9. Sixteen rows: no shape fits them in one wave (15 clusters of 9), so
    the fewest keys a thread that launch at all (16, clusters of 13) run in
    waves; the indexer sums 16 queries per block with its histograms. With
    every score equal the threshold bin holds whole rows, beyond the gathered
    list: the refinement path, and the lowest indices win."""
    wl = small_workload(batch=1, q_len=S, total_len=200000, top_k=2048, seed=1206 + S)
    cpu = make_inputs(wl)
    if zero:
        cpu["kI"].zero_()
    got = decode_vs_oracle(dsa, wl, cpu)
    if zero:
        assert all(got[0, s].tolist() == list(range(2048)) for s in range(S))
