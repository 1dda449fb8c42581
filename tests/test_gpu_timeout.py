"""The device failure path, made to happen without faulting the GPU: the
indexer's pipeline waits are given a zero budget (dsa_set_wait_budget), so
the first wait that is not already complete gives up. The kernel must drain
its copies and tensor-core work, free its tensor memory and report the
timeout in the workspace status word; the next call with the default budget
must be correct (the context stays usable)."""
import numpy as np
import pytest
import torch

from dsa_inputs import make_inputs, small_workload
from tests._helpers import TOL_16BIT, f64_inputs, rel_l2, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from top_sparse_attention_chunked_gb300 import build_lib, dsa as D
    build_lib.build()
    D.load_library()
    return D


@pytest.mark.parametrize("q_len,prefill", [(1, False), (8, False), (64, True)])
def test_wait_that_runs_out_is_reported_and_the_next_call_is_correct(dsa, q_len, prefill):
    import oracle.dsa_oracle as O
    wl = small_workload(batch=2, q_len=q_len, total_len=6000, num_q_heads=24, num_kv_heads=2,
                        top_k=512, kv_dtype="fp16", seed=600 + q_len)
    cpu = make_inputs(wl)
    dev = to_device(cpu)
    p = dsa.problem_for(wl)
    op = dsa.DSA_OP_PREFILL if prefill else dsa.DSA_OP_DECODE
    ws = dsa.alloc_workspace(p, op)
    out = torch.empty(wl.batch, wl.q_len, wl.num_q_heads, 128, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(wl.batch, wl.q_len, wl.top_k, dtype=torch.int32, device="cuda")
    fn = dsa.dsa_sparse_attn_prefill if prefill else dsa.dsa_sparse_attn_decode

    def call():
        fn(p, dev["q"], dev["qI"], dev["w"], dev["kI"], dev["k"], dev["v"], None, None, idx, out, ws)

    try:
        dsa.dsa_set_wait_budget(0)
        call()
        with pytest.raises(dsa.DsaError) as e:
            dsa.dsa_read_device_status(ws)
        assert e.value.status == dsa.DSA_ERR_TIMEOUT
    finally:
        dsa.dsa_set_wait_budget(-1)
    # the context is usable and the same call with the default budget is right
    call()
    assert dsa.dsa_read_device_status(ws) == 0
    f = f64_inputs(cpu)
    gidx = idx.cpu().numpy()
    rows = [(0, 0), (1, q_len - 1)]
    for b, s in rows:
        n = O.visible_len(int(f["total_len"][b]), q_len, s)
        ref = O.index_scores_row(f["qI"][b, s], f["w"][b, s], f["kI"][b], n)
        kth = np.sort(ref)[::-1][wl.top_k - 1]
        diff = np.setxor1d(gidx[b, s], O.topk_select_row(ref, wl.top_k))
        assert (np.abs(ref[diff] - kth) <= 1e-5 * kth).all()
    att = O.sparse_attention(f["q"], f["k"], f["v"], gidx, 2, rows=rows)
    got = out.float().cpu().numpy().astype(np.float64)
    sel = np.array(rows)
    assert rel_l2(got[sel[:, 0], sel[:, 1]], att[sel[:, 0], sel[:, 1]]) <= TOL_16BIT
