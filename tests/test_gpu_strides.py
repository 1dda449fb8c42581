"""K / V caches in another layout through dsa_problem.kv_strides (the
boundary's batch / token / head strides): a BNSH cache [B, Hkv, cap, 128]
gives the same selection and output as the token-major cache holding the same
values (the same arithmetic, so bit for bit), and matches the oracle. Decode
(BF16, FP16, INT8) and prefill (BF16, on the tensor-core path)."""
import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
from dsa_inputs import make_inputs, small_workload
from tests._helpers import TOL_16BIT, TOL_INT8, f64_inputs, rel_l2, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from top_sparse_attention_chunked_gb300 import build_lib, dsa as D
    build_lib.build()
    D.load_library()
    return D


def _run(D, wl, dev, k, v, prefill, strides):
    p = D.problem_for(wl, kv_strides=strides)
    ws = D.alloc_workspace(p, D.DSA_OP_PREFILL if prefill else D.DSA_OP_DECODE)
    ws.fill_(0xA5)
    out = torch.empty(wl.batch, wl.q_len, wl.num_q_heads, 128, dtype=D._TORCH_DT[p.out_dtype],
                      device="cuda")
    idx = torch.empty(wl.batch, wl.q_len, wl.top_k, dtype=torch.int32, device="cuda")
    fn = D.dsa_sparse_attn_prefill if prefill else D.dsa_sparse_attn_decode
    fn(p, dev["q"], dev["qI"], dev["w"], dev["kI"], k, v, dev["k_scale"], dev["v_scale"], idx, out, ws)
    torch.cuda.synchronize()
    assert D.dsa_read_device_status(ws) == 0
    return idx.cpu().numpy(), out.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("kv,q_len,prefill", [("bf16", 4, False), ("fp16", 1, False),
                                              ("int8", 8, False), ("bf16", 64, True),
                                              ("fp16", 40, True)])
def test_bnsh_cache_equals_token_major(dsa, kv, q_len, prefill):
    wl = small_workload(batch=2, q_len=q_len, total_len=3000, num_q_heads=24, num_kv_heads=2,
                        top_k=512, kv_dtype=kv, seed=800 + q_len)
    cpu = make_inputs(wl)
    dev = to_device(cpu)
    B, cap, H = wl.batch, wl.cap, wl.num_kv_heads
    kb = dev["k"].permute(0, 2, 1, 3).contiguous()     # [B, Hkv, cap, 128]
    vb = dev["v"].permute(0, 2, 1, 3).contiguous()
    strides = (H * cap * 128, 128, cap * 128)
    idx0, out0 = _run(dsa, wl, dev, dev["k"], dev["v"], prefill, None)
    idx1, out1 = _run(dsa, wl, dev, kb, vb, prefill, strides)
    assert (idx0 == idx1).all()
    assert np.array_equal(out0, out1), "the layout changed the arithmetic"
    f = f64_inputs(cpu)
    rows = [(0, 0), (1, q_len - 1), (0, q_len // 2)]
    att = O.sparse_attention(f["q"], f["k"], f["v"], idx1, H, f["k_scale"], f["v_scale"], rows=rows)
    sel = np.array(rows)
    tol = TOL_INT8 if kv == "int8" else TOL_16BIT
    assert rel_l2(out1[sel[:, 0], sel[:, 1]], att[sel[:, 0], sel[:, 1]]) <= tol


def test_strides_are_validated(dsa):
    wl = small_workload(batch=1, q_len=1, total_len=300, num_q_heads=8, num_kv_heads=2, top_k=16)
    for bad in [(300 * 2 * 128, 64, 128), (1, 256, 128), (300 * 2 * 128, 256, 0)]:
        p = dsa.problem_for(wl, kv_strides=bad)
        with pytest.raises(dsa.DsaError) as e:   # rejected before anything runs
            dsa.dsa_workspace_size(p, dsa.DSA_OP_DECODE)
        assert e.value.status == dsa.DSA_ERR_INVALID_ARG
    # the cache writes take only the default layout
    p = dsa.problem_for(wl, kv_strides=(300 * 2 * 128, 128, 300 * 128))
    cpu = make_inputs(wl)
    dev = to_device(cpu)
    kI_new = torch.zeros(1, 1, 64, dtype=torch.bfloat16, device="cuda")
    kv_new = torch.zeros(1, 1, 2, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_cache_append(p, kI_new, kv_new, kv_new, dev["kI"], dev["k"], dev["v"])
    assert e.value.status == dsa.DSA_ERR_UNSUPPORTED
