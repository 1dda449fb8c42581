"""The built calls composed the way a decoding layer runs them, each stage
checked against the oracle on the previous stage's GPU output:

  1. dsa_rmsnorm_rotary on q, k (head dim 128) and qI, kI (index dim 64) at
     positions T_b - S + s (within the fp32 error bound);
  2. dsa_cache_append of kI, k, v into caches holding T_b - S past rows
     (bit-exact, INT8 quantised on write);
  3. dsa_sparse_attn_decode over the appended caches (selection within the
     tie band, output within the relative-L2 tolerance).
"""
import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
from dsa_inputs import make_append_inputs, make_rope_inputs, to_f64
from tests._helpers import TOL_16BIT, TOL_INT8, check_selection, rel_l2
from tests.test_gpu_rmsnorm_rotary import check as check_rope

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from top_sparse_attention_chunked_gb300 import build_lib, dsa as D
    build_lib.build()
    D.load_library()
    return D


def rope_stage(D, raw, S, T, cap, seed):
    """raw [B, S, H, Dh] bf16 -> rotated [B, S, H, Dh] bf16 at positions T_b - S + s."""
    B, _, H, Dh = raw.shape
    inp = make_rope_inputs(B * S, H, Dh, Dh, cap, "bf16", "fp32", seed=seed)
    inp["x"] = raw.reshape(B * S, H, Dh).contiguous()
    inp["positions"] = torch.tensor([T[b] - S + s for b in range(B) for s in range(S)],
                                    dtype=torch.int32)
    y = torch.empty(B * S, H, Dh, dtype=torch.bfloat16, device="cuda")
    D.dsa_rmsnorm_rotary(inp["x"].cuda(), inp["gamma"].cuda(), y, eps=1e-6,
                         cos_cache=inp["cos"].cuda(), sin_cache=inp["sin"].cuda(),
                         positions=inp["positions"].cuda(), rotary_dim=Dh)
    torch.cuda.synchronize()
    got = y.cpu()
    check_rope(inp, got, Dh, 1e-6, cap)
    return got.reshape(B, S, H, Dh)


@pytest.mark.parametrize("kv", ["fp16", "int8"])
def test_rope_append_decode(dsa, kv):
    D = dsa
    B, S, Hq, Hkv, cap, k = 2, 4, 8, 2, 3072, 256
    T = [3000, 1777]
    g = torch.Generator().manual_seed(71)
    q_raw = torch.randn(B, S, Hq, 128, generator=g).to(torch.bfloat16)
    qI_raw = torch.randn(B, S, 16, 64, generator=g).to(torch.bfloat16)
    w = torch.rand(B, S, 16, generator=g)
    app = make_append_inputs(B, S, Hkv, cap, T, "bf16", kv, seed=72, specials=False)
    # the past rows of the caches are ordinary values, not sentinels
    for b in range(B):
        app["kI"][b, T[b]:] = 0
    # 1. RMSNorm + RoPE of every new vector
    q = rope_stage(D, q_raw, S, T, cap, 1)
    qI = rope_stage(D, qI_raw, S, T, cap, 2)
    app["k_new"] = rope_stage(D, app["k_new"], S, T, cap, 3)
    app["kI_new"] = rope_stage(D, app["kI_new"].reshape(B, S, 1, 64), S, T, cap, 4).reshape(B, S, 64)
    # 2. append into the caches
    p = D.make_problem(batch=B, q_len=S, total_len=T, top_k=k, num_q_heads=Hq,
                       num_kv_heads=Hkv, cache_capacity=cap, q_dtype="bf16", kv_dtype=kv)
    dev = {n: (v.cuda() if isinstance(v, torch.Tensor) else v) for n, v in app.items()}
    D.dsa_cache_append(p, dev["kI_new"], dev["k_new"], dev["v_new"], dev["kI"], dev["k"], dev["v"],
                       dev["k_scale"], dev["v_scale"])
    torch.cuda.synchronize()
    f = {n: to_f64(v) if isinstance(v, torch.Tensor) else v for n, v in app.items()}
    kI_o, k_o, v_o, ks_o, vs_o = O.cache_append(f["kI"], f["k"], f["v"], f["k_scale"], f["v_scale"],
                                                f["kI_new"], f["k_new"], f["v_new"], T, kv)
    assert torch.equal(dev["kI"].cpu(), torch.from_numpy(kI_o).to(torch.bfloat16))
    assert np.array_equal(to_f64(dev["k"].cpu()), k_o) and np.array_equal(to_f64(dev["v"].cpu()), v_o)
    if kv == "int8":
        assert np.array_equal(dev["k_scale"].cpu().numpy(), ks_o.astype(np.float32))
    # 3. decode over the appended caches
    ws = D.alloc_workspace(p, D.DSA_OP_DECODE)
    out = torch.empty(B, S, Hq, 128, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(B, S, k, dtype=torch.int32, device="cuda")
    D.dsa_sparse_attn_decode(p, q.cuda(), qI.cuda(), w.cuda(), dev["kI"], dev["k"], dev["v"],
                             dev["k_scale"], dev["v_scale"], idx, out, ws)
    torch.cuda.synchronize()
    assert D.dsa_read_device_status(ws) == 0
    idx_h = idx.cpu().numpy()
    qI64, w64 = to_f64(qI), w.double().numpy()
    for b in range(B):
        for s in range(S):
            n = O.visible_len(T[b], S, s)
            ref = O.index_scores_row(qI64[b, s], w64[b, s], kI_o[b], n)
            check_selection(ref, idx_h[b, s], k)
    att = O.sparse_attention(to_f64(q), k_o, v_o, idx_h, Hkv, ks_o, vs_o, 0.0)
    err = rel_l2(out.float().cpu().numpy().astype(np.float64), att)
    assert err <= (TOL_INT8 if kv == "int8" else TOL_16BIT), err
