"""dsa_rope_append (one launch) against the chain it replaces: four
dsa_rmsnorm_rotary calls (q and k_new in the q dtype, qI and kI_new in BF16,
positions total_len[b] - q_len + s) and dsa_cache_append. Every output — q,
qI, the four caches — must be equal bit for bit; the chain itself is held to
the oracle by the RMSNorm + RoPE and cache-append tests."""
import pytest
import torch

from dsa_inputs import make_append_inputs, make_rope_inputs

pytestmark = pytest.mark.gpu

_TDT = {"bf16": torch.bfloat16, "fp16": torch.float16}


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from top_sparse_attention_chunked_gb300 import build_lib, dsa as D
    build_lib.build()
    D.load_library()
    return D


def _bits(t):
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16)
    if t.dtype == torch.float32:
        return t.view(torch.int32)
    return t


@pytest.mark.parametrize("qd,kv", [("bf16", "bf16"), ("bf16", "fp16"), ("bf16", "int8"),
                                   ("fp16", "fp16"), ("fp16", "int8")])
@pytest.mark.parametrize("rot,rot_i,cdt", [(128, 64, "fp32"), (64, 32, "bf16"), (0, 0, "fp32")])
def test_rope_append_equals_chain(dsa, qd, kv, rot, rot_i, cdt):
    D = dsa
    B, S, Hq, Hkv, cap = 3, 5, 8, 2, 96
    T = [5, 60, 96]
    max_pos = 90                                   # the last positions are clamped
    g = torch.Generator().manual_seed(81)
    q = (torch.randn(B, S, Hq, 128, generator=g) * 3).to(_TDT[qd])
    qI = torch.randn(B, S, 16, 64, generator=g).to(torch.bfloat16)
    app = make_append_inputs(B, S, Hkv, cap, T, qd, kv, seed=82)
    rq = make_rope_inputs(1, 1, 128, max(rot, 2), max_pos, qd, cdt, seed=83)
    ri = make_rope_inputs(1, 1, 64, max(rot_i, 2), max_pos, "bf16", cdt, seed=84)
    gam = {n: (torch.rand(dim, generator=g) + 0.5).cuda() for n, dim in
           (("q", 128), ("k", 128), ("qI", 64), ("kI", 64))}
    cos = rq["cos"].cuda() if rot else None
    sin = rq["sin"].cuda() if rot else None
    cos_i = ri["cos"].cuda() if rot_i else None
    sin_i = ri["sin"].cuda() if rot_i else None
    if rot:
        cos, sin = cos[:, :rot // 2].contiguous(), sin[:, :rot // 2].contiguous()
    if rot_i:
        cos_i, sin_i = cos_i[:, :rot_i // 2].contiguous(), sin_i[:, :rot_i // 2].contiguous()
    pos = torch.tensor([T[b] - S + s for b in range(B) for s in range(S)], dtype=torch.int32).cuda()
    p = D.make_problem(batch=B, q_len=S, total_len=T, top_k=8, num_q_heads=Hq, num_kv_heads=Hkv,
                       cache_capacity=cap, q_dtype=qd, kv_dtype=kv)
    caches = ("kI", "k", "v", "k_scale", "v_scale")

    # the chain
    c = {n: (app[n].cuda() if app[n] is not None else None) for n in caches}
    qa, qIa = q.cuda(), qI.cuda()
    k_new, kI_new, v_new = app["k_new"].cuda(), app["kI_new"].cuda(), app["v_new"].cuda()
    for x, gm, cs, sn, r in ((qa.view(B * S, Hq, 128), gam["q"], cos, sin, rot),
                             (qIa.view(B * S, 16, 64), gam["qI"], cos_i, sin_i, rot_i)):
        D.dsa_rmsnorm_rotary(x, gm, x, eps=1e-5, cos_cache=cs, sin_cache=sn,
                             positions=pos if r else None, rotary_dim=r)
    k_rot = torch.empty_like(k_new)
    kI_rot = torch.empty_like(kI_new)
    D.dsa_rmsnorm_rotary(k_new.view(B * S, Hkv, 128), gam["k"], k_rot.view(B * S, Hkv, 128), eps=1e-5,
                         cos_cache=cos, sin_cache=sin, positions=pos if rot else None, rotary_dim=rot)
    D.dsa_rmsnorm_rotary(kI_new.view(B * S, 1, 64), gam["kI"], kI_rot.view(B * S, 1, 64), eps=1e-5,
                         cos_cache=cos_i, sin_cache=sin_i, positions=pos if rot_i else None,
                         rotary_dim=rot_i)
    D.dsa_cache_append(p, kI_rot, k_rot, v_new, c["kI"], c["k"], c["v"], c["k_scale"], c["v_scale"])

    # one launch
    f = {n: (app[n].cuda() if app[n] is not None else None) for n in caches}
    qb, qIb = q.cuda(), qI.cuda()
    D.dsa_rope_append(p, qb, qIb, k_new, kI_new, v_new, f["kI"], f["k"], f["v"], f["k_scale"],
                      f["v_scale"], gam["q"], gam["k"], gam["qI"], gam["kI"], eps=1e-5,
                      cos=cos, sin=sin, cos_index=cos_i, sin_index=sin_i)
    torch.cuda.synchronize()
    assert D.dsa_last_launches() == ["rope_append_kernel"]
    assert torch.equal(_bits(qb), _bits(qa)), "q"
    assert torch.equal(_bits(qIb), _bits(qIa)), "qI"
    for n in caches:
        if c[n] is not None:
            assert torch.equal(_bits(f[n]), _bits(c[n])), n
    # the new-token inputs are read only
    assert torch.equal(_bits(k_new), _bits(app["k_new"].cuda()))
    assert torch.equal(_bits(kI_new), _bits(app["kI_new"].cuda()))
