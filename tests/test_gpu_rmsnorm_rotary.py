"""GPU parity of dsa_rmsnorm_rotary (through the C ABI) against the oracle's
exact (float64) RMSNorm + rotary embedding. The library computes in fp32 and
rounds once, so each output element must lie within

    E + ulp_out(|exact| + E) / 2,   E = m * (D/2 + 12) * 2^-24,

of the exact value, where m = |y_i cos| + |y_partner sin| for a rotated
element and |y_i| otherwise (y the exact normalised vector): the fp32 sum of
D squares contributes at most D/2 relative units after the square root, and
the scaling, reciprocal, weight and rotation a few more."""
import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
from dsa_inputs import make_rope_inputs, to_f64

pytestmark = pytest.mark.gpu

_MANT = {torch.bfloat16: (7, -126), torch.float16: (10, -14)}
_TDT = {"bf16": torch.bfloat16, "fp16": torch.float16}


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from top_sparse_attention_chunked_gb300 import build_lib, dsa as D
    build_lib.build()
    D.load_library()
    return D


def ulp(v: np.ndarray, dtype) -> np.ndarray:
    mant, emin = _MANT[dtype]
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** emin)))
    return 2.0 ** (np.maximum(e, emin) - mant)


def bound(x64, gamma, eps, cos, sin, pos, r, out_dtype, exact):
    D = x64.shape[-1]
    y = O.rmsnorm_rotary(x64, gamma, eps, None, None, pos, 0)      # normalised, not rotated
    m = np.abs(y)
    h = r // 2
    if h:
        c = np.abs(np.asarray(cos, dtype=np.float64)[np.asarray(pos)])[:, None, :]
        s = np.abs(np.asarray(sin, dtype=np.float64)[np.asarray(pos)])[:, None, :]
        a, b = np.abs(y[..., :h]), np.abs(y[..., h:r])
        m = m.copy()
        m[..., :h] = a * c + b * s
        m[..., h:r] = b * c + a * s
    E = m * (D / 2 + 12) * 2.0 ** -24
    return E + 0.5 * ulp(np.abs(exact) + E, out_dtype)


def run(D, inp, r, eps, y_dtype, in_place=False):
    x = inp["x"].cuda()
    y = x if in_place else torch.empty(x.shape, dtype=y_dtype, device="cuda")
    D.dsa_rmsnorm_rotary(x, inp["gamma"].cuda(), y, eps=eps,
                         cos_cache=None if r == 0 else inp["cos"].cuda(),
                         sin_cache=None if r == 0 else inp["sin"].cuda(),
                         positions=None if r == 0 else inp["positions"].cuda(), rotary_dim=r)
    torch.cuda.synchronize()
    assert D.dsa_last_launches() == ["rmsnorm_rotary_kernel"]
    return y


def check(inp, got, r, eps, max_pos, rows=None):
    x64 = to_f64(inp["x"])
    pos = np.clip(inp["positions"].numpy(), 0, max_pos - 1)
    cos = to_f64(inp["cos"]) if r else None
    sin = to_f64(inp["sin"]) if r else None
    g = to_f64(inp["gamma"])
    if rows is not None:
        x64, pos, got = x64[rows], pos[rows], got[rows]
    exact = O.rmsnorm_rotary(x64, g, eps, cos, sin, pos, r)
    lim = bound(x64, g, eps, cos, sin, pos, r, got.dtype, exact)
    err = np.abs(to_f64(got) - exact)
    bad = np.argwhere(err > lim)
    assert bad.size == 0, (f"{len(bad)} elements outside the fp32 bound; first {tuple(bad[0])}: "
                           f"got {to_f64(got)[tuple(bad[0])]}, exact {exact[tuple(bad[0])]}, "
                           f"bound {lim[tuple(bad[0])]}")


@pytest.mark.parametrize("Dh,r", [(128, 128), (128, 64), (128, 0), (64, 64), (64, 32), (64, 2)])
@pytest.mark.parametrize("xd,yd,cd", [("bf16", "bf16", "fp32"), ("bf16", "fp16", "fp32"),
                                      ("fp16", "fp16", "bf16"), ("fp16", "bf16", "fp32")])
def test_rmsnorm_rotary_parity(dsa, Dh, r, xd, yd, cd):
    N, H, max_pos = 37, 3, 600
    inp = make_rope_inputs(N, H, Dh, r, max_pos, xd, cd, seed=Dh + r, first_pos=550)
    got = run(dsa, inp, r, 1e-6, _TDT[yd]).cpu()   # positions 550..586, the last ones clamped
    check(inp, got, r, 1e-6, max_pos)


def test_rmsnorm_rotary_in_place_matches(dsa):
    inp = make_rope_inputs(64, 4, 128, 128, 256, "bf16", "fp32", seed=3)
    a = run(dsa, inp, 128, 1e-5, torch.bfloat16).cpu()
    b = run(dsa, inp, 128, 1e-5, torch.bfloat16, in_place=True).cpu()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_rmsnorm_rotary_extreme_magnitudes(dsa):
    """BF16 vectors of absmax near 1e30 and 1e-30 (the rescaled paths) and
    eps = 0, where the fp32 sum of squares would overflow or vanish."""
    inp = make_rope_inputs(6, 2, 128, 128, 16, "bf16", "fp32", seed=4)
    x = inp["x"].double()
    for t, scale in enumerate([1e30, 1e-30, 3e37, 1e-36, 1.0, 2.0 ** 60]):
        x[t] = x[t] / x[t].abs().max() * scale
    inp["x"] = x.to(torch.bfloat16)
    got = run(dsa, inp, 128, 0.0, torch.bfloat16).cpu()
    assert torch.isfinite(got.float()).all()
    check(inp, got, 128, 0.0, 16)


def test_rmsnorm_zero_vector_with_eps(dsa):
    inp = make_rope_inputs(4, 2, 64, 64, 8, "fp16", "fp32", seed=5)
    inp["x"][1, 0].zero_()
    got = run(dsa, inp, 64, 1e-6, torch.float16).cpu()
    assert (got[1, 0] == 0).all()
    check(inp, got, 64, 1e-6, 8)


@pytest.mark.parametrize("H,Dh,r", [(24, 128, 128), (16, 64, 32)])
def test_rmsnorm_rotary_prefill_chunk(dsa, H, Dh, r):
    """Full size of the prefill chunk: 8,192 tokens at positions 32,768 ..
    40,959 (the query heads, and the index-query heads with a partial rotary
    width), checked on 512 sampled tokens including the first and last."""
    N, max_pos = 8192, 40960
    inp = make_rope_inputs(N, H, Dh, r, max_pos, "bf16", "fp32", seed=H, first_pos=32768)
    got = run(dsa, inp, r, 1e-6, torch.bfloat16).cpu()
    rng = np.random.default_rng(9)
    rows = np.unique(np.concatenate([[0, N - 1], rng.choice(N, 510, replace=False)]))
    check(inp, got, r, 1e-6, max_pos, rows=rows)
