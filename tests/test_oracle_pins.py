"""Pins for the CPU oracle: each check ties an oracle function to something
other than itself -- values printed on the pages, hand-worked fixtures,
closed forms, invariants, a library routine in a special case, or brute force
on tiny inputs. The mutation tests at the end plant plausible mistakes in a
copy of the oracle and assert that some pin catches each one.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
from dsa_inputs import make_inputs, small_workload, to_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _num(x):
    return float(x) if not isinstance(x, str) else float(x)


# ---------------------------------------------------------------------------
# reusable checks (also driven by the mutation tests)
# ---------------------------------------------------------------------------
def check_topk_fixture(mod):
    for case in _load("topk_tiny.json")["cases"]:
        s = np.array([_num(x) for x in case["scores"]], dtype=np.float64)
        got = mod.topk_select_row(s, case["k"])
        assert got.tolist() == case["expected"], (case, got)


def is_valid_topk(scores, k, sel):
    """Definition of the selection, checked by properties only: right count,
    ascending then -1 padding, every selected >= every unselected, and on the
    threshold value the selected indices all precede the unselected ones."""
    n = len(scores)
    keff = min(k, n)
    sel = np.asarray(sel)
    if sel.shape != (k,) or (sel[keff:] != -1).any():
        return False
    chosen = sel[:keff]
    if (chosen < 0).any() or (chosen >= n).any():
        return False
    if keff > 1 and not (np.diff(chosen) > 0).all():
        return False
    rest = np.setdiff1d(np.arange(n), chosen)
    if len(rest) == 0 or keff == 0:
        return True
    vs = scores[chosen] + 0.0
    vr = scores[rest] + 0.0
    if vs.min() < vr.max():
        return False
    thr = vs.min()
    if vr.max() == thr:
        if chosen[vs == thr].max() > rest[vr == thr].min():
            return False
    return True


def brute_force_topk(scores, k):
    """k rounds of 'take the largest remaining value, lowest index first'."""
    left = list(range(len(scores)))
    picked = []
    for _ in range(min(k, len(scores))):
        best = left[0]
        for i in left[1:]:
            if scores[i] + 0.0 > scores[best] + 0.0:
                best = i
        picked.append(best)
        left.remove(best)
    out = sorted(picked) + [-1] * (k - len(picked))
    return np.array(out)


def check_topk_bruteforce(mod, trials=300):
    rng = np.random.default_rng(0)
    for _ in range(trials):
        n = int(rng.integers(1, 10))
        s = rng.integers(0, 4, size=n).astype(np.float64)
        for k in (1, max(1, n // 2), n, n + 3):
            got = mod.topk_select_row(s, k)
            assert got.tolist() == brute_force_topk(s, k).tolist(), (s, k, got)


def check_indexer_fixture(mod):
    fx = _load("indexer_tiny.json")
    got = mod.index_scores_row(np.array(fx["qI"]), np.array(fx["w"]),
                               np.array(fx["kI"]), len(fx["kI"]))
    assert np.array_equal(got, np.array(fx["expected"])), got


def check_indexer_closed_form(mod):
    """kI_t = c_t u and qI_h = a_h u give qI_h.kI_t = a_h c_t |u|^2, so
    score_t = sum_h w_h max(0, a_h c_t |u|^2) -- with mixed signs of a_h and c_t
    this separates ReLU-per-head from ReLU-after-the-sum and the head weights."""
    rng = np.random.default_rng(1)
    HI, DI, n = 16, 64, 40
    u = rng.standard_normal(DI)
    a = rng.standard_normal(HI)
    c = rng.standard_normal(n)
    w = rng.uniform(0, 1, HI)
    qI = a[:, None] * u[None, :]
    kI = c[:, None] * u[None, :]
    uu = float(u @ u)
    expect = np.array([sum(w[h] * max(0.0, a[h] * c[t] * uu) for h in range(HI))
                       for t in range(n)])
    got = mod.index_scores_row(qI, w, kI, n)
    np.testing.assert_allclose(got, expect, rtol=1e-12, atol=1e-12)


def check_indexer_loops(mod):
    """Pure-Python loops on a tiny random case, including the causal limits of
    S > 1 queries (R1) and a capacity larger than the live length."""
    rng = np.random.default_rng(2)
    B, S, HI, DI, cap = 2, 3, 3, 5, 9
    T = np.array([7, 4])
    qI = rng.standard_normal((B, S, HI, DI))
    w = rng.uniform(0, 1, (B, S, HI))
    kI = rng.standard_normal((B, cap, DI))
    got = mod.index_scores(qI, w, kI, T)
    for b in range(B):
        for s in range(S):
            n = T[b] - S + s + 1
            for t in range(cap):
                if t >= n:
                    assert np.isnan(got[b, s, t])
                    continue
                tot = 0.0
                for h in range(HI):
                    d = 0.0
                    for i in range(DI):
                        d += qI[b, s, h, i] * kI[b, t, i]
                    tot += w[b, s, h] * (d if d > 0 else 0.0)
                assert abs(got[b, s, t] - tot) <= 1e-12 * (1 + abs(tot))


def torch_dense_reference(q, k, v, T, softmax_scale=None):
    """Dense causal GQA attention via torch's scaled_dot_product_attention in
    float64 (the library routine the sparse method reduces to when every
    visible key is selected)."""
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    out = np.zeros(q.shape)
    for b in range(B):
        n_all = int(T[b])
        qt = torch.from_numpy(q[b]).permute(1, 0, 2)                 # [Hq,S,D]
        kt = torch.from_numpy(k[b, :n_all]).permute(1, 0, 2)          # [Hkv,n,D]
        vt = torch.from_numpy(v[b, :n_all]).permute(1, 0, 2)
        kt = kt.repeat_interleave(G, dim=0)
        vt = vt.repeat_interleave(G, dim=0)
        pos = torch.arange(n_all - S, n_all)
        mask = torch.arange(n_all)[None, :] <= pos[:, None]           # [S,n]
        o = torch.nn.functional.scaled_dot_product_attention(
            qt, kt, vt, attn_mask=mask, scale=softmax_scale)
        out[b] = o.permute(1, 0, 2).numpy()
    return out


def check_dense_equivalence(mod):
    wl = small_workload(batch=2, q_len=3, total_len=50, num_q_heads=6,
                        num_kv_heads=2, top_k=64, seed=11)
    inp = {k: to_f64(v) if isinstance(v, torch.Tensor) else v
           for k, v in make_inputs(wl).items()}
    res = mod.sparse_attention_step(inp, wl.num_kv_heads, wl.top_k)
    ref = torch_dense_reference(inp["q"], inp["k"], inp["v"], inp["total_len"])
    np.testing.assert_allclose(res["out"], ref, rtol=1e-10, atol=1e-12)


def check_worked_example(mod, spacing=0):
    """PR #33847's case through the oracle's attention: q = 88 e_0, K codes
    0 and e_0 (k_scale 1), V codes 1 and 0 with value scale 2^120, softmax
    scale 1. ``spacing`` inserts keys with logit -1000 between the two
    candidates (weights e^-1088 are exactly 0 in float64)."""
    fx = _load("int8_rescale_worked_example.json")
    D = 128
    m = 2 + spacing
    q = np.zeros((1, 1, 1, D))
    q[0, 0, 0, 0] = 88.0
    k = np.zeros((1, m, 1, D))
    k[0, m - 1, 0, 0] = 1.0
    k[0, 1:m - 1, 0, 0] = -1000.0 / 88.0
    v = np.zeros((1, m, 1, D))
    v[0, 0, 0, :] = fx["value_codes"][0]
    v[0, m - 1, 0, :] = fx["value_codes"][1]
    ks = np.ones((1, m, 1))
    vs = np.full((1, m, 1), 2.0 ** fx["value_scale_log2"])
    idx = np.arange(m)[None, None, :]
    out = mod.sparse_attention(q, k, v, idx, 1, ks, vs, softmax_scale=1.0)
    expect = 2.0 ** 120 * math.exp(-88) / (1 + math.exp(-88))
    np.testing.assert_allclose(out[0, 0, 0], expect, rtol=1e-12)
    assert round(out[0, 0, 0, 0], 4) == pytest.approx(fx["printed_value"], abs=5e-4)


# ---------------------------------------------------------------------------
# the pins
# ---------------------------------------------------------------------------
def test_topk_golden_fixture():
    check_topk_fixture(O)


def test_topk_bruteforce_tiny():
    check_topk_bruteforce(O)


@pytest.mark.parametrize("seed", range(5))
def test_topk_invariants_tie_heavy(seed):
    rng = np.random.default_rng(100 + seed)
    for _ in range(40):
        n = int(rng.integers(1, 300))
        s = rng.integers(-3, 4, size=n).astype(np.float64)
        if rng.random() < 0.3:
            s[rng.integers(0, n, size=max(1, n // 5))] = -0.0
        for k in (1, max(1, n // 3), n, n + 7):
            assert is_valid_topk(s, k, O.topk_select_row(s, k))


def test_topk_distinct_values_matches_argpartition():
    rng = np.random.default_rng(3)
    for n in (1, 17, 2048, 5000):
        s = rng.permutation(n).astype(np.float64) * 0.5 - 7.0
        for k in (1, min(n, 512), n):
            expect = np.sort(np.argpartition(-s, k - 1)[:k])
            assert O.topk_select_row(s, k)[:k].tolist() == expect.tolist()


def test_indexer_golden_fixture():
    check_indexer_fixture(O)


def test_indexer_closed_form():
    check_indexer_closed_form(O)


def test_indexer_loops_causal():
    check_indexer_loops(O)


def test_visible_len_positions():
    assert O.visible_len(4096, 1, 0) == 4096
    assert [O.visible_len(40960, 8192, s) for s in (0, 8191)] == [32769, 40960]
    with pytest.raises(ValueError):
        O.visible_len(3, 5, 0)


def test_dense_equivalence_when_topk_covers_all():
    check_dense_equivalence(O)


def test_worked_example_large_value_scale():
    for spacing in (0, 1, 15, 40):
        check_worked_example(O, spacing)


def test_permutation_invariance():
    wl = small_workload(batch=1, q_len=1, total_len=300, num_q_heads=8,
                        num_kv_heads=2, top_k=37, seed=5)
    inp = {k: to_f64(v) if isinstance(v, torch.Tensor) else v
           for k, v in make_inputs(wl).items()}
    base = O.sparse_attention_step(inp, 2, wl.top_k)
    perm = np.random.default_rng(0).permutation(wl.total_len)
    p = dict(inp)
    for key in ("kI", "k", "v"):
        p[key] = inp[key][:, perm]
    got = O.sparse_attention_step(p, 2, wl.top_k)
    np.testing.assert_allclose(got["out"], base["out"], rtol=1e-12, atol=1e-13)
    # the selected rows are the same rows, renamed by the permutation
    sel_b = set(base["idx"][0, 0].tolist())
    sel_p = set(perm[got["idx"][0, 0]].tolist())
    assert sel_b == sel_p


def test_uniform_query_gives_mean_of_selected_values():
    wl = small_workload(batch=2, q_len=2, total_len=200, num_q_heads=4,
                        num_kv_heads=2, top_k=50, seed=6)
    inp = {k: to_f64(v) if isinstance(v, torch.Tensor) else v
           for k, v in make_inputs(wl).items()}
    inp["q"] = np.zeros_like(inp["q"])
    res = O.sparse_attention_step(inp, 2, wl.top_k)
    for b in range(2):
        for s in range(2):
            sel = res["idx"][b, s]
            sel = sel[sel >= 0]
            for h in range(4):
                g = h // 2
                np.testing.assert_allclose(res["out"][b, s, h],
                                           inp["v"][b, sel, g].mean(axis=0),
                                           rtol=1e-12, atol=1e-14)


def test_zero_index_keys_select_the_prefix():
    wl = small_workload(batch=1, q_len=4, total_len=100, top_k=30, seed=8)
    inp = {k: to_f64(v) if isinstance(v, torch.Tensor) else v
           for k, v in make_inputs(wl).items()}
    inp["kI"] = np.zeros_like(inp["kI"])
    res = O.sparse_attention_step(inp, 2, 30)
    assert (res["scores"][0, 0, :97] == 0).all()
    for s in range(4):
        assert res["idx"][0, s].tolist() == list(range(30))
    # top_k beyond the visible length: everything, then -1
    res = O.sparse_attention_step(inp, 2, 99)
    assert res["idx"][0, 0].tolist() == list(range(97)) + [-1, -1]


def test_int8_path_reduces_to_plain_values():
    rng = np.random.default_rng(9)
    B, S, Hq, Hkv, D, m = 1, 2, 4, 2, 128, 60
    q = rng.standard_normal((B, S, Hq, D))
    codes_k = rng.integers(-127, 128, (B, m, Hkv, D)).astype(np.float64)
    codes_v = rng.integers(-127, 128, (B, m, Hkv, D)).astype(np.float64)
    idx = np.tile(np.arange(0, m, 2), (B, S, 1))
    ones = np.ones((B, m, Hkv))
    a = O.sparse_attention(q, codes_k, codes_v, idx, Hkv, ones, ones)
    b = O.sparse_attention(q, codes_k, codes_v, idx, Hkv)
    np.testing.assert_array_equal(a, b)
    # and a power-of-two scale scales the values exactly
    a2 = O.sparse_attention(q, codes_k, codes_v, idx, Hkv, ones, 4 * ones)
    np.testing.assert_array_equal(a2, 4 * b)


def test_full_step_on_workload_shapes():
    wl = small_workload(batch=2, q_len=3, total_len=700, top_k=100,
                        kv_dtype="int8", seed=10)
    inp = {k: to_f64(v) if isinstance(v, torch.Tensor) else v
           for k, v in make_inputs(wl).items()}
    res = O.sparse_attention_step(inp, 2, 100)
    assert res["out"].shape == (2, 3, 8, 128)
    for b in range(2):
        for s in range(3):
            n = 700 - 3 + s + 1
            assert is_valid_topk(res["scores"][b, s, :n], 100, res["idx"][b, s])


# ---------------------------------------------------------------------------
# cache append (R11)
# ---------------------------------------------------------------------------
def check_quantize_fixture(mod):
    for case in _load("int8_quantize_tiny.json")["cases"]:
        codes, scale = mod.quantize_row_int8(np.array(case["x"], dtype=np.float64))
        assert codes.tolist() == case["codes"], (case, codes)
        assert float(scale) == case["scale"], (case, scale)


def check_quantize_invariants(mod):
    rng = np.random.default_rng(11)
    for _ in range(200):
        x = (rng.standard_normal(128) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
        codes, scale = mod.quantize_row_int8(x)
        amax = np.abs(x).max()
        # the absmax element maps to +-127 and every code is within range
        assert np.abs(codes.astype(np.int32)).max() == 127
        # scale * 127 recovers the absmax to fp32 rounding
        assert abs(float(scale) * 127.0 - float(amax)) <= 1e-6 * float(amax)
        # rounding to nearest: every value within half a step (plus fp32 slack)
        err = np.abs(x.astype(np.float64) - codes.astype(np.float64) * float(scale))
        assert err.max() <= 0.5 * float(scale) * (1 + 1e-5)


def check_append_positions(mod):
    """B = 2, S = 2, cap = 6, T = (5, 3): the new tokens land in rows 3, 4 of
    sequence 0 and rows 1, 2 of sequence 1; every other row keeps its value."""
    B, S, cap, Hkv = 2, 2, 6, 1
    kI = np.full((B, cap, 2), -9.0)
    k = np.full((B, cap, Hkv, 2), -9.0)
    v = np.full((B, cap, Hkv, 2), -9.0)
    kI_new = np.arange(B * S * 2, dtype=np.float64).reshape(B, S, 2)
    k_new = 10 + np.arange(B * S * Hkv * 2, dtype=np.float64).reshape(B, S, Hkv, 2)
    v_new = 20 + np.arange(B * S * Hkv * 2, dtype=np.float64).reshape(B, S, Hkv, 2)
    out = mod.cache_append(kI, k, v, None, None, kI_new, k_new, v_new, [5, 3], "bf16")
    kI2, k2, v2 = out[0], out[1], out[2]
    rows = {0: (3, 4), 1: (1, 2)}
    for b in range(B):
        for t in range(cap):
            if t in rows[b]:
                s_ = rows[b].index(t)
                assert kI2[b, t].tolist() == kI_new[b, s_].tolist()
                assert k2[b, t].tolist() == k_new[b, s_].tolist()
                assert v2[b, t].tolist() == v_new[b, s_].tolist()
            else:
                assert (kI2[b, t] == -9).all() and (k2[b, t] == -9).all() and (v2[b, t] == -9).all()


def check_round_to(mod):
    """Round-to-nearest-even into the 16-bit formats, worked from their
    definitions: FP16 has 10 fraction bits, largest finite 65,504, subnormal
    step 2^-24; BF16 has 7 fraction bits and FP32's exponent range."""
    f16 = mod.round_to(np.array([65504.0, 65519.0, 65520.0, 1e-6, 2.0 ** -25, 3 * 2.0 ** -25,
                                 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11]), "fp16")
    assert f16[0] == 65504.0
    assert f16[1] == 65504.0                      # below the midpoint to 2^16
    assert np.isposinf(f16[2])                    # the midpoint: ties to even = 2^16, overflow
    assert f16[3] == 17 * 2.0 ** -24              # 1e-6 / 2^-24 = 16.78
    assert f16[4] == 0.0                          # half the smallest step: ties to even (0)
    assert f16[5] == 2 * 2.0 ** -24               # 1.5 steps: ties to even (2)
    assert f16[6] == 1.0                          # 1 + half an ulp: ties to even
    assert f16[7] == 1.0 + 2.0 ** -9              # 1 + 1.5 ulp: ties to even (2 ulp)
    bf = mod.round_to(np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 70000.0, 3.0e38]), "bf16")
    assert bf[0] == 1.0 and bf[1] == 1.0 + 2.0 ** -6
    assert bf[2] == 70144.0                       # 70000 = 1.068 * 2^16: steps of 2^9
    assert bf[3] == 226 * 2.0 ** 120               # 3e38 / 2^120 = 225.7: the nearest step


def test_round_to_ieee_cases():
    check_round_to(O)


def test_quantize_golden_fixture():
    check_quantize_fixture(O)


def test_quantize_invariants():
    check_quantize_invariants(O)


def test_append_positions():
    check_append_positions(O)


def test_append_int8_dequantises_to_within_half_a_step():
    rng = np.random.default_rng(3)
    B, S, cap, Hkv = 1, 3, 8, 2
    new = rng.standard_normal((B, S, Hkv, 128)).astype(np.float32).astype(np.float64)
    zeros = np.zeros((B, cap, Hkv, 128))
    sc = np.zeros((B, cap, Hkv))
    _, k2, _, ks2, _ = O.cache_append(np.zeros((B, cap, 64)), zeros, zeros, sc, sc,
                                      np.zeros((B, S, 64)), new, new, [8], "int8")
    deq = O.dequantize(k2[0, 5:8], ks2[0, 5:8])
    assert np.abs(deq - new[0]).max() <= 0.5 * ks2[0, 5:8].max() * (1 + 1e-5)


# ---------------------------------------------------------------------------
# paged caches (R12)
# ---------------------------------------------------------------------------
def check_gather_pages(mod):
    """block_size 2, pool rows labelled 10*row; table [[2, 0], [1, 3]]:
    sequence 0 is pool rows 4, 5, 0 (3 tokens), sequence 1 rows 2, 3, 6, 7."""
    pool = (10.0 * np.arange(8)).reshape(8, 1)
    view = mod.gather_pages(pool, np.array([[2, 0], [1, 3]]), 2, [3, 4])
    assert view[:, :, 0].tolist() == [[40.0, 50.0, 0.0, 0.0], [20.0, 30.0, 60.0, 70.0]]


def test_gather_pages_hand_case():
    check_gather_pages(O)


# ---------------------------------------------------------------------------
# RMSNorm + rotary embedding (R13)
# ---------------------------------------------------------------------------
def check_rope_fixture(mod):
    for c in _load("rmsnorm_rotary_tiny.json")["cases"]:
        out = mod.rmsnorm_rotary(np.array([c["x"]], dtype=np.float64), c["gamma"], c["eps"],
                                 np.array(c["cos"]), np.array(c["sin"]), [c["position"]],
                                 c["rotary_dim"])
        assert np.allclose(out[0], np.array(c["out"]), rtol=0, atol=1e-12), (c, out)


def check_rope_complex(mod):
    """The rotation as a complex product: (y_i + i y_{i+h}) * exp(i theta_{p,i}),
    with y from the vector norm (||x|| / sqrt(D)) instead of the mean square."""
    rng = np.random.default_rng(5)
    N, H, D, r = 6, 3, 16, 12
    x = rng.standard_normal((N, H, D))
    gamma = rng.uniform(0.5, 1.5, D)
    theta = rng.uniform(-np.pi, np.pi, (9, r // 2))
    pos = rng.integers(0, 9, N)
    eps = 1e-3
    out = mod.rmsnorm_rotary(x, gamma, eps, np.cos(theta), np.sin(theta), pos, r)
    rms = np.sqrt(np.linalg.norm(x, axis=-1, keepdims=True) ** 2 / D + eps)
    y = gamma * x / rms
    h = r // 2
    z = (y[..., :h] + 1j * y[..., h:r]) * np.exp(1j * theta[pos])[:, None, :]
    assert np.allclose(out[..., :h], z.real, atol=1e-12)
    assert np.allclose(out[..., h:r], z.imag, atol=1e-12)
    assert np.allclose(out[..., r:], y[..., r:], atol=1e-12)


def check_rope_scale_invariance(mod):
    """With eps = 0 the output does not depend on the input's scale, and at an
    angle of zero it is x * gamma / rms(x)."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal((4, 2, 8))
    g = rng.uniform(0.5, 2.0, 8)
    ones, zeros = np.ones((3, 4)), np.zeros((3, 4))
    a = mod.rmsnorm_rotary(x, g, 0.0, ones, zeros, [0, 1, 2, 0], 8)
    b = mod.rmsnorm_rotary(37.5 * x, g, 0.0, ones, zeros, [0, 1, 2, 0], 8)
    assert np.allclose(a, b, atol=1e-12)
    assert np.allclose(a, x * g / np.sqrt(np.mean(x * x, axis=-1, keepdims=True)), atol=1e-12)


def test_rope_golden_fixture():
    check_rope_fixture(O)


def test_rope_complex_rotation():
    check_rope_complex(O)


def test_rope_scale_invariance():
    check_rope_scale_invariance(O)


# ---------------------------------------------------------------------------
# floating auxiliary K/V (R14)
# ---------------------------------------------------------------------------
def _aux_case(case):
    f = lambda rows: np.array([[_num(x) for x in r] for r in rows], dtype=np.float64)
    T, S = case["total_len"], case["q_len"]
    q = f(case["q"]).reshape(1, S, 1, -1)
    k = f(case["k_cache"]).reshape(1, T, 1, -1)
    v = f(case["v_cache"]).reshape(1, T, 1, -1)
    ka = f(case["k_aux"]).reshape(1, S, 1, -1)
    va = f(case["v_aux"]).reshape(1, S, 1, -1)
    if "idx_rows" in case:
        idx = np.array(case["idx_rows"], dtype=np.int64).reshape(1, S, -1)
    else:
        idx = np.array(case["idx"], dtype=np.int64).reshape(1, S, -1)
    return q, k, v, ka, va, idx, np.array([T])


def check_aux_fixture(mod):
    cases = _load("aux_kv_tiny.json")["cases"]
    for case in cases:
        q, k, v, ka, va, idx, T = _aux_case(case)
        with np.errstate(invalid="ignore", over="ignore"):
            got = mod.sparse_attention_aux(q, k, v, idx, 1, ka, va, T,
                                           softmax_scale=case["softmax_scale"])
        if "expected" in case:
            assert np.allclose(got[0, 0, 0], case["expected"], rtol=0, atol=1e-9), (case["what"], got)
        elif "expected_rows" in case:
            for s, exp in enumerate(case["expected_rows"]):
                assert np.allclose(got[0, s, 0], exp, rtol=1e-15, atol=0), (case["what"], got)
        else:
            e = math.e
            assert np.allclose(got[0, 0, 0], [2 / (1 + e), 2 * e / (1 + e)], rtol=1e-15), (case["what"], got)


def check_aux_reduces_to_cache(mod):
    """With k_aux / v_aux equal to the cache's new rows the result is the plain
    sparse attention (ties the aux row of key t to cache row t, R1)."""
    wl = small_workload(batch=2, q_len=3, total_len=300, num_q_heads=8, num_kv_heads=2,
                        top_k=64, kv_dtype="bf16", seed=44)
    cpu = make_inputs(wl)
    f = {k: to_f64(v) for k, v in cpu.items() if v is not None and k != "total_len"}
    T = cpu["total_len"].numpy()
    idx = mod.topk(mod.index_scores(f["qI"], f["w"], f["kI"], T), T, 64)
    # make sure the new tokens are selected (the oracle picks by score)
    for b in range(2):
        for s in range(3):
            row = idx[b, s]
            row[:s + 1] = np.arange(T[b] - 3, T[b] - 3 + s + 1)
            idx[b, s] = np.sort(row)
    ka = np.stack([f["k"][b, T[b] - 3:T[b]] for b in range(2)])
    va = np.stack([f["v"][b, T[b] - 3:T[b]] for b in range(2)])
    plain = mod.sparse_attention(f["q"], f["k"], f["v"], idx, 2)
    got = mod.sparse_attention_aux(f["q"], f["k"], f["v"], idx, 2, ka, va, T)
    assert np.allclose(got, plain, rtol=1e-13, atol=0)
    # and a perturbed aux row changes exactly the rows that selected it
    ka2 = ka.copy()
    ka2[1, 0] += 1.0
    got2 = mod.sparse_attention_aux(f["q"], f["k"], f["v"], idx, 2, ka2, va, T)
    changed = ~np.isclose(got2, got, rtol=1e-13, atol=0).all(axis=(2, 3))
    expect = np.zeros((2, 3), dtype=bool)
    expect[1, :] = True   # every query of sequence 1 selected key T-3 (aux row 0)
    assert (changed == expect).all(), changed


def test_aux_golden_fixture():
    check_aux_fixture(O)


def test_aux_reduces_to_plain_attention():
    check_aux_reduces_to_cache(O)


# ---------------------------------------------------------------------------
# mutation tests: plant a mistake in a copy of the oracle, a pin must fail
# ---------------------------------------------------------------------------
class _Mutant:
    """A namespace that forwards to the oracle except for replaced functions;
    replaced functions are resolved through this namespace, so a mutant inner
    helper reaches the outer functions that call it."""

    def __init__(self, **repl):
        g = dict(O.__dict__)
        g.update(repl)
        for name, f in O.__dict__.items():
            if name in repl or not callable(f) or getattr(f, "__module__", "") != O.__name__:
                continue
            if hasattr(f, "__code__"):
                g[name] = type(f)(f.__code__, g, f.__name__, f.__defaults__, f.__closure__)
        self._ns = g

    def __getattr__(self, name):
        return self._ns[name]


def _fails(check, mod):
    try:
        check(mod)
    except AssertionError:
        return True
    return False


def test_mutant_relu_after_head_sum_is_caught():
    def bad(qI_s, w_s, kI_b, n):
        return np.maximum((kI_b[:n] @ qI_s.T) @ w_s, 0.0)
    m = _Mutant(index_scores_row=bad)
    assert _fails(check_indexer_fixture, m) and _fails(check_indexer_closed_form, m)


def test_mutant_dropped_head_weight_is_caught():
    def bad(qI_s, w_s, kI_b, n):
        return np.maximum(kI_b[:n] @ qI_s.T, 0.0).sum(axis=1)
    assert _fails(check_indexer_fixture, _Mutant(index_scores_row=bad))


def test_mutant_transposed_operand_is_caught():
    def bad(qI_s, w_s, kI_b, n):   # heads and dims mixed up where shapes allow
        return np.maximum(kI_b[:n] @ qI_s.T[::-1], 0.0) @ w_s
    assert _fails(check_indexer_fixture, _Mutant(index_scores_row=bad))


def test_mutant_causal_off_by_one_is_caught():
    def bad(T, S, s):
        return T - S + s
    assert _fails(check_indexer_loops, _Mutant(visible_len=bad))


def test_mutant_tie_to_higher_index_is_caught():
    def bad(scores, k):
        v = np.asarray(scores, dtype=np.float64) + 0.0
        n = v.shape[0]
        keff = min(k, n)
        order = np.lexsort((-np.arange(n), -v))
        out = np.full(k, -1, dtype=np.int64)
        out[:keff] = np.sort(order[:keff])
        return out
    m = _Mutant(topk_select_row=bad)
    assert _fails(check_topk_fixture, m) and _fails(check_topk_bruteforce, m)


def test_mutant_wrong_gqa_grouping_is_caught():
    def bad(q, k, v, idx, num_kv_heads, k_scale=None, v_scale=None,
            softmax_scale=0.0, rows=None):
        B, S, Hq, D = q.shape
        scale = softmax_scale if softmax_scale else 1.0 / np.sqrt(D)
        out = np.full(q.shape, np.nan)
        for b in range(B):
            for s in range(S):
                sel = idx[b, s][idx[b, s] >= 0]
                Kb = O.dequantize(k[b, sel], None if k_scale is None else k_scale[b, sel])
                Vb = O.dequantize(v[b, sel], None if v_scale is None else v_scale[b, sel])
                for h in range(Hq):
                    g = h % num_kv_heads          # interleaved instead of consecutive
                    out[b, s, h] = O.attend_row(q[b, s, h], Kb[:, g], Vb[:, g], scale)
        return out
    assert _fails(check_dense_equivalence, _Mutant(sparse_attention=bad))


def test_mutant_wrong_softmax_scale_is_caught():
    def bad(q_h, Kg, Vg, scale):
        logits = (Kg @ q_h) / Kg.shape[1]
        p = np.exp(logits - logits.max())
        return (p / p.sum()) @ Vg
    assert _fails(check_dense_equivalence, _Mutant(attend_row=bad))


def test_mutant_value_scale_dropped_is_caught():
    def bad(codes, scale):
        return codes
    assert _fails(check_worked_example, _Mutant(dequantize=bad))


def test_mutant_round_half_up_is_caught():
    def bad(x):
        x32 = np.asarray(x, dtype=np.float32)
        scale = np.float32(np.float32(np.max(np.abs(x32))) / np.float32(127.0))
        if scale == 0:
            return np.zeros(x32.shape, dtype=np.int8), np.float32(0.0)
        q = np.floor(x32 / scale + np.float32(0.5))
        return np.clip(q, -127, 127).astype(np.int8), scale
    assert _fails(check_quantize_fixture, _Mutant(quantize_row_int8=bad))


def test_mutant_scale_over_128_is_caught():
    def bad(x):
        x32 = np.asarray(x, dtype=np.float32)
        scale = np.float32(np.float32(np.max(np.abs(x32))) / np.float32(128.0))
        if scale == 0:
            return np.zeros(x32.shape, dtype=np.int8), np.float32(0.0)
        return np.clip(np.rint(x32 / scale), -127, 127).astype(np.int8), scale
    m = _Mutant(quantize_row_int8=bad)
    assert _fails(check_quantize_fixture, m) and _fails(check_quantize_invariants, m)


def test_mutant_append_one_row_late_is_caught():
    def bad(kI, k, v, k_scale, v_scale, kI_new, k_new, v_new, total_len, kv_dtype):
        return O.cache_append(kI, k, v, k_scale, v_scale, kI_new, k_new, v_new,
                              [t + 1 if t + 1 <= kI.shape[1] else t for t in total_len], kv_dtype)
    assert _fails(check_append_positions, _Mutant(cache_append=bad))


def test_mutant_page_index_swapped_is_caught():
    def bad(pool, table, block_size, total_len):
        pool = np.asarray(pool)
        table = np.asarray(table)
        B, per_seq = table.shape
        out = np.zeros((B, per_seq * block_size) + pool.shape[1:])
        for b in range(B):
            for t in range(int(total_len[b])):
                out[b, t] = pool[table[b, t % per_seq] * block_size + t // per_seq]
        return out
    assert _fails(check_gather_pages, _Mutant(gather_pages=bad))


def _rope_variant(pairs="half", sin_sign=1.0, eps_outside=False, norm_all_heads=False):
    def f(x, gamma, eps, cos, sin, positions, rotary_dim):
        x = np.asarray(x, dtype=np.float64)
        axis = (-2, -1) if norm_all_heads else -1
        ms = np.mean(x * x, axis=axis, keepdims=True)
        y = x / (np.sqrt(ms) + eps if eps_outside else np.sqrt(ms + eps)) * np.asarray(gamma)
        out = y.copy()
        h = rotary_dim // 2
        pos = np.asarray(positions)
        c = np.asarray(cos)[pos][:, None, :]
        s = sin_sign * np.asarray(sin)[pos][:, None, :]
        if pairs == "half":
            ia, ib = np.arange(h), np.arange(h) + h
        else:
            ia, ib = 2 * np.arange(h), 2 * np.arange(h) + 1
        a, b = y[..., ia], y[..., ib]
        out[..., ia] = a * c - b * s
        out[..., ib] = b * c + a * s
        return out
    return f


def test_mutant_rope_interleaved_pairs_is_caught():
    assert _fails(check_rope_fixture, _Mutant(rmsnorm_rotary=_rope_variant(pairs="interleaved")))


def test_mutant_rope_sin_sign_is_caught():
    assert _fails(check_rope_fixture, _Mutant(rmsnorm_rotary=_rope_variant(sin_sign=-1.0)))


def test_mutant_rope_eps_outside_sqrt_is_caught():
    assert _fails(check_rope_complex, _Mutant(rmsnorm_rotary=_rope_variant(eps_outside=True)))


def test_mutant_rope_norm_over_all_heads_is_caught():
    assert _fails(check_rope_complex, _Mutant(rmsnorm_rotary=_rope_variant(norm_all_heads=True)))


def test_mutant_round_toward_zero_is_caught():
    def bad(values, dtype):
        import torch
        t = torch.as_tensor(np.asarray(values, dtype=np.float64)).to(torch.float32)
        bits = {"bf16": 7, "fp16": 10, "fp32": 23}[dtype]
        m, e = np.frexp(t.numpy().astype(np.float64))
        return np.ldexp(np.trunc(m * 2.0 ** (bits + 1)) / 2.0 ** (bits + 1), e)
    assert _fails(check_round_to, _Mutant(round_to=bad))


def test_mutant_aux_row_off_by_one_is_caught():
    def bad(q, k, v, idx, num_kv_heads, k_aux, v_aux, total_len, k_scale=None, v_scale=None,
            softmax_scale=0.0, rows=None):
        # reads aux row t - (T - S) - 1 (wrapping), a plausible indexing slip
        S = q.shape[1]
        ka = np.roll(k_aux, 1, axis=1)
        va = np.roll(v_aux, 1, axis=1)
        return O.sparse_attention_aux(q, k, v, idx, num_kv_heads, ka, va, total_len, k_scale,
                                      v_scale, softmax_scale, rows)
    m = _Mutant(sparse_attention_aux=bad)
    assert _fails(check_aux_fixture, m) or _fails(check_aux_reduces_to_cache, m)
    assert _fails(check_aux_reduces_to_cache, m)


def test_mutant_aux_ignored_is_caught():
    def bad(q, k, v, idx, num_kv_heads, k_aux, v_aux, total_len, k_scale=None, v_scale=None,
            softmax_scale=0.0, rows=None):
        return O.sparse_attention(q, k, v, idx, num_kv_heads, k_scale, v_scale, softmax_scale, rows)
    assert _fails(check_aux_fixture, _Mutant(sparse_attention_aux=bad))
