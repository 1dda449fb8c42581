"""GPU parity of dsa_cache_append (through the C ABI) against the oracle's
cache append: bit-exact, since the append is a copy, a round-to-nearest
conversion or an INT8 quantisation whose codes are decided in IEEE fp32 on
both sides. Every byte of every cache is compared, so rows the append must not
touch are checked to keep their sentinel values."""
import json
import os

import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
from dsa_inputs import make_append_inputs, make_inputs, small_workload, to_f64
from tests._helpers import TOL_INT8, check_selection, f64_inputs, rel_l2

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
COMBOS = [("bf16", "bf16"), ("bf16", "fp16"), ("bf16", "int8"), ("fp16", "fp16"),
          ("fp16", "int8")]
_TDT = {"bf16": torch.bfloat16, "fp16": torch.float16}
_BITS = {torch.bfloat16: torch.int16, torch.float16: torch.int16}


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from top_sparse_attention_chunked_gb300 import build_lib, dsa as D
    build_lib.build()
    D.load_library()
    return D


def _problem(D, B, S, H, cap, T, qd, kv):
    return D.make_problem(batch=B, q_len=S, total_len=list(T), top_k=1, num_q_heads=H,
                          num_kv_heads=H, cache_capacity=cap, q_dtype=qd, kv_dtype=kv)


def run_append(D, cpu, B, S, H, cap, T, qd, kv):
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in cpu.items()}
    p = _problem(D, B, S, H, cap, T, qd, kv)
    D.dsa_cache_append(p, dev["kI_new"], dev["k_new"], dev["v_new"], dev["kI"], dev["k"],
                       dev["v"], dev["k_scale"], dev["v_scale"])
    torch.cuda.synchronize()
    assert D.dsa_last_launches() == ["cache_append_kernel"]
    return {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in dev.items()}


def oracle_append(cpu, kv):
    f = {k: to_f64(v) if isinstance(v, torch.Tensor) else v for k, v in cpu.items()}
    return O.cache_append(f["kI"], f["k"], f["v"], f["k_scale"], f["v_scale"], f["kI_new"],
                          f["k_new"], f["v_new"], [int(t) for t in cpu["total_len"]], kv)


def _bits_equal(got: torch.Tensor, ref64: np.ndarray, name: str):
    ref = torch.from_numpy(ref64).to(got.dtype)
    if got.dtype in _BITS:
        a, b = got.view(_BITS[got.dtype]), ref.view(_BITS[got.dtype])
    elif got.dtype == torch.float32:
        a, b = got.view(torch.int32), ref.view(torch.int32)
    else:
        a, b = got, ref
    bad = (a != b).nonzero()
    assert bad.shape[0] == 0, (f"{name}: {bad.shape[0]} elements differ, first at "
                               f"{tuple(bad[0].tolist())}: got {got[tuple(bad[0])]} "
                               f"want {ref[tuple(bad[0])]}")


def check_against_oracle(gpu, cpu, kv):
    kI, k, v, ks, vs = oracle_append(cpu, kv)
    _bits_equal(gpu["kI"], kI, "kI")
    _bits_equal(gpu["k"], k, "k")
    _bits_equal(gpu["v"], v, "v")
    if kv == "int8":
        _bits_equal(gpu["k_scale"], ks, "k_scale")
        _bits_equal(gpu["v_scale"], vs, "v_scale")


@pytest.mark.parametrize("qd,kv", COMBOS)
@pytest.mark.parametrize("B,S,H,cap,T", [
    (3, 5, 2, 64, [5, 37, 64]),         # ragged lengths, one sequence filled to capacity
    (1, 1, 2, 4096, [4096]),            # one decode token
    (2, 8, 3, 100, [8, 99]),            # odd KV-head count (odd rows per token)
    (4, 16, 1, 40, [16, 17, 30, 40]),
])
def test_append_bitexact(dsa, qd, kv, B, S, H, cap, T):
    cpu = make_append_inputs(B, S, H, cap, T, qd, kv, seed=B * 100 + S)
    gpu = run_append(dsa, cpu, B, S, H, cap, T, qd, kv)
    check_against_oracle(gpu, cpu, kv)


@pytest.mark.parametrize("qd", ["bf16", "fp16"])
def test_append_int8_golden_rows(dsa, qd):
    """The hand-worked quantisation cases (power-of-two scales, exact ties),
    each padded with zeros to a 128-element row: codes and scales must equal
    the stored values, with no oracle involved."""
    cases = json.load(open(os.path.join(GOLDEN, "int8_quantize_tiny.json")))["cases"]
    B, S, H, cap = 1, len(cases), 1, len(cases) + 3
    cpu = make_append_inputs(B, S, H, cap, [cap], qd, "int8", seed=5, specials=False)
    for s, c in enumerate(cases):
        row = torch.zeros(128)
        row[:len(c["x"])] = torch.tensor(c["x"])
        cpu["k_new"][0, s, 0] = row.to(_TDT[qd])
        cpu["v_new"][0, s, 0] = (-row).to(_TDT[qd])
    gpu = run_append(dsa, cpu, B, S, H, cap, [cap], qd, "int8")
    for s, c in enumerate(cases):
        t = cap - S + s
        n = len(c["codes"])
        assert gpu["k"][0, t, 0, :n].tolist() == c["codes"], c
        assert gpu["v"][0, t, 0, :n].tolist() == [-x for x in c["codes"]], c
        assert (gpu["k"][0, t, 0, n:] == 0).all()
        assert float(gpu["k_scale"][0, t, 0]) == c["scale"]
        assert float(gpu["v_scale"][0, t, 0]) == c["scale"]


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_append_prefill_chunk_8k_on_32k(dsa, kv):
    """Full size of the prefill workload: 8,192 new tokens appended after a
    32,768-token past (2 KV heads), every byte compared."""
    B, S, H, cap, T = 1, 8192, 2, 40960, [40960]
    cpu = make_append_inputs(B, S, H, cap, T, "bf16", kv, seed=77)
    gpu = run_append(dsa, cpu, B, S, H, cap, T, "bf16", kv)
    check_against_oracle(gpu, cpu, kv)


def test_append_decode_256k_int8_rows(dsa):
    """Decode-sized append into a 262,144-row INT8 cache: the 8 new rows equal
    the oracle's, and every other row keeps its bytes (compared on the GPU)."""
    B, S, H, cap, T = 1, 8, 2, 262144, [262144 - 1000]
    cpu = make_append_inputs(B, S, H, cap, T, "bf16", "int8", seed=9)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in cpu.items()}
    before = {k: dev[k].clone() for k in ("kI", "k", "v", "k_scale", "v_scale")}
    p = _problem(dsa, B, S, H, cap, T, "bf16", "int8")
    dsa.dsa_cache_append(p, dev["kI_new"], dev["k_new"], dev["v_new"], dev["kI"], dev["k"],
                         dev["v"], dev["k_scale"], dev["v_scale"])
    torch.cuda.synchronize()
    lo, hi = T[0] - S, T[0]
    for k_ in before:
        assert torch.equal(dev[k_][:, :lo], before[k_][:, :lo]), k_
        assert torch.equal(dev[k_][:, hi:], before[k_][:, hi:]), k_
    for s in range(S):
        for g in range(H):
            for name, src in (("k", "k_new"), ("v", "v_new")):
                codes, sc = O.quantize_row_int8(to_f64(cpu[src][0, s, g]))
                assert dev[name][0, lo + s, g].cpu().numpy().tolist() == codes.tolist()
                assert np.float32(dev[name + "_scale"][0, lo + s, g].item()) == sc
    assert torch.equal(dev["kI"][0, lo:hi].cpu(), cpu["kI_new"][0])


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_append_own_rows_reproduces_cache(dsa, dt):
    """Appending a cache's own last rows (new tokens in the cache's type)
    restores rows that were overwritten, so the cache is bit for bit the
    original and the decode that follows gives the identical output."""
    D = dsa
    wl = small_workload(batch=2, q_len=3, total_len=2500, num_q_heads=8, num_kv_heads=2,
                        top_k=128, q_dtype=dt, kv_dtype=dt, seed=43)
    base = make_inputs(wl)
    T, S = wl.total_len, wl.q_len
    dev = {k_: (v_.cuda() if isinstance(v_, torch.Tensor) else v_) for k_, v_ in base.items()}
    kI_new = dev["kI"][:, T - S:T].clone()
    k_new = dev["k"][:, T - S:T].clone()
    v_new = dev["v"][:, T - S:T].clone()
    orig = {k_: dev[k_].clone() for k_ in ("kI", "k", "v")}
    for k_ in ("kI", "k", "v"):
        dev[k_][:, T - S:T] = 7.0
    p = D.problem_for(wl)
    D.dsa_cache_append(p, kI_new, k_new, v_new, dev["kI"], dev["k"], dev["v"], None, None)
    for k_ in ("kI", "k", "v"):
        assert torch.equal(dev[k_].view(torch.int16), orig[k_].view(torch.int16)), k_
    ws = D.alloc_workspace(p, D.DSA_OP_DECODE)
    outs = []
    for kI_, k_, v_ in ((dev["kI"], dev["k"], dev["v"]), (orig["kI"], orig["k"], orig["v"])):
        out = torch.empty(wl.batch, S, wl.num_q_heads, 128, dtype=D._TORCH_DT[p.out_dtype],
                          device="cuda")
        D.dsa_sparse_attn_decode(p, dev["q"], dev["qI"], dev["w"], kI_, k_, v_, None, None, None,
                                 out, ws)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_append_then_decode_matches_oracle(dsa):
    """The step as a user runs it: append the new tokens (INT8, quantised on
    write), then decode over the cache. The decode output is checked against
    the oracle run on the oracle's appended cache with the GPU's selection."""
    D = dsa
    wl = small_workload(batch=2, q_len=4, total_len=3000, num_q_heads=8, num_kv_heads=2,
                        top_k=256, kv_dtype="int8", seed=41)
    base = make_inputs(wl)
    app = make_append_inputs(wl.batch, wl.q_len, wl.num_kv_heads, wl.cap,
                             [wl.total_len] * wl.batch, "bf16", "int8", seed=42, specials=False)
    for name in ("kI", "k", "v", "k_scale", "v_scale"):
        app[name] = base[name].clone()
    gpu = run_append(D, app, wl.batch, wl.q_len, wl.num_kv_heads, wl.cap,
                     [wl.total_len] * wl.batch, "bf16", "int8")
    kI, k, v, ks, vs = oracle_append(app, "int8")
    cpu = dict(base)
    for name, val in (("kI", gpu["kI"]), ("k", gpu["k"]), ("v", gpu["v"]),
                      ("k_scale", gpu["k_scale"]), ("v_scale", gpu["v_scale"])):
        cpu[name] = val
    dev = {k_: (v_.cuda() if isinstance(v_, torch.Tensor) else v_) for k_, v_ in cpu.items()}
    p = D.problem_for(wl)
    ws = D.alloc_workspace(p, D.DSA_OP_DECODE)
    out = torch.empty(wl.batch, wl.q_len, wl.num_q_heads, 128, dtype=torch.bfloat16,
                      device="cuda")
    idx = torch.empty(wl.batch, wl.q_len, wl.top_k, dtype=torch.int32, device="cuda")
    D.dsa_sparse_attn_decode(p, dev["q"], dev["qI"], dev["w"], dev["kI"], dev["k"], dev["v"],
                             dev["k_scale"], dev["v_scale"], idx, out, ws)
    torch.cuda.synchronize()
    idx_h = idx.cpu().numpy()
    f = f64_inputs(base)
    for b in range(wl.batch):
        for s in range(wl.q_len):
            n = O.visible_len(wl.total_len, wl.q_len, s)
            ref = O.index_scores_row(f["qI"][b, s], f["w"][b, s], kI[b], n)
            check_selection(ref, idx_h[b, s], wl.top_k)
    att = O.sparse_attention(f["q"], k, v, idx_h, wl.num_kv_heads, ks, vs, 0.0)
    err = rel_l2(out.float().cpu().numpy().astype(np.float64), att)
    assert err <= TOL_INT8, err


def near_tie_rows(dt: torch.dtype, nrows: int, seed: int):
    """Rows whose absmax is one element and whose other elements x make
    x / (absmax/127) fall within 2^-12 of a half-integer, preferring the x
    whose fp32 quotient rounds onto the half-integer exactly (a tie made by
    the division's rounding). Returns (rows [nrows, 128] fp32, count of
    rounding-made ties)."""
    rng = np.random.default_rng(seed)
    allv = torch.arange(0, 2 ** 16, dtype=torch.int32).to(torch.int16).view(dt).float().numpy()
    allv = allv[np.isfinite(allv) & (allv > 0)].astype(np.float32)
    amaxes = rng.choice(allv[(allv > 1e-3) & (allv < 1e4)], nrows, replace=False)
    rows = np.zeros((nrows, 128), dtype=np.float32)
    made = 0
    for r, a in enumerate(amaxes):
        sc = np.float32(a / np.float32(127))
        xs = allv[allv < a]
        y = xs.astype(np.float64) / np.float64(sc)
        d = np.abs(np.abs(y - np.rint(y)) - 0.5)
        q = xs / sc
        rn_tie = (np.abs(q - np.rint(q)) == 0.5) & (d > 0)
        cand = np.concatenate([xs[rn_tie], xs[(d <= 2.0 ** -12) & ~rn_tie]])[:127]
        made += int(min(rn_tie.sum(), 127))
        rows[r, 0] = a
        rows[r, 1:1 + cand.size] = cand * rng.choice([-1.0, 1.0], cand.size)
    return rows, made


@pytest.mark.parametrize("qd", ["bf16", "fp16"])
def test_append_int8_near_ties(dsa, qd):
    """Quotients within 2^-12 of a half-integer (among them hundreds that the
    fp32 division rounds onto the half-integer exactly) give the oracle's
    codes bit for bit."""
    rows, made = near_tie_rows(_TDT[qd], 64, seed=3 if qd == "fp16" else 4)
    assert made >= 20
    B, S, H = 1, 32, 1
    cap = S
    cpu = make_append_inputs(B, S, 2, cap, [cap], qd, "int8", seed=6, specials=False)
    cpu["k_new"] = torch.from_numpy(rows[:32].reshape(B, S, 1, 128)).to(_TDT[qd])
    cpu["v_new"] = torch.from_numpy(rows[32:].reshape(B, S, 1, 128)).to(_TDT[qd])
    cpu["k"], cpu["v"] = cpu["k"][:, :, :1].contiguous(), cpu["v"][:, :, :1].contiguous()
    cpu["k_scale"] = cpu["k_scale"][:, :, :1].contiguous()
    cpu["v_scale"] = cpu["v_scale"][:, :, :1].contiguous()
    gpu = run_append(dsa, cpu, B, S, H, cap, [cap], qd, "int8")
    check_against_oracle(gpu, cpu, "int8")
