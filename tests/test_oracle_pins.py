"""Pins of the CPU oracle against things other than itself.

Each pin is independent of the oracle's code: a hand-worked example stored
under tests/golden/, a closed form, a library routine (torch.histc,
torch bf16 conversion, torch silu, a dense matmul), brute force written here
in plain Python, or an invariant of the method.  The last group plants
plausible mistakes in the oracle (on the CPU) and checks that a pin fails.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import mc2_oracle as orc
from moe_expert_dispatch_histc_gb300.workloads import (
    WORKLOADS, make_inputs, as_f64)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _small_case(seed, T=16, H=8, I=4, E=4, k=2, W=2, shared=False):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    if shared:
        w1 = np.repeat(rng.standard_normal((1, H, 2 * I)), E, axis=0)
        w2 = np.repeat(rng.standard_normal((1, I, H)), E, axis=0)
    else:
        w1 = rng.standard_normal((E, H, 2 * I))
        w2 = rng.standard_normal((E, I, H))
    logits = rng.standard_normal((T, E))
    sel = np.argsort(-logits, axis=1, kind="stable")[:, :k].astype(np.int32)
    p = rng.uniform(0.1, 1.0, (T, k))
    p = p / p.sum(axis=1, keepdims=True)
    return x, w1, w2, sel, p


# ---------------------------------------------------------------- histc
def test_histc_matches_torch_histc():
    rng = np.random.default_rng(0)
    for E in (1, 3, 8, 64):
        v = rng.integers(-2, E + 2, size=1000)
        ref = torch.histc(torch.tensor(v, dtype=torch.float64), bins=E, min=0, max=E)
        assert np.array_equal(orc.histc(v, E, 0, E), ref.numpy().astype(np.int64))
        f = rng.uniform(-1, E + 1, size=1000)
        ref = torch.histc(torch.tensor(f), bins=E, min=0, max=E)
        assert np.array_equal(orc.histc(f, E, 0, E), ref.numpy().astype(np.int64))


def test_counts_worked_example():
    g = _golden("counts_worked_example.json")
    sel = np.array(g["selected_experts"], dtype=np.int32)
    E, W = g["E"], g["W"]
    cnt = orc.rank_counts(sel, E, W)
    assert cnt.tolist() == g["num_global"]
    send, recv = orc.send_recv_counts(cnt, W)
    assert [s.tolist() for s in send] == g["send_counts"]
    assert [r.tolist() for r in recv] == g["recv_counts"]
    assert orc.expert_offsets(cnt).tolist() == g["offsets"]
    rows, idx = orc.permute(np.arange(g["T"]), sel, E)
    assert idx.tolist() == g["permute_src"]
    assert rows.tolist() == g["permuted_token"]
    res = orc.block_forward(np.zeros((4, 2)), np.zeros((E, 2, 2)), np.zeros((E, 1, 2)),
                            sel, np.full((4, 2), 0.5), E, W)
    assert res["unpermute_dst"].tolist() == g["unpermute_dst"]


def _brute_counts(sel, E, W):
    T, k = sel.shape
    Tl = T // W
    cnt = [[0] * E for _ in range(W)]
    for t in range(T):
        for j in range(k):
            e = int(sel[t, j])
            if 0 <= e < E:
                cnt[t // Tl][e] += 1
    return cnt


@pytest.mark.parametrize("seed", range(4))
def test_counts_brute_force_and_invariants(seed):
    rng = np.random.default_rng(seed)
    T, k, E, W = 24, 3, 6, 3
    sel = rng.integers(0, E, size=(T, k)).astype(np.int32)
    cnt = orc.rank_counts(sel, E, W)
    assert cnt.tolist() == _brute_counts(sel, E, W)
    assert cnt.sum() == T * k                              # counts sum to T*k
    assert all(cnt[r].sum() == (T // W) * k for r in range(W))
    send, recv = orc.send_recv_counts(cnt, W)
    El = E // W
    assert sum(int(r.sum()) for r in recv) == T * k        # everything sent is received
    for r in range(W):                                     # recv_r[s*El+le] = send_s[r*El+le]
        for s in range(W):
            for le in range(El):
                assert recv[r][s * El + le] == send[s][r * El + le]


def test_counts_skip_invalid_ids():
    sel = np.array([[0, 4], [-1, 1], [3, 3], [2, 5]], dtype=np.int32)
    cnt = orc.rank_counts(sel, 4, 2)
    assert cnt.tolist() == _brute_counts(sel, 4, 2)
    assert cnt.sum() == 5


@pytest.mark.parametrize("seed", range(4))
def test_permutation_is_stable_sort_by_expert(seed):
    rng = np.random.default_rng(seed)
    T, k, E = 30, 4, 7
    sel = rng.integers(0, E, size=(T, k)).astype(np.int32)
    _, idx = orc.permute(np.arange(T), sel, E)
    flat = sel.reshape(-1).tolist()
    brute = sorted(range(T * k), key=lambda i: (flat[i], i))   # (expert, t, j)
    assert idx.tolist() == brute
    assert sorted(idx.tolist()) == list(range(T * k))


def test_permute_then_unpermute_is_identity():
    rng = np.random.default_rng(3)
    T, k, E, H = 32, 4, 8, 5
    x = rng.standard_normal((T, H))
    sel = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    rows, idx = orc.permute(x, sel, E)
    back = orc.unpermute(rows, idx, np.full((T, k), 1.0 / k))
    assert np.array_equal(back, x)                          # 1/k = 2**-2: exact
    # one-hot probs select one slot: still the identity
    oh = np.zeros((T, k))
    oh[np.arange(T), rng.integers(0, k, T)] = 1.0
    assert np.array_equal(orc.unpermute(rows, idx, oh), x)


# ---------------------------------------------------------------- rounding and silu
def test_round_to_bf16_matches_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f) & (np.abs(f) >= 2.0 ** -126) & (np.abs(f) < 3e38)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(orc.round_to_bf16(f.astype(np.float64)), ref)
    # ties go to even
    assert orc.round_to_bf16(np.array([1 + 2 ** -8]))[0] == 1.0
    assert orc.round_to_bf16(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6
    assert orc.round_to_bf16(np.array([0.0]))[0] == 0.0


def test_silu_pins():
    g = np.linspace(-30, 30, 2001)
    ref = torch.nn.functional.silu(torch.tensor(g)).numpy()
    assert np.allclose(orc.silu(g), ref, rtol=1e-14, atol=1e-300)
    assert orc.silu(np.array([0.0]))[0] == 0.0
    assert abs(orc.silu(np.array([50.0]))[0] - 50.0) < 1e-15 * 50
    assert abs(orc.silu(np.array([math.log(3)]))[0] - 0.75 * math.log(3)) < 1e-15


def test_swiglu_closed_form():
    g = _golden("swiglu_closed_form.json")
    ln3 = math.log(3.0)
    gate = np.array(g["w1_gate_over_ln3"]) * ln3
    up = np.array(g["w1_up"])
    w1 = np.concatenate([gate, up], axis=2)
    w2 = np.array(g["w2"])
    sel = np.array(g["selected_experts"], dtype=np.int32)
    probs = np.array(g["probs"])
    out = orc.block_forward(np.array(g["x"]), w1, w2, sel, probs, g["E"], g["W"])["out"]
    assert np.allclose(out, np.array(g["out_over_ln3"]) * ln3, rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------- the block
def _brute_python(x, w1, w2, sel, probs):
    """Plain-Python per-token formula: out[t] = sum_j p * swiglu(x w1[e]) w2[e]."""
    T, H = x.shape
    I = w2.shape[1]
    out = [[0.0] * H for _ in range(T)]
    for t in range(T):
        for j in range(sel.shape[1]):
            e = int(sel[t, j])
            g = [sum(x[t, a] * w1[e, a, n] for a in range(H)) for n in range(2 * I)]
            h = [g[n] / (1.0 + math.exp(-g[n])) * g[I + n] for n in range(I)]
            for c in range(H):
                out[t][c] += probs[t, j] * sum(h[n] * w2[e, n, c] for n in range(I))
    return np.array(out)


@pytest.mark.parametrize("seed", range(3))
def test_block_matches_python_brute_force(seed):
    x, w1, w2, sel, p = _small_case(seed)
    ref = _brute_python(x, w1, w2, sel, p)
    got = orc.block_forward(x, w1, w2, sel, p, E=4, W=2)["out"]
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", range(3))
def test_block_matches_rankwise_alltoallv_flow(seed):
    x, w1, w2, sel, p = _small_case(seed, T=24, E=6, k=3, W=3)
    a = orc.block_forward(x, w1, w2, sel, p, E=6, W=3)["out"]
    b = orc.ep_mc2_forward_emulated(x, w1, w2, sel, p, E=6, W=3)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-13)
    for t in range(0, 24, 5):
        c = orc.brute_force_token(x[t], w1, w2, sel[t], p[t], 6)
        assert np.allclose(a[t], c, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("seed", range(3))
def test_shared_weights_reduce_to_dense_swiglu_mlp(seed):
    x, w1, w2, sel, p = _small_case(seed, T=20, H=16, I=8, E=5, k=3, W=1, shared=True)
    xt = torch.tensor(x)
    g = xt @ torch.tensor(w1[0])
    dense = (torch.nn.functional.silu(g[:, :8]) * g[:, 8:]) @ torch.tensor(w2[0])
    got = orc.block_forward(x, w1, w2, sel, p, E=5, W=1)["out"]
    assert np.allclose(got, dense.numpy(), rtol=1e-12, atol=1e-12)


def test_invalid_ids_contribute_nothing():
    x, w1, w2, sel, p = _small_case(5, T=8, E=4, k=2, W=2)
    bad = sel.copy()
    bad[1, 0] = 4
    bad[6, 1] = -3
    res = orc.block_forward(x, w1, w2, bad, p, E=4, W=2)
    assert res["offsets"][-1] == 14
    assert sorted(res["permute_src"][14:].tolist()) == [2, 13]   # flat t*k+j
    for t in range(8):
        ref = orc.brute_force_token(x[t], w1, w2, bad[t], p[t], 4)
        assert np.allclose(res["out"][t], ref, rtol=1e-13, atol=1e-13)


def test_tiny_workload_end_to_end():
    wl = WORKLOADS["tiny"]
    d = make_inputs(wl, 0)
    x, w1, w2 = (as_f64(d[n], wl.act) for n in ("x", "w1", "w2"))
    res = orc.block_forward(x, w1, w2, d["sel"], d["probs"], wl.E, wl.W, h_dtype="f32")
    b = orc.ep_mc2_forward_emulated(x, w1, w2, d["sel"], d["probs"], wl.E, wl.W, h_dtype="f32")
    assert np.allclose(res["out"], b, rtol=1e-12, atol=1e-15)
    assert res["cnt"].sum() == wl.T * wl.k


# ---------------------------------------------------------------- int8 path
def test_quant_block_integer_parts_by_brute_force():
    rng = np.random.default_rng(0)
    T, H, I, E, k, W = 8, 6, 3, 4, 2, 2
    xq = rng.integers(-127, 128, (T, H)).astype(np.int8)
    w1q = rng.integers(-127, 128, (E, H, 2 * I)).astype(np.int8)
    w2q = rng.integers(-127, 128, (E, I, H)).astype(np.int8)
    xs = rng.uniform(1e-3, 1e-2, T).astype(np.float32)
    w1s = rng.uniform(1e-3, 1e-2, (E, 2 * I)).astype(np.float32)
    w2s = rng.uniform(1e-3, 1e-2, (E, H)).astype(np.float32)
    sel = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    probs = np.full((T, k), 0.5, np.float32)
    r = orc.quant_block_forward(xq, xs, w1q, w1s, w2q, w2s, sel, probs, E, W)
    src = r["permute_src"]
    for p in range(T * k):
        t, j = divmod(int(src[p]), k)
        e = int(sel[t, j])
        for n in range(2 * I):
            acc = sum(int(xq[t, a]) * int(w1q[e, a, n]) for a in range(H))
            assert r["acc1"][p, n] == acc
            assert r["h"].shape == (T * k, I)
        for c in range(H):
            acc2 = sum(int(r["hq"][p, i]) * int(w2q[e, i, c]) for i in range(I))
            assert r["acc2"][p, c] == acc2


def test_quant_worst_case_accumulator_fits_int32():
    K = 3072
    xq = np.full((1, K), -127, np.int8)
    w = np.full((1, K, 2), 127, np.int8)
    w[0, :, 1] = -127
    xs = np.ones(1, np.float32)
    ws = np.ones((1, 2), np.float32)
    w2 = np.ones((1, 1, 4), np.int8)
    r = orc.quant_block_forward(xq, xs, w, ws, w2, np.ones((1, 4), np.float32),
                                np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32), 1, 1)
    assert r["acc1"][0, 0] == -K * 127 * 127
    assert abs(int(r["acc1"][0, 0])) < 2 ** 31


def test_exact_int_matmul_against_python_integers():
    """The float64 route of the integer products equals Python's exact
    integers, including sums far above 2**24 and the int8 extreme -128."""
    rng = np.random.default_rng(3)
    a = rng.integers(-128, 128, (5, 3072)).astype(np.int8)
    b = rng.integers(-128, 128, (3072, 4)).astype(np.int8)
    a[0] = -128
    b[:, 0] = -128
    got = orc.exact_int_matmul(a, b)
    assert got.dtype == np.int64
    for i in range(5):
        for j in range(4):
            assert got[i, j] == sum(int(a[i, t]) * int(b[t, j]) for t in range(3072))
    assert got[0, 0] == 3072 * 128 * 128
    with pytest.raises(AssertionError):
        orc.exact_int_matmul(np.full((1, 2 ** 20), 2 ** 20, np.int64),
                             np.full((2 ** 20, 1), 2 ** 20, np.int64))


def _quant_case(seed):
    """A small int8 block whose scale shapes make transposition mistakes fit:
    E = 2I, so a transposed [E, 2I] channel scale still has the right shape."""
    rng = np.random.default_rng(seed)
    T, H, I, E, k, W = 12, 5, 2, 4, 2, 2
    xq = rng.integers(-127, 128, (T, H)).astype(np.int8)
    w1q = rng.integers(-127, 128, (E, H, 2 * I)).astype(np.int8)
    w2q = rng.integers(-127, 128, (E, I, H)).astype(np.int8)
    xs = rng.uniform(1e-3, 1e-2, T).astype(np.float32)
    w1s = rng.uniform(1e-3, 1e-2, (E, 2 * I)).astype(np.float32)
    w2s = rng.uniform(1e-3, 1e-2, (E, H)).astype(np.float32)
    sel = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    probs = rng.uniform(0.1, 1.0, (T, k)).astype(np.float32)
    return dict(xq=xq, xs=xs, w1q=w1q, w1s=w1s, w2q=w2q, w2s=w2s, sel=sel, probs=probs,
                E=E, W=W, k=k, I=I, H=H)


def test_quant_dequant_equals_float_block_on_dequantised_operands():
    """(x1_scale * x2_scale) * (x1 @ x2) with x1_scale per token (m, 1) and
    x2_scale per channel (1, n): fc1 of the int8 block equals the float block
    run on x = xs[t] * xq[t, :] and w1 = w1q[e] * w1s[e, None, :], so their
    SwiGLU outputs agree; fc2's rows equal (hs[p] * hq[p, :]) @ (w2q[e] *
    w2s[e]), written out here element by element; the output is the
    probability-weighted sum of a token's rows, also written out here."""
    c = _quant_case(0)
    r = orc.quant_block_forward(c["xq"], c["xs"], c["w1q"], c["w1s"], c["w2q"], c["w2s"],
                                c["sel"], c["probs"], c["E"], c["W"])
    xf = c["xs"].astype(np.float64)[:, None] * c["xq"].astype(np.float64)
    w1f = c["w1q"].astype(np.float64) * c["w1s"].astype(np.float64)[:, None, :]
    w2f = c["w2q"].astype(np.float64) * c["w2s"].astype(np.float64)[:, None, :]
    ref = orc.block_forward(xf, w1f, w2f, c["sel"], c["probs"], c["E"], c["W"])
    assert np.allclose(r["h"], ref["h"], rtol=1e-12, atol=0)
    offs, src, k = r["offsets"], r["permute_src"], c["k"]
    n = int(offs[-1])
    for p in range(n):
        e = int(np.searchsorted(offs, p, side="right") - 1)
        for col in range(c["H"]):
            v = sum((float(r["hs"][p]) * int(r["hq"][p, i])) *
                    (int(c["w2q"][e, i, col]) * float(c["w2s"][e, col])) for i in range(c["I"]))
            assert math.isclose(r["y"][p, col], v, rel_tol=1e-12, abs_tol=1e-300)
    T = c["sel"].shape[0]
    for t in range(T):
        for col in range(c["H"]):
            v = 0.0
            for p in range(n):
                if int(src[p]) // k == t:
                    v += float(c["probs"][t, int(src[p]) % k]) * r["y"][p, col]
            assert math.isclose(r["out"][t, col], v, rel_tol=1e-12, abs_tol=1e-300)


def test_requant_rows_ties_worked_example():
    """Hand-worked rows whose h / hs lands exactly on .5 (scales that are powers
    of two, so every quotient is exact): ties go to the even code."""
    g = _golden("requant_ties.json")
    for h, hs, hq in zip(g["h"], g["hs"], g["hq"]):
        q, s = orc.requant_rows(np.array([h]))
        assert float(s[0]) == hs
        assert q[0].astype(int).tolist() == hq


@pytest.mark.parametrize("mutation", ["w1s_transposed", "w1s_wrong_expert", "xs_wrong_token",
                                      "w2s_dropped", "w2s_wrong_expert", "hs_dropped",
                                      "requant_half_away", "requant_by_128"])
def test_planted_quant_mistakes_are_caught(monkeypatch, mutation):
    """Each plausible mistake in the int8 block's scale handling or its
    re-quantisation, planted in the oracle, makes a pin fail."""
    real = orc.quant_block_forward
    real_rq = orc.requant_rows

    def bad(xq, xs, w1q, w1s, w2q, w2s, sel, probs, E, W, hq_override=None):
        if mutation == "w1s_transposed":
            w1s = np.ascontiguousarray(w1s.T)
        elif mutation == "w1s_wrong_expert":
            w1s = np.roll(w1s, 1, axis=0)
        elif mutation == "xs_wrong_token":
            xs = xs[::-1].copy()
        elif mutation == "w2s_dropped":
            w2s = np.ones_like(w2s)
        elif mutation == "w2s_wrong_expert":
            w2s = np.roll(w2s, 1, axis=0)
        res = real(xq, xs, w1q, w1s, w2q, w2s, sel, probs, E, W, hq_override=hq_override)
        if mutation == "hs_dropped":   # fc2 dequantised without the row scale
            res["y"] = res["y"] / res["hs"].astype(np.float64)[:, None]
            res["out"] = orc.unpermute(res["y"], res["permute_src"], probs,
                                       valid_rows=int(res["offsets"][-1]))
        return res

    def bad_rq(h):
        h32 = np.asarray(h, dtype=np.float64).astype(np.float32)
        amax = np.abs(h32).max(axis=1)
        if mutation == "requant_by_128":
            hs = np.where(amax > 0, amax / np.float32(128.0), np.float32(1.0)).astype(np.float32)
            q = np.rint(h32 / hs[:, None])
        else:   # requant_half_away: ties away from zero
            hs = np.where(amax > 0, amax / np.float32(127.0), np.float32(1.0)).astype(np.float32)
            v = (h32 / hs[:, None]).astype(np.float32)
            q = np.sign(v) * np.floor(np.abs(v) + 0.5)
        return np.clip(q, -127, 127).astype(np.int8), hs

    if mutation.startswith("requant"):
        monkeypatch.setattr(orc, "requant_rows", bad_rq)
    else:
        monkeypatch.setattr(orc, "quant_block_forward", bad)
    failures = 0
    for fn in (test_quant_dequant_equals_float_block_on_dequantised_operands,
               test_requant_rows_ties_worked_example, test_requant_rows_properties):
        try:
            fn()
        except (AssertionError, ValueError, IndexError):
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake {mutation}"


def test_requant_rows_properties():
    rng = np.random.default_rng(1)
    h = rng.standard_normal((50, 37)) * rng.uniform(1e-3, 10, (50, 1))
    h[3] = 0.0
    hq, hs = orc.requant_rows(h)
    assert hq.dtype == np.int8 and np.abs(hq.astype(int)).max() <= 127
    nz = np.abs(h).max(axis=1) > 0
    assert np.all(np.abs(hq[nz].astype(int)).max(axis=1) == 127)   # the row max maps to +-127
    assert np.all(hq[3] == 0) and hs[3] == 1.0
    err = np.abs(hq.astype(np.float64) * hs[:, None] - h)
    assert np.all(err <= hs[:, None] * (0.5 + 1e-5))


# ---------------------------------------------------------------- backward
def _bwd_case(T, H, I, E, k, W, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    w1 = rng.standard_normal((E, H, 2 * I)) * 0.3
    w2 = rng.standard_normal((E, I, H)) * 0.3
    sel = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    probs = rng.uniform(0.1, 1.0, (T, k)).astype(np.float32)
    dout = rng.standard_normal((T, H))
    return x, w1, w2, sel, probs, dout


def _torch_token_forward(x, w1, w2, sel, probs, E):
    """The block written per token with torch ops (no permutation, no groups):
    out[t] = sum over valid slots of probs[t, j] * SwiGLU(x[t] @ w1[e]) @ w2[e]."""
    T, k = sel.shape
    I = w2.shape[1]
    rows = []
    for t in range(T):
        acc = torch.zeros(x.shape[1], dtype=torch.float64)
        for j in range(k):
            e = int(sel[t, j])
            if not 0 <= e < E:
                continue
            g = x[t] @ w1[e]
            acc = acc + probs[t, j] * ((torch.nn.functional.silu(g[:I]) * g[I:]) @ w2[e])
        rows.append(acc)
    return torch.stack(rows)


@pytest.mark.parametrize("seed", [0, 1])
def test_backward_matches_torch_autograd(seed):
    T, H, I, E, k, W = 6, 8, 4, 4, 2, 2
    x, w1, w2, sel, probs, dout = _bwd_case(T, H, I, E, k, W, seed)
    sel[2, 1] = 9  # one invalid slot: no gradient through it
    r = orc.block_backward(x, w1, w2, sel, probs, dout, E, W)
    tx, tw1, tw2 = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (x, w1, w2))
    tp = torch.tensor(probs.astype(np.float64), requires_grad=True)
    out = _torch_token_forward(tx, tw1, tw2, sel, tp, E)
    (out * torch.from_numpy(dout)).sum().backward()
    for name, t in (("dx", tx), ("dw1", tw1), ("dw2", tw2), ("dprobs", tp)):
        assert np.allclose(r[name], t.grad.numpy(), rtol=1e-10, atol=1e-12), name
    assert r["dprobs"][2, 1] == 0.0


def test_backward_by_finite_differences():
    T, H, I, E, k, W = 4, 6, 3, 3, 2, 1
    x, w1, w2, sel, probs, dout = _bwd_case(T, H, I, E, k, W, 5)
    r = orc.block_backward(x, w1, w2, sel, probs, dout, E, W)

    def loss(x_, w1_, w2_, p_):
        return float((orc.block_forward(x_, w1_, w2_, sel, p_, E, W)["out"] * dout).sum())
    eps = 1e-6
    rng = np.random.default_rng(6)
    for name, arr in (("dx", x), ("dw1", w1), ("dw2", w2), ("dprobs", probs)):
        for _ in range(3):
            idx = tuple(int(rng.integers(0, n)) for n in arr.shape)
            args = [x, w1, w2, probs.astype(np.float64)]
            pos = {"dx": 0, "dw1": 1, "dw2": 2, "dprobs": 3}[name]
            plus, minus = [a.copy() for a in args], [a.copy() for a in args]
            plus[pos][idx] += eps
            minus[pos][idx] -= eps
            fd = (loss(*plus) - loss(*minus)) / (2 * eps)
            assert math.isclose(r[name][idx], fd, rel_tol=1e-5, abs_tol=1e-7), (name, idx)


def test_backward_prob_gradient_identity():
    """out is linear in probs: sum_j probs[t, j] * dprobs[t, j] = out[t] . dout[t]."""
    x, w1, w2, sel, probs, dout = _bwd_case(8, 8, 4, 4, 3, 2, 7)
    r = orc.block_backward(x, w1, w2, sel, probs, dout, 4, 2)
    out = orc.block_forward(x, w1, w2, sel, probs, 4, 2)["out"]
    lhs = (probs.astype(np.float64) * r["dprobs"]).sum(axis=1)
    assert np.allclose(lhs, (out * dout).sum(axis=1), rtol=1e-12, atol=1e-12)


def test_silu_grad_pins():
    a = torch.linspace(-30, 30, 241, dtype=torch.float64, requires_grad=True)
    torch.nn.functional.silu(a).sum().backward()
    assert np.allclose(orc.silu_grad(a.detach().numpy()), a.grad.numpy(), rtol=1e-12, atol=1e-14)
    assert orc.silu_grad(np.array([0.0]))[0] == 0.5


@pytest.mark.parametrize("mutation", ["silu_grad_sign", "no_prob_in_dy", "transposed_dw2"])
def test_planted_backward_mistakes_are_caught(monkeypatch, mutation):
    if mutation == "silu_grad_sign":
        real = orc.silu_grad
        monkeypatch.setattr(orc, "silu_grad", lambda a: real(-np.asarray(a)))
    elif mutation == "no_prob_in_dy":
        real = orc.block_backward

        def bad(x, w1, w2, sel, probs, dout, E, W, h_dtype=None):
            return real(x, w1, w2, sel, np.ones_like(probs), dout, E, W, h_dtype)
        monkeypatch.setattr(orc, "block_backward", bad)
    else:
        real = orc.block_backward

        def bad(x, w1, w2, sel, probs, dout, E, W, h_dtype=None):
            r = real(x, w1, w2, sel, probs, dout, E, W, h_dtype)
            r["dw2"] = r["dw2"][:, ::-1, :]
            return r
        monkeypatch.setattr(orc, "block_backward", bad)
    failures = 0
    for fn in (lambda: test_backward_matches_torch_autograd(0), test_backward_by_finite_differences):
        try:
            fn()
        except (AssertionError, ValueError, IndexError):
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake {mutation}"


# ---------------------------------------------------- quantised matmul + reduce-scatter
def _mmrs_inputs(W, m, k, n, seed):
    rng = np.random.default_rng(seed)
    x1 = rng.integers(-127, 128, (W, m, k)).astype(np.int8)
    x2 = rng.integers(-127, 128, (W, k, n)).astype(np.int8)
    x1s = rng.uniform(1e-3, 1e-2, (W, m)).astype(np.float32)
    x2s = rng.uniform(1e-3, 1e-2, (W, n)).astype(np.float32)
    return x1, x1s, x2, x2s


def test_mm_reduce_scatter_by_brute_force():
    """Element by element: sum over ranks and over k of
    x1_scale * x2_scale * x1 * x2, in plain Python integers and floats."""
    W, m, k, n = 3, 6, 5, 6
    x1, x1s, x2, x2s = _mmrs_inputs(W, m, k, n, 0)
    acc, total, per_rank = orc.mm_reduce_scatter(x1, x1s, x2, x2s)
    for i in range(m):
        for c in range(n):
            want = 0.0
            for r in range(W):
                a = sum(int(x1[r, i, q]) * int(x2[r, q, c]) for q in range(k))
                assert acc[r, i, c] == a
                want += float(x1s[r, i]) * float(x2s[r, c]) * a
            assert math.isclose(total[i, c], want, rel_tol=1e-12, abs_tol=1e-15)
    # rank r receives rows [r*m/W, (r+1)*m/W)
    for r in range(W):
        assert np.array_equal(per_rank[r], total[r * (m // W):(r + 1) * (m // W)])


def test_mm_reduce_scatter_one_rank_is_a_dequantised_matmul():
    x1, x1s, x2, x2s = _mmrs_inputs(1, 16, 64, 8, 1)
    _, total, per_rank = orc.mm_reduce_scatter(x1, x1s, x2, x2s)
    ref = torch.from_numpy(x1[0].astype(np.float64)) @ torch.from_numpy(x2[0].astype(np.float64))
    ref = (torch.from_numpy(x1s[0].astype(np.float64))[:, None] *
           torch.from_numpy(x2s[0].astype(np.float64))[None, :]) * ref
    assert np.allclose(total, ref.numpy(), rtol=1e-13, atol=0)
    assert per_rank.shape == (1, 16, 8)


def test_mm_reduce_scatter_shared_scales_is_one_long_matmul():
    """With the same scales on every rank, the sum over ranks of x1_r @ x2_r is
    one matmul over the concatenated reduction axis (block matrix product)."""
    W, m, k, n = 4, 8, 32, 6
    x1, x1s, x2, x2s = _mmrs_inputs(W, m, k, n, 2)
    x1s[:] = x1s[0]
    x2s[:] = x2s[0]
    _, total, _ = orc.mm_reduce_scatter(x1, x1s, x2, x2s)
    a = np.concatenate(list(x1), axis=1).astype(np.float64)          # [m, W*k]
    b = np.concatenate(list(x2), axis=0).astype(np.float64)          # [W*k, n]
    ref = (x1s[0].astype(np.float64)[:, None] * x2s[0].astype(np.float64)[None, :]) * (a @ b)
    assert np.allclose(total, ref, rtol=1e-13, atol=0)


def test_mm_reduce_scatter_sum_is_independent_of_rank_order():
    W, m, k, n = 4, 8, 16, 5
    x1, x1s, x2, x2s = _mmrs_inputs(W, m, k, n, 3)
    perm = np.array([2, 0, 3, 1])
    _, t0, _ = orc.mm_reduce_scatter(x1, x1s, x2, x2s)
    _, t1, _ = orc.mm_reduce_scatter(x1[perm], x1s[perm], x2[perm], x2s[perm])
    assert np.allclose(t0, t1, rtol=1e-13, atol=0)


def test_tolerance_rule():
    ref = np.array([1.0, -2.0, 4.0])
    assert orc.bf16_tolerance_ok(ref + 1e-4, ref)[0]
    assert not orc.bf16_tolerance_ok(ref + np.array([0, 0, 0.05]), ref)[0]     # max rule
    assert not orc.bf16_tolerance_ok(ref * 1.003, ref)[0]                      # mean rule


# ---------------------------------------------------------------- planted mistakes
def _mut_swap_gate_up(gu):
    I = gu.shape[1] // 2
    return orc.silu(gu[:, I:]) * gu[:, :I]


def _mut_sign(g):
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(g))


@pytest.mark.parametrize("mutation", ["drop_channel_scale", "first_rank_only",
                                      "scatter_columns"])
def test_planted_reduce_scatter_mistakes_are_caught(monkeypatch, mutation):
    real = orc.mm_reduce_scatter

    def bad(x1q, x1s, x2q, x2s):
        W, m, _ = x1q.shape
        if mutation == "drop_channel_scale":
            return real(x1q, x1s, x2q, np.ones_like(x2s))
        if mutation == "first_rank_only":
            acc, total, _ = real(x1q[:1], x1s[:1], x2q[:1], x2s[:1])
            return acc, total, total.reshape(W, m // W, -1) if m % W == 0 else None
        acc, total, _ = real(x1q, x1s, x2q, x2s)       # scatter_columns
        return acc, total, np.stack(np.split(total, W, axis=1)) if total.shape[1] % W == 0 \
            else total.reshape(W, m // W, -1)
    monkeypatch.setattr(orc, "mm_reduce_scatter", bad)
    failures = 0
    for fn in (test_mm_reduce_scatter_by_brute_force,
               test_mm_reduce_scatter_one_rank_is_a_dequantised_matmul,
               test_mm_reduce_scatter_shared_scales_is_one_long_matmul):
        try:
            fn()
        except (AssertionError, ValueError, IndexError):
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake {mutation}"


@pytest.mark.parametrize("mutation", ["swap_gate_up", "silu_sign", "transposed_recv",
                                      "unstable_permute", "drop_prob", "off_by_one_rank"])
def test_planted_mistakes_are_caught(monkeypatch, mutation):
    """Each plausible mistake, planted in the oracle, makes some pin fail."""
    if mutation == "swap_gate_up":
        monkeypatch.setattr(orc, "swiglu", _mut_swap_gate_up)
    elif mutation == "silu_sign":
        monkeypatch.setattr(orc, "silu", _mut_sign)
    elif mutation == "transposed_recv":
        def bad(num_global, W):
            El = num_global.shape[1] // W
            send = [num_global[r].copy() for r in range(W)]
            recv = [num_global[:, r * El:(r + 1) * El].T.reshape(-1).copy() for r in range(W)]
            return send, recv
        monkeypatch.setattr(orc, "send_recv_counts", bad)
    elif mutation == "unstable_permute":
        real = orc.permute

        def bad(hidden, sel, E=None):
            rows, idx = real(hidden, sel, E)
            return rows[::-1], idx[::-1]
        monkeypatch.setattr(orc, "permute", bad)
    elif mutation == "drop_prob":
        real_un = orc.unpermute
        monkeypatch.setattr(orc, "unpermute",
                            lambda y, i, p, valid_rows=None: real_un(y, i, np.ones_like(p), valid_rows))
    elif mutation == "off_by_one_rank":
        def bad(sel, E, W):
            T, k = sel.shape
            Tl = T // W
            return np.stack([orc.histc(sel[max(0, r * Tl - 1):(r + 1) * Tl - 1].reshape(-1), E, 0, E)
                             for r in range(W)])
        monkeypatch.setattr(orc, "rank_counts", bad)
    failures = 0
    for fn in (test_counts_worked_example, test_permute_then_unpermute_is_identity,
               test_swiglu_closed_form, lambda: test_block_matches_python_brute_force(0),
               lambda: test_block_matches_rankwise_alltoallv_flow(0),
               lambda: test_counts_brute_force_and_invariants(0),
               lambda: test_permutation_is_stable_sort_by_expert(0)):
        try:
            fn()
        except (AssertionError, ValueError, IndexError):
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake {mutation}"


def test_backward_gradients_are_local_to_experts_and_tokens():
    """The chain rule keeps the block's gradients local: an expert's dw1, dw2
    depend only on the rows routed to it, a token's dx and dprobs only on its
    own k slots.  The full oracle must equal reduced problems built from one
    expert (its routed tokens as single-slot tokens) or one token (with its k
    experts); the full-size GPU backward test relies on this."""
    rng = np.random.default_rng(5)
    T, H, I, E, k, W = 24, 16, 8, 6, 2, 2
    x = rng.standard_normal((T, H))
    w1 = rng.standard_normal((E, H, 2 * I)) * 0.3
    w2 = rng.standard_normal((E, I, H)) * 0.3
    sel = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    probs = rng.uniform(0.1, 1.0, (T, k))
    dout = rng.standard_normal((T, H))
    full = orc.block_backward(x, w1, w2, sel, probs, dout, E, W)
    for e in range(E):
        ts, js = np.nonzero(sel == e)
        if len(ts) == 0:
            assert not full["dw1"][e].any() and not full["dw2"][e].any()
            continue
        red = orc.block_backward(x[ts], w1[e:e + 1], w2[e:e + 1], np.zeros((len(ts), 1), np.int32),
                                 probs[ts, js][:, None], dout[ts], 1, 1)
        assert np.allclose(full["dw1"][e], red["dw1"][0], rtol=1e-12, atol=1e-12)
        assert np.allclose(full["dw2"][e], red["dw2"][0], rtol=1e-12, atol=1e-12)
    for t in range(T):
        red = orc.block_backward(x[t:t + 1], w1[sel[t]], w2[sel[t]], np.arange(k, dtype=np.int32)[None],
                                 probs[t:t + 1], dout[t:t + 1], k, 1)
        assert np.allclose(full["dx"][t], red["dx"][0], rtol=1e-12, atol=1e-12)
        assert np.allclose(full["dprobs"][t], red["dprobs"][0], rtol=1e-12, atol=1e-12)
