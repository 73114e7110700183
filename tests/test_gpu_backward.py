"""Backward of the block on the GPU against the CPU oracle (float64 chain rule
of the forward, pinned by torch autograd and finite differences).

Tolerance: the GPU path rounds G, dG, probs*h and the transposed weights to
bf16 (relative 2^-9 each) and keeps the gathered gradient rows as scaled
fp16 (2^-11) before the next matmul, so its gradients carry a few bf16 ulps:
max|err| <= 2e-2 * max|ref| and sum|err| / sum|ref| <= 1e-2 per output
(dx, dw1, dw2, dprobs)."""
import numpy as np
import pytest
import torch

from oracle import mc2_oracle as orc
from moe_expert_dispatch_histc_gb300 import binding as B, block as blk
from moe_expert_dispatch_histc_gb300.workloads import (WORKLOADS, Workload, as_f64,
                                                       bf16_bits_to_f32, f32_to_bf16_bits,
                                                       make_inputs)

from gpu_util import ensure_built, random_shapes, to_np

pytestmark = pytest.mark.gpu


def _tol(got, ref, what, max_rel=2e-2, mean_rel=1e-2):
    ok, a, m = orc.bf16_tolerance_ok(got, ref, max_rel=max_rel, mean_rel=mean_rel)
    assert ok, f"{what}: max|err|/max|ref| = {a:.3e}, mean rel = {m:.3e}"
    return a, m


def gpu_backward(wl, seed=0, sel=None, keep_g=False):
    """One backward call on the GPU; returns (got, status, inputs, dout bits)."""
    ensure_built()
    inp = make_inputs(wl, seed)
    if sel is not None:
        inp["sel"] = np.ascontiguousarray(sel.astype(np.int32))
    rng = np.random.default_rng(seed + 100)
    dout_bits = f32_to_bf16_bits(rng.standard_normal((wl.T, wl.H)).astype(np.float32))
    d = blk.inputs_to_device(inp, wl)
    b = blk.alloc_buffers(wl)
    shape = blk.shape_of(wl)
    B.mc2_moe_counts(shape, d["sel"], b.cnt, b.recv, b.offsets, b.permute_src, b.unpermute_dst,
                     b.ws, b.dev_status)
    w1t = torch.empty(wl.E, 2 * wl.I, wl.H, dtype=torch.bfloat16, device="cuda")
    w2t = torch.empty(wl.E, wl.H, wl.I, dtype=torch.bfloat16, device="cuda")
    B.mc2_transpose_weights(shape, d["w1"], d["w2"], w1t, w2t)
    dout = torch.from_numpy(dout_bits.view(np.int16)).view(torch.bfloat16).cuda()
    g = None
    if keep_g:   # the training forward keeps the pre-activation rows
        g = torch.empty(wl.T * wl.k, 2 * wl.I, dtype=torch.bfloat16, device="cuda")
        h = torch.empty(wl.T * wl.k, wl.I, dtype=torch.bfloat16, device="cuda")
        B.mc2_alltoallv_gmm_keep(shape, d["x"], d["w1"], b.offsets, b.permute_src, h, g,
                                 b.dev_status)
    ws = torch.empty(B.mc2_backward_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    dx = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device="cuda")
    dw1 = torch.empty(wl.E, wl.H, 2 * wl.I, dtype=torch.float32, device="cuda")
    dw2 = torch.empty(wl.E, wl.I, wl.H, dtype=torch.float32, device="cuda")
    dprobs = torch.empty(wl.T, wl.k, dtype=torch.float32, device="cuda")
    B.mc2_moe_backward(shape, d["x"], d["probs"], d["w1"], w1t, w2t, dout, b.offsets, b.permute_src,
                       b.unpermute_dst, dx, dw1, dw2, dprobs, ws, b.dev_status, g=g)
    torch.cuda.synchronize()
    # transposes are exact copies
    assert torch.equal(w1t.view(torch.int16), d["w1"].transpose(1, 2).contiguous().view(torch.int16))
    assert torch.equal(w2t.view(torch.int16), d["w2"].transpose(1, 2).contiguous().view(torch.int16))
    got = dict(dx=to_np(dx), dw1=to_np(dw1), dw2=to_np(dw2), dprobs=to_np(dprobs))
    return got, int(b.dev_status.item()), inp, dout_bits


def run_backward(wl, seed=0, sel=None, keep_g=False):
    got, status, inp, dout_bits = gpu_backward(wl, seed, sel, keep_g)
    x, w1, w2 = (as_f64(inp[n], wl.act) for n in ("x", "w1", "w2"))
    ref = orc.block_backward(x, w1, w2, inp["sel"], inp["probs"],
                             bf16_bits_to_f32(dout_bits).astype(np.float64), wl.E, wl.W,
                             h_dtype="bf16")
    return got, ref, status


BWD = [
    Workload("bwd_small", 256, 256, 128, 8, 2, 2, "bf16"),
    Workload("bwd_ragged", 384, 320, 192, 6, 3, 3, "bf16"),       # partial tiles in M and N
    Workload("bwd_many_experts", 512, 512, 256, 32, 4, 4, "bf16"),
    Workload("bwd_multi_tile", 2048, 1024, 512, 16, 4, 4, "bf16"),  # ~512 rows per expert
]


@pytest.mark.parametrize("wl", BWD, ids=lambda w: w.name)
def test_backward_parity(wl):
    got, ref, status = run_backward(wl, seed=1)
    assert status == 0
    for name in ("dx", "dw1", "dw2", "dprobs"):
        _tol(got[name], ref[name], name)


@pytest.mark.parametrize("mode", [1, 2], ids=["single_cta", "cta_pairs"])
@pytest.mark.parametrize("wl", [BWD[1], BWD[3]], ids=lambda w: w.name)
def test_backward_parity_under_each_tiling(wl, mode):
    """The two dgrad GEMMs on single-CTA tiles and on CTA pairs, forced: both
    within the tolerance."""
    B.mc2_set_tile_pairing(mode)
    try:
        got, ref, status = run_backward(wl, seed=2)
    finally:
        B.mc2_set_tile_pairing(0)
    assert status == 0
    for name in ("dx", "dw1", "dw2", "dprobs"):
        _tol(got[name], ref[name], name)


@pytest.mark.parametrize("wl", random_shapes(303, 6, "bf16"), ids=lambda w: w.name)
def test_backward_random_shapes(wl):
    """Seeded random shapes (ragged in every dimension, odd expert counts,
    top-k 1 to 8): every gradient within the tolerance."""
    got, ref, status = run_backward(wl, seed=7)
    assert status == 0
    for name in ("dx", "dw1", "dw2", "dprobs"):
        _tol(got[name], ref[name], f"{wl.name}: {name}")


@pytest.mark.parametrize("wl", [
    Workload("bwd_k10", 128, 192, 64, 16, 10, 4, "bf16"),           # top-k past 8
    Workload("bwd_single_expert", 128, 128, 64, 1, 1, 1, "bf16"),   # a dense SwiGLU MLP
    Workload("bwd_one_token_per_rank", 4, 128, 64, 8, 2, 4, "bf16"),
], ids=lambda w: w.name)
def test_backward_large_topk_and_degenerate(wl):
    """Top-k beyond 8 (the dx sum's generic loop), one expert, one token per
    logical rank: every gradient within the tolerance."""
    got, ref, status = run_backward(wl, seed=8)
    assert status == 0
    for name in ("dx", "dw1", "dw2", "dprobs"):
        _tol(got[name], ref[name], f"{wl.name}: {name}")


def test_backward_invalid_ids_and_empty_experts():
    """Invalid slots get dprobs 0 and no gradient; experts without rows get zero
    weight gradients."""
    wl = Workload("bwd_sparse", 256, 256, 128, 8, 2, 2, "bf16")
    rng = np.random.default_rng(3)
    sel = np.stack([rng.choice([1, 5], 2, replace=False) for _ in range(wl.T)]).astype(np.int32)
    sel[7, 0], sel[100, 1] = -1, 8
    got, ref, status = run_backward(wl, seed=3, sel=sel)
    assert status & B.MC2_DEV_BAD_EXPERT_ID
    assert got["dprobs"][7, 0] == 0.0 and got["dprobs"][100, 1] == 0.0
    for e in (0, 2, 3, 4, 6, 7):
        assert not got["dw1"][e].any() and not got["dw2"][e].any()
    for name in ("dx", "dw1", "dw2", "dprobs"):
        _tol(got[name], ref[name], name)


def test_backward_empty_batch():
    """No tokens: every expert's weight gradients are written as zeros (the
    outputs start uninitialised) and nothing is flagged."""
    wl = Workload("bwd_empty", 0, 256, 128, 8, 2, 2, "bf16")
    got, status, _, _ = gpu_backward(wl, seed=0)
    assert status == 0
    assert got["dw1"].shape == (8, 256, 256) and not got["dw1"].any()
    assert got["dw2"].shape == (8, 128, 256) and not got["dw2"].any()


def test_backward_with_kept_pre_activation_is_bitwise_the_recompute():
    wl = BWD[3]
    got_r, _, st_r = run_backward(wl, seed=4)
    got_k, _, st_k = run_backward(wl, seed=4, keep_g=True)
    assert st_r == 0 and st_k == 0
    for name in ("dx", "dw1", "dw2", "dprobs"):
        assert np.array_equal(got_r[name], got_k[name]), name


def test_training_forward_h_against_the_oracle():
    """mc2_alltoallv_gmm_keep: h from the kept bf16 pre-activation, within the
    block's forward tolerance of the oracle's h; g = the oracle's G rows."""
    ensure_built()
    wl = BWD[3]
    inp = make_inputs(wl, 5)
    d = blk.inputs_to_device(inp, wl)
    b = blk.alloc_buffers(wl)
    shape = blk.shape_of(wl)
    B.mc2_moe_counts(shape, d["sel"], b.cnt, b.recv, b.offsets, b.permute_src, b.unpermute_dst,
                     b.ws, b.dev_status)
    g = torch.empty(wl.T * wl.k, 2 * wl.I, dtype=torch.bfloat16, device="cuda")
    h = torch.empty(wl.T * wl.k, wl.I, dtype=torch.bfloat16, device="cuda")
    B.mc2_alltoallv_gmm_keep(shape, d["x"], d["w1"], b.offsets, b.permute_src, h, g, b.dev_status)
    torch.cuda.synchronize()
    x, w1, w2 = (as_f64(inp[n], wl.act) for n in ("x", "w1", "w2"))
    ref = orc.block_backward(x, w1, w2, inp["sel"], inp["probs"], np.zeros((wl.T, wl.H)), wl.E,
                             wl.W, h_dtype="bf16")
    nvalid = ref["g"].shape[0]
    ok, a, m = orc.bf16_tolerance_ok(to_np(g)[:nvalid], ref["g"])
    assert ok, (a, m)
    ok, a, m = orc.bf16_tolerance_ok(to_np(h)[:nvalid], ref["h"])
    assert ok, (a, m)
    assert int(b.dev_status.item()) == 0


def test_backward_full_size_sampled():
    """The uniform workload at full size, in the configuration the bench
    times (G kept by the training forward).  The oracle cannot run the whole
    problem in seconds, but the chain rule keeps gradients local: an expert's
    dw1 and dw2 depend only on the rows routed to it, and a token's dx and
    dprobs only on its own k slots.  Reduced problems -- one expert with its
    routed tokens as single-slot tokens, one token with its k experts -- give
    the oracle's exact values for sampled experts and tokens."""
    wl = WORKLOADS["uniform"]
    got, status, inp, dout_bits = gpu_backward(wl, seed=6, keep_g=True)
    assert status == 0
    sel, probs = inp["sel"], inp["probs"]
    x = as_f64(inp["x"], wl.act)
    dout = bf16_bits_to_f32(dout_bits).astype(np.float64)
    counts = np.bincount(sel.reshape(-1), minlength=wl.E)
    for e in (int(np.argmax(counts)), int(np.argmin(counts)), 17):
        ts, js = np.nonzero(sel == e)
        ref = orc.block_backward(x[ts], as_f64(inp["w1"][e:e + 1], wl.act),
                                 as_f64(inp["w2"][e:e + 1], wl.act),
                                 np.zeros((len(ts), 1), np.int32), probs[ts, js][:, None],
                                 dout[ts], 1, 1, h_dtype="bf16")
        _tol(got["dw1"][e], ref["dw1"][0], f"dw1[{e}]")
        _tol(got["dw2"][e], ref["dw2"][0], f"dw2[{e}]")
    toks = np.random.default_rng(0).choice(wl.T, 12, replace=False)
    ref_dx, ref_dp = [], []
    for t in toks:
        es = sel[t]
        ref = orc.block_backward(x[t:t + 1], as_f64(inp["w1"][es], wl.act),
                                 as_f64(inp["w2"][es], wl.act),
                                 np.arange(wl.k, dtype=np.int32)[None], probs[t:t + 1],
                                 dout[t:t + 1], wl.k, 1, h_dtype="bf16")
        ref_dx.append(ref["dx"][0])
        ref_dp.append(ref["dprobs"][0])
    _tol(got["dx"][toks], np.stack(ref_dx), "dx (sampled tokens)")
    _tol(got["dprobs"][toks], np.stack(ref_dp), "dprobs (sampled tokens)")
