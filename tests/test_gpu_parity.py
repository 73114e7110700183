"""Parity of the CUDA path with the CPU oracle, through the C ABI.

Integer outputs (counts, recv counts, offsets, permutation indices) must be
bit-exact.  Floating-point outputs must satisfy the block's rule
max|err| <= 1e-2 * max|ref| and sum|err| / sum|ref| <= 2e-3 against the
float64 oracle (h is compared after the oracle rounds it to the activation
dtype, as the block materialises it).  Small shapes are compared in full;
the named full-size workloads in the launch configuration of the benchmark
(one mc2_moe_forward call) are compared on sampled tokens and rows.
"""
import numpy as np
import pytest
import torch

from oracle import mc2_oracle as orc
from moe_expert_dispatch_histc_gb300 import binding as B
from moe_expert_dispatch_histc_gb300.workloads import (WORKLOADS, Workload, as_f64, make_inputs,
                                                       make_routing)

from gpu_util import F64Experts, ensure_built, random_shapes, run_gpu, to_np

pytestmark = pytest.mark.gpu

H_DTYPE = {"f32": "f32", "bf16": "bf16"}


def _counts_exact(wl, inp, b):
    res_cnt = orc.rank_counts(inp["sel"], wl.E, wl.W)
    send, recv = orc.send_recv_counts(res_cnt, wl.W)
    offsets = orc.expert_offsets(res_cnt)
    _, src = orc.permute(np.arange(wl.T), inp["sel"], wl.E)
    dst = np.empty_like(src)
    dst[src] = np.arange(src.shape[0])
    assert np.array_equal(to_np(b.cnt), res_cnt), "cnt (all_gather of histc) differs"
    assert np.array_equal(to_np(b.recv), np.stack(recv)), "recv_counts differ"
    assert np.array_equal(to_np(b.offsets), offsets), "expert offsets differ"
    assert np.array_equal(to_np(b.permute_src), src), "permute_src differs"
    assert np.array_equal(to_np(b.unpermute_dst), dst), "unpermute_dst differs"
    return src, offsets


def _tol(got, ref, what):
    ok, a, m = orc.bf16_tolerance_ok(got, ref)
    assert ok, f"{what}: max|err|/max|ref| = {a:.3e} (<= 1e-2), mean rel = {m:.3e} (<= 2e-3)"
    return a, m


def test_selftest_wait_times_out_and_reports():
    ensure_built()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.mc2_selftest_wait(20_000_000, st)          # 20 ms on a barrier nothing completes
    torch.cuda.synchronize()
    assert int(st.item()) & B.MC2_DEV_TIMEOUT


@pytest.fixture(params=[1, 2], ids=["three_launches", "one_cluster"])
def counts_path(request):
    """Force one of the two counts passes for the test."""
    ensure_built()
    B.mc2_set_counts_path(request.param)
    yield request.param
    B.mc2_set_counts_path(0)


def _run_counts(wl, sel):
    from moe_expert_dispatch_histc_gb300 import block as blk
    d_sel = torch.from_numpy(np.ascontiguousarray(sel.astype(np.int32))).cuda()
    b = blk.alloc_buffers(wl)
    B.mc2_moe_counts(blk.shape_of(wl), d_sel, b.cnt, b.recv, b.offsets, b.permute_src,
                     b.unpermute_dst, b.ws, b.dev_status)
    torch.cuda.synchronize()
    return b


@pytest.mark.parametrize("name", ["tiny", "uniform", "skew", "int8", "decode"])
def test_counts_bit_exact(name, counts_path):
    wl = WORKLOADS[name]
    wlc = wl.scaled(act="bf16") if wl.act == "i8" else wl
    inp = {"sel": make_routing(wlc, 0)[0]}   # the counts read the ids only
    b = _run_counts(wlc, inp["sel"])
    _counts_exact(wlc, inp, b)
    assert int(b.dev_status.item()) == 0


COUNTS_SHAPES = [
    Workload("w1_ragged", 1000, 64, 64, 16, 3, 1, "bf16"),        # one rank, ragged last chunk
    Workload("many_ranks", 1024, 64, 64, 1024, 2, 1024, "bf16"),  # W = E = 1024: three launches only
    Workload("big_e", 2048, 64, 64, 1024, 8, 8, "bf16"),          # E = 1024 tables in shared memory
    Workload("long_chunks", 65536, 64, 64, 8, 4, 2, "bf16"),      # 16 CTAs, 512-entry chunks
]


@pytest.mark.parametrize("wl", COUNTS_SHAPES, ids=lambda w: w.name)
def test_counts_shapes_bit_exact(wl, counts_path):
    inp = make_inputs(wl, 3)
    b = _run_counts(wl, inp["sel"])
    _counts_exact(wl, inp, b)
    assert int(b.dev_status.item()) == 0


def test_counts_invalid_ids_every_value(counts_path):
    """-2, -1, E and a large id are all invalid: counted nowhere, sorted last."""
    wl = Workload("bad_counts", 512, 64, 64, 16, 4, 4, "bf16")
    inp = make_inputs(wl, 4)
    sel = inp["sel"].copy()
    sel[0, 0], sel[5, 1], sel[200, 3], sel[511, 2], sel[300, 0] = -2, -1, 16, 1 << 30, -(1 << 31)
    inp["sel"] = sel
    b = _run_counts(wl, sel)
    _counts_exact(wl, inp, b)
    assert int(b.dev_status.item()) & B.MC2_DEV_BAD_EXPERT_ID


SMALL = [
    Workload("tiny", 64, 256, 128, 8, 2, 2, "f32"),
    Workload("multi_mtile", 1024, 256, 128, 8, 2, 2, "bf16"),       # ~256 rows/expert, ragged
    Workload("ragged_n", 384, 320, 192, 6, 3, 3, "bf16"),           # partial n-tiles of fc1 and fc2
    Workload("many_experts", 256, 512, 256, 64, 8, 4, "bf16"),      # ~32 rows/expert
    Workload("k1", 200, 128, 64, 4, 1, 2, "bf16"),
    Workload("fp32_ragged", 96, 192, 64, 4, 2, 2, "f32"),
    Workload("e1024", 2048, 128, 64, 1024, 2, 8, "bf16"),         # the largest E: 1025-entry prefix
]


@pytest.fixture(params=[1, 2], ids=["single_cta", "cta_pairs"])
def pairing(request):
    """Force one grouped-GEMM tiling (single CTAs or CTA pairs) for the test."""
    ensure_built()
    B.mc2_set_tile_pairing(request.param)
    yield request.param
    B.mc2_set_tile_pairing(0)


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_block_parity_full(wl, pairing):
    inp, d, b = run_gpu(wl, seed=1)
    src, offsets = _counts_exact(wl, inp, b)
    x, w1, w2 = (as_f64(inp[n], wl.act) for n in ("x", "w1", "w2"))
    ref = orc.block_forward(x, w1, w2, inp["sel"], inp["probs"], wl.E, wl.W, h_dtype=H_DTYPE[wl.act])
    nvalid = int(offsets[-1])
    _tol(to_np(b.h)[:nvalid], ref["h"], "h (fc1 + SwiGLU)")
    _tol(to_np(b.out), ref["out"], "out (fc2 + combine)")
    assert int(b.dev_status.item()) == 0


# Degenerate forms of the method: one expert (the block is a dense SwiGLU
# MLP), one expert per logical rank, one token per logical rank.
DEGENERATE = [
    Workload("single_expert", 256, 128, 64, 1, 1, 1, "bf16"),
    Workload("one_expert_per_rank", 128, 128, 64, 4, 2, 4, "bf16"),
    Workload("one_token_per_rank", 4, 128, 64, 8, 2, 4, "bf16"),
]

LARGE_K = [
    Workload("k10", 128, 192, 64, 16, 10, 4, "bf16"),        # top-k past the combine's unrolled forms
    Workload("k_eq_E12", 96, 128, 128, 12, 12, 3, "bf16"),   # every token on every expert
    Workload("k40_f32", 64, 128, 64, 64, 40, 4, "f32"),      # 40 slots per token
]


@pytest.mark.parametrize("wl", LARGE_K + DEGENERATE, ids=lambda w: w.name)
def test_large_topk_and_degenerate_parity(wl, pairing):
    """Top-k beyond 8 (the combine's generic loop, many slots per token in
    the counts and the gather), k = E, and the degenerate shapes: counts and
    indices bit-exact, h and out within the tolerance, on both tilings."""
    inp, d, b = run_gpu(wl, seed=11)
    src, offsets = _counts_exact(wl, inp, b)
    x, w1, w2 = (as_f64(inp[n], wl.act) for n in ("x", "w1", "w2"))
    ref = orc.block_forward(x, w1, w2, inp["sel"], inp["probs"], wl.E, wl.W, h_dtype=H_DTYPE[wl.act])
    nvalid = int(offsets[-1])
    assert nvalid == wl.R
    _tol(to_np(b.h)[:nvalid], ref["h"], f"{wl.name}: h")
    _tol(to_np(b.out), ref["out"], f"{wl.name}: out")
    assert int(b.dev_status.item()) == 0


@pytest.mark.parametrize("wl", random_shapes(101, 10, "bf16") + random_shapes(102, 4, "f32"),
                         ids=lambda w: w.name)
def test_random_shapes_parity(wl, pairing):
    """Seeded random shapes -- ragged tiles in every dimension, expert counts
    that are not powers of two, top-k from 1 to 8, one to four logical ranks:
    counts and indices bit-exact, h and out within the tolerance, on both
    tilings."""
    inp, d, b = run_gpu(wl, seed=3)
    src, offsets = _counts_exact(wl, inp, b)
    x, w1, w2 = (as_f64(inp[n], wl.act) for n in ("x", "w1", "w2"))
    ref = orc.block_forward(x, w1, w2, inp["sel"], inp["probs"], wl.E, wl.W, h_dtype=H_DTYPE[wl.act])
    nvalid = int(offsets[-1])
    _tol(to_np(b.h)[:nvalid], ref["h"], f"{wl.name}: h")
    _tol(to_np(b.out), ref["out"], f"{wl.name}: out")
    assert int(b.dev_status.item()) == 0


@pytest.mark.parametrize("wl", SMALL[:3], ids=lambda w: w.name)
def test_segments_equal_single_call(wl):
    _, _, b1 = run_gpu(wl, seed=2)
    _, _, b2 = run_gpu(wl, seed=2, segments=True)
    assert torch.equal(b1.out, b2.out) and torch.equal(b1.h, b2.h)


@pytest.mark.parametrize("wl", [SMALL[1], Workload("i8_events", 512, 256, 128, 8, 2, 2, "i8")],
                         ids=lambda w: w.name)
def test_gemm_events_bracket_the_fc1_kernel(wl):
    """mc2_set_gemm_events (how the benchmark times the fc1 kernel alone): the
    two events land around the kernel, inside the fc1 call's own span, and
    the results are bitwise those of a run without them."""
    from moe_expert_dispatch_histc_gb300 import block as blk
    ensure_built()
    inp = make_inputs(wl, 6)
    d = blk.inputs_to_device(inp, wl)
    b = blk.alloc_buffers(wl)
    blk.prepack(wl, d, b)
    shape = blk.shape_of(wl)
    st = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in ev[1:3]:  # a first record creates the CUDA events
        e.record(st)
    B.mc2_moe_counts(shape, d["sel"], b.cnt, b.recv, b.offsets, b.permute_src, b.unpermute_dst,
                     b.ws, b.dev_status)
    ev[0].record(st)
    B.mc2_set_gemm_events(ev[1], ev[2])
    try:
        B.mc2_alltoallv_gmm(shape, d["x"], d["xs"], d["w1"], d["w1s"], b.offsets, b.permute_src,
                            b.ws, b.h, b.h_scale, b.dev_status)
    finally:
        B.mc2_set_gemm_events(None, None)
    ev[3].record(st)
    B.mc2_gmm_alltoallv(shape, b.h, b.h_scale, d["w2"], d["w2s"], b.offsets, b.permute_src,
                        b.unpermute_dst, d["probs"], b.ws, b.out, b.dev_status)
    torch.cuda.synchronize()
    kernel_ms, call_ms = ev[1].elapsed_time(ev[2]), ev[0].elapsed_time(ev[3])
    assert 0 < kernel_ms <= call_ms
    assert ev[0].elapsed_time(ev[1]) >= 0 and ev[2].elapsed_time(ev[3]) >= 0
    _, _, b0 = run_gpu(wl, seed=6)
    assert torch.equal(b0.h.view(torch.uint8), b.h.view(torch.uint8))
    assert torch.equal(b0.out.view(torch.uint8), b.out.view(torch.uint8))
    assert int(b.dev_status.item()) == 0


def test_fc2_alone_on_oracle_h():
    """fc2 + combine fed the oracle's h: isolates the combine segment."""
    wl = SMALL[1]
    inp, d, b = run_gpu(wl, seed=3)
    x, w1, w2 = (as_f64(inp[n], wl.act) for n in ("x", "w1", "w2"))
    ref = orc.block_forward(x, w1, w2, inp["sel"], inp["probs"], wl.E, wl.W, h_dtype="bf16")
    h_ref = torch.from_numpy(ref["h"].astype(np.float32)).to(torch.bfloat16).cuda()
    h = torch.zeros_like(b.h)
    h[:h_ref.shape[0]] = h_ref
    from moe_expert_dispatch_histc_gb300 import block as blk
    B.mc2_gmm_alltoallv(blk.shape_of(wl), h, None, d["w2"], None, b.offsets, b.permute_src,
                        b.unpermute_dst, d["probs"], b.ws, b.out, b.dev_status)
    torch.cuda.synchronize()
    _tol(to_np(b.out), ref["out"], "out from oracle h")


@pytest.mark.parametrize("name", ["uniform", "skew"])
def test_tilings_equal_bitwise_full_size(name):
    """Every tiling accumulates each output in the same K order: the
    full-size h and out are identical bit for bit on single CTAs and on CTA
    pairs."""
    wl = WORKLOADS[name]
    res = []
    for mode in (1, 2):
        B.mc2_set_tile_pairing(mode)
        try:
            _, _, b = run_gpu(wl, seed=5)
        finally:
            B.mc2_set_tile_pairing(0)
        assert int(b.dev_status.item()) == 0
        res.append(b)
    for b in res[1:]:
        assert torch.equal(res[0].h.view(torch.int16), b.h.view(torch.int16))
        assert torch.equal(res[0].out.view(torch.int16), b.out.view(torch.int16))


def test_determinism_bitwise(pairing):
    wl = SMALL[1]
    _, _, b1 = run_gpu(wl, seed=4)
    _, _, b2 = run_gpu(wl, seed=4)
    assert torch.equal(b1.out.view(torch.int16), b2.out.view(torch.int16))
    assert torch.equal(b1.h.view(torch.int16), b2.h.view(torch.int16))


@pytest.mark.parametrize("wl", [SMALL[1], SMALL[3]], ids=lambda w: w.name)
def test_launch_overlap_changes_nothing(wl):
    """Programmatic dependent launch on or off: bitwise the same block."""
    ensure_built()
    try:
        B.mc2_set_launch_overlap(0)
        _, _, b0 = run_gpu(wl, seed=7)
    finally:
        B.mc2_set_launch_overlap(1)
    _, _, b1 = run_gpu(wl, seed=7)
    assert torch.equal(b0.out.view(torch.int16), b1.out.view(torch.int16))
    assert torch.equal(b0.h.view(torch.int16), b1.h.view(torch.int16))
    assert int(b1.dev_status.item()) == 0


COMBINE_SHAPES = [
    Workload("c_multi_mtile", 1024, 256, 128, 8, 2, 2, "bf16"),
    Workload("c_ragged_n", 384, 320, 192, 6, 3, 3, "bf16"),     # k = 3; H = 320: a partial tile
    Workload("c_k8", 512, 512, 128, 16, 8, 4, "bf16"),
    Workload("c_k1", 200, 128, 64, 4, 1, 2, "bf16"),
    Workload("c_fp32", 96, 192, 64, 4, 2, 2, "f32"),
    Workload("c_k10", 128, 256, 64, 16, 10, 2, "bf16"),         # k > 8: the separate kernel
]


@pytest.mark.parametrize("wl", COMBINE_SHAPES + random_shapes(505, 6, "bf16"),
                         ids=lambda w: w.name)
def test_fused_combine_equals_separate_bitwise(wl, pairing):
    """The combine inside the fc2 kernel and the separate combine kernel sum
    the same products in the same slot order: bitwise the same output, also
    with invalid ids and a token whose every slot is invalid (a zero row)."""
    inp = make_inputs(wl, 12)
    sel = inp["sel"].copy()
    sel[0, :] = wl.E                     # token 0: no valid slot
    sel[5 % wl.T, 0] = -1
    sel[wl.T - 1, wl.k - 1] = 1 << 20
    inp["sel"] = np.ascontiguousarray(sel)
    outs = []
    for mode in (0, 1):   # separate kernel, then fused into fc2
        B.mc2_set_combine_path(mode)
        try:
            _, _, b = run_gpu(wl, inputs=inp)
        finally:
            B.mc2_set_combine_path(0)
        outs.append(b)
        assert int(b.dev_status.item()) == B.MC2_DEV_BAD_EXPERT_ID
    o0, o1 = outs[0].out, outs[1].out
    iv = torch.int32 if o0.dtype == torch.float32 else torch.int16
    assert torch.equal(o0.view(iv), o1.view(iv)), "fused combine differs from the separate kernel"
    assert float(o1[0].abs().max()) == 0.0
    x, w1, w2 = (as_f64(inp[n], wl.act) for n in ("x", "w1", "w2"))
    ref = orc.block_forward(x, w1, w2, inp["sel"], inp["probs"], wl.E, wl.W,
                            h_dtype=H_DTYPE[wl.act])
    _tol(to_np(o1), ref["out"], "out with the fused combine")


@pytest.mark.parametrize("name", ["uniform", "skew"])
def test_fused_combine_full_size_repeated_calls(name):
    """The fused combine at full size (CTA pairs, many tokens completing in
    the last tiles, so both the local sums and the deferred list are used):
    three fc2 calls in a row on one workspace (counters and list re-armed by
    every call) give the separate kernel's bits each time."""
    from moe_expert_dispatch_histc_gb300 import block as blk
    wl = WORKLOADS[name]
    inp, d, b = run_gpu(wl, seed=13)
    ref = b.out.clone()
    try:
        B.mc2_set_combine_path(1)
        for _ in range(3):
            b.out.zero_()
            B.mc2_gmm_alltoallv(blk.shape_of(wl), b.h, None, d["w2"], None, b.offsets,
                                b.permute_src, b.unpermute_dst, d["probs"], b.ws, b.out,
                                b.dev_status)
            torch.cuda.synchronize()
            assert torch.equal(ref.view(torch.int16), b.out.view(torch.int16))
    finally:
        B.mc2_set_combine_path(0)
    assert int(b.dev_status.item()) == 0


def _unfused(wl, seed, out=None):
    from moe_expert_dispatch_histc_gb300 import block as blk
    inp = make_inputs(wl, seed)
    d = blk.inputs_to_device(inp, wl)
    b = blk.alloc_buffers(wl)
    xp = torch.empty(wl.T * wl.k, wl.H, dtype=torch.bfloat16, device="cuda")
    blk.run_unfused(wl, d, b, xp)
    torch.cuda.synchronize()
    return inp, d, b, xp


@pytest.mark.parametrize("wl", [w for w in SMALL if w.act == "bf16"], ids=lambda w: w.name)
def test_unfused_baseline_equals_fused_block(wl):
    """Materialised permute + plain grouped fc1, then fc2 + combine: the same
    h and out bits as the fused block, and xp[p] = x[permute_src[p] / k]."""
    inp, d, b, xp = _unfused(wl, 10)
    src, offsets = _counts_exact(wl, inp, b)
    xa = as_f64(inp["x"], wl.act)
    ref = orc.block_forward(xa, as_f64(inp["w1"], wl.act), as_f64(inp["w2"], wl.act), inp["sel"],
                            inp["probs"], wl.E, wl.W, h_dtype="bf16")
    nvalid = int(offsets[-1])
    _tol(to_np(b.h)[:nvalid], ref["h"], "non-fused h")
    _tol(to_np(b.out), ref["out"], "non-fused out")
    x = torch.from_numpy(inp["x"].view(np.int16)).cuda()
    assert torch.equal(xp.view(torch.int16), x[torch.from_numpy(src // wl.k).cuda().long()])
    _, _, bf = run_gpu(wl, seed=10)
    assert torch.equal(b.h.view(torch.int16), bf.h.view(torch.int16))
    assert torch.equal(b.out.view(torch.int16), bf.out.view(torch.int16))
    assert int(b.dev_status.item()) == 0


def test_unfused_baseline_full_size_uniform():
    """The non-fused path at full size against the float64 oracle (every
    element), and bitwise against the fused block."""
    wl = WORKLOADS["uniform"]
    inp, _, b, _ = _unfused(wl, 0)
    src, offsets = _counts_exact(wl, inp, b)
    ref = orc.block_forward(as_f64(inp["x"], wl.act), F64Experts(inp["w1"], wl.act),
                            F64Experts(inp["w2"], wl.act), inp["sel"], inp["probs"], wl.E, wl.W,
                            h_dtype="bf16")
    _tol(to_np(b.h)[:int(offsets[-1])], ref["h"], "non-fused h (full size)")
    _tol(to_np(b.out), ref["out"], "non-fused out (full size)")
    _, _, bf = run_gpu(wl, seed=0)
    assert torch.equal(b.out.view(torch.int16), bf.out.view(torch.int16))
    assert int(b.dev_status.item()) == 0


# ------------------------------------------------------------------ edge cases
def _custom(wl, sel, seed=5):
    inp = make_inputs(wl, seed)
    inp["sel"] = np.ascontiguousarray(sel.astype(np.int32))
    return inp


def _check_custom(wl, inp, expect_bad=False):
    inp, d, b = run_gpu(wl, inputs=inp)
    src, offsets = _counts_exact(wl, inp, b)
    x, w1, w2 = (as_f64(inp[n], wl.act) for n in ("x", "w1", "w2"))
    ref = orc.block_forward(x, w1, w2, inp["sel"], inp["probs"], wl.E, wl.W, h_dtype="bf16")
    nvalid = int(offsets[-1])
    if nvalid:
        _tol(to_np(b.h)[:nvalid], ref["h"], "h")
    _tol(to_np(b.out), ref["out"], "out")
    status = int(b.dev_status.item())
    assert bool(status & B.MC2_DEV_BAD_EXPERT_ID) == expect_bad
    assert not status & B.MC2_DEV_TIMEOUT


def test_all_tokens_to_one_expert(pairing):
    wl = Workload("one_expert", 512, 256, 128, 8, 1, 2, "bf16")
    _check_custom(wl, _custom(wl, np.full((512, 1), 5)))


def test_most_experts_empty(pairing):
    wl = Workload("sparse", 300, 256, 128, 16, 2, 2, "bf16")
    sel = np.stack([np.full(300, 3), np.full(300, 12)], axis=1)
    _check_custom(wl, _custom(wl, sel))


def test_invalid_ids_are_flagged_and_skipped(pairing):
    wl = Workload("bad_ids", 64, 256, 128, 8, 2, 2, "bf16")
    inp = make_inputs(wl, 6)
    sel = inp["sel"].copy()
    sel[3, 0], sel[17, 1], sel[40, 0] = 8, -1, 1000
    _check_custom(wl, _custom(wl, sel, seed=6), expect_bad=True)


def test_zero_routing_weights(pairing):
    """Slots with probability 0 (and a token whose every weight is 0) add
    nothing: out matches the oracle, and the all-zero token's row is 0."""
    wl = Workload("zero_probs", 512, 256, 128, 8, 4, 2, "bf16")
    inp = make_inputs(wl, 9)
    probs = inp["probs"].copy()
    probs[::3, 1] = 0.0
    probs[7, :] = 0.0
    inp["probs"] = np.ascontiguousarray(probs)
    inp, d, b = run_gpu(wl, inputs=inp)
    x, w1, w2 = (as_f64(inp[n], wl.act) for n in ("x", "w1", "w2"))
    ref = orc.block_forward(x, w1, w2, inp["sel"], inp["probs"], wl.E, wl.W, h_dtype="bf16")
    _tol(to_np(b.out), ref["out"], "out with zero weights")
    assert float(b.out[7].float().abs().max()) == 0.0
    assert int(b.dev_status.item()) == 0


def test_empty_input():
    wl = Workload("empty", 0, 256, 128, 8, 2, 2, "bf16")
    inp, d, b = run_gpu(wl)
    assert to_np(b.cnt).sum() == 0 and to_np(b.offsets).sum() == 0


# ------------------------------------------------------------------ full size
@pytest.mark.parametrize("name", ["uniform", "skew", "decode"])
def test_full_size_full(name):
    """The named workloads at full size, in the launch configuration of the
    benchmark (one mc2_moe_forward call): counts and indices bit-exact, and
    every element of h and out within the tolerance of the float64 oracle."""
    wl = WORKLOADS[name]
    inp, d, b = run_gpu(wl, seed=0)
    src, offsets = _counts_exact(wl, inp, b)
    x = as_f64(inp["x"], wl.act)
    w1, w2 = F64Experts(inp["w1"], wl.act), F64Experts(inp["w2"], wl.act)
    ref = orc.block_forward(x, w1, w2, inp["sel"], inp["probs"], wl.E, wl.W, h_dtype="bf16")
    nvalid = int(offsets[-1])
    _tol(to_np(b.h)[:nvalid], ref["h"], f"{name}: h (all rows)")
    _tol(to_np(b.out), ref["out"], f"{name}: out (all tokens)")
    # the first and last row of the busiest expert and the last token
    cnt = np.diff(offsets)
    e_big = int(np.argmax(cnt))
    for p in (int(offsets[e_big]), int(offsets[e_big + 1]) - 1):
        _tol(to_np(b.h)[p:p + 1], ref["h"][p:p + 1], f"{name}: h row {p}")
    _tol(to_np(b.out)[-1:], ref["out"][-1:], f"{name}: last token")
    assert int(b.dev_status.item()) == 0
