"""Parity of the int8 path with the oracle (int64 accumulators, float64
dequant), through the C ABI.

The int8 products run on bf16 tensor cores with K summed in exact chunks, so
the int32 accumulators must equal the oracle's exactly.  The per-row
re-quantisation decides integers from floats; both sides decide in float32,
so codes may differ only where h / hs lands within a few fp32 ulp of a .5 tie
(the GPU's silu uses the fast exponential): at most 1 code, on a tiny fraction
of elements.  fc2 is therefore checked exactly on the GPU's own h_q.
"""
import numpy as np
import pytest
import torch

from oracle import mc2_oracle as orc
from moe_expert_dispatch_histc_gb300 import binding as B
from moe_expert_dispatch_histc_gb300 import block as blk
from moe_expert_dispatch_histc_gb300.workloads import WORKLOADS, Workload, make_inputs

from gpu_util import ensure_built, random_shapes, to_np

pytestmark = pytest.mark.gpu


def _run(wl, inp, out):
    ensure_built()
    d = blk.inputs_to_device(inp, wl)
    b = blk.alloc_buffers(wl, out=out)
    blk.prepack(wl, d, b, out=out)
    blk.run_segments(wl, d, b, out=out)
    torch.cuda.synchronize()
    return d, b


@pytest.fixture(params=[0, 1, 2], ids=["wide", "single_cta", "cta_pairs"])
def pairing(request):
    """Force one int8 GEMM tiling for the test: the default 128 x 256 tiles
    (K chunks folded in TMEM), 128 x 128 tiles, or 256 x 128 CTA pairs."""
    ensure_built()
    B.mc2_set_tile_pairing(request.param)
    yield request.param
    B.mc2_set_tile_pairing(0)


SMALL_I8 = [
    Workload("i8_small", 256, 256, 128, 8, 2, 2, "i8"),
    Workload("i8_chunk_edge", 128, 2112, 192, 4, 2, 2, "i8"),    # K = 33 k-blocks: chunks 16+16+1
    Workload("i8_k3072", 64, 3072, 1536, 4, 2, 2, "i8"),         # three full chunks, two in fc2
    Workload("i8_k4096", 96, 4096, 320, 4, 2, 2, "i8"),          # four chunks (two folds); I % 128 = 64
    Workload("i8_fc2_k3072", 64, 320, 3072, 4, 2, 2, "i8"),      # fc2 K = 3072; H % 256 = 64
]


@pytest.mark.parametrize("wl", SMALL_I8, ids=lambda w: w.name)
def test_int8_fc1_accumulators_exact(wl, pairing):
    inp = make_inputs(wl, 7)
    d, b = _run(wl, inp, out="i32")
    ref = orc.quant_block_forward(inp["x"], inp["xs"], inp["w1"], inp["w1s"], inp["w2"],
                                  inp["w2s"], inp["sel"], inp["probs"], wl.E, wl.W)
    n = int(ref["offsets"][-1])
    assert np.array_equal(to_np(b.h)[:n].astype(np.int64), ref["acc1"])
    assert int(b.dev_status.item()) == 0


@pytest.mark.parametrize("K", [3072, 4096])
def test_int8_worst_case_magnitudes_exact(pairing, K):
    """All values +-127: |acc| = K * 127^2 (49.5M at K = 3072, 66.1M at
    K = 4096) > 2^24, exact only by chunking (and, for the wide tiles, by
    folding the chunks into int32 in TMEM)."""
    wl = Workload("i8_worst", 64, K, 128, 2, 1, 1, "i8")
    inp = make_inputs(wl, 0)
    inp["x"] = np.full_like(inp["x"], 127)
    inp["x"][1::2] = -127
    inp["w1"] = np.full_like(inp["w1"], -127)
    inp["w1"][:, :, 1::3] = 127
    d, b = _run(wl, inp, out="i32")
    ref = orc.quant_block_forward(inp["x"], inp["xs"], inp["w1"], inp["w1s"], inp["w2"],
                                  inp["w2s"], inp["sel"], inp["probs"], wl.E, wl.W)
    assert np.abs(ref["acc1"]).max() == K * 127 * 127
    assert np.array_equal(to_np(b.h).astype(np.int64), ref["acc1"])


@pytest.mark.parametrize("K", [2048, 3072, 4096])
def test_int8_worst_case_dequant_tilings_bitwise(K):
    """All values +-127 in long same-sign runs: most fc1 sums lie past 2^24
    (up to 47M at K = 4096), where fp32(acc) rounds.  The wide tiles form
    fp32(acc) with one fp32 add of the two chunks' exact sums at K = 2048 and
    by converting the folded int32 sums beyond; the 128 x 128 tiles convert
    the exact int32 sums.  h_q, its scales and the block output must agree bit
    for bit, and the output stays within the tolerance of the oracle."""
    wl = Workload("i8_worst_dq", 64, K, 128, 2, 1, 1, "i8")
    inp = make_inputs(wl, 1)
    inp["x"] = np.full_like(inp["x"], 127)
    inp["x"][1::2] = -127
    inp["x"][2::4, ::5] = -127
    inp["w1"] = np.full_like(inp["w1"], 127)
    inp["w1"][:, :, 1::3] = -127
    inp["w1"][:, ::7, :] = -inp["w1"][:, ::7, :]
    res = []
    for mode in (0, 1):
        B.mc2_set_tile_pairing(mode)
        try:
            d, b = _run(wl, inp, out="bf16")
            res.append((to_np(b.h), to_np(b.h_scale), to_np(b.out)))
            assert int(b.dev_status.item()) == 0
        finally:
            B.mc2_set_tile_pairing(0)
    for a, c in zip(res[0], res[1]):
        assert np.array_equal(a.view(np.uint8), c.view(np.uint8))
    ref = orc.quant_block_forward(inp["x"], inp["xs"], inp["w1"], inp["w1s"], inp["w2"],
                                  inp["w2s"], inp["sel"], inp["probs"], wl.E, wl.W)
    assert (np.abs(ref["acc1"]) > 2 ** 24).mean() > 0.5  # most sums round in fp32
    ok, a, m = orc.bf16_tolerance_ok(res[0][2], ref["out"])
    assert ok, f"out: max {a:.3e}, mean {m:.3e}"


def _check_block(wl, inp, expect_bad=False):
    """The int8 block through its entry points against the oracle: scales to
    fp32 rounding and codes to +-1 at ties, fc2 exactly on the GPU's own h_q,
    the output within the block's tolerance; the device status word."""
    d, b = _run(wl, inp, out="bf16")
    hq = to_np(b.h)
    hs = to_np(b.h_scale)
    ref = orc.quant_block_forward(inp["x"], inp["xs"], inp["w1"], inp["w1s"], inp["w2"],
                                  inp["w2s"], inp["sel"], inp["probs"], wl.E, wl.W)
    n = int(ref["offsets"][-1])
    assert np.array_equal(to_np(b.offsets), ref["offsets"])
    # re-quantisation: scales agree to fp32 rounding, codes to +-1 at ties
    assert np.allclose(hs[:n], ref["hs"], rtol=1e-5, atol=0)
    diff = np.abs(hq[:n].astype(int) - ref["hq"].astype(int))
    assert diff.max() <= 1 and (diff > 0).mean() < 1e-3
    # fc2 exactly on the GPU's own h_q
    acc2 = torch.empty((wl.R, wl.H), dtype=torch.int32, device="cuda")
    B.mc2_gmm_alltoallv(blk.shape_of(wl, "i32"), b.h, None, d["w2"], None, b.offsets,
                        b.permute_src, None, None, b.ws, acc2, b.dev_status)
    torch.cuda.synchronize()
    ref2 = orc.quant_block_forward(inp["x"], inp["xs"], inp["w1"], inp["w1s"], inp["w2"],
                                   inp["w2s"], inp["sel"], inp["probs"], wl.E, wl.W,
                                   hq_override=(hq[:n], hs[:n]))
    assert np.array_equal(to_np(acc2)[:n].astype(np.int64), ref2["acc2"])
    # the block output (bf16) within the block's tolerance of the float64 oracle
    ok, a, m = orc.bf16_tolerance_ok(to_np(b.out), ref["out"])
    assert ok, f"out: max {a:.3e}, mean {m:.3e}"
    status = int(b.dev_status.item())
    assert bool(status & B.MC2_DEV_BAD_EXPERT_ID) == expect_bad
    assert not status & B.MC2_DEV_TIMEOUT
    return ref


@pytest.mark.parametrize("wl", SMALL_I8, ids=lambda w: w.name)
def test_int8_block_parity(wl, pairing):
    _check_block(wl, make_inputs(wl, 8))


@pytest.mark.parametrize("wl", random_shapes(202, 10, "i8"), ids=lambda w: w.name)
def test_int8_random_shapes(wl, pairing):
    """Seeded random shapes on every int8 tiling: fc1's int32 accumulators
    bit-exact, then the whole block against the oracle."""
    inp = make_inputs(wl, 5)
    d, b = _run(wl, inp, out="i32")
    ref = orc.quant_block_forward(inp["x"], inp["xs"], inp["w1"], inp["w1s"], inp["w2"],
                                  inp["w2s"], inp["sel"], inp["probs"], wl.E, wl.W)
    n = int(ref["offsets"][-1])
    assert np.array_equal(to_np(b.h)[:n].astype(np.int64), ref["acc1"])
    _check_block(wl, inp)


def _with_sel(wl, sel, seed):
    inp = make_inputs(wl, seed)
    inp["sel"] = np.ascontiguousarray(np.asarray(sel).astype(np.int32))
    return inp


def test_int8_all_tokens_to_one_expert(pairing):
    """Every token on expert 5, the seven others empty: 512 rows make four row
    tiles of one expert, K = 3072 runs in three exact chunks; fc1's int32
    accumulators exact, the block within tolerance."""
    wl = Workload("i8_one_expert", 512, 3072, 256, 8, 1, 2, "i8")
    inp = _with_sel(wl, np.full((512, 1), 5), 3)
    d, b = _run(wl, inp, out="i32")
    ref = orc.quant_block_forward(inp["x"], inp["xs"], inp["w1"], inp["w1s"], inp["w2"],
                                  inp["w2s"], inp["sel"], inp["probs"], wl.E, wl.W)
    assert np.array_equal(to_np(b.h)[:512].astype(np.int64), ref["acc1"])
    _check_block(wl, inp)


def test_int8_large_topk(pairing):
    """Twelve slots per token (the combine's generic loop) on sixteen experts."""
    wl = Workload("i8_k12", 96, 256, 128, 16, 12, 4, "i8")
    _check_block(wl, make_inputs(wl, 9))


def test_int8_most_experts_empty(pairing):
    wl = Workload("i8_sparse", 300, 256, 128, 16, 2, 2, "i8")
    _check_block(wl, _with_sel(wl, np.stack([np.full(300, 3), np.full(300, 12)], axis=1), 4))


def test_int8_invalid_ids_are_flagged_and_skipped():
    wl = Workload("i8_bad_ids", 64, 256, 128, 8, 2, 2, "i8")
    sel = make_inputs(wl, 6)["sel"].copy()
    sel[3, 0], sel[17, 1], sel[40, 0] = 8, -1, 1000
    _check_block(wl, _with_sel(wl, sel, 6), expect_bad=True)


def test_int8_empty_input():
    wl = Workload("i8_empty", 0, 256, 128, 8, 2, 2, "i8")
    d, b = _run(wl, make_inputs(wl, 0), out="bf16")
    assert to_np(b.cnt).sum() == 0 and to_np(b.offsets).sum() == 0
    assert int(b.dev_status.item()) == 0


def test_int8_full_size_full():
    """The int8 workload at full size through the block's entry points: the
    row scales and codes of the re-quantisation against the oracle (codes
    within 1 at fp32 ties), fc2's int32 accumulators exact on the GPU's own
    codes, and every output element within the block's tolerance."""
    wl = WORKLOADS["int8"]
    inp = make_inputs(wl, 0)
    d, b = _run(wl, inp, out="bf16")
    hq, hs = to_np(b.h), to_np(b.h_scale)
    ref = orc.quant_block_forward(inp["x"], inp["xs"], inp["w1"], inp["w1s"], inp["w2"],
                                  inp["w2s"], inp["sel"], inp["probs"], wl.E, wl.W)
    n = int(ref["offsets"][-1])
    assert np.array_equal(to_np(b.offsets), ref["offsets"])
    assert np.array_equal(to_np(b.permute_src), ref["permute_src"])
    assert np.allclose(hs[:n], ref["hs"], rtol=1e-5, atol=0)
    diff = np.abs(hq[:n].astype(int) - ref["hq"].astype(int))
    assert diff.max() <= 1 and (diff > 0).mean() < 1e-3
    ok, a, m = orc.bf16_tolerance_ok(to_np(b.out), ref["out"])
    assert ok, f"int8 out (all tokens): max {a:.3e}, mean {m:.3e}"
    acc2 = torch.empty((wl.R, wl.H), dtype=torch.int32, device="cuda")
    B.mc2_gmm_alltoallv(blk.shape_of(wl, "i32"), b.h, None, d["w2"], None, b.offsets,
                        b.permute_src, None, None, b.ws, acc2, b.dev_status)
    torch.cuda.synchronize()
    ref2 = orc.quant_block_forward(inp["x"], inp["xs"], inp["w1"], inp["w1s"], inp["w2"],
                                   inp["w2s"], inp["sel"], inp["probs"], wl.E, wl.W,
                                   hq_override=(hq[:n], hs[:n]))
    assert np.array_equal(to_np(acc2)[:n].astype(np.int64), ref2["acc2"])
    assert int(b.dev_status.item()) == 0


def test_int8_full_size_accumulators_full(pairing):
    """The int8 workload at full size: fc1 sums K = 3072 in three exact chunks
    and fc2 K = 1536 in two, and every CTA takes several tiles, so the TMEM
    chunk-slot ring wraps many times.  Every element of both int32
    accumulators (fc2 on random int8 rows) bit-exact against the oracle."""
    wl = WORKLOADS["int8"]
    inp = make_inputs(wl, 3)
    d, b = _run(wl, inp, out="i32")
    ref = orc.quant_block_forward(inp["x"], inp["xs"], inp["w1"], inp["w1s"], inp["w2"],
                                  inp["w2s"], inp["sel"], inp["probs"], wl.E, wl.W)
    n = int(ref["offsets"][-1])
    assert np.array_equal(to_np(b.permute_src), ref["permute_src"])
    assert np.array_equal(to_np(b.h)[:n].astype(np.int64), ref["acc1"])
    rng = np.random.default_rng(11)
    hq = rng.integers(-127, 128, (wl.R, wl.I)).astype(np.int8)
    acc2 = torch.empty((wl.R, wl.H), dtype=torch.int32, device="cuda")
    B.mc2_gmm_alltoallv(blk.shape_of(wl, "i32"), torch.from_numpy(hq).cuda(), None, d["w2"], None,
                        b.offsets, b.permute_src, None, None, b.ws, acc2, b.dev_status)
    torch.cuda.synchronize()
    ref2 = orc.quant_block_forward(inp["x"], inp["xs"], inp["w1"], inp["w1s"], inp["w2"],
                                   inp["w2s"], inp["sel"], inp["probs"], wl.E, wl.W,
                                   hq_override=(hq[:n], np.ones(n, np.float32)))
    assert np.array_equal(to_np(acc2)[:n].astype(np.int64), ref2["acc2"])
    assert int(b.dev_status.item()) == 0


@pytest.mark.parametrize("wl", [Workload("i8_mid", 2048, 1024, 512, 16, 4, 4, "i8"),
                                Workload("i8_mid3", 1024, 3072, 1536, 16, 4, 4, "i8")],
                         ids=lambda w: w.name)
def test_int8_tilings_equal_bitwise(wl):
    """Every int8 GEMM tiling accumulates each output's K chunks exactly and
    dequantises alike: h_q, its scales and the block output are identical
    bit for bit (workloads with several tiles per CTA and per CTA pair; the
    second folds a chunk in fc1)."""
    inp = make_inputs(wl, 4)
    res = []
    for mode in (0, 1, 2):
        B.mc2_set_tile_pairing(mode)
        try:
            d, b = _run(wl, inp, out="bf16")
            res.append((to_np(b.h), to_np(b.h_scale), to_np(b.out)))
            assert int(b.dev_status.item()) == 0
        finally:
            B.mc2_set_tile_pairing(0)
    for other in res[1:]:
        for a, c in zip(res[0], other):
            assert np.array_equal(a.view(np.uint8), c.view(np.uint8))
