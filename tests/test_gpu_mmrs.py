"""Quantised matmul + reduce-scatter over logical ranks on the GPU, against
the CPU oracle.  Two forms: the two-pass one writes every rank's int32
partial product to the workspace (checked bit-exact); the fused one keeps
them on chip, and its bf16 result must equal the two-pass result bit for bit
(the same fma per rank, in rank order).  Both within the block's tolerance
rule of the float64 oracle."""
import numpy as np
import pytest
import torch

from oracle import mc2_oracle as orc
from moe_expert_dispatch_histc_gb300 import binding as B

from gpu_util import ensure_built

pytestmark = pytest.mark.gpu


def _align(v, a=256):
    return (v + a - 1) // a * a


@pytest.fixture(autouse=True)
def _default_path():
    yield
    B.mc2_set_mmrs_path(0)


def _call(s, d, ws, m, n, path):
    B.mc2_set_mmrs_path(path)
    out = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.mc2_mm_reduce_scatter_i8(s, d[0], d[1], d[2], d[3], out, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert B.mc2_last_launch_count() == (2 if path == 0 else 4)
    return out


def _run(W, m, k, n, seed=0, worst=False):
    ensure_built()
    rng = np.random.default_rng(seed)
    if worst:   # every product at the int8 extreme with one sign: |acc| = k * 127^2 per rank
        x1 = np.full((W, m, k), 127, np.int8)
        x2 = np.full((W, k, n), -127, np.int8)
    else:
        x1 = rng.integers(-127, 128, (W, m, k)).astype(np.int8)
        x2 = rng.integers(-127, 128, (W, k, n)).astype(np.int8)
    x1s = rng.uniform(1e-3, 1e-2, (W, m)).astype(np.float32)
    x2s = rng.uniform(1e-3, 1e-2, (W, n)).astype(np.float32)
    s = B.MmrsShape(m, k, n, W)
    nbytes = B.mc2_mm_reduce_scatter_workspace_bytes(s)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    d = [torch.from_numpy(a).cuda() for a in (x1, x1s, x2, x2s)]
    out = _call(s, d, ws, m, n, 1)
    fused = _call(s, d, ws, m, n, 0)
    assert torch.equal(fused.view(torch.int16), out.view(torch.int16)), \
        "fused result differs from the two-pass result"
    acc, total, per_rank = orc.mm_reduce_scatter(x1, x1s, x2, x2s)
    # workspace: bf16 x1 [W*m, k], bf16 x2 [W, k, n], int32 partials [W*m, n]
    off = _align(W * m * k * 2) + _align(W * k * n * 2)
    got_acc = ws[off:off + W * m * n * 4].view(torch.int32).view(W, m, n).cpu().numpy()
    assert np.array_equal(got_acc, acc), "int32 partial products differ"
    got = out.float().cpu().numpy()
    ok, a, b = orc.bf16_tolerance_ok(got, total)
    assert ok, (a, b)
    for r in range(W):   # each rank's reduce-scatter block
        blk = got[r * (m // W):(r + 1) * (m // W)]
        assert np.array_equal(blk, got.reshape(W, m // W, n)[r])
    return got, total


@pytest.mark.parametrize("W,m,k,n", [(1, 64, 256, 128), (2, 64, 256, 128), (4, 256, 1024, 320),
                                     (8, 136, 512, 192), (3, 300, 1088, 64), (2, 512, 3072, 128),
                                     (1, 512, 2048, 576), (8, 776, 128, 320)])
def test_mm_reduce_scatter_parity(W, m, k, n):
    _run(W, m, k, n, seed=W * 7 + k)


def _random_mmrs_shapes(seed, n):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        W = int(rng.choice([1, 2, 3, 4, 8]))
        out.append((W, W * int(rng.integers(1, 80)), 64 * int(rng.integers(1, 40)),
                    64 * int(rng.integers(1, 10))))
    return out


@pytest.mark.parametrize("W,m,k,n", _random_mmrs_shapes(404, 8))
def test_mm_reduce_scatter_random_shapes(W, m, k, n):
    """Seeded random shapes (ragged row and column tiles, one to three K
    chunks, odd rank counts): bitwise equal to the two-pass form, int32
    partials exact, the result within the tolerance."""
    _run(W, m, k, n, seed=m + k + n)


@pytest.mark.parametrize("k", [2048, 4096])
def test_mm_reduce_scatter_worst_case_accumulators(k):
    """Every product -127*127: |acc| = k * 127^2 > 2^24 per rank (33 M at
    k = 2048, 66 M at k = 4096), exact in int32 (1024-long exact chunks; at
    k = 4096 the fused form has one accumulator set in TMEM instead of two).
    With two chunks the fused form rounds their fp32 sum once, which must
    equal the two-pass form's conversion of the exact int32 sum bit for bit."""
    _run(2, 128, k, 128, worst=True)


def test_mm_reduce_scatter_empty_and_rejected():
    ensure_built()
    s = B.MmrsShape(0, 256, 128, 2)
    ws = torch.empty(B.mc2_mm_reduce_scatter_workspace_bytes(s), dtype=torch.uint8, device="cuda")
    x2 = torch.zeros(2, 256, 128, dtype=torch.int8, device="cuda")
    x2s = torch.ones(2, 128, device="cuda")
    for path in (0, 1):
        B.mc2_set_mmrs_path(path)
        assert B.mc2_mm_reduce_scatter_i8(s, None, None, x2, x2s, None, ws, None) == B.MC2_OK
    bad = B.MmrsShape(6, 256, 128, 4)   # m not divisible by W
    assert B.mc2_mm_reduce_scatter_i8(bad, x2, x2s, x2, x2s, x2, ws, None,
                                      check=False) == B.MC2_ERR_INVALID_ARG


@pytest.mark.parametrize("W,m,k,n", [(2, 8192, 512, 2048), (2, 4096, 3072, 2048),
                                     (8, 4096, 1024, 4096)])
def test_mm_reduce_scatter_many_tiles_per_cluster(W, m, k, n):
    """Shapes where every CTA pair of the fused kernel takes three or more
    output tiles (256-column tiles with two accumulator sets at k = 512;
    128-column tiles with three K chunks at k = 3072; the benchmarked
    W8 m4096 k1024 n4096), so accumulators and barrier phases are reused
    across tiles.  The fused result must equal the two-pass result bit for
    bit; sampled rows of both, and the two-pass int32 partials, against the
    oracle on those rows."""
    ensure_built()
    rng = np.random.default_rng(k + n)
    x1 = rng.integers(-127, 128, (W, m, k)).astype(np.int8)
    x2 = rng.integers(-127, 128, (W, k, n)).astype(np.int8)
    x1s = rng.uniform(1e-3, 1e-2, (W, m)).astype(np.float32)
    x2s = rng.uniform(1e-3, 1e-2, (W, n)).astype(np.float32)
    s = B.MmrsShape(m, k, n, W)
    ws = torch.empty(B.mc2_mm_reduce_scatter_workspace_bytes(s), dtype=torch.uint8, device="cuda")
    d = [torch.from_numpy(a).cuda() for a in (x1, x1s, x2, x2s)]
    two = _call(s, d, ws, m, n, 1)
    off = _align(W * m * k * 2) + _align(W * k * n * 2)
    acc = ws[off:off + W * m * n * 4].view(torch.int32).view(W, m, n)
    fused = _call(s, d, ws, m, n, 0)
    assert torch.equal(fused.view(torch.int16), two.view(torch.int16)), \
        "fused result differs from the two-pass result"
    rows = np.sort(np.concatenate([rng.choice(m, 14, replace=False), [0, m - 1]]))
    ref_acc, ref_total, _ = orc.mm_reduce_scatter(x1[:, rows], x1s[:, rows], x2, x2s)
    assert np.array_equal(acc[:, torch.from_numpy(rows).cuda()].cpu().numpy(), ref_acc)
    ok, a, b = orc.bf16_tolerance_ok(fused.float().cpu().numpy()[rows], ref_total)
    assert ok, (a, b)
