"""Host-side checks of the C ABI: the library loads, exports what the header
declares, applies its argument rules and launches nothing on bad input.
None of these calls reaches the GPU."""
import pytest

from moe_expert_dispatch_histc_gb300 import binding as B
from moe_expert_dispatch_histc_gb300.build import build
from moe_expert_dispatch_histc_gb300.workloads import WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def built():
    build()
    return B.lib()


def test_header_symbols_are_exported():
    names = B.header_functions()
    assert "mc2_moe_counts" in names and "mc2_alltoallv_gmm" in names
    assert "mc2_gmm_alltoallv" in names
    L = B.lib()
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/mc2moe.h but not exported"


def test_binding_covers_header():
    assert set(B.header_functions()) <= set(B._SIGS)


def _shape(**kw):
    base = dict(T=64, H=256, I=128, E=8, k=2, W=2, act="bf16", out=None)
    base.update(kw)
    return B.Shape.make(**base)


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_named_workloads_are_valid(name):
    wl = WORKLOADS[name]
    s = B.Shape.make(wl.T, wl.H, wl.I, wl.E, wl.k, wl.W, wl.act)
    assert B.mc2_check_shape(s) == B.MC2_OK
    assert B.mc2_workspace_bytes(s) > 0


@pytest.mark.parametrize("kw", [
    dict(E=9), dict(T=63), dict(k=9), dict(k=0), dict(H=200), dict(I=100), dict(H=0),
    dict(E=2048, W=2), dict(W=0), dict(T=-2), dict(act="i32", out="i32"), dict(act="f32", out="bf16"),
    dict(act="bf16", out="i32"), dict(act="bf16", out="f32"),
])
def test_shape_rules_reject(kw):
    s = _shape(**kw)
    assert B.mc2_check_shape(s) == B.MC2_ERR_INVALID_ARG
    assert B.mc2_workspace_bytes(s) == 0


def test_shape_rules_accept_edges():
    for kw in (dict(T=0), dict(k=8), dict(W=1, T=3), dict(E=1, k=1, W=1), dict(act="f32", out="f32"),
               dict(act="i8", out="bf16"), dict(act="i8", out="i32"), dict(H=64, I=64)):
        assert B.mc2_check_shape(_shape(**kw)) == B.MC2_OK, kw


def test_workspace_is_deterministic_and_aligned():
    s = _shape(T=4096, H=2048, I=768, E=64, k=8, W=4)
    a, b = B.mc2_workspace_bytes(s), B.mc2_workspace_bytes(s)
    assert a == b and a % 256 == 0
    # the fc2 rows of the combine dominate: R * H fp16 values plus one fp32
    # decode factor per 64 columns
    assert a >= 4096 * 8 * 2048 * 2 + 4096 * 8 * (2048 // 64) * 4


def test_null_pointers_are_rejected_before_any_launch():
    s = _shape()
    fake = 1 << 40  # never dereferenced: validation fails first
    assert B.mc2_moe_counts(s, fake, fake, fake, fake, fake, fake, None, None, stream=0,
                            check=False) == B.MC2_ERR_INVALID_ARG
    assert B.mc2_moe_counts(s, None, fake, fake, fake, fake, fake, fake, None, stream=0,
                            check=False) == B.MC2_ERR_INVALID_ARG
    assert B.mc2_alltoallv_gmm(s, fake, None, None, None, fake, fake, fake, fake, None,
                               stream=0, check=False) == B.MC2_ERR_INVALID_ARG
    assert B.mc2_gmm_alltoallv(s, fake, None, fake, None, fake, fake, fake, None, fake, fake,
                               stream=0, check=False) == B.MC2_ERR_INVALID_ARG
    # scales are for the int8 path only
    assert B.mc2_alltoallv_gmm(s, fake, fake, fake, None, fake, fake, fake, fake, None,
                               stream=0, check=False) == B.MC2_ERR_INVALID_ARG
    bad = _shape(E=9)
    assert B.mc2_moe_forward(bad, *([fake] * 17), None, stream=0,
                             check=False) == B.MC2_ERR_INVALID_ARG
    assert B.mc2_selftest_wait(1000, None, stream=0, check=False) == B.MC2_ERR_INVALID_ARG


def test_int8_empty_batch_accepts_null_arrays_and_launches_nothing():
    """T = 0: the per-token and per-row arrays are empty, so x, the scales,
    permute_src and h may be NULL; the calls succeed without touching the
    device (the stream argument is never used).  With tokens present the
    scales are required."""
    fake = 1 << 40
    s = _shape(T=0, act="i8", out="bf16")
    assert B.mc2_alltoallv_gmm(s, None, None, None, None, fake, None, fake, None, None,
                               stream=0, check=False) == B.MC2_OK
    assert B.mc2_gmm_alltoallv(s, None, None, None, None, fake, None, None, None, fake, None,
                               stream=0, check=False) == B.MC2_OK
    s = _shape(act="i8", out="bf16")
    assert B.mc2_alltoallv_gmm(s, fake, None, fake, fake, fake, fake, fake, fake, fake,
                               stream=0, check=False) == B.MC2_ERR_INVALID_ARG
    assert B.mc2_gmm_alltoallv(s, fake, None, fake, fake, fake, fake, fake, fake, fake, fake,
                               stream=0, check=False) == B.MC2_ERR_INVALID_ARG


def test_misaligned_pointers_are_rejected():
    s = _shape()
    fake = 1 << 40
    odd = fake + 8          # 8-byte aligned only
    assert B.mc2_moe_counts(s, odd, fake, fake, fake, fake, fake, fake, None, stream=0,
                            check=False) == B.MC2_ERR_INVALID_ARG
    assert B.mc2_moe_counts(s, fake, fake, fake, fake, fake, fake, fake + 16, None, stream=0,
                            check=False) == B.MC2_ERR_INVALID_ARG     # ws needs 256 bytes
    assert B.mc2_alltoallv_gmm(s, odd, None, fake, None, fake, fake, fake, fake, None,
                               stream=0, check=False) == B.MC2_ERR_INVALID_ARG
    assert B.mc2_gmm_alltoallv(s, fake, None, fake, None, fake, fake, fake, fake, fake, odd,
                               stream=0, check=False) == B.MC2_ERR_INVALID_ARG
    # the allocation-free counts take the same pointer rule (on this machine a
    # call that got past it would fail its device lookup with MC2_ERR_CUDA)
    for i in range(6):
        ptrs = [fake] * 6
        ptrs[i] = odd
        assert B.mc2_moe_counts_static(s, *ptrs, None, stream=0,
                                       check=False) == B.MC2_ERR_INVALID_ARG, i


def test_forward_validates_every_segment_before_enqueuing():
    """A bad fc1 or fc2 argument is reported before the counts are launched
    (with no GPU here, a launch would have failed with MC2_ERR_CUDA)."""
    s = _shape()
    fake = 1 << 40
    args = dict(x=fake, x_scale=None, sel=fake, probs=fake, w1=fake, w1_scale=None, w2=fake,
                w2_scale=None, cnt=fake, recv=fake, offsets=fake, permute_src=fake,
                unpermute_dst=fake, h=fake, h_scale=None, out=fake, ws=fake)
    for bad in (dict(x=None), dict(w2=None), dict(out=fake + 4), dict(h_scale=fake)):
        a = {**args, **bad}
        assert B.mc2_moe_forward(s, *a.values(), None, stream=0,
                                 check=False) == B.MC2_ERR_INVALID_ARG, bad


def test_baseline_path_argument_rules():
    fake = 1 << 40
    s = _shape()
    assert B.mc2_permute_rows(s, fake, fake, None, stream=0, check=False) == B.MC2_ERR_INVALID_ARG
    assert B.mc2_permute_rows(s, fake + 8, fake, fake, stream=0,
                              check=False) == B.MC2_ERR_INVALID_ARG
    assert B.mc2_gmm_swiglu(s, fake, fake, None, fake, None, stream=0,
                            check=False) == B.MC2_ERR_INVALID_ARG
    assert B.mc2_gmm_swiglu(_shape(E=9), fake, fake, fake, fake, None, stream=0,
                            check=False) == B.MC2_ERR_INVALID_ARG
    for act in ("f32", "i8"):  # the baseline path is bf16 only
        sa = _shape(act=act)
        assert B.mc2_permute_rows(sa, fake, fake, fake, stream=0,
                                  check=False) == B.MC2_ERR_UNSUPPORTED
        assert B.mc2_gmm_swiglu(sa, fake, fake, fake, fake, None, stream=0,
                                check=False) == B.MC2_ERR_UNSUPPORTED


def test_mm_reduce_scatter_rules():
    ok = B.MmrsShape(64, 256, 128, 2)
    assert B.mc2_mm_reduce_scatter_workspace_bytes(ok) >= 2 * 64 * 128 * 4
    for bad in (B.MmrsShape(63, 256, 128, 2), B.MmrsShape(64, 200, 128, 2),
                B.MmrsShape(64, 256, 100, 2), B.MmrsShape(64, 4160, 128, 2),
                B.MmrsShape(64, 256, 128, 0), B.MmrsShape(-2, 256, 128, 2)):
        assert B.mc2_mm_reduce_scatter_workspace_bytes(bad) == 0
        assert B.mc2_mm_reduce_scatter_i8(bad, None, None, None, None, None, None, None,
                                          stream=0, check=False) == B.MC2_ERR_INVALID_ARG
    fake = 1 << 40
    assert B.mc2_mm_reduce_scatter_i8(ok, fake, fake, fake, fake, fake, fake + 16, None,
                                      stream=0, check=False) == B.MC2_ERR_INVALID_ARG
    assert B.mc2_mm_reduce_scatter_i8(ok, None, fake, fake, fake, fake, fake, None,
                                      stream=0, check=False) == B.MC2_ERR_INVALID_ARG


def test_prepack_is_a_noop_for_float_paths_and_checks_int8_args():
    fake = 1 << 40
    assert B.mc2_prepack_weights(_shape(), None, None, None, stream=0, check=False) == B.MC2_OK
    s8 = _shape(act="i8")
    assert B.mc2_prepack_weights(s8, fake, None, fake, stream=0, check=False) == B.MC2_ERR_INVALID_ARG
    assert B.mc2_check_shape(_shape(act="i8", H=4160)) == B.MC2_ERR_INVALID_ARG   # K > 4096
    # int8 dequant mode needs every scale; the raw int32 test mode takes none for h
    assert B.mc2_alltoallv_gmm(s8, fake, None, fake, fake, fake, fake, fake, fake, fake,
                               stream=0, check=False) == B.MC2_ERR_INVALID_ARG
    s8raw = _shape(act="i8", out="i32")
    assert B.mc2_alltoallv_gmm(s8raw, fake, None, fake, None, fake, fake, fake, fake, fake,
                               stream=0, check=False) == B.MC2_ERR_INVALID_ARG


def test_status_strings():
    for st in range(6):
        assert B.status_str(st)
    assert B.status_str(99) == "unknown status"
    assert B.status_str(B.MC2_OK) == "ok"


def test_gemm_events_hook_rejects_events_that_do_not_exist_yet():
    """torch creates a CUDA event at its first record; before that the
    binding refuses it instead of passing a NULL handle.  None clears."""
    import torch
    with pytest.raises(ValueError):
        B.mc2_set_gemm_events(torch.cuda.Event(enable_timing=True), None)
    B.mc2_set_gemm_events(None, None)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        B.lib()
