"""The allocation-free counts entry point (mc2_moe_counts_static).

Some callers cannot allocate device memory themselves -- a plugin whose host
application owns every device allocation, or a service with a device-memory
budget fixed at start-up -- so they cannot provide the workspace that
mc2_moe_counts takes.  mc2_moe_counts_static uses a fixed scratch array
inside the library instead.  These tests call it through the C ABI and
compare it with mc2_moe_counts on two calls in a row (different inputs, so
the second call also shows that the first call's leftover scratch does not
leak into the result).  The file is named to be collected last.
"""
import pytest
import torch

from moe_expert_dispatch_histc_gb300 import binding as B
from moe_expert_dispatch_histc_gb300 import block as blk
from moe_expert_dispatch_histc_gb300.build import build
from moe_expert_dispatch_histc_gb300.workloads import WORKLOADS, make_routing


def _outs(wl):
    i32 = dict(dtype=torch.int32, device="cuda")
    return [torch.full((wl.W, wl.E), -7, **i32), torch.full((wl.W, wl.E), -7, **i32),
            torch.full((wl.E + 1,), -7, **i32), torch.full((wl.R,), -7, **i32),
            torch.full((wl.R,), -7, **i32), torch.zeros(1, **i32)]


@pytest.mark.gpu
def test_counts_static_matches_workspace_counts_twice():
    build()
    for name, seed in (("skew", 0), ("uniform", 3)):
        wl = WORKLOADS[name]
        sel, _ = make_routing(wl, seed)
        d_sel = torch.from_numpy(sel).cuda()
        shape = blk.shape_of(wl)
        ws = torch.empty(B.mc2_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
        ref = _outs(wl)
        B.mc2_moe_counts(shape, d_sel, *ref[:5], ws, ref[5])
        got = _outs(wl)
        B.mc2_moe_counts_static(shape, d_sel, *got)
        torch.cuda.synchronize()
        for a, b in zip(ref, got):
            assert torch.equal(a, b), f"{name}: static-scratch counts differ from mc2_moe_counts"


@pytest.mark.gpu
def test_counts_static_rejects_shapes_beyond_its_scratch():
    """A shape whose tables exceed the fixed scratch returns
    MC2_ERR_UNSUPPORTED and launches nothing.  Every buffer passed is a real
    device buffer of the size the shape asks for, so even a broken size check
    would launch on valid memory."""
    build()
    # (E + 1) * W * ceil(T*k/W/256) = 1025 * 8 * 64 > 131072
    T, E, k, W = 131072, 1024, 1, 8
    big = B.Shape.make(T, 64, 64, E, k, W, "bf16")
    i32 = dict(dtype=torch.int32, device="cuda")
    sel = torch.zeros((T, k), **i32)
    cnt, recv = torch.full((W, E), -7, **i32), torch.full((W, E), -7, **i32)
    offsets = torch.full((E + 1,), -7, **i32)
    src, dst = torch.full((T * k,), -7, **i32), torch.full((T * k,), -7, **i32)
    st = torch.zeros(1, **i32)
    assert B.mc2_moe_counts_static(big, sel, cnt, recv, offsets, src, dst, st,
                                   check=False) == B.MC2_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert int(cnt.min()) == -7 and int(cnt.max()) == -7, "a rejected call wrote its outputs"
    assert int(st.item()) == 0
