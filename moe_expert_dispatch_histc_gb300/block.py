"""Device-memory plumbing around the C ABI: move seeded inputs to the GPU,
allocate the outputs and workspace the block writes, and call the library.

Nothing here computes any step of the block; every step runs in libmc2moe.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import binding as B
from .workloads import Workload

_TORCH_ACT = {"f32": torch.float32, "bf16": torch.bfloat16, "i8": torch.int8}


def shape_of(wl: Workload, out: str | None = None) -> B.Shape:
    return B.Shape.make(wl.T, wl.H, wl.I, wl.E, wl.k, wl.W, wl.act, out)


def _act_tensor(a: np.ndarray, act: str, device) -> torch.Tensor:
    if act == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(device)


def inputs_to_device(inp: dict, wl: Workload, device="cuda") -> dict:
    d = {
        "sel": torch.from_numpy(np.ascontiguousarray(inp["sel"])).to(device),
        "probs": torch.from_numpy(np.ascontiguousarray(inp["probs"])).to(device),
        "x": _act_tensor(inp["x"], wl.act, device),
        "w1": _act_tensor(inp["w1"], wl.act, device),
        "w2": _act_tensor(inp["w2"], wl.act, device),
    }
    for k in ("xs", "w1s", "w2s"):
        d[k] = torch.from_numpy(inp[k]).to(device) if k in inp else None
    return d


@dataclass
class BlockBuffers:
    cnt: torch.Tensor
    recv: torch.Tensor
    offsets: torch.Tensor
    permute_src: torch.Tensor
    unpermute_dst: torch.Tensor
    h: torch.Tensor
    h_scale: torch.Tensor | None
    out: torch.Tensor
    ws: torch.Tensor
    dev_status: torch.Tensor


def alloc_buffers(wl: Workload, device="cuda", out: str | None = None) -> BlockBuffers:
    shape = shape_of(wl, out)
    R = wl.R
    i32 = torch.int32
    if wl.act == "i8":
        h = torch.empty((R, 2 * wl.I) if out == "i32" else (R, wl.I),
                        dtype=torch.int32 if out == "i32" else torch.int8, device=device)
        h_scale = None if out == "i32" else torch.empty(R, dtype=torch.float32, device=device)
        o = torch.empty((R, wl.H) if out == "i32" else (wl.T, wl.H),
                        dtype=torch.int32 if out == "i32" else torch.bfloat16, device=device)
    else:
        h = torch.empty((R, wl.I), dtype=_TORCH_ACT[wl.act], device=device)
        h_scale = None
        o = torch.empty((wl.T, wl.H), dtype=_TORCH_ACT[wl.act], device=device)
    ws_bytes = B.mc2_workspace_bytes(shape)
    if ws_bytes == 0:
        raise ValueError(f"shape rejected by the library: {wl}")
    return BlockBuffers(
        cnt=torch.empty((wl.W, wl.E), dtype=i32, device=device),
        recv=torch.empty((wl.W, wl.E), dtype=i32, device=device),
        offsets=torch.empty(wl.E + 1, dtype=i32, device=device),
        permute_src=torch.empty(R, dtype=i32, device=device),
        unpermute_dst=torch.empty(R, dtype=i32, device=device),
        h=h, h_scale=h_scale, out=o,
        ws=torch.empty(ws_bytes, dtype=torch.uint8, device=device),
        dev_status=torch.zeros(1, dtype=i32, device=device),
    )


def prepack(wl: Workload, d: dict, b: BlockBuffers, stream=None, out: str | None = None):
    """Once per weight set: the int8 path's bf16 weight copies in the workspace
    (a no-op for the other activation types)."""
    return B.mc2_prepack_weights(shape_of(wl, out), d["w1"], d["w2"], b.ws, stream=stream)


def run_block(wl: Workload, d: dict, b: BlockBuffers, stream=None, out: str | None = None):
    """One pass of the whole block through the single C entry point."""
    shape = shape_of(wl, out)
    return B.mc2_moe_forward(shape, d["x"], d["xs"], d["sel"], d["probs"], d["w1"], d["w1s"],
                             d["w2"], d["w2s"], b.cnt, b.recv, b.offsets, b.permute_src,
                             b.unpermute_dst, b.h, b.h_scale, b.out, b.ws, b.dev_status,
                             stream=stream)


def run_segments(wl: Workload, d: dict, b: BlockBuffers, stream=None, out: str | None = None):
    """The block as its three C entry points, in order."""
    shape = shape_of(wl, out)
    B.mc2_moe_counts(shape, d["sel"], b.cnt, b.recv, b.offsets, b.permute_src, b.unpermute_dst,
                     b.ws, b.dev_status, stream=stream)
    B.mc2_alltoallv_gmm(shape, d["x"], d["xs"], d["w1"], d["w1s"], b.offsets, b.permute_src,
                        b.ws, b.h, b.h_scale, b.dev_status, stream=stream)
    if out == "i32":
        return
    B.mc2_gmm_alltoallv(shape, b.h, b.h_scale, d["w2"], d["w2s"], b.offsets, b.permute_src,
                        b.unpermute_dst, d["probs"], b.ws, b.out, b.dev_status, stream=stream)


def run_unfused(wl: Workload, d: dict, b: BlockBuffers, xp: torch.Tensor, stream=None):
    """The non-fused baseline: counts, materialised permute into xp [T*k, H],
    plain grouped fc1 + SwiGLU, then fc2 + combine (bf16 only)."""
    shape = shape_of(wl)
    B.mc2_moe_counts(shape, d["sel"], b.cnt, b.recv, b.offsets, b.permute_src, b.unpermute_dst,
                     b.ws, b.dev_status, stream=stream)
    B.mc2_permute_rows(shape, d["x"], b.permute_src, xp, stream=stream)
    B.mc2_gmm_swiglu(shape, xp, d["w1"], b.offsets, b.h, b.dev_status, stream=stream)
    B.mc2_gmm_alltoallv(shape, b.h, None, d["w2"], None, b.offsets, b.permute_src, b.unpermute_dst,
                        d["probs"], b.ws, b.out, b.dev_status, stream=stream)
