"""Helpers shared by the GPU tests: run the CUDA path on seeded inputs and
bring results back; lazily widen stored weights to float64 for the oracle."""
from __future__ import annotations

import numpy as np
import torch

from moe_expert_dispatch_histc_gb300 import block as blk
from moe_expert_dispatch_histc_gb300.build import build
from moe_expert_dispatch_histc_gb300.workloads import as_f64, make_inputs

_built = False


def ensure_built():
    global _built
    if not _built:
        build()
        _built = True


class F64Experts:
    """w[e] -> float64 copy of expert e's weights, converted on every use and
    not kept, so the oracle can walk a weight set whose float64 copy would
    not fit in host memory (the decode workload's w1 is 12.9 GB in float64)."""

    def __init__(self, arr, act):
        self.arr, self.act = arr, act
        self.shape = arr.shape

    def __getitem__(self, e):
        return as_f64(self.arr[int(e)], self.act)


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.numpy()


def run_gpu(wl, seed=0, inputs=None, segments=False, out=None):
    ensure_built()
    inp = make_inputs(wl, seed) if inputs is None else inputs
    d = blk.inputs_to_device(inp, wl)
    b = blk.alloc_buffers(wl, out=out)
    blk.prepack(wl, d, b, out=out)
    if segments:
        blk.run_segments(wl, d, b, out=out)
    else:
        blk.run_block(wl, d, b, out=out)
    torch.cuda.synchronize()
    return inp, d, b


def random_shapes(seed, n, act):
    """n seeded random block shapes within the library's rules: W in {1, 2, 4},
    E a multiple of W up to 16 W, k up to min(E, 8), T a multiple of W up to
    150 W, H and I multiples of 64 (64..512, 64..384) -- ragged tiles in every
    dimension and expert counts that are not powers of two."""
    from moe_expert_dispatch_histc_gb300.workloads import Workload
    rng = np.random.default_rng(seed)
    shapes = []
    for i in range(n):
        W = int(rng.choice([1, 2, 4]))
        E = W * int(rng.integers(1, 17))
        k = int(rng.integers(1, min(E, 8) + 1))
        T = W * int(rng.integers(1, 151))
        H = 64 * int(rng.integers(1, 9))
        I = 64 * int(rng.integers(1, 7))
        shapes.append(Workload(f"rand{i}_T{T}_H{H}_I{I}_E{E}_k{k}_W{W}", T, H, I, E, k, W, act))
    return shapes
