"""Seeded synthetic inputs for the MoE expert block.

This module draws random numbers and nothing else: it holds none of the
block's arithmetic (no counting, permutation, matmul, SwiGLU or combine).
Both the CUDA path's tests/bench and the CPU oracle consume what it returns,
so the two sides always see identical inputs.

The router output (``selected_experts``, ``routing_weights``) is an *input*
to the block: in the ``ep_mc2_forward`` call of "NPU Training Operators -
MC2" (section "Migration checks", the suggested dispatcher call) the experts
function receives ``routing_weights`` and ``selected_experts`` from the
caller.  The router is therefore generated here, as the workloads state it:
logits ~ N(0, 1) (plus a per-expert bias for the skewed workload), softmax,
top-k with ties broken towards the lower expert index, and the k kept
probabilities renormalised to sum to one.

Named workloads (sizes are what the names say):

* ``tiny``     T=64    H=256  I=128  E=8   k=2 W=2  fp32 activations/weights
* ``uniform``  T=4096  H=2048 I=768  E=64  k=8 W=4  bf16, near-uniform load
* ``skew``     T=16384 H=2048 I=768  E=128 k=8 W=8  bf16, Zipf(s=1.2) bias
* ``int8``     T=8192  H=3072 I=1536 E=64  k=4 W=8  int8 + fp32 scales
* ``decode``   T=256   H=4096 I=1536 E=128 k=8 W=8  bf16, weight-bound

Weights: fc1 ``w1`` is [E, H, 2I] (gate columns [0, I), up columns [I, 2I)),
fc2 ``w2`` is [E, I, H]; both are used as ``x @ w``.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "get_workload", "make_routing", "make_inputs",
    "f32_to_bf16_bits", "bf16_bits_to_f32",
]


@dataclass(frozen=True)
class Workload:
    name: str
    T: int          # tokens
    H: int          # hidden size
    I: int          # per-expert intermediate size (fc1 emits 2I: gate | up)
    E: int          # experts
    k: int          # top-k
    W: int          # logical expert-parallel ranks
    act: str        # "f32" | "bf16" | "i8"
    routing: str = "normal"   # "normal" | "zipf"
    init_std: float = 0.02

    @property
    def R(self) -> int:
        """Permuted rows: every (token, slot) pair once."""
        return self.T * self.k

    @property
    def E_local(self) -> int:
        return self.E // self.W

    @property
    def flops(self) -> int:
        """Algorithmic flops of one block: fc1 (2*R*H*2I) + fc2 (2*R*I*H)."""
        return 6 * self.R * self.H * self.I

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 64, 256, 128, 8, 2, 2, "f32"),
    "uniform": Workload("uniform", 4096, 2048, 768, 64, 8, 4, "bf16"),
    "skew": Workload("skew", 16384, 2048, 768, 128, 8, 8, "bf16", routing="zipf"),
    "int8": Workload("int8", 8192, 3072, 1536, 64, 4, 8, "i8"),
    "decode": Workload("decode", 256, 4096, 1536, 128, 8, 8, "bf16"),
}


def get_workload(name: str) -> Workload:
    return WORKLOADS[name]


# --------------------------------------------------------------------------
# bf16 storage.  numpy has no bf16 dtype, so bf16 tensors are carried as
# uint16 bit patterns.  Conversion from fp32 rounds to nearest-even.
# --------------------------------------------------------------------------
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# Router (input to the block)
# --------------------------------------------------------------------------
def _softmax_topk_renorm(logits: np.ndarray, k: int):
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z, dtype=np.float32)
    p = p / p.sum(axis=1, keepdims=True, dtype=np.float32)
    # stable sort of -p: equal probabilities keep the lower expert index first
    order = np.argsort(-p, axis=1, kind="stable")[:, :k]
    top = np.take_along_axis(p, order, axis=1).astype(np.float32)
    top = top / top.sum(axis=1, keepdims=True, dtype=np.float32)
    return order.astype(np.int32), top.astype(np.float32)


def zipf_bias(E: int, s: float = 1.2) -> np.ndarray:
    """2*log of a Zipf(s) weight per expert, expert e <-> rank e+1, unshuffled.
    The Zipf normalising constant cancels in softmax, so it is left out."""
    return (2.0 * (-s) * np.log(np.arange(1, E + 1, dtype=np.float64))).astype(np.float32)


def make_routing(wl: Workload, seed: int):
    rng = np.random.default_rng([seed, 1])
    logits = rng.standard_normal((wl.T, wl.E), dtype=np.float32)
    if wl.routing == "zipf":
        logits = logits + zipf_bias(wl.E)[None, :]
    return _softmax_topk_renorm(logits, wl.k)


def make_inputs(wl: Workload, seed: int = 0) -> dict:
    """All inputs of one block, as numpy arrays.

    Returned keys:
      sel   int32 [T, k]    selected experts
      probs f32   [T, k]    renormalised routing weights
      x     [T, H]          f32 (tiny), uint16 bf16 bits (bf16), int8 (i8)
      w1    [E, H, 2I]      same dtype convention as x
      w2    [E, I, H]       same dtype convention as x
      xs    f32 [T]         per-token scale        (i8 only)
      w1s   f32 [E, 2I]     per-channel fc1 scale  (i8 only)
      w2s   f32 [E, H]      per-channel fc2 scale  (i8 only)
    """
    sel, probs = make_routing(wl, seed)
    out = {"sel": sel, "probs": probs}
    T, H, I, E = wl.T, wl.H, wl.I, wl.E
    if wl.act in ("f32", "bf16"):
        def normal(shape, stream):
            r = np.random.default_rng([seed, stream])
            return r.standard_normal(shape, dtype=np.float32) * np.float32(wl.init_std)
        x, w1, w2 = normal((T, H), 2), normal((E, H, 2 * I), 3), normal((E, I, H), 4)
        if wl.act == "bf16":
            x, w1, w2 = f32_to_bf16_bits(x), f32_to_bf16_bits(w1), f32_to_bf16_bits(w2)
        out.update(x=x, w1=w1, w2=w2)
    elif wl.act == "i8":
        def ints(shape, stream):
            r = np.random.default_rng([seed, stream])
            return r.integers(-127, 128, size=shape, dtype=np.int8)

        def scales(shape, stream):
            r = np.random.default_rng([seed, stream])
            return r.uniform(1e-3, 1e-2, size=shape).astype(np.float32)
        out.update(x=ints((T, H), 2), w1=ints((E, H, 2 * I), 3), w2=ints((E, I, H), 4),
                   xs=scales((T,), 5), w1s=scales((E, 2 * I), 6), w2s=scales((E, H), 7))
    else:
        raise ValueError(f"unknown activation dtype {wl.act!r}")
    return out


def as_f64(a: np.ndarray, act: str) -> np.ndarray:
    """Exact float64 view of an input array stored under the dtype convention above."""
    if act == "bf16" and a.dtype == np.uint16:
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a, dtype=np.float64)
