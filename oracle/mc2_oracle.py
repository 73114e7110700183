"""CPU oracle for the MC2 MoE expert block -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this module.  The CUDA library never calls it
and shares no code with it; the two meet only through the seeded inputs of
``moe_expert_dispatch_histc_gb300.workloads``.

It is written to be slow and obviously correct: float64 throughout (int64 for
the int8 path), numpy matmul as the only library step, no blocking or fusion.
Integer products go through a float64 matmul whose every partial sum is
checked to stay below 2**53, so they are exact (``exact_int_matmul``).

Sources (page title, then section):

[EP]  "NPU Training Operators - MC2" (shaojiemike.top), section "Execution
      path" (执行路径): the data flow of ep_mc2_forward, which this file
      enumerates in the page's order as
        1 flatten the token rows to [T, H];
        2 count each rank's (token, slot) pairs per expert with histc over E
          bins on [0, E];
        3 gather every rank's counts (all_gather over the EP group);
        4 a rank sends its own counts;
        5 it receives, from every source rank, the counts of its local
          experts' column range;
        6 permute the token rows by expert;
        7 dispatch exchange fused with the fc1 grouped matmul;
        8 SwiGLU;
        9 fc2 grouped matmul fused with the combine exchange;
       10 unpermute, weighting each row by its routing probability.
[BG]  same page, "Background constraints" (背景约束): dispatch = AllToAllv then
      GroupedMatmul; combine = GroupedMatmul then AllToAllv.
[MIG] same page, "Migration checks" (迁移检查): num_experts % ep_size == 0; a
      rank's experts start at ep_rank * num_local_experts; selected_experts in
      [0, num_experts); fc1_weight = gate_up_proj, fc2_weight = down_proj.
[RSQ] "torch_npu.npu_mm_reduce_scatter_base" (Ascend op-plugin docs),
      "Function description" (功能说明): quantised output
      (x1_scale * x2_scale) * (x1 @ x2 + bias); "Parameters" (参数说明):
      x1_scale (m, 1) fp32 per token, x2_scale (1, n) fp32 per channel,
      output bf16 by default, non-zero bias unsupported; the op itself is
      output = reducescatter(...) over world_size ranks with reduce_op 'sum',
      and m must be divisible by world_size.

Readings where the pages are silent (each also listed in the design notes):
  * ids outside [0, E) are invalid [MIG]; they are left out of every count
    and every matmul and contribute nothing to the combine.  (torch.histc
    itself would put the value E into the last bin; ``histc`` below keeps
    that library behaviour and the block filters ids first.)
  * logical rank r owns tokens [r*T/W, (r+1)*T/W).
  * permute sorts the flattened (token, slot) pairs by expert, stably, so
    equal experts keep (token asc, slot asc) order; ``sorted_indices[p]`` is
    the flat index t*k+j of permuted row p.  ``unpermute_dst`` is its inverse.
  * gate = fc1 columns [0, I), up = columns [I, 2I); h = silu(gate) * up,
    silu(g) = g / (1 + exp(-g)).
  * h is materialised in the activation dtype (bf16 rounding, or fp32 for the
    fp32 workload); the fc2 result stays unrounded until the combine, whose
    output is the only other rounding (done by the caller of the oracle).
  * int8: between fc1 and fc2 the SwiGLU output is re-quantised per row,
    symmetric: hs = max|h| / 127 (1 when the row is all zero),
    hq = round-half-even(h / hs) clamped to [-127, 127].  That decision is
    taken in float32, the precision of the CUDA path.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "histc", "round_to_bf16", "round_to_f32", "silu", "swiglu",
    "rank_counts", "send_recv_counts", "permute", "unpermute",
    "expert_offsets", "grouped_matmul", "block_forward", "ep_mc2_forward_emulated",
    "brute_force_token", "quant_block_forward", "requant_rows", "mm_reduce_scatter",
    "exact_int_matmul",
    "silu_grad", "block_backward", "ORACLE_UNPINNED",
]

# Functions with no pin independent of this file (see tests/test_oracle_pins.py).
ORACLE_UNPINNED = ()


# ---------------------------------------------------------------------------
# Rounding helpers (the block materialises h in the activation dtype)
# ---------------------------------------------------------------------------
def round_to_bf16(v: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (8 significant bits),
    ties to even, returned as float64.  Normal range only (|v| >= 2**-126),
    plus exact zero -- far wider than any value this block produces."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)                       # v = m * 2**e, 0.5 <= |m| < 1
    q = np.rint(m * 256.0) / 256.0           # 8 significant bits, half-even
    return np.ldexp(q, e)


def round_to_f32(v: np.ndarray) -> np.ndarray:
    return np.asarray(v, dtype=np.float64).astype(np.float32).astype(np.float64)


_ROUND = {"bf16": round_to_bf16, "f32": round_to_f32, None: lambda v: v}


# ---------------------------------------------------------------------------
# Step 2 [EP]: torch.histc semantics
# ---------------------------------------------------------------------------
def histc(values: np.ndarray, bins: int, vmin: float, vmax: float) -> np.ndarray:
    """Histogram with torch.histc semantics: ``bins`` equal-width bins over
    [vmin, vmax]; values outside are ignored; a value equal to vmax falls in
    the last bin.  Returned as int64 counts."""
    v = np.asarray(values, dtype=np.float64).reshape(-1)
    inside = (v >= vmin) & (v <= vmax)
    width = (vmax - vmin) / bins
    b = np.floor((v[inside] - vmin) / width).astype(np.int64)
    b = np.minimum(b, bins - 1)
    return np.array([np.count_nonzero(b == i) for i in range(bins)], dtype=np.int64)


def _valid(sel: np.ndarray, E: int) -> np.ndarray:
    return (sel >= 0) & (sel < E)


def rank_counts(sel: np.ndarray, E: int, W: int) -> np.ndarray:
    """Steps 2-3 [EP] for all W logical ranks: row r is rank r's histc of its
    own tokens' selected experts; stacking the rows is the all_gather result
    num_global [W, E] (row = source rank).  Invalid ids are dropped first [MIG]."""
    T, k = sel.shape
    assert T % W == 0 and E % W == 0
    Tl = T // W
    rows = []
    for r in range(W):
        s = sel[r * Tl:(r + 1) * Tl].reshape(-1)
        s = s[_valid(s, E)]
        rows.append(histc(s, bins=E, vmin=0, vmax=E))
    return np.stack(rows)


def send_recv_counts(num_global: np.ndarray, W: int):
    """Steps 4-5 [EP]: send_counts of rank r is its own histogram [E];
    recv_counts of rank r is num_global[:, r*E_l:(r+1)*E_l].reshape(-1),
    i.e. source-rank-major [W * E_l]."""
    E = num_global.shape[1]
    El = E // W
    send = [num_global[r].copy() for r in range(W)]
    recv = [num_global[:, r * El:(r + 1) * El].reshape(-1).copy() for r in range(W)]
    return send, recv


# ---------------------------------------------------------------------------
# Steps 6 and 10 [EP]: permute / unpermute
# ---------------------------------------------------------------------------
def permute(hidden: np.ndarray, sel: np.ndarray, E: int | None = None):
    """Permute: stable sort of the flattened (token, slot) pairs by expert.
    Returns (permuted rows, sorted_indices) with permuted[p] = hidden[
    sorted_indices[p] // k].  Ids outside [0, E) sort after every valid one."""
    T, k = sel.shape
    flat = sel.reshape(-1).astype(np.int64)
    ok = flat >= 0 if E is None else _valid(flat, E)
    key = np.where(ok, flat, np.iinfo(np.int64).max)
    sorted_indices = np.argsort(key, kind="stable")
    return hidden[sorted_indices // k], sorted_indices


def unpermute(permuted_out: np.ndarray, sorted_indices: np.ndarray,
              probs: np.ndarray, valid_rows: int | None = None) -> np.ndarray:
    """Unpermute with probs: put each permuted row back at its flat (token,
    slot) index, scale by routing_weights[t, j] and sum the k slots of each
    token, slots in ascending order.  Rows p >= valid_rows (invalid ids) add
    nothing."""
    T, k = probs.shape
    R = sorted_indices.shape[0]
    n = R if valid_rows is None else valid_rows
    Hd = permuted_out.shape[1]
    back = np.zeros((R, Hd), dtype=np.float64)
    back[sorted_indices[:n]] = permuted_out[:n]
    back = back.reshape(T, k, Hd)
    out = np.zeros((T, Hd), dtype=np.float64)
    for j in range(k):
        out += probs[:, j:j + 1].astype(np.float64) * back[:, j, :]
    return out


def expert_offsets(num_global: np.ndarray) -> np.ndarray:
    """Start row of each expert in the expert-major permuted buffer:
    exclusive prefix sum of the per-expert totals over all ranks, [E + 1]."""
    tot = num_global.sum(axis=0)
    return np.concatenate([[0], np.cumsum(tot)]).astype(np.int64)


# ---------------------------------------------------------------------------
# Steps 7-9 [EP]: grouped matmul and SwiGLU
# ---------------------------------------------------------------------------
def silu(g: np.ndarray) -> np.ndarray:
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):         # exp(-g) = inf for g << 0 gives -0.0
        return g / (1.0 + np.exp(-g))


def swiglu(gu: np.ndarray) -> np.ndarray:
    """SwiGLU of a gate|up row block [n, 2I] -> [n, I] (gate_up_proj [MIG])."""
    I = gu.shape[1] // 2
    return silu(gu[:, :I]) * gu[:, I:]


def grouped_matmul(rows: np.ndarray, weights: np.ndarray, group_sizes) -> np.ndarray:
    """npu_grouped_matmul semantics: consecutive row groups, group g of size
    group_sizes[g] multiplied by weights[g]."""
    outs, start = [], 0
    for g, n in enumerate(group_sizes):
        n = int(n)
        outs.append(rows[start:start + n] @ weights[g])
        start += n
    assert start == rows.shape[0]
    if not outs:
        return np.zeros((0, weights.shape[2]))
    return np.concatenate(outs, axis=0)


# ---------------------------------------------------------------------------
# The block in the single-device, expert-major layout (what the GPU computes)
# ---------------------------------------------------------------------------
def block_forward(x, w1, w2, sel, probs, E, W, h_dtype=None):
    """Whole block, steps 1-10 [EP], with the W logical ranks' exchanges
    folded into one expert-major buffer.  x [T, H], w1 [E, H, 2I],
    w2 [E, I, H], sel [T, k], probs [T, k]; float64 in, float64 out.

    Returns a dict: cnt [W, E], send (list), recv (list), offsets [E + 1],
    permute_src [R] (= sorted_indices), unpermute_dst [R], h [R_valid, I]
    (rounded to h_dtype), out [T, H] (unrounded)."""
    T, k = sel.shape
    x = np.asarray(x, dtype=np.float64).reshape(T, -1)          # step 1
    num_global = rank_counts(sel, E, W)                          # steps 2-3
    send, recv = send_recv_counts(num_global, W)                 # steps 4-5
    offsets = expert_offsets(num_global)
    permuted, sorted_indices = permute(x, sel, E)                # step 6
    nvalid = int(offsets[-1])
    tot = num_global.sum(axis=0)
    g = grouped_matmul(permuted[:nvalid], w1, tot)               # step 7
    h = _ROUND[h_dtype](swiglu(g))                               # step 8
    y = grouped_matmul(h, w2, tot)                               # step 9
    out = unpermute(y, sorted_indices, probs, valid_rows=nvalid)  # step 10
    unpermute_dst = np.empty_like(sorted_indices)
    unpermute_dst[sorted_indices] = np.arange(sorted_indices.shape[0])
    return dict(cnt=num_global, send=send, recv=recv, offsets=offsets,
                permute_src=sorted_indices, unpermute_dst=unpermute_dst,
                h=h, y=y, out=out)


# ---------------------------------------------------------------------------
# The block as the pages run it: W ranks, explicit AllToAllv by the counts
# ---------------------------------------------------------------------------
def ep_mc2_forward_emulated(x, w1, w2, sel, probs, E, W, h_dtype=None):
    """Steps 1-10 [EP] rank by rank.  Each logical rank permutes its own
    tokens; the dispatch AllToAllv [BG] moves, from every source rank s to
    every destination rank d, the contiguous chunk of s's permuted rows whose
    experts lie in d's range [d*E_l, (d+1)*E_l) [MIG], sized by send_counts;
    rank d splits what it received by recv_counts (source-major) and runs
    each row through its expert's fc1, SwiGLU and fc2; the combine AllToAllv
    returns every chunk to its source, which unpermutes with its probs.
    Returns out [T, H] (float64, unrounded)."""
    T, k = sel.shape
    H = x.shape[1]
    Tl, El = T // W, E // W
    x = np.asarray(x, dtype=np.float64)
    num_global = rank_counts(sel, E, W)
    send, recv = send_recv_counts(num_global, W)
    # each source rank permutes its own tokens (step 6)
    perm_rows, perm_idx, chunks = [], [], []
    for s in range(W):
        sel_s = sel[s * Tl:(s + 1) * Tl]
        rows, idx = permute(x[s * Tl:(s + 1) * Tl], sel_s, E)
        perm_rows.append(rows)
        perm_idx.append(idx)
        # split s's permuted rows into per-destination chunks by send_counts
        sizes = [int(send[s][d * El:(d + 1) * El].sum()) for d in range(W)]
        starts = np.concatenate([[0], np.cumsum(sizes)])
        chunks.append([rows[starts[d]:starts[d + 1]] for d in range(W)])
    # dispatch AllToAllv: rank d receives chunk (s -> d) for s = 0..W-1
    returned = [[None] * W for _ in range(W)]
    for d in range(W):
        recv_buf = np.concatenate([chunks[s][d] for s in range(W)], axis=0)
        counts = recv[d].reshape(W, El)            # [source, local expert]
        assert recv_buf.shape[0] == int(counts.sum())
        y_buf = np.empty((recv_buf.shape[0], H))
        pos = 0
        for s in range(W):
            for le in range(El):
                n = int(counts[s, le])
                e = d * El + le
                g = recv_buf[pos:pos + n] @ w1[e]                     # step 7
                h = _ROUND[h_dtype](swiglu(g))                        # step 8
                y_buf[pos:pos + n] = h @ w2[e]                        # step 9
                pos += n
        # combine AllToAllv: chunk for source s goes back to s
        pos = 0
        for s in range(W):
            n = int(counts[s].sum())
            returned[s][d] = y_buf[pos:pos + n]
            pos += n
    out = np.zeros((T, H))
    for s in range(W):
        back = np.concatenate(returned[s], axis=0)
        nvalid = int(send[s].sum())
        out[s * Tl:(s + 1) * Tl] = unpermute(back, perm_idx[s],
                                             probs[s * Tl:(s + 1) * Tl], valid_rows=nvalid)  # step 10
    return out


# ---------------------------------------------------------------------------
# Backward of the block [EP]: the gradient of sum(out * dout) with respect to
# x, w1, w2 and probs, taken step by step back through steps 10 .. 6.
# (The pages name the fused operators AllToAllGroupedMatmul /
# GroupedMatmulAllToAll; their backward is the chain rule of the same flow.)
# ---------------------------------------------------------------------------
def silu_grad(a: np.ndarray) -> np.ndarray:
    """d silu(a) / da = s(a) * (1 + a * (1 - s(a))), s the logistic function."""
    a = np.asarray(a, dtype=np.float64)
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-a))
    return s * (1.0 + a * (1.0 - s))


def block_backward(x, w1, w2, sel, probs, dout, E, W, h_dtype=None):
    """Gradients of L = sum(block_forward(...).out * dout).

    Reading: h enters fc2 as materialised (rounded to h_dtype); its rounding
    passes gradients through unchanged (derivative 1), so dh flows back into
    the SwiGLU at the unrounded pre-activation G.  Ids outside [0, E) take no
    part in the block and get no gradient (their dprobs is 0).

    step 10  out[t] = sum_j probs[t, j] * Y[p(t, j)]
             -> dY[p] = probs[t, j] * dout[t];  dprobs[t, j] = Y[p] . dout[t]
    step 9   Y_e = h_e @ w2[e]   -> dh_e = dY_e @ w2[e]^T;  dw2[e] = h_e^T @ dY_e
    step 8   h = silu(a) * b     -> da = dh * b * silu'(a);  db = dh * silu(a)
    step 7   G_e = Xp_e @ w1[e]  -> dXp_e = dG_e @ w1[e]^T;  dw1[e] = Xp_e^T @ dG_e
    step 6   Xp[p] = x[t(p)]     -> dx[t] = sum over valid slots of dXp[p(t, j)]

    Returns a dict with dx [T, H], dw1 [E, H, 2I], dw2 [E, I, H], dprobs [T, k]
    and the intermediates (g, h, y, dy, dh, dg, dxp) in permuted-row order."""
    T, k = sel.shape
    x = np.asarray(x, dtype=np.float64).reshape(T, -1)
    H = x.shape[1]
    I = w2.shape[1]
    num_global = rank_counts(sel, E, W)
    offsets = expert_offsets(num_global)
    permuted, src = permute(x, sel, E)
    nvalid = int(offsets[-1])
    tot = num_global.sum(axis=0)
    xp = permuted[:nvalid]
    g = grouped_matmul(xp, w1, tot)
    h = _ROUND[h_dtype](swiglu(g))
    y = grouped_matmul(h, w2, tot)
    tok, slot = src[:nvalid] // k, src[:nvalid] % k
    dout = np.asarray(dout, dtype=np.float64)
    p_rows = probs.astype(np.float64)[tok, slot]
    dy = p_rows[:, None] * dout[tok]                                    # step 10
    dprobs = np.zeros((T, k))
    dprobs[tok, slot] = np.einsum("ph,ph->p", y, dout[tok])
    dh = np.zeros((nvalid, I))
    dw2 = np.zeros((E, I, H))
    dg = np.zeros((nvalid, 2 * I))
    dxp = np.zeros((nvalid, H))
    dw1 = np.zeros((E, H, 2 * I))
    for e in range(E):
        a0, a1 = int(offsets[e]), int(offsets[e + 1])
        if a0 == a1:
            continue
        dh[a0:a1] = dy[a0:a1] @ w2[e].T                                 # step 9
        dw2[e] = h[a0:a1].T @ dy[a0:a1]
    gate, up = g[:, :I], g[:, I:]
    dg[:, :I] = dh * up * silu_grad(gate)                               # step 8
    dg[:, I:] = dh * silu(gate)
    for e in range(E):
        a0, a1 = int(offsets[e]), int(offsets[e + 1])
        if a0 == a1:
            continue
        dxp[a0:a1] = dg[a0:a1] @ w1[e].T                                # step 7
        dw1[e] = xp[a0:a1].T @ dg[a0:a1]
    dx = np.zeros((T, H))
    for j in range(k):                                                  # step 6
        m = slot == j
        np.add.at(dx, tok[m], dxp[m])
    return dict(dx=dx, dw1=dw1, dw2=dw2, dprobs=dprobs, g=g, h=h, y=y, dy=dy, dh=dh,
                dg=dg, dxp=dxp, offsets=offsets, permute_src=src)


def brute_force_token(x_t, w1, w2, sel_t, probs_t, E, h_dtype=None):
    """out[t] = sum_j probs[t, j] * swiglu(x[t] @ w1[e_j]) @ w2[e_j], with no
    counts and no permutation (the meaning of the block, one token)."""
    acc = np.zeros(w2.shape[2])
    for j in range(len(sel_t)):
        e = int(sel_t[j])
        if not (0 <= e < E):
            continue
        g = np.asarray(x_t, dtype=np.float64)[None, :] @ w1[e]
        h = _ROUND[h_dtype](swiglu(g))
        acc += float(probs_t[j]) * (h @ w2[e])[0]
    return acc


# ---------------------------------------------------------------------------
# int8 path [RSQ]: (x1_scale * x2_scale) * (x1 @ x2), no bias
# ---------------------------------------------------------------------------
def exact_int_matmul(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Integer matrix product a @ b, exact, returned as int64.

    Computed as a float64 library matmul: every product and every partial
    sum is an integer of magnitude at most K * max|a| * max|b|, and below
    2**53 each of them is a float64 exactly, so the result does not depend
    on the library's summation order.  The bound is checked first."""
    a = np.asarray(a)
    b = np.asarray(b)
    K = a.shape[-1]
    ma = int(np.abs(a.astype(np.int64)).max(initial=0))
    mb = int(np.abs(b.astype(np.int64)).max(initial=0))
    assert K * ma * mb < 2 ** 53, "integer product too large for an exact float64 sum"
    return (a.astype(np.float64) @ b.astype(np.float64)).astype(np.int64)


def requant_rows(h: np.ndarray):
    """Symmetric per-row int8 re-quantisation of h, decided in float32:
    hs = fp32(max|h|) / 127 (1 when the row is all zero);
    hq = round-half-even(fp32(h) / hs) clamped to [-127, 127]."""
    h32 = np.asarray(h, dtype=np.float64).astype(np.float32)
    amax = np.abs(h32).max(axis=1) if h32.shape[1] else np.zeros(h32.shape[0], np.float32)
    hs = np.where(amax > 0, amax / np.float32(127.0), np.float32(1.0)).astype(np.float32)
    q = np.rint((h32 / hs[:, None]).astype(np.float32))
    hq = np.clip(q, -127, 127).astype(np.int8)
    return hq, hs


def quant_block_forward(xq, xs, w1q, w1s, w2q, w2s, sel, probs, E, W, hq_override=None):
    """int8 block.  fc1: acc1 = xq @ w1q (exact, int64); G = (xs[t] * w1s[e])
    * acc1 per [RSQ]; h = SwiGLU(G); (hq, hs) = requant_rows(h);
    fc2: acc2 = hq @ w2q (exact, int64); Y = (hs[p] * w2s[e]) * acc2;
    out = unpermute(Y, probs).  When ``hq_override=(hq, hs)`` is given, fc2
    consumes it instead (used to check fc2 exactly on another producer's hq).
    Returns a dict with the int64 accumulators and the float64 results."""
    T, k = sel.shape
    num_global = rank_counts(sel, E, W)
    offsets = expert_offsets(num_global)
    tok, sorted_indices = permute(np.arange(T), sel, E)        # token of each row
    nvalid = int(offsets[-1])
    I = w2q.shape[1]
    H = w2q.shape[2]
    acc1 = np.zeros((nvalid, 2 * I), dtype=np.int64)
    g = np.zeros((nvalid, 2 * I))
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a == b:
            continue
        acc1[a:b] = exact_int_matmul(xq[tok[a:b]], w1q[e])
        scale = xs[tok[a:b]].astype(np.float64)[:, None] * w1s[e].astype(np.float64)[None, :]
        g[a:b] = scale * acc1[a:b]
    h = swiglu(g)
    hq, hs = requant_rows(h) if hq_override is None else hq_override
    acc2 = np.zeros((nvalid, H), dtype=np.int64)
    y = np.zeros((nvalid, H))
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a == b:
            continue
        acc2[a:b] = exact_int_matmul(hq[a:b], w2q[e])
        y[a:b] = (hs[a:b].astype(np.float64)[:, None] * w2s[e].astype(np.float64)[None, :]) * acc2[a:b]
    out = unpermute(y, sorted_indices, probs, valid_rows=nvalid)
    return dict(cnt=num_global, offsets=offsets, permute_src=sorted_indices,
                acc1=acc1, h=h, hq=hq, hs=hs, acc2=acc2, y=y, out=out)


def mm_reduce_scatter(x1q, x1s, x2q, x2s):
    """Quantised matmul + reduce-scatter over W ranks [RSQ].
    x1q [W, m, k] int8, x1s [W, m], x2q [W, k, n] int8, x2s [W, n].
    Each rank's partial is (x1_scale * x2_scale) * (x1 @ x2) with the product
    exact in int64; the reduce is the sum over ranks (float64 here); rank r
    receives rows [r*m/W, (r+1)*m/W) of the sum.
    Returns (acc [W, m, n] int64, total [m, n] float64, per_rank [W, m/W, n])."""
    W, m, _ = x1q.shape
    n = x2q.shape[2]
    assert m % W == 0
    acc = np.zeros((W, m, n), dtype=np.int64)
    total = np.zeros((m, n))
    for r in range(W):
        acc[r] = exact_int_matmul(x1q[r], x2q[r])
        scale = x1s[r].astype(np.float64)[:, None] * x2s[r].astype(np.float64)[None, :]
        total += scale * acc[r]
    per_rank = total.reshape(W, m // W, n)
    return acc, total, per_rank


def bf16_tolerance_ok(got: np.ndarray, ref: np.ndarray, max_rel=1e-2, mean_rel=2e-3):
    """The block's floating-point acceptance rule: max|err| <= 1e-2 * max|ref|
    and sum|err| / sum|ref| <= 2e-3.  Returns (ok, max_err_ratio, mean_rel_err)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    mref = float(np.abs(ref).max()) if ref.size else 0.0
    sref = float(np.abs(ref).sum()) if ref.size else 0.0
    a = float(err.max()) / mref if mref > 0 else float(err.max() if err.size else 0.0)
    b = float(err.sum()) / sref if sref > 0 else float(err.sum() if err.size else 0.0)
    return (a <= max_rel and b <= mean_rel), a, b

