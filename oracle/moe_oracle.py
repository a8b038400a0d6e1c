"""CPU oracle for the routed Mixture-of-Experts expert-MLP layer, forward and backward.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, fp64 statement of
what the layer computes.  It exists so that the CUDA library can be checked
against it.  Only the test suite, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import it; the library itself
never does, and this module imports nothing from the library.

Source: "LigerCute -- native CUTLASS + NVSHMEM kernels" (the liger-cute-kernels
0.8.3 package README):

* Overview: buffers are sized from the total routed-token capacity, not a
  per-expert capacity, which keeps execution valid under CUDA Graphs.
* LigerMoE design, Forward pass: routed tokens are sorted (by expert) before
  the main loop, the MMA warps run the expert MLP, and a final local combine
  applies the router weights after every expert result has arrived.
* LigerMoE design, Backward pass: routed expert-output gradients first, then
  activation recomputation, input gradients and expert-weight gradients
  (accumulated across token-tile batches), and a final local dispatch that
  reduces the routed dX back to the original tokens.

The pages name no activation; the expert MLP here is SwiGLU:
``f_e(x) = (silu(x W_gate[e]) * (x W_up[e])) W_down[e]`` with
``silu(z) = z / (1 + exp(-z))``.  Layouts: ``w_gate, w_up`` [E, D, I],
``w_down`` [E, I, D], ``x`` [T, D], ``topk_ids``/``topk_w`` [T, K].

Every floating-point result is computed in fp64 from inputs widened exactly
(bf16 values are exact in fp64); nothing is rounded in between.  Integer
outputs (counts, offsets, permutation) are exact.

Parity pins (tests/test_oracle_*.py): the permutation against a brute-force
scan and its invariants; the forward against a dense masked per-token loop, the
K=1 plain-MLP case, linearity in the router weights and a hand-derived scalar
case; the backward against fp64 central finite differences, the
<dW, W> = sum w <dY, f_e(x)> identity for the two weights the output is linear
in, and exact zeros for empty experts.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "capacity", "route_permute", "expert_mlp_fwd", "combine", "expert_mlp_bwd",
    "moe_forward", "moe_backward", "silu", "sigmoid",
]


def sigmoid(z):
    """Logistic function 1 / (1 + exp(-z)) in fp64."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    """SiLU(z) = z * sigmoid(z)."""
    z = np.asarray(z, dtype=np.float64)
    return z * sigmoid(z)


def silu_grad(z):
    """d/dz silu(z) = sigmoid(z) * (1 + z * (1 - sigmoid(z)))."""
    s = sigmoid(z)
    return s * (1.0 + z * (1.0 - s))


def capacity(T: int, K: int, E: int, align: int) -> int:
    """Rows of every expert-sorted buffer: the total routed-token count plus the
    worst-case padding of each expert to ``align`` rows, rounded up to ``align``
    (Overview: sized from the total routed-token capacity)."""
    R = T * K
    c = R + E * (align - 1)
    return ((c + align - 1) // align) * align


def route_permute(topk_ids, topk_w, x, E: int, align: int):
    """Sort the T*K routed slots by expert into one padded, expert-contiguous order.

    (LigerMoE design, Forward pass: routed tokens are sorted before the main
    loop.)  A slot is the flat index j = t*K + k.  Counting sort with key
    (expert, j): within an expert, slots keep ascending j.  Each expert's
    segment starts at ``offsets[e]`` and is padded to a multiple of ``align``.

    Returns a dict:
      counts   [E]      int64  slots routed to each expert
      offsets  [E+1]    int64  offsets[0]=0, offsets[e+1]=offsets[e]+ceil(counts[e]/align)*align
      perm_src [cap]    int64  flat slot j placed at sorted row s, -1 on padding rows
      inv_perm [T*K]    int64  sorted row s of flat slot j (inv_perm[perm_src[s]] == s)
      w_perm   [cap]    f64    router weight of the slot at row s, 0 on padding
      x_perm   [cap, D] f64    x[t] of the slot at row s, 0 on padding (rows < offsets[E])
    Rows at and beyond offsets[E] hold perm_src=-1, w_perm=0, x_perm=0.
    """
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, K = ids.shape
    R = T * K
    flat = ids.reshape(-1)
    if R and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    w = np.asarray(topk_w, dtype=np.float64).reshape(-1)
    cap = capacity(T, K, E, align)

    counts = np.zeros(E, dtype=np.int64)
    for j in range(R):
        counts[flat[j]] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + (counts[e] + align - 1) // align * align

    perm_src = np.full(cap, -1, dtype=np.int64)
    inv_perm = np.empty(R, dtype=np.int64)
    next_row = offsets[:-1].copy()
    for j in range(R):  # ascending j, so the order inside an expert is stable
        e = flat[j]
        s = next_row[e]
        next_row[e] += 1
        perm_src[s] = j
        inv_perm[j] = s

    w_perm = np.zeros(cap, dtype=np.float64)
    real = perm_src >= 0
    w_perm[real] = w[perm_src[real]]

    x_perm = None
    if x is not None:
        x = np.asarray(x, dtype=np.float64)
        x_perm = np.zeros((cap, x.shape[1]), dtype=np.float64)
        x_perm[real] = x[perm_src[real] // K]
    return dict(counts=counts, offsets=offsets, perm_src=perm_src, inv_perm=inv_perm,
                w_perm=w_perm, x_perm=x_perm)


def _expert_rows(offsets, e):
    return slice(int(offsets[e]), int(offsets[e + 1]))


def expert_mlp_fwd(x_perm, w_gate, w_up, w_down, offsets, experts=None):
    """Per-expert SwiGLU MLP over the expert-sorted rows (LigerMoE design,
    Forward pass: the MMA warps execute the expert MLP).

    For the rows s of expert e: G = x_perm[s] W_gate[e], U = x_perm[s] W_up[e],
    A = silu(G) * U, y_perm[s] = A W_down[e].  Padding rows are zero in, zero out.
    ``experts`` restricts the work to a subset; rows of other experts are NaN.
    The weights may be indexable per expert (e.g. a list holding only the experts
    that are computed).
    """
    x_perm = np.asarray(x_perm, dtype=np.float64)
    E = len(offsets) - 1
    D = x_perm.shape[1]
    y = np.full((x_perm.shape[0], D), np.nan if experts is not None else 0.0)
    if experts is None:
        y[int(offsets[E]):] = 0.0
    for e in (range(E) if experts is None else experts):
        rows = _expert_rows(offsets, e)
        xe = x_perm[rows]
        g = xe @ np.asarray(w_gate[e], dtype=np.float64)
        u = xe @ np.asarray(w_up[e], dtype=np.float64)
        a = silu(g) * u
        y[rows] = a @ np.asarray(w_down[e], dtype=np.float64)
    return y


def combine(src_perm, inv_perm, topk_w, T: int, K: int):
    """Reduce the K routed rows of every token back to the token (LigerMoE design:
    the forward's local combine applies the router weights; the backward's local
    dispatch reduces the routed dX with weight one).

    out[t] = sum_k w[t,k] * src_perm[inv_perm[t*K+k]]   (w = 1 when topk_w is None)
    """
    src = np.asarray(src_perm, dtype=np.float64)
    inv = np.asarray(inv_perm, dtype=np.int64)
    out = np.zeros((T, src.shape[1]), dtype=np.float64)
    w = None if topk_w is None else np.asarray(topk_w, dtype=np.float64).reshape(T, K)
    for k in range(K):
        rows = src[inv[np.arange(T) * K + k]]
        out += rows if w is None else w[:, k:k + 1] * rows
    return out


def expert_mlp_bwd(dy, x_perm, perm_src, w_perm, offsets, w_gate, w_up, w_down, K: int,
                   experts=None):
    """Backward of the routed expert MLP on the expert-sorted rows (LigerMoE
    design, Backward pass).

    Per row s of expert e, with t = perm_src[s] // K:
      dy_s  = w_perm[s] * dy[t]             routed expert-output gradient
      G, U  = x_s W_gate[e], x_s W_up[e]    activation recomputation
      A     = silu(G) * U
      dA    = dy_s W_down[e]^T
      dG    = dA * U * silu'(G),  dU = dA * silu(G)
      dx_perm[s] = dG W_gate[e]^T + dU W_up[e]^T     input gradient
      dW_down[e] = sum_s A^T dy_s,  dW_gate[e] = sum_s x_s^T dG,  dW_up[e] = sum_s x_s^T dU
    Padding rows carry zero gradient.  Experts with no rows get dW == 0.
    ``experts`` restricts the work: dx_perm rows of other experts are NaN and the
    three weight gradients come back as dicts {e: array} over the listed experts.
    """
    dy = np.asarray(dy, dtype=np.float64)
    x_perm = np.asarray(x_perm, dtype=np.float64)
    perm_src = np.asarray(perm_src, dtype=np.int64)
    w_perm = np.asarray(w_perm, dtype=np.float64)
    E = len(offsets) - 1
    todo = list(range(E) if experts is None else experts)
    D = x_perm.shape[1]
    I = np.asarray(w_gate[todo[0]]).shape[1] if todo else 0
    if experts is None:
        dx_perm = np.zeros(x_perm.shape)
        dw_gate = np.zeros((E, D, I))
        dw_up = np.zeros((E, D, I))
        dw_down = np.zeros((E, I, D))
    else:
        dx_perm = np.full(x_perm.shape, np.nan)
        dw_gate, dw_up, dw_down = {}, {}, {}
    for e in todo:
        rows = _expert_rows(offsets, e)
        src = perm_src[rows]
        real = src >= 0
        dys = np.zeros((src.shape[0], D))
        dys[real] = w_perm[rows][real, None] * dy[src[real] // K]
        xe = x_perm[rows]
        wg = np.asarray(w_gate[e], dtype=np.float64)
        wu = np.asarray(w_up[e], dtype=np.float64)
        wd = np.asarray(w_down[e], dtype=np.float64)
        g = xe @ wg
        u = xe @ wu
        a = silu(g) * u
        da = dys @ wd.T
        dg = da * u * silu_grad(g)
        du = da * silu(g)
        dx_perm[rows] = dg @ wg.T + du @ wu.T
        dw_down[e] = a.T @ dys
        dw_gate[e] = xe.T @ dg
        dw_up[e] = xe.T @ du
    return dx_perm, dw_gate, dw_up, dw_down


def _tokens_of_expert(ids, e):
    """Token indices t and slot indices k with ids[t, k] == e."""
    t, k = np.nonzero(ids == e)
    return t, k


def moe_forward(x, topk_ids, topk_w, w_gate, w_up, w_down):
    """The whole layer by its definition, without any permutation:
    Y[t] = sum_k w[t,k] * f_{ids[t,k]}(x[t])."""
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(topk_ids, dtype=np.int64)
    w = np.asarray(topk_w, dtype=np.float64)
    E = len(w_gate)
    y = np.zeros_like(x)
    for e in range(E):
        t, k = _tokens_of_expert(ids, e)
        if t.size == 0:
            continue
        xe = x[t]
        a = silu(xe @ np.asarray(w_gate[e], np.float64)) * (xe @ np.asarray(w_up[e], np.float64))
        fe = a @ np.asarray(w_down[e], np.float64)
        np.add.at(y, t, w[t, k][:, None] * fe)
    return y


def moe_backward(x, topk_ids, topk_w, w_gate, w_up, w_down, dy, weight_grads=True):
    """Gradients of L = sum(Y * dY) for the whole layer by its definition:
    returns dX [T,D], dW_gate [E,D,I], dW_up [E,D,I], dW_down [E,I,D] (routing fixed).
    With ``weight_grads=False`` only dX is computed (the dW slots are None)."""
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(topk_ids, dtype=np.int64)
    w = np.asarray(topk_w, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    E = len(w_gate)
    D = x.shape[1]
    dx = np.zeros_like(x)
    dwg = dwu = dwd = None
    for e in range(E):
        t, k = _tokens_of_expert(ids, e)
        if t.size == 0:
            continue
        wg = np.asarray(w_gate[e], np.float64)
        wu = np.asarray(w_up[e], np.float64)
        wd = np.asarray(w_down[e], np.float64)
        xe = x[t]
        g = xe @ wg
        u = xe @ wu
        a = silu(g) * u
        dys = w[t, k][:, None] * dy[t]
        da = dys @ wd.T
        dg = da * u * silu_grad(g)
        du = da * silu(g)
        np.add.at(dx, t, dg @ wg.T + du @ wu.T)
        if weight_grads:
            if dwg is None:
                I = wg.shape[1]
                dwg, dwu, dwd = np.zeros((E, D, I)), np.zeros((E, D, I)), np.zeros((E, I, D))
            dwd[e] = a.T @ dys
            dwg[e] = xe.T @ dg
            dwu[e] = xe.T @ du
    if weight_grads and dwg is None:   # no expert received a token
        I = np.asarray(w_gate[0]).shape[1]
        dwg, dwu, dwd = np.zeros((E, D, I)), np.zeros((E, D, I)), np.zeros((E, I, D))
    return dx, dwg, dwu, dwd
