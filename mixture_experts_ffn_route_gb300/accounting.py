"""Algorithmic work of one layer forward: flops and HBM bytes per kernel.

These are the roofline numerators (no padding rows, no re-reads): a weight
matrix of an expert that receives at least one row is read once, activations
are read and written once.  Sizes: T tokens, H hidden, E experts, k top-k,
I intermediate, A = T*k assignments, n_e rows of expert e.
"""
from __future__ import annotations

import numpy as np

BF16 = 2
F32 = 4
I32 = 4
MX8 = 1 + 1 / 32  # an FP8 code plus its share of the E8M0 scale of its group of 32
MX4 = 0.5 + 1 / 32  # an E2M1 code (half a byte) plus its share of the scale


def _counts(counts, has_shared, T):
    c = np.asarray(counts, dtype=np.int64)
    n_active = int((c > 0).sum()) + (1 if has_shared and T > 0 else 0)
    rows = int(c.sum()) + (T if has_shared else 0)
    return rows, n_active


def gemm1_flops(counts, H, I, has_shared=0, T=0):
    rows, _ = _counts(counts, has_shared, T)
    return 2 * rows * H * (2 * I)


def gemm2_flops(counts, H, I, has_shared=0, T=0):
    rows, _ = _counts(counts, has_shared, T)
    return 2 * rows * I * H


def router_flops(T, H, E):
    return 2 * T * H * E


def gemm1_bytes(counts, H, I, has_shared=0, T=0, w_bytes=BF16, x_bytes=BF16, act_bytes=BF16):
    """W1 of every active expert (H x 2I), its input rows (H; gathered from the
    token rows by the permutation) and Act rows (I).  The A8W8 form reads int8
    weights (w_bytes 1), fp16 token codes and writes fp32 Act (act_bytes 4)."""
    rows, n_active = _counts(counts, has_shared, T)
    return n_active * H * 2 * I * w_bytes + rows * H * x_bytes + rows * I * act_bytes


def gemm2_bytes(counts, H, I, has_shared=0, T=0, w_bytes=BF16, act_bytes=BF16, out_bytes=F32):
    """W2 of every active expert (I x H), Act rows in (bf16, or fp16 codes),
    expert output rows out (fp32; bf16 in the bf16 inference forward)."""
    rows, n_active = _counts(counts, has_shared, T)
    return n_active * I * H * w_bytes + rows * I * act_bytes + rows * H * out_bytes


def dispatch_bytes(T, H, k):
    """Expert ids in (twice: count and place); perm and inv out.  The permuted
    token rows are not materialised (Linear1 gathers them)."""
    A = T * k
    return 2 * A * I32 + 2 * A * I32


def dispatch_payload_bytes(T, H, k):
    """The permuted activation block alone, T*k rows of H bf16 values."""
    return T * k * H * BF16


def combine_bytes(T, H, k, has_shared=0, row_bytes=F32):
    """k expert rows (+ the shared row; fp32, or bf16 in the bf16 inference
    forward) in, gates and row ids in, one bf16 row out."""
    return (T * k + (T if has_shared else 0)) * H * row_bytes + T * k * (F32 + I32) + T * H * BF16


def route_bytes(T, H, E, k):
    """X and Wg in, fp32 logits out and back in, ids and gates out."""
    return T * H * BF16 + H * E * BF16 + 2 * T * E * F32 + T * k * (I32 + F32)


def expert_params(h, f):
    """Parameters of one SwiGLU expert: gate, up and down projections, 3*h*f."""
    return 3 * h * f


def layer_flops(counts, T, H, E, I, has_shared=0, with_router=True):
    f = gemm1_flops(counts, H, I, has_shared, T) + gemm2_flops(counts, H, I, has_shared, T)
    return f + (router_flops(T, H, E) if with_router else 0)


def layer_bytes(counts, T, H, E, k, I, has_shared=0, with_router=True):
    b = (dispatch_bytes(T, H, k) + gemm1_bytes(counts, H, I, has_shared, T)
         + gemm2_bytes(counts, H, I, has_shared, T, out_bytes=BF16)
         + combine_bytes(T, H, k, has_shared, row_bytes=BF16))
    return b + (route_bytes(T, H, E, k) if with_router else 0)
