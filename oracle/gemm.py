"""Dequantise-then-float64 GEMM: dense, grouped contiguous, grouped masked.

Sources (page titles and sections):
  * HALOps "GEMM" API, ``dense_gemm``: output = input @ weight^T + bias, BF16
    output written in place; alpha float32 [1] (required for w4a4-nvfp4), bias
    [N] BF16 (w8a8-mxfp8 only).
  * HALOps "GEMM" API, ``batch_gemm``: output[b] = input[b] @ weight[b]^T with a
    per-batch alpha [B] and bias [B, N].
  * HALOps "GEMM" API, ``group_masked_gemm``: input [E * max_m, K], weight
    [E, N, K]; masked_m[e] valid rows per expert, padded rows are skipped.
  * cuDNN frontend "Grouped GEMM + dGLU (SM100)", Tensors/layouts and Step 1:
    groups contiguous in M, described by padded_offsets (cumulative 256-aligned
    group ends, valid_m = padded_offsets[-1]); ref[m, n] = alpha_g-scaled
    sum_k dequantize(A[m, k]) * dequantize(B[n, k, g]).

Readings (also listed in the design notes):
  G1  dequantize(x) = element value * scale value; the sum is taken in float64
      by a library matmul over the dequantised matrices; the output is
      compared with the unrounded float64 value.
  G2  alpha multiplies the sum once (alpha * sum + bias); a missing alpha is 1,
      a missing bias is 0.
  G3  Contiguous groups: every row in [0, off[L-1]) belongs to the group g with
      off[g-1] <= row < off[g] (off[-1] = 0), including the zero pad rows a
      group carries up to its 256-aligned end; rows >= off[L-1] are not
      written.
  G4  Masked groups: rows e*max_m + i with i < min(masked_m[e], max_m) are
      written; every other row is left untouched.
  G5  Error bound for a GPU result y against ref (per element):
      |y - ref| <= 2^-8 |ref| + 2^-20 |alpha_g| sum_k |a_k b_k|.
"""

import numpy as np


def _alpha_bias(alpha, bias, n_groups, n):
    a = np.ones(n_groups) if alpha is None else np.asarray(alpha, dtype=np.float64).reshape(n_groups)
    b = np.zeros((n_groups, n)) if bias is None else np.asarray(bias, dtype=np.float64).reshape(n_groups, n)
    return a, b


def dense(a_deq, b_deq, alpha=None, bias=None):
    """ref = alpha * (A @ B^T) + bias and the bound term |alpha| * (|A| @ |B|^T).

    a_deq [M, K] and b_deq [N, K] are float64 dequantised operands.
    """
    a_deq = np.asarray(a_deq, dtype=np.float64)
    b_deq = np.asarray(b_deq, dtype=np.float64)
    al, bi = _alpha_bias(alpha, bias, 1, b_deq.shape[0])
    ref = al[0] * (a_deq @ b_deq.T) + bi[0][None, :]
    mag = abs(al[0]) * (np.abs(a_deq) @ np.abs(b_deq).T)
    return ref, mag


def group_of_rows_contig(padded_offsets, m_rows):
    """Group index of each row under G3 (-1 for rows >= off[L-1])."""
    off = np.asarray(padded_offsets, dtype=np.int64)
    rows = np.arange(m_rows)
    g = np.searchsorted(off, rows, side="right")  # first g with off[g] > row
    return np.where(rows < (off[-1] if len(off) else 0), g, -1)


def grouped_contig(a_deq, b_deq, padded_offsets, alpha=None, bias=None):
    """Contiguous grouped GEMM under G3.

    a_deq [M, K]; b_deq [L, N, K]; returns (ref [M, N], mag [M, N], written [M])
    where rows with written == False keep whatever the output held before.
    """
    a_deq = np.asarray(a_deq, dtype=np.float64)
    b_deq = np.asarray(b_deq, dtype=np.float64)
    L, N, _ = b_deq.shape
    M = a_deq.shape[0]
    al, bi = _alpha_bias(alpha, bias, L, N)
    grp = group_of_rows_contig(padded_offsets, M)
    ref = np.zeros((M, N))
    mag = np.zeros((M, N))
    for g in range(L):
        rows = np.nonzero(grp == g)[0]
        if rows.size == 0:
            continue
        ref[rows] = al[g] * (a_deq[rows] @ b_deq[g].T) + bi[g][None, :]
        mag[rows] = abs(al[g]) * (np.abs(a_deq[rows]) @ np.abs(b_deq[g]).T)
    return ref, mag, grp >= 0


def grouped_rows(a_deq, b_deq, expert_ids, alpha=None, bias=None):
    """Contiguous grouped GEMM with a per-row expert index (HALOps
    group_contiguous_gemm: "expert_ids maps each token row to its expert",
    groups packed without per-expert padding).

    Reading G6: a row whose id lies outside [0, L), or that breaks the
    non-decreasing order the page requires (its id is below the id of the row
    before it, whatever that id is), is not written.  Returns (ref [M, N], mag [M, N], written [M]).
    """
    a_deq = np.asarray(a_deq, dtype=np.float64)
    b_deq = np.asarray(b_deq, dtype=np.float64)
    L, N, _ = b_deq.shape
    ids = np.asarray(expert_ids, dtype=np.int64)
    M = a_deq.shape[0]
    al, bi = _alpha_bias(alpha, bias, L, N)
    ref = np.zeros((M, N))
    mag = np.zeros((M, N))
    written = np.zeros(M, dtype=bool)
    for m in range(M):
        g = int(ids[m])
        if g < 0 or g >= L or (m > 0 and g < ids[m - 1]):
            continue
        ref[m] = al[g] * (b_deq[g] @ a_deq[m]) + bi[g]
        mag[m] = abs(al[g]) * (np.abs(b_deq[g]) @ np.abs(a_deq[m]))
        written[m] = True
    return ref, mag, written


def grouped_masked(a_deq, b_deq, masked_m, max_m, alpha=None, bias=None):
    """Masked grouped GEMM under G4.

    a_deq [E * max_m, K]; b_deq [E, N, K]; returns (ref, mag, written [E*max_m]).
    """
    a_deq = np.asarray(a_deq, dtype=np.float64)
    b_deq = np.asarray(b_deq, dtype=np.float64)
    E, N, _ = b_deq.shape
    al, bi = _alpha_bias(alpha, bias, E, N)
    ref = np.zeros((E * max_m, N))
    mag = np.zeros((E * max_m, N))
    written = np.zeros(E * max_m, dtype=bool)
    for e in range(E):
        cnt = min(int(masked_m[e]), max_m)
        if cnt <= 0:
            continue
        rows = np.arange(e * max_m, e * max_m + cnt)
        ref[rows] = al[e] * (a_deq[rows] @ b_deq[e].T) + bi[e][None, :]
        mag[rows] = abs(al[e]) * (np.abs(a_deq[rows]) @ np.abs(b_deq[e]).T)
        written[rows] = True
    return ref, mag, written


def within_bound(y, ref, mag, rel=2.0 ** -8, acc=2.0 ** -20):
    """Element-wise check of G5; returns (ok mask, excess ratio)."""
    y = np.asarray(y, dtype=np.float64)
    tol = rel * np.abs(ref) + acc * mag
    err = np.abs(y - ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(tol > 0, err / tol, np.where(err > 0, np.inf, 0.0))
    return err <= tol, ratio
