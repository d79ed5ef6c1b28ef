"""Shared test helpers: conversions and the error metrics (no method arithmetic)."""

import numpy as np
import torch


def to_np64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a float32 / bfloat16 tensor."""
    return t.detach().to("cpu").float().numpy().astype(np.float64)


def to_np32(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").float().numpy()


def rel_fro(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def max_row_rel(got, ref) -> float:
    """Largest per-row error ||got_i - ref_i|| / max(||ref_i||, rms row norm) over the rows of a 2-D array.

    A whole-tensor Frobenius norm can hide one wrong row or a wrong tail tile
    (one bad row of 2048 moves it by about 0.02); this bounds every row on its
    own.  A row whose reference nearly cancels (a one-element row of dB at
    rank 1, say) is measured against the root-mean-square row norm instead of
    its own tiny norm: a wrong row still shows an error of about one rms row.
    """
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if got.ndim == 1:
        got, ref = got[None, :], ref[None, :]
    if not ref.size:
        return 0.0
    num = np.linalg.norm(got - ref, axis=1)
    den = np.linalg.norm(ref, axis=1)
    rms = np.linalg.norm(ref) / np.sqrt(ref.shape[0])
    den = np.maximum(den, rms if rms > 0 else 1.0)
    return float((num / den).max())


def assert_close(got, ref, tol, what=""):
    """Both bounds of the GEMM parity bar: the whole tensor and every row."""
    e, er = rel_fro(got, ref), max_row_rel(got, ref)
    assert e < tol and er < tol, "%s: relative Frobenius %.3e, worst row %.3e (bound %.1e)" % (what, e, er, tol)


def t_save_tol(k: int) -> float:
    """Bound on the relative error of t_save = X A^T (bf16 operands, float32
    accumulation on the tensor cores) against the float64 product.  The
    products are exact; each of the k accumulation steps can lose up to 2^-23
    of the running sum, and for zero-mean terms the sum grows like sqrt(k)
    times a term while the error grows like k, so the relative error is of order
    sqrt(k) 2^-23 (1.2e-5 measured at k = 11008).  Four times that, and never
    below 1e-5."""
    return max(1e-5, 4.0 * (k ** 0.5) * 2.0 ** -23)


# Relative Frobenius bound for bf16-in / fp32-accumulate products against the
# float64 oracle, as the benchmark spec fixes it; applied to the whole tensor
# and to every row.
GEMM_TOL = 2e-2
