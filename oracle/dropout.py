"""LoRA dropout: the counter-based mask and the linear layer with the dropped branch input.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Every page's LoRA configuration sets ``lora_dropout = 0.05`` (P1 tutorial
"QLoRA: fine-tuning 7B on a 24 GB card", section 3.3; tbr8.org section 4;
fedte.cc section 2).  Dropout acts on the input of the LoRA branch only: the
branch computes B A (x * m / (1 - p)) with m a 0/1 mask kept with probability
1 - p (inverted dropout, so the expectation is unchanged), and the frozen path
sees x itself.  Backpropagation through the fixed mask gives

    T  = (X * M) A^T / (1 - p)             [M, r]
    Y  = X Wdeq^T + s T B^T
    U  = dY B
    dX = dY Wdeq + s (U A) * M / (1 - p)
    dA = s U^T (X * M) / (1 - p)
    dB = s dY^T T

The mask is drawn by Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel
random numbers: as easy as 1, 2, 3", SC 2011), written here from that
definition: element e = row * k + col of an [m, k] input uses word e mod 4 of
Philox(counter = (e div 4 as two 32-bit words, offset as two 32-bit words),
key = seed as two 32-bit words); the element is kept when that word is at
least floor(p * 2^32).  The packed mask holds one bit per element: byte
(row, c) covers columns 8c .. 8c+7, bit t (least significant first) column 8c + t.
"""

from __future__ import annotations

import numpy as np

M0, M1 = 0xD2511F53, 0xCD9E8D57          # round multipliers
W0, W1 = 0x9E3779B9, 0xBB67AE85          # key increments (golden ratio, sqrt(3) - 1)
MASK32 = 0xFFFFFFFF


def philox4x32_10(ctr, key):
    """Philox4x32 with 10 rounds on arrays of counters ``ctr`` [..., 4] and keys [..., 2]
    (uint32 values held in uint64 arrays).  Returns [..., 4] uint32."""
    c = [np.asarray(ctr[..., i], dtype=np.uint64) for i in range(4)]
    k0 = np.asarray(key[..., 0], dtype=np.uint64)
    k1 = np.asarray(key[..., 1], dtype=np.uint64)
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + W0) & MASK32
            k1 = (k1 + W1) & MASK32
        p0 = np.uint64(M0) * c[0]            # full 64-bit products of two 32-bit words
        p1 = np.uint64(M1) * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(MASK32)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(MASK32)
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return np.stack([x.astype(np.uint32) for x in c], axis=-1)


def keep_threshold(p: float) -> int:
    """floor(p * 2^32): a word at or above it keeps its element."""
    if not 0.0 <= p < 1.0:
        raise ValueError("dropout probability must be in [0, 1)")
    return int(np.floor(np.float64(np.float32(p)) * 4294967296.0))


def keep_mask(seed: int, offset: int, m: int, k: int, p: float) -> np.ndarray:
    """Boolean [m, k]: True where the element is kept."""
    e = np.arange(m * k, dtype=np.uint64)
    grp = e >> np.uint64(2)
    ctr = np.stack([grp & np.uint64(MASK32), grp >> np.uint64(32),
                    np.full_like(grp, offset & MASK32), np.full_like(grp, (offset >> 32) & MASK32)], axis=-1)
    key = np.stack([np.full_like(grp, seed & MASK32), np.full_like(grp, (seed >> 32) & MASK32)], axis=-1)
    words = philox4x32_10(ctr, key)
    w = words[np.arange(m * k), (e & np.uint64(3)).astype(np.int64)]
    return (w.astype(np.uint64) >= np.uint64(keep_threshold(p))).reshape(m, k)


def pack_mask(keep: np.ndarray) -> np.ndarray:
    """uint8 [m, ceil(k/8)] with bit t of byte (row, c) = keep[row, 8c + t]."""
    keep = np.asarray(keep, dtype=bool)
    return np.packbits(keep, axis=1, bitorder="little")


def unpack_mask(packed: np.ndarray, k: int) -> np.ndarray:
    return np.unpackbits(np.asarray(packed, dtype=np.uint8), axis=1, bitorder="little", count=k).astype(bool)


def lora_forward(x, wdeq, a, b, alpha: float, r: int, keep, p: float):
    """``(Y, T)`` of the layer with dropout on the branch input (float64)."""
    x, wdeq, a, b = (np.asarray(v, dtype=np.float64) for v in (x, wdeq, a, b))
    s = float(alpha) / float(r)
    xd = x * np.asarray(keep, dtype=np.float64) / (1.0 - p)
    t = xd @ a.T
    return x @ wdeq.T + s * (t @ b.T), t


def lora_backward(dy, x, wdeq, a, b, alpha: float, r: int, keep, p: float, t=None):
    """``(dX, dA, dB)`` through the fixed mask (float64)."""
    dy, x, wdeq, a, b = (np.asarray(v, dtype=np.float64) for v in (dy, x, wdeq, a, b))
    s = float(alpha) / float(r)
    keep = np.asarray(keep, dtype=np.float64)
    xd = x * keep / (1.0 - p)
    if t is None:
        t = xd @ a.T
    u = dy @ b
    dx = dy @ wdeq + s * (u @ a) * keep / (1.0 - p)
    da = s * (u.T @ xd)
    db = s * (dy.T @ np.asarray(t, dtype=np.float64))
    return dx, da, db
