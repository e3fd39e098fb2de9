"""Philox4x32-10, written from its published definition.

Source: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel Random Numbers: As Easy as 1, 2,
3", SC'11 -- the Philox-4x32 bijection with R = 10 rounds.

One round maps the counter (c0, c1, c2, c3) under the round key (k0, k1) to

    (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0))

with M0 = 0xD2511F53 and M1 = 0xCD9E8D57 (32x32 -> 64-bit products split into high and low words). The
key is bumped by the Weyl constants W0 = 0x9E3779B9, W1 = 0xBB67AE85 between rounds, so round r uses
(k0 + r*W0, k1 + r*W1) mod 2^32.

Test infrastructure: only tests/, the smoke check and the CPU-baseline leg of the benchmark use this
module. It shares no code with the CUDA path.
"""
from __future__ import annotations

import numpy as np

M0 = 0xD2511F53
M1 = 0xCD9E8D57
W0 = 0x9E3779B9
W1 = 0xBB67AE85
MASK32 = 0xFFFFFFFF
ROUNDS = 10


def philox4x32_10(ctr, key):
    """Scalar Philox4x32-10 on Python ints: ctr = (c0, c1, c2, c3), key = (k0, k1) -> 4 words."""
    c0, c1, c2, c3 = (int(v) & MASK32 for v in ctr)
    k0, k1 = (int(v) & MASK32 for v in key)
    for r in range(ROUNDS):
        if r:
            k0 = (k0 + W0) & MASK32
            k1 = (k1 + W1) & MASK32
        p0 = M0 * c0
        p1 = M1 * c2
        c0, c1, c2, c3 = ((p1 >> 32) ^ c1 ^ k0) & MASK32, p1 & MASK32, ((p0 >> 32) ^ c3 ^ k1) & MASK32, p0 & MASK32
    return c0, c1, c2, c3


def philox4x32_10_np(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox4x32-10 over numpy arrays (broadcast); returns four uint64 arrays < 2^32."""
    u = np.uint64
    m32 = u(MASK32)
    c0, c1, c2, c3, k0, k1 = (np.asarray(v, dtype=np.uint64) & m32 for v in (c0, c1, c2, c3, k0, k1))
    c0, c1, c2, c3, k0, k1 = np.broadcast_arrays(c0, c1, c2, c3, k0, k1)
    c0, c1, c2, c3, k0, k1 = (np.array(v, dtype=np.uint64) for v in (c0, c1, c2, c3, k0, k1))
    for r in range(ROUNDS):
        if r:
            k0 = (k0 + u(W0)) & m32
            k1 = (k1 + u(W1)) & m32
        p0 = u(M0) * c0          # < 2^64: exact in uint64
        p1 = u(M1) * c2
        n0 = ((p1 >> u(32)) ^ c1 ^ k0) & m32
        n2 = ((p0 >> u(32)) ^ c3 ^ k1) & m32
        c0, c1, c2, c3 = n0, p1 & m32, n2, p0 & m32
    return c0, c1, c2, c3


def token_words(tokens, seed: int, row_id: int, step) -> np.ndarray:
    """The 32-bit Philox output word assigned to each token index of one row.

    Counter layout (a reading: the workload fixes only "key = seed, counter = (row, step)", not how a
    token index enters the counter): key = (seed mod 2^32, seed >> 32), counter = (v >> 2, row_id,
    step mod 2^32, step >> 32), and token v takes output word v & 3, so one Philox call serves four
    consecutive tokens.

    ``step`` may be a scalar (result shaped like ``tokens``) or a 1-D array of steps (result shaped
    [len(step), len(tokens)]).
    """
    v = np.asarray(tokens, dtype=np.int64).reshape(-1)
    seed = int(seed) & ((1 << 64) - 1)
    steps = np.asarray(step, dtype=np.uint64)
    scalar = steps.ndim == 0
    steps = steps.reshape(-1, 1)
    g = (v >> 2).astype(np.uint64).reshape(1, -1)
    out = philox4x32_10_np(g, int(row_id) & MASK32, steps & np.uint64(MASK32), steps >> np.uint64(32),
                           seed & MASK32, seed >> 32)
    words = np.stack(out, axis=-1)                     # [S, N, 4]
    sel = np.take_along_axis(words, (v & 3).reshape(1, -1, 1).astype(np.int64), axis=-1)[..., 0]
    if scalar:
        return sel[0].reshape(np.shape(tokens))
    return sel
