"""Reference of the GEMM's exact-chunk plan rule (test infrastructure).

Every activation code has |q_x| <= 127, so a run of K-products over the range
R is exact in fp32 for output row o when 127 * sum_{k in R} |Q_w[o,k]| is at
most 2^24 - 1 (every partial sum is then an integer fp32 holds exactly). For
each block of 128 weight rows the plan is the longest run length L, in units
of 64 K-elements with runs starting at multiples of L, among 16 * 2^j
(shorter than K) and all of K, that satisfies the bound for every row and
run; 16 (1024 products, or all of K when it is shorter) always does.
"""
import numpy as np

LIMIT = (1 << 24) - 1


def candidates(num_kb):
    c = []
    L = 16
    while L < num_kb and len(c) < 15:
        c.append(L)
        L *= 2
    c.append(num_kb)
    return c


def max_run_sum(absq_kb, L):
    """Largest sum over runs of L K-blocks (rows of per-block |q| sums)."""
    n = absq_kb.shape[1]
    best = 0
    for s in range(0, n, L):
        best = max(best, int(absq_kb[:, s:s + L].sum(axis=1).max()))
    return best


def plan(Qw):
    N, K = Qw.shape
    num_kb = (K + 63) // 64
    out = []
    for b0 in range(0, N, 128):
        blk = np.abs(Qw[b0:b0 + 128].astype(np.int64))
        pad = num_kb * 64 - K
        if pad:
            blk = np.pad(blk, ((0, 0), (0, pad)))
        kb = blk.reshape(blk.shape[0], num_kb, 64).sum(axis=2)
        best = min(16, num_kb)
        for L in candidates(num_kb):
            if 127 * max_run_sum(kb, L) <= LIMIT:
                best = max(best, L)
        out.append(best)
    return np.array(out, dtype=np.int32)


def plan_is_safe(Qw, kchunk):
    N, K = Qw.shape
    num_kb = (K + 63) // 64
    for i, b0 in enumerate(range(0, N, 128)):
        L = int(kchunk[i]) * 64
        blk = np.abs(Qw[b0:b0 + 128].astype(np.int64))
        for s in range(0, K, L):
            if 127 * int(blk[:, s:s + L].sum(axis=1).max()) > LIMIT:
                return False
    return True
