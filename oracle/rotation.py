"""Rotation construction R = U · (H_d / sqrt(d)) · P_br, in fp64.

Test infrastructure only (see the package docstring).

[OSCAR news] "OSCARの違い": the key basis U_Q is the eigenbasis of the query
covariance C_Q = (1/N) Σ_n q_nᵀ q_n; the value basis U_S is the eigenbasis of
the score-weighted value covariance C_S = (1/N) Vᵀ Sᵀ S V; the composite
rotations are R_K = U_Q · H_Had · P_br and R_V = U_S · H_Had · P_br, where U
aligns channels with attention importance, the Hadamard factor equalises
importance across channels and the bit-reversal permutation P_br spreads each
importance level across the quantisation groups.

[Escha log] part 2, fix 3: the calibration-free rotation is the Sylvester
Hadamard matrix divided by sqrt(head_dim), built by repeated doubling
[[h, h], [h, -h]], identical in every layer.

Readings where the pages are silent:
* row-vector convention: a head vector x is rotated as x · R, so that
  (q R)(k R)ᵀ = q kᵀ for orthogonal R;
* the Hadamard factor has the full size d (the page builds it at head_dim);
* eigenvectors are ordered by descending eigenvalue, and each is signed so
  that its entry of largest magnitude is positive (lowest index on a tie);
* P_br acts on columns: (x · P_br)[j] = x[bitrev(j)], bitrev over log2(d) bits;
* the 1/N normalisation of a covariance does not change its eigenvectors.
"""

import numpy as np


def hadamard(n):
    """Sylvester Hadamard matrix of order n (a power of two), entries ±1, fp64.

    Built by the doubling construction of [Escha log] fix 3: start from [[1]]
    and replace h by [[h, h], [h, -h]] until the order reaches n.
    """
    if n < 1 or (n & (n - 1)) != 0:
        raise ValueError("Hadamard order must be a power of two")
    h = np.ones((1, 1), dtype=np.float64)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def bitrev_indices(d):
    """bitrev(j) for j in [0, d): j's log2(d)-bit binary representation reversed."""
    if d < 1 or (d & (d - 1)) != 0:
        raise ValueError("d must be a power of two")
    nbits = d.bit_length() - 1
    out = np.zeros(d, dtype=np.int64)
    for j in range(d):
        r = 0
        for b in range(nbits):
            if j & (1 << b):
                r |= 1 << (nbits - 1 - b)
        out[j] = r
    return out


def eig_desc(C):
    """Eigen-decomposition of a symmetric matrix, descending, sign-canonical.

    Returns (w, U) with C = U diag(w) Uᵀ, w[0] >= w[1] >= ..., and every
    column of U signed so that its largest-magnitude entry is positive (the
    lowest row index wins a tie in magnitude).  [OSCAR news] "OSCARの違い":
    U_Q / U_S are the eigenvectors of the covariance.
    """
    C = np.asarray(C, dtype=np.float64)
    if C.ndim != 2 or C.shape[0] != C.shape[1]:
        raise ValueError("covariance must be square")
    Cs = 0.5 * (C + C.T)
    w, U = np.linalg.eigh(Cs)
    order = np.argsort(-w, kind="stable")
    w = w[order]
    U = U[:, order].copy()
    for j in range(U.shape[1]):
        col = U[:, j]
        i = int(np.argmax(np.abs(col)))  # argmax returns the lowest index on ties
        if col[i] < 0:
            U[:, j] = -col
    return w, U


def block_hadamard(d, block):
    """The d×d block-diagonal matrix with d/block copies of H_block / sqrt(block).

    block = d gives the full normalised Hadamard.  [OSCAR news] "OSCARの違い"
    names the Hadamard factor without a size; a block smaller than d confines
    the mixing to channels of similar importance (consecutive eigen-directions),
    which is the case in which P_br's spreading of each importance level over
    the quantisation groups matters.
    """
    if block < 1 or (block & (block - 1)) != 0 or d % block != 0:
        raise ValueError("block must be a power of two dividing d")
    Hb = hadamard(block) / np.sqrt(block)
    M = np.zeros((d, d))
    for i in range(d // block):
        M[i * block:(i + 1) * block, i * block:(i + 1) * block] = Hb
    return M


def build_rotation(C, d, use_bitrev=True, hadamard_block=None):
    """R = U · H · P_br in fp64 (row-vector convention x · R), with H the
    normalised Hadamard of size d, or block-diagonal with blocks of
    hadamard_block (block_hadamard).

    C is the d×d covariance (C_Q for keys, C_S for values) or None for the
    calibration-free rotation U = I of [Escha log] fix 3.  With
    use_bitrev=False the permutation is left out, so cov=None gives exactly
    the page's Hadamard / sqrt(head_dim).
    Returns (R, w) where w are the descending eigenvalues (None when C is None).
    """
    if C is None:
        U = np.eye(d)
        w = None
    else:
        C = np.asarray(C, dtype=np.float64)
        if C.shape != (d, d):
            raise ValueError("covariance shape must be (d, d)")
        w, U = eig_desc(C)
    block = d if hadamard_block is None else int(hadamard_block)
    M = U @ block_hadamard(d, block)
    if use_bitrev:
        M = M[:, bitrev_indices(d)]  # column j takes column bitrev(j)
    return M, w


def covariance(X):
    """C = (1/N) Σ_n x_nᵀ x_n for the rows x_n of X (N×d), fp64.

    [OSCAR news] "OSCARの違い": the empirical query covariance C_Q.
    """
    X = np.asarray(X, dtype=np.float64)
    return X.T @ X / X.shape[0]


def value_covariance(S, V):
    """C_S = (1/N) Vᵀ Sᵀ S V with S the N×M attention-score matrix, V M×d.

    [OSCAR news] "OSCARの違い": the score-weighted value covariance.  N is the
    number of calibration query rows of S (the normalisation does not change
    the eigenvectors).
    """
    S = np.asarray(S, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    SV = S @ V
    return SV.T @ SV / S.shape[0]
