"""PSAC low-rank key compensation (oracle, test infrastructure only).

"QuantWM" (Innovations, item 3; Methodology): principal-subspace attention
compensation restores the remaining key error along the dominant subspace of
the queries with low-rank projections.  Reading:

* U [d, r] = the top-r eigenvectors of the uncentred second moment
  C = (1/n) sum_t q_t q_t^T of one head's historical queries, eigenvalues in
  descending order; each column is signed so its largest-magnitude entry is
  positive (ties to the lower index).
* each cached token stores coeff_t = fp16_rne(U^T (k_t - k_hat_t)).
* the cached logit gains  tau (U^T q) . coeff_t.

With r = d, U U^T = I and k_hat + U coeff = k up to the fp16 rounding of the
coefficients, so the compensated logits equal the unquantised ones.
"""

from __future__ import annotations

import numpy as np

F64 = np.float64


def second_moment(Qhist):
    Q = np.asarray(Qhist, F64)
    return (Q.T @ Q) / Q.shape[0]


def fix_signs(U):
    U = np.array(U, F64)
    for j in range(U.shape[1]):
        i = int(np.argmax(np.abs(U[:, j])))
        if U[i, j] < 0:
            U[:, j] = -U[:, j]
    return U


def psac_basis(Qhist, r, centred=False):
    """Top-r eigenvectors (fp64 [d, r]) of the historical-query second moment."""
    Q = np.asarray(Qhist, F64)
    if centred:
        Q = Q - Q.mean(axis=0, keepdims=True)
    C = second_moment(Q)
    w, V = np.linalg.eigh(C)               # ascending eigenvalues
    order = np.argsort(-w, kind="stable")
    return fix_signs(V[:, order[:r]]), w[order[:r]]


def psac_coeff(K, Khat, U):
    """fp16 coefficients U^T (k - k_hat) for rows of K, Khat [n, d]; U [d, r] (fp32 values)."""
    resid = np.asarray(K, F64) - np.asarray(Khat, F64)
    return (resid @ np.asarray(U, F64)).astype(np.float16)
