"""Test infrastructure (not part of the product path): the reverse mode of the
KDA recurrence in its chunked (WY/UT) form, plain fp64 numpy.

The pages name the chunked form for training ("code-audit", finding
dual-kda-execution-regimes: chunked KDA for prefill and training, fused
recurrent KDA for one-token decode) and print no gradient; this is the exact
reverse mode of the chunk-level forward below, written out step by step.  It
is the reference a chunked GPU backward is checked against, and it is itself
pinned (tests/test_oracle_chunked_backward.py) by equality with the
recurrent reverse mode of kdaref.c (which finite differences pin).

Forward of one chunk of L tokens of one (sequence, head), state S (K x V) at
its start, Gam_r = g_0 + ... + g_r per channel, Gam_L = Gam_{L-1}:
    Kbar = k e^{Gam},  Ktil = k e^{-Gam},  Khat = k e^{Gam_L - Gam},
    Qbar = scale q e^{Gam}
    A_kk[r, s] = beta_r <Kbar_r, Ktil_s>   (s < r),   T = (I + A_kk)^{-1}
    W = T diag(beta) Kbar,   Ut = T diag(beta) V,   U = Ut - W S
    A_qk[r, s] = <Qbar_r, Ktil_s>   (s <= r)
    O = Qbar S + A_qk U,   S' = diag(e^{Gam_L}) S + Khat^T U
No sub-chunk references are needed in fp64 for the decays the tests use.
Parity: pinned by the recurrent reverse mode (not against the pages, which
print no gradient).
"""
import numpy as np


def _pieces(qc, kc, vc, gc, bc, scale):
    L = qc.shape[0]
    gam = np.cumsum(gc, axis=0)                 # [L, K]
    gl = gam[-1]
    kbar = kc * np.exp(gam)
    ktil = kc * np.exp(-gam)
    khat = kc * np.exp(gl[None, :] - gam)
    qbar = scale * qc * np.exp(gam)
    akk = np.tril(bc[:, None] * (kbar @ ktil.T), -1)
    T = np.linalg.inv(np.eye(L) + akk)
    bk = bc[:, None] * kbar
    bv = bc[:, None] * vc
    W = T @ bk
    Ut = T @ bv
    aqk = np.tril(qbar @ ktil.T)
    return dict(gam=gam, gl=gl, kbar=kbar, ktil=ktil, khat=khat, qbar=qbar, akk=akk, T=T,
                bk=bk, bv=bv, W=W, Ut=Ut, aqk=aqk)


def chunk_forward(qc, kc, vc, gc, bc, S, scale=1.0):
    """(O [L, V], S' [K, V]) of one chunk from its start state S."""
    p = _pieces(qc, kc, vc, gc, bc, scale)
    U = p["Ut"] - p["W"] @ S
    O = p["qbar"] @ S + p["aqk"] @ U
    S_next = np.exp(p["gl"])[:, None] * S + p["khat"].T @ U
    return O, S_next


def chunk_backward(qc, kc, vc, gc, bc, S, dO, dS_next, scale=1.0):
    """Gradients of one chunk: (dq, dk, dv, dg [L, .], dbeta [L], dS [K, V])
    given dL/dO and dL/dS' of the chunk and its start state S."""
    p = _pieces(qc, kc, vc, gc, bc, scale)
    T, W, aqk = p["T"], p["W"], p["aqk"]
    kbar, ktil, khat, qbar = p["kbar"], p["ktil"], p["khat"], p["qbar"]
    U = p["Ut"] - W @ S
    decay = np.exp(p["gl"])                                  # [K]
    L = qc.shape[0]
    # through O = Qbar S + A_qk U and S' = diag(e^{Gam_L}) S + Khat^T U
    dU = aqk.T @ dO + khat @ dS_next
    dS = qbar.T @ dO + decay[:, None] * dS_next - W.T @ dU
    daqk = np.tril(dO @ U.T)
    dqbar = dO @ S.T + daqk @ ktil
    dktil = daqk.T @ qbar
    dkhat = U @ dS_next.T
    # U = Ut - W S;  W = T Bk, Ut = T Bv
    dW = -dU @ S.T
    dT = dW @ p["bk"].T + dU @ p["bv"].T
    dbk = T.T @ dW
    dbv = T.T @ dU
    # T = (I + A_kk)^{-1}, A_kk strictly lower triangular
    dakk = np.tril(-T.T @ dT @ T.T, -1)
    # A_kk[r, s] = beta_r <Kbar_r, Ktil_s>
    kk = kbar @ ktil.T
    dbeta = np.sum(dakk * kk, axis=1)
    dkbar = bc[:, None] * (dakk @ ktil)
    dktil = dktil + (bc[:, None] * dakk).T @ kbar
    # Bk = diag(beta) Kbar, Bv = diag(beta) V
    dbeta = dbeta + np.sum(dbk * kbar, axis=1) + np.sum(dbv * vc, axis=1)
    dkbar = dkbar + bc[:, None] * dbk
    dv = bc[:, None] * dbv
    # the decay factors
    gam, gl = p["gam"], p["gl"]
    dk = dkbar * np.exp(gam) + dktil * np.exp(-gam) + dkhat * np.exp(gl[None, :] - gam)
    dq = scale * dqbar * np.exp(gam)
    dgam = dkbar * kbar - dktil * ktil - dkhat * khat + dqbar * qbar
    dgl = np.sum(dkhat * khat, axis=0) + np.sum(dS_next * (decay[:, None] * S), axis=1)
    dgam[L - 1] += dgl
    dg = np.cumsum(dgam[::-1], axis=0)[::-1]               # Gam_r = sum_{i <= r} g_i
    return dq, dk, dv, dg, dbeta, dS


def chunked_backward(q, k, v, g, beta, dO, cu_seqlens=None, scale=1.0, initial_state=None,
                     dS_final=None, chunk=64):
    """The reverse mode in chunks of ``chunk`` tokens, with the same arguments
    and results as oracle.recurrent_backward (fp64 arrays)."""
    q, k, v, g, beta, dO = (np.asarray(a, dtype=np.float64) for a in (q, k, v, g, beta, dO))
    N, H, K = q.shape
    V = v.shape[-1]
    cu = [0, N] if cu_seqlens is None else [int(c) for c in np.asarray(cu_seqlens)]
    B = len(cu) - 1
    dq, dk, dg = (np.zeros((N, H, K)) for _ in range(3))
    dv = np.zeros((N, H, V))
    dbeta = np.zeros((N, H))
    dS0 = np.zeros((B, H, K, V))
    for b in range(B):
        t0, t1 = cu[b], cu[b + 1]
        starts = list(range(t0, t1, chunk))
        for h in range(H):
            S = (np.zeros((K, V)) if initial_state is None
                 else np.asarray(initial_state, dtype=np.float64)[b, h].copy())
            states = []
            for c0 in starts:           # chunk-start states
                c1 = min(c0 + chunk, t1)
                states.append(S)
                _, S = chunk_forward(q[c0:c1, h], k[c0:c1, h], v[c0:c1, h], g[c0:c1, h],
                                     beta[c0:c1, h], S, scale)
            dS = (np.zeros((K, V)) if dS_final is None
                  else np.asarray(dS_final, dtype=np.float64)[b, h].copy())
            for c0, Sc in zip(reversed(starts), reversed(states)):
                c1 = min(c0 + chunk, t1)
                r = chunk_backward(q[c0:c1, h], k[c0:c1, h], v[c0:c1, h], g[c0:c1, h],
                                   beta[c0:c1, h], Sc, dO[c0:c1, h], dS, scale)
                dq[c0:c1, h], dk[c0:c1, h], dv[c0:c1, h], dg[c0:c1, h], dbeta[c0:c1, h] = r[:5]
                dS = r[5]
            dS0[b, h] = dS
    return dq, dk, dv, dg, dbeta, dS0
